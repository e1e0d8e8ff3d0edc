// Split-K form of the CTA-pair GEMM for launches whose output tiles are too few to fill the
// chip (the row-parallel GEMMs of a small layer: T = 2048 tokens, h = 3072 gives 96 tiles of
// 256 x 256, 1.26 rounds on 76 CTA pairs, each with a 192-block K-loop).
//
// A thread-block cluster holds S CTA pairs (2S CTAs) that share one output tile at a time. Pair
// p runs the p-th of S contiguous parts of the tile's K range, which for a row-parallel GEMM is
// the shard-ordered range: pair p owns a group of consecutive shards (a whole group when S
// divides the shard count). The S fp32 partial tiles are then summed on chip in ascending pair
// order, (P_0 + P_1) + P_2 ..., chunk by chunk: pair p receives the running sum of pairs
// 0..p-1 in its shared memory, adds its own TMEM accumulator, and sends the sum on to pair
// p + 1 with st.async remote stores whose byte count completes the receiver's mbarrier; the
// last pair converts to bf16 and stores the tile with TMA. This is the method's g (or f) sum
// done between SMs, through distributed shared memory instead of an all-reduce.
//
// Everything else follows the single-pair kernel in mptp_gemm.cuh (warp roles, ring of TMA
// stages, double-buffered TMEM accumulators, bounded waits with abort): only the cluster
// geometry (pair p = CTA ranks 2p, 2p+1; commits multicast to its two ranks) and the epilogue
// differ. Store epilogue only; four epilogue warps.
#pragma once

#include "mptp_gemm.cuh"

namespace mptp {

constexpr int SPLIT_NE = 4;
constexpr int XCH_BYTES_PER_WARP = 32 * 32 * 4;  // one fp32 chunk: 32 rows x 32 columns

// Remote store of 16 bytes into the shared memory of another CTA of the cluster; the byte count
// completes on the receiver's mbarrier (both are shared::cluster addresses).
__device__ __forceinline__ void st_async_v4(uint32_t addr, uint4 v, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
                 : "memory");
}
// Arrive on a barrier of another CTA of the cluster, ordering this thread's earlier shared-memory
// reads before it at cluster scope.
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait on a barrier that another CTA of the cluster arrives on.
__device__ __forceinline__ bool wait_bounded_cluster(uint64_t* bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait_acq_cluster(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.budget_ns) {
            if (c.status) atomicOr(c.status, DEV_TIMEOUT);
            *c.abort_flag = 1u;
            return false;
        }
    }
}

template <int BN_, int S_>
struct SplitCfg {
    static constexpr int BN = BN_;
    static constexpr int S = S_;                 // CTA pairs per cluster
    static constexpr int BNH = BN / 2;
    static constexpr int NE = SPLIT_NE;
    static constexpr int NUM_THREADS = 64 + 32 * NE;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BNH * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = BN <= 128 ? 256 : 512;
    static constexpr int STG_BYTES = NE * STG_BYTES_PER_WARP;
    static constexpr int XCH_BYTES = NE * XCH_BYTES_PER_WARP;
    static constexpr int MAX_STAGES = 8;
    static constexpr int FIT_STAGES = static_cast<int>((SMEM_LIMIT - 1024 - 768 - STG_BYTES - XCH_BYTES) / STAGE_BYTES);
    static constexpr int STAGES = FIT_STAGES < MAX_STAGES ? FIT_STAGES : MAX_STAGES;
    // full, empty per stage; tmem full x2, tmem empty x2, drain; per epilogue warp: received, free
    static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * NE;
    static constexpr size_t SMEM_BYTES =
        1024 + size_t(STAGES) * STAGE_BYTES + STG_BYTES + XCH_BYTES + 8 * NUM_BARS + 16;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory per block");
    static_assert(STAGES >= 4, "pipeline depth");
    static_assert(S >= 2 && 2 * S <= 8, "CTA pairs per cluster (portable cluster size)");
    static_assert(BN % 32 == 0 && BN <= 256, "pair tile width");
};

// Parts of a K range [kb_begin, kb_end) split over S pairs: pair p runs [lo, hi).
__host__ __device__ inline void split_range(int kb_begin, int kb_end, int S, int p, int& lo, int& hi) {
    const int L = kb_end - kb_begin;
    lo = kb_begin + (L * p) / S;
    hi = kb_begin + (L * (p + 1)) / S;
}

template <int BN, int S>
__global__ void __launch_bounds__(SplitCfg<BN, S>::NUM_THREADS, 1)
    gemm_split_kernel(const __grid_constant__ TmapSet maps, const GemmArgs args) {
    using Cfg = SplitCfg<BN, S>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int BNH = Cfg::BNH;
    constexpr int NE = Cfg::NE;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t* stg_base = smem + STAGES * Cfg::STAGE_BYTES;
    uint8_t* xch_base = stg_base + Cfg::STG_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(xch_base + Cfg::XCH_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tfull_bar = bars + 2 * STAGES;
    uint64_t* tempty_bar = bars + 2 * STAGES + 2;
    uint64_t* drain_bar = bars + 2 * STAGES + 4;
    uint64_t* recv_bar = bars + 2 * STAGES + 5;       // [NE]: the previous pair's chunk has landed
    uint64_t* free_bar = recv_bar + NE;                // [NE]: the next pair has consumed our last chunk
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t pr = rank & 1u;         // rank in the CTA pair
    const int pc = static_cast<int>(rank >> 1);  // pair in the cluster: its part of the K range
    const uint32_t base = rank & ~1u;      // the pair's leader
    const bool leader = (pr == 0);
    const uint16_t pair_mask = static_cast<uint16_t>(0x3u << base);
    const int cl = static_cast<int>(blockIdx.x) / (2 * S);
    const int num_cl = static_cast<int>(gridDim.x) / (2 * S);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 2);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 2 * NE);
        }
        mbar_init(drain_bar, 1);
        for (int e = 0; e < NE; ++e) {
            mbar_init(&recv_bar[e], 1);  // the receiver's own expect_tx arrival; the bytes complete it
            mbar_init(&free_bar[e], 1);  // one arrival from the receiving warp
        }
        *abort_flag = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&maps.a);
        prefetch_tensormap(&maps.b);
        if (pc == S - 1) prefetch_tensormap(&maps.o0);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // every CTA's barriers exist before any cross-CTA arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{args.status, abort_flag, args.budget_ns};
    grid_dependency_wait();
    grid_launch_dependents();

    const ProbInfo& p = args.pr;
    int k_lo, k_hi;
    split_range(p.kb_begin, p.kb_end, S, pc, k_lo, k_hi);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (every CTA) ----------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const CUtensorMap* tmA = &maps.a;
            const CUtensorMap* tmB = &maps.b;
            for (int u = cl; u < p.num_units && ok; u += num_cl) {
                int m_blk, ucol;
                decode_unit(p, u, m_blk, ucol);
                const int arow = m_blk * 2 * BM + static_cast<int>(pr) * BM;
                const int bcol = ucol * BN + static_cast<int>(pr) * BNH;
                for (int kb = k_lo; kb < k_hi; ++kb) {
                    if (!wait_bounded(&empty_bar[stage], phase ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[stage]), base);
                    mbar_arrive_expect_tx_cluster(full_leader, Cfg::STAGE_BYTES);
                    uint8_t* a_dst = sA + stage * Cfg::A_BYTES;
                    uint8_t* b_dst = sB + stage * Cfg::B_BYTES;
                    if (p.a_mn == 2) {
                        tma_load_3d_pair(a_dst, tmA, full_leader, 0, kb * BK, arow / 64);
                    } else if (p.a_mn) {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d_pair(a_dst + j * 8192, tmA, full_leader, arow + j * 64, kb * BK);
                    } else {
                        tma_load_2d_pair(a_dst, tmA, full_leader, kb * BK, arow);
                    }
                    if (p.b_mn == 2) {
                        tma_load_3d_pair(b_dst, tmB, full_leader, 0, kb * BK, bcol / 64);
                    } else if (p.b_mn) {
#pragma unroll
                        for (int j = 0; j < BNH / 64; ++j)
                            tma_load_2d_pair(b_dst + j * 8192, tmB, full_leader, bcol + j * 64, kb * BK);
                    } else {
                        tma_load_2d_pair(b_dst, tmB, full_leader, kb * BK, bcol);
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // ---------------- MMA issuer (each pair's leader) ----------------
            auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
                const bool got = mbar_test_wait(bar, parity) || wait_bounded(bar, parity, ctl);
                return __all_sync(0xffffffffu, got) != 0;
            };
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tcount = 0;
            bool ok = true;
            const bool a_mn = p.a_mn != 0, b_mn = p.b_mn != 0;
            const uint32_t idesc = make_idesc_bf16(2 * BM, BN, a_mn, b_mn);
            const uint32_t a_lbo = a_mn ? 8192u : 16u, b_lbo = b_mn ? 8192u : 16u;
            const uint64_t a_kstep = a_mn ? (2048u >> 4) : (32u >> 4);
            const uint64_t b_kstep = b_mn ? (2048u >> 4) : (32u >> 4);
            const uint64_t ad_base = make_sdesc_sw128(smem_u32(sA), a_lbo, 1024);
            const uint64_t bd_base = make_sdesc_sw128(smem_u32(sB), b_lbo, 1024);
            for (int u = cl; u < p.num_units && ok; u += num_cl, ++tcount) {
                const uint32_t buf = tcount & 1u;
                const uint32_t tph = (tcount >> 1) & 1u;
                if (!wait_all(&tempty_bar[buf], tph ^ 1u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                for (int kb = k_lo; kb < k_hi; ++kb) {
                    if (!wait_all(&full_bar[stage], phase)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad0 = ad_base + static_cast<uint64_t>(stage) * (Cfg::A_BYTES >> 4);
                    const uint64_t bd0 = bd_base + static_cast<uint64_t>(stage) * (Cfg::B_BYTES >> 4);
                    umma_bf16_pair_elect(d_tmem, ad0, bd0, idesc, kb > k_lo ? 1u : 0u);
#pragma unroll
                    for (int k = 1; k < BK / UMMA_K; ++k)
                        umma_bf16_pair_acc_elect(d_tmem, ad0 + k * a_kstep, bd0 + k * b_kstep, idesc);
                    umma_commit_pair_multicast_elect(&empty_bar[stage], pair_mask);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair_multicast_elect(&tfull_bar[buf], pair_mask);
            }
            umma_commit_pair_elect(drain_bar);
            wait_drain(drain_bar, 0, args.status);
        }
    } else {
        // ---------------- epilogue (NE warps, every CTA) ----------------
        // Per 32-column chunk: this pair's fp32 partial from TMEM; plus the running sum of the
        // pairs before it (received in this warp's exchange buffer); then either sent on to the
        // next pair (same rank in its pair, same warp) or, in the last pair, stored as bf16.
        constexpr int CHUNKS = BN / 32;
        const int e = warp - 2;
        const int q = warp & 3;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* stg = stg_base + e * STG_BYTES_PER_WARP;
        // Row `lane` of the exchange chunk: 128 bytes, 16-byte piece j at slot (j + lane) % 8.
        uint8_t* xrow = xch_base + e * XCH_BYTES_PER_WARP + lane * 128;
        const bool has_prev = pc > 0, has_next = pc < S - 1;
        // The same buffer and barriers in the next pair's CTA of this rank, and the free barrier in
        // the previous pair's (only ranks inside the cluster are mapped).
        const uint32_t xrow_next = has_next ? mapa_shared(smem_u32(xrow), rank + 2) : 0u;
        const uint32_t recv_next = has_next ? mapa_shared(smem_u32(&recv_bar[e]), rank + 2) : 0u;
        const uint32_t free_prev = has_prev ? mapa_shared(smem_u32(&free_bar[e]), rank - 2) : 0u;
        int sbuf = 0;
        uint32_t tcount = 0, xr = 0, xs = 0;  // tiles; chunks received; chunks sent
        bool ok = true;
        for (int u = cl; u < p.num_units && ok; u += num_cl, ++tcount) {
            int m_blk, ucol;
            decode_unit(p, u, m_blk, ucol);
            const int row0 = m_blk * 2 * BM + static_cast<int>(pr) * BM + q * 32;
            const uint32_t buf = tcount & 1u;
            const uint32_t tph = (tcount >> 1) & 1u;
            bool got = true;
            if (lane == 0) got = wait_bounded(&tfull_bar[buf], tph, ctl);
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r[32];
#pragma unroll 1
            for (int cc = 0; cc < CHUNKS && ok; ++cc) {
                tmem_ld32(tmem_base + lane_addr + buf * BN + cc * 32, r);
                tmem_ld_wait(r);
                if (cc == CHUNKS - 1) {  // accumulator drained: hand it back to the pair's MMA
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[buf]), base));
                }
                if (has_prev) {
                    if (lane == 0) mbar_arrive_expect_tx(&recv_bar[e], XCH_BYTES_PER_WARP);
                    bool rg = wait_bounded_cluster(&recv_bar[e], xr & 1u, ctl);
                    ++xr;
                    if (__all_sync(0xffffffffu, rg) == 0) {
                        ok = false;
                        break;
                    }
                    // running sum of the pairs before this one, then this pair's partial
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint4 v = *reinterpret_cast<const uint4*>(xrow + (((j + lane) & 7) << 4));
                        r[4 * j + 0] = __float_as_uint(__uint_as_float(v.x) + __uint_as_float(r[4 * j + 0]));
                        r[4 * j + 1] = __float_as_uint(__uint_as_float(v.y) + __uint_as_float(r[4 * j + 1]));
                        r[4 * j + 2] = __float_as_uint(__uint_as_float(v.z) + __uint_as_float(r[4 * j + 2]));
                        r[4 * j + 3] = __float_as_uint(__uint_as_float(v.w) + __uint_as_float(r[4 * j + 3]));
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive_release_cluster(free_prev);  // the buffer may be refilled
                }
                if (has_next) {
                    bool fg = true;
                    if (lane == 0) fg = wait_bounded_cluster(&free_bar[e], (xs & 1u) ^ 1u, ctl);
                    ++xs;
                    if (__shfl_sync(0xffffffffu, fg ? 1 : 0, 0) == 0) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_async_v4(xrow_next + (((j + lane) & 7) << 4),
                                    make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]), recv_next);
                } else {
                    const int col0 = ucol * BN + cc * 32;
                    if (col0 < p.N) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                        stage_and_store(&maps.o0, stg, sbuf, lane, pk, col0, row0);
                    }
                }
            }
        }
        if (!has_next && lane == 0) bulk_wait_group<0>();
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) spin_ns(ABORT_SETTLE_NS);
        __syncthreads();
    }
    cluster_sync_all();  // every remote store into this CTA and every MMA reading it are done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int BN, int S>
inline void split_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int clusters, cudaStream_t stream) {
    using Cfg = SplitCfg<BN, S>;
    cfg->gridDim = dim3(2 * S * clusters, 1, 1);
    cfg->blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
    cfg->dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2 * S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg->attrs = attr;
    cfg->numAttrs = 2;
}

// Clusters of S pairs that can be resident at once (0 if the kernel cannot run as such).
template <int BN, int S>
inline int resident_split_clusters(int num_sms) {
    using Cfg = SplitCfg<BN, S>;
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev] != 0) return cached[dev] > 0 ? cached[dev] : 0;
    auto kern = gemm_split_kernel<BN, S>;
    int clusters = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::SMEM_BYTES)) ==
        cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[2];
        split_config<BN, S>(&cfg, attr, num_sms / (2 * S), nullptr);
        cfg.numAttrs = 1;  // the cluster shape only
        if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) clusters = 0;
    }
    cudaGetLastError();
    if (clusters > num_sms / (2 * S)) clusters = num_sms / (2 * S);
    if (dev >= 0 && dev < 64) cached[dev] = clusters > 0 ? clusters : -1;
    return clusters > 0 ? clusters : 0;
}

template <int BN, int S>
inline cudaError_t launch_gemm_split(const TmapSet& maps, const GemmArgs& args, int num_sms, cudaStream_t stream) {
    using Cfg = SplitCfg<BN, S>;
    auto kern = gemm_split_kernel<BN, S>;
    if (args.pr.b_mn && (BN % 128 != 0 || (args.pr.b_mn == 2 && BN != 256))) return cudaErrorInvalidValue;
    const int resident = resident_split_clusters<BN, S>(num_sms);
    if (resident <= 0) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    int use = args.pr.num_units < resident ? args.pr.num_units : resident;
    if (use > 0) {  // as few clusters as give the same number of rounds
        const int rounds = (args.pr.num_units + use - 1) / use;
        use = (args.pr.num_units + rounds - 1) / rounds;
    }
    if (use <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[2];
    split_config<BN, S>(&cfg, attr, use, stream);
    e = cudaLaunchKernelEx(&cfg, kern, maps, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mptp
