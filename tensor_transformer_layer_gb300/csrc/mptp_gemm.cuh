// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues.
//
//   C[M, N] = sum_k  A(m, k) * B(k, n),   bf16 inputs, fp32 accumulation in TMEM.
//
// One CTA per SM (grid = min(work units, SMs)); 192 threads:
//   warp 0      TMA producer (one elected lane): 128x64 A tile + BNx64 B tile per
//               stage into a STAGES-deep shared-memory ring, 128-byte swizzle.
//   warp 1      TMEM allocator (whole warp) and MMA issuer (one lane): 4 x
//               tcgen05.mma (M=128, N=BN, K=16) per stage into one of two TMEM
//               accumulators (double buffer: 2*BN fp32 columns).
//   warps 2..5  epilogue: tcgen05.ld 32 rows x 32 columns per warp (TMEM lane
//               quarter = warp % 4, thread = output row), fused math, bf16 store
//               or cross-entropy partials. Runs while the MMA fills the other
//               accumulator.
//
// A work unit is one 128-row block and `tiles_per_unit` consecutive BN-wide
// column tiles (1 for plain GEMMs; several for the cross-entropy, whose epilogue
// keeps running per-row statistics over the unit). The K-loop runs over K
// blocks [kb_begin, kb_end) in ascending order, so a K range that covers shards
// 0..t-1 of a row-parallel GEMM sums the shard partials in shard order inside
// the accumulator: the g / f all-reduce of the method becomes the K-loop.
//
// Operand majorness: K-major = K contiguous in global memory (row-major [rows, K]),
// MN-major = M (or N) contiguous (row-major [K, rows]); both are loaded by TMA
// with the 128-byte swizzle and described to the MMA without any transpose copy.
//
// Every mbarrier wait is bounded by a time budget; on expiry the kernel sets
// MP_DEV_TIMEOUT in the status word, raises a CTA-wide abort flag, waits (with a
// fixed bound) for its own TMA loads and MMAs in flight, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>

#include "mptp_ptx.cuh"

namespace mptp {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int NUM_THREADS = 192;
constexpr int NUM_EPI_WARPS = 4;
constexpr uint32_t DEV_TIMEOUT = 0x1u;
constexpr uint32_t DEV_TARGET_RANGE = 0x2u;
constexpr unsigned long long DRAIN_BUDGET_NS = 1000000000ull;  // 1 s

enum EpiKind : int {
    EPI_STORE = 0,  // out0 = bf16(acc)
    EPI_GELU = 1,   // out0 = bf16(GeLU(acc)); out1 (nullable) = bf16(acc)
    EPI_DGELU = 2,  // out0 = bf16(acc * GeLU'(aux)), aux = bf16 U
    EPI_CE = 3,     // per-row online max / sum-exp / target logit over the unit
};

struct GemmArgs {
    int M, N;                 // output extent (masking of the ragged tails)
    int num_m_blocks;         // ceil(M / BM)
    int num_units;            // num_m_blocks * unit columns
    int tiles_per_unit;       // BN-wide column tiles per unit
    int kb_begin, kb_end;     // K blocks (of BK) to accumulate, ascending
    __nv_bfloat16* out0;
    long long ld0;
    __nv_bfloat16* out1;
    long long ld1;
    const __nv_bfloat16* aux;
    long long ld_aux;
    // cross-entropy epilogue
    const int32_t* target;
    float* ws;                // [P][3][M] fp32: max, sum-exp, target logit
    int v_valid;
    uint32_t* status;         // nullable
    unsigned long long budget_ns;
};

template <int BN_>
struct GemmCfg {
    static constexpr int BN = BN_;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = (BN == 256) ? 4 : 6;
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tmem full x2, tmem empty x2, drain
    static constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + 8 * NUM_BARS + 16;
};

struct Ctl {
    uint32_t* status;
    volatile uint32_t* abort_flag;
    unsigned long long budget_ns;
};

// Bounded wait. false = gave up (budget spent or another role aborted).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const Ctl& c) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.budget_ns) {
            if (c.status) atomicOr(c.status, DEV_TIMEOUT);
            *c.abort_flag = 1u;
            return false;
        }
    }
}

// Teardown wait with a fixed bound, independent of the abort flag.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > DRAIN_BUDGET_NS) {
            if (status) atomicOr(status, DEV_TIMEOUT);
            return;
        }
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float gelu_f(float u) {
    return 0.5f * u * (1.0f + erff(u * 0.70710678118654752f));
}

__device__ __forceinline__ float gelu_prime_f(float u) {
    const float cdf = 0.5f * (1.0f + erff(u * 0.70710678118654752f));
    const float pdf = 0.39894228040143268f * expf(-0.5f * u * u);
    return cdf + u * pdf;
}

__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&p)[16]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
    d[0] = make_uint4(p[0], p[1], p[2], p[3]);
    d[1] = make_uint4(p[4], p[5], p[6], p[7]);
    d[2] = make_uint4(p[8], p[9], p[10], p[11]);
    d[3] = make_uint4(p[12], p[13], p[14], p[15]);
}

template <int BN, bool A_MN, bool B_MN, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmArgs args) {
    using Cfg = GemmCfg<BN>;
    constexpr int STAGES = Cfg::STAGES;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * Cfg::STAGE_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tfull_bar = bars + 2 * STAGES;
    uint64_t* tempty_bar = bars + 2 * STAGES + 2;
    uint64_t* drain_bar = bars + 2 * STAGES + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], NUM_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{args.status, abort_flag, args.budget_ns};

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_mask = 0, issued_parity = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                const int m_blk = u % args.num_m_blocks;
                const int n_blk0 = (u / args.num_m_blocks) * args.tiles_per_unit;
                for (int nt = 0; nt < args.tiles_per_unit && ok; ++nt) {
                    const int n_blk = n_blk0 + nt;
                    for (int kb = args.kb_begin; kb < args.kb_end; ++kb) {
                        if (!wait_bounded(&empty_bar[stage], phase ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full_bar[stage], Cfg::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * Cfg::A_BYTES;
                        uint8_t* b_dst = sB + stage * Cfg::B_BYTES;
                        if (A_MN) {
#pragma unroll
                            for (int j = 0; j < BM / 64; ++j)
                                tma_load_2d(a_dst + j * 8192, &tmA, &full_bar[stage], m_blk * BM + j * 64, kb * BK);
                        } else {
                            tma_load_2d(a_dst, &tmA, &full_bar[stage], kb * BK, m_blk * BM);
                        }
                        if (B_MN) {
#pragma unroll
                            for (int j = 0; j < BN / 64; ++j)
                                tma_load_2d(b_dst + j * 8192, &tmB, &full_bar[stage], n_blk * BN + j * 64, kb * BK);
                        } else {
                            tma_load_2d(b_dst, &tmB, &full_bar[stage], kb * BK, n_blk * BN);
                        }
                        issued_mask |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // No TMA load of ours may still be landing when the CTA exits.
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s)) wait_drain(&full_bar[s], (issued_parity >> s) & 1u, args.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t IDESC = make_idesc_bf16(BM, BN, A_MN, B_MN);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tcount = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
                for (int nt = 0; nt < args.tiles_per_unit && ok; ++nt, ++tcount) {
                    const uint32_t buf = tcount & 1u;
                    const uint32_t tph = (tcount >> 1) & 1u;
                    if (!wait_bounded(&tempty_bar[buf], tph ^ 1u, ctl)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    for (int kb = args.kb_begin; kb < args.kb_end; ++kb) {
                        if (!wait_bounded(&full_bar[stage], phase, ctl)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_base = smem_u32(sA + stage * Cfg::A_BYTES);
                        const uint32_t b_base = smem_u32(sB + stage * Cfg::B_BYTES);
#pragma unroll
                        for (int k = 0; k < BK / UMMA_K; ++k) {
                            const uint64_t ad = A_MN ? make_sdesc_sw128(a_base + k * 2048, 8192, 1024)
                                                     : make_sdesc_sw128(a_base + k * 32, 16, 1024);
                            const uint64_t bd = B_MN ? make_sdesc_sw128(b_base + k * 2048, 8192, 1024)
                                                     : make_sdesc_sw128(b_base + k * 32, 16, 1024);
                            umma_bf16(d_tmem, ad, bd, IDESC, (kb > args.kb_begin || k > 0) ? 1u : 0u);
                        }
                        umma_commit(&empty_bar[stage]);  // frees the stage when these MMAs finish
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit(&tfull_bar[buf]);  // accumulator ready for the epilogue
                }
            }
            // Every MMA of ours must finish before TMEM is freed.
            umma_commit(drain_bar);
            wait_drain(drain_bar, 0, args.status);
        }
    } else {
        // ---------------- epilogue (warps 2..5) ----------------
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row_in_tile = q * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint32_t tcount = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < args.num_units && ok; u += gridDim.x) {
            const int m_blk = u % args.num_m_blocks;
            const int ucol = u / args.num_m_blocks;
            const int n_blk0 = ucol * args.tiles_per_unit;
            const int row = m_blk * BM + row_in_tile;
            const bool row_ok = row < args.M;
            // cross-entropy running state (natural-log units)
            float run_m = -INFINITY, run_s = 0.0f, z_tgt = 0.0f;
            int tgt = -1;
            if (EPI == EPI_CE && row_ok) tgt = args.target[row];

            for (int nt = 0; nt < args.tiles_per_unit; ++nt, ++tcount) {
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
                const int n_blk = n_blk0 + nt;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    const int col0 = n_blk * BN + c * 32;
                    uint32_t r[32];
                    tmem_ld32(tmem_base + lane_addr + buf * BN + c * 32, r);
                    tmem_ld_wait(r);
                    if (col0 >= args.N) continue;  // ragged N tail (whole 32-column chunks)
                    if constexpr (EPI == EPI_STORE) {
                        if (row_ok) {
                            uint32_t p[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                p[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                            store_row32(args.out0 + row * args.ld0 + col0, p);
                        }
                    } else if constexpr (EPI == EPI_GELU) {
                        if (row_ok) {
                            uint32_t p[16];
                            if (args.out1 != nullptr) {
#pragma unroll
                                for (int j = 0; j < 16; ++j)
                                    p[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                                store_row32(args.out1 + row * args.ld1 + col0, p);
                            }
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                p[j] = pack_bf16x2(gelu_f(__uint_as_float(r[2 * j])),
                                                   gelu_f(__uint_as_float(r[2 * j + 1])));
                            store_row32(args.out0 + row * args.ld0 + col0, p);
                        }
                    } else if constexpr (EPI == EPI_DGELU) {
                        if (row_ok) {
                            const uint4* src = reinterpret_cast<const uint4*>(args.aux + row * args.ld_aux + col0);
                            uint32_t uw[16];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint4 w = src[j];
                                uw[4 * j + 0] = w.x;
                                uw[4 * j + 1] = w.y;
                                uw[4 * j + 2] = w.z;
                                uw[4 * j + 3] = w.w;
                            }
                            uint32_t p[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float g0 = __uint_as_float(r[2 * j]) * gelu_prime_f(bf16_lo(uw[j]));
                                const float g1 = __uint_as_float(r[2 * j + 1]) * gelu_prime_f(bf16_hi(uw[j]));
                                p[j] = pack_bf16x2(g0, g1);
                            }
                            store_row32(args.out0 + row * args.ld0 + col0, p);
                        }
                    } else {  // EPI_CE
                        const int lim = args.v_valid - col0;  // valid columns in this chunk
                        if (lim > 0) {
                            constexpr float LOG2E = 1.4426950408889634f;
                            float mx = -INFINITY;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float x = (j < lim) ? __uint_as_float(r[j]) : -INFINITY;
                                mx = fmaxf(mx, x);
                            }
                            if (mx > run_m) {
                                run_s *= ex2_approx((run_m - mx) * LOG2E);
                                run_m = mx;
                            }
                            const float mb = run_m * LOG2E;
                            float acc = 0.0f;
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float e = ex2_approx(fmaf(__uint_as_float(r[j]), LOG2E, -mb));
                                acc += (j < lim) ? e : 0.0f;
                            }
                            run_s += acc;
                            const unsigned dt = static_cast<unsigned>(tgt - col0);
                            if (dt < 32u && static_cast<int>(dt) < lim) {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (static_cast<int>(dt) == j) z_tgt = __uint_as_float(r[j]);
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty_bar[buf]);
            }
            if (!ok) break;
            if constexpr (EPI == EPI_CE) {
                if (row_ok) {
                    float* w = args.ws + static_cast<long long>(ucol) * 3 * args.M;
                    w[row] = run_m;
                    w[args.M + row] = run_s;
                    w[2 * args.M + row] = z_tgt;
                }
            }
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// Host-side launcher (grid = min(units, SMs), one CTA per SM).
template <int BN, bool A_MN, bool B_MN, int EPI>
inline cudaError_t launch_gemm_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& args,
                                  int num_sms, cudaStream_t stream) {
    using Cfg = GemmCfg<BN>;
    auto kern = gemm_tc_kernel<BN, A_MN, B_MN, EPI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    const int grid = args.num_units < num_sms ? args.num_units : num_sms;
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, NUM_THREADS, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, args);
    return cudaGetLastError();
}

}  // namespace mptp
