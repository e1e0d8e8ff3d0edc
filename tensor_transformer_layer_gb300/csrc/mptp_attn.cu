// Entry point of the head-parallel self-attention block (forward): mp_attn_fwd.
//
// "Megatron-LM: Training Multi-Billion Parameter Language Models Using Model
// Parallelism", section 3.4 "Attention Head Parallelism in the Self-Attention Block",
// and "Megatron-LM, annotated", section 3.2 "The attention block": the Q, K, V
// projections are split by columns so that each of the t shards holds whole heads,
// every head runs its (causal, GPT-2 style) softmax attention alone, and the output
// projection is split by rows with the shards' partial outputs summed (g).
//
//   QKV = X Wqkv                 column-parallel GEMM (all shards' heads in one launch)
//   O_h = softmax(Q_h K_h^T / sqrt d + causal) V_h    fused attention kernel below
//   out = sum_i O_i Wo_i          row-parallel GEMM, shards in ascending order in the K-loop
//
// Attention kernel: one CTA per (sequence, head, 128-query tile), 192 threads:
//   warp 0      TMA producer: the Q tile once, then K and V tiles (128 keys) into a
//               2-stage ring. Head width D is loaded as D/32 boxes of 32 columns with
//               the 64-byte swizzle.
//   warp 1      TMEM allocator and MMA issuer: S_j = Q K_j^T (M = N = 128, K = D) into
//               one of two TMEM buffers, PV_j = P_j V_j (M = 128, N = D, K = 128) into
//               one of two more, issued in the order S_{j+1}, PV_j so the tensor core
//               works on the next scores while the softmax runs.
//   warps 2..5  softmax and correction, thread = query row: two passes over S_j
//               (masked max, then exp2 with the 1/sqrt(d) scale folded in), P_j written
//               as bf16 into 128-byte-swizzled shared memory (the A operand of PV_j),
//               running max m and sum l; O is accumulated in registers as
//               O = O * alpha_j + PV_j, alpha_j = exp(m_{j-1} - m_j); finally O / l is
//               stored with TMA.
// Key tiles above the diagonal are skipped; the diagonal tile is masked.
#include "mptp_gemm.cuh"
#include "mptp_internal.h"

namespace mptp {

constexpr int ATT_BQ = 128;  // queries per CTA
constexpr int ATT_BKV = 128; // keys per tile
constexpr int ATT_THREADS = 192;

template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 96, "head width");
    static constexpr int NB = D / 32;                 // 32-column boxes per tile row
    static constexpr int BOX_BYTES = 128 * 64;        // 128 rows x 32 bf16
    static constexpr int Q_BYTES = NB * BOX_BYTES;
    static constexpr int KV_BYTES = 2 * NB * BOX_BYTES;   // K tile + V tile
    static constexpr int P_BYTES = ATT_BQ * ATT_BKV * 2;  // two 64-key blocks, 128-byte swizzle
    static constexpr int STG_BYTES = 4 * STG_BYTES_PER_WARP;
    static constexpr int NUM_BARS = 1 + 2 * 2 + 2 * 2 * 4 + 1;  // + drain
    static constexpr size_t SMEM_BYTES =
        1024 + Q_BYTES + 2 * KV_BYTES + 2 * P_BYTES + STG_BYTES + 8 * NUM_BARS + 16;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory per block");
    static constexpr uint32_t TMEM_COLS = 512;  // S: 2 x 128 columns, PV: 2 x 128 (D used)
};

struct AttnArgs {
    int b, s, h, heads, nq;  // nq = s / 128 query tiles per sequence
    float scale_log2;        // log2(e) / sqrt(D)
    uint32_t* status;
    unsigned long long budget_ns;
};

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQKV, const __grid_constant__ CUtensorMap tmO,
                    const AttnArgs args) {
    using Cfg = AttnCfg<D>;
    constexpr int NB = Cfg::NB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sKV = sQ + Cfg::Q_BYTES;                  // stage st: K at st*KV_BYTES, V after it
    uint8_t* sP = sKV + 2 * Cfg::KV_BYTES;             // buffer pb at pb*P_BYTES
    uint8_t* stg_base = sP + 2 * Cfg::P_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stg_base + Cfg::STG_BYTES);
    uint64_t* q_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = bars + 3;
    uint64_t* s_full = bars + 5;
    uint64_t* s_empty = bars + 7;
    uint64_t* p_full = bars + 9;
    uint64_t* p_empty = bars + 11;
    uint64_t* pv_full = bars + 13;
    uint64_t* pv_empty = bars + 15;
    uint64_t* drain_bar = bars + 17;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Longest (most key tiles) query tiles first.
    const int per_tile = args.b * args.heads;
    const int qt = args.nq - 1 - static_cast<int>(blockIdx.x) / per_tile;
    const int rem = static_cast<int>(blockIdx.x) % per_tile;
    const int seq = rem / args.heads;
    const int head = rem % args.heads;
    const int n = qt + 1;                       // key tiles 0..qt (causal)
    const int row_base = seq * args.s;          // first token row of this sequence
    const int h = args.h;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(drain_bar, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 4);
            mbar_init(&p_full[i], 4);
            mbar_init(&p_empty[i], 1);
            mbar_init(&pv_full[i], 1);
            mbar_init(&pv_empty[i], 4);
        }
        *abort_flag = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmQKV);
        prefetch_tensormap(&tmO);
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
            mbar_arrive_expect_tx(q_full, Cfg::Q_BYTES);
            for (int c = 0; c < NB; ++c)
                tma_load_2d(sQ + c * Cfg::BOX_BYTES, &tmQKV, q_full, head * D + c * 32, row_base + qt * ATT_BQ);
            for (int j = 0; j < n; ++j) {
                const int st = j & 1;
                if (!wait_bounded(&kv_empty[st], ((j >> 1) & 1) ^ 1u, ctl)) break;
                mbar_arrive_expect_tx(&kv_full[st], Cfg::KV_BYTES);
                uint8_t* k_dst = sKV + st * Cfg::KV_BYTES;
                uint8_t* v_dst = k_dst + NB * Cfg::BOX_BYTES;
                for (int c = 0; c < NB; ++c) {
                    tma_load_2d(k_dst + c * Cfg::BOX_BYTES, &tmQKV, &kv_full[st], h + head * D + c * 32,
                                row_base + j * ATT_BKV);
                    tma_load_2d(v_dst + c * Cfg::BOX_BYTES, &tmQKV, &kv_full[st], 2 * h + head * D + c * 32,
                                row_base + j * ATT_BKV);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t IDESC_S = make_idesc_bf16(ATT_BQ, ATT_BKV, false, false);
            constexpr uint32_t IDESC_PV = make_idesc_bf16(ATT_BQ, D, false, true);
            bool ok = wait_bounded(q_full, 0, ctl);
            auto issue_s = [&](int j) -> bool {
                const int sb = j & 1;
                if (!wait_bounded(&s_empty[sb], ((j >> 1) & 1) ^ 1u, ctl)) return false;
                if (!wait_bounded(&kv_full[j & 1], (j >> 1) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sKV + (j & 1) * Cfg::KV_BYTES);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 1) * Cfg::BOX_BYTES + (k & 1) * 32;
                    umma_bf16(tmem_base + sb * 128, make_sdesc_sw64(q0 + off, 16, 512),
                              make_sdesc_sw64(k0 + off, 16, 512), IDESC_S, k > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[sb]);
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int pb = j & 1;
                if (!wait_bounded(&p_full[pb], (j >> 1) & 1, ctl)) return false;
                if (!wait_bounded(&pv_empty[pb], ((j >> 1) & 1) ^ 1u, ctl)) return false;
                tc_fence_after();
                const uint32_t p0 = smem_u32(sP + pb * Cfg::P_BYTES);
                const uint32_t v0 = smem_u32(sKV + (j & 1) * Cfg::KV_BYTES + NB * Cfg::BOX_BYTES);
#pragma unroll
                for (int k = 0; k < ATT_BKV / 16; ++k) {
                    const uint64_t ad = make_sdesc_sw128(p0 + (k >> 2) * (ATT_BQ * 128) + (k & 3) * 32, 16, 1024);
                    const uint64_t bd = make_sdesc_sw64(v0 + k * 1024, Cfg::BOX_BYTES, 512);
                    umma_bf16(tmem_base + 256 + pb * 128, ad, bd, IDESC_PV, k > 0 ? 1u : 0u);
                }
                umma_commit(&kv_empty[j & 1]);  // K_j (read by S_j) and V_j are free
                umma_commit(&p_empty[pb]);
                umma_commit(&pv_full[pb]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; j < n && ok; ++j) {
                if (j + 1 < n) ok = issue_s(j + 1);
                if (ok) ok = issue_pv(j);
            }
            // Every MMA must finish before TMEM is freed.
            umma_commit(drain_bar);
            wait_drain(drain_bar, 0, args.status);
        }
    } else {
        // ---------------- softmax / correction (warps 2..5) ----------------
        const int q = warp & 3;
        const int qrow = q * 32 + lane;                 // query row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const float c2 = args.scale_log2;
        float m = -INFINITY, l = 0.0f;
        float O[D];
#pragma unroll
        for (int i = 0; i < D; ++i) O[i] = 0.0f;
        float alpha0 = 0.0f, alpha1 = 0.0f;  // correction factor of the tile in each buffer
        bool ok = true;

        auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool got = true;
            if (lane == 0) got = wait_bounded(bar, parity, ctl);
            return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        };
        auto softmax = [&](int j) -> bool {
            const int sb = j & 1;
            if (!wait_lane0(&s_full[sb], (j >> 1) & 1)) return false;
            tc_fence_after();
            const bool diag = (j == qt);
            const uint32_t sbase = tmem_base + lane_addr + sb * 128;
            // pass 1: row max of the (masked) raw scores
            float mx = -INFINITY;
#pragma unroll 1
            for (int c = 0; c < ATT_BKV / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(sbase + c * 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const bool masked = diag && (c * 32 + i > qrow);
                    mx = fmaxf(mx, masked ? -INFINITY : __uint_as_float(r[i]));
                }
            }
            const float m_new = fmaxf(m, mx);
            const float a_new = ex2_approx((m - m_new) * c2);
            if (sb) alpha1 = a_new; else alpha0 = a_new;
            const float mb = m_new * c2;
            // P_j may be written once PV_{j-2} has read this buffer.
            if (!wait_lane0(&p_empty[sb], ((j >> 1) & 1) ^ 1u)) return false;
            uint8_t* prow = sP + sb * Cfg::P_BYTES + qrow * 128;
            const int sw = qrow & 7;
            float rowsum = 0.0f;
            // pass 2: P = exp2(s * c2 - m_new * c2), bf16 into the swizzled P tile
#pragma unroll 1
            for (int c = 0; c < ATT_BKV / 32; ++c) {
                uint32_t r[32];
                tmem_ld32(sbase + c * 32, r);
                tmem_ld_wait(r);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float pr[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int col = c * 32 + 2 * i + e;
                        const bool masked = diag && (col > qrow);
                        pr[e] = masked ? 0.0f : ex2_approx(fmaf(__uint_as_float(r[2 * i + e]), c2, -mb));
                        rowsum += pr[e];
                    }
                    pk[i] = pack_bf16x2(pr[0], pr[1]);
                }
                // 32 keys = four 16-byte chunks of row qrow in 64-key block c/2.
                uint8_t* blk = prow + (c >> 1) * (ATT_BQ * 128);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int u = (c & 1) * 4 + v;
                    *reinterpret_cast<uint4*>(blk + ((u ^ sw) << 4)) =
                        make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            l = l * a_new + rowsum;
            m = m_new;
            fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&s_empty[sb]);
                mbar_arrive(&p_full[sb]);
            }
            return true;
        };
        auto correct = [&](int j) -> bool {
            const int pb = j & 1;
            if (!wait_lane0(&pv_full[pb], (j >> 1) & 1)) return false;
            tc_fence_after();
            const float a = pb ? alpha1 : alpha0;
#pragma unroll
            for (int c = 0; c < NB; ++c) {
                uint32_t r[32];
                tmem_ld32(tmem_base + lane_addr + 256 + pb * 128 + c * 32, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int i = 0; i < 32; ++i) O[c * 32 + i] = fmaf(O[c * 32 + i], a, __uint_as_float(r[i]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pv_empty[pb]);
            return true;
        };

        ok = softmax(0);
        for (int j = 0; j < n && ok; ++j) {
            if (j + 1 < n) ok = softmax(j + 1);
            if (ok) ok = correct(j);
        }
        if (ok) {
            const float inv = 1.0f / l;
            uint8_t* stg = stg_base + (warp - 2) * STG_BYTES_PER_WARP;
            int sbuf = 0;
#pragma unroll
            for (int c = 0; c < NB; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(O[c * 32 + 2 * i] * inv, O[c * 32 + 2 * i + 1] * inv);
                stage_and_store(&tmO, stg, sbuf, lane, pk, head * D + c * 32, row_base + qt * ATT_BQ + q * 32);
            }
            if (lane == 0) bulk_wait_group<0>();
        }
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) spin_ns(ABORT_SETTLE_NS);
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

template <int D>
static cudaError_t launch_attn(const CUtensorMap& tmQKV, const CUtensorMap& tmO, const AttnArgs& a,
                               cudaStream_t s) {
    using Cfg = AttnCfg<D>;
    auto kern = attn_fwd_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    kern<<<a.b * a.heads * a.nq, ATT_THREADS, Cfg::SMEM_BYTES, s>>>(tmQKV, tmO, a);
    return cudaGetLastError();
}

}  // namespace mptp

using namespace mptp;

extern "C" mp_status mp_attn_fwd(const mp_bf16* X, const mp_bf16* Wqkv, const mp_bf16* Wo, mp_bf16* out,
                                 mp_bf16* QKV, mp_bf16* O, int b, int s, int h, int heads, int t,
                                 uint32_t* d_status, void* stream) {
    if (b < 0 || s < 0 || h <= 0 || heads <= 0 || t < 1) return MP_ERR_INVALID_ARG;
    if (h % heads != 0 || heads % t != 0) return MP_ERR_UNSUPPORTED_SHAPE;
    const int d = h / heads;
    if ((d != 64 && d != 96) || h % 64 != 0 || s % ATT_BQ != 0)
        return MP_ERR_UNSUPPORTED_SHAPE;
    const long long T = static_cast<long long>(b) * s;
    if (T == 0) return MP_OK;
    if (!X || !Wqkv || !Wo || !out || !QKV || !O) return MP_ERR_INVALID_ARG;
    const void* ptrs[] = {X, Wqkv, Wo, out, QKV, O};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MP_ERR_MISALIGNED;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MP_ERR_MISALIGNED;
    int sms = 0;
    mp_status st = check_device(&sms);
    if (st != MP_OK) return st;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const unsigned long long budget = wait_budget_ns();
    const double Tb = 2.0 * T, hb = 2.0 * h;

    // QKV = X Wqkv: all shards' heads in one column-parallel launch (Wqkv MN-major).
    TmapSet m1{};
    if (!make_tmap_bf16(&m1.a, X, h, T, h, 64, BM) || !make_tmap_bf16(&m1.b, Wqkv, 3 * h, h, 3 * h, 64, 64) ||
        !make_tmap_bf16_out(&m1.o0, QKV, 3 * h, T, 3 * h))
        return MP_ERR_CUDA;
    GemmArgs a1{};
    a1.pr.M = static_cast<int>(T);
    a1.pr.N = 3 * h;
    a1.pr.num_m_blocks = ceil_div(T, 2 * BM);
    a1.pr.num_units = a1.pr.num_m_blocks * ceil_div(3 * h, 256);
    a1.pr.n_fastest = n_fastest_order(Tb * h, hb * 3 * h);
    a1.pr.kb_end = h / BK;
    a1.pr.b_mn = 1;
    a1.tiles_per_unit = 1;
    a1.status = d_status;
    a1.budget_ns = budget;
    if (launch_gemm_tc<256, EPI_STORE, 4>(m1, a1, sms, cs) != cudaSuccess) return MP_ERR_CUDA;

    // Per-head causal attention.
    CUtensorMap tq, to;
    if (!make_tmap_bf16_sw64(&tq, QKV, 3 * h, T, 3 * h, 32, ATT_BQ) || !make_tmap_bf16_out(&to, O, h, T, h))
        return MP_ERR_CUDA;
    AttnArgs aa{};
    aa.b = b;
    aa.s = s;
    aa.h = h;
    aa.heads = heads;
    aa.nq = s / ATT_BQ;
    aa.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    aa.status = d_status;
    aa.budget_ns = budget;
    cudaError_t e = d == 64 ? launch_attn<64>(tq, to, aa, cs) : launch_attn<96>(tq, to, aa, cs);
    if (e != cudaSuccess) return MP_ERR_CUDA;

    // out = sum_i O_i Wo_i: the K-loop runs over the heads' columns in ascending order, i.e.
    // shard 0's heads, then shard 1's, ... (the g sum; a K block may span two shards).
    TmapSet m3{};
    if (!make_tmap_bf16(&m3.a, O, h, T, h, 64, BM) || !make_tmap_bf16(&m3.b, Wo, h, h, h, 64, 64) ||
        !make_tmap_bf16_out(&m3.o0, out, h, T, h))
        return MP_ERR_CUDA;
    GemmArgs a3{};
    a3.pr.M = static_cast<int>(T);
    a3.pr.N = h;
    a3.pr.num_m_blocks = ceil_div(T, 2 * BM);
    a3.pr.num_units = a3.pr.num_m_blocks * ceil_div(h, 256);
    a3.pr.n_fastest = n_fastest_order(Tb * h, hb * h);
    a3.pr.kb_begin = 0;
    a3.pr.kb_end = h / BK;
    a3.pr.b_mn = 1;
    a3.tiles_per_unit = 1;
    a3.status = d_status;
    a3.budget_ns = budget;
    if (launch_gemm_tc<256, EPI_STORE, 4>(m3, a3, sms, cs) != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}
