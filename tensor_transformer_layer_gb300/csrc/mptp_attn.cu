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
// Attention kernel: one CTA per (sequence, head, 128-query tile), 320 threads:
//   warp 0      TMA producer: the Q tile once, then K tiles (128 keys) into a 3-stage
//               ring that runs two tiles ahead, and V tiles into a ring of their own
//               (2 stages at D = 96, 3 at D = 64), so that a K load never waits for a
//               PV product and a V load never waits for a score product. Head width D
//               is loaded as D/32 boxes of 32 columns with the 64-byte swizzle.
//   warp 1      TMEM allocator and MMA issuer: S_j = Q K_j^T (M = N = 128, K = D) into
//               one of two TMEM buffers, PV_j = P_j V_j (M = 128, N = D, K = 128) into
//               one of two more, issued in the order S_{j+1}, PV_j so the tensor core
//               works on the next scores while the softmax runs.
//   warps 2..9  softmax and correction, two warps per 32-row quarter (thread = query
//               row), each taking 64 of the 128 key columns and half of the head's
//               output columns. Its half of S_j is read from TMEM once (the buffer is
//               released right after); masked row max over eight independent chains,
//               exchanged with the partner warp through a shared slot and an mbarrier;
//               exp2 with the 1/sqrt(d) scale folded in, P_j written as bf16 into
//               128-byte-swizzled shared memory (the A operand of PV_j); running max m
//               and partial sums l; O accumulated in registers as O * alpha_j + PV_j,
//               alpha_j = exp(m_{j-1} - m_j); finally O / (l_0 + l_1) is stored.
// Key tiles above the diagonal are skipped; the diagonal tile is masked.
#include "mptp_gemm.cuh"
#include "mptp_internal.h"

namespace mptp {

constexpr int ATT_BQ = 128;  // queries per CTA
constexpr int ATT_BKV = 128; // keys per tile
constexpr int ATT_THREADS = 320;

template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 96, "head width");
    static constexpr int NB = D / 32;                 // 32-column boxes per tile row
    static constexpr int BOX_BYTES = 128 * 64;        // 128 rows x 32 bf16
    static constexpr int Q_BYTES = NB * BOX_BYTES;
    static constexpr int KV_TILE_BYTES = NB * BOX_BYTES;  // one K or one V tile
    static constexpr int KST = 3;                          // K ring stages
    static constexpr int VST = D == 64 ? 3 : 2;            // V ring stages
    static constexpr int P_BYTES = ATT_BQ * ATT_BKV * 2;  // two 64-key blocks, 128-byte swizzle
    static constexpr int XCHG_BYTES = 2 * 2 * ATT_BQ * 4;  // [parity][half][row] fp32
    // q_full, K ring, V ring, S/P/PV full+empty pairs, drain, 4 exchange barriers
    static constexpr int NUM_BARS = 1 + 2 * KST + 2 * VST + 2 * 2 * 3 + 1 + 4;
    static constexpr size_t SMEM_BYTES =
        1024 + Q_BYTES + (KST + VST) * KV_TILE_BYTES + 2 * P_BYTES + XCHG_BYTES + 8 * NUM_BARS + 16;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory per block");
    static constexpr uint32_t TMEM_COLS = 512;  // S: 2 x 128 columns, PV: 2 x 128 (D used)
};

struct AttnArgs {
    __nv_bfloat16* O;        // [b s, h] attention output
    int b, s, h, heads, nq;  // nq = s / 128 query tiles per sequence
    float scale_log2;        // log2(e) / sqrt(D)
    uint32_t* status;
    unsigned long long budget_ns;
};

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQKV, const AttnArgs args) {
    using Cfg = AttnCfg<D>;
    constexpr int NB = Cfg::NB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;
    uint8_t* sK = sQ + Cfg::Q_BYTES;                       // K stage st at st * KV_TILE_BYTES
    uint8_t* sV = sK + Cfg::KST * Cfg::KV_TILE_BYTES;      // V stage st at st * KV_TILE_BYTES
    uint8_t* sP = sV + Cfg::VST * Cfg::KV_TILE_BYTES;      // buffer pb at pb * P_BYTES
    float* xchg = reinterpret_cast<float*>(sP + 2 * Cfg::P_BYTES);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * Cfg::P_BYTES + Cfg::XCHG_BYTES);
    constexpr int KST = Cfg::KST, VST = Cfg::VST;
    uint64_t* q_full = bars;
    uint64_t* k_full = bars + 1;
    uint64_t* k_empty = k_full + KST;
    uint64_t* v_full = k_empty + KST;
    uint64_t* v_empty = v_full + VST;
    uint64_t* s_full = v_empty + VST;
    uint64_t* s_empty = s_full + 2;
    uint64_t* p_full = s_empty + 2;
    uint64_t* p_empty = p_full + 2;
    uint64_t* pv_full = p_empty + 2;
    uint64_t* pv_empty = pv_full + 2;
    uint64_t* drain_bar = pv_empty + 2;
    uint64_t* xchg_bar = drain_bar + 1;  // one per row quarter: the two warps of the quarter
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
        for (int i = 0; i < KST; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < VST; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 8);
            mbar_init(&p_full[i], 8);
            mbar_init(&p_empty[i], 1);
            mbar_init(&pv_full[i], 1);
            mbar_init(&pv_empty[i], 8);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&xchg_bar[i], 2);
        *abort_flag = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmQKV);
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
            // Tile j of K (column block 1 of QKV) or V (block 2) into a ring stage.
            auto load = [&](int j, int which, uint64_t* full, uint64_t* empty, uint8_t* ring, int stages) -> bool {
                const int st = j % stages;
                if (!wait_bounded(&empty[st], ((j / stages) & 1) ^ 1u, ctl)) return false;
                mbar_arrive_expect_tx(&full[st], Cfg::KV_TILE_BYTES);
                uint8_t* dst = ring + st * Cfg::KV_TILE_BYTES;
                for (int c = 0; c < NB; ++c)
                    tma_load_2d(dst + c * Cfg::BOX_BYTES, &tmQKV, &full[st], which * h + head * D + c * 32,
                                row_base + j * ATT_BKV);
                return true;
            };
            constexpr int LEAD = KST - 1;  // K tiles loaded ahead of the V tile of the same index
            bool ok = true;
            for (int j = 0; j < LEAD && j < n && ok; ++j) ok = load(j, 1, k_full, k_empty, sK, KST);
            for (int j = 0; j < n && ok; ++j) {
                if (j + LEAD < n) ok = load(j + LEAD, 1, k_full, k_empty, sK, KST);
                if (ok) ok = load(j, 2, v_full, v_empty, sV, VST);
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
                const int ks = j % KST;
                if (!wait_bounded(&s_empty[sb], ((j >> 1) & 1) ^ 1u, ctl)) return false;
                if (!wait_bounded(&k_full[ks], (j / KST) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t q0 = smem_u32(sQ), k0 = smem_u32(sK + ks * Cfg::KV_TILE_BYTES);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 1) * Cfg::BOX_BYTES + (k & 1) * 32;
                    umma_bf16(tmem_base + sb * 128, make_sdesc_sw64(q0 + off, 16, 512),
                              make_sdesc_sw64(k0 + off, 16, 512), IDESC_S, k > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[sb]);
                umma_commit(&k_empty[ks]);  // K_j is free once S_j is done
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int pb = j & 1;
                if (!wait_bounded(&p_full[pb], (j >> 1) & 1, ctl)) return false;
                if (!wait_bounded(&pv_empty[pb], ((j >> 1) & 1) ^ 1u, ctl)) return false;
                const int vs = j % VST;
                if (!wait_bounded(&v_full[vs], (j / VST) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t p0 = smem_u32(sP + pb * Cfg::P_BYTES);
                const uint32_t v0 = smem_u32(sV + vs * Cfg::KV_TILE_BYTES);
#pragma unroll
                for (int k = 0; k < ATT_BKV / 16; ++k) {
                    const uint64_t ad = make_sdesc_sw128(p0 + (k >> 2) * (ATT_BQ * 128) + (k & 3) * 32, 16, 1024);
                    const uint64_t bd = make_sdesc_sw64(v0 + k * 1024, Cfg::BOX_BYTES, 512);
                    umma_bf16(tmem_base + 256 + pb * 128, ad, bd, IDESC_PV, k > 0 ? 1u : 0u);
                }
                umma_commit(&v_empty[vs]);  // V_j is free
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
        // ---------------- softmax / correction (warps 2..9) ----------------
        const int q = warp & 3;                         // TMEM lane quarter
        const int half = (warp - 2) >> 2;               // key columns [64 half, +64), O columns [D/2 half, +D/2)
        const int qrow = q * 32 + lane;                 // query row within the tile
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const float c2 = args.scale_log2;
        constexpr int DH = D / 2;                       // output columns per warp
        float m = -INFINITY, l = 0.0f;
        float O[DH];
#pragma unroll
        for (int i = 0; i < DH; ++i) O[i] = 0.0f;
        float alpha0 = 0.0f, alpha1 = 0.0f;  // correction factor of the tile in each buffer
        uint32_t xphase = 0;
        bool ok = true;

        auto wait_lane0 = [&](uint64_t* bar, uint32_t parity) -> bool {
            bool got = true;
            if (lane == 0) got = wait_bounded(bar, parity, ctl);
            return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
        };
        // Exchange one value per row with the partner warp of this quarter (bounded wait).
        auto exchange = [&](float mine, float& theirs) -> bool {
            float* slot = xchg + (xphase & 1) * (2 * ATT_BQ);
            slot[half * ATT_BQ + qrow] = mine;
            __syncwarp();
            if (lane == 0) mbar_arrive(&xchg_bar[q]);
            const bool got = wait_lane0(&xchg_bar[q], xphase & 1);
            __syncwarp();  // orders lane 0's acquire before every lane's read
            xphase ^= 1u;
            theirs = slot[(half ^ 1) * ATT_BQ + qrow];
            return got;
        };
        auto softmax = [&](int j) -> bool {
            const int sb = j & 1;
            bool good = wait_lane0(&s_full[sb], (j >> 1) & 1);
            if (good) good = wait_lane0(&p_empty[sb], ((j >> 1) & 1) ^ 1u);  // PV_{j-2} read this P buffer
            tc_fence_after();
            // Key columns of this warp's half at or left of the diagonal: all 64 off the diagonal tile.
            const int lim = (j == qt) ? qrow - half * 64 + 1 : 64;
            const uint32_t sbase = tmem_base + lane_addr + sb * 128 + half * 64;
            uint32_t ra[32], rb[32];  // S row, columns [0, 32) and [32, 64) of this half
            float mx = -INFINITY;
            if (good) {
                tmem_ld32(sbase, ra);
                tmem_ld32(sbase + 32, rb);
                tmem_wait_ld();
                reg_fence32(ra);
                reg_fence32(rb);
                // S_j is in registers: its TMEM buffer may take S_{j+2}.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[sb]);
                // pass 1: row max, eight independent chains
                float m8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
                if (lim >= 64) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        m8[i & 7] = fmaxf(m8[i & 7], __uint_as_float(ra[i]));
                        m8[(i + 4) & 7] = fmaxf(m8[(i + 4) & 7], __uint_as_float(rb[i]));
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        m8[i & 7] = fmaxf(m8[i & 7], i < lim ? __uint_as_float(ra[i]) : -INFINITY);
                        m8[(i + 4) & 7] = fmaxf(m8[(i + 4) & 7], i + 32 < lim ? __uint_as_float(rb[i]) : -INFINITY);
                    }
                }
                mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                           fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
            }
            float other = -INFINITY;
            const bool xok = exchange(good ? mx : __int_as_float(0x7fc00000), other);
            if (!good || !xok || other != other) return false;  // NaN from the partner: it failed
            const float m_new = fmaxf(m, fmaxf(mx, other));
            const float a_new = ex2_approx((m - m_new) * c2);
            if (sb) alpha1 = a_new; else alpha0 = a_new;
            const float mb = m_new * c2;
            // pass 2: P = exp2(s * c2 - m_new * c2) as bf16 into 64-key block `half` of the P tile
            float s8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) s8[k] = 0.0f;
            uint8_t* prow = sP + sb * Cfg::P_BYTES + half * (ATT_BQ * 128) + qrow * 128;
            const int sw = qrow & 7;
            // One 32-column register block; `base` = its first column. Every 8 columns are
            // stored as one 16-byte chunk u of the row (128-byte swizzle: chunk u ^ (row & 7)).
            auto expo = [&](const uint32_t(&r)[32], int base) {
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t pk[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int e = 8 * g + 2 * i;
                        float p0 = ex2_approx(fmaf(__uint_as_float(r[e]), c2, -mb));
                        float p1 = ex2_approx(fmaf(__uint_as_float(r[e + 1]), c2, -mb));
                        if (lim < base + 32) {
                            p0 = base + e < lim ? p0 : 0.0f;
                            p1 = base + e + 1 < lim ? p1 : 0.0f;
                        }
                        s8[(2 * i) & 7] += p0;
                        s8[(2 * i + 1) & 7] += p1;
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    const int u = base / 8 + g;
                    *reinterpret_cast<uint4*>(prow + ((u ^ sw) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            };
            expo(ra, 0);
            expo(rb, 32);
            const float rowsum = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
            l = l * a_new + rowsum;  // this warp's partial row sum
            m = m_new;
            fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
            return true;
        };
        auto correct = [&](int j) -> bool {
            const int pb = j & 1;
            if (!wait_lane0(&pv_full[pb], (j >> 1) & 1)) return false;
            tc_fence_after();
            const float a = pb ? alpha1 : alpha0;
            const uint32_t pv = tmem_base + lane_addr + 256 + pb * 128 + half * DH;
            // 16-column chunks, two loads in flight at a time
#pragma unroll
            for (int c0 = 0; c0 < DH / 16; c0 += 2) {
                uint32_t r0[16], r1[16];
                tmem_ld16(pv + c0 * 16, r0);
                if (c0 + 1 < DH / 16) tmem_ld16(pv + (c0 + 1) * 16, r1);
                tmem_wait_ld();
                reg_fence16(r0);
                if (c0 + 1 < DH / 16) reg_fence16(r1);
#pragma unroll
                for (int i = 0; i < 16; ++i) O[c0 * 16 + i] = fmaf(O[c0 * 16 + i], a, __uint_as_float(r0[i]));
                if (c0 + 1 < DH / 16) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        O[(c0 + 1) * 16 + i] = fmaf(O[(c0 + 1) * 16 + i], a, __uint_as_float(r1[i]));
                }
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
        float l_other = 0.0f;
        if (ok) ok = exchange(l, l_other);
        if (ok) {
            const float inv = 1.0f / (l + l_other);
            uint4* dst = reinterpret_cast<uint4*>(args.O + static_cast<long long>(row_base + qt * ATT_BQ + qrow) * h +
                                                  head * D + half * DH);
#pragma unroll
            for (int v = 0; v < DH / 8; ++v)
                dst[v] = make_uint4(pack_bf16x2(O[8 * v] * inv, O[8 * v + 1] * inv),
                                    pack_bf16x2(O[8 * v + 2] * inv, O[8 * v + 3] * inv),
                                    pack_bf16x2(O[8 * v + 4] * inv, O[8 * v + 5] * inv),
                                    pack_bf16x2(O[8 * v + 6] * inv, O[8 * v + 7] * inv));
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
static cudaError_t launch_attn(const CUtensorMap& tmQKV, const AttnArgs& a, cudaStream_t s) {
    using Cfg = AttnCfg<D>;
    auto kern = attn_fwd_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    kern<<<a.b * a.heads * a.nq, ATT_THREADS, Cfg::SMEM_BYTES, s>>>(tmQKV, a);
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
    CUtensorMap tq;
    if (!make_tmap_bf16_sw64(&tq, QKV, 3 * h, T, 3 * h, 32, ATT_BQ)) return MP_ERR_CUDA;
    AttnArgs aa{};
    aa.O = reinterpret_cast<__nv_bfloat16*>(O);
    aa.b = b;
    aa.s = s;
    aa.h = h;
    aa.heads = heads;
    aa.nq = s / ATT_BQ;
    aa.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    aa.status = d_status;
    aa.budget_ns = budget;
    cudaError_t e = d == 64 ? launch_attn<64>(tq, aa, cs) : launch_attn<96>(tq, aa, cs);
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
