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
// Attention kernel: one CTA per (sequence, head, pair of consecutive 128-query tiles
// 2p and 2p+1), 384 threads, the longest pairs launched first. The two query tiles
// ("A" = 2p, "B" = 2p+1) share every K and V tile they both need (causal: keys 0..2p for
// A, 0..2p+1 for B), so each K/V tile is loaded once for 256 queries.
//   warpgroup 0 (64 or 72 registers a thread): warp 0 is the TMA producer: both Q tiles once, then
//               K tiles into a ring that runs ahead and V tiles into a ring of their own
//               (head width D loaded as D/32 boxes of 32 columns, 64-byte swizzle). Warp 1
//               allocates TMEM and issues the products: the whole warp runs the issue loop
//               and one elected lane issues. Warps 2 and 3 only lend their registers.
//               TMEM holds S_A, S_B (128 columns each) and the output accumulators O_A, O_B
//               (D columns, at 256 and 384). Per key tile j and query tile g it issues
//               PV_g(j) (O_g += P_g V_j, P_g read from TMEM) and then S_g(j+1) = Q_g K_{j+1}^T;
//               while one tile's softmax runs, the tensor core works on the other tile.
//   warpgroups 1, 2 (216 or 208 registers a thread): softmax of tile A and of tile B; thread =
//               query row (the TMEM lane quarter of the warp), all 128 key columns. The
//               score row is read from TMEM once; row max over four chains of three-input
//               maxima. The running max is raised lazily: only when it grows by more than
//               2^8 in the exp2 domain are O (in TMEM) and the row sum rescaled by
//               alpha = exp2((m_old - m_new) log2(e) / sqrt(d)); otherwise the stale max
//               is kept (P entries stay <= 256, and O and the sum use the same max, so
//               the final quotient is unchanged). P = exp2(s log2(e)/sqrt(d) - m ...) is
//               packed to bf16 and stored over the first 64 columns of S_g, where the next
//               PV reads it. After the last tile O / l is read from TMEM, staged in the
//               shared memory of the group's Q tile (free by then) and written by TMA stores.
// Key tiles above the diagonal are skipped; the diagonal tile is masked.
#include <type_traits>

#include "mptp_gemm.cuh"
#include "mptp_internal.h"

namespace mptp {

constexpr int ATT_BQ = 128;   // queries per tile (two tiles per CTA)
constexpr int ATT_BKV = 128;  // keys per tile
constexpr int ATT_THREADS = 384;  // warpgroup 0: TMA, MMA, two idle warps; 1, 2: softmax
constexpr float ATT_RESCALE_LOG2 = 8.0f;  // lazy rescale threshold on the max, exp2 domain

template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 96, "head width");
    static constexpr int NB = D / 32;                     // 32-column boxes per tile row
    static constexpr int BOX_BYTES = 128 * 64;            // 128 rows x 32 bf16
    static constexpr int Q_BYTES = NB * BOX_BYTES;        // one query tile
    static constexpr int KV_TILE_BYTES = NB * BOX_BYTES;  // one K or one V tile
    // Registers a thread in warpgroup 0 and in the softmax warpgroups (setmaxnreg); the launch
    // gives 384 x 168, so 128 x REGS_CTRL + 256 x REGS_SOFTMAX must not exceed it. The splits
    // without spills: the MMA issuer needs more than 64 at D = 96 (six-step products).
    static constexpr int REGS_CTRL = D == 64 ? 64 : 72;
    static constexpr int REGS_SOFTMAX = D == 64 ? 216 : 208;
    static_assert(128 * REGS_CTRL + 256 * REGS_SOFTMAX <= ATT_THREADS * 168, "register split");
    static constexpr int KST = D == 64 ? 4 : 3;           // K ring stages
    static constexpr int VST = D == 64 ? 4 : 3;           // V ring stages
    // q_full per query tile, K ring, V ring, s_full/p_full/o_full per query tile, drain
    static constexpr int NUM_BARS = 2 + 2 * KST + 2 * VST + 2 * 3 + 1;
    static constexpr size_t SMEM_BYTES = 1024 + 2 * Q_BYTES + (KST + VST) * KV_TILE_BYTES + 8 * NUM_BARS + 16;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory per block");
    // S_A, S_B: 128 columns each (P_g, bf16, overwrites the first 64 columns of S_g);
    // O_A, O_B: D columns at 256 and 384.
    static constexpr uint32_t TMEM_COLS = 512;
};

struct AttnArgs {
    __nv_bfloat16* O;        // [b s, h] attention output
    int b, s, h, heads, nq;  // nq = s / 128 query tiles per sequence
    int npairs;              // ceil(nq / 2) query-tile pairs per sequence
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
    constexpr int KST = Cfg::KST, VST = Cfg::VST;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem;                                    // tile g at g * Q_BYTES
    uint8_t* sK = sQ + 2 * Cfg::Q_BYTES;                   // K stage st at st * KV_TILE_BYTES
    uint8_t* sV = sK + KST * Cfg::KV_TILE_BYTES;           // V stage st at st * KV_TILE_BYTES
    uint64_t* bars = reinterpret_cast<uint64_t*>(sV + VST * Cfg::KV_TILE_BYTES);
    uint64_t* q_full = bars;  // [2]: query tile g landed
    uint64_t* k_full = bars + 2;
    uint64_t* k_empty = k_full + KST;
    uint64_t* v_full = k_empty + KST;
    uint64_t* v_empty = v_full + VST;
    uint64_t* s_full = v_empty + VST;   // [2]: S_g computed (and every earlier product of tile g)
    uint64_t* p_full = s_full + 2;      // [2]: P_g written to TMEM (and O_g rescaled)
    uint64_t* o_full = p_full + 2;      // [2]: the last PV_g done
    uint64_t* drain_bar = o_full + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Longest pairs (most key tiles) first.
    const int per_pair = args.b * args.heads;
    const int pr = args.npairs - 1 - static_cast<int>(blockIdx.x) / per_pair;
    const int rem = static_cast<int>(blockIdx.x) % per_pair;
    const int seq = rem / args.heads;
    const int head = rem % args.heads;
    const int qt_a = 2 * pr, qt_b = 2 * pr + 1;
    const bool has_b = qt_b < args.nq;
    const int n_a = qt_a + 1;                   // key tiles of A (causal)
    const int n_b = has_b ? qt_b + 1 : 0;       // key tiles of B
    const int n = has_b ? n_b : n_a;            // key tiles loaded
    const int row_base = seq * args.s;          // first token row of this sequence
    const int h = args.h;

    constexpr int LEAD = KST - 1;  // K tiles loaded ahead of the V tile of the same index
    // Tile j of K (column block 1 of QKV) or V (block 2) into ring stage st, once the stage is free.
    auto issue_kv = [&](int j, int which, uint64_t* full, uint8_t* ring, int st) {
        mbar_arrive_expect_tx(&full[st], Cfg::KV_TILE_BYTES);
        uint8_t* dst = ring + st * Cfg::KV_TILE_BYTES;
        for (int c = 0; c < NB; ++c)
            tma_load_2d(dst + c * Cfg::BOX_BYTES, &tmQKV, &full[st], which * h + head * D + c * 32,
                        row_base + j * ATT_BKV);
    };
    if (threadIdx.x == 0) {
        mbar_init(&q_full[0], 1);
        mbar_init(&q_full[1], 1);
        mbar_init(drain_bar, 1);
        for (int i = 0; i < KST; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < VST; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&s_full[g], 1);
            mbar_init(&p_full[g], 4);
            mbar_init(&o_full[g], 1);
        }
        *abort_flag = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
        // The producer thread issues the first loads (K tile 0, the Q tiles, then the next LEAD - 1
        // K tiles, whose ring stages are still free) now, so that their latency overlaps the rest
        // of the set-up; QKV is read only once the grid that writes it has completed. Each Q tile
        // has a barrier of its own, so S_A(0) starts as soon as K_0 and Q_A have landed.
        prefetch_tensormap(&tmQKV);
        grid_dependency_wait();
        issue_kv(0, 1, k_full, sK, 0);
        for (int g = 0; g < (has_b ? 2 : 1); ++g) {
            mbar_arrive_expect_tx(&q_full[g], Cfg::Q_BYTES);
            for (int c = 0; c < NB; ++c)
                tma_load_2d(sQ + g * Cfg::Q_BYTES + c * Cfg::BOX_BYTES, &tmQKV, &q_full[g], head * D + c * 32,
                            row_base + (g ? qt_b : qt_a) * ATT_BQ);
        }
        for (int j = 1; j < LEAD && j < n; ++j) issue_kv(j, 1, k_full, sK, j);
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
    // Launched as the QKV GEMM's programmatic dependent: QKV is read only after that grid completes.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp < 4) {
        reg_dealloc<Cfg::REGS_CTRL>();
        if (warp == 0) {
            if (lane == 0) {
                // ---------------- TMA producer ----------------
                // (Both Q tiles and K tiles 0 .. LEAD - 1 went out during the set-up.)
                auto load = [&](int j, int which, uint64_t* full, uint64_t* empty, uint8_t* ring, int stages) -> bool {
                    const int st = j % stages;
                    if (!wait_bounded(&empty[st], ((j / stages) & 1) ^ 1u, ctl)) return false;
                    issue_kv(j, which, full, ring, st);
                    return true;
                };
                bool ok = true;
                for (int j = 0; j < n && ok; ++j) {
                    if (j + LEAD < n) ok = load(j + LEAD, 1, k_full, k_empty, sK, KST);
                    if (ok) ok = load(j, 2, v_full, v_empty, sV, VST);
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer ----------------
            // The whole warp runs this loop (operands stay warp-uniform); one elected lane issues
            // each product and commit.
            // Per key tile j and query tile g: PV_g(j) reads P_g from TMEM, then S_g(j+1)
            // overwrites the same columns. Products issued by one thread run in issue order,
            // so S_g(j+1) cannot overtake the read of P_g(j); the commit after S_g(j+1) also
            // covers PV_g(j), so s_full tells the softmax group that O_g is current.
            constexpr uint32_t IDESC_S = make_idesc_bf16(ATT_BQ, ATT_BKV, false, false);
            constexpr uint32_t IDESC_PV = make_idesc_bf16(ATT_BQ, D, false, true);
            auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
                const bool got = wait_bounded(bar, parity, ctl);
                return __all_sync(0xffffffffu, got) != 0;
            };
            // Descriptors are computed once; an operand at byte offset o from a base is that
            // base's descriptor advanced by o >> 4 in its address field.
            const uint64_t q_desc = make_sdesc_sw64(smem_u32(sQ), 16, 512);
            const uint64_t k_desc = make_sdesc_sw64(smem_u32(sK), 16, 512);
            const uint64_t v_desc = make_sdesc_sw64(smem_u32(sV), Cfg::BOX_BYTES, 512);
            auto s_mma = [&](int g, int j) {
                const uint64_t qd = q_desc + static_cast<uint32_t>((g * Cfg::Q_BYTES) >> 4);
                const uint64_t kd = k_desc + static_cast<uint32_t>(((j % KST) * Cfg::KV_TILE_BYTES) >> 4);
                const uint32_t d_tmem = tmem_base + g * 128;
    #pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k >> 1) * Cfg::BOX_BYTES + (k & 1) * 32) >> 4;
                    umma_bf16_elect(d_tmem, qd + off, kd + off, IDESC_S, k > 0 ? 1u : 0u);
                }
                umma_commit_elect(&s_full[g]);
            };
            auto pv_mma = [&](int g, int j) {
                const uint64_t vd = v_desc + static_cast<uint32_t>(((j % VST) * Cfg::KV_TILE_BYTES) >> 4);
                const uint32_t d_tmem = tmem_base + 256 + g * 128;
                const uint32_t a_tmem = tmem_base + g * 128;
                const uint32_t acc0 = j > 0 ? 1u : 0u;
    #pragma unroll
                for (int k = 0; k < ATT_BKV / 16; ++k)
                    umma_bf16_ts_elect(d_tmem, a_tmem + k * 8, vd + ((k * 1024) >> 4), IDESC_PV, k > 0 ? 1u : acc0);
            };
            bool ok = wait_all(&k_full[0], 0) && wait_all(&q_full[0], 0);
            if (ok) {
                tc_fence_after();
                s_mma(0, 0);
                if (has_b) {
                    ok = wait_all(&q_full[1], 0);
                    if (ok) {
                        tc_fence_after();
                        s_mma(1, 0);
                    }
                }
                umma_commit_elect(&k_empty[0]);
            }
            for (int j = 0; j < n && ok; ++j) {
                ok = wait_all(&v_full[j % VST], (j / VST) & 1);
                bool k_next = false;  // K tile j + 1 waited for
                for (int g = 0; g < 2 && ok; ++g) {
                    const int ng = g ? n_b : n_a;
                    if (j >= ng) continue;
                    if (!wait_all(&p_full[g], j & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    pv_mma(g, j);
                    if (j + 1 < ng) {
                        if (!k_next) {
                            if (!wait_all(&k_full[(j + 1) % KST], ((j + 1) / KST) & 1)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            k_next = true;
                        }
                        s_mma(g, j + 1);
                    } else {
                        umma_commit_elect(&o_full[g]);
                    }
                }
                if (!ok) break;
                umma_commit_elect(&v_empty[j % VST]);                  // V tile free once both PVs are done
                if (k_next) umma_commit_elect(&k_empty[(j + 1) % KST]);  // K tile free after both S
            }
            // Every MMA must finish before TMEM is freed.
            umma_commit_elect(drain_bar);
            wait_drain(drain_bar, 0, args.status);
        }
    } else {
        reg_alloc<Cfg::REGS_SOFTMAX>();
        // ---------------- softmax (warps 4..7: tile A, 8..11: tile B) ----------------
        const int g = (warp - 4) >> 2;
        const int q = warp & 3;                         // TMEM lane quarter
        const int qrow = q * 32 + lane;                 // query row within the tile
        const int qt = g ? qt_b : qt_a;
        const int ng = g ? n_b : n_a;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t s_addr = tmem_base + lane_addr + g * 128;
        const uint32_t o_addr = tmem_base + lane_addr + 256 + g * 128;
        const float c2 = args.scale_log2;
        float m = -INFINITY, l = 0.0f;
        bool ok = true;

        // Every lane polls (one warp instruction either way, and no divergent branch).
        auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
            const bool got = wait_bounded(bar, parity, ctl);
            return __all_sync(0xffffffffu, got) != 0;
        };
        for (int j = 0; j < ng && ok; ++j) {
            if (!wait_all(&s_full[g], j & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t r[4][32];  // the score row, 128 columns; then P packed in r[0], r[1]
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(s_addr + c * 32, r[c]);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 4; ++c) reg_fence32(r[c]);
            // Key columns at or left of the diagonal: all 128 off the diagonal tile (the
            // common case, warp-uniform, compiled without masking).
            const bool diag = (j == qt);
            const int lim = qrow + 1;
            auto sv = [&](int e) { return __uint_as_float(r[e >> 5][e & 31]); };
            float m4[4];
            auto row_max = [&](auto masked) {
                auto v = [&](int e) { return (!decltype(masked)::value || e < lim) ? sv(e) : -INFINITY; };
#pragma unroll
                for (int k = 0; k < 4; ++k) m4[k] = max3f(v(2 * k), v(2 * k + 1), -INFINITY);
#pragma unroll
                for (int e = 8; e < ATT_BKV; e += 8)
#pragma unroll
                    for (int k = 0; k < 4; ++k) m4[k] = max3f(m4[k], v(e + 2 * k), v(e + 2 * k + 1));
            };
            if (diag)
                row_max(std::true_type{});
            else
                row_max(std::false_type{});
            const float mx = fmaxf(max3f(m4[0], m4[1], m4[2]), m4[3]);
            bool rescale = false;
            float alpha = 1.0f;
            if (j == 0) {
                m = mx;
            } else if ((mx - m) * c2 > ATT_RESCALE_LOG2) {
                alpha = ex2_approx((m - mx) * c2);
                m = mx;
                l *= alpha;
                rescale = true;
            }
            // P = exp2(s c2 - m c2); column pair k (keys 2k, 2k+1) packed as bf16x2 into word k
            // of r (word k <= 2k has been read by then).
            const float2 c2v = make_float2(c2, c2);
            const float2 nmb = make_float2(-m * c2, -m * c2);
            float2 s4[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) s4[k] = make_float2(0.0f, 0.0f);
            auto exp_pack = [&](auto masked) {
#pragma unroll
                for (int k = 0; k < ATT_BKV / 2; ++k) {
                    const float2 x = fma2(make_float2(sv(2 * k), sv(2 * k + 1)), c2v, nmb);
                    float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                    if (decltype(masked)::value) {
                        p.x = 2 * k < lim ? p.x : 0.0f;
                        p.y = 2 * k + 1 < lim ? p.y : 0.0f;
                    }
                    s4[k & 3] = add2(s4[k & 3], p);
                    r[k >> 5][k & 31] = pack_bf16x2(p.x, p.y);
                }
            };
            if (diag)
                exp_pack(std::true_type{});
            else
                exp_pack(std::false_type{});
            const float2 s2 = add2(add2(s4[0], s4[1]), add2(s4[2], s4[3]));
            l += s2.x + s2.y;
            // P_g into the first 64 columns of S_g (the A operand of PV).
            tmem_st32(s_addr, r[0]);
            tmem_st32(s_addr + 32, r[1]);
            // Rows whose max rose: O_g *= alpha in TMEM before the next PV adds to it (the
            // last PV_g is complete: s_full covered it).
            if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int c = 0; c < NB; ++c) {
                    uint32_t o[32];
                    tmem_ld32(o_addr + c * 32, o);
                    tmem_wait_ld();
                    reg_fence32(o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(o_addr + c * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[g]);
        }
        // O / l after the last PV, through shared memory and TMA stores: each warp stages its 32
        // rows as NB 32 x 32 boxes (64-byte swizzle: 16-byte piece j of row r at j ^ ((r >> 1) & 3))
        // in the Q tile's space, which no product reads any more, and stores them whole.
        if (ok && ng > 0 && wait_all(&o_full[g], 0)) {
            tc_fence_after();
            const float inv = 1.0f / l;
            uint8_t* stg = sQ + g * Cfg::Q_BYTES + q * (NB * 2048);
            const int sw = (lane >> 1) & 3;
#pragma unroll 1
            for (int c = 0; c < NB; ++c) {
                uint32_t o[32];
                tmem_ld32(o_addr + c * 32, o);
                tmem_wait_ld();
                reg_fence32(o);
                uint8_t* row = stg + c * 2048 + lane * 64;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    *reinterpret_cast<uint4*>(row + ((v ^ sw) << 4)) = make_uint4(
                        pack_bf16x2(__uint_as_float(o[8 * v]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                        pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                        pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                        pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
            }
            fence_proxy_async_smem();  // the stores are read by TMA (async proxy)
            __syncwarp();
            if (lane == 0) {
                for (int c = 0; c < NB; ++c)
                    tma_store_2d(&tmO, stg + c * 2048, head * D + c * 32, row_base + qt * ATT_BQ + q * 32);
                bulk_commit_group();
                bulk_wait_group<0>();  // written before the CTA exits
            }
            __syncwarp();
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
static cudaError_t launch_attn(const CUtensorMap& tmQKV, const CUtensorMap& tmO, const AttnArgs& a, cudaStream_t s) {
    using Cfg = AttnCfg<D>;
    auto kern = attn_fwd_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    e = launch_pdl(kern, dim3(a.b * a.heads * a.npairs), dim3(ATT_THREADS), Cfg::SMEM_BYTES, s, tmQKV, tmO, a);
    return e != cudaSuccess ? e : cudaGetLastError();
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
    int b1f = 0;
    if (!make_tmap_bf16(&m1.a, X, h, T, h, 64, BM) || !(b1f = make_tmap_mn_operand(&m1.b, Wqkv, 3 * h, h, 3 * h)) ||
        !make_tmap_bf16_out(&m1.o0, QKV, 3 * h, T, 3 * h))
        return MP_ERR_CUDA;
    GemmArgs a1{};
    a1.pr.M = static_cast<int>(T);
    a1.pr.N = 3 * h;
    a1.pr.num_m_blocks = ceil_div(T, 2 * BM);
    a1.pr.num_units = a1.pr.num_m_blocks * ceil_div(3 * h, 256);
    a1.pr.n_fastest = n_fastest_order(Tb * h, hb * 3 * h);
    a1.pr.kb_end = h / BK;
    a1.pr.b_mn = b1f;
    a1.tiles_per_unit = 1;
    a1.status = d_status;
    a1.budget_ns = budget;
    if (launch_gemm_tc<256, EPI_STORE, 4>(m1, a1, sms, cs) != cudaSuccess) return MP_ERR_CUDA;

    // Per-head causal attention.
    CUtensorMap tq;
    CUtensorMap to;  // O in 32 x 32 boxes, 64-byte swizzle (the kernel's staging layout)
    if (!make_tmap_bf16_sw64(&tq, QKV, 3 * h, T, 3 * h, 32, ATT_BQ) || !make_tmap_bf16_out(&to, O, h, T, h))
        return MP_ERR_CUDA;
    AttnArgs aa{};
    aa.O = reinterpret_cast<__nv_bfloat16*>(O);
    aa.b = b;
    aa.s = s;
    aa.h = h;
    aa.heads = heads;
    aa.nq = s / ATT_BQ;
    aa.npairs = (aa.nq + 1) / 2;
    aa.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(d));
    aa.status = d_status;
    aa.budget_ns = budget;
    cudaError_t e = d == 64 ? launch_attn<64>(tq, to, aa, cs) : launch_attn<96>(tq, to, aa, cs);
    if (e != cudaSuccess) return MP_ERR_CUDA;

    // out = sum_i O_i Wo_i: the K-loop runs over the heads' columns in ascending order, i.e.
    // shard 0's heads, then shard 1's, ... (the g sum; a K block may span two shards).
    TmapSet m3{};
    int b3f = 0;
    if (!make_tmap_bf16(&m3.a, O, h, T, h, 64, BM) || !(b3f = make_tmap_mn_operand(&m3.b, Wo, h, h, h)) ||
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
    a3.pr.b_mn = b3f;
    a3.tiles_per_unit = 1;
    a3.status = d_status;
    a3.budget_ns = budget;
    if (launch_gemm_tc<256, EPI_STORE, 4>(m3, a3, sms, cs) != cudaSuccess) return MP_ERR_CUDA;
    return MP_OK;
}
