// Persistent, warp-specialised tcgen05 GEMM for sm_103a with fused epilogues,
// run by CTA pairs (thread-block clusters of 2, tcgen05 cta_group::2).
//
//   C[M, N] = sum_k  A(m, k) * B(k, n),   bf16 inputs, fp32 accumulation in TMEM.
//
// A pair computes a 256 x BN output tile: CTA r (r = rank in the pair) owns rows
// [256 i + 128 r, +128) of the tile and holds in its shared memory those 128 rows
// of A and columns [BN/2 r, +BN/2) of B; the leader (r = 0) issues one
// tcgen05.mma with M = 256 that reads both CTAs' shared memory and writes each
// CTA's 128 x BN accumulator into that CTA's TMEM. Per SM this halves the B
// traffic, so a stage is 32 KB (BN = 256) and the ring holds 6 or 7 stages.
//
// Grid = 2 x the fewest co-resident pairs that finish the units in the fewest
// rounds; 64 + 32*NE threads per CTA:
//   warp 0      TMA producer (one lane) in each CTA: its A and B halves per
//               stage, completion signalled on the leader's `full` barrier.
//   warp 1      TMEM allocator (whole warp, both CTAs) and, in the leader only,
//               the MMA issuer: the whole warp runs the issue loop (so descriptors
//               and addresses stay in uniform registers) and one elected lane issues
//               4 x tcgen05.mma (K = 16) per stage into one of two TMEM accumulators
//               (BN fp32 columns each per CTA); its commits arrive on the `empty` /
//               `tmem full` barriers of both CTAs.
//   warps 2..   NE epilogue warps (4 or 8) in each CTA: tcgen05.ld 32 rows x 32
//               columns (TMEM lane quarter = warp % 4, thread = output row; with 8
//               warps two warps share a quarter and split the columns), fused math,
//               then bf16 rows staged in a 64-byte-swizzled shared box per warp and
//               written by TMA stores (32x32 boxes), or cross-entropy partials.
//               An accumulator is
//               handed back (to the leader) as soon as its last columns are in
//               registers, so it overlaps the next tile's MMAs.
//
// A work unit is one 256-row block and `tiles_per_unit` consecutive BN-wide
// column tiles (1 for plain GEMMs; several for the cross-entropy, whose epilogue
// keeps running per-row statistics over the unit). The K-loop runs over K
// blocks [kb_begin, kb_end) in ascending order, so a K range that covers shards
// 0..t-1 of a row-parallel GEMM sums the shard partials in shard order inside
// the accumulator: the g / f all-reduce of the method becomes the K-loop.
//
// Operand majorness: K-major = K contiguous in global memory (row-major [rows, K]),
// MN-major = M (or N) contiguous (row-major [K, rows]); both are loaded by TMA
// with the 128-byte swizzle and described to the MMA without any transpose copy.
// An MN-major operand's stage is two 64-column blocks per CTA, loaded by one 3-D
// box (majorness flag 2) or two 2-D boxes (flag 1).
//
// Every mbarrier wait is bounded by a time budget; on expiry the kernel sets
// MP_DEV_TIMEOUT in the status word, raises a CTA-wide abort flag, lets its own
// TMA loads and MMAs in flight finish (bounded), meets its peer at the cluster
// barrier, frees TMEM and returns.
#pragma once

#include <cuda_bf16.h>

#include <cstdlib>

#include "mptp_launch.cuh"
#include "mptp_ptx.cuh"

namespace mptp {

constexpr int BM = 128;       // rows per CTA (a pair covers 2 * BM)
constexpr int BK = 64;        // K per stage: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int STG_BYTES_PER_WARP = 2 * 2048;  // two 32x32 bf16 staging boxes
constexpr uint32_t DEV_TIMEOUT = 0x1u;
constexpr uint32_t DEV_TARGET_RANGE = 0x2u;
constexpr unsigned long long DRAIN_BUDGET_NS = 1000000000ull;  // 1 s
constexpr unsigned long long ABORT_SETTLE_NS = 50000ull;       // in-flight copies land well within this

enum EpiKind : int {
    EPI_STORE = 0,  // o0 = bf16(acc)
    EPI_GELU = 1,   // o0 = bf16(GeLU(acc)); o1 (when has_out1) = bf16(acc)
    EPI_DGELU = 2,  // o0 = bf16(acc * GeLU'(aux)), aux = bf16 U
    EPI_CE = 3,     // per-row online max / sum-exp / target logit over the unit
    EPI_DZ = 4,     // o0 = bf16(dloss * (exp(acc - lse) - [col == target])), 0 on padding columns
    EPI_ACC = 5,    // fp32 accumulation across launches into `acc` (tensor map o1); the last launch
                    // stores bf16 o0
};

enum AccMode : int {
    ACC_FIRST = 0,  // acc = C          (TMA store of fp32 boxes through o1)
    ACC_MID = 1,    // acc += C         (TMA reduction: the add is done at L2, no read back)
    ACC_LAST = 2,   // o0 = bf16(acc + C)
    ACC_ONLY = 3,   // o0 = bf16(C)
};

// The GEMM of a launch.
struct ProbInfo {
    int M, N;                 // output extent (masking of the ragged tails)
    int num_m_blocks;         // ceil(M / (2 * BM)): 256-row blocks, one per pair tile
    int num_units;            // num_m_blocks * unit columns
    int n_fastest;            // unit order: 0 = row blocks fastest, 1 = column units fastest
    int kb_begin, kb_end;     // K blocks (of BK) to accumulate, ascending
    int a_mn, b_mn;           // operand majorness: 0 = K contiguous; 1 = M (N) contiguous, loaded as
                              // 64-wide 2-D boxes; 2 = the same through a 3-D map (one box per stage)
};

struct GemmArgs {
    ProbInfo pr;
    int tiles_per_unit;       // BN-wide column tiles per unit (cross-entropy: several)
    // epilogue operands that are not written through tensor maps
    const __nv_bfloat16* aux; // U for GeLU'
    long long ld_aux;
    int has_out1;             // GeLU: also store U (tensor map o1)
    // cross-entropy epilogues
    const int32_t* target;
    float* ws;                // [P][3][M] fp32: max, sum-exp, target logit
    int v_valid;
    int col_off;              // global vocabulary index of output column 0 (backward: shard offset)
    const float* lse;         // backward: per-token log-sum-exp (NaN = invalid target)
    const float* dloss;       // backward: per-token upstream gradient
    // fp32 accumulation across launches
    float* acc;
    long long ld_acc;
    int acc_mode;
    uint32_t* status;         // nullable
    unsigned long long budget_ns;
};

// Tensor maps of a launch: the two operands and the epilogue outputs.
struct TmapSet {
    CUtensorMap a;
    CUtensorMap b;
    CUtensorMap o0;
    CUtensorMap o1;
};

constexpr size_t SMEM_LIMIT = 232448;  // opt-in shared memory per block on sm_103

template <int BN_, int EPI, int NE_>
struct GemmCfg {
    static constexpr int BN = BN_;             // tile width of the pair
    static constexpr int BNH = BN / 2;         // B columns held per CTA
    static constexpr int NE = NE_;
    static constexpr int NUM_THREADS = 64 + 32 * NE;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BNH * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr uint32_t TMEM_COLS = BN <= 128 ? 256 : 512;  // two accumulators, power of two
    // staging per epilogue warp: two 32 x 32 boxes, bf16 (2 KB each) or, accumulating, fp32 (4 KB)
    static constexpr int STG_PER_WARP = EPI == EPI_ACC ? 2 * 4096 : STG_BYTES_PER_WARP;
    static constexpr int STG_BYTES = EPI == EPI_CE ? 0 : NE * STG_PER_WARP;
    static constexpr int MAX_STAGES = 8;
    static constexpr int FIT_STAGES = static_cast<int>((SMEM_LIMIT - 1024 - 512 - STG_BYTES) / STAGE_BYTES);
    static constexpr int STAGES = FIT_STAGES < MAX_STAGES ? FIT_STAGES : MAX_STAGES;
    static constexpr int NUM_BARS = 2 * STAGES + 5;  // full, empty, tmem full x2, tmem empty x2, drain
    static constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + STG_BYTES + 8 * NUM_BARS + 16;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory per block");
    static_assert(STAGES >= 4, "pipeline depth");
    static_assert(BN == 128 || BN == 224 || BN == 256, "pair tile width");
    static_assert(BN != 224 || NE == 4, "224-wide tiles: four epilogue warps (7 column chunks each)");
    static_assert(NE == 4 || NE == 8, "4 or 8 epilogue warps");
    static_assert(EPI != EPI_CE || NE == 4, "cross-entropy epilogue keeps one thread per row");
    static_assert(EPI != EPI_ACC || NE == 4, "accumulating epilogue uses four warps");
};

struct Ctl {
    uint32_t* status;
    volatile uint32_t* abort_flag;
    unsigned long long budget_ns;
};

// Bounded wait. false = gave up (budget spent or another role of this CTA aborted).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, const Ctl& c) {
    auto probe = [&]() { return mbar_try_wait(bar, parity); };
    if (probe()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (probe()) return true;
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

__device__ __forceinline__ void spin_ns(unsigned long long ns) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < ns) {
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Standard normal CDF and density from one exponential, with erf taken from the
// rational approximation of Abramowitz & Stegun, Handbook of Mathematical
// Functions, eq. 7.1.26 (|error of erf| <= 1.5e-7 for x >= 0):
//   erf(x) = 1 - (a1 s + a2 s^2 + a3 s^3 + a4 s^4 + a5 s^5) e^{-x^2},  s = 1 / (1 + p x).
// With x = |u| / sqrt 2 and q = (1 - erf(x)) / 2, Phi(u) = 1 - q for u >= 0 and q
// for u < 0; phi(u) = e^{-x^2} / sqrt(2 pi) reuses the same exponential, and
// GeLU(u) = u Phi(u) = max(u, 0) - |u| q. In fp32 with the hardware ex2/rcp
// approximations the CDF error stays below 1e-6, far under the bf16 output spacing.
// Two values at a time: the arithmetic runs as packed two-lane instructions.
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
struct NormalCdfPdf2 {
    float2 a;      // |u|
    float2 nq;     // -q = -(1 - erf(|u| / sqrt 2)) / 2
    float2 e;      // e^{-u^2 / 2}
};
__device__ __forceinline__ NormalCdfPdf2 normal_tail2(float2 u) {
    constexpr float P_OVER_SQRT2 = 0.23164189f;   // 0.3275911 / sqrt 2
    constexpr float NEG_HALF_LOG2E = -0.72134752f;  // e^{-u^2/2} = 2^{u^2 * this}
    // -a_k / 2, so that the polynomial times e gives -q directly
    constexpr float C1 = -0.127414796f, C2 = 0.142248368f, C3 = -0.7107068705f, C4 = 0.7265760135f,
                    C5 = -0.5307027145f;
    auto dup = [](float c) { return make_float2(c, c); };
    NormalCdfPdf2 r;
    r.a = make_float2(fabsf(u.x), fabsf(u.y));
    const float2 d = fma2(r.a, dup(P_OVER_SQRT2), dup(1.0f));
    const float2 s = make_float2(rcp_approx(d.x), rcp_approx(d.y));
    float2 poly = fma2(s, dup(C5), dup(C4));
    poly = fma2(poly, s, dup(C3));
    poly = fma2(poly, s, dup(C2));
    poly = fma2(poly, s, dup(C1));
    poly = mul2(poly, s);
    const float2 w = mul2(mul2(u, u), dup(NEG_HALF_LOG2E));
    r.e = make_float2(ex2_approx(w.x), ex2_approx(w.y));
    r.nq = mul2(poly, r.e);
    return r;
}
// GeLU(u) = max(u, 0) - |u| q.
__device__ __forceinline__ float2 gelu2(float2 u) {
    const NormalCdfPdf2 t = normal_tail2(u);
    return fma2(t.a, t.nq, make_float2(fmaxf(u.x, 0.0f), fmaxf(u.y, 0.0f)));
}
// GeLU'(u) = Phi(u) + u phi(u).
__device__ __forceinline__ float2 gelu_prime2(float2 u) {
    constexpr float INV_SQRT_2PI = 0.39894228040143268f;
    const NormalCdfPdf2 t = normal_tail2(u);
    const float2 cdf = make_float2(u.x >= 0.0f ? 1.0f + t.nq.x : -t.nq.x, u.y >= 0.0f ? 1.0f + t.nq.y : -t.nq.y);
    return fma2(u, mul2(t.e, make_float2(INV_SQRT_2PI, INV_SQRT_2PI)), cdf);
}

// One warp writes its 32 rows x 32 columns of bf16 (thread = row) into one of its
// two staging boxes, in the 64-byte-swizzled layout the output tensor map uses
// (16-byte chunk j of row r sits at chunk j ^ ((r >> 1) & 3)), then lane 0 stores
// the box with TMA at (x = first column, y = first row). Out-of-range rows and
// columns are clipped by the TMA unit.
__device__ __forceinline__ void stage_and_store(const CUtensorMap* map, uint8_t* stg, int& sbuf, int lane,
                                                const uint32_t (&p)[16], int x, int y) {
    if (lane == 0) bulk_wait_group_read<1>();  // the store that last used this box has read it
    __syncwarp();
    uint8_t* row = stg + sbuf * 2048 + lane * 64;
    const int sw = (lane >> 1) & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map, stg + sbuf * 2048, x, y);
        bulk_commit_group();
    }
    sbuf ^= 1;
}

// The fp32 form: 32 rows x 32 columns (128-byte rows, 16-byte chunk j of row r at chunk
// j ^ (r & 7), the 128-byte swizzle) in one of the warp's two 4 KB boxes, then lane 0 either
// stores the box or adds it into global memory with a TMA reduction.
__device__ __forceinline__ void stage_and_store_f32(const CUtensorMap* map, uint8_t* stg, int& sbuf, int lane,
                                                    const uint32_t (&v)[32], int x, int y, bool add) {
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    uint8_t* row = stg + sbuf * 4096 + lane * 128;
    const int sw = lane & 7;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (add)
            tma_reduce_add_2d(map, stg + sbuf * 4096, x, y);
        else
            tma_store_2d(map, stg + sbuf * 4096, x, y);
        bulk_commit_group();
    }
    sbuf ^= 1;
}

__device__ __forceinline__ void decode_unit(const ProbInfo& p, int lu, int& m_blk, int& ucol) {
    if (p.n_fastest) {
        const int ncols = p.num_units / p.num_m_blocks;
        ucol = lu % ncols;
        m_blk = lu / ncols;
    } else {
        m_blk = lu % p.num_m_blocks;
        ucol = lu / p.num_m_blocks;
    }
}

template <int BN, int EPI, int NE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GemmCfg<BN, EPI, NE>::NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ TmapSet maps, const GemmArgs args) {
    using Cfg = GemmCfg<BN, EPI, NE>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int BNH = Cfg::BNH;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t* stg_base = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stg_base + Cfg::STG_BYTES);
    uint64_t* full_bar = bars;                // leader: both CTAs' loads of a stage landed
    uint64_t* empty_bar = bars + STAGES;      // each CTA: the pair's MMAs finished reading a stage
    uint64_t* tfull_bar = bars + 2 * STAGES;  // each CTA: accumulator ready
    uint64_t* tempty_bar = bars + 2 * STAGES + 2;  // leader: both CTAs' epilogues drained an accumulator
    uint64_t* drain_bar = bars + 2 * STAGES + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 2);   // one expect_tx arrival from each CTA's producer
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 2 * NE);  // every epilogue warp of both CTAs
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&maps.a);
        prefetch_tensormap(&maps.b);
        if (EPI != EPI_CE) prefetch_tensormap(&maps.o0);
        if ((EPI == EPI_GELU && args.has_out1) || (EPI == EPI_ACC && args.acc_mode <= ACC_MID))
            prefetch_tensormap(&maps.o1);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any cross-CTA arrival
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{args.status, abort_flag, args.budget_ns};
    // The set-up above overlaps the previous kernel's tail when this grid was launched as its
    // programmatic dependent; no global memory is touched before the previous grid completes.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const ProbInfo& p = args.pr;
            const CUtensorMap* tmA = &maps.a;
            const CUtensorMap* tmB = &maps.b;
            for (int u = pair; u < p.num_units && ok; u += num_pairs) {
                int m_blk, ucol;
                decode_unit(p, u, m_blk, ucol);
                const int n_blk0 = ucol * args.tiles_per_unit;
                const int arow = m_blk * 2 * BM + static_cast<int>(rank) * BM;  // this CTA's A rows
                for (int nt = 0; nt < args.tiles_per_unit && ok; ++nt) {
                    const int bcol = (n_blk0 + nt) * BN + static_cast<int>(rank) * BNH;  // this CTA's B columns
                    for (int kb = p.kb_begin; kb < p.kb_end; ++kb) {
                        if (!wait_bounded(&empty_bar[stage], phase ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[stage]), 0);
                        mbar_arrive_expect_tx_cluster(full_leader, Cfg::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * Cfg::A_BYTES;
                        uint8_t* b_dst = sB + stage * Cfg::B_BYTES;
                        if (p.a_mn == 2) {  // all 64-wide M blocks of the stage in one 3-D box
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
        }
    } else if (warp == 1) {
        if (leader) {
            // ---------------- MMA issuer (leader CTA) ----------------
            // The whole warp runs the issue loop, so that the operands stay warp-uniform; one
            // elected lane issues each product and commit. Waits are polled by every lane.
            auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
                const bool got = mbar_test_wait(bar, parity) || wait_bounded(bar, parity, ctl);
                return __all_sync(0xffffffffu, got) != 0;
            };
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tcount = 0;
            bool ok = true;
            const ProbInfo& p = args.pr;
            const bool a_mn = p.a_mn != 0, b_mn = p.b_mn != 0;
            for (int u = pair; u < p.num_units && ok; u += num_pairs) {
                const uint32_t idesc = make_idesc_bf16(2 * BM, BN, a_mn, b_mn);
                // Descriptor of a stage's first K slice; the k-th slice is that descriptor
                // advanced in its address field (>> 4) by 2048 B (MN-major) or 32 B (K-major).
                const uint32_t a_lbo = a_mn ? 8192u : 16u, b_lbo = b_mn ? 8192u : 16u;
                const uint64_t a_kstep = a_mn ? (2048u >> 4) : (32u >> 4);
                const uint64_t b_kstep = b_mn ? (2048u >> 4) : (32u >> 4);
                const uint64_t ad_base = make_sdesc_sw128(smem_u32(sA), a_lbo, 1024);
                const uint64_t bd_base = make_sdesc_sw128(smem_u32(sB), b_lbo, 1024);
                for (int nt = 0; nt < args.tiles_per_unit && ok; ++nt, ++tcount) {
                    const uint32_t buf = tcount & 1u;
                    const uint32_t tph = (tcount >> 1) & 1u;
                    if (!wait_all(&tempty_bar[buf], tph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + buf * BN;
                    // The issuing thread is on the critical path: one stage's four MMAs take 512
                    // tensor cycles, and everything else it does per stage must fit beside them.
                    // Stage descriptors are the stage-0 ones advanced in their address field.
                    for (int kb = p.kb_begin; kb < p.kb_end; ++kb) {
                        if (!wait_all(&full_bar[stage], phase)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad0 = ad_base + static_cast<uint64_t>(stage) * (Cfg::A_BYTES >> 4);
                        const uint64_t bd0 = bd_base + static_cast<uint64_t>(stage) * (Cfg::B_BYTES >> 4);
                        umma_bf16_pair_elect(d_tmem, ad0, bd0, idesc, kb > p.kb_begin ? 1u : 0u);
#pragma unroll
                        for (int k = 1; k < BK / UMMA_K; ++k)
                            umma_bf16_pair_acc_elect(d_tmem, ad0 + k * a_kstep, bd0 + k * b_kstep, idesc);
                        umma_commit_pair_multicast_elect(&empty_bar[stage], 0x3);  // frees the stage in both CTAs
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!ok) break;
                    umma_commit_pair_multicast_elect(&tfull_bar[buf], 0x3);  // accumulators ready in both CTAs
                }
            }
            // Every MMA of the pair must finish before either CTA frees TMEM or exits.
            umma_commit_pair_elect(drain_bar);
            wait_drain(drain_bar, 0, args.status);
        }
    } else {
        // ---------------- epilogue (NE warps, both CTAs) ----------------
        constexpr int CHUNKS = BN / 32;
        constexpr int MY_CHUNKS = CHUNKS / (NE / 4);
        const int e = warp - 2;                      // epilogue warp index
        const int q = warp & 3;                      // TMEM lane quarter this warp may access
        const int c_begin = (e >> 2) * MY_CHUNKS;    // column half (8 warps) or all columns (4)
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* stg = stg_base + e * Cfg::STG_PER_WARP;
        int sbuf = 0;
        uint32_t tcount = 0;
        bool ok = true;
        const ProbInfo& p = args.pr;
        const CUtensorMap* tmO0 = &maps.o0;
        for (int u = pair; u < p.num_units && ok; u += num_pairs) {
            int m_blk, ucol;
            decode_unit(p, u, m_blk, ucol);
            const int n_blk0 = ucol * args.tiles_per_unit;
            const int row0 = m_blk * 2 * BM + static_cast<int>(rank) * BM + q * 32;  // this warp's 32 rows
            const int row = row0 + lane;
            const bool row_ok = row < p.M;
            // cross-entropy running state (natural-log units)
            float run_m = -INFINITY, run_s = 0.0f, z_tgt = 0.0f;
            int tgt = -1;
            if ((EPI == EPI_CE || EPI == EPI_DZ) && row_ok) tgt = args.target[row];
            // cross-entropy backward row state: lse in log2 units, upstream gradient
            float lse2 = 0.0f, dl = 0.0f;
            if (EPI == EPI_DZ && row_ok) {
                lse2 = args.lse[row] * 1.4426950408889634f;
                dl = args.dloss[row];
                if (!(lse2 == lse2)) {  // invalid target (NaN log-sum-exp): no gradient for this token
                    lse2 = 0.0f;
                    dl = 0.0f;
                    tgt = -1;
                }
            }

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
                // Chunk pipeline: the TMEM load (and, for GeLU', the U row segment) of
                // chunk cc+1 is in flight while chunk cc is computed and stored.
                auto issue = [&](int cc, uint32_t (&rr)[32], uint32_t (&uu)[16]) {
                    const int c = c_begin + cc;
                    if constexpr (EPI == EPI_DGELU) {
                        const int col0 = n_blk * BN + c * 32;
                        if (row_ok && col0 < p.N) {
                            const uint4* src = reinterpret_cast<const uint4*>(args.aux + row * args.ld_aux + col0);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint4 w = src[j];
                                uu[4 * j + 0] = w.x;
                                uu[4 * j + 1] = w.y;
                                uu[4 * j + 2] = w.z;
                                uu[4 * j + 3] = w.w;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) uu[j] = 0u;
                        }
                    }
                    tmem_ld32(tmem_base + lane_addr + buf * BN + c * 32, rr);
                };
                auto finish = [&](int cc, const uint32_t (&r)[32], const uint32_t (&uw)[16]) {
                    const int c = c_begin + cc;
                    const int col0 = n_blk * BN + c * 32;
                    if (col0 >= p.N) return;  // ragged N tail (whole 32-column chunks)
                    // One 32-column bf16 row segment per thread, staged and TMA-stored.
                    if constexpr (EPI == EPI_STORE) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                        stage_and_store(tmO0, stg, sbuf, lane, pk, col0, row0);
                    } else if constexpr (EPI == EPI_GELU) {
                        uint32_t pk[16];
                        if (args.has_out1) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                            stage_and_store(&maps.o1, stg, sbuf, lane, pk, col0, row0);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float2 g = gelu2(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])));
                            pk[j] = pack_bf16x2(g.x, g.y);
                        }
                        stage_and_store(tmO0, stg, sbuf, lane, pk, col0, row0);
                    } else if constexpr (EPI == EPI_DGELU) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float2 gp = gelu_prime2(make_float2(bf16_lo(uw[j]), bf16_hi(uw[j])));
                            const float2 g = mul2(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), gp);
                            pk[j] = pack_bf16x2(g.x, g.y);
                        }
                        stage_and_store(tmO0, stg, sbuf, lane, pk, col0, row0);
                    } else if constexpr (EPI == EPI_DZ) {
                        // dZ = dloss * (softmax - onehot) on valid columns, 0 on padding.
                        constexpr float LOG2E = 1.4426950408889634f;
                        const int gcol0 = args.col_off + col0;
                        const int lim = args.v_valid - gcol0;
                        const unsigned dt = static_cast<unsigned>(tgt - gcol0);
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float g[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const int jj = 2 * j + e2;
                                float pr = ex2_approx(fmaf(__uint_as_float(r[jj]), LOG2E, -lse2));
                                if (static_cast<int>(dt) == jj && dt < 32u) pr -= 1.0f;
                                g[e2] = (jj < lim && dl != 0.0f) ? dl * pr : 0.0f;
                            }
                            pk[j] = pack_bf16x2(g[0], g[1]);
                        }
                        stage_and_store(tmO0, stg, sbuf, lane, pk, col0, row0);
                    } else if constexpr (EPI == EPI_ACC) {
                        if (args.acc_mode == ACC_ONLY || args.acc_mode == ACC_LAST) {
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                            if (args.acc_mode == ACC_LAST && row_ok) {
                                const float4* src = reinterpret_cast<const float4*>(args.acc + row * args.ld_acc + col0);
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const float4 a4 = src[j];
                                    v[4 * j] += a4.x;
                                    v[4 * j + 1] += a4.y;
                                    v[4 * j + 2] += a4.z;
                                    v[4 * j + 3] += a4.w;
                                }
                            }
                            uint32_t pk[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                            stage_and_store(tmO0, stg, sbuf, lane, pk, col0, row0);
                        } else {
                            stage_and_store_f32(&maps.o1, stg, sbuf, lane, r, col0, row0, args.acc_mode == ACC_MID);
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
                                const float ev = ex2_approx(fmaf(__uint_as_float(r[j]), LOG2E, -mb));
                                acc += (j < lim) ? ev : 0.0f;
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
                };
                // Last columns of this accumulator are in registers: hand it back to the leader's MMA.
                auto release = [&]() {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty_bar[buf]), 0));
                };
                uint32_t ra[32], rb[32], ua[16], ub[16];
                issue(0, ra, ua);
#pragma unroll 1
                for (int cc = 0; cc < MY_CHUNKS; cc += 2) {
                    tmem_ld_wait(ra);
                    if (cc + 1 < MY_CHUNKS)
                        issue(cc + 1, rb, ub);
                    else
                        release();
                    finish(cc, ra, ua);
                    if (cc + 1 < MY_CHUNKS) {
                        tmem_ld_wait(rb);
                        if (cc + 2 < MY_CHUNKS)
                            issue(cc + 2, ra, ua);
                        else
                            release();
                        finish(cc + 1, rb, ub);
                    }
                }
            }
            if (!ok) break;
            if constexpr (EPI == EPI_CE) {
                if (row_ok) {
                    float* w = args.ws + static_cast<long long>(ucol) * 3 * p.M;
                    w[row] = run_m;
                    w[p.M + row] = run_s;
                    w[2 * p.M + row] = z_tgt;
                }
            }
        }
        // All of this warp's TMA stores must have landed before the kernel ends.
        if (EPI != EPI_CE && lane == 0) bulk_wait_group<0>();
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    // After an abort some TMA loads issued by this CTA may never have been consumed;
    // give them a fixed time to land before this CTA (or, via the cluster barrier,
    // the leader whose barrier they signal) can exit. The flag is final here.
    if (*abort_flag) {
        if (threadIdx.x == 0) spin_ns(ABORT_SETTLE_NS);
        __syncthreads();
    }
    cluster_sync_all();  // the leader's MMAs (which read this CTA's shared memory) are done
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
}

// Number of CTA pairs that can be resident at once for one kernel instantiation.
template <int BN, int EPI, int NE>
inline int resident_pairs(int num_sms) {
    using Cfg = GemmCfg<BN, EPI, NE>;
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tc_kernel<BN, EPI, NE>, &cfg) != cudaSuccess ||
        clusters <= 0) {
        cudaGetLastError();
        clusters = num_sms / 2;
    }
    if (clusters > num_sms / 2) clusters = num_sms / 2;
    if (dev >= 0 && dev < 64) cached[dev] = clusters;
    return clusters;
}

// Host-side launcher: grid = 2 x min(units, resident pairs, max_pairs if > 0), one CTA per SM.
template <int BN, int EPI, int NE>
inline cudaError_t launch_gemm_tc(const TmapSet& maps, const GemmArgs& args, int num_sms, cudaStream_t stream,
                                  int max_pairs = 0) {
    using Cfg = GemmCfg<BN, EPI, NE>;
    auto kern = gemm_tc_kernel<BN, EPI, NE>;
    if (BN % 128 != 0 && args.pr.b_mn) return cudaErrorInvalidValue;  // MN-major B needs 64-column boxes per CTA
    if (args.pr.b_mn == 2 && BN != 256) return cudaErrorInvalidValue;  // 3-D B box: two 64-column blocks per CTA
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    int pairs = resident_pairs<BN, EPI, NE>(num_sms);
    if (max_pairs > 0 && max_pairs < pairs) pairs = max_pairs;
    int use = args.pr.num_units < pairs ? args.pr.num_units : pairs;
    // As few pairs as give the same number of rounds of units: the same time, and the idle
    // SMs leave power headroom to the busy ones under the board's power cap.
    if (use > 0) {
        const int rounds = (args.pr.num_units + use - 1) / use;
        use = (args.pr.num_units + rounds - 1) / rounds;
    }
    if (use <= 0) return cudaSuccess;
    e = launch_pdl(kern, dim3(2 * use), dim3(Cfg::NUM_THREADS), Cfg::SMEM_BYTES, stream, maps, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mptp
