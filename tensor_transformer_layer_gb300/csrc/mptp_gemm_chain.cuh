// A chain of dependent GEMMs in one persistent launch: the MLP block's forward
// (K1 then K2) or backward (K3, then K4, K5a, K5b), or one vocabulary shard of the
// cross-entropy backward (K10, then K12 and K11), with no kernel boundary between
// them.
//
// Why. Each separate GEMM launch ends in a part-empty last round of tiles, an
// epilogue with nothing to hide behind and a teardown, and the next launch
// cannot load its first operand until every CTA of the previous one has
// finished. At small layers (T = 2048 tokens, h = 1536: 20-26 us of MMA work a
// GEMM) that costs 7-10 us a launch. Here the units of all GEMMs of a direction
// form one list in a fixed order. The host gives each CTA pair its positions in the
// list (a greedy list-scheduling pass over the pairs, cached per shape; a list too long
// for the tables runs as separate launches instead, although the kernel can also take
// positions round-robin, pair p taking p, p + P, p + 2P, ...). A unit that reads another GEMM's output
// waits, once before its first load, for the part of it that it reads:
//   K2 unit (row block m, column tile n)   needs K1's row block m
//   K4 unit (m, n)                         needs K3's row block m
//   K5a unit (h block i, f tile j)         needs K3's column tile j
//   K5b                                    needs nothing (Y and dZ are inputs)
//   K12 unit (m, n)                        needs K10's row block m (dZ rows)
//   K11 unit (i, j)                        needs K10's column tile i (dZ columns)
// Each epilogue warp of the producing GEMM adds one to its tile's row-block counter
// and column-tile counter after the tile's TMA stores have completed (release adds);
// the consumer's TMA producer polls one counter with acquire loads. Every output
// tile is still computed by one CTA pair over the same ascending K-loop as the
// separate kernels, so the results are bitwise the same. (Waiting per 256-column
// tile instead, streaming behind the producer GEMM, was measured: the acquire
// fences it puts on the producer thread's path every few K blocks cost more than
// the earlier start gained.)
//
// No hand-out. Every warp role of both CTAs of a pair walks the same list
// positions and decodes them from tables in its own shared memory, so the pair
// needs no communication beyond the pipeline barriers the separate kernel has.
// (A work queue claimed with an atomic and handed to the roles through shared
// memory was measured first: the release-ordered arrives it needs on the
// producer's and the MMA warp's paths stall them until their outstanding memory
// operations complete, and it ran 30-40 % slower per unit.)
//
// Progress. Every unit's dependencies come earlier in the list, and each pair
// runs its units in list order. The lowest-numbered unfinished unit therefore has
// all of its inputs, and its pair has finished every earlier unit of its own, so
// it is never blocked, provided its CTAs are resident. The grid is sized to the
// pairs the device holds at once (one CTA per SM); CTAs that start before the
// previous kernel in the stream has left the SMs wait only for that kernel, which
// does not depend on them. A kernel running beside this one on another stream can
// keep a pair off the device while the resident pairs wait for it; every wait is
// bounded (MP_DEV_TIMEOUT, as in mptp_gemm.cuh), so that ends the launch with an
// error instead of a hang, and the entry points document that these launches run
// alone on the device.
//
// Workspace (caller-owned, zero before first use): word 1 counts the CTAs that have
// finished; after the control words come the row-block counters and the column-tile
// counters of the first GEMM (K1 or K3). The last CTA to finish zeroes all of it
// again, so consecutive launches on one stream can share it.
#pragma once

#include <type_traits>

#include "mptp.h"
#include "mptp_gemm.cuh"

namespace mptp {

constexpr int CHAIN_MAX_PROBS = 4;
constexpr int CHAIN_MAX_SEGS = 64;
constexpr int CHAIN_MAX_PAIRS = 96;      // CTA pairs a launch may have (GB300: 76)
constexpr int CHAIN_MAX_SCHED = 4096;    // list positions a precomputed schedule may hold
constexpr int CHAIN_MAX_PER_PAIR = 480;  // ... and one pair's share of them
constexpr int CHAIN_CTL_WORDS = 64;  // word 1: finished CTAs; padding to 256 bytes
constexpr int CHAIN_BN = 256;
static_assert(CHAIN_BN == 4 * BK, "a dependency tile is four K blocks");
constexpr int CHAIN_FWD = 0;         // problem 0: GeLU epilogue (optionally also U), others: store
constexpr int CHAIN_BWD = 1;         // problem 0: GeLU' epilogue (reads U), others: store
// Cross-entropy backward, one vocabulary shard: problem 0 (K10) turns recomputed logits into dZ
// (softmax minus one-hot, times the upstream gradient), problem 1 (K12) accumulates dX across the
// shards' launches in fp32, problem 2 (K11) stores dE.
constexpr int CHAIN_CE = 2;

enum ChainDep : int {
    DEP_NONE = 0,
    DEP_ROWS = 1,  // unit (m, n) reads problem 0's row block m (every column tile of it)
    DEP_COLS = 2,  // unit (i, j) reads problem 0's column tile j (every row block of it)
    DEP_COLS_M = 3,  // unit (i, j) reads problem 0's column tile i (its row block indexes them)
};

struct ChainProb {
    ProbInfo pr;   // M, N, row blocks, units, K range, operand majorness (pr.n_fastest not used here)
    int ncols;     // column tiles a row block has
    int group;     // unit order: row blocks in groups of `group`, row blocks fastest within a group
    int dep;       // ChainDep on problem 0
};

// A run of consecutive units (in a problem's own order) in the chain's list.
struct ChainSeg {
    int prob, first, count;
};

struct ChainArgs {
    ChainProb p[CHAIN_MAX_PROBS];
    ChainSeg seg[CHAIN_MAX_SEGS];
    int nsegs;
    int total_units;
    uint32_t* ctl;            // workspace control words (word 1: CTAs finished)
    uint32_t* row_done;       // workspace: per row block of problem 0, epilogue warps that finished a tile
    uint32_t* col_done;       // workspace: per column tile of problem 0, the same count
    int num_counters;         // row_done and col_done are one array of this many words
    const __nv_bfloat16* aux;  // backward: U (GeLU' operand), row pitch ld_aux
    long long ld_aux;
    int has_out1;             // forward: problem 0 also stores U through its o1 map
    // cross-entropy backward (CHAIN_CE)
    const int32_t* target;    // [T] target id of each token
    const float* lse;         // [T] log-sum-exp of each token's logits (NaN: no gradient)
    const float* dloss;       // [T] upstream gradient of each token's loss
    int v_valid;              // vocabulary columns below this are real, the rest padding
    int col_off;              // first vocabulary column of this launch's shard
    const float* acc;         // [T, ld_acc] fp32 dX accumulator (read by the last shard)
    long long ld_acc;
    int acc_mode;             // ACC_FIRST: store it (o1 map), ACC_MID: add to it, ACC_LAST: read it, store bf16
    uint32_t* status;         // nullable
    unsigned long long budget_ns;
    // Which list positions each pair runs. sched = 0: pair p runs p, p + P, p + 2P, ... (P pairs).
    // sched = 1: pair p runs sched_pos[sched_first[p] .. sched_first[p + 1]), increasing, as the
    // host's list-scheduling pass assigned them (a greedy simulation of the pairs taking the list in
    // order, so the positions each pair gets are increasing and every unit's inputs come earlier).
    int sched;
    uint16_t sched_first[CHAIN_MAX_PAIRS + 1];
    uint16_t sched_pos[CHAIN_MAX_SCHED];
};

struct ChainMaps {
    TmapSet m[CHAIN_MAX_PROBS];
};

template <int NE_, int CHAIN_>
struct ChainCfg {
    using Base = GemmCfg<CHAIN_BN, EPI_STORE, NE_>;
    static constexpr int NE = NE_;
    static constexpr int BN = CHAIN_BN;
    static constexpr int BNH = BN / 2;
    static constexpr int NUM_THREADS = Base::NUM_THREADS;
    static constexpr int A_BYTES = Base::A_BYTES;
    static constexpr int B_BYTES = Base::B_BYTES;
    static constexpr int STAGE_BYTES = Base::STAGE_BYTES;
    static constexpr uint32_t TMEM_COLS = Base::TMEM_COLS;
    // two staging boxes a warp: 32 x 32 bf16 (2 KB), or fp32 (4 KB) where dX is accumulated
    static constexpr int STG_PER_WARP = CHAIN_ == CHAIN_CE ? 2 * 4096 : STG_BYTES_PER_WARP;
    static constexpr int STG_BYTES = NE * STG_PER_WARP;
    // problem table, list segments, this pair's list positions, TMEM slot and flags words
    static constexpr int EXTRA = CHAIN_MAX_PROBS * 40 + CHAIN_MAX_SEGS * 12 + CHAIN_MAX_PER_PAIR * 2 + 16;
    // Six stages with either epilogue width (eight warps' bf16 staging boxes, or four warps' fp32
    // boxes, leave 8 bytes to spare).
    static constexpr int STAGES = 6;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr size_t SMEM_BYTES = 1024 + size_t(STAGES) * STAGE_BYTES + STG_BYTES + 8 * NUM_BARS + EXTRA;
    static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory per block");
    static_assert(STAGES >= 4, "pipeline depth");
    static_assert(NE == 4 || NE == 8, "4 or 8 epilogue warps");
    static_assert(CHAIN_ != CHAIN_CE || NE == 4, "the cross-entropy chain uses four epilogue warps");
};

// A problem's fields as the kernel uses them, copied once into shared memory at start-up (the
// parameter arrays are indexed at run time; reads through them are slow and would be repeated
// after every inline-asm memory clobber of the issue loops).
struct ChainProbS {
    int kb_begin, kb_end, a_mn, b_mn;
    int dep;
    int M, N, ncols, num_m_blocks, group;
};
static_assert(sizeof(ChainProbS) == 40, "problem table entry size assumed by ChainCfg::EXTRA");

// Position in a problem's order -> (row block, column tile): groups of `group` row blocks,
// row blocks fastest within a group (group 1 is plain row-major order).
__device__ __forceinline__ void chain_decode(const ChainProbS& p, int lu, int& m_blk, int& ncol) {
    const int per_group = p.group * p.ncols;
    const int gi = lu / per_group;
    const int r = lu - gi * per_group;
    const int left = p.num_m_blocks - gi * p.group;
    const int rows = left < p.group ? left : p.group;
    m_blk = gi * p.group + r % rows;
    ncol = r / rows;
}

// Calls f(std::integral_constant<int, I>) for problem I = prob, so that f's code for each problem
// reads that problem's parameters and tensor maps at fixed offsets: the compiler then keeps them
// in uniform registers, as the single-GEMM kernel has them, instead of reloading them through a
// run-time index on every issue (which measured 20-25 % slower per unit).
template <int CHAIN, typename F>
__device__ __forceinline__ void chain_dispatch(int prob, F&& f) {
    if (prob == 0) {
        f(std::integral_constant<int, 0>{});
    } else if (CHAIN == CHAIN_FWD || prob == 1) {
        f(std::integral_constant<int, 1>{});
    } else if (CHAIN == CHAIN_CE || prob == 2) {
        f(std::integral_constant<int, 2>{});
    } else {
        f(std::integral_constant<int, 3>{});
    }
}

// Walks list positions in increasing order for one warp role: the problem, row block and column
// tile of position g, from the shared-memory tables (a segment cursor that only moves forward).
struct ListCursor {
    int seg = 0, base = 0;
    __device__ __forceinline__ void unit(const ChainSeg* segs, const ChainProbS* probs, int g, int& prob, int& m_blk,
                                         int& ncol) {
        while (g >= base + segs[seg].count) base += segs[seg++].count;
        prob = segs[seg].prob;
        chain_decode(probs[prob], segs[seg].first + (g - base), m_blk, ncol);
    }
};

// Bounded wait until a completion counter reaches `target`: acquire loads (the counter's release
// adds by the producing warps form one release sequence, so the load that reads the final count
// synchronizes with every one of them), with a short sleep between reads so that waiting producers
// do not crowd the counter's cache line; then the async-proxy fence the TMA loads that follow need.
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t target, const Ctl& c) {
    if (ld_acquire_gpu(ctr) < target) {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(ctr) < target) {
            if (*c.abort_flag) return false;
            if (globaltimer_ns() - t0 > c.budget_ns) {
                if (c.status) atomicOr(c.status, DEV_TIMEOUT);
                *c.abort_flag = 1u;
                return false;
            }
            __nanosleep(256);
        }
    }
    fence_proxy_async_global();
    return true;
}

template <int NE, int CHAIN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(ChainCfg<NE, CHAIN>::NUM_THREADS, 1)
    gemm_chain_kernel(const __grid_constant__ ChainMaps maps, const __grid_constant__ ChainArgs args) {
    using Cfg = ChainCfg<NE, CHAIN>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int BN = Cfg::BN;
    constexpr int BNH = Cfg::BNH;
    constexpr uint32_t WARPS_PER_TILE = 2 * NE;  // epilogue warps of both CTAs, each publishes its share

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t* stg_base = smem + STAGES * Cfg::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stg_base + Cfg::STG_BYTES);
    uint64_t* full_bar = bars;
    uint64_t* empty_bar = bars + STAGES;
    uint64_t* tfull_bar = bars + 2 * STAGES;
    uint64_t* tempty_bar = bars + 2 * STAGES + 2;
    uint64_t* drain_bar = bars + 2 * STAGES + 4;
    ChainProbS* probs = reinterpret_cast<ChainProbS*>(bars + Cfg::NUM_BARS);  // problem table
    ChainSeg* segs = reinterpret_cast<ChainSeg*>(probs + CHAIN_MAX_PROBS);  // the list's segments
    uint16_t* my_pos = reinterpret_cast<uint16_t*>(segs + CHAIN_MAX_SEGS);   // this pair's list positions
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(my_pos + CHAIN_MAX_PER_PAIR);
    volatile uint32_t* abort_flag = tmem_slot + 1;
    volatile uint32_t* last_cta = tmem_slot + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = (rank == 0);
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

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
        *abort_flag = 0u;
        *last_cta = 0u;
        fence_mbarrier_init();
        fence_proxy_async_smem();
    }
    if (threadIdx.x >= 64 && threadIdx.x < 64 + CHAIN_MAX_PROBS) {  // lanes of the first epilogue warp
        const int i = threadIdx.x - 64;
        const ChainProb& p = args.p[i];
        ChainProbS q;
        q.kb_begin = p.pr.kb_begin;
        q.kb_end = p.pr.kb_end;
        q.a_mn = p.pr.a_mn;
        q.b_mn = p.pr.b_mn;
        q.dep = p.dep;
        q.M = p.pr.M;
        q.N = p.pr.N;
        q.ncols = p.ncols;
        q.num_m_blocks = p.pr.num_m_blocks;
        q.group = p.group;
        probs[i] = q;
    }
    if (threadIdx.x >= 96 && threadIdx.x < 96 + CHAIN_MAX_SEGS) {  // lanes of the second epilogue warp pair
        const int i = threadIdx.x - 96;
        if (i < args.nsegs) segs[i] = args.seg[i];
    }
    int my_count;  // list positions this pair runs
    if (args.sched) {
        const int b = args.sched_first[pair];
        my_count = args.sched_first[pair + 1] - b;
        for (int i = threadIdx.x; i < my_count; i += blockDim.x) my_pos[i] = args.sched_pos[b + i];
    } else {
        my_count = pair < args.total_units ? (args.total_units - 1 - pair) / num_pairs + 1 : 0;
    }
    if (warp == 0 && lane == 0) {
        for (int i = 0; i < CHAIN_MAX_PROBS; ++i) {
            if ((i >= 2 && CHAIN == CHAIN_FWD) || (i >= 3 && CHAIN == CHAIN_CE)) break;
            prefetch_tensormap(&maps.m[i].a);
            prefetch_tensormap(&maps.m[i].b);
            prefetch_tensormap(&maps.m[i].o0);
        }
        if (CHAIN == CHAIN_CE && args.acc_mode != ACC_LAST) prefetch_tensormap(&maps.m[1].o1);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const Ctl ctl{args.status, abort_flag, args.budget_ns};
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const int dep_ncols = probs[0].ncols, dep_mblocks = probs[0].num_m_blocks;
            ListCursor cur;
            for (int k = 0; k < my_count && ok; ++k) {
                const int g = args.sched ? my_pos[k] : pair + k * num_pairs;
                int prob, m_blk, ncol;
                cur.unit(segs, probs, g, prob, m_blk, ncol);
                chain_dispatch<CHAIN>(prob, [&](auto PI) {
                    constexpr int I = decltype(PI)::value;
                    const ChainProb& P = args.p[I];
                    const CUtensorMap* tmA = &maps.m[I].a;
                    const CUtensorMap* tmB = &maps.m[I].b;
                    const int kb_begin = P.pr.kb_begin, kb_end = P.pr.kb_end, a_mn = P.pr.a_mn, b_mn = P.pr.b_mn;
                    // K1, K3 (problem 0) and K5b (problem 3) read only inputs: no dependency code at all.
                    constexpr bool MAY_DEP = I == 1 || (CHAIN != CHAIN_FWD && I == 2);
                    const int dep = MAY_DEP ? P.dep : DEP_NONE;
                    const int arow = m_blk * 2 * BM + static_cast<int>(rank) * BM;
                    const int bcol = ncol * BN + static_cast<int>(rank) * BNH;
                    // A unit that reads problem 0's output waits, once, for the whole row block (K2, K4)
                    // or column tile (K5a) of it to be complete. The producer thread issues every load of
                    // the pair, so nothing else is added to its K-loop.
                    if (MAY_DEP && dep != DEP_NONE) {
                        const bool rows = dep == DEP_ROWS;
                        const uint32_t* ctr = rows ? args.row_done + m_blk
                                                   : args.col_done + (dep == DEP_COLS_M ? m_blk : ncol);
                        const uint32_t target = WARPS_PER_TILE * static_cast<uint32_t>(rows ? dep_ncols : dep_mblocks);
                        if (!wait_count(ctr, target, ctl)) {
                            ok = false;
                            return;
                        }
                    }
                    for (int kb = kb_begin; kb < kb_end; ++kb) {
                        if (!wait_bounded(&empty_bar[stage], phase ^ 1u, ctl)) {
                            ok = false;
                            break;
                        }
                        const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[stage]), 0);
                        mbar_arrive_expect_tx_cluster(full_leader, Cfg::STAGE_BYTES);
                        uint8_t* a_dst = sA + stage * Cfg::A_BYTES;
                        uint8_t* b_dst = sB + stage * Cfg::B_BYTES;
                        if (a_mn == 2) {
                            tma_load_3d_pair(a_dst, tmA, full_leader, 0, kb * BK, arow / 64);
                        } else if (a_mn) {
#pragma unroll
                            for (int j = 0; j < BM / 64; ++j)
                                tma_load_2d_pair(a_dst + j * 8192, tmA, full_leader, arow + j * 64, kb * BK);
                        } else {
                            tma_load_2d_pair(a_dst, tmA, full_leader, kb * BK, arow);
                        }
                        if (b_mn == 2) {
                            tma_load_3d_pair(b_dst, tmB, full_leader, 0, kb * BK, bcol / 64);
                        } else if (b_mn) {
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
                });
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // ---------------- MMA issuer (leader CTA, whole warp) ----------------
            auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool {
                const bool got = mbar_test_wait(bar, parity) || wait_bounded(bar, parity, ctl);
                return __all_sync(0xffffffffu, got) != 0;
            };
            int stage = 0;
            uint32_t phase = 0;
            uint32_t tcount = 0;
            bool ok = true;
            ListCursor cur;
            for (int k = 0; k < my_count && ok; ++k) {
                const int g = args.sched ? my_pos[k] : pair + k * num_pairs;
                int prob, m_blk, ncol;
                cur.unit(segs, probs, g, prob, m_blk, ncol);
                const uint32_t buf = tcount & 1u;
                const uint32_t tph = (tcount >> 1) & 1u;
                ++tcount;
                if (!wait_all(&tempty_bar[buf], tph ^ 1u)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * BN;
                // The K-loop of problem I. Its K range and operand majorness are read from the kernel
                // parameters at a fixed index, so the compiler keeps them and the descriptors built
                // from them in uniform registers, where tcgen05.mma takes its operands (values read
                // through the run-time problem index would be moved there on every issue).
                auto k_loop = [&](auto PI) {
                    constexpr int I = decltype(PI)::value;
                    const int kb_begin = args.p[I].pr.kb_begin, kb_end = args.p[I].pr.kb_end;
                    const bool a_mn = args.p[I].pr.a_mn != 0, b_mn = args.p[I].pr.b_mn != 0;
                    const uint32_t idesc = make_idesc_bf16(2 * BM, BN, a_mn, b_mn);
                    // Descriptor of a stage's first K slice; the k-th slice is that descriptor
                    // advanced in its address field (>> 4) by 2048 B (MN-major) or 32 B (K-major).
                    const uint64_t ad_base = make_sdesc_sw128(smem_u32(sA), a_mn ? 8192u : 16u, 1024);
                    const uint64_t bd_base = make_sdesc_sw128(smem_u32(sB), b_mn ? 8192u : 16u, 1024);
                    const uint64_t a_kstep = a_mn ? (2048u >> 4) : (32u >> 4);
                    const uint64_t b_kstep = b_mn ? (2048u >> 4) : (32u >> 4);
                    for (int kb = kb_begin; kb < kb_end; ++kb) {
                        if (!wait_all(&full_bar[stage], phase)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t ad0 = ad_base + static_cast<uint64_t>(stage) * (Cfg::A_BYTES >> 4);
                        const uint64_t bd0 = bd_base + static_cast<uint64_t>(stage) * (Cfg::B_BYTES >> 4);
                        umma_bf16_pair_elect(d_tmem, ad0, bd0, idesc, kb > kb_begin ? 1u : 0u);
#pragma unroll
                        for (int k = 1; k < BK / UMMA_K; ++k)
                            umma_bf16_pair_acc_elect(d_tmem, ad0 + k * a_kstep, bd0 + k * b_kstep, idesc);
                        umma_commit_pair_multicast_elect(&empty_bar[stage], 0x3);
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                };
                chain_dispatch<CHAIN>(prob, k_loop);
                if (!ok) break;
                umma_commit_pair_multicast_elect(&tfull_bar[buf], 0x3);
            }
            umma_commit_pair_elect(drain_bar);
            wait_drain(drain_bar, 0, args.status);
        }
    } else {
        // ---------------- epilogue (NE warps, both CTAs) ----------------
        constexpr int CHUNKS = BN / 32;
        constexpr int MY_CHUNKS = CHUNKS / (NE / 4);
        const int e = warp - 2;
        const int q = warp & 3;
        const int c_begin = (e >> 2) * MY_CHUNKS;
        const uint32_t lane_addr = static_cast<uint32_t>(q * 32) << 16;
        uint8_t* stg = stg_base + e * Cfg::STG_PER_WARP;
        int sbuf = 0;
        uint32_t tcount = 0;
        ListCursor cur;
        bool ok = true;
        for (int k = 0; k < my_count && ok; ++k) {
            const int g = args.sched ? my_pos[k] : pair + k * num_pairs;
            int prob, m_blk, ncol;
            cur.unit(segs, probs, g, prob, m_blk, ncol);
            const uint32_t buf = tcount & 1u;
            const uint32_t tph = (tcount >> 1) & 1u;
            ++tcount;
            bool have = true;
            if (lane == 0) have = wait_bounded(&tfull_bar[buf], tph, ctl);
            have = __shfl_sync(0xffffffffu, have ? 1 : 0, 0) != 0;
            if (!have) break;
            tc_fence_after();
            chain_dispatch<CHAIN>(prob, [&](auto PI) {
                constexpr int I = decltype(PI)::value;
                // problem 0 carries the activation epilogue and publishes its tiles
                constexpr bool ACT = (I == 0);
                const int M = args.p[I].pr.M, N = args.p[I].pr.N;
                const CUtensorMap* tmO0 = &maps.m[I].o0;
                const int row0 = m_blk * 2 * BM + static_cast<int>(rank) * BM + q * 32;
                const int row = row0 + lane;
                const bool row_ok = row < M;
                // Cross-entropy backward, problem 0: this row's log-sum-exp (log2 units), upstream
                // gradient and target; a NaN log-sum-exp (invalid target) gives the row no gradient.
                float lse2 = 0.0f, dl = 0.0f;
                int tgt = -1;
                if constexpr (CHAIN == CHAIN_CE && ACT) {
                    if (row_ok) {
                        tgt = args.target[row];
                        lse2 = args.lse[row] * 1.4426950408889634f;
                        dl = args.dloss[row];
                        if (!(lse2 == lse2)) {
                            lse2 = 0.0f;
                            dl = 0.0f;
                            tgt = -1;
                        }
                    }
                }
                // bf16 boxes: with fp32 boxes in the same staging (cross-entropy), box k of either
                // kind starts at 4 KB k, so a box never overlaps the other one in flight.
                auto store_bf16 = [&](const uint32_t (&pk)[16], int col0) {
                    stage_and_store(tmO0, CHAIN == CHAIN_CE ? stg + sbuf * 2048 : stg, sbuf, lane, pk, col0, row0);
                };
                auto issue = [&](int cc, uint32_t (&rr)[32], uint32_t (&uu)[16]) {
                    const int c = c_begin + cc;
                    if constexpr (CHAIN == CHAIN_BWD && ACT) {
                        const int col0 = ncol * BN + c * 32;
                        if (row_ok && col0 < N) {
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
                    const int col0 = ncol * BN + c * 32;
                    if (col0 >= N) return;
                    uint32_t pk[16];
                    if constexpr (CHAIN == CHAIN_FWD && ACT) {
                        if (args.has_out1) {
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                            stage_and_store(&maps.m[0].o1, stg, sbuf, lane, pk, col0, row0);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float2 gv = gelu2(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])));
                            pk[j] = pack_bf16x2(gv.x, gv.y);
                        }
                    } else if constexpr (CHAIN == CHAIN_BWD && ACT) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const float2 gp = gelu_prime2(make_float2(bf16_lo(uw[j]), bf16_hi(uw[j])));
                            const float2 gv =
                                mul2(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), gp);
                            pk[j] = pack_bf16x2(gv.x, gv.y);
                        }
                    } else if constexpr (CHAIN == CHAIN_CE && ACT) {
                        // dZ = dloss (exp(z - lse) - [column == target]), 0 on padding columns.
                        constexpr float LOG2E = 1.4426950408889634f;
                        const int gcol0 = args.col_off + col0;
                        const int lim = args.v_valid - gcol0;
                        const unsigned dt = static_cast<unsigned>(tgt - gcol0);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float gz[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const int jj = 2 * j + e2;
                                float pr = ex2_approx(fmaf(__uint_as_float(r[jj]), LOG2E, -lse2));
                                if (static_cast<int>(dt) == jj && dt < 32u) pr -= 1.0f;
                                gz[e2] = (jj < lim && dl != 0.0f) ? dl * pr : 0.0f;
                            }
                            pk[j] = pack_bf16x2(gz[0], gz[1]);
                        }
                    } else if constexpr (CHAIN == CHAIN_CE && I == 1) {
                        // dX across the shards' launches: the first stores its fp32 tile, the middle
                        // ones add theirs at L2 (TMA reductions), the last adds the accumulator in
                        // registers and stores bf16; one addition per shard, in shard order.
                        if (args.acc_mode != ACC_LAST) {
                            stage_and_store_f32(&maps.m[1].o1, stg, sbuf, lane, r, col0, row0, args.acc_mode == ACC_MID);
                            return;
                        }
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        if (row_ok) {
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
#pragma unroll
                        for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                    }
                    store_bf16(pk, col0);
                };
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
                if constexpr (ACT) {
                    // Publish this warp's share of the tile once its stores have landed in global memory.
                    if (lane == 0) {
                        bulk_wait_group<0>();
                        fence_proxy_async_global();
                        red_release_gpu_add(args.row_done + m_blk, 1u);
                        red_release_gpu_add(args.col_done + ncol, 1u);
                    }
                    __syncwarp();
                }
            });
        }
        if (lane == 0) bulk_wait_group<0>();
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (threadIdx.x == 0) spin_ns(ABORT_SETTLE_NS);
        __syncthreads();
    }
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
    // The last CTA to finish returns the workspace to zeros for the next launch. Every other CTA
    // has stopped claiming, polling and publishing before it counts itself finished.
    if (threadIdx.x == 0) {
        __threadfence();
        const uint32_t done = atomicAdd(args.ctl + 1, 1u);
        if (done == gridDim.x - 1) {
            __threadfence();
            *last_cta = 1u;
        }
    }
    __syncthreads();
    if (*last_cta) {
        for (int i = threadIdx.x; i < args.num_counters; i += blockDim.x) args.row_done[i] = 0u;
        __syncthreads();
        if (threadIdx.x == 0) {
            args.ctl[0] = 0u;
            args.ctl[1] = 0u;
        }
    }
}

// Host side of the list scheduling (mptp_mlp_fused.cu), for the other users of the chain kernel.
// A problem of M x N outputs over K blocks [kb_begin, kb_end) (operand majorness as ProbInfo),
// units in groups of `group` row blocks.
ChainProb chain_problem(int M, int N, int kb_begin, int kb_end, int a_mn, int b_mn, int group);
// Bytes of zeroed counters a chain over a first problem of M0 x N0 outputs needs (control words,
// one per 256-row block and per 256-column tile), rounded up to 256.
size_t chain_counter_bytes(int M0, int N0);
// One cross-entropy backward shard in one launch: problems 0 (K10), 1 (K12, DEP_ROWS) and 2 (K11,
// DEP_COLS_M) set up in `a`; `counters` holds chain_counter_bytes of zeros, and is zero again
// when the launch ends. CHAIN_NO_SCHEDULE (nothing launched) when the list does not fit the
// schedule tables.
mp_status launch_chain_ce(const ChainMaps& m, ChainArgs& a, int sms, cudaStream_t s, uint32_t* counters);
// Returned by the host side when a list has no precomputed schedule (more positions than
// CHAIN_MAX_SCHED, or a pair's share beyond CHAIN_MAX_PER_PAIR); the callers then run the same
// GEMMs as separate launches. (The kernel's round-robin order, which needs no tables, leaves pairs
// waiting on dependencies that a schedule places after other work: measured 20-40 % slower than the
// separate launches at T = 16384 and 32768.)
constexpr mp_status CHAIN_NO_SCHEDULE = static_cast<mp_status>(-1);

template <int NE, int CHAIN>
inline int chain_resident_pairs(int num_sms) {
    using Cfg = ChainCfg<NE, CHAIN>;
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    auto kern = gemm_chain_kernel<NE, CHAIN>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::SMEM_BYTES)) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    cfg.blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        clusters = num_sms / 2;
    }
    if (clusters > num_sms / 2) clusters = num_sms / 2;
    if (clusters > CHAIN_MAX_PAIRS) clusters = CHAIN_MAX_PAIRS;
    if (dev >= 0 && dev < 64) cached[dev] = clusters;
    return clusters;
}

// Grid = 2 x `pairs` (the pairs the schedule in args was made for; at most the resident pairs).
template <int NE, int CHAIN>
inline cudaError_t launch_gemm_chain(const ChainMaps& maps, const ChainArgs& args, int pairs, cudaStream_t stream) {
    using Cfg = ChainCfg<NE, CHAIN>;
    auto kern = gemm_chain_kernel<NE, CHAIN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg::SMEM_BYTES));
    if (e != cudaSuccess) return e;
    if (pairs <= 0) return cudaSuccess;
    e = launch_pdl(kern, dim3(2 * pairs), dim3(Cfg::NUM_THREADS), Cfg::SMEM_BYTES, stream, maps, args);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace mptp
