// Entry points of the sharded MLP block with each direction in one launch:
// mp_mlp_fwd_fused (K1 and K2) and mp_mlp_bwd_fused (K3, K4, K5a, K5b), run by
// the chain kernel of mptp_gemm_chain.cuh.
//
// They compute what mp_mlp_fwd_shards / mp_mlp_bwd_shards compute ("Megatron-LM:
// Training Multi-Billion Parameter Language Models Using Model Parallelism",
// section 3.4; "Tensor and pipeline parallelism, and choosing a layout",
// Proposition (Megatron MLP split)), tile for tile with the same K-loops, so every
// output equals theirs bit for bit. What changes is the schedule: the second GEMM
// of the forward starts on a row block as soon as the first has completed that
// row block, and in the backward the f sum (K4) and the weight gradients (K5a,
// K5b) run beside K3 and each other on whichever CTA pairs are free. That overlap is the method's own ("Tensor and pipeline parallelism, and
// choosing a layout", the remarks after the Proposition: the backward all-reduce
// of dX overlaps the weight-gradient GEMMs), done inside one grid.
#include <algorithm>
#include <cstdlib>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <vector>

#include "mptp_gemm_chain.cuh"
#include "mptp_internal.h"

namespace mptp {
namespace {

mp_status check_shape(int T, int h, int f, int t, int s0, int n) {
    if (T < 0 || h <= 0 || f <= 0 || t < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || f % t != 0 || (f / t) % 64 != 0) return MP_ERR_UNSUPPORTED_SHAPE;
    if (s0 < 0 || n < 1 || s0 > t - n) return MP_ERR_INVALID_ARG;
    return MP_OK;
}

// Control words, then one completion counter per 256-row block and per 256-column tile of Y (dU).
size_t workspace_need(int T, int f) {
    const size_t words = CHAIN_CTL_WORDS + static_cast<size_t>(ceil_div(T, 2 * BM)) + ceil_div(f, CHAIN_BN);
    return (words * 4 + 255) / 256 * 256;
}

ChainProb chain_prob(int M, int N, int kb_begin, int kb_end, int a_mn, int b_mn, int group) {
    ChainProb c{};
    c.pr.M = M;
    c.pr.N = N;
    c.pr.num_m_blocks = ceil_div(M, 2 * BM);
    c.ncols = ceil_div(N, CHAIN_BN);
    c.pr.num_units = c.pr.num_m_blocks * c.ncols;
    c.pr.kb_begin = kb_begin;
    c.pr.kb_end = kb_end;
    c.pr.a_mn = a_mn;
    c.pr.b_mn = b_mn;
    c.group = group < 1 ? 1 : (group > c.pr.num_m_blocks ? c.pr.num_m_blocks : group);
    c.dep = DEP_NONE;
    return c;
}

// Units of row group gi of a problem (rows [gi * group, ...)), as a run of its own order.
ChainSeg row_group(const ChainProb& c, int prob, int gi) {
    const int first_row = gi * c.group;
    const int rows = (c.pr.num_m_blocks - first_row) < c.group ? (c.pr.num_m_blocks - first_row) : c.group;
    return ChainSeg{prob, first_row * c.ncols, rows * c.ncols};
}

// The list: problem 0's row groups, each followed (after `lag` more groups) by the same rows of
// problem 1, then problems 2.. whole. Problem 1 reads problem 0 by rows, so every unit comes
// after the units it reads.
bool build_list(ChainArgs& a, int nprobs, int lag) {
    const int ng = ceil_div(a.p[0].pr.num_m_blocks, a.p[0].group);
    int n = 0;
    for (int g = 0; g < ng + lag; ++g) {
        if (g < ng) a.seg[n++] = row_group(a.p[0], 0, g);
        if (g >= lag) a.seg[n++] = row_group(a.p[1], 1, g - lag);
        if (n > CHAIN_MAX_SEGS - 4) return false;
    }
    for (int i = 2; i < nprobs; ++i) a.seg[n++] = ChainSeg{i, 0, a.p[i].pr.num_units};
    a.nsegs = n;
    a.total_units = 0;
    for (int i = 0; i < n; ++i) a.total_units += a.seg[i].count;
    return true;
}

// Fewest row blocks per group that keep the list within the segment table.
int min_row_group(int m_blocks) { return ceil_div(m_blocks, (CHAIN_MAX_SEGS - 4) / 2); }

// Epilogue warps of the chain kernel: eight where the GeLU / GeLU' tiles have short K-loops (their
// epilogue also waits for its stores to land before publishing), four elsewhere. Measured at
// h <= 2048: equal or up to 2 % faster with eight (8192 x 1536); at h = 3072 four are 1 % faster.
bool chain_ne8(int h) { return h <= 2048; }

// Where one launch measured no slower than the separate launches (CUDA events, same box): every
// width at T <= 8192 (1-10 % faster over the layer sweep), and h >= 2304 at T = 16384 (forward 1-4 %,
// backward 6 % faster). At T = 16384 with h <= 1920 and T = 32768 with h = 1536 the one-launch
// forward was 2-7 % slower and the backward about 1 %; those layers run the separate launches.
bool chain_pays(int T, int h) { return T <= 8192 || h >= 2304; }

// Host copy of the kernel's position decode (chain_decode).
void decode_host(const ChainProb& p, int lu, int& m_blk, int& ncol) {
    const int per_group = p.group * p.ncols;
    const int gi = lu / per_group;
    const int r = lu - gi * per_group;
    const int left = p.pr.num_m_blocks - gi * p.group;
    const int rows = left < p.group ? left : p.group;
    m_blk = gi * p.group + r % rows;
    ncol = r / rows;
}

// Cost model of the list-scheduling pass, in K-block times (one 64-deep stage of a 256 x 256 tile).
constexpr double SCHED_UNIT = 0.5;  // per-unit overhead (pipeline turn-over)
constexpr double SCHED_EPI = 3.0;   // a problem-0 tile's epilogue and store, after its last MMA
constexpr double SCHED_LAT = 1.0;   // a published tile reaching the waiting producer

struct Schedule {
    std::vector<uint16_t> first, pos;
    double makespan = 0.0;
};

// Greedy list scheduling of the list over `pairs` CTA pairs: each position, in order, goes to the
// pair that is free first (the lowest index among equals); a unit that reads problem 0's output
// starts once the row block or column tile it reads is complete. Each pair's positions come out
// increasing. Returns false when the schedule would not fit the kernel's tables (the callers then
// run the separate launches).
bool list_schedule(const ChainArgs& a, int pairs, Schedule& out) {
    out.makespan = 0.0;
    if (a.total_units > CHAIN_MAX_SCHED || pairs > CHAIN_MAX_PAIRS || pairs < 1) return false;
    const ChainProb& p0 = a.p[0];
    // completion times of problem 0's row blocks and column tiles (the last of their tiles)
    std::vector<double> row_done(static_cast<size_t>(p0.pr.num_m_blocks), 0.0), col_done(static_cast<size_t>(p0.ncols), 0.0);
    using Slot = std::pair<double, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> freeq;
    for (int q = 0; q < pairs; ++q) freeq.push({0.0, q});
    std::vector<std::vector<uint16_t>> mine(pairs);
    int g = 0;
    for (int si = 0; si < a.nsegs; ++si) {
        const ChainSeg& sg = a.seg[si];
        const ChainProb& p = a.p[sg.prob];
        const int L = p.pr.kb_end - p.pr.kb_begin;
        for (int i = 0; i < sg.count; ++i, ++g) {
            int m_blk, ncol;
            decode_host(p, sg.first + i, m_blk, ncol);
            const Slot f = freeq.top();
            freeq.pop();
            double cur = f.first + SCHED_UNIT;
            if (p.dep == DEP_ROWS) cur = std::max(cur, row_done[static_cast<size_t>(m_blk)] + SCHED_LAT);
            if (p.dep == DEP_COLS) cur = std::max(cur, col_done[static_cast<size_t>(ncol)] + SCHED_LAT);
            if (p.dep == DEP_COLS_M) cur = std::max(cur, col_done[static_cast<size_t>(m_blk)] + SCHED_LAT);
            cur += L;
            if (sg.prob == 0) {
                row_done[static_cast<size_t>(m_blk)] = std::max(row_done[static_cast<size_t>(m_blk)], cur + SCHED_EPI);
                col_done[static_cast<size_t>(ncol)] = std::max(col_done[static_cast<size_t>(ncol)], cur + SCHED_EPI);
            }
            mine[f.second].push_back(static_cast<uint16_t>(g));
            freeq.push({cur, f.second});
            out.makespan = std::max(out.makespan, cur + (sg.prob == 0 ? SCHED_EPI : 0.0));
        }
    }
    out.first.assign(static_cast<size_t>(pairs) + 1, 0);
    out.pos.clear();
    for (int q = 0; q < pairs; ++q) {
        if (mine[q].size() > static_cast<size_t>(CHAIN_MAX_PER_PAIR)) return false;
        out.first[q] = static_cast<uint16_t>(out.pos.size());
        out.pos.insert(out.pos.end(), mine[q].begin(), mine[q].end());
    }
    out.first[pairs] = static_cast<uint16_t>(out.pos.size());
    return true;
}

// The list and schedule of a launch. The rows of problems 0 and 1 go in groups of G row blocks
// (problem 1's group g after problem 0's group g + lag); every (G, lag) with G a power of two up to
// the row blocks and lag up to 3 is scheduled by the list-scheduling pass and the shortest
// simulated makespan is kept (the first of equals). Cached by the problems' geometry and the pair
// count. If no schedule fits the kernel's tables, groups of min_row_group rows, lag 0 and no
// schedule (launch_chain_ne then answers CHAIN_NO_SCHEDULE).
struct Plan {
    int group = 1, lag = 0;
    Schedule sched;  // empty: none fits the tables
};

bool plan_chain(ChainArgs& a, int nprobs, int pairs) {
    std::vector<int> key{nprobs, pairs};
    for (int i = 0; i < nprobs; ++i) {
        const ChainProb& p = a.p[i];
        key.insert(key.end(), {p.pr.num_m_blocks, p.ncols, p.pr.kb_begin, p.pr.kb_end, p.dep, p.group});
    }
    static std::mutex mu;
    static std::map<std::vector<int>, Plan> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it == cache.end()) {
        const int mb = a.p[0].pr.num_m_blocks;
        Plan best;
        best.group = std::max(1, min_row_group(mb));
        bool have = false;
        for (int G = 1; G <= 2 * mb; G *= 2) {
            const int g = std::min(G, mb);
            if (g < min_row_group(mb)) continue;
            for (int lag = 0; lag <= 3; ++lag) {
                if (lag > 0 && lag >= ceil_div(mb, g)) break;
                ChainArgs& t = a;  // scratch use of the caller's args; the chosen plan is applied below
                t.p[0].group = g;
                t.p[1].group = g;
                if (!build_list(t, nprobs, lag)) continue;
                Schedule sc;
                if (!list_schedule(t, pairs, sc)) continue;
                if (!have || sc.makespan < best.sched.makespan) {
                    best.group = g;
                    best.lag = lag;
                    best.sched = std::move(sc);
                    have = true;
                }
            }
            if (G >= mb) break;
        }
        if (cache.size() >= 256) cache.clear();
        it = cache.emplace(key, std::move(best)).first;
    }
    const Plan& pl = it->second;
    a.p[0].group = pl.group;
    a.p[1].group = pl.group;
    if (!build_list(a, nprobs, pl.lag)) return false;
    a.sched = pl.sched.first.empty() ? 0 : 1;
    if (a.sched) {
        std::copy(pl.sched.first.begin(), pl.sched.first.end(), a.sched_first);
        std::copy(pl.sched.pos.begin(), pl.sched.pos.end(), a.sched_pos);
    }
    return true;
}

// CTA pairs of a chain launch: every pair the device holds at once, at most one per unit.
template <int NE, int CHAIN>
int chain_pairs(int sms, int nprobs, const ChainArgs& a) {
    int units = 0;
    for (int i = 0; i < nprobs; ++i) units += a.p[i].pr.num_units;
    const int r = chain_resident_pairs<NE, CHAIN>(sms);
    return r < units ? r : units;
}

template <int NE, int CHAIN>
mp_status launch_chain_ne(const ChainMaps& m, ChainArgs& a, int nprobs, int sms, cudaStream_t s) {
    const int pairs = chain_pairs<NE, CHAIN>(sms, nprobs, a);
    if (!plan_chain(a, nprobs, pairs)) return MP_ERR_UNSUPPORTED_SHAPE;
    if (!a.sched) return CHAIN_NO_SCHEDULE;
    return launch_gemm_chain<NE, CHAIN>(m, a, pairs, s) == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

template <int CHAIN>
mp_status launch_chain(const ChainMaps& m, ChainArgs& a, int nprobs, int sms, cudaStream_t s, int h) {
    return chain_ne8(h) ? launch_chain_ne<8, CHAIN>(m, a, nprobs, sms, s) : launch_chain_ne<4, CHAIN>(m, a, nprobs, sms, s);
}

mp_status check_workspace(void* ws, size_t bytes, int T, int f) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return MP_ERR_WORKSPACE;
    if (bytes < workspace_need(T, f)) return MP_ERR_WORKSPACE;
    return MP_OK;
}

}  // namespace

ChainProb chain_problem(int M, int N, int kb_begin, int kb_end, int a_mn, int b_mn, int group) {
    return chain_prob(M, N, kb_begin, kb_end, a_mn, b_mn, group);
}

size_t chain_counter_bytes(int M0, int N0) {
    const size_t words = CHAIN_CTL_WORDS + static_cast<size_t>(ceil_div(M0, 2 * BM)) + ceil_div(N0, CHAIN_BN);
    return (words * 4 + 255) / 256 * 256;
}

mp_status launch_chain_ce(const ChainMaps& m, ChainArgs& a, int sms, cudaStream_t s, uint32_t* counters) {
    a.ctl = counters;
    a.row_done = counters + CHAIN_CTL_WORDS;
    a.col_done = a.row_done + a.p[0].pr.num_m_blocks;
    a.num_counters = a.p[0].pr.num_m_blocks + a.p[0].ncols;
    return launch_chain_ne<4, CHAIN_CE>(m, a, 3, sms, s);
}

}  // namespace mptp

using namespace mptp;

extern "C" size_t mp_mlp_fused_workspace_bytes(int T, int h, int f, int t) {
    if (check_shape(T, h, f, t, 0, t) != MP_OK) return 0;
    return workspace_need(T, f);
}

extern "C" mp_status mp_mlp_fwd_fused(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, mp_bf16* Z, mp_bf16* Y,
                                      mp_bf16* U_save, int T, int h, int f, int t, int shard_begin, int shard_count,
                                      void* workspace, size_t workspace_bytes, uint32_t* d_status, void* stream) {
    mp_status st = check_shape(T, h, f, t, shard_begin, shard_count);
    if (st != MP_OK) return st;
    if (T == 0) return MP_OK;
    if (!X || !A || !B || !Z || !Y) return MP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Z) || !aligned16(Y) ||
        (U_save && !aligned16(U_save)) || (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return MP_ERR_MISALIGNED;
    if ((st = check_workspace(workspace, workspace_bytes, T, f)) != MP_OK) return st;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    if (!chain_pays(T, h))
        return mp_mlp_fwd_shards(X, A, B, Z, Y, U_save, T, h, f, t, shard_begin, shard_count, d_status, stream);
    const int fs = f / t;
    const int c0 = shard_begin * fs, nc = shard_count * fs;

    ChainMaps m{};
    ChainArgs a{};
    // K1: U = X A_r (A MN-major), Y = GeLU(U), over the range's columns.
    int b1 = 0;
    if (!make_tmap_bf16(&m.m[0].a, X, h, T, h, 64, BM) || !(b1 = make_tmap_mn_operand(&m.m[0].b, A + c0, nc, h, f)) ||
        !make_tmap_bf16_out(&m.m[0].o0, Y + c0, nc, T, f) ||
        !make_tmap_bf16_out(&m.m[0].o1, U_save ? U_save + c0 : Y + c0, nc, T, f))
        return MP_ERR_CUDA;
    // K2: Z = sum_i Y_i B_i over the range's K blocks, ascending (the g sum).
    int b2 = 0;
    if (!make_tmap_bf16(&m.m[1].a, Y, f, T, f, 64, BM) || !(b2 = make_tmap_mn_operand(&m.m[1].b, B, h, f, h)) ||
        !make_tmap_bf16_out(&m.m[1].o0, Z, h, T, h))
        return MP_ERR_CUDA;
    // K1 and K2 take their row grouping from the plan (launch_chain).
    a.p[0] = chain_prob(T, nc, 0, h / BK, 0, b1, 1);
    a.p[1] = chain_prob(T, h, c0 / BK, (c0 + nc) / BK, 0, b2, 1);
    a.p[1].dep = DEP_ROWS;
    uint32_t* ws = static_cast<uint32_t*>(workspace);
    a.ctl = ws;
    a.row_done = ws + CHAIN_CTL_WORDS;
    a.col_done = a.row_done + a.p[0].pr.num_m_blocks;
    a.num_counters = a.p[0].pr.num_m_blocks + a.p[0].ncols;
    a.has_out1 = U_save ? 1 : 0;
    a.status = d_status;
    a.budget_ns = wait_budget_ns();
    st = launch_chain<CHAIN_FWD>(m, a, 2, sms, static_cast<cudaStream_t>(stream), h);
    if (st == CHAIN_NO_SCHEDULE)  // too many tiles for the schedule tables: the separate launches
        return mp_mlp_fwd_shards(X, A, B, Z, Y, U_save, T, h, f, t, shard_begin, shard_count, d_status, stream);
    return st;
}

extern "C" mp_status mp_mlp_bwd_fused(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, const mp_bf16* U,
                                      const mp_bf16* Y, const mp_bf16* dZ, mp_bf16* dX, mp_bf16* dA, mp_bf16* dB,
                                      mp_bf16* dU_ws, int T, int h, int f, int t, int shard_begin, int shard_count,
                                      void* workspace, size_t workspace_bytes, uint32_t* d_status, void* stream) {
    mp_status st = check_shape(T, h, f, t, shard_begin, shard_count);
    if (st != MP_OK) return st;
    if (!A || !B || !dA || !dB) return MP_ERR_INVALID_ARG;
    if (T > 0 && (!X || !U || !Y || !dZ || !dX || !dU_ws)) return MP_ERR_INVALID_ARG;
    const void* ptrs[] = {X, A, B, U, Y, dZ, dX, dA, dB, dU_ws};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MP_ERR_MISALIGNED;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MP_ERR_MISALIGNED;
    if (T > 0 && (st = check_workspace(workspace, workspace_bytes, T, f)) != MP_OK) return st;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int fs = f / t;
    const int c0 = shard_begin * fs, nc = shard_count * fs;
    if (T == 0) {
        // Empty batch: the range's weight gradients are sums over zero tokens.
        if (cudaMemset2DAsync(dA + c0, size_t(f) * 2, 0, size_t(nc) * 2, size_t(h), s) != cudaSuccess ||
            cudaMemsetAsync(dB + size_t(c0) * h, 0, size_t(nc) * h * 2, s) != cudaSuccess)
            return MP_ERR_CUDA;
        return MP_OK;
    }

    if (!chain_pays(T, h))
        return mp_mlp_bwd_shards(X, A, B, U, Y, dZ, dX, dA, dB, dU_ws, T, h, f, t, shard_begin, shard_count, d_status,
                                 stream);
    ChainMaps m{};
    ChainArgs a{};
    // K3: dU_r = (dZ B_r^T) * GeLU'(U_r); both operands K-major.
    if (!make_tmap_bf16(&m.m[0].a, dZ, h, T, h, 64, BM) ||
        !make_tmap_bf16(&m.m[0].b, B + size_t(c0) * h, h, nc, h, 64, CHAIN_BN / 2) ||
        !make_tmap_bf16_out(&m.m[0].o0, dU_ws + c0, nc, T, f))
        return MP_ERR_CUDA;
    // K4: dX = sum_i dU_i A_i^T over the range's K blocks, ascending (the f sum).
    if (!make_tmap_bf16(&m.m[1].a, dU_ws, f, T, f, 64, BM) ||
        !make_tmap_bf16(&m.m[1].b, A, f, h, f, 64, CHAIN_BN / 2) || !make_tmap_bf16_out(&m.m[1].o0, dX, h, T, h))
        return MP_ERR_CUDA;
    // K5a: dA_r = X^T dU_r (M = h, N = nc, K = T), both operands MN-major.
    int a5 = 0, b5 = 0;
    if (!(a5 = make_tmap_mn_operand(&m.m[2].a, X, h, T, h)) || !(b5 = make_tmap_mn_operand(&m.m[2].b, dU_ws + c0, nc, T, f)) ||
        !make_tmap_bf16_out(&m.m[2].o0, dA + c0, nc, h, f))
        return MP_ERR_CUDA;
    // K5b: dB_r = Y_r^T dZ (M = nc, N = h, K = T), both operands MN-major.
    int a6 = 0, b6 = 0;
    if (!(a6 = make_tmap_mn_operand(&m.m[3].a, Y + c0, nc, T, f)) || !(b6 = make_tmap_mn_operand(&m.m[3].b, dZ, h, T, h)) ||
        !make_tmap_bf16_out(&m.m[3].o0, dB + size_t(c0) * h, h, nc, h))
        return MP_ERR_CUDA;
    // K3 and K4 take their row grouping from the plan (launch_chain).
    a.p[0] = chain_prob(T, nc, 0, h / BK, 0, 0, 1);
    a.p[1] = chain_prob(T, h, c0 / BK, (c0 + nc) / BK, 0, 0, 1);
    a.p[1].dep = DEP_ROWS;
    // dA: row blocks fastest (X^T's panels are the smaller operand); dB: row-major.
    a.p[2] = chain_prob(h, nc, 0, ceil_div(T, BK), a5, b5, ceil_div(h, 2 * BM));
    a.p[2].dep = DEP_COLS;
    a.p[3] = chain_prob(nc, h, 0, ceil_div(T, BK), a6, b6, 1);
    uint32_t* ws = static_cast<uint32_t*>(workspace);
    a.ctl = ws;
    a.row_done = ws + CHAIN_CTL_WORDS;
    a.col_done = a.row_done + a.p[0].pr.num_m_blocks;
    a.num_counters = a.p[0].pr.num_m_blocks + a.p[0].ncols;
    a.aux = reinterpret_cast<const __nv_bfloat16*>(U + c0);
    a.ld_aux = f;
    a.status = d_status;
    a.budget_ns = wait_budget_ns();
    st = launch_chain<CHAIN_BWD>(m, a, 4, sms, s, h);
    if (st == CHAIN_NO_SCHEDULE)  // too many tiles for the schedule tables: the separate launches
        return mp_mlp_bwd_shards(X, A, B, U, Y, dZ, dX, dA, dB, dU_ws, T, h, f, t, shard_begin, shard_count, d_status,
                                 stream);
    return st;
}
