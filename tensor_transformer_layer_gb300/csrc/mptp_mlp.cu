// Entry points of the sharded MLP block: mp_mlp_fwd and mp_mlp_bwd.
//
// Forward ("Megatron-LM: Training Multi-Billion Parameter Language Models Using
// Model Parallelism", section 3.4, column-parallel then row-parallel GEMM;
// "Tensor and pipeline parallelism, and choosing a layout", Proposition (Megatron
// MLP split), steps 1-3):
//   K1  U = X A, Y = GeLU(U)       all t column shards of A in one launch
//   K2  Z = sum_i Y_i B_i          K-loop over shards 0..t-1, TMEM accumulation
// Backward (Proposition steps 4-5):
//   K3  dU = (G B^T) * GeLU'(U)
//   K4  dX = sum_i dU_i A_i^T      K-loop over shards 0..t-1 (the f sum)
//   K5  dA = X^T dU, dB = Y^T G    both operands MN-major, K = T
// K4 and K5 are independent once dU exists. Megatron overlaps the backward all-reduce
// of dX with the weight-gradient GEMMs ("Tensor and pipeline parallelism, and choosing
// a layout", the discussion after the Proposition on the communication ratio); here
// the f sum of dX is inside K4's K-loop, and the overlap becomes K4, K5a and K5b side
// by side on disjoint sets of CTA pairs (the caller's stream plus two side streams),
// so that none of them ends in a part-empty last wave of tiles.
//
// Shard ranges. mp_mlp_fwd_shards / mp_mlp_bwd_shards run the work of shards
// [s0, s0 + n) only: K1, K3 and K5 over the range's f/t-wide column (or row) blocks,
// K2 and K4 over the range's K blocks, so Z (dX) is the partial output those shards
// contribute before the g (f) all-reduce. mp_mlp_fwd and mp_mlp_bwd are the full
// range [0, t). Every output element runs the same K-loop whichever range it is
// computed in, so a range's Y, U, dU, dA and dB blocks equal the full call's bitwise.
#include <cstdlib>
#include <cstring>

#include "mptp_gemm.cuh"
#include "mptp_gemm_split.cuh"
#include "mptp_internal.h"

namespace mptp {

static mp_status check_mlp_shape(int T, int h, int f, int t) {
    if (T < 0 || h <= 0 || f <= 0 || t < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || f % t != 0 || (f / t) % 64 != 0) return MP_ERR_UNSUPPORTED_SHAPE;
    return MP_OK;
}

static mp_status check_shard_range(int t, int s0, int n) {
    if (s0 < 0 || n < 1 || s0 > t - n) return MP_ERR_INVALID_ARG;
    return MP_OK;
}

// One GEMM of a launch: C[M, N] over K blocks [kb_begin, kb_end). a_bytes / b_bytes
// are the sizes of the A (M side) and B (N side) operands, for the unit order.
static ProbInfo problem(int M, int N, int bn, int kb_begin, int kb_end, bool a_mn, bool b_mn, double a_bytes,
                        double b_bytes) {
    ProbInfo p{};
    p.M = M;
    p.N = N;
    p.num_m_blocks = ceil_div(M, 2 * BM);  // 256-row blocks: one per CTA-pair tile
    p.num_units = p.num_m_blocks * ceil_div(N, bn);
    p.n_fastest = n_fastest_order(a_bytes, b_bytes);
    p.kb_begin = kb_begin;
    p.kb_end = kb_end;
    p.a_mn = a_mn ? 1 : 0;
    p.b_mn = b_mn ? 1 : 0;
    return p;
}

// Backward schedule of K4, K5a, K5b: MPTP_BWD_SCHEDULE = "serial" | "overlap"; unset or
// anything else picks the side-by-side schedule when its estimated makespan is at least
// 6 % below the serial one. Measured on GB300 over h in {768..3072}, T in {512..8192}:
// it wins 1-50 % where the estimate says >= 7 %, and loses up to 5 % at h = 3072 with
// T >= 4096 (estimate <= 5.5 %), where three GEMMs' operand panels crowd L2.
enum class BwdSchedule { Auto, Serial, Overlap };
static BwdSchedule bwd_schedule() {
    const char* v = std::getenv("MPTP_BWD_SCHEDULE");
    if (v != nullptr && std::strcmp(v, "serial") == 0) return BwdSchedule::Serial;
    if (v != nullptr && std::strcmp(v, "overlap") == 0) return BwdSchedule::Overlap;
    return BwdSchedule::Auto;
}

// Cost of one output tile in K-block times: its K blocks plus about two for the epilogue.
constexpr int EPI_KB = 2;

// Epilogue warps of K1 and K3 (GeLU, GeLU'). A launch's last tile is epilogued after its last
// MMA with nothing to hide behind: with few K blocks per CTA pair (the layer at T = 2048,
// h = 1536: 72 a pair) eight warps halve that tail (K3's 10.6 -> 6.3 us, K1's 5.4 -> 4.0 us;
// the step -1 %), while on long launches four measured 0.2-0.8 % faster (fewer warps beside the
// MMA issuer). The store-only GEMMs keep four: eight were 1 % slower there.
constexpr int SHORT_LAUNCH_KB = 256;  // K blocks a pair runs, at most, for eight epilogue warps

template <int EPI>
static cudaError_t launch_gelu_epi(const TmapSet& m, const GemmArgs& a, int sms, cudaStream_t s) {
    const int pairs = resident_pairs<256, EPI, 4>(sms);
    const bool short_launch = ceil_div(a.pr.num_units, pairs) * (a.pr.kb_end - a.pr.kb_begin) <= SHORT_LAUNCH_KB;
    return short_launch ? launch_gemm_tc<256, EPI, 8>(m, a, sms, s) : launch_gemm_tc<256, EPI, 4>(m, a, sms, s);
}

// Tile width of K4 (dX = dU A^T, N = h, B operand K-major). 224-wide tiles cut h = 3072
// into 14 column units instead of 12, so T = 4096 gives 224 units: 2.95 rounds of 76 CTA
// pairs, against 2.53 rounds of 256-wide tiles whose last round leaves half the pairs idle.
constexpr int K4_BN = 224;

// Split-K for the row-parallel GEMMs (K2, K4) when their output tiles do not fill the chip:
// the two CTA pairs of a cluster share a 256-wide tile, each over half of the shard-ordered K
// range, and the partials are summed on chip (mptp_gemm_split.cuh). Costs in K-block times:
// one pair per tile, `bn` wide, takes rounds x L x bn / 256; two pairs take
// rounds x ceil(L / 2) plus about SPLIT_HOP_KB for the on-chip sum. The split is taken when it
// is at least 10 % cheaper and each pair keeps at least 16 K blocks (T = 2048, h = 3072: 96
// tiles on 36 clusters, 292 against 384; the forward 5.6 % faster). Measured and not kept:
// 128-wide split tiles (at T = 2048, h = 1536 the forward took 81 us against 68 us unsplit), and
// clusters of three or four pairs, which fit only 23 or 15 at a time on the 152-SM GB300 and beat
// two pairs at no layer shape of the Megatron-LM sweep.
constexpr int SPLIT_PAIRS = 2;
constexpr int SPLIT_HOP_KB = 4;
constexpr int SPLIT_MIN_KB = 16;

static long long tiles_of(int M, int N, int bn) { return static_cast<long long>(ceil_div(M, 2 * BM)) * ceil_div(N, bn); }

// True when the split kernel should run this GEMM (M x N, L K blocks) instead of the
// single-pair kernel with BN1-wide tiles.
template <int BN1>
static bool use_split(int M, int N, int L, int sms) {
    const int pairs = resident_pairs<BN1, EPI_STORE, 4>(sms);
    const int clusters = resident_split_clusters<256, SPLIT_PAIRS>(sms);
    if (clusters <= 0 || L < SPLIT_MIN_KB * SPLIT_PAIRS) return false;
    const long long one = (tiles_of(M, N, BN1) + pairs - 1) / pairs * L * BN1;  // x 1/256 K-block times
    const long long two =
        ((tiles_of(M, N, 256) + clusters - 1) / clusters * ceil_div(L, SPLIT_PAIRS) + SPLIT_HOP_KB) * 256;
    return two * 10 <= one * 9;
}

static GemmArgs launch_args(uint32_t* status) {
    GemmArgs a{};
    a.tiles_per_unit = 1;
    a.status = status;
    a.budget_ns = wait_budget_ns();
    return a;
}

}  // namespace mptp

using namespace mptp;

extern "C" mp_status mp_mlp_fwd_shards(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, mp_bf16* Z,
                                       mp_bf16* Y, mp_bf16* U_save, int T, int h, int f, int t, int shard_begin,
                                       int shard_count, uint32_t* d_status, void* stream) {
    mp_status st = check_mlp_shape(T, h, f, t);
    if (st != MP_OK) return st;
    if ((st = check_shard_range(t, shard_begin, shard_count)) != MP_OK) return st;
    if (T == 0) return MP_OK;
    if (!X || !A || !B || !Z || !Y) return MP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Z) || !aligned16(Y) ||
        (U_save && !aligned16(U_save)) || (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return MP_ERR_MISALIGNED;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const double Tb = 2.0 * T, hb = 2.0 * h;
    // The range's columns of A, Y and U: [c0, c0 + nc), whole 64-wide blocks (f/t % 64 == 0).
    const int fs = f / t;
    const int c0 = shard_begin * fs, nc = shard_count * fs;

    // K1: column-parallel GEMM + GeLU over the range's columns: U = X A_r (A MN-major), Y = GeLU(U).
    TmapSet m1{};
    int b1 = 0;
    if (!make_tmap_bf16(&m1.a, X, h, T, h, 64, BM) || !(b1 = make_tmap_mn_operand(&m1.b, A + c0, nc, h, f)) ||
        !make_tmap_bf16_out(&m1.o0, Y + c0, nc, T, f) ||
        (U_save && !make_tmap_bf16_out(&m1.o1, U_save + c0, nc, T, f)))
        return MP_ERR_CUDA;
    GemmArgs a1 = launch_args(d_status);
    a1.pr = problem(T, nc, 256, 0, h / BK, false, true, Tb * h, hb * nc);
    a1.pr.b_mn = b1;
    a1.has_out1 = U_save ? 1 : 0;
    if (launch_gelu_epi<EPI_GELU>(m1, a1, sms, s) != cudaSuccess) return MP_ERR_CUDA;

    // K2: row-parallel GEMM Z = sum_i Y_i B_i over the range; K blocks of shard i are
    // [i*f/t, (i+1)*f/t) / BK, visited for i = s0..s0+n-1 in order, all into the same
    // accumulator (the g sum).
    TmapSet m2{};
    int b2 = 0;
    if (!make_tmap_bf16(&m2.a, Y, f, T, f, 64, BM) || !(b2 = make_tmap_mn_operand(&m2.b, B, h, f, h)) ||
        !make_tmap_bf16_out(&m2.o0, Z, h, T, h))
        return MP_ERR_CUDA;
    GemmArgs a2 = launch_args(d_status);
    a2.pr = problem(T, h, 256, c0 / BK, (c0 + nc) / BK, false, true, Tb * nc, hb * nc);
    a2.pr.b_mn = b2;
    const bool split2 = use_split<256>(T, h, nc / BK, sms);
    if ((split2 ? launch_gemm_split<256, SPLIT_PAIRS>(m2, a2, sms, s) : launch_gemm_tc<256, EPI_STORE, 4>(m2, a2, sms, s)) !=
        cudaSuccess)
        return MP_ERR_CUDA;
    return MP_OK;
}

extern "C" mp_status mp_mlp_fwd(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, mp_bf16* Z, mp_bf16* Y,
                                mp_bf16* U_save, int T, int h, int f, int t, uint32_t* d_status, void* stream) {
    return mp_mlp_fwd_shards(X, A, B, Z, Y, U_save, T, h, f, t, 0, t, d_status, stream);
}

extern "C" mp_status mp_mlp_bwd_shards(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, const mp_bf16* U,
                                       const mp_bf16* Y, const mp_bf16* dZ, mp_bf16* dX, mp_bf16* dA, mp_bf16* dB,
                                       mp_bf16* dU_ws, int T, int h, int f, int t, int shard_begin, int shard_count,
                                       uint32_t* d_status, void* stream) {
    mp_status st = check_mlp_shape(T, h, f, t);
    if (st != MP_OK) return st;
    if ((st = check_shard_range(t, shard_begin, shard_count)) != MP_OK) return st;
    if (!A || !B || !dA || !dB) return MP_ERR_INVALID_ARG;
    if (T > 0 && (!X || !U || !Y || !dZ || !dX || !dU_ws)) return MP_ERR_INVALID_ARG;
    const void* ptrs[] = {X, A, B, U, Y, dZ, dX, dA, dB, dU_ws};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MP_ERR_MISALIGNED;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MP_ERR_MISALIGNED;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // The range's columns of U, Y, dU, dA and rows of B, dB: [c0, c0 + nc).
    const int fs = f / t;
    const int c0 = shard_begin * fs, nc = shard_count * fs;
    if (T == 0) {
        // Empty batch: the range's weight gradients are sums over zero tokens.
        if (cudaMemset2DAsync(dA + c0, size_t(f) * 2, 0, size_t(nc) * 2, size_t(h), s) != cudaSuccess ||
            cudaMemsetAsync(dB + size_t(c0) * h, 0, size_t(nc) * h * 2, s) != cudaSuccess)
            return MP_ERR_CUDA;
        return MP_OK;
    }
    const double Tb = 2.0 * T, hb = 2.0 * h, fb = 2.0 * nc;

    // K3: dU_r = (dZ B_r^T) * GeLU'(U_r).  A operand dZ [T,h] (K-major), B operand the range's rows
    // of B [f,h] (K-major).
    TmapSet m3{};
    if (!make_tmap_bf16(&m3.a, dZ, h, T, h, 64, BM) || !make_tmap_bf16(&m3.b, B + size_t(c0) * h, h, nc, h, 64, 128) ||
        !make_tmap_bf16_out(&m3.o0, dU_ws + c0, nc, T, f))
        return MP_ERR_CUDA;
    GemmArgs a3 = launch_args(d_status);
    a3.pr = problem(T, nc, 256, 0, h / BK, false, false, Tb * h, fb * h);
    a3.aux = reinterpret_cast<const __nv_bfloat16*>(U + c0);
    a3.ld_aux = f;
    if (launch_gelu_epi<EPI_DGELU>(m3, a3, sms, s) != cudaSuccess) return MP_ERR_CUDA;

    // K4: dX = sum_i dU_i A_i^T.  A operand dU [T,f] (K-major), B operand A [h,f] (K-major); K blocks of
    // shard i are [i*f/t, (i+1)*f/t) / BK, visited for i = s0..s0+n-1 in order (the f sum).
    TmapSet m4{};
    if (!make_tmap_bf16(&m4.a, dU_ws, f, T, f, 64, BM) || !make_tmap_bf16(&m4.b, A, f, h, f, 64, K4_BN / 2) ||
        !make_tmap_bf16_out(&m4.o0, dX, h, T, h))
        return MP_ERR_CUDA;
    GemmArgs a4 = launch_args(d_status);
    a4.pr = problem(T, h, K4_BN, c0 / BK, (c0 + nc) / BK, false, false, Tb * nc, hb * nc);

    // K5a: dA_r = X^T dU_r (M = h, N = nc, K = T).  Both operands MN-major.
    TmapSet m5{};
    int a5f = 0, b5f = 0;
    if (!(a5f = make_tmap_mn_operand(&m5.a, X, h, T, h)) ||
        !(b5f = make_tmap_mn_operand(&m5.b, dU_ws + c0, nc, T, f)) || !make_tmap_bf16_out(&m5.o0, dA + c0, nc, h, f))
        return MP_ERR_CUDA;
    GemmArgs a5 = launch_args(d_status);
    a5.pr = problem(h, nc, 256, 0, ceil_div(T, BK), true, true, Tb * h, Tb * nc);
    a5.pr.a_mn = a5f;
    a5.pr.b_mn = b5f;

    // K5b: dB_r = Y_r^T dZ (M = nc, N = h, K = T).  Both operands MN-major.
    TmapSet m6{};
    int a6f = 0, b6f = 0;
    if (!(a6f = make_tmap_mn_operand(&m6.a, Y + c0, nc, T, f)) || !(b6f = make_tmap_mn_operand(&m6.b, dZ, h, T, h)) ||
        !make_tmap_bf16_out(&m6.o0, dB + size_t(c0) * h, h, nc, h))
        return MP_ERR_CUDA;
    GemmArgs a6 = launch_args(d_status);
    a6.pr = problem(nc, h, 256, 0, ceil_div(T, BK), true, true, Tb * nc, Tb * h);
    a6.pr.a_mn = a6f;
    a6.pr.b_mn = b6f;

    // Every output tile is computed by the same K-loop whichever pairs run it, so both
    // schedules give bitwise identical results.
    const int pairs = resident_pairs<256, EPI_STORE, 4>(sms);
    const int units[3] = {a4.pr.num_units, a5.pr.num_units, a6.pr.num_units};
    const int cost[3] = {a4.pr.kb_end - a4.pr.kb_begin + EPI_KB, a5.pr.kb_end - a5.pr.kb_begin + EPI_KB,
                         a6.pr.kb_end - a6.pr.kb_begin + EPI_KB};
    int split[3] = {pairs, pairs, pairs};
    const BwdSchedule mode = bwd_schedule();
    bool overlap = false;
    if (mode != BwdSchedule::Serial && pairs >= 3) {
        const long long side = split_pairs(pairs, 3, units, cost, split);
        overlap = mode == BwdSchedule::Overlap || side * 100 <= serial_makespan(pairs, 3, units, cost) * 94;
    }
    if (overlap) {
        std::lock_guard<std::mutex> lock(side_stream_mutex());
        SideStreams* ss = side_streams(s);
        if (ss != nullptr) {
            bool ok = cudaEventRecord(ss->fork, s) == cudaSuccess &&
                      cudaStreamWaitEvent(ss->s[0], ss->fork, 0) == cudaSuccess &&
                      cudaStreamWaitEvent(ss->s[1], ss->fork, 0) == cudaSuccess;
            if (!ok) return MP_ERR_CUDA;
            ok = launch_gemm_tc<K4_BN, EPI_STORE, 4>(m4, a4, sms, s, split[0]) == cudaSuccess;
            ok = launch_gemm_tc<256, EPI_STORE, 4>(m5, a5, sms, ss->s[0], split[1]) == cudaSuccess && ok;
            ok = launch_gemm_tc<256, EPI_STORE, 4>(m6, a6, sms, ss->s[1], split[2]) == cudaSuccess && ok;
            // Join even after a failed launch, so the caller's stream never runs ahead of the side streams.
            for (int i = 0; i < 2; ++i)
                ok = cudaEventRecord(ss->join[i], ss->s[i]) == cudaSuccess &&
                     cudaStreamWaitEvent(s, ss->join[i], 0) == cudaSuccess && ok;
            return ok ? MP_OK : MP_ERR_CUDA;
        }
    }
    const bool split4 = use_split<K4_BN>(T, h, nc / BK, sms);
    if (split4) {
        // The split kernel's 256-wide tiles: B boxes of 128 rows per CTA.
        if (!make_tmap_bf16(&m4.b, A, f, h, f, 64, 128)) return MP_ERR_CUDA;
        a4.pr = problem(T, h, 256, c0 / BK, (c0 + nc) / BK, false, false, Tb * nc, hb * nc);
    }
    if ((split4 ? launch_gemm_split<256, SPLIT_PAIRS>(m4, a4, sms, s) : launch_gemm_tc<K4_BN, EPI_STORE, 4>(m4, a4, sms, s)) !=
            cudaSuccess ||
        launch_gemm_tc<256, EPI_STORE, 4>(m5, a5, sms, s) != cudaSuccess ||
        launch_gemm_tc<256, EPI_STORE, 4>(m6, a6, sms, s) != cudaSuccess)
        return MP_ERR_CUDA;
    return MP_OK;
}

extern "C" mp_status mp_mlp_bwd(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, const mp_bf16* U,
                                const mp_bf16* Y, const mp_bf16* dZ, mp_bf16* dX, mp_bf16* dA, mp_bf16* dB,
                                mp_bf16* dU_ws, int T, int h, int f, int t, uint32_t* d_status, void* stream) {
    return mp_mlp_bwd_shards(X, A, B, U, Y, dZ, dX, dA, dB, dU_ws, T, h, f, t, 0, t, d_status, stream);
}
