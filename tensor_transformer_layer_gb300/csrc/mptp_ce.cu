// Entry points of the vocab-parallel fused output GEMM + cross-entropy
// ("Megatron-LM: Training Multi-Billion Parameter Language Models Using Model
// Parallelism", section 3.4, "Output Embedding Parallelism and the Fused
// Cross-Entropy Optimization", steps 1-6).
//
//   K6  logits X E_p^T per (128-token block, vocabulary partition p); the
//       epilogue keeps, per token, the running max m_p, the sum of exp(z - m_p)
//       and the target logit, and writes the triple; logits stay on chip.
//   K7  per token: M = max_p m_p, S = sum_p s_p exp(m_p - M),
//       loss = M + log S - z_target (the page's two all-reduces and final step); on request
//       also lse = M + log S, the per-token log-sum-exp the backward needs.
#include "mptp_gemm.cuh"
#include "mptp_internal.h"

namespace mptp {

// K7 layout: lane = token (every load of a partition plane is one coalesced 128-byte line per
// warp). A block's W warps (W = 8 when G = 8, else 4) form W / G token groups of 32 tokens, and
// the G warps of a group split the partitions (share j takes j, j + G, j + 2G, ...). With few
// tokens G = 8 puts every partition's load in flight at once; with many, G = 1 is one thread
// per token over all partitions. Each warp issues CMB_LOADS partitions' loads before reducing
// them; a group's G partial (max, sum) pairs are merged in shared memory.
constexpr int CMB_WARPS = 8;  // warps per block at most
constexpr int CMB_LOADS = 8;  // partitions a warp loads before reducing them

// Fold partials (m_j, s_j) into the running (M, S): M = max, S = sum s_j exp(m_j - M), the
// running sum rescaled when M grows; partitions with no valid column (s = 0, m = -inf) skip.
__device__ __forceinline__ void lse_fold(float& M, float& S, const float (&mm)[CMB_LOADS], const float (&ss)[CMB_LOADS]) {
    float cm = mm[0];
#pragma unroll
    for (int j = 1; j < CMB_LOADS; ++j) cm = fmaxf(cm, mm[j]);
    const float nM = fmaxf(M, cm);
    if (nM == -INFINITY) return;
    S = (M == -INFINITY) ? 0.0f : S * expf(M - nM);
#pragma unroll
    for (int j = 0; j < CMB_LOADS; ++j)
        if (ss[j] > 0.0f) S += ss[j] * expf(mm[j] - nM);
    M = nM;
}

// SPLIT = false is the G = 1 form (no merge, fewer registers, more resident threads).
template <bool SPLIT>
__global__ void __launch_bounds__(32 * CMB_WARPS) ce_combine_kernel(const float* __restrict__ ws,
                                                                    const int32_t* __restrict__ target,
                                                                    float* __restrict__ loss,
                                                                    float* __restrict__ lse_out, int T, int P, int G,
                                                                    int chunk_cols, int v_valid, uint32_t* status) {
    grid_dependency_wait();  // the partials of the logit GEMM before it
    __shared__ float sM[SPLIT ? CMB_WARPS : 1][32], sS[SPLIT ? CMB_WARPS : 1][32];
    if (!SPLIT) G = 1;
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int grp = w / G, share = w % G;
    const int r = (blockIdx.x * (static_cast<int>(blockDim.x >> 5) / G) + grp) * 32 + lane;
    const bool valid = r < T;
    const long long stride = 3ll * T;
    float M = -INFINITY, S = 0.0f;
    if (valid) {
        for (int p0 = share; p0 < P; p0 += G * CMB_LOADS) {
            float mm[CMB_LOADS], ss[CMB_LOADS];
#pragma unroll
            for (int j = 0; j < CMB_LOADS; ++j) {
                const int p = p0 + j * G;
                mm[j] = (p < P) ? ws[p * stride + r] : -INFINITY;
                ss[j] = (p < P) ? ws[p * stride + T + r] : 0.0f;
            }
            lse_fold(M, S, mm, ss);
        }
    }
    if constexpr (SPLIT) {
        sM[w][lane] = M;
        sS[w][lane] = S;
        __syncthreads();
        if (share != 0 || !valid) return;
        float mm[CMB_LOADS], ss[CMB_LOADS];
#pragma unroll
        for (int j = 0; j < CMB_LOADS; ++j) {
            mm[j] = j < G ? sM[w + j][lane] : -INFINITY;
            ss[j] = j < G ? sS[w + j][lane] : 0.0f;
        }
        M = -INFINITY;
        S = 0.0f;
        lse_fold(M, S, mm, ss);
    } else if (!valid) {
        return;
    }
    const int tg = target[r];
    if (tg < 0 || tg >= v_valid) {
        loss[r] = __int_as_float(0x7fc00000);
        if (lse_out) lse_out[r] = __int_as_float(0x7fc00000);  // no gradient flows from this token
        if (status) atomicOr(status, DEV_TARGET_RANGE);
        return;
    }
    const float z = ws[(tg / chunk_cols) * stride + 2ll * T + r];
    const float l = M + logf(S);
    loss[r] = l - z;
    if (lse_out) lse_out[r] = l;
}
static_assert(CMB_WARPS <= CMB_LOADS, "a group's merge folds up to CMB_WARPS pairs in one pass");

// Warps per token group: the largest of 1, 2, 4, 8 that keeps the grid within about 27 warps a
// SM (measured on T = 8192, 32768 and 131172 tokens with 40 partitions: splitting further only
// adds blocks once the loads in flight already cover the DRAM latency).
static int combine_group(long long T, int sms) {
    const long long token_warps = (T + 31) / 32;
    int G = CMB_WARPS;
    while (G > 1 && token_warps * G > 27ll * sms) G >>= 1;
    return G;
}

static mp_status check_ce_shape(int T, int h, int v_pad, int v_valid, int t) {
    if (T < 0 || h <= 0 || v_pad <= 0 || t < 1 || v_valid < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || v_pad % (128 * t) != 0 || v_valid > v_pad) return MP_ERR_UNSUPPORTED_SHAPE;
    return MP_OK;
}

}  // namespace mptp

using namespace mptp;

extern "C" size_t mp_vocab_ce_workspace_bytes(int T, int v_pad, int t) { return ce_plan_workspace(T, v_pad, t, 0); }

extern "C" mp_status mp_vocab_ce_partials(const mp_bf16* X, const mp_bf16* E, const int32_t* target,
                                          void* workspace, size_t workspace_bytes, int T, int h, int v_pad,
                                          int v_valid, int t, uint32_t* d_status, void* stream) {
    mp_status st = check_ce_shape(T, h, v_pad, v_valid, t);
    if (st != MP_OK) return st;
    if (T == 0) return MP_OK;
    if (!X || !E || !target || !workspace) return MP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(E) || !aligned16(target) || !aligned16(workspace) ||
        (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return MP_ERR_MISALIGNED;
    // The partition follows the workspace given (the preferred plan when it fits).
    if (workspace_bytes < ce_plan_workspace(T, v_pad, t, workspace_bytes)) return MP_ERR_WORKSPACE;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    CePlan plan;
    ce_plan(T, v_pad, t, workspace_bytes, &plan);

    TmapSet m{};
    if (!make_tmap_bf16(&m.a, X, h, T, h, 64, BM) || !make_tmap_bf16(&m.b, E, h, v_pad, h, 64, plan.bn / 2))
        return MP_ERR_CUDA;
    GemmArgs a{};
    a.pr.M = T;
    a.pr.N = v_pad;
    a.pr.num_m_blocks = ceil_div(T, 2 * BM);  // 256-row blocks: one per CTA-pair tile
    a.pr.num_units = a.pr.num_m_blocks * plan.P;
    a.pr.n_fastest = 0;
    a.pr.kb_begin = 0;
    a.pr.kb_end = h / BK;
    a.pr.a_mn = 0;
    a.pr.b_mn = 0;
    a.tiles_per_unit = plan.tiles_per_unit;
    a.target = target;
    a.ws = static_cast<float*>(workspace);
    a.v_valid = v_valid;
    a.status = d_status;
    a.budget_ns = wait_budget_ns();
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = (plan.bn == 256) ? launch_gemm_tc<256, EPI_CE, 4>(m, a, sms, s)
                                     : launch_gemm_tc<128, EPI_CE, 4>(m, a, sms, s);
    return e == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

static mp_status ce_combine(const void* workspace, size_t workspace_bytes, const int32_t* target, float* loss,
                            float* lse, int T, int v_pad, int v_valid, int t, uint32_t* d_status, void* stream) {
    if (T < 0 || v_pad <= 0 || t < 1 || v_valid < 1) return MP_ERR_INVALID_ARG;
    if (v_pad % (128 * t) != 0 || v_valid > v_pad) return MP_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MP_OK;
    if (!workspace || !target || !loss) return MP_ERR_INVALID_ARG;
    if (!aligned16(workspace) || !aligned16(target) || !aligned16(loss) || (lse && !aligned16(lse)) ||
        (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return MP_ERR_MISALIGNED;
    if (workspace_bytes < ce_plan_workspace(T, v_pad, t, workspace_bytes)) return MP_ERR_WORKSPACE;
    int sms = 0;
    mp_status st = check_device(&sms);
    if (st != MP_OK) return st;
    CePlan plan;
    ce_plan(T, v_pad, t, workspace_bytes, &plan);
    const int G = combine_group(T, sms);
    const int W = G == CMB_WARPS ? CMB_WARPS : 4;  // warps per block
    const cudaError_t e = launch_pdl(G > 1 ? ce_combine_kernel<true> : ce_combine_kernel<false>,
                                     dim3(ceil_div(T, 32 * (W / G))), dim3(32 * W),
                                     0, static_cast<cudaStream_t>(stream), static_cast<const float*>(workspace),
                                     target, loss, lse, T, plan.P, G, plan.chunk_cols, v_valid, d_status);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}

extern "C" mp_status mp_vocab_ce_combine(const void* workspace, size_t workspace_bytes, const int32_t* target,
                                         float* loss, int T, int v_pad, int v_valid, int t, uint32_t* d_status,
                                         void* stream) {
    return ce_combine(workspace, workspace_bytes, target, loss, nullptr, T, v_pad, v_valid, t, d_status, stream);
}

static mp_status vocab_ce(const mp_bf16* X, const mp_bf16* E, const int32_t* target, float* loss, float* lse,
                          void* workspace, size_t workspace_bytes, int T, int h, int v_pad, int v_valid, int t,
                          uint32_t* d_status, void* stream) {
    mp_status st = check_ce_shape(T, h, v_pad, v_valid, t);
    if (st != MP_OK) return st;
    if (T == 0) return MP_OK;
    if (!loss) return MP_ERR_INVALID_ARG;
    if (!aligned16(loss) || (lse && !aligned16(lse))) return MP_ERR_MISALIGNED;
    st = mp_vocab_ce_partials(X, E, target, workspace, workspace_bytes, T, h, v_pad, v_valid, t, d_status, stream);
    if (st != MP_OK) return st;
    return ce_combine(workspace, workspace_bytes, target, loss, lse, T, v_pad, v_valid, t, d_status, stream);
}

extern "C" mp_status mp_vocab_ce(const mp_bf16* X, const mp_bf16* E, const int32_t* target, float* loss,
                                 void* workspace, size_t workspace_bytes, int T, int h, int v_pad, int v_valid,
                                 int t, uint32_t* d_status, void* stream) {
    return vocab_ce(X, E, target, loss, nullptr, workspace, workspace_bytes, T, h, v_pad, v_valid, t, d_status,
                    stream);
}

extern "C" mp_status mp_vocab_ce_lse(const mp_bf16* X, const mp_bf16* E, const int32_t* target, float* loss,
                                     float* lse, void* workspace, size_t workspace_bytes, int T, int h, int v_pad,
                                     int v_valid, int t, uint32_t* d_status, void* stream) {
    if (T > 0 && !lse) return MP_ERR_INVALID_ARG;
    return vocab_ce(X, E, target, loss, lse, workspace, workspace_bytes, T, h, v_pad, v_valid, t, d_status, stream);
}
