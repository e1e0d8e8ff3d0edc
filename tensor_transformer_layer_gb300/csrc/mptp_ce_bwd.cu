// Entry point of the vocab-parallel cross-entropy backward: mp_vocab_ce_bwd.
//
// The pages describe the fused forward only ("Megatron-LM: Training Multi-Billion
// Parameter Language Models Using Model Parallelism", section 3.4, "Output Embedding
// Parallelism and the Fused Cross-Entropy Optimization"); the backward is the plain
// derivative of softmax cross-entropy: dZ = dloss * (softmax(z) - onehot(target)),
// dX = dZ E, dE = dZ^T X. It keeps the forward's vocabulary partition: for shard i
// (rows [i v_pad/t, (i+1) v_pad/t) of E), in ascending order,
//   K10  z_i = X E_i^T recomputed; the epilogue turns it into dZ_i (bf16) from the
//        per-token log-sum-exp, so only one shard of logit gradients exists at a time;
//   K11  dE_i = dZ_i^T X  (both operands MN-major);
//   K12  dX += dZ_i E_i   (fp32 accumulation across shards in shard order - the sum the
//        forward's all-reduce would carry: shard 0's tiles are stored, later shards' tiles
//        added at L2 by TMA reductions, and the last shard adds the accumulator in registers
//        and stores bf16).
// Shard by shard, each shard's three GEMMs run as one launch of the chain kernel
// (mptp_gemm_chain.cuh): a K12 tile starts on a block of tokens once K10 has written
// that block's dZ rows, a K11 tile once K10 has written its 256 vocabulary columns,
// so the GEMMs share the SMs instead of each ending in a part-empty wave. The tiles
// and K-loops are the separate kernels' (MPTP_CE_BWD_CHAIN=0 runs those instead, as does a
// shard with more tiles than the chain's schedule table holds), so the gradients are the
// same bit for bit. With every shard's dZ in the workspace (one
// pass), the three GEMMs run once each over the whole vocabulary.
// The log-sum-exp comes from the forward: either exported by it (mp_vocab_ce_lse, then
// mp_vocab_ce_bwd_lse), or rebuilt from its loss: lse = loss + z_target, with z_target
// = X[r] . E[target[r]] recomputed in fp32 (K9, mp_vocab_ce_bwd).
#include <cstdlib>

#include "mptp_gemm_chain.cuh"
#include "mptp_internal.h"

namespace mptp {

// One warp per token: lse[r] = loss[r] + X[r] . E[target[r]] (fp32 accumulation of
// bf16 products); NaN and MP_DEV_TARGET_RANGE for a target outside [0, v_valid).
__global__ void __launch_bounds__(256) ce_lse_kernel(const __nv_bfloat16* __restrict__ X,
                                                     const __nv_bfloat16* __restrict__ E,
                                                     const int32_t* __restrict__ target,
                                                     const float* __restrict__ loss, float* __restrict__ lse, int T,
                                                     int h, int v_valid, uint32_t* status) {
    grid_dependency_wait();  // the kernels that wrote the loss (and X) before it
    grid_launch_dependents();
    const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= T) return;
    const int tg = target[r];
    if (tg < 0 || tg >= v_valid) {
        if (lane == 0) {
            lse[r] = __int_as_float(0x7fc00000);
            if (status) atomicOr(status, DEV_TARGET_RANGE);
        }
        return;
    }
    const uint4* xr = reinterpret_cast<const uint4*>(X + static_cast<long long>(r) * h);
    const uint4* er = reinterpret_cast<const uint4*>(E + static_cast<long long>(tg) * h);
    float acc = 0.0f;
    for (int i = lane; i < h / 8; i += 32) {
        const uint4 a = xr[i], b = er[i];
        const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc = fmaf(bf16_lo(aw[j]), bf16_lo(bw[j]), acc);
            acc = fmaf(bf16_hi(aw[j]), bf16_hi(bw[j]), acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) lse[r] = loss[r] + acc;
}

// Workspace: lse [T] fp32, then either (shard by shard, t > 1) the chain kernel's counters, an fp32
// dX accumulator [T, h] and one shard's dZ [T, v_pad / t] bf16, or (one pass, `chunks` = 1) every
// shard's dZ [T, v_pad] bf16.
struct CeBwdLayout {
    size_t lse_off, ctr_off, ctr_bytes, acc_off, dz_off, total;
    int chunks;  // vocabulary chunks processed one after another: t (shard by shard) or 1
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static bool ce_bwd_layout(int T, int h, int v_pad, int t, bool one_pass, CeBwdLayout* L) {
    if (T < 0 || h <= 0 || t < 1 || v_pad <= 0 || v_pad % (128 * t) != 0) return false;
    L->chunks = one_pass ? 1 : t;
    const size_t vc = static_cast<size_t>(v_pad / L->chunks);
    L->lse_off = 0;
    L->ctr_off = align256(size_t(T) * 4);
    L->ctr_bytes = L->chunks == 1 ? 0 : chain_counter_bytes(T, static_cast<int>(vc));  // one chunk: no chain
    L->acc_off = L->ctr_off + L->ctr_bytes;
    L->dz_off = L->acc_off + (L->chunks == 1 ? 0 : align256(size_t(T) * h * 4));  // one chunk: no accumulator
    L->total = L->dz_off + align256(size_t(T) * vc * 2);
    return true;
}

}  // namespace mptp

using namespace mptp;

extern "C" size_t mp_vocab_ce_bwd_workspace_bytes(int T, int h, int v_pad, int t) {
    CeBwdLayout L;
    if (!ce_bwd_layout(T, h, v_pad, t, false, &L)) return 0;
    return L.total;
}

extern "C" size_t mp_vocab_ce_bwd_workspace_bytes_one_pass(int T, int h, int v_pad, int t) {
    CeBwdLayout L;
    if (!ce_bwd_layout(T, h, v_pad, t, true, &L)) return 0;
    return L.total;
}

// The backward from either the forward's loss (lse rebuilt by K9) or its exported lse.
static mp_status ce_bwd(const mp_bf16* X, const mp_bf16* E, const int32_t* target, const float* loss,
                        const float* lse_in, const float* dloss, mp_bf16* dX, mp_bf16* dE, void* workspace,
                        size_t workspace_bytes, int T, int h, int v_pad, int v_valid, int t, uint32_t* d_status,
                        void* stream) {
    if (T < 0 || h <= 0 || v_pad <= 0 || t < 1 || v_valid < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || v_pad % (128 * t) != 0 || v_valid > v_pad) return MP_ERR_UNSUPPORTED_SHAPE;
    if (!E || !dE) return MP_ERR_INVALID_ARG;
    if (T > 0 && (!X || !target || !(loss || lse_in) || !dloss || !dX || !workspace)) return MP_ERR_INVALID_ARG;
    const void* ptrs[] = {X, E, target, loss, lse_in, dloss, dX, dE, workspace};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MP_ERR_MISALIGNED;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MP_ERR_MISALIGNED;
    CeBwdLayout lay, one;
    ce_bwd_layout(T, h, v_pad, t, false, &lay);
    ce_bwd_layout(T, h, v_pad, t, true, &one);
    if (T > 0 && workspace_bytes < lay.total) return MP_ERR_WORKSPACE;
    if (workspace_bytes >= one.total) lay = one;  // room for every shard's dZ: one pass
    int sms = 0;
    mp_status st = check_device(&sms);
    if (st != MP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // No tokens: the embedding gradient is a sum over zero tokens.
        return cudaMemsetAsync(dE, 0, size_t(v_pad) * h * 2, s) == cudaSuccess ? MP_OK : MP_ERR_CUDA;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    float* lse_ws = reinterpret_cast<float*>(ws + lay.lse_off);
    float* acc = reinterpret_cast<float*>(ws + lay.acc_off);
    __nv_bfloat16* dz = reinterpret_cast<__nv_bfloat16*>(ws + lay.dz_off);
    const __nv_bfloat16* Xb = reinterpret_cast<const __nv_bfloat16*>(X);
    const __nv_bfloat16* Eb = reinterpret_cast<const __nv_bfloat16*>(E);

    const float* lse = lse_in;
    if (lse == nullptr) {
        if (launch_pdl(ce_lse_kernel, dim3(ceil_div(T, 8)), dim3(256), 0, s, Xb, Eb, target, loss, lse_ws, T, h,
                       v_valid, d_status) != cudaSuccess ||
            cudaGetLastError() != cudaSuccess)
            return MP_ERR_CUDA;
        lse = lse_ws;
    }

    // Vocabulary chunks of vs columns (whole shards, in shard order): one chunk when the
    // workspace holds every shard's dZ, else one shard at a time.
    const int C = lay.chunks;
    const int vs = v_pad / C;
    const double Tb = 2.0 * T, hb = 2.0 * h, vb = 2.0 * vs;
    const unsigned long long budget = wait_budget_ns();
    const char* chain_env = std::getenv("MPTP_CE_BWD_CHAIN");
    const bool chain_off = chain_env && chain_env[0] == '0' && chain_env[1] == '\0';
    // The chain only where a shard's list fits the precomputed schedule (T up to about 32k tokens
    // at v_pad / t = 6400): beyond it the chain would take its units round-robin, which leaves
    // pairs waiting on dependencies that a schedule would have placed after other work.
    const long long mbT = ceil_div(T, 2 * BM), ncv = ceil_div(vs, CHAIN_BN), nch = ceil_div(h, CHAIN_BN);
    const long long chain_units = mbT * ncv + mbT * nch + ncv * nch;  // a shard's K10, K12, K11 tiles
    if (C > 1 && !chain_off && chain_units <= CHAIN_MAX_SCHED) {
        // Each shard's K10, K12 and K11 in one chain launch; its counters start at zero and every
        // launch returns them to zero for the next.
        uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + lay.ctr_off);
        if (cudaMemsetAsync(ctr, 0, lay.ctr_bytes, s) != cudaSuccess) return MP_ERR_CUDA;
        for (int i = 0; i < C; ++i) {
            const __nv_bfloat16* Ei = Eb + static_cast<long long>(i) * vs * h;
            __nv_bfloat16* dEi = reinterpret_cast<__nv_bfloat16*>(dE) + static_cast<long long>(i) * vs * h;
            ChainMaps m{};
            ChainArgs a{};
            // problem 0, K10: z_i = X E_i^T -> dZ_i (both operands K-major)
            if (!make_tmap_bf16(&m.m[0].a, X, h, T, h, 64, BM) ||
                !make_tmap_bf16(&m.m[0].b, Ei, h, vs, h, 64, CHAIN_BN / 2) ||
                !make_tmap_bf16_out(&m.m[0].o0, dz, vs, T, vs))
                return MP_ERR_CUDA;
            a.p[0] = chain_problem(T, vs, 0, h / BK, 0, 0, 1);
            // problem 1, K12: dX (+)= dZ_i E_i (E_i MN-major), reads K10's rows
            int b12 = 0;
            if (!make_tmap_bf16(&m.m[1].a, dz, vs, T, vs, 64, BM) || !(b12 = make_tmap_mn_operand(&m.m[1].b, Ei, h, vs, h)) ||
                !make_tmap_bf16_out(&m.m[1].o0, dX, h, T, h) || !make_tmap_f32_out(&m.m[1].o1, acc, h, T, h))
                return MP_ERR_CUDA;
            a.p[1] = chain_problem(T, h, 0, vs / BK, 0, b12, 1);
            a.p[1].dep = DEP_ROWS;
            // problem 2, K11: dE_i = dZ_i^T X (both MN-major), tile i of its rows reads K10's column tile i
            int a11 = 0, b11 = 0;
            if (!(a11 = make_tmap_mn_operand(&m.m[2].a, dz, vs, T, vs)) || !(b11 = make_tmap_mn_operand(&m.m[2].b, X, h, T, h)) ||
                !make_tmap_bf16_out(&m.m[2].o0, dEi, h, vs, h))
                return MP_ERR_CUDA;
            a.p[2] = chain_problem(vs, h, 0, ceil_div(T, BK), a11, b11, ceil_div(vs, 2 * BM));
            a.p[2].dep = DEP_COLS_M;
            a.target = target;
            a.lse = lse;
            a.dloss = dloss;
            a.v_valid = v_valid;
            a.col_off = i * vs;
            a.acc = acc;
            a.ld_acc = h;
            a.acc_mode = i == 0 ? ACC_FIRST : (i == C - 1 ? ACC_LAST : ACC_MID);
            a.status = d_status;
            a.budget_ns = budget;
            st = launch_chain_ce(m, a, sms, s, ctr);
            if (st == CHAIN_NO_SCHEDULE && i == 0) break;  // no schedule: the separate launches below
            if (st != MP_OK) return st;
        }
        if (st == MP_OK) return MP_OK;
    }
    for (int i = 0; i < C; ++i) {
        const __nv_bfloat16* Ei = Eb + static_cast<long long>(i) * vs * h;
        __nv_bfloat16* dEi = reinterpret_cast<__nv_bfloat16*>(dE) + static_cast<long long>(i) * vs * h;

        // K10: z_i = X E_i^T -> dZ_i (bf16, [T, vs]) in the workspace.
        TmapSet m10{};
        if (!make_tmap_bf16(&m10.a, X, h, T, h, 64, BM) || !make_tmap_bf16(&m10.b, Ei, h, vs, h, 64, 128) ||
            !make_tmap_bf16_out(&m10.o0, dz, vs, T, vs))
            return MP_ERR_CUDA;
        GemmArgs a10{};
        a10.pr.M = T;
        a10.pr.N = vs;
        a10.pr.num_m_blocks = ceil_div(T, 2 * BM);
        a10.pr.num_units = a10.pr.num_m_blocks * ceil_div(vs, 256);
        a10.pr.n_fastest = n_fastest_order(Tb * h, vb * h);
        a10.pr.kb_begin = 0;
        a10.pr.kb_end = h / BK;
        a10.tiles_per_unit = 1;
        a10.target = target;
        a10.v_valid = v_valid;
        a10.col_off = i * vs;
        a10.lse = lse;
        a10.dloss = dloss;
        a10.status = d_status;
        a10.budget_ns = budget;
        if (launch_gemm_tc<256, EPI_DZ, 8>(m10, a10, sms, s) != cudaSuccess) return MP_ERR_CUDA;

        // K11: dE_i = dZ_i^T X (M = vs, N = h, K = T; both operands MN-major).
        TmapSet m11{};
        int a11f = 0, b11f = 0;
        if (!(a11f = make_tmap_mn_operand(&m11.a, dz, vs, T, vs)) || !(b11f = make_tmap_mn_operand(&m11.b, X, h, T, h)) ||
            !make_tmap_bf16_out(&m11.o0, dEi, h, vs, h))
            return MP_ERR_CUDA;
        GemmArgs a11{};
        a11.pr.M = vs;
        a11.pr.N = h;
        a11.pr.num_m_blocks = ceil_div(vs, 2 * BM);
        a11.pr.num_units = a11.pr.num_m_blocks * ceil_div(h, 256);
        a11.pr.n_fastest = n_fastest_order(Tb * vs, Tb * h);
        a11.pr.kb_begin = 0;
        a11.pr.kb_end = ceil_div(T, BK);
        a11.pr.a_mn = a11f;
        a11.pr.b_mn = b11f;
        a11.tiles_per_unit = 1;
        a11.status = d_status;
        a11.budget_ns = budget;
        if (launch_gemm_tc<256, EPI_STORE, 4>(m11, a11, sms, s) != cudaSuccess) return MP_ERR_CUDA;

        // K12: dX (+)= dZ_i E_i (M = T, N = h, K = vs; A K-major, B = E_i MN-major), shards in order.
        TmapSet m12{};
        int b12f = 0;
        if (!make_tmap_bf16(&m12.a, dz, vs, T, vs, 64, BM) || !(b12f = make_tmap_mn_operand(&m12.b, Ei, h, vs, h)) ||
            !make_tmap_bf16_out(&m12.o0, dX, h, T, h) || (C > 1 && !make_tmap_f32_out(&m12.o1, acc, h, T, h)))
            return MP_ERR_CUDA;
        GemmArgs a12{};
        a12.pr.M = T;
        a12.pr.N = h;
        a12.pr.num_m_blocks = ceil_div(T, 2 * BM);
        a12.pr.num_units = a12.pr.num_m_blocks * ceil_div(h, 256);
        a12.pr.n_fastest = n_fastest_order(Tb * vs, vb * h);
        a12.pr.kb_begin = 0;
        a12.pr.kb_end = vs / BK;
        a12.pr.a_mn = 0;
        a12.pr.b_mn = b12f;
        a12.tiles_per_unit = 1;
        a12.acc = C == 1 ? nullptr : acc;  // one pass: ACC_ONLY, no fp32 accumulator
        a12.ld_acc = h;
        a12.acc_mode = (C == 1) ? ACC_ONLY : (i == 0 ? ACC_FIRST : (i == C - 1 ? ACC_LAST : ACC_MID));
        a12.status = d_status;
        a12.budget_ns = budget;
        if (launch_gemm_tc<256, EPI_ACC, 4>(m12, a12, sms, s) != cudaSuccess) return MP_ERR_CUDA;
    }
    return MP_OK;
}

extern "C" mp_status mp_vocab_ce_bwd(const mp_bf16* X, const mp_bf16* E, const int32_t* target, const float* loss,
                                     const float* dloss, mp_bf16* dX, mp_bf16* dE, void* workspace,
                                     size_t workspace_bytes, int T, int h, int v_pad, int v_valid, int t,
                                     uint32_t* d_status, void* stream) {
    if (T > 0 && !loss) return MP_ERR_INVALID_ARG;
    return ce_bwd(X, E, target, loss, nullptr, dloss, dX, dE, workspace, workspace_bytes, T, h, v_pad, v_valid, t,
                  d_status, stream);
}

extern "C" mp_status mp_vocab_ce_bwd_lse(const mp_bf16* X, const mp_bf16* E, const int32_t* target, const float* lse,
                                         const float* dloss, mp_bf16* dX, mp_bf16* dE, void* workspace,
                                         size_t workspace_bytes, int T, int h, int v_pad, int v_valid, int t,
                                         uint32_t* d_status, void* stream) {
    if (T > 0 && !lse) return MP_ERR_INVALID_ARG;
    return ce_bwd(X, E, target, nullptr, lse, dloss, dX, dE, workspace, workspace_bytes, T, h, v_pad, v_valid, t,
                  d_status, stream);
}
