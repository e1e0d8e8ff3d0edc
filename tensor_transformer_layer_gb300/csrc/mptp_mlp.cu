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
#include "mptp_gemm.cuh"
#include "mptp_internal.h"

namespace mptp {

static mp_status check_mlp_shape(int T, int h, int f, int t) {
    if (T < 0 || h <= 0 || f <= 0 || t < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || f % t != 0 || (f / t) % 64 != 0) return MP_ERR_UNSUPPORTED_SHAPE;
    return MP_OK;
}

// a_bytes / b_bytes: sizes of the A (M side) and B (N side) operands, for the unit order.
static GemmArgs base_args(int M, int N, int bn, int kb_begin, int kb_end, double a_bytes, double b_bytes,
                          uint32_t* status) {
    GemmArgs a{};
    a.M = M;
    a.N = N;
    a.num_m_blocks = ceil_div(M, 2 * BM);  // 256-row blocks: one per CTA-pair tile
    a.tiles_per_unit = 1;
    a.num_units = a.num_m_blocks * ceil_div(N, bn);
    a.n_fastest = n_fastest_order(a_bytes, b_bytes);
    a.kb_begin = kb_begin;
    a.kb_end = kb_end;
    a.status = status;
    a.budget_ns = wait_budget_ns();
    return a;
}

}  // namespace mptp

using namespace mptp;

extern "C" mp_status mp_mlp_fwd(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, mp_bf16* Z, mp_bf16* Y,
                                mp_bf16* U_save, int T, int h, int f, int t, uint32_t* d_status, void* stream) {
    mp_status st = check_mlp_shape(T, h, f, t);
    if (st != MP_OK) return st;
    if (T == 0) return MP_OK;
    if (!X || !A || !B || !Z || !Y) return MP_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(A) || !aligned16(B) || !aligned16(Z) || !aligned16(Y) ||
        (U_save && !aligned16(U_save)) || (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return MP_ERR_MISALIGNED;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const double Tb = 2.0 * T, hb = 2.0 * h;
    CUtensorMap tmX, tmA, tmY, tmB, tmYo, tmUo, tmZo;
    if (!make_tmap_bf16(&tmX, X, h, T, h, 64, BM) || !make_tmap_bf16(&tmA, A, f, h, f, 64, 64) ||
        !make_tmap_bf16(&tmY, Y, f, T, f, 64, BM) || !make_tmap_bf16(&tmB, B, h, f, h, 64, 64) ||
        !make_tmap_bf16_out(&tmYo, Y, f, T, f) || !make_tmap_bf16_out(&tmZo, Z, h, T, h) ||
        !make_tmap_bf16_out(&tmUo, U_save ? static_cast<const void*>(U_save) : static_cast<const void*>(Y), f, T, f))
        return MP_ERR_CUDA;

    // K1: column-parallel GEMM + GeLU over all shards' columns.
    GemmArgs a1 = base_args(T, f, 256, 0, h / BK, Tb * h, hb * f, d_status);
    a1.out0 = reinterpret_cast<__nv_bfloat16*>(Y);
    a1.ld0 = f;
    a1.out1 = reinterpret_cast<__nv_bfloat16*>(U_save);
    a1.ld1 = f;
    if (launch_gemm_tc<256, false, true, EPI_GELU, 8>(tmX, tmA, tmYo, tmUo, a1, sms, s) != cudaSuccess)
        return MP_ERR_CUDA;

    // K2: row-parallel GEMM; K blocks of shard i are [i*f/t, (i+1)*f/t) / BK, visited
    // for i = 0..t-1 in order, all into the same accumulator (the g sum).
    const int fs = f / t;
    GemmArgs a2 = base_args(T, h, 256, 0 * (fs / BK), t * (fs / BK), Tb * f, hb * f, d_status);
    a2.out0 = reinterpret_cast<__nv_bfloat16*>(Z);
    a2.ld0 = h;
    if (launch_gemm_tc<256, false, true, EPI_STORE, 4>(tmY, tmB, tmZo, tmZo, a2, sms, s) != cudaSuccess)
        return MP_ERR_CUDA;
    return MP_OK;
}

extern "C" mp_status mp_mlp_bwd(const mp_bf16* X, const mp_bf16* A, const mp_bf16* B, const mp_bf16* U,
                                const mp_bf16* Y, const mp_bf16* dZ, mp_bf16* dX, mp_bf16* dA, mp_bf16* dB,
                                mp_bf16* dU_ws, int T, int h, int f, int t, uint32_t* d_status, void* stream) {
    mp_status st = check_mlp_shape(T, h, f, t);
    if (st != MP_OK) return st;
    if (!A || !B || !dA || !dB) return MP_ERR_INVALID_ARG;
    if (T > 0 && (!X || !U || !Y || !dZ || !dX || !dU_ws)) return MP_ERR_INVALID_ARG;
    const void* ptrs[] = {X, A, B, U, Y, dZ, dX, dA, dB, dU_ws};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return MP_ERR_MISALIGNED;
    if (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)) return MP_ERR_MISALIGNED;
    int sms = 0;
    if ((st = check_device(&sms)) != MP_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // Empty batch: the weight gradients are sums over zero tokens.
        if (cudaMemsetAsync(dA, 0, size_t(h) * f * 2, s) != cudaSuccess ||
            cudaMemsetAsync(dB, 0, size_t(f) * h * 2, s) != cudaSuccess)
            return MP_ERR_CUDA;
        return MP_OK;
    }

    // K3: dU = (dZ B^T) * GeLU'(U).  A operand dZ [T,h] (K-major), B operand B [f,h] (K-major).
    const double Tb = 2.0 * T, hb = 2.0 * h, fb = 2.0 * f;
    CUtensorMap tm_dZ_k, tm_B_k, tm_dU_o;
    if (!make_tmap_bf16(&tm_dZ_k, dZ, h, T, h, 64, BM) || !make_tmap_bf16(&tm_B_k, B, h, f, h, 64, 128) ||
        !make_tmap_bf16_out(&tm_dU_o, dU_ws, f, T, f))
        return MP_ERR_CUDA;
    GemmArgs a3 = base_args(T, f, 256, 0, h / BK, Tb * h, fb * h, d_status);
    a3.out0 = reinterpret_cast<__nv_bfloat16*>(dU_ws);
    a3.ld0 = f;
    a3.aux = reinterpret_cast<const __nv_bfloat16*>(U);
    a3.ld_aux = f;
    if (launch_gemm_tc<256, false, false, EPI_DGELU, 8>(tm_dZ_k, tm_B_k, tm_dU_o, tm_dU_o, a3, sms, s) !=
        cudaSuccess)
        return MP_ERR_CUDA;

    // K4: dX = sum_i dU_i A_i^T.  A operand dU [T,f] (K-major), B operand A [h,f] (K-major).
    CUtensorMap tm_dU_k, tm_A_k, tm_dX_o;
    if (!make_tmap_bf16(&tm_dU_k, dU_ws, f, T, f, 64, BM) || !make_tmap_bf16(&tm_A_k, A, f, h, f, 64, 128) ||
        !make_tmap_bf16_out(&tm_dX_o, dX, h, T, h))
        return MP_ERR_CUDA;
    const int fs = f / t;
    GemmArgs a4 = base_args(T, h, 256, 0 * (fs / BK), t * (fs / BK), Tb * f, hb * f, d_status);
    a4.out0 = reinterpret_cast<__nv_bfloat16*>(dX);
    a4.ld0 = h;
    if (launch_gemm_tc<256, false, false, EPI_STORE, 4>(tm_dU_k, tm_A_k, tm_dX_o, tm_dX_o, a4, sms, s) !=
        cudaSuccess)
        return MP_ERR_CUDA;

    // K5a: dA = X^T dU (M = h, N = f, K = T).  Both operands MN-major.
    CUtensorMap tm_X_mn, tm_dU_mn, tm_dA_o;
    if (!make_tmap_bf16(&tm_X_mn, X, h, T, h, 64, 64) || !make_tmap_bf16(&tm_dU_mn, dU_ws, f, T, f, 64, 64) ||
        !make_tmap_bf16_out(&tm_dA_o, dA, f, h, f))
        return MP_ERR_CUDA;
    GemmArgs a5 = base_args(h, f, 256, 0, ceil_div(T, BK), Tb * h, Tb * f, d_status);
    a5.out0 = reinterpret_cast<__nv_bfloat16*>(dA);
    a5.ld0 = f;
    if (launch_gemm_tc<256, true, true, EPI_STORE, 4>(tm_X_mn, tm_dU_mn, tm_dA_o, tm_dA_o, a5, sms, s) !=
        cudaSuccess)
        return MP_ERR_CUDA;

    // K5b: dB = Y^T dZ (M = f, N = h, K = T).  Both operands MN-major.
    CUtensorMap tm_Y_mn, tm_dZ_mn, tm_dB_o;
    if (!make_tmap_bf16(&tm_Y_mn, Y, f, T, f, 64, 64) || !make_tmap_bf16(&tm_dZ_mn, dZ, h, T, h, 64, 64) ||
        !make_tmap_bf16_out(&tm_dB_o, dB, h, f, h))
        return MP_ERR_CUDA;
    GemmArgs a6 = base_args(f, h, 256, 0, ceil_div(T, BK), Tb * f, Tb * h, d_status);
    a6.out0 = reinterpret_cast<__nv_bfloat16*>(dB);
    a6.ld0 = h;
    if (launch_gemm_tc<256, true, true, EPI_STORE, 4>(tm_Y_mn, tm_dZ_mn, tm_dB_o, tm_dB_o, a6, sms, s) !=
        cudaSuccess)
        return MP_ERR_CUDA;
    return MP_OK;
}
