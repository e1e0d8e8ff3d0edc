// mp_vocab_ce_noalloc: the fused vocab-parallel cross-entropy for callers that
// cannot allocate device memory.
//
// Who needs it: a process whose device memory is owned by someone else's pool
// and that is not allowed to call cudaMalloc/cudaFree itself, for instance a
// serving runtime that reserves all of HBM at start-up and forbids any later
// allocation (cudaMalloc and cudaFree can synchronise the device and stall every
// stream), or a host framework whose memory accounting must see every byte.
// Such a caller cannot hand mp_vocab_ce a workspace of its own, so this entry
// point takes the per-token partition triples from a fixed-size static device
// array (4 MiB). CUDA places that array in device memory when it loads the code
// module that holds it: with lazy module loading (the CUDA default) that is the
// first call of this entry point on a device, T = 0 included, and not when the
// library is loaded. A caller whose pool later takes the rest of HBM makes one
// such call before it reserves the pool (or runs with CUDA_MODULE_LOADING=EAGER).
// From then on the device holds the 4 MiB until the process exits.
//
// The caller still passes X, E, the targets and the loss buffer; nothing here
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
#include "mptp_internal.h"

// Scratch for the triples: fp32 [P][3][T], at most MP_CE_NOALLOC_MAX_FLOATS floats.
// In host code this name is only a host-side stand-in; kernels must be given the
// device address obtained below.
static __device__ __align__(256) float g_ce_scratch[MP_CE_NOALLOC_MAX_FLOATS];

namespace {

// Device address of g_ce_scratch on the current device. Looked up on every call (a host-side
// query, no device work), so that a context re-created after cudaDeviceReset never receives a
// stale address. The first lookup on a device loads the module and places the array.
mp_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MP_ERR_NO_DEVICE;
    }
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_ce_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return MP_ERR_CUDA;
    }
    *out = p;
    return MP_OK;
}

}  // namespace

extern "C" mp_status mp_vocab_ce_noalloc(const mp_bf16* X, const mp_bf16* E, const int32_t* target, float* loss,
                                         int T, int h, int v_pad, int v_valid, int t, uint32_t* d_status,
                                         void* stream) {
    if (T < 0 || h <= 0 || v_pad <= 0 || t < 1 || v_valid < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || v_pad % (128 * t) != 0 || v_valid > v_pad) return MP_ERR_UNSUPPORTED_SHAPE;
    // The triples must fit in the static array (in the partition that fits it best); larger
    // problems are refused before any launch.
    const size_t need = mptp::ce_plan_workspace(T, v_pad, t, sizeof(g_ce_scratch));
    if (need > sizeof(g_ce_scratch) || (T > 0 && need == 0)) return MP_ERR_WORKSPACE;
    int sms = 0;
    mp_status st = mptp::check_device(&sms);
    if (st != MP_OK) return st;
    // Also for T = 0: the lookup places the array on this device (see the file comment).
    void* ws = nullptr;
    if ((st = scratch_address(&ws)) != MP_OK) return st;
    if (T == 0) return MP_OK;
    // Every (partition, token) triple is written by the partials kernel before the
    // combine reads it, so the array needs no clearing between calls.
    return mp_vocab_ce(X, E, target, loss, ws, sizeof(g_ce_scratch), T, h, v_pad, v_valid, t, d_status, stream);
}
