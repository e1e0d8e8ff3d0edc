// mp_vocab_ce_noalloc: the fused vocab-parallel cross-entropy for callers that
// cannot allocate device memory.
//
// Who needs it: a process whose device memory is owned by someone else's pool
// and that is not allowed to call cudaMalloc/cudaFree itself, for instance a
// serving runtime that reserves all of HBM at start-up and forbids any later
// allocation (cudaMalloc and cudaFree can synchronise the device and stall every
// stream), or a host framework whose memory accounting must see every byte.
// Such a caller cannot hand mp_vocab_ce a workspace of its own, so this entry
// point takes the per-token partition triples from a fixed-size array that the
// library reserves in device memory when it is loaded (every GPU that loads the
// library holds these 4 MiB until the process exits).
//
// The caller still passes X, E, the targets and the loss buffer; nothing here
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
#include <mutex>

#include "mptp_internal.h"

// Scratch for the triples: fp32 [P][3][T], at most MP_CE_NOALLOC_MAX_FLOATS floats.
// In host code this name is only a host-side stand-in; kernels must be given the
// device address obtained below.
static __device__ __align__(256) float g_ce_scratch[MP_CE_NOALLOC_MAX_FLOATS];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_ce_scratch on the current device, looked up once per
// device (the first call on a device does this, with that device current).
mp_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return MP_ERR_NO_DEVICE;
    }
    if (dev < 0 || dev >= kMaxDevices) return MP_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_ce_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MP_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MP_OK;
}

}  // namespace

extern "C" mp_status mp_vocab_ce_noalloc(const mp_bf16* X, const mp_bf16* E, const int32_t* target, float* loss,
                                         int T, int h, int v_pad, int v_valid, int t, uint32_t* d_status,
                                         void* stream) {
    if (T < 0 || h <= 0 || v_pad <= 0 || t < 1 || v_valid < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || v_pad % (128 * t) != 0 || v_valid > v_pad) return MP_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MP_OK;
    // The triples must fit in the static array; larger problems are refused before any launch.
    const size_t need = mp_vocab_ce_workspace_bytes(T, v_pad, t);
    if (need == 0 || need > sizeof(g_ce_scratch)) return MP_ERR_WORKSPACE;
    int sms = 0;
    mp_status st = mptp::check_device(&sms);
    if (st != MP_OK) return st;
    void* ws = nullptr;
    if ((st = scratch_address(&ws)) != MP_OK) return st;
    // Every (partition, token) triple is written by the partials kernel before the
    // combine reads it, so the array needs no clearing between calls.
    return mp_vocab_ce(X, E, target, loss, ws, sizeof(g_ce_scratch), T, h, v_pad, v_valid, t, d_status, stream);
}
