// Entry point of the vocab-parallel input embedding: mp_vocab_embed.
//
// "Megatron-LM: Training Multi-Billion Parameter Language Models Using Model
// Parallelism", section 3.4, "Input Embedding Parallelism": E [v_pad, h] is split
// along the vocabulary into t row blocks; shard i looks up the ids inside its range
// and yields zeros elsewhere; the g all-reduce sums the shards. Each valid id is owned
// by exactly one shard, so the sum is that shard's row, bit for bit: the kernel finds
// the owner from the id and copies its row once (16-byte vectors, one warp per token),
// which is the HBM-bound minimum (read T rows of E, write T rows).
#include <cuda_bf16.h>

#include "mptp_internal.h"
#include "mptp_launch.cuh"
#include "mptp_ptx.cuh"

namespace mptp {

__global__ void __launch_bounds__(256) vocab_embed_kernel(const int32_t* __restrict__ ids,
                                                          const uint4* __restrict__ E, uint4* __restrict__ out,
                                                          int T, int hv, int vs, int t, int v_valid,
                                                          uint32_t* status) {
    grid_dependency_wait();  // the kernels that wrote the ids (or E) before it
    grid_launch_dependents();
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < T; r += warps) {
        const int id = __ldg(ids + r);
        // Owner shard of the id (none for ids outside [0, v_valid)).
        const int shard = (id >= 0 && id < v_valid) ? id / vs : -1;
        uint4* dst = out + static_cast<long long>(r) * hv;
        if (shard < 0 || shard >= t) {
            for (int i = lane; i < hv; i += 32) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            if (lane == 0 && status) atomicOr(status, 0x2u);
            continue;
        }
        const uint4* src = E + (static_cast<long long>(shard) * vs + (id - shard * vs)) * hv;
        // 8 vectors per lane in flight before any store (h up to 2048 per pass).
        for (int base = 0; base < hv; base += 8 * 32) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * 32 + lane;
                if (i < hv) v[j] = __ldg(src + i);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * 32 + lane;
                if (i < hv) __stcs(dst + i, v[j]);
            }
        }
    }
}

}  // namespace mptp

using namespace mptp;

extern "C" mp_status mp_vocab_embed(const int32_t* ids, const mp_bf16* E, mp_bf16* out, int T, int h, int v_pad,
                                    int v_valid, int t, uint32_t* d_status, void* stream) {
    if (T < 0 || h <= 0 || v_pad <= 0 || t < 1 || v_valid < 1) return MP_ERR_INVALID_ARG;
    if (h % 64 != 0 || v_pad % (128 * t) != 0 || v_valid > v_pad) return MP_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return MP_OK;
    if (!ids || !E || !out) return MP_ERR_INVALID_ARG;
    if (!aligned16(ids) || !aligned16(E) || !aligned16(out) ||
        (d_status && (reinterpret_cast<uintptr_t>(d_status) & 3u)))
        return MP_ERR_MISALIGNED;
    int sms = 0;
    mp_status st = check_device(&sms);
    if (st != MP_OK) return st;
    const int blocks_needed = ceil_div(T, 8);
    const int grid = blocks_needed < sms * 8 ? blocks_needed : sms * 8;
    const cudaError_t e = launch_pdl(vocab_embed_kernel, dim3(grid), dim3(256), 0, static_cast<cudaStream_t>(stream), ids,
                                     reinterpret_cast<const uint4*>(E), reinterpret_cast<uint4*>(out), T, h / 8,
                                     v_pad / t, t, v_valid, d_status);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? MP_OK : MP_ERR_CUDA;
}
