// Kernel launch with programmatic stream serialization (programmatic dependent launch), shared
// by every entry point.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>

namespace mptp {

// MPTP_PDL=0 launches the kernels without programmatic stream serialization.
inline bool pdl_enabled() {
    const char* v = std::getenv("MPTP_PDL");
    return !(v != nullptr && v[0] == '0');
}

// Launch with programmatic stream serialization: the kernel may start while the previous kernel
// in the stream is finishing, and waits for it (grid_dependency_wait) before touching global
// memory. Cluster dimensions come from the kernel's own attribute.
template <typename Kern, typename... Args>
inline cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace mptp
