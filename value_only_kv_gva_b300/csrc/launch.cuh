// launch.cuh -- host-side launch helpers shared by the kernel launchers.
#pragma once

#include <cstring>

#include <cuda_runtime.h>

namespace gva {

// cudaError_t of the calling host thread's last failed CUDA call (gva_last_cuda_error).
inline thread_local int g_last_cuda_error = 0;

// Programmatic dependent launch is requested only where it has a kernel to follow:
// always for eager launches, and during stream capture only when every node the
// launch will depend on is a kernel node.
inline bool pdl_allowed(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    const cudaGraphNode_t *deps = nullptr;
    size_t n = 0;
    if (cudaStreamGetCaptureInfo(s, &st, nullptr, nullptr, &deps, nullptr, &n) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (st != cudaStreamCaptureStatusActive) return true;
    if (n == 0 || deps == nullptr) return false;
    for (size_t i = 0; i < n; ++i) {
        cudaGraphNodeType t;
        if (cudaGraphNodeGetType(deps[i], &t) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        if (t != cudaGraphNodeTypeKernel) return false;
    }
    return true;
}

template <typename Kern, typename... Params>
cudaError_t launch(Kern kernel, dim3 grid, dim3 block, size_t smem, void *stream,
                   const Params &...params) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_allowed(cfg.stream) ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, params...);
}

inline int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) g_last_cuda_error = (int)e;
    return e == cudaSuccess ? GVA_OK : GVA_ERR_CUDA;
}

}  // namespace gva
