// Launch helper shared by the translation units that own kernels: every
// launch goes through cudaLaunchKernelEx with programmatic stream
// serialisation (so a kernel's prologue overlaps its predecessor's tail) and,
// where asked, a thread-block cluster shape or a cooperative launch (every
// CTA of the grid resident at once: the launch fails rather than run a grid
// whose CTAs wait on each other but cannot all be resident).
#pragma once

#include <utility>

#include <cuda_runtime.h>

#include "../../include/awq_moe.h"

namespace awq {

template <typename Kernel>
inline awq_status set_smem(Kernel k, int bytes)
{
    // Per-function attribute; cheap enough to set on every call and keeps the
    // library free of per-device state.
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess
               ? AWQ_OK
               : AWQ_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
inline awq_status launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem, int cluster_x,
                            bool cooperative, cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return err == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
inline awq_status launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, int smem, int cluster_x,
                         cudaStream_t stream, Args &&...args)
{
    return launch_ex(kernel, grid, block, smem, cluster_x, false, stream, std::forward<Args>(args)...);
}

}  // namespace awq
