// agmm_kernels.cu -- kernel selection and launch for the fused all-gather
// matmul (the fused kernel itself: agmm_fused_kernel.cuh), and the unfused
// path's gather kernel.
#include "kernel_params.h"

namespace agmm {
namespace {

// Copies shard r (blockIdx.y) to rows [r*m_pd, (r+1)*m_pd) of the gathered
// buffer: the decomposed path's all-gather (AllGather-GEMM tutorial, local
// store phase), here a device-local copy.
__global__ void __launch_bounds__(256) agmm_gather_rows(const __grid_constant__ GatherParams g) {
  const int r = blockIdx.y;
  const uint4* __restrict__ src = g.src[r];
  uint4* __restrict__ dst = g.dst + (int64_t)r * g.vec_per_shard;
  const int64_t n = g.vec_per_shard;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 v0 = __ldg(src + i);
    const uint4 v1 = __ldg(src + i + stride);
    const uint4 v2 = __ldg(src + i + 2 * stride);
    const uint4 v3 = __ldg(src + i + 3 * stride);
    dst[i] = v0;
    dst[i + stride] = v1;
    dst[i + 2 * stride] = v2;
    dst[i + 3 * stride] = v3;
  }
  for (; i < n; i += stride) dst[i] = __ldg(src + i);
}

KernelFn select_kernel(const KernelKey& k) {
  if (k.path == kPathSwap) return select_swap_kernel(k);
  return k.atoms == 2 ? select_rows_kernel_a2(k) : select_rows_kernel_a1(k);
}

}  // namespace

cudaError_t prepare_agmm_kernel(const KernelKey& key, size_t smem_bytes, int cluster_x,
                                int* max_active) {
  KernelFn fn = select_kernel(key);
  if (!fn) return cudaErrorInvalidValue;
  // Always the device maximum: plans of different sizes share a kernel, and a
  // later plan must never lower the limit an earlier plan launches with.
  if (smem_bytes > kMaxDynSmem) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxDynSmem);
  if (e != cudaSuccess) return e;
  if (cluster_x > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  if (max_active) {
    if (cluster_x > 1) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)cluster_x, 1, 1);
      cfg.blockDim = dim3(kThreads, 1, 1);
      cfg.dynamicSmemBytes = smem_bytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = (unsigned)cluster_x;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      e = cudaOccupancyMaxActiveClusters(max_active, fn, &cfg);
    } else {
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(max_active, fn, kThreads, smem_bytes);
    }
  }
  return e;
}

cudaError_t launch_agmm_kernel(const KernelKey& key, const KernelParams& p, dim3 grid, int cluster_x,
                               size_t smem_bytes, bool cooperative, cudaStream_t stream) {
  KernelFn fn = select_kernel(key);
  if (!fn) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[3];
  unsigned na = 0;
  if (cluster_x > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster_x;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  } else if (p.pdl) {
    // Programmatic dependent launch: this grid's prologue may overlap the
    // previous kernel's tail; the kernel waits (griddepcontrol.wait) before
    // its first global-memory access.
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

cudaError_t launch_gather_kernel(const GatherParams& g, int P, int blocks_per_shard,
                                 cudaStream_t stream) {
  agmm_gather_rows<<<dim3((unsigned)blocks_per_shard, (unsigned)P, 1), 256, 0, stream>>>(g);
  return cudaGetLastError();
}

}  // namespace agmm
