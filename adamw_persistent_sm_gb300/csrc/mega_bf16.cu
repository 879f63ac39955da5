// mega_bf16.cu - the megakernel instantiated for __nv_bfloat16 operands.
#include "mega.cuh"
#include "launch.h"

cudaError_t mt_prepare_mega_bf16(size_t smem, int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(mt_megakernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mt_opkernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, mt_megakernel<__nv_bfloat16>, MT_THREADS, smem);
}

cudaError_t mt_launch_mega_bf16(const KArgs& a, int grid, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mt_megakernel<__nv_bfloat16>, a);
}

cudaError_t mt_launch_op_bf16(const KArgs& a, int grid, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(MT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mt_opkernel<__nv_bfloat16>, a);
}
