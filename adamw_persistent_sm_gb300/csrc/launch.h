// launch.h - host launchers of the two megakernel instantiations.
#pragma once
#include <cuda_runtime.h>
#include "plan.h"

cudaError_t mt_launch_mega_f32(const KArgs& a, int grid, size_t smem, cudaStream_t st);
cudaError_t mt_launch_mega_bf16(const KArgs& a, int grid, size_t smem, cudaStream_t st);
cudaError_t mt_prepare_mega_f32(size_t smem, int* blocks_per_sm);
cudaError_t mt_prepare_mega_bf16(size_t smem, int* blocks_per_sm);
// single-op harness kernel (same arguments and shared memory as the update)
cudaError_t mt_launch_op_f32(const KArgs& a, int grid, size_t smem, cudaStream_t st);
cudaError_t mt_launch_op_bf16(const KArgs& a, int grid, size_t smem, cudaStream_t st);
