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

// host.cu: every host-side check of mt_train_update (MT_OK or the status the
// launch would return before enqueueing anything)
int mt_check_update_args(const float* params, const void* shadow, const float* grads, const float* adam_m,
                         const float* adam_v, const int32_t* tokens, const struct mt_hparams* hp,
                         const void* arena, int64_t arena_bytes);
