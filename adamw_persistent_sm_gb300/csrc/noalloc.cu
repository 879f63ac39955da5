// noalloc.cu - mt_train_update_noalloc: the training-update launch with its
// arena in a fixed device array owned by this library, for callers that may
// not allocate device memory themselves.
//
// The array is a file-scope __device__ variable of MT_NOALLOC_ARENA_BYTES.
// The CUDA runtime places it in device memory when this file's module is
// loaded on a device, and it stays there until the process exits.  Host code
// must not pass the array's name to a kernel: on the host that name is only a
// stand-in symbol, not a device address.  The device address is looked up
// with cudaGetSymbolAddress on every call, with the caller's device current,
// so it stays right after a cudaDeviceReset reloads the module.
#include <cuda_runtime.h>
#include <string.h>

#include "../../include/moe_train.h"
#include "launch.h"
#include "plan.h"

static __device__ __align__(256) unsigned char g_noalloc_arena[MT_NOALLOC_ARENA_BYTES];

namespace {

// Device address of the array on the current device.
int noalloc_arena(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_arena);
  if (e != cudaSuccess || !p) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  *out = p;
  return MT_OK;
}

}  // namespace

extern "C" int32_t mt_train_update_noalloc(float* params, void* shadow, float* grads, float* adam_m,
                                           float* adam_v, const int32_t* tokens, const mt_hparams* hp,
                                           mt_outputs* out, void* stream) {
  const int64_t need = mt_arena_bytes(hp);
  if (need < 0) return (int32_t)(-need);
  if (need > (int64_t)MT_NOALLOC_ARENA_BYTES) return MT_ERR_ARENA_SMALL;
  void* arena = nullptr;
  int st = noalloc_arena(&arena);
  if (st) return st;
  // every check of the launch comes before anything is enqueued
  st = mt_check_update_args(params, shadow, grads, adam_m, adam_v, tokens, hp, arena,
                            (int64_t)MT_NOALLOC_ARENA_BYTES);
  if (st) return st;
  // The array keeps whatever the previous call left in it.  The barrier
  // words and the status word must start at zero; the rest of the header
  // (the running loss of the update) is kept for later microbatches.
  if (cudaMemsetAsync(arena, 0, offsetof(ArenaHdr, micro_index), (cudaStream_t)stream) != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_CUDA;
  }
  st = mt_train_update(params, shadow, grads, adam_m, adam_v, tokens, hp, arena, (int64_t)MT_NOALLOC_ARENA_BYTES,
                       stream);
  if (st) return st;
  if (out) return mt_read_outputs(arena, out, stream);
  return MT_OK;
}
