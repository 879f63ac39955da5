// noalloc.cu - mt_train_update_noalloc: the training-update launch with its
// arena in a fixed device array owned by this library, for callers that may
// not allocate device memory themselves.
//
// The array is a file-scope __device__ variable of MT_NOALLOC_ARENA_BYTES.
// The CUDA runtime places it in device memory when this file's module is
// loaded on a device, and it stays there until the process exits.  Host code
// must not pass the array's name to a kernel: on the host that name is only a
// stand-in symbol, not a device address.  The device address is looked up
// once per device with cudaGetSymbolAddress (with that device current) and
// cached.
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "../../include/moe_train.h"
#include "plan.h"

static __device__ __align__(256) unsigned char g_noalloc_arena[MT_NOALLOC_ARENA_BYTES];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the array on the current device (looked up once per device).
int noalloc_arena(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MT_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_arena);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return MT_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
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
