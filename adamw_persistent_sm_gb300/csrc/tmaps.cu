// tmaps.cu - TMA tensor maps of the bf16 operands of the tensor-core
// products.  Every map describes one whole 2-D buffer (layers and experts
// stacked along the outer dimension) with a 64 x 64 box and the 128-byte
// swizzle that the tcgen05 shared-memory descriptors expect.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "../../include/moe_train.h"
#include "tmaps.h"

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;

void resolve() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
          cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
}

// rows x cols bf16 matrix at base (row stride = cols elements)
bool encode(CUtensorMap* m, const void* base, long long rows, long long cols) {
  if (!g_encode || !base || rows <= 0 || cols <= 0) return false;
  if (((uintptr_t)base & 15) || ((cols * 2) & 15)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

int mt_build_tensor_maps(KArgs* a, void* shadow) {
  std::call_once(g_once, resolve);
  if (!g_encode) return MT_ERR_CUDA;
  const MtDims& D = a->D;
  const long long L = D.L, T = D.T, d = D.d, hq = D.hq, E = D.E, F = D.F, V = D.V, Pm = D.Pmax;
  char* ar = a->arena;
  const char* w = (const char*)shadow;
  auto P = [&](int pid) { return (const void*)(w + a->poff[pid] * 2); };
  auto A = [&](int id) { return (const void*)(ar + a->aoff[id]); };
  bool ok = true;
  ok &= encode(&a->maps[MAP_R], A(A_R), L * T, d);
  ok &= encode(&a->maps[MAP_WQKV], P(P_WQKV), L * 3 * hq, d);
  ok &= encode(&a->maps[MAP_O], A(A_O), L * T, hq);
  ok &= encode(&a->maps[MAP_WO], P(P_WO), L * d, hq);
  ok &= encode(&a->maps[MAP_XS], A(A_XS), L * Pm, d);
  ok &= encode(&a->maps[MAP_WGATE], P(P_WGATE), L * E * F, d);
  ok &= encode(&a->maps[MAP_WUP], P(P_WUP), L * E * F, d);
  ok &= encode(&a->maps[MAP_ACT], A(A_ACT), L * Pm, F);
  ok &= encode(&a->maps[MAP_WDOWN], P(P_WDOWN), L * E * d, F);
  ok &= encode(&a->maps[MAP_RF], A(A_RF), T, d);
  ok &= encode(&a->maps[MAP_WLM], P(P_LM_HEAD), V, d);
  ok &= encode(&a->maps[MAP_DLOGITS], A(A_DLOGITS), T, V);
  ok &= encode(&a->maps[MAP_DY], A(A_DY), Pm, d);
  ok &= encode(&a->maps[MAP_DGU], A(A_DGU), Pm, 2 * F);
  ok &= encode(&a->maps[MAP_DXO], A(A_DXO), T, d);
  ok &= encode(&a->maps[MAP_DQKV], A(A_DQKV), T, 3 * hq);
  ok &= encode(&a->maps[MAP_QKV], A(A_QKV), L * T, 3 * hq);
  ok &= encode(&a->maps[MAP_DOUT], A(A_DO), T, hq);
  return ok ? MT_OK : MT_ERR_ARG;
}

int mt_build_debug_maps(KArgs* a, const void* A, long long a_rows, long long a_cols, const void* B,
                        long long b_rows, long long b_cols) {
  std::call_once(g_once, resolve);
  if (!g_encode) return MT_ERR_CUDA;
  bool ok = encode(&a->maps[MAP_R], A, a_rows, a_cols);
  ok &= encode(&a->maps[MAP_WQKV], B, b_rows, b_cols);
  return ok ? MT_OK : MT_ERR_ARG;
}
