// tmaps.cu - TMA tensor maps of the tensor-core products.  Every map
// describes one whole 2-D buffer (layers and experts stacked along the outer
// dimension).  Operand maps (bf16) have a 64 x 64 box and the 128-byte
// swizzle that the tcgen05 shared-memory descriptors expect; epilogue maps
// have a 32 x 32 box whose rows are swizzled over their own width (64 bytes
// for bf16, 128 for fp32), the layout the epilogue warps stage in shared
// memory for bulk stores and aux loads.
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

// rows x cols matrix at base (row stride = cols elements), box bc x br
bool encode_box(CUtensorMap* m, const void* base, long long rows, long long cols, bool f32, unsigned bc,
                unsigned br, CUtensorMapSwizzle sw) {
  const long long es = f32 ? 4 : 2;
  if (!g_encode || !base || rows <= 0 || cols <= 0) return false;
  if (((uintptr_t)base & 15) || ((cols * es) & 15)) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(cols * es)};
  cuuint32_t box[2] = {bc, br};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
// product operands: bf16, 64 x 64 boxes, 128-byte swizzle
bool encode(CUtensorMap* m, const void* base, long long rows, long long cols) {
  return encode_box(m, base, rows, cols, false, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}
// epilogue boxes: 32 rows x 32 columns (64 bytes per bf16 row, 128 per fp32 row)
bool encode_epi(CUtensorMap* m, const void* base, long long rows, long long cols, bool f32) {
  return encode_box(m, base, rows, cols, f32, 32, 32, f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

}  // namespace

int mt_build_tensor_maps(KArgs* a, void* shadow) {
  std::call_once(g_once, resolve);
  if (!g_encode) return MT_ERR_CUDA;
  const MtDims& D = a->D;
  const long long L = D.L, T = D.T, d = D.d, hq = D.hq, E = D.E, F = D.F, V = D.V, Pm = D.Pmax;
  const long long AL = a->act_layers;       // layers of expert activations the arena keeps
  const long long U = D.U;                  // weight slots of the per-layer tensors
  char* ar = a->arena;
  const char* w = (const char*)shadow;
  auto P = [&](int pid) { return (const void*)(w + a->poff[pid] * 2); };
  auto A = [&](int id) { return (const void*)(ar + a->aoff[id]); };
  bool ok = true;
  ok &= encode(&a->maps[MAP_R], A(A_R), L * T, d);
  ok &= encode(&a->maps[MAP_WQKV], P(P_WQKV), U * 3 * hq, d);
  ok &= encode(&a->maps[MAP_O], A(A_O), L * T, hq);
  ok &= encode(&a->maps[MAP_WO], P(P_WO), U * d, hq);
  ok &= encode(&a->maps[MAP_XS], A(A_XS), L * Pm, d);
  ok &= encode(&a->maps[MAP_WGATE], P(P_WGATE), U * E * F, d);
  ok &= encode(&a->maps[MAP_WUP], P(P_WUP), U * E * F, d);
  ok &= encode(&a->maps[MAP_ACT], A(A_ACT), AL * Pm, F);
  ok &= encode(&a->maps[MAP_WDOWN], P(P_WDOWN), U * E * d, F);
  ok &= encode(&a->maps[MAP_RF], A(A_RF), T, d);
  ok &= encode(&a->maps[MAP_WLM], P(P_LM_HEAD), V, d);
  ok &= encode(&a->maps[MAP_DLOGITS], A(A_DLOGITS), T, V);
  ok &= encode(&a->maps[MAP_DY], A(A_DY), Pm, d);
  ok &= encode(&a->maps[MAP_DGU], A(A_DGU), Pm, 2 * F);
  ok &= encode(&a->maps[MAP_DXO], A(A_DXO), T, d);
  ok &= encode(&a->maps[MAP_DQKV], A(A_DQKV), T, 3 * hq);
  ok &= encode(&a->maps[MAP_QKV], A(A_QKV), L * T, 3 * hq);
  ok &= encode(&a->maps[MAP_DOUT], A(A_DO), T, hq);
  ok &= encode(&a->maps[MAP_DZB], A(A_DZB), T, 64);
  ok &= encode(&a->maps[MAP_R2], A(A_R2), L * T, d);
  ok &= encode_epi(&a->maps[MAP_E_QKV], A(A_QKV), L * T, 3 * hq, false);
  ok &= encode_epi(&a->maps[MAP_E_GU], A(A_GU), AL * Pm, 2 * F, false);
  ok &= encode_epi(&a->maps[MAP_E_ACT], A(A_ACT), AL * Pm, F, false);
  ok &= encode_epi(&a->maps[MAP_E_DGU], A(A_DGU), Pm, 2 * F, false);
  ok &= encode_box(&a->maps[MAP_E_DLOGITS], A(A_DLOGITS), T, V, false, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= encode_box(&a->maps[MAP_E_QKV64], A(A_QKV), L * T, 3 * hq, false, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= encode_epi(&a->maps[MAP_E_DO], A(A_DO), T, hq, false);
  ok &= encode_epi(&a->maps[MAP_E_O], A(A_O), L * T, hq, false);
  ok &= encode_epi(&a->maps[MAP_E_Y], A(A_Y), L * Pm, d, true);
  ok &= encode_epi(&a->maps[MAP_E_DRF], A(A_DRF), T, d, true);
  ok &= encode_epi(&a->maps[MAP_E_DXS], A(A_DXS), Pm, d, true);
  ok &= encode_epi(&a->maps[MAP_E_DR], A(A_DR), T, d, true);
  ok &= encode_epi(&a->maps[MAP_E_XM], A(A_XM), L * T, d, true);
  ok &= encode_epi(&a->maps[MAP_E_X], A(A_X), (L + 1) * T, d, true);
  ok &= encode_box(&a->maps[MAP_E_DQKV], A(A_DQKV), T, 3 * hq, false, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= encode_box(&a->maps[MAP_E_OROW], A(A_O), L * T, hq, false, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (a->use_dsg) {
    const long long rows = (long long)D.B * D.H * D.S;
    ok &= encode_box(&a->maps[MAP_E_DS], A(A_DSG), rows, D.S, false, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B);
    ok &= encode_box(&a->maps[MAP_E_DSL], A(A_DSG), rows, D.S, false, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  return ok ? MT_OK : MT_ERR_ARG;
}

int mt_build_debug_maps(KArgs* a, const void* A, long long a_rows, long long a_cols, const void* B,
                        long long b_rows, long long b_cols, const void* C, long long c_rows, long long c_cols,
                        bool c_f32, int a_rpb, int b_rpb) {
  std::call_once(g_once, resolve);
  if (!g_encode) return MT_ERR_CUDA;
  bool ok = encode_box(&a->maps[MAP_R], A, a_rows, a_cols, false, 64, (unsigned)a_rpb, CU_TENSOR_MAP_SWIZZLE_128B);
  ok &= encode_box(&a->maps[MAP_WQKV], B, b_rows, b_cols, false, 64, (unsigned)b_rpb, CU_TENSOR_MAP_SWIZZLE_128B);
  if (C) ok &= encode_epi(&a->maps[c_f32 ? MAP_E_Y : MAP_E_QKV], C, c_rows, c_cols, c_f32);
  return ok ? MT_OK : MT_ERR_ARG;
}
