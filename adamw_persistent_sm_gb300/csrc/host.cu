// host.cu - the C ABI (include/moe_train.h): argument checks, the parameter
// layout, the arena plan, tensor maps and the cooperative launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "../../include/moe_train.h"
#include "launch.h"
#include "plan.h"
#include "tmaps.h"
#include "gemm_tc.cuh"

static_assert(sizeof(mt_hparams) == 128, "mt_hparams layout is part of the ABI");
static_assert(sizeof(mt_outputs) == 40 + 4 * MT_MAX_LAYERS * MT_MAX_EXPERTS + 12, "mt_outputs layout");

namespace {

constexpr long long kAlign = 1024;
constexpr int kNch = MT_MAX_CTAS;

long long round_up(long long x, long long a) { return (x + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Dimension and hyperparameter checks shared by every entry point.
int check_hparams(const mt_hparams* hp) {
  if (!hp) return MT_ERR_ARG;
  if (hp->vocab <= 0 || hp->d_model <= 0 || hp->n_layers <= 0 || hp->n_heads <= 0 ||
      hp->head_dim <= 0 || hp->n_experts <= 0 || hp->top_k <= 0 || hp->d_ff <= 0 ||
      hp->batch <= 0 || hp->seq <= 0)
    return MT_ERR_ARG;
  if (hp->precision != MT_PREC_FP32 && hp->precision != MT_PREC_BF16) return MT_ERR_ARG;
  if (hp->flags & ~(uint32_t)MT_FLAGS_ALL) return MT_ERR_ARG;
  if (hp->micro_count <= 0 || hp->micro_index < 0 || hp->micro_index >= hp->micro_count) return MT_ERR_ARG;
  if (hp->step < 1) return MT_ERR_ARG;
  if ((hp->flags & MT_FLAG_SELECTIVE_EXPERTS) && hp->expert_step < 1) return MT_ERR_ARG;
  if (hp->n_unique_layers < 0 || hp->n_unique_layers > hp->n_layers || hp->reserved0 != 0) return MT_ERR_ARG;
  if (!(hp->lr >= 0.f) || !(hp->beta1 >= 0.f && hp->beta1 < 1.f) || !(hp->beta2 >= 0.f && hp->beta2 < 1.f) ||
      !(hp->eps > 0.f) || !(hp->weight_decay >= 0.f) || !(hp->clip_norm > 0.f) || !(hp->clip_eps >= 0.f) ||
      !(hp->norm_eps > 0.f) || !(hp->rope_theta > 0.f) || !(hp->loss_coef >= 0.f) || hp->wait_timeout_ns < 0)
    return MT_ERR_ARG;
  // shapes the kernels implement
  if (hp->n_layers > MT_MAX_LAYERS || hp->n_experts > MT_MAX_EXPERTS || hp->top_k > 8 ||
      hp->top_k > hp->n_experts)
    return MT_ERR_UNSUPPORTED;
  if (hp->head_dim != 16 && hp->head_dim != 64) return MT_ERR_UNSUPPORTED;
  if (hp->d_model % 32 != 0 || hp->d_model > 768) return MT_ERR_UNSUPPORTED;
  if (hp->d_ff % 64 != 0) return MT_ERR_UNSUPPORTED;
  if (hp->seq < 2) return MT_ERR_UNSUPPORTED;
  if (hp->vocab % 8 != 0) return MT_ERR_UNSUPPORTED;
  if ((long long)hp->n_experts * hp->d_model * 4 > 160 * 1024) return MT_ERR_UNSUPPORTED;  // router staged in smem
  const long long T = (long long)hp->batch * hp->seq;
  if (T * hp->top_k + (long long)hp->n_experts * MT_TILE_M > (1LL << 30)) return MT_ERR_UNSUPPORTED;
  if ((long long)hp->vocab * T > (1LL << 40)) return MT_ERR_UNSUPPORTED;
  return MT_OK;
}

// The bf16 model runs only on the tensor-core path: 128-row tiles over tokens
// and expert rows, 256-column tiles over features, 128-query / 128-key
// attention blocks of head_dim 64.  Other bf16 shapes are refused.
bool tc_shapes_ok(const mt_hparams* hp) {
  const long long T = (long long)hp->batch * hp->seq;
  const int hq = hp->n_heads * hp->head_dim;
  return T % 128 == 0 && hp->d_model % 256 == 0 && hq % 256 == 0 && hp->vocab % 256 == 0 &&
         hp->d_ff % 256 == 0 && hp->head_dim == 64 && hp->seq % 128 == 0;
}

void make_plan(const mt_hparams* hp, MtPlan* P) {
  MtDims& D = P->D;
  D.V = hp->vocab; D.d = hp->d_model; D.L = hp->n_layers; D.H = hp->n_heads; D.hd = hp->head_dim;
  D.hq = D.H * D.hd; D.E = hp->n_experts; D.K = hp->top_k; D.F = hp->d_ff; D.B = hp->batch;
  D.S = hp->seq; D.T = D.B * D.S;
  D.U = hp->n_unique_layers > 0 ? hp->n_unique_layers : hp->n_layers;
  D.Pmax = (int)round_up((long long)D.T * D.K + (long long)D.E * (MT_TILE_M - 1), MT_TILE_M);
  D.nch = kNch;
  D.op_bytes = hp->precision == MT_PREC_BF16 ? 2 : 4;
  const long long T = D.T, d = D.d, L = D.L, ob = D.op_bytes, Pm = D.Pmax;
  long long sz[A_COUNT];
  sz[A_HDR] = sizeof(ArenaHdr);
  sz[A_ROPE] = (long long)D.S * (D.hd / 2) * 2 * 4;
  sz[A_X] = (L + 1) * T * d * 4;
  sz[A_XM] = L * T * d * 4;
  sz[A_INV1] = L * T * 4;
  sz[A_INV2] = L * T * 4;
  sz[A_R] = L * T * d * ob;
  sz[A_QKV] = L * T * 3 * D.hq * ob;
  sz[A_O] = L * T * D.hq * ob;
  sz[A_LSE] = L * D.B * D.H * (long long)D.S * 4;
  sz[A_R2] = L * T * d * ob;
  sz[A_Z] = L * T * D.E * 4;
  sz[A_IDX] = L * T * D.K * 4;
  sz[A_WGT] = L * T * D.K * 4;
  sz[A_CNT] = L * (long long)D.nch * D.E * 4;
  sz[A_OFFS] = L * (D.E + 1) * 4;
  sz[A_PERM] = L * Pm * 4;
  sz[A_INVM] = L * T * D.K * 4;
  sz[A_XS] = L * Pm * d * ob;
  // memory rule MT_FLAG_RECOMPUTE_EXPERT_ACT: one layer of expert activations
  const long long AL = (hp->flags & MT_FLAG_RECOMPUTE_EXPERT_ACT) ? 1 : L;
  sz[A_GU] = AL * Pm * 2 * D.F * ob;
  sz[A_ACT] = AL * Pm * D.F * ob;
  sz[A_Y] = L * Pm * d * 4;
  sz[A_RF] = T * d * ob;
  sz[A_INVF] = T * 4;
  sz[A_CEPART] = T * ((D.V + 127) / 128) * 2 * 4;
  sz[A_CETGT] = T * 4;
  sz[A_DLOGITS] = T * D.V * ob;
  sz[A_TOKLOSS] = T * 4;
  sz[A_DX] = T * d * 4;
  sz[A_DXO] = T * d * ob;
  sz[A_DY] = Pm * d * ob;
  sz[A_DZ] = T * D.E * 4;
  sz[A_DZB] = T * 64 * 2;
  sz[A_DGU] = Pm * 2 * D.F * ob;
  sz[A_DXS] = Pm * d * 4;
  sz[A_DR2] = T * d * 4;
  sz[A_DO] = T * D.hq * ob;
  sz[A_DSUM] = T * D.H * 4;
  sz[A_DQKV] = T * 3 * D.hq * ob;
  // dS^T of one layer for the dQ product of the tcgen05 attention backward
  // (memory rule MT_FLAG_RECOMPUTE_ATTN_DS: not kept, dQ recomputes it)
  const bool keep_ds = hp->precision == MT_PREC_BF16 && !(hp->flags & MT_FLAG_RECOMPUTE_ATTN_DS);
  sz[A_DSG] = keep_ds ? (long long)D.B * D.H * D.S * D.S * 2 : 0;
  sz[A_DR] = T * d * 4;
  sz[A_DRF] = T * d * 4;
  sz[A_PART] = (long long)D.nch * (D.E + 2) * d * 4;
  sz[A_KPART] = 8LL * 3 * D.hq * d * 4;
  sz[A_NORMPART] = (long long)MT_OPT_RANGES * D.nch * 8;
  sz[A_DEP] = dep_words(D) * 4;
  // the per-CTA trace exists only in arenas sized for traced launches
  sz[A_TRACE] = (hp->flags & MT_FLAG_TRACE) ? (long long)D.nch * MT_TRACE_WORDS * 8 : 0;
  long long off = 0;
  for (int i = 0; i < A_COUNT; ++i) {
    P->aoff[i] = off;
    P->abytes[i] = sz[i];
    off = round_up(off + sz[i], kAlign);
  }
  P->arena_bytes = off;
  // parameters: per-layer tensors are stacked over the U weight slots
  const long long V = D.V, E = D.E, F = D.F, hq = D.hq, U = D.U;
  long long pn[P_COUNT];
  pn[P_EMB] = V * d;
  pn[P_ATTN_NORM] = U * d;
  pn[P_WQKV] = U * 3 * hq * d;
  pn[P_WO] = U * d * hq;
  pn[P_MOE_NORM] = U * d;
  pn[P_ROUTER] = U * E * d;
  pn[P_WGATE] = U * E * F * d;
  pn[P_WUP] = U * E * F * d;
  pn[P_WDOWN] = U * E * d * F;
  pn[P_FINAL_NORM] = d;
  pn[P_LM_HEAD] = V * d;
  long long po = 0;
  for (int i = 0; i < P_COUNT; ++i) {
    P->poff[i] = po;
    P->pnumel[i] = pn[i];
    po = round_up(po + pn[i], 64);
  }
  P->n_params = po;
}

const char* kParamNames[P_COUNT] = {"emb",     "attn_norm", "wqkv",   "wo",         "moe_norm", "router",
                                    "w_gate",  "w_up",      "w_down", "final_norm", "lm_head"};

struct DevState {
  size_t smem_f32 = 0, smem_bf16 = 0;   // dynamic shared memory the kernel was prepared for
  int sms = 0;
  int bps_f32 = 0, bps_bf16 = 0;
};
std::mutex g_mu;
DevState g_dev[64];

size_t smem_bytes(const MtDims& D, bool tc) {
  size_t attn = (size_t)(4 * 64 * 65 + 2 * 64 * 65 + 128) * 4;
  size_t simt = (size_t)SG_BM * SG_CPAD * 4;
  size_t router = 1024 + (size_t)D.E * D.d * 4 + 64 * 4;   // ring barriers, router weights, counts
  // column reductions: staged 1/rms and router gradients, token-lane partials
  const int er = D.E <= 4 ? 4 : D.E <= 16 ? 16 : D.E <= 32 ? 32 : 64;
  const int cw = D.E <= 16 ? 4 : D.E <= 32 ? 2 : 1;
  size_t col = 1024 + (size_t)(256 + 256 * D.E + 3 * (er + 1) * 64 * cw) * 4;
  size_t embed = (size_t)(2 * 4096 + 8) * 4;                // embedding backward: match list
  size_t need = attn > simt ? attn : simt;
  if (router > need) need = router;
  if (embed > need) need = embed;
  if (col > need) need = col;
  if (tc && MT_TC_SMEM > need) need = MT_TC_SMEM;
  return need;
}


// Set the kernel's shared-memory limit (once per size and device) and return
// the cooperative grid: one CTA per SM.
int prepare_launch(bool bf16, size_t smem, int* grid) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MT_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DevState& ds = g_dev[dev];
  if (!ds.sms) {
    if (cudaDeviceGetAttribute(&ds.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MT_ERR_CUDA;
  }
  int* bps = bf16 ? &ds.bps_bf16 : &ds.bps_f32;
  size_t& prepared = bf16 ? ds.smem_bf16 : ds.smem_f32;
  if (prepared != smem) {
    cudaError_t e = bf16 ? mt_prepare_mega_bf16(smem, bps) : mt_prepare_mega_f32(smem, bps);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return MT_ERR_LAUNCH;
    }
    prepared = smem;
  }
  if (*bps < 1) return MT_ERR_LAUNCH;
  *grid = ds.sms < kNch ? ds.sms : kNch;
  return MT_OK;
}

int launch_update(int op, int layer, float* params, void* shadow, float* grads, float* adam_m, float* adam_v,
                  const int32_t* tokens, const mt_hparams* hp, void* arena, int64_t arena_bytes, void* stream);

}  // namespace

// Every host-side check of a training-update launch, in the order the launch
// makes them; nothing is enqueued.
int mt_check_update_args(const float* params, const void* shadow, const float* grads, const float* adam_m,
                         const float* adam_v, const int32_t* tokens, const mt_hparams* hp, const void* arena,
                         int64_t arena_bytes) {
  int st = check_hparams(hp);
  if (st) return st;
  const bool bf16 = hp->precision == MT_PREC_BF16;
  if (!params || !grads || !adam_m || !adam_v || !tokens || !arena) return MT_ERR_ARG;
  if (bf16 && !shadow) return MT_ERR_ARG;
  if (!aligned(params, 256) || !aligned(grads, 256) || !aligned(adam_m, 256) || !aligned(adam_v, 256) ||
      !aligned(arena, 256) || !aligned(tokens, 16) || (shadow && !aligned(shadow, 256)))
    return MT_ERR_ARG;
  MtPlan P;
  make_plan(hp, &P);
  if (arena_bytes < P.arena_bytes) return MT_ERR_ARENA_SMALL;
  if (bf16 && !tc_shapes_ok(hp)) return MT_ERR_UNSUPPORTED;
  return MT_OK;
}

extern "C" {

int64_t mt_param_count(const mt_hparams* hp) {
  int st = check_hparams(hp);
  if (st) return -st;
  MtPlan P;
  make_plan(hp, &P);
  return P.n_params;
}

int32_t mt_param_layout(const mt_hparams* hp, mt_tensor_desc* out, int32_t cap) {
  int st = check_hparams(hp);
  if (st) return -st;
  if (cap > 0 && !out) return -MT_ERR_ARG;
  MtPlan P;
  make_plan(hp, &P);
  const long long L = P.D.U, d = hp->d_model, E = hp->n_experts, F = hp->d_ff, V = hp->vocab;
  const long long hq = (long long)hp->n_heads * hp->head_dim;
  // per-layer tensors have one slot per distinct layer (U = n_layers unless looped)
  const long long shapes[P_COUNT][4] = {{V, d}, {L, d}, {L, 3 * hq, d}, {L, d, hq}, {L, d}, {L, E, d},
                                        {L, E, F, d}, {L, E, F, d}, {L, E, d, F}, {d}, {V, d}};
  const int ndims[P_COUNT] = {2, 2, 3, 3, 2, 3, 4, 4, 4, 1, 2};
  for (int i = 0; i < P_COUNT && i < cap; ++i) {
    mt_tensor_desc& t = out[i];
    memset(&t, 0, sizeof(t));
    strncpy(t.name, kParamNames[i], sizeof(t.name) - 1);
    t.offset = P.poff[i];
    t.numel = P.pnumel[i];
    t.ndim = ndims[i];
    for (int k = 0; k < ndims[i]; ++k) t.shape[k] = shapes[i][k];
    t.weight_decay = 1;
  }
  return P_COUNT;
}

int64_t mt_arena_bytes(const mt_hparams* hp) {
  int st = check_hparams(hp);
  if (st) return -st;
  MtPlan P;
  make_plan(hp, &P);
  return P.arena_bytes;
}

int32_t mt_arena_init(void* arena, int64_t arena_bytes, void* stream) {
  if (!arena || !aligned(arena, 256) || arena_bytes < (int64_t)sizeof(ArenaHdr)) return MT_ERR_ARG;
  cudaError_t e = cudaMemsetAsync(arena, 0, sizeof(ArenaHdr), (cudaStream_t)stream);
  return e == cudaSuccess ? MT_OK : MT_ERR_CUDA;
}

int32_t mt_train_update(float* params, void* shadow, float* grads, float* adam_m, float* adam_v,
                        const int32_t* tokens, const mt_hparams* hp, void* arena, int64_t arena_bytes,
                        void* stream) {
  return launch_update(0, 0, params, shadow, grads, adam_m, adam_v, tokens, hp, arena, arena_bytes, stream);
}

int32_t mt_debug_run(int32_t op, int32_t layer, float* params, void* shadow, float* grads, float* adam_m,
                     float* adam_v, const int32_t* tokens, const mt_hparams* hp, void* arena,
                     int64_t arena_bytes, void* stream) {
  if (op < MT_OP_ATTN_FWD || op > MT_OP_CLIP_ADAMW) return MT_ERR_ARG;
  int st = check_hparams(hp);
  if (st) return st;
  if (layer < 0 || layer >= hp->n_layers) return MT_ERR_ARG;
  return launch_update(op, layer, params, shadow, grads, adam_m, adam_v, tokens, hp, arena, arena_bytes, stream);
}

}  // extern "C"

namespace {
// One launch of the update (op == 0) or of one op of the single-op harness.
int launch_update(int op, int layer, float* params, void* shadow, float* grads, float* adam_m, float* adam_v,
                  const int32_t* tokens, const mt_hparams* hp, void* arena, int64_t arena_bytes, void* stream) {
  int st = mt_check_update_args(params, shadow, grads, adam_m, adam_v, tokens, hp, arena, arena_bytes);
  if (st) return st;
  const bool bf16 = hp->precision == MT_PREC_BF16;
  MtPlan P;
  make_plan(hp, &P);
  const bool want_tc = bf16;

  int grid = 0;
  st = prepare_launch(bf16, smem_bytes(P.D, want_tc), &grid);
  if (st) return st;
  const size_t smem = smem_bytes(P.D, want_tc);

  KArgs* a = new KArgs();
  memset(a, 0, sizeof(KArgs));
  a->D = P.D;
  a->lr = hp->lr; a->beta1 = hp->beta1; a->beta2 = hp->beta2; a->eps = hp->eps; a->wd = hp->weight_decay;
  a->clip = hp->clip_norm; a->clip_eps = hp->clip_eps; a->norm_eps = hp->norm_eps;
  a->rope_theta = hp->rope_theta;
  const bool selective = (hp->flags & MT_FLAG_SELECTIVE_EXPERTS) != 0;
  // every target of an update weighs 1 / (its targets); under selective
  // updates each microbatch is an update of the shared tensors
  const double ntargets = (double)hp->batch * (hp->seq - 1) * (selective ? 1 : hp->micro_count);
  a->coef = hp->loss_coef > 0.f ? hp->loss_coef : (float)(1.0 / ntargets);
  a->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
  a->micro_index = hp->micro_index;
  a->micro_count = hp->micro_count;
  const bool last = hp->micro_index == hp->micro_count - 1;
  const bool opt = !(hp->flags & MT_FLAG_NO_OPTIMIZER);
  a->run_opt = opt && (last || selective);
  auto group = [&](int gi, long long step, float gscale, int r0, int nr) {
    OptGroup& g = a->ogrp[gi];
    g.ibc1 = (float)(1.0 / (1.0 - pow((double)hp->beta1, (double)step)));
    g.ibc2 = (float)(1.0 / (1.0 - pow((double)hp->beta2, (double)step)));
    g.gscale = gscale;
    g.r0 = r0;
    g.nr = nr;
  };
  auto range = [&](int ri, long long off, long long n, int gi, int first) {
    a->orng[ri] = OptRange{off, n, gi, first};
  };
  const unsigned all = (1u << P_COUNT) - 1u;
  const unsigned experts = (1u << P_WGATE) | (1u << P_WUP) | (1u << P_WDOWN);
  if (!selective) {
    // one clipped AdamW step over every tensor after the last microbatch
    a->acc_mask = hp->micro_index > 0 ? all : 0u;
    a->n_ranges = 0;
    if (a->run_opt) {
      range(0, 0, P.n_params, 0, 1);
      group(0, hp->step, 1.0f, 0, 1);
      a->n_ranges = 1;
    }
  } else {
    // shared tensors (all but the expert products): a step after every
    // microbatch; expert tensors: gradients summed over micro_count
    // microbatches, a step on their mean after the last
    a->acc_mask = hp->micro_index > 0 ? experts : 0u;
    a->n_ranges = 0;
    if (opt) {
      const long long e0 = P.poff[P_WGATE], e1 = P.poff[P_FINAL_NORM];
      range(0, 0, e0, 0, 1);
      range(1, e1, P.n_params - e1, 0, 0);
      group(0, hp->step, 1.0f, 0, 2);
      a->n_ranges = 2;
      if (last) {
        range(2, e0, e1 - e0, 1, 1);
        group(1, hp->expert_step, 1.0f / (float)hp->micro_count, 2, 1);
        a->n_ranges = 3;
      }
    }
  }
  a->flags = hp->flags;
  a->timeout_ns = hp->wait_timeout_ns > 0 ? hp->wait_timeout_ns : 4000000000LL;
  a->n_params = P.n_params;
  a->master = params; a->shadow = shadow; a->grads = grads; a->adam_m = adam_m; a->adam_v = adam_v;
  a->tokens = tokens;
  a->arena = (char*)arena;
  memcpy(a->poff, P.poff, sizeof(a->poff));
  memcpy(a->aoff, P.aoff, sizeof(a->aoff));
  a->use_tc = want_tc ? 1 : 0;
  a->use_dsg = bf16 && P.abytes[A_DSG] > 0;
  a->act_layers = (hp->flags & MT_FLAG_RECOMPUTE_EXPERT_ACT) ? 1 : hp->n_layers;
  // counters need whole 128-row blocks on both sides of every hand-off
  a->deps = bf16 && !(hp->flags & MT_FLAG_BARRIERS_ONLY);
  a->smem_bytes = (int)smem;
  if (want_tc) {
    int ms = mt_build_tensor_maps(a, shadow);
    if (ms != MT_OK) { delete a; return ms; }
  }
  a->debug_op = op;
  a->dbg_layer = layer;
  cudaError_t e = op ? (bf16 ? mt_launch_op_bf16(*a, grid, smem, (cudaStream_t)stream)
                             : mt_launch_op_f32(*a, grid, smem, (cudaStream_t)stream))
                     : (bf16 ? mt_launch_mega_bf16(*a, grid, smem, (cudaStream_t)stream)
                             : mt_launch_mega_f32(*a, grid, smem, (cudaStream_t)stream));
  delete a;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  return MT_OK;
}
}  // namespace

extern "C" {

int32_t mt_read_outputs(const void* arena, mt_outputs* out, void* stream) {
  if (!arena || !out) return MT_ERR_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MT_ERR_CUDA;
  ArenaHdr h;
  if (cudaMemcpy(&h, arena, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MT_ERR_CUDA;
  memset(out, 0, sizeof(*out));
  out->status = h.status;
  out->error_site = h.error_site;
  out->micro_index = h.micro_index;
  out->optimizer_ran = h.optimizer_ran;
  out->loss = h.loss;
  out->loss_update = h.loss_update;
  out->grad_norm = h.grad_norm;
  out->clip_coef = h.clip_coef;
  out->n_ctas = h.n_ctas;
  out->n_phases = h.n_phases;
  memcpy(out->expert_counts, h.expert_counts, sizeof(out->expert_counts));
  out->experts_updated = h.experts_updated;
  out->expert_grad_norm = h.expert_grad_norm;
  out->expert_clip_coef = h.expert_clip_coef;
  return h.status;
}

int32_t mt_debug_view(const void* arena, const mt_hparams* hp, int32_t which, int32_t layer, mt_view* out) {
  int st = check_hparams(hp);
  if (st) return st;
  if (!arena || !out) return MT_ERR_ARG;
  MtPlan P;
  make_plan(hp, &P);
  const MtDims& D = P.D;
  if (layer < 0 || layer > D.L) return MT_ERR_ARG;
  if (layer == D.L && which != MT_VIEW_HIDDEN) return MT_ERR_ARG;
  char* base = (char*)arena;
  const long long T = D.T;
  switch (which) {
    case MT_VIEW_ROUTER_LOGITS:
      *out = {base + P.aoff[A_Z] + (long long)layer * T * D.E * 4, T * D.E, 4}; break;
    case MT_VIEW_TOPK_IDX:
      *out = {base + P.aoff[A_IDX] + (long long)layer * T * D.K * 4, T * D.K, 4}; break;
    case MT_VIEW_TOPK_W:
      *out = {base + P.aoff[A_WGT] + (long long)layer * T * D.K * 4, T * D.K, 4}; break;
    case MT_VIEW_ROUTE_OFFS:
      *out = {base + P.aoff[A_OFFS] + (long long)layer * (D.E + 1) * 4, D.E + 1, 4}; break;
    case MT_VIEW_ROUTE_PERM:
      *out = {base + P.aoff[A_PERM] + (long long)layer * D.Pmax * 4, D.Pmax, 4}; break;
    case MT_VIEW_TOK_LOSS:
      *out = {base + P.aoff[A_TOKLOSS], T, 4}; break;
    case MT_VIEW_TRACE:
      if (!(hp->flags & MT_FLAG_TRACE)) return MT_ERR_ARG;
      *out = {base + P.aoff[A_TRACE], (long long)D.nch * MT_TRACE_WORDS, 8}; break;
    case MT_VIEW_HIDDEN:
      *out = {base + P.aoff[A_X] + (long long)layer * T * D.d * 4, T * D.d, 4}; break;
    case MT_VIEW_LOGITS:
      *out = {base + P.aoff[A_DLOGITS], T * D.V, D.op_bytes}; break;
    case MT_VIEW_QKV:
      *out = {base + P.aoff[A_QKV] + (long long)layer * T * 3 * D.hq * D.op_bytes, T * 3 * D.hq, D.op_bytes}; break;
    case MT_VIEW_ATTN_O:
      *out = {base + P.aoff[A_O] + (long long)layer * T * D.hq * D.op_bytes, T * D.hq, D.op_bytes}; break;
    case MT_VIEW_LSE:
      *out = {base + P.aoff[A_LSE] + (long long)layer * D.B * D.H * D.S * 4, (long long)D.B * D.H * D.S, 4}; break;
    case MT_VIEW_DOUT:
      *out = {base + P.aoff[A_DO], T * D.hq, D.op_bytes}; break;
    case MT_VIEW_DSUM:
      *out = {base + P.aoff[A_DSUM], (long long)D.B * D.H * D.S, 4}; break;
    case MT_VIEW_DQKV:
      *out = {base + P.aoff[A_DQKV], T * 3 * D.hq, D.op_bytes}; break;
    case MT_VIEW_XMID:
      *out = {base + P.aoff[A_XM] + (long long)layer * T * D.d * 4, T * D.d, 4}; break;
    case MT_VIEW_R2:
      *out = {base + P.aoff[A_R2] + (long long)layer * T * D.d * D.op_bytes, T * D.d, D.op_bytes}; break;
    case MT_VIEW_EXPERT_IN:
      *out = {base + P.aoff[A_XS] + (long long)layer * D.Pmax * D.d * D.op_bytes, (long long)D.Pmax * D.d,
              D.op_bytes}; break;
    case MT_VIEW_FINAL_NORM:
      *out = {base + P.aoff[A_RF], T * D.d, D.op_bytes}; break;
    case MT_VIEW_DX:
      *out = {base + P.aoff[A_DX], T * D.d, 4}; break;
    default:
      return MT_ERR_ARG;
  }
  return MT_OK;
}

int32_t mt_debug_gemm(const void* A, int32_t a_mn, const void* B, int32_t b_mn, float* C, int32_t M, int32_t N,
                      int32_t K, int32_t rag, const int32_t* offs, int32_t nseg, int32_t precision, int32_t use_tc,
                      void* arena, int64_t arena_bytes, void* stream) {
  if (!A || !B || !C || !arena || M <= 0 || N <= 0 || K <= 0) return MT_ERR_ARG;
  if (arena_bytes < (int64_t)sizeof(ArenaHdr) || !aligned(arena, 256)) return MT_ERR_ARG;
  if (precision != MT_PREC_FP32 && precision != MT_PREC_BF16) return MT_ERR_ARG;
  if (rag < 0 || rag > 2 || (rag && (!offs || nseg <= 0))) return MT_ERR_ARG;
  if (rag == 1 && a_mn) return MT_ERR_ARG;
  if (rag == 2 && !(a_mn && b_mn)) return MT_ERR_ARG;
  const bool bf16 = precision == MT_PREC_BF16;
  // bf16 operands run on the tensor cores only; the CUDA-core engine is the
  // fp32 model's
  if (bf16 && !(use_tc & 1)) return MT_ERR_UNSUPPORTED;
  const bool tc = bf16;
  const int out_mode = tc ? ((use_tc >> 1) & 3) : 0;     // use_tc bits 1-2: output mode (tensor cores only)
  if (out_mode == 3) return MT_ERR_ARG;
  if (tc && (M % 128 || N % 256 || K % 64)) return MT_ERR_UNSUPPORTED;
  if (tc && (!aligned(A, 16) || !aligned(B, 16))) return MT_ERR_ARG;
  const size_t smem = tc ? (size_t)MT_TC_SMEM : (size_t)SG_BM * SG_CPAD * 4;
  int grid = 0;
  int st = prepare_launch(bf16, smem, &grid);
  if (st) return st;
  KArgs* a = new KArgs();
  memset(a, 0, sizeof(KArgs));
  a->arena = (char*)arena;
  a->timeout_ns = 4000000000LL;
  a->debug_gemm = 1;
  a->dbg_a = A; a->dbg_b = B; a->dbg_c = C;
  a->dbg_m = M; a->dbg_n = N; a->dbg_k = K; a->dbg_a_mn = a_mn; a->dbg_b_mn = b_mn;
  a->dbg_rag = rag; a->dbg_nseg = rag ? nseg : 0; a->dbg_offs = offs;
  a->dbg_out_mode = out_mode;
  a->dbg_tma = tc && (use_tc & 8) && rag != 2 && out_mode < 2;
  a->use_tc = tc ? 1 : 0;
  if (tc) {
    const long long segs = rag == 1 ? nseg : 1;
    const long long ar = a_mn ? K : M, ac = a_mn ? M : K;
    const long long br = (b_mn ? K : N) * segs, bc = b_mn ? N : K;
    // use_tc bit 4: K-major operands in one 128-row (A) / 256-row (B) box per K block
    const bool tall = (use_tc & 16) != 0;
    a->dbg_a_rpb = (tall && !a_mn && rag != 2) ? 128 : 64;
    a->dbg_b_rpb = (tall && !b_mn && rag != 2) ? 256 : 64;
    int ms = mt_build_debug_maps(a, A, ar, ac, B, br, bc, a->dbg_tma ? C : nullptr, M, N, out_mode == 0,
                                 a->dbg_a_rpb, a->dbg_b_rpb);
    if (ms != MT_OK) { delete a; return ms; }
  }
  cudaError_t e = bf16 ? mt_launch_mega_bf16(*a, grid, smem, (cudaStream_t)stream)
                       : mt_launch_mega_f32(*a, grid, smem, (cudaStream_t)stream);
  delete a;
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MT_ERR_LAUNCH;
  }
  return MT_OK;
}

const char* mt_status_string(int32_t s) {
  switch (s) {
    case MT_OK: return "ok";
    case MT_ERR_ARG: return "invalid argument";
    case MT_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MT_ERR_ARENA_SMALL: return "arena too small";
    case MT_ERR_LAUNCH: return "kernel launch failed";
    case MT_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MT_ERR_DEVICE_BOUNDS: return "device-side index out of range";
    case MT_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

}  // extern "C"

// ---------------------------------------------------------------------------
// fp32 -> bf16 compute copy
// ---------------------------------------------------------------------------
static __global__ void sync_shadow_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                          long long n) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

extern "C" int32_t mt_sync_shadow(const float* master, void* shadow_bf16, int64_t n, void* stream) {
  if (!master || !shadow_bf16 || n < 0) return MT_ERR_ARG;
  if (n == 0) return MT_OK;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  sync_shadow_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(master, (__nv_bfloat16*)shadow_bf16, n);
  return cudaGetLastError() == cudaSuccess ? MT_OK : MT_ERR_LAUNCH;
}
