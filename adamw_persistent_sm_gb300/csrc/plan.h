// plan.h - layout of parameters and of the activation arena, shared by the
// host planner (host.cu) and the megakernel (mega.cuh).
//
// The arena holds every value that crosses a phase boundary of the update
// (the "planned GPU-memory arena" of "How a training megakernel works",
// section "4 - Scheduling and storage").  Offsets are fixed per dimensions,
// so one plan serves every launch with the same hyperparameters.
#pragma once
#include <stdint.h>
#include <cuda.h>

#define MT_TILE_M 128           // routing pads each expert segment to this many rows
#define MT_NMAPS 40

// parameter tensors, in flat-buffer order
enum ParamId {
  P_EMB = 0, P_ATTN_NORM, P_WQKV, P_WO, P_MOE_NORM, P_ROUTER, P_WGATE, P_WUP, P_WDOWN,
  P_FINAL_NORM, P_LM_HEAD, P_COUNT
};

// arena buffers
enum ArenaId {
  A_HDR = 0,   // control header (ArenaHdr)
  A_ROPE,      // fp32 [S][hd/2][2] cos, sin
  A_X,         // fp32 [L+1][T][d] residual stream entering each layer (L: final)
  A_XM,        // fp32 [L][T][d] residual stream after attention
  A_INV1,      // fp32 [L][T] attention RMSNorm 1/rms
  A_INV2,      // fp32 [L][T] expert RMSNorm 1/rms
  A_R,         // op   [L][T][d] attention RMSNorm output
  A_QKV,       // op   [L][T][3hq] q,k after RoPE, v
  A_O,         // op   [L][T][hq] attention output
  A_LSE,       // fp32 [L][B*H][S] attention row log-sum-exp
  A_R2,        // op   [L][T][d] expert RMSNorm output
  A_Z,         // fp32 [L][T][E] router logits
  A_IDX,       // i32  [L][T][K] chosen experts (slot 0 best)
  A_WGT,       // fp32 [L][T][K] renormalised router weights
  A_CNT,       // i32  [L][NCH][E] per-chunk expert counts
  A_OFFS,      // i32  [L][E+1] padded segment starts
  A_PERM,      // i32  [L][Pmax] assignment at each sorted row (-1 pad)
  A_INVM,      // i32  [L][T*K] sorted row of each assignment
  A_XS,        // op   [L][Pmax][d] expert inputs in expert order
  A_GU,        // op   [L][Pmax][2F] gate and up pre-activations [g | u]
  A_ACT,       // op   [L][Pmax][F] silu(g) * u
  A_Y,         // fp32 [L][Pmax][d] expert outputs
  A_RF,        // op   [T][d] final RMSNorm output
  A_INVF,      // fp32 [T]
  A_CEPART,    // fp32 [T][ceil(V/128)][2] per column tile (max, sum exp(l - max)) of the logits
  A_CETGT,     // fp32 [T] logit of the target token
  A_DLOGITS,   // op   [T][V] logits from the LM head, overwritten in place by dlogits
  A_TOKLOSS,   // fp32 [T]
  A_DX,        // fp32 [T][d] gradient wrt the residual stream
  A_DXO,       // op   [T][d] operand copy of A_DX
  A_DY,        // op   [Pmax][d] gradient wrt expert outputs
  A_DZ,        // fp32 [T][E] gradient wrt router logits
  A_DZB,       // bf16 [T][64] A_DZ rounded to bf16, columns E..63 zero (operand of the router-weight gradient)
  A_DGU,       // op   [Pmax][2F] gradient wrt [g | u]
  A_DXS,       // fp32 [Pmax][d] gradient wrt expert inputs
  A_DR2,       // fp32 [T][d] gradient wrt expert RMSNorm output
  A_DO,        // op   [T][hq] gradient wrt attention output
  A_DSUM,      // fp32 [B*H][S] rowsum(dO * O) of the attention backward
  A_DQKV,      // op   [T][3hq] gradient wrt q,k,v (before RoPE)
  A_DSG,       // bf16 [B*H*S][S] dS^T of one layer's attention backward (keys x queries; tensor-core path)
  A_DR,        // fp32 [T][d] gradient wrt attention RMSNorm output
  A_DRF,       // fp32 [T][d] gradient wrt final RMSNorm output
  A_PART,      // fp32 [NCH][E+2][d] column-reduction partials
  A_KPART,     // fp32 [<= 8 x 3hq x d] split-K partial tiles of weight gradients
  A_NORMPART,  // fp32 [NCH] squared-norm partials (double precision accumulate)
  A_DEP,       // u32  dependency counters and work tickets (layout below), zeroed by the first phase
  A_TRACE,     // i64  [NCH][MT_TRACE_WORDS] barrier pairs, then job stamps
  A_COUNT
};


// TMA tensor maps (bf16 operands of the tensor-core products), one per 2-D
// buffer; per-layer and per-expert tensors are addressed through the outer
// coordinate of a map over the whole stack.
enum MapId {
  MAP_R = 0, MAP_WQKV, MAP_O, MAP_WO, MAP_XS, MAP_WGATE, MAP_WUP, MAP_ACT, MAP_WDOWN, MAP_RF,
  MAP_WLM, MAP_DLOGITS, MAP_DY, MAP_DGU, MAP_DXO, MAP_DQKV, MAP_QKV, MAP_DOUT, MAP_DZB, MAP_R2,
  // 32 x 32 boxes of the epilogues' bulk stores and aux loads: bf16 with the
  // 64-byte swizzle, fp32 with the 128-byte swizzle
  MAP_E_QKV, MAP_E_GU, MAP_E_ACT, MAP_E_DGU,
  MAP_E_DLOGITS,  // (32 rows x 64 columns, 128-byte swizzle)
  MAP_E_DO, MAP_E_O,
  MAP_E_Y, MAP_E_DRF, MAP_E_DXS, MAP_E_DR, MAP_E_XM, MAP_E_X,
  MAP_E_DQKV,   // 32 rows x 64 columns, 128-byte swizzle: the attention backward's dq, dk, dv rows
  MAP_E_OROW,   // 32 rows x 64 columns, 128-byte swizzle: the attention forward's output rows
  MAP_E_DS,     // 128 rows x 64 columns, 128-byte swizzle: dS^T tiles stored by the dK/dV job
  MAP_E_DSL,    // 64 x 64, 128-byte swizzle: dS^T boxes loaded by the dQ product
  MAP_E_QKV64,  // 32 rows x 64 columns, 128-byte swizzle: q,k,v rows of the qkv product
  MAP_COUNT
};
static_assert(MAP_COUNT <= MT_NMAPS, "too many tensor maps");

struct MtDims {
  int V, d, L, H, hd, hq, E, K, F, B, S, T;
  int U;       // distinct layers (weight slots); layer visit l uses slot l % U
  int Pmax;    // rows of expert-ordered buffers: T*K + E*(MT_TILE_M-1), rounded up to MT_TILE_M
  int nch;     // maximum number of CTAs (chunks) the arena was sized for
  int op_bytes;
};

// Control header at the start of the arena.  Each word the barrier spins on
// sits in its own 128-byte line.
struct ArenaHdr {
  unsigned int bar_count; unsigned int pad0[31];
  unsigned int bar_gen;   unsigned int pad1[31];
  int status; int error_site; int pad2[30];
  // outputs (mirrors mt_outputs)
  int micro_index, optimizer_ran;
  float loss, loss_update, grad_norm, clip_coef;
  int n_ctas, n_phases;
  int expert_counts[16 * 64];
  // second optimizer group (expert tensors under MT_FLAG_SELECTIVE_EXPERTS)
  int experts_updated;
  float expert_grad_norm, expert_clip_coef;
};

// Dependency counters.  Each layer owns one counter per 128-row block of
// every hand-off that runs without a grid barrier; a producer adds 1 when it
// has stored its part of a block, a consumer waits until the block's counter
// reaches the number of producer parts.  After the L layers come the work
// tickets (dynamically scheduled jobs take item numbers from them).
enum DepKind {
  DEP_QKV = 0,   // [T/128] q,k,v tiles stored (target: 3hq/256 column tiles)
  DEP_O,         // [T/128] attention items stored (target: H)
  DEP_XMID,      // [T/128] out-projection tiles stored (target: d/256)
  DEP_RN,        // [T/128] 32-token combine groups stored (next layer's norm rows; target 4)
  DEP_DR,        // [T/128] qkv dgrad tiles stored (attention-norm backward rows; target: d/256)
  DEP_ACT,       // [Pmax/128] gate/up tiles stored (target: 2F/256)
  DEP_KINDS
};
#define MT_DEP_GROUP 32         // tokens per combine item when counters are on
#define MT_TICKETS 16           // ticket counters per layer (plus one set for the head)
// Work tickets.  Per layer: the attention jobs and every tensor-core product
// (tiles drawn in index order by whichever CTA is free); the head's set (layer
// index L) holds the LM-head products and the optimizer sweep.
enum TicketId {
  TK_ADAMW = 0,
  TK_QKV, TK_WO, TK_GATEUP, TK_DOWN,
  TK_DOWN_DGRAD, TK_DOWN_WGRAD, TK_GU_DGRAD, TK_GU_WGRAD, TK_WO_DGRAD, TK_WO_WGRAD, TK_QKV_DGRAD, TK_QKV_WGRAD,
  TK_GATEUP_AGAIN,              // the gate/up product re-run in the backward (memory rule)
  TK_ROUTER_WGRAD,              // the router-weight gradient product
  TK_COUNT_,
  // the head's set: LM-head products and the optimizer ranges
  TK_LM = TK_QKV, TK_LM_DGRAD = TK_WO, TK_LM_WGRAD = TK_GATEUP,
  TK_ADAMW_R1 = TK_DOWN, TK_ADAMW_R2 = TK_DOWN_DGRAD
};
static_assert(TK_COUNT_ <= MT_TICKETS, "ticket ids exceed a layer's ticket set");
__host__ __device__ inline long long dep_blocks(const MtDims& D, int kind) {
  return kind == DEP_ACT ? D.Pmax / MT_TILE_M : (D.T + MT_TILE_M - 1) / MT_TILE_M;
}
__host__ __device__ inline long long dep_layer_words(const MtDims& D) {
  return (DEP_KINDS - 1) * dep_blocks(D, DEP_QKV) + dep_blocks(D, DEP_ACT);
}
__host__ __device__ inline long long dep_offset(const MtDims& D, int l, int kind) {
  return (long long)l * dep_layer_words(D) + (long long)kind * dep_blocks(D, DEP_QKV);
}
__host__ __device__ inline long long ticket_offset(const MtDims& D, int l, int id) {
  return (long long)D.L * dep_layer_words(D) + (long long)l * MT_TICKETS + id;
}
__host__ __device__ inline long long dep_words(const MtDims& D) {
  return (long long)D.L * dep_layer_words(D) + (long long)(D.L + 1) * MT_TICKETS;
}

// The optimizer of one launch: up to MT_OPT_RANGES contiguous ranges of the
// flat parameter / gradient / moment buffers, each in one of two groups.  A
// group is one clipped AdamW step: its own global norm (over the gradients of
// its ranges, times gscale), its own bias corrections.
#define MT_OPT_RANGES 3
struct OptRange {
  long long off, n;             // element range (off and n multiples of 4)
  int group;                    // 0 or 1
  int first;                    // the group's first range (writes the group's outputs)
};
struct OptGroup {
  float ibc1, ibc2;             // 1 / (1 - beta^t) for this group's step t
  float gscale;                 // the step uses gscale * (summed gradient)
  int r0, nr;                   // its ranges: orng[r0 .. r0+nr-1] (norm partial slots alike)
};

struct KArgs {
  MtDims D;
  float lr, beta1, beta2, eps, wd, clip, clip_eps, norm_eps, coef, rope_theta;
  float decay;                  // 1 - lr * weight_decay, in double on the host
  int micro_index, micro_count, run_opt;
  unsigned acc_mask;            // bit p: parameter tensor p's gradient is added to the buffer (else overwritten)
  int n_ranges;                 // optimizer ranges this launch (0: no optimizer)
  OptRange orng[MT_OPT_RANGES];
  OptGroup ogrp[2];
  unsigned int flags;
  long long timeout_ns;
  long long n_params;
  float* master;
  void* shadow;
  float* grads;
  float* adam_m;
  float* adam_v;
  const int* tokens;
  char* arena;
  long long poff[P_COUNT];      // element offsets of each tensor in the flat buffers
  long long aoff[A_COUNT];      // byte offsets of each arena buffer
  int debug_op;                 // single-op harness (mt_opkernel): MT_OP_* and its layer
  int dbg_layer;
  int debug_gemm;               // test harness: run only the product described below
  const void* dbg_a; const void* dbg_b; float* dbg_c;
  int dbg_m, dbg_n, dbg_k, dbg_a_mn, dbg_b_mn, dbg_rag, dbg_nseg;
  int dbg_out_mode;             // 0 fp32 C, 1 bf16 C (written over the fp32 buffer), 2 accumulators read only
  int dbg_tma;                  // C written by the bulk-store epilogue (map MAP_E_Y fp32 / MAP_E_QKV bf16)
  int dbg_a_rpb, dbg_b_rpb;     // rows per TMA box of the harness's A and B maps
  const int* dbg_offs;
  int use_tc;                   // tcgen05 GEMMs (bf16 only)
  int use_dsg;                  // dQ as a product over stored dS^T (A_DSG, MAP_E_DS/DSL; bf16 only)
  int deps;                     // dependency counters replace the grid barriers they cover
  int act_layers;               // layers of [g | u] and silu(g) u the arena keeps: L, or 1 when the
                                // backward re-runs each layer's gate/up product (memory rule)
  int smem_bytes;               // dynamic shared memory of the launch
  CUtensorMap maps[MT_NMAPS];
};

// host-side plan (host.cu)
struct MtPlan {
  MtDims D;
  long long aoff[A_COUNT];
  long long abytes[A_COUNT];
  long long arena_bytes;
  long long poff[P_COUNT];
  long long pnumel[P_COUNT];
  long long n_params;
};
