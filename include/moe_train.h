/*
 * moe_train.h - C ABI of the GB300 training-update megakernel.
 *
 * One call of mt_train_update() runs one microbatch of a complete training
 * update of a top-K-of-E mixture-of-experts transformer as ONE persistent
 * cooperative CUDA kernel resident on every SM: forward pass, next-token
 * cross-entropy, backward pass and - after the last microbatch of an update -
 * global-norm clipping and AdamW.  This is the operation described by the
 * Latch pages: "How a training megakernel works", sections "One training
 * update" (forward, loss, backward, optimizer), "From two weights to 200
 * million" (TinyMoE: attention + expert layers, top-2 of 16 routing, AdamW),
 * "1 - Describe the model and update" (bf16 attention, token_topk,
 * route_order, ragged_mm, global-norm clipping, AdamW), "4 - Scheduling and
 * storage" (phases across all SMs, grid-wide barriers, a planned activation
 * arena, FP32 master weights and Adam moments with BF16 matrix products) and
 * "How GPUs usually run it" (16 microbatches, one kernel per microbatch, one
 * optimizer update after the last).
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller (allocated
 *    e.g. through torch).  The library never allocates device memory and
 *    never frees caller memory.  Pointers must be 256-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Work is enqueued asynchronously on it; the call returns after the launch.
 *  - Every entry point returns an mt_status (0 = MT_OK).  Argument errors are
 *    detected on the host before anything is enqueued.  Device-side failures
 *    (a bounded wait that ran out) are reported in the arena's status word,
 *    read with mt_read_outputs().
 *  - Thread safety: calls on different arenas may run concurrently; calls
 *    that share an arena must be ordered on one stream.
 */
#ifndef MOE_TRAIN_H_
#define MOE_TRAIN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mt_status {
  MT_OK = 0,
  MT_ERR_ARG = 1,             /* null / misaligned pointer, bad size or hyperparameter */
  MT_ERR_UNSUPPORTED = 2,     /* dimensions outside what the kernels implement */
  MT_ERR_ARENA_SMALL = 3,     /* arena_bytes < mt_arena_bytes(hp) */
  MT_ERR_LAUNCH = 4,          /* CUDA error at launch (e.g. cooperative grid too large) */
  MT_ERR_DEVICE_TIMEOUT = 5,  /* a device-side bounded wait ran out (status word) */
  MT_ERR_DEVICE_BOUNDS = 6,   /* a device-side index check failed (status word) */
  MT_ERR_CUDA = 7             /* other CUDA runtime error */
} mt_status;

enum { MT_PREC_FP32 = 0, MT_PREC_BF16 = 1 };

/* hp.flags bits (any other bit is MT_ERR_ARG) */
enum {
  MT_FLAG_TRACE = 1u << 0,        /* record per-CTA phase timestamps in the arena */
  MT_FLAG_NO_OPTIMIZER = 1u << 3, /* skip clip + AdamW even on the last microbatch */
  MT_FLAG_TEST_STALL = 1u << 4,   /* test only: CTA 0 never arrives at the first grid
                                     barrier, so the others' bounded waits run out */
  MT_FLAG_BARRIERS_ONLY = 1u << 5, /* separate every phase by a grid barrier, even where
                                     per-block dependency counters would do (same
                                     results bit for bit; for comparison) */
  /* Memory rules ("Open problems", Generality 2: what is stored and what is
   * recomputed).  Each trades arena bytes for work. */
  MT_FLAG_RECOMPUTE_ATTN_DS = 1u << 7, /* bf16: keep no dS^T of the attention backward
                                          (batch*heads*seq^2 bf16 per launch); the dQ items
                                          recompute P and dS instead of reading it (same
                                          values up to fp32 summation order) */
  MT_FLAG_RECOMPUTE_EXPERT_ACT = 1u << 9, /* keep the expert activations [g | u] and
                                          silu(g) u of one layer instead of all L
                                          ((L-1) * Pmax * 3 * d_ff operands fewer); the backward
                                          re-runs each layer's gate/up product first (bit for
                                          bit the same values) */
  /* Selective updates ("Results", "Other measured compiler work": shared
   * weights update every microbatch, experts every 16).  The shared tensors
   * (every tensor but w_gate, w_up, w_down) get their gradients overwritten
   * and a clipped AdamW step (step t = hp.step, norm over the shared
   * gradients) after EVERY microbatch, each microbatch weighing its targets
   * 1 / (batch*(seq-1)).  The expert tensors' gradients are summed over the
   * micro_count microbatches of a period (overwritten at micro_index 0); after
   * the last one they get a clipped AdamW step (t = hp.expert_step, norm over
   * their gradients) on the mean, sum / micro_count.  mt_outputs reports the
   * shared step in grad_norm / clip_coef and the expert step in
   * expert_grad_norm / expert_clip_coef / experts_updated. */
  MT_FLAG_SELECTIVE_EXPERTS = 1u << 8,
  MT_FLAGS_ALL = (1u << 0) | (1u << 3) | (1u << 4) | (1u << 5) | (1u << 7) | (1u << 8) | (1u << 9)
};

/*
 * Hyperparameters and dimensions of one microbatch launch (host struct,
 * copied at call time).  Model: vocab V, d_model d, n_layers L, n_heads H of
 * head_dim hd (H*hd may differ from d), n_experts E, top_k K, expert width
 * d_ff F; this microbatch holds batch x seq tokens.
 * Implemented shapes (else MT_ERR_UNSUPPORTED): d a multiple of 32 and at
 * most 768; hd 16 or 64; F a multiple of 64; E <= 64 with E*d*4 <= 160 KiB;
 * K <= min(8, E); V a multiple of 8; L <= 16; seq >= 2.  The bf16 model
 * runs on the tensor cores only (tcgen05 products and attention) and
 * additionally needs seq a multiple of 128, d, H*hd, V and F multiples of
 * 256, and hd = 64.
 */
typedef struct mt_hparams {
  int32_t vocab, d_model, n_layers, n_heads, head_dim, n_experts, top_k, d_ff;
  int32_t batch, seq;
  int32_t precision;          /* MT_PREC_FP32 (exact fp32 FMAs, no TF32) | MT_PREC_BF16 */
  int32_t micro_index;        /* 0 overwrites the gradients, > 0 adds into them */
  int32_t micro_count;        /* optimizer runs when micro_index == micro_count - 1 */
  uint32_t flags;
  int64_t step;               /* AdamW step t (1-based) used for bias correction */
  float lr, beta1, beta2, eps, weight_decay;
  float clip_norm, clip_eps;  /* c = min(1, clip_norm / (||g|| + clip_eps)) */
  float norm_eps;             /* RMSNorm epsilon */
  float rope_theta;           /* rotary base */
  float loss_coef;            /* per-target CE coefficient; 0 -> 1/(batch*(seq-1)*micro_count) */
  int64_t wait_timeout_ns;    /* bound on every device-side wait; 0 -> 4e9 ns */
  int64_t expert_step;        /* MT_FLAG_SELECTIVE_EXPERTS: AdamW step t of the expert tensors */
  int32_t n_unique_layers;    /* looped model ("Results", "Other measured compiler work": repeated
                                 layers share weights and accumulate gradients across visits):
                                 U distinct layers, layer visit l (0 <= l < n_layers) uses weight
                                 slot l mod U, and each slot's gradient is the sum over its visits.
                                 0 = n_layers (no looping); else 1 <= U <= n_layers.  The per-layer
                                 parameter tensors are stacked over the U slots. */
  int32_t reserved0;          /* must be 0 */
} mt_hparams;

/* One parameter tensor inside the flat fp32 parameter buffer. */
typedef struct mt_tensor_desc {
  char name[24];
  int64_t offset;             /* element offset into the flat buffer (multiple of 64) */
  int64_t numel;
  int32_t ndim;
  int64_t shape[4];
  int32_t weight_decay;       /* 1: AdamW decay applies (every tensor, by design) */
} mt_tensor_desc;

#define MT_MAX_LAYERS 16
#define MT_MAX_EXPERTS 64
#define MT_MAX_CTAS 512

/* Results of the last launch on an arena (see mt_read_outputs). */
typedef struct mt_outputs {
  int32_t status;             /* mt_status of the device side (0 = ok) */
  int32_t error_site;         /* which wait / check failed (internal code) */
  int32_t micro_index;        /* microbatch the values below belong to */
  int32_t optimizer_ran;      /* 1 if clip + AdamW ran in this launch */
  float loss;                 /* this microbatch's sum of coef * CE */
  float loss_update;          /* running sum over the microbatches of this update */
  float grad_norm;            /* ||g||_2 before clipping (valid if optimizer_ran) */
  float clip_coef;            /* min(1, clip/(norm+eps))  (valid if optimizer_ran) */
  int32_t n_ctas;             /* grid size of the launch */
  int32_t n_phases;           /* grid-wide barriers passed */
  int32_t expert_counts[MT_MAX_LAYERS * MT_MAX_EXPERTS]; /* tokens routed to [layer][expert] */
  int32_t experts_updated;    /* MT_FLAG_SELECTIVE_EXPERTS: 1 if the expert step ran */
  float expert_grad_norm;     /* its norm of the mean expert gradient, before clipping */
  float expert_clip_coef;     /* and its clip coefficient */
} mt_outputs;

/* Number of parameters (elements of the flat fp32 buffers params/grads/m/v).
 * Defined by: "How a training megakernel works", "From two weights to 200
 * million" (the model's weights: attention and expert layers) with the sizes
 * of hp.  Errors: a negative mt_status (see check rules above). */
int64_t mt_param_count(const mt_hparams* hp);

/* Defined by: "How a training megakernel works", "From two weights to 200
 * million" (attention + expert layers with a router) and "1 - Describe the
 * model and update" (the model's parameter names are kept).
 * Fill out[0..min(cap, n)-1] with the parameter layout; returns the number of
 * tensors n (11) or a negative mt_status.  Order: emb [V,d], attn_norm [L,d],
 * wqkv [L,3*H*hd,d], wo [L,d,H*hd], moe_norm [L,d], router [L,E,d],
 * w_gate [L,E,F,d], w_up [L,E,F,d], w_down [L,E,d,F], final_norm [d],
 * lm_head [V,d]; every matrix is [out, in]. */
int32_t mt_param_layout(const mt_hparams* hp, mt_tensor_desc* out, int32_t cap);

/* Defined by: "How a training megakernel works", "4 - Scheduling and storage"
 * (values passed between phases live in a planned GPU-memory arena).
 * Bytes of caller-provided device arena the launch needs (worst case over
 * routing), or a negative mt_status.  With MT_FLAG_TRACE in hp->flags the
 * arena also holds the per-CTA trace (MT_VIEW_TRACE), so traced launches
 * need an arena sized with that flag.  bf16 models also hold one layer's
 * attention-backward dS^T, batch * heads * seq^2 bf16 values, unless the
 * memory rule MT_FLAG_RECOMPUTE_ATTN_DS is set; an arena must be sized with
 * the flags of the launches that use it. */
int64_t mt_arena_bytes(const mt_hparams* hp);

/* Zero the arena's control header (barrier and status words).  Call once after
 * allocating an arena, and again after a device-side error.  Defined by: same
 * section (the grid-wide barriers between phases); the pages' per-update
 * scalar fills are not needed because the barrier resets itself.
 * Errors: MT_ERR_ARG (null or misaligned arena), MT_ERR_CUDA. */
int32_t mt_arena_init(void* arena, int64_t arena_bytes, void* stream);

/* Write the bf16 compute copy of the fp32 master parameters:
 * shadow[i] = bf16(master[i]) for i < n (round to nearest even).  Defined by:
 * "4 - Scheduling and storage" (FP32 master weights, BF16 matrix products).
 * Both pointers are caller-owned device memory.  Errors: MT_ERR_ARG,
 * MT_ERR_LAUNCH. */
int32_t mt_sync_shadow(const float* master, void* shadow_bf16, int64_t n, void* stream);

/*
 * One microbatch of the training update, as one persistent kernel launch.
 * Defined by: "How a training megakernel works", "One training update"
 * (forward, loss, backward, optimizer step), "What Latch does" (one
 * persistent GPU program resident across the SMs; steps 1-4: bf16 attention,
 * token_topk, route_order, ragged_mm, global-norm clipping and AdamW, phases
 * with grid-wide barriers, the arena, FP32 master weights and moments with
 * BF16 products) and "How GPUs usually run it" (one kernel per microbatch,
 * one optimizer update after the last microbatch of the published batch).
 *   params  fp32 [n]   master weights (updated in place by the optimizer)
 *   shadow  bf16 [n]   compute copy (read by bf16 products, rewritten by AdamW);
 *                      may be NULL when hp->precision == MT_PREC_FP32
 *   grads   fp32 [n]   gradient sum over the update's microbatches
 *                      (overwritten when micro_index == 0)
 *   adam_m, adam_v fp32 [n]  Adam moments (updated by the optimizer)
 *   tokens  int32 [batch, seq] token ids in [0, vocab), device memory
 *   arena   device scratch of arena_bytes >= mt_arena_bytes(hp), 256-B aligned,
 *           initialised once with mt_arena_init; holds activations, routing
 *           buffers, the status word and the outputs block.
 * Position s of each sequence is trained to predict token s+1; the last
 * position has no target.
 */
int32_t mt_train_update(float* params, void* shadow, float* grads, float* adam_m,
                        float* adam_v, const int32_t* tokens, const mt_hparams* hp,
                        void* arena, int64_t arena_bytes, void* stream);

/* Synchronise `stream` and copy the outputs block of the arena to *out.
 * Returns out->status (MT_OK if the device side succeeded), or MT_ERR_ARG /
 * MT_ERR_CUDA for host-side failures.  Defined by: "One training update" (the
 * loss) and "1 - Describe the model and update" (global-norm clipping: the
 * norm and coefficient). */
int32_t mt_read_outputs(const void* arena, mt_outputs* out, void* stream);

/* Capacity of the per-CTA trace (MT_VIEW_TRACE) */
enum { MT_TRACE_PHASES = 512, MT_TRACE_JOBS = 1024, MT_TRACE_WORDS = 2 * (512 + 1024) };

/* Debug views into the arena after a launch (device pointers into the arena,
 * owned by the arena's owner).  which: see MT_VIEW_* ; layer selects the
 * layer for per-layer buffers.  Defined by: "5 - Generation and compilation"
 * (the generated program's comparison and numerical-check commands).
 * Errors: MT_ERR_ARG (unknown view or layer, trace view of an untraced
 * arena). */
enum {
  MT_VIEW_ROUTER_LOGITS = 0,  /* fp32 [T, E] */
  MT_VIEW_TOPK_IDX = 1,       /* int32 [T, K] */
  MT_VIEW_TOPK_W = 2,         /* fp32 [T, K] */
  MT_VIEW_ROUTE_OFFS = 3,     /* int32 [E+1] padded segment starts (multiples of 128) */
  MT_VIEW_ROUTE_PERM = 4,     /* int32 [Pmax] assignment t*K+k at each sorted row, -1 = pad */
  MT_VIEW_TOK_LOSS = 5,       /* fp32 [T] coef * CE per position */
  MT_VIEW_TRACE = 6,          /* int64 [CTA][MT_TRACE_WORDS] (hp->flags must hold
                                 MT_FLAG_TRACE, else MT_ERR_ARG): per CTA, for
                                 grid barrier p < MT_TRACE_PHASES the pair (t_arrive,
                                 t_leave) at [2p], then from [2*MT_TRACE_PHASES] for job
                                 stamp j < MT_TRACE_JOBS the pair (t_end, job id); ns */
  MT_VIEW_HIDDEN = 7,         /* fp32 [T, d] residual stream entering `layer` (layer = L: final) */
  MT_VIEW_LOGITS = 8,         /* operand type [T, V]: LM-head logits (bf16 or fp32), overwritten
                                 in place by dlogits during the same launch */
  /* Buffers the single-op harness (mt_debug_run) reads and writes.  "op" is
   * the operand type: bf16 for MT_PREC_BF16, fp32 for MT_PREC_FP32. */
  MT_VIEW_QKV = 9,            /* op [T, 3*H*hd] of `layer`: q and k after RoPE, v; head h owns
                                 columns h*hd..(h+1)*hd-1 of each of the three blocks */
  MT_VIEW_ATTN_O = 10,        /* op [T, H*hd] of `layer`: attention output */
  MT_VIEW_LSE = 11,           /* fp32 [B*H, S] of `layer`: row log-sum-exp of the scaled scores;
                                 natural log for MT_PREC_FP32, base-2 log for MT_PREC_BF16
                                 (log2 of the row sum of exp2(log2(e) q.k / sqrt(hd))) */
  MT_VIEW_DOUT = 12,          /* op [T, H*hd]: gradient wrt the attention output (one layer at a time) */
  MT_VIEW_DSUM = 13,          /* fp32 [B*H, S]: rowsum(dO * O) of the attention backward */
  MT_VIEW_DQKV = 14,          /* op [T, 3*H*hd]: gradient wrt q, k (before RoPE) and v */
  MT_VIEW_XMID = 15,          /* fp32 [T, d] of `layer`: residual stream after attention */
  MT_VIEW_R2 = 16,            /* op [T, d] of `layer`: expert RMSNorm output (router input) */
  MT_VIEW_EXPERT_IN = 17,     /* op [Pmax, d] of `layer`: expert inputs in expert order (rows of
                                 MT_VIEW_ROUTE_PERM; pad rows zero) */
  MT_VIEW_FINAL_NORM = 18,    /* op [T, d]: final RMSNorm output (LM-head input) */
  MT_VIEW_DX = 19             /* fp32 [T, d]: gradient wrt the residual stream; after an update,
                                 wrt the embedding output (the rows the embedding backward sums) */
};
typedef struct mt_view {
  void* ptr;
  int64_t numel;
  int32_t elem_bytes;
} mt_view;
int32_t mt_debug_view(const void* arena, const mt_hparams* hp, int32_t which, int32_t layer,
                      mt_view* out);

/*
 * Single-op parity harness (tests): run ONE step of the update on inputs the
 * caller has written into the arena (through mt_debug_view pointers) and into
 * the parameter buffers, with the same device code the update uses.  Every
 * op is one cooperative launch on `stream`; its outputs are read back through
 * mt_debug_view and mt_read_outputs.  Arguments are those of mt_train_update
 * (hp describes the model and the microbatch; the arena must be initialised
 * with mt_arena_init and sized by mt_arena_bytes(hp)) plus:
 *   op     one of MT_OP_*;
 *   layer  the layer whose per-layer buffers the op reads and writes.
 * Errors as mt_train_update; MT_ERR_ARG for an unknown op or layer.
 */
enum {
  /* Causal attention forward ("1 - Describe the model and update": bf16
   * attention): MT_VIEW_QKV -> MT_VIEW_ATTN_O, MT_VIEW_LSE. */
  MT_OP_ATTN_FWD = 1,
  /* Causal attention backward: MT_VIEW_QKV, MT_VIEW_ATTN_O, MT_VIEW_LSE (as the
   * forward left them) and MT_VIEW_DOUT -> MT_VIEW_DSUM, MT_VIEW_DQKV. */
  MT_OP_ATTN_BWD = 2,
  /* Expert RMSNorm, router logits, token_topk and route_order with the
   * dispatch gather (same section): MT_VIEW_XMID and the moe_norm / router
   * parameters -> MT_VIEW_R2, MT_VIEW_ROUTER_LOGITS, MT_VIEW_TOPK_IDX,
   * MT_VIEW_TOPK_W, MT_VIEW_ROUTE_OFFS, MT_VIEW_ROUTE_PERM, MT_VIEW_EXPERT_IN
   * and the expert counts of mt_outputs. */
  MT_OP_ROUTER = 3,
  /* LM head and fused next-token cross-entropy ("2 - Capture": labels and
   * coefficients): MT_VIEW_FINAL_NORM, lm_head, tokens -> MT_VIEW_TOK_LOSS,
   * the loss of mt_outputs and dlogits in MT_VIEW_LOGITS. */
  MT_OP_LM_CE = 4,
  /* Global-norm clipping and AdamW ("1 - Describe the model and update"):
   * params, grads, adam_m, adam_v (hp->step, lr, ...) -> updated params, m, v,
   * the bf16 shadow, and grad_norm / clip_coef of mt_outputs. */
  MT_OP_CLIP_ADAMW = 5
};
int32_t mt_debug_run(int32_t op, int32_t layer, float* params, void* shadow, float* grads, float* adam_m,
                     float* adam_v, const int32_t* tokens, const mt_hparams* hp, void* arena,
                     int64_t arena_bytes, void* stream);

/*
 * mt_train_update_noalloc - the same launch as mt_train_update, but with no
 * arena argument: the scratch arena is a fixed array of MT_NOALLOC_ARENA_BYTES
 * that this library keeps in device memory.  The paper has no counterpart to
 * this entry point.
 *
 * Who it is for: callers that are handed pointers to their tensors but may not
 * allocate device memory themselves - for example a plug-in running inside a
 * host application whose device memory is all owned by that application's
 * own pool, or a service that has fixed its device-memory budget at start-up
 * and may not call cudaMalloc (which can also block on device-wide work) while
 * it serves.  The caller still passes every input and output (params, shadow,
 * grads, adam_m, adam_v, tokens, out); this call makes no device allocation.
 *
 * Limits and behaviour:
 *  - Only models with mt_arena_bytes(hp) <= MT_NOALLOC_ARENA_BYTES (16 MiB,
 *    e.g. the tiny configuration, which needs about 8.8 MiB) are accepted;
 *    larger ones return MT_ERR_ARENA_SMALL and nothing is enqueued.
 *  - The array occupies MT_NOALLOC_ARENA_BYTES on every device where the
 *    library's code is loaded, until the process exits.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress), so the address stays right after a
 *    cudaDeviceReset reloads the library's module; the first call on a device
 *    also loads the module there, so make it before any stream capture.
 *  - Every argument check (as mt_train_update's) runs before anything is
 *    enqueued: a call that returns an error has written nothing.
 *  - Every call uses the same array, which keeps what the previous call left
 *    in it; each call clears the barrier and status words it needs at zero.
 *    Calls whose execution overlaps on the GPU (different streams, or
 *    different host threads on one device) race on the array and must be
 *    serialised by the caller.
 *  - out (host pointer, may be NULL): when given, the call synchronises
 *    `stream` and copies the launch's outputs block to *out, returning
 *    out->status; when NULL the call returns after the launch is enqueued.
 */
#define MT_NOALLOC_ARENA_BYTES (16u << 20)
int32_t mt_train_update_noalloc(float* params, void* shadow, float* grads, float* adam_m, float* adam_v,
                                const int32_t* tokens, const mt_hparams* hp, mt_outputs* out, void* stream);

/*
 * Test harness: one matrix product C = A * B^T through the megakernel's product
 * engine (tcgen05 tensor cores for MT_PREC_BF16, which then needs bit 0 of
 * use_tc set, else MT_ERR_UNSUPPORTED; the fp32 model's CUDA-core engine for
 * MT_PREC_FP32), fp32 accumulation, fp32 C.  Used by the tests to check
 * every operand layout of the update's products ("1 - Describe the model and
 * update": dense products and ragged_mm) in isolation.
 *   rag = 0: A is [M,K] (a_mn = 0) or [K,M] (a_mn = 1); B is [N,K] (b_mn = 0)
 *            or [K,N] (b_mn = 1); C is [M,N].
 *   rag = 1: ragged rows.  A [M,K] (a_mn must be 0) is split into nseg row
 *            segments at offs (device int32 [nseg+1], multiples of 128, the
 *            last <= M); segment e multiplies B[e] ([nseg][N][K] or
 *            [nseg][K][N]); rows past offs[nseg] are not written.
 *   rag = 2: ragged reduction.  A [K,M], B [K,N] (a_mn = b_mn = 1); segment e
 *            reduces rows offs[e]..offs[e+1] into C[e] ([nseg][M][N]).
 * use_tc: bit 0 selects the tensor cores; on that path bits 1-2 select the
 * output (0: fp32 C; 1: bf16 C written over the start of the C buffer; 2: the
 * accumulators are read from tensor memory and dropped - a timing mode); bit 3
 * writes an fp32 or bf16 C (rag 0 or 1) by bulk tensor stores from the
 * epilogue's shared-memory window, the path the update's products take.
 * A and B are bf16 (MT_PREC_BF16) or fp32 (MT_PREC_FP32) device arrays.  The
 * tensor-core path needs M a multiple of 128, N a multiple of 256 and K a
 * multiple of 64.
 * arena: >= 4 KiB device scratch initialised with mt_arena_init.
 */
int32_t mt_debug_gemm(const void* A, int32_t a_mn, const void* B, int32_t b_mn, float* C, int32_t M, int32_t N,
                      int32_t K, int32_t rag, const int32_t* offs, int32_t nseg, int32_t precision, int32_t use_tc,
                      void* arena, int64_t arena_bytes, void* stream);

/* Stable text for a status code. */
const char* mt_status_string(int32_t status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_TRAIN_H_ */
