"""ctypes binding of the C ABI in include/moe_train.h.

Argument marshalling only: every step of the training update runs in the
CUDA library.  Pointers are plain integers (e.g. ``tensor.data_ptr()``);
streams are ``cudaStream_t`` values as integers (``torch.cuda.current_stream()
.cuda_stream``).  The library is loaded from this package directory; if it
is missing the import of a symbol fails loudly - there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

from . import _build

MT_OK = 0
MT_ERR_ARG = 1
MT_ERR_UNSUPPORTED = 2
MT_ERR_ARENA_SMALL = 3
MT_ERR_LAUNCH = 4
MT_ERR_DEVICE_TIMEOUT = 5
MT_ERR_DEVICE_BOUNDS = 6
MT_ERR_CUDA = 7

MT_PREC_FP32 = 0
MT_PREC_BF16 = 1

MT_FLAG_TRACE = 1 << 0
MT_FLAG_NO_OPTIMIZER = 1 << 3
MT_FLAG_TEST_STALL = 1 << 4
MT_FLAG_BARRIERS_ONLY = 1 << 5
MT_FLAG_RECOMPUTE_ATTN_DS = 1 << 7
MT_FLAG_SELECTIVE_EXPERTS = 1 << 8
MT_FLAG_RECOMPUTE_EXPERT_ACT = 1 << 9

MT_MAX_LAYERS = 16
MT_MAX_EXPERTS = 64

MT_VIEW_ROUTER_LOGITS = 0
MT_VIEW_TOPK_IDX = 1
MT_VIEW_TOPK_W = 2
MT_VIEW_ROUTE_OFFS = 3
MT_VIEW_ROUTE_PERM = 4
MT_VIEW_TOK_LOSS = 5
MT_VIEW_TRACE = 6
MT_MAX_CTAS = 512                     # arena buffers are sized for up to this many CTAs
MT_TRACE_PHASES = 512                 # per CTA: barrier (arrive, leave) pairs, then
MT_TRACE_JOBS = 1024                  # (end time, job id) pairs
MT_TRACE_WORDS = 2 * (MT_TRACE_PHASES + MT_TRACE_JOBS)
MT_VIEW_HIDDEN = 7
MT_VIEW_LOGITS = 8
MT_VIEW_QKV = 9
MT_VIEW_ATTN_O = 10
MT_VIEW_LSE = 11
MT_VIEW_DOUT = 12
MT_VIEW_DSUM = 13
MT_VIEW_DQKV = 14
MT_VIEW_XMID = 15
MT_VIEW_R2 = 16
MT_VIEW_EXPERT_IN = 17
MT_VIEW_FINAL_NORM = 18
MT_VIEW_DX = 19

MT_OP_ATTN_FWD = 1
MT_OP_ATTN_BWD = 2
MT_OP_ROUTER = 3
MT_OP_LM_CE = 4
MT_OP_CLIP_ADAMW = 5


class mt_hparams(C.Structure):
    _fields_ = [
        ("vocab", C.c_int32), ("d_model", C.c_int32), ("n_layers", C.c_int32),
        ("n_heads", C.c_int32), ("head_dim", C.c_int32), ("n_experts", C.c_int32),
        ("top_k", C.c_int32), ("d_ff", C.c_int32), ("batch", C.c_int32), ("seq", C.c_int32),
        ("precision", C.c_int32), ("micro_index", C.c_int32), ("micro_count", C.c_int32),
        ("flags", C.c_uint32), ("step", C.c_int64),
        ("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
        ("weight_decay", C.c_float), ("clip_norm", C.c_float), ("clip_eps", C.c_float),
        ("norm_eps", C.c_float), ("rope_theta", C.c_float), ("loss_coef", C.c_float),
        ("wait_timeout_ns", C.c_int64), ("expert_step", C.c_int64),
        ("n_unique_layers", C.c_int32), ("reserved0", C.c_int32),
    ]


class mt_tensor_desc(C.Structure):
    _fields_ = [("name", C.c_char * 24), ("offset", C.c_int64), ("numel", C.c_int64),
                ("ndim", C.c_int32), ("shape", C.c_int64 * 4), ("weight_decay", C.c_int32)]


class mt_outputs(C.Structure):
    _fields_ = [("status", C.c_int32), ("error_site", C.c_int32), ("micro_index", C.c_int32),
                ("optimizer_ran", C.c_int32), ("loss", C.c_float), ("loss_update", C.c_float),
                ("grad_norm", C.c_float), ("clip_coef", C.c_float), ("n_ctas", C.c_int32),
                ("n_phases", C.c_int32),
                ("expert_counts", C.c_int32 * (MT_MAX_LAYERS * MT_MAX_EXPERTS)),
                ("experts_updated", C.c_int32), ("expert_grad_norm", C.c_float),
                ("expert_clip_coef", C.c_float)]


class mt_view(C.Structure):
    _fields_ = [("ptr", C.c_void_p), ("numel", C.c_int64), ("elem_bytes", C.c_int32)]


_P = C.c_void_p
_SIGNATURES = {
    "mt_param_count": (C.c_int64, [C.POINTER(mt_hparams)]),
    "mt_param_layout": (C.c_int32, [C.POINTER(mt_hparams), C.POINTER(mt_tensor_desc), C.c_int32]),
    "mt_arena_bytes": (C.c_int64, [C.POINTER(mt_hparams)]),
    "mt_arena_init": (C.c_int32, [_P, C.c_int64, _P]),
    "mt_sync_shadow": (C.c_int32, [_P, _P, C.c_int64, _P]),
    "mt_train_update": (C.c_int32, [_P, _P, _P, _P, _P, _P, C.POINTER(mt_hparams), _P, C.c_int64, _P]),
    "mt_read_outputs": (C.c_int32, [_P, C.POINTER(mt_outputs), _P]),
    "mt_debug_view": (C.c_int32, [_P, C.POINTER(mt_hparams), C.c_int32, C.c_int32, C.POINTER(mt_view)]),
    "mt_status_string": (C.c_char_p, [C.c_int32]),
    "mt_train_update_noalloc": (C.c_int32, [_P, _P, _P, _P, _P, _P, C.POINTER(mt_hparams),
                                            C.POINTER(mt_outputs), _P]),
    "mt_debug_run": (C.c_int32, [C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P, C.POINTER(mt_hparams), _P,
                                 C.c_int64, _P]),
    "mt_debug_gemm": (C.c_int32, [_P, C.c_int32, _P, C.c_int32, _P, C.c_int32, C.c_int32, C.c_int32,
                                  C.c_int32, _P, C.c_int32, C.c_int32, C.c_int32, _P, C.c_int64, _P]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False) -> C.CDLL:
    """Load the in-tree CUDA library (optionally building it first)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library {_build.LIB} is missing: run __graft_entry__.build()")
        _build.build()
    lib = C.CDLL(_build.LIB)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def hparams(cfg, micro_index: int = 0, flags: int = 0, step: int | None = None,
            wait_timeout_ns: int = 0, loss_coef: float = 0.0, expert_step: int = 1) -> mt_hparams:
    """mt_hparams from any object with the configuration's attribute names."""
    hp = mt_hparams()
    hp.vocab, hp.d_model, hp.n_layers = cfg.vocab, cfg.d_model, cfg.n_layers
    hp.n_heads, hp.head_dim, hp.n_experts = cfg.n_heads, cfg.head_dim, cfg.n_experts
    hp.top_k, hp.d_ff, hp.batch, hp.seq = cfg.top_k, cfg.d_ff, cfg.batch, cfg.seq
    hp.precision = MT_PREC_BF16 if cfg.precision == "bf16" else MT_PREC_FP32
    hp.micro_index, hp.micro_count = micro_index, cfg.micro_count
    hp.flags = flags
    hp.step = cfg.step if step is None else step
    hp.lr, hp.beta1, hp.beta2, hp.eps = cfg.lr, cfg.beta1, cfg.beta2, cfg.eps
    hp.weight_decay, hp.clip_norm, hp.clip_eps = cfg.weight_decay, cfg.clip_norm, cfg.clip_eps
    hp.norm_eps, hp.rope_theta = cfg.norm_eps, cfg.rope_theta
    hp.loss_coef = loss_coef
    hp.wait_timeout_ns = wait_timeout_ns
    hp.expert_step = expert_step
    hp.n_unique_layers = getattr(cfg, "n_unique_layers", 0)
    return hp


# ---- thin wrappers with the C names ---------------------------------------
def mt_param_count(hp: mt_hparams) -> int:
    return load().mt_param_count(C.byref(hp))


def mt_param_layout(hp: mt_hparams) -> list[dict]:
    lib = load()
    n = lib.mt_param_layout(C.byref(hp), None, 0)
    if n < 0:
        raise ValueError(f"mt_param_layout: {status_string(-n)}")
    arr = (mt_tensor_desc * n)()
    lib.mt_param_layout(C.byref(hp), arr, n)
    return [dict(name=t.name.decode(), offset=t.offset, numel=t.numel,
                 shape=tuple(t.shape[i] for i in range(t.ndim)), weight_decay=t.weight_decay)
            for t in arr]


def mt_arena_bytes(hp: mt_hparams) -> int:
    return load().mt_arena_bytes(C.byref(hp))


def mt_arena_init(arena: int, nbytes: int, stream: int = 0) -> int:
    return load().mt_arena_init(arena, nbytes, stream)


def mt_sync_shadow(master: int, shadow: int, n: int, stream: int = 0) -> int:
    return load().mt_sync_shadow(master, shadow, n, stream)


def mt_train_update(params: int, shadow: int, grads: int, adam_m: int, adam_v: int, tokens: int,
                    hp: mt_hparams, arena: int, arena_bytes: int, stream: int = 0) -> int:
    return load().mt_train_update(params, shadow, grads, adam_m, adam_v, tokens, C.byref(hp),
                                  arena, arena_bytes, stream)


MT_NOALLOC_ARENA_BYTES = 16 << 20


def mt_train_update_noalloc(params: int, shadow: int, grads: int, adam_m: int, adam_v: int,
                            tokens: int, hp: mt_hparams, out: mt_outputs | None = None,
                            stream: int = 0) -> int:
    """Training-update launch whose scratch arena is the library's fixed
    device array (no device allocation by the caller or the library)."""
    return load().mt_train_update_noalloc(params, shadow, grads, adam_m, adam_v, tokens, C.byref(hp),
                                          C.byref(out) if out is not None else None, stream)


def mt_read_outputs(arena: int, stream: int = 0) -> mt_outputs:
    out = mt_outputs()
    load().mt_read_outputs(arena, C.byref(out), stream)
    return out


def mt_debug_view(arena: int, hp: mt_hparams, which: int, layer: int = 0) -> mt_view:
    v = mt_view()
    st = load().mt_debug_view(arena, C.byref(hp), which, layer, C.byref(v))
    if st != MT_OK:
        raise ValueError(f"mt_debug_view: {status_string(st)}")
    return v


def mt_debug_run(op: int, layer: int, params: int, shadow: int, grads: int, adam_m: int, adam_v: int,
                 tokens: int, hp: mt_hparams, arena: int, arena_bytes: int, stream: int = 0) -> int:
    return load().mt_debug_run(op, layer, params, shadow, grads, adam_m, adam_v, tokens, C.byref(hp),
                               arena, arena_bytes, stream)


def mt_debug_gemm(A: int, a_mn: int, B_: int, b_mn: int, C_: int, M: int, N: int, K: int, rag: int,
                  offs: int, nseg: int, precision: int, use_tc: int, arena: int, arena_bytes: int,
                  stream: int = 0) -> int:
    return load().mt_debug_gemm(A, a_mn, B_, b_mn, C_, M, N, K, rag, offs, nseg, precision, use_tc,
                                arena, arena_bytes, stream)


def status_string(st: int) -> str:
    return load().mt_status_string(st).decode()
