"""Host-side checks of the C ABI: the library loads, exports every entry
point the header declares, reports the parameter layout of the seeded inputs,
sizes the arena monotonically, and rejects bad arguments before touching a
GPU.  No compute call is made."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import moe_inputs as mi
from adamw_persistent_sm_gb300 import binding as B
from adamw_persistent_sm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return B.load(build_if_missing=True)


def header_functions():
    text = open(os.path.join(ROOT, "include", "moe_train.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\**\s*(mt_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_function(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_library_is_in_tree(lib):
    assert os.path.dirname(_build.LIB) == os.path.join(ROOT, "adamw_persistent_sm_gb300")


@pytest.mark.parametrize("name", ["tiny", "b2", "top8"])
def test_param_layout_matches_inputs(lib, name):
    cfg = mi.get_config(name)
    hp = B.hparams(cfg)
    assert B.mt_param_count(hp) == mi.param_count(cfg)
    lay = B.mt_param_layout(hp)
    shapes = mi.param_shapes(cfg)
    assert [t["name"] for t in lay] == [n for n, _ in shapes]
    for t, (_, s) in zip(lay, shapes):
        assert t["shape"] == s
        assert t["offset"] % 64 == 0
        assert t["weight_decay"] == 1
    ends = [t["offset"] + t["numel"] for t in lay]
    assert all(e <= o for e, o in zip(ends, [t["offset"] for t in lay][1:]))


def test_param_count_of_published_stand_in(lib):
    # 219,132,672 with an untied head (the page quotes 199,837,056 for TinyMoE)
    assert B.mt_param_count(B.hparams(mi.get_config("b2"))) == 219_132_672
    # 8 x (2d + 4d^2 + E d + 3 E F d) + 2 V d + d with E=32, F=256
    assert B.mt_param_count(B.hparams(mi.get_config("top8"))) == 219_230_976


def test_arena_grows_with_tokens(lib):
    cfg = mi.get_config("b2")
    sizes = [B.mt_arena_bytes(B.hparams(cfg.replace(batch=b))) for b in (1, 2, 4, 8)]
    assert all(s > 0 for s in sizes)
    assert sizes == sorted(sizes) and len(set(sizes)) == 4


def _bad(cfg, **kw):
    return B.hparams(cfg.replace(**kw)) if kw else B.hparams(cfg)


@pytest.mark.parametrize("kw,code", [
    (dict(vocab=0), B.MT_ERR_ARG),
    (dict(head_dim=32), B.MT_ERR_UNSUPPORTED),
    (dict(d_model=1024), B.MT_ERR_UNSUPPORTED),
    (dict(top_k=9, n_experts=16), B.MT_ERR_UNSUPPORTED),
    (dict(n_experts=65), B.MT_ERR_UNSUPPORTED),
    (dict(d_ff=100), B.MT_ERR_UNSUPPORTED),
    (dict(seq=1), B.MT_ERR_UNSUPPORTED),
    (dict(lr=float("nan")), B.MT_ERR_ARG),
    (dict(beta2=1.0), B.MT_ERR_ARG),
    (dict(micro_count=0), B.MT_ERR_ARG),
])
def test_bad_hparams_are_rejected(lib, kw, code):
    hp = _bad(mi.get_config("tiny"), **kw)
    assert B.mt_param_count(hp) == -code
    assert B.mt_arena_bytes(hp) == -code


def test_train_update_argument_checks(lib):
    cfg = mi.get_config("tiny")
    hp = B.hparams(cfg)
    need = B.mt_arena_bytes(hp)
    fake = 1 << 20                      # aligned, never dereferenced: checks fail first
    args = [fake, 0, fake, fake, fake, fake]
    assert B.mt_train_update(0, 0, fake, fake, fake, fake, hp, fake, need) == B.MT_ERR_ARG
    assert B.mt_train_update(*args, hp, fake + 4, need) == B.MT_ERR_ARG          # misaligned arena
    assert B.mt_train_update(*args, hp, fake, need - 1) == B.MT_ERR_ARENA_SMALL
    hb = B.hparams(mi.get_config("b2"))
    assert B.mt_train_update(*args, hb, fake, B.mt_arena_bytes(hb)) == B.MT_ERR_ARG   # bf16 needs shadow
    hp.micro_index = 1
    assert B.mt_train_update(*args, hp, fake, need) == B.MT_ERR_ARG               # index >= count
    assert B.mt_arena_init(0, 1024) == B.MT_ERR_ARG
    assert B.status_string(B.MT_ERR_DEVICE_TIMEOUT) == "device-side wait timed out"


def test_struct_sizes_match_header(lib):
    assert C.sizeof(B.mt_hparams) == 128
    assert C.sizeof(B.mt_outputs) == 40 + 4 * 16 * 64 + 12


def test_trace_arena_is_sized_by_the_trace_flag():
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("tiny")
    plain = B.mt_arena_bytes(B.hparams(cfg))
    traced = B.mt_arena_bytes(B.hparams(cfg, flags=B.MT_FLAG_TRACE))
    per_cta = B.MT_TRACE_WORDS * 8
    assert traced - plain >= B.MT_MAX_CTAS * per_cta
    assert traced - plain < B.MT_MAX_CTAS * per_cta + 4096
    assert plain <= B.MT_NOALLOC_ARENA_BYTES


def test_arena_holds_the_attention_ds_buffer_unless_recomputed():
    """bf16 models keep one layer's dS^T (batch x heads x seq^2 bf16) for the
    dQ product; the memory rule MT_FLAG_RECOMPUTE_ATTN_DS drops it, and the
    fp32 model never holds it."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("b2")
    ds = cfg.batch * cfg.n_heads * cfg.seq * cfg.seq * 2
    keep = B.mt_arena_bytes(B.hparams(cfg))
    drop = B.mt_arena_bytes(B.hparams(cfg, flags=B.MT_FLAG_RECOMPUTE_ATTN_DS))
    assert ds <= keep - drop < ds + 4096
    tiny = B.mt_arena_bytes(B.hparams(mi.get_config("tiny")))
    assert tiny <= B.MT_NOALLOC_ARENA_BYTES


def test_unknown_flags_and_untiled_bf16_shapes_are_refused():
    """Retired or unknown flag bits are argument errors; a bf16 model whose
    shapes the tensor-core tiles do not cover is refused (there is no
    CUDA-core fallback for bf16)."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("b2")
    for bit in (1, 2, 6, 10, 31):
        assert B.mt_arena_bytes(B.hparams(cfg, flags=1 << bit)) == -B.MT_ERR_ARG
    fake = 1 << 20
    args = (fake, fake, fake, fake, fake, fake)
    bad = B.hparams(cfg.replace(seq=1000))          # not a multiple of 128
    need = B.mt_arena_bytes(bad)
    assert need > 0
    assert B.mt_train_update(*args, bad, fake, need) == B.MT_ERR_UNSUPPORTED
    bad = B.hparams(cfg.replace(d_ff=320))          # not a multiple of 256
    assert B.mt_train_update(*args, bad, fake, B.mt_arena_bytes(bad)) == B.MT_ERR_UNSUPPORTED


def test_memory_rule_keeps_one_layer_of_expert_activations():
    """MT_FLAG_RECOMPUTE_EXPERT_ACT drops (L-1) layers of [g | u] and
    silu(g) u: (L-1) * Pmax * 3 * d_ff operand values."""
    from adamw_persistent_sm_gb300 import binding as B
    for name in ("b2", "b32", "tiny"):
        cfg = mi.get_config(name)
        keep = B.mt_arena_bytes(B.hparams(cfg))
        drop = B.mt_arena_bytes(B.hparams(cfg, flags=B.MT_FLAG_RECOMPUTE_EXPERT_ACT))
        T, K, E = cfg.tokens_per_micro, cfg.top_k, cfg.n_experts
        pmax = -(-(T * K + E * 127) // 128) * 128
        ob = 2 if cfg.precision == "bf16" else 4
        saved = (cfg.n_layers - 1) * pmax * 3 * cfg.d_ff * ob
        assert saved - 4096 < keep - drop <= saved + 4096, (name, keep - drop, saved)


@pytest.mark.parametrize("name", ["tiny", "b2", "top8"])
def test_debug_views_are_disjoint_buffers_inside_the_arena(lib, name):
    """Every debug view of the first and the last layer lies inside the arena
    that mt_arena_bytes plans, with its documented shape; views of different
    buffers do not overlap and start on 1024-byte boundaries; the trace view
    exists only when the trace flag sizes the arena for it.  Host arithmetic
    only: the arena address is never dereferenced."""
    cfg = mi.get_config(name)
    hp = B.hparams(cfg)
    need = B.mt_arena_bytes(hp)
    base = 1 << 40
    T, d, E, K = cfg.batch * cfg.seq, cfg.d_model, cfg.n_experts, cfg.top_k
    hq = cfg.n_heads * cfg.head_dim
    op = 2 if cfg.precision == "bf16" else 4
    shapes = {B.MT_VIEW_ROUTER_LOGITS: (T * E, 4), B.MT_VIEW_TOPK_IDX: (T * K, 4), B.MT_VIEW_TOPK_W: (T * K, 4),
              B.MT_VIEW_ROUTE_OFFS: (E + 1, 4), B.MT_VIEW_TOK_LOSS: (T, 4), B.MT_VIEW_HIDDEN: (T * d, 4),
              B.MT_VIEW_XMID: (T * d, 4), B.MT_VIEW_DX: (T * d, 4), B.MT_VIEW_QKV: (T * 3 * hq, op),
              B.MT_VIEW_ATTN_O: (T * hq, op), B.MT_VIEW_R2: (T * d, op), B.MT_VIEW_FINAL_NORM: (T * d, op)}
    views = [getattr(B, k) for k in dir(B) if k.startswith("MT_VIEW_") and k != "MT_VIEW_TRACE"]
    spans = []
    for which in views:
        for layer in (0, cfg.n_layers - 1):
            v = B.mt_debug_view(base, hp, which, layer)
            lo = v.ptr - base
            hi = lo + v.numel * v.elem_bytes
            assert 0 <= lo < hi <= need, (which, layer)
            if which in shapes:
                assert (v.numel, v.elem_bytes) == shapes[which], which
            if layer == 0:
                assert lo % 1024 == 0, which
                spans.append((lo, hi, which))
    spans.sort()
    for (_, a1, wa), (b0, _, wb) in zip(spans, spans[1:]):
        assert a1 <= b0, (wa, wb)
    # the residual stream entering the final norm (layer L) exists too
    v = B.mt_debug_view(base, hp, B.MT_VIEW_HIDDEN, cfg.n_layers)
    assert v.ptr - base + v.numel * v.elem_bytes <= need
    with pytest.raises(ValueError):
        B.mt_debug_view(base, hp, B.MT_VIEW_TRACE, 0)
    ht = B.hparams(cfg, flags=B.MT_FLAG_TRACE)
    v = B.mt_debug_view(base, ht, B.MT_VIEW_TRACE, 0)
    assert 0 <= v.ptr - base and v.ptr - base + v.numel * v.elem_bytes <= B.mt_arena_bytes(ht)
