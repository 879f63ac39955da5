"""Single-op parity: each step of the update run alone through mt_debug_run
(the update's own device code) on seeded inputs, compared element by element
with the oracle function that defines it.

Ops and the passages that define them ("How a training megakernel works",
section "1 - Describe the model and update"): causal attention forward and
backward (``bf16_sdpa.sdpa``), the expert RMSNorm + router with
``token_topk`` and ``route_order`` and the dispatch gather, the LM head with
the fused next-token cross-entropy ("2 - Capture": labels and
coefficients), and global-norm clipping + AdamW.

Sizes: the 32x1024 and 1x4096 (top-8) shapes of the update, where the
oracle evaluates sampled (batch, head) pairs or token rows one by one, and
the tiny fp32 model in full.  Tolerances follow from the arithmetic of each
path and are stated beside each assertion.
"""
import math

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity_util import rel_l2, to_np

pytestmark = pytest.mark.gpu

CASES = ["tiny", "b32", "top8"]


def _trainer(cfg):
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    return MoETrainer(cfg, "cuda:0")


def _put(tr, which, layer, arr, dtype):
    v = tr.debug_view(which, layer, dtype)
    v.copy_(torch.as_tensor(np.ascontiguousarray(arr, dtype=np.float32).reshape(-1)).to(dtype).to(v.device))


def _get(tr, which, layer, dtype, shape):
    return to_np(tr.debug_view(which, layer, dtype)).reshape(shape)


def _opdtype(cfg):
    return torch.bfloat16 if cfg.precision == "bf16" else torch.float32


def _ok(tr):
    from adamw_persistent_sm_gb300 import binding as B
    out = tr.outputs()
    assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
    return out


def _heads(cfg, x, block):
    """[T, 3hq] or [T, hq] -> the (b, h) slices of column block ``block``."""
    B_, S, H, hd = cfg.batch, cfg.seq, cfg.n_heads, cfg.head_dim
    hq = H * hd
    return x[:, block * hq:(block + 1) * hq].reshape(B_, S, H, hd).transpose(0, 2, 1, 3)


def _pairs(cfg, n=6):
    """(batch, head) pairs the oracle evaluates: all for small shapes, else a
    seeded sample that includes the first and the last pair."""
    B_, H = cfg.batch, cfg.n_heads
    allp = [(b, h) for b in range(B_) for h in range(H)]
    if len(allp) <= 8:
        return allp
    rng = np.random.default_rng(5)
    pick = rng.choice(len(allp), size=n - 2, replace=False)
    return sorted({allp[0], allp[-1], *[allp[i] for i in pick]})


def _attn_inputs(cfg, seed):
    bf = cfg.precision == "bf16"
    T, hq = cfg.tokens_per_micro, cfg.n_heads * cfg.head_dim
    return mi.normal_operand((T, 3 * hq), seed, 1.0, bf16=bf)


def _run_attn_fwd(cfg, tr, qkv):
    from adamw_persistent_sm_gb300 import binding as B
    dt = _opdtype(cfg)
    _put(tr, B.MT_VIEW_QKV, 0, qkv, dt)
    tr.debug_run(B.MT_OP_ATTN_FWD, 0)
    _ok(tr)
    T, hq = cfg.tokens_per_micro, cfg.n_heads * cfg.head_dim
    o = _get(tr, B.MT_VIEW_ATTN_O, 0, dt, (T, hq))
    lse = _get(tr, B.MT_VIEW_LSE, 0, torch.float32, (cfg.batch, cfg.n_heads, cfg.seq))
    if cfg.precision == "bf16":
        lse = lse * math.log(2.0)          # this path keeps base-2 log-sum-exp
    return o, lse


@pytest.mark.parametrize("name", CASES)
def test_attention_forward(name):
    """o = softmax(q k^T / sqrt(hd), keys j <= i) v and the row log-sum-exp.
    bf16: P is rounded to bf16 for the PV product and o is stored in bf16
    (2^-9 relative each), the scores and sums are fp32: per element
    |err| <= 8e-3 |o| + 8e-3 (v has unit scale), lse within 2e-4.  fp32: 1e-5."""
    cfg = mi.get_config(name)
    tr = _trainer(cfg)
    qkv = _attn_inputs(cfg, 100)
    o, lse = _run_attn_fwd(cfg, tr, qkv)
    q, k, v = (_heads(cfg, qkv.astype(np.float64), i) for i in range(3))
    og = _heads(cfg, o, 0)
    bf = cfg.precision == "bf16"
    # the first query of every sequence sees only itself: o = v exactly
    np.testing.assert_array_equal(og[:, :, 0, :], v[:, :, 0, :])
    for b, h in _pairs(cfg):
        ref = oracle.causal_attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1])[0, 0]
        err = np.abs(og[b, h] - ref)
        if bf:
            assert np.all(err <= 8e-3 * np.abs(ref) + 8e-3), (b, h, float(err.max()))
            assert rel_l2(og[b, h], ref) < 5e-3, (b, h)
        else:
            assert rel_l2(og[b, h], ref) < 1e-5, (b, h)
        lref = oracle.causal_logsumexp(q[b, h], k[b, h])
        assert np.max(np.abs(lse[b, h] - lref)) < (2e-4 if bf else 1e-5), (b, h)


@pytest.mark.parametrize("name", ["b32", "top8"])
def test_attention_forward_rising_scores(name):
    """Keys whose scale grows along the sequence (1 at the first position, 6
    at the last), so that a row's later key blocks exceed the maximum of its
    first block by far more than 2^8 in exp2 units: the online softmax must
    rescale the row's accumulated output and sum by large factors mid-item
    (a stale or dropped rescale shows as an error of the size of o).  The
    input is checked to force that (from the fp64 scores) and the output is
    held to the bounds of the forward test."""
    cfg = mi.get_config(name)
    tr = _trainer(cfg)
    qkv = _attn_inputs(cfg, 110).copy()
    S, hq = cfg.seq, cfg.n_heads * cfg.head_dim
    pos = np.arange(cfg.tokens_per_micro) % S
    qkv[:, hq:2 * hq] *= (1.0 + 5.0 * pos / S)[:, None].astype(np.float32)
    qkv = mi.round_to_bf16(qkv)
    o, lse = _run_attn_fwd(cfg, tr, qkv)
    q, k, v = (_heads(cfg, qkv.astype(np.float64), i) for i in range(3))
    og = _heads(cfg, o, 0)
    scale_l2 = 1.0 / math.sqrt(cfg.head_dim) / math.log(2.0)
    moved = 0
    for b, h in _pairs(cfg):
        s = (q[b, h] @ k[b, h].T) * scale_l2
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
        first = s[:, :128].max(axis=1)
        moved += int(np.sum(s.max(axis=1) > first + 8.0))
        ref = oracle.causal_attention(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1])[0, 0]
        err = np.abs(og[b, h] - ref)
        assert np.all(err <= 8e-3 * np.abs(ref) + 8e-3), (b, h, float(err.max()))
        assert rel_l2(og[b, h], ref) < 5e-3, (b, h)
        lref = oracle.causal_logsumexp(q[b, h], k[b, h])
        assert np.max(np.abs(lse[b, h] - lref)) < 2e-4 * max(1.0, float(np.max(np.abs(lref)))), (b, h)
    assert moved > 100, moved


@pytest.mark.parametrize("name", CASES)
def test_attention_backward(name):
    """dq, dk (RoPE undone) and dv of the causal attention, from q, k, v, the
    forward's o and lse, and dO.  bf16: P and dS are rounded to bf16 for the
    products: per (b, h) relative L2 within 1e-2, and per element
    |err| <= 0.02 M + 0.02 |ref| where M is the root-sum-square size of the
    terms the output row sums (10x the 2^-9 rounding).  fp32: 1e-5."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    tr = _trainer(cfg)
    qkv = _attn_inputs(cfg, 200)
    _run_attn_fwd(cfg, tr, qkv)
    T, hq = cfg.tokens_per_micro, cfg.n_heads * cfg.head_dim
    bf = cfg.precision == "bf16"
    do = mi.normal_operand((T, hq), 201, 1.0, bf16=bf)
    dt = _opdtype(cfg)
    _put(tr, B.MT_VIEW_DOUT, 0, do, dt)
    tr.debug_run(B.MT_OP_ATTN_BWD, 0)
    _ok(tr)
    dqkv = _get(tr, B.MT_VIEW_DQKV, 0, dt, (T, 3 * hq))
    q, k, v = (_heads(cfg, qkv.astype(np.float64), i) for i in range(3))
    dout = _heads(cfg, do.astype(np.float64), 0)
    cos, sin = oracle.rope_tables(cfg.seq, cfg.head_dim, cfg.rope_theta)
    got = [_heads(cfg, dqkv, i) for i in range(3)]
    scale = 1.0 / math.sqrt(cfg.head_dim)
    worst = 0.0
    for b, h in _pairs(cfg):
        sl = (slice(b, b + 1), slice(h, h + 1))
        dq, dk, dv = oracle.causal_attention_backward(dout[sl], q[sl], k[sl], v[sl])
        refs = [oracle.rope_backward(dq, cos, sin)[0, 0], oracle.rope_backward(dk, cos, sin)[0, 0], dv[0, 0]]
        # Size of the terms each output row sums: the bf16 rounding of P and dS
        # (2^-9 relative) perturbs a row by ~2^-9 of this, whatever cancels.
        P = oracle.moe_oracle._causal_probs(q[b, h], k[b, h])
        dP = dout[b, h] @ v[b, h].T
        dS = P * (dP - np.sum(dP * P, axis=1, keepdims=True))
        ms = lambda x: np.mean(x * x, axis=1)
        # dS = P (dP - D) is formed in fp32 from dP and D summed in different
        # orders: where they cancel exactly (the first query) an fp32 residue
        # of their size remains
        dS2 = dS * dS + (1e-3 * P * (np.abs(dP) + np.abs(np.sum(dP * P, axis=1, keepdims=True)))) ** 2
        terms = [np.sqrt(dS2 @ ms(k[b, h])) * scale,
                 np.sqrt(dS2.T @ ms(q[b, h])) * scale,
                 np.sqrt((P * P).T @ ms(dout[b, h]))]
        for i, ref in enumerate(refs):
            g = got[i][b, h]
            if bf:
                assert rel_l2(g, ref) < 1e-2, ("qkv"[i], b, h, rel_l2(g, ref))
                bound = 0.02 * terms[i][:, None] + 0.02 * np.abs(ref)
                ratio = float(np.max(np.abs(g - ref) / bound))
                worst = max(worst, ratio)
                assert ratio <= 1.0, ("qkv"[i], b, h, ratio)
            else:
                assert rel_l2(g, ref) < 1e-5, ("qkv"[i], b, h, rel_l2(g, ref))
    print(f"\n{name}: worst element error / bound {worst:.3f}")


def _padded_offsets(counts, tile=128):
    offs = np.zeros(len(counts) + 1, dtype=np.int64)
    offs[1:] = np.cumsum((np.asarray(counts) + tile - 1) // tile * tile)
    return offs


@pytest.mark.parametrize("name", CASES)
def test_router_topk_route_order(name):
    """Expert RMSNorm, fp32 router logits, token_topk (ties to the lower
    expert: two experts get identical router rows) and route_order with the
    dispatch gather.  Logits within 2e-5 (|z| + rms z) of float64 (fp32
    products); r2 within bf16 rounding; choices, weights, the stable order,
    the 128-row padded segments, the gathered rows and the expert counts
    exact for the GPU's own logits."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    tr = _trainer(cfg)
    T, d, E, K = cfg.tokens_per_micro, cfg.d_model, cfg.n_experts, cfg.top_k
    x = mi.normal_operand((T, d), 300, 0.05)
    g = mi.normal_operand((d,), 301, 0.1, mean=1.0)
    wr = mi.normal_operand((E, d), 302, 0.02)
    wr[3] = wr[1]                                   # identical logits: ties go to the lower index
    tr.view(tr.params, "moe_norm")[0].copy_(torch.as_tensor(g))
    tr.view(tr.params, "router")[0].copy_(torch.as_tensor(wr))
    _put(tr, B.MT_VIEW_XMID, 0, x, torch.float32)
    tr.debug_run(B.MT_OP_ROUTER, 0)
    out = _ok(tr)
    dt = _opdtype(cfg)
    z = _get(tr, B.MT_VIEW_ROUTER_LOGITS, 0, torch.float32, (T, E))
    r2 = _get(tr, B.MT_VIEW_R2, 0, dt, (T, d))
    idx = to_np(tr.debug_view(B.MT_VIEW_TOPK_IDX, 0, torch.int32)).astype(np.int64).reshape(T, K)
    w = _get(tr, B.MT_VIEW_TOPK_W, 0, torch.float32, (T, K))
    offs = to_np(tr.debug_view(B.MT_VIEW_ROUTE_OFFS, 0, torch.int32)).astype(np.int64)
    perm = to_np(tr.debug_view(B.MT_VIEW_ROUTE_PERM, 0, torch.int32)).astype(np.int64)
    xs = _get(tr, B.MT_VIEW_EXPERT_IN, 0, dt, (-1, d))
    # logits and normalised rows against float64
    r_ref, _ = oracle.rmsnorm(x.astype(np.float64), g.astype(np.float64), cfg.norm_eps)
    z_ref = r_ref @ wr.astype(np.float64).T
    assert np.all(np.abs(z - z_ref) <= 2e-5 * (np.abs(z_ref) + np.sqrt(np.mean(z_ref ** 2))))
    rtol = 4e-3 if cfg.precision == "bf16" else 1e-6
    assert np.all(np.abs(r2 - r_ref) <= rtol * np.abs(r_ref) + 1e-6)
    np.testing.assert_array_equal(z[:, 1], z[:, 3])
    # choices and weights on the GPU's own logits
    idx_ref, w_ref, _ = oracle.token_topk(z, K)
    np.testing.assert_array_equal(idx, idx_ref)
    np.testing.assert_allclose(w, w_ref, rtol=0, atol=1e-5)
    tie = np.sum(np.any(idx == 1, axis=1) & ~np.any(idx == 3, axis=1) & (np.sort(z, 1)[:, -K] == z[:, 1]))
    print(f"\n{name}: {tie} tokens whose last chosen slot was a tie between experts 1 and 3")
    # stable counting sort, padded segments, gathered rows, counts
    o_perm, counts, o_offs, _ = oracle.route_order(idx, E)
    np.testing.assert_array_equal(offs, _padded_offsets(counts))
    for e in range(E):
        seg = perm[offs[e]:offs[e] + counts[e]]
        np.testing.assert_array_equal(seg, o_perm[o_offs[e]:o_offs[e + 1]])
        assert np.all(perm[offs[e] + counts[e]:offs[e + 1]] == -1)
        np.testing.assert_array_equal(xs[offs[e]:offs[e] + counts[e]], r2[seg // K])
        assert not np.any(xs[offs[e] + counts[e]:offs[e + 1]])
        assert out.expert_counts[e] == counts[e]


def _ce_rows(cfg):
    """Token rows the oracle evaluates: all for small shapes, else a seeded
    sample plus the last position of the first and last sequences."""
    T, S = cfg.tokens_per_micro, cfg.seq
    if T <= 256:
        return np.arange(T)
    rng = np.random.default_rng(7)
    rows = set(rng.choice(T, size=254, replace=False).tolist()) | {S - 1, T - 1, 0, T - 2}
    return np.array(sorted(rows))


@pytest.mark.parametrize("name", CASES)
def test_lm_head_cross_entropy(name):
    """Logits = rf W_lm^T, per-position coef * (lse - logit[target]) with the
    last position of every sequence unlabelled, and dlogits = coef (softmax -
    onehot) written over the logits.  The log-sum-exp partials and the target
    logit come from fp32 accumulators: per-position loss within 1e-5
    relative.  bf16: dlogits come from the stored bf16 logits and are stored
    in bf16: per element |err| <= 1e-2 |ref| + 2e-3 max|row|.  fp32: 1e-5."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    tr = _trainer(cfg)
    T, d, V, S = cfg.tokens_per_micro, cfg.d_model, cfg.vocab, cfg.seq
    bf = cfg.precision == "bf16"
    rf = mi.normal_operand((T, d), 400, 1.0, bf16=bf)
    w = mi.normal_operand((V, d), 401, 0.02, bf16=bf)
    tr.view(tr.params, "lm_head").copy_(torch.as_tensor(w))
    tr.sync_shadow()
    tok = mi.make_tokens(cfg, 0)
    dt = _opdtype(cfg)
    _put(tr, B.MT_VIEW_FINAL_NORM, 0, rf, dt)
    tr.debug_run(B.MT_OP_LM_CE, 0, tokens=torch.as_tensor(tok).cuda())
    out = _ok(tr)
    tl = to_np(tr.debug_view(B.MT_VIEW_TOK_LOSS))
    dl = tr.debug_view(B.MT_VIEW_LOGITS, 0, dt).view(T, V)
    coef = 1.0 / (cfg.batch * (S - 1))
    assert out.loss == pytest.approx(float(np.sum(tl)), rel=1e-6)
    flat = tok.reshape(-1)
    rows = _ce_rows(cfg)
    got = to_np(dl[torch.as_tensor(rows).cuda()])
    W = w.astype(np.float64)
    total = 0.0
    for i, t in enumerate(rows):
        logits = rf[t].astype(np.float64) @ W.T
        m = logits.max()
        lse = m + math.log(np.sum(np.exp(logits - m)))
        p = np.exp(logits - lse)
        if t % S == S - 1:                          # no target
            assert tl[t] == 0.0 and not np.any(got[i])
            continue
        tgt = flat[t + 1]
        ref_loss = coef * (lse - logits[tgt])
        assert abs(tl[t] - ref_loss) <= 1e-5 * abs(ref_loss), (t, tl[t], ref_loss)
        ref = coef * p
        ref[tgt] -= coef
        if bf:
            assert np.all(np.abs(got[i] - ref) <= 1e-2 * np.abs(ref) + 2e-3 * np.abs(ref).max()), t
        else:
            assert rel_l2(got[i], ref) < 1e-5, t
        total += ref_loss
    if len(rows) == T:                              # every position evaluated
        assert out.loss == pytest.approx(total, rel=1e-5)


@pytest.mark.parametrize("name", CASES)
def test_clip_adamw(name):
    """n = ||g||, c = min(1, clip / (n + 1e-6)), decoupled decay, bias-corrected
    AdamW at step t = 3, over every parameter (the flat buffer as one
    tensor), with the fp32 hyperparameters the C ABI carries.  fp32
    arithmetic with a fast division: m and v within 5e-7 of their two terms,
    p within 2.4e-7 of the decayed weight plus the Adam step's relative error
    (1e-6 plus what it inherits from m and v), n and c within 1e-6, and the
    bf16 shadow is the round-to-nearest-even copy of p."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    tr = _trainer(cfg)
    n = tr.n_params
    gstd = 1.2 * cfg.clip_norm / math.sqrt(n)        # norm ~1.2 x clip: the clip is active
    p0 = mi.normal_operand((n,), 500, 0.02)
    g0 = mi.normal_operand((n,), 501, gstd)
    m0 = mi.normal_operand((n,), 502, 0.5 * gstd)
    v0 = mi.normal_operand((n,), 503, gstd) ** 2
    for buf, arr in ((tr.params, p0), (tr.grads, g0), (tr.adam_m, m0), (tr.adam_v, v0)):
        buf.copy_(torch.as_tensor(arr))
    tr.debug_run(B.MT_OP_CLIP_ADAMW, 0, step=3)
    out = _ok(tr)
    # the C ABI carries the hyperparameters in fp32 (beta2 = 0.95f, ...): the
    # oracle takes those same values
    f32 = lambda x: float(np.float32(x))
    hyp = dict(lr=f32(cfg.lr), beta1=f32(cfg.beta1), beta2=f32(cfg.beta2), eps=f32(cfg.eps),
               weight_decay=f32(cfg.weight_decay), clip_norm=f32(cfg.clip_norm), clip_eps=f32(cfg.clip_eps))
    ref_p, ref_m, ref_v, norm, c = oracle.clip_adamw(
        {"all": p0.astype(np.float64)}, {"all": g0}, {"all": m0}, {"all": v0}, step=3, **hyp)
    assert out.grad_norm == pytest.approx(norm, rel=1e-6)
    assert out.clip_coef == pytest.approx(c, rel=1e-6)
    assert c < 1.0
    p = tr.params.cpu().numpy().astype(np.float64)
    m = tr.adam_m.cpu().numpy().astype(np.float64)
    v = tr.adam_v.cpu().numpy().astype(np.float64)
    b1, b2 = hyp["beta1"], hyp["beta2"]
    cg = c * g0.astype(np.float64)
    ref_p, ref_m, ref_v = ref_p["all"], ref_m["all"], ref_v["all"]
    # m and v: a few fp32 roundings of their two terms
    tm = b1 * np.abs(m0) + (1 - b1) * np.abs(cg)
    tv = b2 * v0 + (1 - b2) * cg * cg
    assert np.all(np.abs(m - ref_m) <= 5e-7 * tm + 1e-30)
    assert np.all(np.abs(v - ref_v) <= 5e-7 * tv + 1e-30)
    # p: the decayed weight's rounding plus the Adam step's relative error,
    # which inherits m's and v's (large where their terms cancel)
    decayed = p0.astype(np.float64) * (1.0 - hyp["lr"] * hyp["weight_decay"])
    step = decayed - ref_p
    rel_step = 1e-6 + 6e-7 * tm / np.maximum(np.abs(ref_m), 1e-300) + 3e-7 * tv / np.maximum(ref_v, 1e-300)
    assert np.all(np.abs(p - ref_p) <= 2.4e-7 * np.abs(decayed) + rel_step * np.abs(step) + 1e-12)
    if tr.shadow is not None:
        assert torch.equal(tr.shadow, tr.params.bfloat16())
