"""Pins of the CPU oracle to facts other than itself: the pages' worked
example, closed forms, library routines, finite differences, brute force and
invariants.  All CPU-only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def tiny(**kw):
    return mi.get_config("tiny", **kw)


# --------------------------------------------------------------------------
# "How a training megakernel works", section "One training update"
# --------------------------------------------------------------------------
def test_worked_example_matches_page():
    g = json.load(open(os.path.join(GOLD, "worked_example.json")))
    r = oracle.worked_example(**g["inputs"])
    for key, val in g["printed"].items():
        if key == "L_after_printed":
            assert abs(r["L_after"] - val) < 5e-6          # printed rounded to 2 s.f.
        else:
            assert r[key] == pytest.approx(val, abs=1e-15), key
    assert r["L_after"] == pytest.approx(g["exact"]["L_after"], rel=1e-12)


# --------------------------------------------------------------------------
# Elementary steps against library routines and closed forms
# --------------------------------------------------------------------------
def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(0)
    x, g = rng.normal(size=(7, 48)), rng.normal(size=48)
    y, _ = oracle.rmsnorm(x, g, 1e-5)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (48,), torch.tensor(g), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13, atol=1e-14)


def test_rmsnorm_backward_matches_autograd():
    rng = np.random.default_rng(1)
    x, g, dy = rng.normal(size=(5, 32)), rng.normal(size=32), rng.normal(size=(5, 32))
    y, inv = oracle.rmsnorm(x, g, 1e-5)
    dx, dg = oracle.rmsnorm_backward(dy, x, inv, g)
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(g, requires_grad=True)
    torch.nn.functional.rms_norm(xt, (32,), gt, eps=1e-5).backward(torch.tensor(dy))
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-11, atol=1e-13)


def test_causal_attention_matches_sdpa():
    rng = np.random.default_rng(2)
    q, k, v = (rng.normal(size=(2, 3, 20, 16)) for _ in range(3))
    o = oracle.causal_attention(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=True)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_causal_attention_backward_matches_autograd():
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.normal(size=(1, 2, 17, 8)) for _ in range(4))
    dq, dk, dv = oracle.causal_attention_backward(do, q, k, v)
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True).backward(
        torch.tensor(do))
    for a, b in ((dq, qt), (dk, kt), (dv, vt)):
        np.testing.assert_allclose(a, b.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_causal_logsumexp_matches_torch():
    rng = np.random.default_rng(22)
    q, k = rng.normal(size=(9, 16)), rng.normal(size=(9, 16))
    lse = oracle.causal_logsumexp(q, k)
    s = torch.tensor(q @ k.T / 4.0)
    s = s.masked_fill(~torch.tril(torch.ones(9, 9, dtype=torch.bool)), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), rtol=1e-14)
    # p = exp(s - lse) is the oracle's softmax
    p = oracle.moe_oracle._causal_probs(q, k)
    np.testing.assert_allclose(p, np.exp(s.numpy() - lse[:, None]), rtol=1e-12, atol=1e-300)


def test_first_query_attends_only_to_itself():
    rng = np.random.default_rng(4)
    q, k, v = (rng.normal(size=(1, 1, 9, 4)) for _ in range(3))
    o = oracle.causal_attention(q, k, v)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], rtol=0, atol=1e-15)


def test_rope_properties():
    """Rotation: preserves pair norms; q.k after rotation depends only on the
    position difference; rope_backward inverts rope."""
    hd, S = 16, 40
    cos, sin = oracle.rope_tables(S, hd, 1e4)
    rng = np.random.default_rng(5)
    a, b = rng.normal(size=hd), rng.normal(size=hd)
    A = oracle.rope(np.tile(a, (S, 1)), cos, sin)
    Bm = oracle.rope(np.tile(b, (S, 1)), cos, sin)
    np.testing.assert_allclose(np.linalg.norm(A, axis=1), np.linalg.norm(a), rtol=1e-13)
    dots = A @ Bm.T
    for delta in (0, 3, 11):
        diag = np.array([dots[i + delta, i] for i in range(S - delta)])
        np.testing.assert_allclose(diag, diag[0], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(oracle.rope_backward(A, cos, sin), np.tile(a, (S, 1)), atol=1e-13)
    # position 0 is the identity; angle of pair i at position 1 is theta^(-2i/hd)
    np.testing.assert_allclose(A[0], a, atol=1e-15)
    i = 3
    ang = 1e4 ** (-2 * i / hd)
    assert A[1, i] == pytest.approx(a[i] * math.cos(ang) - a[i + hd // 2] * math.sin(ang))


def test_silu_against_torch():
    g = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(oracle.silu(g), torch.nn.functional.silu(torch.tensor(g)).numpy(),
                               rtol=1e-14, atol=1e-15)
    gt = torch.tensor(g, requires_grad=True)
    torch.nn.functional.silu(gt).sum().backward()
    np.testing.assert_allclose(oracle.silu_grad(g), gt.grad.numpy(), rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------
# token_topk and route_order: brute force and textbook stable sort
# --------------------------------------------------------------------------
@pytest.mark.parametrize("E,K", [(4, 2), (16, 2), (32, 8), (5, 5)])
def test_token_topk_brute_force(E, K):
    rng = np.random.default_rng(E * 100 + K)
    z = rng.integers(-3, 3, size=(300, E)).astype(np.float32)   # many exact ties
    z[:100] = rng.normal(size=(100, E)).astype(np.float32)
    idx, w, p = oracle.token_topk(z, K)
    for t in range(z.shape[0]):
        brute = sorted(range(E), key=lambda e: (-float(z[t, e]), e))[:K]
        assert list(idx[t]) == brute
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)        # slot 0 is the largest weight


def test_route_order_is_stable_counting_sort():
    rng = np.random.default_rng(7)
    for E, K, T in ((4, 2, 64), (16, 2, 500), (32, 8, 300)):
        z = rng.normal(size=(T, E)).astype(np.float32)
        idx, _, _ = oracle.token_topk(z, K)
        perm, counts, offsets, inv = oracle.route_order(idx, E)
        flat = idx.reshape(-1)
        np.testing.assert_array_equal(perm, np.argsort(flat, kind="stable"))
        np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
        assert offsets[-1] == T * K and np.all(np.diff(offsets) == counts)
        np.testing.assert_array_equal(inv[perm], np.arange(T * K))
        assert counts.sum() == T * K


# --------------------------------------------------------------------------
# Clip + AdamW: library routine, closed forms
# --------------------------------------------------------------------------
def _hp(**kw):
    base = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                clip_norm=1.0, clip_eps=1e-6)
    base.update(kw)
    return base


def test_clip_adamw_matches_torch_over_steps():
    rng = np.random.default_rng(8)
    shapes = {"a": (5, 7), "b": (11,), "c": (3, 2, 4)}
    p = {k: rng.normal(size=s) for k, s in shapes.items()}
    m = {k: np.zeros(s) for k, s in shapes.items()}
    v = {k: np.zeros(s) for k, s in shapes.items()}
    tp = [torch.tensor(p[k], requires_grad=True) for k in shapes]
    opt = torch.optim.AdamW(tp, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    for step in range(1, 5):
        scale = [0.3, 3.0, 0.05, 10.0][step - 1]       # some steps clip, some do not
        g = {k: scale * rng.normal(size=s) for k, s in shapes.items()}
        p, m, v, n, c = oracle.clip_adamw(p, g, m, v, step=step, **_hp())
        for t, k in zip(tp, shapes):
            t.grad = torch.tensor(g[k])
        tn = torch.nn.utils.clip_grad_norm_(tp, 1.0)
        assert n == pytest.approx(float(tn), rel=1e-13)
        opt.step()
        for t, k in zip(tp, shapes):
            np.testing.assert_allclose(p[k], t.detach().numpy(), rtol=1e-12, atol=1e-15)


def test_adamw_first_step_closed_form():
    """With m = v = 0 and t = 1 the bias corrections cancel:
    p1 = p0 (1 - lr wd) - lr * g' / (|g'| + eps), g' = c g."""
    rng = np.random.default_rng(9)
    p0 = {"w": rng.normal(size=100)}
    g = {"w": rng.normal(size=100) * 0.01}
    z = {"w": np.zeros(100)}
    hp = _hp(clip_norm=0.05)
    p1, m1, v1, n, c = oracle.clip_adamw(p0, g, z, z, step=1, **hp)
    assert c == pytest.approx(min(1.0, 0.05 / (np.linalg.norm(g["w"]) + 1e-6)))
    gc = c * g["w"]
    expect = p0["w"] * (1 - 1e-4) - 1e-3 * gc / (np.abs(gc) + 1e-8)
    np.testing.assert_allclose(p1["w"], expect, rtol=1e-9, atol=1e-15)
    # ||c g|| = min(n, clip) up to the clip_eps in the denominator
    assert np.linalg.norm(gc) == pytest.approx(min(n, 0.05 * n / (n + 1e-6)), rel=1e-12)


# --------------------------------------------------------------------------
# Whole update on the tiny configuration
# --------------------------------------------------------------------------
@pytest.fixture(scope="module")
def tiny_setup():
    cfg = tiny()
    return cfg, mi.make_params(cfg), mi.make_tokens(cfg, 0)


def test_initial_loss_near_log_vocab(tiny_setup):
    cfg, P, tok = tiny_setup
    loss = oracle.loss_only(P, tok, cfg)
    assert abs(loss - math.log(cfg.vocab)) < 0.05


def test_loss_matches_torch_cross_entropy(tiny_setup):
    cfg, P, tok = tiny_setup
    D = oracle.Dims.of(cfg)
    coef = 1.0 / oracle.n_targets(*tok.shape)
    loss, _, dbg = oracle.forward_backward(oracle.to64(P), tok, D, coef, {}, backward=False)
    logits = torch.tensor(dbg["logits"]).view(cfg.batch, cfg.seq, cfg.vocab)
    ref = torch.nn.functional.cross_entropy(logits[:, :-1].reshape(-1, cfg.vocab),
                                            torch.tensor(tok[:, 1:]).long().reshape(-1))
    assert loss == pytest.approx(float(ref), rel=1e-13)


def test_hand_backward_matches_float64_autograd(tiny_setup):
    from torch_model import grads as autograd_grads
    cfg, P, tok = tiny_setup
    r = oracle.train_update(P, [tok], cfg)
    coef = 1.0 / oracle.n_targets(*tok.shape)
    loss, g = autograd_grads(P, tok, cfg, coef)
    assert r.loss == pytest.approx(loss, rel=1e-12)
    for k in g:
        np.testing.assert_allclose(r.grads[k], g[k], rtol=1e-9, atol=1e-13, err_msg=k)


def test_hand_backward_finite_differences(tiny_setup):
    """Central differences in float64 on sampled coordinates of every tensor,
    plus one random-direction directional derivative over all parameters."""
    cfg, P, tok = tiny_setup
    r = oracle.train_update(P, [tok], cfg)
    P64 = oracle.to64(P)
    rng = np.random.default_rng(10)
    h = 1e-5
    for name, arr in P64.items():
        flat = arr.reshape(-1)
        g = r.grads[name].reshape(-1)
        picks = list(rng.choice(flat.size, size=min(4, flat.size), replace=False))
        picks.append(int(np.argmax(np.abs(g))))
        for i in picks:
            old = flat[i]
            flat[i] = old + h
            lp = oracle.loss_only(P64, tok, cfg)
            flat[i] = old - h
            lm = oracle.loss_only(P64, tok, cfg)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[i]) <= 1e-6 * abs(g[i]) + 2e-9, (name, i, fd, g[i])
    direction = {k: rng.normal(size=v.shape) for k, v in P64.items()}
    eps = 1e-6
    plus = {k: P64[k] + eps * direction[k] for k in P64}
    minus = {k: P64[k] - eps * direction[k] for k in P64}
    fd = (oracle.loss_only(plus, tok, cfg) - oracle.loss_only(minus, tok, cfg)) / (2 * eps)
    an = sum(float(np.sum(r.grads[k] * direction[k])) for k in P64)
    assert fd == pytest.approx(an, rel=1e-6)


def test_accumulation_equals_one_big_batch():
    """Sum of microbatch gradients with coefficient 1/(all targets) equals the
    gradient of the concatenated batch."""
    cfg = tiny(batch=1, micro_count=3)
    P = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    acc = oracle.train_update(P, toks, cfg)
    big = oracle.train_update(P, [np.concatenate(toks, axis=0)], cfg.replace(batch=3, micro_count=1))
    assert acc.loss == pytest.approx(big.loss, rel=1e-12)
    for k in acc.grads:
        np.testing.assert_allclose(acc.grads[k], big.grads[k], rtol=1e-10, atol=1e-15)
    # and evaluating a microbatch one sequence at a time changes nothing
    split = oracle.train_update(P, [np.concatenate(toks, axis=0)], cfg.replace(batch=3, micro_count=1),
                                seqs_per_block=1)
    for k in acc.grads:
        np.testing.assert_allclose(split.grads[k], big.grads[k], rtol=1e-10, atol=1e-15)


def test_causality(tiny_setup):
    """Changing token s leaves every earlier position's loss unchanged except
    position s-1, whose target it is."""
    cfg, P, tok = tiny_setup
    D = oracle.Dims.of(cfg)
    P64 = oracle.to64(P)
    _, tl0, _ = oracle.forward_backward(P64, tok, D, 1.0, {}, backward=False)
    s = 20
    tok2 = tok.copy()
    tok2[0, s] = (tok2[0, s] + 1) % cfg.vocab
    _, tl1, _ = oracle.forward_backward(P64, tok2, D, 1.0, {}, backward=False)
    np.testing.assert_allclose(tl1[:s - 1], tl0[:s - 1], rtol=1e-12, atol=1e-14)
    assert tl1[s - 1] != tl0[s - 1]
    np.testing.assert_allclose(tl1[cfg.seq:], tl0[cfg.seq:], rtol=1e-12, atol=1e-14)


def test_single_expert_is_dense_swiglu():
    """E = 1, K = 1: the expert layer is a dense SwiGLU feed-forward."""
    cfg = tiny(n_experts=1, top_k=1)
    P = oracle.to64(mi.make_params(cfg))
    D = oracle.Dims.of(cfg)
    rng = np.random.default_rng(11)
    r2 = rng.normal(size=(30, cfg.d_model))
    out, c = oracle.moe_forward(r2, 0, P, D)
    g = r2 @ P["w_gate"][0, 0].T
    u = r2 @ P["w_up"][0, 0].T
    ref = (torch.nn.functional.silu(torch.tensor(g)).numpy() * u) @ P["w_down"][0, 0].T
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_all_experts_is_softmax_mixture():
    """K = E: every expert is chosen and the weights are the full softmax."""
    cfg = tiny(n_experts=4, top_k=4)
    P = oracle.to64(mi.make_params(cfg))
    D = oracle.Dims.of(cfg)
    rng = np.random.default_rng(12)
    r2 = rng.normal(size=(25, cfg.d_model))
    out, _ = oracle.moe_forward(r2, 1, P, D)
    p = torch.softmax(torch.tensor(r2 @ P["router"][1].T), dim=-1).numpy()
    ref = np.zeros_like(out)
    for e in range(4):
        h = oracle.silu(r2 @ P["w_gate"][1, e].T) * (r2 @ P["w_up"][1, e].T)
        ref += p[:, e:e + 1] * (h @ P["w_down"][1, e].T)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_unrouted_expert_gets_zero_gradient():
    """An expert no token is routed to receives exactly zero gradient, and its
    router row only receives gradient through nothing (dz is zero off the
    chosen experts)."""
    cfg = tiny()
    P = oracle.to64(mi.make_params(cfg))
    D = oracle.Dims.of(cfg)
    rng = np.random.default_rng(13)
    r2 = np.abs(rng.normal(size=(40, cfg.d_model))) + 1.0   # all entries positive
    P["router"][0, 3, :] = -1.0                               # z_3 = -sum(r2) << 0
    out, c = oracle.moe_forward(r2, 0, P, D)
    assert c["counts"][3] == 0 and c["counts"][:3].sum() == 40 * cfg.top_k
    grads = {k: np.zeros_like(v) for k, v in P.items()}
    dout = rng.normal(size=out.shape)
    oracle.moe_backward(dout, r2, c, 0, P, D, grads)
    for name in ("w_gate", "w_up", "w_down"):
        assert not np.any(grads[name][0, 3])
        for e in range(3):
            assert np.any(grads[name][0, e]) == (c["counts"][e] > 0)
    assert not np.any(grads["router"][0, 3])


# --------------------------------------------------------------------------
# Expert choice made on given router logits (the GPU's, in the parity tests)
# --------------------------------------------------------------------------
def _own_logits(P, tok, cfg):
    D = oracle.Dims.of(cfg)
    _, _, dbg = oracle.forward_backward(oracle.to64(P), tok, D, 1.0, {}, keep_cache=True,
                                        backward=False)
    return [c["moe"]["z"] for c in dbg["caches"]]


def test_route_logits_equal_to_own_logits_change_nothing(tiny_setup):
    cfg, P, tok = tiny_setup
    own = oracle.train_update(P, [tok], cfg)
    forced = oracle.train_update(P, [tok], cfg, route_logits=[_own_logits(P, tok, cfg)])
    assert forced.loss == own.loss
    for k in own.grads:
        np.testing.assert_array_equal(forced.grads[k], own.grads[k], err_msg=k)
        np.testing.assert_array_equal(forced.params[k], own.params[k], err_msg=k)


def test_route_logits_choose_experts_and_backward_matches_finite_differences(tiny_setup):
    """With other logits deciding the choice, (1) each layer's chosen experts
    are token_topk of those logits, (2) the weights are the oracle's own
    probabilities renormalised over that choice, and (3) the hand backward is
    the derivative of the loss with that choice held fixed (central
    differences in float64)."""
    cfg, P, tok = tiny_setup
    D = oracle.Dims.of(cfg)
    rng = np.random.default_rng(21)
    T = tok.size
    rz = [rng.normal(size=(T, cfg.n_experts)) for _ in range(cfg.n_layers)]
    own_z = _own_logits(P, tok, cfg)
    P64 = oracle.to64(P)
    _, _, dbg = oracle.forward_backward(P64, tok, D, 1.0, {}, keep_cache=True, backward=False,
                                        route_logits=rz)
    n_diff = 0
    for l, c in enumerate(dbg["caches"]):
        idx, _, _ = oracle.token_topk(rz[l], cfg.top_k)
        np.testing.assert_array_equal(c["moe"]["idx"], idx)
        own_idx, _, _ = oracle.token_topk(own_z[l] if l == 0 else c["moe"]["z"], cfg.top_k)
        n_diff += int(np.sum(np.any(np.sort(own_idx, 1) != np.sort(idx, 1), axis=1)))
        p = oracle.softmax(c["moe"]["z"])
        pk = np.take_along_axis(p, idx, axis=1)
        np.testing.assert_allclose(c["moe"]["w"], pk / pk.sum(1, keepdims=True), rtol=1e-14)
    assert n_diff > T // 2          # the given logits really change the choices
    r = oracle.train_update(P, [tok], cfg, route_logits=[rz])
    h = 1e-5
    for name, arr in P64.items():
        flat = arr.reshape(-1)
        g = r.grads[name].reshape(-1)
        picks = list(rng.choice(flat.size, size=min(3, flat.size), replace=False))
        picks.append(int(np.argmax(np.abs(g))))
        for i in picks:
            old = flat[i]
            flat[i] = old + h
            lp = oracle.loss_only(P64, tok, cfg, route_logits=rz)
            flat[i] = old - h
            lm = oracle.loss_only(P64, tok, cfg, route_logits=rz)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[i]) <= 1e-6 * abs(g[i]) + 2e-9, (name, i, fd, g[i])


def test_pooled_oracle_equals_serial_oracle():
    """The tests' process-pool evaluation of the oracle (one block of
    sequences per worker, gradients summed, one clip + AdamW) gives the serial
    oracle's update."""
    from parity_util import pooled_oracle_update
    cfg = tiny(batch=3, micro_count=2)
    P = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    serial = oracle.train_update(P, toks, cfg)
    pooled = pooled_oracle_update(cfg, toks, workers=2)
    assert pooled.loss == pytest.approx(serial.loss, rel=1e-13)
    assert pooled.grad_norm == pytest.approx(serial.grad_norm, rel=1e-13)
    for k in serial.grads:
        np.testing.assert_allclose(pooled.grads[k], serial.grads[k], rtol=1e-11, atol=1e-16)
        # Adam divides by sqrt(v): summation-order rounding of tiny gradients is amplified
        np.testing.assert_allclose(pooled.params[k], serial.params[k], rtol=1e-9, atol=1e-16)
    for a, b in zip(pooled.tok_loss, serial.tok_loss):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-16)


# --------------------------------------------------------------------------
# Selective updates: the two special cases are plain updates
# --------------------------------------------------------------------------
def test_selective_all_experts_is_gradient_accumulation():
    """With every tensor in the expert group nothing updates until the end,
    and the step on the mean gradient is the accumulated update's step."""
    cfg = tiny(batch=1, micro_count=3)
    P = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    acc = oracle.train_update(P, toks, cfg)
    sel = oracle.selective_updates(P, toks, cfg, expert_names=tuple(P))
    for k in P:
        # coefficient 1/31 per microbatch, then / 3, against 1/93: rounding only
        np.testing.assert_allclose(sel.expert_grads[k] / 3, acc.grads[k], rtol=1e-10, atol=1e-16)
        np.testing.assert_allclose(sel.params[k], acc.params[k], rtol=1e-9, atol=1e-15)
    assert sel.expert_norm == pytest.approx(acc.grad_norm, rel=1e-12)


def test_selective_all_shared_is_one_update_per_microbatch():
    """With no expert group every microbatch is one whole update at step
    index 1, 2, 3 with the state carried over."""
    cfg = tiny(batch=1, micro_count=3)
    P = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    sel = oracle.selective_updates(P, toks, cfg, expert_names=())
    st, m, v = P, None, None
    for i, t in enumerate(toks):
        r = oracle.train_update(st, [t], cfg.replace(micro_count=1, step=i + 1), m=m, v=v)
        st, m, v = r.params, r.m, r.v
        assert sel.losses[i] == pytest.approx(r.loss, rel=1e-12)
        assert sel.shared_norms[i] == pytest.approx(r.grad_norm, rel=1e-12)
    for k in P:
        np.testing.assert_allclose(sel.params[k], st[k], rtol=1e-12, atol=1e-16)


def test_selective_first_shared_step_and_expert_step():
    """The first microbatch's shared step is the plain single-microbatch
    update's step on those tensors (clipping off: the norm is then over
    different sets but unused), and the expert step is one AdamW step at
    t = 1 on the mean of the period's expert gradients: with clipping off,
    -lr * sign(mean g) - lr * wd * p up to eps."""
    cfg = tiny(batch=1, micro_count=3, clip_norm=1e6)
    P = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    one = oracle.selective_updates(P, toks[:1], cfg)
    plain = oracle.train_update(P, toks[:1], cfg.replace(micro_count=1))
    for k in P:
        if k not in oracle.EXPERT_TENSORS:
            np.testing.assert_allclose(one.params[k], plain.params[k], rtol=1e-12, atol=1e-16)
    full = oracle.selective_updates(P, toks, cfg)
    for k in oracle.EXPERT_TENSORS:
        g = full.expert_grads[k] / 3
        p0 = P[k].astype(np.float64)
        expect = p0 * (1 - cfg.lr * cfg.weight_decay) - cfg.lr * g / (np.abs(g) + cfg.eps)
        np.testing.assert_allclose(full.params[k], expect, rtol=1e-9, atol=1e-15)
        # and differs from stepping on the sum by the eps term only where |g| ~ eps
        assert np.any(full.expert_grads[k])


# --------------------------------------------------------------------------
# Looped model: repeated layers share weights, gradients add over visits
# --------------------------------------------------------------------------
def test_looped_model_is_the_unrolled_model_with_tied_weights():
    """A model of U distinct layers visited L times equals the L-layer model
    whose layer l holds a copy of slot l mod U: same loss, and each slot's
    gradient is the sum of the unrolled layers' gradients over its visits."""
    cfg = tiny(n_layers=4, n_unique_layers=2)
    P = mi.make_params(cfg)
    tok = mi.make_tokens(cfg, 0)
    looped = oracle.train_update(P, [tok], cfg)
    unrolled_cfg = cfg.replace(n_unique_layers=0)
    U = {k: (np.stack([v[l % 2] for l in range(4)]) if v.ndim >= 2 and k not in ("emb", "lm_head") else v)
         for k, v in P.items()}
    un = oracle.train_update(U, [tok], unrolled_cfg)
    assert looped.loss == pytest.approx(un.loss, rel=1e-13)
    for k, g in looped.grads.items():
        if k in ("emb", "lm_head", "final_norm"):
            np.testing.assert_allclose(g, un.grads[k], rtol=1e-11, atol=1e-16)
        else:
            # visits 0, 2 use slot 0 and visits 1, 3 slot 1
            np.testing.assert_allclose(g, un.grads[k][0:2] + un.grads[k][2:4], rtol=1e-10, atol=1e-15, err_msg=k)


def test_looped_backward_finite_differences():
    """Central differences on the looped model (one layer visited twice)."""
    cfg = tiny(n_layers=2, n_unique_layers=1)
    P = oracle.to64(mi.make_params(cfg))
    tok = mi.make_tokens(cfg, 0)
    r = oracle.train_update(P, [tok], cfg)
    rng = np.random.default_rng(31)
    h = 1e-5
    for name in ("wqkv", "wo", "moe_norm", "router", "w_gate", "w_down", "attn_norm"):
        flat = P[name].reshape(-1)
        g = r.grads[name].reshape(-1)
        for i in [int(np.argmax(np.abs(g))), *rng.choice(flat.size, size=2, replace=False)]:
            old = flat[i]
            flat[i] = old + h
            lp = oracle.loss_only(P, tok, cfg)
            flat[i] = old - h
            lm = oracle.loss_only(P, tok, cfg)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[i]) <= 1e-6 * abs(g[i]) + 2e-9, (name, i, fd, g[i])
