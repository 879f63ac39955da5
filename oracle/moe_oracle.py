"""Plain, slow CPU oracle (NumPy, float64) for one MoE training update.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  It shares no code, table or constant
generator with the CUDA library; it reads the same seeded fp32 weights and
int32 tokens (``moe_inputs``) and upcasts them to float64.

What it computes follows the Latch pages:

* "How a training megakernel works", section "One training update": a
  training update is forward pass -> loss -> backward pass (chain rule) ->
  optimizer step; the two-weight example of that section is
  :func:`worked_example`.
* same page, "From two weights to 200 million": TinyMoE is attention plus
  expert layers in which a router sends each token to two of sixteen small
  feed-forward networks; AdamW keeps running averages of the gradients and
  of their squares.
* same page, "1 - Describe the model and update": the custom operations are
  bf16 attention (:func:`causal_attention`), ``token_topk``
  (:func:`token_topk`), ``route_order`` (:func:`route_order`) and
  ``ragged_mm`` (the per-expert products inside :func:`moe_forward`);
  global-norm clipping and AdamW are plain tensor arithmetic
  (:func:`clip_adamw`).
* same page, "2 - Capture ...": the objective takes ``(labels,
  coefficients)`` -- read here as next-token labels with one coefficient per
  target equal to 1 / (number of targets in the whole update).
* same page, "How GPUs usually run it": gradients of all microbatches of the
  published batch are summed before the one optimizer update.

Every function below is the plain definition of its step: there is no
blocking, fusion or reordering beyond looping over experts, (batch, head)
pairs and independent sequences.  The backward pass is derived by hand and
checked against finite differences and float64 autograd in the tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F64 = np.float64


# ---------------------------------------------------------------------------
# The pages' two-weight example ("How a training megakernel works",
# section "One training update").
# ---------------------------------------------------------------------------
def worked_example(x=2.0, t=1.0, w1=0.5, w2=1.5, eta=0.1) -> dict:
    """h = w1*x, y = w2*h, L = (y - t)^2 / 2, hand backprop, one SGD step."""
    h = w1 * x
    y = w2 * h
    L = 0.5 * (y - t) ** 2
    dL_dy = y - t
    dL_dw2 = dL_dy * h
    dL_dh = dL_dy * w2
    dL_dw1 = dL_dh * x
    w1_new = w1 - eta * dL_dw1
    w2_new = w2 - eta * dL_dw2
    h2 = w1_new * x
    y2 = w2_new * h2
    L2 = 0.5 * (y2 - t) ** 2
    return dict(h=h, y=y, L=L, dL_dy=dL_dy, dL_dw2=dL_dw2, dL_dh=dL_dh,
                dL_dw1=dL_dw1, w1_new=w1_new, w2_new=w2_new, h_after=h2,
                y_after=y2, L_after=L2)


# ---------------------------------------------------------------------------
# Elementary steps
# ---------------------------------------------------------------------------
def rmsnorm(x, g, eps):
    """y = x / sqrt(mean(x^2) + eps) * g over the last axis; returns (y, inv)."""
    inv = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x * inv * g, inv


def rmsnorm_backward(dy, x, inv, g):
    """Gradients of y = x*inv*g: returns (dx, dg) with dg summed over rows.

    With a = dy*g and xh = x*inv:  dx = inv * (a - xh * mean(a*xh)).
    """
    xh = x * inv
    a = dy * g
    dx = inv * (a - xh * np.mean(a * xh, axis=-1, keepdims=True))
    dg = np.sum(dy * xh, axis=0)
    return dx, dg


def rope_tables(seq, head_dim, theta):
    """Angles pos * theta^(-2i/head_dim) for pos < seq, i < head_dim/2."""
    half = head_dim // 2
    pos = np.arange(seq, dtype=F64)[:, None]
    freq = theta ** (-2.0 * np.arange(half, dtype=F64) / head_dim)
    ang = pos * freq[None, :]
    return np.cos(ang), np.sin(ang)


def rope(x, cos, sin):
    """Rotate-half rotary embedding on the last axis of x [..., S, hd]:
    pair (i, i + hd/2) is rotated by the angle of (pos, i)."""
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def rope_backward(dy, cos, sin):
    """Transpose of :func:`rope` (rotation by the negative angle)."""
    half = dy.shape[-1] // 2
    d1, d2 = dy[..., :half], dy[..., half:]
    return np.concatenate([d1 * cos + d2 * sin, d2 * cos - d1 * sin], axis=-1)


def _causal_probs(q, k):
    """Softmax of q k^T / sqrt(hd) with keys j <= query i, for one (b, h)."""
    S, hd = q.shape
    s = (q @ k.T) / math.sqrt(hd)
    s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=1, keepdims=True)


def causal_attention(q, k, v):
    """o = softmax(q k^T / sqrt(hd) + causal mask) v for q,k,v [B, H, S, hd]."""
    B, H, S, hd = q.shape
    o = np.empty_like(q)
    for b in range(B):
        for h in range(H):
            o[b, h] = _causal_probs(q[b, h], k[b, h]) @ v[b, h]
    return o


def causal_logsumexp(q, k):
    """Row log-sum-exp of the scaled causal scores q k^T / sqrt(hd) (keys
    j <= i) for one (batch, head): the normaliser of the attention softmax."""
    S, hd = q.shape
    s = (q @ k.T) / math.sqrt(hd)
    s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    m = s.max(axis=1)
    return m + np.log(np.sum(np.exp(s - m[:, None]), axis=1))


def causal_attention_backward(do, q, k, v):
    """Gradients of :func:`causal_attention` wrt q, k, v (P recomputed)."""
    B, H, S, hd = q.shape
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    scale = 1.0 / math.sqrt(hd)
    for b in range(B):
        for h in range(H):
            p = _causal_probs(q[b, h], k[b, h])
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            ds = p * (dp - np.sum(dp * p, axis=1, keepdims=True))
            dq[b, h] = (ds @ k[b, h]) * scale
            dk[b, h] = (ds.T @ q[b, h]) * scale
    return dq, dk, dv


def softmax(z, axis=-1):
    z = z - z.max(axis=axis, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=axis, keepdims=True)


def silu(g):
    return g / (1.0 + np.exp(-g))


def silu_grad(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


# ---------------------------------------------------------------------------
# Routing: token_topk and route_order ("1 - Describe the model and update")
# ---------------------------------------------------------------------------
def token_topk(z, k):
    """Top-k experts per token from router logits z [T, E].

    p = softmax(z); the k largest p in descending order, equal values going
    to the lower expert index (slot 0 = best).  softmax is strictly monotone,
    so ordering by z is ordering by p.  Weights are renormalised over the k
    chosen experts: w_j = p_j / sum_chosen p.  Returns (idx int32 [T,k],
    w float64 [T,k], p float64 [T,E]).
    """
    p = softmax(z.astype(F64))
    order = np.argsort(-z, axis=1, kind="stable")   # stable: ties keep lower index first
    idx = order[:, :k].astype(np.int32)
    pk = np.take_along_axis(p, idx, axis=1)
    w = pk / pk.sum(axis=1, keepdims=True)
    return idx, w, p


def route_order(idx, n_experts):
    """Expert-sorted order of the T*k assignments a = t*k + slot.

    A stable counting sort by expert: within an expert, assignments keep
    ascending a.  Returns (perm [T*k] assignment at each sorted position,
    counts [E], offsets [E+1] unpadded, inv [T*k] sorted position of each
    assignment).
    """
    flat = idx.reshape(-1).astype(np.int64)
    counts = np.zeros(n_experts, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(n_experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = offsets[:-1].copy()
    perm = np.empty(flat.size, dtype=np.int64)
    inv = np.empty(flat.size, dtype=np.int64)
    for a, e in enumerate(flat):
        perm[fill[e]] = a
        inv[a] = fill[e]
        fill[e] += 1
    return perm, counts, offsets, inv


# ---------------------------------------------------------------------------
# Model
# ---------------------------------------------------------------------------
@dataclass
class Dims:
    vocab: int
    d: int
    L: int
    H: int
    hd: int
    E: int
    K: int
    F: int
    eps: float
    theta: float
    U: int = 0          # looped model: distinct layers; visit l uses weights l mod U (0: U = L)

    @staticmethod
    def of(cfg) -> "Dims":
        return Dims(cfg.vocab, cfg.d_model, cfg.n_layers, cfg.n_heads, cfg.head_dim,
                    cfg.n_experts, cfg.top_k, cfg.d_ff, cfg.norm_eps, cfg.rope_theta,
                    getattr(cfg, "n_unique_layers", 0))

    def slot(self, l: int) -> int:
        """Weights of layer visit l ("Results", "Other measured compiler work":
        the looped model's repeated layers share weights; gradients of a
        slot accumulate over its visits)."""
        return l % (self.U or self.L)


def to64(params: dict) -> dict:
    return {k: np.asarray(v, dtype=F64) for k, v in params.items()}


def moe_forward(r2, l, P, D: Dims, route_z=None):
    """Router, top-k, route_order and the per-expert SwiGLU products of one
    expert layer (weights of layer slot l).  Returns the weighted combination
    [T, d] and a cache.

    ``route_z`` (optional, [T, E]): logits on which the top-k *choice* is made
    instead of this layer's own logits.  The weights are still the oracle's
    own softmax probabilities of the chosen experts, renormalised over them,
    so only the discrete choice comes from ``route_z``.  This is the check
    the pages' routing statement implies ("token_topk" then "route_order" on a
    given set of router logits): with another implementation's logits the
    oracle reproduces that implementation's expert choices, and every other
    step stays the plain fp64 definition.
    """
    T = r2.shape[0]
    z = r2 @ P["router"][l].T                        # [T, E]
    idx, w, p = token_topk(z, D.K)
    if route_z is not None:
        idx, _, _ = token_topk(np.asarray(route_z), D.K)
        pk = np.take_along_axis(p, idx, axis=1)
        w = pk / pk.sum(axis=1, keepdims=True)
    perm, counts, offsets, inv = route_order(idx, D.E)
    xs = r2[perm // D.K]                              # rows in expert order
    g = np.zeros((T * D.K, D.F))
    u = np.zeros((T * D.K, D.F))
    a = np.zeros((T * D.K, D.F))
    y = np.zeros((T * D.K, D.d))
    for e in range(D.E):
        rows = slice(offsets[e], offsets[e + 1])
        g[rows] = xs[rows] @ P["w_gate"][l, e].T
        u[rows] = xs[rows] @ P["w_up"][l, e].T
        a[rows] = silu(g[rows]) * u[rows]
        y[rows] = a[rows] @ P["w_down"][l, e].T
    inv_tk = inv.reshape(T, D.K)
    out = np.zeros((T, D.d))
    for s in range(D.K):                              # fixed slot order
        out += w[:, s:s + 1] * y[inv_tk[:, s]]
    cache = dict(z=z, idx=idx, w=w, perm=perm, counts=counts, offsets=offsets,
                 inv=inv, xs=xs, g=g, u=u, a=a, y=y)
    return out, cache


def moe_backward(dout, r2, c, l, P, D: Dims, grads):
    """Backward of :func:`moe_forward`; returns d r2 and adds weight grads."""
    T = r2.shape[0]
    inv_tk = c["inv"].reshape(T, D.K)
    w = c["w"]
    dy = np.zeros_like(c["y"])
    dw = np.zeros((T, D.K))
    for s in range(D.K):
        rows = inv_tk[:, s]
        dy[rows] = w[:, s:s + 1] * dout
        dw[:, s] = np.sum(dout * c["y"][rows], axis=1)
    dxs = np.zeros_like(c["xs"])
    for e in range(D.E):
        rows = slice(c["offsets"][e], c["offsets"][e + 1])
        da = dy[rows] @ P["w_down"][l, e]
        grads["w_down"][l, e] += dy[rows].T @ c["a"][rows]
        g, u = c["g"][rows], c["u"][rows]
        dg = da * u * silu_grad(g)
        du = da * silu(g)
        dxs[rows] = dg @ P["w_gate"][l, e] + du @ P["w_up"][l, e]
        grads["w_gate"][l, e] += dg.T @ c["xs"][rows]
        grads["w_up"][l, e] += du.T @ c["xs"][rows]
    dr2 = np.zeros_like(r2)
    for s in range(D.K):                              # direct per-row sum, fixed order
        dr2 += dxs[inv_tk[:, s]]
    # Renormalised weights are the softmax of the chosen logits, so
    # dz_i = w_i (dw_i - sum_j w_j dw_j) on chosen experts and 0 elsewhere.
    dz = np.zeros((T, D.E))
    mean_dw = np.sum(w * dw, axis=1, keepdims=True)
    dz_chosen = w * (dw - mean_dw)
    for s in range(D.K):
        dz[np.arange(T), c["idx"][:, s]] += dz_chosen[:, s]
    grads["router"][l] += dz.T @ r2
    dr2 += dz @ P["router"][l]
    return dr2


def forward_backward(P: dict, tokens: np.ndarray, D: Dims, coef: float, grads: dict,
                     keep_cache: bool = False, backward: bool = True, route_logits=None):
    """Loss of one block of independent sequences and its gradients, added to
    ``grads``.  ``tokens`` is int [B, S]; ``coef`` multiplies every target's
    cross-entropy.  ``route_logits`` (optional) is a per-layer list of [B*S, E]
    logits on which each layer's expert choice is made (see
    :func:`moe_forward`).  Returns (loss, per_token_loss [B*S], debug)."""
    B, S = tokens.shape
    T = B * S
    tok = tokens.reshape(-1)
    cos, sin = rope_tables(S, D.hd, D.theta)

    def heads(t2d):
        return t2d.reshape(B, S, D.H, D.hd).transpose(0, 2, 1, 3)

    def unheads(t4d):
        return t4d.transpose(0, 2, 1, 3).reshape(T, D.H * D.hd)

    hq = D.H * D.hd
    x = P["emb"][tok].copy()
    caches = []
    for l in range(D.L):
        x_in = x
        w = D.slot(l)                                # weights of this layer visit
        r, inv = rmsnorm(x_in, P["attn_norm"][w], D.eps)
        qkv = r @ P["wqkv"][w].T
        q = rope(heads(qkv[:, :hq]), cos, sin)
        k = rope(heads(qkv[:, hq:2 * hq]), cos, sin)
        v = heads(qkv[:, 2 * hq:])
        o = unheads(causal_attention(q, k, v))
        x_mid = x_in + o @ P["wo"][w].T
        r2, inv2 = rmsnorm(x_mid, P["moe_norm"][w], D.eps)
        moe_out, mc = moe_forward(r2, w, P, D,
                                  None if route_logits is None else route_logits[l])
        x = x_mid + moe_out
        caches.append(dict(x_in=x_in, r=r, inv=inv, q=q, k=k, v=v, o=o,
                           x_mid=x_mid, r2=r2, inv2=inv2, moe=mc))
    rf, invf = rmsnorm(x, P["final_norm"], D.eps)
    logits = rf @ P["lm_head"].T                      # [T, V]

    # Next-token cross entropy: position s predicts tok[b, s+1]; the last
    # position of each sequence has no target.
    has_target = np.ones((B, S), dtype=bool)
    has_target[:, -1] = False
    has_target = has_target.reshape(-1)
    target = np.zeros((B, S), dtype=np.int64)
    target[:, :-1] = tokens[:, 1:]
    target = target.reshape(-1)
    m = logits.max(axis=1, keepdims=True)
    lse = (m + np.log(np.sum(np.exp(logits - m), axis=1, keepdims=True)))[:, 0]
    tok_loss = np.where(has_target, coef * (lse - logits[np.arange(T), target]), 0.0)
    loss = float(np.sum(tok_loss))
    if not backward:
        dbg = dict(lse=lse, logits=logits, rf=rf)
        if keep_cache:
            dbg["caches"] = caches
        return loss, tok_loss, dbg
    dlogits = np.exp(logits - lse[:, None])
    dlogits[np.arange(T), target] -= 1.0
    dlogits *= np.where(has_target, coef, 0.0)[:, None]
    del logits

    # ---- backward ------------------------------------------------------
    grads["lm_head"] += dlogits.T @ rf
    drf = dlogits @ P["lm_head"]
    del dlogits
    dx, dgf = rmsnorm_backward(drf, x, invf, P["final_norm"])
    grads["final_norm"] += dgf
    for l in reversed(range(D.L)):
        c = caches[l]
        w = D.slot(l)                                # gradients of a slot add over its visits
        # expert half: x = x_mid + moe(rmsnorm(x_mid))
        dr2 = moe_backward(dx, c["r2"], c["moe"], w, P, D, grads)
        dxm, dg2 = rmsnorm_backward(dr2, c["x_mid"], c["inv2"], P["moe_norm"][w])
        grads["moe_norm"][w] += dg2
        dx = dx + dxm
        # attention half: x_mid = x_in + attn(rmsnorm(x_in)) Wo^T
        grads["wo"][w] += dx.T @ c["o"]
        do = heads(dx @ P["wo"][w])
        dq, dk, dv = causal_attention_backward(do, c["q"], c["k"], c["v"])
        dqkv = np.concatenate([unheads(rope_backward(dq, cos, sin)),
                               unheads(rope_backward(dk, cos, sin)),
                               unheads(dv)], axis=1)
        grads["wqkv"][w] += dqkv.T @ c["r"]
        dr = dqkv @ P["wqkv"][w]
        dxa, dg1 = rmsnorm_backward(dr, c["x_in"], c["inv"], P["attn_norm"][w])
        grads["attn_norm"][w] += dg1
        dx = dx + dxa
    np.add.at(grads["emb"], tok, dx)

    debug = {}
    if keep_cache:
        debug = dict(caches=caches, lse=lse, rf=rf)
    else:
        debug = dict(router=[dict(z=c["moe"]["z"], idx=c["moe"]["idx"], w=c["moe"]["w"],
                                  perm=c["moe"]["perm"], counts=c["moe"]["counts"])
                             for c in caches])
    return loss, tok_loss, debug


# ---------------------------------------------------------------------------
# Optimizer: global-norm clip + AdamW ("1 - Describe the model and update")
# ---------------------------------------------------------------------------
def global_norm(grads: dict) -> float:
    return math.sqrt(sum(float(np.sum(np.asarray(g, F64) ** 2)) for g in grads.values()))


def clip_adamw(params, grads, m, v, *, lr, beta1, beta2, eps, weight_decay,
               clip_norm, clip_eps, step):
    """One clipped AdamW step on float64 copies; returns (p, m, v, norm, coef).

    n = ||g||_2 over every tensor; c = min(1, clip / (n + clip_eps)); g <- c g;
    p <- p (1 - lr wd); m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
    p <- p - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).
    Decoupled weight decay applies to every tensor.
    """
    n = global_norm(grads)
    c = min(1.0, clip_norm / (n + clip_eps))
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    new_p, new_m, new_v = {}, {}, {}
    for name in params:
        g = c * np.asarray(grads[name], F64)
        p = np.asarray(params[name], F64) * (1.0 - lr * weight_decay)
        mm = beta1 * np.asarray(m[name], F64) + (1.0 - beta1) * g
        vv = beta2 * np.asarray(v[name], F64) + (1.0 - beta2) * g * g
        p = p - lr * (mm / bc1) / (np.sqrt(vv / bc2) + eps)
        new_p[name], new_m[name], new_v[name] = p, mm, vv
    return new_p, new_m, new_v, n, c


# ---------------------------------------------------------------------------
# One complete update
# ---------------------------------------------------------------------------
@dataclass
class UpdateResult:
    loss: float
    grads: dict
    grad_norm: float
    clip_coef: float
    params: dict
    m: dict
    v: dict
    tok_loss: list = field(default_factory=list)
    debug: list = field(default_factory=list)


def n_targets(batch, seq) -> int:
    return batch * (seq - 1)


def train_update(params: dict, micro_tokens: list, cfg, m=None, v=None,
                 seqs_per_block: int | None = None, keep_cache=False,
                 route_logits=None) -> UpdateResult:
    """Forward, loss, backward over every microbatch (gradients summed), then
    one clipped AdamW step.

    ``coefficients``: every target of the update weighs 1 / (total targets),
    so the reported loss is the mean next-token cross-entropy of the update.
    ``seqs_per_block`` optionally evaluates a microbatch a few sequences at a
    time; sequences never interact in this model, so the sum is unchanged.
    ``route_logits`` (optional): per microbatch, a per-layer list of
    [batch*seq, E] logits on which the expert choices are made (see
    :func:`moe_forward`).
    """
    D = Dims.of(cfg)
    P = to64(params)
    total_targets = sum(n_targets(*t.shape) for t in micro_tokens)
    coef = 1.0 / total_targets
    grads = {k: np.zeros_like(p) for k, p in P.items()}
    loss = 0.0
    tok_losses, debugs = [], []
    for mi_, tokens in enumerate(micro_tokens):
        B, S = tokens.shape
        step_b = B if seqs_per_block is None else seqs_per_block
        parts = []
        for b0 in range(0, B, step_b):
            rz = None
            if route_logits is not None:
                rows = slice(b0 * S, min(b0 + step_b, B) * S)
                rz = [np.asarray(z)[rows] for z in route_logits[mi_]]
            lo, tl, dbg = forward_backward(P, tokens[b0:b0 + step_b], D, coef, grads,
                                           keep_cache=keep_cache, route_logits=rz)
            loss += lo
            parts.append(tl)
            debugs.append(dbg)
        tok_losses.append(np.concatenate(parts))
    if m is None:
        m = {k: np.zeros_like(p) for k, p in P.items()}
    if v is None:
        v = {k: np.zeros_like(p) for k, p in P.items()}
    new_p, new_m, new_v, n, c = clip_adamw(
        P, grads, m, v, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
        weight_decay=cfg.weight_decay, clip_norm=cfg.clip_norm, clip_eps=cfg.clip_eps,
        step=cfg.step)
    return UpdateResult(loss=loss, grads=grads, grad_norm=n, clip_coef=c, params=new_p,
                        m=new_m, v=new_v, tok_loss=tok_losses, debug=debugs)


def loss_only(params: dict, tokens: np.ndarray, cfg, coef: float | None = None,
              route_logits=None) -> float:
    """Loss of one microbatch (for finite differences)."""
    D = Dims.of(cfg)
    P = to64(params)
    if coef is None:
        coef = 1.0 / n_targets(*tokens.shape)
    loss, _, _ = forward_backward(P, tokens, D, coef, {}, backward=False,
                                  route_logits=route_logits)
    return loss


# ---------------------------------------------------------------------------
# Selective updates (*Results*, "Other measured compiler work": shared weights
# update every microbatch, experts every 16)
# ---------------------------------------------------------------------------
EXPERT_TENSORS = ("w_gate", "w_up", "w_down")


@dataclass
class SelectiveResult:
    params: dict
    m: dict
    v: dict
    losses: list            # loss of each microbatch (mean CE over its targets)
    shared_norms: list      # ||g|| of the shared tensors at each microbatch
    shared_coefs: list
    expert_norm: float      # ||mean expert gradient|| at the end of the period
    expert_coef: float
    shared_grads: dict      # shared gradients of the last microbatch
    expert_grads: dict      # expert gradients summed over the period


def selective_updates(params: dict, micro_tokens: list, cfg, m=None, v=None, step: int = 1,
                      expert_step: int = 1, expert_names=EXPERT_TENSORS,
                      route_logits=None) -> SelectiveResult:
    """One period of selective updates over ``micro_tokens``.

    Every microbatch i: forward and backward at the current weights, every
    target weighing 1 / (targets of the microbatch); the shared tensors (all
    but ``expert_names``) take one clipped AdamW step at step index step + i
    (norm over the shared gradients).  The expert tensors' gradients are
    summed over the microbatches; after the last one the experts take one
    clipped AdamW step at ``expert_step`` on the mean (sum / number of
    microbatches, norm over that mean).
    """
    D = Dims.of(cfg)
    P = to64(params)
    m = {k: np.zeros_like(p) for k, p in P.items()} if m is None else to64(m)
    v = {k: np.zeros_like(p) for k, p in P.items()} if v is None else to64(v)
    shared = [k for k in P if k not in expert_names]
    experts = [k for k in P if k in expert_names]
    hyper = dict(lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
                 weight_decay=cfg.weight_decay, clip_norm=cfg.clip_norm, clip_eps=cfg.clip_eps)
    acc = {k: np.zeros_like(P[k]) for k in experts}
    losses, norms, coefs = [], [], []
    grads = {}
    for i, tokens in enumerate(micro_tokens):
        grads = {k: np.zeros_like(p) for k, p in P.items()}
        coef = 1.0 / n_targets(*tokens.shape)
        rz = None if route_logits is None else route_logits[i]
        loss, _, _ = forward_backward(P, tokens, D, coef, grads, route_logits=rz)
        losses.append(loss)
        for k in experts:
            acc[k] += grads[k]
        if shared:
            sp, sm, sv, n, c = clip_adamw({k: P[k] for k in shared}, {k: grads[k] for k in shared},
                                          {k: m[k] for k in shared}, {k: v[k] for k in shared},
                                          step=step + i, **hyper)
            P.update(sp); m.update(sm); v.update(sv)
            norms.append(n); coefs.append(c)
    n_e, c_e = 0.0, 1.0
    if experts:
        mean = {k: acc[k] / len(micro_tokens) for k in experts}
        ep, em, ev, n_e, c_e = clip_adamw({k: P[k] for k in experts}, mean, {k: m[k] for k in experts},
                                          {k: v[k] for k in experts}, step=expert_step, **hyper)
        P.update(ep); m.update(em); v.update(ev)
    return SelectiveResult(params=P, m=m, v=v, losses=losses, shared_norms=norms, shared_coefs=coefs,
                           expert_norm=n_e, expert_coef=c_e,
                           shared_grads={k: grads[k] for k in shared}, expert_grads=acc)
