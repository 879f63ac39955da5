"""An independent float64 PyTorch (CPU) statement of the MoE forward pass,
used only to cross-check the oracle's hand-derived backward through autograd.

It is written from the model definition with library ops (scaled dot-product
attention, rms_norm, silu, cross_entropy, topk) and shares no code with the
oracle.  The routing decision is not differentiable; ``torch.topk`` orders
ties differently from the oracle, so tests use inputs without ties.
"""
import math

import torch
import torch.nn.functional as F


def _rope(x, pos_theta):
    cos, sin = pos_theta
    half = x.shape[-1] // 2
    x1, x2 = x[..., :half], x[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1)


def loss_fn(P, tokens, cfg, coef):
    """Next-token CE of one microbatch times ``coef`` per target (sum)."""
    B, S = tokens.shape
    d, H, hd, E, K = cfg.d_model, cfg.n_heads, cfg.head_dim, cfg.n_experts, cfg.top_k
    tok = torch.as_tensor(tokens, dtype=torch.long)
    pos = torch.arange(S, dtype=torch.float64)[:, None]
    inv_freq = cfg.rope_theta ** (-torch.arange(0, hd, 2, dtype=torch.float64) / hd)
    ang = pos * inv_freq[None, :]
    cs = (torch.cos(ang), torch.sin(ang))
    x = P["emb"][tok]                                   # [B, S, d]
    for l in range(cfg.n_layers):
        r = F.rms_norm(x, (d,), P["attn_norm"][l], eps=cfg.norm_eps)
        qkv = r @ P["wqkv"][l].T
        q, k, v = qkv.split(H * hd, dim=-1)
        q = q.view(B, S, H, hd).transpose(1, 2)
        k = k.view(B, S, H, hd).transpose(1, 2)
        v = v.view(B, S, H, hd).transpose(1, 2)
        q, k = _rope(q, cs), _rope(k, cs)
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        o = o.transpose(1, 2).reshape(B, S, H * hd)
        x = x + o @ P["wo"][l].T
        r2 = F.rms_norm(x, (d,), P["moe_norm"][l], eps=cfg.norm_eps)
        z = r2 @ P["router"][l].T                       # [B, S, E]
        p = torch.softmax(z, dim=-1)
        top_p, top_i = torch.topk(p, K, dim=-1)
        w = top_p / top_p.sum(dim=-1, keepdim=True)
        out = torch.zeros_like(x)
        for e in range(E):
            h = F.silu(r2 @ P["w_gate"][l, e].T) * (r2 @ P["w_up"][l, e].T)
            ye = h @ P["w_down"][l, e].T
            we = (w * (top_i == e)).sum(dim=-1, keepdim=True)
            out = out + we * ye
        x = x + out
    rf = F.rms_norm(x, (d,), P["final_norm"], eps=cfg.norm_eps)
    logits = rf @ P["lm_head"].T
    ce = F.cross_entropy(logits[:, :-1].reshape(-1, cfg.vocab), tok[:, 1:].reshape(-1),
                         reduction="sum")
    return ce * coef


def grads(params_np, tokens, cfg, coef):
    P = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in params_np.items()}
    loss = loss_fn(P, tokens, cfg, coef)
    loss.backward()
    return float(loss), {k: t.grad.numpy() for k, t in P.items()}
