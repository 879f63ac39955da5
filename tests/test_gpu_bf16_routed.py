"""GPU parity of the bf16-product configurations with the expert choices
taken from the GPU's own router logits.

The oracle runs live (float64, a pool of worker processes) and makes each
layer's top-k choice on the router logits the GPU computed for that layer -
the check the pages' routing statement implies ("token_topk" and
"route_order" applied to a given set of logits; the GPU's choices on its
logits are checked bit for bit in test_gpu_bf16.py).  Everything else on the
oracle side - the logits used for the weights, every product, the loss, the
backward, clip and AdamW - is its own float64 arithmetic.  This separates the
kernels' numerical error from the routing flips of near-tied tokens, which
move whole token contributions between experts and dominate the comparison
against the oracle's own routing.

Gates (asserted, unchanged from the bf16 policy, *Results* - "Numerical
scope"): loss and per-position losses within 1e-2; every gradient tensor
within 0.08 relative L2; every updated weight tensor within 1e-2 relative L2;
the gradient norm within 0.08; the first Adam moment within 0.08 and the
second, quadratic in the gradient, within 0.16.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from parity_util import (BF16_GRAD_TOL, BF16_LOSS_TOL, BF16_PARAM_TOL, pooled_oracle_update,
                         rel_l2, to_np)

pytestmark = pytest.mark.gpu


def run_with_logits(cfg, params, micro_tokens, flags=0):
    """Run the update microbatch by microbatch, reading every layer's router
    logits after each launch (the next launch overwrites them)."""
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = MoETrainer(cfg, "cuda:0", flags=flags)
    tr.load_params(params)
    T, E = cfg.tokens_per_micro, cfg.n_experts
    logits, tok_loss = [], []
    for i, tok in enumerate(micro_tokens):
        tr.micro_step(torch.as_tensor(tok).cuda(), i)
        out = tr.outputs()
        assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
        logits.append([tr.debug_view(B.MT_VIEW_ROUTER_LOGITS, l).cpu().numpy()
                       .astype(np.float64).reshape(T, E) for l in range(cfg.n_layers)])
        tok_loss.append(to_np(tr.debug_view(B.MT_VIEW_TOK_LOSS)))
    return tr, out, logits, tok_loss


@pytest.mark.parametrize("name,rule", [("b2", None), ("b32", None), ("accum16", None),
                                       ("b2", "RECOMPUTE_ATTN_DS")])
def test_bf16_update_with_gpu_routing(name, rule):
    """rule: a memory rule whose path differs from the default (dQ recomputes
    P and dS instead of reading the stored dS^T)."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    flags = getattr(B, "MT_FLAG_" + rule) if rule else 0
    tr, out, logits, tok_loss = run_with_logits(cfg, params, toks, flags)
    ref = pooled_oracle_update(cfg, toks, route_logits=logits)
    print(f"\n{name} (GPU routing): loss {out.loss_update:.6f} (oracle {ref.loss:.6f}), "
          f"|g| {out.grad_norm:.5f} (oracle {ref.grad_norm:.5f})")
    assert abs(out.loss_update - ref.loss) / ref.loss < BF16_LOSS_TOL
    for i in range(cfg.micro_count):
        assert rel_l2(tok_loss[i], ref.tok_loss[i]) < BF16_LOSS_TOL, i
    assert abs(out.grad_norm - ref.grad_norm) / ref.grad_norm < BF16_GRAD_TOL
    worst = {}
    for pname, _ in mi.param_shapes(cfg):
        g = to_np(tr.view(tr.grads, pname))
        p = to_np(tr.view(tr.params, pname))
        m = to_np(tr.view(tr.adam_m, pname))
        v = to_np(tr.view(tr.adam_v, pname))
        eg = rel_l2(g, ref.grads[pname])
        ep = rel_l2(p, ref.params[pname])
        em = rel_l2(m, ref.m[pname])
        ev = rel_l2(v, ref.v[pname])
        dp = rel_l2(p - params[pname], ref.params[pname] - params[pname].astype(np.float64))
        print(f"  {pname:10s} grad {eg:.5f}  updated weight {ep:.6f}  (step {dp:.4f})  "
              f"m {em:.5f}  v {ev:.5f}")
        worst[pname] = (eg, ep, em, ev)
    del tr
    torch.cuda.empty_cache()
    for pname, (eg, ep, em, ev) in worst.items():
        assert eg < BF16_GRAD_TOL, (pname, "grad", eg)
        assert ep < BF16_PARAM_TOL, (pname, "updated weight", ep)
        assert em < BF16_GRAD_TOL, (pname, "adam m", em)
        assert ev < 2 * BF16_GRAD_TOL, (pname, "adam v", ev)


def test_residual_stream_drift_per_layer():
    """Relative L2 distance between the GPU's residual stream entering each
    layer and the oracle's, on the 2x1024 configuration: with the GPU's
    expert choices (the bf16 products' own error) and with the oracle's own
    choices (the same plus routing flips)."""
    import oracle
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("b2")
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    tr, out, logits, _ = run_with_logits(cfg, params, toks)
    T, d = cfg.tokens_per_micro, cfg.d_model
    hidden = [to_np(tr.debug_view(B.MT_VIEW_HIDDEN, l)).reshape(T, d) for l in range(cfg.n_layers)]
    del tr
    torch.cuda.empty_cache()
    D = oracle.Dims.of(cfg)
    P = oracle.to64(params)
    rows = []
    for label, rz in (("GPU routing", logits[0]), ("own routing", None)):
        _, _, dbg = oracle.forward_backward(P, toks[0], D, 1.0, {}, keep_cache=True, backward=False,
                                            route_logits=rz)
        xs = [c["x_in"] for c in dbg["caches"]]
        drift = [rel_l2(hidden[l], xs[l]) for l in range(cfg.n_layers)]
        rows.append((label, drift))
        print(f"\n{label}: " + " ".join(f"{x:.2e}" for x in drift))
    forced = rows[0][1]
    assert forced[0] == 0.0 or forced[0] < 1e-6       # the embedding rows are copied exactly
    assert max(forced) < 1e-2, forced                  # measured at most 5.7e-3 over 8 layers
