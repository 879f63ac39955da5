"""Selective updates on the GPU against the oracle (*Results*, "Other
measured compiler work": shared weights update every microbatch, experts
every 16 - here every ``micro_count`` microbatches, 4 in the tests).

MT_FLAG_SELECTIVE_EXPERTS: after every microbatch the shared tensors take a
clipped AdamW step (step index advancing per microbatch); the expert tensors
sum their gradients over the period and step once on the mean after its last
microbatch.  The tiny fp32 model runs two periods at 1e-4; the 2x1024 bf16
model runs one period with the expert choices taken from the GPU's router
logits, under the bf16 gates.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity_util import (BF16_GRAD_TOL, BF16_LOSS_TOL, BF16_PARAM_TOL, TINY_TOL, rel_l2, to_np)

pytestmark = pytest.mark.gpu


def _period(tr, cfg, toks, step0, expert_step, gpu_routing):
    from adamw_persistent_sm_gb300 import binding as B
    T, E = cfg.tokens_per_micro, cfg.n_experts
    losses, norms, logits = [], [], []
    for i, tok in enumerate(toks):
        tr.micro_step(torch.as_tensor(tok).cuda(), i, step=step0 + i, flags=B.MT_FLAG_SELECTIVE_EXPERTS,
                      expert_step=expert_step)
        out = tr.outputs()
        assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
        assert out.optimizer_ran == 1
        assert out.experts_updated == (1 if i == len(toks) - 1 else 0)
        losses.append(out.loss)
        norms.append(out.grad_norm)
        if gpu_routing:
            logits.append([tr.debug_view(B.MT_VIEW_ROUTER_LOGITS, l).cpu().numpy().astype(np.float64)
                           .reshape(T, E) for l in range(cfg.n_layers)])
    return out, losses, norms, (logits if gpu_routing else None)


def _compare(tr, cfg, ref, out, losses, norms, tol_loss, tol_grad, tol_param):
    for i, (lo, n) in enumerate(zip(losses, norms)):
        assert abs(lo - ref.losses[i]) / ref.losses[i] < tol_loss, (i, lo, ref.losses[i])
        assert abs(n - ref.shared_norms[i]) / ref.shared_norms[i] < tol_grad, (i, n, ref.shared_norms[i])
    assert abs(out.expert_grad_norm - ref.expert_norm) / ref.expert_norm < tol_grad
    worst = {}
    for name, _ in mi.param_shapes(cfg):
        g_ref = ref.expert_grads[name] if name in oracle.EXPERT_TENSORS else ref.shared_grads[name]
        e = (rel_l2(to_np(tr.view(tr.grads, name)), g_ref),
             rel_l2(to_np(tr.view(tr.params, name)), ref.params[name]),
             rel_l2(to_np(tr.view(tr.adam_m, name)), ref.m[name]),
             rel_l2(to_np(tr.view(tr.adam_v, name)), ref.v[name]))
        worst[name] = e
        print(f"  {name:10s} grad {e[0]:.2e} weight {e[1]:.2e} m {e[2]:.2e} v {e[3]:.2e}")
    for name, (g, p, m, v) in worst.items():
        assert g < tol_grad and m < tol_grad and v < 2 * tol_grad, (name, g, m, v)
        assert p < tol_param, (name, p)


def test_tiny_two_periods():
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    cfg = mi.get_config("tiny", micro_count=4)
    params = mi.make_params(cfg)
    tr = MoETrainer(cfg, "cuda:0")
    tr.load_params(params)
    P, M, V = params, None, None
    for period in range(2):
        toks = mi.make_step_tokens(cfg, period + 1)
        out, losses, norms, _ = _period(tr, cfg, toks, 1 + 4 * period, period + 1, False)
        ref = oracle.selective_updates(P, toks, cfg, m=M, v=V, step=1 + 4 * period, expert_step=period + 1)
        P, M, V = ref.params, ref.m, ref.v
        print(f"\nperiod {period + 1}: losses {['%.5f' % x for x in losses]}")
        _compare(tr, cfg, ref, out, losses, norms, TINY_TOL, TINY_TOL, TINY_TOL)


def test_b2_one_period_with_gpu_routing():
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    cfg = mi.get_config("b2", micro_count=4)
    params = mi.make_params(cfg)
    tr = MoETrainer(cfg, "cuda:0")
    tr.load_params(params)
    toks = mi.make_update_tokens(cfg)
    out, losses, norms, logits = _period(tr, cfg, toks, 1, 1, True)
    ref = oracle.selective_updates(params, toks, cfg, route_logits=logits)
    print(f"\nb2 selective: losses {['%.5f' % x for x in losses]} (oracle {['%.5f' % x for x in ref.losses]})")
    _compare(tr, cfg, ref, out, losses, norms, BF16_LOSS_TOL, BF16_GRAD_TOL, BF16_PARAM_TOL)
