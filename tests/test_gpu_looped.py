"""The looped model on the GPU against the oracle (*Results*, "Other
measured compiler work": looped TinyMoE - repeated layers share weights and
accumulate gradients across visits).

hp.n_unique_layers = U: layer visit l runs with the weights of slot l mod U,
and every slot's gradient is the sum over its visits (the backward writes the
last visit of a slot and adds the earlier ones).  Tiny fp32 with one layer
visited twice at 1e-4; the 2x1024 trunk with 4 distinct layers visited twice
each, with the GPU's expert choices, under the bf16 gates.
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from parity_util import (BF16_GRAD_TOL, BF16_LOSS_TOL, BF16_PARAM_TOL, TINY_TOL, pooled_oracle_update,
                         rel_l2, run_gpu_update, to_np)
from test_gpu_bf16_routed import run_with_logits

pytestmark = pytest.mark.gpu


def _check(tr, out, ref, cfg, tol_loss, tol_grad, tol_param):
    assert abs(out.loss_update - ref.loss) / ref.loss < tol_loss
    assert abs(out.grad_norm - ref.grad_norm) / ref.grad_norm < tol_grad
    for name, shape in mi.param_shapes(cfg):
        assert tuple(tr.layout[name]["shape"]) == tuple(shape)
        g = rel_l2(to_np(tr.view(tr.grads, name)), ref.grads[name])
        p = rel_l2(to_np(tr.view(tr.params, name)), ref.params[name])
        print(f"  {name:10s} grad {g:.2e} weight {p:.2e}")
        assert g < tol_grad, (name, g)
        assert p < tol_param, (name, p)


@pytest.mark.parametrize("L,U", [(2, 1), (4, 2)])
def test_tiny_looped(L, U):
    cfg = mi.get_config("tiny", n_layers=L, n_unique_layers=U)
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    tr, out = run_gpu_update(cfg, params, toks)
    ref = oracle.train_update(params, toks, cfg)
    _check(tr, out, ref, cfg, TINY_TOL, TINY_TOL, TINY_TOL)


def test_b2_trunk_looped_with_gpu_routing():
    cfg = mi.get_config("looped", batch=2)
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    tr, out, logits, _ = run_with_logits(cfg, params, toks)
    ref = pooled_oracle_update(cfg, toks, route_logits=logits)
    print(f"\nlooped 2x1024: loss {out.loss_update:.6f} (oracle {ref.loss:.6f})")
    _check(tr, out, ref, cfg, BF16_LOSS_TOL, BF16_GRAD_TOL, BF16_PARAM_TOL)
