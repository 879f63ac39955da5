"""GPU parity of the bf16-product configurations at their full sizes, against
oracle values stored by tests/golden/make_golden.py (float64, seeded sample
coordinates): loss within 1e-2, every gradient tensor within 0.08 relative
L2 and every updated tensor within 1e-2 relative L2 on the samples."""
import numpy as np
import pytest

import moe_inputs as mi
from parity_util import (BF16_GRAD_TOL, BF16_LOSS_TOL, BF16_PARAM_TOL, load_golden, rel_l2,
                         run_gpu_update, to_np)

pytestmark = pytest.mark.gpu


def check_against_golden(cfg, tr, out, gold):
    report = {}
    assert abs(out.loss_update - gold["loss"]) / gold["loss"] < BF16_LOSS_TOL
    assert abs(out.grad_norm - gold["grad_norm"]) / gold["grad_norm"] < BF16_GRAD_TOL
    for name, _ in mi.param_shapes(cfg):
        idx = gold[f"{name}.idx"]
        g = to_np(tr.view(tr.grads, name).reshape(-1)[idx])
        p = to_np(tr.view(tr.params, name).reshape(-1)[idx])
        eg = rel_l2(g, gold[f"{name}.grad"])
        ep = rel_l2(p, gold[f"{name}.param"])
        report[name] = (eg, ep)
        assert eg < BF16_GRAD_TOL, (name, eg)
        assert ep < BF16_PARAM_TOL, (name, ep)
    return report


@pytest.mark.parametrize("name", ["b2", "top8", "b32", "accum16"])
def test_bf16_update_matches_oracle(name):
    gold = load_golden(name)
    assert gold is not None, f"missing tests/golden/oracle_{name}.npz (run make_golden.py)"
    cfg = mi.get_config(name)
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    tr, out = run_gpu_update(cfg, params, toks)
    rep = check_against_golden(cfg, tr, out, gold)
    print(name, {k: (round(a, 5), round(b, 6)) for k, (a, b) in rep.items()})
    if cfg.micro_count == 1:
        from adamw_persistent_sm_gb300 import binding as B
        tl = to_np(tr.debug_view(B.MT_VIEW_TOK_LOSS))
        assert rel_l2(tl, gold["tok_loss"]) < BF16_LOSS_TOL
    del tr
