"""A multi-step training run checked against the oracle after every update
(*Results* - "Faster execution" times fresh, mid and late training states;
this is the short synthetic version of such a run).

Both sides carry their own state - the GPU its fp32 master weights, bf16
shadow and Adam moments in device memory, the oracle its float64 copies - so
the bias corrections of steps t > 1, the non-zero moments and the round trip
of the state through every launch are all compared.  New seeded tokens each
step.  The tiny fp32 model runs 10 updates at 1e-4; the bf16 models (5 updates
at 2x1024, 2 at 1x4096 top-8) run with
the expert choices taken from the GPU's router logits (as in
test_gpu_bf16_routed.py) under the bf16 gates.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity_util import (BF16_GRAD_TOL, BF16_LOSS_TOL, BF16_PARAM_TOL, TINY_TOL, rel_l2, to_np)

pytestmark = pytest.mark.gpu


def _run(name, steps, gpu_routing):
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    cfg = mi.get_config(name)
    params = mi.make_params(cfg)
    tr = MoETrainer(cfg, "cuda:0")
    tr.load_params(params)
    P = oracle.to64(params)
    M = V = None
    T, E = cfg.tokens_per_micro, cfg.n_experts
    rows = []
    for t in range(1, steps + 1):
        toks = mi.make_step_tokens(cfg, t)
        logits = []
        for i, tok in enumerate(toks):
            tr.micro_step(torch.as_tensor(tok).cuda(), i, step=t)
            if gpu_routing:
                assert tr.outputs().status == B.MT_OK
                logits.append([tr.debug_view(B.MT_VIEW_ROUTER_LOGITS, l).cpu().numpy().astype(np.float64)
                               .reshape(T, E) for l in range(cfg.n_layers)])
        out = tr.outputs()
        assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
        ref = oracle.train_update(P, toks, cfg.replace(step=t), m=M, v=V,
                                  route_logits=logits if gpu_routing else None)
        P, M, V = ref.params, ref.m, ref.v
        errs = {"loss": abs(out.loss_update - ref.loss) / ref.loss,
                "norm": abs(out.grad_norm - ref.grad_norm) / ref.grad_norm}
        for pname, _ in mi.param_shapes(cfg):
            errs[pname] = (rel_l2(to_np(tr.view(tr.grads, pname)), ref.grads[pname]),
                           rel_l2(to_np(tr.view(tr.params, pname)), ref.params[pname]),
                           rel_l2(to_np(tr.view(tr.adam_m, pname)), ref.m[pname]),
                           rel_l2(to_np(tr.view(tr.adam_v, pname)), ref.v[pname]))
        worst = [max(e[i] for k, e in errs.items() if isinstance(e, tuple)) for i in range(4)]
        print(f"\n{name} step {t}: loss {out.loss_update:.6f} (oracle {ref.loss:.6f}) "
              f"worst grad {worst[0]:.2e} weight {worst[1]:.2e} m {worst[2]:.2e} v {worst[3]:.2e}")
        rows.append(errs)
    return cfg, rows


def test_tiny_ten_updates():
    _, rows = _run("tiny", 10, gpu_routing=False)
    for t, errs in enumerate(rows, 1):
        for k, e in errs.items():
            for x in (e if isinstance(e, tuple) else (e,)):
                assert x < TINY_TOL, (t, k, x)


@pytest.mark.parametrize("name,steps", [("b2", 5), ("top8", 2)])
def test_bf16_updates_with_gpu_routing(name, steps):
    _, rows = _run(name, steps, gpu_routing=True)
    for t, errs in enumerate(rows, 1):
        assert errs["loss"] < BF16_LOSS_TOL, (t, errs["loss"])
        assert errs["norm"] < BF16_GRAD_TOL, (t, errs["norm"])
        for k, e in errs.items():
            if isinstance(e, tuple):
                g, p, m, v = e
                assert g < BF16_GRAD_TOL and m < BF16_GRAD_TOL and v < 2 * BF16_GRAD_TOL, (t, k, e)
                assert p < BF16_PARAM_TOL, (t, k, e)
