"""Helpers of the GPU parity tests: run an update through the C ABI and
compare it with the oracle's values."""
import os

import numpy as np
import torch

import moe_inputs as mi

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

# tolerances of the two numerical policies
TINY_TOL = 1e-4                       # fp32: loss, every gradient, every updated tensor
BF16_LOSS_TOL = 1e-2                  # bf16 products: loss and updated weights
BF16_PARAM_TOL = 1e-2
BF16_GRAD_TOL = 0.08                  # relative L2 per gradient tensor


def rel_l2(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def run_gpu_update(cfg, params, micro_tokens, flags=0, trainer=None, step=None):
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = trainer or MoETrainer(cfg, "cuda:0", flags=flags)
    if trainer is None:
        tr.load_params(params)
    tr.update([torch.as_tensor(t).cuda() for t in micro_tokens], step=step)
    out = tr.outputs()
    assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
    return tr, out


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def load_golden(name):
    path = os.path.join(GOLD, f"oracle_{name}.npz")
    if not os.path.exists(path):
        return None
    return dict(np.load(path))
