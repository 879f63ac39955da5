"""Write sampled oracle outputs for the large configurations.

Calls only the CPU oracle (and the seeded input generators): for each
configuration it runs one complete update in float64 and stores the loss,
the gradient norm, the clip coefficient, the per-position losses, every
tensor's gradient norm, and gradients / updated weights at seeded sample
coordinates.  The GPU parity tests compare the CUDA path against these.

Usage:  python tests/golden/make_golden.py b2 top8 b32 accum16
Microbatches are evaluated one sequence at a time (sequences never interact
in this model, so the sums are unchanged and memory stays small).
"""
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import moe_inputs as mi  # noqa: E402
import oracle  # noqa: E402

N_SAMPLES = 4096
SAMPLE_SEED = 2024


def sample_indices(name, arr, cfg, tokens_all, k):
    """Seeded coordinates of one tensor; embedding samples come from rows of
    tokens present in the update (other rows have zero gradient)."""
    rng = np.random.default_rng(SAMPLE_SEED + k)
    n = arr.size
    if name == "emb":
        rows = np.unique(np.concatenate([t.reshape(-1) for t in tokens_all]))
        cand = (rows[:, None] * cfg.d_model + np.arange(cfg.d_model)[None, :]).reshape(-1)
        return np.sort(rng.choice(cand, size=min(N_SAMPLES, cand.size), replace=False))
    return np.sort(rng.choice(n, size=min(N_SAMPLES, n), replace=False))


def make(name):
    cfg = mi.get_config(name)
    t0 = time.time()
    params = mi.make_params(cfg)
    toks = mi.make_update_tokens(cfg)
    r = oracle.train_update(params, toks, cfg, seqs_per_block=1)
    out = dict(loss=r.loss, grad_norm=r.grad_norm, clip_coef=r.clip_coef,
               tok_loss=np.concatenate(r.tok_loss))
    for k, (pname, _) in enumerate(mi.param_shapes(cfg)):
        g = r.grads[pname]
        idx = sample_indices(pname, g, cfg, toks, k)
        out[f"{pname}.idx"] = idx
        out[f"{pname}.grad"] = g.reshape(-1)[idx]
        out[f"{pname}.param"] = r.params[pname].reshape(-1)[idx]
        out[f"{pname}.grad_norm"] = np.linalg.norm(g)
    path = os.path.join(HERE, f"oracle_{name}.npz")
    np.savez_compressed(path, **out)
    print(f"{name}: loss {r.loss:.6f} |g| {r.grad_norm:.5f} c {r.clip_coef:.5f} "
          f"({time.time() - t0:.0f} s) -> {os.path.relpath(path, ROOT)}", flush=True)


if __name__ == "__main__":
    for n in sys.argv[1:] or ["b2", "top8"]:
        make(n)
