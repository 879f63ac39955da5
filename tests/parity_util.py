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


# ---------------------------------------------------------------------------
# The oracle over many sequences, one block of sequences per worker process.
# Sequences never interact in this model, so the update's gradient is the sum
# of the blocks' gradients; the clip + AdamW step then runs once on the sum.
# Workers are started with "spawn" (never forked from a process that holds a
# CUDA context) and regenerate the seeded weights themselves.
# ---------------------------------------------------------------------------
_WORKER_P = {}


def _oracle_block(job):
    import oracle
    cfg, tokens, coef, route_rows = job
    key = (cfg.name, cfg.n_experts, cfg.top_k, cfg.d_ff, cfg.n_layers, cfg.n_unique_layers)
    if key not in _WORKER_P:
        _WORKER_P.clear()
        _WORKER_P[key] = oracle.to64(mi.make_params(cfg))
    P = _WORKER_P[key]
    D = oracle.Dims.of(cfg)
    grads = {k: np.zeros_like(v) for k, v in P.items()}
    loss, parts = 0.0, []
    S = tokens.shape[1]
    for b in range(tokens.shape[0]):
        rz = None if route_rows is None else [z[b * S:(b + 1) * S] for z in route_rows]
        lo, tl, _ = oracle.forward_backward(P, tokens[b:b + 1], D, coef, grads, route_logits=rz)
        loss += lo
        parts.append(tl)
    return loss, np.concatenate(parts), grads


def oracle_workers() -> int:
    """Worker count for the pooled oracle: the host cores (at most 16), bounded by
    about 6 GB of host memory per worker (float64 weights, gradients and one
    sequence's activations at d 768, V 32000)."""
    cores = len(os.sched_getaffinity(0))
    try:
        mem = os.sysconf("SC_PHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError):
        mem = 64 << 30
    try:
        with open("/sys/fs/cgroup/memory.max") as f:
            lim = f.read().strip()
        if lim != "max":
            mem = min(mem, int(lim))
    except OSError:
        pass
    return max(1, min(cores, 16, int((mem - (16 << 30)) // (6 << 30))))


def pooled_oracle_update(cfg, micro_tokens, route_logits=None, workers=None):
    """oracle.train_update evaluated by a pool of worker processes.

    route_logits: per microbatch, a per-layer list of [batch*seq, E] logits on
    which the expert choices are made (None: the oracle's own choices).
    Returns an oracle.UpdateResult (tok_loss per microbatch)."""
    import multiprocessing as mp

    import oracle
    workers = workers or oracle_workers()
    total_targets = sum(oracle.n_targets(*t.shape) for t in micro_tokens)
    coef = 1.0 / total_targets
    jobs, owner = [], []
    for m, tokens in enumerate(micro_tokens):
        B, S = tokens.shape
        n = max(1, min(B, -(-B * len(micro_tokens) // workers)))
        for b0 in range(0, B, n):
            b1 = min(B, b0 + n)
            rows = None
            if route_logits is not None:
                rows = [np.asarray(z)[b0 * S:b1 * S] for z in route_logits[m]]
            jobs.append((cfg, tokens[b0:b1], coef, rows))
            owner.append(m)
    threads = max(1, len(os.sched_getaffinity(0)) // workers)
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    for k in saved:
        os.environ[k] = str(threads)
    try:
        with mp.get_context("spawn").Pool(workers) as pool:
            results = pool.map(_oracle_block, jobs, chunksize=1)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    grads = None
    loss = 0.0
    tok_parts = [[] for _ in micro_tokens]
    for (lo, tl, g), m in zip(results, owner):       # fixed order: microbatch, then sequence
        loss += lo
        tok_parts[m].append(tl)
        if grads is None:
            grads = g
        else:
            for k in grads:
                grads[k] += g[k]
    del results
    P = oracle.to64(mi.make_params(cfg))
    zeros = {k: np.zeros_like(v) for k, v in P.items()}
    new_p, new_m, new_v, n, c = oracle.clip_adamw(
        P, grads, zeros, zeros, lr=cfg.lr, beta1=cfg.beta1, beta2=cfg.beta2, eps=cfg.eps,
        weight_decay=cfg.weight_decay, clip_norm=cfg.clip_norm, clip_eps=cfg.clip_eps,
        step=cfg.step)
    return oracle.UpdateResult(loss=loss, grads=grads, grad_norm=n, clip_coef=c, params=new_p,
                               m=new_m, v=new_v, tok_loss=[np.concatenate(p) for p in tok_parts])
