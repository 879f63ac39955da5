"""Seeded synthetic inputs for the MoE training update.

This module holds no arithmetic of the method: it names the five workload
configurations, lists the parameter tensors with their shapes, and draws the
seeded initial weights and token ids.  Both the CUDA path (through the tests
and the benchmark) and the CPU oracle take their inputs from here, so the two
sides see bit-identical fp32 weights and int32 tokens.

Workloads (one GPU, one update each):

* ``tiny``    - vocab 256, d 64, 2 layers, 4 heads of 16, 4 experts top-2,
                d_ff 128, batch 2 x 32, fp32 compute.
* ``b2``      - vocab 32000, d 768, 8 layers, 12 heads of 64, 16 experts top-2,
                d_ff 512, batch 2 x 1024, bf16 products / fp32 state.
* ``b32``     - as ``b2`` with batch 32 x 1024 (one microbatch).
* ``accum16`` - as ``b2`` with 16 microbatches of 8 x 1024, one optimizer step.
* ``top8``    - as ``b2`` but 32 experts of d_ff 256, top-8, batch 1 x 4096,
                Zipf(1.1) token ids.
* ``looped``  - as ``b32`` with 4 distinct layers visited twice each (8 layer
                visits; visit l uses the weights of layer l mod 4).

The model is the pages' "TinyMoE" stand-in ("How a training megakernel works",
section "From two weights to 200 million": attention plus expert layers whose
router sends each token to two of sixteen small feed-forward networks, trained
with AdamW); the exact sizes above are this project's choice because the pages
do not print them.
"""
from __future__ import annotations

import copy
from dataclasses import dataclass, field, asdict

import numpy as np

WEIGHT_SEED = 1740          # arbitrary; borrowed from the seed the pages' full run names
TOKEN_SEED = 1741           # + micro_index


@dataclass
class MoEConfig:
    name: str
    vocab: int
    d_model: int
    n_layers: int
    n_heads: int
    head_dim: int
    n_experts: int
    top_k: int
    d_ff: int
    batch: int
    seq: int
    micro_count: int = 1
    precision: str = "bf16"          # "fp32" | "bf16"
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.95
    eps: float = 1e-8
    weight_decay: float = 0.1
    clip_norm: float = 1.0
    clip_eps: float = 1e-6
    norm_eps: float = 1e-5
    rope_theta: float = 1e4
    init_std: float = 0.02
    out_std: float = 0.02            # attention out-proj and expert down-proj
    token_dist: str = "uniform"      # "uniform" | "zipf1.1"
    step: int = 1                    # AdamW step index t (1-based)
    n_unique_layers: int = 0         # looped model: distinct layers (0 = n_layers)

    @property
    def tokens_per_micro(self) -> int:
        return self.batch * self.seq

    @property
    def tokens_per_update(self) -> int:
        return self.batch * self.seq * self.micro_count

    def replace(self, **kw) -> "MoEConfig":
        c = copy.copy(self)
        for k, v in kw.items():
            if not hasattr(c, k):
                raise AttributeError(k)
            setattr(c, k, v)
        return c

    def as_dict(self) -> dict:
        return asdict(self)


_BASE = dict(vocab=32000, d_model=768, n_layers=8, n_heads=12, head_dim=64,
             n_experts=16, top_k=2, d_ff=512, precision="bf16", lr=3e-4,
             out_std=0.02 / np.sqrt(16.0))

CONFIGS: dict[str, MoEConfig] = {
    "tiny": MoEConfig(name="tiny", vocab=256, d_model=64, n_layers=2, n_heads=4,
                      head_dim=16, n_experts=4, top_k=2, d_ff=128, batch=2, seq=32,
                      precision="fp32", lr=1e-3, out_std=0.02),
    "b2": MoEConfig(name="b2", batch=2, seq=1024, **_BASE),
    "b32": MoEConfig(name="b32", batch=32, seq=1024, **_BASE),
    "accum16": MoEConfig(name="accum16", batch=8, seq=1024, micro_count=16, **_BASE),
    "top8": MoEConfig(name="top8", batch=1, seq=4096, token_dist="zipf1.1",
                      **{**_BASE, "n_experts": 32, "top_k": 8, "d_ff": 256}),
    # looped ("SMELT-style") model: the same trunk with 4 distinct layers,
    # each visited twice (visit l uses the weights of layer l mod 4)
    "looped": MoEConfig(name="looped", batch=32, seq=1024, n_unique_layers=4, **_BASE),
}


def get_config(name: str, **overrides) -> MoEConfig:
    return CONFIGS[name].replace(**overrides) if overrides else copy.copy(CONFIGS[name])


def param_shapes(cfg: MoEConfig) -> list[tuple[str, tuple[int, ...]]]:
    """Parameter tensors in their canonical order, stacked over layers.

    ``wqkv`` rows are [q; k; v], head h owning rows h*head_dim..(h+1)*head_dim-1
    inside each block; every matrix is stored [out, in] (row = output feature).
    """
    V, d, E, F = cfg.vocab, cfg.d_model, cfg.n_experts, cfg.d_ff
    L = cfg.n_unique_layers or cfg.n_layers          # per-layer tensors: one slot per distinct layer
    hq = cfg.n_heads * cfg.head_dim
    return [
        ("emb", (V, d)),
        ("attn_norm", (L, d)),
        ("wqkv", (L, 3 * hq, d)),
        ("wo", (L, d, hq)),
        ("moe_norm", (L, d)),
        ("router", (L, E, d)),
        ("w_gate", (L, E, F, d)),
        ("w_up", (L, E, F, d)),
        ("w_down", (L, E, d, F)),
        ("final_norm", (d,)),
        ("lm_head", (V, d)),
    ]


NORM_GAINS = ("attn_norm", "moe_norm", "final_norm")
OUT_PROJ = ("wo", "w_down")


def param_count(cfg: MoEConfig) -> int:
    return int(sum(int(np.prod(s)) for _, s in param_shapes(cfg)))


def make_params(cfg: MoEConfig, seed: int = WEIGHT_SEED) -> dict[str, np.ndarray]:
    """Seeded fp32 initial weights: N(0, init_std) drawn in fp64 and rounded to
    fp32; ``wo`` and ``w_down`` use ``out_std``; RMSNorm gains are 1."""
    rng = np.random.default_rng(seed)
    out: dict[str, np.ndarray] = {}
    for name, shape in param_shapes(cfg):
        if name in NORM_GAINS:
            out[name] = np.ones(shape, dtype=np.float32)
        else:
            std = cfg.out_std if name in OUT_PROJ else cfg.init_std
            out[name] = rng.normal(0.0, std, size=shape).astype(np.float32)
    return out


def zipf_probs(vocab: int, s: float = 1.1) -> np.ndarray:
    """P(id = r-1) proportional to r**-s for rank r = 1..vocab (truncated, normalised)."""
    r = np.arange(1, vocab + 1, dtype=np.float64)
    p = r ** (-s)
    return p / p.sum()


def make_tokens(cfg: MoEConfig, micro_index: int = 0) -> np.ndarray:
    """Seeded int32 token ids [batch, seq] for one microbatch."""
    rng = np.random.default_rng(TOKEN_SEED + micro_index)
    shape = (cfg.batch, cfg.seq)
    if cfg.token_dist == "uniform":
        return rng.integers(0, cfg.vocab, size=shape, dtype=np.int32)
    if cfg.token_dist == "zipf1.1":
        return rng.choice(cfg.vocab, size=shape, p=zipf_probs(cfg.vocab, 1.1)).astype(np.int32)
    raise ValueError(cfg.token_dist)


def make_update_tokens(cfg: MoEConfig) -> list[np.ndarray]:
    """Token ids of every microbatch of one update."""
    return [make_tokens(cfg, i) for i in range(cfg.micro_count)]


def zeros_like_params(cfg: MoEConfig) -> dict[str, np.ndarray]:
    return {name: np.zeros(shape, dtype=np.float32) for name, shape in param_shapes(cfg)}


# ---------------------------------------------------------------------------
# Seeded operands for the single-op tests (draws only)
# ---------------------------------------------------------------------------
def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 copy of x holding the nearest bfloat16 values (ties to even), so
    that a bf16 device buffer and a float64 host copy hold the same numbers."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16 << 16
    return (b & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


def normal_operand(shape, seed: int, std: float = 1.0, mean: float = 0.0,
                   bf16: bool = False) -> np.ndarray:
    """Seeded N(mean, std) fp32 array; bf16-representable when ``bf16``."""
    x = np.random.default_rng(seed).normal(mean, std, size=shape).astype(np.float32)
    return round_to_bf16(x) if bf16 else x


def make_step_tokens(cfg: MoEConfig, step: int) -> list[np.ndarray]:
    """Token ids of every microbatch of update number ``step`` (1-based) of a
    multi-step run; step 1 draws the same ids as :func:`make_update_tokens`."""
    base = 0 if step == 1 else 100003 * step
    return [make_tokens(cfg, base + i) for i in range(cfg.micro_count)]
