"""GB300 training-update megakernel for a top-K-of-E mixture-of-experts
transformer: one persistent CUDA kernel per microbatch runs the forward pass,
next-token cross-entropy, backward pass, global-norm clipping and AdamW.

The compute path is the CUDA library built from ``csrc/`` (C ABI in
``include/moe_train.h``); :mod:`.binding` marshals arguments to it and
:mod:`.trainer` allocates device buffers through torch.
"""
from . import binding  # noqa: F401

__all__ = ["binding", "build", "MoETrainer"]


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def __getattr__(name):
    if name == "MoETrainer":
        from .trainer import MoETrainer
        return MoETrainer
    raise AttributeError(name)
