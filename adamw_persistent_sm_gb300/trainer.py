"""Device buffers for the training update, allocated through torch.

PyTorch supplies device memory and streams only; every step of the update
runs in the CUDA library through :mod:`.binding`.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B


class StatusError(RuntimeError):
    pass


def _check(st: int, what: str) -> None:
    if st != B.MT_OK:
        raise StatusError(f"{what}: {B.status_string(st)} ({st})")


class MoETrainer:
    """Flat fp32 parameters, bf16 shadow, gradients, Adam moments and the
    arena for one model configuration on the current CUDA device."""

    def __init__(self, cfg, device: str | torch.device = "cuda", flags: int = 0,
                 wait_timeout_ns: int = 0):
        if not torch.cuda.is_available():
            raise RuntimeError("MoETrainer needs a CUDA device")
        self.lib = B.load()
        self.cfg = cfg
        self.device = torch.device(device)
        self.flags = flags
        self.wait_timeout_ns = wait_timeout_ns
        hp = B.hparams(cfg, flags=flags)      # MT_FLAG_TRACE adds the trace to the arena
        n = B.mt_param_count(hp)
        if n < 0:
            raise StatusError(f"mt_param_count: {B.status_string(-n)}")
        self.n_params = n
        self.layout = {t["name"]: t for t in B.mt_param_layout(hp)}
        dev = self.device
        self.params = torch.zeros(n, dtype=torch.float32, device=dev)
        self.bf16 = cfg.precision == "bf16"
        self.shadow = torch.zeros(n, dtype=torch.bfloat16, device=dev) if self.bf16 else None
        self.grads = torch.zeros(n, dtype=torch.float32, device=dev)
        self.adam_m = torch.zeros(n, dtype=torch.float32, device=dev)
        self.adam_v = torch.zeros(n, dtype=torch.float32, device=dev)
        self.arena_bytes = B.mt_arena_bytes(hp)
        if self.arena_bytes < 0:
            raise StatusError(f"mt_arena_bytes: {B.status_string(-self.arena_bytes)}")
        self.arena = torch.empty(self.arena_bytes, dtype=torch.uint8, device=dev)
        self.reset_arena()

    # ---- plumbing -----------------------------------------------------------
    @property
    def stream(self) -> int:
        return torch.cuda.current_stream(self.device).cuda_stream

    def reset_arena(self) -> None:
        _check(B.mt_arena_init(self.arena.data_ptr(), self.arena_bytes, self.stream), "mt_arena_init")

    def view(self, buf: torch.Tensor, name: str) -> torch.Tensor:
        t = self.layout[name]
        return buf[t["offset"]:t["offset"] + t["numel"]].view(t["shape"])

    def load_params(self, named: dict) -> None:
        """Copy named fp32 arrays into the flat master buffer and refresh the
        bf16 shadow."""
        for name, arr in named.items():
            src = torch.as_tensor(np.ascontiguousarray(arr, dtype=np.float32))
            self.view(self.params, name).copy_(src.view(self.layout[name]["shape"]))
        self.sync_shadow()

    def sync_shadow(self) -> None:
        if self.shadow is not None:
            _check(B.mt_sync_shadow(self.params.data_ptr(), self.shadow.data_ptr(), self.n_params,
                                    self.stream), "mt_sync_shadow")

    def named(self, buf: torch.Tensor) -> dict:
        return {name: self.view(buf, name) for name in self.layout}

    def hparams(self, micro_index: int = 0, step: int | None = None, flags: int | None = None,
                expert_step: int = 1):
        return B.hparams(self.cfg, micro_index=micro_index, step=step,
                         flags=self.flags if flags is None else flags,
                         wait_timeout_ns=self.wait_timeout_ns, expert_step=expert_step)

    # ---- the update ---------------------------------------------------------
    def micro_step(self, tokens: torch.Tensor, micro_index: int = 0, step: int | None = None,
                   flags: int | None = None, expert_step: int = 1) -> None:
        """Enqueue one microbatch launch (tokens: int32 [batch, seq] on the device)."""
        assert tokens.dtype == torch.int32 and tokens.is_cuda and tokens.is_contiguous()
        hp = self.hparams(micro_index, step, flags, expert_step)
        st = B.mt_train_update(self.params.data_ptr(),
                               self.shadow.data_ptr() if self.shadow is not None else 0,
                               self.grads.data_ptr(), self.adam_m.data_ptr(), self.adam_v.data_ptr(),
                               tokens.data_ptr(), hp, self.arena.data_ptr(), self.arena_bytes,
                               self.stream)
        _check(st, "mt_train_update")

    def update(self, micro_tokens: list, step: int | None = None, flags: int | None = None) -> None:
        for i, tok in enumerate(micro_tokens):
            self.micro_step(tok, i, step, flags)

    def debug_run(self, op: int, layer: int = 0, tokens: torch.Tensor | None = None,
                  step: int | None = None) -> None:
        """One op of the single-op harness on the buffers of this trainer."""
        if tokens is None:           # ops that read no token ids still take a valid buffer
            tokens = torch.zeros(self.cfg.batch, self.cfg.seq, dtype=torch.int32, device=self.device)
        tok = tokens.data_ptr()
        hp = self.hparams(0, step)
        st = B.mt_debug_run(op, layer, self.params.data_ptr(),
                            self.shadow.data_ptr() if self.shadow is not None else 0,
                            self.grads.data_ptr(), self.adam_m.data_ptr(), self.adam_v.data_ptr(),
                            tok, hp, self.arena.data_ptr(), self.arena_bytes, self.stream)
        _check(st, "mt_debug_run")

    def outputs(self) -> B.mt_outputs:
        return B.mt_read_outputs(self.arena.data_ptr(), self.stream)

    def debug_view(self, which: int, layer: int = 0, dtype=torch.float32) -> torch.Tensor:
        """A torch tensor aliasing a buffer inside the arena."""
        v = B.mt_debug_view(self.arena.data_ptr(), self.hparams(), which, layer)
        off = v.ptr - self.arena.data_ptr()
        nbytes = v.numel * v.elem_bytes
        return self.arena[off:off + nbytes].view(dtype)
