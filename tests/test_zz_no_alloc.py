"""mt_train_update_noalloc: the training-update launch whose scratch arena
is the library's own fixed device array, for callers that may not allocate
device memory (e.g. a plug-in whose host application owns all device memory).

Two calls in a row through the C ABI - a first AdamW step and a second step
on new tokens - must give the same loss, gradients, weights and Adam moments
as the regular entry point with a caller-allocated arena.  Runs last so that
a failure here cannot hide any other test's result, and needs no state from
other tests."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from parity_util import TINY_TOL, rel_l2, to_np

pytestmark = pytest.mark.gpu


def test_noalloc_matches_regular_entry_point_on_two_calls():
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer

    cfg = mi.get_config("tiny")
    hp = B.hparams(cfg)
    assert 0 < B.mt_arena_bytes(hp) <= B.MT_NOALLOC_ARENA_BYTES
    params = mi.make_params(cfg)
    calls = [(1, torch.as_tensor(mi.make_tokens(cfg, 0)).cuda()),
             (2, torch.as_tensor(mi.make_tokens(cfg, 5)).cuda())]

    # regular entry point, caller-allocated arena
    ref = MoETrainer(cfg, "cuda:0")
    ref.load_params(params)
    # the same state for the no-allocation entry point, in plain torch buffers
    p = ref.params.clone()
    g = torch.zeros_like(ref.grads)
    m = torch.zeros_like(ref.adam_m)
    v = torch.zeros_like(ref.adam_v)
    stream = torch.cuda.current_stream().cuda_stream

    for step, tok in calls:
        ref.micro_step(tok, 0, step=step)
        out_ref = ref.outputs()
        assert out_ref.status == B.MT_OK

        out = B.mt_outputs()
        st = B.mt_train_update_noalloc(p.data_ptr(), 0, g.data_ptr(), m.data_ptr(), v.data_ptr(),
                                       tok.data_ptr(), B.hparams(cfg, step=step), out, stream)
        assert st == B.MT_OK, B.status_string(st)
        assert out.status == B.MT_OK and out.optimizer_ran == 1
        assert abs(out.loss - out_ref.loss) <= TINY_TOL * abs(out_ref.loss)
        assert abs(out.grad_norm - out_ref.grad_norm) <= TINY_TOL * out_ref.grad_norm
        for name in ref.layout:
            for mine, theirs in ((p, ref.params), (g, ref.grads), (m, ref.adam_m), (v, ref.adam_v)):
                a, b = to_np(ref.view(mine, name)), to_np(ref.view(theirs, name))
                assert rel_l2(a, b) <= TINY_TOL, (step, name)


def test_noalloc_rejects_a_model_larger_than_its_array():
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("b2")
    hp = B.hparams(cfg)
    assert B.mt_arena_bytes(hp) > B.MT_NOALLOC_ARENA_BYTES
    fake = 1 << 20          # never dereferenced: the size check fails first
    st = B.mt_train_update_noalloc(fake, fake, fake, fake, fake, fake, hp, None, 0)
    assert st == B.MT_ERR_ARENA_SMALL
