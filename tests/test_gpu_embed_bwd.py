"""Embedding backward with one token id at every position of a 32 x 1024
batch.  The embedding is a row gather, so its gradient is a scatter-add:
dE[v] = sum over the positions t with tok[t] = v of dx_t, added in
ascending t ("How a training megakernel works", section "1 - Describe the
model and update").  Here every match falls into the vocabulary rows of
one CTA, whose match list fills and is added in several rounds (flushes in
the middle of the scan).  The row must equal the position-ordered fp32 sum
of the dx rows the kernel read (debug view) bit for bit, and every other
row must be zero."""
import numpy as np
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


def test_embedding_backward_repeated_token_equals_ordered_sum():
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    cfg = mi.get_config("b32")
    tr = MoETrainer(cfg, "cuda:0", flags=B.MT_FLAG_NO_OPTIMIZER)
    tr.load_params(mi.make_params(cfg))
    vid = 7
    tok = torch.full((cfg.batch, cfg.seq), vid, dtype=torch.int32, device="cuda:0")
    tr.update([tok])
    out = tr.outputs()
    assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
    torch.cuda.synchronize()
    T, d = cfg.batch * cfg.seq, cfg.d_model
    dx = tr.debug_view(B.MT_VIEW_DX, 0, torch.float32)[:T * d].view(T, d).cpu().numpy()
    dE = tr.named(tr.grads)["emb"].cpu().numpy()
    ref = np.zeros(d, dtype=np.float32)
    for t in range(T):
        ref = ref + dx[t]            # fp32 adds in ascending position, as the kernel does
    assert np.array_equal(dE[vid], ref)
    assert np.count_nonzero(np.delete(dE, vid, axis=0)) == 0
