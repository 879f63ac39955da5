"""Runtime behaviour on the GPU: a bounded grid-barrier wait that runs out
(no GPU fault: one CTA never arrives, the others give up after 2 ms and the
status word says so), recovery after mt_arena_init, an out-of-range token
reported without a fault, and the per-CTA phase trace."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle
from parity_util import TINY_TOL

pytestmark = pytest.mark.gpu


def _trainer(cfg, **kw):
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = MoETrainer(cfg, "cuda:0", **kw)
    tr.load_params(mi.make_params(cfg))
    return tr


def test_barrier_timeout_is_reported_and_recoverable():
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("tiny")
    tr = _trainer(cfg, wait_timeout_ns=2_000_000)
    toks = [torch.as_tensor(t).cuda() for t in mi.make_update_tokens(cfg)]
    tr.update(toks, flags=B.MT_FLAG_TEST_STALL)
    out = tr.outputs()
    assert out.status == B.MT_ERR_DEVICE_TIMEOUT
    assert out.error_site == 1                     # the grid barrier
    # the context is intact: re-initialise the arena and run a normal update
    tr.load_params(mi.make_params(cfg))
    tr.grads.zero_()
    tr.reset_arena()
    tr.update(toks, flags=0)
    out = tr.outputs()
    assert out.status == B.MT_OK
    ref = oracle.train_update(mi.make_params(cfg), mi.make_update_tokens(cfg), cfg)
    assert abs(out.loss - ref.loss) / ref.loss < TINY_TOL


def test_out_of_range_token_sets_bounds_status():
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("tiny")
    tr = _trainer(cfg)
    tok = mi.make_tokens(cfg, 0)
    tok[1, 5] = cfg.vocab                        # one past the end: clamped and reported
    tr.update([torch.as_tensor(tok).cuda()])
    out = tr.outputs()
    assert out.status == B.MT_ERR_DEVICE_BOUNDS and out.error_site == 2
    tr.reset_arena()


def test_phase_trace():
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config("tiny")
    tr = _trainer(cfg, flags=B.MT_FLAG_TRACE)
    tr.update([torch.as_tensor(t).cuda() for t in mi.make_update_tokens(cfg)])
    out = tr.outputs()
    assert out.status == B.MT_OK
    tv = tr.debug_view(B.MT_VIEW_TRACE, 0, torch.int64).cpu().numpy().reshape(-1, B.MT_TRACE_WORDS)
    tv = tv[:, :2 * B.MT_TRACE_PHASES].reshape(-1, B.MT_TRACE_PHASES, 2)
    tv = tv[:out.n_ctas, :out.n_phases]
    assert np.all(tv[:, :, 1] >= tv[:, :, 0])
    assert np.all(np.diff(tv[:, :, 0], axis=1) >= 0)
    # every CTA leaves barrier p at about the same time
    spread = tv[:, :, 1].max(axis=0) - tv[:, :, 1].min(axis=0)
    assert np.median(spread) < 1_000_000
