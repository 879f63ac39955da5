"""The attention forward on tcgen05 (TMEM accumulators, TMA-fed K/V ring,
softmax warps) against the warp-level mma.sync forward on the same inputs:
both round P to bf16 before the PV product and accumulate in fp32, so the
update agrees up to accumulation order."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from parity_util import rel_l2, to_np

pytestmark = pytest.mark.gpu


def _run(cfg, flags):
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = MoETrainer(cfg, "cuda:0", flags=flags)
    tr.load_params(mi.make_params(cfg))
    tr.update([torch.as_tensor(t).cuda() for t in mi.make_update_tokens(cfg)], flags=flags | B.MT_FLAG_NO_OPTIMIZER)
    out = tr.outputs()
    assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
    return tr, out


@pytest.mark.parametrize("name", ["b2", "top8"])
def test_tcgen05_forward_matches_mma_sync(name):
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    t_tm, o_tm = _run(cfg, 0)
    t_ms, o_ms = _run(cfg, B.MT_FLAG_MMA_SYNC_ATTN)
    assert abs(o_tm.loss - o_ms.loss) / o_ms.loss < 2e-3
    tl_tm = to_np(t_tm.debug_view(B.MT_VIEW_TOK_LOSS))
    tl_ms = to_np(t_ms.debug_view(B.MT_VIEW_TOK_LOSS))
    assert rel_l2(tl_tm, tl_ms) < 1e-2
    # the first layer's attention output feeds the rest of the forward: compare
    # the hidden state entering layer 1 (fp32 residual stream)
    h_tm = to_np(t_tm.debug_view(B.MT_VIEW_HIDDEN, 1))
    h_ms = to_np(t_ms.debug_view(B.MT_VIEW_HIDDEN, 1))
    assert rel_l2(h_tm, h_ms) < 5e-3
    g_tm, g_ms = t_tm.named(t_tm.grads), t_ms.named(t_ms.grads)
    for k in ("wqkv", "wo", "attn_norm", "lm_head"):
        assert rel_l2(to_np(g_tm[k]), to_np(g_ms[k])) < 0.05, k
