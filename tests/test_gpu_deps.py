"""Per-block dependency counters against grid barriers.  With counters on
(the default wherever the tensor-core products and attention run), the
hand-offs qkv -> attention -> out-projection -> router, gate/up -> down,
combine -> next layer and (backward) qkv dgrad -> attention-norm backward
wait per 128-row block instead of at a grid barrier, the attention-norm
backward hands its rows to the next layer's expert-combine backward on the
same CTA,
and attention items are drawn from ticket counters.  Every item still
computes the same values in the same order, so the update must equal the
barrier-only schedule bit for bit."""
import pytest
import torch

import moe_inputs as mi

pytestmark = pytest.mark.gpu


def _run(cfg, flags):
    from adamw_persistent_sm_gb300 import binding as B
    from adamw_persistent_sm_gb300.trainer import MoETrainer
    tr = MoETrainer(cfg, "cuda:0", flags=flags)
    tr.load_params(mi.make_params(cfg))
    tr.update([torch.as_tensor(t).cuda() for t in mi.make_update_tokens(cfg)])
    out = tr.outputs()
    assert out.status == B.MT_OK, (B.status_string(out.status), out.error_site)
    torch.cuda.synchronize()
    return tr, out


@pytest.mark.parametrize("name", ["b2", "top8"])
def test_counters_equal_barriers_bit_for_bit(name):
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    t_dep, o_dep = _run(cfg, 0)
    t_bar, o_bar = _run(cfg, B.MT_FLAG_BARRIERS_ONLY)
    assert o_dep.loss == o_bar.loss
    assert o_dep.grad_norm == o_bar.grad_norm
    assert torch.equal(t_dep.grads, t_bar.grads)
    assert torch.equal(t_dep.params, t_bar.params)
    assert torch.equal(t_dep.adam_m, t_bar.adam_m)
    assert torch.equal(t_dep.adam_v, t_bar.adam_v)
    # five forward barriers per layer, the backward's qkv dgrad -> norm
    # backward barrier (counters) and, above layer 0, the norm backward ->
    # next layer's expert-combine backward barrier (same token chunk per CTA)
    # are gone
    assert o_bar.n_phases - o_dep.n_phases == 7 * cfg.n_layers - 1


def test_counters_are_deterministic_across_launches():
    cfg = mi.get_config("b2")
    t1, o1 = _run(cfg, 0)
    t2, o2 = _run(cfg, 0)
    assert o1.loss == o2.loss
    assert torch.equal(t1.params, t2.params)


@pytest.mark.parametrize("name", ["b2", "tiny"])
def test_expert_activation_recompute_is_bit_identical(name):
    """The memory rule that re-runs each layer's gate/up product in the
    backward (one layer of expert activations kept) gives the default plan's
    update bit for bit: same tiles, same inputs, same accumulation order."""
    from adamw_persistent_sm_gb300 import binding as B
    cfg = mi.get_config(name)
    base, _ = _run(cfg, 0)
    rule, _ = _run(cfg, B.MT_FLAG_RECOMPUTE_EXPERT_ACT)
    assert rule.arena_bytes < base.arena_bytes
    for buf in ("grads", "params", "adam_m", "adam_v"):
        assert torch.equal(getattr(base, buf), getattr(rule, buf)), buf
