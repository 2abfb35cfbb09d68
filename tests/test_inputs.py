"""The seeded synthetic inputs (CPU): the same seed gives the same tensors, the recipe's
distributions hold (mean / spread / ranges), and the core inputs have unit q, k rows."""
import math

import torch

from gated_deltanet_linear_conv_gb300 import inputs as I


def test_mixer_inputs_are_deterministic_per_seed():
    a = I.make_mixer_inputs(7, [5, 64, 3], conv_state_std=1.0, S0_std=0.02)
    b = I.make_mixer_inputs(7, [5, 64, 3], conv_state_std=1.0, S0_std=0.02)
    c = I.make_mixer_inputs(8, [5, 64, 3], conv_state_std=1.0, S0_std=0.02)
    for name in ('mixed_qkv', 'conv_w', 'conv_state', 'a', 'b', 'A_log', 'dt_bias', 'z', 'norm_w', 'S0'):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert not torch.equal(a.mixed_qkv, c.mixed_qkv)
    assert a.cu_seqlens().tolist() == [0, 5, 69, 72]


def test_mixer_recipe_distributions():
    inp = I.make_mixer_inputs(1, [64])                  # the prefill recipe at 64 tokens
    sh = inp.shape
    assert inp.mixed_qkv.shape == (64, sh.C) and inp.mixed_qkv.dtype == torch.bfloat16
    x = inp.mixed_qkv.float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    assert abs(inp.conv_w.float().std().item() - 0.25) < 0.01
    assert inp.conv_state is None and inp.S0 is None       # zero states are passed as None
    assert 0.0 <= inp.A_log.min().item() and inp.A_log.max().item() <= math.log(16.0)
    assert -1.0 <= inp.dt_bias.min().item() and inp.dt_bias.max().item() <= 1.0
    assert abs(inp.norm_w.mean().item() - 1.0) < 0.05 and inp.norm_w.std().item() < 0.2
    assert inp.z.shape == (64, sh.Nv, sh.Dv)


def test_random_lengths_stay_in_range():
    inp = I.make_mixer_inputs(3, random_lengths=(16, 5, 9), shape=I.MixerShape(1, 2, 64, 64))
    assert len(inp.lengths) == 16 and all(5 <= L <= 9 for L in inp.lengths)
    assert inp.total_tokens == sum(inp.lengths)


def test_tiny_core_workload_has_unit_keys():
    c = I.workload('tiny_core_t256')
    assert c.q.shape == (256, 2, 64) and c.v.shape == (256, 2, 64)
    for t in (c.q, c.k):
        n = t.double().norm(dim=-1)
        assert torch.allclose(n, torch.ones_like(n), atol=1e-5)
