"""Seeded synthetic inputs for the Gated DeltaNet mixer workloads.

Shared by the tests, the bench and the oracle checks.  This module holds
random draws, dtype casts and shapes only -- none of the mixer's arithmetic.
Every draw comes from one CPU ``torch.Generator`` seeded per workload, in
fp32, in a fixed order, then cast; the exact host tensors are what both the
CUDA path and the oracle consume.

Draw order: lengths (packed workloads) -> mixed_qkv -> conv_w -> conv_state
-> a -> b -> A_log -> dt_bias -> z -> norm_w -> S0.

"N(m, s)" means mean m and standard deviation s.
"""

import math
from dataclasses import dataclass, field

import torch


@dataclass
class MixerShape:
    Nk: int
    Nv: int
    Dk: int
    Dv: int

    @property
    def C(self):
        return 2 * self.Nk * self.Dk + self.Nv * self.Dv


QWEN_SHAPE = MixerShape(Nk=16, Nv=32, Dk=128, Dv=128)


@dataclass
class MixerInputs:
    shape: MixerShape
    lengths: list
    mixed_qkv: torch.Tensor          # [tokens, C]
    conv_w: torch.Tensor             # [C, 4]
    conv_state: torch.Tensor         # [N, C, 3] or None (zeros)
    a: torch.Tensor                  # [tokens, Nv]
    b: torch.Tensor                  # [tokens, Nv]
    A_log: torch.Tensor              # [Nv] fp32
    dt_bias: torch.Tensor            # [Nv] fp32
    z: torch.Tensor                  # [tokens, Nv, Dv]
    norm_w: torch.Tensor             # [Dv] fp32
    S0: torch.Tensor                 # [N, Nv, Dk, Dv] fp32 or None (zeros)
    extra: dict = field(default_factory=dict)

    @property
    def num_seqs(self):
        return len(self.lengths)

    @property
    def total_tokens(self):
        return int(sum(self.lengths))

    def cu_seqlens(self):
        cu = [0]
        for L in self.lengths:
            cu.append(cu[-1] + int(L))
        return torch.tensor(cu, dtype=torch.int32)


def _normal(gen, shape, mean, std):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * std + mean


def _uniform(gen, shape, lo, hi):
    return torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo


def make_mixer_inputs(seed, lengths=None, shape=QWEN_SHAPE, dtype=torch.bfloat16,
                      conv_w_std=0.25, conv_state_std=None, A_log_range=(0.0, math.log(16.0)),
                      S0_std=None, random_lengths=None, conv_bias_std=None):
    """Draw one mixer workload.

    lengths: list of per-sequence token counts, or None when ``random_lengths``
    = (num_seqs, lo, hi) asks for lengths ~ U[lo, hi] (inclusive).
    conv_state_std / S0_std: None means a zero state (passed as None).
    """
    gen = torch.Generator().manual_seed(seed)
    if random_lengths is not None:
        n, lo, hi = random_lengths
        lengths = [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]
    lengths = [int(L) for L in lengths]
    T = sum(lengths)
    N = len(lengths)
    C = shape.C
    mixed = _normal(gen, (T, C), 0.0, 1.0).to(dtype)
    conv_w = _normal(gen, (C, 4), 0.0, conv_w_std).to(dtype)
    conv_state = None
    if conv_state_std is not None:
        conv_state = _normal(gen, (N, C, 3), 0.0, conv_state_std).to(dtype)
    a = _normal(gen, (T, shape.Nv), 0.0, 1.0).to(dtype)
    b = _normal(gen, (T, shape.Nv), 0.0, 1.0).to(dtype)
    A_log = _uniform(gen, (shape.Nv,), A_log_range[0], A_log_range[1])
    dt_bias = _uniform(gen, (shape.Nv,), -1.0, 1.0)
    z = _normal(gen, (T, shape.Nv, shape.Dv), 0.0, 1.0).to(dtype)
    norm_w = _normal(gen, (shape.Dv,), 1.0, 0.1)
    S0 = None
    if S0_std is not None:
        S0 = _normal(gen, (N, shape.Nv, shape.Dk, shape.Dv), 0.0, S0_std)
    extra = {}
    if conv_bias_std is not None:
        extra['conv_bias'] = _normal(gen, (C,), 0.0, conv_bias_std).to(dtype)
    return MixerInputs(shape, lengths, mixed, conv_w, conv_state, a, b, A_log, dt_bias, z,
                       norm_w, S0, extra)


@dataclass
class CoreInputs:
    """Inputs of the delta-rule core alone (q, k, v, gate pre-activations)."""
    shape: MixerShape
    lengths: list
    q: torch.Tensor      # [tokens, Nk, Dk], unit rows
    k: torch.Tensor      # [tokens, Nk, Dk], unit rows
    v: torch.Tensor      # [tokens, Nv, Dv]
    a: torch.Tensor      # [tokens, Nv]
    b: torch.Tensor      # [tokens, Nv]
    A_log: torch.Tensor  # [Nv]
    dt_bias: torch.Tensor
    S0: torch.Tensor     # [N, Nv, Dk, Dv] or None

    def cu_seqlens(self):
        cu = [0]
        for L in self.lengths:
            cu.append(cu[-1] + int(L))
        return torch.tensor(cu, dtype=torch.int32)


def _unit_rows(x):
    # a N(0, I) vector divided by its length is uniform on the unit sphere
    return x / x.norm(dim=-1, keepdim=True)


def make_core_inputs(seed, lengths, shape, dtype=torch.float32, S0_std=None,
                     A_log_range=(0.0, math.log(16.0))):
    """q, k ~ uniform on the unit sphere (normalised N(0, 1)), v, a, b ~ N(0, 1),
    A_log ~ U(A_log_range), dt_bias ~ U(-1, 1).  Draw order q -> k -> v -> a ->
    b -> A_log -> dt_bias -> S0."""
    gen = torch.Generator().manual_seed(seed)
    T = sum(int(L) for L in lengths)
    N = len(lengths)
    q = _unit_rows(_normal(gen, (T, shape.Nk, shape.Dk), 0.0, 1.0)).to(dtype)
    k = _unit_rows(_normal(gen, (T, shape.Nk, shape.Dk), 0.0, 1.0)).to(dtype)
    v = _normal(gen, (T, shape.Nv, shape.Dv), 0.0, 1.0).to(dtype)
    a = _normal(gen, (T, shape.Nv), 0.0, 1.0).to(dtype)
    b = _normal(gen, (T, shape.Nv), 0.0, 1.0).to(dtype)
    A_log = _uniform(gen, (shape.Nv,), A_log_range[0], A_log_range[1])
    dt_bias = _uniform(gen, (shape.Nv,), -1.0, 1.0)
    S0 = None
    if S0_std is not None:
        S0 = _normal(gen, (N, shape.Nv, shape.Dk, shape.Dv), 0.0, S0_std)
    return CoreInputs(shape, [int(L) for L in lengths], q, k, v, a, b, A_log, dt_bias, S0)


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

WORKLOADS = {
    'tiny_core_t256': dict(kind='core', seed=0, lengths=[256],
                           shape=MixerShape(2, 2, 64, 64)),
    'prefill_t4096': dict(kind='mixer', seed=1, lengths=[4096]),
    'decode_b256': dict(kind='decode', seed=2, lengths=[1] * 256),
    'varlen_16seq': dict(kind='mixer', seed=3, random_lengths=(16, 512, 8192)),
    'prefill_t131072': dict(kind='mixer', seed=4, lengths=[131072],
                            A_log_range=(-4.0, 0.0)),
}


def workload(name):
    """Draw one of the five named workloads.

    tiny_core_t256  : B=1, T=256, Nk=Nv=2, Dk=Dv=64, fp32 core inputs, zero state.
    prefill_t4096   : B=1, T=4096, C=8192 bf16 mixed_qkv, zero conv/recurrent state.
    decode_b256     : B=256 sequences, one token each; conv state N(0,1) bf16,
                      recurrent state N(0, 0.02) fp32.
    varlen_16seq    : 16 sequences, lengths ~ U[512, 8192], packed; recurrent
                      state N(0, 0.02) per sequence; zero conv state.
    prefill_t131072 : B=1, T=131072, A_log ~ U(-4, 0) (slow decay).
    """
    spec = dict(WORKLOADS[name])
    kind = spec.pop('kind')
    if kind == 'core':
        return make_core_inputs(spec['seed'], spec['lengths'], spec['shape'])
    if kind == 'decode':
        return make_mixer_inputs(spec['seed'], spec['lengths'], conv_state_std=1.0,
                                 S0_std=0.02)
    if name == 'varlen_16seq':
        return make_mixer_inputs(spec['seed'], random_lengths=spec['random_lengths'],
                                 S0_std=0.02)
    return make_mixer_inputs(spec['seed'], spec['lengths'],
                             A_log_range=spec.get('A_log_range', (0.0, math.log(16.0))))


# ---------------------------------------------------------------------------
# generic seeded draws for tests of single steps
# ---------------------------------------------------------------------------

def draw_normal(seed, shape, mean=0.0, std=1.0, dtype=torch.float32):
    """N(mean, std) of the given shape from a generator seeded with ``seed``."""
    gen = torch.Generator().manual_seed(seed)
    return _normal(gen, tuple(shape), mean, std).to(dtype)


def draw_uniform(seed, shape, lo, hi, dtype=torch.float32):
    """U(lo, hi) of the given shape from a generator seeded with ``seed``."""
    gen = torch.Generator().manual_seed(seed)
    return _uniform(gen, tuple(shape), lo, hi).to(dtype)
