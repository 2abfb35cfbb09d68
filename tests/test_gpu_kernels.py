"""Parity of every CUDA entry point with the fp64 oracle at small sizes that
still span several tiles, ragged tails, empty sequences and both head sizes.
All calls go through the C ABI (libgdn.so via the ctypes binding)."""

import math

import numpy as np
import pytest
import torch

import oracle as O
from gated_deltanet_linear_conv_gb300 import gdn
from gated_deltanet_linear_conv_gb300 import inputs as I
from helpers import TOL_BF16, TOL_F32, assert_close, np64

pytestmark = pytest.mark.gpu

SHAPES = [I.MixerShape(2, 4, 128, 128), I.MixerShape(2, 2, 64, 64)]


def cuda(t):
    return None if t is None else t.cuda()


# ------------------------------------------------------------------ rmsnorm

@pytest.mark.parametrize('dim', [64, 128])
@pytest.mark.parametrize('xdt', [torch.float32, torch.bfloat16])
@pytest.mark.parametrize('rows', [0, 1, 1237])
def test_gated_rmsnorm(dim, xdt, rows):
    x = I.draw_normal(1, (rows, dim), dtype=xdt)
    z = I.draw_normal(2, (rows, dim), dtype=xdt)
    w = I.draw_normal(3, (dim,), 1.0, 0.1)
    y = gdn.gated_rmsnorm(cuda(x), cuda(z), cuda(w), 1e-6, torch.float32)
    torch.cuda.synchronize()
    if rows == 0:
        return
    ref = O.gated_rmsnorm(np64(x), np64(z), np64(w), 1e-6)
    assert_close(np64(y), ref, TOL_F32)
    yb = gdn.gated_rmsnorm(cuda(x), cuda(z), cuda(w), 1e-6, torch.bfloat16)
    assert_close(np64(yb), ref, TOL_BF16)


# ------------------------------------------------------------------ gating

@pytest.mark.parametrize('dt', [torch.float32, torch.bfloat16])
def test_gating(dt):
    rows, Nv = 777, 6
    a = I.draw_normal(4, (rows, Nv), 0.0, 3.0, dtype=dt)
    b = I.draw_normal(5, (rows, Nv), 0.0, 3.0, dtype=dt)
    A_log = I.draw_uniform(6, (Nv,), -4.0, math.log(16.0))
    dt_bias = I.draw_uniform(7, (Nv,), -1.0, 1.0)
    g, beta = gdn.gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    rg, rb = O.gating(np64(a), np64(b), np64(A_log), np64(dt_bias))
    assert_close(np64(g), rg, TOL_F32)
    assert_close(np64(beta), rb, TOL_F32)


# ------------------------------------------------------------------ conv + gating

def _conv_case(shape, dt, lengths, seed=11, state=True, bias=True):
    return I.make_mixer_inputs(seed, lengths, shape, dtype=dt,
                               conv_state_std=1.0 if state else None,
                               conv_bias_std=0.1 if bias else None)


def _run_conv(inp, cu, out_dtype, in_place=False, state=True):
    sh = inp.shape
    cs_in = cuda(inp.conv_state) if state else None
    if in_place:
        cs_out = cs_in
    else:
        cs_out = torch.empty(inp.num_seqs, sh.C, 3, dtype=inp.mixed_qkv.dtype, device='cuda')
    res = gdn.conv_gating(cuda(inp.mixed_qkv), cuda(inp.conv_w), cuda(inp.a), cuda(inp.b),
                          cuda(inp.A_log), cuda(inp.dt_bias), sh.Nk, sh.Nv, sh.Dk, sh.Dv,
                          cu_seqlens=cuda(cu), num_seqs=inp.num_seqs,
                          conv_bias=cuda(inp.extra.get('conv_bias')), conv_state_in=cs_in,
                          conv_state_out=cs_out, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return res, cs_out


def _oracle_conv(inp, cu, state=True):
    sh = inp.shape
    return O.conv_gating(np64(inp.mixed_qkv), np64(inp.conv_w), np64(inp.a), np64(inp.b),
                         np64(inp.A_log), np64(inp.dt_bias), sh.Nk, sh.Nv, sh.Dk, sh.Dv,
                         cu_seqlens=None if cu is None else cu.numpy(), num_seqs=inp.num_seqs,
                         conv_bias=np64(inp.extra.get('conv_bias')),
                         conv_state=np64(inp.conv_state) if state else None)


@pytest.mark.parametrize('shape', SHAPES, ids=['d128', 'd64'])
@pytest.mark.parametrize('dt', [torch.float32, torch.bfloat16], ids=['f32', 'bf16'])
def test_conv_gating_varlen(shape, dt):
    lengths = [1, 2, 5, 0, 37, 64, 130, 3]
    inp = _conv_case(shape, dt, lengths)
    cu = inp.cu_seqlens()
    (q, k, v, g, beta), cs_out = _run_conv(inp, cu, torch.float32)
    ref = _oracle_conv(inp, cu)
    for name, got in (('q', q), ('k', k), ('v', v), ('g', g), ('beta', beta)):
        assert_close(np64(got), ref[name], TOL_F32, what=name)
    np.testing.assert_array_equal(np64(cs_out), ref['conv_state'])
    gdn.check_device_error()


@pytest.mark.parametrize('shape', SHAPES, ids=['d128', 'd64'])
def test_conv_gating_in_place_state_and_bf16_out(shape):
    lengths = [2, 70, 1, 19]
    inp = _conv_case(shape, torch.bfloat16, lengths, seed=12)
    cu = inp.cu_seqlens()
    ref = _oracle_conv(inp, cu)
    (q, k, v, g, beta), cs = _run_conv(inp, cu, torch.bfloat16, in_place=True)
    np.testing.assert_array_equal(np64(cs), ref['conv_state'])
    for name, got in (('q', q), ('k', k), ('v', v)):
        assert_close(np64(got), ref[name], TOL_BF16, what=name)


@pytest.mark.parametrize('lengths', [[1, 2, 5, 0, 37, 64, 130, 3], [0, 16, 0, 2, 30, 0], [40]],
                         ids=['mixed', 'empties', 'one'])
def test_conv_gating_state_out_without_state_in(lengths):
    """The tiled bf16 path writes the new conv state from its staged rows when there is no
    state in (zeros before a sequence's first token, and for empty sequences)."""
    shape = SHAPES[0]
    inp = _conv_case(shape, torch.bfloat16, lengths, seed=14, state=False)
    cu = inp.cu_seqlens()
    (q, k, v, g, beta), cs_out = _run_conv(inp, cu, torch.bfloat16, state=False)
    ref = _oracle_conv(inp, cu, state=False)
    np.testing.assert_array_equal(np64(cs_out), ref['conv_state'])
    for name, got in (('q', q), ('k', k), ('v', v)):
        assert_close(np64(got), ref[name], TOL_BF16, what=name)
    gdn.check_device_error()


@pytest.mark.parametrize('bias,state', [(True, True), (False, False), (False, True)],
                         ids=['bias_state', 'plain', 'state'])
@pytest.mark.parametrize('odt', [torch.float32, torch.bfloat16], ids=['f32', 'bf16'])
def test_conv_gating_tiled_64_wide_heads(bias, state, odt):
    """The tiled bf16 kernel with 64-wide q/k heads (8 lanes per head in the L2 norm) on a
    shape whose channels fill whole 1024-channel blocks (Nk = 8, Nv = 16: C = 2048), with and
    without bias and conv state, ragged and empty sequences, every channel block rotating
    over the CTAs."""
    shape = I.MixerShape(8, 16, 64, 64)
    lengths = [1, 40, 0, 3, 130, 17, 64, 2]
    inp = _conv_case(shape, torch.bfloat16, lengths, seed=15, state=state, bias=bias)
    cu = inp.cu_seqlens()
    (q, k, v, g, beta), cs_out = _run_conv(inp, cu, odt, state=state)
    ref = _oracle_conv(inp, cu, state=state)
    tol = TOL_F32 if odt == torch.float32 else TOL_BF16
    for name, got in (('q', q), ('k', k), ('v', v)):
        assert_close(np64(got), ref[name], tol, what=name)
    for name, got in (('g', g), ('beta', beta)):
        assert_close(np64(got), ref[name], TOL_F32, what=name)
    np.testing.assert_array_equal(np64(cs_out), ref['conv_state'])
    gdn.check_device_error()


def test_conv_gating_equal_batches_no_state():
    shape = SHAPES[0]
    inp = _conv_case(shape, torch.bfloat16, [33, 33, 33], seed=13, state=False, bias=False)
    (q, k, v, g, beta), cs_out = _run_conv(inp, None, torch.float32, state=False)
    ref = _oracle_conv(inp, None, state=False)
    for name, got in (('q', q), ('k', k), ('v', v), ('g', g), ('beta', beta)):
        assert_close(np64(got), ref[name], TOL_F32, what=name)
    np.testing.assert_array_equal(np64(cs_out), ref['conv_state'])


# ------------------------------------------------------------------ recurrent decode

@pytest.mark.parametrize('shape', SHAPES + [I.MixerShape(1, 2, 128, 64), I.MixerShape(2, 2, 64, 128)],
                         ids=['d128', 'd64', 'k128v64', 'k64v128'])
def test_recurrent_decode_multi_token(shape):
    lengths = [1, 4, 2, 3]                   # one-token decode and multi-token verify
    c = I.make_core_inputs(21, lengths, shape, S0_std=0.5)
    g, beta = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
    gt, bt = torch.tensor(g, dtype=torch.float32), torch.tensor(beta, dtype=torch.float32)
    cu = c.cu_seqlens()
    state = cuda(c.S0.clone())
    o = gdn.recurrent_decode(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), state, 0.3,
                             cu_seqlens=cuda(cu), out_dtype=torch.float32)
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt), 0.3,
                                          np64(c.S0), cu.numpy())
    assert_close(np64(o), ro, TOL_F32)
    assert_close(np64(state), rS, TOL_F32)


@pytest.mark.parametrize('shape', SHAPES, ids=['d128', 'd64'])
def test_recurrent_decode_step_states(shape):
    """Draft + verify decode (1 + 3 tokens per sequence): the state after every
    token equals the recurrence over that prefix, and restarting from one of
    them (a rollback to the last accepted token) reproduces the rest."""
    lengths = [4, 4, 4]
    c = I.make_core_inputs(57, lengths, shape, dtype=torch.float32, S0_std=0.1)
    gt, bt = _core_gates(c)
    cu = c.cu_seqlens()
    S = cuda(c.S0.clone())
    steps = torch.empty(sum(lengths), shape.Nv, shape.Dk, shape.Dv, device='cuda')
    o = gdn.recurrent_decode(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), S, 0.3,
                             cu_seqlens=cuda(cu), out_dtype=torch.float32, step_states=steps)
    torch.cuda.synchronize()
    cu_l = cu.tolist()
    for s in range(len(lengths)):
        b0, b1 = cu_l[s], cu_l[s + 1]
        for j in range(b1 - b0):
            sub = slice(b0, b0 + j + 1)
            _, Sj = O.recurrent_gated_delta_rule(np64(c.q[sub]), np64(c.k[sub]), np64(c.v[sub]), np64(gt[sub]),
                                                 np64(bt[sub]), 0.3, np64(c.S0[s:s + 1]))
            assert_close(np64(steps[b0 + j]), Sj[0], TOL_F32, what=(s, j))
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt), 0.3,
                                          np64(c.S0), cu.numpy())
    assert_close(np64(o), ro, TOL_F32)
    assert_close(np64(S), rS, TOL_F32)
    for s in range(len(lengths)):
        assert torch.equal(steps[cu_l[s + 1] - 1], S[s])        # the last step is the final state
    # roll sequence 1 back to its second token and replay its last two tokens
    b0 = cu_l[1]
    S1 = steps[b0 + 1:b0 + 2].clone()
    tail = slice(b0 + 2, b0 + 4)
    o_tail = gdn.recurrent_decode(cuda(c.q[tail]), cuda(c.k[tail]), cuda(c.v[tail]), cuda(gt[tail]),
                                  cuda(bt[tail]), S1, 0.3, num_seqs=1, out_dtype=torch.float32)
    torch.testing.assert_close(o_tail, o[tail], rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(S1[0], S[1], rtol=1e-5, atol=1e-6)


def test_gpu_gating_feeds_decode():
    """gdn_gating + gdn_recurrent_decode on the tiny workload vs the oracle."""
    c = I.workload('tiny_core_t256')
    sh = c.shape
    g, beta = gdn.gating(cuda(c.a), cuda(c.b), cuda(c.A_log), cuda(c.dt_bias))
    state = torch.zeros(1, sh.Nv, sh.Dk, sh.Dv, device='cuda')
    o = gdn.recurrent_decode(cuda(c.q), cuda(c.k), cuda(c.v), g, beta, state, 1 / 8,
                             num_seqs=1, out_dtype=torch.float32)
    rg, rb = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), rg, rb, 1 / 8)
    assert_close(np64(o), ro, TOL_F32)
    assert_close(np64(state), rS, TOL_F32)


# ------------------------------------------------------------------ fused decode

@pytest.mark.parametrize('shape', SHAPES + [I.MixerShape(1, 4, 128, 128)], ids=['d128', 'd64', 'r4'])
def test_decode_fused_two_steps(shape):
    B = 5
    inp = I.make_mixer_inputs(31, [2] * B, shape, conv_state_std=1.0, S0_std=0.05)
    sh = inp.shape
    mixed = inp.mixed_qkv.view(B, 2, sh.C)
    a = inp.a.view(B, 2, sh.Nv)
    b = inp.b.view(B, 2, sh.Nv)
    z = inp.z.view(B, 2, sh.Nv, sh.Dv)
    cs, S = cuda(inp.conv_state.clone()), cuda(inp.S0.clone())
    rcs, rS = np64(inp.conv_state), np64(inp.S0)
    for step in range(2):
        y = gdn.decode_fused(cuda(mixed[:, step].contiguous()), cuda(inp.conv_w), cs,
                             cuda(a[:, step].contiguous()), cuda(b[:, step].contiguous()),
                             cuda(inp.A_log), cuda(inp.dt_bias), S, cuda(z[:, step].contiguous()),
                             cuda(inp.norm_w), sh.Nk, sh.Nv, sh.Dk, sh.Dv, out_dtype=torch.float32)
        ref = O.decode_step(np64(mixed[:, step]), np64(inp.conv_w), rcs, np64(a[:, step]),
                            np64(b[:, step]), np64(inp.A_log), np64(inp.dt_bias), rS,
                            np64(z[:, step]), np64(inp.norm_w), sh.Nk, sh.Nv, sh.Dk, sh.Dv)
        rcs, rS = ref['conv_state'], ref['state']
        assert_close(np64(y), ref['y'], TOL_F32, what=step)
        assert_close(np64(S), rS, TOL_F32, what=step)
        np.testing.assert_array_equal(np64(cs), rcs)


# ------------------------------------------------------------------ chunk prefill

CHUNK_LENGTHS = [[1], [63], [64], [65], [200], [0, 5, 0, 70, 128, 1]]


def _core_gates(c):
    g, beta = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
    return torch.tensor(g, dtype=torch.float32), torch.tensor(beta, dtype=torch.float32)


@pytest.mark.parametrize('fp32', [True, False], ids=['fp32', 'tc'])
@pytest.mark.parametrize('shape', SHAPES, ids=['d128', 'd64'])
@pytest.mark.parametrize('lengths', CHUNK_LENGTHS, ids=lambda L: 'L' + '_'.join(map(str, L)))
def test_chunk_prefill_varlen(fp32, shape, lengths):
    # the main entry point takes bf16 q/k/v (tensor cores at 128-wide heads);
    # the fp32 entry point takes fp32 q/k/v.  The oracle sees the same values.
    c = I.make_core_inputs(41, lengths, shape, dtype=torch.float32 if fp32 else torch.bfloat16,
                           S0_std=0.1)
    gt, bt = _core_gates(c)
    cu = c.cu_seqlens()
    o, ST = gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), 0.2,
                              initial_state=cuda(c.S0), cu_seqlens=cuda(cu),
                              out_dtype=torch.float32, fp32=fp32)
    torch.cuda.synchronize()
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt), 0.2,
                                          np64(c.S0), cu.numpy())
    tol = TOL_F32 if fp32 else TOL_BF16
    if sum(lengths) > 0:
        assert_close(np64(o), ro, tol)
    assert_close(np64(ST), rS, tol)
    gdn.check_device_error()


@pytest.mark.parametrize('fp32', [True, False], ids=['fp32', 'tc'])
def test_chunk_prefill_zero_state_bf16_io(fp32):
    shape = SHAPES[0]
    c = I.make_core_inputs(42, [300], shape, dtype=torch.bfloat16)
    gt, bt = _core_gates(c)
    o, ST = gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), 1 / math.sqrt(128),
                              out_dtype=torch.bfloat16, fp32=fp32)
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt),
                                          1 / math.sqrt(128))
    assert_close(np64(o), ro, TOL_BF16)
    assert_close(np64(ST), rS, TOL_F32 if fp32 else TOL_BF16)


def test_chunk_in_place_state():
    shape = SHAPES[0]
    c = I.make_core_inputs(43, [100, 150], shape, S0_std=0.1)
    gt, bt = _core_gates(c)
    cu = c.cu_seqlens()
    S = cuda(c.S0.clone())
    o, _ = gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), 0.2,
                             initial_state=S, final_state=S, cu_seqlens=cuda(cu), out_dtype=torch.float32)
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt), 0.2,
                                          np64(c.S0), cu.numpy())
    assert_close(np64(S), rS, TOL_BF16)
    assert_close(np64(o), ro, TOL_BF16)


def test_tiny_workload_chunked_vs_recurrent():
    """The tiny fp32 workload: GPU chunk path vs GPU recurrent path vs the oracle."""
    c = I.workload('tiny_core_t256')
    sh = c.shape
    g, beta = gdn.gating(cuda(c.a), cuda(c.b), cuda(c.A_log), cuda(c.dt_bias))
    o_c, S_c = gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), g, beta, 1 / 8, out_dtype=torch.float32)
    o_f, S_f = gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), g, beta, 1 / 8,
                                 out_dtype=torch.float32, fp32=True)
    state = torch.zeros(1, sh.Nv, sh.Dk, sh.Dv, device='cuda')
    o_r = gdn.recurrent_decode(cuda(c.q), cuda(c.k), cuda(c.v), g, beta, state, 1 / 8, num_seqs=1,
                               out_dtype=torch.float32)
    rg, rb = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), rg, rb, 1 / 8)
    assert_close(np64(o_c), ro, TOL_BF16)
    assert_close(np64(S_c), rS, TOL_BF16)
    assert_close(np64(o_f), ro, TOL_F32)
    assert_close(np64(S_f), rS, TOL_F32)
    assert_close(np64(o_r), ro, TOL_F32)
    assert_close(np64(state), rS, TOL_F32)
    assert_close(np64(o_c), np64(o_r), TOL_BF16)


# ------------------------------------------------------------------ whole prefill path

@pytest.mark.parametrize('fuse_norm', [True, False], ids=['fused_norm', 'separate_norm'])
def test_mixer_prefill_small_end_to_end(fuse_norm):
    shape = SHAPES[0]
    inp = I.make_mixer_inputs(51, [90, 1, 200], shape, conv_state_std=1.0, S0_std=0.05)
    sh = inp.shape
    cu = inp.cu_seqlens()
    cs_out = torch.empty(inp.num_seqs, sh.C, 3, dtype=torch.bfloat16, device='cuda')
    y, S = gdn.mixer_prefill(cuda(inp.mixed_qkv), cuda(inp.conv_w), cuda(inp.a), cuda(inp.b),
                             cuda(inp.A_log), cuda(inp.dt_bias), cuda(inp.z), cuda(inp.norm_w),
                             sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=cuda(cu),
                             conv_state_in=cuda(inp.conv_state), conv_state_out=cs_out,
                             initial_state=cuda(inp.S0), out_dtype=torch.float32, fuse_norm=fuse_norm)
    ref = O.mixer_prefill(np64(inp.mixed_qkv), np64(inp.conv_w), np64(inp.a), np64(inp.b),
                          np64(inp.A_log), np64(inp.dt_bias), np64(inp.z), np64(inp.norm_w),
                          sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=cu.numpy(),
                          conv_state=np64(inp.conv_state), initial_state=np64(inp.S0))
    assert_close(np64(y), ref['y'], TOL_BF16)
    assert_close(np64(S), ref['state'], TOL_BF16)
    np.testing.assert_array_equal(np64(cs_out), ref['conv_state'])


@pytest.mark.parametrize('odt', [torch.float32, torch.bfloat16], ids=['f32', 'bf16'])
@pytest.mark.parametrize('lengths', [[300], [40], [64], [130, 0, 64, 7]],
                         ids=['one_seq', 'one_partial_chunk', 'one_full_chunk', 'packed'])
def test_chunk_prefill_gated_norm(lengths, odt):
    """Chunk prefill with the gated RMSNorm in its epilogue: against the oracle
    (recurrence, then the norm) and against the two separate calls.  One
    sequence runs the cooperative launch, the packed batch the two launches."""
    shape = SHAPES[0]
    c = I.make_core_inputs(61, lengths, shape, dtype=torch.bfloat16, S0_std=0.1)
    gt, bt = _core_gates(c)
    cu = c.cu_seqlens()
    T = sum(lengths)
    z = I.draw_normal(62, (T, shape.Nv, shape.Dv), dtype=torch.bfloat16)
    w = I.draw_normal(63, (shape.Dv,), mean=1.0, std=0.1)
    packed = len(lengths) > 1
    args = (cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt))
    y, ST = gdn.chunk_prefill_gated_norm(*args, cuda(z), cuda(w), 0.2, initial_state=cuda(c.S0),
                                         cu_seqlens=cuda(cu) if packed else None, num_seqs=len(lengths),
                                         out_dtype=odt)
    torch.cuda.synchronize()
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt), 0.2,
                                          np64(c.S0), cu.numpy())
    ry = O.gated_rmsnorm(ro, np64(z), np64(w), 1e-6)
    assert_close(np64(y), ry, TOL_BF16)
    assert_close(np64(ST), rS, TOL_BF16)
    # the fused call normalises o as a bf16 o would be stored
    o2, _ = gdn.chunk_prefill(*args, 0.2, initial_state=cuda(c.S0), cu_seqlens=cuda(cu) if packed else None,
                              num_seqs=len(lengths), out_dtype=torch.bfloat16)
    y2 = gdn.gated_rmsnorm(o2, cuda(z), cuda(w), 1e-6, out_dtype=odt)
    if odt == torch.float32:
        assert_close(np64(y), np64(y2), 1e-5, row_tol=1e-4)
    else:
        assert_close(np64(y), np64(y2), TOL_BF16)
    gdn.check_device_error()


def test_device_error_flag_on_bad_cu_seqlens():
    """A non-monotone cu_seqlens is caught on the device, skipped and reported."""
    shape = SHAPES[1]
    c = I.make_core_inputs(44, [10, 10], shape)
    gt, bt = _core_gates(c)
    bad = torch.tensor([0, 15, 12], dtype=torch.int32)     # second sequence ends before it starts
    gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), 1.0,
                      cu_seqlens=cuda(bad), out_dtype=torch.float32)
    with pytest.raises(RuntimeError, match='device error'):
        gdn.check_device_error()
    gdn.check_device_error()      # the flag was cleared


# ------------------------------------------------------------------ one long sequence, split in two

@pytest.mark.parametrize('T,odt,state', [(2048, torch.float32, 'in'), (2100, torch.float32, 'in_place'),
                                         (4000, torch.bfloat16, 'none'), (2100, torch.bfloat16, 'no_final')],
                         ids=['T2048_f32_S0', 'T2100_f32_inplace', 'T4000_bf16_zero', 'T2100_bf16_nofinal'])
def test_chunk_prefill_one_long_sequence(T, odt, state):
    """One sequence of 32 chunks or more runs split in two segments (the second segment's
    scan from a zero state and its transition-map scan beside the first segment's, then
    the fix-up of the second segment's outputs and of the final state): against the
    oracle, whole chunks and a ragged last chunk, with and without initial and final
    states."""
    shape = SHAPES[0]
    c = I.make_core_inputs(81, [T], shape, dtype=torch.bfloat16, S0_std=0.1,
                           A_log_range=(-4.0, 0.0))           # slow decay: the entry state matters
    gt, bt = _core_gates(c)
    S0 = cuda(c.S0) if state in ('in', 'in_place') else None
    ST = S0 if state == 'in_place' else None
    o, S = gdn.chunk_prefill(cuda(c.q), cuda(c.k), cuda(c.v), cuda(gt), cuda(bt), 0.2, initial_state=S0,
                             final_state=ST, out_dtype=odt, want_final_state=state != 'no_final')
    torch.cuda.synchronize()
    gdn.check_device_error()
    ro, rS = O.chunk_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), np64(gt), np64(bt), 0.2,
                                      np64(c.S0) if S0 is not None else None)
    assert_close(np64(o), ro, TOL_BF16)
    if state != 'no_final':
        assert_close(np64(S), rS, TOL_BF16)
    else:
        assert S is None


# ------------------------------------------------------------------ draft + verify decode, both states

def test_verify_decode_rolls_back_conv_and_recurrent_state():
    """A multi-token (1 + 3 tokens) decode step of the mixer core with the rollback
    points of both caches: the conv state after every token (gdn_conv_state_steps)
    against the oracle's state after each prefix, bit for bit, and the recurrent
    state after every token (gdn_recurrent_decode_steps).  Rolling sequence 1 back to
    its second token and replaying its last two tokens from the two kept states
    reproduces the first pass."""
    shape = SHAPES[0]
    lengths = [4, 4, 4]
    inp = I.make_mixer_inputs(77, lengths, shape, dtype=torch.bfloat16, conv_state_std=1.0, S0_std=0.05)
    sh = inp.shape
    cu = inp.cu_seqlens()
    cu_l = cu.tolist()
    x, w = cuda(inp.mixed_qkv), cuda(inp.conv_w)
    cs_in = cuda(inp.conv_state)
    conv_steps = gdn.conv_state_steps(x, sh.Nk, sh.Nv, sh.Dk, sh.Dv, conv_state_in=cs_in, cu_seqlens=cuda(cu))
    cs_out = torch.empty_like(cs_in)
    q, k, v, g, beta = gdn.conv_gating(x, w, cuda(inp.a), cuda(inp.b), cuda(inp.A_log), cuda(inp.dt_bias),
                                       sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=cuda(cu), conv_state_in=cs_in,
                                       conv_state_out=cs_out, out_dtype=torch.float32)
    S = cuda(inp.S0.clone())
    rec_steps = torch.empty(sum(lengths), sh.Nv, sh.Dk, sh.Dv, device='cuda')
    o = gdn.recurrent_decode(q, k, v, g, beta, S, 1.0, cu_seqlens=cuda(cu), out_dtype=torch.float32,
                             step_states=rec_steps)
    torch.cuda.synchronize()
    gdn.check_device_error()
    # every step's conv state against the oracle's state after that prefix (raw copies: exact)
    xs = np64(inp.mixed_qkv)
    for s in range(len(lengths)):
        for j in range(lengths[s]):
            _, st = O.causal_conv1d(xs[cu_l[s]:cu_l[s] + j + 1], np64(inp.conv_w), None, np64(inp.conv_state[s]))
            np.testing.assert_array_equal(np64(conv_steps[cu_l[s] + j]), st)
        assert torch.equal(conv_steps[cu_l[s + 1] - 1], cs_out[s])       # the last step is the new state
    ref = O.mixer_prefill(xs, np64(inp.conv_w), np64(inp.a), np64(inp.b), np64(inp.A_log), np64(inp.dt_bias),
                          np64(inp.z), np64(inp.norm_w), sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=cu.numpy(),
                          conv_state=np64(inp.conv_state), initial_state=np64(inp.S0))
    assert_close(np64(o), ref['o'], TOL_F32)
    # roll sequence 1 back to its second token (keep both states there) and replay tokens 2-3
    b0 = cu_l[1]
    tail = slice(b0 + 2, b0 + 4)
    cs1 = conv_steps[b0 + 1].unsqueeze(0).contiguous()
    S1 = rec_steps[b0 + 1].unsqueeze(0).clone()
    q2, k2, v2, g2, beta2 = gdn.conv_gating(cuda(inp.mixed_qkv[tail].contiguous()), w, cuda(inp.a[tail].contiguous()),
                                            cuda(inp.b[tail].contiguous()), cuda(inp.A_log), cuda(inp.dt_bias),
                                            sh.Nk, sh.Nv, sh.Dk, sh.Dv, num_seqs=1, conv_state_in=cs1,
                                            out_dtype=torch.float32)
    o2 = gdn.recurrent_decode(q2, k2, v2, g2, beta2, S1, 1.0, num_seqs=1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    torch.testing.assert_close(o2, o[tail], rtol=1e-5, atol=1e-6)
    torch.testing.assert_close(S1[0], S[1], rtol=1e-5, atol=1e-6)
