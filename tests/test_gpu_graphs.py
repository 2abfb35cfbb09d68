"""A mixed batch in one CUDA graph: a packed multi-sequence prefill (solve and
scan launches), a one-sequence prefill (the cooperative launch) and a fused
decode step of other sequences, captured once and replayed with new inputs
copied into the captured buffers -- the launch sequence of a serving step with
no host synchronisation inside.  Each replay is checked against the oracle."""

import numpy as np
import pytest
import torch

import oracle as O
from gated_deltanet_linear_conv_gb300 import gdn
from gated_deltanet_linear_conv_gb300 import inputs as I
from helpers import TOL_BF16, TOL_F32, assert_close, np64

pytestmark = pytest.mark.gpu

SHAPE = I.MixerShape(2, 4, 128, 128)


def _prefill_bufs(inp):
    """Device copies of a prefill batch's inputs plus every output buffer."""
    sh = inp.shape
    T, N = inp.total_tokens, inp.num_seqs
    d = {name: getattr(inp, name).cuda() for name in
         ('mixed_qkv', 'conv_w', 'a', 'b', 'A_log', 'dt_bias', 'z', 'norm_w', 'conv_state', 'S0')}
    d['cu'] = inp.cu_seqlens().cuda()
    d['cs_out'] = torch.empty(N, sh.C, 3, dtype=torch.bfloat16, device='cuda')
    d['ST'] = torch.empty(N, sh.Nv, sh.Dk, sh.Dv, device='cuda')
    bf = torch.bfloat16
    d['bufs'] = dict(q=torch.empty(T, sh.Nk, sh.Dk, dtype=bf, device='cuda'),
                     k=torch.empty(T, sh.Nk, sh.Dk, dtype=bf, device='cuda'),
                     v=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'),
                     g=torch.empty(T, sh.Nv, device='cuda'), beta=torch.empty(T, sh.Nv, device='cuda'),
                     o=torch.empty(T, sh.Nv, sh.Dv, dtype=bf, device='cuda'),
                     y=torch.empty(T, sh.Nv, sh.Dv, dtype=torch.float32, device='cuda'),
                     workspace=torch.empty(gdn.chunk_prefill_workspace_size(N, T, sh.Nk, sh.Nv, sh.Dk, sh.Dv),
                                           dtype=torch.uint8, device='cuda'))
    return d


def _run_prefill(d, sh):
    gdn.mixer_prefill(d['mixed_qkv'], d['conv_w'], d['a'], d['b'], d['A_log'], d['dt_bias'], d['z'],
                      d['norm_w'], sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=d['cu'],
                      conv_state_in=d['conv_state'], conv_state_out=d['cs_out'], initial_state=d['S0'],
                      final_state=d['ST'], out_dtype=torch.float32, bufs=d['bufs'], fuse_norm=False)


def _check_prefill(d, inp):
    sh = inp.shape
    ref = O.mixer_prefill(np64(inp.mixed_qkv), np64(inp.conv_w), np64(inp.a), np64(inp.b),
                          np64(inp.A_log), np64(inp.dt_bias), np64(inp.z), np64(inp.norm_w),
                          sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=inp.cu_seqlens().numpy(),
                          conv_state=np64(inp.conv_state), initial_state=np64(inp.S0))
    assert_close(np64(d['bufs']['y']), ref['y'], TOL_BF16)
    assert_close(np64(d['ST']), ref['state'], TOL_BF16)
    np.testing.assert_array_equal(np64(d['cs_out']), ref['conv_state'])


def _load(d, inp):
    """Copy a new batch (same shapes, its own weights too) into the captured input buffers."""
    for name in ('mixed_qkv', 'conv_w', 'a', 'b', 'A_log', 'dt_bias', 'z', 'norm_w', 'conv_state', 'S0'):
        d[name].copy_(getattr(inp, name))


def test_mixed_prefill_and_decode_in_one_graph():
    sh = SHAPE
    packed = [I.make_mixer_inputs(70 + i, [130, 70, 1], sh, conv_state_std=1.0, S0_std=0.05) for i in range(2)]
    single = [I.make_mixer_inputs(80 + i, [200], sh, conv_state_std=1.0, S0_std=0.05) for i in range(2)]
    dec = [I.make_mixer_inputs(90 + i, [1] * 3, sh, conv_state_std=1.0, S0_std=0.05) for i in range(2)]
    P, S = _prefill_bufs(packed[0]), _prefill_bufs(single[0])
    D = {name: getattr(dec[0], name).cuda() for name in
         ('mixed_qkv', 'conv_w', 'a', 'b', 'A_log', 'dt_bias', 'z', 'norm_w', 'conv_state', 'S0')}
    Dy = torch.empty(3, sh.Nv, sh.Dv, device='cuda')

    def step():
        _run_prefill(P, sh)
        _run_prefill(S, sh)
        gdn.decode_fused(D['mixed_qkv'], D['conv_w'], D['conv_state'], D['a'], D['b'], D['A_log'],
                         D['dt_bias'], D['S0'], D['z'], D['norm_w'], sh.Nk, sh.Nv, sh.Dk, sh.Dv,
                         out_dtype=torch.float32, y=Dy)

    step()                               # the library's per-device set-up happens outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for rep in range(2):
        _load(P, packed[rep])
        _load(S, single[rep])
        _load(D, dec[rep])
        graph.replay()
        torch.cuda.synchronize()
        _check_prefill(P, packed[rep])
        _check_prefill(S, single[rep])
        inp = dec[rep]
        ref = O.decode_step(np64(inp.mixed_qkv), np64(inp.conv_w), np64(inp.conv_state), np64(inp.a),
                            np64(inp.b), np64(inp.A_log), np64(inp.dt_bias), np64(inp.S0), np64(inp.z),
                            np64(inp.norm_w), sh.Nk, sh.Nv, sh.Dk, sh.Dv)
        assert_close(np64(Dy), ref['y'], TOL_F32)
        assert_close(np64(D['S0']), ref['state'], TOL_F32)
        np.testing.assert_array_equal(np64(D['conv_state']), ref['conv_state'])
    gdn.check_device_error()
