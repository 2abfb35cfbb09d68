"""gdn_chunk_prefill_static: the chunk prefill for callers that cannot
allocate device memory (hosts that reserve the device up front and give the
library no allocator).  It runs on the library's fixed scratch array instead of
a caller workspace.  This file sorts last so that a stop-at-first-failure run
has already run every other test; it also passes on its own in a fresh
process.  Calls go straight through the C ABI."""

import ctypes
import math

import pytest
import torch

import oracle as O
from gated_deltanet_linear_conv_gb300 import gdn
from gated_deltanet_linear_conv_gb300 import inputs as I
from helpers import TOL_BF16, assert_close, np64

pytestmark = pytest.mark.gpu


def _static_call(q, k, v, g, beta, scale, S0, ST, o, cu, num_seqs):
    T, Nk, Dk = q.shape
    Nv, Dv = v.shape[1], v.shape[2]
    d = gdn.gdn_dims(num_seqs, T, Nk, Nv, Dk, Dv)
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    st = gdn.lib().gdn_chunk_prefill_static(
        ctypes.byref(d), ptr(cu), q.data_ptr(), k.data_ptr(), v.data_ptr(), gdn.GDN_BF16,
        g.data_ptr(), beta.data_ptr(), float(scale), ptr(S0), ST.data_ptr(), o.data_ptr(),
        gdn.GDN_F32, torch.cuda.current_stream().cuda_stream)
    assert st == gdn.GDN_OK, gdn.lib().gdn_last_error_string()


def test_static_scratch_matches_workspace_call_twice():
    shape = I.MixerShape(2, 4, 128, 128)
    lengths = [130, 64, 1, 300]
    cu = I.make_core_inputs(91, lengths, shape, dtype=torch.bfloat16, S0_std=0.1).cu_seqlens().cuda()
    for call, seed in enumerate((91, 92)):          # two calls in a row, different data
        c = I.make_core_inputs(seed, lengths, shape, dtype=torch.bfloat16, S0_std=0.1)
        q, k, v = c.q.cuda(), c.k.cuda(), c.v.cuda()
        g = (-torch.nn.functional.softplus(c.a.float())).cuda()
        beta = torch.sigmoid(c.b.float()).cuda()
        S0 = c.S0.cuda()
        o_ref, S_ref = gdn.chunk_prefill(q, k, v, g, beta, 1 / math.sqrt(128), initial_state=S0,
                                         cu_seqlens=cu, out_dtype=torch.float32)
        o = torch.empty_like(o_ref)
        ST = torch.empty_like(S_ref)
        _static_call(q, k, v, g, beta, 1 / math.sqrt(128), S0, ST, o, cu, len(lengths))
        torch.cuda.synchronize()
        assert_close(np64(o), np64(o_ref), TOL_BF16, what=call)
        assert_close(np64(ST), np64(S_ref), TOL_BF16, what=call)
    gdn.check_device_error()


def test_static_scratch_one_sequence_twice():
    """One sequence takes the one-sequence launch (solve and scan overlapped, the ready
    flags and the item counter cleared in the shared array by every call): two calls in
    a row with different data, at the full head count, against the workspace call and
    the oracle."""
    shape = I.MixerShape(16, 32, 128, 128)
    T = 1000
    assert gdn.chunk_prefill_workspace_size(1, T, 16, 32, 128, 128) <= 32 << 20
    for call, seed in enumerate((93, 94)):
        c = I.make_core_inputs(seed, [T], shape, dtype=torch.bfloat16, S0_std=0.05)
        g, beta = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
        gt, bt = torch.tensor(g, dtype=torch.float32).cuda(), torch.tensor(beta, dtype=torch.float32).cuda()
        q, k, v, S0 = c.q.cuda(), c.k.cuda(), c.v.cuda(), c.S0.cuda()
        scale = 1 / math.sqrt(128)
        o_ref, S_ref = gdn.chunk_prefill(q, k, v, gt, bt, scale, initial_state=S0, out_dtype=torch.float32)
        o = torch.empty_like(o_ref)
        ST = torch.empty_like(S_ref)
        _static_call(q, k, v, gt, bt, scale, S0, ST, o, None, 1)
        torch.cuda.synchronize()
        assert_close(np64(o), np64(o_ref), TOL_BF16, what=call)
        assert_close(np64(ST), np64(S_ref), TOL_BF16, what=call)
        ro, rS = O.chunk_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), g, beta, scale, np64(c.S0))
        assert_close(np64(o), ro, TOL_BF16, what=call)
        assert_close(np64(ST), rS, TOL_BF16, what=call)
    gdn.check_device_error()


def test_static_scratch_long_single_sequence():
    """One sequence's solve tiles go through a fixed ring, so the fixed scratch holds a
    sequence far longer than its tiles would need one by one (8192 tokens, 32 heads)."""
    shape = I.MixerShape(16, 32, 128, 128)
    T = 8192
    c = I.make_core_inputs(95, [T], shape, dtype=torch.bfloat16, S0_std=0.05)
    g, beta = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
    gt, bt = torch.tensor(g, dtype=torch.float32).cuda(), torch.tensor(beta, dtype=torch.float32).cuda()
    q, k, v, S0 = c.q.cuda(), c.k.cuda(), c.v.cuda(), c.S0.cuda()
    o_ref, S_ref = gdn.chunk_prefill(q, k, v, gt, bt, 1.0, initial_state=S0, out_dtype=torch.float32)
    o = torch.empty_like(o_ref)
    ST = torch.empty_like(S_ref)
    _static_call(q, k, v, gt, bt, 1.0, S0, ST, o, None, 1)
    torch.cuda.synchronize()
    assert_close(np64(o), np64(o_ref), TOL_BF16)
    assert_close(np64(ST), np64(S_ref), TOL_BF16)
    gdn.check_device_error()


def test_static_scratch_rejects_too_large():
    # a packed batch keeps one tile per (chunk, head): 4 x 32768 tokens at 32 heads is far past it
    T, N, Nk, Nv, D = 131072, 4, 16, 32, 128
    d = gdn.gdn_dims(N, T, Nk, Nv, D, D)
    x = torch.empty(16, dtype=torch.bfloat16, device='cuda')      # never read: rejected before launch
    f = torch.empty(16, device='cuda')
    st = gdn.lib().gdn_chunk_prefill_static(
        ctypes.byref(d), None, x.data_ptr(), x.data_ptr(), x.data_ptr(), gdn.GDN_BF16, f.data_ptr(),
        f.data_ptr(), 1.0, None, f.data_ptr(), x.data_ptr(), gdn.GDN_BF16,
        torch.cuda.current_stream().cuda_stream)
    assert st == gdn.GDN_ERR_INVALID_ARG
    assert b'scratch' in gdn.lib().gdn_last_error_string()
