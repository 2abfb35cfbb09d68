"""Parity at the five named workloads' full sizes, in the launch configuration
bench.py times (one packed call per step).  The oracle runs its fp64 chunked
form (pinned to the token-by-token recurrence in test_oracle.py); the packed
long workloads are compared on whole sequences chosen up front, or on the
first and last 4096 tokens and the final state."""

import numpy as np
import pytest
import torch

import oracle as O
from gated_deltanet_linear_conv_gb300 import gdn
from gated_deltanet_linear_conv_gb300 import inputs as I
from helpers import TOL_BF16, TOL_F32, TOL_ROW_Y_BF16, assert_close, np64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def cuda(t):
    return None if t is None else t.cuda()


def _gpu_prefill(inp, final_state=True, fuse_norm=False):
    """The whole prefill path; also returns the core output o (None with the norm fused)."""
    sh = inp.shape
    cu = inp.cu_seqlens()
    cs_out = torch.empty(inp.num_seqs, sh.C, 3, dtype=inp.mixed_qkv.dtype, device='cuda')
    o = None if fuse_norm else torch.empty(inp.total_tokens, sh.Nv, sh.Dv, dtype=torch.bfloat16, device='cuda')
    y, S = gdn.mixer_prefill(cuda(inp.mixed_qkv), cuda(inp.conv_w), cuda(inp.a), cuda(inp.b),
                             cuda(inp.A_log), cuda(inp.dt_bias), cuda(inp.z), cuda(inp.norm_w),
                             sh.Nk, sh.Nv, sh.Dk, sh.Dv, cu_seqlens=cuda(cu),
                             conv_state_in=cuda(inp.conv_state), conv_state_out=cs_out,
                             initial_state=cuda(inp.S0), out_dtype=torch.bfloat16, fuse_norm=fuse_norm,
                             bufs=None if o is None else {'o': o})
    torch.cuda.synchronize()
    gdn.check_device_error()
    return y, S, cs_out, o


def _oracle_seq(inp, s, keep=None, segment=4096):
    """The oracle's prefill of sequence s, streamed in segments with state carry."""
    sh = inp.shape
    cu = inp.cu_seqlens().tolist()
    bos, eos = cu[s], cu[s + 1]
    cs = None if inp.conv_state is None else np64(inp.conv_state[s:s + 1])
    S = None if inp.S0 is None else np64(inp.S0[s:s + 1])
    ys, os_ = {}, {}
    for a in range(bos, eos, segment):
        b = min(a + segment, eos)
        sl = slice(a, b)
        kp = None if keep is None else keep[a - bos:b - bos]
        r = O.mixer_prefill(np64(inp.mixed_qkv[sl]), np64(inp.conv_w), np64(inp.a[sl]), np64(inp.b[sl]),
                            np64(inp.A_log), np64(inp.dt_bias), np64(inp.z[sl]), np64(inp.norm_w),
                            sh.Nk, sh.Nv, sh.Dk, sh.Dv, conv_state=cs, initial_state=S,
                            use_chunked=True)
        cs, S = r['conv_state'], r['state']
        if kp is None or kp.any():
            ys[a] = r['y']
            os_[a] = r['o']
    return ys, S[0], cs[0], os_


@pytest.mark.parametrize('fuse_norm', [False, True], ids=['separate_norm', 'fused_norm'])
def test_prefill_t4096(fuse_norm):
    inp = I.workload('prefill_t4096')
    y, S, cs, o = _gpu_prefill(inp, fuse_norm=fuse_norm)
    ys, S_ref, cs_ref, os_ = _oracle_seq(inp, 0)
    assert_close(np64(y), ys[0], TOL_BF16, row_tol=TOL_ROW_Y_BF16)
    if o is not None:
        assert_close(np64(o), os_[0], TOL_BF16)
    assert_close(np64(S[0]), S_ref, TOL_BF16)
    np.testing.assert_array_equal(np64(cs[0]), cs_ref)


def test_decode_b256():
    inp = I.workload('decode_b256')
    sh = inp.shape
    cs, St = cuda(inp.conv_state.clone()), cuda(inp.S0.clone())
    y = gdn.decode_fused(cuda(inp.mixed_qkv), cuda(inp.conv_w), cs, cuda(inp.a), cuda(inp.b),
                         cuda(inp.A_log), cuda(inp.dt_bias), St, cuda(inp.z), cuda(inp.norm_w),
                         sh.Nk, sh.Nv, sh.Dk, sh.Dv, out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref = O.decode_step(np64(inp.mixed_qkv), np64(inp.conv_w), np64(inp.conv_state), np64(inp.a),
                        np64(inp.b), np64(inp.A_log), np64(inp.dt_bias), np64(inp.S0), np64(inp.z),
                        np64(inp.norm_w), sh.Nk, sh.Nv, sh.Dk, sh.Dv)
    assert_close(np64(y), ref['y'], TOL_F32)
    assert_close(np64(St), ref['state'], TOL_F32)
    np.testing.assert_array_equal(np64(cs), ref['conv_state'])


def test_varlen_16seq():
    inp = I.workload('varlen_16seq')
    assert inp.num_seqs == 16 and all(512 <= L <= 8192 for L in inp.lengths)
    y, S, cs, o = _gpu_prefill(inp)
    cu = inp.cu_seqlens().tolist()
    for s in range(inp.num_seqs):                 # every sequence: outputs, final and conv states
        ys, S_ref, cs_ref, os_ = _oracle_seq(inp, s, segment=8192)
        assert_close(np64(y[cu[s]:cu[s + 1]]), ys[cu[s]], TOL_BF16, row_tol=TOL_ROW_Y_BF16, what=s)
        assert_close(np64(o[cu[s]:cu[s + 1]]), os_[cu[s]], TOL_BF16, what=s)
        assert_close(np64(S[s]), S_ref, TOL_BF16, what=s)
        np.testing.assert_array_equal(np64(cs[s]), cs_ref)


def test_prefill_t131072_first_last_and_state():
    inp = I.workload('prefill_t131072')
    T = inp.total_tokens
    y, S, cs, o = _gpu_prefill(inp)
    y_first, o_first = np64(y[:4096]), np64(o[:4096])
    y_last, o_last = np64(y[T - 4096:]), np64(o[T - 4096:])
    del y, o
    keep = np.zeros(T, dtype=bool)
    keep[:4096] = True
    keep[T - 4096:] = True
    ys, S_ref, cs_ref, os_ = _oracle_seq(inp, 0, keep=keep)
    assert_close(y_first, ys[0], TOL_BF16, row_tol=TOL_ROW_Y_BF16)
    assert_close(y_last, ys[T - 4096], TOL_BF16, row_tol=TOL_ROW_Y_BF16)
    assert_close(o_first, os_[0], TOL_BF16)
    assert_close(o_last, os_[T - 4096], TOL_BF16)
    assert_close(np64(S[0]), S_ref, TOL_BF16)
    np.testing.assert_array_equal(np64(cs[0]), cs_ref)
