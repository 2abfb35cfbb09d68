"""Failure detection without a GPU fault: the bounded device waits of the
chunk-prefill scan.  A test hook launches the one-sequence prefill with no
solve work, so no chunk's ready flag is ever published and every scan's first
wait runs out (while none of its copies or products is in flight).  The call
must come back with the device error flag raised (code 2), and the same
process must then run a normal prefill that matches the oracle."""

import ctypes
import math
import time

import pytest
import torch

import oracle as O
from gated_deltanet_linear_conv_gb300 import gdn
from gated_deltanet_linear_conv_gb300 import inputs as I
from helpers import TOL_BF16, assert_close, np64

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_then_a_clean_call():
    shape = I.MixerShape(2, 4, 128, 128)
    T = 300
    c = I.make_core_inputs(71, [T], shape, dtype=torch.bfloat16)
    g, beta = O.gating(np64(c.a), np64(c.b), np64(c.A_log), np64(c.dt_bias))
    gt = torch.tensor(g, dtype=torch.float32).cuda()
    bt = torch.tensor(beta, dtype=torch.float32).cuda()
    q, k, v = c.q.cuda(), c.k.cuda(), c.v.cuda()
    ws_bytes = gdn.chunk_prefill_workspace_size(1, T, shape.Nk, shape.Nv, shape.Dk, shape.Dv)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device='cuda')
    o = torch.empty(T, shape.Nv, shape.Dv, dtype=torch.bfloat16, device='cuda')
    d = gdn.gdn_dims(1, T, shape.Nk, shape.Nv, shape.Dk, shape.Dv)
    gdn.check_device_error()                      # nothing pending from earlier tests
    wait_ns = 20_000_000                          # 20 ms
    t0 = time.perf_counter()
    st = gdn.lib().gdn_test_chunk_wait_timeout(
        ctypes.byref(d), q.data_ptr(), k.data_ptr(), v.data_ptr(), gt.data_ptr(), bt.data_ptr(),
        o.data_ptr(), ws.data_ptr(), ws_bytes, wait_ns, torch.cuda.current_stream().cuda_stream)
    assert st == gdn.GDN_OK, gdn.lib().gdn_last_error_string()
    with pytest.raises(RuntimeError, match='bounded wait timed out'):
        gdn.check_device_error()
    assert time.perf_counter() - t0 < 10.0
    gdn.check_device_error()                      # the flag was read and cleared

    # the context is still usable: a normal call on the same buffers matches the oracle
    o2, S2 = gdn.chunk_prefill(q, k, v, gt, bt, 1 / math.sqrt(128), out_dtype=torch.float32, workspace=ws)
    torch.cuda.synchronize()
    gdn.check_device_error()
    ro, rS = O.recurrent_gated_delta_rule(np64(c.q), np64(c.k), np64(c.v), g, beta, 1 / math.sqrt(128))
    assert_close(np64(o2), ro, TOL_BF16)
    assert_close(np64(S2), rS, TOL_BF16)


def test_timeout_hook_rejects_bad_bounds():
    d = gdn.gdn_dims(1, 64, 2, 4, 128, 128)
    x = torch.empty(16, device='cuda')
    st = gdn.lib().gdn_test_chunk_wait_timeout(ctypes.byref(d), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                               x.data_ptr(), x.data_ptr(), x.data_ptr(), x.data_ptr(), 64,
                                               100, torch.cuda.current_stream().cuda_stream)
    assert st == gdn.GDN_ERR_INVALID_ARG
