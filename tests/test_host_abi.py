"""CPU-only checks of the C ABI: the library builds and loads, exports every
symbol include/gdn.h declares, and rejects bad arguments on the host before
any CUDA call (no compute is launched here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope='module')
def lib():
    from gated_deltanet_linear_conv_gb300 import _build, gdn
    _build.build()
    return gdn.lib()


def header_symbols():
    text = open(os.path.join(ROOT, 'include', 'gdn.h')).read()
    return sorted(set(re.findall(r'^(?:int|const char\*)\s+(gdn_\w+)\(', text, re.M)))


def test_header_symbols_exported(lib):
    from gated_deltanet_linear_conv_gb300 import gdn
    syms = header_symbols()
    assert len(syms) >= 10
    for s in syms:
        assert hasattr(lib, s), s
    assert set(syms) == set(gdn.EXPORTS)
    assert lib.gdn_version() >> 16 == 1


def _dims(*v):
    from gated_deltanet_linear_conv_gb300 import gdn
    return gdn.gdn_dims(*v)


def test_invalid_arguments_rejected_on_host(lib):
    from gated_deltanet_linear_conv_gb300 import gdn
    E = gdn
    # Nv not a multiple of Nk
    d = _dims(1, 10, 3, 4, 128, 128)
    st = lib.gdn_chunk_prefill(ctypes.byref(d), None, None, None, None, 0, None, None, 1.0, None,
                               None, None, 0, None, 0, None)
    assert st == E.GDN_ERR_INVALID_ARG and b'multiple' in lib.gdn_last_error_string()
    # unsupported head size
    d = _dims(1, 10, 2, 4, 96, 128)
    st = lib.gdn_recurrent_decode(ctypes.byref(d), None, None, None, None, 0, None, None, 1.0, None,
                                  None, 0, None)
    assert st == E.GDN_ERR_UNSUPPORTED
    # tokens not divisible into equal sequences without cu_seqlens
    d = _dims(3, 10, 2, 4, 128, 128)
    st = lib.gdn_conv_gating(ctypes.byref(d), None, None, 0, None, None, None, None, None, None,
                             None, None, 1.0, 1e-6, None, None, None, 0, None, None, None)
    assert st == E.GDN_ERR_INVALID_ARG
    # NULL required pointer
    d = _dims(1, 16, 2, 4, 128, 128)
    st = lib.gdn_conv_gating(ctypes.byref(d), None, None, 0, None, None, None, None, None, None,
                             None, None, 1.0, 1e-6, None, None, None, 0, None, None, None)
    assert st == E.GDN_ERR_INVALID_ARG and b'NULL' in lib.gdn_last_error_string()
    # misaligned pointer
    st = lib.gdn_gated_rmsnorm(4, 128, 0x1008, 0, 0x2000, 0, 0x3000, 1e-6, 0x4000, 0, None)
    assert st == E.GDN_ERR_INVALID_ARG and b'aligned' in lib.gdn_last_error_string()
    # bad dtype code
    st = lib.gdn_gating(4, 2, 0x1000, 0x2000, 7, 0x3000, 0x4000, 0x5000, 0x6000, None)
    assert st == E.GDN_ERR_INVALID_ARG
    # fused decode needs one token per sequence
    d = _dims(2, 4, 2, 4, 128, 128)
    st = lib.gdn_decode_fused(ctypes.byref(d), 0x1000, 0, 0x1000, None, 0x1000, 0x1000, 0x1000,
                              0x1000, 0x1000, 1.0, 1e-6, 0x1000, 0x1000, 0x1000, 1e-6, 0x1000, 0, None)
    assert st == E.GDN_ERR_INVALID_ARG
    # the fused chunk + gated-norm call checks its sizes like the chunk prefill
    d = _dims(1, 10, 3, 4, 128, 128)
    st = lib.gdn_chunk_prefill_gated_norm(ctypes.byref(d), None, None, None, None, 0, None, None, 1.0, None,
                                          None, None, 0, None, 1e-6, None, 0, None, 0, None)
    assert st == E.GDN_ERR_INVALID_ARG and b'multiple' in lib.gdn_last_error_string()
    # per-step decode states are required by the steps variant
    d = _dims(1, 4, 2, 4, 128, 128)
    st = lib.gdn_recurrent_decode_steps(ctypes.byref(d), None, 0x1000, 0x1000, 0x1000, 0, 0x1000, 0x1000, 1.0,
                                        0x1000, None, 0x1000, 0, None)
    assert st == E.GDN_ERR_INVALID_ARG and b'step_states' in lib.gdn_last_error_string()
    n = ctypes.c_size_t(99)
    assert lib.gdn_chunk_prefill_workspace_size(ctypes.byref(_dims(1, 64, 2, 4, 128, 128)),
                                                ctypes.byref(n)) == 0


def test_binding_rejects_cpu_tensors(lib):
    import torch
    from gated_deltanet_linear_conv_gb300 import gdn
    x = torch.zeros(4, 128)
    with pytest.raises(ValueError):
        gdn.gated_rmsnorm(x, x, torch.ones(128))
