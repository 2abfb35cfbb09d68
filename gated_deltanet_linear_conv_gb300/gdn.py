"""Thin ctypes binding of libgdn.so (the C ABI declared in include/gdn.h).

Argument marshalling only: every step of the mixer runs in the library's
CUDA kernels.  Tensors are torch CUDA tensors (torch supplies device memory
and the current stream); they must be contiguous and on the current device.
There is no fallback: if libgdn.so is missing or a call fails, a
RuntimeError is raised.
"""

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, 'libgdn.so')

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_CUDA, GDN_ERR_DEVICE = range(5)
GDN_BF16, GDN_F32 = 0, 1

EXPORTS = ('gdn_version', 'gdn_last_error_string', 'gdn_check_device_error', 'gdn_conv_gating',
           'gdn_conv_state_steps',
           'gdn_gating', 'gdn_chunk_prefill_workspace_size', 'gdn_chunk_prefill',
           'gdn_chunk_prefill_fp32', 'gdn_chunk_prefill_static', 'gdn_chunk_prefill_gated_norm',
           'gdn_recurrent_decode', 'gdn_recurrent_decode_steps',
           'gdn_gated_rmsnorm', 'gdn_decode_fused', 'gdn_test_chunk_wait_timeout')


class gdn_dims(ctypes.Structure):
    _fields_ = [('num_seqs', ctypes.c_int32), ('total_tokens', ctypes.c_int32),
                ('num_k_heads', ctypes.c_int32), ('num_v_heads', ctypes.c_int32),
                ('head_k_dim', ctypes.c_int32), ('head_v_dim', ctypes.c_int32)]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_DIMS = ctypes.POINTER(gdn_dims)

_SIGS = {
    'gdn_version': ([], _I),
    'gdn_last_error_string': ([], ctypes.c_char_p),
    'gdn_check_device_error': ([_P], _I),
    'gdn_conv_gating': ([_DIMS, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _F, _F,
                         _P, _P, _P, _I, _P, _P, _P], _I),
    'gdn_gating': ([_I64, ctypes.c_int32, _P, _P, _I, _P, _P, _P, _P, _P], _I),
    'gdn_conv_state_steps': ([_DIMS, _P, _P, _I, _P, _P, _P], _I),
    'gdn_chunk_prefill_workspace_size': ([_DIMS, ctypes.POINTER(_SZ)], _I),
    'gdn_chunk_prefill': ([_DIMS, _P, _P, _P, _P, _I, _P, _P, _F, _P, _P, _P, _I, _P, _SZ, _P], _I),
    'gdn_chunk_prefill_fp32': ([_DIMS, _P, _P, _P, _P, _I, _P, _P, _F, _P, _P, _P, _I, _P], _I),
    'gdn_chunk_prefill_static': ([_DIMS, _P, _P, _P, _P, _I, _P, _P, _F, _P, _P, _P, _I, _P], _I),
    'gdn_chunk_prefill_gated_norm': ([_DIMS, _P, _P, _P, _P, _I, _P, _P, _F, _P, _P, _P, _I, _P, _F, _P, _I,
                                      _P, _SZ, _P], _I),
    'gdn_recurrent_decode': ([_DIMS, _P, _P, _P, _P, _I, _P, _P, _F, _P, _P, _I, _P], _I),
    'gdn_recurrent_decode_steps': ([_DIMS, _P, _P, _P, _P, _I, _P, _P, _F, _P, _P, _P, _I, _P], _I),
    'gdn_gated_rmsnorm': ([_I64, ctypes.c_int32, _P, _I, _P, _I, _P, _F, _P, _I, _P], _I),
    'gdn_decode_fused': ([_DIMS, _P, _I, _P, _P, _P, _P, _P, _P, _P, _F, _F, _P, _P, _P, _F,
                          _P, _I, _P], _I),
    'gdn_test_chunk_wait_timeout': ([_DIMS, _P, _P, _P, _P, _P, _P, _P, _SZ, _I64, _P], _I),
}


def lib():
    """Load libgdn.so once (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError('libgdn.so is not built (%s); run __graft_entry__.build()' % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status, name):
    if status != GDN_OK:
        msg = lib().gdn_last_error_string().decode()
        raise RuntimeError('%s failed (status %d): %s' % (name, status, msg))


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError('expected a CUDA tensor')
    if not t.is_contiguous():
        raise ValueError('expected a contiguous tensor')
    return t.data_ptr()


def _dt(t):
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise ValueError('unsupported dtype %s' % t.dtype)


def _tdt(code):
    return torch.bfloat16 if code == GDN_BF16 else torch.float32


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _dims(num_seqs, total, Nk, Nv, Dk, Dv):
    return gdn_dims(int(num_seqs), int(total), int(Nk), int(Nv), int(Dk), int(Dv))


def _f32(t):
    if t is None or t.dtype == torch.float32:
        return t
    raise ValueError('expected a float32 tensor')


def check_device_error():
    """Synchronise the current stream and raise if a kernel flagged bad metadata."""
    _check(lib().gdn_check_device_error(_stream()), 'gdn_check_device_error')


def conv_gating(mixed_qkv, conv_w, a, b, A_log, dt_bias, Nk, Nv, Dk, Dv, cu_seqlens=None,
                num_seqs=1, conv_bias=None, conv_state_in=None, conv_state_out=None,
                q_scale=None, l2_eps=1e-6, out_dtype=torch.bfloat16, out=None):
    """gdn_conv_gating.  Returns (q, k, v, g, beta); ``out`` may supply them."""
    T = mixed_qkv.shape[0]
    if cu_seqlens is not None:
        num_seqs = cu_seqlens.numel() - 1
    if q_scale is None:
        q_scale = 1.0 / math.sqrt(Dk)
    dev = mixed_qkv.device
    if out is None:
        q = torch.empty(T, Nk, Dk, dtype=out_dtype, device=dev)
        k = torch.empty(T, Nk, Dk, dtype=out_dtype, device=dev)
        v = torch.empty(T, Nv, Dv, dtype=out_dtype, device=dev)
        g = torch.empty(T, Nv, dtype=torch.float32, device=dev)
        beta = torch.empty(T, Nv, dtype=torch.float32, device=dev)
    else:
        q, k, v, g, beta = out
    for t in (conv_w, a, b) + tuple(x for x in (conv_bias, conv_state_in, conv_state_out) if x is not None):
        if t.dtype != mixed_qkv.dtype:
            raise ValueError('conv_w, a, b, conv_bias and conv states share the dtype of mixed_qkv')
    d = _dims(num_seqs, T, Nk, Nv, Dk, Dv)
    st = lib().gdn_conv_gating(ctypes.byref(d), _ptr(cu_seqlens), _ptr(mixed_qkv), _dt(mixed_qkv),
                               _ptr(conv_w), _ptr(conv_bias), _ptr(conv_state_in),
                               _ptr(conv_state_out), _ptr(a), _ptr(b), _ptr(_f32(A_log)),
                               _ptr(_f32(dt_bias)), float(q_scale), float(l2_eps), _ptr(q), _ptr(k),
                               _ptr(v), _dt(q), _ptr(g), _ptr(beta), _stream())
    _check(st, 'gdn_conv_gating')
    return q, k, v, g, beta


def conv_state_steps(mixed_qkv, Nk, Nv, Dk, Dv, conv_state_in=None, cu_seqlens=None, num_seqs=1, out=None):
    """gdn_conv_state_steps: the conv state after every token, [tokens, C, 3]."""
    T, C = mixed_qkv.shape
    if cu_seqlens is not None:
        num_seqs = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty(T, C, 3, dtype=mixed_qkv.dtype, device=mixed_qkv.device)
    if conv_state_in is not None and conv_state_in.dtype != mixed_qkv.dtype:
        raise ValueError('conv_state_in shares the dtype of mixed_qkv')
    d = _dims(num_seqs, T, Nk, Nv, Dk, Dv)
    st = lib().gdn_conv_state_steps(ctypes.byref(d), _ptr(cu_seqlens), _ptr(mixed_qkv), _dt(mixed_qkv),
                                    _ptr(conv_state_in), _ptr(out), _stream())
    _check(st, 'gdn_conv_state_steps')
    return out


def gating(a, b, A_log, dt_bias, out=None):
    """gdn_gating.  a, b [rows, Nv].  Returns (g, beta) fp32."""
    rows, Nv = a.shape
    if out is None:
        g = torch.empty(rows, Nv, dtype=torch.float32, device=a.device)
        beta = torch.empty_like(g)
    else:
        g, beta = out
    st = lib().gdn_gating(rows, Nv, _ptr(a), _ptr(b), _dt(a), _ptr(_f32(A_log)), _ptr(_f32(dt_bias)),
                          _ptr(g), _ptr(beta), _stream())
    _check(st, 'gdn_gating')
    return g, beta


def chunk_prefill_workspace_size(num_seqs, total, Nk, Nv, Dk, Dv):
    d = _dims(num_seqs, total, Nk, Nv, Dk, Dv)
    n = _SZ(0)
    _check(lib().gdn_chunk_prefill_workspace_size(ctypes.byref(d), ctypes.byref(n)),
           'gdn_chunk_prefill_workspace_size')
    return n.value


def chunk_prefill(q, k, v, g, beta, scale=1.0, initial_state=None, final_state=None,
                  cu_seqlens=None, num_seqs=1, out_dtype=torch.bfloat16, o=None, workspace=None,
                  fp32=False, want_final_state=True):
    """gdn_chunk_prefill (or gdn_chunk_prefill_fp32).  Returns (o, final_state)."""
    T, Nk, Dk = q.shape
    Nv, Dv = v.shape[1], v.shape[2]
    if cu_seqlens is not None:
        num_seqs = cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(T, Nv, Dv, dtype=out_dtype, device=q.device)
    if final_state is None and want_final_state:
        final_state = torch.empty(num_seqs, Nv, Dk, Dv, dtype=torch.float32, device=q.device)
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError('q, k, v must share a dtype')
    d = _dims(num_seqs, T, Nk, Nv, Dk, Dv)
    if fp32:
        st = lib().gdn_chunk_prefill_fp32(ctypes.byref(d), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v),
                                          _dt(q), _ptr(_f32(g)), _ptr(_f32(beta)), float(scale),
                                          _ptr(_f32(initial_state)), _ptr(_f32(final_state)), _ptr(o),
                                          _dt(o), _stream())
        _check(st, 'gdn_chunk_prefill_fp32')
        return o, final_state
    ws_bytes = chunk_prefill_workspace_size(num_seqs, T, Nk, Nv, Dk, Dv)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = lib().gdn_chunk_prefill(ctypes.byref(d), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _dt(q),
                                 _ptr(_f32(g)), _ptr(_f32(beta)), float(scale),
                                 _ptr(_f32(initial_state)), _ptr(_f32(final_state)), _ptr(o), _dt(o),
                                 _ptr(workspace), ws_bytes if workspace is not None else 0, _stream())
    _check(st, 'gdn_chunk_prefill')
    return o, final_state


def chunk_prefill_gated_norm(q, k, v, g, beta, z, norm_w, scale=1.0, initial_state=None,
                             final_state=None, cu_seqlens=None, num_seqs=1, norm_eps=1e-6,
                             out_dtype=torch.bfloat16, y=None, workspace=None, want_final_state=True):
    """gdn_chunk_prefill_gated_norm: chunk prefill with the gated RMSNorm fused into its
    output.  Returns (y, final_state)."""
    T, Nk, Dk = q.shape
    Nv, Dv = v.shape[1], v.shape[2]
    if cu_seqlens is not None:
        num_seqs = cu_seqlens.numel() - 1
    if y is None:
        y = torch.empty(T, Nv, Dv, dtype=out_dtype, device=q.device)
    if final_state is None and want_final_state:
        final_state = torch.empty(num_seqs, Nv, Dk, Dv, dtype=torch.float32, device=q.device)
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise ValueError('q, k, v must share a dtype')
    d = _dims(num_seqs, T, Nk, Nv, Dk, Dv)
    ws_bytes = chunk_prefill_workspace_size(num_seqs, T, Nk, Nv, Dk, Dv)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    st = lib().gdn_chunk_prefill_gated_norm(
        ctypes.byref(d), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(_f32(g)),
        _ptr(_f32(beta)), float(scale), _ptr(_f32(initial_state)), _ptr(_f32(final_state)), _ptr(z),
        _dt(z), _ptr(_f32(norm_w)), float(norm_eps), _ptr(y), _dt(y), _ptr(workspace),
        ws_bytes if workspace is not None else 0, _stream())
    _check(st, 'gdn_chunk_prefill_gated_norm')
    return y, final_state


def recurrent_decode(q, k, v, g, beta, state, scale=1.0, cu_seqlens=None, num_seqs=None,
                     out_dtype=torch.bfloat16, o=None, step_states=None):
    """gdn_recurrent_decode: state [N, Nv, Dk, Dv] fp32 is updated in place.  Returns o.
    With ``step_states`` ([tokens, Nv, Dk, Dv] fp32) it calls gdn_recurrent_decode_steps,
    which also writes the state after every token."""
    T, Nk, Dk = q.shape
    Nv, Dv = v.shape[1], v.shape[2]
    if cu_seqlens is not None:
        num_seqs = cu_seqlens.numel() - 1
    if num_seqs is None:
        num_seqs = state.shape[0]
    if o is None:
        o = torch.empty(T, Nv, Dv, dtype=out_dtype, device=q.device)
    d = _dims(num_seqs, T, Nk, Nv, Dk, Dv)
    args = (ctypes.byref(d), _ptr(cu_seqlens), _ptr(q), _ptr(k), _ptr(v), _dt(q), _ptr(_f32(g)),
            _ptr(_f32(beta)), float(scale), _ptr(_f32(state)))
    if step_states is None:
        st = lib().gdn_recurrent_decode(*args, _ptr(o), _dt(o), _stream())
        _check(st, 'gdn_recurrent_decode')
    else:
        st = lib().gdn_recurrent_decode_steps(*args, _ptr(_f32(step_states)), _ptr(o), _dt(o), _stream())
        _check(st, 'gdn_recurrent_decode_steps')
    return o


def gated_rmsnorm(x, z, w, eps=1e-6, out_dtype=torch.bfloat16, y=None):
    """gdn_gated_rmsnorm over the last axis of x (any leading shape)."""
    dim = x.shape[-1]
    rows = x.numel() // dim
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype, device=x.device)
    st = lib().gdn_gated_rmsnorm(rows, dim, _ptr(x), _dt(x), _ptr(z), _dt(z), _ptr(_f32(w)), float(eps),
                                 _ptr(y), _dt(y), _stream())
    _check(st, 'gdn_gated_rmsnorm')
    return y


def decode_fused(mixed_qkv, conv_w, conv_state, a, b, A_log, dt_bias, state, z, norm_w, Nk, Nv,
                 Dk, Dv, conv_bias=None, q_scale=None, l2_eps=1e-6, norm_eps=1e-6,
                 out_dtype=torch.bfloat16, y=None):
    """gdn_decode_fused: one token per sequence; conv_state and state updated in place."""
    B = mixed_qkv.shape[0]
    if q_scale is None:
        q_scale = 1.0 / math.sqrt(Dk)
    if y is None:
        y = torch.empty(B, Nv, Dv, dtype=out_dtype, device=mixed_qkv.device)
    d = _dims(B, B, Nk, Nv, Dk, Dv)
    st = lib().gdn_decode_fused(ctypes.byref(d), _ptr(mixed_qkv), _dt(mixed_qkv), _ptr(conv_w),
                                _ptr(conv_bias), _ptr(conv_state), _ptr(a), _ptr(b),
                                _ptr(_f32(A_log)), _ptr(_f32(dt_bias)), float(q_scale), float(l2_eps),
                                _ptr(_f32(state)), _ptr(z), _ptr(_f32(norm_w)), float(norm_eps), _ptr(y),
                                _dt(y), _stream())
    _check(st, 'gdn_decode_fused')
    return y


def mixer_prefill(mixed_qkv, conv_w, a, b, A_log, dt_bias, z, norm_w, Nk, Nv, Dk, Dv,
                  cu_seqlens=None, num_seqs=1, conv_bias=None, conv_state_in=None,
                  conv_state_out=None, initial_state=None, final_state=None, q_scale=None,
                  l2_eps=1e-6, norm_eps=1e-6, act_dtype=torch.bfloat16, out_dtype=torch.bfloat16,
                  bufs=None, fuse_norm=None):
    """The prefill path: conv_gating -> chunk_prefill -> gated_rmsnorm.  With ``fuse_norm``
    (and shapes that run on the tensor cores: bf16, 128-wide heads) the chunk prefill and
    the norm are one call (gdn_chunk_prefill_gated_norm).  By default (None) that call is
    taken for a single sequence, where the norm runs beside the sequential scan and the
    call measured faster than the two separate ones on a GB300 (119.2 vs 111.1 + 18.9 us at
    4096 tokens); packed batches take the two calls (their fused form applies the norm in
    the scan's output epilogue, which paces the scan).

    ``bufs`` (optional dict) supplies preallocated q, k, v, g, beta, o, y."""
    bufs = bufs or {}
    out = None
    if 'q' in bufs:
        out = (bufs['q'], bufs['k'], bufs['v'], bufs['g'], bufs['beta'])
    q, k, v, g, beta = conv_gating(mixed_qkv, conv_w, a, b, A_log, dt_bias, Nk, Nv, Dk, Dv,
                                   cu_seqlens, num_seqs, conv_bias, conv_state_in, conv_state_out,
                                   q_scale, l2_eps, act_dtype, out)
    if fuse_norm is None:
        fuse_norm = num_seqs == 1
    if fuse_norm and act_dtype == torch.bfloat16 and z.dtype == torch.bfloat16 and Dk == 128 and Dv == 128:
        return chunk_prefill_gated_norm(q, k, v, g, beta, z, norm_w, 1.0, initial_state, final_state,
                                        cu_seqlens, num_seqs, norm_eps, out_dtype, bufs.get('y'),
                                        bufs.get('workspace'))
    o, S = chunk_prefill(q, k, v, g, beta, 1.0, initial_state, final_state, cu_seqlens, num_seqs,
                         act_dtype, bufs.get('o'), bufs.get('workspace'))
    y = gated_rmsnorm(o, z, norm_w, norm_eps, out_dtype, bufs.get('y'))
    return y, S
