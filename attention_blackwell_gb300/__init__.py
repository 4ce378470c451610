"""GB300-native fused exact attention: a thin ctypes binding over libfa.so.

Every step of the computation runs in the library's CUDA kernels; this module
only marshals arguments (torch tensors -> device pointers, the current CUDA
stream) and turns status codes into exceptions.  It never falls back to any
other implementation: if ``lib/libfa.so`` is missing, every call raises.

Build the library with ``python -m attention_blackwell_gb300.build``.
"""
import ctypes
import os

import torch

__all__ = ["fwd", "set_fwd_kernel", "fwd_pairs_resident", "set_bwd_kernel", "bwd_pairs_resident", "set_schedule_order", "bwd", "bwd_workspace", "exp2_emu", "selftest_timeout", "set_tuning", "set_debug_counters", "device_status", "num_sms", "FAError", "library_path", "lib"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libfa.so")
_lib = None

HEAD_DIM = 128


class FAError(RuntimeError):
    """A libfa call returned a non-zero status."""

    def __init__(self, code, what):
        self.code = code
        super().__init__("%s: %s (%d)" % (what, _status_string(code), code))


def library_path():
    return _LIB_PATH


def lib():
    """The loaded libfa.so (ctypes.CDLL); raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError("libfa.so is not built (%s); run `python -m attention_blackwell_gb300.build`"
                               % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        vp, i, f, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_int64
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_status_string.argtypes = [i]
        L.fa_num_sms.restype = i
        L.fa_num_sms.argtypes = []
        L.fa_set_tuning.restype = i
        L.fa_set_tuning.argtypes = [i, f]
        L.fa_set_fwd_kernel.restype = i
        L.fa_set_fwd_kernel.argtypes = [i]
        L.fa_fwd_pairs_resident.restype = i
        L.fa_fwd_pairs_resident.argtypes = []
        L.fa_set_bwd_kernel.restype = i
        L.fa_set_bwd_kernel.argtypes = [i]
        L.fa_bwd_pairs_resident.restype = i
        L.fa_bwd_pairs_resident.argtypes = []
        L.fa_set_schedule_order.restype = i
        L.fa_set_schedule_order.argtypes = [i]
        L.fa_fwd.restype = i
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp]
        sz = ctypes.c_size_t
        L.fa_bwd_workspace_size.restype = sz
        L.fa_bwd_workspace_size.argtypes = [i, i, i, i, i, i]
        L.fa_bwd_stages.restype = i
        L.fa_bwd_stages.argtypes = [i] + [vp] * 9 + [i, i, i, i, i, f, i, vp, i, i, vp, sz, vp]
        L.fa_bwd.restype = i
        L.fa_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp, i, i, vp, sz, vp]
        L.fa_get_device_status.restype = i
        L.fa_get_device_status.argtypes = [vp, vp]
        L.fa_exp2_emu.restype = i
        L.fa_exp2_emu.argtypes = [vp, vp, i64, vp]
        L.fa_selftest_timeout.restype = i
        L.fa_selftest_timeout.argtypes = [vp]
        L.fa_set_debug_counters.restype = i
        L.fa_set_debug_counters.argtypes = [vp, vp, vp]
        _lib = L
    return _lib


def _status_string(code):
    try:
        return lib().fa_status_string(int(code)).decode()
    except Exception:  # library missing while formatting an error
        return "status"


def _check(rc, what):
    if rc != 0:
        raise FAError(rc, what)


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, name, dtype):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def set_bwd_kernel(kernel=0):
    """Backward main kernel for later calls: 0 one CTA per 128-key tile (the
    default), 1 CTA pairs per 256-key block (fixed length, d = 128)."""
    _check(lib().fa_set_bwd_kernel(int(kernel)), "fa_set_bwd_kernel")


def set_schedule_order(order=0):
    """Order of the work units for later calls: 0 the cost-ordered schedule
    (the default), 1 plain enumeration (for testing the scheduler)."""
    _check(lib().fa_set_schedule_order(int(order)), "fa_set_schedule_order")


def bwd_pairs_resident():
    """CTA pairs backward kernel 1 keeps resident (0 before its first launch)."""
    return int(lib().fa_bwd_pairs_resident())


def fwd_pairs_resident():
    """CTA pairs forward kernel 2 keeps resident (0 before its first launch)."""
    return int(lib().fa_fwd_pairs_resident())


def num_sms():
    n = lib().fa_num_sms()
    if n < 0:
        raise FAError(n, "fa_num_sms")
    return n


def set_tuning(exp2_emu_sixteenths=0, tau=8.0):
    """Process-wide forward tuning (sixteenths of exp2 on the FMA pipe, 0-4;
    rescale threshold tau)."""
    _check(lib().fa_set_tuning(int(exp2_emu_sixteenths), float(tau)), "fa_set_tuning")


def set_fwd_kernel(kernel=2):
    """Forward kernel for later calls: 0 ping-pong 128x128 tiles, 2 CTA pairs
    with 256-key blocks (the default)."""
    _check(lib().fa_set_fwd_kernel(int(kernel)), "fa_set_fwd_kernel")


def fwd(q, k, v, causal=False, alpha=None, cu_seqlens=None, max_seqlen=None, out=None, lse=None, stream=None):
    """Forward attention.  Returns (o, lse).

    Fixed length: q [B,N,Hq,d], k/v [B,N,Hkv,d] bf16 -> o like q,
    lse float32 [B,Hq,N].  Varlen: q [T,Hq,d], k/v [T,Hkv,d],
    cu_seqlens int32 [B+1] on the device, max_seqlen -> o [T,Hq,d],
    lse [Hq,T].  d = 128, 64 or 256.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, torch.bfloat16)
    varlen = cu_seqlens is not None
    if varlen:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        if q.dim() != 3:
            raise ValueError("varlen q must be [T, Hq, d]")
        T, Hq, d = q.shape
        Hkv = k.shape[1]
        B, N = cu_seqlens.numel() - 1, T
        if max_seqlen is None:
            raise ValueError("varlen needs max_seqlen")
        lse_shape = (Hq, T)
    else:
        if q.dim() != 4:
            raise ValueError("q must be [B, N, Hq, d]")
        B, N, Hq, d = q.shape
        Hkv = k.shape[2]
        max_seqlen = N
        lse_shape = (B, Hq, N)
    if k.shape != v.shape or k.shape[:-2] != q.shape[:-2]:
        raise ValueError("k and v must match q's leading shape")
    if alpha is None:
        alpha = 1.0 / (d ** 0.5)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(lse_shape, dtype=torch.float32, device=q.device)
    _need(out, "out", torch.bfloat16)
    _need(lse, "lse", torch.float32)
    rc = lib().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, N, d, float(alpha),
                      1 if causal else 0, _ptr(cu_seqlens), int(max_seqlen), _stream(stream))
    _check(rc, "fa_fwd")
    return out, lse


def _shapes(q, k, cu_seqlens, max_seqlen):
    if cu_seqlens is not None:
        T, Hq, d = q.shape
        return cu_seqlens.numel() - 1, T, Hq, k.shape[1], d, max_seqlen
    B, N, Hq, d = q.shape
    return B, N, Hq, k.shape[2], d, N


def bwd_workspace(B, Hq, N, deterministic=False, varlen=False, device=None, d=HEAD_DIM):
    """A uint8 CUDA tensor large enough for fa_bwd (N = total tokens if varlen)."""
    n = lib().fa_bwd_workspace_size(int(B), int(Hq), int(N), int(d), int(bool(deterministic)), int(bool(varlen)))
    if n == 0:
        raise ValueError("invalid sizes for the backward workspace")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def bwd(q, k, v, o, lse, do, causal=False, alpha=None, cu_seqlens=None, max_seqlen=None, deterministic=False,
        workspace=None, dq=None, dk=None, dv=None, stages=7, stream=None):
    """Backward attention.  Returns (dq, dk, dv); layouts as in fwd, d = 128,
    64 or 256.

    ``stages`` selects the launches (1 preprocess, 2 main, 4 postprocess);
    the default runs all three.
    """
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _need(t, n, torch.bfloat16)
    _need(lse, "lse", torch.float32)
    varlen = cu_seqlens is not None
    if varlen:
        _need(cu_seqlens, "cu_seqlens", torch.int32)
        if max_seqlen is None:
            raise ValueError("varlen needs max_seqlen")
    B, N, Hq, Hkv, d, ms = _shapes(q, k, cu_seqlens, max_seqlen)
    if alpha is None:
        alpha = 1.0 / (d ** 0.5)
    if workspace is None:
        workspace = bwd_workspace(B, Hq, N, deterministic, varlen, device=q.device, d=d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _need(t, n, torch.bfloat16)
    rc = lib().fa_bwd_stages(int(stages), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                             _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, float(alpha), 1 if causal else 0,
                             _ptr(cu_seqlens), int(ms), int(bool(deterministic)), _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(rc, "fa_bwd")
    return dq, dk, dv


def set_debug_counters(visits=None, inner=None, rescales=None):
    """Arm (tensors) or disarm (None) the kernels' debug counters: int32
    visits / inner and int64 rescales[2] CUDA tensors the caller zeroes."""
    for t, n, dt in ((visits, "visits", torch.int32), (inner, "inner", torch.int32), (rescales, "rescales", torch.int64)):
        if t is not None:
            _need(t, n, dt)
    _check(lib().fa_set_debug_counters(_ptr(visits), _ptr(inner), _ptr(rescales)), "fa_set_debug_counters")


def device_status(workspace=None, stream=None):
    """Synchronise the stream and return (and clear) the device status code."""
    return lib().fa_get_device_status(_ptr(workspace), _stream(stream))


def exp2_emu(x, stream=None):
    """The forward kernel's FMA-pipe 2^x on a float32 CUDA tensor."""
    _need(x, "x", torch.float32)
    y = torch.empty_like(x)
    _check(lib().fa_exp2_emu(_ptr(x), _ptr(y), x.numel(), _stream(stream)), "fa_exp2_emu")
    return y


def selftest_timeout(stream=None):
    """Enqueue the failure-detection diagnostic (a bounded wait on a barrier
    nothing arrives at); device_status() afterwards reports the timeout."""
    _check(lib().fa_selftest_timeout(_stream(stream)), "fa_selftest_timeout")
