"""exp2 emulation (Cody-Waite + degree-3 Horner), float32, and its coefficient fit.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

FlashAttention-4 blog, section "Faster exponential: split 2^x between MUFU.EX2
and FMA": 2^x = 2^n 2^f with n = floor(x), f in [0,1); 2^f approximated by
p0 + p1 f + p2 f^2 + p3 f^3 in Horner form with p0 = 1 and p1..p3 chosen to
minimise the relative error on [0,1) (the authors used Sollya and print
p1 ~ 0.6951, p2 ~ 0.2276, p3 ~ 0.0771); 2^n applied by adding n to the
exponent bits.  FlashAttention-4 paper summary §3.1.3 / Table 2: max relative
error 8.77e-5 in float32.

The float32 evaluation lives in ``exp2_poly.c`` (fused multiply-adds, like the
FMA units the section names); this module compiles it on first use, loads it
with ctypes, and fits the coefficients with its own linear-programming
minimax (scipy.optimize.linprog), not Sollya.
"""
import ctypes
import functools
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "exp2_poly.c")
_LIB = os.path.join(_HERE, "_build", "libexp2_poly.so")


def build(force=False):
    """Compile exp2_poly.c into oracle/_build/libexp2_poly.so (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + ".%d.tmp" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                           _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB)
    return _LIB


@functools.lru_cache(maxsize=None)
def _lib():
    lib = ctypes.CDLL(build())
    f = ctypes.c_float
    lib.exp2_poly.restype = f
    lib.exp2_poly.argtypes = [f, f, f, f]
    lib.exp2_poly_many.restype = None
    lib.exp2_poly_many.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_long, f, f, f]
    lib.exp2_poly_max_rel_err.restype = ctypes.c_double
    lib.exp2_poly_max_rel_err.argtypes = [ctypes.c_uint32, ctypes.c_uint32, f, f, f,
                                          ctypes.POINTER(ctypes.c_float)]
    return lib


@functools.lru_cache(maxsize=None)
def fit_coefficients(grid=20001):
    """(p1, p2, p3) minimising max |p(f) - 2^f| / 2^f on [0,1], p0 = 1.

    Linear program in (p1, p2, p3, e): minimise e subject to
    -e <= (1 + p1 f + p2 f^2 + p3 f^3 - 2^f) / 2^f <= e on a dense grid.
    Returned rounded to float32.
    """
    from scipy.optimize import linprog

    f = np.linspace(0.0, 1.0, grid)
    t = np.exp2(f)
    a = np.stack([f / t, f ** 2 / t, f ** 3 / t], axis=1)
    b = (t - 1.0) / t
    ones = np.ones((grid, 1))
    a_ub = np.vstack([np.hstack([a, -ones]), np.hstack([-a, -ones])])
    b_ub = np.concatenate([b, -b])
    res = linprog([0, 0, 0, 1], A_ub=a_ub, b_ub=b_ub,
                  bounds=[(None, None)] * 3 + [(0, None)], method="highs")
    if not res.success:
        raise RuntimeError("exp2 coefficient fit failed: " + res.message)
    return tuple(float(np.float32(c)) for c in res.x[:3])


def exp2_poly(x, coeffs=None):
    """Element-wise emulated 2^x in float32 (array in, float32 array out)."""
    p1, p2, p3 = coeffs or fit_coefficients()
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    y = np.empty_like(x)
    _lib().exp2_poly_many(x.ctypes.data, y.ctypes.data, x.size, p1, p2, p3)
    return y


def max_rel_err_unit_interval(coeffs=None, lo=0.0, hi_exclusive=1.0):
    """Exhaustive max relative error over every float32 in [lo, hi_exclusive)."""
    p1, p2, p3 = coeffs or fit_coefficients()
    lo_bits = int(np.float32(lo).view(np.uint32))
    hi_bits = int(np.float32(hi_exclusive).view(np.uint32)) - 1
    arg = ctypes.c_float()
    err = _lib().exp2_poly_max_rel_err(lo_bits, hi_bits, p1, p2, p3, ctypes.byref(arg))
    return err, arg.value
