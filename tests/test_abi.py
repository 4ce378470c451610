"""The C-ABI library builds, loads without a GPU, exports every function that
include/*.h declares, and rejects bad arguments before touching the GPU.
CPU only: no compute call is made."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from attention_blackwell_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = declared_functions()
    assert {"fa_fwd", "fa_get_device_status", "fa_status_string", "fa_exp2_emu"} <= names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    lib.fa_status_string.restype = ctypes.c_char_p
    assert lib.fa_status_string(0) == b"FA_OK"
    for code in range(-1, -7, -1):
        assert lib.fa_status_string(code).startswith(b"FA_ERR_")


def test_fwd_rejects_bad_arguments_on_the_host(lib):
    f = lib.fa_fwd
    vp, i, fl = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.restype = i
    f.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, fl, i, vp, i, vp]
    P = 0x10000  # never dereferenced: every call below fails validation first
    ok = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, N=128, d=128, alpha=0.1, causal=0, cu=None, ms=0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["Hq"], a["Hkv"], a["N"], a["d"],
                 a["alpha"], a["causal"], a["cu"], a["ms"], None)

    assert call(q=None) == -1
    assert call(B=0) == -1
    assert call(N=-1) == -1
    assert call(Hq=3) == -1            # Hq % Hkv
    assert call(alpha=0.0) == -1
    assert call(alpha=float("inf")) == -1
    assert call(causal=2) == -1
    assert call(d=96) == -2            # d is 64, 128 or 256
    assert call(d=512) == -2
    assert call(d=256, cu=P, ms=1 << 20) == -2   # d = 256 varlen: the same limits
    assert call(d=256, B=5000, cu=P, ms=128) == -2
    assert call(cu=P, ms=0) == -1      # varlen without max_seqlen
    assert call(cu=P, ms=1 << 20) == -2
    assert call(B=5000, cu=P, ms=128) == -2
    assert call(o=P + 8) == -3


def test_set_tuning_validation(lib):
    lib.fa_set_tuning.argtypes = [ctypes.c_int, ctypes.c_float]
    assert lib.fa_set_tuning(5, 8.0) == -2
    assert lib.fa_set_tuning(-1, 8.0) == -2
    assert lib.fa_set_tuning(4, 8.0) == 0
    assert lib.fa_set_tuning(0, -1.0) == -1
    assert lib.fa_set_tuning(0, 8.0) == 0


def test_forward_kernel_selector(lib):
    """Kernels 0 and 2 are accepted, others rejected; no GPU call is made and
    the pair kernel reports no resident pairs before it has ever been launched."""
    assert lib.fa_fwd_pairs_resident() == 0
    for k in (0, 2):
        assert lib.fa_set_fwd_kernel(k) == 0
    assert lib.fa_set_fwd_kernel(1) == -1
    assert lib.fa_set_fwd_kernel(3) == -1
    assert lib.fa_set_fwd_kernel(-1) == -1
    assert lib.fa_set_fwd_kernel(2) == 0


def test_backward_kernel_selector(lib):
    """Kernels 0-1 are accepted, others rejected; no GPU call is made."""
    assert lib.fa_bwd_pairs_resident() == 0
    for k in (0, 1):
        assert lib.fa_set_bwd_kernel(k) == 0
    assert lib.fa_set_bwd_kernel(2) == -1
    assert lib.fa_set_bwd_kernel(-1) == -1
    assert lib.fa_set_bwd_kernel(0) == 0


def test_schedule_order_selector(lib):
    """Orders 0 (cost-ordered, the default) and 1 (plain enumeration) are
    accepted, others rejected; no GPU call is made."""
    for k in (1, 0):
        assert lib.fa_set_schedule_order(k) == 0
    assert lib.fa_set_schedule_order(2) == -1
    assert lib.fa_set_schedule_order(-1) == -1
    assert lib.fa_set_schedule_order(0) == 0


def test_workspace_size_depends_on_head_dim(lib):
    """Host arithmetic only: the fp32 dQ accumulator scales with d."""
    f = lib.fa_bwd_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 6
    n64, n128, n256 = f(2, 4, 1000, 64, 0, 0), f(2, 4, 1000, 128, 0, 0), f(2, 4, 1000, 256, 0, 0)
    assert 0 < n64 < n128 < n256
    assert n128 - n64 >= 2 * 4 * 1000 * 64 * 4        # B*N*Hq rows of 64 more floats
    assert n256 - n128 >= 2 * 4 * 1000 * 128 * 4
    # d = 256 deterministic: two semaphore sets of one per 64-row query step
    assert f(2, 4, 1000, 256, 1, 0) - n256 >= 2 * 4 * (2000 // 64) * 4
    assert f(2, 4, 1000, 96, 0, 0) == 0 and f(2, 4, 1000, 512, 0, 0) == 0


def test_varlen_workspace_holds_the_head_group_partial_sums(lib):
    """Host arithmetic only: at d = 64 / 128 a varlen workspace also holds
    fp32 dK and dV partial sums, [2][Hkv][T][d] with Hkv <= Hq / 16 when the
    work is split by query-head group: Hq * T * d / 2 bytes."""
    f = lib.fa_bwd_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 6
    for d in (64, 128):
        fixed, packed = f(1, 32, 5000, d, 0, 0), f(4, 32, 5000, d, 0, 1)   # T = 5000 both
        assert packed - fixed >= 32 * 5000 * d // 2 >= 2 * (32 // 16) * 5000 * d * 4
    # d = 256 never splits: only the work list and offsets are added
    assert f(4, 32, 5000, 256, 0, 1) - f(1, 32, 5000, 256, 0, 0) < 32 * 5000 * 256 // 2


def test_noalloc_returns_fa_bwd_codes_on_the_host(lib):
    """fa_bwd_noalloc runs fa_bwd's argument checks first, so both entry
    points give the same code for the same bad arguments (unbuilt head dims:
    FA_ERR_UNSUPPORTED); none of these calls reaches the GPU."""
    vp, i, fl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    na, bw = lib.fa_bwd_noalloc, lib.fa_bwd
    na.restype = bw.restype = i
    na.argtypes = [vp] * 9 + [i, i, i, i, i, fl, i, vp, i, i, vp]
    bw.argtypes = [vp] * 9 + [i, i, i, i, i, fl, i, vp, i, i, vp, sz, vp]
    P = 0x10000
    ok = dict(p=P, B=1, Hq=2, Hkv=2, N=128, d=128, alpha=0.1, causal=0, cu=None, ms=0, det=0)
    cases = [dict(d=512), dict(d=96), dict(p=None), dict(B=0), dict(Hq=3), dict(alpha=0.0), dict(causal=2),
             dict(det=2), dict(cu=P, ms=0), dict(cu=P, ms=1 << 20), dict(p=P + 8), dict(d=96, p=P + 8)]
    for kw in cases:
        a = dict(ok, **kw)
        ptrs = [a["p"]] * 9
        args = ptrs + [a["B"], a["Hq"], a["Hkv"], a["N"], a["d"], a["alpha"], a["causal"], a["cu"], a["ms"], a["det"]]
        r_na = na(*args, None)
        r_bw = bw(*args, P, 1 << 40, None)
        assert r_na == r_bw and r_na < 0, (kw, r_na, r_bw)
    assert na(*([P] * 9 + [1, 2, 2, 128, 96, 0.1, 0, None, 0, 0]), None) == -2
