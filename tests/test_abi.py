"""The C-ABI library loads, exports every symbol include/fa.h declares, and rejects bad arguments on the
host before launching anything (CPU only: no call here reaches the GPU)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_17_gb300 as fa
    if not os.path.exists(fa.LIB_PATH):
        from exact_io_aware_17_gb300 import build
        build.build()
    fa.load_library()
    return fa


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_binding_exports(fa):
    assert _declared_functions() == sorted(fa.EXPORTS)


def test_library_exports_every_declared_symbol(fa):
    out = subprocess.run(["nm", "-D", "--defined-only", fa.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(fa_[a-z0-9_]+)$", out, flags=re.M))
    for name in _declared_functions():
        assert name in exported, name
        assert getattr(fa.load_library(), name) is not None


def test_binding_fails_loudly_without_library(tmp_path):
    code = ("import exact_io_aware_17_gb300 as fa\n"
            "try:\n    fa.load_library(%r)\nexcept RuntimeError as e:\n    print('raised', e)\n" % str(tmp_path / "missing.so"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=ROOT)
    assert "raised" in r.stdout


FAKE = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced: every call below fails its checks
MISALIGNED = ctypes.c_void_p(0x10008)


def _fwd(lib, ptrs=None, B=1, H=1, N=8, d=64, scale=0.125):
    p = ptrs or [FAKE] * 5
    return lib.fa_fwd(*p, B, H, N, d, scale, None)


def test_fwd_argument_checks(fa):
    lib = fa.load_library()
    assert _fwd(lib, [None, FAKE, FAKE, FAKE, FAKE]) == fa.FA_ERR_INVALID_ARG
    assert "q is NULL" in fa.fa_last_error_string()
    assert _fwd(lib, [FAKE, FAKE, MISALIGNED, FAKE, FAKE]) == fa.FA_ERR_INVALID_ARG
    assert "v is not 16-byte aligned" in fa.fa_last_error_string()
    for kw in (dict(B=0), dict(H=0), dict(N=0), dict(d=0), dict(N=-5)):
        assert _fwd(lib, **kw) == fa.FA_ERR_INVALID_ARG, kw
    for scale in (0.0, -1.0, float("nan"), float("inf")):
        assert _fwd(lib, scale=scale) == fa.FA_ERR_INVALID_ARG, scale
    for d in (16, 32, 96, 256):
        assert _fwd(lib, d=d) == fa.FA_ERR_UNSUPPORTED, d
        assert "d must be 64 or 128" in fa.fa_last_error_string()
    assert _fwd(lib, B=1 << 16, H=1 << 16) == fa.FA_ERR_INVALID_ARG


def test_fwd_f32_argument_checks(fa):
    lib = fa.load_library()
    args = [FAKE] * 5
    assert lib.fa_fwd_f32(*args, 1, 1, 8, 130, 0.1, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_f32(*args, 1, 1, 8, 18, 0.1, None) == fa.FA_ERR_UNSUPPORTED
    assert lib.fa_fwd_f32(None, *args[1:], 1, 1, 8, 16, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_fwd_f32(*args, 1, 1, 0, 16, 0.1, None) == fa.FA_ERR_INVALID_ARG


def test_bwd_argument_checks(fa):
    lib = fa.load_library()
    need = fa.fa_bwd_workspace_size(2, 3, 100, 64)
    ptrs = [FAKE] * 9

    def call(ws=FAKE, ws_bytes=need, d=64, N=100, p=None):
        return lib.fa_bwd(*(p or ptrs), 2, 3, N, d, 0.125, ws, ws_bytes, None)

    assert call(ws=None) == fa.FA_ERR_INVALID_ARG
    assert call(ws=ctypes.c_void_p(0x10010)) == fa.FA_ERR_INVALID_ARG        # not 256-byte aligned
    assert "256-byte" in fa.fa_last_error_string()
    assert call(ws_bytes=need - 1) == fa.FA_ERR_INVALID_ARG
    assert "workspace holds" in fa.fa_last_error_string()
    assert call(d=32) == fa.FA_ERR_UNSUPPORTED
    assert call(N=0) == fa.FA_ERR_INVALID_ARG
    bad = list(ptrs)
    bad[4] = None
    assert call(p=bad) == fa.FA_ERR_INVALID_ARG and "dout is NULL" in fa.fa_last_error_string()


def test_workspace_size_formula(fa):
    def r256(x):
        return (x + 255) // 256 * 256
    for B, H, N, d in ((1, 1, 1, 64), (4, 16, 2048, 64), (1, 16, 8192, 128), (2, 3, 100, 128)):
        rows = B * H * N
        padded = B * H * ((N + 127) // 128 * 128)
        assert fa.fa_bwd_workspace_size(B, H, N, d) == r256(rows * d * 4) + 2 * r256(padded * 4)
    assert fa.fa_bwd_workspace_size(0, 1, 1, 64) == 0


def test_error_string_is_replaced_by_the_next_failure(fa):
    lib = fa.load_library()
    _fwd(lib, B=0)
    assert "B, H, N, d must be >= 1" in fa.fa_last_error_string()
    _fwd(lib, d=32)
    assert "d must be 64 or 128" in fa.fa_last_error_string()


def test_kernel_launch_counter_counts_nothing_without_launches(fa):
    """fa_kernel_launches counts enqueued kernels only: calls rejected before any launch leave it alone."""
    before = fa.fa_kernel_launches()
    assert before >= 0
    lib = fa.load_library()
    assert lib.fa_fwd(None, None, None, None, None, 1, 1, 8, 64, 0.125, None) == 1   # FA_ERR_INVALID_ARG
    assert fa.fa_kernel_launches() == before


def test_test_switch_is_off_by_default_and_ignores_the_environment(fa):
    """The failure-path switch is an explicit call only: the library source reads no environment variable."""
    import glob
    for src in glob.glob(os.path.join(ROOT, "exact_io_aware_17_gb300", "csrc", "*")):
        assert "getenv" not in open(src).read(), src
    fa.fa_test_force_wait_timeout(True)
    fa.fa_test_force_wait_timeout(False)


def test_pending_timing_request_changes_no_argument_check(fa):
    """With a fa_debug_time_bwd_main request pending, rejected backward calls still fail their checks before
    anything is launched (host only; that they also consume the request is checked on the GPU)."""
    lib = fa.load_library()
    ptrs = [FAKE] * 9
    lib.fa_debug_time_bwd_main(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000))   # never recorded
    launches = fa.fa_kernel_launches()
    assert lib.fa_bwd(*ptrs, 1, 1, 0, 64, 0.125, FAKE, 1 << 20, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 0, 64, 0.125, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_kernel_launches() == launches
