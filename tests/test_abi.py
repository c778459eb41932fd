"""The C-ABI library builds, loads and exports every declared entry point.

No compute call is made here (no GPU needed); only host-side validation paths.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mtpspec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?(?:int|size_t|int64_t|char)\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from mtp_speculative_decoding_draft_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("mtp_draft", "spec_verify", "spec_step", "mtp_workspace_size", "spec_verify_workspace_size",
              "mtp_get_status", "mtp_clear_status", "mtp_error_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), "missing export %s" % n


def test_host_side_validation_without_gpu(lib):
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    L = bd.library()
    dims = bd.make_dims(1, 4096, 32, 8, 128, 12288, 151936, 4099)
    n = L.mtp_workspace_size(ctypes.byref(dims), 3)
    assert n > 3 * 4096 * 4
    assert L.mtp_workspace_size(ctypes.byref(dims), 0) == 0           # k outside 1..8
    assert L.mtp_workspace_size(ctypes.byref(dims), 9) == 0
    bad = bd.make_dims(1, 4096, 32, 6, 128, 12288, 151936, 4099)      # Hq % Hkv != 0
    assert L.mtp_workspace_size(ctypes.byref(bad), 3) == 0
    bad = bd.make_dims(1, 4096, 32, 8, 96, 12288, 151936, 4099)       # unsupported head size
    assert L.mtp_workspace_size(ctypes.byref(bad), 3) == 0
    # verification from hidden states: a stochastic shape whose (row, 256-token
    # tile) items reach 2^31 is refused (a 32-bit claim counter walks them);
    # greedy has no such counter
    assert bd.fused_workspace_size(1 << 20, 8, 256 * 256, 64, 1) == 0
    assert bd.fused_workspace_size(1 << 20, 8, 256 * 256, 64, 0) > 0
    assert bd.fused_workspace_size((1 << 20) - 1, 8, 256 * 256, 64, 1) > 0
    # argument errors are reported before any device work
    assert L.spec_verify(4, 0, 100, 1.0, 0, None, None, None, None, None, None, None, None, None, 0, None) == -1
    assert L.spec_verify(4, 3, 100, 1.0, 0, None, None, None, None, None, None, None, None, None, 0, None) == -1
    assert L.mtp_draft(None, None, None, None, None, None, None, 3, 1.0, 0, None, None, None, None, 0, None) == -1
    assert L.mtp_draft_modules(ctypes.byref(dims), None, 1, None, None, None, 3, 1.0, 0, None, None, None,
                               None, 0, None) == -1                   # no modules
    mods = (bd.MtpModule * 4)()
    assert L.mtp_draft_modules(ctypes.byref(dims), mods, 4, None, None, None, 3, 1.0, 0, None, None, None,
                               None, 0, None) == -1                   # more modules than depths
    assert L.spec_step_modules(ctypes.byref(dims), mods, 0, None, None, None, 3, 1.0, 0, None, None, None,
                               None, None, None, None, None, None, None, 0, None) == -1
    assert L.mtp_draft_dynamic(ctypes.byref(dims), None, None, None, None, None, None, 3, 1.0, 0, 0.5, None, None,
                               None, None, None, 0, None) == -1       # no weights, no k_eff
    assert L.spec_verify_dynamic(4, 0, 100, 1.0, 0, None, None, None, None, None, None, None, None, None, None, 0,
                                 None) == -1
    assert L.mtp_draft_reduced(ctypes.byref(dims), None, None, None, 0, None, None, None, None, None, 3, 1.0, 0,
                               None, None, None, None, 0, None) == -1   # no weights, no map
    assert L.mtp_selftest_wait_timeout(None, None) == -1                # no status word
    assert L.mtp_selftest_wait_timeout(ctypes.c_void_p(2), None) == -1  # misaligned status word
    assert L.mtp_error_string(-3) == b"workspace too small"
    assert L.spec_verify_workspace_size(4, 3, 100) >= 4


def test_variant_arguments_are_checked_on_the_host(lib):
    """The next rows' own argument rules, before any device work: each call
    with valid arguments gets as far as the workspace-size check (-3, no
    workspace given); the same call with one bad value is refused (-1).
    The pointers are never dereferenced on these paths."""
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    L = bd.library()
    dims = bd.make_dims(1, 256, 4, 2, 64, 768, 5003, 300)
    w = bd.MtpWeights(*[ctypes.c_void_p(4096 * (i + 1)) for i in range(len(bd.WEIGHT_FIELDS))])
    h, tok, kc, vc, cl, ud, dt, dl, ke = [ctypes.c_void_p(1 << (20 + i)) for i in range(9)]
    ws = ctypes.c_void_p(1 << 30)

    def dynamic(stop_p):
        return L.mtp_draft_dynamic(ctypes.byref(dims), ctypes.byref(w), h, tok, kc, vc, cl, 3, 1.0, 1,
                                   ctypes.c_float(stop_p), ud, dt, dl, ke, ws, 0, None)

    assert dynamic(0.5) == -3 and dynamic(0.0) == -3
    for bad in (-0.5, float("nan"), float("inf")):       # stop_p must be finite and >= 0
        assert dynamic(bad) == -1

    head, vmap = ctypes.c_void_p(1 << 26), ctypes.c_void_p(1 << 27)

    def reduced(n):
        return L.mtp_draft_reduced(ctypes.byref(dims), ctypes.byref(w), head, vmap, n, h, tok, kc, vc, cl, 3, 1.0,
                                   1, ud, dt, dl, ws, 0, None)

    assert reduced(128) == -3 and reduced(5003) == -3
    assert reduced(127) == -1 and reduced(5004) == -1      # 128 <= N <= V


def test_noalloc_limit_counts_the_draft_only_layout(lib):
    """mtp_draft_noalloc keeps no logits and no verifier state in its scratch:
    at d 4096, F 12288, V 151936 a batch of 4 passes the 4 MiB limit (and then
    fails on its missing weights, before any device work) while a batch of 5,
    which takes the tensor-core path's buffers, is refused."""
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    L = bd.library()
    for B, want in ((4, -1), (5, -5)):
        dims = bd.make_dims(B, 4096, 32, 8, 128, 12288, 151936, 4099)
        assert L.mtp_draft_noalloc(ctypes.byref(dims), None, None, None, None, None, None, 3, 1.0, 0, None, None,
                                   None, None, None) == want


def test_trace_read_needs_the_trace_build(lib):
    """The launch trace exists only in the library built with MTP_TRACE; the
    default build answers MTP_ERR_UNSUPPORTED_SHAPE without touching a GPU."""
    from mtp_speculative_decoding_draft_gb300 import binding as bd
    assert bd.library().mtp_trace_read(None, 0) == -2
    with pytest.raises(bd.MtpError):
        bd.trace_read(4)


def test_trace_build_variant_compiles():
    from mtp_speculative_decoding_draft_gb300 import build
    path = build.build(variant="trace")
    L = ctypes.CDLL(path)
    assert hasattr(L, "mtp_trace_read")
    assert L.mtp_trace_read(None, 5) == -1      # a null buffer for 5 records
