"""The C-ABI library loads, exports every declared entry point, and rejects
bad arguments on the host before touching a GPU (CPU only: no call here
reaches CUDA)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="needs nvcc to build the library")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_51_gb300 import binding, build
    build.build()
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("spec_verify", "spec_verify_ex", "spec_verify_workspace_size",
              "spec_verify_host", "spec_philox_fill", "spec_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in spec_verify.h but not exported"


def test_workspace_size(lib):
    from speculative_decoding_verification_51_gb300 import binding
    assert binding.workspace_size(4, 3, 1024) > 0
    assert binding.workspace_size(256, 3, 151936) >= 256 * 4 * 75 * 16  # one partial per chunk
    assert binding.workspace_size(-1, 3, 1024) == 0
    assert binding.workspace_size(4, 32, 1024) == 0   # K above 31
    assert binding.workspace_size(4, 3, 1020) == 0    # V not a multiple of 8
    assert binding.workspace_size(4, 3, 4) == 0       # V below 8


def _call(lib, B=2, K=3, V=64, logits=0x10000, dtype=1, probs=0x20000, ids=0x30000,
          num=0x40000, temp=0x50000, out=0x60000, nacc=0x70000, ws=0x80000, ws_bytes=1 << 30):
    vp = ctypes.c_void_p
    return lib.spec_verify(vp(logits), dtype, vp(probs), vp(ids), vp(num), vp(temp),
                           ctypes.c_uint64(0), B, K, V, vp(out), vp(nacc), vp(ws), ws_bytes,
                           vp(0))


def test_host_side_errors(lib):
    from speculative_decoding_verification_51_gb300 import binding as bd
    assert _call(lib, B=-1) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, K=32) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, V=4) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, dtype=7) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, V=1020) == bd.SPEC_ERR_UNSUPPORTED
    assert _call(lib, B=0) == bd.SPEC_OK            # nothing to do, nothing enqueued
    assert _call(lib, logits=0) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, num=0) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, ids=0) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, ws=0) == bd.SPEC_ERR_INVALID_ARG
    assert _call(lib, logits=0x10008) == bd.SPEC_ERR_UNSUPPORTED   # not 16-byte aligned
    assert _call(lib, probs=0x20004) == bd.SPEC_ERR_UNSUPPORTED
    assert _call(lib, ws=0x80010) == bd.SPEC_ERR_WORKSPACE         # not 256-byte aligned
    assert _call(lib, ws_bytes=16) == bd.SPEC_ERR_WORKSPACE
    assert lib.spec_philox_fill(0, None, -1, None, None) == bd.SPEC_ERR_INVALID_ARG
    assert lib.spec_philox_fill(0, None, 0, None, None) == bd.SPEC_OK
    assert lib.spec_status_str(4) == b"SPEC_ERR_WORKSPACE"
    assert lib.spec_verify_status_ptr(ctypes.c_void_p(0x1000)) == 0x100C
    assert bd.host_small_bytes(3, 2) == 5 * 256


def test_typical_host_side_errors(lib):
    """spec_verify_typical rejects a NaN threshold and bad sizes on the host."""
    from speculative_decoding_verification_51_gb300 import binding as bd
    vp = ctypes.c_void_p

    def call(theta, B=2, K=3, V=64, ws=0x80000):
        return lib.spec_verify_typical(vp(0x10000), 1, vp(0x30000), vp(0x40000), vp(0x50000),
                                       ctypes.c_float(theta), ctypes.c_uint64(0), B, K, V,
                                       vp(0x60000), vp(0x70000), vp(ws), 1 << 30, vp(0),
                                       ctypes.c_uint32(0), None, None, None)
    assert call(float("nan")) == bd.SPEC_ERR_INVALID_ARG
    assert call(0.1, K=32) == bd.SPEC_ERR_INVALID_ARG
    assert call(0.1, V=1020) == bd.SPEC_ERR_UNSUPPORTED
    assert call(0.1, B=0) == bd.SPEC_OK
    assert call(float("inf"), ws=0x80010) == bd.SPEC_ERR_WORKSPACE


def test_early_exit_host_side_errors(lib):
    """spec_verify_early_exit checks as spec_verify_ex does, plus seed_dev alignment."""
    from speculative_decoding_verification_51_gb300 import binding as bd
    vp = ctypes.c_void_p

    def call(B=2, K=3, V=64, seed_dev=None, ws=0x80000):
        return lib.spec_verify_early_exit(vp(0x10000), 1, vp(0x20000), vp(0x30000), vp(0x40000),
                                          vp(0x50000), ctypes.c_uint64(0), B, K, V, vp(0x60000),
                                          vp(0x70000), vp(ws), 1 << 30, vp(0), ctypes.c_uint32(0),
                                          None, None, None, None if seed_dev is None else vp(seed_dev))
    assert call(K=32) == bd.SPEC_ERR_INVALID_ARG
    assert call(V=1020) == bd.SPEC_ERR_UNSUPPORTED
    assert call(B=0) == bd.SPEC_OK
    assert call(seed_dev=0x90004) == bd.SPEC_ERR_INVALID_ARG   # not 8-byte aligned
    assert call(ws=0x80010) == bd.SPEC_ERR_WORKSPACE


@pytest.mark.parametrize("entry", ["spec_verify_all_rows", "spec_verify_by_request"])
def test_forced_path_host_side_errors(lib, entry):
    """The two forced-path entry points check as spec_verify_ex does, plus
    seed_dev alignment and a NULL entry among the events."""
    from speculative_decoding_verification_51_gb300 import binding as bd
    vp = ctypes.c_void_p
    fn = getattr(lib, entry)

    def call(B=2, K=3, V=64, seed_dev=None, ws=0x80000, events=None):
        return fn(vp(0x10000), 1, vp(0x20000), vp(0x30000), vp(0x40000), vp(0x50000),
                  ctypes.c_uint64(0), B, K, V, vp(0x60000), vp(0x70000), vp(ws), 1 << 30, vp(0),
                  ctypes.c_uint32(0), None, None, None,
                  None if seed_dev is None else vp(seed_dev), events)
    assert call(K=32) == bd.SPEC_ERR_INVALID_ARG
    assert call(V=1020) == bd.SPEC_ERR_UNSUPPORTED
    assert call(B=0) == bd.SPEC_OK
    assert call(seed_dev=0x90004) == bd.SPEC_ERR_INVALID_ARG
    assert call(ws=0x80010) == bd.SPEC_ERR_WORKSPACE
    ev = (ctypes.c_void_p * 6)(*([0x1000] * 5 + [0]))
    assert call(events=ev) == bd.SPEC_ERR_INVALID_ARG


def test_path_query_rejects_bad_sizes(lib):
    """spec_verify_path answers -1 for sizes or dtypes no call accepts."""
    assert lib.spec_verify_path(256, 32, 151936, 1) == -1   # K above the maximum
    assert lib.spec_verify_path(256, 3, 1020, 1) == -1      # V not a multiple of 8
    assert lib.spec_verify_path(256, 3, 151936, 7) == -1    # no such dtype
    assert lib.spec_verify_path(-1, 3, 151936, 1) == -1


def test_lmhead_host_side_errors(lib):
    """spec_lmhead_logits / spec_verify_lmhead reject bad sizes and pointers
    before any launch."""
    from speculative_decoding_verification_51_gb300 import binding as bd
    vp = ctypes.c_void_p

    def proj(rows=4, H=64, V=64, hid=0x10000, w=0x20000, out=0x30000, st=0x40000):
        return lib.spec_lmhead_logits(vp(hid), vp(w), rows, H, V, vp(out), vp(st), vp(0))
    assert proj(H=96) == bd.SPEC_ERR_UNSUPPORTED      # H not a multiple of 64
    assert proj(V=1020) == bd.SPEC_ERR_UNSUPPORTED    # V not a multiple of 8
    assert proj(H=0) == bd.SPEC_ERR_INVALID_ARG
    assert proj(rows=-1) == bd.SPEC_ERR_INVALID_ARG
    assert proj(rows=0) == bd.SPEC_OK
    assert proj(hid=0) == bd.SPEC_ERR_INVALID_ARG
    assert proj(st=0) == bd.SPEC_ERR_INVALID_ARG
    assert proj(w=0x20008) == bd.SPEC_ERR_UNSUPPORTED  # not 16-byte aligned

    assert lib.spec_verify_lmhead_workspace_size(4, 3, 64, 96) == 0
    n = lib.spec_verify_lmhead_workspace_size(4, 3, 64, 128)
    assert n >= lib.spec_verify_workspace_size(4, 3, 64) + 4 * 4 * 128 * 2

    def fused(B=4, K=3, V=64, H=128, hid=0x10000, ws_bytes=None):
        return lib.spec_verify_lmhead(vp(hid), vp(0x20000), H, vp(0x30000), vp(0x40000),
                                      vp(0x50000), vp(0x60000), vp(0x70000), ctypes.c_uint64(0),
                                      B, K, V, vp(0x80000), vp(0x90000), vp(0x100000),
                                      n if ws_bytes is None else ws_bytes, vp(0),
                                      ctypes.c_uint32(0), None, None, None)
    assert fused(H=96) == bd.SPEC_ERR_UNSUPPORTED
    assert fused(K=32) == bd.SPEC_ERR_INVALID_ARG
    assert fused(B=0) == bd.SPEC_OK
    assert fused(hid=0) == bd.SPEC_ERR_INVALID_ARG
    assert fused(ws_bytes=n - 1) == bd.SPEC_ERR_WORKSPACE
