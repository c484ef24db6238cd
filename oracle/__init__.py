"""Float64 CPU oracle of the batched speculative-sampling verifier.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package.  The product path (the CUDA library and its binding)
never loads it and never falls back to it.

The arithmetic lives in ``spec_verify_oracle.c`` (plain C, float64,
``-ffp-contract=off``, no fast-math); this module compiles it with the host
``gcc`` into ``oracle/_build/`` and wraps it with ctypes.  See the C file's
header for the definitions it restates and the readings it takes where the
source pages are silent.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(the pages' worked ratio, closed forms, brute force on tiny vocabularies, a
chi-square test of losslessness, the Philox known-answer vectors and planted
mistakes that the pins must catch).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_verify_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIB = None

ROW_W = 4  # per-row diagnostics: p(x_j), q(x_j), u_j, accepted (-1 untested)
R_PX, R_QX, R_U, R_ACCEPT = 0, 1, 2, 3
REQ_W = 9  # per-request: mode, n_acc, emit row, u', mass, lo, hi, probe lo, probe hi
Q_MODE, Q_NACC, Q_EROW, Q_UEMIT, Q_MASS, Q_LO, Q_HI, Q_PLO, Q_PHI = range(9)
MODE_BAD, MODE_GREEDY, MODE_RESIDUAL, MODE_BONUS, MODE_FALLBACK, MODE_TYPICAL = -1, 0, 1, 2, 3, 4
RULE_LOSSLESS, RULE_TYPICAL = 0, 1

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math"]


def lib_path(src: str = _SRC, tag: str = "") -> str:
    return os.path.join(_BUILD, f"liboracle{tag}_{platform.machine()}.so")


def build(src: str = _SRC, out: str | None = None, extra: list[str] | None = None) -> str:
    """Compile the oracle (or a variant of its source) with gcc; return the .so path."""
    out = out or lib_path(src)
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src) and not extra:
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", *CFLAGS, *(extra or []), "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    vp, i32, u64, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_int64
    lib.oracle_spec_verify.restype = i32
    lib.oracle_spec_verify.argtypes = [vp, i32, vp, vp, vp, vp, u64, i32, i32, i32,
                                       vp, vp, vp, vp, vp, vp, vp, i32]
    lib.oracle_spec_verify_rule.restype = i32
    lib.oracle_spec_verify_rule.argtypes = [vp, i32, vp, vp, vp, vp, u64, i32, i32, i32,
                                            vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                            ctypes.c_double]
    lib.oracle_tree_verify.restype = i32
    lib.oracle_tree_verify.argtypes = [vp, i32, vp, vp, vp, vp, vp, u64, i32, i32, i32,
                                       vp, vp, vp, vp, vp, vp, vp, vp, i32]
    lib.oracle_philox_blocks.restype = None
    lib.oracle_philox_blocks.argtypes = [vp, vp, i64, vp]
    lib.oracle_row_uniforms.restype = None
    lib.oracle_row_uniforms.argtypes = [u64, u64, ctypes.c_uint32,
                                        ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_double)]
    lib.oracle_uniform_from_bits.restype = ctypes.c_double
    lib.oracle_uniform_from_bits.argtypes = [ctypes.c_uint32]
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the compiled oracle (building it first if needed)."""
    global _LIB
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _LOCK:
        if _LIB is None:
            _LIB = _declare(ctypes.CDLL(build()))
        return _LIB


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def spec_verify(target_logits: np.ndarray, draft_probs: np.ndarray | None,
                draft_ids: np.ndarray, num_draft: np.ndarray, temperature: np.ndarray,
                seed: int, *, logits_dtype: str | None = None,
                req_index: np.ndarray | None = None, uniforms: np.ndarray | None = None,
                probe: np.ndarray | None = None, n_threads: int = 0, lib=None,
                typical_threshold: float | None = None) -> dict:
    """Run the oracle.

    target_logits: [B, K+1, V] float32, or uint16 bf16 bit patterns.
    draft_probs:   [B, K, V] float32 (None only if every request is greedy).
    draft_ids [B, K] int32, num_draft [B] int32, temperature [B] float32.
    uniforms: None (Philox(seed, b, j)) or [B, K+1, 2] float64 used as given.
    req_index: global request index per local request (Philox counter).
    probe: [B] int32 token ids whose emission-CDF interval is reported.
    typical_threshold: None for the lossless rule, else the hard threshold of
    the typical-acceptance rule.
    """
    lib = lib or load()
    tl = np.ascontiguousarray(target_logits)
    if logits_dtype is None:
        logits_dtype = "bf16" if tl.dtype == np.uint16 else "f32"
    if logits_dtype == "bf16":
        assert tl.dtype in (np.uint16, np.int16), tl.dtype
        dt = 1
    else:
        tl = np.ascontiguousarray(tl, dtype=np.float32)
        dt = 0
    B, K1, V = tl.shape
    K = K1 - 1
    dp = None if draft_probs is None else np.ascontiguousarray(draft_probs, dtype=np.float32)
    if dp is not None:
        assert dp.shape == (B, K, V), (dp.shape, (B, K, V))
    di = np.ascontiguousarray(draft_ids, dtype=np.int32).reshape(B, K)
    nd = np.ascontiguousarray(num_draft, dtype=np.int32).reshape(B)
    tp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    ri = None if req_index is None else np.ascontiguousarray(req_index, dtype=np.int64).reshape(B)
    un = None if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, K1, 2)
    pr = None if probe is None else np.ascontiguousarray(probe, dtype=np.int32).reshape(B)
    out_ids = np.empty((B, K1), dtype=np.int32)
    out_nacc = np.empty((B,), dtype=np.int32)
    row_diag = np.empty((B, K1, ROW_W), dtype=np.float64)
    req_diag = np.empty((B, REQ_W), dtype=np.float64)
    if typical_threshold is None:
        n_bad = lib.oracle_spec_verify(_ptr(tl), dt, _ptr(dp), _ptr(di), _ptr(nd), _ptr(tp),
                                       ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _ptr(ri),
                                       _ptr(un), _ptr(pr), _ptr(out_ids), _ptr(out_nacc),
                                       _ptr(row_diag), _ptr(req_diag), int(n_threads))
    else:
        n_bad = lib.oracle_spec_verify_rule(
            _ptr(tl), dt, _ptr(dp), _ptr(di), _ptr(nd), _ptr(tp),
            ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _ptr(ri), _ptr(un), _ptr(pr),
            _ptr(out_ids), _ptr(out_nacc), _ptr(row_diag), _ptr(req_diag), int(n_threads),
            RULE_TYPICAL, float(typical_threshold))
    if n_bad < 0:
        raise ValueError("oracle_spec_verify rejected its arguments")
    return {"out_ids": out_ids, "out_num_accepted": out_nacc, "row_diag": row_diag,
            "req_diag": req_diag, "n_bad": int(n_bad)}


def tree_verify(target_logits: np.ndarray, draft_probs: np.ndarray | None,
                tree_tokens: np.ndarray, tree_parents: np.ndarray, num_nodes: np.ndarray,
                temperature: np.ndarray, seed: int, *, logits_dtype: str | None = None,
                req_index: np.ndarray | None = None, uniforms: np.ndarray | None = None,
                probe: np.ndarray | None = None, n_threads: int = 0, lib=None) -> dict:
    """Token-tree verification by the oracle.

    target_logits: [B, N, V] float32, or uint16 bf16 bit patterns (row v: the
    target's logits for the token after node v).  draft_probs [B, N, V]
    float32 (row c: the distribution node c's token was drawn from; row 0
    unused) or None.  tree_tokens / tree_parents [B, N] int32 (node 0 is the
    root), num_nodes [B], temperature [B].
    uniforms: None (Philox) or [B, N, 2]: lane 0 of entry c - 1 is child c's
    acceptance uniform, lane 1 of entry v node v's emission uniform.
    """
    lib = lib or load()
    tl = np.ascontiguousarray(target_logits)
    if logits_dtype is None:
        logits_dtype = "bf16" if tl.dtype == np.uint16 else "f32"
    if logits_dtype == "bf16":
        assert tl.dtype in (np.uint16, np.int16), tl.dtype
        dt = 1
    else:
        tl = np.ascontiguousarray(tl, dtype=np.float32)
        dt = 0
    B, N, V = tl.shape
    dp = None if draft_probs is None else np.ascontiguousarray(draft_probs, dtype=np.float32)
    if dp is not None:
        assert dp.shape == (B, N, V), (dp.shape, (B, N, V))
    tt = np.ascontiguousarray(tree_tokens, dtype=np.int32).reshape(B, N)
    tpar = np.ascontiguousarray(tree_parents, dtype=np.int32).reshape(B, N)
    nn = np.ascontiguousarray(num_nodes, dtype=np.int32).reshape(B)
    tp = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    ri = None if req_index is None else np.ascontiguousarray(req_index, dtype=np.int64).reshape(B)
    un = None if uniforms is None else np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, N, 2)
    pr = None if probe is None else np.ascontiguousarray(probe, dtype=np.int32).reshape(B)
    out_ids = np.empty((B, N), dtype=np.int32)
    out_nacc = np.empty((B,), dtype=np.int32)
    out_last = np.empty((B,), dtype=np.int32)
    node_diag = np.empty((B, N, ROW_W), dtype=np.float64)
    req_diag = np.empty((B, REQ_W), dtype=np.float64)
    n_bad = lib.oracle_tree_verify(_ptr(tl), dt, _ptr(dp), _ptr(tt), _ptr(tpar), _ptr(nn),
                                   _ptr(tp), ctypes.c_uint64(seed & (2**64 - 1)), B, N, V,
                                   _ptr(ri), _ptr(un), _ptr(pr), _ptr(out_ids), _ptr(out_nacc),
                                   _ptr(out_last), _ptr(node_diag), _ptr(req_diag),
                                   int(n_threads))
    if n_bad < 0:
        raise ValueError("oracle_tree_verify rejected its arguments")
    return {"out_ids": out_ids, "out_num_accepted": out_nacc, "out_last_node": out_last,
            "node_diag": node_diag, "req_diag": req_diag, "n_bad": int(n_bad)}


def philox_blocks(ctrs: np.ndarray, key: tuple[int, int], lib=None) -> np.ndarray:
    """Philox4x32-10 blocks: ctrs [n, 4] uint32 -> [n, 4] uint32."""
    lib = lib or load()
    c = np.ascontiguousarray(ctrs, dtype=np.uint32).reshape(-1, 4)
    k = np.asarray(key, dtype=np.uint32).reshape(2)
    out = np.empty_like(c)
    lib.oracle_philox_blocks(_ptr(c), _ptr(k), c.shape[0], _ptr(out))
    return out


def row_uniforms(seed: int, b: int, j: int, lib=None) -> tuple[float, float]:
    """(u_accept, u_emit) of row j of request b."""
    lib = lib or load()
    ua, ue = ctypes.c_double(), ctypes.c_double()
    lib.oracle_row_uniforms(ctypes.c_uint64(seed), ctypes.c_uint64(b), j,
                            ctypes.byref(ua), ctypes.byref(ue))
    return ua.value, ue.value


def uniform_from_bits(x: int, lib=None) -> float:
    lib = lib or load()
    return lib.oracle_uniform_from_bits(x)


def omp_threads() -> int:
    """Threads the oracle uses by default (OMP_NUM_THREADS, else the cores)."""
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v and v.isdigit() else (os.cpu_count() or 1)
