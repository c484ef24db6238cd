"""ctypes binding of the spec_verify C ABI (include/spec_verify.h).

Argument marshalling only: tensors are checked for device, dtype, shape and
contiguity, their device pointers and the current CUDA stream are passed to
the library, and a non-OK status raises.  Every step of verification runs in
the library's kernels; there is no fallback.  torch is used for allocation
(outputs, workspace) and for the stream handle.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

SPEC_OK, SPEC_ERR_INVALID_ARG, SPEC_ERR_UNSUPPORTED, SPEC_ERR_CUDA, SPEC_ERR_WORKSPACE = range(5)
SPEC_F32, SPEC_BF16 = 0, 1
BADBIT = {"num_draft": 1, "temperature": 2, "draft_id": 4, "empty_row": 8, "no_probs": 16,
          "timeout": 32, "tree": 64}
MODE_BAD, MODE_GREEDY, MODE_RESIDUAL, MODE_BONUS, MODE_FALLBACK, MODE_TYPICAL = -1, 0, 1, 2, 3, 4
MAX_K = 31
# kernels of one call, in launch order: the request-by-request verifier
# (spec_verify_by_request, and spec_verify where verify_path() is 1), and the
# all-rows verifier (spec_verify_all_rows, and spec_verify where it is 0)
KERNELS = ("k_prep", "k_verify")
KERNELS_ALL_ROWS = ("k_plan", "k_row_stats", "k_accept_all", "k_sample", "k_emit")
N_KERNELS = len(KERNELS)
N_MARKS = 6  # events a profiled call records

_LOCK = threading.Lock()
_LIB = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)}")


def _declare(lib):
    vp, i32, u32, u64, i64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64,
                                  ctypes.c_int64, ctypes.c_size_t)
    lib.spec_status_str.restype = ctypes.c_char_p
    lib.spec_status_str.argtypes = [i32]
    lib.spec_verify_workspace_size.restype = sz
    lib.spec_verify_workspace_size.argtypes = [i32, i32, i32]
    lib.spec_verify_status_ptr.restype = vp
    lib.spec_verify_status_ptr.argtypes = [vp]
    common = [vp, i32, vp, vp, vp, vp, u64, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.spec_verify.restype = i32
    lib.spec_verify.argtypes = common
    lib.spec_verify_ex.restype = i32
    lib.spec_verify_ex.argtypes = common + [u32, vp, vp, vp]
    lib.spec_verify_dev_seed.restype = i32
    lib.spec_verify_dev_seed.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, i32, i32, vp, vp, vp,
                                         sz, vp, u32, vp, vp, vp]
    lib.spec_verify_early_exit.restype = i32
    lib.spec_verify_early_exit.argtypes = common + [u32, vp, vp, vp, vp]
    lib.spec_verify_all_rows.restype = i32
    lib.spec_verify_all_rows.argtypes = common + [u32, vp, vp, vp, vp, vp]
    lib.spec_verify_by_request.restype = i32
    lib.spec_verify_by_request.argtypes = common + [u32, vp, vp, vp, vp, vp]
    lib.spec_verify_path.restype = i32
    lib.spec_verify_path.argtypes = [i32, i32, i32, i32]
    lib.spec_verify_lmhead_workspace_size.restype = sz
    lib.spec_verify_lmhead_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.spec_verify_lmhead.restype = i32
    lib.spec_verify_lmhead.argtypes = [vp, vp, i32, vp, vp, vp, vp, vp, u64, i32, i32, i32, vp, vp,
                                       vp, sz, vp, u32, vp, vp, vp]
    lib.spec_lmhead_logits.restype = i32
    lib.spec_lmhead_logits.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    lib.spec_verify_tree_workspace_size.restype = sz
    lib.spec_verify_tree_workspace_size.argtypes = [i32, i32, i32]
    lib.spec_verify_tree.restype = i32
    lib.spec_verify_tree.argtypes = [vp, i32, vp, vp, vp, vp, vp, u64, i32, i32, i32, vp, vp, vp,
                                     vp, sz, vp, u32, vp, vp, vp]
    lib.spec_verify_typical.restype = i32
    lib.spec_verify_typical.argtypes = [vp, i32, vp, vp, vp, ctypes.c_float, u64, i32, i32, i32,
                                        vp, vp, vp, sz, vp, u32, vp, vp, vp]
    lib.spec_verify_profiled.restype = i32
    lib.spec_verify_profiled.argtypes = common + [vp]
    lib.spec_verify_host_small_bytes.restype = sz
    lib.spec_verify_host_small_bytes.argtypes = [i32, i32]
    lib.spec_verify_host.restype = i32
    lib.spec_verify_host.argtypes = [vp, i32, vp, vp, vp, vp, u64, i32, i32, i32, vp, vp, vp, vp,
                                     vp, vp, sz, vp]
    lib.spec_philox_fill.restype = i32
    lib.spec_philox_fill.argtypes = [u64, vp, i64, vp, vp]
    return lib


def library_path() -> str:
    return _build.lib_path()


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            path = _build.lib_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"spec_verify CUDA library missing ({path}); build it with "
                    "`python -m speculative_decoding_verification_51_gb300.build`")
            _LIB = _declare(ctypes.CDLL(path))
        return _LIB


def status_str(status: int) -> str:
    return lib().spec_status_str(int(status)).decode()


def workspace_size(B: int, K: int, V: int) -> int:
    return int(lib().spec_verify_workspace_size(B, K, V))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype, shape=None, device=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def new_workspace(B: int, K: int, V: int, device) -> torch.Tensor:
    n = workspace_size(B, K, V)
    if n == 0:
        raise ValueError(f"unsupported sizes B={B} K={K} V={V}")
    return torch.empty(n, dtype=torch.uint8, device=device)


def spec_verify(target_logits: torch.Tensor, draft_probs: torch.Tensor | None,
                draft_ids: torch.Tensor, num_draft: torch.Tensor, temperature: torch.Tensor,
                seed: int, *, out_ids: torch.Tensor | None = None,
                out_num_accepted: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, stream=None, request_offset: int = 0,
                debug: bool = False, dev_status: torch.Tensor | None = None,
                seed_dev: torch.Tensor | None = None, early_exit: bool = False,
                all_rows: bool = False, by_request: bool = False):
    """Verify drafts on the GPU (see include/spec_verify.h for the semantics).

    seed_dev: a one-element int64 CUDA tensor; if given, the kernels read the
    seed from it when they run (spec_verify_dev_seed, for CUDA graph capture)
    and `seed` is ignored.
    early_exit: the K + 1-pass form of reading each request's rows only up to
    its first rejection (spec_verify_early_exit); same outputs.
    all_rows: read and check every row 0..num_draft[b] in one streaming pass
    (spec_verify_all_rows); same outputs except that an all -inf sampling row
    after the first rejection makes the request bad.
    by_request: the request-by-request verifier at any B
    (spec_verify_by_request).  Without either flag the call runs the one
    verify_path() names.
    Returns (out_ids [B, K+1] int32, out_num_accepted [B] int32), plus
    (dbg_rows [B, K+1, 4], dbg_req [B, 4]) when debug=True.
    """
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    if target_logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    elif target_logits.dtype == torch.float32:
        dt = SPEC_F32
    else:
        raise ValueError("target_logits must be bfloat16 or float32")
    _check(target_logits, "target_logits", target_logits.dtype)
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, K, V), dev)
    _check(draft_ids, "draft_ids", torch.int32, (B, K), dev)
    _check(num_draft, "num_draft", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    if out_ids is None:
        out_ids = torch.empty((B, K1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(out_ids, "out_ids", torch.int32, (B, K1), dev)
    _check(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    if workspace is None:
        workspace = new_workspace(B, K, V, dev)
    dbg_rows = dbg_req = None
    if debug:
        dbg_rows = torch.empty((B, K1, 4), dtype=torch.float32, device=dev)
        dbg_req = torch.empty((B, 4), dtype=torch.float32, device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,), dev)
    if seed_dev is not None:
        _check(seed_dev, "seed_dev", torch.int64, (1,), dev)
    with torch.cuda.device(dev):
        st = _stream(stream)
        if all_rows or by_request:
            if all_rows and by_request:
                raise ValueError("all_rows and by_request exclude each other")
            fn = lib().spec_verify_all_rows if all_rows else lib().spec_verify_by_request
            rc = fn(
                _p(target_logits), dt, _p(draft_probs), _p(draft_ids), _p(num_draft),
                _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _p(out_ids),
                _p(out_num_accepted), _p(workspace), workspace.numel(), st,
                ctypes.c_uint32(request_offset & 0xFFFFFFFF), _p(dbg_rows), _p(dbg_req),
                _p(dev_status), _p(seed_dev), None)
        elif early_exit:
            rc = lib().spec_verify_early_exit(
                _p(target_logits), dt, _p(draft_probs), _p(draft_ids), _p(num_draft),
                _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _p(out_ids),
                _p(out_num_accepted), _p(workspace), workspace.numel(), st,
                ctypes.c_uint32(request_offset & 0xFFFFFFFF), _p(dbg_rows), _p(dbg_req),
                _p(dev_status), _p(seed_dev))
        elif seed_dev is not None:
            rc = lib().spec_verify_dev_seed(
                _p(target_logits), dt, _p(draft_probs), _p(draft_ids), _p(num_draft),
                _p(temperature), _p(seed_dev), B, K, V, _p(out_ids), _p(out_num_accepted),
                _p(workspace), workspace.numel(), st, ctypes.c_uint32(request_offset & 0xFFFFFFFF),
                _p(dbg_rows), _p(dbg_req), _p(dev_status))
        elif debug or request_offset or dev_status is not None:
            rc = lib().spec_verify_ex(
                _p(target_logits), dt, _p(draft_probs), _p(draft_ids), _p(num_draft),
                _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _p(out_ids),
                _p(out_num_accepted), _p(workspace), workspace.numel(), st,
                ctypes.c_uint32(request_offset & 0xFFFFFFFF), _p(dbg_rows), _p(dbg_req),
                _p(dev_status))
        else:
            rc = lib().spec_verify(
                _p(target_logits), dt, _p(draft_probs), _p(draft_ids), _p(num_draft),
                _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _p(out_ids),
                _p(out_num_accepted), _p(workspace), workspace.numel(), st)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify")
    if debug:
        return out_ids, out_num_accepted, dbg_rows, dbg_req
    return out_ids, out_num_accepted


def spec_verify_typical(target_logits: torch.Tensor, draft_ids: torch.Tensor,
                        num_draft: torch.Tensor, temperature: torch.Tensor, threshold: float,
                        seed: int, *, out_ids: torch.Tensor | None = None,
                        out_num_accepted: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None,
                        request_offset: int = 0, debug: bool = False,
                        dev_status: torch.Tensor | None = None):
    """Typical-acceptance verification on the GPU (include/spec_verify.h,
    spec_verify_typical): drafts are kept while p_j(x_j) >= threshold.

    Returns (out_ids, out_num_accepted), plus (dbg_rows, dbg_req) when debug=True.
    """
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, K+1, V]")
    B, K1, V = target_logits.shape
    K = K1 - 1
    dev = target_logits.device
    if target_logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    elif target_logits.dtype == torch.float32:
        dt = SPEC_F32
    else:
        raise ValueError("target_logits must be bfloat16 or float32")
    _check(target_logits, "target_logits", target_logits.dtype)
    _check(draft_ids, "draft_ids", torch.int32, (B, K), dev)
    _check(num_draft, "num_draft", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    if out_ids is None:
        out_ids = torch.empty((B, K1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(out_ids, "out_ids", torch.int32, (B, K1), dev)
    _check(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    if workspace is None:
        workspace = new_workspace(B, K, V, dev)
    dbg_rows = dbg_req = None
    if debug:
        dbg_rows = torch.empty((B, K1, 4), dtype=torch.float32, device=dev)
        dbg_req = torch.empty((B, 4), dtype=torch.float32, device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,), dev)
    with torch.cuda.device(dev):
        rc = lib().spec_verify_typical(
            _p(target_logits), dt, _p(draft_ids), _p(num_draft), _p(temperature),
            ctypes.c_float(threshold), ctypes.c_uint64(seed & (2**64 - 1)), B, K, V,
            _p(out_ids), _p(out_num_accepted), _p(workspace), workspace.numel(),
            _stream(stream), ctypes.c_uint32(request_offset & 0xFFFFFFFF), _p(dbg_rows),
            _p(dbg_req), _p(dev_status))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_typical")
    if debug:
        return out_ids, out_num_accepted, dbg_rows, dbg_req
    return out_ids, out_num_accepted


def spec_verify_tree(target_logits: torch.Tensor, draft_probs: torch.Tensor | None,
                     tree_tokens: torch.Tensor, tree_parents: torch.Tensor,
                     num_nodes: torch.Tensor, temperature: torch.Tensor, seed: int, *,
                     workspace: torch.Tensor | None = None, stream=None, request_offset: int = 0,
                     debug: bool = False, dev_status: torch.Tensor | None = None):
    """Token-tree verification on the GPU (include/spec_verify.h,
    spec_verify_tree).  Returns (out_ids [B, N], out_num_accepted [B],
    out_last_node [B]), plus (dbg_nodes [B, N, 4], dbg_req [B, 4]) when debug."""
    if target_logits.dim() != 3:
        raise ValueError("target_logits must be [B, N, V]")
    B, N, V = target_logits.shape
    dev = target_logits.device
    if target_logits.dtype == torch.bfloat16:
        dt = SPEC_BF16
    elif target_logits.dtype == torch.float32:
        dt = SPEC_F32
    else:
        raise ValueError("target_logits must be bfloat16 or float32")
    _check(target_logits, "target_logits", target_logits.dtype)
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, N, V), dev)
    _check(tree_tokens, "tree_tokens", torch.int32, (B, N), dev)
    _check(tree_parents, "tree_parents", torch.int32, (B, N), dev)
    _check(num_nodes, "num_nodes", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    out_ids = torch.empty((B, N), dtype=torch.int32, device=dev)
    out_nacc = torch.empty((B,), dtype=torch.int32, device=dev)
    out_last = torch.empty((B,), dtype=torch.int32, device=dev)
    if workspace is None:
        n = int(lib().spec_verify_tree_workspace_size(B, N, V))
        if n == 0:
            raise ValueError("unsupported tree size")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    dbg_nodes = dbg_req = None
    if debug:
        dbg_nodes = torch.empty((B, N, 4), dtype=torch.float32, device=dev)
        dbg_req = torch.empty((B, 4), dtype=torch.float32, device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,), dev)
    with torch.cuda.device(dev):
        rc = lib().spec_verify_tree(
            _p(target_logits), dt, _p(draft_probs), _p(tree_tokens), _p(tree_parents),
            _p(num_nodes), _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, N, V,
            _p(out_ids), _p(out_nacc), _p(out_last), _p(workspace), workspace.numel(),
            _stream(stream), ctypes.c_uint32(request_offset & 0xFFFFFFFF), _p(dbg_nodes),
            _p(dbg_req), _p(dev_status))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_tree")
    if debug:
        return out_ids, out_nacc, out_last, dbg_nodes, dbg_req
    return out_ids, out_nacc, out_last


def spec_verify_profiled(target_logits, draft_probs, draft_ids, num_draft, temperature, seed,
                         out_ids, out_num_accepted, workspace, events, stream=None,
                         all_rows: bool = False, by_request: bool = False) -> None:
    """spec_verify (all_rows=True: spec_verify_all_rows; by_request=True:
    spec_verify_by_request) with N_MARKS torch.cuda.Event marks around its
    kernels: events[i] -> events[i + 1] brackets kernel i of KERNELS
    (KERNELS_ALL_ROWS for the all-rows verifier).  The events must already
    have been recorded once, so that they exist."""
    B, K1, V = target_logits.shape
    dt = SPEC_BF16 if target_logits.dtype == torch.bfloat16 else SPEC_F32
    if len(events) != N_MARKS:
        raise ValueError(f"need {N_MARKS} events")
    handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    with torch.cuda.device(target_logits.device):
        args = (_p(target_logits), dt, _p(draft_probs), _p(draft_ids), _p(num_draft),
                _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, K1 - 1, V, _p(out_ids),
                _p(out_num_accepted), _p(workspace), workspace.numel(), _stream(stream))
        if all_rows or by_request:
            fn = lib().spec_verify_all_rows if all_rows else lib().spec_verify_by_request
            rc = fn(*args, ctypes.c_uint32(0), None, None, None, None, handles)
        else:
            rc = lib().spec_verify_profiled(*args, handles)
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_profiled")


def verify_path(B: int, K: int, V: int, dtype: torch.dtype, device=None) -> int:
    """1 if spec_verify runs the request-by-request verifier for these sizes
    on `device` (default: the current CUDA device), 0 if the all-rows pass."""
    dt = SPEC_BF16 if dtype == torch.bfloat16 else SPEC_F32
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        r = lib().spec_verify_path(B, K, V, dt)
    if r < 0:
        raise SpecVerifyError(SPEC_ERR_INVALID_ARG, "spec_verify_path")
    return r


def status_word(workspace: torch.Tensor) -> torch.Tensor:
    """The device status word of the last call that used `workspace` (a view)."""
    return workspace[12:16].view(torch.int32)


def host_small_bytes(B: int, K: int) -> int:
    return int(lib().spec_verify_host_small_bytes(B, K))


def spec_verify_host(h_logits: torch.Tensor, h_probs: torch.Tensor | None, h_ids: torch.Tensor,
                     h_num: torch.Tensor, h_temp: torch.Tensor, seed: int,
                     h_out_ids: torch.Tensor, h_out_nacc: torch.Tensor, d_logits: torch.Tensor,
                     d_probs: torch.Tensor | None, d_small: torch.Tensor,
                     workspace: torch.Tensor, stream=None) -> None:
    """Host-buffer variant: copies in, verifies, copies out (asynchronous)."""
    B, K1, V = h_logits.shape
    K = K1 - 1
    dt = SPEC_BF16 if h_logits.dtype == torch.bfloat16 else SPEC_F32
    for t, n in ((h_logits, "h_logits"), (h_ids, "h_ids"), (h_num, "h_num"), (h_temp, "h_temp"),
                 (h_out_ids, "h_out_ids"), (h_out_nacc, "h_out_nacc")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    with torch.cuda.device(d_logits.device):
        rc = lib().spec_verify_host(
            _p(h_logits), dt, _p(h_probs), _p(h_ids), _p(h_num), _p(h_temp),
            ctypes.c_uint64(seed & (2**64 - 1)), B, K, V, _p(h_out_ids), _p(h_out_nacc),
            _p(d_logits), _p(d_probs), _p(d_small), _p(workspace), workspace.numel(),
            _stream(stream))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_host")


def philox_fill(seed: int, ctrs: torch.Tensor, stream=None) -> torch.Tensor:
    """Philox4x32-10 of the library: ctrs [n, 4] int32 (bit patterns) on the GPU."""
    _check(ctrs, "ctrs", torch.int32)
    out = torch.empty_like(ctrs)
    with torch.cuda.device(ctrs.device):
        rc = lib().spec_philox_fill(ctypes.c_uint64(seed & (2**64 - 1)), _p(ctrs),
                                    ctrs.numel() // 4, _p(out), _stream(stream))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_philox_fill")
    return out


def lmhead_logits(hidden: torch.Tensor, lm_head: torch.Tensor, *, out: torch.Tensor | None = None,
                  dev_status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """bf16 logits = hidden [rows, H] @ lm_head [V, H]^T on the tensor cores
    (include/spec_verify.h, spec_lmhead_logits)."""
    if hidden.dim() != 2 or lm_head.dim() != 2 or hidden.shape[1] != lm_head.shape[1]:
        raise ValueError("hidden must be [rows, H] and lm_head [V, H]")
    rows, H = hidden.shape
    V = lm_head.shape[0]
    dev = hidden.device
    _check(hidden, "hidden", torch.bfloat16, device=dev)
    _check(lm_head, "lm_head", torch.bfloat16, device=dev)
    if out is None:
        out = torch.empty((rows, V), dtype=torch.bfloat16, device=dev)
    _check(out, "out", torch.bfloat16, (rows, V), dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(dev_status, "dev_status", torch.int32, (1,), dev)
    with torch.cuda.device(dev):
        rc = lib().spec_lmhead_logits(_p(hidden), _p(lm_head), rows, H, V, _p(out), _p(dev_status),
                                      _stream(stream))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_lmhead_logits")
    return out


def spec_verify_lmhead(hidden: torch.Tensor, lm_head: torch.Tensor, draft_probs: torch.Tensor | None,
                       draft_ids: torch.Tensor, num_draft: torch.Tensor, temperature: torch.Tensor,
                       seed: int, *, logits_out: torch.Tensor | None = None,
                       out_ids: torch.Tensor | None = None,
                       out_num_accepted: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, stream=None, request_offset: int = 0,
                       debug: bool = False, dev_status: torch.Tensor | None = None):
    """Verification with the logits produced in the call from hidden states
    (include/spec_verify.h, spec_verify_lmhead).

    hidden [B, K+1, H] bf16, lm_head [V, H] bf16.  Returns (out_ids,
    out_num_accepted, logits_out) plus (dbg_rows, dbg_req) when debug=True.
    """
    if hidden.dim() != 3 or lm_head.dim() != 2 or hidden.shape[2] != lm_head.shape[1]:
        raise ValueError("hidden must be [B, K+1, H] and lm_head [V, H]")
    B, K1, H = hidden.shape
    K, V = K1 - 1, lm_head.shape[0]
    dev = hidden.device
    _check(hidden, "hidden", torch.bfloat16, device=dev)
    _check(lm_head, "lm_head", torch.bfloat16, device=dev)
    if draft_probs is not None:
        _check(draft_probs, "draft_probs", torch.float32, (B, K, V), dev)
    _check(draft_ids, "draft_ids", torch.int32, (B, K), dev)
    _check(num_draft, "num_draft", torch.int32, (B,), dev)
    _check(temperature, "temperature", torch.float32, (B,), dev)
    if logits_out is None:
        logits_out = torch.empty((B, K1, V), dtype=torch.bfloat16, device=dev)
    _check(logits_out, "logits_out", torch.bfloat16, (B, K1, V), dev)
    if out_ids is None:
        out_ids = torch.empty((B, K1), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(out_ids, "out_ids", torch.int32, (B, K1), dev)
    _check(out_num_accepted, "out_num_accepted", torch.int32, (B,), dev)
    if workspace is None:
        n = int(lib().spec_verify_lmhead_workspace_size(B, K, V, H))
        if n == 0:
            raise ValueError(f"unsupported sizes B={B} K={K} V={V} H={H}")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev)
    dbg_rows = dbg_req = None
    if debug:
        dbg_rows = torch.empty((B, K1, 4), dtype=torch.float32, device=dev)
        dbg_req = torch.empty((B, 4), dtype=torch.float32, device=dev)
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (1,), dev)
    with torch.cuda.device(dev):
        rc = lib().spec_verify_lmhead(
            _p(hidden), _p(lm_head), H, _p(logits_out), _p(draft_probs), _p(draft_ids),
            _p(num_draft), _p(temperature), ctypes.c_uint64(seed & (2**64 - 1)), B, K, V,
            _p(out_ids), _p(out_num_accepted), _p(workspace), workspace.numel(), _stream(stream),
            ctypes.c_uint32(request_offset & 0xFFFFFFFF), _p(dbg_rows), _p(dbg_req),
            _p(dev_status))
    if rc != SPEC_OK:
        raise SpecVerifyError(rc, "spec_verify_lmhead")
    if debug:
        return out_ids, out_num_accepted, logits_out, dbg_rows, dbg_req
    return out_ids, out_num_accepted, logits_out
