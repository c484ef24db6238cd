"""spec_verify_noalloc, the entry point for callers that cannot allocate device
memory (an engine that already owns every byte of the GPU for its weights and
KV cache, or a plugin host that hands over only input and output buffers):
it must give the same results as spec_verify with a caller-provided
workspace, call after call, and refuse sizes its fixed scratch cannot hold.

Collected last on purpose (file name), so that a run stopping at the first
failure has run every other test before this one.  It needs nothing from the
other tests and passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_51_gb300 import binding
from speculative_decoding_verification_51_gb300 import build as _build
from speculative_decoding_verification_51_gb300 import workloads as W

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 8 << 20  # SPEC_NOALLOC_SCRATCH_BYTES in include/spec_verify.h


def _noalloc_fn():
    _build.build()
    lib = binding.lib()
    f = lib.spec_verify_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    f.restype = i32
    f.argtypes = [vp, i32, vp, vp, vp, vp, ctypes.c_uint64, i32, i32, i32, vp, vp, vp]
    return f


def _call(f, w, seed, out, nacc):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dt = binding.SPEC_BF16 if w.target_logits.dtype == torch.bfloat16 else binding.SPEC_F32
    return f(p(w.target_logits), dt, p(w.draft_probs), p(w.draft_ids), p(w.num_draft),
             p(w.temperature), ctypes.c_uint64(seed), w.B, w.K, w.V, p(out), p(nacc),
             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    f = _noalloc_fn()
    w = W.make_workload(4, device="cuda")  # the largest-vocabulary workload fits the scratch
    assert binding.workspace_size(w.B, w.K, w.V) <= NOALLOC_SCRATCH_BYTES
    for seed in (11, 12):  # two calls in a row share (and reuse) the scratch array
        want_ids, want_n = binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids,
                                               w.num_draft, w.temperature, seed)
        out = torch.full((w.B, w.K + 1), -7, dtype=torch.int32, device="cuda")
        nacc = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        assert _call(f, w, seed, out, nacc) == binding.SPEC_OK
        torch.cuda.synchronize()
        # the two paths run the same kernels: bit-identical results expected
        assert np.array_equal(out.cpu().numpy(), want_ids.cpu().numpy())
        assert np.array_equal(nacc.cpu().numpy(), want_n.cpu().numpy())


def test_noalloc_rejects_sizes_beyond_its_scratch():
    f = _noalloc_fn()
    w = W.make_workload(1, device="cuda")  # small real buffers; never read
    B, K, V = 4096, 8, 151936              # needs far more than 8 MiB of scratch
    assert binding.workspace_size(B, K, V) > NOALLOC_SCRATCH_BYTES
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = f(p(w.target_logits), binding.SPEC_F32, p(w.draft_probs), p(w.draft_ids),
           p(w.num_draft), p(w.temperature), ctypes.c_uint64(0), B, K, V, p(w.draft_ids),
           p(w.num_draft), ctypes.c_void_p(0))
    assert rc == binding.SPEC_ERR_WORKSPACE
