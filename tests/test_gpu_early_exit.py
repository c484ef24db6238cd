"""The verifiers that stop reading a request's rows at its first rejection
(spec_verify_by_request, request by request in one persistent kernel, and
spec_verify_early_exit, one pass per draft position) against the all-rows
verifier (spec_verify_all_rows) and the float64 oracle (GPU).

All three give every row they read the same arithmetic and the same Philox
uniforms, so their outputs must be identical element by element, and so must
the per-row diagnostics of every row both read (rows 0..a_b); rows the
early-exit verifiers never read report NaN with accept = -1, and those two
agree on every diagnostic.
"""
import numpy as np
import pytest
import torch

from gpu_common import (assert_excused_within_bound, check_parity, custom_workload, ensure_built,
                        run_gpu)
from speculative_decoding_verification_51_gb300 import binding
from speculative_decoding_verification_51_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _all3(w, **kw):
    """(all rows, K + 1 passes, request by request)"""
    par = run_gpu(w, all_rows=True, **kw)
    ee = run_gpu(w, early_exit=True, **kw)
    br = run_gpu(w, by_request=True, **kw)
    return par, ee, br


def _assert_same(w, par, ee, br=None):
    if br is not None:  # the two early-exit verifiers agree on everything
        for a, b in zip(ee, br):
            assert np.array_equal(a, b, equal_nan=True)
    ids, nacc, rows, req = par
    ids2, nacc2, rows2, req2 = ee
    assert np.array_equal(nacc, nacc2)
    assert np.array_equal(ids, ids2)
    assert np.array_equal(req, req2, equal_nan=True)
    n = w.num_draft.cpu().numpy()
    for b in range(len(nacc)):
        if nacc[b] < 0:
            assert np.isnan(rows2[b, :, :3]).all() and (rows2[b, :, 3] == -1).all()
            continue
        read = int(nacc[b]) + 1          # rows 0..a_b were read
        assert np.array_equal(rows[b, :read], rows2[b, :read], equal_nan=True), b
        assert np.isnan(rows2[b, read:, :3]).all() and (rows2[b, read:, 3] == -1).all(), b
        assert nacc[b] <= n[b]


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_early_exit_equals_all_rows(cid):
    w = W.make_workload(cid, device="cuda")
    par, ee, br = _all3(w)
    _assert_same(w, par, ee, br)
    # the workload exercises early rejections, full acceptance and bonus rows
    nacc, n = par[1], w.num_draft.cpu().numpy()
    if cid >= 3:
        assert (nacc < n).any() and (nacc == n).any()
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cid,B", [(3, 24), (4, 256), (5, 64)])
def test_early_exit_oracle_parity(cid, B):
    w = W.make_workload(cid, device="cuda").leading(B)
    rep = check_parity(w, f"early_exit_config{cid}_B{B}", early_exit=True)
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    assert_excused_within_bound(rep)


def test_early_exit_more_seeds_and_offset():
    for s in (3, 4, 5):
        w = W.make_workload(4, device="cuda", gen_seed=100 + s)
        w.seed = 77 * s
        par, ee, br = _all3(w, request_offset=1000 * s)
        _assert_same(w, par, ee, br)


def test_early_exit_k0_greedy_and_bad_requests():
    # K = 0: one pass, every request takes its bonus row
    w = W.make_workload(3, device="cuda", B=16, K=0, V=4096)
    par, ee, br = _all3(w)
    _assert_same(w, par, ee, br)
    # all greedy, a bad draft id after the first rejection, a bad num_draft and
    # a bad temperature: flagged exactly as the all-rows pass flags them
    w = W.make_workload(5, device="cuda", B=32, V=8192)
    w.temperature[:16] = 0.0
    ids = w.draft_ids.clone()
    n = w.num_draft.clone()
    n[3] = 8
    ids[3, 7] = 8192           # out of range, at the last draft position
    n[5] = 9                   # above K
    w.temperature[6] = float("nan")
    w.draft_ids, w.num_draft = ids, n
    st1 = torch.zeros(1, dtype=torch.int32, device="cuda")
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    st3 = torch.zeros(1, dtype=torch.int32, device="cuda")
    par = run_gpu(w, all_rows=True, dev_status=st1)
    ee = run_gpu(w, early_exit=True, dev_status=st2)
    br = run_gpu(w, dev_status=st3, by_request=True)
    _assert_same(w, par, ee, br)
    assert par[1][3] == -1 and par[1][5] == -1 and par[1][6] == -1
    assert int(st1.item()) == int(st2.item()) == int(st3.item())
    s = int(st2.item())
    assert s & binding.BADBIT["draft_id"] and s & binding.BADBIT["num_draft"]
    assert s & binding.BADBIT["temperature"]


def test_early_exit_skips_rows_after_the_first_rejection():
    """A sampling row after a certain rejection is never read: made all -inf,
    it turns the all-rows verdict into 'bad request' (the row is checked) but
    leaves the early-exit verdict equal to that on any finite row."""
    ensure_built()
    w = W.make_workload(3, device="cuda", B=8, K=4, V=2048)
    w.temperature[:] = 1.0
    w.num_draft[:] = 4
    lg = w.target_logits
    x0 = w.draft_ids[:, 0].long()
    # draft 0 has p = 0 under the target: rejected for certain
    lg[torch.arange(8, device="cuda"), 0, x0] = float("-inf")
    ref = run_gpu(w, early_exit=True)
    lg[2, 3, :] = float("-inf")          # request 2, row 3 (never read)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    par = run_gpu(w, dev_status=st, all_rows=True)
    ee = run_gpu(w, early_exit=True)
    br = run_gpu(w, by_request=True)
    for a, b in zip(ee, br):
        assert np.array_equal(a, b, equal_nan=True)
    assert (ref[1] == 0).all()
    assert par[1][2] == -1 and int(st.item()) & binding.BADBIT["empty_row"]
    assert np.array_equal(ee[0], ref[0]) and np.array_equal(ee[1], ref[1])
    keep = np.arange(8) != 2
    assert np.array_equal(par[0][keep], ee[0][keep])


def test_early_exit_graph_replay_with_device_seed():
    """The K + 1 passes and the draws have a fixed launch sequence: captured
    once, replayed with a new seed in device memory, they give the direct
    call's result for that seed."""
    ensure_built()
    w = W.make_workload(4, device="cuda", B=64)
    B, K, V = w.B, w.K, w.V
    ws = binding.new_workspace(B, K, V, w.target_logits.device)
    out_ids = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    out_nacc = torch.empty((B,), dtype=torch.int32, device="cuda")
    seed_buf = torch.zeros(1, dtype=torch.int64, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                            w.temperature, 0, out_ids=out_ids, out_num_accepted=out_nacc,
                            workspace=ws, seed_dev=seed_buf, early_exit=True)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                            w.temperature, 0, out_ids=out_ids, out_num_accepted=out_nacc,
                            workspace=ws, seed_dev=seed_buf, early_exit=True)
    for seed in (5, 123456789, 2**40 + 3):
        seed_buf.fill_(seed)
        g.replay()
        torch.cuda.synchronize()
        ids, nacc = binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids,
                                        w.num_draft, w.temperature, seed)
        torch.cuda.synchronize()
        assert torch.equal(ids, out_ids) and torch.equal(nacc, out_nacc)


def test_early_exit_31_drafts():
    """K = 31, the largest draft count: 32 passes, drafts mostly the row
    argmax so that long accepted prefixes reach the late passes."""
    rng = np.random.default_rng(31)
    B, K, V = 24, 31, 3000
    l = rng.normal(0, 1.5, (B, K + 1, V))
    q = rng.dirichlet(np.ones(V), (B, K))
    ids = l[:, :K].argmax(-1)
    ids[::5, 20] = rng.integers(0, V, (B + 4) // 5)  # some late rejections
    q[np.arange(B)[:, None], np.arange(K)[None], ids] = 1e-4
    n = np.where(np.arange(B) % 3 == 0, K, rng.integers(0, K + 1, B))
    T = np.where(np.arange(B) % 4 == 0, 0.0, 0.2)
    w = custom_workload(l, q, ids, n, T, bf16=True, seed=31)
    par, ee, br = _all3(w)
    _assert_same(w, par, ee, br)
    assert par[1].max() >= 20  # some request got past pass 20
    rep = check_parity(w, "early_exit_K31", early_exit=True)
    assert not rep.failures, rep.failures[:5]
