"""Typical acceptance ("投机采样", 验收标准, Typical Acceptance) on the GPU
against the oracle's typical rule: drafts are kept while the target's
probability of them reaches a hard threshold; the next token is the target's
own draw at the row after the kept prefix (GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (assert_excused_within_bound, check_parity_typical, custom_workload,
                        run_gpu_typical)
from speculative_decoding_verification_51_gb300 import binding
from speculative_decoding_verification_51_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _assert_ok(rep):
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    assert_excused_within_bound(rep)


@pytest.mark.parametrize("cid,theta", [(1, 1e-3), (1, 0.02), (2, 1e-3), (2, 0.05),
                                       (3, 1e-4), (3, 0.01), (4, 1e-3), (4, 0.1), (5, 0.003)])
def test_typical_parity(cid, theta):
    w = W.make_workload(cid, device="cuda")
    rep, (ids, nacc, rows, req), ref = check_parity_typical(w, theta, f"typical{cid}_{theta}")
    _assert_ok(rep)
    T = w.temperature.cpu().numpy()
    samp = (T > 0) & (nacc >= 0)
    # every sampling request draws its next token from p (mode 4) on both sides
    assert (req[samp, 0] == binding.MODE_TYPICAL).all()
    assert (ref["req_diag"][samp, oracle.Q_MODE] == oracle.MODE_TYPICAL).all()
    assert (req[samp, 1] == nacc[samp]).all()
    del w
    torch.cuda.empty_cache()


def test_typical_thresholds_split_the_drafts():
    """On the Zipf workload the chosen thresholds keep some drafts and refuse
    others, so both branches of the rule are exercised above."""
    w = W.make_workload(3, device="cuda")
    frac = []
    for theta in (1e-4, 0.01):
        _, nacc = run_gpu_typical(w, theta, debug=False)
        n = w.num_draft.cpu().numpy()
        frac.append(nacc.sum() / n.sum())
    assert 0.0 < frac[1] < frac[0] < 1.0, frac


@pytest.mark.parametrize("bf16", [False, True])
def test_typical_extremes(bf16):
    """theta = -inf keeps every draft with p > 0; theta = +inf keeps none;
    a draft the target gives probability 0 is never kept."""
    rng = np.random.default_rng(5)
    B, K, V = 48, 4, 4096
    logits = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    logits[::3, 2, :] = np.where(np.arange(V) == ids[::3, 2, None], -np.inf, logits[::3, 2, :])
    num = np.full(B, K, np.int32)
    temp = np.full(B, 0.9, np.float32)
    w = custom_workload(logits, None, ids, num, temp, bf16=bf16, seed=77)
    for theta, want in ((-math.inf, None), (math.inf, 0)):
        rep, (out, nacc, _, _), ref = check_parity_typical(w, theta, f"typical_ext_{theta}")
        _assert_ok(rep)
        if want is None:
            exp = np.where(np.arange(B) % 3 == 0, 2, K)
            assert (nacc == exp).all()
        else:
            assert (nacc == 0).all()


def test_typical_mixed_greedy_and_shard_offset():
    """Greedy requests keep exact-match verification; a shard with a request
    offset draws the uniforms of its global indices."""
    w = W.make_workload(4, device="cuda")
    full, _, _ = check_parity_typical(w, 0.05, "typical4_full")
    _assert_ok(full)
    ids_all, nacc_all = run_gpu_typical(w, 0.05, debug=False)
    sub = w.subset(list(range(100, 180)))
    ids_s, nacc_s = run_gpu_typical(sub, 0.05, debug=False, request_offset=100)
    assert np.array_equal(ids_s, ids_all[100:180])
    assert np.array_equal(nacc_s, nacc_all[100:180])


def test_typical_ignores_draft_probs_and_reports_bad_requests():
    """No draft distribution is needed; bad requests still get -1 and their
    status bits."""
    rng = np.random.default_rng(6)
    B, K, V = 8, 3, 1024
    logits = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    num = np.full(B, K, np.int32)
    temp = np.ones(B, np.float32)
    num[1] = K + 1
    temp[2] = -1.0
    ids[3, 0] = V
    w = custom_workload(logits, None, ids, num, temp, bf16=False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nacc = run_gpu_typical(w, 1e-3, debug=False, dev_status=st)
    assert (nacc[[1, 2, 3]] == -1).all() and (out[[1, 2, 3]] == -1).all()
    assert (nacc[[0, 4, 5, 6, 7]] >= 0).all()
    s = int(st.item())
    assert s & binding.BADBIT["num_draft"] and s & binding.BADBIT["temperature"]
    assert s & binding.BADBIT["draft_id"] and not s & binding.BADBIT["no_probs"]


def test_typical_emission_law():
    """With theta above every probability nothing is kept and the token at
    row 0 is drawn from p_0: chi-square of 2^18 GPU draws against p_0."""
    from scipy.stats import chisquare
    B, K, V = 1 << 18, 1, 64
    rng = np.random.default_rng(9)
    row = rng.normal(0, 1, (K + 1, V)).astype(np.float32)
    logits = np.broadcast_to(row, (B, K + 1, V))
    w = custom_workload(logits, None, np.zeros((B, K), np.int32), np.full(B, K, np.int32),
                        np.ones(B, np.float32), bf16=False, seed=123)
    out, nacc = run_gpu_typical(w, 2.0, debug=False)
    assert (nacc == 0).all()
    p = np.exp(row[0].astype(np.float64) - row[0].max())
    p /= p.sum()
    obs = np.bincount(out[:, 0], minlength=V)
    assert chisquare(obs, p * B).pvalue > 1e-4


def test_typical_tiny_temperatures():
    """Point-mass target rows (temperatures down to 1e-44): a draft is kept
    iff it is one of its row's maxima and their share passes the threshold."""
    rng = np.random.default_rng(17)
    B, K, V = 40, 3, 5000
    logits = rng.normal(0, 3, (B, K + 1, V)).astype(np.float32)
    logits += rng.choice([-60.0, 0.0, 35.0], (B, 1, 1)).astype(np.float32)
    ids = np.where(rng.random((B, K)) < 0.6, logits[:, :K].argmax(-1),
                   rng.integers(0, V, (B, K))).astype(np.int32)
    num = rng.integers(0, K + 1, B).astype(np.int32)
    temps = [1e-3, 1e-8, 1e-10, 1e-20, 1e-30, 1e-38, 1e-44]
    temp = np.array([temps[b % len(temps)] for b in range(B)], np.float32)
    w = custom_workload(logits, None, ids, num, temp, bf16=True, seed=5)
    rep, _, _ = check_parity_typical(w, 0.05, "typical_tiny_T")
    _assert_ok(rep)
