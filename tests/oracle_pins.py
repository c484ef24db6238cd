"""Pins of the float64 oracle: facts fixed by the source pages and by the
mathematics, checked against the oracle without trusting it.

Each ``pin_*`` takes a loaded oracle library and raises AssertionError when
the oracle disagrees.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on copies of the oracle with planted
mistakes and requires each mistake to trip at least one pin.

Sources (web pages, by title and section):
  [P1] 深入推测解码：从概念到实现 -- 保证原始分布 (the acceptance rule, the
       q=0.4/p=0.2 example, the residual), 伪代码 (break at first mismatch).
  [P2] RTP-LLM Speculative Engine 深度解析 -- 拒绝采样算法.
  [P3] 投机采样 -- 第三步..第五步, output-length cases, 调整分布 (the
       output equals sampling from p), Blockwise Parallel Decoding example,
       验收标准 / 精确匹配, and Typical Acceptance (a hard threshold on the
       target's probability of each draft, longest kept prefix).
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- helpers

def _run(lib, logits, q, ids, n, T, seed=0, **kw):
    logits = np.asarray(logits, dtype=np.float32)
    B, K1, V = logits.shape
    q = None if q is None else np.asarray(q, dtype=np.float32).reshape(B, K1 - 1, V)
    return oracle.spec_verify(logits, q, np.asarray(ids, np.int32).reshape(B, K1 - 1),
                              np.asarray(n, np.int32).reshape(B),
                              np.asarray(T, np.float32).reshape(B), seed, lib=lib, **kw)


def _tile(x, B):
    x = np.asarray(x)
    return np.ascontiguousarray(np.broadcast_to(x, (B,) + x.shape))


def _softmax64(l, T):
    """Independent float64 softmax (Python loop, libm exp, sequential sum)."""
    s = [v / T for v in l]
    M = max(s)
    e = [math.exp(v - M) for v in s]
    Z = 0.0
    for v in e:
        Z += v
    return [v / Z for v in e]


def _inv_cdf(w, u):
    S = 0.0
    for v in w:
        S += v
    t = u * S
    C = 0.0
    for x, v in enumerate(w):
        C += v
        if C >= t:
            return x
    return len(w) - 1


def straight_line(logit_rows, q_rows, draft, n, T, u_acc, u_emit):
    """A second, independent restatement of the method for tiny inputs.

    logit_rows: n+1 rows of floats, q_rows: n rows, draft: n ids,
    u_acc/u_emit: per-row uniforms.  Returns (accepted, tokens).
    """
    out = []
    for j in range(n):
        row = logit_rows[j]
        if T == 0.0:
            top = int(np.argmax(row))  # numpy argmax returns the first maximum
            if top == draft[j]:
                out.append(draft[j])
                continue
            return j, out + [top]
        p = _softmax64(row, T)
        px, qx = p[draft[j]], float(q_rows[j][draft[j]])
        if px > 0.0 and (qx == 0.0 or u_acc[j] <= px / qx):
            out.append(draft[j])
            continue
        r = [max(0.0, a - float(b)) for a, b in zip(p, q_rows[j])]
        if sum(r) > 0.0:
            return j, out + [_inv_cdf(r, u_emit[j])]
        return j, out + [_inv_cdf(p, u_emit[j])]
    row = logit_rows[n]
    if T == 0.0:
        return n, out + [int(np.argmax(row))]
    return n, out + [_inv_cdf(_softmax64(row, T), u_emit[n])]


# ---------------------------------------------------------------- pins

def pin_philox_kat(lib):
    """Philox4x32-10 equals the published known-answer vectors."""
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "philox4x32_10_kat.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        out = oracle.philox_blocks(np.array([v[0:4]], np.uint32), (v[4], v[5]), lib=lib)
        assert [int(x) for x in out[0]] == v[6:10], (r, [hex(int(x)) for x in out[0]])


def pin_uniform_map(lib):
    """u = ((x >> 8) + 1) 2^-24: the ends of (0, 1] and exact steps."""
    assert lib.oracle_uniform_from_bits(0) == 2.0 ** -24
    assert lib.oracle_uniform_from_bits(0xFFFFFFFF) == 1.0
    assert lib.oracle_uniform_from_bits(0x100) == 2.0 * 2.0 ** -24
    assert lib.oracle_uniform_from_bits(0xFF) == 2.0 ** -24


def pin_uniform_lanes(lib):
    """Row j of request b: lane 0 drives acceptance, lane 1 the emission."""
    V, K, B, seed = 4, 2, 3, 0x1234_5678_9ABC
    l = np.zeros((B, K + 1, V), np.float32)
    q = np.full((B, K, V), 0.25, np.float32)
    ids = np.zeros((B, K), np.int32)
    r = _run(lib, l, q, ids, [K] * B, [1.0] * B, seed=seed)
    for b in range(B):
        for j in range(K):
            blk = oracle.philox_blocks(np.array([[b, j, 0, 0]], np.uint32),
                                       (seed & 0xFFFFFFFF, seed >> 32), lib=lib)[0]
            assert r["row_diag"][b, j, oracle.R_U] == ((int(blk[0]) >> 8) + 1) * 2.0 ** -24
        blk = oracle.philox_blocks(np.array([[b, K, 0, 0]], np.uint32),
                                   (seed & 0xFFFFFFFF, seed >> 32), lib=lib)[0]
        assert r["req_diag"][b, oracle.Q_UEMIT] == ((int(blk[1]) >> 8) + 1) * 2.0 ** -24


def pin_worked_ratio(lib):
    """[P1] 保证原始分布 3b: q=0.4, p=0.2 -> accepted with probability 1/2."""
    g = json.load(open(os.path.join(GOLDEN, "worked_ratio.json")))
    p = np.array([g["p_draft_token"], 0.5, 0.3])
    q = np.array([g["q_draft_token"], 0.3, 0.3], np.float32)
    l = np.log(p).astype(np.float32)
    # exact: accept iff u <= p/q, over a grid of uniforms (lane 0)
    grid = (np.arange(4096) + 0.5) / 4096
    B = grid.size
    uni = np.zeros((B, 2, 2))
    uni[:, 0, 0] = grid
    uni[:, :, 1] = 0.5
    r = _run(lib, _tile(l[None].repeat(2, 0), B), _tile(q[None], B), np.zeros((B, 1)),
             [1] * B, [1.0] * B, uniforms=uni)
    ratio = r["row_diag"][:, 0, oracle.R_PX] / r["row_diag"][:, 0, oracle.R_QX]
    assert np.allclose(ratio, g["accept_probability"], rtol=1e-6)
    acc = r["out_num_accepted"] == 1
    far = np.abs(grid - g["accept_probability"]) > 1e-6
    assert np.array_equal(acc[far], (grid <= g["accept_probability"])[far])
    # Monte Carlo with the Philox stream: 10^6 requests
    B = 1_000_000
    r = _run(lib, _tile(l[None].repeat(2, 0), B), _tile(q[None], B), np.zeros((B, 1)),
             [1] * B, [1.0] * B, seed=7)
    f = float(np.mean(r["out_num_accepted"] == 1))
    sigma = math.sqrt(0.25 / B)
    assert abs(f - g["accept_probability"]) < 5 * sigma, f


def pin_equal_probs_always_accept(lib):
    """[P1] 3a / [P3] 第三步: p >= q accepts; constant logits give p = q = 2^-10
    exactly, so every draft is accepted and the bonus is drawn from p."""
    V, K, B = 1024, 4, 2000
    l = np.zeros((B, K + 1, V), np.float32)
    q = np.full((B, K, V), 2.0 ** -10, np.float32)
    rng = np.random.default_rng(3)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    r = _run(lib, l, q, ids, [K] * B, [1.0] * B, seed=11)
    assert np.all(r["out_num_accepted"] == K)
    assert np.array_equal(r["out_ids"][:, :K], ids)
    assert np.all(r["req_diag"][:, oracle.Q_MODE] == oracle.MODE_BONUS)
    u2 = r["req_diag"][:, oracle.Q_UEMIT]
    # inverse CDF of the uniform distribution: C(x) = (x+1)/1024 exactly
    assert np.array_equal(r["out_ids"][:, K], np.ceil(u2 * V).astype(np.int32) - 1)
    # p > q (p = 1/2 on the draft token, q = 1/4) also always accepts
    l2 = np.full((B, 2, 4), math.log(1 / 6), np.float32)
    l2[:, 0, 0] = math.log(1 / 2)
    q2 = np.full((B, 1, 4), 0.25, np.float32)
    r = _run(lib, l2, q2, np.zeros((B, 1)), [1] * B, [1.0] * B, seed=12)
    assert np.all(r["out_num_accepted"] == 1)


def pin_zero_target_prob_never_accepted(lib):
    """p(x) = 0 accepts with probability p/q = 0, for every u in (0, 1]; the
    residual max(0, p - q) is 0 at x, so x is never re-emitted."""
    V, B = 6, 4097
    l = np.zeros((B, 2, V), np.float32)
    l[:, 0, 2] = -np.inf
    q = np.full((B, 1, V), 1.0 / V, np.float32)
    uni = np.zeros((B, 2, 2))
    uni[:, 0, 0] = np.r_[2.0 ** -24, (np.arange(B - 2) + 1) / (B - 1), 1.0]
    uni[:, 0, 1] = np.r_[1.0, (np.arange(B - 2) + 1) / (B - 1), 2.0 ** -24]
    r = _run(lib, l, q, np.full((B, 1), 2), [1] * B, [1.0] * B, uniforms=uni)
    assert np.all(r["out_num_accepted"] == 0)
    assert not np.any(r["out_ids"][:, 0] == 2)
    # q(x) = 0 as well: still rejected (p = 0 decides); q(x) = 0 < p(x): accepted
    q0 = q.copy()
    q0[:, 0, 2] = 0.0
    r = _run(lib, l, q0, np.full((B, 1), 2), [1] * B, [1.0] * B, uniforms=uni)
    assert np.all(r["out_num_accepted"] == 0)
    l1 = np.zeros((B, 2, V), np.float32)
    r = _run(lib, l1, q0, np.full((B, 1), 2), [1] * B, [1.0] * B, uniforms=uni)
    assert np.all(r["out_num_accepted"] == 1)


def pin_residual_support(lib):
    """[P3] 调整分布: a rejected x has q(x) > p(x), so max(0, p - q) puts no
    mass on it; every resampled token has p > q."""
    rng = np.random.default_rng(5)
    B, K, V = 20000, 1, 7
    l = rng.normal(0, 1.5, (B, K + 1, V)).astype(np.float32)
    dl = l[:, :K] + rng.normal(0, 1.0, (B, K, V))
    q = np.exp(dl - dl.max(-1, keepdims=True))
    q = (q / q.sum(-1, keepdims=True)).astype(np.float32)
    cdf = np.cumsum(q[:, 0].astype(np.float64), -1)
    cdf /= cdf[:, -1:]
    ids = np.minimum((cdf < rng.random((B, 1))).sum(-1), V - 1).astype(np.int32)[:, None]
    r = _run(lib, l, q, ids, [K] * B, [1.0] * B, seed=9)
    rej = r["out_num_accepted"] == 0
    assert rej.sum() > 1000
    for b in np.flatnonzero(rej)[:3000]:
        p = _softmax64(l[b, 0].astype(np.float64).tolist(), 1.0)
        x = r["out_ids"][b, 0]
        assert p[x] > q[b, 0, x], (b, x, p[x], q[b, 0, x])
        assert p[ids[b, 0]] < q[b, 0, ids[b, 0]]


def pin_output_shape(lib):
    """[P3] output-length cases: 1 <= length <= n+1; the accepted prefix is the
    drafts; -1 after the emitted token; the bonus only when all accepted."""
    rng = np.random.default_rng(6)
    B, K, V = 4000, 5, 9
    l = rng.normal(0, 1.0, (B, K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), (B, K)).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    n = rng.integers(0, K + 1, B).astype(np.int32)
    T = np.where(rng.random(B) < 0.3, 0.0, rng.uniform(0.3, 2.0, B)).astype(np.float32)
    r = _run(lib, l, q, ids, n, T, seed=4)
    assert r["n_bad"] == 0
    a = r["out_num_accepted"]
    assert np.all((a >= 0) & (a <= n))
    for b in range(B):
        assert np.array_equal(r["out_ids"][b, :a[b]], ids[b, :a[b]])
        assert 0 <= r["out_ids"][b, a[b]] < V
        assert np.all(r["out_ids"][b, a[b] + 1:] == -1)
        mode = r["req_diag"][b, oracle.Q_MODE]
        if T[b] > 0:
            assert (mode == oracle.MODE_BONUS) == (a[b] == n[b]), (b, mode, a[b], n[b])
        assert r["req_diag"][b, oracle.Q_EROW] == a[b]


def pin_greedy_example(lib):
    """[P3] Blockwise Parallel Decoding example, exact-match acceptance."""
    g = json.load(open(os.path.join(GOLDEN, "greedy_bpd_example.json")))
    vocab = {w: i for i, w in enumerate(g["vocab"])}
    V, K = len(vocab), len(g["draft"])
    l = np.full((1, K + 1, V), -3.0, np.float32)
    for j, w in enumerate(g["target_top1"]):
        l[0, j, vocab[w]] = 2.0
    ids = np.array([[vocab[w] for w in g["draft"]]], np.int32)
    r = _run(lib, l, None, ids, [K], [0.0])
    a = int(r["out_num_accepted"][0])
    assert a == g["expected_num_accepted"]
    assert [g["vocab"][i] for i in r["out_ids"][0, :a + 1]] == g["expected_out"]
    assert np.all(r["out_ids"][0, a + 1:] == -1)


def pin_greedy_ties(lib):
    """Greedy target token = the lowest index among equal maxima (numpy.argmax
    returns the first maximum)."""
    rng = np.random.default_rng(8)
    B, K, V = 3000, 3, 16
    l = rng.integers(-2, 3, (B, K + 1, V)).astype(np.float32)  # many ties
    top = l.argmax(-1)
    ids = np.where(rng.random((B, K)) < 0.6, top[:, :K], rng.integers(0, V, (B, K)))
    r = _run(lib, l, None, ids, [K] * B, [0.0] * B)
    for b in range(B):
        a = r["out_num_accepted"][b]
        assert np.array_equal(ids[b, :a], top[b, :a])
        assert a == K or ids[b, a] != top[b, a]
        assert r["out_ids"][b, a] == top[b, a]


def pin_softmax_vs_scipy(lib):
    """p_j(x_j) = softmax(l_j / T)[x_j] (scipy, float64) to 1e-13 relative."""
    from scipy.special import softmax
    rng = np.random.default_rng(10)
    B, K, V = 64, 3, 1000
    l = rng.normal(0, 3.0, (B, K + 1, V)).astype(np.float32)
    q = np.full((B, K, V), 1e-30, np.float32)  # tiny q: every draft accepted
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    T = rng.uniform(0.2, 3.0, B).astype(np.float32)
    r = _run(lib, l, q, ids, [K] * B, T)
    assert np.all(r["out_num_accepted"] == K)
    for b in range(B):
        for j in range(K):
            ref = softmax(l[b, j].astype(np.float64) / np.float64(T[b]))[ids[b, j]]
            assert abs(r["row_diag"][b, j, oracle.R_PX] - ref) <= 1e-13 * ref


def pin_temperature(lib):
    """softmax(l / T) at T equals softmax(l') at T = 1 for l' = l / T, when
    l / T is exact in float32 (T a power of two)."""
    rng = np.random.default_rng(12)
    B, K, V = 200, 2, 50
    l = rng.normal(0, 2.0, (B, K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), (B, K)).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    r1 = _run(lib, l, q, ids, [K] * B, [4.0] * B, seed=2)
    r2 = _run(lib, l / np.float32(4.0), q, ids, [K] * B, [1.0] * B, seed=2)
    assert np.array_equal(r1["out_ids"], r2["out_ids"])
    assert np.allclose(r1["row_diag"][..., oracle.R_PX], r2["row_diag"][..., oracle.R_PX],
                       rtol=1e-15, atol=0, equal_nan=True)
    # a vanishing temperature makes p one-hot at the maximum
    r3 = _run(lib, l, q, ids, [K] * B, [1e-30] * B, seed=2)
    top = l.argmax(-1)
    for b in range(B):
        a = r3["out_num_accepted"][b]
        assert np.array_equal(ids[b, :a], top[b, :a])
        assert r3["out_ids"][b, a] == top[b, a]


def pin_inverse_cdf_ends(lib):
    """Inverse CDF = smallest x with C(x) >= u' S: u' = 1 lands on the last
    token of positive mass, a tiny u' on the first (zero-mass tokens skipped)."""
    p = np.array([0.1, 0.6, 0.3, 0.0])
    q = np.array([[0.7, 0.1, 0.1, 0.1]], np.float32)  # residual [0, .5, .2, 0]
    l = np.log(np.maximum(p, 1e-300)).astype(np.float32)
    l[3] = -np.inf
    L = np.stack([l, l])[None]
    for u2, want in ((1.0, 2), (2.0 ** -24, 1), (0.5 / 0.7 - 1e-5, 1), (0.5 / 0.7 + 1e-5, 2)):
        uni = np.array([[[1.0, u2], [0.5, 0.5]]])
        r = _run(lib, L, q[None], [[0]], [1], [1.0], uniforms=uni)
        assert r["out_num_accepted"][0] == 0
        assert r["out_ids"][0, 0] == want, (u2, r["out_ids"][0])


def pin_zero_residual_fallback(lib):
    """An unnormalised q >= p everywhere leaves max(0, p - q) with no mass; the
    token is then drawn from p itself."""
    p = np.array([0.1, 0.2, 0.3, 0.4])
    l = np.log(p).astype(np.float32)
    q = np.full((1, 1, 4), 0.5, np.float32)
    for u2, want in ((0.05, 0), (0.25, 1), (0.55, 2), (0.95, 3)):
        uni = np.array([[[1.0, u2], [0.5, 0.5]]])
        r = _run(lib, np.stack([l, l])[None], q, [[1]], [1], [1.0], uniforms=uni)
        assert r["out_num_accepted"][0] == 0
        assert r["req_diag"][0, oracle.Q_MODE] == oracle.MODE_FALLBACK
        assert r["out_ids"][0, 0] == want


def pin_bad_inputs(lib):
    """Malformed requests give -1 outputs and are counted; good ones are not
    disturbed."""
    V, K = 8, 2
    l = np.zeros((7, K + 1, V), np.float32)
    l[6, 1, :] = -np.inf             # a sampling row with no finite logit
    q = np.full((7, K, V), 1 / V, np.float32)
    ids = np.ones((7, K), np.int32)
    ids[3, 1] = V                    # draft id out of range
    n = np.array([K, -1, K + 1, K, K, K, K], np.int32)
    T = np.array([1.0, 1.0, 1.0, 1.0, np.nan, -0.5, 1.0], np.float32)
    r = _run(lib, l, q, ids, n, T)
    assert r["n_bad"] == 6
    assert r["out_num_accepted"][0] == K
    for b in range(1, 7):
        assert r["out_num_accepted"][b] == -1 and np.all(r["out_ids"][b] == -1)
    T2 = T.copy()
    T2[4] = np.inf
    r = _run(lib, l[4:5], q[4:5], ids[4:5], n[4:5], T2[4:5])
    assert r["n_bad"] == 1
    # the draft id beyond num_draft is never looked at
    ids2 = ids[:1].copy()
    ids2[0, 1] = -5
    r = _run(lib, l[:1], q[:1], ids2, [1], [1.0])
    assert r["n_bad"] == 0


def pin_unused_rows_ignored(lib):
    """Rows j > n_b and draft ids j >= n_b are never read: poisoning them
    changes nothing."""
    rng = np.random.default_rng(13)
    B, K, V = 500, 4, 12
    l = rng.normal(0, 1.0, (B, K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), (B, K)).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    n = rng.integers(0, K + 1, B).astype(np.int32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    r1 = _run(lib, l, q, ids, n, T, seed=1)
    l2, q2, ids2 = l.copy(), q.copy(), ids.copy()
    for b in range(B):
        l2[b, n[b] + 1:] = np.nan
        q2[b, n[b]:] = np.nan
        ids2[b, n[b]:] = -1
    r2 = _run(lib, l2, q2, ids2, n, T, seed=1)
    assert np.array_equal(r1["out_ids"], r2["out_ids"])
    assert np.array_equal(r1["out_num_accepted"], r2["out_num_accepted"])


def pin_request_index(lib):
    """A request's result depends only on its own data and its global index."""
    rng = np.random.default_rng(14)
    B, K, V = 64, 3, 10
    l = rng.normal(0, 1.0, (B, K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), (B, K)).astype(np.float32)
    ids = rng.integers(0, V, (B, K)).astype(np.int32)
    T = np.ones(B, np.float32)
    full = _run(lib, l, q, ids, [K] * B, T, seed=77)
    sel = np.array([5, 17, 40, 63])
    part = _run(lib, l[sel], q[sel], ids[sel], [K] * 4, T[sel], seed=77, req_index=sel)
    assert np.array_equal(full["out_ids"][sel], part["out_ids"])


def pin_brute_force(lib):
    """Exhaustive agreement with ``straight_line`` on tiny vocabularies: every
    draft tuple in V^K, a grid of uniforms, greedy and sampling."""
    rng = np.random.default_rng(15)
    for V, K in ((2, 3), (3, 2), (5, 2), (8, 1), (4, 3)):
        tuples = np.array(list(itertools.product(range(V), repeat=K)), np.int32)
        l = rng.normal(0, 1.2, (K + 1, V)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.7, K).astype(np.float32)
        grid = (np.arange(16) + 0.5) / 16
        for T in (0.0, 0.7, 1.0):
            reps = tuples.shape[0] * grid.size
            B = reps
            ids = np.repeat(tuples, grid.size, 0)
            uni = np.empty((B, K + 1, 2))
            gi = np.tile(np.arange(grid.size), tuples.shape[0])
            for j in range(K + 1):
                uni[:, j, 0] = grid[(gi + 3 * j) % grid.size]
                uni[:, j, 1] = grid[(gi * 5 + j) % grid.size]
            r = _run(lib, _tile(l, B), _tile(q, B), ids, [K] * B, [T] * B, uniforms=uni)
            lr = l.astype(np.float64).tolist()
            T32 = float(np.float32(T))
            for b in range(B):
                a, toks = straight_line(lr, q, ids[b].tolist(), K, T32,
                                        uni[b, :, 0].tolist(), uni[b, :, 1].tolist())
                assert r["out_num_accepted"][b] == a, (V, K, T, b)
                assert r["out_ids"][b, :a + 1].tolist() == toks, (V, K, T, b)


def _law(p, q):
    """Closed form of one slot: P(accept) = sum_x min(p, q); the emitted token's
    law q min(1, p/q) + (1 - alpha) norm(max(0, p - q)), which equals p."""
    alpha = np.minimum(p, q).sum()
    r = np.maximum(p - q, 0)
    emit = q * np.minimum(1.0, np.divide(p, q, out=np.ones_like(p), where=q > 0)) \
        + (1 - alpha) * r / r.sum()
    return alpha, emit


def pin_lossless_closed_form(lib):
    """[P3] 调整分布 / [P1] 保证原始分布: the emitted token's law is p.  The
    two-path sum is checked algebraically, then against 10^6 oracle trials
    (chi-square per slot, acceptance frequencies, and P(a = k))."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(16)
    for V, seed in ((5, 21), (8, 22)):
        K = 3
        l = rng.normal(0, 1.0, (K + 1, V)).astype(np.float32)
        q = rng.dirichlet(np.ones(V), K).astype(np.float32)
        p = np.array([_softmax64(l[j].astype(np.float64).tolist(), 1.0) for j in range(K + 1)])
        qd = q.astype(np.float64)
        alphas = []
        for j in range(K):
            alpha, emit = _law(p[j], qd[j] / qd[j].sum())
            assert np.allclose(emit, p[j], atol=1e-12)
            alphas.append(np.minimum(p[j], qd[j]).sum())
        B = 1_000_000
        draw = np.empty((B, K), np.int32)
        for j in range(K):
            cdf = np.cumsum(qd[j] / qd[j].sum())
            draw[:, j] = np.minimum(np.searchsorted(cdf, rng.random(B), side="right"), V - 1)
        r = _run(lib, _tile(l, B), _tile(q, B), draw, [K] * B, [1.0] * B, seed=seed)
        a = r["out_num_accepted"]
        for j in range(K + 1):
            reach = a >= j
            tok = r["out_ids"][reach, j]
            obs = np.bincount(tok, minlength=V)
            exp_ = p[j] * reach.sum()
            assert chisquare(obs, exp_).pvalue > 1e-3, (V, j, obs, exp_)
        for k in range(K + 1):
            pk = np.prod(alphas[:k]) * (1 - alphas[k] if k < K else 1.0)
            f = np.mean(a == k)
            assert abs(f - pk) < 5 * math.sqrt(pk * (1 - pk) / B) + 1e-9, (V, k, f, pk)


# ------------------------------------------------- typical acceptance

def straight_line_typical(logit_rows, draft, n, T, theta, u_emit):
    """Independent restatement of the typical-acceptance rule ([P3] 验收标准,
    Typical Acceptance): keep the longest prefix of drafts whose target
    probability reaches the hard threshold; the next token is the target's
    own draw (sampling) or argmax (greedy) at the row after the prefix."""
    out = []
    for j in range(n):
        row = logit_rows[j]
        if T == 0.0:
            top = int(np.argmax(row))
            if top == draft[j]:
                out.append(draft[j])
                continue
            return j, out + [top]
        p = _softmax64(row, T)
        if p[draft[j]] > 0.0 and p[draft[j]] >= theta:
            out.append(draft[j])
            continue
        return j, out + [_inv_cdf(p, u_emit[j])]
    row = logit_rows[n]
    if T == 0.0:
        return n, out + [int(np.argmax(row))]
    return n, out + [_inv_cdf(_softmax64(row, T), u_emit[n])]


def pin_typical_brute_force(lib):
    """Typical acceptance agrees with ``straight_line_typical`` on every draft
    tuple of tiny vocabularies, over thresholds and a grid of uniforms; it
    reads no draft distribution (q is not passed)."""
    rng = np.random.default_rng(17)
    for V, K in ((3, 3), (5, 2), (8, 1)):
        tuples = np.array(list(itertools.product(range(V), repeat=K)), np.int32)
        l = rng.normal(0, 1.5, (K + 1, V)).astype(np.float32)
        l[0, V - 1] = -np.inf  # one token the target never produces
        grid = (np.arange(8) + 0.5) / 8
        for T in (0.0, 0.8):
            for theta in (-1.0, 0.05, 0.2, 0.45, 2.0):
                B = tuples.shape[0] * grid.size
                ids = np.repeat(tuples, grid.size, 0)
                uni = np.empty((B, K + 1, 2))
                gi = np.tile(np.arange(grid.size), tuples.shape[0])
                for j in range(K + 1):
                    uni[:, j, 0] = grid[(gi + j) % grid.size]
                    uni[:, j, 1] = grid[(gi * 3 + j) % grid.size]
                r = _run(lib, _tile(l, B), None, ids, [K] * B, [T] * B, uniforms=uni,
                         typical_threshold=theta)
                assert r["n_bad"] == 0
                lr = l.astype(np.float64).tolist()
                T32 = float(np.float32(T))
                for b in range(B):
                    a, toks = straight_line_typical(lr, ids[b].tolist(), K, T32, theta,
                                                    uni[b, :, 1].tolist())
                    assert r["out_num_accepted"][b] == a, (V, K, T, theta, b)
                    assert r["out_ids"][b, :a + 1].tolist() == toks, (V, K, T, theta, b)


def pin_typical_threshold_boundary(lib):
    """The threshold is inclusive: constant logits over V = 2^k give
    p = 2^-k exactly, so theta = 2^-k keeps every draft and the next float
    above it keeps none; then the emitted token is the target's own draw at
    row 0.  A draft with p = 0 is never kept, whatever the threshold."""
    V, K, B = 16, 3, 64
    l = np.zeros((B, K + 1, V), np.float32)
    ids = np.tile(np.arange(K, dtype=np.int32), (B, 1))
    r = _run(lib, l, None, ids, [K] * B, [1.0] * B, typical_threshold=1.0 / V)
    assert (r["out_num_accepted"] == K).all()
    r = _run(lib, l, None, ids, [K] * B, [1.0] * B,
             typical_threshold=float(np.nextafter(1.0 / V, 1.0)))
    assert (r["out_num_accepted"] == 0).all()
    assert (r["req_diag"][:, oracle.Q_EROW] == 0).all()
    u = r["req_diag"][:, oracle.Q_UEMIT]
    assert r["out_ids"][:, 0].tolist() == [min(V - 1, math.ceil(x * V) - 1) for x in u]
    l2 = l.copy()
    l2[:, 1, 1] = -np.inf
    r = _run(lib, l2, None, ids, [K] * B, [1.0] * B, typical_threshold=-5.0)
    assert (r["out_num_accepted"] == 1).all()


def pin_typical_closed_form(lib):
    """Per slot, typical acceptance keeps x_j ~ q with probability
    sum over {x : p(x) >= theta} of q(x); the token after the kept prefix
    follows p at its row.  Checked against 4 * 10^5 oracle trials."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(18)
    V, K, B = 6, 3, 400_000
    l = rng.normal(0, 1.0, (K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), K)
    p = np.array([_softmax64(l[j].astype(np.float64).tolist(), 1.0) for j in range(K + 1)])
    theta = float(np.median(p[:K]))
    alphas = [q[j][p[j] >= theta].sum() for j in range(K)]
    draw = np.empty((B, K), np.int32)
    for j in range(K):
        draw[:, j] = np.minimum(np.searchsorted(np.cumsum(q[j]), rng.random(B), side="right"),
                                V - 1)
    r = _run(lib, _tile(l, B), None, draw, [K] * B, [1.0] * B, seed=31,
             typical_threshold=theta)
    a = r["out_num_accepted"]
    for k in range(K + 1):
        pk = np.prod(alphas[:k]) * (1 - alphas[k] if k < K else 1.0)
        f = np.mean(a == k)
        assert abs(f - pk) < 5 * math.sqrt(pk * (1 - pk) / B) + 1e-9, (k, f, pk)
    for j in range(K + 1):
        sel = a == j
        tok = r["out_ids"][sel, j]
        obs = np.bincount(tok, minlength=V)
        assert chisquare(obs, p[j] * sel.sum()).pvalue > 1e-3, (j, obs)


# ------------------------------------------------- token-tree verification

def _run_tree(lib, logits, q, tok, par, n, T, seed=0, **kw):
    logits = np.asarray(logits, dtype=np.float32)
    B, N, V = logits.shape
    q = None if q is None else np.asarray(q, dtype=np.float32).reshape(B, N, V)
    return oracle.tree_verify(logits, q, np.asarray(tok, np.int32).reshape(B, N),
                              np.asarray(par, np.int32).reshape(B, N),
                              np.asarray(n, np.int32).reshape(B),
                              np.asarray(T, np.float32).reshape(B), seed, lib=lib, **kw)


def _children(par, n, v):
    return [c for c in range(v + 1, n) if par[c] == v]


def straight_line_tree(rows, q, tok, par, n, T, ua, ue):
    """Independent restatement of the tree walk ([P3] 验证方案, token tree
    verification; residual chain over siblings) for tiny trees: returns
    (accepted tokens, emitted token, last node)."""
    v, path = 0, []
    while True:
        kids = _children(par, n, v)
        if T == 0.0:
            g = int(np.argmax(rows[v]))
            hit = [c for c in kids if tok[c] == g]
            if not hit:
                return path, g, v
            path.append(tok[hit[0]])
            v = hit[0]
            continue
        r = np.array(_softmax64(list(rows[v]), T))
        emit = r
        nxt = None
        for i, c in enumerate(kids):
            qc = np.asarray(q[c], dtype=np.float64)
            x = tok[c]
            if r[x] > 0 and (qc[x] == 0 or ua[c] <= r[x] / qc[x]):
                nxt = c
                break
            res = np.maximum(r - qc, 0.0)
            if res.sum() > 0:
                emit = res
                if i + 1 < len(kids):
                    r = res / res.sum()
            else:
                emit = r
        if nxt is not None:
            path.append(tok[nxt])
            v = nxt
            continue
        return path, _inv_cdf(list(emit), ue[v]), v


def _random_tree(rng, N, n):
    par = np.full(N, -1, np.int32)
    for c in range(1, n):
        par[c] = rng.integers(0, c)
    return par


def pin_tree_chain_is_chain(lib):
    """A trie whose every node has one child is a chain of drafts: tree
    verification then returns exactly what the chain verifier returns (same
    Philox blocks, same rules), for greedy and sampling rows, bonus, residual
    and zero-residual cases."""
    rng = np.random.default_rng(19)
    B, K, V = 64, 4, 24
    l = rng.normal(0, 1.5, (B, K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V) * 0.5, (B, K)).astype(np.float32)
    q[::7] *= 3.0  # unnormalised q: residuals without mass occur
    ids = np.array([[rng.choice(V, p=q[b, j] / q[b, j].sum()) for j in range(K)] for b in range(B)],
                   np.int32)
    ids[::5] = l[::5, :K].argmax(-1)  # long accepted prefixes
    n = rng.integers(0, K + 1, B).astype(np.int32)
    T = np.where(rng.random(B) < 0.3, 0.0, rng.uniform(0.5, 1.5, B)).astype(np.float32)
    chain = _run(lib, l, q, ids, n, T, seed=77)
    tq = np.zeros((B, K + 1, V), np.float32)
    tq[:, 1:] = q
    tok = np.zeros((B, K + 1), np.int32)
    tok[:, 1:] = ids
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    tree = _run_tree(lib, l, tq, tok, par, n + 1, T, seed=77)
    assert np.array_equal(tree["out_num_accepted"], chain["out_num_accepted"])
    assert np.array_equal(tree["out_ids"], chain["out_ids"])
    assert np.array_equal(tree["out_last_node"], chain["out_num_accepted"])


def pin_tree_brute_force(lib):
    """Agreement with ``straight_line_tree`` on many random tiny tries (with
    repeated sibling tokens), greedy and sampling, over a grid of uniforms."""
    rng = np.random.default_rng(20)
    for V, N in ((3, 6), (5, 7), (8, 5)):
        B = 300
        l = rng.normal(0, 1.2, (B, N, V)).astype(np.float32)
        q = rng.dirichlet(np.ones(V) * 0.8, (B, N)).astype(np.float32)
        tok = rng.integers(0, V, (B, N)).astype(np.int32)
        par = np.stack([_random_tree(rng, N, N) for _ in range(B)])
        n = rng.integers(1, N + 1, B).astype(np.int32)
        T = np.where(rng.random(B) < 0.35, 0.0, rng.uniform(0.6, 1.4, B)).astype(np.float32)
        uni = rng.random((B, N, 2)) * 0.999 + 0.0005
        r = _run_tree(lib, l, q, tok, par, n, T, uniforms=uni)
        assert r["n_bad"] == 0
        for b in range(B):
            ua = {c: uni[b, c - 1, 0] for c in range(1, N)}
            ue = uni[b, :, 1]
            path, e, v = straight_line_tree(l[b].astype(np.float64), q[b], tok[b].tolist(),
                                            par[b].tolist(), int(n[b]), float(T[b]), ua, ue)
            a = int(r["out_num_accepted"][b])
            assert a == len(path), (V, N, b)
            assert r["out_ids"][b, :a].tolist() == path, (V, N, b)
            assert int(r["out_ids"][b, a]) == e, (V, N, b)
            assert int(r["out_last_node"][b]) == v, (V, N, b)


def pin_tree_first_token_law(lib):
    """Children drawn independently from q and tested along the residual
    chain leave the first token of the output distributed as the target's p
    at the root (chi-square over 4 * 10^5 tries of a root with three
    children), and the first child is kept with probability sum min(p, q)."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(21)
    V, N, B = 6, 4, 400_000
    l = rng.normal(0, 1.0, (N, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V)).astype(np.float32)
    qd = q.astype(np.float64)
    p = np.array(_softmax64(l[0].astype(np.float64).tolist(), 1.0))
    cdf = np.cumsum(qd / qd.sum())
    tok = np.zeros((B, N), np.int32)
    for c in range(1, N):
        tok[:, c] = np.minimum(np.searchsorted(cdf, rng.random(B), side="right"), V - 1)
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    r = _run_tree(lib, _tile(l, B), _tile(np.tile(q, (N, 1)), B), tok, par, np.full(B, N),
                  np.ones(B), seed=41)
    first = r["out_ids"][:, 0]
    obs = np.bincount(first, minlength=V)
    assert chisquare(obs, p * B).pvalue > 1e-3, obs
    kept1 = np.mean((r["out_num_accepted"] == 1) & (r["out_last_node"] == 1))
    alpha = np.minimum(p, qd / qd.sum()).sum()
    assert abs(kept1 - alpha) < 5 * math.sqrt(alpha * (1 - alpha) / B), (kept1, alpha)


def pin_tree_bad_inputs(lib):
    """Malformed tries give -1 outputs and are counted; good requests are not
    affected: a parent at or after its child, a token outside [0, V), a node
    count outside [1, N], a negative temperature, children without q."""
    V, N = 8, 4
    l = np.zeros((6, N, V), np.float32)
    q = np.full((6, N, V), 1.0 / V, np.float32)
    tok = np.ones((6, N), np.int32)
    par = np.tile(np.array([-1, 0, 1, 2], np.int32), (6, 1))
    n = np.full(6, N, np.int32)
    T = np.ones(6, np.float32)
    par[1, 2] = 2          # parent not before the child
    tok[2, 3] = V          # token out of range
    n[3] = 0               # no root
    T[4] = -1.0            # bad temperature
    r = _run_tree(lib, l, q, tok, par, n, T)
    assert r["n_bad"] == 4
    assert (r["out_num_accepted"][1:5] == -1).all() and (r["out_ids"][1:5] == -1).all()
    assert r["out_num_accepted"][0] >= 0 and r["out_num_accepted"][5] >= 0
    r2 = _run_tree(lib, l[:1], None, tok[:1], par[:1], n[:1], T[:1])
    assert r2["n_bad"] == 1  # sampling children without their q


def pin_tree_unused_nodes_ignored(lib):
    """Nodes at or beyond num_nodes are never read: poisoning their logits,
    tokens, parents and q changes nothing."""
    rng = np.random.default_rng(22)
    B, N, V = 40, 6, 10
    l = rng.normal(0, 1, (B, N, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), (B, N)).astype(np.float32)
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    par = np.stack([_random_tree(rng, N, N) for _ in range(B)])
    n = rng.integers(1, N, B).astype(np.int32)
    T = np.where(rng.random(B) < 0.4, 0.0, 1.0).astype(np.float32)
    a = _run_tree(lib, l, q, tok, par, n, T, seed=3)
    l2, q2, tok2, par2 = l.copy(), q.copy(), tok.copy(), par.copy()
    for b in range(B):
        l2[b, n[b]:] = np.nan
        q2[b, n[b]:] = np.nan
        tok2[b, n[b]:] = -7
        par2[b, n[b]:] = 99
    c = _run_tree(lib, l2, q2, tok2, par2, n, T, seed=3)
    assert np.array_equal(a["out_ids"], c["out_ids"])
    assert np.array_equal(a["out_num_accepted"], c["out_num_accepted"])


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
