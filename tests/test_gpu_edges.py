"""Edge cases, degenerate inputs, error paths and properties of the CUDA path
(GPU)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_common import (assert_excused_within_bound, check_parity, custom_workload, ensure_built,
                        run_gpu)
from speculative_decoding_verification_51_gb300 import binding
from speculative_decoding_verification_51_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def test_philox_matches_oracle_bit_for_bit():
    ensure_built()
    rng = np.random.default_rng(0)
    n = 1 << 20
    ctrs = rng.integers(0, 2**32, (n, 4), dtype=np.uint64).astype(np.uint32)
    ctrs[:4] = [[0, 0, 0, 0], [0xFFFFFFFF] * 4, [1, 2, 3, 4], [5, 0, 0, 0]]
    for seed in (0, 0xDEADBEEF, 0xA409382299F31D0 | (1 << 63)):
        key = (seed & 0xFFFFFFFF, seed >> 32)
        want = oracle.philox_blocks(ctrs, key)
        got = binding.philox_fill(seed, torch.from_numpy(ctrs.view(np.int32)).cuda())
        assert np.array_equal(got.cpu().numpy().view(np.uint32), want)


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("V", [8, 1024, 2048, 2056, 5000, 8200, 16392])
def test_ragged_vocab_sizes(V, bf16):
    rng = np.random.default_rng(V + bf16)
    B, K = 37, 4
    l = rng.normal(0, 2.0, (B, K + 1, V))
    dl = l[:, :K] + rng.normal(0, 1.0, (B, K, V))
    q = np.exp(dl - dl.max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    ids = np.array([[rng.choice(V, p=q[b, j]) for j in range(K)] for b in range(B)])
    n = rng.integers(0, K + 1, B)
    T = np.where(rng.random(B) < 0.3, 0.0, rng.uniform(0.4, 1.6, B))
    w = custom_workload(l, q, ids, n, T, bf16=bf16, seed=V)
    rep = check_parity(w, f"ragged_V{V}_{'bf16' if bf16 else 'f32'}")
    assert not rep.failures, rep.failures[:5]


@pytest.mark.parametrize("K", [0, 1, 31])
def test_draft_count_extremes(K):
    rng = np.random.default_rng(K)
    B, V = 16, 3000
    l = rng.normal(0, 1.0, (B, K + 1, V))
    q = rng.dirichlet(np.ones(V), (B, K)) if K else np.zeros((B, 0, V))
    ids = rng.integers(0, V, (B, K))
    # make most drafts likely to be accepted so that long prefixes occur
    if K:
        ids[:, :] = l[:, :K].argmax(-1)
        q[np.arange(B)[:, None], np.arange(K)[None], ids] = 1e-6
    n = np.full(B, K)
    T = np.where(np.arange(B) % 2 == 0, 0.0, 1.0)
    w = custom_workload(l, q, ids, n, T, bf16=True, seed=K)
    rep = check_parity(w, f"K{K}")
    assert not rep.failures, rep.failures[:5]


def test_equal_probs_accept_everything_and_bonus_is_exact():
    B, K, V = 64, 4, 1024
    l = np.zeros((B, K + 1, V))
    q = np.full((B, K, V), 2.0 ** -10)
    rng = np.random.default_rng(1)
    ids = rng.integers(0, V, (B, K))
    w = custom_workload(l, q, ids, [K] * B, [1.0] * B, bf16=True, seed=5)
    out, nacc, rows, req = run_gpu(w)
    assert np.all(nacc == K)
    assert np.array_equal(out[:, :K], ids)
    for b in range(B):
        u2 = oracle.row_uniforms(5, b, K)[1]
        assert out[b, K] == math.ceil(u2 * V) - 1
        assert req[b, 0] == binding.MODE_BONUS


def test_zero_target_probability_is_never_accepted():
    B, V = 512, 64
    l = np.zeros((B, 2, V))
    l[:, 0, 7] = -np.inf
    q = np.full((B, 1, V), 1.0 / V)
    w = custom_workload(l, q, np.full((B, 1), 7), [1] * B, [1.0] * B, bf16=False, seed=3)
    out, nacc, _, _ = run_gpu(w)
    assert np.all(nacc == 0)
    assert not np.any(out[:, 0] == 7)


@pytest.mark.parametrize("path", ["auto", "all_rows", "by_request"])
def test_bad_inputs_flagged_and_isolated(path):
    kw = {} if path == "auto" else {path: True}
    rng = np.random.default_rng(2)
    B, K, V = 8, 2, 256
    l = rng.normal(0, 1, (B, K + 1, V))
    l[6, 0, :] = -np.inf               # sampling row without a finite logit (read by both)
    q = rng.dirichlet(np.ones(V), (B, K))
    ids = rng.integers(0, V, (B, K))
    ids[3, 1] = V                      # draft id out of range
    n = np.array([K, -1, K + 1, K, K, K, K, 1])
    T = np.array([1.0, 1.0, 1.0, 1.0, np.nan, -0.5, 1.0, 0.0])
    w = custom_workload(l, q, ids, n, T, bf16=True, seed=1)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, nacc, _, _ = run_gpu(w, dev_status=st, **kw)
    bits = int(st.item())
    assert bits == (binding.BADBIT["num_draft"] | binding.BADBIT["temperature"] |
                    binding.BADBIT["draft_id"] | binding.BADBIT["empty_row"])
    for b in (1, 2, 3, 4, 5, 6):
        assert nacc[b] == -1 and np.all(out[b] == -1)
    ref = oracle.spec_verify(**W.to_numpy(w))
    for b in (0, 7):
        assert nacc[b] == ref["out_num_accepted"][b]
        assert np.array_equal(out[b], ref["out_ids"][b])
    # missing draft probabilities only hurt sampling requests
    w2 = custom_workload(l[[0, 7]], None, ids[[0, 7]], n[[0, 7]], T[[0, 7]], bf16=True)
    ensure_built()
    o2, n2 = binding.spec_verify(w2.target_logits, None, w2.draft_ids, w2.num_draft,
                                 w2.temperature, 0, dev_status=st, **kw)
    assert int(st.item()) == binding.BADBIT["no_probs"]
    assert n2[0].item() == -1 and n2[1].item() == ref["out_num_accepted"][7]


def test_unused_rows_and_ids_are_never_read():
    w = W.make_workload(4, device="cuda", B=64, V=20000)
    a = run_gpu(w)
    n = w.num_draft.long()
    tl = w.target_logits.clone()
    dp = w.draft_probs.clone()
    for b in range(w.B):
        tl[b, n[b] + 1:] = float("nan")
        dp[b, n[b]:] = float("nan")
    w2 = W.Workload(w.spec, tl, dp, w.draft_ids, w.num_draft, w.temperature, w.seed)
    b_ = run_gpu(w2)
    assert np.array_equal(a[0], b_[0]) and np.array_equal(a[1], b_[1])


def test_greedy_ties_lowest_index():
    rng = np.random.default_rng(4)
    B, K, V = 200, 3, 4096
    l = rng.integers(-3, 3, (B, K + 1, V)).astype(np.float64)   # massive ties
    top = l.argmax(-1)
    ids = np.where(rng.random((B, K)) < 0.7, top[:, :K], rng.integers(0, V, (B, K)))
    w = custom_workload(l, None, ids, [K] * B, [0.0] * B, bf16=True)
    out, nacc, _, _ = run_gpu(w)
    ref = oracle.spec_verify(**W.to_numpy(w))
    assert np.array_equal(out, ref["out_ids"]) and np.array_equal(nacc, ref["out_num_accepted"])


def test_request_offset_shards_agree():
    w = W.make_workload(3, device="cuda", B=48, V=12000)
    full = run_gpu(w)
    parts = []
    for lo, hi in ((0, 20), (20, 48)):
        s = w.subset(list(range(lo, hi)))
        parts.append(run_gpu(s, request_offset=lo))
    assert np.array_equal(full[0], np.concatenate([p[0] for p in parts]))
    assert np.array_equal(full[1], np.concatenate([p[1] for p in parts]))


def test_deterministic_and_seed_sensitive():
    w = W.make_workload(4, device="cuda", B=64, V=30000)
    a, b = run_gpu(w), run_gpu(w)
    assert np.array_equal(a[0], b[0])
    w.seed = 12345
    c = run_gpu(w)
    assert not np.array_equal(a[0], c[0])


def test_host_buffer_entry_point_matches():
    w = W.make_workload(2, device="cuda")
    want = run_gpu(w, debug=False)
    B, K1, V = w.target_logits.shape
    K = K1 - 1
    h = {k: getattr(w, k).cpu().pin_memory() for k in
         ("target_logits", "draft_probs", "draft_ids", "num_draft", "temperature")}
    out = torch.empty((B, K1), dtype=torch.int32).pin_memory()
    nacc = torch.empty((B,), dtype=torch.int32).pin_memory()
    d_l = torch.empty_like(w.target_logits)
    d_p = torch.empty_like(w.draft_probs)
    small = torch.empty(binding.host_small_bytes(B, K), dtype=torch.uint8, device="cuda")
    ws = binding.new_workspace(B, K, V, "cuda")
    binding.spec_verify_host(h["target_logits"], h["draft_probs"], h["draft_ids"],
                             h["num_draft"], h["temperature"], w.seed, out, nacc, d_l, d_p,
                             small, ws)
    torch.cuda.synchronize()
    assert np.array_equal(out.numpy(), want[0]) and np.array_equal(nacc.numpy(), want[1])


@pytest.mark.parametrize("pinned", [True, False])
def test_host_buffer_rows_only_and_whole_copies(pinned):
    """spec_verify_host on the largest vocabulary (leading 64 requests):
    pinned host buffers take the copy kernels that move only the rows the
    verifier reads (the device buffers start as garbage, so a row it reads
    but did not copy shows); pageable buffers take whole-tensor copies.
    Both give the device call's outputs."""
    w = W.make_workload(4, device="cuda").leading(64)
    want = run_gpu(w, debug=False)
    B, K1, V = w.target_logits.shape
    K = K1 - 1
    h = {k: getattr(w, k).cpu() for k in
         ("target_logits", "draft_probs", "draft_ids", "num_draft", "temperature")}
    if pinned:
        h = {k: t.pin_memory() for k, t in h.items()}
    out = torch.empty((B, K1), dtype=torch.int32)
    nacc = torch.empty((B,), dtype=torch.int32)
    if pinned:
        out, nacc = out.pin_memory(), nacc.pin_memory()
    d_l = torch.full_like(w.target_logits, float("nan"))
    d_p = torch.full_like(w.draft_probs, float("nan"))
    small = torch.empty(binding.host_small_bytes(B, K), dtype=torch.uint8, device="cuda")
    ws = binding.new_workspace(B, K, V, "cuda")
    for seed in (w.seed, w.seed + 1):
        binding.spec_verify_host(h["target_logits"], h["draft_probs"], h["draft_ids"],
                                 h["num_draft"], h["temperature"], seed, out, nacc, d_l, d_p,
                                 small, ws)
        torch.cuda.synchronize()
        ref = run_gpu(w, debug=False) if seed == w.seed else None
        if seed != w.seed:
            ids2, nacc2 = binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids,
                                              w.num_draft, w.temperature, seed)
            torch.cuda.synchronize()
            ref = (ids2.cpu().numpy(), nacc2.cpu().numpy())
        assert np.array_equal(out.numpy(), ref[0]) and np.array_equal(nacc.numpy(), ref[1])
    assert (want[1] < w.num_draft.cpu().numpy()).any()  # residual draws took q rows


def test_misaligned_and_small_workspace_rejected():
    ensure_built()
    w = W.make_workload(1, device="cuda")
    B, K1, V = w.target_logits.shape
    ws = binding.new_workspace(B, K1 - 1, V, "cuda")
    with pytest.raises(binding.SpecVerifyError) as e:
        binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                            w.temperature, 0, workspace=ws[:64])
    assert e.value.status == binding.SPEC_ERR_WORKSPACE
    big = torch.zeros(B * K1 * V + 1, dtype=torch.float32, device="cuda")
    shifted = big[1:].view(B, K1, V)   # 4-byte offset: not 16-byte aligned
    with pytest.raises(binding.SpecVerifyError) as e:
        binding.spec_verify(shifted, w.draft_probs, w.draft_ids, w.num_draft, w.temperature, 0)
    assert e.value.status == binding.SPEC_ERR_UNSUPPORTED


def test_status_word_in_workspace():
    w = W.make_workload(1, device="cuda")
    B, K1, V = w.target_logits.shape
    ws = binding.new_workspace(B, K1 - 1, V, "cuda")
    bad_t = torch.full_like(w.temperature, -1.0)
    binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft, bad_t, 0,
                        workspace=ws)
    assert int(binding.status_word(ws).item()) == binding.BADBIT["temperature"]
    binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                        w.temperature, 0, workspace=ws)
    assert int(binding.status_word(ws).item()) == 0


def test_lossless_chi_square_on_gpu():
    """The emitted token at slot j, given the request reached it, follows p_j
    (10^6 requests through the CUDA path; no oracle involved)."""
    from scipy.stats import chisquare
    rng = np.random.default_rng(17)
    V, K, B = 8, 3, 1_000_000
    l = rng.normal(0, 1.0, (K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), K).astype(np.float32)
    p = np.exp(l.astype(np.float64) - l.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    ids = np.empty((B, K), np.int32)
    for j in range(K):
        cdf = np.cumsum(q[j].astype(np.float64) / q[j].sum())
        ids[:, j] = np.minimum(np.searchsorted(cdf, rng.random(B), side="right"), V - 1)
    ensure_built()
    dev = "cuda"
    tl = torch.from_numpy(l).to(dev)[None].expand(B, K + 1, V).contiguous()
    dp = torch.from_numpy(q).to(dev)[None].expand(B, K, V).contiguous()
    out, nacc = binding.spec_verify(tl, dp, torch.from_numpy(ids).to(dev),
                                    torch.full((B,), K, dtype=torch.int32, device=dev),
                                    torch.ones(B, device=dev), 99)
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    for j in range(K + 1):
        reach = nacc >= j
        obs = np.bincount(out[reach, j], minlength=V)
        assert chisquare(obs, p[j] * reach.sum()).pvalue > 1e-3, (j, obs)
    alpha = [np.minimum(p[j], q[j]).sum() for j in range(K)]
    for k in range(K + 1):
        pk = np.prod(alpha[:k]) * (1 - alpha[k] if k < K else 1.0)
        f = np.mean(nacc == k)
        assert abs(f - pk) < 5 * math.sqrt(pk * (1 - pk) / B) + 1e-9


def test_device_seed_and_graph_replay():
    """The seed read from device memory gives the same result as the seed
    passed by value, and a call captured in a CUDA graph replays with the
    seed written before each replay."""
    ensure_built()
    w = W.make_workload(3, device="cuda")
    B, K = w.B, w.K
    ws = binding.new_workspace(B, K, w.V, torch.device("cuda"))
    out = torch.empty((B, K + 1), dtype=torch.int32, device="cuda")
    nacc = torch.empty((B,), dtype=torch.int32, device="cuda")
    seed = torch.tensor([123456789], dtype=torch.int64, device="cuda")

    def call(**kw):
        binding.spec_verify(w.target_logits, w.draft_probs, w.draft_ids, w.num_draft,
                            w.temperature, kw.pop("s", 0), out_ids=out, out_num_accepted=nacc,
                            workspace=ws, **kw)

    call(s=123456789)
    torch.cuda.synchronize()
    want = (out.clone(), nacc.clone())
    call(seed_dev=seed)
    torch.cuda.synchronize()
    assert torch.equal(out, want[0]) and torch.equal(nacc, want[1])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(seed_dev=seed, stream=s)
    for sd in (77, 123456789, 2**40 + 3):
        seed.fill_(sd)
        g.replay()
        torch.cuda.synchronize()
        got = (out.clone(), nacc.clone())
        call(s=sd)
        torch.cuda.synchronize()
        assert torch.equal(got[0], out) and torch.equal(got[1], nacc), sd


def _tiny_temperature_workload(bf16: bool):
    """Rows whose offsets RN(max * log2(e) / T) run far past 2^24: tiny
    temperatures, maxima of both signs and of larger magnitude, and exact
    ties at the maximum in some rows."""
    rng = np.random.default_rng(29 + bf16)
    B, K, V = 40, 3, 5000
    l = rng.normal(0, 3.0, (B, K + 1, V))
    l += rng.choice([-60.0, -2.0, 0.0, 35.0], (B, 1, 1))
    for b in range(0, B, 3):  # two or three tokens share the maximum
        for j in range(K + 1):
            top = l[b, j].max() + 1.0
            l[b, j, rng.choice(V, 2 + (b % 2), replace=False)] = top
    dl = l[:, :K] + rng.normal(0, 1.0, (B, K, V))
    q = np.exp(dl - dl.max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    ids = np.array([[l[b, j].argmax() if (b + j) % 2 == 0 else rng.choice(V, p=q[b, j])
                     for j in range(K)] for b in range(B)])
    n = rng.integers(0, K + 1, B)
    temps = [1e-3, 1e-6, 1e-8, 1e-10, 1e-20, 1e-30, 1e-38, 1e-44]
    T = np.array([temps[b % len(temps)] for b in range(B)])
    return l, q, ids, n, T


@pytest.mark.parametrize("bf16", [False, True])
def test_tiny_temperatures_match_oracle(bf16):
    """Very small positive temperatures make softmax(l / T) a point mass on
    the row's maxima; the one-FFMA weight offset must not overflow there."""
    l, q, ids, n, T = _tiny_temperature_workload(bf16)
    w = custom_workload(l, q, ids, n, T, bf16=bf16, seed=7)
    rep = check_parity(w, f"tiny_T_{'bf16' if bf16 else 'f32'}")
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    # where p is a point mass, every emitted token is one of the row's maxima
    out, nacc, _, _ = run_gpu(w)
    lv = w.target_logits.float().cpu().numpy()
    for b in range(len(n)):
        if T[b] <= 1e-8 and nacc[b] >= 0:
            row = lv[b, nacc[b]]
            assert row[out[b, nacc[b]]] == row.max(), b


def _wide_vocab_workload(bf16: bool, V: int = 300008, B: int = 12, K: int = 3, seed: int = 41):
    """More than 128 chunks of 2048 tokens per row (V = 300008: 147 chunks,
    the last one 1000 tokens): the pairwise row merges and the block-by-block
    chunk picks that shorter vocabularies never reach."""
    rng = np.random.default_rng(seed + bf16)
    l = rng.normal(0, 2.0, (B, K + 1, V))
    dl = l[:, :K] + rng.normal(0, 1.0, (B, K, V))
    q = np.exp(dl - dl.max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    ids = np.array([[rng.choice(V, p=q[b, j]) for j in range(K)] for b in range(B)])
    n = rng.integers(0, K + 1, B)
    n[:2] = K  # at least two requests can reach the bonus row
    T = np.where(np.arange(B) % 4 == 3, 0.0, rng.uniform(0.5, 1.5, B))
    return custom_workload(l, q, ids, n, T, bf16=bf16, seed=seed)


@pytest.mark.parametrize("bf16", [False, True])
def test_more_than_128_chunks(bf16):
    w = _wide_vocab_workload(bf16)
    rep = check_parity(w, f"wide_V300008_{'bf16' if bf16 else 'f32'}")
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    # the early exit merges its rows inside k_row_stats: same outputs
    par = run_gpu(w)
    ee = run_gpu(w, early_exit=True)
    assert np.array_equal(par[0], ee[0]) and np.array_equal(par[1], ee[1])


def test_many_requests_small_vocabulary():
    """B = 5000 requests (several passes of k_plan's scan, 5000 acceptance
    CTAs, 10000 draw slots) over a 1024-token vocabulary."""
    rng = np.random.default_rng(43)
    B, K, V = 5000, 2, 1024
    l = rng.normal(0, 2.0, (B, K + 1, V))
    dl = l[:, :K] + rng.normal(0, 0.7, (B, K, V))
    q = np.exp(dl - dl.max(-1, keepdims=True))
    q /= q.sum(-1, keepdims=True)
    cq = q.cumsum(-1)
    ids = (cq < rng.random((B, K, 1))).sum(-1).clip(0, V - 1)  # x_j ~ q_j
    n = rng.integers(0, K + 1, B)
    T = np.where(rng.random(B) < 0.2, 0.0, rng.uniform(0.5, 1.5, B))
    w = custom_workload(l, q, ids, n, T, bf16=True, seed=43)
    rep = check_parity(w, "B5000_V1024")
    assert not rep.failures, rep.failures[:5]
    assert_excused_within_bound(rep)


def test_residual_without_mass_falls_back_to_p():
    """q_j = 2 p_j on every row (a draft distribution that is not normalised):
    a rejected draft leaves max(0, p - q) = 0 everywhere, and the token at the
    rejected row is drawn from p with the row's emission uniform instead."""
    rng = np.random.default_rng(53)
    B, K, V = 48, 3, 3000
    l = rng.normal(0, 2.0, (B, K + 1, V)).astype(np.float32)
    T = rng.uniform(0.6, 1.4, B)
    z = l[:, :K].astype(np.float64) / T[:, None, None]
    p = np.exp(z - z.max(-1, keepdims=True))
    p /= p.sum(-1, keepdims=True)
    q = (2.0 * p).astype(np.float32)
    cp = p.cumsum(-1)
    ids = (cp < rng.random((B, K, 1))).sum(-1).clip(0, V - 1)  # x_j ~ p_j
    n = np.full(B, K)
    w = custom_workload(l, q, ids, n, T, bf16=False, seed=53)
    rep = check_parity(w, "zero_residual_fallback")
    assert not rep.failures, rep.failures[:5]
    _, nacc, _, req = run_gpu(w)
    rejected = nacc < n
    assert rejected.sum() >= 10
    assert (req[rejected, 0] == oracle.MODE_FALLBACK).all()
    assert (req[~rejected, 0] == oracle.MODE_BONUS).all()
