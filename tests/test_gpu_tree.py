"""Token-tree verification on the GPU against the float64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_common import ensure_built
from speculative_decoding_verification_51_gb300 import binding
from tree_common import compare_tree, make_tree_workload, random_parents

pytestmark = pytest.mark.gpu


def _run(w, **kw):
    ensure_built()
    res = binding.spec_verify_tree(w.logits, w.probs, w.tokens, w.parents, w.nodes, w.temp,
                                   w.seed, debug=True, **kw)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in res]


def _check(w, tag):
    inp = w.to_numpy()
    ids, nacc, last, dbg, _ = _run(w)
    ref = oracle.tree_verify(**inp)
    rep = compare_tree(inp, ids, nacc, last, dbg, ref)
    print(f"[{tag}] {rep.summary()}")
    assert not rep.failures, rep.failures[:5]
    assert rep.excused < 1e-4 * rep.rows, rep.summary()
    return rep, (ids, nacc, last)


@pytest.mark.parametrize("B,N,V,bf16,width", [
    (64, 8, 1024, False, 1.0),
    (64, 16, 32000, True, 0.5),
    (16, 32, 128256, True, 0.3),
    (48, 12, 5000, False, 0.8),
    (40, 6, 2056, True, 1.0),
])
def test_tree_parity(B, N, V, bf16, width):
    w = make_tree_workload(B, N, V, bf16=bf16, seed=B + N + V, width=width)
    rep, (ids, nacc, last) = _check(w, f"tree_B{B}_N{N}_V{V}")
    assert rep.greedy > 0 and rep.sampling > 0
    assert (nacc > 0).any()  # some drafts were kept


def test_tree_chain_shape_matches_chain_verifier():
    """A trie with one child per node is verified exactly like the chain of
    its drafts (same uniforms, same rules): GPU tree vs GPU chain, and both
    against the oracle."""
    rng = np.random.default_rng(3)
    B, K, V = 64, 5, 4096
    w = make_tree_workload(B, K + 1, V, bf16=True, seed=11)
    par = np.tile(np.arange(-1, K, dtype=np.int32), (B, 1))
    w.parents = torch.from_numpy(par).cuda()
    ids, nacc, last, dbg, _ = _run(w)
    chain_probs = w.probs[:, 1:].contiguous()
    chain_ids = w.tokens[:, 1:].contiguous()
    cids, cnacc = binding.spec_verify(w.logits, chain_probs, chain_ids, w.nodes - 1, w.temp,
                                      w.seed)
    torch.cuda.synchronize()
    cids, cnacc = cids.cpu().numpy(), cnacc.cpu().numpy()
    inp = w.to_numpy()
    ref = oracle.tree_verify(**inp)
    rep = compare_tree(inp, ids, nacc, last, dbg, ref)
    assert not rep.failures, rep.failures[:5]
    # the two GPU verifiers agree wherever neither sits on an excused near-tie
    agree = (cnacc == nacc) & (cids == ids).all(1)
    assert agree.mean() > 0.97, agree.mean()
    assert np.array_equal(last[agree], nacc[agree])


def test_tree_greedy_is_bit_exact_and_bad_tries_are_flagged():
    rng = np.random.default_rng(5)
    B, N, V = 16, 8, 1024
    w = make_tree_workload(B, N, V, bf16=False, seed=5, greedy_frac=1.0)
    par = w.parents.cpu().numpy()
    tok = w.tokens.cpu().numpy()
    nodes = w.nodes.cpu().numpy()
    nodes[:] = N
    par[1, 3] = 5            # parent after the child
    tok[2, 4] = V            # token out of range
    nodes[3] = 0             # no root
    w.parents = torch.from_numpy(par).cuda()
    w.tokens = torch.from_numpy(tok).cuda()
    w.nodes = torch.from_numpy(nodes).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ensure_built()
    ids, nacc, last = [t.cpu().numpy() for t in binding.spec_verify_tree(
        w.logits, w.probs, w.tokens, w.parents, w.nodes, w.temp, w.seed, dev_status=st)]
    assert (nacc[1:4] == -1).all() and (ids[1:4] == -1).all() and (last[1:4] == -1).all()
    s = int(st.item())
    assert s & binding.BADBIT["tree"] and s & binding.BADBIT["draft_id"]
    assert s & binding.BADBIT["num_draft"]
    ref = oracle.tree_verify(**w.to_numpy())
    good = np.array([b for b in range(B) if b not in (1, 2, 3)])
    assert np.array_equal(ids[good], ref["out_ids"][good])
    assert np.array_equal(nacc[good], ref["out_num_accepted"][good])
    assert np.array_equal(last[good], ref["out_last_node"][good])


def test_tree_first_token_law():
    """Three children drawn independently from q below the root: the first
    output token follows p at the root (chi-square over 2^17 GPU walks)."""
    from scipy.stats import chisquare
    B, N, V = 1 << 17, 4, 64
    rng = np.random.default_rng(9)
    row = rng.normal(0, 1, (N, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V)).astype(np.float32)
    cdf = np.cumsum(q.astype(np.float64) / q.sum())
    tok = np.zeros((B, N), np.int32)
    for c in range(1, N):
        tok[:, c] = np.minimum(np.searchsorted(cdf, rng.random(B), side="right"), V - 1)
    par = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    ensure_built()
    logits = torch.from_numpy(np.broadcast_to(row, (B, N, V)).copy()).cuda()
    probs = torch.from_numpy(np.broadcast_to(q, (B, N, V)).copy()).cuda()
    ids, nacc, last = binding.spec_verify_tree(
        logits, probs, torch.from_numpy(tok).cuda(), torch.from_numpy(par).cuda(),
        torch.full((B,), N, dtype=torch.int32, device="cuda"),
        torch.ones(B, dtype=torch.float32, device="cuda"), 4242)
    first = ids[:, 0].cpu().numpy()
    p = np.exp(row[0].astype(np.float64) - row[0].max())
    p /= p.sum()
    assert chisquare(np.bincount(first, minlength=V), p * B).pvalue > 1e-4


def test_tree_request_offset():
    """A shard with a request offset draws the uniforms of its global indices."""
    w = make_tree_workload(48, 10, 3000, bf16=True, seed=21)
    ids, nacc, last, _, _ = _run(w)
    ensure_built()
    sl = slice(16, 40)
    sub = [t[sl].contiguous() for t in (w.logits, w.probs, w.tokens, w.parents, w.nodes, w.temp)]
    sids, snacc, slast = binding.spec_verify_tree(*sub, w.seed, request_offset=16)
    assert np.array_equal(sids.cpu().numpy(), ids[sl])
    assert np.array_equal(snacc.cpu().numpy(), nacc[sl])
    assert np.array_equal(slast.cpu().numpy(), last[sl])


def test_tree_tiny_temperatures():
    """Temperatures far below 1 (point masses on the maxima) through the tree
    walk's merges, acceptances and sibling residuals."""
    B = 40
    w = make_tree_workload(B, 8, 5000, bf16=True, seed=77, width=0.6)
    temps = [1e-3, 1e-8, 1e-10, 1e-20, 1e-30, 1e-38, 1e-44, 0.0]
    w.temp = torch.tensor([temps[b % len(temps)] for b in range(B)], dtype=torch.float32,
                          device=w.temp.device)
    rep, _ = _check(w, "tree_tiny_T")
    assert rep.sampling > 0 and rep.greedy > 0


def test_tree_more_than_128_chunks():
    """V = 300008 (147 chunks of 2048 tokens): the walk's row merges and chunk
    picks past 128 chunks."""
    w = make_tree_workload(8, 6, 300008, bf16=True, seed=91, width=0.5)
    rep, _ = _check(w, "tree_V300008")
    assert rep.sampling > 0
