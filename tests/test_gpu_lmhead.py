"""The tcgen05 LM-head projection (spec_lmhead_logits) against the float64
oracle and against a plain PyTorch float32 matmul (GPU).

Tolerance: the kernel sums float32 products in its own order and rounds once
to bf16; the oracle sums exactly.  A float32 sum of H products is within
H * 2^-24 * sum|h_k w_k| of the exact one (the standard bound for recursive
summation, doubled here for the tensor cores' internal order), and the bf16
rounding adds half an ulp of the result.  Every logit must lie within that
bound; logits that differ from the oracle's bf16 value at all must be rare
(they sit within the float32 error of a rounding boundary, or cancel).
"""
import numpy as np
import pytest
import torch

from gpu_common import ensure_built
from oracle import lmhead as LM
from speculative_decoding_verification_51_gb300 import binding

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _ulp(a, b):
    a = a.astype(np.int32)
    b = b.astype(np.int32)
    oa = np.where(a & 0x8000, -(a & 0x7FFF), a & 0x7FFF)
    ob = np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(oa - ob)


def _bf16_ulp(x):
    """Spacing of bf16 numbers at |x| (float64)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return np.ldexp(1.0, np.frexp(ax)[1] - 8)


def _within_bound(out_bits, exact, abs_sum, H):
    got = LM.bf16_bits_to_f64(out_bits)
    bound = 0.5 * _bf16_ulp(got) + 2.0 * H * 2.0 ** -24 * abs_sum
    return np.abs(got - exact) <= bound


def _inputs(rows, H, V, seed, wscale=None):
    g = torch.Generator(device="cpu").manual_seed(seed)
    hid = torch.randn(rows, H, generator=g).to(torch.bfloat16)
    w = (torch.randn(V, H, generator=g) * (wscale or H ** -0.5)).to(torch.bfloat16)
    return hid.cuda(), w.cuda()


@pytest.mark.parametrize("rows,H,V", [(200, 128, 4104), (1, 64, 8), (129, 192, 2056)])
def test_lmhead_matches_oracle(rows, H, V):
    ensure_built()
    hid, w = _inputs(rows, H, V, rows + H + V)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.lmhead_logits(hid, w, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    hb, wb = _bits(hid), _bits(w)
    ref = LM.lmhead_logits(hb, wb)
    exact = LM.lmhead_logits_f64(hb, wb)
    abs_sum = np.abs(LM.bf16_bits_to_f64(hb)) @ np.abs(LM.bf16_bits_to_f64(wb)).T
    ok = _within_bound(_bits(out), exact, abs_sum, H)
    assert ok.all(), np.argwhere(~ok)[:5]
    d = _ulp(_bits(out), ref)
    assert (d > 0).mean() < 0.02
    assert (d <= 1).mean() > 0.999  # more than 1 ulp only where the sum cancels


@pytest.mark.parametrize("rows,H,V", [(658, 1024, 151936), (256, 4096, 32000)])
def test_lmhead_matches_torch(rows, H, V):
    ensure_built()
    hid, w = _inputs(rows, H, V, 7)
    out = binding.lmhead_logits(hid, w)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    ref = (hid.float() @ w.float().T).to(torch.bfloat16)
    torch.backends.cuda.matmul.allow_tf32 = prev
    torch.cuda.synchronize()
    d = _ulp(_bits(out), _bits(ref))
    assert (d > 0).mean() < 0.02
    assert (d <= 1).mean() > 0.999
    # a sampled block checked against the float64 oracle within the bound
    rs = slice(100, 140)
    vs = slice(V - 300, V)
    hb, wb = _bits(hid[rs]), _bits(w[vs])
    exact = LM.lmhead_logits_f64(hb, wb)
    abs_sum = np.abs(LM.bf16_bits_to_f64(hb)) @ np.abs(LM.bf16_bits_to_f64(wb)).T
    assert _within_bound(_bits(out[rs, vs]), exact, abs_sum, H).all()


# ------------------------------------------------ the fused verifier (spec_verify_lmhead)

import parity  # noqa: E402
import oracle  # noqa: E402
from speculative_decoding_verification_51_gb300 import workloads as W  # noqa: E402


def _fused_check(B, K, V, H, seed, w=None, **kw):
    ensure_built()
    if w is None:
        w = W.make_lmhead_workload(B, K, V, H, seed=seed, **kw)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids, nacc, logits, rows, req = binding.spec_verify_lmhead(
        w.hidden, w.lm_head, w.draft_probs, w.draft_ids, w.num_draft, w.temperature, w.seed,
        debug=True, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ids, nacc, rows = ids.cpu().numpy(), nacc.cpu().numpy(), rows.cpu().numpy()
    inp = W.lmhead_to_numpy(w)
    # the oracle's own logits: exact sums (integer operands), one bf16 rounding
    lo = LM.lmhead_logits(inp["hidden"].reshape(-1, H), inp["lm_head"]).reshape(B, K + 1, V)
    n = inp["num_draft"]
    got = _bits(logits)
    for b in range(B):  # the rows the verifier reads are written, bit for bit
        assert np.array_equal(got[b, : n[b] + 1], lo[b, : n[b] + 1]), b
    vin = {"target_logits": lo, "draft_probs": inp["draft_probs"], "draft_ids": inp["draft_ids"],
           "num_draft": n, "temperature": inp["temperature"], "seed": inp["seed"]}
    ref = oracle.spec_verify(**vin)
    rep = parity.compare(vin, ids, nacc, rows, ref)
    print(f"[lmhead B{B} K{K} V{V} H{H}] {rep.summary()}")
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    assert rep.excused < 1e-4 * rep.rows, rep.summary()
    return rep


@pytest.mark.parametrize("B,K,V,H,greedy", [(40, 4, 4104, 128, 0.25), (24, 3, 2056, 64, 1.0),
                                            (33, 5, 8200, 192, 0.0)])
def test_fused_verify_small(B, K, V, H, greedy):
    rep = _fused_check(B, K, V, H, seed=B + V, greedy_frac=greedy)
    if greedy == 1.0:
        assert rep.sampling == 0
    if greedy == 0.0:
        assert rep.greedy == 0


def test_fused_verify_largest_vocabulary():
    """The largest-vocabulary shape (B=256, K=3, V=151936, ragged num_draft,
    25% greedy) with hidden size 1024."""
    rep = _fused_check(256, 3, 151936, 1024, seed=4)
    assert rep.greedy > 0 and rep.sampling > 0


def test_fused_verify_tiny_temperatures():
    """The projection epilogue's running row statistics at temperatures down
    to 1e-44 (offsets RN(max * log2(e) / T) far past 2^24)."""
    B, K, V, H = 32, 3, 4104, 128
    w = W.make_lmhead_workload(B, K, V, H, seed=71, greedy_frac=0.2)
    temps = torch.tensor([1e-3, 1e-8, 1e-10, 1e-20, 1e-30, 1e-38, 1e-44, 0.7])
    t = temps[torch.arange(B) % len(temps)].to(w.temperature.device)
    w.temperature = torch.where(w.temperature > 0, t, w.temperature).contiguous()
    rep = _fused_check(B, K, V, H, seed=71, w=w)
    assert rep.sampling > 0
