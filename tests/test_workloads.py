"""The seeded input generator: shapes, determinism, structure (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_51_gb300 import workloads as W


@pytest.mark.parametrize("cid", [1, 2])
def test_shapes_and_determinism(cid):
    a, b = W.make_workload(cid), W.make_workload(cid)
    s = W.SPECS[cid]
    assert a.target_logits.shape == (s.B, s.K + 1, s.V)
    assert a.draft_probs.shape == (s.B, s.K, s.V)
    assert a.target_logits.dtype == (torch.bfloat16 if s.dtype == "bf16" else torch.float32)
    for x, y in ((a.target_logits, b.target_logits), (a.draft_probs, b.draft_probs),
                 (a.draft_ids, b.draft_ids), (a.temperature, b.temperature)):
        assert torch.equal(x, y)
    assert torch.allclose(a.draft_probs.sum(-1), torch.ones(()), atol=1e-4)


@pytest.mark.parametrize("cid", [3, 4, 5])
def test_small_versions_of_large_recipes(cid):
    w = W.make_workload(cid, B=16, V=4096)
    n = w.num_draft.long()
    pos = torch.arange(w.K)[None]
    assert torch.all(w.draft_ids[pos >= n[:, None]] == -1)
    ok = w.draft_ids[pos < n[:, None]]
    assert torch.all((ok >= 0) & (ok < w.V))
    if cid == 4:
        assert torch.all((n >= 0) & (n <= 3))
    if cid == 5:
        assert torch.all((n >= 1) & (n <= 8))
        assert torch.all((w.temperature >= 0.3) & (w.temperature <= 1.5))


def test_config2_half_greedy_and_oracle_runs():
    w = W.make_workload(2)
    assert torch.equal(w.temperature[1::2], torch.zeros(4))
    assert torch.equal(w.temperature[0::2], torch.ones(4))
    r = oracle.spec_verify(**W.to_numpy(w))
    assert r["n_bad"] == 0
    a = r["out_num_accepted"]
    assert np.all((a >= 0) & (a <= w.K))


def test_counts():
    nd = torch.tensor([0, 3, 1])
    assert W.valid_rows(nd) == 7 and W.positions(nd) == 4


def test_named_workload_is_one_input_set():
    """The generator runs on the host whatever the target device, so a named
    workload is the same inputs everywhere; repeated builds return their own
    tensors (the host cache hands out copies)."""
    a = W.make_workload(3, B=8, V=2048)
    b = W.make_workload(3, B=8, V=2048)
    assert a.target_logits.data_ptr() != b.target_logits.data_ptr()
    a.target_logits.zero_()
    c = W.make_workload(3, B=8, V=2048)
    assert torch.equal(b.target_logits, c.target_logits)
    assert not torch.equal(a.target_logits, c.target_logits)


@pytest.mark.gpu
@pytest.mark.parametrize("cid", [2, 4])
def test_device_copy_equals_host_build(cid):
    h = W.make_workload(cid, device="cpu")
    d = W.make_workload(cid, device="cuda")
    for k in ("target_logits", "draft_probs", "draft_ids", "num_draft", "temperature"):
        assert torch.equal(getattr(h, k), getattr(d, k).cpu()), k
