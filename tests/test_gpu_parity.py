"""CUDA path vs the float64 oracle on the five measured workloads, at full size
and in the launch configuration the benchmark times (GPU)."""
import pytest
import torch

from gpu_common import assert_excused_within_bound, assert_excused_within_rate, check_parity
from speculative_decoding_verification_51_gb300 import binding
from speculative_decoding_verification_51_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_workload_parity(cid):
    w = W.make_workload(cid, device="cuda")
    rep = check_parity(w, f"config{cid}")
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    assert_excused_within_bound(rep)
    del w
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B", [32, 128])
def test_config5_sweep_prefixes(B):
    w = W.make_workload(5, device="cuda").leading(B)
    rep = check_parity(w, f"config5_B{B}")
    assert not rep.failures, rep.failures[:5]
    assert_excused_within_bound(rep)


@pytest.mark.parametrize("cid,seed", [(3, 7), (4, 8), (4, 9), (5, 10)])
def test_more_seeds(cid, seed):
    w = W.make_workload(cid, device="cuda", gen_seed=seed)
    w.seed = seed * 1000 + 1
    rep = check_parity(w, f"config{cid}_seed{seed}")
    assert not rep.failures, rep.failures[:5]
    assert_excused_within_rate(rep, w.V)


@pytest.mark.parametrize("cid", [1, 2, 3])
def test_workload_parity_by_request(cid):
    """The smaller workloads, where spec_verify runs the all-rows pass, through
    the request-by-request verifier."""
    w = W.make_workload(cid, device="cuda")
    rep = check_parity(w, f"config{cid}_by_request", by_request=True)
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    assert_excused_within_bound(rep)


def test_path_follows_the_sm_count():
    """spec_verify runs request by request from B = 2.1 x the SM count up."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    b0 = (21 * sms + 9) // 10  # the smallest B with 10 B >= 21 SMs
    for B, want in ((b0 - 1, 0), (b0, 1), (512, 1), (64, 0), (1, 0)):
        assert binding.verify_path(B, 3, 151936, torch.bfloat16) == want, (B, sms)
    assert binding.verify_path(512, 3, 97 * 2048, torch.bfloat16) == 0  # rows too long
    assert binding.verify_path(512, 3, 151936, torch.float32) == 1


def test_large_batch_by_request():
    """Config 4's recipe at B = 1024: spec_verify verifies request by request,
    each CTA claiming about seven requests in turn (the claim order, the two
    request records and the pass ring reused many times)."""
    w = W.make_workload(4, device="cuda", B=1024)
    assert binding.verify_path(w.B, w.K, w.V, w.target_logits.dtype) == 1
    rep = check_parity(w, "config4_B1024")
    assert not rep.failures, rep.failures[:5]
    assert rep.max_p_rel <= 1e-5
    assert_excused_within_rate(rep, w.V)
    del w
    torch.cuda.empty_cache()
