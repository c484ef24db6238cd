"""CUDA path vs the float64 oracle on the five measured workloads, at full size
and in the launch configuration the benchmark times (GPU)."""
import pytest
import torch

from gpu_common import assert_excused_within_bound, assert_excused_within_rate, check_parity
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
