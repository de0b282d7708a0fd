"""GPU parity of the segment-parallel inter-chunk scan (padded calls with few,
long chains): each chain's chunks are cut into segments; the transition and
offset of every segment but the last are computed in parallel, a combine forms
the entry states E_{s+1} = M_s E_s + C_s in fp32, and all segments' outputs are
computed in parallel from their entry states (the seg / comb kernels of the
cuDNN-frontend sm90 KDA page, Conversation).  Every head against the fp64
oracle element by element; deterministic across runs and under injected warp
stalls; the default schedule of the few-chain long workload."""
import numpy as np
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import assert_norm_close, assert_parity, gpu_prefill, oracle_prefill, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _run(inp, **over):
    import kda_chunked_prefill_02_gb300 as K
    with K.overrides(**over):
        sched = K.prefill_schedule(inp.q)
        out, fin = gpu_prefill(inp)
    return sched, out, fin


@pytest.mark.parametrize("case,nseg", [(dict(B=1, T=12300, H=2), 2),      # last segment short
                                       (dict(B=1, T=12300, H=2), 3),
                                       (dict(B=2, T=8192 + 37, H=3, init_std=None), 2),
                                       (dict(B=1, T=64 * 64 * 5, H=1), 5)])
def test_scan_matches_oracle(case, nseg):
    inp = inputs.prefill_inputs(1400 + nseg + case["T"] % 97, **case)
    sched, out, fin = _run(inp, scan_segments=nseg)
    assert sched["scan_segments"] == nseg, sched
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "scan, %d segments" % nseg)
    # the one-pass recurrence on the same inputs: both within tolerance of the
    # oracle, and close to each other
    _, out1, fin1 = _run(inp, scan_segments=1, segment_chunks=0)
    assert_parity(out1, fin1, ro, rf, "one pass")
    assert rel_fro(to_np(fin), to_np(fin1)) <= 1e-2


def test_scan_bit_identical_across_runs_and_under_stalls():
    inp = inputs.prefill_inputs(1450, B=1, T=12300, H=2)
    _, ref_out, ref_fin = _run(inp, scan_segments=3)
    for seed in (0, 1, 2, 3):
        _, out, fin = _run(inp, scan_segments=3, stall_seed=seed)
        assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin), seed


def test_scan_without_final_state_and_zero_initial_state():
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(1451, B=1, T=8192 + 64, H=2, init_std=None)
    d = inp.to("cuda")
    with K.overrides(scan_segments=2):
        out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, output_final_state=False)
    torch.cuda.synchronize()
    assert fin is None
    ro, rf = oracle_prefill(inp)
    assert_parity(out, None, ro, rf, "scan, no final state")


def test_scan_with_fused_norm():
    """The output pass of the scan carries the fused gated RMSNorm (the
    operator pass writes no outputs)."""
    import kda_chunked_prefill_02_gb300 as K
    from oracle.norm import gated_rmsnorm
    inp = inputs.prefill_inputs(1452, B=1, T=8192 + 100, H=2)
    gen = torch.Generator().manual_seed(3)
    gate = (torch.randn(inp.v.shape, generator=gen) * 2).to(torch.bfloat16)
    w = (torch.rand(128, generator=gen) + 0.5).float()
    d = inp.to("cuda")
    with K.overrides(scan_segments=2):
        plain_out, plain_fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
        out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                 out_gate=gate.cuda(), norm_weight=w.cuda(), norm_eps=1e-6)
    torch.cuda.synchronize()
    same = gated_rmsnorm(to_np(plain_out), gate.float().numpy(), w.numpy(), 1e-6)
    assert_norm_close(to_np(out), same)
    assert torch.equal(fin, plain_fin)


def test_few_chain_long_workload_takes_the_scan():
    """B=1, T=131072, H=8 (the long workload with a quarter of its heads): the
    default schedule is the scan; every head against the oracle."""
    inp = inputs.config_inputs("long_h8")
    sched, out, fin = _run(inp)
    assert sched["scan_segments"] >= 2, sched
    ro, rf = oracle_prefill(inp)
    og, fg = to_np(out), to_np(fin)
    worst = max(float(np.abs(og[..., h, :] - ro[..., h, :]).max()) for h in range(8))
    worst_st = max(rel_fro(fg[:, h], rf[:, h]) for h in range(8))
    print("long_h8 (scan, %d segments): worst out max-abs %.3e, worst final-state rel Frobenius %.3e"
          % (sched["scan_segments"], worst, worst_st))
    assert_parity(out, fin, ro, rf, "long_h8")
    assert worst_st <= 1e-2
