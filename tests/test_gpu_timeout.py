"""The bounded-wait path of the kernels, exercised without faulting the GPU.

Every mbarrier wait in the prep and state kernels is bounded; a wait that runs
out writes KDA_ERR_TIMEOUT to the status word, and the CTA winds down: the
epilogue warps agree on stopping through the OR-reduction of the chunk
barrier, and before TMEM and shared memory are released every copy still in
flight and every product already issued is waited for (with the full 200 ms
bound).  A call's overrides can lower the bound of the working waits and turn
on a probe: the first wait of every CTA for a tensor-core product then waits
on an mbarrier that nothing arrives on, so it runs out while that product and
the tile copies are still in flight.  The call must still return, the device
must stay usable, and the next normal call on the same stream must give the
oracle's result (the
failure detection plan of the build: device-side timeouts reported through a
status word, the context kept alive; the TMEM-dealloc ordering of the
TensorRT-LLM MQA-logits page)."""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import assert_parity, oracle_prefill

pytestmark = pytest.mark.gpu

KDA_ERR_TIMEOUT = 4


def _call(d, status, **kw):
    import kda_chunked_prefill_02_gb300 as K
    return K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                         cu_seqlens=d.cu_seqlens, device_status=status, **kw)


@pytest.mark.parametrize("stage", ["prep", "state"])
@pytest.mark.parametrize("kernel", ["slab", "head"])
def test_wait_that_runs_out_is_reported_and_the_context_survives(stage, kernel):
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(1201, B=2, T=64 * 6 + 9, H=3)
    d = inp.to("cuda")
    ws = torch.empty(K.workspace_size(d.q, d.v), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with K.overrides(state_kernel=kernel, segment_chunks=0):
        if stage == "state":   # records from a normal prep, then a state pass that times out
            _call(d, status, workspace=ws, stage="prep")
            torch.cuda.synchronize()
            assert status.item() == 0
        with K.overrides(state_kernel=kernel, segment_chunks=0, wait_limit_ns=2000, timeout_probe=True):
            _call(d, status, workspace=ws, stage=stage)
        torch.cuda.synchronize()            # returns: no hang, no fault
        assert status.item() == KDA_ERR_TIMEOUT
        # the same stream, the same workspace, a normal call: the oracle's result
        status.zero_()
        out, fin = _call(d, status, workspace=ws)
        torch.cuda.synchronize()
    assert status.item() == 0
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "after a timed-out %s call" % stage)


def test_timeout_in_the_segmented_schedule_and_under_stalls():
    """Both streams of the segmented schedule wind down; also with the stall
    hook on, so that the probe's wait runs out at many different points of
    the other warps' work."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(1202, B=1, T=64 * 9 + 3, H=4)
    d = inp.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for seed in (0, 5):
        status.zero_()
        with K.overrides(segment_chunks=2, wait_limit_ns=2000, timeout_probe=True, stall_seed=seed):
            _call(d, status)
        torch.cuda.synchronize()
        assert status.item() == KDA_ERR_TIMEOUT, seed
    status.zero_()
    with K.overrides(segment_chunks=2):
        out, fin = _call(d, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "segmented call after timed-out calls")


def test_production_calls_ignore_the_environment(monkeypatch):
    """Names that earlier builds read from the environment change nothing: a
    call with them set gives the bits of a call without them."""
    inp = inputs.prefill_inputs(1203, B=1, T=64 * 9 + 3, H=4)
    d = inp.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _call(d, status)
    torch.cuda.synchronize()
    for name, val in (("KDA_STALL_INJECT", "3"), ("KDA_STATE_KERNEL", "slab"),
                      ("KDA_SEGMENT_CHUNKS", "1"), ("KDA_SEGMENT_PDL", "0")):
        monkeypatch.setenv(name, val)
    got = _call(d, status)
    torch.cuda.synchronize()
    assert torch.equal(ref[0], got[0]) and torch.equal(ref[1], got[1])


def test_timeout_in_the_scan():
    """The operator, combine-fed and output passes of the segment-parallel scan
    wind down like the other passes."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(1204, B=1, T=8192 + 64, H=2)
    d = inp.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with K.overrides(scan_segments=2, wait_limit_ns=2000, timeout_probe=True):
        _call(d, status)
    torch.cuda.synchronize()
    assert status.item() == KDA_ERR_TIMEOUT
    status.zero_()
    with K.overrides(scan_segments=2):
        out, fin = _call(d, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "scan after a timed-out scan")


def test_timeout_in_the_tensor_core_verify():
    """The tensor-core verify kernel's first product wait runs out under the
    probe: the call returns, the status says so, and a normal call on the same
    stream then matches the oracle."""
    import numpy as np
    import kda_chunked_prefill_02_gb300 as K
    import oracle
    vi = inputs.verify_inputs(1205, R=20, D=6, H=2)
    d = vi.to("cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = d.state_pool.clone()
    with K.overrides(verify_kernel="tensor", wait_limit_ns=2000, timeout_probe=True):
        K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, device_status=status)
    torch.cuda.synchronize()
    assert status.item() == KDA_ERR_TIMEOUT
    status.zero_()
    pool = d.state_pool.clone()
    with K.overrides(verify_kernel="tensor"):
        out = K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, device_status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    o_ref, _ = oracle.verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted)
    assert np.abs(out.float().cpu().numpy() - o_ref).max() <= 2e-2
