"""Bit-identical results under injected warp stalls.

An overrides stall_seed launches the kernel instantiations with the stall hook:
at every injection site (before and after each barrier, mbarrier wait,
tensor-core issue, copy issue and hand-off of the prep, state and verify
kernels) a quarter of the warps, chosen by a hash of the seed, block, warp, site
and iteration, spin for 0..4095 cycles.  Only the timing changes, so every
output, final state, workspace record and verify pool must equal the
unperturbed run's bit for bit; a missing barrier or a buffer reused too early
would show as a difference.  Each case also runs twice without stalls (the
plain run is deterministic)."""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs

pytestmark = pytest.mark.gpu

SEEDS = (1, 2, 3)


def _prefill(d, seed, **over):
    import kda_chunked_prefill_02_gb300 as K
    ws = torch.full((K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    with K.overrides(stall_seed=seed or 0, **over):
        out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                 cu_seqlens=d.cu_seqlens, workspace=ws)
        torch.cuda.synchronize()
    return out.cpu(), fin.cpu()


def _same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


@pytest.mark.parametrize("kernel", ["slab", "head"])
@pytest.mark.parametrize("case", [dict(B=2, T=64 * 5 + 17, H=3),
                                  dict(lengths=[17, 0, 16, 130, 1, 64], H=2)])
def test_prefill_bit_identical_under_stalls(kernel, case):
    inp = inputs.prefill_inputs(900 + len(case), **case)
    d = inp.to("cuda")
    ref = _prefill(d, 0, state_kernel=kernel, segment_chunks=0)
    assert _same(ref, _prefill(d, 0, state_kernel=kernel, segment_chunks=0))
    for seed in SEEDS:
        got = _prefill(d, seed, state_kernel=kernel, segment_chunks=0)
        assert _same(ref, got), "seed %d changed the result" % seed


def test_segmented_bit_identical_under_stalls():
    """Two streams, programmatic launches and the state carried between
    segments, with stalls in both kernels."""
    inp = inputs.prefill_inputs(910, B=1, T=64 * 9 + 3, H=4)
    d = inp.to("cuda")
    ref = _prefill(d, 0, segment_chunks=2)
    for seed in SEEDS:
        assert _same(ref, _prefill(d, seed, segment_chunks=2)), seed


def test_prep_records_bit_identical_under_stalls():
    """The per-chunk records of the prep kernel alone (every operand image)."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(911, lengths=[200, 64, 5], H=2)
    d = inp.to("cuda")

    def records(seed):
        ws = torch.full((K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens),), 0xFF,
                        dtype=torch.uint8, device="cuda")
        with K.overrides(stall_seed=seed or 0):
            K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                          cu_seqlens=d.cu_seqlens, workspace=ws, stage="prep")
            torch.cuda.synchronize()
        L = K.workspace_layout(d.q, cu_seqlens=d.cu_seqlens)
        n = int(L.max_chunks) * 2 * int(L.record_bytes)
        return ws[L.records:L.records + n].cpu()

    ref = records(0)
    for seed in SEEDS:
        assert torch.equal(ref, records(seed)), seed


def test_norm_bit_identical_under_stalls():
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(912, B=1, T=200, H=2)
    d = inp.to("cuda")
    gen = torch.Generator().manual_seed(913)
    gate = (torch.randn(inp.v.shape, generator=gen) * 2).to(torch.bfloat16).cuda()
    w = (torch.rand(128, generator=gen) + 0.5).float().cuda()

    def run(seed):
        with K.overrides(stall_seed=seed or 0):
            out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                     out_gate=gate, norm_weight=w)
            torch.cuda.synchronize()
        return out.cpu(), fin.cpu()

    ref = run(0)
    for seed in SEEDS:
        assert _same(ref, run(seed)), seed


@pytest.mark.parametrize("kernel,D", [("sequential", 4), ("tensor", 4), ("tensor", 11)])
@pytest.mark.parametrize("pool_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("replay", [False, True])
def test_verify_bit_identical_under_stalls(pool_dtype, replay, kernel, D):
    import kda_chunked_prefill_02_gb300 as K
    vi = inputs.verify_inputs(914, R=40, D=D, H=3)
    d = vi.to("cuda")
    pool0 = d.state_pool.to(pool_dtype)

    def run(seed):
        pool = pool0.clone()
        with K.overrides(stall_seed=seed or 0, verify_kernel=kernel):
            out = K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, slot=d.slot,
                               replay_only=replay)
            torch.cuda.synchronize()
        return (pool.cpu(),) if replay else (out.cpu(), pool.cpu())

    ref = run(0)
    for seed in SEEDS:
        assert _same(ref, run(seed)), seed
