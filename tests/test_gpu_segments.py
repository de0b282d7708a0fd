"""GPU parity of the segmented schedule of padded calls: the tokens are cut into
segments, the state pass of one segment runs on a second stream beside the
prep of the next, and every chain's state passes between segments in fp32
through the workspace.  Forced through the call's overrides on small shapes: bit
for bit equal to the one-pass call with the same state kernel (the chunk steps
are the same, the state crosses a segment boundary exactly), and within the
tolerances of the fp64 oracle.  The long workload at full size takes this
schedule by default (test_gpu_prefill.test_full_size_configs)."""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import assert_parity, oracle_prefill, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _run(d, **kw):
    """One call on a workspace filled with 0xff bytes (NaN as fp32 / bf16), so
    that a record or carried state read before it is written shows."""
    import kda_chunked_prefill_02_gb300 as K
    ws = torch.full((K.workspace_size(d.q, d.v),), 0xFF, dtype=torch.uint8, device="cuda")
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                             workspace=ws, **kw)
    torch.cuda.synchronize()
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("kernel", ["slab", "head"])
@pytest.mark.parametrize("case,seg", [(dict(B=1, T=64 * 9 + 5, H=2), 2),
                                      (dict(B=2, T=64 * 5, H=3, init_std=None), 1),
                                      (dict(B=3, T=64 * 4 + 63, H=1), 3),
                                      (dict(B=1, T=200, H=2), 100)])
def test_segments_equal_one_pass(kernel, case, seg):
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(800 + seg + case["T"], **case)
    d = inp.to("cuda")
    with K.overrides(state_kernel=kernel, segment_chunks=seg):
        sch = K.prefill_schedule(d.q)
        assert sch["segmented"] and sch["segment_chunks"] == min(seg, -(-case["T"] // 64))
        assert sch["whole_chain"] == (kernel == "head")
        out_s, fin_s = _run(d)
    with K.overrides(state_kernel=kernel, segment_chunks=0):
        assert not K.prefill_schedule(d.q)["segmented"]
        out_1, fin_1 = _run(d)
    assert torch.equal(out_s, out_1) and torch.equal(fin_s, fin_1)
    ro, rf = oracle_prefill(inp)
    assert_parity(out_s, fin_s, ro, rf, "segmented, %s kernel" % kernel)


def test_segments_in_place_state():
    """initial_state and final_state the same buffer: the first segment reads
    it, only the last one writes it."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(851, B=2, T=64 * 6 + 10, H=2)
    d = inp.to("cuda")
    ro, rf = oracle_prefill(inp)
    st = d.initial_state.clone()
    with K.overrides(segment_chunks=2):
        out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=st, final_state=st)
        torch.cuda.synchronize()
    assert fin.data_ptr() == st.data_ptr()
    assert_parity(out, st, ro, rf, "segmented, in-place state")


def test_segments_with_fused_norm():
    """The fused gated RMSNorm in the segmented schedule (whole-chain kernel):
    the gate pointer moves with the segment."""
    import kda_chunked_prefill_02_gb300 as K
    from oracle.norm import gated_rmsnorm
    inp = inputs.prefill_inputs(852, B=2, T=64 * 5 + 7, H=2)
    gen = torch.Generator().manual_seed(853)
    gate = (torch.randn(inp.v.shape, generator=gen) * 2).to(torch.bfloat16)
    w = (torch.rand(128, generator=gen) + 0.5).float()
    d = inp.to("cuda")
    kw = dict(out_gate=gate.cuda(), norm_weight=w.cuda(), norm_eps=1e-6)
    with K.overrides(segment_chunks=2):
        assert K.prefill_schedule(d.q, norm=True)["whole_chain"]
        out_s, fin_s = _run(d, **kw)
    with K.overrides(segment_chunks=0):
        out_1, fin_1 = _run(d, **kw)
    assert torch.equal(out_s, out_1) and torch.equal(fin_s, fin_1)
    ro, rf = oracle_prefill(inp)
    ref = gated_rmsnorm(ro, gate.float().numpy(), w.numpy(), 1e-6)
    assert rel_fro(to_np(out_s), ref) <= 2e-2
    assert rel_fro(to_np(fin_s), rf) <= 1e-2


def test_segments_strided_views():
    """Strided (non-contiguous) inputs: each segment's base pointers advance by
    its first token times the token stride."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(854, B=2, T=64 * 4 + 1, H=2)
    d = inp.to("cuda")
    # views into a wider buffer: heads interleaved with a dummy head
    def widen(t):
        shape = list(t.shape)
        shape[2] = 3
        w = torch.zeros(shape, dtype=t.dtype, device=t.device)
        w[:, :, 0:3:2] = t
        return w[:, :, 0:3:2]
    q, k, v, g = (widen(t) for t in (d.q, d.k, d.v, d.g))
    b = torch.zeros(d.beta.shape[0], d.beta.shape[1], 3, device="cuda")
    b[:, :, 0:3:2] = d.beta
    beta = b[:, :, 0:3:2]
    assert not q.is_contiguous()
    with K.overrides(segment_chunks=1):
        out_s, fin_s = K.kda_prefill(q, k, v, g, beta, initial_state=d.initial_state)
        torch.cuda.synchronize()
    with K.overrides(segment_chunks=0):
        out_1, fin_1 = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
        torch.cuda.synchronize()
    assert torch.equal(out_s, out_1) and torch.equal(fin_s, fin_1)


def test_default_schedule_of_the_long_workload():
    """On a 152-SM GB300 the long workload (B 1, T 131072, H 32) takes the
    segmented schedule with the whole-chain state kernel on 32 SMs; the
    full-size parity test then runs it."""
    import kda_chunked_prefill_02_gb300 as K
    q = torch.empty(1, 131072, 32, 128, dtype=torch.bfloat16, device="meta")
    with K.overrides():
        sch = K.prefill_schedule(q)
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("schedule constants are for 152 SMs")
    assert sch["segmented"] and sch["whole_chain"] and sch["prep_ctas"] == 120
    assert sch["scan_segments"] == 0 and sch["segment_chunks"] % 8 == 0


def test_segments_without_programmatic_launch():
    """no_pdl: the prep grids of consecutive segments run strictly one after the
    other; same bits as with the programmatic launch."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(855, B=1, T=64 * 11 + 3, H=3)
    d = inp.to("cuda")
    with K.overrides(segment_chunks=2):
        a = _run(d)
    with K.overrides(segment_chunks=2, no_pdl=True):
        b = _run(d)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("kernel,seg", [("head", 0), ("slab", 0), ("head", 2), ("slab", 2)])
def test_output_tensor_store_into_strided_out(kernel, seg):
    """The state kernels store the output rows by tensor store through a map of
    `out` with the caller's strides: a row-padded out view (token and head
    strides not dense) gets the same bits as a dense one, and the padding
    between rows stays untouched."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(856, B=2, T=64 * 4 + 9, H=3)
    d = inp.to("cuda")
    with K.overrides(state_kernel=kernel, segment_chunks=seg):
        ref, _ = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
        big = torch.full(d.v.shape[:-1] + (128 + 24,), 7.0, dtype=torch.bfloat16, device="cuda")
        out = big[..., :128]
        K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state, out=out)
        torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert bool((big[..., 128:] == 7.0).all())


def test_segmented_call_in_a_cuda_graph():
    """A segmented call captured into a CUDA graph (after one call outside the
    capture created the second stream and its events) replays to the bits of
    the uncaptured segmented call; replaying twice gives the same bits."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(857, B=1, T=64 * 6 + 5, H=2)
    d = inp.to("cuda")
    ws = torch.empty(K.workspace_size(d.q, d.v), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d.v)
    fin = torch.empty_like(d.initial_state)
    with K.overrides(segment_chunks=2):
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state, out=out,
                          final_state=fin, workspace=ws, stream=s)
        torch.cuda.synchronize()
        ref_out, ref_fin = out.clone(), fin.clone()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state, out=out,
                          final_state=fin, workspace=ws, stream=s)
        for _ in range(2):
            out.zero_()
            fin.zero_()
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "segmented call replayed from a CUDA graph")


def test_segments_without_final_state():
    """output_final_state=False: the segments still carry the state between
    them through the workspace; the outputs are those of one pass."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(858, B=2, T=64 * 5 + 3, H=2)
    d = inp.to("cuda")
    with K.overrides(segment_chunks=2):
        out_s, fin_s = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                     output_final_state=False)
        torch.cuda.synchronize()
    with K.overrides(segment_chunks=0):
        out_1, _ = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
        torch.cuda.synchronize()
    assert fin_s is None
    assert torch.equal(out_s, out_1)
