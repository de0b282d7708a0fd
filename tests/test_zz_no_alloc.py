"""The allocation-free prefill entry point, kda_prefill_noalloc.

Some callers of this library cannot allocate device memory at the point where
they run KDA prefill (a device-memory budget owned by another runtime, or a
latency-critical loop where cudaMalloc is not allowed), so they cannot pass a
workspace.  kda_prefill_noalloc runs the same kernels on a scratch array built
into the library.  This test calls it through the C ABI twice in a row, on two
different problems, and checks each result against the workspace-based
kda_prefill with the tolerances the other parity tests use (and bit for bit,
since the same kernels run); it also runs a padded problem in segments (the
segmented schedule keeps its carried state in the scratch too) and checks
that a problem too large for the built-in scratch is refused cleanly.

It sits in a file of its own, collected last, and works both alone in a fresh
process and after the other tests.
"""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import OUT_ATOL, STATE_RTOL, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _both(inp):
    import kda_chunked_prefill_02_gb300 as K
    from kda_chunked_prefill_02_gb300.kda import kda_prefill_noalloc
    d = inp.to("cuda")
    ref_out, ref_fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta,
                                     initial_state=d.initial_state, cu_seqlens=d.cu_seqlens)
    out = torch.full_like(ref_out, float("nan"))
    fin = torch.full_like(ref_fin, float("nan"))
    kda_prefill_noalloc(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                        cu_seqlens=d.cu_seqlens, out=out, final_state=fin)
    torch.cuda.synchronize()
    return ref_out, ref_fin, out, fin


def test_noalloc_matches_workspace_prefill_on_two_calls():
    """Two different problems in a row: each result within the parity
    tolerances of the workspace-based call, and in fact the same bits (the same
    kernels run on the same inputs)."""
    cases = [inputs.prefill_inputs(101, lengths=[300, 0, 77, 1], H=4),
             inputs.prefill_inputs(102, B=2, T=257, H=3)]
    for inp in cases:
        ref_out, ref_fin, out, fin = _both(inp)
        o, r = to_np(out), to_np(ref_out)
        assert abs(o - r).max() <= OUT_ATOL
        assert rel_fro(to_np(fin), to_np(ref_fin)) <= STATE_RTOL
        assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_noalloc_segmented_schedule_within_the_limit():
    """A padded problem near the scratch limit (2048 tokens x 12 heads) run in
    segments: the state carried between segments and the second stream both
    use the built-in scratch; the bits equal the workspace-based call's."""
    import kda_chunked_prefill_02_gb300 as K
    from kda_chunked_prefill_02_gb300.kda import NOALLOC_MAX_WORKSPACE_BYTES
    inp = inputs.prefill_inputs(104, B=1, T=2048, H=12)
    assert K.workspace_size(inp.q, inp.v) <= NOALLOC_MAX_WORKSPACE_BYTES
    for seg in (8, 3):
        with K.overrides(segment_chunks=seg):
            assert K.prefill_schedule(inp.q, num_sms=152)["segmented"]
            ref_out, ref_fin, out, fin = _both(inp)
        assert torch.equal(out, ref_out) and torch.equal(fin, ref_fin)


def test_noalloc_refuses_problems_beyond_its_scratch():
    import kda_chunked_prefill_02_gb300 as K
    from kda_chunked_prefill_02_gb300.kda import (NOALLOC_MAX_WORKSPACE_BYTES, KdaError,
                                                  kda_prefill_noalloc)
    inp = inputs.prefill_inputs(103, B=1, T=4096, H=8)
    d = inp.to("cuda")
    assert K.workspace_size(d.q, d.v) > NOALLOC_MAX_WORKSPACE_BYTES
    out = torch.zeros_like(d.v)
    with pytest.raises(KdaError) as e:
        kda_prefill_noalloc(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state, out=out)
    assert e.value.status == 2  # KDA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert not out.any()        # nothing was launched
