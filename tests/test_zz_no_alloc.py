"""The allocation-free prefill entry point, kda_prefill_noalloc.

Some callers of this library cannot allocate device memory at the point where
they run KDA prefill (a device-memory budget owned by another runtime, or a
latency-critical loop where cudaMalloc is not allowed), so they cannot pass a
workspace.  kda_prefill_noalloc runs the same kernels on a scratch array built
into the library.  This test calls it through the C ABI twice in a row, on two
different problems, and checks each result against the workspace-based
kda_prefill with the tolerances the other parity tests use; it also checks that
a problem too large for the built-in scratch is refused cleanly.

It sits in a file of its own, collected last, and works both alone in a fresh
process and after the other tests.
"""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import OUT_ATOL, STATE_RTOL, rel_fro, to_np

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_prefill_on_two_calls():
    import kda_chunked_prefill_02_gb300 as K
    from kda_chunked_prefill_02_gb300.kda import kda_prefill_noalloc
    cases = [inputs.prefill_inputs(101, lengths=[300, 0, 77, 1], H=4),
             inputs.prefill_inputs(102, B=2, T=257, H=3)]
    for inp in cases:
        d = inp.to("cuda")
        ref_out, ref_fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta,
                                         initial_state=d.initial_state, cu_seqlens=d.cu_seqlens)
        out = torch.full_like(ref_out, float("nan"))
        fin = torch.full_like(ref_fin, float("nan"))
        kda_prefill_noalloc(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                            cu_seqlens=d.cu_seqlens, out=out, final_state=fin)
        torch.cuda.synchronize()
        o, r = to_np(out), to_np(ref_out)
        assert abs(o - r).max() <= OUT_ATOL
        assert rel_fro(to_np(fin), to_np(ref_fin)) <= STATE_RTOL


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
