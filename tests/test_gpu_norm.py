"""GPU parity of the gated RMSNorm fused into the state pass's output epilogue
(out = o / sqrt(mean_c o_c^2 + eps) * w * sigmoid(gate), per token and head)
against the fp64 oracle: the sequential recurrence's outputs followed by
oracle.norm.gated_rmsnorm."""
import numpy as np
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import STATE_RTOL, assert_norm_close, oracle_prefill, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _case(inp, seed, eps):
    import kda_chunked_prefill_02_gb300 as K
    from oracle.norm import gated_rmsnorm
    gen = torch.Generator().manual_seed(seed)
    gate = (torch.randn(inp.v.shape, generator=gen) * 2).to(torch.bfloat16)
    w = (torch.rand(128, generator=gen) + 0.5).float()
    d = inp.to("cuda")
    # the plain call on the kernel the norm takes (the whole-chain kernel)
    with K.overrides(state_kernel="head"):
        plain_out, plain_fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                             cu_seqlens=d.cu_seqlens)
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                             cu_seqlens=d.cu_seqlens, out_gate=gate.cuda(), norm_weight=w.cuda(),
                             norm_eps=eps)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(inp)
    g64, w64 = gate.float().numpy(), w.numpy()
    # 1) the norm itself, on the same kernel's unnormalised output
    assert_norm_close(to_np(out), gated_rmsnorm(to_np(plain_out), g64, w64, eps))
    # 2) against the oracle end to end; rows of small RMS amplify the recurrence's
    # own (separately tested) error, so the whole tensor is compared relatively
    ref = gated_rmsnorm(ro, g64, w64, eps)
    assert rel_fro(to_np(out), ref) <= 2e-2
    assert rel_fro(to_np(fin), rf) <= STATE_RTOL
    # the state pass is the same: the final state does not depend on the norm
    assert torch.equal(fin, plain_fin)


@pytest.mark.parametrize("case", [dict(B=1, T=256, H=2), dict(B=2, T=200, H=3),
                                  dict(lengths=[17, 0, 16, 130], H=2)])
def test_fused_norm_matches_oracle(case):
    inp = inputs.prefill_inputs(600 + sum(case.get("lengths", [case.get("T", 0)])), **case)
    _case(inp, 7, 1e-6)


def test_fused_norm_large_eps():
    inp = inputs.prefill_inputs(611, B=1, T=130, H=2)
    _case(inp, 8, 0.5)


def test_fused_norm_needs_both_operands():
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(612, B=1, T=64, H=2)
    d = inp.to("cuda")
    gate = torch.zeros(d.v.shape, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(K.KdaError) as e:
        from kda_chunked_prefill_02_gb300.kda import _prefill_args, lib, _check, _stream_handle, workspace_size
        import ctypes
        out = torch.empty_like(d.v)
        ws = torch.empty(workspace_size(d.q, d.v), dtype=torch.uint8, device="cuda")
        a = _prefill_args(d.q, d.k, d.v, d.g, d.beta, None, None, out, None, True, 1.0, ws, None, 64)
        a.out_gate = ctypes.c_void_p(gate.data_ptr())
        a.gate_stride = a.out_stride
        _check(lib().kda_prefill(ctypes.byref(a), _stream_handle(None)))
    assert e.value.status == 1
