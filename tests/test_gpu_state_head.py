"""GPU parity of the one-CTA-per-chain state kernel (all 128 value columns per
CTA), forced through the call's overrides on shapes where the default would pick
the 32-column slab kernel: against the fp64 oracle, and against the slab
kernel on the same inputs (same chunk step, same MMA K order)."""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import assert_parity, gpu_prefill, oracle_prefill

pytestmark = pytest.mark.gpu


def _with_kernel(name, inp):
    import kda_chunked_prefill_02_gb300 as K
    with K.overrides(state_kernel=name):
        out, fin = gpu_prefill(inp)
        torch.cuda.synchronize()
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("case", [dict(B=1, T=256, H=2), dict(B=2, T=1000, H=3),
                                  dict(lengths=[17, 0, 16], H=2), dict(lengths=[1025, 0, 31], H=2),
                                  dict(lengths=[1, 64, 65, 127, 128, 129], H=2)])
def test_head_kernel_matches_oracle_and_slab_kernel(case):
    inp = inputs.prefill_inputs(500 + sum(case.get("lengths", [case.get("T", 0)])), **case)
    out_h, fin_h = _with_kernel("head", inp)
    out_s, fin_s = _with_kernel("slab", inp)
    ro, rf = oracle_prefill(inp)
    assert_parity(out_h, fin_h, ro, rf, "head kernel")
    assert (out_h.float() - out_s.float()).abs().max().item() <= 1e-2
    assert torch.allclose(fin_h, fin_s, rtol=1e-4, atol=1e-6)


def test_head_kernel_zero_initial_state_and_continuation():
    inp = inputs.prefill_inputs(561, B=1, T=300, H=2, init_std=None)
    out_h, fin_h = _with_kernel("head", inp)
    ro, rf = oracle_prefill(inp)
    assert_parity(out_h, fin_h, ro, rf, "head kernel, zero initial state")
