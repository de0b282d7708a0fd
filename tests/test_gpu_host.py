"""GPU checks of kda_prefill_host: prefill with every tensor in page-locked host
memory, copies overlapped with the kernels piece by piece.  Padded pieces carry
each chain's state on the device, so the result must equal the device-buffer
kda_prefill bit for bit; varlen pieces are runs of whole sequences, also
bitwise equal.  Small shapes are also checked against the oracle."""
import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import assert_parity, oracle_prefill

pytestmark = pytest.mark.gpu


def _pinned(t):
    return None if t is None else t.contiguous().pin_memory()


def _both(inp, piece_tokens):
    import kda_chunked_prefill_02_gb300 as K
    d = inp.to("cuda")
    ref_out, ref_fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                     cu_seqlens=d.cu_seqlens)
    hq, hk, hv, hg, hb = (_pinned(t) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    h0 = _pinned(inp.initial_state)
    cu = None if inp.cu_seqlens is None else inp.cu_seqlens.contiguous()
    out, fin = K.kda_prefill_host(hq, hk, hv, hg, hb, initial_state=h0, cu_seqlens=cu,
                                  piece_tokens=piece_tokens)
    torch.cuda.synchronize()
    return ref_out.cpu(), ref_fin.cpu(), out, fin


@pytest.mark.parametrize("B,T,H,piece", [(1, 1000, 4, 256), (3, 777, 2, 128), (2, 64, 3, 0),
                                         (1, 4096, 2, 1024)])
def test_padded_pieces_bitwise_equal_device_call(B, T, H, piece):
    inp = inputs.prefill_inputs(200 + T, B=B, T=T, H=H)
    ref_out, ref_fin, out, fin = _both(inp, piece)
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)


@pytest.mark.parametrize("lengths,piece", [([300, 0, 77, 1, 640], 384), ([17, 0, 16], 0),
                                           ([1500, 20, 900], 512)])
def test_varlen_sequence_groups_bitwise_equal_device_call(lengths, piece):
    inp = inputs.prefill_inputs(300 + sum(lengths), lengths=lengths, H=3)
    ref_out, ref_fin, out, fin = _both(inp, piece)
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)


def test_host_call_matches_oracle():
    inp = inputs.prefill_inputs(401, B=2, T=300, H=2)
    _, _, out, fin = _both(inp, 128)
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "host call")


def test_host_call_refuses_small_staging():
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(402, B=1, T=256, H=2)
    hq, hk, hv, hg, hb = (_pinned(t) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(K.KdaError) as e:
        K.kda_prefill_host(hq, hk, hv, hg, hb, staging=small)
    assert e.value.status == 1


@pytest.mark.parametrize("piece", [16384, 8192])
def test_host_pieces_take_the_segmented_schedule(piece):
    """Long pieces of 32 chains: the device call takes the segmented schedule,
    the host-buffer call's pieces the segmented (16384 tokens) or the one-pass
    (8192) schedule, all with the whole-chain state kernel, the state passing
    between segments and between pieces exactly, so both give the same bits;
    two heads are checked against the oracle."""
    from kda_test_util import head_subset
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(403, B=1, T=16384, H=32)
    with K.overrides(state_kernel="head"):
        assert K.prefill_schedule(inp.q, num_sms=152)["segmented"]
        ref_out, ref_fin, out, fin = _both(inp, piece)
    assert torch.equal(out, ref_out)
    assert torch.equal(fin, ref_fin)
    sub = head_subset(inp, [0, 31])
    ro, rf = oracle_prefill(sub)
    assert_parity(out[:, :, [0, 31]], fin[:, [0, 31]], ro, rf, "segmented host pieces")
