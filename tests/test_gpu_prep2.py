"""GPU checks of the two-CTAs-per-SM prep kernel (KDA_PREP_KERNEL=2): its
per-chunk records equal the one-CTA kernel's bit for bit (same operations in
the same order, inputs read from global memory instead of TMA tiles), and a
whole prefill with it matches the fp64 oracle."""
import os

import pytest
import torch

from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import assert_parity, oracle_prefill

pytestmark = pytest.mark.gpu


class _env:
    def __init__(self, **kv):
        self.kv = kv

    def __enter__(self):
        self.old = {k: os.environ.get(k) for k in self.kv}
        for k, v in self.kv.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = str(v)

    def __exit__(self, *exc):
        for k, v in self.old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def _records(d, kernel, **kw):
    import kda_chunked_prefill_02_gb300 as K
    ws = torch.full((K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    with _env(KDA_PREP_KERNEL=kernel, KDA_SEGMENT_CHUNKS=0):
        K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                      cu_seqlens=d.cu_seqlens, workspace=ws, stage="prep", **kw)
        torch.cuda.synchronize()
    L = K.workspace_layout(d.q, cu_seqlens=d.cu_seqlens)
    H = d.q.shape[-2]
    return ws[L.records:L.records + int(L.max_chunks) * H * int(L.record_bytes)].cpu()


@pytest.mark.parametrize("case", [dict(B=1, T=256, H=2), dict(B=2, T=64 * 3 + 17, H=3),
                                  dict(lengths=[17, 0, 300, 64, 65, 1], H=2),
                                  dict(B=1, T=64 * 40, H=5)])
def test_prep2_records_equal_prep1(case):
    inp = inputs.prefill_inputs(990 + len(case), **case)
    d = inp.to("cuda")
    a = _records(d, "1")
    b = _records(d, "2")
    if d.cu_seqlens is not None:
        # only the records of existing chunks are compared
        nrec = sum(-(-n // 64) for n in inp.lengths) * d.q.shape[-2]
        a, b = a[:nrec * 82432], b[:nrec * 82432]
    if not torch.equal(a, b):
        diff = (a != b).nonzero().flatten()
        first = int(diff[0])
        raise AssertionError("records differ: %d bytes, first at record %d offset %d"
                             % (diff.numel(), first // 82432, first % 82432))


def test_prep2_beta_probabilities_and_scale():
    inp = inputs.prefill_inputs(995, B=1, T=130, H=2)
    d = inp.to("cuda")
    beta = torch.sigmoid(d.beta)
    d2 = type(d)(d.q, d.k, d.v, d.g, beta, d.initial_state, d.cu_seqlens, list(d.lengths))
    a = _records(d2, "1", beta_is_logit=False, scale=0.5)
    b = _records(d2, "2", beta_is_logit=False, scale=0.5)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name,heads", [("varlen", [0, 13, 31]), ("padded", [0, 15])])
def test_prep2_full_size_against_oracle(name, heads):
    from kda_test_util import head_subset
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.config_inputs(name)
    d = inp.to("cuda")
    with _env(KDA_PREP_KERNEL="2", KDA_SEGMENT_CHUNKS=0):
        out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                 cu_seqlens=d.cu_seqlens)
        torch.cuda.synchronize()
    with _env(KDA_PREP_KERNEL="1", KDA_SEGMENT_CHUNKS=0):
        out1, fin1 = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                   cu_seqlens=d.cu_seqlens)
        torch.cuda.synchronize()
    assert torch.equal(out, out1) and torch.equal(fin, fin1)
    sub = head_subset(inp, heads)
    ro, rf = oracle_prefill(sub)
    assert_parity(out[..., heads, :], fin[:, heads], ro, rf, name + " (two-CTA prep)")
