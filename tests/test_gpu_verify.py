"""GPU parity of kda_verify against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import OUT_ATOL, rel_fro, to_np

pytestmark = pytest.mark.gpu


def _run(vi, **kw):
    import kda_chunked_prefill_02_gb300 as K
    d = vi.to("cuda")
    pool = d.state_pool.clone()
    out = K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, slot=d.slot, **kw)
    torch.cuda.synchronize()
    return out, pool


def _check(vi, out, pool, rows=None, **kw):
    R = vi.q.shape[0]
    rows = list(range(R)) if rows is None else list(rows)
    sl = torch.tensor(rows, dtype=torch.int32) if vi.slot is None else vi.slot[rows]
    o_ref, st_ref = oracle.verify(vi.q[rows], vi.k[rows], vi.v[rows], vi.g[rows], vi.beta[rows],
                                  vi.state_pool, vi.accepted[rows], slot=sl, **kw)
    err = np.abs(to_np(out[rows]) - o_ref).max()
    assert err <= OUT_ATOL, err
    slots = np.array(rows) if vi.slot is None else vi.slot[rows].numpy()
    st = to_np(pool[torch.as_tensor(slots).long().cuda()])
    assert rel_fro(st, st_ref) <= 1e-4
    # untouched slots keep their values bit for bit
    untouched = sorted(set(range(vi.state_pool.shape[0])) - set(
        (np.arange(R) if vi.slot is None else vi.slot.numpy()).tolist()))
    if untouched:
        assert torch.equal(pool[untouched].cpu(), vi.state_pool[untouched])


def test_verify_small_with_slots():
    vi = inputs.verify_inputs(11, R=9, D=4, H=3, pool_size=13, permute_slots=True)
    vi.accepted[:3] = torch.tensor([0, 4, 1], dtype=torch.int32)
    out, pool = _run(vi)
    _check(vi, out, pool)


@pytest.mark.parametrize("D", [1, 7, 16])
def test_verify_draft_counts_logit_and_scale(D):
    vi = inputs.verify_inputs(12 + D, R=5, D=D, H=2)
    logit = D != 7
    if not logit:  # beta given as probabilities
        vi.beta = torch.sigmoid(vi.beta)
    out, pool = _run(vi, beta_is_logit=logit, scale=0.5)
    _check(vi, out, pool, beta_is_logit=logit, scale=0.5)


def test_verify_bad_accepted_is_reported_not_faulted():
    import kda_chunked_prefill_02_gb300 as K
    vi = inputs.verify_inputs(21, R=4, D=4, H=2)
    vi.accepted[2] = 9
    d = vi.to("cuda")
    pool = d.state_pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, device_status=status)
    torch.cuda.synchronize()
    assert status.item() == 1
    assert torch.equal(pool[2].cpu(), vi.state_pool[2])   # skipped request untouched


def test_verify_full_config_sampled():
    """256 requests x 4 drafts x 32 heads; oracle on 24 sampled requests."""
    vi = inputs.config_inputs("verify")
    out, pool = _run(vi)
    rows = np.random.default_rng(0).choice(vi.q.shape[0], 24, replace=False)
    _check(vi, out, pool, rows=sorted(rows.tolist()))
