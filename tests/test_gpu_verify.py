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


def test_verify_full_config():
    """256 requests x 4 drafts x 32 heads: every request against the oracle
    (outputs element by element, the stored state of every request and head)."""
    vi = inputs.config_inputs("verify")
    out, pool = _run(vi)
    _check(vi, out, pool)
    o_ref, st_ref = oracle.verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted,
                                  slot=vi.slot)
    og = to_np(out)
    per_req = np.abs(og - o_ref).reshape(og.shape[0], -1).max(1)
    print("verify: worst out max-abs %.3e (request %d)" % (per_req.max(), int(per_req.argmax())))


def _bf16_case(seed, R=6, D=4, H=2, **kw):
    vi = inputs.verify_inputs(seed, R=R, D=D, H=H, **kw)
    vi.state_pool = vi.state_pool.to(torch.bfloat16).float()  # the pool's exact values
    return vi


def test_verify_bf16_pool():
    """bf16 state pool: read widened exactly, drafts in fp32, state written back
    rounded to nearest even.  Outputs against the oracle run from the same bf16
    values; the stored state within a bf16 rounding of the oracle's."""
    import kda_chunked_prefill_02_gb300 as K
    vi = _bf16_case(31, permute_slots=True, pool_size=9)
    d = vi.to("cuda")
    pool = d.state_pool.to(torch.bfloat16)
    out = K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, slot=d.slot)
    torch.cuda.synchronize()
    rows = list(range(vi.q.shape[0]))
    o_ref, st_ref = oracle.verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted,
                                  slot=vi.slot)
    assert np.abs(to_np(out) - o_ref).max() <= OUT_ATOL
    st = to_np(pool[vi.slot.long().cuda()])
    assert rel_fro(st, st_ref) <= 1e-2
    # the written states are the bf16 rounding of a state within tolerance; untouched
    # rows (accepted 0) keep their bits
    for r in rows:
        if vi.accepted[r] == 0:
            assert torch.equal(pool[int(vi.slot[r])].cpu(), vi.state_pool[int(vi.slot[r])].to(torch.bfloat16))


@pytest.mark.parametrize("bf16", [False, True])
def test_verify_replay_only_commits_the_accepted_drafts(bf16):
    """Replay-only: only the first accepted[r] drafts run, nothing but the state
    is written (out is not touched), and the state equals the one a normal
    verify stores."""
    import kda_chunked_prefill_02_gb300 as K
    vi = _bf16_case(41, R=7) if bf16 else inputs.verify_inputs(41, R=7, D=4, H=2)
    vi.accepted[:3] = torch.tensor([0, 4, 2], dtype=torch.int32)
    d = vi.to("cuda")
    dt = torch.bfloat16 if bf16 else torch.float32
    pool_a = d.state_pool.to(dt).clone()   # .to() returns the tensor itself when dt matches
    pool_b = d.state_pool.to(dt).clone()
    K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool_a, d.accepted)
    assert K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool_b, d.accepted, replay_only=True) is None
    torch.cuda.synchronize()
    assert torch.equal(pool_a, pool_b)
    _, st_ref = oracle.verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted)
    assert rel_fro(to_np(pool_b[:vi.q.shape[0]]), st_ref) <= (1e-2 if bf16 else 1e-4)


def test_verify_no_requests():
    """R = 0 requests: the call succeeds, writes nothing and leaves the pool."""
    import kda_chunked_prefill_02_gb300 as K
    vi = inputs.verify_inputs(41, R=3, D=4, H=2)
    d = vi.to("cuda")
    pool = d.state_pool.clone()
    out = K.kda_verify(d.q[:0], d.k[:0], d.v[:0], d.g[:0], d.beta[:0], pool, d.accepted[:0])
    torch.cuda.synchronize()
    assert out.shape == (0, 4, 2, 128)
    assert torch.equal(pool.cpu(), vi.state_pool)
