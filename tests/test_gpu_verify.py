"""GPU parity of kda_verify against the fp64 oracle (through the C ABI), for
both kernels: the sequential one (every draft on the CUDA cores in fp32; the
stored state within 1e-4 relative Frobenius of the oracle's) and the
tensor-core one (the drafts as one WY-form chunk with tf32 products and an
fp32 state update; within 2e-3, which is about the tf32 rounding of the
state-dependent terms, 2^-11 relative, accumulated over the 128-term products
and the chunk's drafts)."""
import contextlib

import numpy as np
import pytest
import torch

import oracle
from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import OUT_ATOL, rel_fro, to_np

pytestmark = pytest.mark.gpu

KERNELS = ["sequential", "tensor"]
STATE_TOL = {"sequential": 1e-4, "tensor": 2e-3, None: 2e-3}
_kernel = None   # the kernel the current test runs (None: the library's choice)


def _ctx():
    import kda_chunked_prefill_02_gb300 as K
    return K.overrides(verify_kernel=_kernel) if _kernel else contextlib.nullcontext()


@pytest.fixture(params=KERNELS)
def kernel(request):
    global _kernel
    _kernel = request.param
    yield request.param
    _kernel = None


def _run(vi, **kw):
    import kda_chunked_prefill_02_gb300 as K
    d = vi.to("cuda")
    pool = d.state_pool.clone()
    with _ctx():
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
    assert rel_fro(st, st_ref) <= STATE_TOL[_kernel], rel_fro(st, st_ref)
    # untouched slots keep their values bit for bit
    untouched = sorted(set(range(vi.state_pool.shape[0])) - set(
        (np.arange(R) if vi.slot is None else vi.slot.numpy()).tolist()))
    if untouched:
        assert torch.equal(pool[untouched].cpu(), vi.state_pool[untouched])


def test_verify_small_with_slots(kernel):
    vi = inputs.verify_inputs(11, R=9, D=4, H=3, pool_size=13, permute_slots=True)
    vi.accepted[:3] = torch.tensor([0, 4, 1], dtype=torch.int32)
    out, pool = _run(vi)
    _check(vi, out, pool)


@pytest.mark.parametrize("D", [1, 4, 7, 8, 16])
def test_verify_draft_counts_logit_and_scale(kernel, D):
    vi = inputs.verify_inputs(12 + D, R=5, D=D, H=2)
    logit = D != 7
    if not logit:  # beta given as probabilities
        vi.beta = torch.sigmoid(vi.beta)
    out, pool = _run(vi, beta_is_logit=logit, scale=0.5)
    _check(vi, out, pool, beta_is_logit=logit, scale=0.5)


def test_verify_bad_accepted_is_reported_not_faulted(kernel):
    import kda_chunked_prefill_02_gb300 as K
    vi = inputs.verify_inputs(21, R=4, D=4, H=2)
    vi.accepted[2] = 9
    d = vi.to("cuda")
    pool = d.state_pool.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with _ctx():
        K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted, device_status=status)
    torch.cuda.synchronize()
    assert status.item() == 1
    assert torch.equal(pool[2].cpu(), vi.state_pool[2])   # skipped request untouched


@pytest.mark.parametrize("D", [4, 8, 16])
def test_verify_full_config(kernel, D):
    """256 requests x D drafts x 32 heads (the verify workload at D = 4; the
    same draw at 8 and 16 drafts): every request against the oracle (outputs
    element by element, the stored state of every request and head)."""
    vi = inputs.config_inputs("verify") if D == 4 else inputs.verify_inputs(4, R=256, D=D, H=32)
    out, pool = _run(vi)
    _check(vi, out, pool)
    o_ref, st_ref = oracle.verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted,
                                  slot=vi.slot)
    og = to_np(out)
    per_req = np.abs(og - o_ref).reshape(og.shape[0], -1).max(1)
    print("verify %s D=%d: worst out max-abs %.3e (request %d)" % (kernel, D, per_req.max(),
                                                                 int(per_req.argmax())))


def _bf16_case(seed, R=6, D=4, H=2, **kw):
    vi = inputs.verify_inputs(seed, R=R, D=D, H=H, **kw)
    vi.state_pool = vi.state_pool.to(torch.bfloat16).float()  # the pool's exact values
    return vi


def test_verify_bf16_pool(kernel):
    """bf16 state pool: read widened exactly, drafts in fp32, state written back
    rounded to nearest even.  Outputs against the oracle run from the same bf16
    values; the stored state within a bf16 rounding of the oracle's."""
    import kda_chunked_prefill_02_gb300 as K
    vi = _bf16_case(31, permute_slots=True, pool_size=9)
    d = vi.to("cuda")
    pool = d.state_pool.to(torch.bfloat16)
    with _ctx():
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
def test_verify_replay_only_commits_the_accepted_drafts(kernel, bf16):
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
    with _ctx():
        K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool_a, d.accepted)
        assert K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool_b, d.accepted, replay_only=True) is None
    torch.cuda.synchronize()
    assert torch.equal(pool_a, pool_b)
    _, st_ref = oracle.verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted)
    assert rel_fro(to_np(pool_b[:vi.q.shape[0]]), st_ref) <= (1e-2 if bf16 else STATE_TOL[kernel])


def test_verify_no_requests(kernel):
    """R = 0 requests: the call succeeds, writes nothing and leaves the pool."""
    import kda_chunked_prefill_02_gb300 as K
    vi = inputs.verify_inputs(41, R=3, D=4, H=2)
    d = vi.to("cuda")
    pool = d.state_pool.clone()
    with _ctx():
        out = K.kda_verify(d.q[:0], d.k[:0], d.v[:0], d.g[:0], d.beta[:0], pool, d.accepted[:0])
    torch.cuda.synchronize()
    assert out.shape == (0, 4, 2, 128)
    assert torch.equal(pool.cpu(), vi.state_pool)


def test_verify_kernels_agree_and_extreme_gates():
    """Both kernels on the same draws, including gates far below the
    production bound (-20 and -1e4, which empty a key row in one draft) and
    zero gates: each within its tolerance of the oracle, so within the sum of
    them of each other; no non-finite value anywhere."""
    import kda_chunked_prefill_02_gb300 as K
    global _kernel
    vi = inputs.verify_inputs(61, R=6, D=12, H=3)
    vi.g[0, 3] = -1e4
    vi.g[1, :, 1] = -20.0
    vi.g[2] = 0.0
    vi.accepted[:4] = torch.tensor([12, 5, 1, 9], dtype=torch.int32)
    res = {}
    for kern in KERNELS:
        _kernel = kern
        try:
            out, pool = _run(vi)
        finally:
            _kernel = None
        assert torch.isfinite(out.float()).all() and torch.isfinite(pool).all()
        res[kern] = (out, pool)
        _kernel = kern
        try:
            _check(vi, out, pool)
        finally:
            _kernel = None
    d = (res["sequential"][0].float() - res["tensor"][0].float()).abs().max().item()
    assert d <= 2 * OUT_ATOL


def test_verify_default_kernel_choice():
    """The library takes the sequential kernel for every draft count up to 16
    (measured faster on GB300 than the tensor-core kernel there); the tensor-core
    kernel runs when a call's overrides ask for it."""
    import kda_chunked_prefill_02_gb300 as K
    for D, kern in ((4, "sequential"), (8, "sequential"), (16, "sequential")):
        vi = inputs.verify_inputs(70 + D, R=3, D=D, H=2)
        d = vi.to("cuda")
        outs = {}
        for name in (None, kern):
            pool = d.state_pool.clone()
            with (K.overrides(verify_kernel=name) if name else contextlib.nullcontext()):
                outs[name] = (K.kda_verify(d.q, d.k, d.v, d.g, d.beta, pool, d.accepted), pool)
        torch.cuda.synchronize()
        assert torch.equal(outs[None][0], outs[kern][0]) and torch.equal(outs[None][1], outs[kern][1])
