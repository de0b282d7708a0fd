"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same seeded inputs (optionally on a subset of heads or
sequences), and compare within the stated tolerances:
  out: max |gpu - oracle| <= 2e-2 (bf16 outputs)
  final state: ||gpu - oracle||_F / ||oracle||_F <= 1e-2 (fp32 state)
"""
import numpy as np
import torch

OUT_ATOL = 2e-2
STATE_RTOL = 1e-2


def to_np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def gpu_prefill(inp, **kw):
    import kda_chunked_prefill_02_gb300 as K
    d = inp.to("cuda")
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                             cu_seqlens=d.cu_seqlens, **kw)
    torch.cuda.synchronize()
    return out, fin


def head_subset(inp, heads):
    """The same inputs restricted to the given heads (for the oracle)."""
    from kda_chunked_prefill_02_gb300.inputs import PrefillInputs
    h = list(heads)
    sel = lambda t: t[..., h, :]
    return PrefillInputs(sel(inp.q), sel(inp.k), sel(inp.v), sel(inp.g), inp.beta[..., h],
                         None if inp.initial_state is None else inp.initial_state[:, h],
                         inp.cu_seqlens, list(inp.lengths))


def oracle_prefill(inp, **kw):
    import oracle
    return oracle.prefill(inp.q, inp.k, inp.v, inp.g, inp.beta, cu_seqlens=inp.cu_seqlens,
                          initial_state=inp.initial_state, **kw)


def rel_fro(a, b):
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def assert_parity(out_gpu, fin_gpu, out_ref, fin_ref, what=""):
    og = to_np(out_gpu)
    err = np.abs(og - out_ref).max() if og.size else 0.0
    assert np.isfinite(og).all(), "%s: non-finite outputs" % what
    assert err <= OUT_ATOL, "%s: out max-abs error %.3e > %.1e" % (what, err, OUT_ATOL)
    if fin_gpu is not None:
        fg = to_np(fin_gpu)
        rf = rel_fro(fg, fin_ref)
        assert np.isfinite(fg).all(), "%s: non-finite final state" % what
        assert rf <= STATE_RTOL, "%s: final-state rel Frobenius %.3e > %.1e" % (what, rf, STATE_RTOL)
    return err


def assert_norm_close(out, same):
    """The kernel normalises fp32 o and rounds the result to bf16; `same`
    normalises the bf16-rounded o in fp64.  Each rounding is at most 2^-8 of
    the value, and a relative change of o moves the normalised value by at most
    about twice as much, so the two differ by at most about 1.2 % of the
    output (+ a little absolute slack for values near zero)."""
    err = np.abs(out - same) - (1.6e-2 * np.abs(same) + 2e-3)
    assert err.max() <= 0, float(err.max())
