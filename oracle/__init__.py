"""KDA oracle -- TEST INFRASTRUCTURE ONLY.

Plain CPU implementations of what the KDA prefill / verify path computes, used
to check the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py`` (its cpu_baseline leg and ``--impl reference`` arm) may import
this package.  The product package never imports it and shares no code with
it; the only thing both sides use is the seeded input generator module, which
holds none of the method's arithmetic.

Contents
  * ``prefill`` / ``verify``: ctypes wrappers around ``kda_oracle.c``, the
    sequential token-by-token fp64 recurrence
        S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T,
        o_t = scale * S_t^T q_t
    (Kimi Delta Attention as named by the TensorRT-LLM "Kimi K3 KDA prefill"
    page, Description; fp64 oracle practice from the cuDNN-frontend sm90 KDA
    page, Conversation).
  * ``norm.gated_rmsnorm``: the gated RMSNorm of the output (a reading of the
    TensorRT-LLM "Kimi K3 work for Rubin (SM107)" page; formula in norm.py).
  * ``chunked``: an independent numpy fp64 restatement in chunked (WY / UT)
    form, used only to pin the sequential oracle by brute force on tiny inputs
    and to give reference values for per-chunk intermediates.

Parity status: every function here is pinned by tests/test_oracle.py against
hand-evaluated examples, closed forms, exact-retrieval identities, brute force
and invariants; none is "parity unpinned".
"""
import ctypes

import numpy as np

from . import build as _build

_lib = None


def _bind(lib):
    """Declare the C entry points' signatures on a loaded oracle library."""
    d = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    lib.kda_oracle_prefill.restype = ctypes.c_int
    lib.kda_oracle_prefill.argtypes = [i64, i64p, i64, i64, i64, d, d, d, d, d,
                                       ctypes.c_int, ctypes.c_double, d, d, d]
    lib.kda_oracle_verify.restype = ctypes.c_int
    lib.kda_oracle_verify.argtypes = [i64, i64, i64, i64, i64, d, d, d, d, d,
                                      ctypes.c_int, ctypes.c_double, d, i64p, i64p, d, d]
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


def _f64(x):
    """Widen to a C-contiguous float64 numpy array (exact for bf16 / fp32)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        if str(x.dtype) != "torch.float64":
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64))


def _ptr(a, ty=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ty))


def prefill(q, k, v, g, beta, *, cu_seqlens=None, initial_state=None,
            beta_is_logit=True, scale=1.0, return_threads=False):
    """Sequential fp64 KDA prefill.

    Padded mode (cu_seqlens None): q, k, g [B, T, H, K]; v [B, T, H, V];
    beta [B, T, H]; out [B, T, H, V].  Varlen mode: q, k, g [T_total, H, K],
    v [T_total, H, V], beta [T_total, H], cu_seqlens int [N+1].
    initial_state [N, H, K, V] or None (zeros).  Returns (out, final_state)
    as float64 arrays (and the OpenMP thread count if return_threads).
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    if cu_seqlens is None:
        B, T, H, K = q.shape
        cu = np.arange(B + 1, dtype=np.int64) * T
        lead = (B, T)
    else:
        cu = _i64(cu_seqlens)
        H, K = q.shape[1], q.shape[2]
        lead = (q.shape[0],)
    V = v.shape[-1]
    N = cu.shape[0] - 1
    Tt = int(cu[-1])
    qf, kf, gf = (t.reshape(Tt, H, K) for t in (q, k, g))
    vf = v.reshape(Tt, H, V)
    bf = beta.reshape(Tt, H)
    h0 = None if initial_state is None else _f64(initial_state).reshape(N, H, K, V)
    out = np.zeros((Tt, H, V), dtype=np.float64)
    hT = np.zeros((N, H, K, V), dtype=np.float64)
    used = _load().kda_oracle_prefill(
        N, _ptr(cu, ctypes.c_int64), H, K, V, _ptr(qf), _ptr(kf), _ptr(vf), _ptr(gf), _ptr(bf),
        int(bool(beta_is_logit)), float(scale),
        _ptr(h0) if h0 is not None else None, _ptr(out), _ptr(hT))
    out = out.reshape(*lead, H, V)
    if return_threads:
        return out, hT, used
    return out, hT


def verify(q, k, v, g, beta, state_pool, accepted, *, slot=None, beta_is_logit=True,
           scale=1.0, return_threads=False):
    """Sequential fp64 MTP verify.

    q, k, g [R, D, H, K]; v [R, D, H, V]; beta [R, D, H]; state_pool
    [P, H, K, V]; accepted int [R] in 0..D; slot int [R] or None (= r).
    Returns (out [R, D, H, V], stored_state [R, H, K, V]).
    """
    q, k, v, g, beta, pool = (_f64(t) for t in (q, k, v, g, beta, state_pool))
    R, D, H, K = q.shape
    V = v.shape[-1]
    acc = _i64(accepted)
    sl = None if slot is None else _i64(slot)
    out = np.zeros((R, D, H, V), dtype=np.float64)
    pool_out = np.zeros((R, H, K, V), dtype=np.float64)
    used = _load().kda_oracle_verify(
        R, D, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
        int(bool(beta_is_logit)), float(scale), _ptr(pool),
        _ptr(sl, ctypes.c_int64) if sl is not None else None, _ptr(acc, ctypes.c_int64),
        _ptr(out), _ptr(pool_out))
    if return_threads:
        return out, pool_out, used
    return out, pool_out
