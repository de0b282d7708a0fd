"""Chunked (WY / UT) restatement of the KDA recurrence in numpy fp64.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  A second, independent
derivation of the same function as the sequential oracle, written from the
algebra rather than from the token loop.  Used (a) to pin the sequential
oracle by brute force on tiny inputs and (b) to give reference values for the
per-chunk intermediates that the CUDA path materialises.

For one chain (sequence, head) and one chunk of C tokens with entry state S0
(K x V), with beta already a probability:

  Gam[i]  = sum_{t<=i} g_t                       (in-chunk inclusive gate cumsum:
                                                  the "prefix row" of the
                                                  TensorRT-LLM K1 scan, page 1)
  gam     = Gam[C-1]                              (the "chunk total")
  A'[i,j] = sum_c k_i[c] k_j[c] exp(Gam_i[c] - Gam_j[c])      j < i
  A       = Diag(beta) * strict_lower(A')
  T       = (I + A)^{-1}                          (UT transform; dense solve here)
  W       = T Diag(beta) (K * exp(Gam))
  U       = T Diag(beta) V
  Vnew    = U - W S0
  Aqk[i,j]= sum_c q_i[c] k_j[c] exp(Gam_i[c] - Gam_j[c])      j <= i
  O       = (Q * exp(Gam)) S0 + Aqk Vnew
  S1      = Diag(exp gam) S0 + (K * exp(gam - Gam))^T Vnew

Derivation: unrolling S_t = S'_t + k_t u_t^T with S'_t = Diag(exp g_t) S_{t-1}
and u_t = beta_t (v_t - S'_t^T k_t) over the chunk gives
(I + A) Vnew = Diag(beta) V - Diag(beta)(K * exp Gam) S0, i.e. Vnew = U - W S0.

Exponents are only evaluated for j <= i (Gam_i - Gam_j <= 0), so no term
overflows; meant for tiny inputs only.
"""
import numpy as np


def _sigmoid(b):
    return 1.0 / (1.0 + np.exp(-b))


def _decay_pair(Gam, inclusive):
    """exp(Gam_i[c] - Gam_j[c]) for j <= i (inclusive) or j < i, else 0. [C,C,K]"""
    C = Gam.shape[0]
    diff = Gam[:, None, :] - Gam[None, :, :]
    ii = np.arange(C)[:, None]
    jj = np.arange(C)[None, :]
    mask = (jj <= ii) if inclusive else (jj < ii)
    return np.exp(np.where(mask[:, :, None], diff, -np.inf))


def chunk_step(S0, q, k, v, g, beta):
    """One chunk.  q,k,g [C,K]; v [C,V]; beta [C] (probabilities); S0 [K,V].

    Returns a dict with O [C,V], S1 [K,V] and the intermediates Gam, gam,
    A (beta-scaled strict lower), T, W, U, Vnew, Aqk, Qt (= Q e^Gam),
    Kh (= K e^{gam-Gam}), Qp (= Qt - Aqk W), Oloc (= Aqk U).
    """
    C = q.shape[0]
    Gam = np.cumsum(g, axis=0)
    gam = Gam[-1]
    Ap = np.einsum("ic,jc,ijc->ij", k, k, _decay_pair(Gam, inclusive=False))
    A = beta[:, None] * Ap
    T = np.linalg.solve(np.eye(C) + A, np.eye(C))
    Tb = T * beta[None, :]
    W = Tb @ (k * np.exp(Gam))
    U = Tb @ v
    Vnew = U - W @ S0
    Aqk = np.einsum("ic,jc,ijc->ij", q, k, _decay_pair(Gam, inclusive=True))
    Qt = q * np.exp(Gam)
    O = Qt @ S0 + Aqk @ Vnew
    Kh = k * np.exp(gam[None, :] - Gam)
    S1 = np.exp(gam)[:, None] * S0 + Kh.T @ Vnew
    return dict(O=O, S1=S1, Gam=Gam, gam=gam, A=A, T=T, W=W, U=U, Vnew=Vnew, Aqk=Aqk,
                Qt=Qt, Kh=Kh, Qp=Qt - Aqk @ W, Oloc=Aqk @ U)


def prefill_chunked(q, k, v, g, b, *, cu_seqlens, initial_state=None, beta_is_logit=True,
                    scale=1.0, chunk=64):
    """Chunked fp64 KDA prefill over packed sequences (varlen layout).

    q,k,g [T_total,H,K]; v [T_total,H,V]; b [T_total,H]; cu_seqlens [N+1].
    Returns (out [T_total,H,V], final [N,H,K,V]).
    """
    q = np.asarray(q, np.float64) * scale
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g = np.asarray(g, np.float64)
    b = np.asarray(b, np.float64)
    beta = _sigmoid(b) if beta_is_logit else b
    cu = np.asarray(cu_seqlens, np.int64)
    N = cu.shape[0] - 1
    Tt, H, K = q.shape
    V = v.shape[-1]
    out = np.zeros((Tt, H, V))
    final = np.zeros((N, H, K, V))
    for n in range(N):
        for h in range(H):
            S = np.zeros((K, V)) if initial_state is None else np.array(
                initial_state[n, h], dtype=np.float64)
            for t0 in range(int(cu[n]), int(cu[n + 1]), chunk):
                t1 = min(t0 + chunk, int(cu[n + 1]))
                r = chunk_step(S, q[t0:t1, h], k[t0:t1, h], v[t0:t1, h], g[t0:t1, h],
                               beta[t0:t1, h])
                out[t0:t1, h] = r["O"]
                S = r["S1"]
            final[n, h] = S
    return out, final
