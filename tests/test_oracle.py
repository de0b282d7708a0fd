"""Pins for the fp64 KDA oracle (CPU only).

Each test checks the sequential oracle against something other than itself:
hand-evaluated examples, closed forms, exact-retrieval identities, brute force
in an independently derived chunked form, and structural invariants.  The set
is chosen so that a plausible slip in the oracle (dropped decay, decay on the
wrong axis, wrong sign in the delta, S k instead of S^T k, reading the state
before instead of after the write, a missing beta, the sigmoid on the wrong
side) fails at least one of them.
"""
import json
import os

import numpy as np

from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, T, H, K, V, gate=5.0, norm=True):
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    if norm:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, V))
    g = -gate / (1.0 + np.exp(-rng.standard_normal((T, H, K))))
    b = rng.standard_normal((T, H))
    return q, k, v, g, b


def _basis_keys(rng, T, K):
    """Signed standard basis vectors in distinct channels: exactly orthonormal."""
    perm = rng.permutation(K)[:T]
    sign = rng.choice([-1.0, 1.0], size=T)
    k = np.zeros((T, K))
    k[np.arange(T), perm] = sign
    return k


def test_hand_examples(oracle):
    """Hand-evaluated rational examples (tests/golden/hand_examples.json)."""
    with open(os.path.join(GOLDEN, "hand_examples.json")) as f:
        ex = json.load(f)["examples"]
    for e in ex:
        K, V = e["K"], e["V"]
        T = len(e["beta"])
        q = np.array(e["q"], float).reshape(T, 1, K)
        k = np.array(e["k"], float).reshape(T, 1, K)
        v = np.array(e["v"], float).reshape(T, 1, V)
        g = np.array(e["g"], float).reshape(T, 1, K)
        b = np.array(e["beta"], float).reshape(T, 1)
        S0 = np.array(e["S0"], float).reshape(1, 1, K, V)
        out, fin = oracle.prefill(q, k, v, g, b, cu_seqlens=[0, T], initial_state=S0,
                                  beta_is_logit=False)
        np.testing.assert_allclose(out.reshape(T, V), np.array(e["out"]), rtol=0, atol=1e-14)
        np.testing.assert_allclose(fin.reshape(K, V), np.array(e["final"]), rtol=0, atol=1e-14)


def test_beta_zero_gate_zero_identity(oracle):
    """beta = 0 and g = 0 leave the state untouched: o_t = scale * S0^T q_t."""
    rng = np.random.default_rng(1)
    T, H, K, V = 37, 2, 8, 5
    q, k, v, _, _ = _rand(rng, T, H, K, V)
    S0 = rng.standard_normal((1, H, K, V))
    out, fin = oracle.prefill(q, k, v, np.zeros((T, H, K)), np.zeros((T, H)), cu_seqlens=[0, T],
                              initial_state=S0, beta_is_logit=False, scale=0.5)
    np.testing.assert_array_equal(fin, S0)
    np.testing.assert_allclose(out, 0.5 * np.einsum("hkv,thk->thv", S0[0], q), atol=1e-13)


def test_beta_zero_pure_decay_closed_form(oracle):
    """beta = 0: S_t = Diag(exp(sum_{s<=t} g_s)) S0 (decay acts on key rows)."""
    rng = np.random.default_rng(2)
    T, H, K, V = 29, 3, 8, 5          # K != V: decaying the wrong axis cannot pass
    q, k, v, g, _ = _rand(rng, T, H, K, V, gate=0.3)
    S0 = rng.standard_normal((1, H, K, V))
    out, fin = oracle.prefill(q, k, v, g, np.zeros((T, H)), cu_seqlens=[0, T],
                              initial_state=S0, beta_is_logit=False)
    dec = np.exp(np.cumsum(g, axis=0))                     # [T,H,K]
    St = dec[..., None] * S0[0][None]                      # [T,H,K,V]
    np.testing.assert_allclose(out, np.einsum("thkv,thk->thv", St, q), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fin[0], St[-1], rtol=1e-12, atol=1e-14)


def test_exact_retrieval_orthonormal_keys(oracle):
    """g = 0, beta = 1, exactly orthonormal keys, S0 = 0: querying with k_j at
    any t >= j returns v_j exactly."""
    rng = np.random.default_rng(3)
    T, K, V = 48, 128, 128
    k = _basis_keys(rng, T, K)
    v = rng.standard_normal((T, V))
    jq = np.array([rng.integers(0, t + 1) for t in range(T)])
    q = k[jq]
    out, fin = oracle.prefill(q[:, None], k[:, None], v[:, None], np.zeros((T, 1, K)),
                              np.ones((T, 1)), cu_seqlens=[0, T], beta_is_logit=False)
    np.testing.assert_array_equal(out[:, 0], v[jq])
    np.testing.assert_array_equal(fin[0, 0], k.T @ v)


def test_retrieval_overwrites_nonzero_state(oracle):
    """beta = 1 and a unit key: right after the write S_t^T k_t = v_t, whatever
    the prior state and gate (the delta rule replaces what the key retrieved)."""
    rng = np.random.default_rng(4)
    T, K, V = 20, 32, 12
    k = _basis_keys(rng, T, K)
    v = rng.standard_normal((T, V))
    g = -rng.uniform(0, 3, (T, K))
    S0 = rng.standard_normal((1, 1, K, V))
    out, _ = oracle.prefill(k[:, None], k[:, None], v[:, None], g[:, None], np.ones((T, 1)),
                            cu_seqlens=[0, T], initial_state=S0, beta_is_logit=False)
    np.testing.assert_allclose(out[:, 0], v, rtol=0, atol=1e-14)


def test_matrix_definition_form(oracle):
    """The literal matrix form (I - b k k^T) Diag(e^g) S + b k v^T, o = S^T q."""
    rng = np.random.default_rng(5)
    T, H, K, V = 23, 2, 7, 4
    q, k, v, g, b = _rand(rng, T, H, K, V, gate=1.0)
    S0 = rng.standard_normal((1, H, K, V))
    out, fin = oracle.prefill(q, k, v, g, b, cu_seqlens=[0, T], initial_state=S0)
    beta = 1.0 / (1.0 + np.exp(-b))
    for h in range(H):
        S = S0[0, h].copy()
        for t in range(T):
            kk = k[t, h][:, None]
            S = (np.eye(K) - beta[t, h] * kk @ kk.T) @ np.diag(np.exp(g[t, h])) @ S \
                + beta[t, h] * kk @ v[t, h][None, :]
            np.testing.assert_allclose(out[t, h], S.T @ q[t, h], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(fin[0, h], S, rtol=1e-11, atol=1e-12)


def test_scalar_closed_form_with_sigmoid(oracle):
    """K = V = 1: s_t = (1 - beta k^2) e^g s_{t-1} + beta k v with beta = sigmoid(b),
    checked against the unrolled form prod(a) s0 + sum_j (prod_{r>j} a_r) c_j."""
    rng = np.random.default_rng(6)
    T = 40
    k, v, q = rng.standard_normal(T), rng.standard_normal(T), rng.standard_normal(T)
    g = -rng.uniform(0, 1, T)
    b = rng.standard_normal(T)
    s0 = 0.7
    beta = 1.0 / (1.0 + np.exp(-b))
    a = (1 - beta * k * k) * np.exp(g)
    c = beta * k * v
    s = np.array([np.prod(a[:t + 1]) * s0 + sum(np.prod(a[j + 1:t + 1]) * c[j]
                                                for j in range(t + 1)) for t in range(T)])
    out, fin = oracle.prefill(q[:, None, None], k[:, None, None], v[:, None, None],
                              g[:, None, None], b[:, None], cu_seqlens=[0, T],
                              initial_state=np.full((1, 1, 1, 1), s0))
    np.testing.assert_allclose(out[:, 0, 0], s * q, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(fin.ravel()[0], s[-1], rtol=1e-11)


def test_chunked_form_equals_sequential(oracle):
    """Brute force: the independently derived chunked (WY/UT) form with a dense
    solve equals the token loop, for many chunk sizes, K=V in {8,128}, and
    varlen batches with an empty and a length-1 sequence."""
    rng = np.random.default_rng(7)
    for K, V, lens in [(8, 8, [37, 0, 1, 50]), (128, 128, [70, 0, 1, 9])]:
        Tt, H = sum(lens), 2
        cu = np.concatenate([[0], np.cumsum(lens)])
        q, k, v, g, b = _rand(rng, Tt, H, K, V)
        S0 = 0.1 * rng.standard_normal((len(lens), H, K, V))
        ref_out, ref_fin = oracle.prefill(q, k, v, g, b, cu_seqlens=cu, initial_state=S0,
                                          scale=0.75)
        for C in (1, 2, 3, 5, 16, 64):
            out, fin = chunked.prefill_chunked(q, k, v, g, b, cu_seqlens=cu, initial_state=S0,
                                               scale=0.75, chunk=C)
            np.testing.assert_allclose(out, ref_out, rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(fin, ref_fin, rtol=1e-9, atol=1e-11)


def test_varlen_independence_and_permutation(oracle):
    """A packed call equals per-sequence calls, and permuting the sequences
    permutes the results (bit for bit)."""
    rng = np.random.default_rng(8)
    lens = [13, 0, 1, 40, 7]
    H, K, V = 2, 8, 6
    cu = np.concatenate([[0], np.cumsum(lens)])
    q, k, v, g, b = _rand(rng, sum(lens), H, K, V)
    S0 = rng.standard_normal((len(lens), H, K, V))
    out, fin = oracle.prefill(q, k, v, g, b, cu_seqlens=cu, initial_state=S0)
    for n in range(len(lens)):
        sl = slice(cu[n], cu[n + 1])
        o1, f1 = oracle.prefill(q[sl], k[sl], v[sl], g[sl], b[sl], cu_seqlens=[0, lens[n]],
                                initial_state=S0[n:n + 1])
        np.testing.assert_array_equal(o1, out[sl])
        np.testing.assert_array_equal(f1[0], fin[n])
    perm = [3, 0, 4, 2, 1]
    plens = [lens[p] for p in perm]
    pcu = np.concatenate([[0], np.cumsum(plens)])
    idx = np.concatenate([np.arange(cu[p], cu[p + 1]) for p in perm]).astype(int)
    po, pf = oracle.prefill(q[idx], k[idx], v[idx], g[idx], b[idx], cu_seqlens=pcu,
                            initial_state=S0[perm])
    np.testing.assert_array_equal(po, out[idx])
    np.testing.assert_array_equal(pf, fin[perm])


def test_continuation_chains_final_to_initial(oracle):
    """Prefill of x[0:T] equals prefill of x[0:m] followed by prefill of x[m:T]
    started from the first call's final state, for every split point m."""
    rng = np.random.default_rng(9)
    T, H, K, V = 21, 2, 8, 8
    q, k, v, g, b = _rand(rng, T, H, K, V)
    S0 = rng.standard_normal((1, H, K, V))
    out, fin = oracle.prefill(q, k, v, g, b, cu_seqlens=[0, T], initial_state=S0)
    for m in range(T + 1):
        o1, f1 = oracle.prefill(q[:m], k[:m], v[:m], g[:m], b[:m], cu_seqlens=[0, m],
                                initial_state=S0)
        o2, f2 = oracle.prefill(q[m:], k[m:], v[m:], g[m:], b[m:], cu_seqlens=[0, T - m],
                                initial_state=f1)
        np.testing.assert_array_equal(np.concatenate([o1, o2]), out)
        np.testing.assert_array_equal(f2, fin)


def test_linearity_in_values_and_state(oracle):
    """With k, g, beta fixed, (out, final) is linear in (V, S0) jointly."""
    rng = np.random.default_rng(10)
    T, H, K, V = 33, 2, 8, 6
    q, k, v1, g, b = _rand(rng, T, H, K, V)
    v2 = rng.standard_normal(v1.shape)
    S1, S2 = rng.standard_normal((2, 1, H, K, V))
    a1, a2 = 0.7, -1.3
    f = lambda vv, ss: oracle.prefill(q, k, vv, g, b, cu_seqlens=[0, T], initial_state=ss)
    o1, h1 = f(v1, S1)
    o2, h2 = f(v2, S2)
    o3, h3 = f(a1 * v1 + a2 * v2, a1 * S1 + a2 * S2)
    np.testing.assert_allclose(o3, a1 * o1 + a2 * o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(h3, a1 * h1 + a2 * h2, rtol=1e-11, atol=1e-12)


def test_gate_extreme_forgets_state(oracle):
    """g = -1e4 (exp underflows to 0): each step forgets the state entirely, so
    S_t = beta_t k_t v_t^T and o_t = beta_t (k_t . q_t) v_t."""
    rng = np.random.default_rng(11)
    T, H, K, V = 9, 2, 8, 6
    q, k, v, _, b = _rand(rng, T, H, K, V)
    S0 = rng.standard_normal((1, H, K, V))
    out, fin = oracle.prefill(q, k, v, np.full((T, H, K), -1e4), b, cu_seqlens=[0, T],
                              initial_state=S0)
    beta = 1.0 / (1.0 + np.exp(-b))
    np.testing.assert_allclose(out, (beta * np.einsum("thk,thk->th", k, q))[..., None] * v,
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(fin[0], beta[-1][:, None, None] * k[-1][:, :, None]
                               * v[-1][:, None, :], rtol=1e-12, atol=1e-14)


def test_verify_matches_prefill_prefixes(oracle):
    """Verify = one short chunk per request: its outputs are the prefill outputs
    of the drafts, its stored state is the prefill final state after the
    accepted prefix (accepted 0 leaves the slot's state), read via slot."""
    rng = np.random.default_rng(12)
    R, D, H, K, V, P = 5, 4, 2, 8, 6, 7
    q, k, v, g, b = (x.reshape(R, D, H, -1) if x.ndim == 3 else x.reshape(R, D, H)
                     for x in _rand(rng, R * D, H, K, V))
    pool = rng.standard_normal((P, H, K, V))
    acc = np.array([0, 4, 1, 2, 3])
    slot = np.array([6, 0, 3, 2, 5])
    out, st = oracle.verify(q, k, v, g, b, pool, acc, slot=slot)
    for r in range(R):
        o, f = oracle.prefill(q[r], k[r], v[r], g[r], b[r], cu_seqlens=[0, D],
                              initial_state=pool[slot[r]][None])
        np.testing.assert_array_equal(out[r], o)
        a = acc[r]
        _, fa = oracle.prefill(q[r, :a], k[r, :a], v[r, :a], g[r, :a], b[r, :a],
                               cu_seqlens=[0, a], initial_state=pool[slot[r]][None])
        np.testing.assert_array_equal(st[r], fa[0])


# ---- gated RMSNorm of the output (oracle/norm.py), pinned by closed forms


def test_gated_rmsnorm_constant_row_closed_form():
    """o = c (every channel): mean(o^2) = c^2, so y = c / sqrt(c^2 + eps) * w * sigmoid(g)."""
    from oracle.norm import gated_rmsnorm
    V = 128
    c, eps = -3.0, 0.25
    w = np.linspace(0.5, 2.0, V)
    g = np.linspace(-4.0, 4.0, V)
    y = gated_rmsnorm(np.full((2, V), c), np.tile(g, (2, 1)), w, eps)
    expect = c / np.sqrt(c * c + eps) * w / (1.0 + np.exp(-g))
    assert np.allclose(y, np.tile(expect, (2, 1)), rtol=0, atol=1e-15)


def test_gated_rmsnorm_scale_invariance_and_gate_limits():
    """With eps = 0: y(lambda o) = sign(lambda) y(o); a gate of +40 gives plain
    RMSNorm times w (the rows then have mean square w^2 weighted), a gate of 0
    halves it, and a one-hot row o = a e_j gives sqrt(V) sign(a) w_j at j."""
    from oracle.norm import gated_rmsnorm
    rng = np.random.default_rng(7)
    V = 128
    o = rng.standard_normal((3, V))
    w = rng.uniform(0.5, 1.5, V)
    g = rng.standard_normal((3, V))
    y = gated_rmsnorm(o, g, w, 0.0)
    assert np.allclose(gated_rmsnorm(7.5 * o, g, w, 0.0), y, rtol=1e-13, atol=1e-14)
    assert np.allclose(gated_rmsnorm(-0.2 * o, g, w, 0.0), -y, rtol=1e-13, atol=1e-14)
    plain = gated_rmsnorm(o, np.full_like(g, 40.0), np.ones(V), 0.0)
    assert np.allclose(np.mean(plain * plain, axis=-1), 1.0, rtol=0, atol=1e-12)
    half = gated_rmsnorm(o, np.zeros_like(g), np.ones(V), 0.0)
    assert np.allclose(half, 0.5 * plain, rtol=0, atol=1e-15)
    e = np.zeros(V)
    e[5] = -2.0
    y1 = gated_rmsnorm(e, np.full(V, 40.0), w, 0.0)
    assert abs(y1[5] - (-np.sqrt(V) * w[5])) < 1e-12 and np.count_nonzero(y1) == 1
