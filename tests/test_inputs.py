"""The seeded input generators (CPU): the recipe both the CUDA path's tests and
the oracle are fed from -- determinism, value ranges, and the structure of the
varlen and verify workloads."""
import numpy as np
import torch

from kda_chunked_prefill_02_gb300 import inputs


def test_same_seed_same_values_and_streams_are_independent():
    a = inputs.prefill_inputs(5, B=2, T=70, H=3)
    b = inputs.prefill_inputs(5, B=2, T=70, H=3)
    for x, y in zip((a.q, a.k, a.v, a.g, a.beta, a.initial_state),
                    (b.q, b.k, b.v, b.g, b.beta, b.initial_state)):
        assert torch.equal(x, y)
    c = inputs.prefill_inputs(6, B=2, T=70, H=3)
    assert not torch.equal(a.q, c.q)
    # one stream per tensor: q does not depend on whether a state was drawn
    d = inputs.prefill_inputs(5, B=2, T=70, H=3, init_std=None)
    assert d.initial_state is None and torch.equal(a.q, d.q) and torch.equal(a.g, d.g)


def test_value_recipe():
    inp = inputs.prefill_inputs(7, B=1, T=512, H=4)
    for t in (inp.q, inp.k):
        assert t.dtype == torch.bfloat16
        n = t.float().norm(dim=-1)
        assert torch.all((n - 1).abs() < 2e-2)         # unit norm up to bf16 rounding
    g = inp.g
    assert g.dtype == torch.float32 and torch.all(g < 0) and torch.all(g > -5)
    assert abs(float(g.mean()) + 2.5) < 0.1             # -5 sigmoid(N(0,1)) has mean -2.5
    assert inp.beta.dtype == torch.float32 and abs(float(inp.beta.std()) - 1) < 0.1
    s0 = inp.initial_state
    assert s0.shape == (1, 4, 128, 128) and abs(float(s0.std()) - 0.02) < 1e-3


def test_varlen_lengths_structure():
    for seed in range(5):
        lens = inputs.varlen_lengths(seed, 8, 32768)
        assert len(lens) == 8 and sum(lens) == 32768 and lens.count(1) >= 1
        assert sum(1 for x in lens if x % 64) >= 3 and max(lens) <= 8192
    inp = inputs.prefill_inputs(2, lengths=inputs.varlen_lengths(2, 8, 32768), H=1)
    cu = inp.cu_seqlens.numpy()
    assert cu[0] == 0 and cu[-1] == inp.total_tokens == 32768 and np.all(np.diff(cu) >= 0)
    assert inp.q.shape == (32768, 1, 128) and inp.initial_state.shape == (8, 1, 128, 128)


def test_verify_workload_structure():
    vi = inputs.verify_inputs(9, R=40, D=4, H=2, pool_size=50, permute_slots=True)
    assert vi.q.shape == (40, 4, 2, 128) and vi.state_pool.shape == (50, 2, 128, 128)
    acc = vi.accepted.numpy()
    assert acc.min() >= 0 and acc.max() <= 4 and len(set(acc.tolist())) > 1
    slots = vi.slot.numpy()
    assert len(set(slots.tolist())) == 40 and slots.min() >= 0 and slots.max() < 50


def test_prefix_sample_keeps_sequence_heads():
    inp = inputs.prefill_inputs(11, lengths=[100, 3, 0, 70], H=2)
    sub = inputs.prefix_sample(inp, 64)
    assert sub.lengths == [64, 3, 0, 64]
    cu = inp.cu_seqlens.tolist()
    assert torch.equal(sub.q[:64], inp.q[:64])
    assert torch.equal(sub.q[64:67], inp.q[cu[1]:cu[1] + 3])
    assert torch.equal(sub.q[67:], inp.q[cu[3]:cu[3] + 64])
