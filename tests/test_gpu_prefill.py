"""GPU parity of kda_prefill against the fp64 oracle (through the C ABI).

Element-by-element on small seeded inputs that span several chunks and a
ragged tail; on sampled heads at the full workload sizes; plus the edge cases
(empty and length-1 sequences, strided views, in-place state, extreme gates,
determinism, bad cu_seqlens)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from kda_chunked_prefill_02_gb300 import inputs
from kda_test_util import (assert_parity, gpu_prefill, head_subset, oracle_prefill, rel_fro,
                           to_np)

pytestmark = pytest.mark.gpu


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).view(torch.bfloat16).float().numpy()


def _unswizzle_bf16(img, rows, f16=False):
    """[rows x 64] bf16 (or fp16) block stored with the 128-byte swizzle -> float array."""
    r = np.arange(rows)[:, None]
    c = np.arange(64)[None, :]
    off = r * 128 + (((c // 8) ^ (r % 8)) * 16) + (c % 8) * 2
    u16 = np.frombuffer(img.tobytes(), dtype=np.uint16)
    if f16:
        return u16[off // 2].view(np.float16).astype(np.float64)
    return _bf16(u16[off // 2])


def decode_record(raw):
    """Workspace record (include/kda.h layout) -> dict of Qt (scale Q e^Gam), W,
    Kt (fp16), Aqk (fp16), U, eg."""
    a1 = np.concatenate([_unswizzle_bf16(raw[0:16384], 128), _unswizzle_bf16(raw[16384:32768], 128)], 1)
    kt = _unswizzle_bf16(raw[32768:49152], 128, f16=True)
    aqk = _unswizzle_bf16(raw[49152:57344], 64, f16=True)
    u = _unswizzle_bf16(raw[57344:73728], 128).T     # stored as U^T: 128 value rows x 64 tokens
    eg = np.frombuffer(raw[73728:74240].tobytes(), dtype=np.float32)
    return dict(Qt=a1[:64], W=a1[64:], Kt=kt, Aqk=aqk, U=u, eg=eg)


def test_prep_stage_intermediates():
    """Steps A1-A5 alone: every per-chunk record matches the chunked fp64 form."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(5, B=2, T=200, H=2)
    d = inp.to("cuda")
    ws, L = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, scale=0.8, prep_only=True)
    torch.cuda.synchronize()
    raw = ws.cpu().numpy()
    q, k, v, g, b = (to_np(t) for t in (inp.q, inp.k, inp.v, inp.g, inp.beta))
    beta = 1.0 / (1.0 + np.exp(-b))
    cps = 4
    for bb in range(2):
        for c in range(cps):
            t0, t1 = 64 * c, min(64 * c + 64, 200)
            n = t1 - t0
            for h in range(2):
                r = (bb * cps + c) * 2 + h
                rec = decode_record(raw[L.records + r * L.record_bytes:L.records + (r + 1) * L.record_bytes])
                ref = chunked.chunk_step(np.zeros((128, 128)), 0.8 * q[bb, t0:t1, h], k[bb, t0:t1, h],
                                         v[bb, t0:t1, h], g[bb, t0:t1, h], beta[bb, t0:t1, h])
                for name, got, want in (("W", rec["W"][:n], ref["W"]), ("U", rec["U"][:n], ref["U"]),
                                        ("Qt", rec["Qt"][:n], ref["Qt"]), ("Aqk", rec["Aqk"][:n, :n], ref["Aqk"]),
                                        ("Kt", rec["Kt"][:, :n], ref["Kh"].T)):
                    assert rel_fro(got, want) < 1e-2, (name, bb, c, h, rel_fro(got, want))
                np.testing.assert_allclose(rec["eg"], np.exp(ref["gam"]), rtol=1e-5, atol=1e-30)
                # Aqk is masked to j <= i
                assert not np.any(np.triu(rec["Aqk"], 1)), "Aqk above the diagonal"
                for name, tail in (("W", rec["W"][n:]), ("U", rec["U"][n:]), ("Qt", rec["Qt"][n:]),
                                   ("Aqk", rec["Aqk"][n:]), ("Aqk cols", rec["Aqk"][:, n:]),
                                   ("Kt", rec["Kt"][:, n:])):
                    assert not np.any(tail), name


def test_tiny_config():
    inp = inputs.config_inputs("tiny")
    out, fin = gpu_prefill(inp)
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "tiny")


@pytest.mark.parametrize("lengths,H", [([17, 0, 16], 2), ([1024], 4), ([1025, 0, 31], 2),
                                       ([1, 64, 65, 127, 128, 129], 3)])
def test_varlen_small_shapes(lengths, H):
    inp = inputs.prefill_inputs(7 + len(lengths), lengths=lengths, H=H)
    out, fin = gpu_prefill(inp)
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, str(lengths))
    for n, L in enumerate(lengths):  # zero-length sequences keep their state exactly
        if L == 0:
            assert torch.equal(fin[n].cpu(), inp.initial_state[n])


def test_padded_ragged_tail_no_initial_state():
    inp = inputs.prefill_inputs(31, B=3, T=333, H=2, init_std=None)
    out, fin = gpu_prefill(inp)
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "padded T=333")


def test_beta_probabilities_scale_and_extreme_gates():
    inp = inputs.prefill_inputs(41, B=2, T=192, H=2)
    inp.beta = torch.sigmoid(inp.beta)
    inp.g[0, 10:12] = -1e4        # forget everything
    inp.g[0, 70:90, 0] = -20.0    # beyond the in-block gate floor
    inp.g[1, :, 1] = 0.0          # no decay on one head
    out, fin = gpu_prefill(inp, beta_is_logit=False, scale=0.7)
    ro, rf = oracle_prefill(inp, beta_is_logit=False, scale=0.7)
    assert_parity(out, fin, ro, rf, "beta prob / scale / gates")


def test_strided_views_match_contiguous():
    """Row-padded q/k/v/g/out views (token and head strides not dense) give the
    same bits as contiguous tensors: declared strides are honoured."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(51, B=2, T=130, H=3)
    d = inp.to("cuda")
    ref_out, ref_fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)

    def pad(t, extra):
        big = torch.zeros(t.shape[:-1] + (t.shape[-1] + extra,), dtype=t.dtype, device=t.device)
        big[..., :t.shape[-1]] = t
        return big[..., :t.shape[-1]]

    q, k, v, g = pad(d.q, 64), pad(d.k, 8), pad(d.v, 128), pad(d.g, 4)
    beta = torch.zeros(2, 130, 3, 5, device="cuda")[..., 1]
    beta.copy_(d.beta)
    out = pad(torch.empty_like(d.v), 16)
    K.kda_prefill(q, k, v, g, beta, initial_state=d.initial_state, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out)


def test_in_place_state_and_continuation():
    """final_state may alias initial_state; prefill of x[:m] then x[m:] from the
    first call's final state equals one call."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(61, B=1, T=300, H=2)
    d = inp.to("cuda")
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
    st = d.initial_state.clone()
    m = 100
    o1, _ = K.kda_prefill(d.q[:, :m], d.k[:, :m], d.v[:, :m], d.g[:, :m], d.beta[:, :m],
                          initial_state=st, final_state=st)
    o2, _ = K.kda_prefill(d.q[:, m:], d.k[:, m:], d.v[:, m:], d.g[:, m:], d.beta[:, m:],
                          initial_state=st, final_state=st)
    torch.cuda.synchronize()
    ro, rf = oracle_prefill(inp)
    assert_parity(torch.cat([o1, o2], 1), st, ro, rf, "continuation")
    assert_parity(out, fin, ro, rf, "single call")


def test_bit_identical_across_runs():
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(71, lengths=[300, 1, 0, 700], H=4)
    d = inp.to("cuda")
    a = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                      cu_seqlens=d.cu_seqlens)
    b = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                      cu_seqlens=d.cu_seqlens)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_bad_cu_seqlens_reported_not_faulted():
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(81, lengths=[40, 30], H=2)
    d = inp.to("cuda")
    cu = torch.tensor([0, 50, 45], dtype=torch.int32, device="cuda")  # decreasing, wrong end
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                             cu_seqlens=cu, device_status=status)
    torch.cuda.synchronize()
    assert status.item() == 1
    assert torch.equal(fin, d.initial_state)  # no chunk was processed


def _per_head_errors(out, fin, ro, rf):
    """Worst out max-abs error and worst final-state relative Frobenius error
    over the heads, each with its head index."""
    og, fg = to_np(out), to_np(fin)
    H = og.shape[-2]
    out_err = [float(np.abs(og[..., h, :] - ro[..., h, :]).max()) if og.size else 0.0 for h in range(H)]
    st_err = [rel_fro(fg[:, h], rf[:, h]) for h in range(H)]
    return (max(out_err), int(np.argmax(out_err))), (max(st_err), int(np.argmax(st_err)))


@pytest.mark.parametrize("name,schedules", [("padded", [None, 0]), ("varlen", [None]),
                                            ("long", [None, 0])])
def test_full_size_configs(name, schedules):
    """The full workloads in the launch configuration the bench times, every
    head against the oracle element by element (out max-abs, final state
    relative Frobenius per head); the padded and long workloads also in one
    pass (no segments), which must give the same tolerance."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.config_inputs(name)
    ro, rf = oracle_prefill(inp)
    for seg in schedules:
        with K.overrides(segment_chunks=seg):
            out, fin = gpu_prefill(inp)
        (eo, ho), (es, hs) = _per_head_errors(out, fin, ro, rf)
        print("%s (segments %s): worst out max-abs %.3e (head %d), worst final-state rel "
              "Frobenius %.3e (head %d)" % (name, "default" if seg is None else seg, eo, ho, es, hs))
        assert_parity(out, fin, ro, rf, name)
        assert es <= 1e-2, (name, seg, hs, es)
        del out, fin


def test_split_stages_equal_one_call():
    """kda_prefill_prep followed by kda_prefill_state gives the bits of kda_prefill."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(91, lengths=[129, 0, 64, 1], H=2)
    d = inp.to("cuda")
    a = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                      cu_seqlens=d.cu_seqlens)
    ws = torch.empty(K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens), dtype=torch.uint8,
                     device="cuda")
    K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                  cu_seqlens=d.cu_seqlens, workspace=ws, stage="prep")
    b = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                      cu_seqlens=d.cu_seqlens, workspace=ws, stage="state")
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_padded_zero_length_keeps_the_state():
    """B sequences of T = 0 tokens: no chunk at all, the final state is the
    initial one bit for bit (both state kernels)."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(701, B=2, T=64, H=3)
    d = inp.to("cuda")
    q, k, v, g, b = (t[:, :0].contiguous() for t in (d.q, d.k, d.v, d.g, d.beta))
    for kern in ("slab", "head"):
        with K.overrides(state_kernel=kern):
            out, fin = K.kda_prefill(q, k, v, g, b, initial_state=d.initial_state)
            torch.cuda.synchronize()
        assert out.numel() == 0
        assert torch.equal(fin, d.initial_state)


def test_many_heads_sampled():
    """H = 300 heads (grids and record indexing far past the workloads' 32),
    ragged T; oracle on a few heads."""
    inp = inputs.prefill_inputs(702, B=1, T=150, H=300)
    out, fin = gpu_prefill(inp)
    heads = [0, 1, 137, 299]
    sub = head_subset(inp, heads)
    ro, rf = oracle_prefill(sub)
    assert_parity(out[:, :, heads], fin[:, heads], ro, rf, "H=300")


def test_state_pass_takes_longest_sequences_first():
    """The chunk table ranks varlen sequences by chunk count, longest first
    (ties by index), for the order of the state pass's CTAs; results do not
    depend on it."""
    import kda_chunked_prefill_02_gb300 as K
    lengths = [17, 0, 300, 64, 65, 1]            # chunks 1, 0, 5, 1, 2, 1
    inp = inputs.prefill_inputs(95, lengths=lengths, H=2)
    d = inp.to("cuda")
    ws = torch.full((K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                             cu_seqlens=d.cu_seqlens, workspace=ws)
    torch.cuda.synchronize()
    L = K.workspace_layout(d.q, cu_seqlens=d.cu_seqlens)
    order = ws[L.seq_order:L.seq_order + 4 * len(lengths)].cpu().view(torch.int32).tolist()
    assert order == [2, 4, 0, 3, 5, 1]
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "longest-first order")


@pytest.mark.parametrize("nseq", [1000, 1100])
def test_many_sequences_order_paths(nseq):
    """Up to 1024 sequences the chunk table ranks them longest first; beyond,
    the state pass takes them in index order.  Both give the oracle's result."""
    import numpy as np
    import kda_chunked_prefill_02_gb300 as K
    rng = np.random.default_rng(nseq)
    lengths = [int(x) for x in rng.integers(0, 5, nseq)]
    lengths[7] = 130                                   # one sequence of three chunks
    inp = inputs.prefill_inputs(97, lengths=lengths, H=1)
    d = inp.to("cuda")
    ws = torch.full((K.workspace_size(d.q, d.v, cu_seqlens=d.cu_seqlens),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    out, fin = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                             cu_seqlens=d.cu_seqlens, workspace=ws)
    torch.cuda.synchronize()
    L = K.workspace_layout(d.q, cu_seqlens=d.cu_seqlens)
    order = ws[L.seq_order:L.seq_order + 4 * nseq].cpu().view(torch.int32).tolist()
    if nseq <= 1024:
        assert order[0] == 7 and sorted(order) == list(range(nseq))
        counts = [-(-n // 64) for n in lengths]
        assert all(counts[order[i]] >= counts[order[i + 1]] for i in range(nseq - 1))
    else:
        assert order == list(range(nseq))
    ro, rf = oracle_prefill(inp)
    assert_parity(out, fin, ro, rf, "%d sequences" % nseq)


def test_empty_batch_launches_nothing():
    """B = 0 sequences: nothing to compute, the call succeeds with empty outputs
    (no grid of zero CTAs is launched); the same through the split stages."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(703, B=1, T=100, H=2)
    d = inp.to("cuda")
    q, k, v, g, b = (t[:0] for t in (d.q, d.k, d.v, d.g, d.beta))
    out, fin = K.kda_prefill(q, k, v, g, b)
    torch.cuda.synchronize()
    assert out.shape == (0, 100, 2, 128) and fin.shape == (0, 2, 128, 128)
    ws = torch.empty(K.workspace_size(q, v), dtype=torch.uint8, device="cuda")
    for stage in ("prep", "state"):
        K.kda_prefill(q, k, v, g, b, workspace=ws, stage=stage)
    torch.cuda.synchronize()


def test_side_stream_without_workspace():
    """A call on a side stream with no workspace: the binding allocates the
    workspace and outputs on that stream (so the caching allocator cannot give
    their memory to other work while the kernels run), and the result equals
    the call on the current stream bit for bit."""
    import kda_chunked_prefill_02_gb300 as K
    inp = inputs.prefill_inputs(1301, B=1, T=64 * 9 + 3, H=4)
    d = inp.to("cuda")
    ref = K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    outs = []
    for _ in range(3):   # freed workspaces are reused across the calls
        outs.append(K.kda_prefill(d.q, d.k, d.v, d.g, d.beta, initial_state=d.initial_state,
                                  stream=side))
        junk = torch.full((1 << 22,), 7, dtype=torch.uint8, device="cuda")  # current-stream work
        del junk
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    for out, fin in outs:
        assert torch.equal(out, ref[0]) and torch.equal(fin, ref[1])
