"""CPU-only checks of the C ABI: the library loads, exports every function that
include/*.h declares, and refuses bad arguments on the host (before any CUDA
call, so these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def K():
    from kda_chunked_prefill_02_gb300 import build, kda
    build.build()
    return kda


def _declared(header):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"\b(kda_[a-z_0-9]+)\s*\(", src))


def test_exports_every_declared_symbol(K):
    lib = K.lib()
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            names |= _declared(h)
    assert {"kda_prefill", "kda_verify", "kda_prefill_workspace_size",
            "kda_status_string"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert lib.kda_abi_version() == 6


def _args(K, **kw):
    a = K.PrefillArgs()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: validation fails first
    a.q = a.k = a.v = a.g = a.beta = a.out = fake
    for f in ("q_stride", "k_stride", "v_stride", "g_stride", "out_stride"):
        setattr(a, f, K._i64x3(4 * 256 * 128, 2 * 128, 128))
    a.beta_stride = K._i64x3(512, 2, 1)
    a.batch, a.seqlen, a.num_seqs, a.num_heads = 1, 256, 1, 2
    a.head_dim_k = a.head_dim_v = 128
    a.chunk = 64
    a.beta_is_logit = 1
    a.scale = 1.0
    a.workspace = ctypes.c_void_p(1 << 30)
    a.workspace_bytes = K.lib().kda_prefill_workspace_size(ctypes.byref(a))
    for k_, v_ in kw.items():
        setattr(a, k_, v_)
    return a


def test_host_validation(K):
    lib = K.lib()
    run = lambda a: lib.kda_prefill(ctypes.byref(a), None)
    assert run(_args(K, head_dim_k=64)) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, head_dim_v=256)) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, chunk=32)) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, q_stride=K._i64x3(4 * 256 * 128, 2 * 128 + 3, 128))) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, g_stride=K._i64x3(0, 2 * 128 + 2, 128))) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, q=ctypes.c_void_p((1 << 20) + 2))) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, num_seqs=2)) == K.KDA_ERR_INVALID_ARG
    assert run(_args(K, num_heads=0)) == K.KDA_ERR_INVALID_ARG
    assert run(_args(K, workspace_bytes=100)) == K.KDA_ERR_INVALID_ARG
    assert run(_args(K, workspace=ctypes.c_void_p((1 << 30) + 64))) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, q=None)) == K.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill(None, None) == K.KDA_ERR_INVALID_ARG
    assert lib.kda_prefill_workspace_size(None) == 0


def test_workspace_plan(K):
    lib = K.lib()
    a = _args(K)
    L = K.WorkspaceLayout()
    assert lib.kda_prefill_workspace_layout(ctypes.byref(a), ctypes.byref(L)) == 0
    assert L.max_chunks == 4                        # padded: ceil(256 / 64)
    assert L.total == lib.kda_prefill_workspace_size(ctypes.byref(a))
    offs = [L.records, L.chunk_offset, L.status, L.state_carry]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    # padded: one fp32 128 x 128 state per chain (batch 1 x 2 heads) carried between segments,
    # after the per-segment record counters (one int32 per chunk of a sequence, + 1)
    assert L.total == L.state_carry + 2 * 128 * 128 * 4
    assert L.status < L.prep_counters and L.prep_counters + 4 * 5 <= L.state_carry
    assert L.record_bytes == 74240 and L.chunk_offset >= L.records + 8 * L.record_bytes
    # varlen upper bound on chunks: floor(T / 64) + N
    a2 = _args(K, cu_seqlens=ctypes.c_void_p(1 << 12), num_seqs=3, seqlen=130)
    assert lib.kda_prefill_workspace_layout(ctypes.byref(a2), ctypes.byref(L)) == 0
    assert L.max_chunks == 130 // 64 + 3
    # varlen: the state-pass order of the sequences, int32 [N], after the chunk table
    assert L.seq_order >= L.chunk_offset + 4 * 4 and L.seq_order % 256 == 0
    assert L.status >= L.seq_order + 3 * 4


def test_verify_validation(K):
    lib = K.lib()
    a = K.VerifyArgs()
    a.head_dim_k = a.head_dim_v = 128
    a.num_requests, a.num_drafts, a.num_heads, a.pool_size = 4, 17, 2, 4
    assert lib.kda_verify(ctypes.byref(a), None) == K.KDA_ERR_UNSUPPORTED
    a.num_drafts = 4
    assert lib.kda_verify(ctypes.byref(a), None) == K.KDA_ERR_INVALID_ARG  # null pointers
    a.num_requests = 0
    assert lib.kda_verify(ctypes.byref(a), None) == 0                      # nothing to do


def test_status_strings(K):
    for s in range(5):
        assert K.status_string(s).startswith("KDA_")


def test_verify_refuses_misaligned_state_pool(K):
    """The verify kernel moves the state in 16-byte vectors: a pool pointer that
    is not 16-byte aligned is refused on the host, before any CUDA call."""
    lib = K.lib()
    a = K.VerifyArgs()
    fake = ctypes.c_void_p(1 << 20)
    a.q = a.k = a.v = a.g = a.beta = a.out = a.accepted = fake
    a.state_pool = ctypes.c_void_p((1 << 20) + 4)
    for f in ("q_stride", "k_stride", "v_stride", "g_stride", "out_stride"):
        setattr(a, f, K._i64x3(4 * 2 * 128, 2 * 128, 128))
    a.beta_stride = K._i64x3(8, 2, 1)
    a.head_dim_k = a.head_dim_v = 128
    a.num_requests, a.num_drafts, a.num_heads, a.pool_size = 2, 4, 2, 2
    assert lib.kda_verify(ctypes.byref(a), None) == K.KDA_ERR_UNSUPPORTED


def test_verify_refuses_rows_it_cannot_move_in_16_byte_pieces(K):
    """Verify moves draft rows and state blocks in 16-byte pieces, so a
    misaligned pointer or stride is refused on the host (no CUDA call)."""
    lib = K.lib()

    def args(**kw):
        a = K.VerifyArgs()
        fake = ctypes.c_void_p(1 << 20)
        a.q = a.k = a.v = a.g = a.beta = a.out = a.state_pool = a.accepted = fake
        for f in ("q_stride", "k_stride", "v_stride", "g_stride", "out_stride"):
            setattr(a, f, K._i64x3(4 * 2 * 128, 2 * 128, 128))
        a.beta_stride = K._i64x3(8, 2, 1)
        a.head_dim_k = a.head_dim_v = 128
        a.num_requests, a.num_drafts, a.num_heads, a.pool_size = 2, 4, 2, 2
        for k_, v_ in kw.items():
            setattr(a, k_, v_)
        return a

    run = lambda a: lib.kda_verify(ctypes.byref(a), None)
    assert run(args(q=ctypes.c_void_p((1 << 20) + 2))) == K.KDA_ERR_UNSUPPORTED
    assert run(args(g=ctypes.c_void_p((1 << 20) + 4))) == K.KDA_ERR_UNSUPPORTED
    assert run(args(k_stride=K._i64x3(4 * 2 * 128, 2 * 128 + 4, 128))) == K.KDA_ERR_UNSUPPORTED
    assert run(args(g_stride=K._i64x3(4 * 2 * 128, 2 * 128 + 2, 128))) == K.KDA_ERR_UNSUPPORTED


def _sched(K, num_sms=152, **kw):
    a = _args(K, **kw)
    a.overrides = K._current_overrides()
    s = K.Schedule()
    assert K.lib().kda_prefill_schedule(ctypes.byref(a), num_sms, ctypes.byref(s)) == 0
    return (s.segmented, s.whole_chain, s.segment_chunks, s.prep_ctas)


def test_prefill_schedule(K, monkeypatch):
    """Host-side schedule choice (no GPU call): segments only for few long
    padded chains, with the state kernel that leaves prep the most SMs.  The
    process environment plays no part (the names earlier builds read are set
    here to values that would change the schedule); only the call's overrides
    do."""
    monkeypatch.setenv("KDA_SEGMENT_CHUNKS", "3")
    monkeypatch.setenv("KDA_STATE_KERNEL", "slab")
    monkeypatch.setenv("KDA_STALL_INJECT", "7")
    # 32 chains of 2048 chunks: whole-chain state CTAs on 32 SMs, prep on 120
    # (joined by a second prep grid on the state SMs once each state pass ends)
    s32 = _sched(K, batch=1, num_seqs=1, seqlen=131072, num_heads=32)
    assert s32[:2] == (1, 1) and s32[3] == 120 and s32[2] % 8 == 0
    # 8 chains: the segment-parallel scan (test_scan_schedule_and_workspace);
    # with the scan ruled out, slab state CTAs (4 per chain) on 32 SMs beside
    # prep on 120
    with K.overrides(scan_segments=1):
        s8 = _sched(K, batch=1, num_seqs=1, seqlen=131072, num_heads=8)
    assert s8[:2] == (1, 0) and s8[3] == 120 and s8[2] % 8 == 0
    # the padded workload (64 chains of 64 chunks): two segments, whole-chain
    # state CTAs on 64 SMs, prep on 88 (measured 0.360 ms against 0.399 one pass)
    assert _sched(K, batch=4, num_seqs=4, seqlen=4096, num_heads=16) == (1, 1, 48, 88)
    # short sequences and varlen: one pass
    assert _sched(K, batch=1, num_seqs=1, seqlen=256, num_heads=2) == (0, 0, 0, 152)
    assert _sched(K, batch=1, num_seqs=1, seqlen=4096, num_heads=32)[0] == 0
    # 16384 tokens of 32 heads: segmented (measured 0.69 ms against 0.75 one pass)
    assert _sched(K, batch=1, num_seqs=1, seqlen=16384, num_heads=32)[:2] == (1, 1)
    assert _sched(K, cu_seqlens=ctypes.c_void_p(1 << 12), num_seqs=8, seqlen=32768,
                  num_heads=32) == (0, 1, 0, 152)
    # two chains: the slab pass (2048 steps) dominates and prep is short, so
    # moving prep beside it gains little
    assert _sched(K, batch=1, num_seqs=1, seqlen=131072, num_heads=2)[0] == 0
    # the fused norm needs whole rows: whole-chain kernel in either schedule
    assert _sched(K, batch=1, num_seqs=1, seqlen=131072, num_heads=32,
                  out_gate=ctypes.c_void_p(1))[1] == 1
    # overrides
    with K.overrides(segment_chunks=0):
        assert _sched(K, batch=1, num_seqs=1, seqlen=131072, num_heads=32)[0] == 0
    with K.overrides(segment_chunks=3):
        assert _sched(K, batch=1, num_seqs=1, seqlen=256, num_heads=2) == (1, 0, 3, 144)
    with K.overrides(segment_chunks=3, state_kernel="head"):
        assert _sched(K, batch=1, num_seqs=1, seqlen=256, num_heads=2) == (1, 1, 3, 150)
    with K.overrides(segment_chunks=3, prep_ctas=40):
        assert _sched(K, batch=1, num_seqs=1, seqlen=256, num_heads=2) == (1, 0, 3, 40)
    with K.overrides(state_kernel="head"):
        assert _sched(K, batch=1, num_seqs=1, seqlen=4096, num_heads=2) == (0, 1, 0, 152)
    # negative scan segment counts are refused
    a = _args(K, batch=1, num_seqs=1, seqlen=256, num_heads=2)
    o = K._make_overrides()
    o.scan_segments = -2
    a.overrides = ctypes.pointer(o)
    assert K.lib().kda_prefill(ctypes.byref(a), None) == K.KDA_ERR_INVALID_ARG


def _sched_full(K, num_sms=152, **kw):
    a = _args(K, **kw)
    a.overrides = K._current_overrides()
    s = K.Schedule()
    assert K.lib().kda_prefill_schedule(ctypes.byref(a), num_sms, ctypes.byref(s)) == 0
    return s


def test_scan_schedule_and_workspace(K):
    """The segment-parallel scan: chosen for few long padded chains (a quarter
    of the long workload's heads or fewer), never for the long workload itself
    or varlen calls; forced and ruled out by the overrides; its workspace room
    as include/kda.h states (host only)."""
    long = dict(batch=1, num_seqs=1, seqlen=131072)
    for H in (1, 2, 4, 8):
        s = _sched_full(K, num_heads=H, **long)
        assert s.scan_segments >= 2 and s.segmented == 0 and s.whole_chain == 1, H
        assert (s.scan_segments - 1) * s.scan_chunks < 2048 <= s.scan_segments * s.scan_chunks
    assert _sched_full(K, num_heads=32, **long).scan_segments == 0
    assert _sched_full(K, cu_seqlens=ctypes.c_void_p(1 << 12), num_seqs=8, seqlen=32768,
                       num_heads=2).scan_segments == 0
    with K.overrides(scan_segments=1):       # never: the two-stream schedule instead
        s = _sched_full(K, num_heads=8, **long)
        assert s.scan_segments == 0 and s.segmented == 1
    with K.overrides(scan_segments=3):       # 12300 tokens: 193 chunks, room for 3
        s = _sched_full(K, batch=1, num_seqs=1, seqlen=12300, num_heads=2)
        assert (s.scan_segments, s.scan_chunks) == (3, 65)
    with K.overrides(scan_segments=9):       # clamped to the room
        assert _sched_full(K, batch=1, num_seqs=1, seqlen=12300, num_heads=2).scan_segments == 3
    with K.overrides(scan_segments=2):       # no room below 128 chunks: not run
        assert _sched_full(K, batch=1, num_seqs=1, seqlen=8000, num_heads=2).scan_segments == 0
    lib = K.lib()
    L = K.WorkspaceLayout()
    a = _args(K, num_heads=8, **long)
    assert lib.kda_prefill_workspace_layout(ctypes.byref(a), ctypes.byref(L)) == 0
    assert L.scan_max_segments == 32 and L.scan >= L.state_carry + 8 * 65536
    assert L.total - L.scan >= (3 * 32 - 2) * 8 * 65536
    a = _args(K, batch=1, num_seqs=1, seqlen=131072, num_heads=65)   # too many chains
    assert lib.kda_prefill_workspace_layout(ctypes.byref(a), ctypes.byref(L)) == 0
    assert L.scan_max_segments == 0
    a = _args(K)
    assert K.lib().kda_prefill_schedule(ctypes.byref(a), 0, ctypes.byref(K.Schedule())) == \
        K.KDA_ERR_INVALID_ARG


def test_host_call_staging_plan(K):
    """kda_prefill_host's staging size (host only): the default piece, growth
    with the piece length, the clamp to the input, a lower bound of two piece
    buffers + the chain states + one piece's workspace, and refusals of bad
    piece lengths and bad host cu_seqlens."""
    import torch
    B, T, H = 2, 10000, 4
    q = torch.empty(B, T, H, 128, dtype=torch.bfloat16)
    assert K.host_staging_size(q, q) == K.host_staging_size(q, q, piece_tokens=2048) > 0
    sizes = [K.host_staging_size(q, q, piece_tokens=p) for p in (64, 512, 4096, 10048, 20480)]
    assert sizes[0] < sizes[1] < sizes[2] < sizes[3] == sizes[4]
    per_tok = 3 * 256 + 512 + 4 + 256          # q, k, v, g, beta in; out back
    P = 512
    ws = K.workspace_size(torch.empty(B, P, H, 128, dtype=torch.bfloat16), q)
    assert sizes[1] >= 2 * B * P * H * per_tok + B * H * 128 * 128 * 4 + ws
    for bad in (100, -64):
        assert K.host_staging_size(q, q, piece_tokens=bad) == 0

    cu = torch.tensor([0, 3000, 3001, 3001, 8001, 8065], dtype=torch.int32)
    qv = torch.empty(8065, H, 128, dtype=torch.bfloat16)
    good = K.host_staging_size(qv, qv, cu_seqlens=cu, piece_tokens=64)
    assert good >= 2 * 5000 * H * per_tok      # whole sequences: the longest one fits a buffer
    for i, val in ((0, 1), (2, 2000), (5, 8000)):   # cu[0] != 0, decreasing, end != T
        bad = cu.clone()
        bad[i] = val
        assert K.host_staging_size(qv, qv, cu_seqlens=bad) == 0


def test_size_limits_refused_on_host(K):
    """Calls past the kernels' index ranges are refused before any CUDA call:
    more than 65535 sequences or heads in a prefill (grid dimensions), and
    verify with R * H at or beyond 2^31 items."""
    lib = K.lib()
    run = lambda a: lib.kda_prefill(ctypes.byref(a), None)
    assert run(_args(K, batch=65536, num_seqs=65536)) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, num_heads=65536)) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, seqlen=1 << 31)) == K.KDA_ERR_UNSUPPORTED
    a = K.VerifyArgs()
    fake = ctypes.c_void_p(1 << 20)
    a.q = a.k = a.v = a.g = a.beta = a.out = a.state_pool = a.accepted = fake
    for f in ("q_stride", "k_stride", "v_stride", "g_stride", "out_stride"):
        setattr(a, f, K._i64x3(4 * 2 * 128, 2 * 128, 128))
    a.beta_stride = K._i64x3(8, 2, 1)
    a.head_dim_k = a.head_dim_v = 128
    a.num_requests, a.num_drafts, a.num_heads, a.pool_size = 65535, 4, 65535, 65535
    assert lib.kda_verify(ctypes.byref(a), None) == K.KDA_ERR_UNSUPPORTED


def test_no_fallback_without_the_library_or_a_gpu(K, monkeypatch, tmp_path):
    """The product path never computes on the CPU: CPU tensors are refused, and
    a missing libkda.so is an error, not a detour."""
    import torch
    from kda_chunked_prefill_02_gb300 import inputs
    inp = inputs.prefill_inputs(3, B=1, T=70, H=2)
    with pytest.raises(ValueError, match="CUDA tensor"):
        K.kda_prefill(inp.q, inp.k, inp.v, inp.g, inp.beta, out=torch.empty_like(inp.v),
                      final_state=torch.empty(1, 2, 128, 128), workspace=torch.empty(1, dtype=torch.uint8))
    vi = inputs.verify_inputs(3, R=2, D=2, H=1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        K.kda_verify(vi.q, vi.k, vi.v, vi.g, vi.beta, vi.state_pool, vi.accepted)
    monkeypatch.setattr(K, "_lib", None)
    monkeypatch.setattr(K, "LIB_PATH", str(tmp_path / "libkda.so"))
    with pytest.raises(RuntimeError, match="not built"):
        K.workspace_size(inp.q, inp.v)


def test_noalloc_capacity_as_documented(K):
    """kda_prefill_noalloc's scratch holds the workspace of 2048 tokens x 13
    heads (and 8192 x 3), but not 2048 x 14 (host-side sizes only)."""
    import torch
    lim = K.NOALLOC_MAX_WORKSPACE_BYTES
    size = lambda T, H: K.workspace_size(torch.empty(1, T, H, 128, dtype=torch.bfloat16),
                                         torch.empty(1, T, H, 128, dtype=torch.bfloat16))
    assert size(2048, 13) <= lim < size(2048, 14)
    assert size(8192, 3) <= lim < size(8192, 4)


def test_noalloc_checks_arguments_before_the_size(K):
    """kda_prefill_noalloc runs kda_prefill's argument checks first: a bad
    argument comes back as KDA_ERR_INVALID_ARG / KDA_ERR_UNSUPPORTED exactly as
    from kda_prefill (never as an oversize problem), dimensions whose sizes
    would wrap size_t are refused, and a well-formed problem past the scratch
    is KDA_ERR_UNSUPPORTED.  All before any CUDA call."""
    lib = K.lib()
    f = lib.kda_prefill_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(K.PrefillArgs), ctypes.c_void_p]
    run = lambda a: f(ctypes.byref(a), None)
    assert run(_args(K, num_seqs=-1)) == K.KDA_ERR_INVALID_ARG
    assert run(_args(K, batch=-3, num_seqs=-3)) == K.KDA_ERR_INVALID_ARG
    assert run(_args(K, num_heads=0)) == K.KDA_ERR_INVALID_ARG
    assert run(_args(K, chunk=32)) == K.KDA_ERR_UNSUPPORTED
    assert run(_args(K, q=None)) == K.KDA_ERR_INVALID_ARG
    assert f(None, None) == K.KDA_ERR_INVALID_ARG
    # well formed but larger than the scratch (2048 tokens x 14 heads)
    assert run(_args(K, seqlen=2048, num_heads=14)) == K.KDA_ERR_UNSUPPORTED
    # sizes that would overflow the workspace plan are refused, not wrapped
    huge = _args(K, cu_seqlens=ctypes.c_void_p(1 << 12), batch=1, num_seqs=60000,
                 seqlen=(1 << 31) - 1, num_heads=60000)
    assert run(huge) != K.KDA_OK
    assert lib.kda_prefill_workspace_size(ctypes.byref(huge)) > 0   # representable here
    L = K.WorkspaceLayout()
    big = _args(K, batch=1 << 41, num_seqs=1 << 41, seqlen=1 << 30, num_heads=1 << 20)
    assert lib.kda_prefill_workspace_size(ctypes.byref(big)) == 0
    assert lib.kda_prefill_workspace_layout(ctypes.byref(big), ctypes.byref(L)) == K.KDA_ERR_INVALID_ARG
