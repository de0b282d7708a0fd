"""ctypes binding of libkda.so (include/kda.h): argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
only turns torch tensors into pointers, strides and sizes, allocates outputs
and the workspace through torch (the library itself allocates nothing), and
raises on any status other than KDA_OK.  There is no fallback: if the library
is missing or a tensor is not on a CUDA device, the call fails.
"""
import contextlib
import contextvars
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_CUDA, KDA_ERR_TIMEOUT = range(5)
HEAD_DIM = 128
CHUNK = 64

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i64x3 = ctypes.c_int64 * 3


class Overrides(ctypes.Structure):
    """kda_overrides: test and measurement overrides of the library's choices."""
    _fields_ = [("state_kernel", ctypes.c_int32), ("segment_chunks", ctypes.c_int32),
                ("prep_ctas", ctypes.c_int32), ("no_pdl", ctypes.c_int32),
                ("stall_seed", ctypes.c_uint32), ("scan_segments", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("timeout_probe", ctypes.c_int32),
                ("verify_kernel", ctypes.c_int32)]


_STATE_KERNELS = {None: 0, "slab": 1, "head": 2}
_overrides_var = contextvars.ContextVar("kda_overrides", default=None)


def _make_overrides(state_kernel=None, segment_chunks=None, prep_ctas=None, no_pdl=False,
                    stall_seed=0, wait_limit_ns=0, scan_segments=0, timeout_probe=False,
                    verify_kernel=None):
    o = Overrides()
    o.state_kernel = _STATE_KERNELS[state_kernel]
    o.segment_chunks = -1 if segment_chunks is None else int(segment_chunks)
    o.prep_ctas = int(prep_ctas or 0)
    o.no_pdl = 1 if no_pdl else 0
    o.stall_seed = int(stall_seed or 0)
    o.wait_limit_ns = int(wait_limit_ns or 0)
    o.scan_segments = int(scan_segments or 0)
    o.timeout_probe = 1 if timeout_probe else 0
    o.verify_kernel = {None: 0, "sequential": 1, "tensor": 2}[verify_kernel]
    return o


@contextlib.contextmanager
def overrides(**kw):
    """Within the block, calls of this module pass these kda_overrides to the
    library (tests and measurements): state_kernel ("slab" | "head"),
    segment_chunks (0: never segment, n: segments of n chunks), prep_ctas,
    no_pdl, stall_seed, wait_limit_ns, scan_segments (1: never run the
    segment-parallel scan, n >= 2: run it with n segments), timeout_probe,
    verify_kernel ("sequential" | "tensor").  Nothing is taken from the
    environment."""
    tok = _overrides_var.set(_make_overrides(**kw))
    try:
        yield
    finally:
        _overrides_var.reset(tok)


def _current_overrides():
    o = _overrides_var.get()
    return None if o is None else ctypes.pointer(o)


class PrefillArgs(ctypes.Structure):
    _fields_ = [("q", _p), ("k", _p), ("v", _p), ("g", _p), ("beta", _p), ("out", _p),
                ("q_stride", _i64x3), ("k_stride", _i64x3), ("v_stride", _i64x3),
                ("g_stride", _i64x3), ("beta_stride", _i64x3), ("out_stride", _i64x3),
                ("initial_state", _p), ("final_state", _p), ("cu_seqlens", _p),
                ("batch", _i64), ("seqlen", _i64), ("num_seqs", _i64), ("num_heads", _i64),
                ("head_dim_k", _i64), ("head_dim_v", _i64),
                ("chunk", ctypes.c_int32), ("beta_is_logit", ctypes.c_int32),
                ("scale", ctypes.c_float),
                ("workspace", _p), ("workspace_bytes", ctypes.c_size_t),
                ("device_status", _p), ("out_gate", _p), ("gate_stride", _i64x3),
                ("norm_weight", _p), ("norm_eps", ctypes.c_float),
                ("overrides", ctypes.POINTER(Overrides))]


class PrefillHostArgs(ctypes.Structure):
    _fields_ = [("args", PrefillArgs), ("staging", _p), ("staging_bytes", ctypes.c_size_t),
                ("piece_tokens", _i64)]


class VerifyArgs(ctypes.Structure):
    _fields_ = [("q", _p), ("k", _p), ("v", _p), ("g", _p), ("beta", _p), ("out", _p),
                ("q_stride", _i64x3), ("k_stride", _i64x3), ("v_stride", _i64x3),
                ("g_stride", _i64x3), ("beta_stride", _i64x3), ("out_stride", _i64x3),
                ("state_pool", _p), ("pool_size", _i64), ("slot", _p), ("accepted", _p),
                ("num_requests", _i64), ("num_drafts", _i64), ("num_heads", _i64),
                ("head_dim_k", _i64), ("head_dim_v", _i64),
                ("beta_is_logit", ctypes.c_int32), ("scale", ctypes.c_float),
                ("device_status", _p), ("pool_dtype", ctypes.c_int32),
                ("replay_only", ctypes.c_int32), ("overrides", ctypes.POINTER(Overrides))]


KDA_POOL_F32, KDA_POOL_BF16 = 0, 1


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [("records", ctypes.c_size_t), ("record_bytes", ctypes.c_size_t),
                ("chunk_offset", ctypes.c_size_t), ("status", ctypes.c_size_t),
                ("total", ctypes.c_size_t), ("max_chunks", _i64),
                ("state_carry", ctypes.c_size_t), ("seq_order", ctypes.c_size_t),
                ("scan", ctypes.c_size_t), ("scan_max_segments", _i64),
                ("prep_counters", ctypes.c_size_t)]


class Schedule(ctypes.Structure):
    _fields_ = [("segmented", ctypes.c_int32), ("whole_chain", ctypes.c_int32),
                ("segment_chunks", ctypes.c_int32), ("prep_ctas", ctypes.c_int32),
                ("scan_segments", ctypes.c_int32), ("scan_chunks", ctypes.c_int32)]


_lib = None


def lib():
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkda.so is not built; run `python -m "
                               "kda_chunked_prefill_02_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        L.kda_prefill_workspace_size.restype = ctypes.c_size_t
        L.kda_prefill_workspace_size.argtypes = [ctypes.POINTER(PrefillArgs)]
        L.kda_prefill_workspace_layout.restype = ctypes.c_int
        L.kda_prefill_workspace_layout.argtypes = [ctypes.POINTER(PrefillArgs),
                                                   ctypes.POINTER(WorkspaceLayout)]
        L.kda_prefill_schedule.restype = ctypes.c_int
        L.kda_prefill_schedule.argtypes = [ctypes.POINTER(PrefillArgs), ctypes.c_int,
                                           ctypes.POINTER(Schedule)]
        for name in ("kda_prefill", "kda_prefill_prep", "kda_prefill_state"):
            f = getattr(L, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.POINTER(PrefillArgs), _p]
        L.kda_prefill_host_staging_size.restype = ctypes.c_size_t
        L.kda_prefill_host_staging_size.argtypes = [ctypes.POINTER(PrefillHostArgs)]
        L.kda_prefill_host.restype = ctypes.c_int
        L.kda_prefill_host.argtypes = [ctypes.POINTER(PrefillHostArgs), _p]
        L.kda_verify.restype = ctypes.c_int
        L.kda_verify.argtypes = [ctypes.POINTER(VerifyArgs), _p]
        L.kda_status_string.restype = ctypes.c_char_p
        L.kda_status_string.argtypes = [ctypes.c_int]
        L.kda_abi_version.restype = ctypes.c_int
        L.kda_abi_version.argtypes = []
        _lib = L
    return _lib


class KdaError(RuntimeError):
    def __init__(self, status):
        self.status = status
        super().__init__(lib().kda_status_string(status).decode())


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _check(status):
    if status != KDA_OK:
        raise KdaError(status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _on_stream(stream, like):
    """Context in which torch allocations belong to `stream` (None or a CPU
    tensor: the current stream)."""
    if stream is None or not getattr(like, "is_cuda", False):
        return contextlib.nullcontext()
    return torch.cuda.stream(stream)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(name, t, dtype):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


def _strides3(t, varlen, last_is_channel=True):
    """(batch, token, head) element strides; the channel dim must be contiguous."""
    s = t.stride()
    if last_is_channel:
        if s[-1] != 1:
            raise ValueError("the channel (last) dim must have stride 1")
        s = s[:-1]
    return (0, s[0], s[1]) if varlen else (s[0], s[1], s[2])


def _prefill_args(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, beta_is_logit,
                  scale, workspace, device_status, chunk, out_gate=None, norm_weight=None,
                  norm_eps=1e-6):
    varlen = cu_seqlens is not None
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.float32), ("out", out, torch.bfloat16),
                        ("initial_state", initial_state, torch.float32),
                        ("final_state", final_state, torch.float32),
                        ("cu_seqlens", cu_seqlens, torch.int32),
                        ("device_status", device_status, torch.int32)):
        _need_cuda(name, t, dt)
    for name, t in (("initial_state", initial_state), ("final_state", final_state)):
        if t is not None and not t.is_contiguous():
            raise ValueError("%s must be contiguous [N, H, 128, 128]" % name)
    a = PrefillArgs()
    a.q, a.k, a.v, a.g, a.beta, a.out = (_ptr(t) for t in (q, k, v, g, beta, out))
    a.q_stride = _i64x3(*_strides3(q, varlen))
    a.k_stride = _i64x3(*_strides3(k, varlen))
    a.v_stride = _i64x3(*_strides3(v, varlen))
    a.g_stride = _i64x3(*_strides3(g, varlen))
    a.out_stride = _i64x3(*_strides3(out, varlen))
    a.beta_stride = _i64x3(*_strides3(beta, varlen, last_is_channel=False))
    a.initial_state = _ptr(initial_state)
    a.final_state = _ptr(final_state)
    a.cu_seqlens = _ptr(cu_seqlens)
    if varlen:
        a.batch, a.seqlen, a.num_seqs = 1, q.shape[0], cu_seqlens.shape[0] - 1
        a.num_heads = q.shape[1]
    else:
        a.batch, a.seqlen, a.num_seqs = q.shape[0], q.shape[1], q.shape[0]
        a.num_heads = q.shape[2]
    a.head_dim_k, a.head_dim_v = q.shape[-1], v.shape[-1]
    a.chunk = int(chunk)
    a.beta_is_logit = 1 if beta_is_logit else 0
    a.scale = float(scale)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.device_status = _ptr(device_status)
    if out_gate is not None or norm_weight is not None:
        _need_cuda("out_gate", out_gate, torch.bfloat16)
        _need_cuda("norm_weight", norm_weight, torch.float32)
        if norm_weight is None or not norm_weight.is_contiguous():
            raise ValueError("norm_weight must be a contiguous fp32 [128] CUDA tensor")
        a.out_gate = _ptr(out_gate)
        a.gate_stride = _i64x3(*_strides3(out_gate, varlen))
        a.norm_weight = _ptr(norm_weight)
        a.norm_eps = float(norm_eps)
    a.overrides = _current_overrides()
    return a


def workspace_size(q, v, *, cu_seqlens=None):
    """Workspace bytes that kda_prefill needs for these shapes."""
    a = PrefillArgs()
    if cu_seqlens is not None:
        a.batch, a.seqlen, a.num_seqs = 1, q.shape[0], cu_seqlens.shape[0] - 1
        a.num_heads = q.shape[1]
        a.cu_seqlens = ctypes.c_void_p(1)
    else:
        a.batch, a.seqlen, a.num_seqs = q.shape[0], q.shape[1], q.shape[0]
        a.num_heads = q.shape[2]
    return int(lib().kda_prefill_workspace_size(ctypes.byref(a)))


def workspace_layout(q, *, cu_seqlens=None):
    a = PrefillArgs()
    if cu_seqlens is not None:
        a.batch, a.seqlen, a.num_seqs, a.num_heads = 1, q.shape[0], cu_seqlens.shape[0] - 1, q.shape[1]
        a.cu_seqlens = ctypes.c_void_p(1)
    else:
        a.batch, a.seqlen, a.num_seqs, a.num_heads = q.shape[0], q.shape[1], q.shape[0], q.shape[2]
    L = WorkspaceLayout()
    _check(lib().kda_prefill_workspace_layout(ctypes.byref(a), ctypes.byref(L)))
    return L


def prefill_schedule(q, *, cu_seqlens=None, norm=False, num_sms=None):
    """The schedule kda_prefill runs for q's shape (kda_prefill_schedule):
    dict(segmented, whole_chain, segment_chunks, prep_ctas, scan_segments,
    scan_chunks).  Host only; q may
    live anywhere (only its shape is read).  num_sms defaults to the current
    CUDA device's SM count."""
    a = PrefillArgs()
    if cu_seqlens is not None:
        a.batch, a.seqlen, a.num_seqs, a.num_heads = 1, q.shape[0], cu_seqlens.shape[0] - 1, q.shape[1]
        a.cu_seqlens = ctypes.c_void_p(1)
    else:
        a.batch, a.seqlen, a.num_seqs, a.num_heads = q.shape[0], q.shape[1], q.shape[0], q.shape[2]
    if norm:
        a.out_gate = ctypes.c_void_p(1)
    if num_sms is None:
        num_sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    a.overrides = _current_overrides()
    sch = Schedule()
    _check(lib().kda_prefill_schedule(ctypes.byref(a), int(num_sms), ctypes.byref(sch)))
    return dict(segmented=bool(sch.segmented), whole_chain=bool(sch.whole_chain),
                segment_chunks=sch.segment_chunks, prep_ctas=sch.prep_ctas,
                scan_segments=sch.scan_segments, scan_chunks=sch.scan_chunks)


def kda_prefill(q, k, v, g, beta, *, initial_state=None, cu_seqlens=None, chunk=CHUNK,
                beta_is_logit=True, scale=1.0, out=None, final_state=None,
                output_final_state=True, workspace=None, device_status=None, stream=None,
                prep_only=False, stage=None, out_gate=None, norm_weight=None, norm_eps=1e-6):
    """KDA prefill through the C ABI.

    Padded: q, k, g [B, T, H, 128]; v [B, T, H, 128]; beta [B, T, H].
    Varlen: q, k, g [T_total, H, 128]; beta [T_total, H]; cu_seqlens int32 [N+1]
    on the device.  initial_state fp32 [N, H, 128, 128] or None.
    Returns (out, final_state); with prep_only=True runs steps A1-A5 only and
    returns (workspace, layout).  stage="prep" / "state" run one stage alone
    (the state stage reads the records a previous "prep" call left in
    `workspace`) and return (out, final_state).
    """
    N = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else q.shape[0]
    H = q.shape[-2]
    # Tensors made here belong to the stream the kernels run on, so that the
    # caching allocator cannot hand their memory to other work while the
    # call's kernels still use it.
    with _on_stream(stream, q):
        if out is None:
            out = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device)
        if final_state is None and output_final_state and not prep_only:
            final_state = torch.empty((N, H, q.shape[-1], v.shape[-1]), dtype=torch.float32,
                                      device=q.device)
        if workspace is None:
            nbytes = workspace_size(q, v, cu_seqlens=cu_seqlens)
            workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    a = _prefill_args(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                      beta_is_logit, scale, workspace, device_status, chunk, out_gate, norm_weight,
                      norm_eps)
    fn = {None: lib().kda_prefill, "prep": lib().kda_prefill_prep,
          "state": lib().kda_prefill_state}[stage]
    if prep_only:
        fn = lib().kda_prefill_prep
    _check(fn(ctypes.byref(a), _stream_handle(stream)))
    if prep_only:
        return workspace, workspace_layout(q, cu_seqlens=cu_seqlens)
    return out, final_state


def kda_verify(q, k, v, g, beta, state_pool, accepted, *, slot=None, beta_is_logit=True,
               scale=1.0, out=None, device_status=None, stream=None, replay_only=False):
    """MTP verify through the C ABI; state_pool is updated in place.

    q, k, g [R, D, H, 128]; v [R, D, H, 128]; beta [R, D, H]; state_pool fp32 or
    bf16 [P, H, 128, 128]; accepted (and slot) int32 [R] on the device.  Returns
    out; with replay_only=True only the accepted drafts run, the states are
    stored and nothing else is written (returns None).
    """
    if state_pool is None or state_pool.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("state_pool must be a fp32 or bf16 CUDA tensor")
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.float32), ("state_pool", state_pool, state_pool.dtype),
                        ("accepted", accepted, torch.int32), ("slot", slot, torch.int32),
                        ("device_status", device_status, torch.int32)):
        _need_cuda(name, t, dt)
    if not state_pool.is_contiguous():
        raise ValueError("state_pool must be contiguous [P, H, 128, 128]")
    if out is None and not replay_only:
        with _on_stream(stream, v):
            out = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device)
    if out is not None:
        _need_cuda("out", out, torch.bfloat16)
    a = VerifyArgs()
    a.q, a.k, a.v, a.g, a.beta, a.out = (_ptr(t) for t in (q, k, v, g, beta, out))
    a.pool_dtype = KDA_POOL_BF16 if state_pool.dtype == torch.bfloat16 else KDA_POOL_F32
    a.replay_only = 1 if replay_only else 0
    a.q_stride = _i64x3(*_strides3(q, False))
    a.k_stride = _i64x3(*_strides3(k, False))
    a.v_stride = _i64x3(*_strides3(v, False))
    a.g_stride = _i64x3(*_strides3(g, False))
    a.out_stride = _i64x3(*_strides3(out if out is not None else v, False))
    a.beta_stride = _i64x3(*_strides3(beta, False, last_is_channel=False))
    a.state_pool = _ptr(state_pool)
    a.pool_size = state_pool.shape[0]
    a.slot = _ptr(slot)
    a.accepted = _ptr(accepted)
    a.num_requests, a.num_drafts, a.num_heads = q.shape[0], q.shape[1], q.shape[2]
    a.head_dim_k, a.head_dim_v = q.shape[-1], v.shape[-1]
    a.beta_is_logit = 1 if beta_is_logit else 0
    a.scale = float(scale)
    a.device_status = _ptr(device_status)
    a.overrides = _current_overrides()
    _check(lib().kda_verify(ctypes.byref(a), _stream_handle(stream)))
    return out


NOALLOC_MAX_WORKSPACE_BYTES = 32 << 20


def kda_prefill_noalloc(q, k, v, g, beta, *, initial_state=None, cu_seqlens=None, chunk=CHUNK,
                        beta_is_logit=True, scale=1.0, out=None, final_state=None,
                        device_status=None, stream=None):
    """kda_prefill through the allocation-free entry point: the library uses its
    built-in scratch array instead of a workspace (see kda_prefill_noalloc in
    include/kda.h for the size limit and the rule that calls must not overlap
    on the GPU).  Outputs are still allocated here when not given."""
    L = lib()
    f = L.kda_prefill_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(PrefillArgs), _p]
    N = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else q.shape[0]
    with _on_stream(stream, q):
        if out is None:
            out = torch.empty(v.shape, dtype=torch.bfloat16, device=v.device)
        if final_state is None:
            final_state = torch.empty((N, q.shape[-2], q.shape[-1], v.shape[-1]),
                                      dtype=torch.float32, device=q.device)
    a = _prefill_args(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state,
                      beta_is_logit, scale, None, device_status, chunk)
    _check(f(ctypes.byref(a), _stream_handle(stream)))
    return out, final_state


def _host_args(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, beta_is_logit,
               scale, chunk, staging, piece_tokens, check=True):
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16),
                        ("v", v, torch.bfloat16), ("g", g, torch.float32),
                        ("beta", beta, torch.float32), ("out", out, torch.bfloat16),
                        ("initial_state", initial_state, torch.float32),
                        ("final_state", final_state, torch.float32)):
        if t is None or not check:
            continue
        if t.device.type != "cpu" or not t.is_pinned() or t.dtype != dt or not t.is_contiguous():
            raise ValueError("%s must be a contiguous page-locked host tensor of %s" % (name, dt))
    if cu_seqlens is not None and (cu_seqlens.device.type != "cpu" or cu_seqlens.dtype != torch.int32
                                   or not cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous host int32 tensor here")
    a = PrefillArgs()
    a.q, a.k, a.v, a.g, a.beta, a.out = (_ptr(t) for t in (q, k, v, g, beta, out))
    a.initial_state = _ptr(initial_state)
    a.final_state = _ptr(final_state)
    a.cu_seqlens = _ptr(cu_seqlens)
    if cu_seqlens is not None:
        a.batch, a.seqlen, a.num_seqs, a.num_heads = 1, q.shape[0], cu_seqlens.shape[0] - 1, q.shape[1]
    else:
        a.batch, a.seqlen, a.num_seqs, a.num_heads = q.shape[0], q.shape[1], q.shape[0], q.shape[2]
    a.head_dim_k, a.head_dim_v = q.shape[-1], v.shape[-1]
    a.chunk = int(chunk)
    a.beta_is_logit = 1 if beta_is_logit else 0
    a.scale = float(scale)
    h = PrefillHostArgs()
    h.args = a
    h.staging = _ptr(staging)
    h.staging_bytes = 0 if staging is None else staging.numel() * staging.element_size()
    h.piece_tokens = int(piece_tokens)
    return h


def host_staging_size(q, v, *, cu_seqlens=None, piece_tokens=0):
    """Bytes of device staging kda_prefill_host needs (q, v: host tensors)."""
    h = _host_args(q, q, v, None, None, None, cu_seqlens, None, None, True, 1.0, CHUNK, None,
                   piece_tokens, check=False)
    return int(lib().kda_prefill_host_staging_size(ctypes.byref(h)))


def kda_prefill_host(q, k, v, g, beta, *, initial_state=None, cu_seqlens=None, chunk=CHUNK,
                     beta_is_logit=True, scale=1.0, out=None, final_state=None,
                     output_final_state=True, staging=None, piece_tokens=0, stream=None):
    """KDA prefill with every tensor in page-locked host memory (cu_seqlens a host
    int32 tensor), through the C ABI's kda_prefill_host: the copies in and out
    overlap the kernels piece by piece.  Asynchronous on `stream`; returns the
    host (out, final_state), complete once the stream reaches this point."""
    N = (cu_seqlens.shape[0] - 1) if cu_seqlens is not None else q.shape[0]
    H = q.shape[-2]
    if out is None:
        out = torch.empty(v.shape, dtype=torch.bfloat16, pin_memory=True)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, q.shape[-1], v.shape[-1]), dtype=torch.float32, pin_memory=True)
    if staging is None:
        nbytes = host_staging_size(q, v, cu_seqlens=cu_seqlens, piece_tokens=piece_tokens)
        with (torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()):
            staging = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    h = _host_args(q, k, v, g, beta, initial_state, cu_seqlens, out, final_state, beta_is_logit,
                   scale, chunk, staging, piece_tokens)
    _check(lib().kda_prefill_host(ctypes.byref(h), _stream_handle(stream)))
    return out, final_state
