/*
 * kda.h -- C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * What it computes.  Per chain (one sequence and one head) with a 128 x 128
 * fp32 state S (row = key channel, column = value channel):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = scale * S_t^T q_t
 *
 * "Kimi Delta Attention (KDA) prefill" as named on the TensorRT-LLM page
 * "Kimi K3 KDA prefill: K1 warps finish reading sPartialLast before the next
 * chunk" (Description: in-chunk gate prefix scan and chunk total, fused beta
 * sigmoid, padded equal-length and varlen modes), with the dtypes of the
 * cuDNN-frontend sm90 KDA prefill page (Conversation: BF16 Q/K/V, FP32 gate,
 * beta and state, non-zero initial_state) and the short-chunk MTP verify of the
 * TensorRT-LLM page "Kimi K3 work for Rubin (SM107)" (Description: tcgen05 KDA
 * MTP verify kernel, WY-form chunk, fp32 state pools).
 *
 * Conventions shared by every call.
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device or pinned memory and caches none; scratch memory is
 *    the caller's `workspace`.  (It keeps one CUDA stream and two events per
 *    host thread and device for segmented prefill calls, see kda_prefill.)
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL
 *    = the legacy default stream).  Argument errors found on the host come
 *    back synchronously and launch nothing.
 *  - Element strides are in elements, not bytes.  The channel (last) dim must
 *    have stride 1; every other stride must be a multiple of 8 elements for
 *    bf16 tensors and 4 for fp32 tensors (16-byte rows for 128-bit / TMA
 *    loads), and every base pointer 16-byte aligned.  Layouts that break this
 *    are refused with KDA_ERR_UNSUPPORTED, never read wrongly (the stride
 *    finding on the cuDNN-frontend sm90 KDA page, Conversation).
 *  - head_dim_k = head_dim_v = 128 and chunk = 64 only; anything else is
 *    KDA_ERR_UNSUPPORTED.
 *  - Errors that only the device can see (cu_seqlens not non-decreasing or not
 *    ending at the token count, accepted or slot out of range, a bounded wait
 *    that ran out) are written as a kda_status value to *device_status when it
 *    is non-NULL (a caller-owned device int32 that the caller zeroes); the
 *    kernels then skip the offending work instead of faulting.
 *  - Per-device set-up (the kernels' shared-memory limits, the no-alloc
 *    scratch address) is done on a device's first call and remembered for the
 *    process; after cudaDeviceReset the library must not be called again in
 *    that process.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 6

/*
 * Test and measurement overrides of the library's own choices, passed per call
 * through kda_prefill_args.overrides / kda_verify_args.overrides (NULL = none).
 * Results stay within the stated tolerances whatever is selected (the
 * schedule choices give bitwise-equal results for a given state kernel).
 * Nothing is read from the process environment: a call's kernels and schedule
 * depend only on its arguments.
 *   state_kernel    0: library's choice, 1: 32-column slab CTAs, 2: one
 *                   whole-chain CTA per (sequence, head) (the fused norm
 *                   always takes 2)
 *   segment_chunks  -1: library's choice, 0: never segment, n > 0: segments of
 *                   n chunks (padded calls)
 *   prep_ctas       > 0: prep grid of a forced segmented call (0: choice)
 *   no_pdl          1: no programmatic launch between consecutive prep grids,
 *                   nor of the state pass after a one-pass call's prep
 *   stall_seed      != 0: the kernel instantiations with the stall hook, in
 *                   which a quarter of the warps at each injection site spin
 *                   for a pseudo-random 0..4095 cycles; every result must be
 *                   bit-identical to the run without it
 *   scan_segments   0: library's choice, 1: never run the segment-parallel
 *                   scan, n >= 2: run it with n segments per chain (padded
 *                   calls; clamped to the scan_max_segments of the workspace
 *                   layout, and not run when that is below 2)
 *   wait_limit_ns   > 0: bound of the kernels' working mbarrier waits instead
 *                   of 200 ms (a wait that runs out writes KDA_ERR_TIMEOUT to
 *                   the status word and the CTA winds down; the wind-down's own
 *                   waits for copies and products in flight keep 200 ms)
 *   timeout_probe   1: in every prep, state-pass and tensor-core verify CTA,
 *                   the first wait for a tensor-core product waits instead on
 *                   an mbarrier that nothing arrives on, so that it runs out
 *                   (after wait_limit_ns) with the product and tile copies
 *                   still in flight: the wind-down path, exercised without a
 *                   fault
 *   verify_kernel   kda_verify: 0 library's choice, 1 the sequential kernel
 *                   (every draft on the CUDA cores in fp32), 2 the tensor-core
 *                   kernel (the drafts as one WY-form chunk)
 */
typedef struct kda_overrides {
    int32_t state_kernel;
    int32_t segment_chunks;
    int32_t prep_ctas;
    int32_t no_pdl;
    uint32_t stall_seed;
    int32_t scan_segments;
    int64_t wait_limit_ns;
    int32_t timeout_probe;
    int32_t verify_kernel;
} kda_overrides;

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1,  /* bad pointer / size / cu_seqlens / accepted / slot */
    KDA_ERR_UNSUPPORTED = 2,  /* valid but not supported: dims, chunk, strides, alignment */
    KDA_ERR_CUDA = 3,         /* a CUDA runtime or driver call failed */
    KDA_ERR_TIMEOUT = 4       /* (device_status only) a bounded on-chip wait ran out */
} kda_status;

/*
 * Prefill arguments.
 *
 * Padded mode (cu_seqlens == NULL): B = batch sequences of T = seqlen tokens.
 *   q, k: bf16, g: fp32, element (b, t, h, c) at b*s[0] + t*s[1] + h*s[2] + c
 *   v, out: bf16 (b, t, h, j) likewise with their own strides
 *   beta: fp32 (b, t, h) at b*s[0] + t*s[1] + h*s[2]
 *   num_seqs must equal batch.
 * Varlen mode (cu_seqlens != NULL): num_seqs = N packed sequences over
 *   seqlen = T_total tokens; cu_seqlens is a DEVICE int32 [N+1] with
 *   cu[0] = 0, cu[n] <= cu[n+1], cu[N] = T_total; sequence n owns tokens
 *   cu[n] .. cu[n+1]-1; batch must be 1 and stride [0] is ignored.
 *   Zero-length sequences are allowed: they produce no outputs and their final
 *   state equals their initial state.
 * initial_state: fp32 [N, H, 128, 128] contiguous (row = key) or NULL = zeros.
 * final_state:   fp32 [N, H, 128, 128] contiguous or NULL = not stored.  It may
 *   alias initial_state (in-place update).
 * beta_is_logit: 1 = beta holds logits b and the kernel uses sigmoid(b) (the
 *   fused beta sigmoid); 0 = beta already holds beta in [0, 1].
 * g: log decay per key channel, g <= 0.  Inside the 16-token blocks of a chunk
 *   the interaction terms use the per-token gate floored at -5.4 (the chunk
 *   factorisation's guard against exp overflow): exact for gates >= -5.4 (the
 *   production gate bound is -5), otherwise a term whose true decay is below
 *   e^-5.4 is replaced by one that is also below e^-5.4.  The inter-chunk state
 *   recurrence always uses the exact gates.
 * scale: multiplies q (o_t = scale * S_t^T q_t); 1.0 for the plain recurrence.
 * workspace: device scratch of at least kda_prefill_workspace_size(args) bytes,
 *   256-byte aligned, owned by the caller, used only during the call's kernels
 *   (so it may be reused by the next call on the same stream).
 * Size limits: num_seqs <= 65535 and num_heads <= 65535 per call (the state
 *   pass gives every (sequence, head) chain its own CTA and indexes sequences
 *   and heads by grid dimensions), seqlen < 2^31; larger calls return
 *   KDA_ERR_UNSUPPORTED and launch nothing (split the batch).
 */
typedef struct kda_prefill_args {
    const void* q;              /* bf16 */
    const void* k;              /* bf16 */
    const void* v;              /* bf16 */
    const float* g;             /* fp32 */
    const float* beta;          /* fp32 */
    void* out;                  /* bf16 */
    int64_t q_stride[3];        /* (batch, token, head) element strides */
    int64_t k_stride[3];
    int64_t v_stride[3];
    int64_t g_stride[3];
    int64_t beta_stride[3];
    int64_t out_stride[3];
    const float* initial_state; /* fp32 [N,H,128,128] or NULL */
    float* final_state;         /* fp32 [N,H,128,128] or NULL */
    const int32_t* cu_seqlens;  /* device int32 [N+1] or NULL (padded) */
    int64_t batch;              /* padded: B; varlen: 1 */
    int64_t seqlen;             /* padded: T; varlen: T_total */
    int64_t num_seqs;           /* N (padded: = batch) */
    int64_t num_heads;          /* H >= 1 */
    int64_t head_dim_k;         /* must be 128 */
    int64_t head_dim_v;         /* must be 128 */
    int32_t chunk;              /* must be 64 */
    int32_t beta_is_logit;
    float scale;
    void* workspace;
    size_t workspace_bytes;
    int32_t* device_status;     /* optional device int32 */
    /* Gated RMSNorm fused into the output (out_gate == NULL: off).  A reading of
     * the "gated RMSNorm in the epilogue (fuse_output_norm)" of the TensorRT-LLM
     * page "Kimi K3 work for Rubin (SM107)" (Description), which names it
     * without a formula: per (token, head), over the 128 value channels c,
     *   out_c = o_c / sqrt(mean_c(o_c^2) + norm_eps) * norm_weight[c] * sigmoid(gate_c)
     * with o the attention output in fp32 before rounding.  out_gate: bf16,
     * element (b, t, h, c) at b*gate_stride[0] + t*gate_stride[1] +
     * h*gate_stride[2] + c; norm_weight: fp32 [128].  Both or neither;
     * 16-byte aligned rows (strides multiples of 8) and weight, else
     * KDA_ERR_UNSUPPORTED.  With the norm on, the state pass always runs one CTA
     * per chain (the norm needs whole output rows). */
    const void* out_gate;
    int64_t gate_stride[3];
    const float* norm_weight;
    float norm_eps;
    const kda_overrides* overrides;   /* NULL: the library's choices (see kda_overrides) */
} kda_prefill_args;

/*
 * Bytes of workspace kda_prefill needs for these arguments (depends only on
 * batch, seqlen, num_seqs and num_heads).  Returns 0 if args is NULL.
 */
size_t kda_prefill_workspace_size(const kda_prefill_args* args);

/*
 * KDA prefill: out for every token and (if final_state) the final state of
 * every chain.  Runs the chunked form with 64-token chunks:
 *   A1 chunk table from cu_seqlens (gap-safe for zero-length sequences:
 *      cuDNN-frontend sm90 KDA page, Conversation, "virtual chunk mapping");
 *   A2-A5 per-chunk prep: in-chunk gate cumsum and chunk total, beta sigmoid,
 *      tail masking, gate-scaled operands, the UT transform
 *      (I + Diag(beta) tril(K K^T . decay))^{-1}, W, U and the intra-chunk
 *      attention matrix Aqk;
 *   A6-A7 the serial inter-chunk state pass on tcgen05 tensor cores, per
 *      (sequence, head) chain in four 32-column slab CTAs or one whole-chain
 *      CTA, with the output epilogue (rows stored by TMA tensor stores).
 * Padded calls with few, long chains are run in token segments: the state
 * pass of segment s (on a second stream, joined back into `stream` before
 * the call's work ends) overlaps the prep of segment s+1, which a second prep
 * grid on that stream joins once the state pass ends (both take the
 * segment's records from its counter in prep_counters); the state of every
 * chain passes between segments in fp32 through the workspace's state_carry
 * region, so the results are those of one state pass over the whole
 * sequence.
 * Padded calls with very few chains may instead run the segment-parallel
 * inter-chunk scan (the seg / comb kernels of the cuDNN-frontend sm90 KDA
 * page, Conversation): each chain's chunks are cut into n segments; for every
 * segment but the last, the transition M (the state map of the segment's
 * chunks, taken from the identity with U read as zero) and the offset C (the
 * state the segment leaves from a zero entry) are computed in parallel; a
 * combine kernel then forms the entry states E_{s+1} = M_s E_s + C_s in fp32
 * in a fixed order (E_0 = initial_state), and the outputs of all segments are
 * computed in parallel from their entry states.  The result is deterministic
 * and within the stated tolerances, but not bitwise that of the one-pass
 * state recurrence (the state's rounding path differs).  The second stream and two events are created on a host
 * thread's first segmented call on a device and kept for the thread's life
 * (calls of one thread share them), so segmented calls can be captured into a
 * CUDA graph once one has run outside the capture.
 * Returns KDA_OK once the kernels are enqueued.
 *
 * Segmented calls of one host thread share its second stream, so the state
 * passes of two such calls made from one thread on different caller streams
 * run one after the other (results are unaffected; give each concurrent
 * caller stream its own host thread to overlap them).
 *
 * Tests and measurements can override the kernel and schedule choices per
 * call through args->overrides (see kda_overrides).
 */
kda_status kda_prefill(const kda_prefill_args* args, void* stream);

/*
 * The schedule kda_prefill would run for these arguments on a GPU with
 * num_sms SMs (host only: no device call; honours args->overrides as
 * kda_prefill does).  segmented: 1 if the tokens are cut into
 * segments of segment_chunks chunks, the state pass of one beside the prep
 * of the next, prep on prep_ctas CTAs; whole_chain: 1 if the state pass runs
 * one CTA per chain (all 128 value columns), 0 for four 32-column slab CTAs
 * per chain; scan_segments: n >= 2 if the call runs the segment-parallel scan
 * with n segments of scan_chunks chunks (whole-chain CTAs; then segmented is
 * 0), else 0.  KDA_ERR_INVALID_ARG for NULL pointers or num_sms < 1.
 */
typedef struct kda_schedule {
    int32_t segmented, whole_chain, segment_chunks, prep_ctas;
    int32_t scan_segments, scan_chunks;
} kda_schedule;
kda_status kda_prefill_schedule(const kda_prefill_args* args, int num_sms, kda_schedule* schedule);

/*
 * Runs only steps A1-A5 of kda_prefill and leaves the per-chunk operands in
 * the workspace, laid out as kda_prefill_workspace_layout describes.  Meant for
 * testing the stages one at a time.
 */
kda_status kda_prefill_prep(const kda_prefill_args* args, void* stream);

/*
 * Runs only steps A6-A7 of kda_prefill: the serial state pass and the output
 * epilogue, reading the per-chunk records that a previous kda_prefill_prep
 * with the same arguments and workspace left there.  Together the two calls
 * do exactly what kda_prefill does; split, each stage can be timed alone.
 */
kda_status kda_prefill_state(const kda_prefill_args* args, void* stream);

/*
 * Workspace layout (byte offsets from `workspace`) of the per-chunk records
 * that kda_prefill_prep writes.  Record r = chunk * H + head (chunk is the
 * global chunk index; sequence n owns chunks chunk_offset[n] ..
 * chunk_offset[n+1]-1 in token order) starts at records + r * record_bytes and
 * holds shared-memory images of the state pass's operands.  bf16 images use
 * the 128-byte swizzle (16-byte chunk c of 128-byte row x stored at
 * x*128 + ((c ^ (x mod 8)) * 16)):
 *   [0, 32768)        [Q e^Gam ; W] bf16: key channels 0-63 then 64-127,
 *                     each 128 rows x 128 B; rows 0-63 scale*Q e^Gam, rows
 *                     64-127 W = T Diag(beta)(K e^Gam)
 *   [32768, 49152)    Kt fp16: 128 key rows x 64 tokens, (K e^{gam - Gam})^T
 *   [49152, 57344)    Aqk fp16: 64 token rows x 64 tokens, the masked
 *                     (j <= i) gate-decayed scale*Q K^T of the chunk
 *   [57344, 73728)    U^T bf16, U = T Diag(beta) V: 128 value rows x 64
 *                     tokens (128 B, the swizzle above)
 *   [73728, 74240)    exp(gam) fp32 [128], gam = chunk total of g
 * Rows past a tail chunk's length are zero.  chunk_offset: int32 [N+1].
 * seq_order (varlen): the sequences by descending chunk count (ties by index;
 * index order beyond 1024 sequences), the order in which the state pass's
 * CTAs take them.
 * A segmented kda_prefill (see there) keeps the records of each token segment
 * together: segment s's records follow those of segments 0..s-1, numbered
 * as above within the segment.
 * prep_counters (padded calls): int32 [chunks per sequence + 1], one
 * record counter per segment of a segmented call, from which the prep CTAs of
 * that segment take their records (set to zero at the start of the call).
 * scan (padded calls with at most 64 chains and at least 128 chunks per
 * sequence): room for the segment-parallel scan with up to scan_max_segments
 * = min(32, chunks per sequence / 64) segments: the segments' transitions and
 * offsets, fp32 [(scan_max_segments - 1) * 2, B * H, 128, 128] (block
 * (2 s + w) * B * H + chain, w = 0 transition, 1 offset), then the entry
 * states fp32 [scan_max_segments, B * H, 128, 128].
 */
typedef struct kda_workspace_layout {
    size_t records, record_bytes, chunk_offset, status, total;
    int64_t max_chunks;         /* records per head */
    size_t state_carry;         /* padded calls: fp32 [B, H, 128, 128] */
    size_t seq_order;           /* varlen calls: int32 [N], sequences longest first */
    size_t scan;                /* padded calls: segment-parallel scan buffers (see above) */
    int64_t scan_max_segments;  /* 0 when the layout has no scan room */
    size_t prep_counters;       /* padded calls: int32 per segment (see above) */
} kda_workspace_layout;
kda_status kda_prefill_workspace_layout(const kda_prefill_args* args,
                                        kda_workspace_layout* layout);

/* State pool element types of kda_verify. */
#define KDA_POOL_F32 0
#define KDA_POOL_BF16 1

/*
 * MTP verify: R requests, each with D <= 16 draft tokens, run against a fp32
 * or bf16 state pool (both are accepted, as on the TensorRT-LLM page "Kimi K3
 * work for Rubin (SM107)", Description).  A bf16 pool is read widened to fp32,
 * the drafts run in fp32, and the state written back is rounded to nearest
 * even; it halves the pool traffic.  For request r and head h the state is read from
 * state_pool[slot[r], h] (slot == NULL: slot r), all D drafts go through the
 * recurrence in order and produce outputs, and the state after the first
 * accepted[r] drafts is written back to the same pool slot (accepted 0 leaves
 * it unchanged).  Each state is read before it is written; slots must be
 * distinct across requests.
 *   q, k: bf16, g: fp32, element (r, t, h, c) at r*s[0] + t*s[1] + h*s[2] + c
 *   v, out: bf16 likewise; beta: fp32 (r, t, h)
 *   state_pool: fp32 or bf16 (pool_dtype) [pool_size, H, 128, 128] contiguous
 *   slot, accepted: device int32 [R]; accepted[r] in 0..D, slot[r] in
 *   0..pool_size-1 (out-of-range entries are skipped and reported through
 *   device_status)
 * replay_only = 1 is the commit of accepted drafts (the replay-only mode of
 * the same page): for each request only its first accepted[r] drafts run, no
 * output is written (out may be NULL) and the state after them is stored;
 * accepted 0 leaves the state unchanged.
 * Draft rows and state blocks are moved in 16-byte pieces, so q, k, v, g and
 * state_pool must be 16-byte aligned, the q/k/v strides multiples of 8
 * elements and the g strides multiples of 4; otherwise KDA_ERR_UNSUPPORTED and
 * nothing is launched.  Size limits: R <= 65535, H <= 65535, R * H < 2^31 and
 * pool_size <= 2^30 (else KDA_ERR_UNSUPPORTED).
 */
typedef struct kda_verify_args {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    void* out;
    int64_t q_stride[3];        /* (request, draft, head) element strides */
    int64_t k_stride[3];
    int64_t v_stride[3];
    int64_t g_stride[3];
    int64_t beta_stride[3];
    int64_t out_stride[3];
    void* state_pool;           /* fp32 or bf16 (pool_dtype) [pool_size, H, 128, 128] */
    int64_t pool_size;
    const int32_t* slot;        /* device int32 [R] or NULL */
    const int32_t* accepted;    /* device int32 [R] */
    int64_t num_requests;       /* R */
    int64_t num_drafts;         /* D, 1..16 */
    int64_t num_heads;
    int64_t head_dim_k;         /* must be 128 */
    int64_t head_dim_v;         /* must be 128 */
    int32_t beta_is_logit;
    float scale;
    int32_t* device_status;     /* optional device int32 */
    int32_t pool_dtype;         /* KDA_POOL_F32 or KDA_POOL_BF16 */
    int32_t replay_only;        /* 1: commit mode, see above */
    const kda_overrides* overrides;   /* NULL: none; stall_seed, wait_limit_ns,
                                         timeout_probe and verify_kernel apply */
} kda_verify_args;

kda_status kda_verify(const kda_verify_args* args, void* stream);

/*
 * kda_prefill for callers that cannot allocate device memory.  (The pages have
 * no counterpart to this call; it exists for users of this library.)
 *
 * Who needs it: code that runs inside another runtime's fixed device-memory
 * budget, or in a latency-critical loop where cudaMalloc is not allowed (it can
 * synchronise the device and fragment a memory pool), and therefore cannot hand
 * kda_prefill a workspace.  Same arguments and results as kda_prefill, except
 * that `workspace` / `workspace_bytes` are ignored: the call uses a scratch
 * array of KDA_NOALLOC_MAX_WORKSPACE_BYTES compiled into the library, which
 * every GPU that loads the library keeps in device memory until the process
 * exits.  The caller still passes (and owns) all inputs and outputs.
 *
 * Limits and behaviour:
 *  - Returns KDA_ERR_UNSUPPORTED, launching nothing, when
 *    kda_prefill_workspace_size(args) exceeds KDA_NOALLOC_MAX_WORKSPACE_BYTES
 *    (about 450 chunk-head records of 74,240 bytes, less 64 KB of state per
 *    padded chain: e.g. 2048 tokens x 13 heads, or 8192 tokens x 3 heads).
 *  - The first call on each device looks up the array's device address for
 *    that device (with the device current); make that first call before any
 *    stream capture.  It allocates nothing, here or later.
 *  - Every call on a device shares the one array.  Calls whose kernels overlap
 *    on the GPU (different streams, or different host threads) race on it and
 *    give wrong results: serialise them.  Nothing in the array needs to start
 *    at zero; each call writes what it later reads.
 */
#define KDA_NOALLOC_MAX_WORKSPACE_BYTES ((size_t)32 << 20)
kda_status kda_prefill_noalloc(const kda_prefill_args* args, void* stream);

/*
 * kda_prefill for inputs and outputs that live in host memory.  (The pages have
 * no counterpart; this is a runtime entry of this library for callers that keep
 * their tensors on the host.)
 *
 * args: as for kda_prefill, except that q, k, v, g, beta, out, initial_state and
 * final_state point to PAGE-LOCKED HOST memory (cudaHostAlloc or
 * cudaHostRegister) in the contiguous layouts (padded: q/k/v/g/out
 * [B, T, H, 128], beta [B, T, H]; varlen: [T_total, H, 128] and [T_total, H]),
 * cu_seqlens (varlen) is a HOST int32 array [N + 1], and the stride, workspace
 * and workspace_bytes fields are ignored; the fused output norm is not
 * available here (out_gate must be NULL, else KDA_ERR_UNSUPPORTED).
 * staging: caller-owned device memory, 256-byte aligned, at least
 * kda_prefill_host_staging_size(args) bytes; piece_tokens: tokens per piece, a
 * multiple of 64, or 0 for the library's choice (about a thirty-second of the
 * input, at least 2048 tokens).
 *
 * The work is cut into pieces (padded: a range of chunk-aligned tokens of every
 * sequence, with each chain's state carried from piece to piece on the device,
 * so the result is bitwise that of one kda_prefill call; varlen: runs of whole
 * sequences).  Piece p + 1 is copied in while piece p runs and each piece's
 * output is copied out while later pieces run, on two copy streams (created
 * on a host thread's first call on a device and kept for the thread's life,
 * like kda_prefill's second stream), ordered after the work already on
 * `stream`; when
 * `stream` reaches the point after this call, every output is in host memory.
 * The host buffers and the staging memory must stay valid until then.  Errors:
 * KDA_ERR_INVALID_ARG for missing pointers, unusable shapes or cu_seqlens, or a
 * small / misaligned staging area (nothing is launched); otherwise the statuses
 * of kda_prefill.
 */
typedef struct kda_prefill_host_args {
    kda_prefill_args args;
    void* staging;
    size_t staging_bytes;
    int64_t piece_tokens;
} kda_prefill_host_args;
size_t kda_prefill_host_staging_size(const kda_prefill_host_args* args);
kda_status kda_prefill_host(const kda_prefill_host_args* args, void* stream);

/* Static string naming a status code. */
const char* kda_status_string(kda_status status);

/* KDA_ABI_VERSION of the loaded library. */
int kda_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KDA_H */
