// kda_api.cu -- the C ABI of include/kda.h: host-side argument checks, the
// workspace plan, TMA descriptors and the kernel launches.  Nothing here
// allocates or caches device memory.
#include <stdlib.h>
#include <string.h>

#include "../../include/kda.h"
#include "kda_internal.h"
#include "sm103.cuh"
#include "tmap.h"

using namespace kda;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Upper bound on chunk records per head.
int64_t max_chunks_of(const kda_prefill_args* a) {
    if (a->cu_seqlens == nullptr) return a->batch * ((a->seqlen + kChunk - 1) / kChunk);
    return a->seqlen / kChunk + a->num_seqs;
}

// Segments the workspace has room for in the segment-parallel scan: padded
// calls with at most 64 chains and at least 128 chunks per sequence, one
// segment per 64 chunks up to 32 (0: no scan room).
constexpr int64_t kScanMaxChains = 64, kScanChunksPerSegment = 64;
int64_t scan_max_segments(const kda_prefill_args* a) {
    if (a->cu_seqlens != nullptr || a->batch < 1 || a->num_heads < 1) return 0;
    if (a->batch * a->num_heads > kScanMaxChains) return 0;
    const int64_t cps = (a->seqlen + kChunk - 1) / kChunk;
    const int64_t n = cps / kScanChunksPerSegment;
    if (n < 2) return 0;
    return n < kScanMaxSegments ? n : kScanMaxSegments;
}

bool layout_of(const kda_prefill_args* a, kda_workspace_layout* L) {
    if (a->num_heads < 1 || a->seqlen < 0 || a->num_seqs < 0 || a->batch < 0) return false;
    // Sizes that cannot be described in size_t (with room for the alignment of
    // every region) are refused rather than wrapped.
    constexpr int64_t kMaxDim = (int64_t)1 << 40;
    if (a->seqlen > kMaxDim || a->num_seqs > kMaxDim || a->batch > kMaxDim || a->num_heads > kMaxDim)
        return false;
    const int64_t mc = max_chunks_of(a);
    if (mc < 0) return false;
    const size_t limit = SIZE_MAX / 4;
    if ((size_t)mc > limit / (size_t)a->num_heads) return false;
    const size_t nrec = (size_t)mc * (size_t)a->num_heads;
    if (nrec > limit / kRecBytes) return false;
    const size_t chains = (size_t)(a->cu_seqlens ? a->num_seqs : a->batch);
    if (chains > limit / ((size_t)a->num_heads * kHeadDim * kHeadDim * sizeof(float))) return false;
    size_t o = 0;
    L->max_chunks = mc;
    L->record_bytes = kRecBytes;
    L->records = o; o = align_up(o + nrec * kRecBytes);
    L->chunk_offset = o; o = align_up(o + sizeof(int32_t) * (size_t)(a->num_seqs + 1));
    L->seq_order = o; o = align_up(o + (a->cu_seqlens ? sizeof(int32_t) * (size_t)a->num_seqs : 0));
    L->status = o; o = align_up(o + sizeof(int32_t));
    // padded calls: one record counter per segment of the segmented schedule
    const size_t counters =
        a->cu_seqlens == nullptr ? sizeof(int32_t) * (size_t)((a->seqlen + kChunk - 1) / kChunk + 1) : 0;
    L->prep_counters = o; o = align_up(o + counters);
    // padded calls: the state of every chain between two segments of the
    // segmented schedule (run_prefill)
    const size_t carry = a->cu_seqlens == nullptr
                             ? (size_t)a->batch * (size_t)a->num_heads * kHeadDim * kHeadDim * sizeof(float)
                             : 0;
    L->state_carry = o; o = align_up(o + carry);
    // padded calls with few, long chains: the segment-parallel scan's operators
    // and entry states
    const int64_t smax = scan_max_segments(a);
    L->scan_max_segments = smax;
    const size_t blk = (size_t)kHeadDim * kHeadDim * sizeof(float);
    const size_t scan = smax >= 2 ? (size_t)(3 * smax - 2) * chains * (size_t)a->num_heads * blk : 0;
    L->scan = o; o = align_up(o + scan);
    L->total = o;
    return true;
}

bool strides_ok(const int64_t* s, int64_t mult) {
    for (int i = 0; i < 3; ++i)
        if (s[i] < 0 || (s[i] % mult) != 0) return false;
    return true;
}

// Every argument check of a prefill call except the workspace.
kda_status check_args(const kda_prefill_args* a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->head_dim_k != kHeadDim || a->head_dim_v != kHeadDim || a->chunk != kChunk)
        return KDA_ERR_UNSUPPORTED;
    if (a->num_heads < 1 || a->seqlen < 0 || a->num_seqs < 0 || a->batch < 0)
        return KDA_ERR_INVALID_ARG;
    if (a->cu_seqlens == nullptr) {
        if (a->num_seqs != a->batch) return KDA_ERR_INVALID_ARG;
    } else {
        if (a->batch != 1 || a->num_seqs < 1) return KDA_ERR_INVALID_ARG;
    }
    const bool tokens = a->seqlen > 0 && a->num_seqs > 0;
    if (tokens && (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out))
        return KDA_ERR_INVALID_ARG;
    if (tokens) {
        if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) ||
            !aligned16(a->out))
            return KDA_ERR_UNSUPPORTED;
        if (!strides_ok(a->q_stride, 8) || !strides_ok(a->k_stride, 8) ||
            !strides_ok(a->v_stride, 8) || !strides_ok(a->out_stride, 8) ||
            !strides_ok(a->g_stride, 4) || !strides_ok(a->beta_stride, 1))
            return KDA_ERR_UNSUPPORTED;
    }
    if ((a->initial_state && !aligned16(a->initial_state)) ||
        (a->final_state && !aligned16(a->final_state)))
        return KDA_ERR_UNSUPPORTED;
    // fused gated RMSNorm: both operands or neither
    if ((a->out_gate != nullptr) != (a->norm_weight != nullptr)) return KDA_ERR_INVALID_ARG;
    if (a->out_gate && (!aligned16(a->out_gate) || !aligned16(a->norm_weight) ||
                        !strides_ok(a->gate_stride, 8) || !(a->norm_eps >= 0.f)))
        return KDA_ERR_UNSUPPORTED;
    // the state kernels index sequences and heads by grid dimensions (at most 65535)
    if (a->num_seqs > 65535 || a->num_heads > 65535 || a->seqlen > INT32_MAX)
        return KDA_ERR_UNSUPPORTED;
    kda_workspace_layout L;
    if (!layout_of(a, &L)) return KDA_ERR_INVALID_ARG;
    if (a->overrides && a->overrides->scan_segments < 0) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

// The checks of check_args plus the caller's workspace.
kda_status check_prefill(const kda_prefill_args* a) {
    const kda_status st = check_args(a);
    if (st != KDA_OK) return st;
    kda_workspace_layout L;
    layout_of(a, &L);
    if (!a->workspace || a->workspace_bytes < L.total) return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a->workspace) & (kAlign - 1)) != 0) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

// Draft count from which kda_verify takes the tensor-core kernel by itself.
constexpr int kVerifyWyMinDrafts = 17;

// The call's overrides (tests and measurements), or the library's defaults.
kda_overrides overrides_of(const kda_overrides* o) {
    kda_overrides r;
    memset(&r, 0, sizeof(r));
    r.segment_chunks = -1;
    if (o) r = *o;
    return r;
}
uint64_t wait_limit_of(const kda_overrides& o) {
    return o.wait_limit_ns > 0 ? (uint64_t)o.wait_limit_ns : kWaitLimitNs;
}

void fill_params(const kda_prefill_args* a, const kda_workspace_layout& L, PrefillParams* p) {
    memset(p, 0, sizeof(*p));
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    p->q = static_cast<const __nv_bfloat16*>(a->q);
    p->k = static_cast<const __nv_bfloat16*>(a->k);
    p->v = static_cast<const __nv_bfloat16*>(a->v);
    p->g = a->g;
    p->beta = a->beta;
    p->out = static_cast<__nv_bfloat16*>(a->out);
    for (int i = 0; i < 3; ++i) {
        p->qs[i] = a->q_stride[i]; p->ks[i] = a->k_stride[i]; p->vs[i] = a->v_stride[i];
        p->gs[i] = a->g_stride[i]; p->bs[i] = a->beta_stride[i]; p->os[i] = a->out_stride[i];
    }
    p->h0 = a->initial_state;
    p->hT = a->final_state;
    p->cu = a->cu_seqlens;
    p->chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_offset);
    p->seq_order = a->cu_seqlens ? reinterpret_cast<int32_t*>(ws + L.seq_order) : nullptr;
    p->status = a->device_status ? a->device_status : reinterpret_cast<int32_t*>(ws + L.status);
    p->B = (int)a->batch;
    p->T = (int)a->seqlen;
    p->N = (int)a->num_seqs;
    p->H = (int)a->num_heads;
    p->max_chunks = (int)L.max_chunks;
    p->beta_is_logit = a->beta_is_logit ? 1 : 0;
    p->scale = a->scale;
    p->ws_rec = ws + L.records;
    p->gate = static_cast<const __nv_bfloat16*>(a->out_gate);
    for (int i = 0; i < 3; ++i) p->gts[i] = a->gate_stride[i];
    p->norm_w = a->norm_weight;
    p->norm_eps = a->norm_eps;
    const kda_overrides o = overrides_of(a->overrides);
    p->stall_seed = o.stall_seed;
    p->wait_ns = wait_limit_of(o);
    p->timeout_probe = o.timeout_probe ? 1 : 0;
}

// 4-D input tensor map [channel 128, head, token, batch] with one chunk of
// one head per box.  Returns false if the driver refuses the layout.
bool make_input_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esize,
                    const int64_t* st, int64_t H, int64_t T, int64_t B) {
    const uint64_t tstride = (uint64_t)st[1] * esize;
    const uint64_t bstride = st[0] != 0 ? (uint64_t)st[0] * esize : tstride * (uint64_t)(T > 0 ? T : 1);
    const uint64_t dims[4] = {128, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)st[2] * esize, tstride, bstride};
    const uint32_t box[4] = {128, 1, (uint32_t)kChunk, 1};
    return make_tensor_map(m, dt, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Tensor map of out for the state kernels' tensor stores: [channel
// 128, head, token, batch] with the caller's strides, box [32, 1, 64, 1] and the
// 64-byte swizzle (the layout of the records' value slabs).  base and T are
// those of the launch (a segment's own).  False if the driver refuses the
// layout; the kernel then stores rows one by one.
bool make_out_map(CUtensorMap* m, const kda_prefill_args* a, const void* base, int64_t T) {
    const int64_t B = a->cu_seqlens ? 1 : a->batch, H = a->num_heads;
    if (T <= 0 || B <= 0 || !base) return false;
    const int64_t* st = a->out_stride;
    const uint64_t tstride = (uint64_t)st[1] * 2;
    const uint64_t bstride = st[0] != 0 ? (uint64_t)st[0] * 2 : tstride * (uint64_t)T;
    const uint64_t dims[4] = {128, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)st[2] * 2, tstride, bstride};
    const uint32_t box[4] = {32, 1, (uint32_t)kChunk, 1};
    return make_tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_64B);
}

// Launches the state pass of `p` with the chosen kernel.
cudaError_t launch_state_pass(const kda_prefill_args* a, PrefillParams p, bool head, cudaStream_t s,
                              bool after_prep = false) {
    CUtensorMap om;
    memset(&om, 0, sizeof(om));
    p.out_tma = make_out_map(&om, a, p.out, p.T) ? 1 : 0;
    return head ? launch_state_head(p, om, s, after_prep) : launch_state(p, om, s, after_prep);
}

bool make_prep_maps(const kda_prefill_args* a, PrepMaps* m) {
    const int64_t T = a->seqlen, B = a->cu_seqlens ? 1 : a->batch, H = a->num_heads;
    if (T == 0 || B == 0) return true;
    return make_input_map(&m->q, a->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->q_stride, H, T, B) &&
           make_input_map(&m->k, a->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->k_stride, H, T, B) &&
           make_input_map(&m->v, a->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->v_stride, H, T, B) &&
           make_input_map(&m->g, a->g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a->g_stride, H, T, B);
}

// Which state kernel a sequential call runs: one CTA per chain (all 128 value
// columns) when the 32-column slab CTAs would need more than two waves of SMs;
// below that the slab kernel's shorter step (1.2 against 1.56 us, measured)
// wins.  The two kernels compute the same chunk step.  The overrides'
// state_kernel (tests, measurements) replaces the choice; the fused output norm
// needs whole rows and always takes the whole-chain kernel.
bool whole_chain_kernel(const PrefillParams& p, const kda_overrides& o, int num_sms) {
    if (p.gate) return true;
    if (o.state_kernel == 2) return true;
    if (o.state_kernel == 1) return false;
    return (long long)p.N * p.H * (kHeadDim / kSlab) > 2LL * num_sms;
}

// Segmented schedule of a padded call.  The state pass is one latency-bound
// chain per (sequence, head), prep is throughput-bound over all SMs, and the
// two kernels cannot share an SM (each needs most of its shared memory).  With
// few chains the state pass leaves most SMs idle for its whole length, so the
// tokens are cut into segments: prep of segment s+1 runs on the SMs the state
// pass of segment s leaves free, and once that state pass is done a second
// prep grid on its SMs joins in (both take records from the segment's
// counter).  The choice simulates both streams from per-unit costs measured on
// GB300 (SM clock 2070 MHz, long workload): one (chunk, head) record takes a
// prep CTA 8.3 us on a full GPU and 5 % less on the SMs beside a state pass (a
// fitted value: the prep kernel now measures 7.1 us a record alone, but with
// 7.1 the model picks shorter segments that measure 0.6-1 % slower on the
// long workload and its 16384-token cut, so the constant also carries the
// state pass's slowdown beside the faster prep, which the model leaves out); a
// chunk step takes 1.2 us in the slab kernel (four CTAs per chain) and 1.56 us
// in the whole-chain kernel, 12 % more beside prep;
// every segment adds about 5 us to each stream (launch, start-up, the slowest
// CTA's tail).
//
// The segment-parallel scan (chosen when its estimate wins by 5 %): prep on
// every SM, then the operator pass (2 (n - 1) whole-chain CTAs per chain), the
// combine (one fp32 128 x 128 x 128 product per segment and chain, 6.6 us
// each) and the output pass (n CTAs per chain), each launch adding
// kSegmentUs.  A pass step takes the whole-chain step (1.56 us) unless the
// resident CTAs' record reads (74 KB per step each; the transition and
// offset CTAs of a segment read the same records, so half as many distinct
// ones) need longer at the 4.2 TB/s these reads reach.  Fitted to B 1,
// T 131072, H 1..16 and T 32768, H 8 within 3 % (launch-list durations and
// event-timed calls).
struct Segments {
    bool on = false;
    bool head = false;       // whole-chain state kernel (else slab)
    int chunks = 0;          // chunks of every sequence per segment
    int prep_ctas = 0;       // prep grid while a state pass runs beside it
    int scan_nseg = 0;       // >= 2: segment-parallel scan with this many segments
    int scan_chunks = 0;     //        of this many chunks
};

constexpr double kRecUs = 8.3, kSlabStepUs = 1.2, kHeadStepUs = 1.56;
constexpr double kPrepBeside = 0.95, kStateBeside = 1.12, kSegmentUs = 5.0;
constexpr double kScanCombUs = 6.6, kScanRecordGBs = 4200.0;

// Estimated time of the segment-parallel scan with nseg segments.
double scan_us(long long cps, long long chains, long long nseg, int num_sms) {
    auto waves = [](long long n, long long m) { return (double)((n + m - 1) / m); };
    // step time of a pass whose resident CTAs read `distinct` records per step
    auto step = [&](long long ctas, double share) {
        const double resident = (double)(ctas < num_sms ? ctas : num_sms) * share;
        const double bw_us = resident * (double)kRecBytes / (kScanRecordGBs * 1e3);
        return bw_us > kHeadStepUs ? bw_us : kHeadStepUs;
    };
    const long long L = (cps + nseg - 1) / nseg;
    const long long ops = 2 * (nseg - 1) * chains, outs = nseg * chains;
    return waves(cps * chains, num_sms) * kRecUs + waves(ops, num_sms) * L * step(ops, 0.5) +
           (double)(nseg - 1) * kScanCombUs + waves(outs, num_sms) * L * step(outs, 1.0) + 4.0 * kSegmentUs;
}

// Segment length and count of a scan with (at most) nseg segments: every
// segment but the last has L chunks, the last at least one.
void scan_shape(long long cps, long long nseg, int* out_nseg, int* out_chunks) {
    const long long L = (cps + nseg - 1) / nseg;
    *out_chunks = (int)L;
    *out_nseg = (int)((cps + L - 1) / L);
}

// Estimated time of the segmented schedule.  Prep of segment i (work W_i in
// SM-microseconds) runs on `ctas` SMs from the end of segment i-1's prep,
// P_{i-1}, and on the other num_sms - ctas SMs (the helper grid) from the end of
// segment i-1's state pass, S_{i-1}; its records are shared out dynamically, so
// it ends when the two have done W_i between them (plus half a record of tail).
// The state pass of segment i starts when both P_i and S_{i-1} are reached.  The
// first segment's prep has every SM to itself.
double segmented_us(long long cps, long long chains, long long seg, long long ctas, double step,
                    int num_sms) {
    double P = 0.0, S = 0.0;
    const double hs = (double)(num_sms - ctas);
    for (long long t0 = 0; t0 < cps; t0 += seg) {
        const long long c = cps - t0 < seg ? cps - t0 : seg;
        if (t0 == 0) {
            P = (double)((c * chains + num_sms - 1) / num_sms) * kRecUs + kSegmentUs;
        } else {
            const double W = (double)(c * chains) * kRecUs * kPrepBeside;
            const double alone = P + W / (double)ctas;
            const double end = (hs <= 0.0 || S >= alone) ? alone : (W + (double)ctas * P + hs * S) / ((double)ctas + hs);
            P = end + 0.5 * kRecUs + kSegmentUs;
        }
        S = (P > S ? P : S) + (double)c * step * kStateBeside + kSegmentUs;
    }
    return S;
}

Segments plan_segments(const PrefillParams& p, const kda_overrides& o, int num_sms, int64_t scan_max) {
    Segments sg;
    if (p.cu != nullptr || p.T <= 0 || p.N <= 0 || num_sms < 4) return sg;
    const long long chains = (long long)p.N * p.H, cps = (p.T + kChunk - 1) / kChunk;
    // the scan, when forced (and the workspace has room for it)
    if (o.scan_segments >= 2 && scan_max >= 2) {
        sg.scan_nseg = 1;
        scan_shape(cps, o.scan_segments < scan_max ? o.scan_segments : scan_max, &sg.scan_nseg, &sg.scan_chunks);
        if (sg.scan_nseg < 2) sg.scan_nseg = sg.scan_chunks = 0;
        sg.head = true;
        return sg;
    }
    const long long forced = o.segment_chunks < 0 ? -1 : o.segment_chunks;
    if (forced == 0) return sg;
    const bool allow_slab = !p.gate && o.state_kernel != 2;
    const bool allow_head = p.gate || o.state_kernel != 1;
    auto waves = [](long long n, long long m) { return (double)((n + m - 1) / m); };
    // sequential: prep on every SM, then the state pass (each with its start-up
    // and tail, as a segment's)
    const double one_pass = waves(cps * chains, num_sms) * kRecUs + 2.0 * kSegmentUs +
                            (whole_chain_kernel(p, o, num_sms) ? waves(chains, num_sms) * cps * kHeadStepUs
                                                            : waves(4 * chains, num_sms) * cps * kSlabStepUs);
    double best = one_pass * 0.95;   // segment only for a clear gain
    if (forced > 0) best = 1e300;
    for (int head = 0; head < 2; ++head) {
        if (head ? !allow_head : !allow_slab) continue;
        if (forced > 0 && (bool)head != whole_chain_kernel(p, o, num_sms)) continue;
        const long long state_ctas = head ? chains : 4 * chains;
        long long ctas = num_sms - state_ctas;
        if (ctas < num_sms / 4) {
            if (forced <= 0) continue;  // prep would be starved of SMs
            ctas = num_sms / 4;
        }
        if (forced > 0 && o.prep_ctas > 0) ctas = o.prep_ctas < num_sms ? o.prep_ctas : num_sms;
        const double step = head ? kHeadStepUs : kSlabStepUs;
        if (forced > 0) {
            sg.on = true;
            sg.head = head != 0;
            sg.chunks = (int)(forced < cps ? forced : cps);
            sg.prep_ctas = (int)ctas;
            break;
        }
        // segment lengths of 8, 16, ... chunks (at most 512 candidates)
        const long long stride = 8 * ((cps / 8 + 511) / 512 > 1 ? (cps / 8 + 511) / 512 : 1);
        for (long long seg = stride; seg < cps; seg += stride) {
            const double t = segmented_us(cps, chains, seg, ctas, step, num_sms);
            if (t < best) {
                best = t;
                sg.on = true;
                sg.head = head != 0;
                sg.chunks = (int)seg;
                sg.prep_ctas = (int)ctas;
            }
        }
    }
    // the scan, unless a segment length is forced or the scan is ruled out
    if (forced < 0 && o.scan_segments != 1 && scan_max >= 2 && allow_head) {
        const double cur = sg.on ? best : one_pass;
        double best_scan = cur * 0.95;
        for (long long n = 2; n <= scan_max; ++n) {
            const double t = scan_us(cps, chains, n, num_sms);
            if (t < best_scan) {
                best_scan = t;
                sg = Segments();
                sg.head = true;
                scan_shape(cps, n, &sg.scan_nseg, &sg.scan_chunks);
            }
        }
        if (sg.scan_nseg == 1) sg = Segments();
    }
    return sg;
}

// Runs a planned segmented call: prep of every segment on `s`, the state pass of
// every segment on a second stream, each after its segment's prep and after the
// previous segment's state pass; `s` waits for the last state pass.
// The second stream and the two events of segmented calls: one set per host
// thread and device, created on the first segmented call and kept for the
// thread's life, so that calls recorded into a CUDA graph create nothing.
// Calls of one thread share the set (their state passes queue one after the
// other on it; every dependency goes through the events).
struct SideSet {
    cudaStream_t ss;
    cudaEvent_t ev_prep, ev_done;
};
bool side_set(SideSet* out) {
    constexpr int kMaxDevices = 64;
    thread_local SideSet sets[kMaxDevices] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    SideSet& st = sets[dev];
    if (!st.ss) {
        SideSet n{nullptr, nullptr, nullptr};
        if (cudaStreamCreateWithFlags(&n.ss, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&n.ev_prep, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&n.ev_done, cudaEventDisableTiming) != cudaSuccess) {
            if (n.ev_prep) cudaEventDestroy(n.ev_prep);
            if (n.ss) cudaStreamDestroy(n.ss);
            return false;
        }
        st = n;
    }
    *out = st;
    return true;
}

kda_status run_segments(const kda_prefill_args* a, const PrefillParams& p, const kda_overrides& o,
                        const Segments& sg, const kda_workspace_layout& L, int num_sms,
                        const SideSet& side, cudaStream_t s) {
    cudaStream_t ss = side.ss;
    cudaEvent_t ev_prep = side.ev_prep, ev_done = side.ev_done;
    auto ck = [](cudaError_t e) { return e == cudaSuccess; };
    // the side stream starts after the work already queued on `s`
    bool ok = ck(cudaEventRecord(ev_prep, s)) && ck(cudaStreamWaitEvent(ss, ev_prep, 0));
    float* carry = reinterpret_cast<float*>(static_cast<uint8_t*>(a->workspace) + L.state_carry);
    int32_t* counters = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(a->workspace) + L.prep_counters);
    const int64_t seg_tokens = (int64_t)sg.chunks * kChunk;
    const int64_t nseg = (p.T + seg_tokens - 1) / seg_tokens;
    ok = ok && ck(cudaMemsetAsync(counters, 0, sizeof(int32_t) * (size_t)nseg, s));
    const bool pdl = o.no_pdl == 0;
    // SMs the state pass leaves idle once it is done: a second prep grid there
    // takes records of the segment being prepared from the same counter
    const int helper_ctas = num_sms - sg.prep_ctas;
    size_t rec_base = 0;
    int64_t si = 0;
    for (int64_t t0 = 0; ok && t0 < p.T; t0 += seg_tokens, ++si) {
        const int ts = (int)(p.T - t0 < seg_tokens ? p.T - t0 : seg_tokens);
        const bool first = t0 == 0, last = t0 + ts >= p.T;
        PrefillParams q = p;
        q.q = p.q + t0 * p.qs[1];
        q.k = p.k + t0 * p.ks[1];
        q.v = p.v + t0 * p.vs[1];
        q.g = p.g + t0 * p.gs[1];
        q.beta = p.beta + t0 * p.bs[1];
        q.out = p.out + t0 * p.os[1];
        if (p.gate) q.gate = p.gate + t0 * p.gts[1];
        q.T = ts;
        q.max_chunks = p.B * ((ts + kChunk - 1) / kChunk);
        q.ws_rec = p.ws_rec + rec_base * kRecBytes;
        rec_base += (size_t)q.max_chunks * p.H;
        q.h0 = first ? p.h0 : carry;
        q.hT = last ? p.hT : carry;   // each chain's state is read before it is rewritten
        q.rec_counter = counters + si;
        PrepMaps maps;
        kda_prefill_args sa = *a;
        sa.q = q.q; sa.k = q.k; sa.v = q.v; sa.g = q.g;
        sa.seqlen = ts;
        if (!make_prep_maps(&sa, &maps)) return KDA_ERR_UNSUPPORTED;
        // no state pass runs yet while the first segment is prepared: every SM;
        // later segments: prep_ctas CTAs, joined by the helper grid after the
        // previous segment's state pass (queued before it on the second stream)
        ok = launch_prep(q, maps, first ? num_sms : sg.prep_ctas, s, !first && pdl) == cudaSuccess &&
             (first || helper_ctas < 1 || launch_prep(q, maps, helper_ctas, ss) == cudaSuccess) &&
             ck(cudaEventRecord(ev_prep, s)) && ck(cudaStreamWaitEvent(ss, ev_prep, 0)) &&
             launch_state_pass(a, q, sg.head, ss) == cudaSuccess;
    }
    // join even after a failure, so that nothing queued later on `s` overtakes
    // a state pass already enqueued
    if (ck(cudaEventRecord(ev_done, ss))) ck(cudaStreamWaitEvent(s, ev_done, 0));
    return ok ? KDA_OK : KDA_ERR_CUDA;
}

// Runs a planned segment-parallel scan on `s`: prep of every record on every
// SM, the segments' operators, the combine into entry states, and the outputs
// of every segment from its entry state.
kda_status run_scan(const kda_prefill_args* a, const PrefillParams& p, const Segments& sg,
                    const kda_workspace_layout& L, int num_sms, cudaStream_t s) {
    PrepMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (!make_prep_maps(a, &maps)) return KDA_ERR_UNSUPPORTED;
    if (launch_prep(p, maps, num_sms, s) != cudaSuccess) return KDA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    const size_t blk = (size_t)kHeadDim * kHeadDim;
    PrefillParams q = p;
    q.scan_nseg = sg.scan_nseg;
    q.scan_chunks = sg.scan_chunks;
    q.scan_ops = reinterpret_cast<float*>(ws + L.scan);
    q.scan_entry = q.scan_ops + (size_t)(2 * (L.scan_max_segments - 1)) * p.N * p.H * blk;
    PrefillParams ops = q;
    ops.scan_mode = kScanOps;
    ops.gate = nullptr;   // no outputs in the operator pass
    PrefillParams outp = q;
    outp.scan_mode = kScanOut;
    if (launch_state_pass(a, ops, true, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (launch_scan_combine(q, s) != cudaSuccess) return KDA_ERR_CUDA;
    if (launch_state_pass(a, outp, true, s) != cudaSuccess) return KDA_ERR_CUDA;
    return KDA_OK;
}

kda_status run_prefill(const kda_prefill_args* a, void* stream, int stages) {
    const bool state_pass = (stages & 2) != 0, prep = (stages & 1) != 0;
    kda_status st = check_prefill(a);
    if (st != KDA_OK) return st;
    kda_workspace_layout L;
    layout_of(a, &L);
    PrefillParams p;
    fill_params(a, L, &p);
    int num_sms = 1;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const kda_overrides o = overrides_of(a->overrides);
    if (prep && !a->device_status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), s) != cudaSuccess)
        return KDA_ERR_CUDA;
    if (prep && state_pass) {
        const Segments sg = plan_segments(p, o, num_sms, L.scan_max_segments);
        if (sg.scan_nseg >= 2) return run_scan(a, p, sg, L, num_sms, s);
        SideSet side;
        // without a second stream (none could be created) the call runs in one pass
        if (sg.on && side_set(&side)) return run_segments(a, p, o, sg, L, num_sms, side, s);
    }
    if (prep) {
        PrepMaps pmaps;
        memset(&pmaps, 0, sizeof(pmaps));
        if (!make_prep_maps(a, &pmaps)) return KDA_ERR_UNSUPPORTED;
        if (launch_chunk_table(p, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (launch_prep(p, pmaps, num_sms, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (state_pass) {
        // right after this call's prep: launched programmatically
        if (launch_state_pass(a, p, whole_chain_kernel(p, o, num_sms), s, prep && o.no_pdl == 0) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace

int kda::prefill_check_args(const kda_prefill_args* a) { return (int)check_args(a); }

extern "C" {

size_t kda_prefill_workspace_size(const kda_prefill_args* args) {
    if (!args) return 0;
    kda_workspace_layout L;
    if (!layout_of(args, &L)) return 0;
    return L.total;
}

kda_status kda_prefill_workspace_layout(const kda_prefill_args* args, kda_workspace_layout* layout) {
    if (!args || !layout) return KDA_ERR_INVALID_ARG;
    return layout_of(args, layout) ? KDA_OK : KDA_ERR_INVALID_ARG;
}

kda_status kda_prefill(const kda_prefill_args* args, void* stream) {
    return run_prefill(args, stream, 3);
}

kda_status kda_prefill_schedule(const kda_prefill_args* args, int num_sms, kda_schedule* out) {
    if (!args || !out || num_sms < 1) return KDA_ERR_INVALID_ARG;
    PrefillParams p;
    memset(&p, 0, sizeof(p));
    p.cu = args->cu_seqlens;
    p.T = (int)args->seqlen;
    p.N = (int)args->num_seqs;
    p.H = (int)args->num_heads;
    p.B = (int)args->batch;
    p.gate = static_cast<const __nv_bfloat16*>(args->out_gate);
    const kda_overrides o = overrides_of(args->overrides);
    const Segments sg = plan_segments(p, o, num_sms, scan_max_segments(args));
    const bool scan = sg.scan_nseg >= 2;
    out->segmented = sg.on ? 1 : 0;
    out->whole_chain = (sg.on || scan) ? (sg.head ? 1 : 0) : (whole_chain_kernel(p, o, num_sms) ? 1 : 0);
    out->segment_chunks = sg.on ? sg.chunks : 0;
    out->prep_ctas = sg.on ? sg.prep_ctas : num_sms;
    out->scan_segments = scan ? sg.scan_nseg : 0;
    out->scan_chunks = scan ? sg.scan_chunks : 0;
    return KDA_OK;
}

kda_status kda_prefill_prep(const kda_prefill_args* args, void* stream) {
    return run_prefill(args, stream, 1);
}

kda_status kda_prefill_state(const kda_prefill_args* args, void* stream) {
    return run_prefill(args, stream, 2);
}

kda_status kda_verify(const kda_verify_args* a, void* stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->head_dim_k != kHeadDim || a->head_dim_v != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (a->num_requests < 0 || a->num_heads < 1 || a->num_drafts < 1 || a->pool_size < 0)
        return KDA_ERR_INVALID_ARG;
    if (a->num_drafts > 16) return KDA_ERR_UNSUPPORTED;
    if (a->num_requests == 0) return KDA_OK;
    if (!a->q || !a->k || !a->v || !a->g || !a->beta || (!a->out && !a->replay_only) ||
        !a->state_pool || !a->accepted || a->pool_size < 1)
        return KDA_ERR_INVALID_ARG;
    if (a->pool_dtype != KDA_POOL_F32 && a->pool_dtype != KDA_POOL_BF16) return KDA_ERR_UNSUPPORTED;
    // the kernel numbers the (request, head) items with 32-bit ints
    if (a->num_requests > 65535 || a->num_heads > 65535 || a->pool_size > (1 << 30) ||
        a->num_requests * a->num_heads > INT32_MAX)
        return KDA_ERR_UNSUPPORTED;
    const int64_t* ss[6] = {a->q_stride, a->k_stride, a->v_stride, a->g_stride, a->beta_stride,
                            a->out_stride};
    for (int t = 0; t < 6; ++t)
        for (int i = 0; i < 3; ++i)
            if (ss[t][i] < 0) return KDA_ERR_UNSUPPORTED;
    // Draft rows and state blocks are moved in 16-byte pieces: every q, k, v, g row
    // and the pool must start on a 16-byte boundary.
    auto aligned16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) ||
        !aligned16(a->state_pool))
        return KDA_ERR_UNSUPPORTED;
    for (int i = 0; i < 3; ++i)
        if (a->q_stride[i] % 8 || a->k_stride[i] % 8 || a->v_stride[i] % 8 || a->g_stride[i] % 4)
            return KDA_ERR_UNSUPPORTED;
    int dev = 0, num_sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    VerifyParams p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const __nv_bfloat16*>(a->q);
    p.k = static_cast<const __nv_bfloat16*>(a->k);
    p.v = static_cast<const __nv_bfloat16*>(a->v);
    p.g = a->g;
    p.beta = a->beta;
    p.out = static_cast<__nv_bfloat16*>(a->out);
    for (int i = 0; i < 3; ++i) {
        p.qs[i] = a->q_stride[i]; p.ks[i] = a->k_stride[i]; p.vs[i] = a->v_stride[i];
        p.gs[i] = a->g_stride[i]; p.bs[i] = a->beta_stride[i]; p.os[i] = a->out_stride[i];
    }
    p.pool = a->state_pool;
    p.slot = a->slot;
    p.accepted = a->accepted;
    p.status = a->device_status;
    p.R = (int)a->num_requests;
    p.D = (int)a->num_drafts;
    p.H = (int)a->num_heads;
    p.P = (int)a->pool_size;
    p.beta_is_logit = a->beta_is_logit ? 1 : 0;
    p.scale = a->scale;
    p.pool_bf16 = a->pool_dtype == KDA_POOL_BF16 ? 1 : 0;
    p.replay_only = a->replay_only ? 1 : 0;
    const kda_overrides o = overrides_of(a->overrides);
    if (o.verify_kernel < 0 || o.verify_kernel > 2) return KDA_ERR_INVALID_ARG;
    p.stall_seed = o.stall_seed;
    p.wait_ns = wait_limit_of(o);
    p.timeout_probe = o.timeout_probe ? 1 : 0;
    // The sequential kernel costs four FP32 passes over the state per draft; the
    // tensor-core kernel costs two small products and a few FP32 passes per
    // request, plus a preparation that grows with the drafts.  Measured on
    // GB300 (256 requests x 32 heads, fp32 pool): sequential 0.15 / 0.25 / 0.36 /
    // 0.58 ms at 1 / 4 / 8 / 16 drafts, tensor-core 0.39 / 0.46 / 0.52 / 0.88 ms,
    // so the library takes the sequential kernel for every count it accepts
    // (kVerifyWyMinDrafts is past the limit of 16) and the tensor-core one only
    // when a call's overrides ask for it.
    const bool wy = o.verify_kernel == 2 || (o.verify_kernel == 0 && p.D >= kVerifyWyMinDrafts);
    cudaError_t e = wy ? launch_verify_wy(p, num_sms, static_cast<cudaStream_t>(stream))
                       : launch_verify(p, num_sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape, stride or alignment";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call failed";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded on-chip wait ran out";
    }
    return "unknown kda_status";
}

int kda_abi_version(void) { return KDA_ABI_VERSION; }

}  // extern "C"
