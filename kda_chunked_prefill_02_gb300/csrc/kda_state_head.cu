// kda_state_head.cu -- the serial inter-chunk state pass (steps A6-A7) with one
// CTA per whole chain (sequence n, head h): all 128 value columns of the state.
//
// The chunk step runs in the transposed orientation: the TMEM lanes are the
// 128 value columns of the state, so that both tensor-core products take their
// A operand from TMEM and every operand the threads produce goes to TMEM
// (tcgen05.st) rather than to a shared-memory image behind a proxy fence.  The
// fp32 state itself lives in TMEM as the accumulator of the second product.
// Per chunk, with the record the prep kernel left (Q e^Gam, W, Kt, Aqk, U,
// e^gam):
//   decay             S^T <- S^T Diag(e^gam)                 (threads, in TMEM)
//   P1 (tensor core)  D1^T = S_in^T [Q e^Gam ; W]^T          M = 128 values, N = 128, K = 128 keys
//   epilogue          V_new^T = U^T - D1^T[W part]           (fp16, to TMEM: P23's A operand)
//   P23 (tensor core) [S^T | D1^T[Q part]] += V_new^T [Kt ; Aqk]^T   N = 192 (128 keys + 64 tokens), K = 64
//   epilogue          S^T (the next entry state) -> bf16 to TMEM (P1's A operand);
//                     O^T = D1^T[Q part] = (Q e^Gam) S_in + Aqk V_new -> out (bf16)
// S_in is the chunk's entry state; the decay with the chunk's e^gam is applied
// to the TMEM copy before P23 accumulates Kt V_new onto it.  One instruction
// of M = 128, K = 16 takes about the same time for any N up to 128 on this GPU
// and not much more at N = 192, so the output product rides along with the
// state update.
//
// Warp roles: warp w owns TMEM lane quarter qd = w % 4 (value columns 32 qd ..
// 32 qd + 31, thread = one value column v) and column quarter cq = w / 4: in
// D1 32 tokens of the Q part (cq 0, 1: the output warps) or of the W part
// (cq 2, 3: the V_new warps, two on every SM sub-partition), in the state 32
// keys.  An MMA issue holds its thread for about the product's duration, so P1
// is issued by a thread of an output warp as soon as the chunk barrier has
// published the state operand, and P23 by a thread of a V_new warp (those wait
// for P23 anyway).  The output warps take the output of chunk c while P1 of
// chunk c + 1 runs.  A thread of another output warp issues the output tensor
// stores and the record copies: each record arrives by one 1-D bulk copy into
// one of two stages, issued as soon as the chunk barrier has shown the stage's
// previous chunk finished with it, with an L2 prefetch further ahead.
// Hand-offs are mbarriers and named barriers; every mbarrier wait is bounded,
// and the chunk barrier's OR-reduction of the abort flag makes all warps stop
// at the same chunk.  Every MMA has completed, and every thread that read TMEM
// has waited for its loads and crossed a tcgen05 fence plus a CTA barrier,
// before TMEM is freed (the dealloc ordering of the TensorRT-LLM MQA-logits
// page).
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kHeadThreads = 16 * 32;
// A stage holds one record as the prep kernel wrote it (one bulk copy).
constexpr uint32_t SH_A1 = kRecA1;     // [Q e^Gam ; W] 2 x (128 rows x 128 B), K-major: P1's B operand
constexpr uint32_t SH_KT = kRecKt;     // [Kt ; Aqk] 192 rows x 128 B, K-major: P23's B operand
constexpr uint32_t SH_U = kRecU;       // U^T: 128 value rows x 64 tokens (128-byte swizzle), 16 KB
constexpr uint32_t SH_EG = kRecEg;     // e^gam [128] fp32
constexpr uint32_t kHStageTx = kRecBytes;  // the whole record, one bulk copy
constexpr uint32_t kHStage = 74752;     // kRecBytes rounded up to 1 KB (swizzle atoms)
constexpr int kHStages = 2;
// L2 prefetch of a chain's later records, when the launch's CTAs fit on the GPU
// at once (few chains: the prefetched lines are read before anything evicts
// them); with more CTAs than SMs the prefetches of the resident CTAs evicted
// one another's records before use and cost DRAM traffic (varlen workload,
// 256 chains: 1.056 ms per call without them, 1.096 ms at 4 chunks ahead;
// long workload, 32 chains: 3.973 ms at 2 chunks ahead, 3.991 without).
constexpr int kHPrefetchAhead = 2;
constexpr uint32_t OH_OUT = kHStages * kHStage;   // output rows: 2 images of 4 slabs [64 tokens x 32 values] bf16
constexpr uint32_t kHeadSmem = OH_OUT + 2 * 4 * kSlabImg + 1024;
// TMEM columns (lane = value column v).
constexpr uint32_t TMH_S = 0;      // S^T fp32: keys 0..127 (P23 accumulates onto it)
constexpr uint32_t TMH_D1 = 128;   // D1^T fp32: Q part (tokens 0..63, P23 adds Aqk V_new), then W part
constexpr uint32_t TMH_AS = 256;   // S^T bf16 pairs: keys 0..127 in 64 columns (P1's A operand)
constexpr uint32_t TMH_AV = 320;   // V_new^T fp16 pairs: tokens 0..63 in 32 columns (P23's A operand)
constexpr uint32_t TMH_COLS = 512;
// named barriers (0 is __syncthreads); kBarHOut + q for the output warps of lane quarter q
constexpr uint32_t kBarHVn = 1, kBarHChunk = 2, kBarHNorm = 3, kBarHOut = 4;
static_assert(kRecAqk == kRecKt + 16384, "P23's B operand is Kt followed by Aqk");
static_assert(kRecBytes <= kHStage, "a record fits a stage");

// sigmoid(x) = 1/2 + tanh(x/2)/2, with the hardware tanh approximation
// (relative error ~2^-11, below the bf16 rounding of the output).
__device__ __forceinline__ float sigmoid_fast(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return fmaf(0.5f, t, 0.5f);
}

__device__ __forceinline__ bool warp_wait_h(uint64_t* bar, uint32_t parity, volatile int* abort,
                                            uint64_t limit_ns) {
    const bool ok = mbar_wait(bar, parity, abort, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
    return __uint_as_float(b << 16);
}

// The 32 values x[0..31] of each lane summed over the warp's 32 lanes: after the
// call lane l holds the sum of index l (31 shuffles; each round halves the
// indices a lane keeps).
__device__ __forceinline__ float warp_transpose_sum(float (&x)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int j = 0; j < s; ++j) {
            const float send = upper ? x[j] : x[j + s];
            const float keep = upper ? x[j + s] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return x[0];
}

template <bool kStall>
__global__ void __launch_bounds__(kHeadThreads, 1)
    state_head_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap out_map) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t full[kHStages], p1_done, p2_done, bar_fin, bar_fin2, bar_never;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;
    __shared__ float s_ss[4][64];      // fused norm: partial sums of squares per lane quarter
    __shared__ __align__(16) float s_w[kHeadDim];  // fused norm: weights

    const int h = blockIdx.x;
    // Which chain (and, in the scan modes, which segment and operator) this CTA
    // runs; varlen: the sequences in the order of the chunk table (longest first).
    int n, seg = 0, which = 0;
    if (p.scan_mode == kScanOps) {
        n = (int)blockIdx.y % p.N;
        seg = ((int)blockIdx.y / p.N) >> 1;
        which = ((int)blockIdx.y / p.N) & 1;
    } else if (p.scan_mode == kScanOut) {
        n = (int)blockIdx.y % p.N;
        seg = (int)blockIdx.y / p.N;
    } else {
        n = p.seq_order ? p.seq_order[blockIdx.y] : (int)blockIdx.y;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Scan operator passes: the transition reads U as zero and starts from the
    // identity; neither writes outputs.
    const bool no_out = p.scan_mode == kScanOps;
    const bool zero_u = no_out && which == 0;
    const size_t chain = (size_t)n * p.H + h;

    // Chain extent (cbase: the chain's chunk index of this CTA's first chunk).
    int first, count, seq_len, b, tbase, cbase = 0;
    if (p.cu == nullptr) {
        const int cps = (p.T + kChunk - 1) / kChunk;
        first = n * cps; count = cps; seq_len = p.T; b = n; tbase = 0;
        if (p.scan_mode != kScanOff) {
            cbase = seg * p.scan_chunks;
            first += cbase;
            count = min(p.scan_chunks, cps - cbase);
            if (count < 0) count = 0;
        }
    } else {
        first = p.chunk_off[n];
        count = p.chunk_off[n + 1] - first;
        seq_len = p.cu[n + 1] - p.cu[n];
        b = 0; tbase = p.cu[n];
        if (count < 0) count = 0;
    }

    if (tid == 0) {
        for (int i = 0; i < kHStages; ++i) mbar_init(&full[i], 1);
        mbar_init(&p1_done, 1); mbar_init(&p2_done, 1); mbar_init(&bar_fin, 1); mbar_init(&bar_fin2, 1);
        mbar_init(&bar_never, 1);   // nothing arrives on it (the timeout probe's wait)
        abort_flag = 0;
        fence_mbar_init();
    }
    if (p.gate && tid < kHeadDim) s_w[tid] = p.norm_w[tid];
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, TMH_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Launched programmatically after prep: prep's records are complete and
    // visible from here on (a no-op otherwise).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint32_t tb = tmem_base_sh;
    volatile int* abort = &abort_flag;
    auto fail = [&]() {
        if (atomicExch(&abort_flag, 1) == 0) atomicExch(p.status, 4);
    };
    auto rec_ptr = [&](int c) -> const uint8_t* {
        return p.ws_rec + (size_t)((first + c) * p.H + h) * kRecBytes;
    };

    {
        // ---------------- lane quarter qd (value column v), column quarter cq
        const int qd = warp & 3, cq = warp >> 2;
        const int v = 32 * qd + lane;
        const bool vwarp = cq >= 2;         // V_new warp (W part) or output warp (Q part)
        const int tq = 32 * (cq & 1);       // this warp's first token within its part
        const int k0 = 32 * cq;             // this thread's first key in the state
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const uint32_t d1_col = TMH_D1 + 32 * cq;   // Q part (cq 0, 1) or W part (cq 2, 3)
        // P1: a thread of an output warp; P23: a thread of a V_new warp (those wait
        // for P23 anyway); the record copies: a thread of another V_new warp, once
        // P23 has finished with the stage; the output tensor store of lane
        // quarter qd's slab: a thread of the quarter's second output warp.
        const bool issuer = (warp == 0 && lane == 0);
        const bool issuer2 = (warp == 8 && lane == 0);
        const bool loader = (warp == 9 && lane == 0);
        const bool storer = (cq == 1 && lane == 0);
        // P1 in bf16 (S and the record's rows), P23 in fp16 (V_new, Kt and Aqk)
        const uint32_t id1 = idesc_bf16_f32(128, 128), id2 = idesc_f16_f32(128, 192);
        const size_t blk_off = (size_t)k0 * kHeadDim + v;   // element (k0, v) of a 128 x 128 block
        const size_t st_off = chain * kHeadDim * kHeadDim + blk_off;
        // S^T in bf16 into P1's A operand: keys k0 .. k0 + 31 of lane v.
        auto store_state_operand = [&](const float (&s32)[kSlab]) {
            uint32_t w[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(s32[2 * i], s32[2 * i + 1]);
            tmem_st16(tmem_addr(tb, 32 * qd, TMH_AS + 16 * cq), w);
        };
        // Entry state: the call's initial state, or in the scan the identity
        // (transition), zero (offset) or the combine's entry state E_seg, into
        // TMEM (fp32, keys k0 .. k0 + 31 of lane v; the state lives there) and
        // P1's A operand.
        if (count > 0) {
            const float* h0 = p.h0 ? p.h0 + st_off : nullptr;
            if (p.scan_mode == kScanOps) h0 = nullptr;
            if (p.scan_mode == kScanOut && seg > 0)
                h0 = p.scan_entry + ((size_t)seg * p.N * p.H + chain) * kHeadDim * kHeadDim + blk_off;
            float s0[kSlab];
#pragma unroll
            for (int j = 0; j < kSlab; ++j)
                s0[j] = zero_u ? ((k0 + j == v) ? 1.f : 0.f) : (h0 ? h0[(size_t)j * kHeadDim] : 0.f);
            uint32_t w[kSlab];
#pragma unroll
            for (int j = 0; j < kSlab; ++j) w[j] = __float_as_uint(s0[j]);
            tmem_st16_issue(tmem_addr(tb, 32 * qd, TMH_S + k0), w);
            tmem_st16_issue(tmem_addr(tb, 32 * qd, TMH_S + k0 + 16), w + 16);
            store_state_operand(s0);
        }
        auto issue_load = [&](int c) {
            const int st = c % kHStages;
            mbar_arrive_expect_tx(&full[st], kHStageTx);
            bulk_load(sm + st * kHStage, rec_ptr(c), kRecBytes, &full[st]);
            if (p.rec_prefetch > 0 && c + p.rec_prefetch < count)
                bulk_prefetch_l2(rec_ptr(c + p.rec_prefetch), kRecBytes);
        };
        // P1 of chunk c: D1^T = S^T [Q e^Gam ; W]^T (B: 128 token rows, K-major in
        // two 64-key column blocks; A: S^T from TMEM, 8 columns per 16 keys).
        auto issue_p1 = [&](int c) {
            const uint8_t* sb = sm + (c % kHStages) * kHStage;
            tc_fence_after();
            const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sb + SH_A1));
#pragma unroll
            for (uint32_t k = 0; k < 8; ++k)
                umma_bf16_ta(tb + TMH_D1, tb + TMH_AS + 8 * k, bd + ((k >> 2) * (16384 >> 4) + (k & 3) * 2),
                             id1, k > 0 ? 1u : 0u);
            umma_commit(&p1_done);
        };
        // x: the output warps' O^T values (tokens tq .. tq + 31 of value column v),
        // kept from the end of a chunk to the next one; the V_new warps' U values.
        float x[kSlab];
        // The output of chunk co (O^T in x): the optional gated RMSNorm, then the
        // rows leave by tensor store (chunks inside their sequence; padded calls:
        // every chunk, the tensor map clips the rows past T) or one by one (a
        // varlen tail chunk, which the next sequence's rows follow).
        auto output = [&](int co, bool ok) {
            const int t0 = 64 * (cbase + co);
            if (p.gate) {
                // gated RMSNorm over the 128 channels of each token row: the
                // lanes' squares meet by a transposing warp sum, the four lane
                // quarters' partial sums in shared memory
                float sq[kSlab];
#pragma unroll
                for (int j = 0; j < kSlab; ++j) sq[j] = x[j] * x[j];
                s_ss[qd][tq + lane] = warp_transpose_sum(sq, lane);
                named_bar_sync(kBarHNorm, 256);  // the eight output warps
                const float ms = (s_ss[0][tq + lane] + s_ss[1][tq + lane] + s_ss[2][tq + lane] +
                                  s_ss[3][tq + lane]) * (1.0f / kHeadDim);
                const float rn_l = rsqrtf(ms + p.norm_eps);   // token tq + lane
                const float wv = s_w[v];
                const __nv_bfloat16* gp = p.gate + b * p.gts[0] + h * p.gts[2] + v;
                const int64_t tg0 = (int64_t)tbase + t0 + tq;
#pragma unroll
                for (int j = 0; j < kSlab; ++j) {
                    const float rn = __shfl_sync(0xffffffffu, rn_l, j);
                    float gv = 0.f;
                    if (ok && t0 + tq + j < seq_len) gv = __bfloat162float(gp[(tg0 + j) * p.gts[1]]);
                    x[j] *= rn * wv * sigmoid_fast(gv);
                }
            }
            stall_point<kStall>(p.stall_seed, 3, co);
            const bool by_tma = p.out_tma && (p.cu == nullptr || t0 + kChunk <= seq_len);
            if (by_tma) {
                // One of two images; the stores that read it two outputs ago were
                // done reading before the last chunk barrier (each output commits
                // one bulk group).  An image is 4 slabs (value v / 32) of 64-byte
                // token rows, 16-byte chunk c of row t at t*64 + ((c ^ ((t/2) & 3))
                // << 4); for token tq + j the swizzle depends on (j / 2) % 4 only
                // (tq is a multiple of 32), so four offsets serve all 32 rows.
                uint8_t* const img0 = sm + OH_OUT + (co & 1) * (4 * kSlabImg);
                uint8_t* img = img0 + (uint32_t)tq * 64u;
                uint32_t off[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    off[k] = (uint32_t)(v >> 5) * kSlabImg + ((((uint32_t)(v & 31) >> 3) ^ (uint32_t)k) << 4) +
                             (uint32_t)(v & 7) * 2u;
#pragma unroll
                for (int j = 0; j < kSlab; ++j)
                    *reinterpret_cast<__nv_bfloat16*>(img + (uint32_t)j * 64u + off[(j >> 1) & 3]) =
                        __float2bfloat16_rn(x[j]);
                fence_proxy_async_smem();
                named_bar_sync(kBarHOut + qd, 64);  // the quarter's two output warps: its slab is written
                if (storer) {
                    if (ok && !*abort) {
                        const int tok = (int)(p.cu == nullptr ? t0 : (int64_t)tbase + t0);
                        tma_store_4d(&out_map, kSlab * qd, h, tok, b, img0 + qd * kSlabImg);
                    }
                    bulk_commit();
                }
            } else {
                if (ok) {
                    __nv_bfloat16* dst = p.out + b * p.os[0] + h * p.os[2] + v;
#pragma unroll
                    for (int j = 0; j < kSlab; ++j)
                        if (t0 + tq + j < seq_len)
                            dst[((int64_t)tbase + t0 + tq + j) * p.os[1]] = __float2bfloat16_rn(x[j]);
                }
                if (storer) bulk_commit();   // an empty group: one group per output
            }
        };

        int issued = 0;  // records requested so far (loader thread)
        if (loader)
            for (; issued < kHStages && issued < count; ++issued) issue_load(issued);
        tc_fence_before();
        if (issuer && count > 0 && !mbar_wait(&full[0], 0, abort, p.wait_ns)) fail();
        if (named_bar_or(kBarHChunk, 512, *abort != 0)) count = 0;
        if (issuer && count > 0) issue_p1(0);
        int done = 0;    // chunks finished
        bool out_pending = false;

        for (int c = 0; c < count; ++c) {
            const int st = c % kHStages;
            uint8_t* sb = sm + st * kHStage;
            const uint32_t sb_addr = smem_u32(sb);
            // The record has arrived: the P1 thread waited for it before the chunk
            // barrier that ended the previous chunk (or the one before the loop).
            bool ok = true;
            stall_point<kStall>(p.stall_seed, 1, c);
            // The decay of the entry state by this chunk's e^gam, in TMEM, before
            // P23 adds Kt V_new to it, by the output warps: their own 32 keys
            // (from registers) and those of the V_new warp of the same lane
            // quarter (from TMEM), so that the V_new warps go straight to V_new.
            // The stores complete before the V_new barrier.
            if (!vwarp) {
                const float4* egp = reinterpret_cast<const float4*>(sb + SH_EG);
#pragma unroll
                for (int q16 = 0; q16 < 4; ++q16) {
                    // 16 keys at a time, scaled in place
                    const int kb = k0 + 64 * (q16 >> 1) + 16 * (q16 & 1);
                    uint32_t r[16];
                    tmem_ld16_issue(tb + lane_base + TMH_S + kb, r);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float4 f = egp[kb / 4 + i];
                        asm volatile("" : "+r"(r[4 * i]), "+r"(r[4 * i + 1]), "+r"(r[4 * i + 2]), "+r"(r[4 * i + 3]));
                        r[4 * i] = __float_as_uint(f.x * __uint_as_float(r[4 * i]));
                        r[4 * i + 1] = __float_as_uint(f.y * __uint_as_float(r[4 * i + 1]));
                        r[4 * i + 2] = __float_as_uint(f.z * __uint_as_float(r[4 * i + 2]));
                        r[4 * i + 3] = __float_as_uint(f.w * __uint_as_float(r[4 * i + 3]));
                    }
                    tmem_st16_issue(tmem_addr(tb, 32 * qd, TMH_S + kb), r);
                }
            }
            if (vwarp) {
                // U^T row v, tokens tq .. tq + 31 (four 16-byte chunks), read while
                // P1 runs
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint4 u = *reinterpret_cast<const uint4*>(sb + SH_U + sw128_off(v, tq + 8 * ch));
                    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[8 * ch + 2 * e] = zero_u ? 0.f : bf16_bits_to_float(uw[e] & 0xffffu);
                        x[8 * ch + 2 * e + 1] = zero_u ? 0.f : bf16_bits_to_float(uw[e] >> 16);
                    }
                }
                ok = ok && warp_wait_h((p.timeout_probe && c == 0) ? &bar_never : &p1_done, c & 1, abort, p.wait_ns);
                tc_fence_after();
                if (ok) {
                    // V_new = U - W S_in
                    float d[kSlab];
                    tmem_ld32(tb + lane_base + d1_col, d);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_f16x2(x[2 * i] - d[2 * i], x[2 * i + 1] - d[2 * i + 1]);
                    stall_point<kStall>(p.stall_seed, 2, c);
                    tmem_st16_issue(tmem_addr(tb, 32 * qd, TMH_AV + 16 * (cq & 1)), w);
                }
                tmem_wait_st();   // V_new
                tc_fence_before();
                named_bar_sync(kBarHVn, 512);  // V_new and every thread's decayed state are in TMEM
                if (issuer2 && ok && !*abort) {
                    tc_fence_after();
                    // B = [Kt ; Aqk] (N = 192 rows, K = 64 tokens, K-major); A = V_new^T (all fp16)
                    const uint64_t kt = sdesc_kmajor_sw128(sb_addr + SH_KT);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)
                        umma_bf16_ta(tb + TMH_S, tb + TMH_AV + 8 * k, kt + k * 2, id2, 1u);
                    umma_commit(&p2_done);
                }
                __syncwarp();
            } else {
                tmem_wait_st();   // the decayed state
                tc_fence_before();
                named_bar_arrive(kBarHVn, 512);
                // the previous chunk's output, while P1 of this one runs
                if (out_pending) output(c - 1, ok);
                out_pending = false;
            }
            ok = ok && warp_wait_h(&p2_done, c & 1, abort, p.wait_ns);
            tc_fence_after();
            // (loader) stage st is free: P1 and P23 of chunk c are complete and every
            // thread's reads of it came before the V_new barrier
            if (loader && ok && issued < count) issue_load(issued++);
            if (ok) {
                // the next entry state, and (output warps) this chunk's output rows
                if (!vwarp && !no_out) {
                    tmem_ld32(tb + lane_base + d1_col, x);
                    out_pending = true;
                }
                stall_point<kStall>(p.stall_seed, 4, c);
                if (c + 1 < count) {
                    float d[kSlab];
                    tmem_ld32(tb + lane_base + TMH_S + k0, d);
                    store_state_operand(d);
                }
            } else {
                fail();
            }
            tc_fence_before();
            // (storer) the output image the next chunk writes has been read by its
            // last tensor store; (P1 thread) the next record has arrived before the
            // barrier, so that every thread may read its stage after it
            if (storer) bulk_wait_read_but_last();
            if (issuer && c + 1 < count &&
                !mbar_wait(&full[(c + 1) % kHStages], ((c + 1) / kHStages) & 1, abort, p.wait_ns))
                fail();
            if (named_bar_or(kBarHChunk, 512, *abort != 0)) break;
            done = c + 1;
            if (issuer && c + 1 < count) issue_p1(c + 1);
            stall_point<kStall>(p.stall_seed, 5, c);
        }
        // the last chunk's output
        if (!vwarp && out_pending && done == count && !*abort) output(count - 1, true);
        if (storer) bulk_wait_all();  // the output tensor stores are complete
        // Never leave with a copy in flight (bounded; normally complete).
        if (loader)
            for (int c = done; c < issued; ++c) mbar_wait(&full[c % kHStages], (c / kHStages) & 1, nullptr);
        if (issuer && count > 0) {
            // every product issued has completed before TMEM is released
            umma_commit(&bar_fin);
            mbar_wait(&bar_fin, 0, nullptr);
        }
        if (issuer2 && count > 0) {
            umma_commit(&bar_fin2);
            mbar_wait(&bar_fin2, 0, nullptr);
        }
        // The state after the chain (or the segment): the final state, a scan
        // operator, or nothing (scan segments before the last).
        float* fin = p.hT ? p.hT + st_off : nullptr;
        if (p.scan_mode == kScanOps)
            fin = p.scan_ops + (((size_t)(2 * seg + which)) * p.N * p.H + chain) * kHeadDim * kHeadDim + blk_off;
        if (p.scan_mode == kScanOut && seg != p.scan_nseg - 1) fin = nullptr;
        if (!*abort && fin) {
            // count == 0: the entry state was never stored to TMEM; it is the
            // initial state (or zero / the identity) as read above
            float d[kSlab];
            if (count > 0) {
                tc_fence_after();
                tmem_ld32(tb + lane_base + TMH_S + k0, d);
            } else {
                const float* h0 = p.h0 ? p.h0 + st_off : nullptr;
                if (p.scan_mode == kScanOps) h0 = nullptr;
                if (p.scan_mode == kScanOut && seg > 0)
                    h0 = p.scan_entry + ((size_t)seg * p.N * p.H + chain) * kHeadDim * kHeadDim + blk_off;
#pragma unroll
                for (int j = 0; j < kSlab; ++j)
                    d[j] = zero_u ? ((k0 + j == v) ? 1.f : 0.f) : (h0 ? h0[(size_t)j * kHeadDim] : 0.f);
            }
#pragma unroll
            for (int j = 0; j < kSlab; ++j) fin[(size_t)j * kHeadDim] = d[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TMH_COLS);
}

}  // namespace

cudaError_t launch_state_head(const PrefillParams& p, const CUtensorMap& out_map, cudaStream_t s,
                              bool after_prep) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    static std::atomic<uint64_t> smem_set[2];
    auto kern = p.stall_seed ? state_head_kernel<true> : state_head_kernel<false>;
    cudaError_t e = set_smem_limit_once((const void*)kern, (int)kHeadSmem, smem_set[p.stall_seed ? 1 : 0]);
    if (e != cudaSuccess) return e;
    const int ys = p.scan_mode == kScanOps ? 2 * (p.scan_nseg - 1) : (p.scan_mode == kScanOut ? p.scan_nseg : 1);
    if (ys <= 0) return cudaSuccess;
    dim3 grid(p.H, p.N * ys);
    PrefillParams q = p;
    const long long ctas = (long long)p.H * p.N * ys;
    const int sms = device_sm_count();
    q.rec_prefetch = (sms > 0 && ctas <= sms) ? kHPrefetchAhead : 0;
    return launch_maybe_pdl(kern, grid, dim3(kHeadThreads), kHeadSmem, s, after_prep, q, out_map);
}

namespace {

// ---------------------------------------------------------------- scan combine
// E_{s+1} = M_s E_s + C_s, s = 0 .. nseg - 2, for one chain and a 16-column
// slab of the state (value columns never mix, so the eight slabs of a chain
// run in separate CTAs).  fp32 FMAs in a fixed order (C first, then the key
// index k ascending), so the entry states are bitwise reproducible.
// M_{s+1} and the slab of C_{s+1} are copied into shared memory (cp.async; M
// with a row pitch of 132 floats) while the product of segment s runs; E_s
// stays in shared memory from one segment to the next.  Thread = 4 rows
// (r0 + 32 m, m = 0..3) x 4 columns: per key index one broadcast M value per
// row (the eight rows a warp reads fall on distinct banks) and one float4 of E.
constexpr int kCombThreads = 128;
constexpr int kCombCols = 16;
constexpr int kMPitch = kHeadDim + 4;
constexpr uint32_t kCombSmem =
    (2 * kHeadDim * kMPitch + 2 * kHeadDim * kCombCols + kHeadDim * kCombCols) * sizeof(float);

__device__ __forceinline__ void cp_async16_comb(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kCombThreads) scan_combine_kernel(const PrefillParams p) {
    extern __shared__ __align__(16) float smc[];
    float* Ms[2] = {smc, smc + kHeadDim * kMPitch};           // M[i][k] at i * 132 + k
    float* Cs[2] = {smc + 2 * kHeadDim * kMPitch, smc + 2 * kHeadDim * kMPitch + kHeadDim * kCombCols};
    float* Es = smc + 2 * kHeadDim * kMPitch + 2 * kHeadDim * kCombCols;   // E[k][16 columns]
    const int slab = blockIdx.x, col0 = kCombCols * slab;
    const size_t chain = blockIdx.y, chains = (size_t)p.N * p.H;
    constexpr size_t kBlk = (size_t)kHeadDim * kHeadDim;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int cg = lane & 3, r0 = (lane >> 2) + 8 * w;        // rows r0 + 32 m, columns 4 cg ..
    // M_s and the slab of C_s into shared memory (one cp.async group)
    auto stage = [&](int s, int buf) {
        const float* M = p.scan_ops + ((size_t)(2 * s) * chains + chain) * kBlk;
        const float* C = p.scan_ops + ((size_t)(2 * s + 1) * chains + chain) * kBlk;
        for (int e = tid; e < kHeadDim * kHeadDim / 4; e += kCombThreads)
            cp_async16_comb(Ms[buf] + (e >> 5) * kMPitch + 4 * (e & 31), M + 4 * (size_t)e);
        for (int e = tid; e < kHeadDim * kCombCols / 4; e += kCombThreads)
            cp_async16_comb(Cs[buf] + 4 * e, C + (size_t)(e >> 2) * kHeadDim + col0 + 4 * (e & 3));
        asm volatile("cp.async.commit_group;" ::: "memory");
    };
    if (p.scan_nseg >= 2) stage(0, 0);
    for (int e = tid; e < kHeadDim * kCombCols; e += kCombThreads) {
        const int k = e / kCombCols, j = e % kCombCols;
        Es[e] = p.h0 ? p.h0[chain * kBlk + (size_t)k * kHeadDim + col0 + j] : 0.f;
    }
    for (int s = 0; s + 1 < p.scan_nseg; ++s) {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
        __syncthreads();   // M_s and C_s have landed; E_s is complete; the other buffers are free
        if (s + 2 < p.scan_nseg) stage(s + 1, (s + 1) & 1);
        const float* M = Ms[s & 1];
        const float* C = Cs[s & 1];
        float acc[4][4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 c4 = *reinterpret_cast<const float4*>(C + (r0 + 32 * m) * kCombCols + 4 * cg);
            acc[m][0] = c4.x; acc[m][1] = c4.y; acc[m][2] = c4.z; acc[m][3] = c4.w;
        }
#pragma unroll 4
        for (int k = 0; k < kHeadDim; ++k) {
            const float4 e4 = *reinterpret_cast<const float4*>(Es + k * kCombCols + 4 * cg);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float mv = M[(r0 + 32 * m) * kMPitch + k];
                acc[m][0] = fmaf(mv, e4.x, acc[m][0]);
                acc[m][1] = fmaf(mv, e4.y, acc[m][1]);
                acc[m][2] = fmaf(mv, e4.z, acc[m][2]);
                acc[m][3] = fmaf(mv, e4.w, acc[m][3]);
            }
        }
        __syncthreads();   // every read of E_s is done
        float* out = p.scan_entry + ((size_t)(s + 1) * chains + chain) * kBlk + col0 + 4 * cg;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int r = r0 + 32 * m;
            const float4 v = make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
            *reinterpret_cast<float4*>(Es + r * kCombCols + 4 * cg) = v;
            *reinterpret_cast<float4*>(out + (size_t)r * kHeadDim) = v;
        }
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

}  // namespace

cudaError_t launch_scan_combine(const PrefillParams& p, cudaStream_t s) {
    if (p.N == 0 || p.H == 0 || p.scan_nseg < 2) return cudaSuccess;
    static std::atomic<uint64_t> smem_set;
    cudaError_t e = set_smem_limit_once((const void*)scan_combine_kernel, (int)kCombSmem, smem_set);
    if (e != cudaSuccess) return e;
    dim3 grid(kHeadDim / kCombCols, p.N * p.H);
    scan_combine_kernel<<<grid, kCombThreads, kCombSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
