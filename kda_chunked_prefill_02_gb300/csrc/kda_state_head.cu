// kda_state_head.cu -- the serial inter-chunk state pass (steps A6-A7) with one
// CTA per whole chain (sequence n, head h): all 128 value columns of the state.
//
// A tcgen05.mma of M = 128 and K = 16 takes the same ~100 SM cycles for every
// N <= 128 on this GPU (measured by the MMA throughput probe in the selftest
// library), so one CTA that runs the chunk step at N = 128 costs about what a
// 32-column slab CTA costs, and needs a quarter of the CTAs.  That matters when
// there are more chains than SMs (the slab kernel then runs in several waves),
// and it leaves SMs free for other work.  Per chunk, with the record the prep
// kernel left (W, Q', Kt, U, O_loc, e^gam):
//   P1 (tensor core)  D1 = [W ; Q'] S    M = 128 (64 W rows + 64 Q' rows), N = 128, K = 128
//   epilogue          V_new = U - D1[0:64],  O = O_loc + D1[64:128] -> out (bf16)
//   P2 (tensor core)  D2 = Kt V_new       M = 128 keys, N = 128, K = 64 tokens
//   epilogue          S <- Diag(e^gam) S + D2   (fp32 in registers, bf16 image for P1)
// Warp roles: all 16 warps are the epilogue, warp w owning TMEM lane quarter
// w % 4 and the 32-column quarter w / 4, so a thread holds 32 fp32 state
// values as in the slab kernel.  An MMA issue holds its thread for about the
// product's duration, so P1 is issued by a thread of an output warp (every warp
// waits for P1) and P2 by a thread of a V_new warp (those wait for P2, while
// the output warps compute and store the output rows).  A thread of another
// output warp issues the output tensor stores and the record copies: each
// record arrives by one 1-D bulk copy into one of two stages, issued as soon as
// the chunk barrier has shown the stage's previous chunk finished with it (P2
// complete, every read done, the stores' reads of the staged rows done), with
// an L2 prefetch further ahead.  Hand-offs are
// mbarriers and named barriers; every mbarrier wait is bounded, and the chunk
// barrier's OR-reduction of the abort flag makes all epilogue warps stop at the
// same chunk.  Every MMA has completed, and every thread that read TMEM has
// waited for its loads and crossed a tcgen05 fence plus a CTA barrier, before
// TMEM is freed (the dealloc ordering of the TensorRT-LLM MQA-logits page).
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kHeadThreads = 16 * 32;
constexpr uint32_t SH_A1 = 0;          // [W ; Q'] 2 x (128 rows x 128 B)
constexpr uint32_t SH_KT = 32768;      // Kt 128 rows x 128 B
constexpr uint32_t SH_U = 49152;       // U: 4 value slabs (64-byte swizzle), 16 KB
constexpr uint32_t SH_OL = 65536;      // O_loc, same layout
constexpr uint32_t SH_EG = 81920;      // e^gam [128] fp32
constexpr uint32_t kHStageTx = kRecBytes;  // the whole record, one bulk copy
constexpr uint32_t kHStage = 82944;     // kRecBytes rounded up to 1 KB (swizzle atoms)
constexpr int kHStages = 2;
constexpr int kHPrefetchAhead = 4;
// B operands of P1 and P2, MN-major with the 128-byte swizzle: per K index
// (key for S, token for V_new) two 64-column atoms 1024 B apart, 8-row groups
// 2048 B apart.
constexpr uint32_t kHSbo = 2048;
constexpr uint32_t OH_S = kHStages * kHStage;       // S bf16: 128 key rows (32 KB)
constexpr uint32_t OH_VN = OH_S + 32768;            // V_new bf16: 64 token rows (16 KB)
constexpr uint32_t kHeadSmem = OH_VN + 16384 + 1024;
constexpr uint32_t TMH_D1 = 0, TMH_D2 = 128, TMH_COLS = 256;
constexpr uint32_t kBarHVn = 1, kBarHChunk = 2, kBarHNorm = 3, kBarHOut = 4;  // named barriers (0 is __syncthreads)

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

// Row `r`, columns 32*cq .. 32*cq + 31 of an MN-major image: four 16-byte chunks.
__device__ __forceinline__ void store_quarter(uint8_t* base, int r, int cq, const float* x) {
    uint8_t* rp = base + (r >> 3) * kHSbo + (cq >> 1) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
        const int c = 4 * (cq & 1) + ch;
        *reinterpret_cast<uint4*>(rp + ((c ^ (r & 7)) << 4)) =
            make_uint4(pack_bf16x2(x[8 * ch], x[8 * ch + 1]), pack_bf16x2(x[8 * ch + 2], x[8 * ch + 3]),
                       pack_bf16x2(x[8 * ch + 4], x[8 * ch + 5]), pack_bf16x2(x[8 * ch + 6], x[8 * ch + 7]));
    }
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
    __shared__ float s_ss[4][64];      // fused norm: partial sums of squares per column quarter
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
    const uint32_t tb = tmem_base_sh;
    volatile int* abort = &abort_flag;
    auto fail = [&]() {
        if (atomicExch(&abort_flag, 1) == 0) atomicExch(p.status, 4);
    };
    auto rec_ptr = [&](int c) -> const uint8_t* {
        return p.ws_rec + (size_t)((first + c) * p.H + h) * kRecBytes;
    };

    {
        // ---------------- lane quarter qd, column quarter cq, thread row = key / token
        const int qd = warp & 3, cq = warp >> 2;
        const int row = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        // P1 and the copies: a thread of an output warp; P2: a thread of a V_new
        // warp, which waits for P2 anyway, so that the output warps' work is not
        // held up behind the P2 issue.
        const bool issuer = (warp == 2 && lane == 0);
        const bool issuer2 = (warp == 0 && lane == 0);
        // The output tensor stores and the record copies: a thread of another
        // output warp, so that the P1 thread goes from the chunk barrier straight
        // to the next P1.
        const bool storer = (warp == 3 && lane == 0);
        const uint32_t id = idesc_bf16_f32_bmn(128, 128);
        const uint32_t sS_addr = smem_u32(sm + OH_S), sVn_addr = smem_u32(sm + OH_VN);
        float S[kSlab];
        const size_t blk_off = (size_t)row * kHeadDim + kSlab * cq;   // inside a 128 x 128 block
        const size_t st_off = chain * kHeadDim * kHeadDim + blk_off;
        // Entry state: the call's initial state, or in the scan the identity
        // (transition), zero (offset) or the combine's entry state E_seg.
        const float* h0 = p.h0 ? p.h0 + st_off : nullptr;
        if (p.scan_mode == kScanOps) h0 = nullptr;
        if (p.scan_mode == kScanOut && seg > 0)
            h0 = p.scan_entry + ((size_t)seg * p.N * p.H + chain) * kHeadDim * kHeadDim + blk_off;
        if (zero_u) {
#pragma unroll
            for (int j = 0; j < kSlab; ++j) S[j] = (row == kSlab * cq + j) ? 1.f : 0.f;
        } else if (h0) {
            const float4* src = reinterpret_cast<const float4*>(h0);
#pragma unroll
            for (int x = 0; x < kSlab / 4; ++x) {
                const float4 t = src[x];
                S[4 * x] = t.x; S[4 * x + 1] = t.y; S[4 * x + 2] = t.z; S[4 * x + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kSlab; ++j) S[j] = 0.f;
        }
        // Records of chunks 0 and 1 into the two stages.
        auto issue_load = [&](int c) {
            const int st = c % kHStages;
            mbar_arrive_expect_tx(&full[st], kHStageTx);
            bulk_load(sm + st * kHStage, rec_ptr(c), kRecBytes, &full[st]);
            if (c + kHPrefetchAhead < count) bulk_prefetch_l2(rec_ptr(c + kHPrefetchAhead), kRecBytes);
        };
        int issued = 0;  // records requested so far (storer thread)
        if (storer)
            for (; issued < kHStages && issued < count; ++issued) issue_load(issued);
        store_quarter(sm + OH_S, row, cq, S);
        fence_proxy_async_smem();
        tc_fence_before();
        named_bar_or(kBarHChunk, 512, false);
        int done = 0;    // chunks finished

        for (int c = 0; c < count; ++c) {
            const int st = c % kHStages;
            const uint8_t* sb = sm + st * kHStage;
            const uint32_t sb_addr = smem_u32(sb);
            bool ok = warp_wait_h(&full[st], (c / kHStages) & 1, abort, p.wait_ns);
            stall_point<kStall>(p.stall_seed, 1, c);
            if (issuer && ok) {
                tc_fence_after();
                const uint64_t ad = sdesc_kmajor_sw128(sb_addr + SH_A1);
                const uint64_t bd = sdesc_mnmajor_sw128(sS_addr, 1024u, kHSbo);
#pragma unroll
                for (uint32_t k = 0; k < 8; ++k)
                    umma_bf16(tb + TMH_D1, ad + ((k >> 2) * (16384 >> 4) + (k & 3) * 2),
                              bd + k * ((2 * kHSbo) >> 4), id, k > 0 ? 1u : 0u);
                umma_commit(&p1_done);
            }
            __syncwarp();
            // This thread's U (W rows) or O_loc (Q' rows) values, read while P1 runs.
            uint4 sr[4];
            {
                const uint8_t* src = sb + (qd < 2 ? SH_U : SH_OL) + cq * kSlabImg;
                const int r = qd < 2 ? row : row - 64;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) sr[ch] = *reinterpret_cast<const uint4*>(src + slab_chunk_off(r, ch));
            }
            ok = ok && warp_wait_h((p.timeout_probe && c == 0) ? &bar_never : &p1_done, c & 1, abort, p.wait_ns);
            tc_fence_after();
            float d[kSlab];
            if (ok) {
                tmem_ld32(tb + lane_base + TMH_D1 + kSlab * cq, d);
            }
            if (qd < 2) {
                // V_new = U - W S for token row `row`
                if (ok) {
                    float vn[kSlab];
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const uint32_t uw[4] = {sr[ch].x, sr[ch].y, sr[ch].z, sr[ch].w};
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uw[x]));
                            if (zero_u) f = make_float2(0.f, 0.f);
                            vn[8 * ch + 2 * x] = f.x - d[8 * ch + 2 * x];
                            vn[8 * ch + 2 * x + 1] = f.y - d[8 * ch + 2 * x + 1];
                        }
                    }
                    stall_point<kStall>(p.stall_seed, 2, c);
                    store_quarter(sm + OH_VN, row, cq, vn);
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                named_bar_sync(kBarHVn, 256);  // the eight V_new warps
                if (issuer2 && ok && !*abort) {
                    tc_fence_after();
                    const uint64_t kt = sdesc_kmajor_sw128(sb_addr + SH_KT);
                    const uint64_t bv = sdesc_mnmajor_sw128(sVn_addr, 1024u, kHSbo);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)  // K = 64 tokens
                        umma_bf16(tb + TMH_D2, kt + k * 2, bv + k * ((2 * kHSbo) >> 4), id, k > 0 ? 1u : 0u);
                    umma_commit(&p2_done);
                }
                __syncwarp();
            } else if (!no_out) {
                // O = O_loc + Q' S for token row `row - 64`
                const int i = row - 64, t0 = 64 * (cbase + c);
                const bool valid_row = t0 + i < seq_len;
                const int64_t t = (int64_t)tbase + t0 + i;
                float o[kSlab];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint32_t ow[4] = {sr[ch].x, sr[ch].y, sr[ch].z, sr[ch].w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[x]));
                        o[8 * ch + 2 * x] = f.x + d[8 * ch + 2 * x];
                        o[8 * ch + 2 * x + 1] = f.y + d[8 * ch + 2 * x + 1];
                    }
                }
                if (p.gate) {
                    // gated RMSNorm over the 128 channels of the row: the four column
                    // quarters' sums of squares meet in shared memory
                    uint4 gw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                   make_uint4(0, 0, 0, 0)};
                    if (ok && valid_row) {
                        const uint4* gsrc = reinterpret_cast<const uint4*>(p.gate + b * p.gts[0] + t * p.gts[1] +
                                                                           h * p.gts[2] + kSlab * cq);
#pragma unroll
                        for (int x = 0; x < 4; ++x) gw[x] = gsrc[x];
                    }
                    float ss = 0.f;
#pragma unroll
                    for (int j = 0; j < kSlab; ++j) ss = fmaf(o[j], o[j], ss);
                    s_ss[cq][i] = ss;
                    named_bar_sync(kBarHNorm, 256);  // the eight output warps
                    const float ms = (s_ss[0][i] + s_ss[1][i] + s_ss[2][i] + s_ss[3][i]) * (1.0f / kHeadDim);
                    const float rn = rsqrtf(ms + p.norm_eps);
                    const float4* wq = reinterpret_cast<const float4*>(s_w + kSlab * cq);
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const uint32_t gv[4] = {gw[x].x, gw[x].y, gw[x].z, gw[x].w};
                        const float4 w0 = wq[2 * x], w1 = wq[2 * x + 1];
                        const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[e]));
                            o[8 * x + 2 * e] *= rn * ww[2 * e] * sigmoid_fast(gf.x);
                            o[8 * x + 2 * e + 1] *= rn * ww[2 * e + 1] * sigmoid_fast(gf.y);
                        }
                    }
                }
                stall_point<kStall>(p.stall_seed, 3, c);
                // Rows of a chunk that lies inside its sequence (padded calls: every
                // chunk, the tensor store clips the rows past T) leave by tensor store:
                // each thread writes its bf16 row piece over the O_loc bytes it read
                // (the same 64-byte-swizzled slab layout as the store box), and one
                // thread stores the four slabs.  Rows of a varlen tail chunk, which
                // the next sequence's rows follow, are stored one by one.
                const bool by_tma = p.out_tma && (p.cu == nullptr || t0 + kChunk <= seq_len);
                if (by_tma) {
                    uint8_t* img = sm + st * kHStage + SH_OL + cq * kSlabImg;
#pragma unroll
                    for (int x = 0; x < kSlab / 8; ++x)
                        *reinterpret_cast<uint4*>(img + slab_chunk_off(i, x)) =
                            make_uint4(pack_bf16x2(o[8 * x], o[8 * x + 1]), pack_bf16x2(o[8 * x + 2], o[8 * x + 3]),
                                       pack_bf16x2(o[8 * x + 4], o[8 * x + 5]), pack_bf16x2(o[8 * x + 6], o[8 * x + 7]));
                    fence_proxy_async_smem();
                    named_bar_sync(kBarHOut, 256);  // the eight output warps
                    if (storer && ok && !*abort) {
                        const int tok = (int)(p.cu == nullptr ? t0 : (int64_t)tbase + t0);
#pragma unroll
                        for (int sl = 0; sl < kHeadDim / kSlab; ++sl)
                            tma_store_4d(&out_map, kSlab * sl, h, tok, b, sb + SH_OL + sl * kSlabImg);
                        bulk_commit();
                    }
                } else if (ok && valid_row) {
                    uint4* dst = reinterpret_cast<uint4*>(p.out + b * p.os[0] + t * p.os[1] + h * p.os[2] + kSlab * cq);
#pragma unroll
                    for (int x = 0; x < kSlab / 8; ++x)
                        dst[x] = make_uint4(pack_bf16x2(o[8 * x], o[8 * x + 1]), pack_bf16x2(o[8 * x + 2], o[8 * x + 3]),
                                            pack_bf16x2(o[8 * x + 4], o[8 * x + 5]), pack_bf16x2(o[8 * x + 6], o[8 * x + 7]));
                }
                tc_fence_before();
            }
            ok = ok && warp_wait_h(&p2_done, c & 1, abort, p.wait_ns);
            tc_fence_after();
            if (ok) {
                tmem_ld32(tb + lane_base + TMH_D2 + kSlab * cq, d);
                const float eg = reinterpret_cast<const float*>(sb + SH_EG)[row];
#pragma unroll
                for (int j = 0; j < kSlab; ++j) S[j] = fmaf(eg, S[j], d[j]);
                stall_point<kStall>(p.stall_seed, 4, c);
                if (c + 1 < count) {
                    store_quarter(sm + OH_S, row, cq, S);
                    fence_proxy_async_smem();
                }
            } else {
                fail();
            }
            tc_fence_before();
            if (named_bar_or(kBarHChunk, 512, *abort != 0)) break;
            done = c + 1;
            // stage st is free: P2 of chunk c completed, every read of it is done
            // and (storer) the output tensor stores have read their slabs
            stall_point<kStall>(p.stall_seed, 5, c);
            if (storer && issued < count) {
                bulk_wait_read();
                issue_load(issued++);
            }
        }
        if (storer) {
            bulk_wait_all();  // the output tensor stores are complete
            // Never leave with a copy in flight (bounded; normally complete).
            for (int c = done; c < issued; ++c) mbar_wait(&full[c % kHStages], (c / kHStages) & 1, nullptr);
        }
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
            float4* dst = reinterpret_cast<float4*>(fin);
#pragma unroll
            for (int x = 0; x < kSlab / 4; ++x)
                dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TMH_COLS);
}

}  // namespace

cudaError_t launch_state_head(const PrefillParams& p, const CUtensorMap& out_map, cudaStream_t s) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    static std::atomic<uint64_t> smem_set[2];
    auto kern = p.stall_seed ? state_head_kernel<true> : state_head_kernel<false>;
    cudaError_t e = set_smem_limit_once((const void*)kern, (int)kHeadSmem, smem_set[p.stall_seed ? 1 : 0]);
    if (e != cudaSuccess) return e;
    const int ys = p.scan_mode == kScanOps ? 2 * (p.scan_nseg - 1) : (p.scan_mode == kScanOut ? p.scan_nseg : 1);
    if (ys <= 0) return cudaSuccess;
    dim3 grid(p.H, p.N * ys);
    kern<<<grid, kHeadThreads, kHeadSmem, s>>>(p, out_map);
    return cudaGetLastError();
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
