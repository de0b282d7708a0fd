// kda_state.cu -- the serial inter-chunk state pass of KDA prefill (steps A6-A7).
//
// One CTA owns one chain slab: (sequence n, head h, 32 value columns of the
// 128 x 128 state).  Value columns of the state never interact, so the four
// slabs of a chain run in parallel (the "independent value-row slabs" of the
// cuDNN-frontend sm90 KDA page, Conversation).  Per chunk, with the record the
// prep kernel left in the workspace:
//   P1 (tensor core)  D1 = [Q e^Gam ; W] S      M = 128 (64 Q rows + 64 W rows), K = 128
//   epilogue          V_new = U - D1[64:128]    (fp16 image for P2 and P3, two buffers)
//   P2 (tensor core)  D2 = Kt V_new             M = 128 keys, K = 64 tokens
//   P3 (tensor core)  D1[0:64] += Aqk V_new     -> O = (Q e^Gam) S + Aqk V_new -> out (bf16)
//   epilogue          S <- Diag(e^gam) S + D2   (fp32 in registers, bf16 copy for P1)
// The fp32 state lives in the epilogue threads' registers (thread = key row);
// its bf16 image in shared memory is the B operand of the next chunk's P1.
// P1 runs in bf16, P2 and P3 in fp16 (V_new and the record's Kt and Aqk).
// P3's A operand is the record's 64 Aqk rows; its other 64 rows read the bytes
// after them (the rest of the stage and the next one) and land on the W rows
// of D1, which the V_new epilogue has already consumed.  D1 and the V_new
// image alternate between two buffers, so the output rows of chunk c are read,
// and P3 of chunk c reads V_new, while chunk c + 1 runs.
//
// Warp roles: warp 0 fetches the next chunks' records with 1-D bulk copies
// (three stages) and issues P3 once P2 is queued; warps 1-4 are the epilogue
// (one TMEM lane quarter each: lanes 0-63 the output rows, 64-127 the V_new
// rows), and a thread of a V_new warp issues P1 and P2 right after the
// barriers that publish the operands they need, so the serial chain has no
// hand-off to a separate MMA warp.  Every buffer hand-off is an mbarrier or a
// named barrier, so the reads of one chunk's buffers are ordered before the
// next chunk's writes (the sPartialLast race of the TensorRT-LLM K1 page), and
// every thread that read TMEM has waited for its loads and crossed a tcgen05
// fence plus a CTA barrier before TMEM is freed (the dealloc ordering of the
// TensorRT-LLM MQA-logits page).  All mbarrier waits are bounded; a wait that
// runs out sets KDA_ERR_TIMEOUT, and every epilogue warp still reaches the
// named barriers of that chunk; the chunk barrier's OR-reduction of the abort
// flag makes all of them stop at the same chunk.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kStateThreads = 160;
constexpr uint32_t ST_A1 = 0;          // [Q e^Gam ; W] 2 x (128 rows x 128 B)
constexpr uint32_t ST_KT = 32768;      // [Kt ; Aqk] 192 rows x 128 B
constexpr uint32_t ST_AQK = ST_KT + (kRecAqk - kRecKt);
constexpr uint32_t ST_U = 57344;       // the slab's 32 rows of U^T (128 B: 64 tokens each)
constexpr uint32_t ST_EG = 61440;      // e^gam [128] fp32
constexpr uint32_t kStage = 62464;     // the record's parts, rounded up to 1 KB
constexpr uint32_t kStageTx = 32768 + 24576 + kSlabImg + 512;
constexpr int kStages = 3;
constexpr int kPrefetchAhead = 6;      // chunks between an L2 prefetch and its record's bulk copy
// B operands of P1, P2 and P3, MN-major with the 128-byte swizzle: one 128-byte
// row per K index (key for S, token for V_new) holding the slab's 32 columns,
// 8-row groups 1024 B apart, so each thread stores its own row.
constexpr uint32_t O_S = kStages * kStage;     // S bf16: 128 key rows (16 KB)
constexpr uint32_t O_VN = O_S + 16384;         // V_new fp16: 2 buffers of 64 token rows (8 KB each)
constexpr uint32_t O_OUT = O_VN + 2 * 8192;    // output rows: [64 tokens x 32 values] bf16, 64-byte swizzle
constexpr uint32_t kStateSmem = O_OUT + kSlabImg + 1024;
constexpr uint32_t kRowGroup = 1024;
constexpr uint32_t TM_D1 = 0, TM_D2 = 64, TM_COLS = 128;   // D1: two buffers of 32 columns
constexpr uint32_t kBarVn = 1, kBarChunk = 2, kBarOut = 3;  // named barriers (0 is __syncthreads)
// P3's A operand reads 16 KB from a stage's Aqk: for the last stage the bytes
// past it are the state image's
static_assert((kStages - 1) * kStage + ST_AQK + 16384 <= O_VN, "P3's A operand stays in shared memory");
static_assert(ST_KT + 24576 <= ST_U && ST_U + kSlabImg <= ST_EG && ST_EG + 512 <= kStage, "stage layout");

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
    const bool ok = mbar_wait(bar, parity, abort, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

template <bool kStall>
__global__ void __launch_bounds__(kStateThreads, 1)
    state_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap out_map) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    // p2_issued and p3_done by chunk parity: a waiter may be a chunk behind the
    // arrivals, never two (the chunk barriers in between wait for its work)
    __shared__ uint64_t full[kStages], empty[kStages], p1_done, p2_done, p2_issued[2], p3_done[2], bar_fin,
        bar_fin3, bar_never;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int slab = blockIdx.x, h = blockIdx.y;
    // varlen: the sequences in the order of the chunk table (longest first)
    const int n = p.seq_order ? p.seq_order[blockIdx.z] : (int)blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Chain extent.
    int first, count, seq_len, b, tbase;
    if (p.cu == nullptr) {
        const int cps = (p.T + kChunk - 1) / kChunk;
        first = n * cps; count = cps; seq_len = p.T; b = n; tbase = 0;
    } else {
        first = p.chunk_off[n];
        count = p.chunk_off[n + 1] - first;
        seq_len = p.cu[n + 1] - p.cu[n];
        b = 0; tbase = p.cu[n];
        if (count < 0) count = 0;
    }

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 3);   // P1/P2 read, P3 read, the epilogue's reads
        }
        mbar_init(&p1_done, 1); mbar_init(&p2_done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&p2_issued[i], 1);
            mbar_init(&p3_done[i], 1);
        }
        mbar_init(&bar_fin, 1); mbar_init(&bar_fin3, 1);
        mbar_init(&bar_never, 1);   // nothing arrives on it (the timeout probe's wait)
        abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base_sh, TM_COLS);
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
    const uint32_t id = idesc_bf16_f32_bmn(128, kSlab);       // P1: bf16
    const uint32_t id16 = idesc_f16_f32_bmn(128, kSlab);      // P2, P3: fp16

    if (warp == 0) {
        // ---------------- record fetcher, and P3 once P2 of the chunk is queued
        if (lane == 0) {
            auto load = [&](int c) {
                const int st = c % kStages;
                uint8_t* sb = sm + st * kStage;
                const uint8_t* rp = p.ws_rec + (size_t)((first + c) * p.H + h) * kRecBytes;
                mbar_arrive_expect_tx(&full[st], kStageTx);
                bulk_load(sb + ST_A1, rp + kRecA1, 32768, &full[st]);
                bulk_load(sb + ST_KT, rp + kRecKt, 24576, &full[st]);
                bulk_load(sb + ST_U, rp + kRecU + slab * kSlabImg, kSlabImg, &full[st]);
                bulk_load(sb + ST_EG, rp + kRecEg, 512, &full[st]);
                // Records further ahead are pulled into L2 so that their bulk copies,
                // issued once a stage frees up, do not wait on HBM.
                if (c + kPrefetchAhead < count)
                    bulk_prefetch_l2(p.ws_rec + (size_t)((first + c + kPrefetchAhead) * p.H + h) * kRecBytes,
                                     kRecBytes);
            };
            int issued = 0, p3s = 0;
            for (; issued < kStages && issued < count; ++issued) load(issued);
            for (int c = 0; c < count; ++c) {
                const int st = c % kStages;
                if (!mbar_wait(&p2_issued[c & 1], (c >> 1) & 1, abort, p.wait_ns)) { fail(); break; }
                stall_point<kStall>(p.stall_seed, 1, c);
                {
                    // P3: D1[0:64] += Aqk V_new (A: Aqk rows, K-major; B: V_new, MN-major)
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sm + st * kStage + ST_AQK));
                    const uint64_t bd = sdesc_mnmajor_sw128(smem_u32(sm + O_VN + 8192 * (c & 1)), kRowGroup, kRowGroup);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)
                        umma_bf16(tb + TM_D1 + kSlab * (c & 1), ad + k * 2, bd + k * ((2 * kRowGroup) >> 4), id16, 1u);
                    umma_commit(&p3_done[c & 1]);
                    umma_commit(&empty[st]);
                    p3s = c + 1;
                }
                // the stage of chunk c takes the record kStages chunks on once
                // chunk c is done with it
                if (issued < count) {
                    if (!mbar_wait(&empty[st], (c / kStages) & 1, abort, p.wait_ns)) { fail(); break; }
                    load(issued++);
                }
            }
            // Never leave the CTA with copies or products in flight: wait (bounded)
            // for the last stages issued and the last P3.  In a normal run these
            // completed long ago.
            for (int c = issued - kStages; c < issued; ++c)
                if (c >= 0) mbar_wait(&full[c % kStages], (c / kStages) & 1, nullptr);
            if (p3s > 0) {
                umma_commit(&bar_fin3);
                mbar_wait(&bar_fin3, 0, nullptr);
            }
        }
    } else {
        // ---------------- epilogue (+ MMA issue): TMEM lane quarter qd, thread row = key / token
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const bool vwarp = qd >= 2;                    // D1 rows 64..127: W; 0..63: Q e^Gam
        const bool issuer = (qd == 2 && lane == 0);
        const bool storer = (qd == 0 && lane == 0);
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const uint32_t sS_addr = smem_u32(sm + O_S);
        float S[kSlab];
        const size_t st_off = (((size_t)n * p.H + h) * kHeadDim + row) * kHeadDim + slab * kSlab;
        if (p.h0) {
            const float4* src = reinterpret_cast<const float4*>(p.h0 + st_off);
#pragma unroll
            for (int x = 0; x < kSlab / 4; ++x) {
                const float4 t = src[x];
                S[4 * x] = t.x; S[4 * x + 1] = t.y; S[4 * x + 2] = t.z; S[4 * x + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kSlab; ++j) S[j] = 0.f;
        }
        // Row `row` of an MN-major operand: 32 values (bf16 or fp16) in four
        // swizzled 16-byte chunks.
        auto store_row = [&](uint8_t* base, int r, const float* x, bool f16) {
            uint8_t* rp = base + (r >> 3) * kRowGroup + (r & 7) * 128;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t w[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    w[e] = f16 ? pack_f16x2(x[8 * ch + 2 * e], x[8 * ch + 2 * e + 1])
                               : pack_bf16x2(x[8 * ch + 2 * e], x[8 * ch + 2 * e + 1]);
                *reinterpret_cast<uint4*>(rp + ((ch ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        };
        auto write_state_image = [&]() {
            store_row(sm + O_S, row, S, false);
            fence_proxy_async_smem();
            tc_fence_before();
        };
        // The output rows of chunk co (token row `row` of the chunk): D1 after P3
        // (the buffer of chunk co).  Rows of a chunk inside its sequence (padded:
        // every chunk, the tensor store clips rows past T) leave by one tensor
        // store of the slab, staged in the output image (the box's 64-byte
        // swizzled layout); rows of a varlen tail chunk, which the next
        // sequence's rows follow, are stored one by one.
        auto output = [&](int co) {
            bool ok = warp_wait(&p3_done[co & 1], (co >> 1) & 1, abort, p.wait_ns);
            tc_fence_after();
            const int t0 = 64 * co;
            uint32_t o[kSlab / 2];
            if (ok) {
                float d[kSlab];
                tmem_ld32(tb + lane_base + TM_D1 + kSlab * (co & 1), d);
#pragma unroll
                for (int x = 0; x < kSlab / 2; ++x) o[x] = pack_bf16x2(d[2 * x], d[2 * x + 1]);
            } else {
                fail();
            }
            stall_point<kStall>(p.stall_seed, 4, co);
            const bool by_tma = p.out_tma && (p.cu == nullptr || t0 + kChunk <= seq_len);
            if (by_tma) {
                uint8_t* img = sm + O_OUT;
#pragma unroll
                for (int x = 0; x < kSlab / 8; ++x)
                    *reinterpret_cast<uint4*>(img + slab_chunk_off(row, x)) =
                        make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
                fence_proxy_async_smem();
                named_bar_sync(kBarOut, 64);  // the two output warps
                if (storer && ok && !*abort) {
                    const int tok = (int)(p.cu == nullptr ? t0 : (int64_t)tbase + t0);
                    tma_store_4d(&out_map, kSlab * slab, h, tok, b, img);
                    bulk_commit();
                }
            } else if (ok && t0 + row < seq_len) {
                const int64_t t = (int64_t)tbase + t0 + row;
                uint4* dst = reinterpret_cast<uint4*>(p.out + b * p.os[0] + t * p.os[1] + h * p.os[2] + slab * kSlab);
#pragma unroll
                for (int x = 0; x < kSlab / 8; ++x)
                    dst[x] = make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
            }
            tc_fence_before();
        };
        write_state_image();
        named_bar_or(kBarChunk, 128, false);
        int done = 0;

        for (int c = 0; c < count; ++c) {
            const int st = c % kStages;
            const uint8_t* sb = sm + st * kStage;
            const uint32_t sb_addr = smem_u32(sb);
            const uint32_t d1 = TM_D1 + kSlab * (c & 1);
            bool ok = warp_wait(&full[st], (c / kStages) & 1, abort, p.wait_ns);
            stall_point<kStall>(p.stall_seed, 2, c);
            if (issuer && ok) {
                tc_fence_after();
                // K = 128 keys: A K-major, B (S) MN-major; descriptors built once,
                // only the start address moves per 16-wide K step
                const uint64_t ad = sdesc_kmajor_sw128(sb_addr + ST_A1);
                const uint64_t bd = sdesc_mnmajor_sw128(sS_addr, kRowGroup, kRowGroup);
#pragma unroll
                for (uint32_t k = 0; k < 8; ++k)
                    umma_bf16(tb + d1, ad + ((k >> 2) * (16384 >> 4) + (k & 3) * 2),
                              bd + k * ((2 * kRowGroup) >> 4), id, k > 0 ? 1u : 0u);
                umma_commit(&p1_done);
            }
            __syncwarp();
            if (vwarp) {
                // U of this thread's token (row - 64) in the slab's 32 value
                // columns: column row - 64 of the slab's U^T rows, read while P1 runs.
                uint32_t uw[kSlab / 2];
#pragma unroll
                for (int x = 0; x < kSlab / 2; ++x) {
                    const uint32_t lo = *reinterpret_cast<const uint16_t*>(sb + ST_U + sw128_off(2 * x, row - 64));
                    const uint32_t hi = *reinterpret_cast<const uint16_t*>(sb + ST_U + sw128_off(2 * x + 1, row - 64));
                    uw[x] = lo | (hi << 16);
                }
                ok = ok && warp_wait((p.timeout_probe && c == 0) ? &bar_never : &p1_done, c & 1, abort, p.wait_ns);
                tc_fence_after();
                // V_new = U - W S for token row `row - 64`; stored transposed (K-major over tokens)
                if (ok) {
                    float d[kSlab];
                    tmem_ld32(tb + lane_base + d1, d);
                    float vn[kSlab];
#pragma unroll
                    for (int x = 0; x < kSlab / 2; ++x) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uw[x]));
                        vn[2 * x] = f.x - d[2 * x];
                        vn[2 * x + 1] = f.y - d[2 * x + 1];
                    }
                    stall_point<kStall>(p.stall_seed, 3, c);
                    store_row(sm + O_VN + 8192 * (c & 1), row - 64, vn, true);
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                named_bar_sync(kBarVn, 64);
                if (issuer && ok && !*abort) {
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sb_addr + ST_KT);
                    const uint64_t bd = sdesc_mnmajor_sw128(smem_u32(sm + O_VN + 8192 * (c & 1)), kRowGroup, kRowGroup);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)  // K = 64 tokens: A K-major, B (V_new) MN-major
                        umma_bf16(tb + TM_D2, ad + k * 2, bd + k * ((2 * kRowGroup) >> 4), id16,
                                  k > 0 ? 1u : 0u);
                    umma_commit(&p2_done);
                    umma_commit(&empty[st]);
                    mbar_arrive(&p2_issued[c & 1]);   // the fetcher queues P3 behind P2
                }
                __syncwarp();
            } else if (c > 0) {
                // the previous chunk's output rows, while this chunk's P1 runs
                output(c - 1);
            }
            ok = ok && warp_wait(&p2_done, c & 1, abort, p.wait_ns);
            tc_fence_after();
            if (ok) {
                float d[kSlab];
                tmem_ld32(tb + lane_base + TM_D2, d);
                const float eg = reinterpret_cast<const float*>(sb + ST_EG)[row];
#pragma unroll
                for (int j = 0; j < kSlab; ++j) S[j] = fmaf(eg, S[j], d[j]);
                stall_point<kStall>(p.stall_seed, 5, c);
                write_state_image();
            } else {
                fail();
            }
            // (storer) the output image's previous tensor store has read it
            if (storer) bulk_wait_read();
            // Every epilogue thread takes the same decision: the fetcher warp may set
            // the abort flag at any time, so it is reduced over the barrier.
            if (named_bar_or(kBarChunk, 128, *abort != 0)) break;
            done = c + 1;
            if (issuer) mbar_arrive(&empty[st]);
        }
        // the last chunk's output rows
        if (!vwarp && done == count && count > 0 && !*abort) output(count - 1);
        if (storer) bulk_wait_all();  // the output tensor stores are complete
        if (issuer && count > 0) {
            // every product issued here has completed before TMEM is released
            umma_commit(&bar_fin);
            mbar_wait(&bar_fin, 0, nullptr);
        }
        if (!*abort && p.hT) {
            float4* dst = reinterpret_cast<float4*>(p.hT + st_off);
#pragma unroll
            for (int x = 0; x < kSlab / 4; ++x)
                dst[x] = make_float4(S[4 * x], S[4 * x + 1], S[4 * x + 2], S[4 * x + 3]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tb, TM_COLS);
}

}  // namespace

cudaError_t launch_state(const PrefillParams& p, const CUtensorMap& out_map, cudaStream_t s, bool after_prep) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    static std::atomic<uint64_t> smem_set[2];
    auto kern = p.stall_seed ? state_kernel<true> : state_kernel<false>;
    cudaError_t e = set_smem_limit_once((const void*)kern, (int)kStateSmem, smem_set[p.stall_seed ? 1 : 0]);
    if (e != cudaSuccess) return e;
    dim3 grid(kHeadDim / kSlab, p.H, p.N);
    return launch_maybe_pdl(kern, grid, dim3(kStateThreads), kStateSmem, s, after_prep, p, out_map);
}

}  // namespace kda
