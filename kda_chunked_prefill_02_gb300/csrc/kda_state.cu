// kda_state.cu -- the serial inter-chunk state pass of KDA prefill (steps A6-A7).
//
// One CTA owns one chain slab: (sequence n, head h, 32 value columns of the
// 128 x 128 state).  Value columns of the state never interact, so the four
// slabs of a chain run in parallel (the "independent value-row slabs" of the
// cuDNN-frontend sm90 KDA page, Conversation).  With the per-chunk record of
// the prep kernel (A1 = [W ; Q'], Kt, U, O_loc, e^gam) the chunk recurrence is
//   D1_c  = A1_c S_c                          (128 x 32: W S rows, Q' S rows)
//   V_c   = U_c - D1_c[0:64],   O_c = O_loc_c + D1_c[64:128]
//   S_c+1 = Diag(e^gam_c) S_c + Kt_c V_c.
// Substituting the last line into the first gives
//   D1_c+1 = A1_c+1 (Diag(e^gam_c) S_c) + G_c+1 V_c,   G_c+1 = A1_c+1 Kt_c,
// where G_c+1 (128 x 64) does not depend on the state and is computed one
// chunk ahead, and the first term only needs the state entering chunk c.  So
// the only tensor-core product on the serial chain is G_c+1 V_c (K = 64); the
// state update S_c+1 runs beside it in its own warps.
//
// Warp roles: warp 0 fetches records with 1-D bulk copies (three stages);
// warp 1 owns TMEM and issues every MMA (one thread); warps 2-5 ("X", one TMEM
// lane quarter each) turn D1 into V (bf16 operand of the next products) and O
// (bf16 output); warps 6-9 ("Y") keep the fp32 state in registers (thread =
// key row), update it from D2 = Kt V, write the bf16 image of Diag(e^gam) S and
// convert G to its bf16 operand.  Every hand-off is an mbarrier (arrivals by
// the consumer warps, tcgen05.commit by the issuer), so the reads of one
// chunk's buffers are ordered before the next chunk's writes (the sPartialLast
// race of the TensorRT-LLM K1 page), and every thread that read TMEM has waited
// for its loads and crossed a tcgen05 fence plus a CTA barrier before TMEM is
// freed (the dealloc ordering of the TensorRT-LLM MQA-logits page).  All waits
// are bounded: one that runs out sets KDA_ERR_TIMEOUT and every role stops.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kStateThreads = 320;
constexpr int kStages = 3;
constexpr uint32_t ST_A1 = 0;          // [W ; Q'] 2 x (128 rows x 128 B), K-major A operand
constexpr uint32_t ST_KT = 32768;      // Kt 128 key rows x 64 tokens (SW128)
constexpr uint32_t ST_U = 49152;       // U slab: 64 rows x 32 bf16
constexpr uint32_t ST_OL = 53248;      // O_loc slab
constexpr uint32_t ST_EG = 57344;      // e^gam [128] fp32
constexpr uint32_t kStage = 58368;
constexpr uint32_t kStageTx = 32768 + 16384 + kSlabImg * 2 + 512;
// B operands with N = 32 value columns, MN-major, 64-byte swizzle: one
// 64-byte row per K index (16-byte chunk c of row r at r*64 + ((c ^ ((r>>1)&3)) << 4)),
// 8-row groups 512 B apart; each thread stores its own row.
constexpr uint32_t kRowGroup = 512;
constexpr uint32_t kShBytes = 8192;              // 128 key rows
constexpr uint32_t O_SH = kStages * kStage;     // two buffers: Diag(e^gam_c) S_c (S_0 in buffer 1 first)
constexpr uint32_t O_VN = O_SH + 2 * kShBytes;  // V: 64 token rows, 4 KB
constexpr uint32_t O_G = O_VN + 4096;           // G bf16, K-major A operand: 128 rows x 64 tokens, 16 KB
constexpr uint32_t kStateSmem = O_G + 16384 + 1024;
// TMEM columns (fp32): two D1 accumulators, D2, G.
constexpr uint32_t TM_D1 = 0, TM_D2 = 64, TM_G = 128, TM_COLS = 256;
constexpr uint32_t kBarProlog = 1;  // named barrier: issuer warp + Y warps

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    const bool ok = mbar_wait(bar, parity, abort);
    return __all_sync(0xffffffffu, ok);
}

// Row r of an MN-major N = 32 operand: 32 bf16 in four swizzled 16-byte chunks.
__device__ __forceinline__ void store_row32(uint8_t* base, int r, const float* x) {
    uint8_t* rp = base + r * 64;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4*>(rp + ((ch ^ ((r >> 1) & 3)) << 4)) =
            make_uint4(pack_bf16x2(x[8 * ch], x[8 * ch + 1]), pack_bf16x2(x[8 * ch + 2], x[8 * ch + 3]),
                       pack_bf16x2(x[8 * ch + 4], x[8 * ch + 5]), pack_bf16x2(x[8 * ch + 6], x[8 * ch + 7]));
}

// Unpacks 8 bf16 (one 16-byte chunk) to fp32.
__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[x]));
        f[2 * x] = t.x;
        f[2 * x + 1] = t.y;
    }
}

// 32 consecutive TMEM columns of this warp's lane quarter.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* d) {
    tmem_ld16(taddr, *reinterpret_cast<float(*)[16]>(d));
    tmem_ld16(taddr + 16, *reinterpret_cast<float(*)[16]>(d + 16));
}

__global__ void __launch_bounds__(kStateThreads, 1) state_kernel(const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], empty[kStages], d1_ready[2], d1_free[2];
    __shared__ uint64_t d2_ready, d2_free, g_ready, vn_ready, s_img_ready, g_img_ready;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_flag;

    const int slab = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
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
            mbar_init(&empty[i], 9);  // issuer commit + 4 X warps + 4 Y warps
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&d1_ready[i], 1);
            mbar_init(&d1_free[i], 4);
        }
        mbar_init(&d2_ready, 1);
        mbar_init(&d2_free, 4);
        mbar_init(&g_ready, 1);
        mbar_init(&vn_ready, 2);
        mbar_init(&s_img_ready, 4);
        mbar_init(&g_img_ready, 4);
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
    const uint32_t tb = tmem_base_sh;
    volatile int* abort = &abort_flag;
    auto fail = [&]() {
        if (atomicExch(&abort_flag, 1) == 0) atomicExch(p.status, 4);
    };
    const size_t st_off_base = (((size_t)n * p.H + h) * kHeadDim) * kHeadDim + slab * kSlab;

    if (warp == 0) {
        // ---------------- record fetcher (1-D bulk copies, kStages stages)
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < count; ++c) {
                const int st = c % kStages;
                if (c >= kStages && !mbar_wait(&empty[st], ((c / kStages) - 1) & 1, abort)) { fail(); break; }
                uint8_t* sb = sm + st * kStage;
                const uint8_t* rp = p.ws_rec + (size_t)((first + c) * p.H + h) * kRecBytes;
                mbar_arrive_expect_tx(&full[st], kStageTx);
                bulk_load(sb + ST_A1, rp + kRecA1, 32768, &full[st]);
                bulk_load(sb + ST_KT, rp + kRecKt, 16384, &full[st]);
                bulk_load(sb + ST_U, rp + kRecU + slab * kSlabImg, kSlabImg, &full[st]);
                bulk_load(sb + ST_OL, rp + kRecOl + slab * kSlabImg, kSlabImg, &full[st]);
                bulk_load(sb + ST_EG, rp + kRecEg, 512, &full[st]);
                issued = c + 1;
            }
            // Never leave the CTA with copies in flight.
            for (int c = issued - kStages; c < issued; ++c)
                if (c >= 0) mbar_wait(&full[c % kStages], (c / kStages) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (count > 0) named_bar_sync(kBarProlog, 160);
        if (lane == 0 && count > 0) {
            const uint32_t id32 = idesc_bf16_f32_bmn(128, kSlab), id64 = idesc_bf16_f32_bmn(128, 64);
            const uint32_t sh = smem_u32(sm + O_SH), vnb = smem_u32(sm + O_VN), gb = smem_u32(sm + O_G);
            auto stage_addr = [&](int c) { return smem_u32(sm + (c % kStages) * kStage); };
            // D = A1 * B with A1 K-major (K = 128 keys) and B an MN-major operand
            // (sw64: a N = 32 operand in the 64-byte swizzle; otherwise the
            // N = 64 Kt image in the 128-byte swizzle).  Descriptors are built
            // once per operand base; inside the unrolled K loop only the start
            // address (16-byte units, low bits) changes, so each tcgen05.mma
            // costs an add or two to issue.
            auto mma_a1 = [&](uint32_t d, uint32_t a1, uint32_t bb, uint32_t idesc, bool acc, bool sw64) {
                const uint64_t ad = sdesc_kmajor_sw128(a1);
                const uint64_t bd = sw64 ? sdesc_mnmajor_sw64(bb, kRowGroup, kRowGroup)
                                         : sdesc_mnmajor_sw128(bb, 1024, 1024);
                const uint32_t bstep = sw64 ? (2 * kRowGroup) >> 4 : (2048 >> 4);
#pragma unroll
                for (uint32_t k = 0; k < 8; ++k)
                    umma_bf16(d, ad + ((k >> 2) * (16384 >> 4) + (k & 3) * 2), bd + k * bstep, idesc,
                              (acc || k > 0) ? 1u : 0u);
            };
            // D (+)= A * V with A K-major (K = 64 tokens) and V the MN-major V operand.
            const uint64_t vdesc = sdesc_mnmajor_sw64(vnb, kRowGroup, kRowGroup);
            auto mma_v = [&](uint32_t d, uint32_t a, bool acc) {
                const uint64_t ad = sdesc_kmajor_sw128(a);
#pragma unroll
                for (uint32_t k = 0; k < 4; ++k)
                    umma_bf16(d, ad + k * 2, vdesc + k * ((2 * kRowGroup) >> 4), id32, (acc || k > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(&full[0], 0, abort);
            if (ok) {  // D1_0 = A1_0 S_0 (the Y warps stored S_0 in SH buffer 1)
                tc_fence_after();
                mma_a1(tb + TM_D1, stage_addr(0) + ST_A1, sh + kShBytes, id32, false, true);
                umma_commit(&d1_ready[0]);
            }
            for (int c = 0; ok && c < count; ++c) {
                const bool more = c + 1 < count;
                const uint32_t s0 = stage_addr(c), s1 = stage_addr(c + 1);
                const uint32_t d1 = tb + TM_D1 + 32 * ((c + 1) & 1);
                if (more) {
                    // G_c+1 = A1_c+1 Kt_c (does not depend on the state)
                    if (!(ok = mbar_wait(&full[(c + 1) % kStages], ((c + 1) / kStages) & 1, abort))) break;
                    if (c >= 1 && !(ok = mbar_wait(&g_img_ready, (c - 1) & 1, abort))) break;
                    tc_fence_after();
                    mma_a1(tb + TM_G, s1 + ST_A1, s0 + ST_KT, id64, false, false);
                    umma_commit(&g_ready);
                    // D1_c+1 = A1_c+1 Diag(e^gam_c) S_c  (+ G_c+1 V_c below)
                    if (!(ok = mbar_wait(&s_img_ready, c & 1, abort))) break;
                    if (c >= 1 && !(ok = mbar_wait(&d1_free[(c + 1) & 1], ((c - 1) >> 1) & 1, abort))) break;
                    tc_fence_after();
                    mma_a1(d1, s1 + ST_A1, sh + (c & 1) * kShBytes, id32, false, true);
                }
                // D2 = Kt_c V_c (once the Y warps have read the previous D2)
                if (!(ok = mbar_wait(&vn_ready, c & 1, abort))) break;
                if (c >= 1 && !(ok = mbar_wait(&d2_free, (c - 1) & 1, abort))) break;
                tc_fence_after();
                mma_v(tb + TM_D2, s0 + ST_KT, false);
                umma_commit(&d2_ready);
                umma_commit(&empty[c % kStages]);
                if (more) {
                    if (!(ok = mbar_wait(&g_img_ready, c & 1, abort))) break;
                    tc_fence_after();
                    mma_v(d1, gb, true);
                    umma_commit(&d1_ready[(c + 1) & 1]);
                }
            }
            if (!ok) fail();
        }
    } else if (warp < 6) {
        // ---------------- X warps: D1 -> V (operand) and O (output)
        const int qd = warp & 3, row = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        bool ok = true;
        for (int c = 0; ok && c < count; ++c) {
            const uint8_t* sb = sm + (c % kStages) * kStage;
            if (!(ok = warp_wait(&d1_ready[c & 1], (c >> 1) & 1, abort))) break;
            tc_fence_after();
            float d[kSlab];
            tmem_ld32(tb + lane_base + TM_D1 + 32 * (c & 1), d);
            if (!(ok = warp_wait(&full[c % kStages], (c / kStages) & 1, abort))) break;
            if (qd < 2) {
                // V_c = U_c - W_c S_c for token row `row`
                float vn[kSlab];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    float u[8];
                    unpack8(*reinterpret_cast<const uint4*>(sb + ST_U + slab_chunk_off(row, ch)), u);
#pragma unroll
                    for (int x = 0; x < 8; ++x) vn[8 * ch + x] = u[x] - d[8 * ch + x];
                }
                store_row32(sm + O_VN, row, vn);
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&vn_ready);
            } else {
                // O_c = O_loc_c + Q'_c S_c for token row `row - 64`
                const int i = row - 64, t0 = 64 * c;
                if (t0 + i < seq_len) {
                    uint32_t o[kSlab / 2];
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        float ol[8];
                        unpack8(*reinterpret_cast<const uint4*>(sb + ST_OL + slab_chunk_off(i, ch)), ol);
#pragma unroll
                        for (int x = 0; x < 4; ++x)
                            o[4 * ch + x] = pack_bf16x2(ol[2 * x] + d[8 * ch + 2 * x], ol[2 * x + 1] + d[8 * ch + 2 * x + 1]);
                    }
                    const int64_t t = (int64_t)tbase + t0 + i;
                    uint4* dst = reinterpret_cast<uint4*>(p.out + b * p.os[0] + t * p.os[1] + h * p.os[2] + slab * kSlab);
#pragma unroll
                    for (int x = 0; x < kSlab / 8; ++x)
                        dst[x] = make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
                }
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&d1_free[c & 1]);
                mbar_arrive(&empty[c % kStages]);
            }
        }
        if (!ok) fail();
    } else {
        // ---------------- Y warps: fp32 state (thread = key row), its bf16 image, G operand
        const int qd = warp & 3, row = 32 * qd + lane;
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        float S[kSlab];
        if (p.h0) {
            const float4* src = reinterpret_cast<const float4*>(p.h0 + st_off_base + (size_t)row * kHeadDim);
#pragma unroll
            for (int x = 0; x < kSlab / 4; ++x) {
                const float4 t = src[x];
                S[4 * x] = t.x; S[4 * x + 1] = t.y; S[4 * x + 2] = t.z; S[4 * x + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < kSlab; ++j) S[j] = 0.f;
        }
        bool ok = true;
        if (count > 0) {
            store_row32(sm + O_SH + kShBytes, row, S);  // S_0 for D1_0
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar_sync(kBarProlog, 160);
            // Diag(e^gam_0) S_0 for D1_1
            if ((ok = warp_wait(&full[0], 0, abort)) && count > 1) {
                const float eg0 = reinterpret_cast<const float*>(sm + ST_EG)[row];
                float sh[kSlab];
#pragma unroll
                for (int j = 0; j < kSlab; ++j) sh[j] = eg0 * S[j];
                store_row32(sm + O_SH, row, sh);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_img_ready);
            }
        }
        for (int c = 0; ok && c < count; ++c) {
            const uint8_t* sb = sm + (c % kStages) * kStage;
            const bool more = c + 1 < count;
            // D1_c complete: the G operand and SH buffer (c+1)&1 are free again
            if (!(ok = warp_wait(&d1_ready[c & 1], (c >> 1) & 1, abort))) break;
            if (!(ok = warp_wait(&full[c % kStages], (c / kStages) & 1, abort))) break;
            const float eg = reinterpret_cast<const float*>(sb + ST_EG)[row];
            if (more) {
                // G_c+1 (fp32 in TMEM) -> bf16 K-major operand, row `row`
                if (!(ok = warp_wait(&g_ready, c & 1, abort))) break;
                tc_fence_after();
                uint8_t* gr = sm + O_G + row * 128;
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    float gv[32];
                    tmem_ld32(tb + lane_base + TM_G + 32 * hlf, gv);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int ch = 4 * hlf + q;
                        *reinterpret_cast<uint4*>(gr + ((ch ^ (row & 7)) << 4)) =
                            make_uint4(pack_bf16x2(gv[8 * q], gv[8 * q + 1]), pack_bf16x2(gv[8 * q + 2], gv[8 * q + 3]),
                                       pack_bf16x2(gv[8 * q + 4], gv[8 * q + 5]), pack_bf16x2(gv[8 * q + 6], gv[8 * q + 7]));
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&g_img_ready);
            }
            // S_c+1 = Diag(e^gam_c) S_c + Kt_c V_c
            if (!(ok = warp_wait(&d2_ready, c & 1, abort))) break;
            tc_fence_after();
            float d[kSlab];
            tmem_ld32(tb + lane_base + TM_D2, d);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&d2_free);
#pragma unroll
            for (int j = 0; j < kSlab; ++j) S[j] = fmaf(eg, S[j], d[j]);
            if (c + 2 < count) {
                // Diag(e^gam_c+1) S_c+1 for D1_c+2, into SH buffer (c+1)&1
                if (!(ok = warp_wait(&full[(c + 1) % kStages], ((c + 1) / kStages) & 1, abort))) break;
                const float eg1 = reinterpret_cast<const float*>(sm + ((c + 1) % kStages) * kStage + ST_EG)[row];
                float sh[kSlab];
#pragma unroll
                for (int j = 0; j < kSlab; ++j) sh[j] = eg1 * S[j];
                store_row32(sm + O_SH + ((c + 1) & 1) * kShBytes, row, sh);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_img_ready);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[c % kStages]);
        }
        if (!ok) fail();
        if (!*abort && p.hT) {
            float4* dst = reinterpret_cast<float4*>(p.hT + st_off_base + (size_t)row * kHeadDim);
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

cudaError_t launch_state(const PrefillParams& p, cudaStream_t s) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kStateSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(kHeadDim / kSlab, p.H, p.N);
    state_kernel<<<grid, kStateThreads, kStateSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
