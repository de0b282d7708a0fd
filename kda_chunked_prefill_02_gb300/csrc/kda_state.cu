// kda_state.cu -- the serial inter-chunk state pass of KDA prefill (steps A6-A7).
//
// One CTA owns one chain slab: (sequence n, head h, 32 value columns of the
// 128 x 128 state).  Value columns of the state never interact, so the four
// slabs of a chain run in parallel (the "independent value-row slabs" of the
// cuDNN-frontend sm90 KDA page, Conversation).  Per chunk, with the record the
// prep kernel left in the workspace:
//   P1 (tensor core)  D1 = [W ; Q'] S          M = 128 (64 W rows + 64 Q' rows), K = 128
//   epilogue          V_new = U - D1[0:64],  O = O_loc + D1[64:128] -> out (bf16)
//   P2 (tensor core)  D2 = Kt V_new             M = 128 keys, K = 64 tokens
//   epilogue          S <- Diag(e^gam) S + D2   (fp32 in registers, bf16 copy for P1)
// The fp32 state lives in the epilogue threads' registers (thread = key row);
// its bf16 image in shared memory is the B operand of the next chunk's P1.
//
// Warp roles: warp 0 fetches the next chunks' records with 1-D bulk copies
// (two stages); warps 1-4 are the epilogue (one TMEM lane quarter each), and
// one of their threads issues the MMAs right after the named barrier that
// publishes the operand they need, so the serial chain has no hand-off to a
// separate MMA warp.  Every buffer hand-off is an mbarrier or a named barrier,
// so the reads of one chunk's buffers are ordered before the next chunk's
// writes (the sPartialLast race of the TensorRT-LLM K1 page), and every thread
// that read TMEM has waited for its loads and crossed a tcgen05 fence plus a CTA
// barrier before TMEM is freed (the dealloc ordering of the TensorRT-LLM
// MQA-logits page).  All mbarrier waits are bounded; a wait that runs out sets
// KDA_ERR_TIMEOUT, and every epilogue warp still reaches the named barriers of
// that chunk; the chunk barrier's OR-reduction of the abort flag makes all of
// them stop at the same chunk.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kStateThreads = 160;
constexpr uint32_t ST_A1 = 0;          // [W ; Q'] 2 x (128 rows x 128 B)
constexpr uint32_t ST_KT = 32768;      // Kt 128 rows x 128 B
constexpr uint32_t ST_U = 49152;       // U slab: 64 rows x 32 bf16
constexpr uint32_t ST_OL = 53248;      // O_loc slab
constexpr uint32_t ST_EG = 57344;      // e^gam [128] fp32
constexpr uint32_t kStage = 58368;
constexpr uint32_t kStageTx = 32768 + 16384 + kSlabImg * 2 + 512;
constexpr int kStages = 3;
constexpr int kPrefetchAhead = 6;      // chunks between an L2 prefetch and its record's bulk copy
// B operands of P1 and P2, MN-major with the 128-byte swizzle: one 128-byte
// row per K index (key for S, token for V_new) holding the slab's 32 columns,
// 8-row groups 1024 B apart, so each thread stores its own row.
constexpr uint32_t O_S = kStages * kStage;     // S bf16: 128 key rows (16 KB)
constexpr uint32_t O_VN = O_S + 16384;         // V_new bf16: 64 token rows (8 KB)
constexpr uint32_t kStateSmem = O_VN + 8192 + 1024;
constexpr uint32_t kRowGroup = 1024;
constexpr uint32_t TM_D1 = 0, TM_D2 = 32, TM_COLS = 64;
constexpr uint32_t kBarVn = 1, kBarChunk = 2, kBarOut = 3;  // named barriers (0 is __syncthreads)

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
    __shared__ uint64_t full[kStages], empty[kStages], p1_done, p2_done, bar_fin, bar_never;
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
            mbar_init(&empty[i], 2);
        }
        mbar_init(&p1_done, 1); mbar_init(&p2_done, 1); mbar_init(&bar_fin, 1);
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
    const uint32_t tb = tmem_base_sh;
    volatile int* abort = &abort_flag;
    auto fail = [&]() {
        if (atomicExch(&abort_flag, 1) == 0) atomicExch(p.status, 4);
    };

    if (warp == 0) {
        // ---------------- record fetcher (1-D bulk copies, kStages stages)
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < count; ++c) {
                const int st = c % kStages;
                if (c >= kStages && !mbar_wait(&empty[st], ((c / kStages) - 1) & 1, abort, p.wait_ns)) { fail(); break; }
                stall_point<kStall>(p.stall_seed, 1, c);
                uint8_t* sb = sm + st * kStage;
                const uint8_t* rp = p.ws_rec + (size_t)((first + c) * p.H + h) * kRecBytes;
                mbar_arrive_expect_tx(&full[st], kStageTx);
                bulk_load(sb + ST_A1, rp + kRecA1, 32768, &full[st]);
                bulk_load(sb + ST_KT, rp + kRecKt, 16384, &full[st]);
                bulk_load(sb + ST_U, rp + kRecU + slab * kSlabImg, kSlabImg, &full[st]);
                bulk_load(sb + ST_OL, rp + kRecOl + slab * kSlabImg, kSlabImg, &full[st]);
                bulk_load(sb + ST_EG, rp + kRecEg, 512, &full[st]);
                issued = c + 1;
                // Records further ahead are pulled into L2 so that their bulk copies,
                // issued once a stage frees up, do not wait on HBM.
                if (c + kPrefetchAhead < count)
                    bulk_prefetch_l2(p.ws_rec + (size_t)((first + c + kPrefetchAhead) * p.H + h) * kRecBytes,
                                     kRecBytes);
            }
            // Never leave the CTA with copies in flight: wait (bounded) for the
            // last stages issued.  In a normal run these phases completed long ago.
            for (int c = issued - kStages; c < issued; ++c)
                if (c >= 0) mbar_wait(&full[c % kStages], (c / kStages) & 1, nullptr);
        }
    } else {
        // ---------------- epilogue (+ MMA issue): TMEM lane quarter qd, thread row = key / token
        const int qd = warp & 3;
        const int row = 32 * qd + lane;
        const bool issuer = (qd == 0 && lane == 0);
        const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
        const uint32_t id = idesc_bf16_f32_bmn(128, kSlab);
        const uint32_t sS_addr = smem_u32(sm + O_S), sVn_addr = smem_u32(sm + O_VN);
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
        // Row `row` of an MN-major operand: 32 bf16 in four swizzled 16-byte chunks.
        auto store_row = [&](uint8_t* base, int r, const float* x) {
            uint8_t* rp = base + (r >> 3) * kRowGroup + (r & 7) * 128;
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                *reinterpret_cast<uint4*>(rp + ((ch ^ (r & 7)) << 4)) =
                    make_uint4(pack_bf16x2(x[8 * ch], x[8 * ch + 1]), pack_bf16x2(x[8 * ch + 2], x[8 * ch + 3]),
                               pack_bf16x2(x[8 * ch + 4], x[8 * ch + 5]), pack_bf16x2(x[8 * ch + 6], x[8 * ch + 7]));
        };
        auto write_state_image = [&]() {
            store_row(sm + O_S, row, S);
            fence_proxy_async_smem();
            tc_fence_before();
        };
        write_state_image();
        named_bar_or(kBarChunk, 128, false);

        for (int c = 0; c < count; ++c) {
            const int st = c % kStages;
            const uint8_t* sb = sm + st * kStage;
            const uint32_t sb_addr = smem_u32(sb);
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
                    umma_bf16(tb + TM_D1, ad + ((k >> 2) * (16384 >> 4) + (k & 3) * 2),
                              bd + k * ((2 * kRowGroup) >> 4), id, k > 0 ? 1u : 0u);
                umma_commit(&p1_done);
            }
            // This thread's U (W rows) or O_loc (Q' rows) slab row, read while P1 runs.
            uint4 slab_row[4];
            {
                const uint8_t* src = sb + (qd < 2 ? ST_U : ST_OL);
                const int r = qd < 2 ? row : row - 64;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    slab_row[ch] = *reinterpret_cast<const uint4*>(src + slab_chunk_off(r, ch));
            }
            ok = ok && warp_wait((p.timeout_probe && c == 0) ? &bar_never : &p1_done, c & 1, abort, p.wait_ns);
            tc_fence_after();
            float d[kSlab];
            if (ok) {
                tmem_ld32(tb + lane_base + TM_D1, d);
            }
            if (qd < 2) {
                // V_new = U - W S for token row `row`; stored transposed (K-major over tokens)
                if (ok) {
                    float vn[kSlab];
#pragma unroll
                    for (int ch = 0; ch < 4; ++ch) {
                        const uint4 u = slab_row[ch];
                        const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&uw[x]));
                            vn[8 * ch + 2 * x] = f.x - d[8 * ch + 2 * x];
                            vn[8 * ch + 2 * x + 1] = f.y - d[8 * ch + 2 * x + 1];
                        }
                    }
                    stall_point<kStall>(p.stall_seed, 3, c);
                    store_row(sm + O_VN, row, vn);
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                named_bar_sync(kBarVn, 64);
                if (issuer && ok && !*abort) {
                    tc_fence_after();
                    const uint64_t ad = sdesc_kmajor_sw128(sb_addr + ST_KT);
                    const uint64_t bd = sdesc_mnmajor_sw128(sVn_addr, kRowGroup, kRowGroup);
#pragma unroll
                    for (uint32_t k = 0; k < 4; ++k)  // K = 64 tokens: A K-major, B (V_new) MN-major
                        umma_bf16(tb + TM_D2, ad + k * 2, bd + k * ((2 * kRowGroup) >> 4), id,
                                  k > 0 ? 1u : 0u);
                    umma_commit(&p2_done);
                    umma_commit(&empty[st]);
                }
            } else {
                // O = O_loc + Q' S for token row `row - 64`
                const int i = row - 64;
                const int t0 = 64 * c;
                stall_point<kStall>(p.stall_seed, 4, c);
                uint32_t o[kSlab / 2];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const uint4 ol = slab_row[ch];
                    const uint32_t ow[4] = {ol.x, ol.y, ol.z, ol.w};
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[x]));
                        o[4 * ch + x] = pack_bf16x2(f.x + d[8 * ch + 2 * x], f.y + d[8 * ch + 2 * x + 1]);
                    }
                }
                // Rows of a chunk inside its sequence (padded: every chunk, the tensor
                // store clips rows past T) leave by one tensor store of the slab: each
                // thread writes its row over the O_loc bytes it read (the box's
                // 64-byte-swizzled layout).  Rows of a varlen tail chunk, which the
                // next sequence's rows follow, are stored one by one.
                const bool by_tma = p.out_tma && (p.cu == nullptr || t0 + kChunk <= seq_len);
                if (by_tma) {
                    uint8_t* img = sm + st * kStage + ST_OL;
#pragma unroll
                    for (int x = 0; x < kSlab / 8; ++x)
                        *reinterpret_cast<uint4*>(img + slab_chunk_off(i, x)) =
                            make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
                    fence_proxy_async_smem();
                    named_bar_sync(kBarOut, 64);  // the two output warps
                    if (qd == 2 && lane == 0 && ok && !*abort) {
                        const int tok = (int)(p.cu == nullptr ? t0 : (int64_t)tbase + t0);
                        tma_store_4d(&out_map, kSlab * slab, h, tok, b, img);
                        bulk_commit();
                    }
                } else if (ok && t0 + i < seq_len) {
                    const int64_t t = (int64_t)tbase + t0 + i;
                    uint4* dst = reinterpret_cast<uint4*>(p.out + b * p.os[0] + t * p.os[1] + h * p.os[2] + slab * kSlab);
#pragma unroll
                    for (int x = 0; x < kSlab / 8; ++x)
                        dst[x] = make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]);
                }
                tc_fence_before();
            }
            ok = ok && warp_wait(&p2_done, c & 1, abort, p.wait_ns);
            tc_fence_after();
            if (ok) {
                tmem_ld32(tb + lane_base + TM_D2, d);
                const float eg = reinterpret_cast<const float*>(sb + ST_EG)[row];
#pragma unroll
                for (int j = 0; j < kSlab; ++j) S[j] = fmaf(eg, S[j], d[j]);
                stall_point<kStall>(p.stall_seed, 5, c);
                write_state_image();
            } else {
                fail();
            }
            // The output slab's tensor store has read the stage before the stage is
            // released (the issuer's arrive below follows the barrier).
            if (qd == 2 && lane == 0) bulk_wait_read();
            // Every epilogue thread takes the same decision: the fetcher warp may set
            // the abort flag at any time, so it is reduced over the barrier.
            if (named_bar_or(kBarChunk, 128, *abort != 0)) break;
            if (issuer) mbar_arrive(&empty[st]);
        }
        if (qd == 2 && lane == 0) bulk_wait_all();  // the output tensor stores are complete
        if (issuer && count > 0) {
            // every product issued has completed before TMEM is released
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

cudaError_t launch_state(const PrefillParams& p, const CUtensorMap& out_map, cudaStream_t s) {
    if (p.N == 0 || p.H == 0) return cudaSuccess;
    static std::atomic<uint64_t> smem_set[2];
    auto kern = p.stall_seed ? state_kernel<true> : state_kernel<false>;
    cudaError_t e = set_smem_limit_once((const void*)kern, (int)kStateSmem, smem_set[p.stall_seed ? 1 : 0]);
    if (e != cudaSuccess) return e;
    dim3 grid(kHeadDim / kSlab, p.H, p.N);
    kern<<<grid, kStateThreads, kStateSmem, s>>>(p, out_map);
    return cudaGetLastError();
}

}  // namespace kda
