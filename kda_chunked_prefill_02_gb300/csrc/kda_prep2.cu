// kda_prep2.cu -- the per-chunk preparation (steps A2-A5) with two records in
// flight per SM: two CTAs of 8 warps and about 81 KB of shared memory each, so
// that one CTA's barrier waits, tensor-core waits and memory latencies overlap
// the other's work.  It computes exactly what prep_kernel (kda_prep.cu)
// computes, in the same order of operations, and writes the same records bit
// for bit; the chunked form and the overflow guard are described there.
//
// What changes against the one-CTA-per-SM kernel, to fit the shared memory:
//  * q, k, v and g are read straight from global memory by the threads that
//    use them (latency covered by the other CTA; the next record's rows are
//    asked into L2 ahead), instead of TMA tiles in shared memory;
//  * the operand build of MMA A runs in two channel halves, and MMA A
//    accumulates over them (the same K order as one K = 128 product);
//  * Q e^Gam, the Kt image and e^gam go to the record in global memory from
//    the threads that compute them; epilogue C reads Q e^Gam back from there
//    to form Q' = Q e^Gam - Aqk W, and the final bulk store of [W ; Q']
//    overwrites it;
//  * the [K e^Gam | V] operand of MMA C is built after the UT solve, over the
//    solve's dead fp32 scratch, while MMA B runs.
#include <string.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kP2Threads = 256;

// Dynamic shared memory map (bytes from a 1024-aligned base).
// Region [0, 73728) is reused phase by phase:
//   operand build:  R half (A of MMA A, 128 rows x 128 B) at 0, Y half (B of MMA A,
//                   160 rows x 128 B) at 16384
//   UT solve:       A, T, X (fp32) at 0, 17408, 34816; Aqk (A of MMA B) at 40960,
//                   [T' ; Aqk T'] (A of MMA C) at 49152, T'^T (B of MMA B) at 65536
//   after the solve: [K e^Gam | V] (B of MMA C, MN-major) at 0
//   epilogue C:     record images [W ; Q'] at 0, U at 32768, O_loc at 49152
constexpr uint32_t P_R = 0;
constexpr uint32_t P_Y = 16384;
constexpr uint32_t kYHalf = 160 * 128;
constexpr uint32_t P_A = 0;
constexpr uint32_t P_T = 17408;
constexpr uint32_t P_X = 34816;
constexpr uint32_t P_AQK = 40960;
constexpr uint32_t P_TT = 49152;
constexpr uint32_t P_TTR = 65536;
constexpr uint32_t P_KV = 0;
constexpr uint32_t kKvSbo2 = 4096;
constexpr uint32_t P_SA1 = 0;
constexpr uint32_t P_SU = 32768;
constexpr uint32_t P_SOL = 49152;
constexpr uint32_t P_TOT = 73728;     // fp32 [2][8][128] group decay products (exact, floored)
constexpr uint32_t P_BETA = 81920;    // fp32 [64]
constexpr uint32_t kP2Smem = 82176 + 1024;
constexpr int kPA2 = 68, kPX2 = 40;
constexpr uint32_t TM2_A = 0, TM2_DIAG = 96, TM2_B = 192, TM2_C = 0, TM2_COLS = 256;

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) {
    *reinterpret_cast<uint32_t*>(p) = v;
}
__device__ __forceinline__ void st_bf16(uint8_t* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
    return __ldg(reinterpret_cast<const unsigned int*>(p));
}
// T' = T Diag(beta) entries (i, j), (i, j + 1) into TT (row i, K index j) and
// T'^T (row j, K index i).
__device__ __forceinline__ void store_tprime_pair2(uint8_t* sm, int i, int j, float t0, float t1,
                                                   const float* sBeta) {
    const float a = t0 * sBeta[j], b = t1 * sBeta[j + 1];
    st_u32(sm + P_TT + sw128_off(i, j), pack_bf16x2(a, b));
    st_bf16(sm + P_TTR + sw128_off(j, i), a);
    st_bf16(sm + P_TTR + sw128_off(j + 1, i), b);
}
__device__ __forceinline__ uint32_t yoff_row2(int I, int J, int l) {
    return 8 * I * (I - 1) + 16 * J + l;
}
__device__ __forceinline__ float tf32_round2(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}
// d (16 x 8) = P (16 x 8*ke, pitch pp) * Q (8*ke x 8, pitch pq) over k-steps kb..ke-1
// (warp-level m16n8k8 tf32 MMA, fp32 accumulation, as in the one-CTA kernel).
__device__ __forceinline__ void warp_mma_16x8_2(const float* P, int pp, const float* Q, int pq,
                                                int kb, int ke, float (&d)[4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    d[0] = d[1] = d[2] = d[3] = 0.f;
    for (int ks = kb; ks < ke; ++ks) {
        const int k0 = 8 * ks;
        const uint32_t a0 = __float_as_uint(P[g * pp + k0 + t]), a1 = __float_as_uint(P[(g + 8) * pp + k0 + t]);
        const uint32_t a2 = __float_as_uint(P[g * pp + k0 + t + 4]);
        const uint32_t a3 = __float_as_uint(P[(g + 8) * pp + k0 + t + 4]);
        const uint32_t b0 = __float_as_uint(Q[(k0 + t) * pq + g]), b1 = __float_as_uint(Q[(k0 + t + 4) * pq + g]);
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}
__device__ __forceinline__ void store_tile_tf32_2(float* X, int pq, const float (&d)[4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2*>(X + g * pq + 2 * t) = make_float2(tf32_round2(d[0]), tf32_round2(d[1]));
    *reinterpret_cast<float2*>(X + (g + 8) * pq + 2 * t) = make_float2(tf32_round2(d[2]), tf32_round2(d[3]));
}

// Global addresses of token row `i` of a chunk, channels c, c + 1 (padded:
// batch b; varlen: b = 0 and t0 the packed index).
struct Rows {
    const __nv_bfloat16 *q, *k, *v;
    const float* g;
};
__device__ __forceinline__ Rows rows_of(const PrefillParams& p, const ChunkInfo& ci, int h, int c) {
    Rows r;
    r.q = p.q + ci.b * p.qs[0] + (int64_t)ci.t0 * p.qs[1] + h * p.qs[2] + c;
    r.k = p.k + ci.b * p.ks[0] + (int64_t)ci.t0 * p.ks[1] + h * p.ks[2] + c;
    r.v = p.v + ci.b * p.vs[0] + (int64_t)ci.t0 * p.vs[1] + h * p.vs[2] + c;
    r.g = p.g + ci.b * p.gs[0] + (int64_t)ci.t0 * p.gs[1] + h * p.gs[2] + c;
    return r;
}

template <bool kStall>
__global__ void __launch_bounds__(kP2Threads, 2) prep2_kernel(const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t bar_mma[3];
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrec = p.max_chunks * p.H;
    if (blockIdx.x >= nrec) return;
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar_mma[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, TM2_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;

    // Operand build: thread = key channels c0, c0 + 1 of one channel half and the
    // 8-token group h8 = warp (half hf of 16-token block G); a warp covers the 64
    // channels of the half (one 128-byte operand row) of one token row.
    const int cp2 = 2 * lane, h8 = warp, G = h8 >> 1, hf = h8 & 1;
    // TMEM epilogues: lane quarter qd, column quarters cq and cq + 2.
    const int qd = warp & 3, cq = warp >> 2;
    const float kPFloor = __expf(kGateFloor);
    const float* sBeta = reinterpret_cast<const float*>(sm + P_BETA);

    int rec = blockIdx.x;
    ChunkInfo ci = chunk_info(p, rec / p.H);
    auto load_beta = [&](const ChunkInfo& c, int hh) -> float {
        return (tid < c.len) ? __ldg(p.beta + c.b * p.bs[0] + ((int64_t)c.t0 + tid) * p.bs[1] + hh * p.bs[2])
                             : 0.f;
    };
    // The input rows of a record into L2 (one 256-byte q / k / v row or 512-byte
    // g row per thread).
    auto prefetch_inputs = [&](const ChunkInfo& c, int hh) {
        const int tensor = tid >> 6, i = tid & 63;
        if (c.len > 0 && i < c.len) {
            const Rows r = rows_of(p, c, hh, 0);
            if (tensor == 0) bulk_prefetch_l2(r.q + (int64_t)i * p.qs[1], 256);
            else if (tensor == 1) bulk_prefetch_l2(r.k + (int64_t)i * p.ks[1], 256);
            else if (tensor == 2) bulk_prefetch_l2(r.v + (int64_t)i * p.vs[1], 256);
            else bulk_prefetch_l2(r.g + (int64_t)i * p.gs[1], 512);
        }
    };
    prefetch_inputs(ci, rec % p.H);
    float bcur = load_beta(ci, rec % p.H);
    bool ok = true;
    for (uint32_t it = 0; ci.len > 0; ++it) {
        const int h = rec % p.H;
        const int len = ci.len;
        const int rec_next = rec + gridDim.x;
        const ChunkInfo cn = rec_next < nrec ? chunk_info(p, rec_next / p.H) : ChunkInfo{0, 0, 0, 0, 0};
        if (rec_next >= nrec) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        prefetch_inputs(cn, rec_next % p.H);
        uint8_t* rp = p.ws_rec + (size_t)rec * kRecBytes;
        stall_point<kStall>(p.stall_seed, 1, it);
        if (tid < 64) {
            float bval = bcur;
            if (tid < len && p.beta_is_logit) bval = 1.0f / (1.0f + __expf(-bval));
            reinterpret_cast<float*>(sm + P_BETA)[tid] = tid < len ? bval : 0.f;
        }
        // exp of this thread's gates (channels c0, c0 + 1 of half hh); tokens past
        // the chunk length read as g = 0 (no decay), like zeroed tile rows.
        auto load_p = [&](int hh, float (&p0)[8], float (&p1)[8]) {
            const Rows r = rows_of(p, ci, h, 64 * hh + cp2);
            float2 gv[8];
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                const int i = 8 * h8 + l;
                gv[l] = i < len ? __ldg(reinterpret_cast<const float2*>(r.g + (int64_t)i * p.gs[1]))
                                : make_float2(0.f, 0.f);
            }
#pragma unroll
            for (int l = 0; l < 8; ++l) { p0[l] = __expf(gv[l].x); p1[l] = __expf(gv[l].y); }
        };

        // ---- E1: each 8-token group's decay products (exact, floored) for both halves.
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            float p0[8], p1[8];
            load_p(hh, p0, p1);
            float e0 = 1.f, e1 = 1.f, f0 = 1.f, f1 = 1.f;
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                e0 *= p0[l]; e1 *= p1[l];
                f0 *= fmaxf(p0[l], kPFloor); f1 *= fmaxf(p1[l], kPFloor);
            }
            float* tot = reinterpret_cast<float*>(sm + P_TOT);
            const int c0 = 64 * hh + cp2;
            *reinterpret_cast<float2*>(tot + h8 * 128 + c0) = make_float2(e0, e1);
            *reinterpret_cast<float2*>(tot + 1024 + h8 * 128 + c0) = make_float2(f0, f1);
        }
        stall_point<kStall>(p.stall_seed, 2, it);
        if (tid == 0) bulk_wait_read();  // the previous record's images have left the staging area
        __syncthreads();

        // ---- E2a, per channel half: the MMA A operands R and Y, Q e^Gam, the Kt
        // image and e^gam; MMA A accumulates over the two halves.
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            const int c0 = 64 * hh + cp2, cc = cp2;
            const float* tot = reinterpret_cast<const float*>(sm + P_TOT);
            float p0[8], p1[8];
            load_p(hh, p0, p1);
            float b0[4], b1[4];
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                const float2 u = *reinterpret_cast<const float2*>(tot + (2 * J) * 128 + c0);
                const float2 w = *reinterpret_cast<const float2*>(tot + (2 * J + 1) * 128 + c0);
                b0[J] = u.x * w.x; b1[J] = u.y * w.y;
            }
            const float2 eA = *reinterpret_cast<const float2*>(tot + (2 * G) * 128 + c0);
            const float2 eB = *reinterpret_cast<const float2*>(tot + (2 * G + 1) * 128 + c0);
            const float2 fA = *reinterpret_cast<const float2*>(tot + 1024 + (2 * G) * 128 + c0);
            const float2 fB = *reinterpret_cast<const float2*>(tot + 1024 + (2 * G + 1) * 128 + c0);
            float Bg0 = 1.f, Bg1 = 1.f, E0 = 1.f, E1 = 1.f, Dm0[4], Dm1[4];
            {
                float d0 = 1.f, d1 = 1.f;
#pragma unroll
                for (int J = 0; J < 4; ++J) {
                    if (J < G) { Bg0 *= b0[J]; Bg1 *= b1[J]; }
                    if (J > G) { E0 *= b0[J]; E1 *= b1[J]; }
                    Dm0[J] = d0; Dm1[J] = d1;
                    if (J > G) { d0 *= b0[J]; d1 *= b1[J]; }
                }
            }
            if (h8 == 0)
                *reinterpret_cast<float2*>(rp + kRecEg + c0 * 4) =
                    make_float2(b0[0] * b0[1] * b0[2] * b0[3], b1[0] * b1[1] * b1[2] * b1[3]);
            const float qscale = p.scale;
            const Rows rw = rows_of(p, ci, h, c0);
            uint32_t kw[8];
            {
                // forward over the group: R = [K ac ; Q ac] and Q e^Gam
                float a0 = hf ? Bg0 * eA.x : Bg0, a1 = hf ? Bg1 * eA.y : Bg1;
                float ac0 = hf ? fA.x : 1.f, ac1 = hf ? fA.y : 1.f;
                uint32_t qw[8];
#pragma unroll
                for (int l = 0; l < 8; ++l) {
                    const int i = 8 * h8 + l;
                    kw[l] = i < len ? ldg_u32(rw.k + (int64_t)i * p.ks[1]) : 0u;
                    qw[l] = i < len ? ldg_u32(rw.q + (int64_t)i * p.qs[1]) : 0u;
                }
#pragma unroll
                for (int l = 0; l < 8; ++l) {
                    const int i = 8 * h8 + l;
                    a0 *= p0[l]; a1 *= p1[l];
                    ac0 *= fmaxf(p0[l], kPFloor); ac1 *= fmaxf(p1[l], kPFloor);
                    const float2 kk = bf16x2_to_float2(kw[l]);
                    float2 qq = bf16x2_to_float2(qw[l]);
                    qq.x *= qscale; qq.y *= qscale;
                    st_u32(sm + P_R + sw128_off(i, cc), pack_bf16x2(kk.x * ac0, kk.y * ac1));
                    st_u32(sm + P_R + sw128_off(64 + i, cc), pack_bf16x2(qq.x * ac0, qq.y * ac1));
                    // Q e^Gam into the record's Q' rows (epilogue C subtracts Aqk W)
                    *reinterpret_cast<uint32_t*>(rp + kRecA1 + hh * 16384 + sw128_off(64 + i, cc)) =
                        pack_bf16x2(qq.x * a0, qq.y * a1);
                }
            }
            stall_point<kStall>(p.stall_seed, 3, it);
            {
                // backward over the group: [Yoff ; Yd] and the Kt image
                float z0 = hf ? 1.f : eB.x, z1 = hf ? 1.f : eB.y;
                float zc0 = __frcp_rn(hf ? fA.x * fB.x : fA.x), zc1 = __frcp_rn(hf ? fA.y * fB.y : fA.y);
                float eh0 = 0.f, eh1 = 0.f;
                uint32_t kh0[4], kh1[4];
#pragma unroll
                for (int l = 7; l >= 0; --l) {
                    const int i = 8 * h8 + l;
                    const float2 kk = bf16x2_to_float2(kw[l]);
                    st_u32(sm + P_Y + sw128_off(96 + i, cc), pack_bf16x2(kk.x * zc0, kk.y * zc1));
                    const float kz0 = kk.x * z0, kz1 = kk.y * z1;
#pragma unroll
                    for (int I = 1; I < 4; ++I)
                        if (I > G)
                            st_u32(sm + P_Y + sw128_off(yoff_row2(I, G, 8 * hf + l), cc),
                                   pack_bf16x2(kz0 * Dm0[I], kz1 * Dm1[I]));
                    const float hh0 = kz0 * E0, hh1 = kz1 * E1;
                    if (l & 1) {
                        eh0 = hh0; eh1 = hh1;
                    } else {
                        kh0[l >> 1] = pack_bf16x2(hh0, eh0);
                        kh1[l >> 1] = pack_bf16x2(hh1, eh1);
                    }
                    z0 *= p0[l]; z1 *= p1[l];
                    zc0 *= fmaxf(p0[l], kPFloor); zc1 *= fmaxf(p1[l], kPFloor);
                }
                *reinterpret_cast<uint4*>(rp + kRecKt + sw128_off(c0, 8 * h8)) =
                    make_uint4(kh0[0], kh0[1], kh0[2], kh0[3]);
                *reinterpret_cast<uint4*>(rp + kRecKt + sw128_off(c0 + 1, 8 * h8)) =
                    make_uint4(kh1[0], kh1[1], kh1[2], kh1[3]);
            }
            fence_proxy_async_smem();
            fence_proxy_async_global();  // Q e^Gam is overwritten by this record's bulk store
            stall_point<kStall>(p.stall_seed, 4, it);
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
            if (tid == 0) {
                // MMA A, this channel half: D += R Y^T, N = 160 (off-diagonal and diagonal blocks)
                umma_tile(tb + TM2_A, smem_u32(sm + P_R), 16384, smem_u32(sm + P_Y), kYHalf, 64,
                          idesc_bf16_f32(128, 160), hh > 0);
                umma_commit(&bar_mma[0]);
            }
            // The half's operands are read before the next half overwrites them
            // (two phases of the barrier per record: parity = half).
            ok = __syncthreads_and(tid == 0 ? mbar_wait(&bar_mma[0], (uint32_t)hh, nullptr) : true);
            tc_fence_after();
            if (!ok) break;
        }
        if (!ok) break;
        if (cn.len > 0) bcur = load_beta(cn, rec_next % p.H);

        float* sA = reinterpret_cast<float*>(sm + P_A);
        float* sT = reinterpret_cast<float*>(sm + P_T);
        float* sX = reinterpret_cast<float*>(sm + P_X);
        stall_point<kStall>(p.stall_seed, 5, it);
        // ---- Epilogue A: TMEM rows 0..63 are k rows (-> A, beta-scaled, j < i),
        // rows 64..127 are q rows (-> Aqk, j <= i, bf16 operand of MMA B); this warp
        // takes column blocks J = cq and cq + 2.
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {
            const int J = cq + 2 * jj;
            const bool isq = qd >= 2;
            const int i = 32 * (qd & 1) + lane, I = i >> 4, I0 = 2 * (qd & 1), I1 = I0 + 1;
            const bool lo = lane < 16;
            const float bi = sBeta[i];
            float t0[16], t1[16], tm[16];
            {
                uint32_t r0[16], r1[16], rm[16];
                tmem_ld16_issue(tmem_addr(tb, 32 * qd, TM2_A + yoff_row2(I0, J, 0)), r0);
                tmem_ld16_issue(tmem_addr(tb, 32 * qd, TM2_A + yoff_row2(I1, J, 0)), r1);
                tmem_ld16_issue(tmem_addr(tb, 32 * qd, TM2_DIAG + 16 * J), rm);
                tmem_wait_ld();
                tmem_take16(r0, t0);
                tmem_take16(r1, t1);
                tmem_take16(rm, tm);
            }
            float v[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                const int j = 16 * J + x;
                float val = 0.f;
                if (J < I) val = lo ? t0[x] : t1[x];
                else if (J == I) val = tm[x];
                v[x] = isq ? ((j <= i) ? val : 0.f) : ((j < i) ? tf32_round2(bi * val) : 0.f);
            }
            if (!isq) {
                float4* dst = reinterpret_cast<float4*>(sA + i * kPA2 + 16 * J);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            } else {
                uint32_t w[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) w[x] = pack_bf16x2(v[2 * x], v[2 * x + 1]);
                *reinterpret_cast<uint4*>(sm + P_AQK + sw128_off(i, 16 * J)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(sm + P_AQK + sw128_off(i, 16 * J + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        stall_point<kStall>(p.stall_seed, 6, it);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- UT transform, as in the one-CTA kernel: the four 16 x 16 diagonal
        // inverses by forward substitution (two warps per block, two column pairs
        // per half-warp), then the 16 -> 32 and 32 -> 64 block products on warp
        // MMAs; T' = T Diag(beta) goes to the TT / T'^T operands.
        {
            const int I = warp >> 1, m = lane & 15, s0 = 16 * I;
            float ar[16];
            const float4* arow = reinterpret_cast<const float4*>(sA + (s0 + m) * kPA2 + s0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 t = arow[u];
                ar[4 * u] = t.x; ar[4 * u + 1] = t.y; ar[4 * u + 2] = t.z; ar[4 * u + 3] = t.w;
            }
            const int src = lane & 16;
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                const int l = 8 * (warp & 1) + 4 * pass + 2 * (lane >> 4);
                float xa = (m == l) ? 1.f : 0.f, xb = (m == l + 1) ? 1.f : 0.f;
#pragma unroll
                for (int r = 0; r < 15; ++r) {
                    const float ya = __shfl_sync(0xffffffffu, xa, src + r);
                    const float yb = __shfl_sync(0xffffffffu, xb, src + r);
                    xa = fmaf(-ar[r], ya, xa);
                    xb = fmaf(-ar[r], yb, xb);
                }
                const int i = s0 + m, j = s0 + l;
                *reinterpret_cast<float2*>(sT + i * kPA2 + j) = make_float2(tf32_round2(xa), tf32_round2(xb));
                store_tprime_pair2(sm, i, j, xa, xb, sBeta);
            }
            // zero the 16 x 16 blocks of T' above the diagonal (TT) and below it (T'^T)
            for (int e = tid; e < 12 * 32; e += kP2Threads) {
                const int blkid = e >> 5, rr = (e >> 1) & 15, hc = e & 1;
                const int bi = blkid % 6;
                const int Ib = bi < 3 ? 0 : (bi < 5 ? 1 : 2);
                const int Jb = bi < 3 ? bi + 1 : (bi < 5 ? bi - 1 : 3);
                const int row = blkid < 6 ? 16 * Ib + rr : 16 * Jb + rr;
                const int col = blkid < 6 ? 16 * Jb + 8 * hc : 16 * Ib + 8 * hc;
                *reinterpret_cast<uint4*>(sm + (blkid < 6 ? P_TT : P_TTR) + sw128_off(row, col)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        stall_point<kStall>(p.stall_seed, 7, it);
        __syncthreads();
        const int g4 = lane >> 2, t4 = lane & 3;
        if (warp < 4) {
            // 16 -> 32 in 32-block pb, columns c0..c0+7: X = A_10 T_00, T_10 = -T_11 X
            const int pb = 32 * (warp >> 1), ct = warp & 1, c0 = 8 * ct;
            float* x = sX + (warp >> 1) * 16 * kPX2 + c0;
            float d[4];
            warp_mma_16x8_2(sA + (pb + 16) * kPA2 + pb, kPA2, sT + pb * kPA2 + pb + c0, kPA2, ct, 2, d, lane);
            store_tile_tf32_2(x, kPX2, d, lane);
            stall_point<kStall>(p.stall_seed, 8, it);
            __syncwarp();
            warp_mma_16x8_2(sT + (pb + 16) * kPA2 + pb + 16, kPA2, x, kPX2, 0, 2, d, lane);
            d[0] = -d[0]; d[1] = -d[1]; d[2] = -d[2]; d[3] = -d[3];
            store_tile_tf32_2(sT + (pb + 16) * kPA2 + pb + c0, kPA2, d, lane);
            store_tprime_pair2(sm, pb + 16 + g4, pb + c0 + 2 * t4, d[0], d[1], sBeta);
            store_tprime_pair2(sm, pb + 24 + g4, pb + c0 + 2 * t4, d[2], d[3], sBeta);
        }
        __syncthreads();
        {
            // 32 -> 64, row tile rt, columns c0..c0+7 (all eight warps):
            // X = A[32:, :32] T[:32, :32], then T[32:, :32] = -T[32:, 32:] X
            const int rt = warp >> 2, ct = warp & 3, c0 = 8 * ct;
            float d[4];
            warp_mma_16x8_2(sA + (32 + 16 * rt) * kPA2, kPA2, sT + c0, kPA2, ct, 4, d, lane);
            store_tile_tf32_2(sX + 16 * rt * kPX2 + c0, kPX2, d, lane);
            stall_point<kStall>(p.stall_seed, 9, it);
            __syncthreads();
            warp_mma_16x8_2(sT + (32 + 16 * rt) * kPA2 + 32, kPA2, sX + c0, kPX2, 0, 2 * (rt + 1), d, lane);
            const int r0 = 32 + 16 * rt + g4;
            store_tprime_pair2(sm, r0, c0 + 2 * t4, -d[0], -d[1], sBeta);
            store_tprime_pair2(sm, r0 + 8, c0 + 2 * t4, -d[2], -d[3], sBeta);
        }
        stall_point<kStall>(p.stall_seed, 10, it);
        fence_proxy_async_smem();
        __syncthreads();
        // ---- MMA B: D_b = Aqk T' -> rows 64..127 of the TT operand
        if (tid == 0) {
            tc_fence_after();
            umma_tile(tb + TM2_B, smem_u32(sm + P_AQK), 0, smem_u32(sm + P_TTR), 0, 64,
                      idesc_bf16_f32(128, 64), false);
            umma_commit(&bar_mma[1]);
        }
        // ---- E2b, while MMA B runs: [K e^Gam | V] (B of MMA C, MN-major: token
        // row i, channels contiguous) over the solve's dead fp32 scratch.
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            const int c0 = 64 * hh + cp2;
            const float* tot = reinterpret_cast<const float*>(sm + P_TOT);
            float p0[8], p1[8];
            load_p(hh, p0, p1);
            float Bg0 = 1.f, Bg1 = 1.f;
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                if (J < G) {
                    const float2 u = *reinterpret_cast<const float2*>(tot + (2 * J) * 128 + c0);
                    const float2 w = *reinterpret_cast<const float2*>(tot + (2 * J + 1) * 128 + c0);
                    Bg0 *= u.x * w.x; Bg1 *= u.y * w.y;
                }
            }
            const float2 eA = *reinterpret_cast<const float2*>(tot + (2 * G) * 128 + c0);
            float a0 = hf ? Bg0 * eA.x : Bg0, a1 = hf ? Bg1 * eA.y : Bg1;
            const Rows rw = rows_of(p, ci, h, c0);
            uint32_t kw[8], vw[8];
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                const int i = 8 * h8 + l;
                kw[l] = i < len ? ldg_u32(rw.k + (int64_t)i * p.ks[1]) : 0u;
                vw[l] = i < len ? ldg_u32(rw.v + (int64_t)i * p.vs[1]) : 0u;
            }
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                const int i = 8 * h8 + l;
                a0 *= p0[l]; a1 *= p1[l];
                const float2 kk = bf16x2_to_float2(kw[l]);
                st_u32(sm + P_KV + mn_sw128_off(i, c0, kKvSbo2), pack_bf16x2(kk.x * a0, kk.y * a1));
                st_u32(sm + P_KV + mn_sw128_off(i, 128 + c0, kKvSbo2), vw[l]);
            }
        }
        fence_proxy_async_smem();
        ok = __syncthreads_and(tid == 0 ? mbar_wait(&bar_mma[1], it & 1, nullptr) : true);
        tc_fence_after();
        if (!ok) break;
        stall_point<kStall>(p.stall_seed, 11, it);
        if (qd < 2) {
            const int i = 32 * qd + lane;
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int col = 16 * (cq + 2 * jj);
                float v[16];
                tmem_ld16(tmem_addr(tb, 32 * qd, TM2_B + col), v);
#pragma unroll
                for (int x = 0; x < 16; x += 2)
                    st_u32(sm + P_TT + sw128_off(64 + i, col + x), pack_bf16x2(v[x], v[x + 1]));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA C: [T' ; Aqk T'] [K e^Gam | V] = [W | U ; Aqk W | Aqk U]  (N = 256)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t tt = smem_u32(sm + P_TT), kv = smem_u32(sm + P_KV);
            for (uint32_t k = 0; k < 4; ++k)
                umma_bf16(tb + TM2_C, sdesc_kmajor_sw128(tt + k * 32u),
                          sdesc_mnmajor_sw128(kv + k * 2u * kKvSbo2, 1024u, kKvSbo2),
                          idesc_bf16_f32_bmn(128, 256), k > 0 ? 1u : 0u);
            umma_commit(&bar_mma[2]);
        }
        ok = __syncthreads_and(tid == 0 ? mbar_wait(&bar_mma[2], it & 1, nullptr) : true);
        tc_fence_after();
        if (!ok) break;
        stall_point<kStall>(p.stall_seed, 12, it);
        {
            // ---- Epilogue C: [W ; Q'] rows (Q' = Q e^Gam - Aqk W, Q e^Gam read back
            // from the record) from the first 128 columns and U / O_loc from the
            // last 128, staged as the record's images.
            const int r = 32 * qd + lane, i = r & 63;
            const bool top = qd < 2;
#pragma unroll 1
            for (int jj = 0; jj < 2; ++jj) {
                const int cqv = cq + 2 * jj, half = cqv >> 1;
#pragma unroll 1
                for (int cg2 = 0; cg2 < 2; ++cg2) {
                    float vv[32];
                    tmem_ld32(tmem_addr(tb, 32 * qd, TM2_C + 128 * half + 64 * (cqv & 1) + 32 * cg2), vv);
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {
                        const int col = 64 * (cqv & 1) + 32 * cg2 + 16 * hq;
                        const float* v = vv + 16 * hq;
                        uint32_t w[8];
                        if (half == 0) {
                            if (top) {
#pragma unroll
                                for (int x = 0; x < 8; ++x) w[x] = pack_bf16x2(v[2 * x], v[2 * x + 1]);
                            } else {
                                const uint8_t* qsrc = rp + kRecA1 + (col >> 6) * 16384;
                                const uint4 q0 = *reinterpret_cast<const uint4*>(qsrc + sw128_off(r, col & 63));
                                const uint4 q1 = *reinterpret_cast<const uint4*>(qsrc + sw128_off(r, (col & 63) + 8));
                                const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                                for (int x = 0; x < 8; ++x) {
                                    const float2 q2 = bf16x2_to_float2(qw[x]);
                                    w[x] = pack_bf16x2(q2.x - v[2 * x], q2.y - v[2 * x + 1]);
                                }
                            }
                            uint8_t* img = sm + P_SA1 + (col >> 6) * 16384;
                            *reinterpret_cast<uint4*>(img + sw128_off(r, col & 63)) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4*>(img + sw128_off(r, (col & 63) + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
                        } else {
                            uint8_t* img = sm + (top ? P_SU : P_SOL) + (col >> 5) * kSlabImg;
                            const int c8 = (col & 31) >> 3;
#pragma unroll
                            for (int x = 0; x < 8; ++x) w[x] = pack_bf16x2(v[2 * x], v[2 * x + 1]);
                            *reinterpret_cast<uint4*>(img + slab_chunk_off(i, c8)) = make_uint4(w[0], w[1], w[2], w[3]);
                            *reinterpret_cast<uint4*>(img + slab_chunk_off(i, c8 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                }
            }
        }
        stall_point<kStall>(p.stall_seed, 13, it);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            bulk_store(rp + kRecA1, sm + P_SA1, 32768);
            bulk_store(rp + kRecU, sm + P_SU, 4 * kSlabImg);
            bulk_store(rp + kRecOl, sm + P_SOL, 4 * kSlabImg);
            bulk_commit();
        }
        tc_fence_before();
        __syncthreads();
        rec = rec_next;
        ci = cn;
    }
    if (!ok && tid == 0) atomicExch(p.status, 4);
    if (tid == 0) bulk_wait_all();  // no bulk store may outlive the CTA's shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TM2_COLS);
}

}  // namespace

cudaError_t launch_prep2(const PrefillParams& p, int num_sms, cudaStream_t s, bool overlap_previous) {
    const long long recs = (long long)p.max_chunks * p.H;
    if (recs == 0) return cudaSuccess;
    // the instantiation with the stall hook runs only when a test asks for it
    auto kern = p.stall_seed ? prep2_kernel<true> : prep2_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kP2Smem);
    if (e != cudaSuccess) return e;
    const long long slots = 2LL * num_sms;  // two CTAs per SM
    const unsigned grid = (unsigned)(recs < slots ? recs : slots);
    if (!overlap_previous) {
        kern<<<grid, kP2Threads, kP2Smem, s>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kP2Threads);
    cfg.dynamicSmemBytes = kP2Smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace kda
