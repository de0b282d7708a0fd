// kda_prep.cu -- per-chunk preparation for KDA prefill (steps A1-A5): the chunk
// table, the in-chunk gate cumsum and chunk total, the beta sigmoid, tail
// masking, gate-scaled operands, the intra-chunk interaction matrices on
// tcgen05 tensor cores, the UT transform T = (I + Diag(beta) tril(K K^T . decay))^-1
// and the per-chunk operands the serial state pass consumes.
//
// Per chunk of 64 tokens (rows i, j) and key channel c, with Gam the in-chunk
// inclusive gate cumsum (the TensorRT-LLM K1 "prefix row"; gam = chunk total):
//   A[i,j]   = beta_i sum_c k_i k_j exp(Gam_i - Gam_j)     j <  i
//   Aqk[i,j] =        sum_c q_i k_j exp(Gam_i - Gam_j)     j <= i
//   T = (I + A)^-1,  T' = T Diag(beta)
//   W  = T' (K e^Gam),  U = T' V,  Q' = Q e^Gam - Aqk W,  O_loc = Aqk U
//   Kt = (K e^{gam - Gam})^T,  eg = e^gam
// so that, for the chunk's entry state S, the serial pass only needs
//   V_new = U - W S,  O = Q' S + O_loc,  S <- Diag(eg) S + Kt V_new.
//
// Overflow guard (the "100% NaN at gate -5" hazard on the cuDNN-frontend sm90
// KDA page, Conversation): exp(Gam_i - Gam_j) is never formed as
// exp(Gam_i) * exp(-Gam_j) over the whole chunk.  The chunk is cut into four
// 16-token blocks, and every gate factor is a running product of p = exp(g)
// (one exponential per element):
//   a_l  = prod_{t<=l} p_t   (block start -> token l, <= 1)
//   z_l  = prod_{t>l}  p_t   (token l -> block end,  <= 1)
// For a row block I and an earlier column block J the factor is
//   a_i * exp(sum of the gates of the blocks strictly between) * z_j,
// three factors <= 1.  Inside a block the factor is ac_i / ac_j with ac the
// running product of max(p, e^-5.4) (gate floored at kGateFloor), so that
// 1/ac stays below e^86.4 and fits fp32 / bf16; the floor changes a term only
// when its true decay is already below e^-5.4, and never for gates >= -5.4
// (the production gate bound is -5).
//
// Organisation: a persistent CTA (8 warps) per SM loops over (chunk, head)
// records.  The q, k, v and g tiles of a record arrive by TMA; the next
// record's tiles are requested as soon as the current record's gate phase has
// consumed its inputs, so the loads overlap the tensor-core and solve phases.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads = 256;

// Dynamic shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t O_IQ = 0;          // bf16 [64][128] q tile (TMA, plain rows)
constexpr uint32_t O_IK = 16384;      // bf16 [64][128] k tile
constexpr uint32_t O_IV = 32768;      // bf16 [64][128] v tile
constexpr uint32_t O_IG = 49152;      // fp32 [64][128] g tile
constexpr uint32_t kInBytes = 81920;
constexpr uint32_t O_R = 81920;       // A operand R = [K ac ; Q ac]: 2 x (128 rows x 128 B)
constexpr uint32_t O_Y = 114688;      // B operand [Yoff (96 rows) ; Yd (64 rows)]: 2 x (160 x 128 B)
constexpr uint32_t kYBlock = 160 * 128;
constexpr uint32_t O_KV = 155648;     // B operand [K e^Gam | V], MN-major: 8 token groups x 4 KB
constexpr uint32_t kKvSbo = 4096;     // byte distance between 8-token groups of the KV operand
constexpr uint32_t O_QT = 188416;     // bf16 [64][136] Q e^Gam (row pitch 272 B)
constexpr uint32_t kQtPitch = 272;
constexpr uint32_t O_TOT = 205824;    // fp32 [4][128] block gate totals
constexpr uint32_t O_BETA = 207872;   // fp32 [64] beta
constexpr uint32_t kPrepSmem = 208128 + 1024;
// Scratch of the solve and MMA B / C, over R and Y once MMA A has completed.
constexpr int kPA = 65;               // fp32 row pitch (conflict-free columns)
constexpr uint32_t O_A = 81920;       // fp32 [64][65] beta-scaled A
constexpr uint32_t O_T = 98560;       // fp32 [64][65] T
constexpr uint32_t O_X = 115200;      // fp32 [32][33] products
constexpr uint32_t O_AQK = 119808;    // A operand Aqk: 64 rows x 128 B (rows 64..127 are don't-care)
constexpr uint32_t O_TT = 128000;     // A operand [T' ; Aqk T']: 128 rows x 128 B
constexpr uint32_t O_TTR = 144384;    // B operand T'^T: 64 rows x 128 B
// Staging of the record images written by the last epilogue (over R, Y, KV).
constexpr uint32_t O_SA1 = 81920;     // [W ; Q'] image, 32 KB
constexpr uint32_t O_SU = 114688;     // U image, 16 KB
constexpr uint32_t O_SOL = 131072;    // O_loc image, 16 KB

// TMEM columns.
constexpr uint32_t TM_A = 0, TM_DIAG = 96, TM_B = 192, TM_C = 0, TM_COLS = 256;

__device__ __forceinline__ float2 ld_bf16x2(const uint8_t* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) {
    *reinterpret_cast<uint32_t*>(p) = v;
}
__device__ __forceinline__ void st_bf16(uint8_t* p, float v) {
    *reinterpret_cast<__nv_bfloat16*>(p) = __float2bfloat16_rn(v);
}
// Stores T' = T Diag(beta) entries (i, j) and (i, j + 1) of a computed T block
// into the TT operand (row i, K index j) and the T'^T operand (row j, K index i).
__device__ __forceinline__ void store_tprime_pair(uint8_t* sm, int i, int j, float t0, float t1,
                                                  const float* sBeta) {
    const float a = t0 * sBeta[j], b = t1 * sBeta[j + 1];
    st_u32(sm + O_TT + sw128_off(i, j), pack_bf16x2(a, b));
    st_bf16(sm + O_TTR + sw128_off(j, i), a);
    st_bf16(sm + O_TTR + sw128_off(j + 1, i), b);
}
// Row of the Yoff operand holding column block J as seen from row block I > J:
// block I's group holds its 16*I earlier columns.
__device__ __forceinline__ uint32_t yoff_row(int I, int J, int l) {
    return 8 * I * (I - 1) + 16 * J + l;
}

// Warp-level m16n8k8 tf32 MMA with fp32 accumulation (used for the small block
// products of the UT solve; fragment layouts of the PTX m16n8k8 tf32 shape).
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}
// d (16 x 8 tile) = P (16 x kdim, row pitch pp) * Q (kdim x 8, row pitch pq),
// fp32 matrices in shared memory.  Thread (g = lane/4, t = lane%4) gets
// d0 (g, 2t), d1 (g, 2t+1), d2 (g+8, 2t), d3 (g+8, 2t+1).
__device__ __forceinline__ void warp_mma_16x8(const float* P, int pp, const float* Q, int pq,
                                              int kdim, float (&d)[4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    d[0] = d[1] = d[2] = d[3] = 0.f;
    for (int k0 = 0; k0 < kdim; k0 += 8) {
        const uint32_t a0 = to_tf32(P[g * pp + k0 + t]), a1 = to_tf32(P[(g + 8) * pp + k0 + t]);
        const uint32_t a2 = to_tf32(P[g * pp + k0 + t + 4]), a3 = to_tf32(P[(g + 8) * pp + k0 + t + 4]);
        const uint32_t b0 = to_tf32(Q[(k0 + t) * pq + g]), b1 = to_tf32(Q[(k0 + t + 4) * pq + g]);
        asm volatile(
            "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// Issues the TMA loads of one record's q, k, v, g tiles.
__device__ __forceinline__ void load_inputs(uint8_t* sm, const PrepMaps& m, const ChunkInfo& ci,
                                            int h, uint64_t* bar) {
    mbar_arrive_expect_tx(bar, kInBytes);
    tma_load_4d(sm + O_IQ, &m.q, 0, h, ci.t0, ci.b, bar);
    tma_load_4d(sm + O_IK, &m.k, 0, h, ci.t0, ci.b, bar);
    tma_load_4d(sm + O_IV, &m.v, 0, h, ci.t0, ci.b, bar);
    tma_load_4d(sm + O_IG, &m.g, 0, h, ci.t0, ci.b, bar);
}

__global__ void __launch_bounds__(kPrepThreads, 1)
    prep_kernel(const PrefillParams p, const __grid_constant__ PrepMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t bar_in, bar_mma[3];
    __shared__ uint32_t tmem_base_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrec = p.max_chunks * p.H;
    if (blockIdx.x >= nrec) return;
    if (tid == 0) {
        mbar_init(&bar_in, 1);
        for (int i = 0; i < 3; ++i) mbar_init(&bar_mma[i], 1);
        fence_mbar_init();
        tma_prefetch_desc(&maps.q); tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v); tma_prefetch_desc(&maps.g);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;

    // Thread roles in the gate phases: block G (16 tokens), channels c0, c0 + 1.
    const int G = tid >> 6, c0 = 2 * (tid & 63), blk = c0 >> 6, cc = c0 & 63;
    // Roles in the TMEM epilogues: lane quarter qd, column half.
    const int qd = warp & 3, half = warp >> 2;
    const float kPFloor = __expf(kGateFloor);

    int rec = blockIdx.x;
    ChunkInfo ci = chunk_info(p, rec / p.H);
    if (tid == 0 && ci.len > 0) load_inputs(sm, maps, ci, rec % p.H, &bar_in);
    // beta of the current record, loaded one record ahead (raw value; the
    // sigmoid is applied when it is stored)
    auto load_beta = [&](const ChunkInfo& c, int hh) -> float {
        return (tid < c.len) ? __ldg(p.beta + c.b * p.bs[0] + ((int64_t)c.t0 + tid) * p.bs[1] + hh * p.bs[2])
                             : 0.f;
    };
    float bcur = load_beta(ci, rec % p.H);
    bool ok = true;
    int pend_parity = ci.len > 0 ? 0 : -1;  // parity of an input load still in flight
    for (uint32_t it = 0; ci.len > 0; ++it) {
        const int chunk = rec / p.H, h = rec - chunk * p.H;
        const int len = ci.len;
        const int rec_next = rec + gridDim.x;
        const ChunkInfo cn = rec_next < nrec ? chunk_info(p, rec_next / p.H) : ChunkInfo{0, 0, 0, 0, 0};
        ok = __syncthreads_and(mbar_wait(&bar_in, it & 1, nullptr));
        if (!ok) break;
        pend_parity = -1;
        if (tid < 64) {
            float bval = bcur;
            if (tid < len && p.beta_is_logit) bval = 1.0f / (1.0f + __expf(-bval));
            reinterpret_cast<float*>(sm + O_BETA)[tid] = tid < len ? bval : 0.f;
        }

        // ---- E1: p = exp(g) (masked past the chunk length), block gate totals,
        // and the suffix products z (exact) and zc (floored gate) by a backward pass.
        float p0[16], p1[16], z0[16], z1[16], zc0[16], zc1[16];
        {
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int l = 0; l < 16; ++l) {
                const int i = 16 * G + l;
                float2 gv = *reinterpret_cast<const float2*>(sm + O_IG + i * 512 + c0 * 4);
                if (i >= len) gv = make_float2(0.f, 0.f);
                d0 += gv.x; d1 += gv.y;
                p0[l] = __expf(gv.x); p1[l] = __expf(gv.y);
            }
            float s0 = 1.f, s1 = 1.f, t0 = 1.f, t1 = 1.f;
#pragma unroll
            for (int l = 15; l >= 0; --l) {
                z0[l] = s0; z1[l] = s1; zc0[l] = t0; zc1[l] = t1;
                s0 *= p0[l]; s1 *= p1[l];
                t0 *= fmaxf(p0[l], kPFloor); t1 *= fmaxf(p1[l], kPFloor);
            }
            float* tot = reinterpret_cast<float*>(sm + O_TOT);
            tot[G * 128 + c0] = d0;
            tot[G * 128 + c0 + 1] = d1;
        }
        if (tid == 0) bulk_wait_read();  // the previous record's images have left the staging area
        __syncthreads();

        // ---- E2: the MMA operands and the records that need no MMA.
        {
            const float* tot = reinterpret_cast<const float*>(sm + O_TOT);
            float d0[4], d1[4];
#pragma unroll
            for (int J = 0; J < 4; ++J) { d0[J] = tot[J * 128 + c0]; d1[J] = tot[J * 128 + c0 + 1]; }
            float pre0 = 0.f, pre1 = 0.f, post0 = 0.f, post1 = 0.f;
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                if (J < G) { pre0 += d0[J]; pre1 += d1[J]; }
                if (J > G) { post0 += d0[J]; post1 += d1[J]; }
            }
            const float B0 = __expf(pre0), B1 = __expf(pre1);    // chunk start -> block start
            const float E0 = __expf(post0), E1 = __expf(post1);  // block end -> chunk end
            float Dm0[4], Dm1[4];  // decay over the blocks strictly between G and I
            {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int I = 0; I < 4; ++I) {
                    Dm0[I] = __expf(s0); Dm1[I] = __expf(s1);
                    if (I > G) { s0 += d0[I]; s1 += d1[I]; }
                }
            }
            // 1 / (floored-gate block product): <= e^86.4
            const float ib0 = 1.0f / (fmaxf(p0[0], kPFloor) * zc0[0]);
            const float ib1 = 1.0f / (fmaxf(p1[0], kPFloor) * zc1[0]);
            uint8_t* rp = p.ws_rec + (size_t)rec * kRecBytes;
            if (G == 0)
                *reinterpret_cast<float2*>(rp + kRecEg + c0 * 4) =
                    make_float2(__expf(d0[0] + d0[1] + d0[2] + d0[3]),
                                __expf(d1[0] + d1[1] + d1[2] + d1[3]));
            const float qscale = p.scale;
            const uint32_t bo = blk * 16384u, yb = blk * kYBlock;
            float a0 = 1.f, a1 = 1.f, ac0 = 1.f, ac1 = 1.f;
            float eh0 = 0.f, eh1 = 0.f;
            uint32_t kh0[8], kh1[8];
#pragma unroll
            for (int l = 0; l < 16; ++l) {
                const int i = 16 * G + l;
                const bool valid = i < len;
                a0 *= p0[l]; a1 *= p1[l];
                ac0 *= fmaxf(p0[l], kPFloor); ac1 *= fmaxf(p1[l], kPFloor);
                float2 kk = ld_bf16x2(sm + O_IK + i * 256 + c0 * 2);
                float2 qq = ld_bf16x2(sm + O_IQ + i * 256 + c0 * 2);
                float2 vv = ld_bf16x2(sm + O_IV + i * 256 + c0 * 2);
                if (!valid) { kk = make_float2(0.f, 0.f); qq = kk; vv = kk; }
                qq.x *= qscale; qq.y *= qscale;
                // R = [K ac ; Q ac]
                st_u32(sm + O_R + bo + sw128_off(i, cc), pack_bf16x2(kk.x * ac0, kk.y * ac1));
                st_u32(sm + O_R + bo + sw128_off(64 + i, cc), pack_bf16x2(qq.x * ac0, qq.y * ac1));
                // Yd (diagonal blocks): K / ac = K zc / ac_block
                st_u32(sm + O_Y + yb + sw128_off(96 + i, cc),
                       pack_bf16x2(kk.x * zc0[l] * ib0, kk.y * zc1[l] * ib1));
                // Yoff: column block G seen from each later row block I
#pragma unroll
                for (int I = 1; I < 4; ++I)
                    if (I > G)
                        st_u32(sm + O_Y + yb + sw128_off(yoff_row(I, G, l), cc),
                               pack_bf16x2(kk.x * z0[l] * Dm0[I], kk.y * z1[l] * Dm1[I]));
                // Q e^Gam for Q'
                const float ea0 = a0 * B0, ea1 = a1 * B1;
                st_u32(sm + O_QT + i * kQtPitch + c0 * 2, pack_bf16x2(qq.x * ea0, qq.y * ea1));
                // [K e^Gam | V] (MN-major: token row i, channels contiguous)
                st_u32(sm + O_KV + mn_sw128_off(i, c0, kKvSbo), pack_bf16x2(kk.x * ea0, kk.y * ea1));
                st_u32(sm + O_KV + mn_sw128_off(i, 128 + c0, kKvSbo), pack_bf16x2(vv.x, vv.y));
                // Kt = (K e^{gam - Gam})^T, packed by token pairs
                const float hh0 = kk.x * z0[l] * E0, hh1 = kk.y * z1[l] * E1;
                if ((l & 1) == 0) {
                    eh0 = hh0; eh1 = hh1;
                } else {
                    kh0[l >> 1] = pack_bf16x2(eh0, hh0);
                    kh1[l >> 1] = pack_bf16x2(eh1, hh1);
                }
            }
            // Kt image rows c0, c0 + 1: tokens 16G..16G+15 are 16-byte chunks 2G, 2G+1
            uint8_t* kt = rp + kRecKt;
            *reinterpret_cast<uint4*>(kt + sw128_off(c0, 16 * G)) = make_uint4(kh0[0], kh0[1], kh0[2], kh0[3]);
            *reinterpret_cast<uint4*>(kt + sw128_off(c0, 16 * G + 8)) = make_uint4(kh0[4], kh0[5], kh0[6], kh0[7]);
            *reinterpret_cast<uint4*>(kt + sw128_off(c0 + 1, 16 * G)) = make_uint4(kh1[0], kh1[1], kh1[2], kh1[3]);
            *reinterpret_cast<uint4*>(kt + sw128_off(c0 + 1, 16 * G + 8)) = make_uint4(kh1[4], kh1[5], kh1[6], kh1[7]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        // The input tiles are consumed: fetch the next record's while this one
        // goes through the tensor cores and the solve.
        if (tid == 0 && cn.len > 0) {
            load_inputs(sm, maps, cn, rec_next % p.H, &bar_in);
        }
        if (cn.len > 0) bcur = load_beta(cn, rec_next % p.H);
        if (cn.len > 0) pend_parity = (int)((it + 1) & 1);

        // ---- MMA A: D = R [Yoff ; Yd]^T, N = 160 (off-diagonal and diagonal blocks)
        if (tid == 0) {
            umma_tile(tb + TM_A, smem_u32(sm + O_R), 16384, smem_u32(sm + O_Y), kYBlock, 128,
                      idesc_bf16_f32(128, 160), false);
            umma_commit(&bar_mma[0]);
        }
        ok = __syncthreads_and(mbar_wait(&bar_mma[0], it & 1, nullptr));
        tc_fence_after();
        if (!ok) break;

        float* sA = reinterpret_cast<float*>(sm + O_A);
        float* sT = reinterpret_cast<float*>(sm + O_T);
        float* sX = reinterpret_cast<float*>(sm + O_X);
        const float* sBeta = reinterpret_cast<const float*>(sm + O_BETA);
        {
            // ---- Epilogue A: TMEM rows 0..63 are k rows (-> A, beta-scaled, j < i),
            // rows 64..127 are q rows (-> Aqk, j <= i, bf16 operand of MMA B).
            const bool isq = qd >= 2;
            const int i = 32 * (qd & 1) + lane, I = i >> 4, I0 = 2 * (qd & 1), I1 = I0 + 1;
            const bool lo = lane < 16;
            const float bi = sBeta[i];
#pragma unroll
            for (int jg = 0; jg < 2; ++jg) {
                const int J = 2 * half + jg;
                float t0[16], t1[16], tm[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) { t0[x] = 0.f; t1[x] = 0.f; tm[x] = 0.f; }
                if (J < I0) tmem_ld16(tmem_addr(tb, 32 * qd, TM_A + yoff_row(I0, J, 0)), t0);
                if (J < I1) tmem_ld16(tmem_addr(tb, 32 * qd, TM_A + yoff_row(I1, J, 0)), t1);
                if (J <= I1) tmem_ld16(tmem_addr(tb, 32 * qd, TM_DIAG + 16 * J), tm);
#pragma unroll
                for (int jj = 0; jj < 16; jj += 2) {
                    float v2[2];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int j = 16 * J + jj + e;
                        float val = 0.f;
                        if (J < I) val = lo ? t0[jj + e] : t1[jj + e];
                        else if (J == I) val = tm[jj + e];
                        v2[e] = isq ? ((j <= i) ? val : 0.f) : ((j < i) ? bi * val : 0.f);
                    }
                    const int j = 16 * J + jj;
                    if (!isq) {
                        sA[i * kPA + j] = v2[0];
                        sA[i * kPA + j + 1] = v2[1];
                    } else {
                        st_u32(sm + O_AQK + sw128_off(i, j), pack_bf16x2(v2[0], v2[1]));
                    }
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- UT transform: T = (I + A)^-1 for the unit lower-triangular 64 x 64
        // system, fp32, blocked: four 16 x 16 diagonal inverses by forward
        // substitution, then [[Ta,0],[Aba,Tb]]^-1 = [[Ta^-1,0],[-Tb^-1 Aba Ta^-1, Tb^-1]]
        // at 16 -> 32 and 32 -> 64.  Blocks above the diagonal are never read
        // except the two 16 x 16 ones inside the 32 x 32 diagonal blocks, which
        // are written as zeros.
        if (tid < 64) {
            const int I = tid >> 4, l = tid & 15, s0 = 16 * I;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == l) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                const float* ar = sA + (s0 + r) * kPA + s0;
                float acc[4] = {x[r], 0.f, 0.f, 0.f};
#pragma unroll
                for (int m = 0; m < r; ++m) acc[m & 3] = fmaf(-ar[m], x[m], acc[m & 3]);
                x[r] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(s0 + r) * kPA + s0 + l] = x[r];
            // T' of the diagonal block: column s0+l of TT, row s0+l of T'^T
            const float bl = sBeta[s0 + l];
#pragma unroll
            for (int r = 0; r < 16; ++r) st_bf16(sm + O_TT + sw128_off(s0 + r, s0 + l), x[r] * bl);
            uint32_t w[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) w[r] = pack_bf16x2(x[2 * r] * bl, x[2 * r + 1] * bl);
            *reinterpret_cast<uint4*>(sm + O_TTR + sw128_off(s0 + l, s0)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(sm + O_TTR + sw128_off(s0 + l, s0 + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
        } else {
            // Zero the 16 x 16 blocks of T' above the diagonal (TT: column block
            // J > row block I) and below it in T'^T: 12 blocks x 16 rows x 2 chunks.
            for (int e = tid - 64; e < 12 * 32; e += kPrepThreads - 64) {
                const int blkid = e >> 5, rr = (e >> 1) & 15, half = e & 1;
                const int bi = blkid % 6;
                const int I = bi < 3 ? 0 : (bi < 5 ? 1 : 2);
                const int J = bi < 3 ? bi + 1 : (bi < 5 ? bi - 1 : 3);
                const int row = blkid < 6 ? 16 * I + rr : 16 * J + rr;
                const int col = blkid < 6 ? 16 * J + 8 * half : 16 * I + 8 * half;
                *reinterpret_cast<uint4*>(sm + (blkid < 6 ? O_TT : O_TTR) + sw128_off(row, col)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncthreads();
        // Off-diagonal blocks with warp-level tf32 tensor-core products (fp32
        // accumulation; the result is rounded to bf16 for MMA C anyway).  Each
        // warp owns a column block of its products, so the two dependent
        // products of a level need only a warp barrier between them.
        const int g4 = lane >> 2, t4 = lane & 3;
        if (warp < 4) {
            // 16 -> 32: in 32-block p, X = A_10 T_00, then T_10 = -T_11 X and T_01 = 0
            const int pb = 32 * (warp >> 1), c0 = 8 * (warp & 1);
            float d[4];
            warp_mma_16x8(sA + (pb + 16) * kPA + pb, kPA, sT + pb * kPA + pb + c0, kPA, 16, d, lane);
            float* x = sX + (warp >> 1) * 256;
            x[g4 * 16 + c0 + 2 * t4] = d[0]; x[g4 * 16 + c0 + 2 * t4 + 1] = d[1];
            x[(g4 + 8) * 16 + c0 + 2 * t4] = d[2]; x[(g4 + 8) * 16 + c0 + 2 * t4 + 1] = d[3];
            __syncwarp();
            warp_mma_16x8(sT + (pb + 16) * kPA + pb + 16, kPA, sX + (warp >> 1) * 256 + c0, 16, 16, d, lane);
            float* t10 = sT + (pb + 16) * kPA + pb + c0;
            t10[g4 * kPA + 2 * t4] = -d[0]; t10[g4 * kPA + 2 * t4 + 1] = -d[1];
            t10[(g4 + 8) * kPA + 2 * t4] = -d[2]; t10[(g4 + 8) * kPA + 2 * t4 + 1] = -d[3];
            store_tprime_pair(sm, pb + 16 + g4, pb + c0 + 2 * t4, -d[0], -d[1], sBeta);
            store_tprime_pair(sm, pb + 24 + g4, pb + c0 + 2 * t4, -d[2], -d[3], sBeta);
            float* t01 = sT + pb * kPA + pb + 16 + c0;
            t01[g4 * kPA + 2 * t4] = 0.f; t01[g4 * kPA + 2 * t4 + 1] = 0.f;
            t01[(g4 + 8) * kPA + 2 * t4] = 0.f; t01[(g4 + 8) * kPA + 2 * t4 + 1] = 0.f;
        }
        __syncthreads();
        if (warp < 4) {
            // 32 -> 64: warp w owns columns c0..c0+7 of X = A[32:,:32] T[:32,:32]
            // (both 16-row tiles) and then of T[32:,:32] = -T[32:,32:] X
            const int c0 = 8 * warp;
            float d0[4], d1[4];
            warp_mma_16x8(sA + 32 * kPA, kPA, sT + c0, kPA, 32, d0, lane);
            warp_mma_16x8(sA + 48 * kPA, kPA, sT + c0, kPA, 32, d1, lane);
            float* x = sX + c0;
            x[g4 * 33 + 2 * t4] = d0[0]; x[g4 * 33 + 2 * t4 + 1] = d0[1];
            x[(g4 + 8) * 33 + 2 * t4] = d0[2]; x[(g4 + 8) * 33 + 2 * t4 + 1] = d0[3];
            x[(g4 + 16) * 33 + 2 * t4] = d1[0]; x[(g4 + 16) * 33 + 2 * t4 + 1] = d1[1];
            x[(g4 + 24) * 33 + 2 * t4] = d1[2]; x[(g4 + 24) * 33 + 2 * t4 + 1] = d1[3];
            __syncwarp();
            warp_mma_16x8(sT + 32 * kPA + 32, kPA, sX + c0, 33, 32, d0, lane);
            warp_mma_16x8(sT + 48 * kPA + 32, kPA, sX + c0, 33, 32, d1, lane);
            float* t = sT + 32 * kPA + c0;
            t[g4 * kPA + 2 * t4] = -d0[0]; t[g4 * kPA + 2 * t4 + 1] = -d0[1];
            t[(g4 + 8) * kPA + 2 * t4] = -d0[2]; t[(g4 + 8) * kPA + 2 * t4 + 1] = -d0[3];
            t[(g4 + 16) * kPA + 2 * t4] = -d1[0]; t[(g4 + 16) * kPA + 2 * t4 + 1] = -d1[1];
            t[(g4 + 24) * kPA + 2 * t4] = -d1[2]; t[(g4 + 24) * kPA + 2 * t4 + 1] = -d1[3];
            store_tprime_pair(sm, 32 + g4, c0 + 2 * t4, -d0[0], -d0[1], sBeta);
            store_tprime_pair(sm, 40 + g4, c0 + 2 * t4, -d0[2], -d0[3], sBeta);
            store_tprime_pair(sm, 48 + g4, c0 + 2 * t4, -d1[0], -d1[1], sBeta);
            store_tprime_pair(sm, 56 + g4, c0 + 2 * t4, -d1[2], -d1[3], sBeta);
        }
        fence_proxy_async_smem();
        __syncthreads();
        // ---- MMA B: D_b = Aqk T'  -> rows 64..127 of the TT operand
        if (tid == 0) {
            tc_fence_after();
            umma_tile(tb + TM_B, smem_u32(sm + O_AQK), 0, smem_u32(sm + O_TTR), 0, 64,
                      idesc_bf16_f32(128, 64), false);
            umma_commit(&bar_mma[1]);
        }
        ok = __syncthreads_and(mbar_wait(&bar_mma[1], it & 1, nullptr));
        tc_fence_after();
        if (!ok) break;
        if (qd < 2) {
            const int i = 32 * qd + lane;
#pragma unroll
            for (int cg = 0; cg < 2; ++cg) {
                const int col = 32 * half + 16 * cg;
                float v[16];
                tmem_ld16(tmem_addr(tb, 32 * qd, TM_B + col), v);
#pragma unroll
                for (int x = 0; x < 16; x += 2)
                    st_u32(sm + O_TT + sw128_off(64 + i, col + x), pack_bf16x2(v[x], v[x + 1]));
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA C: [T' ; Aqk T'] [K e^Gam | V] = [W | U ; Aqk W | Aqk U]  (N = 256)
        if (tid == 0) {
            tc_fence_after();
            const uint32_t tt = smem_u32(sm + O_TT), kv = smem_u32(sm + O_KV);
            for (uint32_t k = 0; k < 4; ++k)
                umma_bf16(tb + TM_C, sdesc_kmajor_sw128(tt + k * 32u),
                          sdesc_mnmajor_sw128(kv + k * 2u * kKvSbo, 1024u, kKvSbo),
                          idesc_bf16_f32_bmn(128, 256), k > 0 ? 1u : 0u);
            umma_commit(&bar_mma[2]);
        }
        ok = __syncthreads_and(mbar_wait(&bar_mma[2], it & 1, nullptr));
        tc_fence_after();
        if (!ok) break;
        {
            // ---- Epilogue C: [W ; Q'] rows (Q' = Q e^Gam - Aqk W) from the first 128
            // columns and U / O_loc from the last 128, written as the record's
            // shared-memory images and stored with bulk copies.
            const int r = 32 * qd + lane, i = r & 63;
            const bool top = qd < 2;
#pragma unroll 1
            for (int cg = 0; cg < 8; ++cg) {
                const int col = 16 * cg;
                float v[16];
                tmem_ld16(tmem_addr(tb, 32 * qd, TM_C + 128 * half + col), v);
                if (half == 0) {
                    uint32_t w[8];
                    if (top) {
#pragma unroll
                        for (int x = 0; x < 8; ++x) w[x] = pack_bf16x2(v[2 * x], v[2 * x + 1]);
                    } else {
                        const uint8_t* qt = sm + O_QT + i * kQtPitch + col * 2;
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            const float2 q2 = ld_bf16x2(qt + 4 * x);
                            w[x] = pack_bf16x2(q2.x - v[2 * x], q2.y - v[2 * x + 1]);
                        }
                    }
                    uint8_t* img = sm + O_SA1 + (col >> 6) * 16384;
                    *reinterpret_cast<uint4*>(img + sw128_off(r, col & 63)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(img + sw128_off(r, (col & 63) + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
                } else {
                    uint8_t* img = sm + (top ? O_SU : O_SOL) + (col >> 5) * kSlabImg;
                    const int c8 = (col & 31) >> 3;
                    uint32_t w[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) w[x] = pack_bf16x2(v[2 * x], v[2 * x + 1]);
                    *reinterpret_cast<uint4*>(img + slab_chunk_off(i, c8)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(img + slab_chunk_off(i, c8 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            uint8_t* rp = p.ws_rec + (size_t)rec * kRecBytes;
            bulk_store(rp + kRecA1, sm + O_SA1, 32768);
            bulk_store(rp + kRecU, sm + O_SU, 4 * kSlabImg);
            bulk_store(rp + kRecOl, sm + O_SOL, 4 * kSlabImg);
            bulk_commit();
        }
        tc_fence_before();
        __syncthreads();
        rec = rec_next;
        ci = cn;
    }
    if (!ok && tid == 0) atomicExch(p.status, 4);
    if (tid == 0) bulk_wait_all();  // no bulk store may outlive the CTA's shared memory
    // Never leave with a copy in flight (only possible after a failed wait).
    if (pend_parity >= 0 && tid == 0) mbar_wait(&bar_in, (uint32_t)pend_parity, nullptr);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TM_COLS);
}

// A1: chunk table of packed sequences.  chunk_off[n] = sum_{m<n} ceil(L_m / 64);
// sequences of length 0 own no chunk ("gap-safe" mapping).  cu_seqlens that do
// not start at 0, decrease, or do not end at the token count are reported as
// KDA_ERR_INVALID_ARG and produce an empty table (no chunk is processed).
__global__ void __launch_bounds__(1024) chunk_table_kernel(const PrefillParams p) {
    __shared__ int bad;
    __shared__ int carry;
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        bad = (p.cu[0] != 0 || p.cu[p.N] != p.T) ? 1 : 0;
        carry = 0;
    }
    __syncthreads();
    for (int n = tid; n < p.N; n += blockDim.x)
        if (p.cu[n + 1] < p.cu[n]) atomicOr(&bad, 1);
    __syncthreads();
    if (bad) {
        for (int n = tid; n <= p.N; n += blockDim.x) p.chunk_off[n] = 0;
        if (tid == 0) atomicExch(p.status, 1);
        return;
    }
    for (int base = 0; base < p.N; base += blockDim.x) {
        const int n = base + tid;
        const int cnt = (n < p.N) ? (p.cu[n + 1] - p.cu[n] + kChunk - 1) / kChunk : 0;
        int x = cnt;  // inclusive warp scan
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int excl = carry + (warp > 0 ? wsum[warp - 1] : 0) + x - cnt;
        if (n < p.N) p.chunk_off[n] = excl;
        __syncthreads();
        if (tid == blockDim.x - 1) carry = excl + cnt;
        __syncthreads();
    }
    if (tid == 0) p.chunk_off[p.N] = carry;
}

}  // namespace

cudaError_t launch_chunk_table(const PrefillParams& p, cudaStream_t s) {
    if (p.cu == nullptr) return cudaSuccess;
    chunk_table_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prep(const PrefillParams& p, const PrepMaps& maps, int num_sms, cudaStream_t s) {
    const long long recs = (long long)p.max_chunks * p.H;
    if (recs == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(recs < num_sms ? recs : num_sms);
    prep_kernel<<<grid, kPrepThreads, kPrepSmem, s>>>(p, maps);
    return cudaGetLastError();
}

}  // namespace kda
