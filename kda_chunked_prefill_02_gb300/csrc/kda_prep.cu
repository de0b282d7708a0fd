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
// 16-token blocks.  For a row block I and an earlier column block J the factor
// splits at the end of block J into two factors that are both <= 1:
//   exp(Gam_i - Gam_{e_J}) * exp(Gam_{e_J} - Gam_j).
// Inside a block the split point is the block's 8th token and the per-token
// gate is floored at -10 (kGateClamp), so neither factor exceeds e^80; the
// floor changes a term only when its true decay is already below e^-10.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads = 256;

// Dynamic shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t O_Q = 0;          // bf16 [64][128] q rows (plain), later fp32 A  [64][64]
constexpr uint32_t O_K = 16384;      // bf16 [64][128] k rows,         later fp32 T  [64][64]
constexpr uint32_t O_V = 32768;      // bf16 [64][128] v rows,         later fp32 X  [32][32]
constexpr uint32_t O_G = 49152;      // fp32 [64][128] g rows; then R operand (2 x 16 KB);
                                     // then Aqk operand [128 x 64] + TT operand [128 x 64]
constexpr uint32_t O_RM = 81920;     // Rmid operand (2 x 16 KB); later T'^T operand [64 x 64]
constexpr uint32_t O_YO = 114688;    // Yoff operand, 96 rows (2 x 12 KB)
constexpr uint32_t O_YM = 139264;    // Ymid operand, 64 rows (2 x 8 KB)
constexpr uint32_t O_KV = 155648;    // [K e^Gam | V]^T operand, 256 rows x 64 tokens
constexpr uint32_t O_QT = 188416;    // bf16 [64][136] Q e^Gam (row pitch 272 B)
constexpr uint32_t O_TOT = 205824;   // fp32 [4][128] block gate totals
constexpr uint32_t O_BETA = 207872;  // fp32 [64] beta
constexpr uint32_t kPrepSmem = 208128 + 1024;

// fp32 scratch of the UT solve (row pitch 65 floats: conflict-free column access)
constexpr uint32_t O_AKK = 0, O_T = 16896, O_X = 33792;
constexpr int kPA = 65;
constexpr uint32_t O_AQK = O_G, O_TT = O_G + 16384, O_TTR = O_RM;
constexpr uint32_t kQtPitch = 272;

// TMEM columns.
constexpr uint32_t TM_OFF = 0, TM_MID = 128, TM_B = 192, TM_C = 0, TM_COLS = 256;

__device__ __forceinline__ float2 ld_bf16x2(const uint8_t* p) {
    const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(p);
    return __bfloat1622float2(h);
}
__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) {
    *reinterpret_cast<uint32_t*>(p) = v;
}
// Column offset of (row block I, column block J) inside the Yoff operand:
// block I's group holds its 16*I earlier columns (J = 0..I-1).
__device__ __forceinline__ uint32_t yoff_row(int I, int J, int l) { return 8 * I * (I - 1) + 16 * J + l; }

__global__ void __launch_bounds__(kPrepThreads, 1) prep_kernel(const PrefillParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t bar_mma[3];
    __shared__ uint32_t tmem_base_sh;

    const int rec = blockIdx.x;
    const int chunk = rec / p.H, h = rec - chunk * p.H;
    const ChunkInfo ci = chunk_info(p, chunk);
    if (ci.len <= 0) return;  // beyond the last chunk (varlen upper bound)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar_mma[i], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, TM_COLS);
        tmem_relinquish();
    }

    // ---- L: load q, k, v (bf16) and g (fp32) rows with 128-bit loads; rows at
    // or past the chunk length become zeros (tail masking).
    {
        const int64_t tb = (int64_t)ci.t0;
        for (int it = tid; it < 64 * 16; it += kPrepThreads) {
            const int row = it >> 4, ch = it & 15;
            uint4 vq = make_uint4(0, 0, 0, 0), vk = vq, vv = vq;
            if (row < ci.len) {
                const int64_t t = tb + row;
                vq = __ldg(reinterpret_cast<const uint4*>(p.q + ci.b * p.qs[0] + t * p.qs[1] + h * p.qs[2]) + ch);
                vk = __ldg(reinterpret_cast<const uint4*>(p.k + ci.b * p.ks[0] + t * p.ks[1] + h * p.ks[2]) + ch);
                vv = __ldg(reinterpret_cast<const uint4*>(p.v + ci.b * p.vs[0] + t * p.vs[1] + h * p.vs[2]) + ch);
            }
            *reinterpret_cast<uint4*>(sm + O_Q + row * 256 + ch * 16) = vq;
            *reinterpret_cast<uint4*>(sm + O_K + row * 256 + ch * 16) = vk;
            *reinterpret_cast<uint4*>(sm + O_V + row * 256 + ch * 16) = vv;
        }
        for (int it = tid; it < 64 * 32; it += kPrepThreads) {
            const int row = it >> 5, ch = it & 31;
            float4 vg = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < ci.len) {
                const int64_t t = tb + row;
                vg = __ldg(reinterpret_cast<const float4*>(p.g + ci.b * p.gs[0] + t * p.gs[1] + h * p.gs[2]) + ch);
            }
            *reinterpret_cast<float4*>(sm + O_G + row * 512 + ch * 16) = vg;
        }
        if (tid < 64) {
            float b = 0.f;
            if (tid < ci.len) {
                b = __ldg(p.beta + ci.b * p.bs[0] + (tb + tid) * p.bs[1] + h * p.bs[2]);
                if (p.beta_is_logit) b = 1.0f / (1.0f + __expf(-b));
            }
            reinterpret_cast<float*>(sm + O_BETA)[tid] = b;
        }
    }
    __syncthreads();

    // ---- E1: thread (G, pair) owns tokens 16G..16G+15 of channels 2*pair, 2*pair+1.
    const int G = tid >> 6, pr = tid & 63, c0 = 2 * pr;
    float L0[16], L1[16], C0[16], C1[16];  // local cumsum (raw and floored gates)
    {
        float s0 = 0.f, s1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            const float2 gv = *reinterpret_cast<const float2*>(sm + O_G + (16 * G + l) * 512 + c0 * 4);
            s0 += gv.x; s1 += gv.y;
            u0 += fmaxf(gv.x, kGateClamp); u1 += fmaxf(gv.y, kGateClamp);
            L0[l] = s0; L1[l] = s1; C0[l] = u0; C1[l] = u1;
        }
        float* tot = reinterpret_cast<float*>(sm + O_TOT);
        tot[G * 128 + c0] = s0;
        tot[G * 128 + c0 + 1] = s1;
    }
    __syncthreads();  // block totals visible; the g rows are dead from here on

    // ---- E2: gate factors and the MMA operands.
    //   a  = exp(Gam_i - Gam_{block start - 1})  (<= 1)
    //   z  = exp(Gam_{block end} - Gam_i)         (<= 1)
    //   rm = exp(Gf_i - Gf_m), ym = exp(Gf_m - Gf_i) with Gf the floored-gate
    //        cumsum and m the block's 8th token  (<= e^80 each)
    const int blk = c0 >> 6, cc = c0 & 63;
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
        // Between-block decay for the Yoff groups of later row blocks I > G.
        float Dm0[4], Dm1[4];
        {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int I = 0; I < 4; ++I) {
                Dm0[I] = __expf(s0); Dm1[I] = __expf(s1);
                if (I > G) { s0 += d0[I]; s1 += d1[I]; }
            }
        }
        if (G == 0) {
            const float gam0 = d0[0] + d0[1] + d0[2] + d0[3], gam1 = d1[0] + d1[1] + d1[2] + d1[3];
            *reinterpret_cast<float2*>(p.ws_eg + (size_t)rec * kHeadDim + c0) =
                make_float2(__expf(gam0), __expf(gam1));
        }

        uint32_t kvk0[8], kvk1[8], kvv0[8], kvv1[8], kh0[8], kh1[8];
        float pk0 = 0.f, pk1 = 0.f, pv0 = 0.f, pv1 = 0.f, ph0 = 0.f, ph1 = 0.f;
        const float qscale = p.scale;
#pragma unroll
        for (int l = 0; l < 16; ++l) {
            const int i = 16 * G + l;
            const float a0 = __expf(L0[l]), a1 = __expf(L1[l]);
            const float z0 = __expf(L0[15] - L0[l]), z1 = __expf(L1[15] - L1[l]);
            const float rm0 = __expf(C0[l] - C0[7]), rm1 = __expf(C1[l] - C1[7]);
            const float ym0 = __expf(C0[7] - C0[l]), ym1 = __expf(C1[7] - C1[l]);
            const float2 kk = ld_bf16x2(sm + O_K + i * 256 + c0 * 2);
            float2 qq = ld_bf16x2(sm + O_Q + i * 256 + c0 * 2);
            qq.x *= qscale; qq.y *= qscale;
            const float2 vv = ld_bf16x2(sm + O_V + i * 256 + c0 * 2);
            const uint32_t bo = blk * 16384u;
            // R = [K a ; Q a]  and  Rmid = [K rm ; Q rm]   (A operands, 128 rows)
            st_u32(sm + O_G + bo + sw128_off(i, cc), pack_bf16x2(kk.x * a0, kk.y * a1));
            st_u32(sm + O_G + bo + sw128_off(64 + i, cc), pack_bf16x2(qq.x * a0, qq.y * a1));
            st_u32(sm + O_RM + bo + sw128_off(i, cc), pack_bf16x2(kk.x * rm0, kk.y * rm1));
            st_u32(sm + O_RM + bo + sw128_off(64 + i, cc), pack_bf16x2(qq.x * rm0, qq.y * rm1));
            // Yoff: column block G seen from each later row block I (B operand, 96 rows)
#pragma unroll
            for (int I = 1; I < 4; ++I) {
                if (I > G)
                    st_u32(sm + O_YO + blk * 12288u + sw128_off(yoff_row(I, G, l), cc),
                           pack_bf16x2(kk.x * z0 * Dm0[I], kk.y * z1 * Dm1[I]));
            }
            // Ymid (B operand, 64 rows)
            st_u32(sm + O_YM + blk * 8192u + sw128_off(i, cc), pack_bf16x2(kk.x * ym0, kk.y * ym1));
            // Q e^Gam, kept for Q' in the last epilogue
            st_u32(sm + O_QT + i * kQtPitch + c0 * 2, pack_bf16x2(qq.x * a0 * B0, qq.y * a1 * B1));
            // [K e^Gam | V]^T columns and Kt = (K e^{gam - Gam})^T, packed by token pairs
            const float ke0 = kk.x * a0 * B0, ke1 = kk.y * a1 * B1;
            const float h0v = kk.x * z0 * E0, h1v = kk.y * z1 * E1;
            if ((l & 1) == 0) {
                pk0 = ke0; pk1 = ke1; pv0 = vv.x; pv1 = vv.y; ph0 = h0v; ph1 = h1v;
            } else {
                kvk0[l >> 1] = pack_bf16x2(pk0, ke0);
                kvk1[l >> 1] = pack_bf16x2(pk1, ke1);
                kvv0[l >> 1] = pack_bf16x2(pv0, vv.x);
                kvv1[l >> 1] = pack_bf16x2(pv1, vv.y);
                kh0[l >> 1] = pack_bf16x2(ph0, h0v);
                kh1[l >> 1] = pack_bf16x2(ph1, h1v);
            }
        }
        const int t0c = 16 * G;
        uint4* kv_rows[4] = {
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(c0, t0c)),
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(c0 + 1, t0c)),
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(128 + c0, t0c)),
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(128 + c0 + 1, t0c))};
        uint4* kv_rows_hi[4] = {
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(c0, t0c + 8)),
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(c0 + 1, t0c + 8)),
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(128 + c0, t0c + 8)),
            reinterpret_cast<uint4*>(sm + O_KV + sw128_off(128 + c0 + 1, t0c + 8))};
        *kv_rows[0] = make_uint4(kvk0[0], kvk0[1], kvk0[2], kvk0[3]);
        *kv_rows_hi[0] = make_uint4(kvk0[4], kvk0[5], kvk0[6], kvk0[7]);
        *kv_rows[1] = make_uint4(kvk1[0], kvk1[1], kvk1[2], kvk1[3]);
        *kv_rows_hi[1] = make_uint4(kvk1[4], kvk1[5], kvk1[6], kvk1[7]);
        *kv_rows[2] = make_uint4(kvv0[0], kvv0[1], kvv0[2], kvv0[3]);
        *kv_rows_hi[2] = make_uint4(kvv0[4], kvv0[5], kvv0[6], kvv0[7]);
        *kv_rows[3] = make_uint4(kvv1[0], kvv1[1], kvv1[2], kvv1[3]);
        *kv_rows_hi[3] = make_uint4(kvv1[4], kvv1[5], kvv1[6], kvv1[7]);
        uint4* kt0 = reinterpret_cast<uint4*>(p.ws_kt + (size_t)rec * (kHeadDim * kChunk) + c0 * kChunk + t0c);
        uint4* kt1 = reinterpret_cast<uint4*>(p.ws_kt + (size_t)rec * (kHeadDim * kChunk) + (c0 + 1) * kChunk + t0c);
        kt0[0] = make_uint4(kh0[0], kh0[1], kh0[2], kh0[3]);
        kt0[1] = make_uint4(kh0[4], kh0[5], kh0[6], kh0[7]);
        kt1[0] = make_uint4(kh1[0], kh1[1], kh1[2], kh1[3]);
        kt1[1] = make_uint4(kh1[4], kh1[5], kh1[6], kh1[7]);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;

    bool ok = true;
    // ---- MMA A: D_off = R Yoff^T (N = 96), D_mid = Rmid Ymid^T (N = 64)
    if (tid == 0) {
        umma_tile(tb + TM_OFF, smem_u32(sm + O_G), 16384, smem_u32(sm + O_YO), 12288, 128,
                  idesc_bf16_f32(128, 96), false);
        umma_tile(tb + TM_MID, smem_u32(sm + O_RM), 16384, smem_u32(sm + O_YM), 8192, 128,
                  idesc_bf16_f32(128, 64), false);
        umma_commit(&bar_mma[0]);
    }
    ok = __syncthreads_and(mbar_wait(&bar_mma[0], 0, nullptr));
    tc_fence_after();
    const int qd = warp & 3, half = warp >> 2;
    float* sA = reinterpret_cast<float*>(sm + O_AKK);
    float* sT = reinterpret_cast<float*>(sm + O_T);
    float* sX = reinterpret_cast<float*>(sm + O_X);
    const float* sBeta = reinterpret_cast<const float*>(sm + O_BETA);
    if (ok) {
        // ---- Epilogue A: rows 0..63 of TMEM are k rows (-> A, beta-scaled, j < i),
        // rows 64..127 are q rows (-> Aqk, j <= i, bf16 operand for MMA B).
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
            if (J < I0) tmem_ld16(tmem_addr(tb, 32 * qd, TM_OFF + yoff_row(I0, J, 0)), t0);
            if (J < I1) tmem_ld16(tmem_addr(tb, 32 * qd, TM_OFF + yoff_row(I1, J, 0)), t1);
            if (J <= I1) tmem_ld16(tmem_addr(tb, 32 * qd, TM_MID + 16 * J), tm);
#pragma unroll
            for (int jj = 0; jj < 16; jj += 2) {
                float v2[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int j = 16 * J + jj + e;
                    float val = 0.f;
                    if (J < I) val = lo ? t0[jj + e] : t1[jj + e];
                    else if (J == I) val = tm[jj + e];
                    if (!isq) val = (j < i) ? bi * val : 0.f;
                    else val = (j <= i) ? val : 0.f;
                    v2[e] = val;
                }
                const int j = 16 * J + jj;
                if (!isq) {
                    sA[i * kPA + j] = v2[0];
                    sA[i * kPA + j + 1] = v2[1];
                    st_u32(sm + O_AQK + sw128_off(64 + i, j), 0u);  // zero half of the Aqk operand
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
    // at 16 -> 32 and 32 -> 64.
    if (ok) {
        for (int e = tid; e < 64 * kPA; e += kPrepThreads) sT[e] = 0.f;
        __syncthreads();
        if (tid < 64) {
            const int I = tid >> 4, l = tid & 15, s = 16 * I;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == l) ? 1.f : 0.f;
#pragma unroll
            for (int r = 1; r < 16; ++r) {
                float acc = x[r];
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(-sA[(s + r) * kPA + s + m], x[m], acc);
                x[r] = acc;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(s + r) * kPA + s + l] = x[r];
        }
        __syncthreads();
        for (int e = tid; e < 512; e += kPrepThreads) {  // X = A_10 T_00 (two 32-blocks)
            const int pb = 32 * (e >> 8), r = (e >> 4) & 15, c = e & 15;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                acc = fmaf(sA[(pb + 16 + r) * kPA + pb + m], sT[(pb + m) * kPA + pb + c], acc);
            sX[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < 512; e += kPrepThreads) {  // T_10 = -T_11 X
            const int pb = 32 * (e >> 8), r = (e >> 4) & 15, c = e & 15;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 16; ++m)
                acc = fmaf(sT[(pb + 16 + r) * kPA + pb + 16 + m], sX[(e & 256) + m * 16 + c], acc);
            sT[(pb + 16 + r) * kPA + pb + c] = -acc;
        }
        __syncthreads();
        for (int e = tid; e < 1024; e += kPrepThreads) {  // X = A[32:,:32] T[:32,:32]
            const int r = e >> 5, c = e & 31;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 32; ++m) acc = fmaf(sA[(32 + r) * kPA + m], sT[m * kPA + c], acc);
            sX[r * 33 + c] = acc;
        }
        __syncthreads();
        for (int e = tid; e < 1024; e += kPrepThreads) {  // T[32:,:32] = -T[32:,32:] X
            const int r = e >> 5, c = e & 31;
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < 32; ++m) acc = fmaf(sT[(32 + r) * kPA + 32 + m], sX[m * 33 + c], acc);
            sT[(32 + r) * kPA + c] = -acc;
        }
        __syncthreads();
        // T' = T Diag(beta): rows 0..63 of the TT operand (K-major over j) and
        // T'^T as the B operand of MMA B (row n, K index j).
        for (int e = tid; e < 64 * 32; e += kPrepThreads) {
            const int r = e >> 5, jp = 2 * (e & 31);
            st_u32(sm + O_TT + sw128_off(r, jp),
                   pack_bf16x2(sT[r * kPA + jp] * sBeta[jp], sT[r * kPA + jp + 1] * sBeta[jp + 1]));
            st_u32(sm + O_TTR + sw128_off(r, jp),
                   pack_bf16x2(sT[jp * kPA + r] * sBeta[r], sT[(jp + 1) * kPA + r] * sBeta[r]));
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- MMA B: D_b = [Aqk ; 0] T'  -> rows 64..127 of the TT operand
    if (ok && tid == 0) {
        tc_fence_after();
        umma_tile(tb + TM_B, smem_u32(sm + O_AQK), 0, smem_u32(sm + O_TTR), 0, 64,
                  idesc_bf16_f32(128, 64), false);
        umma_commit(&bar_mma[1]);
    }
    if (ok) ok = __syncthreads_and(mbar_wait(&bar_mma[1], 0, nullptr));
    tc_fence_after();
    if (ok && qd < 2) {
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
    if (ok && tid == 0) {
        tc_fence_after();
        umma_tile(tb + TM_C, smem_u32(sm + O_TT), 0, smem_u32(sm + O_KV), 0, 64,
                  idesc_bf16_f32(128, 256), false);
        umma_commit(&bar_mma[2]);
    }
    if (ok) ok = __syncthreads_and(mbar_wait(&bar_mma[2], 0, nullptr));
    tc_fence_after();
    if (ok) {
        // ---- Epilogue C: W, U (rows 0..63) and Q' = Q e^Gam - Aqk W, O_loc = Aqk U
        // (rows 64..127) to the workspace records.
        const int i = 32 * (qd & 1) + lane;
        const bool top = qd < 2;
        const size_t rb = (size_t)rec * (kChunk * kHeadDim) + (size_t)i * kHeadDim;
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
                uint4* dst = reinterpret_cast<uint4*>((top ? p.ws_w : p.ws_qp) + rb + col);
                dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
                float4* dst = reinterpret_cast<float4*>((top ? p.ws_u : p.ws_ol) + rb + col);
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    dst[x] = make_float4(v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
            }
        }
    }
    if (!ok && tid == 0) atomicExch(p.status, 4);
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

cudaError_t launch_prep(const PrefillParams& p, cudaStream_t s) {
    const long long recs = (long long)p.max_chunks * p.H;
    if (recs == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kPrepSmem);
    if (e != cudaSuccess) return e;
    prep_kernel<<<(unsigned)recs, kPrepThreads, kPrepSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
