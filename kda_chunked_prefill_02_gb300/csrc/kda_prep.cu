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
//   W  = T' (K e^Gam),  U = T' V (stored transposed),  Kt = (K e^{gam - Gam})^T,
//   eg = e^gam
// so that, for the chunk's entry state S, the serial pass only needs
//   V_new = U - W S,  O = (Q e^Gam) S + Aqk V_new,  S <- Diag(eg) S + Kt V_new.
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
// Organisation: a persistent CTA (16 warps) per SM loops over (chunk, head)
// records.  The q, k, v and g tiles of a record arrive by TMA; the next
// record's tiles are requested during the UT solve, so that they land during
// the solve and MMA C.  The record's images leave by bulk copies issued by
// warps that have nothing else to do at that point.  Copies in either
// direction are kept away from the shared-memory-heavy phases (operand build,
// epilogues), which they measurably slow down.
#include <string.h>

#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kPrepThreads = 512;

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
constexpr uint32_t O_QT = 188416;     // Q e^Gam image: 2 column blocks x 64 rows x 128 B (the record's rows 0-63)
// Staging of the record's Kt image (16 KB fp16, the record's bytes) and e^gam
// (512 B), apart from the input tiles, so that the next record's tiles may be
// requested while these images are still being copied out.
constexpr uint32_t O_SKT = 204800;
constexpr uint32_t O_TOT = 221184;    // fp32 [2][8][128] decay products (exact, floored) of 8-token groups
constexpr uint32_t O_BETA = 229376;   // fp32 [64] beta
constexpr uint32_t O_SEG = 229632;
constexpr uint32_t kPrepSmem = 230144 + 1024;
static_assert(kPrepSmem <= 232448, "prep shared memory above the per-block limit");
// The regions live at the same time do not overlap: the input tiles, the MMA A
// operands, the [K e^Gam | V] operand, the Q e^Gam and Kt images, the decay
// products, beta and e^gam.
static_assert(O_IG + 32768 == kInBytes && kInBytes <= O_R, "input tiles");
static_assert(O_R + 2 * 16384 <= O_Y && O_Y + 2 * kYBlock <= O_KV, "MMA A operands");
static_assert(O_KV + 8 * kKvSbo <= O_QT && O_QT + 2 * 8192 <= O_SKT, "KV operand and Q e^Gam image");
static_assert(O_SKT + 16384 <= O_TOT && O_TOT + 2 * 8 * 128 * 4 <= O_BETA, "Kt image and decay products");
static_assert(O_BETA + 64 * 4 <= O_SEG && O_SEG + 128 * 4 + 1024 <= kPrepSmem, "beta and e^gam");
// Scratch of the solve and MMA C, over R and Y once MMA A has completed.
// The fp32 matrices hold tf32-rounded values (operands of the warp MMAs); the
// row pitch 68 (4 mod 32) makes the MMA row-fragment loads and the epilogue's
// float4 row stores conflict-free.
constexpr int kPA = 68;               // fp32 row pitch of A and T
constexpr int kPX = 40;               // fp32 row pitch of the products X (8 mod 32)
constexpr uint32_t O_A = 81920;       // fp32 [64][68] beta-scaled A
constexpr uint32_t O_T = 99328;       // fp32 [64][68] T
constexpr uint32_t O_X = 116736;      // fp32 [32][40] products
constexpr uint32_t O_AQK = 122880;    // Aqk image, fp16: 64 rows x 128 B (the record's, K-major over tokens)
constexpr uint32_t O_TT = 131072;     // A operand [T' ; T']: 128 rows x 128 B
// Staging of the record images written by the last epilogue (over the solve's
// scratch, which MMA C no longer needs).
constexpr uint32_t O_SW = 81920;      // W image: 2 column blocks x 64 rows x 128 B (the record's rows 64-127)
constexpr uint32_t O_SU = 98304;      // U^T image: 128 value rows x 128 B (64 tokens), 16 KB
// The solve's scratch and the last epilogue's staging stay inside R and Y.
static_assert(O_A + 64 * kPA * 4 <= O_T && O_T + 64 * kPA * 4 <= O_X && O_X + 32 * kPX * 4 <= O_AQK,
              "solve scratch");
static_assert(O_AQK + 8192 <= O_TT && O_TT + 16384 <= O_KV, "Aqk image and T' operand");
static_assert(O_SU + 16384 <= O_AQK, "W / U^T staging");

// TMEM columns.
constexpr uint32_t TM_A = 0, TM_DIAG = 96, TM_C = 0, TM_COLS = 256;

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ void st_u32(uint8_t* p, uint32_t v) {
    *reinterpret_cast<uint32_t*>(p) = v;
}
// Stores T' = T Diag(beta) entries (i, j) and (i, j + 1) of a computed T block
// into the TT operand, rows i and 64 + i (MMA C then writes W and U to both
// halves of TMEM's lanes, so that every epilogue warp has work).
__device__ __forceinline__ void store_tprime_pair(uint8_t* sm, int i, int j, float t0, float t1,
                                                  const float* sBeta) {
    const uint32_t ab = pack_bf16x2(t0 * sBeta[j], t1 * sBeta[j + 1]);
    st_u32(sm + O_TT + sw128_off(i, j), ab);
    st_u32(sm + O_TT + sw128_off(64 + i, j), ab);
}
// Row of the Yoff operand holding column block J as seen from row block I > J:
// block I's group holds its 16*I earlier columns.
__device__ __forceinline__ uint32_t yoff_row(int I, int J, int l) {
    return 8 * I * (I - 1) + 16 * J + l;
}

// Warp-level m16n8k8 tf32 MMA with fp32 accumulation (used for the small block
// products of the UT solve; fragment layouts of the PTX m16n8k8 tf32 shape).
__device__ __forceinline__ float tf32_round(float x) { return to_tf32(x); }
// d (16 x 8 tile) = P (16 x 8*ke, row pitch pp) * Q (8*ke x 8, row pitch pq) over
// the k-steps kb .. ke-1 (8 each), fp32 matrices of tf32-rounded values in shared
// memory.  Thread (g = lane/4, t = lane%4) gets d0 (g, 2t), d1 (g, 2t+1),
// d2 (g+8, 2t), d3 (g+8, 2t+1).
__device__ __forceinline__ void warp_mma_16x8(const float* P, int pp, const float* Q, int pq,
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
// Stores a 16 x 8 accumulator tile (fragment layout above) at X (row pitch pq),
// rounded to tf32.
__device__ __forceinline__ void store_tile_tf32(float* X, int pq, const float (&d)[4], int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2*>(X + g * pq + 2 * t) = make_float2(tf32_round(d[0]), tf32_round(d[1]));
    *reinterpret_cast<float2*>(X + (g + 8) * pq + 2 * t) = make_float2(tf32_round(d[2]), tf32_round(d[3]));
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

template <bool kStall>
__global__ void __launch_bounds__(kPrepThreads, 1)
    prep_kernel(const PrefillParams p, const __grid_constant__ PrepMaps maps) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t bar_in, bar_mma[2], bar_fin, bar_never;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int s_rec[3];   // counter mode: first record, then the next record by parity

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nrec = p.max_chunks * p.H;
    if (blockIdx.x >= nrec) return;
    if (tid == 0) {
        mbar_init(&bar_in, 1);
        for (int i = 0; i < 2; ++i) mbar_init(&bar_mma[i], 1);
        mbar_init(&bar_fin, 1);
        mbar_init(&bar_never, 1);   // nothing arrives on it (the timeout probe's wait)
        fence_mbar_init();
        tma_prefetch_desc(&maps.q); tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v); tma_prefetch_desc(&maps.g);
        if (p.rec_counter) {
            // records are taken from the counter, the next one a record ahead so
            // that its inputs can be requested early
            s_rec[2] = atomicAdd(p.rec_counter, 1);
            s_rec[0] = atomicAdd(p.rec_counter, 1);
        }
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;

    // Thread roles in the gate phases: key channels c0, c0 + 1 and the 8-token
    // group h8 (half hf of the 16-token block G).  A warp covers 64 channels
    // (one 128-byte operand row) of one token row per store.
    const int c0 = 2 * (tid & 63), h8 = tid >> 6, G = h8 >> 1, hf = h8 & 1;
    const int blk = c0 >> 6, cc = c0 & 63;
    // Roles in the TMEM epilogues: lane quarter qd, column quarter cq.
    const int qd = warp & 3, cq = warp >> 2;
    const float kPFloor = __expf(kGateFloor);

    const bool counted = p.rec_counter != nullptr;
    int rec = counted ? s_rec[2] : (int)blockIdx.x;
    ChunkInfo ci = rec < nrec ? chunk_info(p, rec / p.H) : ChunkInfo{0, 0, 0, 0, 0};
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
        const int len = ci.len;
        const int rec_next = counted ? s_rec[it & 1] : rec + (int)gridDim.x;
        const ChunkInfo cn = rec_next < nrec ? chunk_info(p, rec_next / p.H) : ChunkInfo{0, 0, 0, 0, 0};
        // This CTA's last record: a grid launched programmatically after this one
        // may start once every CTA has reached this point.
        if (rec_next >= nrec) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        stall_point<kStall>(p.stall_seed, 1, it);
        // Every thread waits on the input mbarrier itself (no CTA barrier here);
        // a wait that ran out is acted on, by all threads alike, at the CTA
        // barrier that ends the gate phase.
        ok = mbar_wait(&bar_in, it & 1, nullptr, p.wait_ns);
        if (ok) pend_parity = -1;
        // the record after the next (read two iterations on, past many barriers;
        // the slot was last read at the top of the previous iteration)
        if (counted && tid == 0 && rec_next < nrec) s_rec[(it + 1) & 1] = atomicAdd(p.rec_counter, 1);
        if (tid < 64) {
            float bval = bcur;
            if (tid < len && p.beta_is_logit) bval = 1.0f / (1.0f + __expf(-bval));
            reinterpret_cast<float*>(sm + O_BETA)[tid] = tid < len ? bval : 0.f;
        }

        // Tokens past the chunk length (the tail of a sequence) read as zeros:
        // k = q = v = 0 and g = 0 (no decay).
        if (len < kChunk) {
            for (int e = tid; e < (kChunk - len) * 80; e += kPrepThreads) {
                const int row = len + e / 80, u = e % 80;
                uint8_t* dst = u < 48 ? sm + (u >> 4) * 16384 + row * 256 + (u & 15) * 16
                                      : sm + O_IG + row * 512 + (u - 48) * 16;
                *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
        }

        // ---- E1: p = exp(g) and the 8-token group's decay products, exact and
        // with the floored gate.  Every decay factor below is a product of these,
        // so the gate phase takes one exponential per element and no more.
        float p0[8], p1[8];
        {
            float e0 = 1.f, e1 = 1.f, f0 = 1.f, f1 = 1.f;
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                const float2 gv = *reinterpret_cast<const float2*>(sm + O_IG + (8 * h8 + l) * 512 + c0 * 4);
                p0[l] = __expf(gv.x); p1[l] = __expf(gv.y);
                e0 *= p0[l]; e1 *= p1[l];
                f0 *= fmaxf(p0[l], kPFloor); f1 *= fmaxf(p1[l], kPFloor);
            }
            float* tot = reinterpret_cast<float*>(sm + O_TOT);
            *reinterpret_cast<float2*>(tot + h8 * 128 + c0) = make_float2(e0, e1);
            *reinterpret_cast<float2*>(tot + 1024 + h8 * 128 + c0) = make_float2(f0, f1);
        }
        stall_point<kStall>(p.stall_seed, 2, it);
        // The previous record's images have left their staging areas (each bulk
        // store is waited for by the lane that issued it).
        if (lane == 0) bulk_wait_read();
        ok = __syncthreads_and(ok);
        if (!ok) break;

        // ---- E2: the MMA operands and the records that need no MMA.  R and Y (MMA
        // A's operands) are written first; the Q e^Gam, [K e^Gam | V] and Kt
        // images, which MMA A does not read, are kept in registers and written
        // while MMA A runs (warp 0, whose lane 0 issues MMA A, writes its share
        // before).
        uint32_t qt_w[8], kv_w[8], v_w[8], kt_w0[4], kt_w1[4];
        {
            const float* tot = reinterpret_cast<const float*>(sm + O_TOT);
            float b0[4], b1[4];  // exact decay of each 16-token block
#pragma unroll
            for (int J = 0; J < 4; ++J) {
                const float2 u = *reinterpret_cast<const float2*>(tot + (2 * J) * 128 + c0);
                const float2 w = *reinterpret_cast<const float2*>(tot + (2 * J + 1) * 128 + c0);
                b0[J] = u.x * w.x; b1[J] = u.y * w.y;
            }
            // exact (eA, eB) and floored (fA, fB) decay of block G's two halves
            const float2 eA = *reinterpret_cast<const float2*>(tot + (2 * G) * 128 + c0);
            const float2 eB = *reinterpret_cast<const float2*>(tot + (2 * G + 1) * 128 + c0);
            const float2 fA = *reinterpret_cast<const float2*>(tot + 1024 + (2 * G) * 128 + c0);
            const float2 fB = *reinterpret_cast<const float2*>(tot + 1024 + (2 * G + 1) * 128 + c0);
            // Bg: chunk start -> block start; E: block end -> chunk end;
            // Dm[I]: the blocks strictly between G and I
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
                *reinterpret_cast<float2*>(sm + O_SEG + c0 * 4) =
                    make_float2(b0[0] * b0[1] * b0[2] * b0[3], b1[0] * b1[1] * b1[2] * b1[3]);
            const float qscale = p.scale;
            const uint32_t bo = blk * 16384u, yb = blk * kYBlock;
            // Byte offset of token row 8 h8 + l (channels cc, cc + 1) in a SW128
            // K-major tile: the row's 16-byte chunk index is XORed with l.
            const uint32_t trow0 = h8 * 1024u + (((uint32_t)cc >> 3) << 4 | ((uint32_t)cc & 7u) << 1);
            auto trow = [&](int l) -> uint32_t { return trow0 ^ (uint32_t)(l * 144); };
            uint8_t* const sR = sm + O_R + bo;
            uint8_t* const sY = sm + O_Y + yb;
            // Forward over the group: the running products a (exact gates, from the
            // chunk start) and ac (floored gates, from the block start).  The second
            // half of a block starts from the first half's product.
            {
                float a0 = hf ? Bg0 * eA.x : Bg0, a1 = hf ? Bg1 * eA.y : Bg1;
                float ac0 = hf ? fA.x : 1.f, ac1 = hf ? fA.y : 1.f;
                uint32_t kw[8], qw[8], vw[8];
                const uint8_t* in = sm + (8 * h8) * 256 + c0 * 2;
#pragma unroll
                for (int l = 0; l < 8; ++l) {
                    kw[l] = *reinterpret_cast<const uint32_t*>(in + O_IK + l * 256);
                    qw[l] = *reinterpret_cast<const uint32_t*>(in + O_IQ + l * 256);
                    vw[l] = *reinterpret_cast<const uint32_t*>(in + O_IV + l * 256);
                }
#pragma unroll
                for (int l = 0; l < 8; ++l) {
                    a0 *= p0[l]; a1 *= p1[l];
                    ac0 *= fmaxf(p0[l], kPFloor); ac1 *= fmaxf(p1[l], kPFloor);
                    const float2 kk = bf16x2_to_float2(kw[l]);
                    float2 qq = bf16x2_to_float2(qw[l]);
                    qq.x *= qscale; qq.y *= qscale;
                    // R = [K ac ; Q ac]
                    st_u32(sR + trow(l), pack_bf16x2(kk.x * ac0, kk.y * ac1));
                    st_u32(sR + 8192 + trow(l), pack_bf16x2(qq.x * ac0, qq.y * ac1));
                    // the record's Q e^Gam rows and [K e^Gam | V], written later
                    qt_w[l] = pack_bf16x2(qq.x * a0, qq.y * a1);
                    kv_w[l] = pack_bf16x2(kk.x * a0, kk.y * a1);
                    v_w[l] = vw[l];
                }
            }
            stall_point<kStall>(p.stall_seed, 3, it);
            // Backward over the group: the suffix products z (exact gates, to the block
            // end) and zc (floored gates); the first half of a block continues through
            // the second half.
            {
                float z0 = hf ? 1.f : eB.x, z1 = hf ? 1.f : eB.y;
                // zc / (floored-gate block product) = 1 / ac: at most e^86.4, since
                // each floored factor is at least e^-5.4
                float zc0 = __frcp_rn(hf ? fA.x * fB.x : fA.x), zc1 = __frcp_rn(hf ? fA.y * fB.y : fA.y);
                float eh0 = 0.f, eh1 = 0.f;
                uint32_t kh0[4], kh1[4], kw[8];
#pragma unroll
                for (int l = 0; l < 8; ++l)
                    kw[l] = *reinterpret_cast<const uint32_t*>(sm + O_IK + (8 * h8 + l) * 256 + c0 * 2);
#pragma unroll
                for (int l = 7; l >= 0; --l) {
                    const float2 kk = bf16x2_to_float2(kw[l]);
                    // Yd (diagonal blocks): K / ac
                    st_u32(sY + 96 * 128 + trow(l), pack_bf16x2(kk.x * zc0, kk.y * zc1));
                    // Yoff: column block G seen from each later row block I (Y row
                    // yoff_row(I, G, 8 hf + l) = 8 I (I - 1) + 8 h8 + l)
                    const float kz0 = kk.x * z0, kz1 = kk.y * z1;
#pragma unroll
                    for (int I = 1; I < 4; ++I)
                        if (I > G)
                            st_u32(sY + 8 * I * (I - 1) * 128 + trow(l), pack_bf16x2(kz0 * Dm0[I], kz1 * Dm1[I]));
                    // Kt = (K e^{gam - Gam})^T in fp16, packed by token pairs
                    const float hh0 = kz0 * E0, hh1 = kz1 * E1;
                    if (l & 1) {
                        eh0 = hh0; eh1 = hh1;
                    } else {
                        kh0[l >> 1] = pack_f16x2(hh0, eh0);
                        kh1[l >> 1] = pack_f16x2(hh1, eh1);
                    }
                    z0 *= p0[l]; z1 *= p1[l];
                    zc0 *= fmaxf(p0[l], kPFloor); zc1 *= fmaxf(p1[l], kPFloor);
                }
#pragma unroll
                for (int x = 0; x < 4; ++x) { kt_w0[x] = kh0[x]; kt_w1[x] = kh1[x]; }
            }
        }
        // The images MMA A does not read: Q e^Gam, [K e^Gam | V] (MN-major: token
        // row i, channels contiguous) and the Kt rows c0, c0 + 1 (tokens 8 h8 ..
        // 8 h8 + 7 are 16-byte chunk h8).
        auto write_late_images = [&]() {
            // token row 8 h8 + l as in E2; the [K e^Gam | V] operand's 8-token
            // groups are kKvSbo apart and its 64-channel atoms 1 KB apart
            const uint32_t t0 = h8 * 1024u + (((uint32_t)cc >> 3) << 4 | ((uint32_t)cc & 7u) << 1);
            uint8_t* const qtb = sm + O_QT + blk * 8192u;
            uint8_t* const kvb = sm + O_KV + h8 * (kKvSbo - 1024u) + blk * 1024u;
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                const uint32_t o = t0 ^ (uint32_t)(l * 144);
                st_u32(qtb + o, qt_w[l]);
                st_u32(kvb + o, kv_w[l]);
                st_u32(kvb + 2048 + o, v_w[l]);
            }
            uint8_t* kt = sm + O_SKT;
            *reinterpret_cast<uint4*>(kt + sw128_off(c0, 8 * h8)) = make_uint4(kt_w0[0], kt_w0[1], kt_w0[2], kt_w0[3]);
            *reinterpret_cast<uint4*>(kt + sw128_off(c0 + 1, 8 * h8)) = make_uint4(kt_w1[0], kt_w1[1], kt_w1[2], kt_w1[3]);
        };
        if (warp == 0) write_late_images();
        stall_point<kStall>(p.stall_seed, 4, it);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            // ---- MMA A: D = R [Yoff ; Yd]^T, N = 160 (off-diagonal and diagonal blocks)
            umma_tile(tb + TM_A, smem_u32(sm + O_R), 16384, smem_u32(sm + O_Y), kYBlock, 128,
                      idesc_bf16_f32(128, 160), false);
            umma_commit(&bar_mma[0]);
        }
        // (no CTA barrier here: nothing reads the late images before the barrier
        // that ends epilogue A)
        if (warp != 0) write_late_images();
        if (cn.len > 0) bcur = load_beta(cn, rec_next % p.H);
        ok = __syncthreads_and(
            tid == 0 ? mbar_wait((p.timeout_probe && it == 0) ? &bar_never : &bar_mma[0], it & 1, nullptr, p.wait_ns)
                     : true);
        tc_fence_after();
        if (!ok) break;

        stall_point<kStall>(p.stall_seed, 5, it);
        float* sA = reinterpret_cast<float*>(sm + O_A);
        float* sT = reinterpret_cast<float*>(sm + O_T);
        float* sX = reinterpret_cast<float*>(sm + O_X);
        const float* sBeta = reinterpret_cast<const float*>(sm + O_BETA);
        {
            // ---- Epilogue A: TMEM rows 0..63 are k rows (-> A, beta-scaled, j < i),
            // rows 64..127 are q rows (-> Aqk, j <= i, the record's fp16 image).
            const bool isq = qd >= 2;
            const int i = 32 * (qd & 1) + lane, I = i >> 4, I0 = 2 * (qd & 1), I1 = I0 + 1;
            const bool lo = lane < 16;
            const float bi = sBeta[i];
            const int J = cq;
            // The three tiles this warp may need, with one wait (a tile the warp's
            // rows do not use is read and ignored; every address lies inside
            // the allocation).
            float t0[16], t1[16], tm[16];
            {
                uint32_t r0[16], r1[16], rm[16];
                tmem_ld16_issue(tmem_addr(tb, 32 * qd, TM_A + yoff_row(I0, J, 0)), r0);
                tmem_ld16_issue(tmem_addr(tb, 32 * qd, TM_A + yoff_row(I1, J, 0)), r1);
                tmem_ld16_issue(tmem_addr(tb, 32 * qd, TM_DIAG + 16 * J), rm);
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
                v[x] = isq ? ((j <= i) ? val : 0.f) : ((j < i) ? tf32_round(bi * val) : 0.f);
            }
            if (!isq) {
                float4* dst = reinterpret_cast<float4*>(sA + i * kPA + 16 * J);
#pragma unroll
                for (int u = 0; u < 4; ++u) dst[u] = make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
            } else {
                uint32_t w[8];
#pragma unroll
                for (int x = 0; x < 8; ++x) w[x] = pack_f16x2(v[2 * x], v[2 * x + 1]);
                *reinterpret_cast<uint4*>(sm + O_AQK + sw128_off(i, 16 * J)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(sm + O_AQK + sw128_off(i, 16 * J + 8)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
        }
        stall_point<kStall>(p.stall_seed, 6, it);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- UT transform: T = (I + A)^-1 for the unit lower-triangular 64 x 64
        // system, blocked: four 16 x 16 diagonal inverses by forward substitution,
        // then [[Ta,0],[Aba,Tb]]^-1 = [[Ta^-1,0],[-Tb^-1 Aba Ta^-1, Tb^-1]] at
        // 16 -> 32 and 32 -> 64.  T' = T Diag(beta) goes to the TT / T'^T operands
        // as each block is produced; the products skip the k-steps that are zero
        // because T is lower triangular, so T's upper blocks are never read.
        {
            // Diagonal blocks: warp (block I, columns l, l + 1 for lanes >= 16 two
            // further), lane row m.  The substitution runs down the rows: once row r
            // is final it is broadcast and every later row subtracts A[m][r] x_r.
            const int I = warp >> 2, m = lane & 15, s0 = 16 * I;
            const int l = 4 * (warp & 3) + 2 * (lane >> 4);
            float ar[16];
            const float4* arow = reinterpret_cast<const float4*>(sA + (s0 + m) * kPA + s0);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 t = arow[u];
                ar[4 * u] = t.x; ar[4 * u + 1] = t.y; ar[4 * u + 2] = t.z; ar[4 * u + 3] = t.w;
            }
            float xa = (m == l) ? 1.f : 0.f, xb = (m == l + 1) ? 1.f : 0.f;
            const int src = lane & 16;
#pragma unroll
            for (int r = 0; r < 15; ++r) {  // A[m][r] = 0 for r >= m: rows <= r are unchanged
                const float ya = __shfl_sync(0xffffffffu, xa, src + r);
                const float yb = __shfl_sync(0xffffffffu, xb, src + r);
                xa = fmaf(-ar[r], ya, xa);
                xb = fmaf(-ar[r], yb, xb);
            }
            const int i = s0 + m, j = s0 + l;
            *reinterpret_cast<float2*>(sT + i * kPA + j) = make_float2(tf32_round(xa), tf32_round(xb));
            store_tprime_pair(sm, i, j, xa, xb, sBeta);
            // Zero the 16 x 16 blocks of T' above the diagonal (column block J >
            // row block I), in both row halves of TT: 6 blocks x 16 rows x 2 chunks.
            if (tid < 6 * 32) {
                const int bi = tid >> 5, rr = (tid >> 1) & 15, hc = tid & 1;
                const int Ib = bi < 3 ? 0 : (bi < 5 ? 1 : 2);
                const int Jb = bi < 3 ? bi + 1 : (bi < 5 ? bi - 1 : 3);
                const int row = 16 * Ib + rr, col = 16 * Jb + 8 * hc;
                *reinterpret_cast<uint4*>(sm + O_TT + sw128_off(row, col)) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(sm + O_TT + sw128_off(64 + row, col)) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        stall_point<kStall>(p.stall_seed, 7, it);
        __syncthreads();
        // Off-diagonal blocks with warp-level tf32 tensor-core products (fp32
        // accumulation; T' is rounded to bf16 for MMA C anyway).
        const int g4 = lane >> 2, t4 = lane & 3;
        if (warp < 4) {
            // 16 -> 32 in 32-block p, columns c0..c0+7: X = A_10 T_00 (T_00 lower
            // triangular: k >= c0), then T_10 = -T_11 X.
            const int pb = 32 * (warp >> 1), ct = warp & 1, c0 = 8 * ct;
            float* x = sX + (warp >> 1) * 16 * kPX + c0;
            float d[4];
            warp_mma_16x8(sA + (pb + 16) * kPA + pb, kPA, sT + pb * kPA + pb + c0, kPA, ct, 2, d, lane);
            store_tile_tf32(x, kPX, d, lane);
            stall_point<kStall>(p.stall_seed, 8, it);
            __syncwarp();
            warp_mma_16x8(sT + (pb + 16) * kPA + pb + 16, kPA, x, kPX, 0, 2, d, lane);
            d[0] = -d[0]; d[1] = -d[1]; d[2] = -d[2]; d[3] = -d[3];
            store_tile_tf32(sT + (pb + 16) * kPA + pb + c0, kPA, d, lane);
            store_tprime_pair(sm, pb + 16 + g4, pb + c0 + 2 * t4, d[0], d[1], sBeta);
            store_tprime_pair(sm, pb + 24 + g4, pb + c0 + 2 * t4, d[2], d[3], sBeta);
        } else if (warp == 13 && lane == 0 && cn.len > 0) {
            // The next record's tiles: E2 has read the current ones, and they land
            // during the rest of the solve and MMA C rather than during the
            // shared-memory-heavy epilogues.
            load_inputs(sm, maps, cn, rec_next % p.H, &bar_in);
        } else if (lane == 0 && warp >= 8 && warp <= 12) {
            // The Aqk, Kt, e^gam and Q e^Gam images leave by bulk copy, one per
            // idle warp (these warps take no part in the 32 -> 64 products).
            uint8_t* rp = p.ws_rec + (size_t)rec * kRecBytes;
            if (warp == 8) bulk_store(rp + kRecAqk, sm + O_AQK, 8192);
            else if (warp == 9) bulk_store(rp + kRecKt, sm + O_SKT, 16384);
            else if (warp == 10) bulk_store(rp + kRecEg, sm + O_SEG, 512);
            else if (warp == 11) bulk_store(rp + kRecA1, sm + O_QT, 8192);
            else bulk_store(rp + kRecA1 + 16384, sm + O_QT + 8192, 8192);
            bulk_commit();
        }
        // The 32 -> 64 products (warps 0-7) read the 16 -> 32 results.
        if (warp < 8) named_bar_sync(2, 256);
        if (cn.len > 0) pend_parity = (int)((it + 1) & 1);
        if (warp < 8) {
            // 32 -> 64, row tile rt (16 rows), columns c0..c0+7:
            // X = A[32:, :32] T[:32, :32] (k >= c0), then T[32:, :32] = -T[32:, 32:] X
            // (row tile rt of T[32:, 32:] is zero beyond k = 16 (rt + 1)).
            const int rt = warp >> 2, ct = warp & 3, c0 = 8 * ct;
            float d[4];
            warp_mma_16x8(sA + (32 + 16 * rt) * kPA, kPA, sT + c0, kPA, ct, 4, d, lane);
            store_tile_tf32(sX + 16 * rt * kPX + c0, kPX, d, lane);
            stall_point<kStall>(p.stall_seed, 9, it);
            named_bar_sync(1, 256);
            warp_mma_16x8(sT + (32 + 16 * rt) * kPA + 32, kPA, sX + c0, kPX, 0, 2 * (rt + 1), d, lane);
            const int r0 = 32 + 16 * rt + g4;
            store_tprime_pair(sm, r0, c0 + 2 * t4, -d[0], -d[1], sBeta);
            store_tprime_pair(sm, r0 + 8, c0 + 2 * t4, -d[2], -d[3], sBeta);
        }
        stall_point<kStall>(p.stall_seed, 10, it);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();

        // ---- MMA C: W = [T' ; T'] (K e^Gam) (N = 128: W in both halves of the
        // lanes) and U^T = V^T T'^T (M = 128 value columns, N = 64 tokens; A is
        // the V half of the [K e^Gam | V] operand, read MN-major).
        if (tid == 0) {
            tc_fence_after();
            const uint32_t tt = smem_u32(sm + O_TT), kv = smem_u32(sm + O_KV);
            for (uint32_t k = 0; k < 4; ++k)
                umma_bf16(tb + TM_C, sdesc_kmajor_sw128(tt + k * 32u),
                          sdesc_mnmajor_sw128(kv + k * 2u * kKvSbo, 1024u, kKvSbo),
                          idesc_bf16_f32_bmn(128, 128), k > 0 ? 1u : 0u);
            for (uint32_t k = 0; k < 4; ++k)
                umma_bf16(tb + TM_C + 128, sdesc_mnmajor_sw128(kv + 2048u + k * 2u * kKvSbo, 1024u, kKvSbo),
                          sdesc_kmajor_sw128(tt + k * 32u), idesc_bf16_f32(128, 64) | (1u << 15),
                          k > 0 ? 1u : 0u);
            umma_commit(&bar_mma[1]);
        }
        ok = __syncthreads_and(tid == 0 ? mbar_wait(&bar_mma[1], it & 1, nullptr, p.wait_ns) : true);
        tc_fence_after();
        if (!ok) break;
        stall_point<kStall>(p.stall_seed, 12, it);
        {
            // ---- Epilogue C, 32 columns per warp, written as the record's
            // shared-memory images and stored with bulk copies: W (cq 0, 1) from
            // the first 128 columns, keys 64 (qd / 2) + 32 cq .. of token row
            // 32 (qd % 2) + lane; U^T (cq 2, 3) from the next 64, tokens
            // 32 (cq - 2) .. of value row 32 qd + lane.
            float v[32];
            tmem_ld32(tmem_addr(tb, 32 * qd, TM_C + (cq < 2 ? 64 * (qd >> 1) + 32 * cq : 128 + 32 * (cq - 2))), v);
            uint32_t w[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) w[x] = pack_bf16x2(v[2 * x], v[2 * x + 1]);
            if (cq < 2) {
                const int i = 32 * (qd & 1) + lane;
                uint8_t* img = sm + O_SW + (qd >> 1) * 8192;
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    *reinterpret_cast<uint4*>(img + sw128_off(i, 32 * cq + 8 * x)) =
                        make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
            } else {
                const int vr = 32 * qd + lane;
#pragma unroll
                for (int x = 0; x < 4; ++x)
                    *reinterpret_cast<uint4*>(sm + O_SU + sw128_off(vr, 32 * (cq - 2) + 8 * x)) =
                        make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
            }
        }
        stall_point<kStall>(p.stall_seed, 13, it);
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            uint8_t* rp = p.ws_rec + (size_t)rec * kRecBytes;
            bulk_store(rp + kRecA1 + 8192, sm + O_SW, 8192);
            bulk_store(rp + kRecA1 + 16384 + 8192, sm + O_SW + 8192, 8192);
            bulk_store(rp + kRecU, sm + O_SU, 16384);
            bulk_commit();
        }
        // Epilogue C's TMEM reads are ordered before the next record's MMA A by
        // this fence and the CTA barrier of the next input wait (the loop's top).
        tc_fence_before();
        rec = rec_next;
        ci = cn;
    }
    if (!ok && tid == 0) {
        atomicExch(p.status, 4);
        // A working wait ran out: every product issued so far completes before
        // the CTA lets go of TMEM and shared memory (bounded).
        umma_commit(&bar_fin);
        mbar_wait(&bar_fin, 0, nullptr);
    }
    if (lane == 0) bulk_wait_all();  // no bulk store may outlive the CTA's shared memory
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
        if (p.seq_order)
            for (int n = tid; n < p.N; n += blockDim.x) p.seq_order[n] = n;
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
    // The order in which the state pass takes the sequences (its CTAs are
    // launched sequence by sequence): longest chain first, so that the chains
    // that set the pass's length start in the first wave of CTAs and the short
    // ones fill in behind them.  Up to 1024 sequences are ranked (ties by
    // index); beyond that the order is the index order.
    if (p.seq_order) {
        __shared__ int cnts[1024];
        if (p.N <= (int)blockDim.x) {
            const int n = tid;
            const int mine = n < p.N ? (p.cu[n + 1] - p.cu[n] + kChunk - 1) / kChunk : 0;
            if (n < p.N) cnts[n] = mine;
            __syncthreads();
            if (n < p.N) {
                int rank = 0;
                for (int m = 0; m < p.N; ++m) {
                    const int cm = cnts[m];
                    rank += (cm > mine || (cm == mine && m < n)) ? 1 : 0;
                }
                p.seq_order[rank] = n;
            }
        } else {
            for (int n = tid; n < p.N; n += blockDim.x) p.seq_order[n] = n;
        }
    }
}

}  // namespace

cudaError_t launch_chunk_table(const PrefillParams& p, cudaStream_t s) {
    if (p.cu == nullptr) return cudaSuccess;
    chunk_table_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prep(const PrefillParams& p, const PrepMaps& maps, int num_sms, cudaStream_t s,
                        bool overlap_previous) {
    if (num_sms < 1) return cudaSuccess;
    const long long recs = (long long)p.max_chunks * p.H;
    if (recs == 0) return cudaSuccess;
    // the instantiation with the stall hook runs only when a test asks for it
    static std::atomic<uint64_t> smem_set[2];
    auto kern = p.stall_seed ? prep_kernel<true> : prep_kernel<false>;
    cudaError_t e = set_smem_limit_once((const void*)kern, (int)kPrepSmem, smem_set[p.stall_seed ? 1 : 0]);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(recs < num_sms ? recs : num_sms);
    if (!overlap_previous) {
        kern<<<grid, kPrepThreads, kPrepSmem, s>>>(p, maps);
        return cudaGetLastError();
    }
    // Programmatic launch: this grid's CTAs may start while the previous prep
    // grid in the stream finishes its last records (it reads nothing that grid
    // writes), so that its tail and this grid's start-up overlap.
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPrepThreads);
    cfg.dynamicSmemBytes = kPrepSmem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p, maps);
}

}  // namespace kda
