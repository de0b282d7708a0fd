// kda_verify_wy.cu -- MTP verify on the tensor cores: the drafts of a request
// form one WY-form chunk (the tcgen05 KDA MTP verify kernel of the TensorRT-LLM
// page "Kimi K3 work for Rubin (SM107)", Description: WY-form chunk, fp32 and
// bf16 state pools, replay-only commit).
//
// Per (request, head) item with entry state S (128 keys x 128 values, fp32),
// D <= 16 drafts and accepted prefix a, with Gam the inclusive prefix over the
// drafts of the gate g (per key channel):
//   A[i,j]   = beta_i sum_c k_i k_j exp(Gam_i - Gam_j)        j <  i
//   Aqk[i,j] = scale sum_c q_i k_j exp(Gam_i - Gam_j)         j <= i
//   T' = (I + A)^-1 Diag(beta),  W = T' (K e^Gam),  U = T' V
//   Q' = scale Q e^Gam - Aqk W,  O_loc = Aqk U
//   P1: D1 = [W ; Q'] S           (tensor cores, kind::tf32, fp32 accumulation)
//       V_new = U - D1[W rows],   O = O_loc + D1[Q' rows]      -> out
//   P2: D2 = Kt_a V_new,  Kt_a[c,j] = k_j[c] exp(Gam_{a-1}[c] - Gam_j[c]) (j < a)
//       S_a = Diag(exp Gam_{a-1}) S + D2                       -> pool (fp32 update)
// which is the sequential recurrence run over the drafts (the derivation of the
// chunked form), with only the state after the accepted prefix stored.  Every
// decay factor is exp of a difference Gam_i - Gam_j <= 0, so no factor can
// overflow whatever the gates.  The tensor-core operands are tf32 (fp32 with a
// 10-bit mantissa; the bf16 operand path of the page is optional and not used);
// the state itself is updated in fp32.
//
// Layout of the products (TMEM lane = output row; tf32 operands in shared
// memory must be K-major, i.e. with the contraction index contiguous):
//   P1 is computed transposed, D1^T = S^T [W ; Q']^T: M = 128 values, N = 32
//   (W rows 0..15, Q' rows 16..31), K = 128 keys.  A = S^T lies in TMEM (lane =
//   value, one key per column), written by the threads as they load the state
//   (lanes = consecutive values: every load is a coalesced 128-byte row piece);
//   B = [W ; Q'] is K-major in shared memory.  The state block arrives by one
//   1-D bulk copy (64 KB fp32 / 32 KB bf16, rows = keys) into one of two
//   staging buffers, requested one item ahead; threads read its columns
//   (lane = value: one 128-byte row piece per key) into TMEM, and read them
//   again for the final update.
//   P2 is computed transposed too, D2^T = V_new^T Kt_a^T: M = 128 values,
//   N = 128 keys, K = 8 or 16 drafts, A = V_new^T (value rows, written by the
//   P1 epilogue), B = Kt_a (key rows); D2^T takes the TMEM columns of S^T, which
//   P1 has finished reading.  Both epilogues run with lane = value column, so
//   that every global store of the updated state is a coalesced row piece.
//
// Organisation: persistent CTAs, one per SM, stream the items.  The state and
// the drafts of item i + 1 are copied in (bulk copy, cp.async) while item i
// runs.  The per-item preparation (gate prefix, the
// pair products with a reduce-scatter over the warp, the triangular solve, W,
// U, Q', O_loc, Kt_a) runs on the CUDA cores.  The product waits are bounded
// like the prefill kernels'; a wait that runs out records KDA_ERR_TIMEOUT and
// the CTA winds down after waiting for the products it issued and its copies.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kWyThreads = 256;
constexpr int kWyMaxDrafts = 16;          // drafts per request (the kernel's kDmax is 8 or 16)
constexpr int kNB = 32;                   // N of P1: W rows 0..15, Q' rows 16..31
// Shared memory (bytes from a 1024-aligned base).
constexpr uint32_t Y_B1 = 0;              // [W ; Q'] fp32 K-major: 4 key blocks of 32 rows x 128 B (16 KB)
constexpr uint32_t kB1Block = kNB * 128;
constexpr uint32_t Y_A2 = 16384;          // Kt_a fp32 K-major: 128 key rows x 128 B (up to 32 drafts)
constexpr uint32_t Y_VN = 32768;          // V_new^T fp32 K-major: 128 value rows x 128 B
constexpr uint32_t Y_Q = 49152;           // drafts: q, k, v bf16 [16][128], g fp32 [16][128]
constexpr uint32_t Y_K = Y_Q + 4096;
constexpr uint32_t Y_V = Y_K + 4096;
constexpr uint32_t Y_G = Y_V + 4096;      // g, turned in place into Gam
constexpr uint32_t Y_U = Y_G + 8192;      // U fp32 [16][128]
constexpr uint32_t Y_OL = Y_U + 8192;     // O_loc fp32 [16][128]
constexpr uint32_t Y_A = Y_OL + 8192;     // A, Aqk, T' fp32 [16][17] each
constexpr int kPs = 17;
constexpr uint32_t Y_AQ = Y_A + 16 * kPs * 4;
constexpr uint32_t Y_TP = Y_AQ + 16 * kPs * 4;
constexpr uint32_t Y_EGA = Y_TP + 16 * kPs * 4;   // exp(Gam_{a-1}) fp32 [128]
constexpr uint32_t Y_BETA = Y_EGA + 512;          // beta fp32 [16]
constexpr uint32_t Y_ST = 92160;                  // two state stagings of 64 KB (rows = keys)
constexpr uint32_t kStBytes = 65536;
constexpr uint32_t kWySmem = Y_ST + 2 * kStBytes + 1024;
constexpr uint32_t TW_S = 0, TW_D1 = 128, TW_COLS = 256;   // S^T (then D2^T), D1^T

__device__ __forceinline__ void cp_async16_wy(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit_wy() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0_wy() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ float bf16f(const uint8_t* p) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(p)) << 16);
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Warp-collective store of 16 consecutive 32-bit columns (no wait).
__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Reduce-scatter of 32 per-lane values over the warp: afterwards lane l holds
// the warp's sum of value l (16 + 8 + 4 + 2 + 1 shuffles; at each level a lane
// keeps the half of its values that its lane bit selects and adds the
// partner's copy of that half).
__device__ __forceinline__ float warp_reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int lvl = 0; lvl < 5; ++lvl) {
        const int half = 16 >> lvl;                // values kept at this level
        const bool up = (lane & half) != 0;
#pragma unroll
        for (int t = 0; t < half; ++t) {
            const float send = up ? v[t] : v[t + half];
            const float keep = up ? v[t + half] : v[t];
            v[t] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
    }
    return v[0];
}

struct WyItem {
    int r, h, slot, acc;
    bool valid;
};

template <bool kBf16, bool kStall, int kDmax>
__global__ void __launch_bounds__(kWyThreads, 1) verify_wy_kernel(const VerifyParams p) {
    extern __shared__ uint8_t smw_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smw_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t bar_p1, bar_p2, bar_fin, bar_never, bar_st[2];
    __shared__ uint32_t tmem_base_sh;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nitems = p.R * p.H, D = p.D;
    if ((int)blockIdx.x >= nitems) return;

    if (tid == 0) {
        mbar_init(&bar_p1, 1);
        mbar_init(&bar_p2, 1);
        mbar_init(&bar_fin, 1);
        mbar_init(&bar_never, 1);   // nothing arrives on it (the timeout probe's wait)
        mbar_init(&bar_st[0], 1);
        mbar_init(&bar_st[1], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, TW_COLS);
        tmem_relinquish();
    }
    // Operand rows that no item writes stay zero: [W ; Q'] rows past D (and the
    // Q' rows in replay-only mode), V_new^T and Kt_a columns past D, the pair
    // matrices' upper triangles.
    for (uint32_t o = tid * 16; o < Y_Q - Y_B1; o += kWyThreads * 16)
        *reinterpret_cast<uint4*>(sm + Y_B1 + o) = make_uint4(0u, 0u, 0u, 0u);
    for (uint32_t o = tid * 4; o < Y_EGA - Y_A; o += kWyThreads * 4) *reinterpret_cast<float*>(sm + Y_A + o) = 0.f;
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base_sh;
    const int q4 = warp & 3, val = 32 * q4 + lane, kh = warp >> 2;   // lane = value column
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;

    auto item_of = [&](int it) -> WyItem {
        WyItem x{0, 0, 0, 0, false};
        if (it >= nitems) return x;
        x.r = it / p.H;
        x.h = it - x.r * p.H;
        x.slot = p.slot ? p.slot[x.r] : x.r;
        x.acc = p.accepted[x.r];
        x.valid = x.slot >= 0 && x.slot < p.P && x.acc >= 0 && x.acc <= D;
        return x;
    };
    // The drafts of item x into the staging rows (one cp.async group).
    auto fetch_drafts = [&](const WyItem& x) {
        if (x.valid) {
            for (int e = tid; e < D * 64; e += kWyThreads) {
                const int t = e >> 6, j = e & 63;
                if (j < 16) {
                    cp_async16_wy(sm + Y_Q + t * 256 + j * 16, p.q + x.r * p.qs[0] + t * p.qs[1] + x.h * p.qs[2] + 8 * j);
                } else if (j < 32) {
                    cp_async16_wy(sm + Y_K + t * 256 + (j - 16) * 16,
                                  p.k + x.r * p.ks[0] + t * p.ks[1] + x.h * p.ks[2] + 8 * (j - 16));
                } else {
                    const int jj = j - 32;   // g: 32 pieces of 16 B; v: the first 16 of them
                    if (jj < 16)
                        cp_async16_wy(sm + Y_V + t * 256 + jj * 16,
                                      p.v + x.r * p.vs[0] + t * p.vs[1] + x.h * p.vs[2] + 8 * jj);
                    cp_async16_wy(sm + Y_G + t * 512 + jj * 16, p.g + x.r * p.gs[0] + t * p.gs[1] + x.h * p.gs[2] + 4 * jj);
                }
            }
        }
        cp_async_commit_wy();
    };
    constexpr uint32_t kRowB = kHeadDim * (kBf16 ? 2 : 4), kPitch = kRowB;
    constexpr uint32_t kStateB = kHeadDim * kRowB;
    uint32_t st_issued[2] = {0u, 0u};   // bulk copies requested per staging buffer (thread 0)
    // The state block of item x into staging buffer b (thread 0, one bulk copy).
    auto fetch_state = [&](const WyItem& x, int b) {
        if (tid == 0 && x.valid) {
            mbar_arrive_expect_tx(&bar_st[b], kStateB);
            bulk_load(sm + Y_ST + b * kStBytes,
                      static_cast<const uint8_t*>(p.pool) + ((size_t)x.slot * p.H + x.h) * kStateB, kStateB,
                      &bar_st[b]);
            ++st_issued[b];
        }
    };

    int it = blockIdx.x;
    WyItem cur = item_of(it);
    fetch_drafts(cur);
    fetch_state(cur, 0);
    uint32_t st_waited[2] = {0u, 0u};   // bulk copies waited for per buffer
    bool ok = true;
    bool mma_issued = false;
    uint32_t n_p1 = 0, n_p2 = 0;   // products waited for so far (the barriers' phases)
    float* gam = reinterpret_cast<float*>(sm + Y_G);
    float* Am = reinterpret_cast<float*>(sm + Y_A);
    float* Aq = reinterpret_cast<float*>(sm + Y_AQ);
    float* Tp = reinterpret_cast<float*>(sm + Y_TP);
    float* sU = reinterpret_cast<float*>(sm + Y_U);
    float* sOL = reinterpret_cast<float*>(sm + Y_OL);
    float* sEga = reinterpret_cast<float*>(sm + Y_EGA);
    float* sBeta = reinterpret_cast<float*>(sm + Y_BETA);

    for (uint32_t k = 0; it < nitems; ++k) {
        const int nit = it + (int)gridDim.x;
        const WyItem nxt = item_of(nit);
        const int a = cur.acc;
        const bool outputs = !p.replay_only;
        const bool state_upd = cur.valid && a > 0;
        const int sb = (int)(k & 1);
        stall_point<kStall>(p.stall_seed, 1, k);
        // The next item's state into the other buffer (its last reader, item
        // k - 1, is done: the loop's closing barrier).
        fetch_state(nxt, sb ^ 1);
        cp_async_wait0_wy();   // this item's drafts have landed
        __syncthreads();
        if (!cur.valid) {
            if (tid == 0 && p.status) atomicExch(p.status, 1);
        } else {
            // ---- gate prefix Gam (in place of g) and beta
            if (tid < kHeadDim) {
                float gv[kDmax];
#pragma unroll
                for (int t = 0; t < kDmax; ++t)
                    if (t < D) gv[t] = gam[t * kHeadDim + tid];
                float acc = 0.f;
#pragma unroll
                for (int t = 0; t < kDmax; ++t)
                    if (t < D) {
                        acc += gv[t];
                        gam[t * kHeadDim + tid] = acc;
                    }
            } else if (tid - kHeadDim < D) {
                const int t = tid - kHeadDim;
                const float b = p.beta[cur.r * p.bs[0] + t * p.bs[1] + cur.h * p.bs[2]];
                sBeta[t] = p.beta_is_logit ? 1.0f / (1.0f + __expf(-b)) : b;
            }
            __syncthreads();
            // ---- pair products: warp w takes rows i = w, w + 8; lane = channels
            // lane + 32 m; the 32 partial sums (A and Aqk against every j) are
            // reduce-scattered so that lane l ends with value l
            for (int i = warp; i < D; i += kWyThreads / 32) {
                float v[32];   // A partials (0..15), Aqk partials (16..31)
#pragma unroll
                for (int x = 0; x < 32; ++x) v[x] = 0.f;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = lane + 32 * m;
                    const float gi = gam[i * kHeadDim + c];
                    const float ki = bf16f(sm + Y_K + i * 256 + 2 * c), qi = bf16f(sm + Y_Q + i * 256 + 2 * c);
#pragma unroll
                    for (int j = 0; j < kDmax; ++j) {
                        if (j <= i) {
                            const float kj = bf16f(sm + Y_K + j * 256 + 2 * c) * __expf(gi - gam[j * kHeadDim + c]);
                            v[j] = fmaf(ki, kj, v[j]);
                            v[16 + j] = fmaf(qi, kj, v[16 + j]);
                        }
                    }
                }
                const float sum = warp_reduce_scatter32(v, lane);
                if (lane < 16) {
                    if (lane < i) Am[i * kPs + lane] = sBeta[i] * sum;
                } else if (lane - 16 <= i) {
                    Aq[i * kPs + lane - 16] = p.scale * sum;
                }
            }
            __syncthreads();
            // ---- T = (I + A)^-1 by forward substitution: warp w solves columns
            // 2w (lanes 0..15) and 2w + 1 (lanes 16..31), lane = row; T' = T Diag(beta)
            {
                const int m = lane & 15, col = 2 * warp + (lane >> 4);
                float x = (m == col) ? 1.f : 0.f;
                for (int r = 0; r + 1 < D; ++r) {
                    const float y = __shfl_sync(0xffffffffu, x, (lane & 16) + r);
                    x = fmaf(-Am[m * kPs + r], y, x);   // A[m][r] = 0 for r >= m
                }
                if (m < D && col < D) Tp[m * kPs + col] = x * sBeta[col];
            }
            __syncthreads();
            // ---- W, U (rows of parity hf), Kt_a and exp(Gam_{a-1}); thread = channel c.
            // Every operand is loaded into registers before the first store, so the
            // loads are not held behind the stores.
            {
                const int c = tid & (kHeadDim - 1), hf = tid >> 7;
                constexpr int kR = kDmax / 2;          // rows of one parity
                float ke[kDmax], vv[kDmax], w[kR], u[kR];
#pragma unroll
                for (int j = 0; j < kDmax; ++j) {
                    ke[j] = j < D ? bf16f(sm + Y_K + j * 256 + 2 * c) * __expf(gam[j * kHeadDim + c]) : 0.f;
                    vv[j] = j < D ? bf16f(sm + Y_V + j * 256 + 2 * c) : 0.f;
                }
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int i = 2 * r + hf;
                    w[r] = 0.f;
                    u[r] = 0.f;
#pragma unroll
                    for (int j = 0; j < kDmax; ++j) {
                        if (j <= i && i < D) {
                            const float t = Tp[i * kPs + j];
                            w[r] = fmaf(t, ke[j], w[r]);
                            u[r] = fmaf(t, vv[j], u[r]);
                        }
                    }
                }
                float kt[kDmax];
                float ga = 0.f;
                if (state_upd) {
                    ga = gam[(a - 1) * kHeadDim + c];
#pragma unroll
                    for (int j = 0; j < kDmax; ++j)
                        kt[j] = (hf == 0 && j < a) ? to_tf32(bf16f(sm + Y_K + j * 256 + 2 * c) *
                                                             __expf(ga - gam[j * kHeadDim + c]))
                                                   : 0.f;
                }
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int i = 2 * r + hf;
                    if (i < D) {
                        *reinterpret_cast<float*>(sm + Y_B1 + f32_kmajor_off(i, c, kB1Block)) = to_tf32(w[r]);
                        sU[i * kHeadDim + c] = u[r];
                    }
                }
                if (state_upd) {
                    if (hf == 0) {
#pragma unroll
                        for (int j = 0; j < kDmax; j += 4)
                            *reinterpret_cast<float4*>(sm + Y_A2 + f32_kmajor_off(c, j, 16384u)) =
                                make_float4(kt[j], kt[j + 1], kt[j + 2], kt[j + 3]);
                    } else {
                        sEga[c] = __expf(ga);
                    }
                }
            }
            __syncthreads();
            // ---- Q' and O_loc (outputs only), again loads first
            if (outputs) {
                const int c = tid & (kHeadDim - 1), hf = tid >> 7;
                constexpr int kR = kDmax / 2;
                float wv[kDmax], uv[kDmax], qp[kR], ol[kR];
#pragma unroll
                for (int j = 0; j < kDmax; ++j) {
                    wv[j] = j < D ? *reinterpret_cast<const float*>(sm + Y_B1 + f32_kmajor_off(j, c, kB1Block)) : 0.f;
                    uv[j] = j < D ? sU[j * kHeadDim + c] : 0.f;
                }
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int i = 2 * r + hf;
                    qp[r] = i < D ? p.scale * bf16f(sm + Y_Q + i * 256 + 2 * c) * __expf(gam[i * kHeadDim + c]) : 0.f;
                    ol[r] = 0.f;
#pragma unroll
                    for (int j = 0; j < kDmax; ++j) {
                        if (j <= i && i < D) {
                            const float aq = Aq[i * kPs + j];
                            qp[r] = fmaf(-aq, wv[j], qp[r]);
                            ol[r] = fmaf(aq, uv[j], ol[r]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    const int i = 2 * r + hf;
                    if (i < D) {
                        *reinterpret_cast<float*>(sm + Y_B1 + f32_kmajor_off(16 + i, c, kB1Block)) = to_tf32(qp[r]);
                        sOL[i * kHeadDim + c] = ol[r];
                    }
                }
            }
            fence_proxy_async_smem();
        }
        stall_point<kStall>(p.stall_seed, 2, k);
        __syncthreads();   // the drafts' staging is free; the operands are written
        fetch_drafts(nxt);
        const bool run_p1 = cur.valid && (outputs || a > 0);
        const uint8_t* stg = sm + Y_ST + sb * kStBytes;
        // S[key][val] from the staging buffer (lanes = consecutive values)
        auto s_at = [&](int key) -> float {
            return kBf16 ? __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(stg + key * kPitch + val * 2) << 16)
                         : *reinterpret_cast<const float*>(stg + key * kPitch + val * 4);
        };
        if (cur.valid) {
            // this item's state has landed (bounded; thread 0 waits, the others at the barrier)
            ok = __syncthreads_and(tid == 0 ? mbar_wait(&bar_st[sb], st_waited[sb] & 1, nullptr, p.wait_ns) : true);
            if (!ok) break;
            if (tid == 0) ++st_waited[sb];
        }
        if (run_p1) {
            // ---- S^T into TMEM: lane = value, 64 keys per thread (columns 64 kh ..)
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16) {
                uint32_t w[16];
#pragma unroll
                for (int x = 0; x < 16; ++x) w[x] = __float_as_uint(s_at(64 * kh + c0 + x));
                tmem_st16_nowait(tb + lane_base + TW_S + 64 * kh + c0, w);
            }
            tmem_wait_st();
            tc_fence_before();
            stall_point<kStall>(p.stall_seed, 3, k);
            __syncthreads();
            tc_fence_after();
            // ---- P1: D1^T = S^T [W ; Q']^T, 16 K steps of 8 keys
            if (tid == 0) {
                const uint32_t b1 = smem_u32(sm + Y_B1);
                const uint32_t id = idesc_tf32_f32(128, kNB, false, false);
#pragma unroll 1
                for (uint32_t st = 0; st < 16; ++st)
                    umma_tf32_ta(tb + TW_D1, tb + TW_S + 8 * st,
                                 sdesc_kmajor_sw128(b1 + (st >> 2) * kB1Block + (st & 3) * 32u), id, st > 0 ? 1u : 0u);
                umma_commit(&bar_p1);
                mma_issued = true;
            }
            ok = __syncthreads_and(tid == 0 ? mbar_wait((p.timeout_probe && n_p1 == 0) ? &bar_never : &bar_p1,
                                                        n_p1 & 1, nullptr, p.wait_ns)
                                            : true);
            tc_fence_after();
            if (!ok) break;
            ++n_p1;
            stall_point<kStall>(p.stall_seed, 4, k);
            // ---- epilogue of P1: warps 0-3 V_new (columns 0..15), warps 4-7 the
            // outputs (columns 16..31); lane = value column
            {
                float d[16];
                tmem_ld16(tb + lane_base + TW_D1 + (kh == 0 ? 0 : 16), d);
                if (kh == 0) {
                    // V_new^T row `val`: drafts in 16-byte pieces (columns past D stay zero)
                    for (int j4 = 0; j4 < D; j4 += 4) {
                        float x[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            x[u] = (j4 + u < D) ? to_tf32(sU[(j4 + u) * kHeadDim + val] - d[j4 + u]) : 0.f;
                        *reinterpret_cast<float4*>(sm + Y_VN + f32_kmajor_off(val, j4, 16384u)) =
                            make_float4(x[0], x[1], x[2], x[3]);
                    }
                    fence_proxy_async_smem();
                } else if (outputs) {
                    for (int i = 0; i < D; ++i)
                        p.out[cur.r * p.os[0] + i * p.os[1] + cur.h * p.os[2] + val] =
                            __float2bfloat16_rn(sOL[i * kHeadDim + val] + d[i]);
                }
            }
            tc_fence_before();
            stall_point<kStall>(p.stall_seed, 5, k);
            __syncthreads();
            tc_fence_after();
        }
        if (state_upd) {
            // ---- P2: D2^T = V_new^T Kt_a^T over the accepted drafts (rounded up
            // to 8), into the columns S^T held
            if (tid == 0) {
                const uint32_t a2 = smem_u32(sm + Y_A2), vn = smem_u32(sm + Y_VN);
                const uint32_t id = idesc_tf32_f32(128, 128, false, false);
                const int steps = (a + 7) >> 3;
                for (int st = 0; st < steps; ++st)
                    umma_tf32(tb + TW_S, sdesc_kmajor_sw128(vn + st * 32u), sdesc_kmajor_sw128(a2 + st * 32u), id,
                              st > 0 ? 1u : 0u);
                umma_commit(&bar_p2);
                mma_issued = true;
            }
            ok = __syncthreads_and(tid == 0 ? mbar_wait(&bar_p2, n_p2 & 1, nullptr, p.wait_ns) : true);
            tc_fence_after();
            if (!ok) break;
            ++n_p2;
            stall_point<kStall>(p.stall_seed, 6, k);
            // ---- S_a[key][val] = exp(Gam_{a-1})[key] S[key][val] + D2^T[val][key]
            // for this thread's value column and 64 keys (S from the staging
            // buffer); lanes = consecutive values, so each store is a 128-byte
            // (fp32) row piece per warp
            {
                uint8_t* dst = static_cast<uint8_t*>(p.pool) + ((size_t)cur.slot * p.H + cur.h) * kStateB +
                               (size_t)val * (kBf16 ? 2 : 4);
#pragma unroll 1
                for (int c0 = 0; c0 < 64; c0 += 32) {
                    float d2[32];
                    tmem_ld32(tb + lane_base + TW_S + 64 * kh + c0, d2);
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int key = 64 * kh + c0 + x;
                        const float n = fmaf(sEga[key], s_at(key), d2[x]);
                        if (kBf16)
                            *reinterpret_cast<__nv_bfloat16*>(dst + (size_t)key * kRowB) = __float2bfloat16_rn(n);
                        else
                            *reinterpret_cast<float*>(dst + (size_t)key * kRowB) = n;
                    }
                }
            }
        }
        tc_fence_before();
        stall_point<kStall>(p.stall_seed, 7, k);
        __syncthreads();   // every read of this item's TMEM and operands is done
        tc_fence_after();
        it = nit;
        cur = nxt;
    }
    if (!ok && tid == 0 && p.status) atomicExch(p.status, 4);
    if (tid == 0 && mma_issued) {
        // every product issued has completed before TMEM is released (bounded)
        umma_commit(&bar_fin);
        mbar_wait(&bar_fin, 0, nullptr);
    }
    cp_async_wait0_wy();   // no copy may land after the CTA has left
    if (tid == 0)
        for (int b = 0; b < 2; ++b)
            while (st_waited[b] < st_issued[b]) {
                mbar_wait(&bar_st[b], st_waited[b] & 1, nullptr);
                ++st_waited[b];
            }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, TW_COLS);
}

template <bool kBf16, bool kStall, int kDmax>
cudaError_t launch_wy_t(const VerifyParams& p, int num_sms, cudaStream_t s) {
    static std::atomic<uint64_t> smem_set;
    cudaError_t e = set_smem_limit_once((const void*)verify_wy_kernel<kBf16, kStall, kDmax>, (int)kWySmem, smem_set);
    if (e != cudaSuccess) return e;
    const long long items = (long long)p.R * p.H;
    const unsigned grid = (unsigned)(items < num_sms ? items : num_sms);
    verify_wy_kernel<kBf16, kStall, kDmax><<<grid, kWyThreads, kWySmem, s>>>(p);
    return cudaGetLastError();
}

template <bool kBf16, bool kStall>
cudaError_t launch_wy_d(const VerifyParams& p, int num_sms, cudaStream_t s) {
    return p.D <= 8 ? launch_wy_t<kBf16, kStall, 8>(p, num_sms, s) : launch_wy_t<kBf16, kStall, 16>(p, num_sms, s);
}

}  // namespace

cudaError_t launch_verify_wy(const VerifyParams& p, int num_sms, cudaStream_t s) {
    if (p.R == 0 || p.H == 0) return cudaSuccess;
    if (p.D < 1 || p.D > kWyMaxDrafts) return cudaErrorInvalidValue;
    if (p.stall_seed)
        return p.pool_bf16 ? launch_wy_d<true, true>(p, num_sms, s) : launch_wy_d<false, true>(p, num_sms, s);
    return p.pool_bf16 ? launch_wy_d<true, false>(p, num_sms, s) : launch_wy_d<false, false>(p, num_sms, s);
}

}  // namespace kda
