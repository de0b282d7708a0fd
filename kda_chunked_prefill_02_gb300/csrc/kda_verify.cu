// kda_verify.cu -- MTP verify: a short draft chunk per request run against a
// fp32 state pool, with the state after the accepted prefix written back.
//
// The drafts of one request form one short chunk of the KDA recurrence (the
// tcgen05 KDA MTP verify kernel and its replay-only commit on the TensorRT-LLM
// page "Kimi K3 work for Rubin (SM107)", Description).  With at most 16 drafts
// the work per (request, head) is ~4 x 16K FMAs against 128 KB of state
// traffic, so the kernel is bound by HBM bandwidth on the state pool.
//
// Organisation: persistent CTAs (two per SM) stream
// (request, head) items.  As soon as an item's state sits in registers, the
// next item's 64 KB state block and draft rows are requested with cp.async, so
// every item's loads overlap the previous item's compute; the updated state
// goes from registers straight to the pool.  Thread (row group rg = lane & 7,
// column group cg = 4*warp + lane / 8) owns the 16 x 4 block of the state at
// key rows 16*rg.., value columns 4*cg..: each staged key-channel value serves
// four columns, and the reductions over key channels (S^T k, S^T q) are 16
// in-thread FMAs per column plus a shuffle reduce-scatter over the row groups
// of the warp (each lane ends with one column's sum; u goes back to all four
// by a gather).  Shared-memory layouts keep every access conflict-free: the
// state's 16-byte chunks are XOR-swizzled by row group, and the staged q, k
// and e^g rows carry 16 bytes of padding after every 128 bytes.
#include "kda_internal.h"
#include "sm103.cuh"

namespace kda {
namespace {

constexpr int kMaxDrafts = 16;
constexpr int kVerifyThreads = 256;
// Staged draft row t (bytes): q bf16 and k bf16 rows of 128, v bf16, e^g fp32,
// the q, k and e^g rows with 16 B of padding after every 128 B (four row groups
// of q / k, two of e^g): row group rg's 16-byte pieces then fall on eight
// distinct bank groups for rg = 0..7.  1360 B per draft keeps two CTAs per SM
// up to 16 drafts with a fp32 pool.
constexpr uint32_t kQRow = 272, kVRow = 256, kERow = 560;
constexpr uint32_t TO_Q = 0, TO_K = kQRow, TO_V = 2 * kQRow, TO_E = 2 * kQRow + kVRow;
constexpr uint32_t kTokBytes = 2 * kQRow + kVRow + kERow;    // 1360
// byte offsets of row group rg in a staged q / k row and in an e^g row
__device__ __forceinline__ uint32_t qk_group(int rg) { return 32u * rg + 16u * (rg >> 2); }
__device__ __forceinline__ uint32_t e_group(int rg) { return 64u * rg + 16u * (rg >> 1); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// Byte offset of 16-byte chunk c of state row r in shared memory (fp32 rows:
// 32 chunks of 4 values; bf16 rows: 16 chunks of 8), XOR-swizzled by the row group.
template <bool kBf16>
__device__ __forceinline__ uint32_t state_chunk(int r, int c) {
    return (uint32_t)r * (kBf16 ? 256u : 512u) + ((uint32_t)(c ^ ((r >> 4) & 7)) << 4);
}
__device__ __forceinline__ float2 bf16x2f(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Column sums over the eight row groups of a warp (lanes rg = 0..7 of one
// column group): a[c] holds this lane's partial sum for column c of its four.
// Reduce-scatter in three shuffle levels (4, 2, 1): the lanes keep half of the
// columns at each level, so lane rg ends with the full sum of column
// ccol(rg) = 2*bit2 + bit1 (4 shuffles instead of the 12 of an all-reduce).  The
// two lanes of a pair (rg, rg^1) add the same two terms, so they hold equal sums.
__device__ __forceinline__ int ccol(int rg) { return (rg >> 1) & 3; }
__device__ __forceinline__ float sum_scatter(const float a[4], int rg) {
    const bool h2 = (rg & 4) != 0, h1 = (rg & 2) != 0;
    const float s0 = __shfl_xor_sync(0xffffffffu, h2 ? a[0] : a[2], 4);
    const float s1 = __shfl_xor_sync(0xffffffffu, h2 ? a[1] : a[3], 4);
    const float c0 = (h2 ? a[2] : a[0]) + s0;  // column 2*h2
    const float c1 = (h2 ? a[3] : a[1]) + s1;  // column 2*h2 + 1
    const float s = __shfl_xor_sync(0xffffffffu, h1 ? c0 : c1, 2);
    float d = (h1 ? c1 : c0) + s;              // column 2*h2 + h1
    d += __shfl_xor_sync(0xffffffffu, d, 1);
    return d;
}
// Inverse of the scatter: lane rg holds x for column ccol(rg); every lane of the
// row-group octet gets all four columns (3 shuffles).
__device__ __forceinline__ void gather4(float x, int rg, float u[4]) {
    const bool h2 = (rg & 4) != 0, h1 = (rg & 2) != 0;
    const float y = __shfl_xor_sync(0xffffffffu, x, 2);
    const float lo = h1 ? y : x, hi = h1 ? x : y;  // columns 2*h2, 2*h2 + 1
    const float lo2 = __shfl_xor_sync(0xffffffffu, lo, 4), hi2 = __shfl_xor_sync(0xffffffffu, hi, 4);
    u[0] = h2 ? lo2 : lo;
    u[1] = h2 ? hi2 : hi;
    u[2] = h2 ? lo : lo2;
    u[3] = h2 ? hi : hi2;
}

struct Item {
    int r, h, slot, acc;
    bool valid;
};

// kBf16: the pool holds bf16 states (read widened to fp32, written back rounded
// to nearest even); otherwise fp32.
template <bool kBf16, bool kStall>
__global__ void __launch_bounds__(kVerifyThreads, 2) verify_kernel(const VerifyParams p) {
    constexpr uint32_t kStateBytes = kHeadDim * kHeadDim * (kBf16 ? 2 : 4);
    extern __shared__ __align__(16) uint8_t smv[];
    __shared__ float s_beta[kMaxDrafts];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = lane & 7, cg = 4 * warp + (lane >> 3);
    const int row0 = 16 * rg, col0 = 4 * cg, cc = ccol(rg);
    const int nitems = p.R * p.H, D = p.D;
    if ((int)blockIdx.x >= nitems) return;
    uint8_t* sst = smv;
    auto tokb = [&](int b) { return smv + kStateBytes + b * D * kTokBytes; };  // draft buffers 0, 1

    auto item_of = [&](int it) -> Item {
        Item x;
        x.r = it / p.H;
        x.h = it - x.r * p.H;
        x.slot = p.slot ? p.slot[x.r] : x.r;
        x.acc = p.accepted[x.r];
        x.valid = x.slot >= 0 && x.slot < p.P && x.acc >= 0 && x.acc <= D;
        return x;
    };
    auto state_of = [&](const Item& x) -> uint8_t* {
        return static_cast<uint8_t*>(p.pool) + ((int64_t)x.slot * p.H + x.h) * (int64_t)kStateBytes;
    };
    auto load_beta = [&](const Item& x) -> float {
        return (tid < D && x.valid) ? p.beta[x.r * p.bs[0] + tid * p.bs[1] + x.h * p.bs[2]] : 0.f;
    };
    // Item x's state block into sst and its draft rows into tb (cp.async, one group).
    auto prefetch = [&](const Item& x, uint8_t* tb) {
        if (x.valid) {
            // Thread tid copies the block's 16-byte chunks tid + 256 j: row r0 + kRows j,
            // chunk c of the row.  r0 < kRows, so the row group (r >> 4) of pass j is
            // j >> 1 (fp32 rows: 8 rows a pass) or j (bf16: 16 rows a pass), a
            // constant of the unrolled pass.
            constexpr int kChunksPerRow = kBf16 ? 16 : 32, kRows = kVerifyThreads / kChunksPerRow;
            const uint8_t* st = state_of(x) + tid * 16;
            const int r0 = tid / kChunksPerRow, c = tid % kChunksPerRow;
            uint8_t* dst = sst + state_chunk<kBf16>(r0, 0);
#pragma unroll
            for (int j = 0; j < kHeadDim / kRows; ++j) {
                const int rgrp = (kBf16 ? j : j >> 1) & 7;
                cp_async16(dst + j * kRows * kChunksPerRow * 16 + ((c ^ rgrp) << 4), st + j * 4096);
            }
            for (int e = tid; e < D * 80; e += kVerifyThreads) {
                const int t = e / 80, j = e - t * 80;
                uint8_t* row = tb + t * kTokBytes;
                if (j < 16) {
                    cp_async16(row + TO_Q + j * 16 + (j >> 3) * 16, p.q + x.r * p.qs[0] + t * p.qs[1] + x.h * p.qs[2] + 8 * j);
                } else if (j < 32) {
                    const int jj = j - 16;
                    cp_async16(row + TO_K + jj * 16 + (jj >> 3) * 16, p.k + x.r * p.ks[0] + t * p.ks[1] + x.h * p.ks[2] + 8 * jj);
                } else if (j < 48) {
                    const int jj = j - 32;
                    cp_async16(row + TO_V + jj * 16, p.v + x.r * p.vs[0] + t * p.vs[1] + x.h * p.vs[2] + 8 * jj);
                } else {
                    const int jj = j - 48;
                    cp_async16(row + TO_E + jj * 16 + (jj >> 3) * 16, p.g + x.r * p.gs[0] + t * p.gs[1] + x.h * p.gs[2] + 4 * jj);
                }
            }
        }
        cp_async_commit();
    };

    int it = blockIdx.x;
    Item cur = item_of(it);
    float bcur = load_beta(cur);
    prefetch(cur, tokb(0));
    Item nxt = it + (int)gridDim.x < nitems ? item_of(it + gridDim.x) : Item{0, 0, 0, 0, false};
    for (int k = 0;; ++k) {
        stall_point<kStall>(p.stall_seed, 1, k);
        cp_async_wait_all();
        __syncthreads();  // this item's state and drafts have landed; the previous item is done
        uint8_t* tb = tokb(k & 1);
        float S[16][4];
        if (cur.valid) {
            for (int e = tid; e < D * kHeadDim; e += kVerifyThreads) {  // e^g in place
                const int t = e >> 7, i = e & (kHeadDim - 1);
                float* ge = reinterpret_cast<float*>(tb + t * kTokBytes + TO_E + i * 4 + (i >> 5) * 16);
                *ge = __expf(*ge);
            }
            if (tid < D) s_beta[tid] = p.beta_is_logit ? 1.0f / (1.0f + __expf(-bcur)) : bcur;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (kBf16) {
                    const uint2 w = *reinterpret_cast<const uint2*>(sst + state_chunk<true>(row0 + i, cg >> 1) +
                                                                    (cg & 1) * 8);
                    const float2 a = bf16x2f(w.x), b = bf16x2f(w.y);
                    S[i][0] = a.x; S[i][1] = a.y; S[i][2] = b.x; S[i][3] = b.y;
                } else {
                    const float4 x = *reinterpret_cast<const float4*>(sst + state_chunk<false>(row0 + i, cg));
                    S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
                }
            }
        } else if (tid == 0 && p.status) {
            atomicExch(p.status, 1);
        }
        stall_point<kStall>(p.stall_seed, 2, k);
        __syncthreads();  // the state block is in registers: its buffer takes the next item
        stall_point<kStall>(p.stall_seed, 3, k);
        prefetch(nxt, tokb((k + 1) & 1));
        const float bnext = load_beta(nxt);
        const int nit = it + gridDim.x;
        const Item after = nit + (int)gridDim.x < nitems ? item_of(nit + gridDim.x) : Item{0, 0, 0, 0, false};
        if (cur.valid) {
            uint8_t* st = state_of(cur);
            // replay-only: run just the accepted drafts; write no output, keep the state
            const int tend = p.replay_only ? cur.acc : D;
            for (int t = 0; t < tend; ++t) {
                const uint8_t* row = tb + t * kTokBytes;
                float kk[16], x[16];
                {
                    const uint4 k0 = *reinterpret_cast<const uint4*>(row + TO_K + qk_group(rg));
                    const uint4 k1 = *reinterpret_cast<const uint4*>(row + TO_K + qk_group(rg) + 16);
                    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float2 f = bf16x2f(kw[w]);
                        kk[2 * w] = f.x; kk[2 * w + 1] = f.y;
                    }
#pragma unroll
                    for (int i = 0; i < 16; i += 4) {
                        const float4 e4 = *reinterpret_cast<const float4*>(row + TO_E + e_group(rg) + 4 * i);
                        x[i] = e4.x; x[i + 1] = e4.y; x[i + 2] = e4.z; x[i + 3] = e4.w;
                    }
                }
                // decay, then u = v - S^T k
                float sk[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 16; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        S[i][c] *= x[i];
                        sk[c] = fmaf(S[i][c], kk[i], sk[c]);
                    }
                // u for this lane's column of the four, then all four to every lane
                const float skc = sum_scatter(sk, rg);
                const float vc = __uint_as_float(
                    (uint32_t)*reinterpret_cast<const uint16_t*>(row + TO_V + 2 * (col0 + cc)) << 16);
                float u[4];
                gather4(s_beta[t] * (vc - skc), rg, u);
                {
                    const uint4 q0 = *reinterpret_cast<const uint4*>(row + TO_Q + qk_group(rg));
                    const uint4 q1 = *reinterpret_cast<const uint4*>(row + TO_Q + qk_group(rg) + 16);
                    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const float2 f = bf16x2f(qw[w]);
                        x[2 * w] = f.x; x[2 * w + 1] = f.y;
                    }
                }
                float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 16; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        S[i][c] = fmaf(kk[i], u[c], S[i][c]);
                        o[c] = fmaf(S[i][c], x[i], o[c]);
                    }
                const float oc = sum_scatter(o, rg);
                if (!(rg & 1) && !p.replay_only)
                    p.out[cur.r * p.os[0] + t * p.os[1] + cur.h * p.os[2] + col0 + cc] =
                        __float2bfloat16_rn(oc * p.scale);
                if (t + 1 == cur.acc) {
                    stall_point<kStall>(p.stall_seed, 4, k);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        if (kBf16)
                            *reinterpret_cast<uint2*>(st + ((row0 + i) * kHeadDim + col0) * 2) =
                                make_uint2(pack_bf16x2(S[i][0], S[i][1]), pack_bf16x2(S[i][2], S[i][3]));
                        else
                            *reinterpret_cast<float4*>(st + ((row0 + i) * kHeadDim + col0) * 4) =
                                make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
                    }
                }
            }
        }
        if (nit >= nitems) break;
        it = nit;
        cur = nxt;
        bcur = bnext;
        nxt = after;
    }
    cp_async_wait_all();  // the last (empty or unused) prefetch group
}

template <bool kBf16, bool kStall>
cudaError_t launch_verify_t(const VerifyParams& p, int num_sms, cudaStream_t s) {
    // the limit is set once per device for the largest draft count
    constexpr size_t kSmemMax = (size_t)kHeadDim * kHeadDim * (kBf16 ? 2 : 4) + 2 * (size_t)kMaxDrafts * kTokBytes;
    static std::atomic<uint64_t> smem_set;
    const size_t smem = (size_t)kHeadDim * kHeadDim * (kBf16 ? 2 : 4) + 2 * (size_t)p.D * kTokBytes;
    cudaError_t e = set_smem_limit_once((const void*)verify_kernel<kBf16, kStall>, (int)kSmemMax, smem_set);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, verify_kernel<kBf16, kStall>, kVerifyThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const long long items = (long long)p.R * p.H;
    const long long cap = (long long)num_sms * per_sm;
    verify_kernel<kBf16, kStall><<<(unsigned)(items < cap ? items : cap), kVerifyThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, int num_sms, cudaStream_t s) {
    if (p.R == 0 || p.H == 0) return cudaSuccess;
    // the instantiations with the stall hook run only when a test asks for them
    if (p.stall_seed)
        return p.pool_bf16 ? launch_verify_t<true, true>(p, num_sms, s) : launch_verify_t<false, true>(p, num_sms, s);
    return p.pool_bf16 ? launch_verify_t<true, false>(p, num_sms, s) : launch_verify_t<false, false>(p, num_sms, s);
}

}  // namespace kda
