// kda_verify.cu -- MTP verify: a short draft chunk per request run against a
// fp32 state pool, with the state after the accepted prefix written back.
//
// The drafts of one request form one short chunk of the KDA recurrence (the
// tcgen05 KDA MTP verify kernel and its replay-only commit on the TensorRT-LLM
// page "Kimi K3 work for Rubin (SM107)", Description).  With at most 16 drafts
// the work per (request, head) is ~4 x 16K FMAs against 128 KB of state
// traffic, so the kernel is bound by HBM bandwidth on the state pool; it runs
// the drafts sequentially on CUDA cores with the state column of each thread
// in registers, which also yields the per-draft outputs directly.
//
// Layout: one CTA per (head, request), 256 threads.  Every draft's q, k, e^g,
// v and beta are staged in shared memory in the same pass as the state load.
// Thread (row group rg = lane & 7, column group cg = 4*warp + lane / 8) owns the
// 16 x 4 block of the state at key rows 16*rg.., value columns 4*cg..: each
// staged key-channel value it reads from shared memory serves four columns,
// and the reductions over key channels (S^T k, S^T q) are 16 in-thread FMAs per
// column plus three shuffle levels over the row groups of the warp.  The
// staged rows are padded by 16 bytes every 16 floats, so the eight row groups
// of a warp read eight different bank quads.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kMaxDrafts = 16;
constexpr int kPadRow = kHeadDim + kHeadDim / 4;   // 160 floats: 16 B of padding per 16 floats
__device__ __forceinline__ int padded(int i) { return i + (i >> 4) * 4; }

__global__ void __launch_bounds__(256, 2)
    verify_kernel(const VerifyParams p) {
    const int h = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int rg = lane & 7, cg = 4 * warp + (lane >> 3);
    const int row0 = 16 * rg, col0 = 4 * cg;
    __shared__ __align__(16) float s_e[kMaxDrafts][kPadRow];
    __shared__ __align__(16) float s_k[kMaxDrafts][kPadRow];
    __shared__ __align__(16) float s_q[kMaxDrafts][kPadRow];
    __shared__ __align__(16) float s_v[kMaxDrafts][kHeadDim];
    __shared__ float s_beta[kMaxDrafts];

    const int slot = p.slot ? p.slot[r] : r;
    const int acc = p.accepted[r];
    if (slot < 0 || slot >= p.P || acc < 0 || acc > p.D) {
        if (tid == 0 && p.status) atomicExch(p.status, 1);
        return;
    }
    float* st = p.pool + ((int64_t)slot * p.H + h) * (kHeadDim * kHeadDim);
    float S[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(st + (row0 + i) * kHeadDim + col0);
        S[i][0] = x.x; S[i][1] = x.y; S[i][2] = x.z; S[i][3] = x.w;
    }
    for (int e = tid; e < p.D * kHeadDim; e += blockDim.x) {
        const int t = e >> 7, i = e & (kHeadDim - 1), pi = padded(i);
        s_q[t][pi] = __bfloat162float(p.q[r * p.qs[0] + t * p.qs[1] + h * p.qs[2] + i]) * p.scale;
        s_k[t][pi] = __bfloat162float(p.k[r * p.ks[0] + t * p.ks[1] + h * p.ks[2] + i]);
        s_e[t][pi] = __expf(p.g[r * p.gs[0] + t * p.gs[1] + h * p.gs[2] + i]);
        s_v[t][i] = __bfloat162float(p.v[r * p.vs[0] + t * p.vs[1] + h * p.vs[2] + i]);
    }
    if (tid < p.D) {
        const float bb = p.beta[r * p.bs[0] + tid * p.bs[1] + h * p.bs[2]];
        s_beta[tid] = p.beta_is_logit ? 1.0f / (1.0f + __expf(-bb)) : bb;
    }
    __syncthreads();

    const int prow = padded(row0);  // the 16 rows of a group are contiguous after padding
    for (int t = 0; t < p.D; ++t) {
        float kk[16], x[16];
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 e4 = *reinterpret_cast<const float4*>(&s_e[t][prow + i]);
            const float4 k4 = *reinterpret_cast<const float4*>(&s_k[t][prow + i]);
            x[i] = e4.x; x[i + 1] = e4.y; x[i + 2] = e4.z; x[i + 3] = e4.w;
            kk[i] = k4.x; kk[i + 1] = k4.y; kk[i + 2] = k4.z; kk[i + 3] = k4.w;
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
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            sk[c] += __shfl_xor_sync(0xffffffffu, sk[c], 1);
            sk[c] += __shfl_xor_sync(0xffffffffu, sk[c], 2);
            sk[c] += __shfl_xor_sync(0xffffffffu, sk[c], 4);
        }
        const float4 v4 = *reinterpret_cast<const float4*>(&s_v[t][col0]);
        const float bt = s_beta[t];
        const float u[4] = {bt * (v4.x - sk[0]), bt * (v4.y - sk[1]), bt * (v4.z - sk[2]), bt * (v4.w - sk[3])};
#pragma unroll
        for (int i = 0; i < 16; i += 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(&s_q[t][prow + i]);
            x[i] = q4.x; x[i + 1] = q4.y; x[i + 2] = q4.z; x[i + 3] = q4.w;
        }
        float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                S[i][c] = fmaf(kk[i], u[c], S[i][c]);
                o[c] = fmaf(S[i][c], x[i], o[c]);
            }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            o[c] += __shfl_xor_sync(0xffffffffu, o[c], 1);
            o[c] += __shfl_xor_sync(0xffffffffu, o[c], 2);
            o[c] += __shfl_xor_sync(0xffffffffu, o[c], 4);
        }
        if (rg < 4) {
            const float oc = rg == 0 ? o[0] : rg == 1 ? o[1] : rg == 2 ? o[2] : o[3];
            p.out[r * p.os[0] + t * p.os[1] + h * p.os[2] + col0 + rg] = __float2bfloat16_rn(oc);
        }
        if (t + 1 == acc) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                *reinterpret_cast<float4*>(st + (row0 + i) * kHeadDim + col0) =
                    make_float4(S[i][0], S[i][1], S[i][2], S[i][3]);
        }
    }
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t s) {
    if (p.R == 0 || p.H == 0) return cudaSuccess;
    dim3 grid(p.H, p.R);
    verify_kernel<<<grid, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kda
