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
// Layout: one CTA per (head, request), 256 threads; the drafts' q, k, e^g, v
// and beta are staged in shared memory in the same pass as the state load;
// lanes 2m and 2m+1 of a warp
// own value column j = 16*warp + m, split over key rows [0,64) and [64,128), so
// the reductions over key channels (S^T k, S^T q) are 64 in-thread FMAs plus one
// lane-pair shuffle, and every pool row is read and written in 64-byte runs.
#include "kda_internal.h"

namespace kda {
namespace {

constexpr int kRows = kHeadDim / 2;
constexpr int kMaxDrafts = 16;

__global__ void __launch_bounds__(256, 2)
    verify_kernel(const VerifyParams p) {
    const int h = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int j = 16 * warp + (lane >> 1), half = lane & 1, r0 = half * kRows;
    // Every draft's inputs, loaded once together with the state so that the
    // request pays one memory latency, not one per draft.
    __shared__ __align__(16) float s_k[kMaxDrafts][kHeadDim];
    __shared__ __align__(16) float s_q[kMaxDrafts][kHeadDim];
    __shared__ __align__(16) float s_e[kMaxDrafts][kHeadDim];
    __shared__ __align__(16) float s_v[kMaxDrafts][kHeadDim];
    __shared__ float s_beta[kMaxDrafts];

    const int slot = p.slot ? p.slot[r] : r;
    const int acc = p.accepted[r];
    if (slot < 0 || slot >= p.P || acc < 0 || acc > p.D) {
        if (tid == 0 && p.status) atomicExch(p.status, 1);
        return;
    }
    float* st = p.pool + ((int64_t)slot * p.H + h) * (kHeadDim * kHeadDim);
    float S[kRows];
#pragma unroll
    for (int c = 0; c < kRows; ++c) S[c] = st[(r0 + c) * kHeadDim + j];
    for (int e = tid; e < p.D * kHeadDim; e += blockDim.x) {
        const int t = e >> 7, i = e & (kHeadDim - 1);
        s_q[t][i] = __bfloat162float(p.q[r * p.qs[0] + t * p.qs[1] + h * p.qs[2] + i]) * p.scale;
        s_k[t][i] = __bfloat162float(p.k[r * p.ks[0] + t * p.ks[1] + h * p.ks[2] + i]);
        s_e[t][i] = __expf(p.g[r * p.gs[0] + t * p.gs[1] + h * p.gs[2] + i]);
        s_v[t][i] = __bfloat162float(p.v[r * p.vs[0] + t * p.vs[1] + h * p.vs[2] + i]);
    }
    if (tid < p.D) {
        const float bb = p.beta[r * p.bs[0] + tid * p.bs[1] + h * p.bs[2]];
        s_beta[tid] = p.beta_is_logit ? 1.0f / (1.0f + __expf(-bb)) : bb;
    }
    __syncthreads();

    for (int t = 0; t < p.D; ++t) {
        // decay, then u = v - S^T k (four partial sums, then the lane pair)
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int c = 0; c < kRows; c += 4) {
            const float4 e = *reinterpret_cast<const float4*>(&s_e[t][r0 + c]);
            const float4 kk = *reinterpret_cast<const float4*>(&s_k[t][r0 + c]);
            S[c] *= e.x; S[c + 1] *= e.y; S[c + 2] *= e.z; S[c + 3] *= e.w;
            a0 = fmaf(S[c], kk.x, a0);
            a1 = fmaf(S[c + 1], kk.y, a1);
            a2 = fmaf(S[c + 2], kk.z, a2);
            a3 = fmaf(S[c + 3], kk.w, a3);
        }
        float sk = (a0 + a1) + (a2 + a3);
        sk += __shfl_xor_sync(0xffffffffu, sk, 1);
        const float bu = s_beta[t] * (s_v[t][j] - sk);
        float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
        for (int c = 0; c < kRows; c += 4) {
            const float4 kk = *reinterpret_cast<const float4*>(&s_k[t][r0 + c]);
            const float4 qq = *reinterpret_cast<const float4*>(&s_q[t][r0 + c]);
            S[c] = fmaf(kk.x, bu, S[c]);
            S[c + 1] = fmaf(kk.y, bu, S[c + 1]);
            S[c + 2] = fmaf(kk.z, bu, S[c + 2]);
            S[c + 3] = fmaf(kk.w, bu, S[c + 3]);
            o0 = fmaf(S[c], qq.x, o0);
            o1 = fmaf(S[c + 1], qq.y, o1);
            o2 = fmaf(S[c + 2], qq.z, o2);
            o3 = fmaf(S[c + 3], qq.w, o3);
        }
        float o = (o0 + o1) + (o2 + o3);
        o += __shfl_xor_sync(0xffffffffu, o, 1);
        if (half == 0) p.out[r * p.os[0] + t * p.os[1] + h * p.os[2] + j] = __float2bfloat16_rn(o);
        if (t + 1 == acc) {
#pragma unroll
            for (int c = 0; c < kRows; ++c) st[(r0 + c) * kHeadDim + j] = S[c];
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
