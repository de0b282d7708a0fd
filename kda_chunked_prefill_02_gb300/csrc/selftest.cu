// selftest.cu -- test-only checks of the sm_103a building blocks in sm103.cuh:
// a single-tile tcgen05 GEMM D = A * B^T (A 128 x 128, B N x 128, bf16, fp32
// accumulation in TMEM) with the operands staged either by threads writing the
// 128-byte-swizzled K-major layout themselves or by TMA with the 128-byte
// swizzle.  Built into its own library (libkda_selftest.so); the product
// library does not contain it.
#include <cuda_runtime.h>

#include "sm103.cuh"
#include "tmap.h"

using namespace kda;

namespace {

__global__ void __launch_bounds__(128)
    umma_selftest_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                         float* __restrict__ D, int N, int use_tma,
                         const __grid_constant__ CUtensorMap map_a,
                         const __grid_constant__ CUtensorMap map_b, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;          // 2 column blocks x 128 rows x 128 B
    uint8_t* sB = smem + 32768;  // 2 column blocks x N rows x 128 B
    __shared__ uint64_t bar_mma, bar_tma;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_tma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (!use_tma) {
        for (int i = tid; i < 128 * 128; i += 128) {
            const int r = i >> 7, c = i & 127;
            *reinterpret_cast<__nv_bfloat16*>(sA + (c >> 6) * 16384 + sw128_off(r, c & 63)) = A[i];
        }
        for (int i = tid; i < N * 128; i += 128) {
            const int r = i >> 7, c = i & 127;
            *reinterpret_cast<__nv_bfloat16*>(sB + (c >> 6) * (N * 128) + sw128_off(r, c & 63)) =
                B[i];
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    bool ok = true;
    if (use_tma) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&bar_tma, (128 + N) * 256);
            for (int kb = 0; kb < 2; ++kb) {
                tma_load_2d(sA + kb * 16384, &map_a, kb * 64, 0, &bar_tma);
                tma_load_2d(sB + kb * N * 128, &map_b, kb * 64, 0, &bar_tma);
            }
        }
        ok = mbar_wait(&bar_tma, 0, nullptr);
    }
    if (tid == 0 && ok) {
        umma_tile(tmem_base, smem_u32(sA), 16384, smem_u32(sB), N * 128, 128,
                  idesc_bf16_f32(128, N), false);
        umma_commit(&bar_mma);
    }
    if (ok) ok = mbar_wait(&bar_mma, 0, nullptr);
    if (!ok) atomicExch(status, 4);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem_addr(tmem_base, warp * 32, c0), v);
            const int row = warp * 32 + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, 256);
}

// D = A B^T with B stored MN-major (B^T as [K rows][N contiguous]); mode bit 0
// clear uses lbo = 1024 (atoms along N adjacent) and sbo = N/64 * 1024, set
// swaps them; mode bit 1 takes A and B as fp16 (copied as 16-bit patterns);
// mode bit 2 stores A MN-major as well (A^T as [K rows][M contiguous]: two
// 64-row atoms 1024 B apart, 8-row K groups 2048 B apart).
__global__ void __launch_bounds__(128)
    umma_mn_selftest_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                            float* __restrict__ D, int N, int mode, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + 32768;
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbo = (uint32_t)(N >= 64 ? N / 64 : 1) * 1024u;
    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    const bool a_mn = (mode & 4) != 0;
    for (int i = tid; i < 128 * 128; i += 128) {
        const int r = i >> 7, c = i & 127;
        if (a_mn)
            *reinterpret_cast<__nv_bfloat16*>(sA + mn_sw128_off(c, r, 2048u)) = A[i];
        else
            *reinterpret_cast<__nv_bfloat16*>(sA + (c >> 6) * 16384 + sw128_off(r, c & 63)) = A[i];
    }
    for (int i = tid; i < N * 128; i += 128) {  // B[n][k] -> MN-major (k, n)
        const int n = i >> 7, k = i & 127;
        *reinterpret_cast<__nv_bfloat16*>(sB + mn_sw128_off(k, n, sbo)) = B[i];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        // mode bit 0: atoms and 8-row groups swapped; bit 1: fp16 operands
        const uint32_t lbo = (mode & 1) == 0 ? 1024u : sbo, sb = (mode & 1) == 0 ? sbo : 1024u;
        const uint32_t id = ((mode & 2) ? idesc_f16_f32_bmn(128, N) : idesc_bf16_f32_bmn(128, N)) |
                            (a_mn ? (1u << 15) : 0u);
        for (int k = 0; k < 8; ++k) {
            const uint32_t kb = k >> 2, kin = (k & 3u) * 32u;
            const uint64_t ad = a_mn ? sdesc_mnmajor_sw128(smem_u32(sA) + (uint32_t)k * 2u * 2048u, 1024u, 2048u)
                                     : sdesc_kmajor_sw128(smem_u32(sA) + kb * 16384 + kin);
            umma_bf16(tmem_base, ad, sdesc_mnmajor_sw128(smem_u32(sB) + (uint32_t)k * 2u * sbo, lbo, sb), id,
                      k > 0 ? 1u : 0u);
        }
        umma_commit(&bar_mma);
    }
    const bool ok = mbar_wait(&bar_mma, 0, nullptr);
    if (!ok) atomicExch(status, 4);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem_addr(tmem_base, warp * 32, c0), v);
            const int row = warp * 32 + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, 256);
}

// D = A B^T, N = 32, with B stored MN-major in the 64-byte swizzle
// (element (k, n) at k*64 + (((n/8) ^ ((k/2) % 4)) * 16) + (n%8)*2; 8-row
// groups 512 B apart).
__global__ void __launch_bounds__(128)
    umma_mn64_selftest_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                              float* __restrict__ D, int* status) {
    constexpr int N = 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + 32768;  // 128 K rows x 64 B = 8 KB
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 32);
        tmem_relinquish();
    }
    for (int i = tid; i < 128 * 128; i += 128) {
        const int r = i >> 7, c = i & 127;
        *reinterpret_cast<__nv_bfloat16*>(sA + (c >> 6) * 16384 + sw128_off(r, c & 63)) = A[i];
    }
    for (int i = tid; i < N * 128; i += 128) {  // B[n][k] -> (k, n)
        const int n = i >> 7, k = i & 127;
        *reinterpret_cast<__nv_bfloat16*>(sB + k * 64 + ((((n >> 3) ^ ((k >> 1) & 3))) << 4) + (n & 7) * 2) = B[i];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        for (int k = 0; k < 8; ++k) {
            const uint32_t kb = k >> 2, kin = (k & 3u) * 32u;
            umma_bf16(tmem_base, sdesc_kmajor_sw128(smem_u32(sA) + kb * 16384 + kin),
                      sdesc_mnmajor_sw64(smem_u32(sB) + (uint32_t)k * 1024u, 512u, 512u),
                      idesc_bf16_f32_bmn(128, N), k > 0 ? 1u : 0u);
        }
        umma_commit(&bar_mma);
    }
    const bool ok = mbar_wait(&bar_mma, 0, nullptr);
    if (!ok) atomicExch(status, 4);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem_addr(tmem_base, warp * 32, c0), v);
            const int row = warp * 32 + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, 32);
}

// D = A B^T with A (128 x 128) held in TMEM (written by the threads with
// tcgen05.st, row m in lane m) and B (N x 128) K-major SW128 in shared memory;
// bf16 or (f16 != 0) fp16 operands, copied as 16-bit patterns.
__global__ void __launch_bounds__(128)
    umma_tmem_a_selftest_kernel(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                                float* __restrict__ D, int N, int f16, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sB = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr uint32_t kACol = 256;  // A occupies columns 256..319, D columns 0..N-1
    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    for (int i = tid; i < N * 128; i += 128) {
        const int r = i >> 7, c = i & 127;
        *reinterpret_cast<__nv_bfloat16*>(sB + (c >> 6) * (N * 128) + sw128_off(r, c & 63)) = B[i];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    {
        const int row = warp * 32 + lane;
        const uint32_t* src = reinterpret_cast<const uint32_t*>(A + row * 128);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t w[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) w[x] = src[16 * j + x];
            tmem_st16(tmem_addr(tb, warp * 32, kACol + 16 * j), w);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sB));
        const uint32_t id = f16 ? idesc_f16_f32(128, N) : idesc_bf16_f32(128, N);
        for (uint32_t k = 0; k < 8; ++k)
            umma_bf16_ta(tb, tb + kACol + 8 * k, bd + (k >> 2) * ((uint32_t)(N * 128) >> 4) + (k & 3) * 2, id,
                         k > 0 ? 1u : 0u);
        umma_commit(&bar_mma);
    }
    const bool ok = mbar_wait(&bar_mma, 0, nullptr);
    if (!ok) atomicExch(status, 4);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem_addr(tb, warp * 32, c0), v);
            const int row = warp * 32 + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// D = A B^T on the tensor cores in tf32 (kind::tf32, fp32 accumulation): A is
// 128 x K and B is N x K fp32 (K a multiple of 8, at most 128; N at most 128),
// each staged K-major (32-wide K blocks of 128-byte rows) or MN-major (per K
// index a 128-byte row of 32 M / N elements, 8-row K groups 1 KB apart,
// 32-wide M / N blocks K/8 KB apart): the operand forms of the tensor-core
// verify kernel.
__global__ void __launch_bounds__(128)
    umma_tf32_selftest_kernel(const float* __restrict__ A, const float* __restrict__ B, float* __restrict__ D,
                              int N, int K, int a_mn, int b_mn, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sA = smem;            // 128 x K fp32
    uint8_t* sB = smem + 65536;    // N x K fp32
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t lbo = (uint32_t)(K / 8) * 1024u;
    if (tid == 0) {
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    // a_mn == 2: A from TMEM, columns 128 .. 128 + K - 1, row m in lane m
    __syncthreads();
    if (a_mn == 2) {
        const int row = warp * 32 + lane;
        for (int c0 = 0; c0 < K; c0 += 16) {
            uint32_t w[16];
#pragma unroll
            for (int x = 0; x < 16; ++x) w[x] = __float_as_uint(A[row * K + c0 + x]);
            tmem_st16(tmem_addr(tmem_base, warp * 32, 128 + c0), w);
        }
    }
    for (int i = tid; i < 128 * K; i += 128) {
        const int m = i / K, k = i % K;
        const uint32_t off = a_mn ? f32_mnmajor_off(m, k, lbo, 1024u) : f32_kmajor_off(m, k, 128u * 128u);
        *reinterpret_cast<float*>(sA + off) = A[i];
    }
    for (int i = tid; i < N * K; i += 128) {
        const int n = i / K, k = i % K;
        const uint32_t off = b_mn ? f32_mnmajor_off(n, k, lbo, 1024u) : f32_kmajor_off(n, k, (uint32_t)N * 128u);
        *reinterpret_cast<float*>(sB + off) = B[i];
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
        const uint32_t a = smem_u32(sA), b = smem_u32(sB);
        const uint32_t id = idesc_tf32_f32(128, N, a_mn == 1, b_mn != 0);
        for (int st = 0; st < K / 8; ++st) {
            const uint64_t ad = a_mn ? sdesc_mnmajor_sw128(a + st * 1024u, lbo, 1024u)
                                     : sdesc_kmajor_sw128(a + (st >> 2) * 16384u + (st & 3) * 32u);
            const uint64_t bd = b_mn ? sdesc_mnmajor_sw128(b + st * 1024u, lbo, 1024u)
                                     : sdesc_kmajor_sw128(b + (st >> 2) * (uint32_t)N * 128u + (st & 3) * 32u);
            if (a_mn == 2)
                umma_tf32_ta(tmem_base, tmem_base + 128 + 8 * st, bd, id, st > 0 ? 1u : 0u);
            else
                umma_tf32(tmem_base, ad, bd, id, st > 0 ? 1u : 0u);
        }
        umma_commit(&bar_mma);
    }
    const bool ok = mbar_wait(&bar_mma, 0, nullptr);
    if (!ok) atomicExch(status, 4);
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem_addr(tmem_base, warp * 32, c0), v);
            const int row = warp * 32 + lane;
#pragma unroll
            for (int i = 0; i < 16; ++i) D[row * N + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, 256);
}

// Throughput of back-to-back MMAs of one shape (operands are zeros: only the
// time matters).  mode: 0 A smem / B MN-major SW128 N=32; 1 A TMEM / B MN-major
// SW128 N=32; 2 A smem / B MN-major SW128 N=128 with 64-column atoms 16 KB
// apart; 3 A smem / B MN-major SW64 N=32; 4 A smem / B K-major N=256;
// 5 A smem / B K-major N=32; 6 A smem / B MN-major SW128 N=64; 7 as 5 with D
// alternating between two TMEM tiles; 8 as 5 with M = 64; 9 as 5 with N = 16.
__global__ void __launch_bounds__(128)
    mma_rate_kernel(int mode, int reps, long long* cycles, int* status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
    __shared__ uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid >> 5;
    for (int i = tid; i < 49152 / 16; i += 128) reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    if (tid == 0) {
        const uint32_t a = smem_u32(sm), bsm = smem_u32(sm + 16384);
        const uint64_t ad = sdesc_kmajor_sw128(a);
        uint64_t bd;
        uint32_t id;
        switch (mode) {
            case 0: case 1: bd = sdesc_mnmajor_sw128(bsm, 1024u, 1024u); id = idesc_bf16_f32_bmn(128, 32); break;
            case 2: bd = sdesc_mnmajor_sw128(bsm, 16384u, 1024u); id = idesc_bf16_f32_bmn(128, 128); break;
            case 3: bd = sdesc_mnmajor_sw64(bsm, 512u, 512u); id = idesc_bf16_f32_bmn(128, 32); break;
            case 4: bd = sdesc_kmajor_sw128(bsm); id = idesc_bf16_f32(128, 256); break;
            case 5: bd = sdesc_kmajor_sw128(bsm); id = idesc_bf16_f32(128, 32); break;
            case 6: bd = sdesc_mnmajor_sw128(bsm, 1024u, 2048u); id = idesc_bf16_f32_bmn(128, 64); break;
            case 8: bd = sdesc_kmajor_sw128(bsm); id = idesc_bf16_f32(64, 32); break;
            case 9: bd = sdesc_kmajor_sw128(bsm); id = idesc_bf16_f32(128, 16); break;
            default: bd = sdesc_kmajor_sw128(bsm); id = idesc_bf16_f32(128, 32); break;
        }
        tc_fence_after();
        const long long t0 = clock64();
        for (int r = 0; r < reps; ++r) {
            if (mode == 1) umma_bf16_ta(tb, tb + 256, bd, id, r > 0 ? 1u : 0u);
            else if (mode == 7) umma_bf16(tb + 64 * (r & 1), ad, bd, id, r > 1 ? 1u : 0u);
            else umma_bf16(tb, ad, bd, id, r > 0 ? 1u : 0u);
        }
        const long long t1 = clock64();
        umma_commit(&bar);
        const bool ok = mbar_wait(&bar, 0, nullptr);
        const long long t2 = clock64();
        if (!ok) atomicExch(status, 4);
        cycles[0] = t1 - t0;  // issue
        cycles[1] = t2 - t0;  // issue + completion
    } else if (warp == 0) {
        // nothing: warp 0's other lanes wait at the barrier
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// to_tf32 (integer round to nearest, ties away from zero) beside the
// conversion instruction, element by element, as bit patterns.
__global__ void tf32_round_selftest_kernel(const float* __restrict__ x, uint32_t* __restrict__ fast,
                                           uint32_t* __restrict__ ref, int n) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const float v = x[i];
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    fast[i] = __float_as_uint(to_tf32(v));
    ref[i] = r;
}

}  // namespace

extern "C" int kda_selftest_umma_tf32(const float* A, const float* B, float* D, int N, int K, int a_mn,
                                      int b_mn, int* status, void* stream) {
    if (N < 16 || N > 128 || (N % 16) != 0 || K < 8 || K > 128 || (K % 8) != 0) return 1;
    if ((a_mn || b_mn) && (K % 8) != 0) return 1;
    if (!a_mn && (K % 32) != 0 && K > 32) return 1;   // K-major: whole 32-wide blocks beyond the first
    const size_t smem = 1024 + 65536 + 65536;
    if (cudaFuncSetAttribute(umma_tf32_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 3;
    umma_tf32_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(A, B, D, N, K, a_mn, b_mn, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_selftest_umma_tmem_a_typed(const void* A, const void* B, float* D, int N, int f16,
                                              int* status, void* stream) {
    if (N < 16 || N > 256 || (N % 16) != 0) return 1;
    const size_t smem = 1024 + 2 * (size_t)N * 128;
    if (cudaFuncSetAttribute(umma_tmem_a_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 3;
    umma_tmem_a_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, D, N, f16 ? 1 : 0, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_selftest_umma_tmem_a(const void* A, const void* B, float* D, int N, int* status,
                                        void* stream) {
    return kda_selftest_umma_tmem_a_typed(A, B, D, N, 0, status, stream);
}

extern "C" int kda_selftest_umma_mn64(const void* A, const void* B, float* D, int* status,
                                      void* stream) {
    const size_t smem = 1024 + 32768 + 8192;
    if (cudaFuncSetAttribute(umma_mn64_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 3;
    umma_mn64_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, D, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_selftest_umma_mn(const void* A, const void* B, float* D, int N, int mode,
                                    int* status, void* stream) {
    if (!(N == 32 || (N >= 64 && N <= 256 && N % 64 == 0))) return 1;
    const size_t smem = 1024 + 32768 + (N >= 64 ? 2 * (size_t)N * 128 : 16384);
    if (cudaFuncSetAttribute(umma_mn_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 3;
    umma_mn_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, D, N, mode, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_selftest_umma(const void* A, const void* B, float* D, int N, int use_tma,
                                 int* status, void* stream) {
    if (N < 16 || N > 256 || (N % 16) != 0) return 1;
    CUtensorMap ma{}, mb{};
    if (use_tma) {
        const uint64_t dims_a[2] = {128, 128}, dims_b[2] = {128, (uint64_t)N};
        const uint64_t strides[1] = {256};
        const uint32_t box_a[2] = {64, 128}, box_b[2] = {64, (uint32_t)N};
        if (!make_tensor_map(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims_a, strides, box_a,
                             CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tensor_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims_b, strides, box_b,
                             CU_TENSOR_MAP_SWIZZLE_128B))
            return 3;
    }
    const size_t smem = 1024 + 32768 + 2 * (size_t)N * 128;
    if (cudaFuncSetAttribute(umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return 3;
    umma_selftest_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)A, (const __nv_bfloat16*)B, D, N, use_tma, ma, mb, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_selftest_tf32_round(const float* x, uint32_t* fast, uint32_t* ref, int n,
                                       void* stream) {
    if (n < 1) return 1;
    tf32_round_selftest_kernel<<<(n + 255) / 256, 256, 0, (cudaStream_t)stream>>>(x, fast, ref, n);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}

extern "C" int kda_selftest_mma_rate(int mode, int reps, long long* cycles, int* status, void* stream) {
    if (mode < 0 || mode > 9 || reps < 1 || reps > 4096) return 1;
    const size_t smem = 1024 + 49152;
    if (cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 3;
    mma_rate_kernel<<<1, 128, smem, (cudaStream_t)stream>>>(mode, reps, cycles, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
