// kda_internal.h -- parameters passed from the host API (kda_api.cu) to the
// prefill / verify kernels, and the launchers each kernel file provides.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

struct kda_prefill_args;

namespace kda {

// Every argument check of kda_prefill except the workspace (a kda_status value).
int prefill_check_args(const kda_prefill_args* a);

// Raises a kernel's dynamic shared-memory limit once per device (the attribute
// stays set for the device's context), so that launches after the first skip
// the driver call.  `done` holds one bit per device.
// The device's SM count, read once per device (0 if it cannot be read).
inline int device_sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cached[dev].load(std::memory_order_acquire);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev].store(n, std::memory_order_release);
    return n;
}

inline cudaError_t set_smem_limit_once(const void* kern, int bytes, std::atomic<uint64_t>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

constexpr int kHeadDim = 128;   // K = V = 128
constexpr int kChunk = 64;      // tokens per chunk
constexpr int kSlab = 32;       // value columns per state-pass CTA
constexpr float kGateFloor = -5.4f;   // per-token gate floor inside 16-token blocks (16 * 5.4 < 87)

// Workspace record per (chunk, head): shared-memory images, written by the prep
// kernel with bulk copies and read back by the state pass with bulk copies.
// [Q e^Gam ; W], Kt and Aqk use the 128-byte swizzle of K-major tcgen05
// operands (16-byte chunk c of 128-byte row r at r*128 + ((c ^ (r & 7)) << 4));
// Aqk follows Kt, so that [Kt ; Aqk] is one 192-row operand.  Kt and Aqk are
// fp16 (the operands of the products with V_new, which the state pass forms
// in fp16: 3 more mantissa bits than bf16 where the rounding of V_new reaches
// the output through 64-term sums).  U is stored transposed, U^T: 128 value
// rows of 64 tokens (128 B, the same swizzle), so that a value column's tokens
// are one row (and a 32-column slab's rows are 4 KB of the record).
constexpr uint32_t kRecA1 = 0;          // [Q e^Gam ; W] bf16: 2 column blocks x 128 rows x 128 B
constexpr uint32_t kRecKt = 32768;      // Kt fp16: 128 key rows x 64 tokens
constexpr uint32_t kRecAqk = 49152;     // Aqk fp16: 64 token rows x 64 tokens
constexpr uint32_t kRecU = 57344;       // U^T bf16: 128 value rows x 64 tokens
constexpr uint32_t kRecEg = 73728;      // e^gam fp32 [128]
constexpr uint32_t kRecBytes = 74240;
constexpr uint32_t kSlabImg = 4096;     // bytes of one 32-column slab (U^T rows, or an output image)

// Byte offset of 16-byte chunk c of row r in a U (or output) slab image.
__host__ __device__ __forceinline__ uint32_t slab_chunk_off(uint32_t r, uint32_t c) {
    return r * 64u + ((c ^ ((r >> 1) & 3u)) << 4);
}

struct PrefillParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    __nv_bfloat16* out;
    int64_t qs[3], ks[3], vs[3], gs[3], bs[3], os[3];
    const float* h0;
    float* hT;
    const int32_t* cu;       // device cu_seqlens (varlen) or nullptr (padded)
    int32_t* chunk_off;      // [N+1] in the workspace (varlen)
    int32_t* seq_order;      // [N] in the workspace (varlen): sequences, longest first
    int32_t* status;         // device status word (never null)
    int B, T, N, H;          // T: per-sequence length (padded) or total tokens (varlen)
    int max_chunks;          // chunk records per head (upper bound)
    int beta_is_logit;
    float scale;
    uint8_t* ws_rec;         // kRecBytes per (chunk, head) record, record r = chunk * H + head
    const __nv_bfloat16* gate;   // gated RMSNorm of the output: gate (nullptr = off)
    int64_t gts[3];              // gate strides (batch, token, head)
    const float* norm_w;         // [128]
    float norm_eps;
    uint32_t stall_seed;         // test hook: timing perturbation (stall_point), 0 = off
    int out_tma;                 // 1: the state kernel got a tensor map of out
    uint64_t wait_ns;            // bound of the kernels' working mbarrier waits (kWaitLimitNs
                                 // unless a test lowers it; wind-down waits keep kWaitLimitNs)
    int timeout_probe;           // test: the first product wait of a CTA waits on an
                                 // mbarrier that nothing arrives on (runs out)
    // Segment-parallel scan of padded calls (whole-chain state kernel only):
    int scan_mode;               // kScanOff, kScanOps or kScanOut
    int scan_chunks;             // chunks per segment
    int scan_nseg;               // segments per chain
    float* scan_ops;             // [(nseg - 1) * 2][B * H] fp32 128 x 128 blocks: M_s, C_s
    float* scan_entry;           // [nseg][B * H] fp32 128 x 128 blocks: E_s (s >= 1 used)
    int32_t* rec_counter;        // prep: records are taken from this counter (starting at 0)
                                 // by every grid given it; nullptr: CTA b takes b, b + grid, ...
    int rec_prefetch;            // whole-chain state kernel: chunks between a record's L2
                                 // prefetch and its bulk copy (0: none); set by its launcher
};

// Modes of the whole-chain state kernel.
//  kScanOff: one pass over each chain (blockIdx.y = sequence).
//  kScanOps: blockIdx.y = (2 s + w) N + n, segment s < nseg - 1: w = 0 its
//            transition M_s (entry = identity, U read as zero), w = 1 its
//            offset C_s (entry = zero); no outputs; the state after the
//            segment goes to scan_ops.
//  kScanOut: blockIdx.y = s N + n: segment s from its entry state (the initial
//            state for s = 0, else scan_entry) with outputs; the last segment
//            stores the final state.
constexpr int kScanOff = 0, kScanOps = 1, kScanOut = 2;
constexpr int kScanMaxSegments = 32;

// Chunk c (global index) -> sequence, token start and length.
struct ChunkInfo {
    int n;        // sequence
    int b;        // batch coordinate used for addressing (padded: n, varlen: 0)
    int t0;       // first token (padded: within the sequence; varlen: packed index)
    int len;      // valid tokens, 1..64 (0 = no such chunk)
    int local;    // chunk index within the sequence
};

__device__ __forceinline__ ChunkInfo chunk_info(const PrefillParams& p, int c) {
    ChunkInfo ci{0, 0, 0, 0, 0};
    if (p.cu == nullptr) {
        const int cps = (p.T + kChunk - 1) / kChunk;
        if (cps == 0 || c >= p.B * cps) return ci;
        ci.n = c / cps;
        ci.b = ci.n;
        ci.local = c - ci.n * cps;
        ci.t0 = ci.local * kChunk;
        ci.len = min(kChunk, p.T - ci.t0);
    } else {
        if (c >= p.chunk_off[p.N]) return ci;
        int lo = 0, hi = p.N;  // find n with chunk_off[n] <= c < chunk_off[n+1]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.chunk_off[mid] <= c) lo = mid; else hi = mid;
        }
        ci.n = lo;
        ci.b = 0;
        ci.local = c - p.chunk_off[lo];
        ci.t0 = p.cu[lo] + ci.local * kChunk;
        ci.len = min(kChunk, p.cu[lo + 1] - ci.t0);
    }
    return ci;
}

// TMA descriptors of the inputs q, k, v (bf16) and g (fp32), each viewed as a
// 4-D tensor [channel 128, head H, token T, batch B] with the caller's strides;
// one box is one chunk of one head: [128, 1, 64, 1].
struct PrepMaps {
    CUtensorMap q, k, v, g;
};

cudaError_t launch_chunk_table(const PrefillParams& p, cudaStream_t s);
// overlap_previous: launched programmatically after another prep grid in the
// same stream (the two may overlap; they must touch disjoint records).
// grid: CTAs (at most one per SM and per record).
cudaError_t launch_prep(const PrefillParams& p, const PrepMaps& maps, int grid, cudaStream_t s,
                        bool overlap_previous = false);
// out_map: tensor map of out, [channel 128, head, token, batch] with a box of
// [32, 1, 64, 1] and the 64-byte swizzle (used when p.out_tma is set).
// after_prep: launched programmatically right after a prep grid in the same
// stream (the state pass's set-up overlaps prep's tail; it waits for prep's
// completion before it reads a record).
cudaError_t launch_state(const PrefillParams& p, const CUtensorMap& out_map, cudaStream_t s,
                         bool after_prep = false);
cudaError_t launch_state_head(const PrefillParams& p, const CUtensorMap& out_map, cudaStream_t s,
                              bool after_prep = false);
// Launches `kern` with the programmatic-serialization attribute when `pdl`.
template <typename... Args>
cudaError_t launch_maybe_pdl(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             bool pdl, Args... args) {
    if (!pdl) {
        kern<<<grid, block, smem, s>>>(args...);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}
// Entry states of the scan: E_{s+1} = M_s E_s + C_s (E_0 = p.h0 or zero) for
// every chain, in fp32 with a fixed summation order.
cudaError_t launch_scan_combine(const PrefillParams& p, cudaStream_t s);

struct VerifyParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const float* beta;
    __nv_bfloat16* out;
    int64_t qs[3], ks[3], vs[3], gs[3], bs[3], os[3];
    void* pool;              // fp32 or bf16 [P, H, 128, 128]
    const int32_t* slot;
    const int32_t* accepted;
    int32_t* status;         // may be null
    int R, D, H, P;
    int beta_is_logit;
    float scale;
    int pool_bf16;           // 1: the pool holds bf16 states
    int replay_only;         // 1: run the accepted drafts only, store the state, no outputs
    uint32_t stall_seed;     // test hook: timing perturbation (stall_point), 0 = off
    uint64_t wait_ns;        // bound of the tensor-core kernel's product waits
    int timeout_probe;       // test: the first product wait runs out (see PrefillParams)
};

// Sequential kernel (every draft on the CUDA cores, fp32).
cudaError_t launch_verify(const VerifyParams& p, int num_sms, cudaStream_t s);
// Tensor-core kernel (the drafts as one WY-form chunk, tf32 products).
cudaError_t launch_verify_wy(const VerifyParams& p, int num_sms, cudaStream_t s);

}  // namespace kda
