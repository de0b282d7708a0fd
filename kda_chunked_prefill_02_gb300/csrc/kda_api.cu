// kda_api.cu -- the C ABI of include/kda.h: host-side argument checks, the
// workspace plan, TMA descriptors and the kernel launches.  Nothing here
// allocates or caches device memory.
#include <stdlib.h>
#include <string.h>

#include "../../include/kda.h"
#include "kda_internal.h"
#include "tmap.h"

using namespace kda;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Upper bound on chunk records per head.
int64_t max_chunks_of(const kda_prefill_args* a) {
    if (a->cu_seqlens == nullptr) return a->batch * ((a->seqlen + kChunk - 1) / kChunk);
    return a->seqlen / kChunk + a->num_seqs;
}

bool layout_of(const kda_prefill_args* a, kda_workspace_layout* L) {
    const int64_t mc = max_chunks_of(a);
    if (mc < 0 || a->num_heads < 1) return false;
    const size_t nrec = (size_t)mc * (size_t)a->num_heads;
    size_t o = 0;
    L->max_chunks = mc;
    L->record_bytes = kRecBytes;
    L->records = o; o = align_up(o + nrec * kRecBytes);
    L->chunk_offset = o; o = align_up(o + sizeof(int32_t) * (size_t)(a->num_seqs + 1));
    L->status = o; o = align_up(o + sizeof(int32_t));
    L->total = o;
    return true;
}

bool strides_ok(const int64_t* s, int64_t mult) {
    for (int i = 0; i < 3; ++i)
        if (s[i] < 0 || (s[i] % mult) != 0) return false;
    return true;
}

kda_status check_prefill(const kda_prefill_args* a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->head_dim_k != kHeadDim || a->head_dim_v != kHeadDim || a->chunk != kChunk)
        return KDA_ERR_UNSUPPORTED;
    if (a->num_heads < 1 || a->seqlen < 0 || a->num_seqs < 0 || a->batch < 0)
        return KDA_ERR_INVALID_ARG;
    if (a->cu_seqlens == nullptr) {
        if (a->num_seqs != a->batch) return KDA_ERR_INVALID_ARG;
    } else {
        if (a->batch != 1 || a->num_seqs < 1) return KDA_ERR_INVALID_ARG;
    }
    const bool tokens = a->seqlen > 0 && a->num_seqs > 0;
    if (tokens && (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->out))
        return KDA_ERR_INVALID_ARG;
    if (tokens) {
        if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) ||
            !aligned16(a->out))
            return KDA_ERR_UNSUPPORTED;
        if (!strides_ok(a->q_stride, 8) || !strides_ok(a->k_stride, 8) ||
            !strides_ok(a->v_stride, 8) || !strides_ok(a->out_stride, 8) ||
            !strides_ok(a->g_stride, 4) || !strides_ok(a->beta_stride, 1))
            return KDA_ERR_UNSUPPORTED;
    }
    if ((a->initial_state && !aligned16(a->initial_state)) ||
        (a->final_state && !aligned16(a->final_state)))
        return KDA_ERR_UNSUPPORTED;
    // fused gated RMSNorm: both operands or neither
    if ((a->out_gate != nullptr) != (a->norm_weight != nullptr)) return KDA_ERR_INVALID_ARG;
    if (a->out_gate && (!aligned16(a->out_gate) || !aligned16(a->norm_weight) ||
                        !strides_ok(a->gate_stride, 8) || !(a->norm_eps >= 0.f)))
        return KDA_ERR_UNSUPPORTED;
    if (a->num_seqs > (1 << 30) || a->num_heads > 65535 || a->seqlen > (int64_t)1 << 31)
        return KDA_ERR_UNSUPPORTED;
    kda_workspace_layout L;
    if (!layout_of(a, &L)) return KDA_ERR_INVALID_ARG;
    if (!a->workspace || a->workspace_bytes < L.total) return KDA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a->workspace) & (kAlign - 1)) != 0) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

void fill_params(const kda_prefill_args* a, const kda_workspace_layout& L, PrefillParams* p) {
    memset(p, 0, sizeof(*p));
    uint8_t* ws = static_cast<uint8_t*>(a->workspace);
    p->q = static_cast<const __nv_bfloat16*>(a->q);
    p->k = static_cast<const __nv_bfloat16*>(a->k);
    p->v = static_cast<const __nv_bfloat16*>(a->v);
    p->g = a->g;
    p->beta = a->beta;
    p->out = static_cast<__nv_bfloat16*>(a->out);
    for (int i = 0; i < 3; ++i) {
        p->qs[i] = a->q_stride[i]; p->ks[i] = a->k_stride[i]; p->vs[i] = a->v_stride[i];
        p->gs[i] = a->g_stride[i]; p->bs[i] = a->beta_stride[i]; p->os[i] = a->out_stride[i];
    }
    p->h0 = a->initial_state;
    p->hT = a->final_state;
    p->cu = a->cu_seqlens;
    p->chunk_off = reinterpret_cast<int32_t*>(ws + L.chunk_offset);
    p->status = a->device_status ? a->device_status : reinterpret_cast<int32_t*>(ws + L.status);
    p->B = (int)a->batch;
    p->T = (int)a->seqlen;
    p->N = (int)a->num_seqs;
    p->H = (int)a->num_heads;
    p->max_chunks = (int)L.max_chunks;
    p->beta_is_logit = a->beta_is_logit ? 1 : 0;
    p->scale = a->scale;
    p->ws_rec = ws + L.records;
    p->gate = static_cast<const __nv_bfloat16*>(a->out_gate);
    for (int i = 0; i < 3; ++i) p->gts[i] = a->gate_stride[i];
    p->norm_w = a->norm_weight;
    p->norm_eps = a->norm_eps;
}

// 4-D input tensor map [channel 128, head, token, batch] with one chunk of
// one head per box.  Returns false if the driver refuses the layout.
bool make_input_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, uint32_t esize,
                    const int64_t* st, int64_t H, int64_t T, int64_t B) {
    const uint64_t tstride = (uint64_t)st[1] * esize;
    const uint64_t bstride = st[0] != 0 ? (uint64_t)st[0] * esize : tstride * (uint64_t)(T > 0 ? T : 1);
    const uint64_t dims[4] = {128, (uint64_t)H, (uint64_t)T, (uint64_t)B};
    const uint64_t strides[3] = {(uint64_t)st[2] * esize, tstride, bstride};
    const uint32_t box[4] = {128, 1, (uint32_t)kChunk, 1};
    return make_tensor_map(m, dt, 4, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool make_prep_maps(const kda_prefill_args* a, PrepMaps* m) {
    const int64_t T = a->seqlen, B = a->cu_seqlens ? 1 : a->batch, H = a->num_heads;
    if (T == 0 || B == 0) return true;
    return make_input_map(&m->q, a->q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->q_stride, H, T, B) &&
           make_input_map(&m->k, a->k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->k_stride, H, T, B) &&
           make_input_map(&m->v, a->v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a->v_stride, H, T, B) &&
           make_input_map(&m->g, a->g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a->g_stride, H, T, B);
}

kda_status run_prefill(const kda_prefill_args* a, void* stream, int stages) {
    const bool state_pass = (stages & 2) != 0, prep = (stages & 1) != 0;
    kda_status st = check_prefill(a);
    if (st != KDA_OK) return st;
    kda_workspace_layout L;
    layout_of(a, &L);
    PrefillParams p;
    fill_params(a, L, &p);
    PrepMaps pmaps;
    memset(&pmaps, 0, sizeof(pmaps));
    int num_sms = 1;
    if (prep && !make_prep_maps(a, &pmaps)) return KDA_ERR_UNSUPPORTED;
    {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return KDA_ERR_CUDA;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (prep) {
        if (!a->device_status && cudaMemsetAsync(p.status, 0, sizeof(int32_t), s) != cudaSuccess)
            return KDA_ERR_CUDA;
        if (launch_chunk_table(p, s) != cudaSuccess) return KDA_ERR_CUDA;
        if (launch_prep(p, pmaps, num_sms, s) != cudaSuccess) return KDA_ERR_CUDA;
    }
    if (state_pass) {
        // One CTA per chain (all 128 value columns) when the 32-column slab CTAs
        // would need more than two waves of SMs: a whole-chain CTA takes about
        // twice as long per chunk step (measured), so below that the slab kernel
        // is as fast or faster.  The two kernels compute the same chunk step.
        // KDA_STATE_KERNEL=head|slab overrides the choice (tests, measurements);
        // the fused output norm needs whole rows and always takes the head kernel.
        const char* force = getenv("KDA_STATE_KERNEL");
        const bool head = p.gate ? true
                          : force && !strcmp(force, "head") ? true
                          : force && !strcmp(force, "slab") ? false
                          : (long long)p.N * p.H * (kHeadDim / kSlab) > 2LL * num_sms;
        if ((head ? launch_state_head(p, s) : launch_state(p, s)) != cudaSuccess) return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

size_t kda_prefill_workspace_size(const kda_prefill_args* args) {
    if (!args) return 0;
    kda_workspace_layout L;
    if (!layout_of(args, &L)) return 0;
    return L.total;
}

kda_status kda_prefill_workspace_layout(const kda_prefill_args* args, kda_workspace_layout* layout) {
    if (!args || !layout) return KDA_ERR_INVALID_ARG;
    return layout_of(args, layout) ? KDA_OK : KDA_ERR_INVALID_ARG;
}

kda_status kda_prefill(const kda_prefill_args* args, void* stream) {
    return run_prefill(args, stream, 3);
}

kda_status kda_prefill_prep(const kda_prefill_args* args, void* stream) {
    return run_prefill(args, stream, 1);
}

kda_status kda_prefill_state(const kda_prefill_args* args, void* stream) {
    return run_prefill(args, stream, 2);
}

kda_status kda_verify(const kda_verify_args* a, void* stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->head_dim_k != kHeadDim || a->head_dim_v != kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (a->num_requests < 0 || a->num_heads < 1 || a->num_drafts < 1 || a->pool_size < 0)
        return KDA_ERR_INVALID_ARG;
    if (a->num_drafts > 16) return KDA_ERR_UNSUPPORTED;
    if (a->num_requests == 0) return KDA_OK;
    if (!a->q || !a->k || !a->v || !a->g || !a->beta || (!a->out && !a->replay_only) ||
        !a->state_pool || !a->accepted || a->pool_size < 1)
        return KDA_ERR_INVALID_ARG;
    if (a->pool_dtype != KDA_POOL_F32 && a->pool_dtype != KDA_POOL_BF16) return KDA_ERR_UNSUPPORTED;
    if (a->num_requests > 65535 || a->num_heads > 65535 || a->pool_size > (1 << 30))
        return KDA_ERR_UNSUPPORTED;
    const int64_t* ss[6] = {a->q_stride, a->k_stride, a->v_stride, a->g_stride, a->beta_stride,
                            a->out_stride};
    for (int t = 0; t < 6; ++t)
        for (int i = 0; i < 3; ++i)
            if (ss[t][i] < 0) return KDA_ERR_UNSUPPORTED;
    // Draft rows and state blocks are moved in 16-byte pieces: every q, k, v, g row
    // and the pool must start on a 16-byte boundary.
    auto aligned16 = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15) == 0; };
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) ||
        !aligned16(a->state_pool))
        return KDA_ERR_UNSUPPORTED;
    for (int i = 0; i < 3; ++i)
        if (a->q_stride[i] % 8 || a->k_stride[i] % 8 || a->v_stride[i] % 8 || a->g_stride[i] % 4)
            return KDA_ERR_UNSUPPORTED;
    int dev = 0, num_sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KDA_ERR_CUDA;
    VerifyParams p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const __nv_bfloat16*>(a->q);
    p.k = static_cast<const __nv_bfloat16*>(a->k);
    p.v = static_cast<const __nv_bfloat16*>(a->v);
    p.g = a->g;
    p.beta = a->beta;
    p.out = static_cast<__nv_bfloat16*>(a->out);
    for (int i = 0; i < 3; ++i) {
        p.qs[i] = a->q_stride[i]; p.ks[i] = a->k_stride[i]; p.vs[i] = a->v_stride[i];
        p.gs[i] = a->g_stride[i]; p.bs[i] = a->beta_stride[i]; p.os[i] = a->out_stride[i];
    }
    p.pool = a->state_pool;
    p.slot = a->slot;
    p.accepted = a->accepted;
    p.status = a->device_status;
    p.R = (int)a->num_requests;
    p.D = (int)a->num_drafts;
    p.H = (int)a->num_heads;
    p.P = (int)a->pool_size;
    p.beta_is_logit = a->beta_is_logit ? 1 : 0;
    p.scale = a->scale;
    p.pool_bf16 = a->pool_dtype == KDA_POOL_BF16 ? 1 : 0;
    p.replay_only = a->replay_only ? 1 : 0;
    return launch_verify(p, num_sms, static_cast<cudaStream_t>(stream)) == cudaSuccess ? KDA_OK
                                                                               : KDA_ERR_CUDA;
}

const char* kda_status_string(kda_status s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG: invalid argument";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED: unsupported shape, stride or alignment";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA: a CUDA call failed";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT: a bounded on-chip wait ran out";
    }
    return "unknown kda_status";
}

int kda_abi_version(void) { return KDA_ABI_VERSION; }

}  // extern "C"
