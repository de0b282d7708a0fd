// kda_host.cu -- KDA prefill from page-locked host buffers (a runtime entry of
// this library; the pages have no counterpart).  The call cuts the work into
// pieces, copies piece p + 1 in while piece p runs through the prefill kernels
// and copies each piece's output back while later pieces run, on two internal
// copy streams around the caller's stream.  Nothing on the host waits.
//
// Pieces: in padded mode a piece is a token range [t0, t0 + len) of every
// sequence, len a multiple of the 64-token chunk, and the state of each chain
// continues from piece to piece in a device state buffer (the in-place
// continuation kda_prefill allows), so the result equals one kda_prefill over
// the whole input.  In varlen mode a piece is a run of whole sequences (they
// are independent), with its own cu_seqlens and state slices.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "../../include/kda.h"

namespace {

constexpr int64_t kD = 128;
constexpr int64_t kChunk = 64;

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }
int64_t up64(int64_t x) { return (x + kChunk - 1) / kChunk * kChunk; }

struct Piece {
    int64_t t0, len;   // token range (padded: within every sequence; varlen: packed)
    int64_t n0, nseq;  // varlen: sequence range
};

struct Plan {
    bool varlen = false;
    int64_t B = 0, T = 0, H = 0, N = 0;
    int64_t Pmax = 0, max_seqs = 0;
    std::vector<Piece> pieces;
    size_t off_q[2], off_k[2], off_v[2], off_g[2], off_b[2], off_o[2], off_s[2];
    size_t off_cu = 0;       // varlen: every piece's rebased cu_seqlens, one after another
    std::vector<int32_t> cu_all;
    std::vector<size_t> cu_at;
    size_t off_ws = 0, ws_bytes = 0, total = 0;
};

// Builds the pieces and the staging layout; false if the arguments are unusable.
bool make_plan(const kda_prefill_host_args* h, Plan* pl) {
    const kda_prefill_args& a = h->args;
    if (a.head_dim_k != kD || a.head_dim_v != kD || a.chunk != kChunk || a.num_heads < 1) return false;
    if (h->piece_tokens < 0 || h->piece_tokens % kChunk) return false;
    pl->H = a.num_heads;
    pl->varlen = a.cu_seqlens != nullptr;
    if (!pl->varlen) {
        if (a.batch < 1 || a.seqlen < 0 || a.num_seqs != a.batch) return false;
        pl->B = a.batch; pl->T = a.seqlen; pl->N = a.batch;
        int64_t P = h->piece_tokens ? h->piece_tokens : up64(std::max<int64_t>((pl->T + 31) / 32, 2048));
        P = std::min(P, std::max<int64_t>(up64(pl->T), kChunk));
        if (pl->T == 0) pl->pieces.push_back({0, 0, 0, 0});
        for (int64_t t0 = 0; t0 < pl->T; t0 += P) pl->pieces.push_back({t0, std::min(P, pl->T - t0), 0, 0});
        pl->Pmax = P;
        pl->max_seqs = pl->B;
    } else {
        if (a.batch != 1 || a.num_seqs < 1 || a.seqlen < 0) return false;
        pl->B = 1; pl->T = a.seqlen; pl->N = a.num_seqs;
        const int32_t* cu = a.cu_seqlens;  // host array here
        if (cu[0] != 0 || cu[pl->N] != pl->T) return false;
        for (int64_t n = 0; n < pl->N; ++n)
            if (cu[n + 1] < cu[n]) return false;
        const int64_t P = h->piece_tokens ? h->piece_tokens : up64(std::max<int64_t>((pl->T + 31) / 32, 2048));
        int64_t n0 = 0;
        while (n0 < pl->N) {
            int64_t n1 = n0 + 1;
            while (n1 < pl->N && cu[n1 + 1] - cu[n0] <= P) ++n1;
            pl->pieces.push_back({cu[n0], cu[n1] - cu[n0], n0, n1 - n0});
            pl->cu_at.push_back(pl->cu_all.size());
            for (int64_t n = n0; n <= n1; ++n) pl->cu_all.push_back(cu[n] - cu[n0]);
            pl->Pmax = std::max<int64_t>(pl->Pmax, cu[n1] - cu[n0]);
            pl->max_seqs = std::max<int64_t>(pl->max_seqs, n1 - n0);
            n0 = n1;
        }
    }
    // Staging: two buffers of piece inputs / output (+ cu_seqlens and states in
    // varlen mode), one state buffer in padded mode, one prefill workspace.
    const size_t tok = (size_t)pl->B * pl->Pmax * pl->H;
    size_t off = 0;
    for (int b = 0; b < 2; ++b) {
        pl->off_q[b] = off; off = up256(off + tok * kD * 2);
        pl->off_k[b] = off; off = up256(off + tok * kD * 2);
        pl->off_v[b] = off; off = up256(off + tok * kD * 2);
        pl->off_g[b] = off; off = up256(off + tok * kD * 4);
        pl->off_b[b] = off; off = up256(off + tok * 4);
        pl->off_o[b] = off; off = up256(off + tok * kD * 2);
        if (pl->varlen || b == 0) {
            pl->off_s[b] = off; off = up256(off + (size_t)pl->max_seqs * pl->H * kD * kD * 4);
        } else {
            pl->off_s[b] = pl->off_s[0];
        }
    }
    pl->off_cu = off;
    off = up256(off + pl->cu_all.size() * 4);
    kda_prefill_args w;
    memset(&w, 0, sizeof(w));
    w.batch = pl->B; w.seqlen = pl->Pmax; w.num_seqs = pl->varlen ? pl->max_seqs : pl->B;
    w.num_heads = pl->H; w.head_dim_k = w.head_dim_v = kD; w.chunk = kChunk;
    w.cu_seqlens = pl->varlen ? reinterpret_cast<const int32_t*>(16) : nullptr;  // only its presence matters
    pl->ws_bytes = kda_prefill_workspace_size(&w);
    pl->off_ws = off;
    pl->total = up256(off + pl->ws_bytes);
    return true;
}

// The copy streams and events of host-buffer calls: one set per host thread
// and device, created on the thread's first call on that device and kept for
// the thread's life (calls of one thread share them; every dependency between
// calls goes through the caller's stream).
struct CopySet {
    cudaStream_t hs = nullptr, ds = nullptr;      // copies in, copies out
    cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_in_done = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
};

bool copy_set(CopySet* out) {
    constexpr int kMaxDevices = 64;
    thread_local CopySet sets[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    CopySet& cs = sets[dev];
    if (!cs.hs) {
        CopySet n;
        auto ev = [](cudaEvent_t* e) { return cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess; };
        bool ok = cudaStreamCreateWithFlags(&n.hs, cudaStreamNonBlocking) == cudaSuccess &&
                  cudaStreamCreateWithFlags(&n.ds, cudaStreamNonBlocking) == cudaSuccess &&
                  ev(&n.ev_start) && ev(&n.ev_end) && ev(&n.ev_in_done);
        for (int b = 0; b < 2 && ok; ++b) ok = ev(&n.ev_in[b]) && ev(&n.ev_comp[b]) && ev(&n.ev_out[b]);
        if (!ok) {
            cudaEvent_t all[] = {n.ev_start, n.ev_end, n.ev_in_done, n.ev_in[0], n.ev_in[1], n.ev_comp[0],
                                 n.ev_comp[1], n.ev_out[0], n.ev_out[1]};
            for (cudaEvent_t e : all)
                if (e) cudaEventDestroy(e);
            if (n.hs) cudaStreamDestroy(n.hs);
            if (n.ds) cudaStreamDestroy(n.ds);
            return false;
        }
        cs = n;
    }
    *out = cs;
    return true;
}

}  // namespace

extern "C" size_t kda_prefill_host_staging_size(const kda_prefill_host_args* h) {
    if (!h) return 0;
    Plan pl;
    return make_plan(h, &pl) ? pl.total : 0;
}

extern "C" kda_status kda_prefill_host(const kda_prefill_host_args* h, void* stream) {
    if (!h) return KDA_ERR_INVALID_ARG;
    const kda_prefill_args& a = h->args;
    if (!a.q || !a.k || !a.v || !a.g || !a.beta || !a.out || !h->staging) return KDA_ERR_INVALID_ARG;
    if (a.out_gate || a.norm_weight) return KDA_ERR_UNSUPPORTED;  // the gate is not staged here
    Plan pl;
    if (!make_plan(h, &pl)) return KDA_ERR_INVALID_ARG;
    if (h->staging_bytes < pl.total || (reinterpret_cast<uintptr_t>(h->staging) & 255))
        return KDA_ERR_INVALID_ARG;
    uint8_t* st = static_cast<uint8_t*>(h->staging);
    const int64_t H = pl.H, T = pl.T, B = pl.B;
    const size_t sblock = (size_t)H * kD * kD * 4;  // one sequence's states
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    CopySet set;
    if (!copy_set(&set)) return KDA_ERR_CUDA;
    cudaStream_t hs = set.hs, ds = set.ds;
    cudaEvent_t ev_start = set.ev_start, ev_end = set.ev_end;
    cudaEvent_t* ev_in = set.ev_in;
    cudaEvent_t* ev_comp = set.ev_comp;
    cudaEvent_t* ev_out = set.ev_out;
    kda_status ret = KDA_OK;
    auto ck = [&](cudaError_t e) {
        if (e != cudaSuccess && ret == KDA_OK) ret = KDA_ERR_CUDA;
        return e == cudaSuccess;
    };
    bool ok = true;
    // Work already queued on the caller's stream (an earlier use of the staging
    // memory) comes first.
    ok = ok && ck(cudaEventRecord(ev_start, cs)) && ck(cudaStreamWaitEvent(hs, ev_start, 0)) &&
         ck(cudaStreamWaitEvent(ds, ev_start, 0));
    float* dstate0 = reinterpret_cast<float*>(st + pl.off_s[0]);
    if (ok && !pl.varlen && a.initial_state)
        ok = ck(cudaMemcpyAsync(dstate0, a.initial_state, (size_t)B * sblock, cudaMemcpyHostToDevice, hs));
    // varlen: all pieces' cu_seqlens in one copy (from pageable memory: the call
    // returns once the host data has been taken)
    if (ok && pl.varlen)
        ok = ck(cudaMemcpyAsync(st + pl.off_cu, pl.cu_all.data(), pl.cu_all.size() * 4, cudaMemcpyHostToDevice, hs));
    // 2-D copy of a token range of every sequence (row = sequence) between the
    // host tensor (T tokens per row) and the piece buffer (len tokens per row).
    auto copy_rows = [&](void* dst, size_t dpitch, const void* src, size_t spitch, size_t width,
                         cudaMemcpyKind kind, cudaStream_t s) -> bool {
        if (width == 0) return true;
        if (B == 1) return ck(cudaMemcpyAsync(dst, src, width, kind, s));
        return ck(cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, (size_t)B, kind, s));
    };
    for (size_t p = 0; p < pl.pieces.size() && ok; ++p) {
        const Piece& pc = pl.pieces[p];
        const int b = (int)(p & 1);
        const int64_t len = pc.len;
        const size_t row_tok = (size_t)H * kD;          // elements per token
        const size_t off_tok = (size_t)pc.t0 * row_tok;  // element offset of t0 in a host row
        // ---- inputs in, once the piece two back has finished with buffer b (in
        // varlen mode also with its state slice, which leaves on the output stream)
        if (p >= 2) ok = ck(cudaStreamWaitEvent(hs, pl.varlen ? ev_out[b] : ev_comp[b], 0));
        const size_t w2 = (size_t)len * row_tok * 2, w4 = (size_t)len * row_tok * 4, wb = (size_t)len * H * 4;
        const size_t hp2 = (size_t)T * row_tok * 2, hp4 = (size_t)T * row_tok * 4, hpb = (size_t)T * H * 4;
        ok = ok && copy_rows(st + pl.off_q[b], w2, static_cast<const uint8_t*>(a.q) + off_tok * 2, hp2, w2,
                             cudaMemcpyHostToDevice, hs);
        ok = ok && copy_rows(st + pl.off_k[b], w2, static_cast<const uint8_t*>(a.k) + off_tok * 2, hp2, w2,
                             cudaMemcpyHostToDevice, hs);
        ok = ok && copy_rows(st + pl.off_v[b], w2, static_cast<const uint8_t*>(a.v) + off_tok * 2, hp2, w2,
                             cudaMemcpyHostToDevice, hs);
        ok = ok && copy_rows(st + pl.off_g[b], w4, reinterpret_cast<const uint8_t*>(a.g) + off_tok * 4, hp4, w4,
                             cudaMemcpyHostToDevice, hs);
        ok = ok && copy_rows(st + pl.off_b[b], wb, reinterpret_cast<const uint8_t*>(a.beta) + pc.t0 * H * 4, hpb,
                             wb, cudaMemcpyHostToDevice, hs);
        if (ok && pl.varlen) {
            if (a.initial_state)
                ok = ck(cudaMemcpyAsync(st + pl.off_s[b], a.initial_state + (size_t)pc.n0 * H * kD * kD,
                                        (size_t)pc.nseq * sblock, cudaMemcpyHostToDevice, hs));
        }
        ok = ok && ck(cudaEventRecord(ev_in[b], hs));
        // ---- the prefill of the piece (after the piece two back's output left buffer b)
        ok = ok && ck(cudaStreamWaitEvent(cs, ev_in[b], 0));
        if (ok && p >= 2) ok = ck(cudaStreamWaitEvent(cs, ev_out[b], 0));
        if (!ok) break;
        kda_prefill_args w = a;
        w.q = st + pl.off_q[b]; w.k = st + pl.off_k[b]; w.v = st + pl.off_v[b];
        w.g = reinterpret_cast<const float*>(st + pl.off_g[b]);
        w.beta = reinterpret_cast<const float*>(st + pl.off_b[b]);
        w.out = st + pl.off_o[b];
        const int64_t s0 = len * H * kD, s1 = H * kD;
        for (int i = 0; i < 3; ++i) {
            const int64_t sv = i == 0 ? s0 : (i == 1 ? s1 : kD);
            w.q_stride[i] = w.k_stride[i] = w.v_stride[i] = w.g_stride[i] = w.out_stride[i] = sv;
        }
        w.beta_stride[0] = len * H; w.beta_stride[1] = H; w.beta_stride[2] = 1;
        w.workspace = st + pl.off_ws;
        w.workspace_bytes = pl.ws_bytes;
        float* dstate = reinterpret_cast<float*>(st + pl.off_s[b]);
        if (!pl.varlen) {
            w.seqlen = len;
            w.initial_state = (p == 0 && !a.initial_state) ? nullptr : dstate0;
            w.final_state = dstate0;
        } else {
            w.batch = 1; w.seqlen = len; w.num_seqs = pc.nseq;
            w.cu_seqlens = reinterpret_cast<const int32_t*>(st + pl.off_cu) + pl.cu_at[p];
            w.initial_state = a.initial_state ? dstate : nullptr;
            w.final_state = a.final_state ? dstate : nullptr;
        }
        const kda_status r = kda_prefill(&w, cs);
        if (r != KDA_OK) { ret = r; ok = false; break; }
        ok = ck(cudaEventRecord(ev_comp[b], cs));
        // ---- output (and varlen final states) out
        ok = ok && ck(cudaStreamWaitEvent(ds, ev_comp[b], 0));
        ok = ok && copy_rows(static_cast<uint8_t*>(a.out) + off_tok * 2, hp2, st + pl.off_o[b], w2, w2,
                             cudaMemcpyDeviceToHost, ds);
        if (ok && pl.varlen && a.final_state)
            ok = ck(cudaMemcpyAsync(a.final_state + (size_t)pc.n0 * H * kD * kD, dstate,
                                    (size_t)pc.nseq * sblock, cudaMemcpyDeviceToHost, ds));
        ok = ok && ck(cudaEventRecord(ev_out[b], ds));
    }
    if (ok && !pl.varlen && a.final_state) {
        ok = ck(cudaStreamWaitEvent(ds, ev_comp[(pl.pieces.size() - 1) & 1], 0)) &&
             ck(cudaMemcpyAsync(a.final_state, dstate0, (size_t)B * sblock, cudaMemcpyDeviceToHost, ds));
    }
    // The caller's stream completes only after every copy has landed (also
    // after a failure, so that nothing queued later on it overtakes a copy).
    if (ck(cudaEventRecord(ev_end, ds))) ck(cudaStreamWaitEvent(cs, ev_end, 0));
    if (ck(cudaEventRecord(set.ev_in_done, hs))) ck(cudaStreamWaitEvent(cs, set.ev_in_done, 0));
    return ret;
}
