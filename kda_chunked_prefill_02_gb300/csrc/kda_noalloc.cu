// kda_noalloc.cu -- kda_prefill_noalloc: KDA prefill for callers that must not
// allocate device memory.
//
// kda_prefill needs a caller-owned workspace.  Some callers cannot provide one:
// code that runs under a fixed device-memory budget owned by another runtime,
// or in a latency-critical loop where cudaMalloc (which can synchronise the
// device and fragment a pool) is not allowed.  This entry point takes the same
// arguments but ignores `workspace` / `workspace_bytes` and uses a scratch
// array compiled into the library instead.
//
// The scratch array lives in device memory of every GPU that loads the library,
// for as long as the process runs, and has a fixed size (kNoAllocScratchBytes).
// In host code the array's name is only a host-side stand-in, so its device
// address is looked up once per device with cudaGetSymbolAddress while that
// device is current, and that address is what the kernels receive.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = KDA_NOALLOC_MAX_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call for that device).
kda_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return KDA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" kda_status kda_prefill_noalloc(const kda_prefill_args* args, void* stream) {
    if (!args) return KDA_ERR_INVALID_ARG;
    // The arguments are checked as kda_prefill checks them (all but the
    // workspace) before the size test, so that bad arguments come back as
    // KDA_ERR_INVALID_ARG and not as an oversize problem.
    const kda_status checked = static_cast<kda_status>(kda::prefill_check_args(args));
    if (checked != KDA_OK) return checked;
    const size_t need = kda_prefill_workspace_size(args);
    if (need > kNoAllocScratchBytes) return KDA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const kda_status st = scratch_on_current_device(&scratch);
    if (st != KDA_OK) return st;
    kda_prefill_args a = *args;
    a.workspace = scratch;
    a.workspace_bytes = kNoAllocScratchBytes;
    return kda_prefill(&a, stream);
}
