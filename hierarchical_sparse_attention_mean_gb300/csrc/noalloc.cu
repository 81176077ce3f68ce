// noalloc.cu -- a variant of the sparse index transpose for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code
// running inside a memory pool they do not own, inside an allocator-free
// runtime, or at a point where allocating would break their memory budget.
// This variant keeps its scratch (one counter per fine key block per slice)
// in a fixed device array that every GPU holding this library carries for the
// life of the process, so the caller passes only inputs and outputs.
#include <string.h>

#include <initializer_list>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "internal.h"

namespace llsa {
namespace {

// Scratch of llsa_index_transpose_noalloc: column counters / scatter cursors.
static __device__ __align__(256) int32_t g_transpose_scratch[LLSA_NOALLOC_TRANSPOSE_MAX_COUNTERS];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (the array's name is only a host-side stand-in in host code).
// The kept address does not survive cudaDeviceReset of that device; the
// header tells such callers to reload the library.
int scratch_on_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LLSA_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_transpose_scratch) != cudaSuccess || !ptr) return LLSA_ERR_CUDA;
        g_scratch_addr[dev] = static_cast<int32_t*>(ptr);
    }
    *out = g_scratch_addr[dev];
    return LLSA_OK;
}

}  // namespace
}  // namespace llsa

using namespace llsa;

static int noalloc_transpose(const llsa_params* p, const int32_t* sel_idx, int32_t* col_ptr, int32_t* row_idx,
                             void* stream);

extern "C" int llsa_index_transpose_noalloc(const llsa_params* p, const int32_t* sel_idx, int32_t* col_ptr,
                                            int32_t* row_idx, void* stream) {
    nvtxRangePushA("llsa_index_transpose_noalloc");
    const int rc = noalloc_transpose(p, sel_idx, col_ptr, row_idx, stream);
    nvtxRangePop();
    return rc;
}

static int noalloc_transpose(const llsa_params* p, const int32_t* sel_idx, int32_t* col_ptr, int32_t* row_idx,
                             void* stream) {
    llsa_sizes z;
    LLSA_TRY(llsa_get_sizes(p, &z));
    if (z.slices == 0) return LLSA_OK;
    for (const void* ptr : {(const void*)sel_idx, (const void*)col_ptr, (const void*)row_idx}) {
        if (!ptr) return LLSA_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return LLSA_ERR_ALIGN;
    }
    if (z.slices * (long long)z.n_blocks > LLSA_NOALLOC_TRANSPOSE_MAX_COUNTERS) return LLSA_ERR_UNSUPPORTED;
    LLSA_TRY(device_ready());
    int32_t* scratch = nullptr;
    LLSA_TRY(scratch_on_current_device(&scratch));
    Shape s;
    memset(&s, 0, sizeof(s));
    s.slices = z.slices;
    s.n = p->n;
    s.T = z.n_blocks;
    s.K1 = z.topk_level[1];
    // the same kernels as llsa_index_transpose; the counters are zeroed on the
    // stream before use, so nothing of an earlier call carries over
    return launch_transpose(s, sel_idx, s.T, s.K1, s.T, col_ptr, row_idx, scratch, static_cast<cudaStream_t>(stream));
}
