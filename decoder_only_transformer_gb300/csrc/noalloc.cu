// noalloc.cu - a SwiGLU entry point that needs no caller-provided or
// library-allocated scratch memory.
//
// tfm_swiglu keeps the hidden activation silu(x W1^T) * (x W3^T), an [M, F]
// matrix, in a workspace the caller allocates.  Some callers cannot allocate
// device memory at the point where they want to run the block: plugins running
// under a host framework that owns the device allocator (and may have handed
// all of the memory to its own pool), and deployments whose device memory is
// budgeted once at start-up, where a later cudaMalloc would fail or break the
// budget.  tfm_swiglu_noalloc gives them the same computation with the hidden
// activation in a fixed array that the library declares in device memory; it
// calls no allocator at all.
//
// The array is kSwigluScratchBytes (16 MiB) per device, reserved on every GPU
// that loads the library until the process exits.  Every call shares it and
// it keeps whatever the last call wrote: the gate/up kernel overwrites all
// M x F entries a call reads, so nothing has to be cleared first.  Calls whose
// kernels overlap on the GPU (different streams, no ordering between them)
// race on the array.
#include <cstdio>
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kSwigluScratchBytes = (size_t)16 << 20;

// The scratch array.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_swiglu_scratch[kSwigluScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices];

// Device address of the array on the current device, looked up once per
// device with that device current.  NULL (and a message) on failure.
void* scratch_address(const char** why) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        *why = "no current CUDA device";
        return nullptr;
    }
    std::lock_guard<std::mutex> lk(g_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_swiglu_scratch);
        if (e != cudaSuccess || !p) {
            *why = cudaGetErrorString(e);
            return nullptr;
        }
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

thread_local char t_msg[256];

}  // namespace

extern "C" {

size_t tfm_swiglu_noalloc_max_bytes(void) { return kSwigluScratchBytes; }

tfm_status tfm_swiglu_noalloc(const void* x, const void* w1, const void* w3, const void* w2,
                              float* y, int64_t M, int32_t D, int32_t F, int32_t accumulate,
                              int32_t mode, void* stream) {
    if (M < 0 || F < 1) {
        snprintf(t_msg, sizeof t_msg, "tfm_swiglu_noalloc: bad sizes M=%lld F=%d", (long long)M, (int)F);
        tfm::set_last_error(t_msg);
        return TFM_EINVAL;
    }
    const size_t need = tfm_swiglu_workspace_bytes(M, F, mode);
    if (need > kSwigluScratchBytes) {
        snprintf(t_msg, sizeof t_msg,
                 "tfm_swiglu_noalloc: M*F activation of %zu bytes exceeds the %zu-byte scratch array",
                 need, kSwigluScratchBytes);
        tfm::set_last_error(t_msg);
        return TFM_EINVAL;
    }
    const char* why = "";
    void* scratch = scratch_address(&why);
    if (!scratch) {
        snprintf(t_msg, sizeof t_msg, "tfm_swiglu_noalloc: scratch address lookup failed: %s", why);
        tfm::set_last_error(t_msg);
        return TFM_ECUDA;
    }
    return tfm_swiglu(x, w1, w3, w2, y, M, D, F, accumulate, scratch, kSwigluScratchBytes, mode,
                      stream);
}

}  // extern "C"
