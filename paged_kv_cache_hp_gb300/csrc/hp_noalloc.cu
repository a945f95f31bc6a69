// hp_noalloc.cu -- hp_gather_noalloc: the gather for callers that cannot allocate device
// memory.
//
// hp_gather needs a small device workspace for its plan (a header and two prefix arrays
// over the sequences).  Most callers allocate it once and pass it in.  Some cannot: a
// plugin hosted by a framework that owns the whole device budget and hands its plugins
// buffers but no allocator, or a latency-critical loop that must not call cudaMalloc or
// cudaFree (both can block, and cudaFree synchronises the device).  For them this file
// keeps the workspace in a fixed array of device memory that the library itself carries:
// it exists on every device that loads the library, for as long as the process runs.
#include <cuda_runtime.h>

#include <mutex>

#include "hp_internal.cuh"

#define HP_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr uint64_t kMaxSeqs = HP_NOALLOC_MAX_SEQS;
// the workspace hp_workspace_bytes reports for kMaxSeqs sequences
constexpr uint64_t kScratchBytes =
    hp::kWsHeaderBytes + 2 * ((8 * (kMaxSeqs + 1) + 255) / 256 * 256);

// The scratch.  In host code this name is only a stand-in for the device array, so the
// host never passes it to a kernel; it passes the device address looked up below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_lock;
void* g_scratch_addr[kMaxDevices];  // device address of g_scratch, per device ordinal

// The scratch's device address on the current device, looked up once per device and kept
// for the process.  A cudaDeviceReset after the first call would leave it stale (the module
// may load elsewhere in the new context); the header states that this is not supported.
int scratch_on_current_device(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HP_ERR_ARG;
    std::lock_guard<std::mutex> hold(g_lock);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return HP_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return HP_OK;
}

}  // namespace

HP_API int hp_gather_noalloc(const hp_paged_desc* desc, void* out, uint64_t out_tokens,
                             int* d_status, void* stream)
{
    if (!desc) return HP_ERR_NULL;
    if (desc->num_seqs > kMaxSeqs) return HP_ERR_NOALLOC_LIMIT;
    void* ws = nullptr;
    const int rc = scratch_on_current_device(&ws);
    if (rc) return rc;
    // The plan writes every scratch field the copy later reads, so whatever a previous
    // call left there needs no clearing.
    return hp_gather(desc, out, out_tokens, ws, kScratchBytes, d_status, stream);
}
