// noalloc.cu -- dr_chunk_fwd_noalloc: the chunkwise forward without a caller-provided
// workspace, for callers that cannot allocate device memory.
//
// Who needs it: code that runs inside a host framework owning all device memory through
// its own pre-reserved pool (a private cudaMalloc there fails or fragments the pool),
// plugin interfaces whose execute callback is not allowed to allocate, and latency-bound
// loops that cannot pay cudaMalloc's implicit device-wide synchronisation.  Such callers
// still pass their inputs and outputs; only the scratch is provided here.
//
// The scratch is one file-scope device array of kNoallocScratchBytes (64 MiB), which every
// GPU that loads libdr.so holds until the process exits.  Host code cannot use the
// array's name as a device address (on the host it names a stand-in object), so the
// device address is looked up with cudaGetSymbolAddress once per device, with that device
// current, on the first call made on that device; make that first call before any stream
// capture begins.  All calls share the array and it keeps the previous call's contents:
// nothing in it needs clearing because the chunk kernels write every scratch element they
// later read, but calls whose work overlaps on the GPU (two streams, or two host threads)
// race on the array and must be serialised by the caller.
#include <mutex>

#include "../../include/dr.h"
#include "chunk_layout.h"
#include "common.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = DR_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
int scratch_address(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DR_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return DR_OK;
}

}  // namespace

extern "C" int dr_chunk_fwd_noalloc(const dr_chunk_desc *desc, const void *q, const void *k,
                                    const void *v, const float *log_alpha, const void *beta,
                                    const float *init_state, void *out, float *final_state,
                                    dr_stream_t stream) {
    size_t need = 0;
    const int rc = dr::chunk_fwd_least_workspace(desc, &need);
    if (rc != DR_OK) return rc;
    if (need > kNoallocScratchBytes) return DR_ERR_WORKSPACE;   // beyond the built-in maximum
    void *scratch = nullptr;
    size_t full = 0;
    dr_chunk_fwd_workspace_bytes(desc, &full);
    if (need > 0 || full > 0) {
        const int st = scratch_address(&scratch);
        if (st != DR_OK) return st;
    }
    return dr_chunk_fwd(desc, q, k, v, log_alpha, beta, init_state, out, final_state, scratch,
                        kNoallocScratchBytes, stream);
}
