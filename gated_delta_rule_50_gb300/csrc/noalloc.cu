// noalloc.cu -- gdn_fwd_noalloc: the forward pass for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running
// inside a CUDA-graph replay whose memory pool is frozen, plugin hosts and
// inference runtimes that own every device allocation and forbid others, or
// C callers without an allocator of their own.  For them this entry point runs
// the ordinary forward with its scratch taken from a fixed, file-scope
// __device__ array instead of a caller buffer.
//
// Limits and caveats (also stated in gdn.h):
//  - The array holds GDN_NOALLOC_SCRATCH_BYTES bytes on every GPU that loads
//    the library, for the life of the process.  Problems whose forward
//    workspace (gdn_fwd_workspace_bytes) is larger are rejected with
//    GDN_ERR_TOO_LARGE before anything is enqueued.
//  - All calls share the one array and it keeps what the last call left.  The
//    forward rewrites every scratch byte it reads and clears its error word at
//    the start of each call, so stale contents never leak into a result; but
//    two calls whose GPU work overlaps (different streams, or different host
//    threads) race on the array and corrupt each other.  Serialise them.
//  - The first call on each device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
gdn_status scratch_for_current_device(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return GDN_ERR_CUDA;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_fwd_noalloc(const gdn_problem *p, const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, const float *h0, void *o, float *g_cum,
                                      void *A, float *h, float *final_state, gdn_stream_t stream) {
    size_t need = gdn_fwd_workspace_bytes(p);
    if (need == 0) return GDN_ERR_INVALID_ARG;
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_TOO_LARGE;
    void *scratch = nullptr;
    gdn_status s = scratch_for_current_device(&scratch);
    if (s != GDN_OK) return s;
    return gdn_fwd(p, q, k, v, g, beta, h0, o, g_cum, A, h, final_state, scratch,
                   (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}
