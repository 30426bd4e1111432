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
//  - The array's address belongs to the CUDA context current at the call.  Outside stream capture
//    every call looks it up afresh (cudaGetSymbolAddress), so a device reset or a caller-made driver
//    context is always served with its own address.  During capture no lookup is made: the address
//    cached for the current context by an earlier call is used, so make one call in each context
//    before capturing; a capture in a context never seen before returns GDN_ERR_CUDA.
//  - A device-side wait that times out leaves its record in the array's error word, which
//    gdn_fwd_noalloc_error() reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gdn.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

// (context, address) pairs of the contexts seen so far; a reset context that gets a recycled handle
// is refreshed by the next lookup made outside capture.
constexpr int kMaxContexts = 64;
std::mutex g_mu;
CUcontext g_ctx[kMaxContexts] = {};
void *g_addr[kMaxContexts] = {};
int g_n = 0;

// Device address of the scratch array in the current context.
gdn_status scratch_for_current_context(cudaStream_t st, void **out) {
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return GDN_ERR_CUDA;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return GDN_ERR_CUDA;
    void *ptr = nullptr;
    // outside capture: look the address up first (this also makes the device's primary context current
    // when the thread has none), then note which context it belongs to
    if (cs == cudaStreamCaptureStatusNone &&
        (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr))
        return GDN_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS || ctx == nullptr) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    int slot = -1;
    for (int i = 0; i < g_n; ++i)
        if (g_ctx[i] == ctx) slot = i;
    if (cs != cudaStreamCaptureStatusNone) {  // no lookup while capturing
        if (slot < 0) return GDN_ERR_CUDA;
        *out = g_addr[slot];
        return GDN_OK;
    }
    if (slot < 0) {
        slot = g_n < kMaxContexts ? g_n++ : kMaxContexts - 1;
        g_ctx[slot] = ctx;
    }
    g_addr[slot] = ptr;
    *out = ptr;
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_fwd_noalloc(const gdn_problem *p, const void *q, const void *k, const void *v,
                                      const float *g, const float *beta, const float *h0, void *o, float *g_cum,
                                      void *A, float *h, float *final_state, gdn_stream_t stream) {
    const size_t need = gdn_fwd_workspace_bytes(p);
    if (need == 0)  // an invalid or unsupported problem: gdn_fwd's own validation gives the status
        return gdn_fwd(p, q, k, v, g, beta, h0, o, g_cum, A, h, final_state, nullptr, 0, stream);
    if (need > (size_t)GDN_NOALLOC_SCRATCH_BYTES) return GDN_ERR_TOO_LARGE;
    void *scratch = nullptr;
    gdn_status s = scratch_for_current_context(reinterpret_cast<cudaStream_t>(stream), &scratch);
    if (s != GDN_OK) return s;
    return gdn_fwd(p, q, k, v, g, beta, h0, o, g_cum, A, h, final_state, scratch,
                   (size_t)GDN_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" gdn_status gdn_fwd_noalloc_error(gdn_stream_t stream) {
    void *scratch = nullptr;
    gdn_status s = scratch_for_current_context(reinterpret_cast<cudaStream_t>(stream), &scratch);
    if (s != GDN_OK) return s;
    return gdn_workspace_error(scratch, stream);
}
