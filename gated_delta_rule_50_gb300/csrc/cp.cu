// cp.cu -- sequence splitting with warmup ("AutoCP" of the FlashQLA pages):
// the trigger rule, the segment geometry and the per-head decay test.
//
// The FlashQLA news page ("FlashQLA's core advantages") and the blog post
// (section 1, Gate-Driven Automatic Intra-Card Context Parallelism) state that
// splitting turns on when batch_size x num_heads <= 40, or <= 56 with
// seq_len >= 8192; that a total of N chunks is cut into segments of L = sqrt(N)
// chunks; and that for decaying heads a warmup of 6-8 chunks from a zero state
// replaces the exact cross-segment correction.  Here batch_size is the number
// of sequences, num_heads the number of value heads and seq_len the longest
// sequence.  A head runs unsplit when any warmup window fails to decay by at
// least a factor 1e-4, since then a zero-state warmup is not an
// accurate start (the error of a window is at most its total decay times the
// state's norm).
#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr double WARMUP_LOG_EPS = -9.210340371976184;  // ln(1e-4)

bool cp_trigger(const Plan &p) {
    const long bh = (long)p.n_seqs * p.Hv;
    return bh <= 40 || (bh <= 56 && p.max_seq_len >= 8192);
}

void cp_geometry(const Plan &p, int *seg_len, int *n_seg) {
    const int N = p.max_seq_chunks;
    int L = (int)std::lround(std::sqrt((double)N));
    if (L < 1) L = 1;
    *seg_len = L;
    *n_seg = (N + L - 1) / L;
}

// One warp per (sequence, value head): serial = 1 when a warmup window's gate sum exceeds ln(eps).
__global__ void k_cp_flags(Plan p, const float *__restrict__ g, int seg_len, int n_seg, int warm,
                           uint8_t *__restrict__ serial) {
    const int s = blockIdx.x, hv = blockIdx.y, lane = threadIdx.x;
    const SeqRange sr = seq_range(p, s);
    const int N = sr.c1 - sr.c0;
    int flag = 0;
    for (int ps = 1; ps < n_seg && ps * seg_len < N; ++ps) {
        const int c0 = max(0, ps * seg_len - warm), c1 = ps * seg_len;
        const int t0 = sr.tok0 + c0 * C, t1 = sr.tok0 + c1 * C;
        double sum = 0.0;  // fp64: the decision does not hang on the summation order
        for (int t = t0 + lane; t < t1; t += 32) sum += (double)g[(size_t)t * p.Hv + hv];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (sum > WARMUP_LOG_EPS) flag = 1;
    }
    if (lane == 0) serial[(size_t)s * p.Hv + hv] = (uint8_t)flag;
}

cudaError_t launch_cp_flags(const Plan &p, const float *g, int seg_len, int n_seg, int warm, uint8_t *serial,
                            cudaStream_t st) {
    k_cp_flags<<<dim3(p.n_seqs, p.Hv), 32, 0, st>>>(p, g, seg_len, n_seg, warm, serial);
    return cudaGetLastError();
}

}  // namespace gdn
