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
//
// The exact split (used when splitting is asked for without warmup) needs no
// decay: the end state of segment p is M_p S_p + h_p, with h_p the segment run
// from a zero state and M_p the segment run with v = 0 from the identity (both
// by the chain kernel), and k_cp_combine scans S_(p+1) = M_p S_p + h_p.
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

// S_(p+1) = M_p S_p + h_p over the segments of one (sequence, value head), S_0 = h0 (or 0), in fp32;
// writes the starting state of every segment after the first.  The value columns are independent:
// grid (n_seqs, Hv, 8) gives each CTA a block of 16 columns; 256 threads, each 8 outputs of a row.
constexpr int CB_COLS = 16, CB_LD = 129;
__global__ void __launch_bounds__(256) k_cp_combine(Plan p, const float *__restrict__ h0, const float *__restrict__ seg_h,
                                                    const float *__restrict__ seg_M, int seg_len, int n_seg,
                                                    float *__restrict__ seg_states) {
    extern __shared__ float smc[];
    float *Ms = smc, *Sb = smc + 128 * CB_LD;  // M_p [128][129]; state block [128][16]
    const int s = blockIdx.x, hv = blockIdx.y, c0 = CB_COLS * blockIdx.z, t = threadIdx.x;
    const SeqRange sr = seq_range(p, s);
    const int nseg_s = (sr.c1 - sr.c0 + seg_len - 1) / seg_len;
    const size_t base = ((size_t)s * p.Hv + hv) * n_seg, KV = (size_t)p.K * p.V;
    for (int idx = t; idx < 128 * CB_COLS; idx += 256) {
        const int k = idx / CB_COLS, c = idx % CB_COLS;
        Sb[idx] = h0 ? h0[((size_t)s * p.Hv + hv) * KV + (size_t)k * p.V + c0 + c] : 0.f;
    }
    const int r = t >> 1, ce = 8 * (t & 1);
    for (int pp = 0; pp + 1 < nseg_s; ++pp) {
        const float *M = seg_M + (base + pp) * KV;
        const float *hp = seg_h + (base + pp) * KV;
        __syncthreads();  // the previous step's reads of Ms are done
        for (int idx = t; idx < 128 * 32; idx += 256) {
            const int k = idx >> 5, q4 = idx & 31;
            const float4 w = reinterpret_cast<const float4 *>(M + (size_t)k * 128)[q4];
            float *d = Ms + k * CB_LD + 4 * q4;
            d[0] = w.x; d[1] = w.y; d[2] = w.z; d[3] = w.w;
        }
        __syncthreads();
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = hp[(size_t)r * p.V + c0 + ce + e];
#pragma unroll 4
        for (int j = 0; j < 128; ++j) {
            const float m = Ms[r * CB_LD + j];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(m, Sb[j * CB_COLS + ce + e], acc[e]);
        }
        __syncthreads();  // every read of the old state block is done
        float *out = seg_states + (base + pp + 1) * KV + (size_t)r * p.V + c0 + ce;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            Sb[r * CB_COLS + ce + e] = acc[e];
            out[e] = acc[e];
        }
    }
}

cudaError_t launch_cp_combine(const Plan &p, const float *h0, const float *seg_h, const float *seg_M, int seg_len,
                              int n_seg, float *seg_states, cudaStream_t st) {
    const int smem = (128 * CB_LD + 128 * CB_COLS) * 4;
    cudaError_t e = cudaFuncSetAttribute(k_cp_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k_cp_combine<<<dim3(p.n_seqs, p.Hv, p.V / CB_COLS), 256, smem, st>>>(p, h0, seg_h, seg_M, seg_len, n_seg,
                                                                         seg_states);
    return cudaGetLastError();
}

}  // namespace gdn
