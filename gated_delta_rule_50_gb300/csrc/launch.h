// launch.h -- internal host launchers shared between the C ABI and the kernel files.
#pragma once
#include <cuda_runtime.h>

#include <cuda.h>

#include "common.cuh"

namespace gdn {

cudaError_t launch_chunk_table(const Plan &p, cudaStream_t st);

// CUDA-core (FFMA) path
cudaError_t launch_simt_prep(const Plan &p, const void *q, const void *k, const float *g, int g_is_cum,
                             const float *beta, float *g_cum, void *A_out, double *gam64, float *A32,
                             float *P32, cudaStream_t st);
cudaError_t launch_simt_scan(const Plan &p, const void *q, const void *k, const void *v, const float *beta,
                             const double *gam64, const float *A32, const float *P32, const float *h0,
                             void *o, float *h, float *ht, cudaStream_t st);
cudaError_t launch_simt_dscan(const Plan &p, const void *q, const void *k, const void *d_o, const float *beta,
                              const double *gam64, const float *A32, const float *P32, const float *dht,
                              float *dSe, float *dh0, cudaStream_t st);
cudaError_t launch_simt_bwd_intra(const Plan &p, const void *q, const void *k, const void *v, const void *d_o,
                                  const float *beta, const double *gam64, const float *A32,
                                  const float *P32, const float *hbuf, const float *dSe, void *dq, void *dk,
                                  void *dv, float *dbeta, float *dg, cudaStream_t st);

// Sequence splitting: each sequence is cut into n_seg segments of
// seg_len chunks.  Warmup: a CP_WARM launch computes every segment's starting state by running `warm`
// chunks from a zero state.  Exact: a CP_SEG launch runs every segment twice -- from a zero state with
// the real v (its contribution h_p) and with v = 0 from the identity (its transition M_p, since the
// recurrence is linear in (v, S)) -- and launch_cp_combine scans S_(p+1) = M_p S_p + h_p.  A CP_MAIN
// launch then runs the segments from their starting states.
enum { CP_WARM = 1, CP_MAIN = 2, CP_SEG = 3 };
struct CpSplit {
    int seg_len, n_seg, warm, mode;
    const uint8_t *serial;  // [n_seqs][Hv] heads whose warmup windows do not decay enough (warmup only)
    float *seg_states;      // [n_seqs][Hv][n_seg][K][V]
    float *seg_h, *seg_M;   // exact: [n_seqs][Hv][n_seg][K][V] contributions and [..][K][K] transitions
};
cudaError_t launch_cp_combine(const Plan &p, const float *h0, const float *seg_h, const float *seg_M, int seg_len,
                              int n_seg, float *seg_states, cudaStream_t st);
bool cp_trigger(const Plan &p);                  // the pages' small batch x heads rule
void cp_geometry(const Plan &p, int *seg_len, int *n_seg);
cudaError_t launch_cp_flags(const Plan &p, const float *g, int seg_len, int n_seg, int warm, uint8_t *serial,
                            cudaStream_t st);

// tensor-core (tcgen05) fused forward: bf16 io, K = V = 128
bool tc_fwd_supported(const Plan &p);
// Per (chunk, value head): A / P operand images (32 KB) and gate vectors (1 KB); see tc_prep.cu.
constexpr size_t TC_TILE_BYTES = 32768, TC_VEC_FLOATS = 256;
cudaError_t launch_tc_prep(const Plan &p, const void *q, const void *k, const float *g, bool g_is_cum,
                           const float *beta, float *g_cum, void *A, float *A32, float *P32, unsigned char *tiles,
                           float *vecs, cudaStream_t st);
cudaError_t launch_tc_fwd(const Plan &p, const void *q, const void *k, const void *v, const unsigned char *tiles,
                          const float *vecs, const float *h0, void *o, float *h, float *ht, cudaStream_t st,
                          const CpSplit *cp = nullptr);

// Zero padding of 64-wide heads to the 128-wide tensor-core tiles (pad.cu): rows [rows][d] bf16 ->
// [rows][128]; slices back [rows][128] -> [rows][d] of bf16 or fp32 elements; states [n][K][V] fp32 <->
// [n][128][128].  Pointers 16-byte aligned.
cudaError_t launch_pad_rows(const void *src, void *dst, size_t rows, int d, cudaStream_t st);
cudaError_t launch_slice_rows(const void *src, void *dst, size_t rows, int d, int elem_bytes, cudaStream_t st);
cudaError_t launch_pad_states(const float *src, float *dst, size_t n, int K, int V, cudaStream_t st);
cudaError_t launch_slice_states(const float *src, float *dst, size_t n, int K, int V, cudaStream_t st);

// TMA map of a [tokens][heads][128] bf16 tensor (64 x 1 x 64 boxes, 128-byte swizzle)
bool make_head_map(CUtensorMap *m, const void *ptr, int heads, const Plan &p);
// TMA map of per-chunk fp32 states [units][128 keys][128 values] as a 2-D tensor of units x 128 rows:
// boxes of 32 values x 128 keys (16 KB), 128-byte swizzle
bool make_state_map(CUtensorMap *m, const float *ptr, size_t units);

// tensor-core reverse scan of the state gradient: bf16 io, K = V = 128
cudaError_t launch_tc_dscan(const Plan &p, const void *q, const void *k, const void *d_o, const float *g_cum,
                            const float *beta, const unsigned char *tiles, const float *dht, float *dSe, float *dh0,
                            cudaStream_t st, const CpSplit *cp = nullptr);

// tensor-core per-chunk gradients (dq, dk, dv, dbeta, dg): bf16 io, K = V = 128
cudaError_t launch_tc_bwd_intra(const Plan &p, const void *q, const void *k, const void *v, const void *d_o,
                                const unsigned char *tiles, const float *vecs, const float *hbuf, const float *dSe,
                                void *dq, void *dk, void *dv, float *dbeta, float *dg, cudaStream_t st);

}  // namespace gdn
