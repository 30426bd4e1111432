// pad.cu -- zero padding of 64-wide heads to the 128-wide tensor-core tiles, and the slices back.
//
// A head size of 64 (K, V or both) runs through the 128-wide kernels on copies whose extra columns
// are zero.  This is exact: with k, q zero past column K and v, the initial state zero past K rows and
// V columns, the state keeps zeros there for every token (each update adds k (.)^T and scales), so the
// outputs' leading columns are the 64-wide results and the trailing ones are discarded.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch.h"

namespace gdn {
namespace {

constexpr int W = 128;  // padded width

// dst [rows][128] <- src [rows][d] (d = 64 or 128), 16-byte chunks, zeros past d.
__global__ void k_pad_rows(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t rows, int d) {
    const size_t n = rows * (W / 8), cpr = (size_t)d / 8;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i >> 4, c = i & 15;
        dst[i] = c < cpr ? src[r * cpr + c] : make_uint4(0, 0, 0, 0);
    }
}

// dst [rows][d] <- the leading d columns of src [rows][128]; cpr = 16-byte chunks per dst row, spr per src row.
__global__ void k_slice_rows(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t rows, size_t cpr,
                             size_t spr) {
    const size_t n = rows * cpr;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / cpr, c = i - r * cpr;
        dst[i] = src[r * spr + c];
    }
}

// dst [n][128][128] <- src [n][K][V] fp32, zeros outside K x V.
__global__ void k_pad_states(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n, int K, int V) {
    const size_t total = n * W * (W / 4), vq = (size_t)V / 4;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t c = i & 31, r = (i >> 5) & 127, s = i >> 12;
        dst[i] = (r < (size_t)K && c < vq) ? src[(s * K + r) * vq + c] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// dst [n][K][V] <- the leading K x V block of src [n][128][128].
__global__ void k_slice_states(const float4 *__restrict__ src, float4 *__restrict__ dst, size_t n, int K, int V) {
    const size_t vq = (size_t)V / 4, total = n * K * vq;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t c = i % vq, rs = i / vq, r = rs % K, s = rs / K;
        dst[i] = src[(s * W + r) * (W / 4) + c];
    }
}

unsigned grid_for(size_t items) {
    const size_t b = (items + 255) / 256;
    return (unsigned)(b < 152 * 16 ? (b ? b : 1) : 152 * 16);
}

}  // namespace

cudaError_t launch_pad_rows(const void *src, void *dst, size_t rows, int d, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    k_pad_rows<<<grid_for(rows * 16), 256, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), rows, d);
    return cudaGetLastError();
}

cudaError_t launch_slice_rows(const void *src, void *dst, size_t rows, int d, int elem_bytes, cudaStream_t st) {
    if (rows == 0) return cudaSuccess;
    const size_t cpr = (size_t)d * elem_bytes / 16, spr = (size_t)W * elem_bytes / 16;
    k_slice_rows<<<grid_for(rows * cpr), 256, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst),
                                                       rows, cpr, spr);
    return cudaGetLastError();
}

cudaError_t launch_pad_states(const float *src, float *dst, size_t n, int K, int V, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    k_pad_states<<<grid_for(n * 4096), 256, 0, st>>>(reinterpret_cast<const float4 *>(src),
                                                     reinterpret_cast<float4 *>(dst), n, K, V);
    return cudaGetLastError();
}

cudaError_t launch_slice_states(const float *src, float *dst, size_t n, int K, int V, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    k_slice_states<<<grid_for(n * (size_t)K * V / 4), 256, 0, st>>>(reinterpret_cast<const float4 *>(src),
                                                                     reinterpret_cast<float4 *>(dst), n, K, V);
    return cudaGetLastError();
}

}  // namespace gdn
