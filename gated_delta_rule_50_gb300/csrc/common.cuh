// common.cuh -- shared host/device definitions of the gated delta rule CUDA library.
//
// Chunking: every sequence is cut into chunks of GDN_CHUNK = 64 tokens from its
// own start (the last chunk of a sequence may be shorter).  A "global chunk"
// index numbers the chunks of all sequences consecutively; in batch mode the
// chunks of sequence b are [b * NC, (b + 1) * NC) with NC = ceil(T / 64); in
// varlen mode their offsets live in a small device table built from
// cu_seqlens.
#pragma once
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int C = GDN_CHUNK;

// Device error word (first 4 bytes of every workspace).
enum : uint32_t { ERR_NONE = 0u, ERR_TIMEOUT = 1u };

struct Plan {
    int B, T, Hq, Hv, K, V, G;
    int n_seqs;
    int NC;             // chunks per sequence (batch mode)
    int total_chunks;   // chunks over all sequences
    int max_seq_chunks; // chunks of the longest sequence
    int max_seq_len;    // tokens of the longest sequence
    int cp_mode, warmup_chunks;
    const int32_t *cu;  // device cu_seqlens (varlen) or nullptr
    int32_t *chunk_off; // device [n_seqs + 1] chunk offsets (varlen) or nullptr
    gdn_dtype io;
    float scale;
    int out_f32;        // bf16 io: o, A, dq, dk, dv written as fp32 (checking mode)
    uint32_t *err;      // device error word
    // test aid (gdn_debug_set_wait): limit of the forward chain's device-side waits, and a chunk whose
    // k / q / operand-image load the chain's producer skips (-1: none)
    unsigned long long wait_ns;
    int drop_load_chunk;
};

struct SeqRange { int tok0, tok1, c0, c1; };  // token span and global chunk span

__host__ __device__ inline SeqRange seq_range(const Plan &p, int s) {
    SeqRange r;
    if (p.cu) {
        r.tok0 = p.cu[s]; r.tok1 = p.cu[s + 1];
        r.c0 = p.chunk_off[s]; r.c1 = p.chunk_off[s + 1];
    } else {
        r.tok0 = s * p.T; r.tok1 = (s + 1) * p.T;
        r.c0 = s * p.NC; r.c1 = (s + 1) * p.NC;
    }
    return r;
}

struct ChunkPos { int seq, tok0, len, local; };

// Global chunk -> (sequence, first token, length).  Varlen uses a binary search
// over the chunk-offset table.
__device__ inline ChunkPos chunk_pos(const Plan &p, int gc) {
    ChunkPos c;
    int s;
    if (p.cu) {
        int lo = 0, hi = p.n_seqs - 1;
        while (lo < hi) {  // last s with chunk_off[s] <= gc
            int mid = (lo + hi + 1) >> 1;
            if (p.chunk_off[mid] <= gc) lo = mid; else hi = mid - 1;
        }
        // skip empty sequences that share the same offset
        s = lo;
        while (s + 1 < p.n_seqs && p.chunk_off[s + 1] <= gc) ++s;
    } else {
        s = gc / p.NC;
    }
    SeqRange r = seq_range(p, s);
    c.seq = s;
    c.local = gc - r.c0;
    c.tok0 = r.tok0 + c.local * C;
    int rem = r.tok1 - c.tok0;
    c.len = rem < C ? rem : C;
    return c;
}

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Workspace carving helper: 256-byte aligned bump allocation inside a caller buffer.
struct Carve {
    size_t off = 0;
    template <typename T> size_t take(size_t count) {
        size_t o = off;
        off = (off + count * sizeof(T) + 255) & ~size_t(255);
        return o;
    }
};

}  // namespace gdn
