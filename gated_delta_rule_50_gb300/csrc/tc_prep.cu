// tc_prep.cu -- per-chunk preparation for the tensor-core chain kernels (bf16 io,
// K = V = 128, chunk 64): the gate cumsum, L, A = (I + L)^{-1} and P, for every
// chunk at once.
//
// These are the intra-chunk quantities of the chunked form (the "A matrix" step
// of the pages' step list; FlashQLA blog post, section 2).  None of them depends
// on the state, so they are computed here, fully in parallel over chunks and
// heads, and the serial state chains only copy them in.  One CTA per (chunk,
// q/k head) forms K K^T and Q K^T once on the tensor cores and loops over the
// group's value heads:
//
//   gam   chunk-local inclusive cumsum of g (or given, for the backward),
//   L     = strict_lower(diag(beta) (D o K K^T)),  D_ri = exp(gam_r - gam_i),
//   A     = (I + L)^{-1}          (blocked, in place, fp32),
//   P     = D o Q K^T             (lower, diagonal included).
//
// Per (chunk, value head) it writes a 32 KB operand image -- A hi, A lo, P hi,
// P lo, each a 64 x 64 bf16 tile in the 128-byte-swizzled K-major layout the
// MMAs read (row r at r * 128, 16-byte chunk c at position c ^ (r & 7)) -- and a
// 1 KB vector block {gam, exp(gam), exp(gam_last - gam), beta} x 64, ready for
// plain bulk copies.  Optionally g_cum, A in the io dtype and fp32 A / P.  Each
// hi / lo pair is staged in shared memory and leaves by two 8 KB bulk copies (the
// P pair while the inverse runs, the A pair while the next head starts): per-thread
// 16-byte stores, each warp store touching 32 rows 128 bytes apart, cost 8 % more.
// The fp32 L / A matrix has an even row stride so that the inverse's block products
// and the L and A rows move pairs of values per shared-memory access.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int DK = 128;
constexpr int NT = 128;

// The k / q tiles are dead once K K^T and Q K^T are in TMEM, so the fp32 scratch reuses their space.
constexpr uint32_t S_KQ = 0;                          // [kb0: K 8K, Q 8K][kb1: K 8K, Q 8K]
constexpr int LMS = 66;                               // row stride of Lm (even: 8-byte row pairs)
constexpr uint32_t S_LM = 0;                          // fp32 [64][LMS]: L, then A in place
constexpr uint32_t S_VEC = S_LM + 64 * LMS * 4;       // gam, Gam, E, beta (64 each)
constexpr int GB_HEADS = 4;
constexpr uint32_t S_GB = S_VEC + 4 * 64 * 4;         // g (or g_cum) and beta of up to GB_HEADS value heads x 64 rows
constexpr uint32_t S_IMG = S_GB + 2 * GB_HEADS * 64 * 4;  // staging of a hi / lo operand image pair (2 x 8 KB)
// fp32 3 x [16][18], used only between the diagonal blocks and the end of the inverse, when no image is staged
constexpr uint32_t S_TB = S_IMG;
constexpr uint32_t S_BAR = S_IMG + 16384;
constexpr uint32_t S_MISC = S_BAR + 16;
constexpr uint32_t SMEM_BYTES = S_MISC + 32 + 1024;
static_assert(S_IMG % 16 == 0 && S_BAR >= 32768 && S_TB + 3 * 16 * 18 * 4 <= S_BAR, "shared memory map");
static_assert(SMEM_BYTES + 1024 <= 233472 / 6, "six CTAs per SM");

constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);

struct PrepArgs {
    const float *g, *beta;
    int g_is_cum;
    float *g_cum;
    void *A;  // [B,T,Hv,64]: bf16, or fp32 when p.out_f32
    float *A32, *P32;
    unsigned char *tiles;  // [chunks][Hv] x 32 KB
    float *vecs;           // [chunks][Hv] x 256
};

__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return sdesc_sw128(a, 16, 1024); }

// Blocked in-place inverse of the unit lower-triangular I + L held in Lm
// ([64][LMS], strictly lower part = L, rest 0); afterwards Lm = (I + L)^{-1}.
// Column blocks of 16 are processed right to left so that the inverted A_IK
// (K > J) and the untouched L_KJ are both available:
//     A_IJ = -(sum_{K=J+1}^{I} A_IK L_KJ) A_JJ.
// Called by the 128 prep threads (named barrier 1).
__device__ void blocked_inverse(float *Lm, float *Tb, int pt) {
    constexpr int LS = LMS, TS = 18;
    float x[16];
    const int b = pt >> 4, jc = pt & 15, base = 16 * b;
    if (pt < 64) {  // diagonal blocks: forward substitution, one column per thread
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i >= jc && i < r) s = fmaf(Lm[(base + r) * LS + base + i], x[i], s);
            x[r] = (r < jc) ? 0.f : (r == jc ? 1.f : -s);
        }
    }
    named_bar(1, 128);
    if (pt < 64) {
#pragma unroll
        for (int r = 0; r < 16; ++r) Lm[(base + r) * LS + base + jc] = x[r];
    }
    if (pt == 0) bulk_wait_read_all();  // the P image has left the staging buffer, which takes A's next
    named_bar(1, 128);
    // Off-diagonal blocks, right to left.  Warp w computes block row I = J + 1 + w as register tiles: lane
    // (rq, cq) owns rows 2 rq, 2 rq + 1 and columns 4 cq .. 4 cq + 3 of the block, reading pairs of
    // adjacent values with 8-byte shared loads (three per 8 FMAs).  Each element is summed in the order K,
    // then k, as the textbook block recursion writes it.
    const int w = pt >> 5, ln = pt & 31, rq = ln >> 2, cq = ln & 3;
    float *Tw = Tb + w * 16 * TS;  // this warp's 16 x 16 T block
    auto ld2 = [](const float *p) { return *reinterpret_cast<const float2 *>(p); };
    auto st2 = [](float *p, float a, float b) { *reinterpret_cast<float2 *>(p) = make_float2(a, b); };
    for (int J = 2; J >= 0; --J) {
        const int I = J + 1 + w;
        if (I <= 3) {
            float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int K = J + 1; K <= I; ++K) {  // T_IJ = sum_K A_IK L_KJ
                const float *arow = Lm + (16 * I + 2 * rq) * LS + 16 * K;
                const float *lcol = Lm + (16 * K) * LS + 16 * J + 4 * cq;
#pragma unroll
                for (int k = 0; k < 16; k += 2) {
                    const float2 xa = ld2(arow + k), xb = ld2(arow + LS + k);
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const float x0 = kk ? xa.y : xa.x, x1 = kk ? xb.y : xb.x;
                        const float2 ya = ld2(lcol + (k + kk) * LS), yb = ld2(lcol + (k + kk) * LS + 2);
                        const float y[4] = {ya.x, ya.y, yb.x, yb.y};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            t0[e] = fmaf(x0, y[e], t0[e]);
                            t1[e] = fmaf(x1, y[e], t1[e]);
                        }
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                st2(Tw + (2 * rq) * TS + 4 * cq + e, t0[e], t0[e + 1]);
                st2(Tw + (2 * rq + 1) * TS + 4 * cq + e, t1[e], t1[e + 1]);
            }
        }
        named_bar(1, 128);  // every L_KJ has been read before the A_IJ below overwrite them
        if (I <= 3) {
            float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};  // A_IJ = -T_IJ A_JJ
            const float *acol = Lm + (16 * J) * LS + 16 * J + 4 * cq;
#pragma unroll
            for (int k = 0; k < 16; k += 2) {
                const float2 xa = ld2(Tw + (2 * rq) * TS + k), xb = ld2(Tw + (2 * rq + 1) * TS + k);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const float x0 = kk ? xa.y : xa.x, x1 = kk ? xb.y : xb.x;
                    const float2 ya = ld2(acol + (k + kk) * LS), yb = ld2(acol + (k + kk) * LS + 2);
                    const float y[4] = {ya.x, ya.y, yb.x, yb.y};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        o0[e] = fmaf(x0, y[e], o0[e]);
                        o1[e] = fmaf(x1, y[e], o1[e]);
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 4; e += 2) {
                st2(Lm + (16 * I + 2 * rq) * LS + 16 * J + 4 * cq + e, -o0[e], -o0[e + 1]);
                st2(Lm + (16 * I + 2 * rq + 1) * LS + 16 * J + 4 * cq + e, -o1[e], -o1[e + 1]);
            }
        }
        named_bar(1, 128);
    }
}

// 8 consecutive values of row r (chunk ch) of a 64-wide tile -> hi and lo 16-byte chunks of the image.
__device__ __forceinline__ void put_split_chunk(unsigned char *hi_tile, unsigned char *lo_tile, int r, int ch,
                                                const float *x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_pair(x[2 * i], x[2 * i + 1], h[i], l[i]);
    const uint32_t off = (uint32_t)r * 128u + ((uint32_t)(ch ^ (r & 7)) << 4);
    *reinterpret_cast<uint4 *>(hi_tile + off) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(lo_tile + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

__global__ void __launch_bounds__(NT, 6)
k_tc_prep(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q, Plan p, PrepArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + S_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *Lm = reinterpret_cast<float *>(sm + S_LM), *Tb = reinterpret_cast<float *>(sm + S_TB);
    float *gam = reinterpret_cast<float *>(sm + S_VEC), *Gm = gam + 64, *Ev = gam + 128, *bet = gam + 192;
    float *wtot = reinterpret_cast<float *>(misc + 4);
    const uint32_t bar_tma = sb + S_BAR, bar_mma = sb + S_BAR + 8;

    const int gc = blockIdx.x, hq = blockIdx.y;
    const ChunkPos cp = chunk_pos(p, gc);
    const int tok0 = cp.tok0, n = cp.len;

    if (t == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sb + S_MISC, 64);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    bool ok = true;
    // g (or g_cum) and beta of row t (threads 0..63) for every value head of the group (up to GB_HEADS;
    // adjacent in memory), loaded now so that the loads overlap the k / q copy and the K K^T product and
    // parked in shared memory once that space is free; rows past the chunk end hold the last value
    const bool gb_staged = p.G <= GB_HEADS;
    float gpre[GB_HEADS], bpre[GB_HEADS];
    if (gb_staged && t < 64) {
        const size_t row = (size_t)(tok0 + (t < n ? t : n - 1)) * p.Hv + (size_t)hq * p.G;
#pragma unroll
        for (int gg = 0; gg < GB_HEADS; ++gg)
            if (gg < p.G) {
                gpre[gg] = (a.g_is_cum || t < n) ? a.g[row + gg] : 0.f;
                bpre[gg] = t < n ? a.beta[row + gg] : 0.f;
            }
    }
    // K K^T (lanes 0..63) and Q K^T (lanes 64..127) of this chunk: D1 = [K; Q] K^T
    if (t == 0) {
        mbar_arrive_expect_tx(bar_tma, 32768);
        tma_load_3d(sb + S_KQ, &tm_k, bar_tma, 0, hq, tok0);
        tma_load_3d(sb + S_KQ + 8192, &tm_q, bar_tma, 0, hq, tok0);
        tma_load_3d(sb + S_KQ + 16384, &tm_k, bar_tma, 64, hq, tok0);
        tma_load_3d(sb + S_KQ + 24576, &tm_q, bar_tma, 64, hq, tok0);
    }
    if (warp == 0) ok = mbar_wait_warp(bar_tma, 0, abort_flag);
    ok = __syncthreads_and(ok) != 0;
    if (ok && t == 0) {
        tc_fence_after();
        for (int blk = 0; blk < 2; ++blk)
            mma_chain<4, 2, 2>(tmem, kdesc(sb + S_KQ + 16384 * blk), kdesc(sb + S_KQ + 16384 * blk), ID_N64, blk);
        mma_commit(bar_mma);
    }
    if (ok && warp == 0) ok = mbar_wait_warp(bar_mma, 0, abort_flag);
    ok = __syncthreads_and(ok) != 0;  // the MMA has read the k / q tiles: their space is scratch from here
    tc_fence_after();
    float *gst = reinterpret_cast<float *>(sm + S_GB), *bst = gst + GB_HEADS * 64;
    if (gb_staged && t < 64) {  // each thread reads back only its own entries
#pragma unroll
        for (int gg = 0; gg < GB_HEADS; ++gg)
            if (gg < p.G) {
                gst[gg * 64 + t] = gpre[gg];
                bst[gg * 64 + t] = bpre[gg];
            }
    }
    for (int g = 0; ok && g < p.G; ++g) {
        const int hv = hq * p.G + g;
        const size_t unit = (size_t)gc * p.Hv + hv;
        // gate cumsum over rows 0..63 (threads 0..63); rows past the chunk end hold the last value
        float x = 0.f, bv = 0.f;
        if (t < 64) {
            if (gb_staged) {
                x = gst[g * 64 + t];
                bv = bst[g * 64 + t];
            } else {
                const size_t gi = (size_t)(tok0 + (t < n ? t : n - 1)) * p.Hv + hv;
                x = (a.g_is_cum || t < n) ? a.g[gi] : 0.f;
                bv = t < n ? a.beta[gi] : 0.f;
            }
            if (!a.g_is_cum) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                if (t == 31) *wtot = x;
            }
        }
        __syncthreads();
        if (t < 64) {
            if (!a.g_is_cum && t >= 32) x += *wtot;
            gam[t] = x;
            bet[t] = bv;
            if (t < n && a.g_cum) a.g_cum[(size_t)(tok0 + t) * p.Hv + hv] = x;
        }
        if (t == 0) bulk_wait_read_all();  // the previous head's A image has left the staging buffer
        __syncthreads();
        const float glast = gam[n - 1];
        if (t < 64) {
            Gm[t] = t < n ? __expf(gam[t]) : 0.f;
            Ev[t] = t < n ? __expf(glast - gam[t]) : 0.f;
        }
        unsigned char *img = a.tiles + unit * 32768;
        // this thread's row of K K^T (t < 64) or Q K^T (t >= 64), read from TMEM in two 32-column halves
        // (half a row at a time keeps the register footprint small)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t raw[32];
            tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * half, raw);
            if (t < 64) {  // L = beta D o K K^T, strictly lower
                const int r = t;
                const float gr = gam[r], br = bet[r];
#pragma unroll
                for (int k = 0; k < 32; k += 2) {  // pairs of entries: 8-byte stores
                    const int i = 32 * half + k;
                    const float l0 = (i < r && r < n) ? br * __expf(gr - gam[i]) * __uint_as_float(raw[k]) : 0.f;
                    const float l1 =
                        (i + 1 < r && r < n) ? br * __expf(gr - gam[i + 1]) * __uint_as_float(raw[k + 1]) : 0.f;
                    *reinterpret_cast<float2 *>(Lm + r * LMS + i) = make_float2(l0, l1);
                }
            } else {  // P = D o Q K^T, lower incl. diagonal -> image (and fp32 copy)
                const int r = t - 64;
                const float gr = gam[r];
                float *p32 = a.P32 ? a.P32 + unit * C * C + (size_t)r * C : nullptr;
#pragma unroll
                for (int cq = 0; cq < 4; ++cq) {
                    const int ch = 4 * half + cq;
                    float pv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * ch + e;
                        pv[e] = (i <= r && r < n) ? __expf(gr - gam[i]) * __uint_as_float(raw[8 * cq + e]) : 0.f;
                    }
                    put_split_chunk(sm + S_IMG, sm + S_IMG + 8192, r, ch, pv);
                    if (p32) {
                        reinterpret_cast<float4 *>(p32)[2 * ch] = make_float4(pv[0], pv[1], pv[2], pv[3]);
                        reinterpret_cast<float4 *>(p32)[2 * ch + 1] = make_float4(pv[4], pv[5], pv[6], pv[7]);
                    }
                }
            }
        }
        if (t >= 64) fence_proxy_async_smem();  // staged P image -> bulk copy
        __syncthreads();
        if (t == 0) {
            bulk_store(img + 16384, sb + S_IMG, 8192);
            bulk_store(img + 24576, sb + S_IMG + 8192, 8192);
            bulk_commit();
        }
        blocked_inverse(Lm, Tb, t);
        {  // A -> image, io-dtype output and fp32 copy: thread holds half a row
            const int r = t >> 1, hh = t & 1;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int ch = 4 * hh + q;
                float vals[8];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float2 v2 = *reinterpret_cast<const float2 *>(Lm + r * LMS + 8 * ch + e);
                    vals[e] = v2.x;
                    vals[e + 1] = v2.y;
                }
                put_split_chunk(sm + S_IMG, sm + S_IMG + 8192, r, ch, vals);
                if (a.A && r < n) {
                    const size_t ao = ((size_t)(tok0 + r) * p.Hv + hv) * C + 8 * ch;
                    if (p.out_f32) {
                        float4 *d = reinterpret_cast<float4 *>(static_cast<float *>(a.A) + ao);
                        d[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
                        d[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
                    } else {
                        const uint4 pk = make_uint4(pack_bf16(vals[0], vals[1]), pack_bf16(vals[2], vals[3]),
                                                    pack_bf16(vals[4], vals[5]), pack_bf16(vals[6], vals[7]));
                        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.A) + ao) = pk;
                    }
                }
                if (a.A32) {
                    float4 *d = reinterpret_cast<float4 *>(a.A32 + unit * C * C + (size_t)r * C + 8 * ch);
                    d[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
                    d[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
                }
            }
        }
        if (t < 64)  // vector block: 256 floats
            reinterpret_cast<float4 *>(a.vecs + unit * 256)[t] = reinterpret_cast<const float4 *>(gam)[t];
        fence_proxy_async_smem();  // staged A image -> bulk copy
        __syncthreads();  // Lm, vectors reused by the next head
        if (t == 0) {
            bulk_store(img, sb + S_IMG, 8192);
            bulk_store(img + 8192, sb + S_IMG + 8192, 8192);
            bulk_commit();
        }
    }
    if (t == 0) bulk_wait_all();
    if (!ok && t == 0) {
        if (atomicCAS(p.err + 1, 0u, 301u) == 0u) {
            p.err[2] = (uint32_t)gc;
            p.err[4] = blockIdx.x + blockIdx.y * gridDim.x;
        }
        atomicOr(p.err, ERR_TIMEOUT);
        mbar_drain(bar_tma, 0);
        mma_commit(bar_mma);
        mbar_drain(bar_mma, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 64);
}

}  // namespace

cudaError_t launch_tc_prep(const Plan &p, const void *q, const void *k, const float *g, bool g_is_cum,
                           const float *beta, float *g_cum, void *A, float *A32, float *P32, unsigned char *tiles,
                           float *vecs, cudaStream_t st) {
    if (p.total_chunks == 0) return cudaSuccess;
    CUtensorMap tk, tq;
    if (!make_head_map(&tk, k, p.Hq, p) || !make_head_map(&tq, q, p.Hq, p)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_tc_prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    PrepArgs a;
    a.g = g;
    a.beta = beta;
    a.g_is_cum = g_is_cum ? 1 : 0;
    a.g_cum = g_cum;
    a.A = A;
    a.A32 = A32;
    a.P32 = P32;
    a.tiles = tiles;
    a.vecs = vecs;
    dim3 grid(p.total_chunks, p.Hq);
    k_tc_prep<<<grid, NT, SMEM_BYTES, st>>>(tk, tq, p, a);
    return cudaGetLastError();
}

}  // namespace gdn
