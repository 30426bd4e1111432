// tc_bwd_intra.cu -- tensor-core per-chunk gradients of the chunked gated delta
// rule (bf16 io, K = V = 128, chunk 64).
//
// One CTA per (chunk, q/k head) loops over the value heads of the group.  It
// needs the chunk-entry state h and the state gradient at the chunk end dSe
// (both from the scans) and the chunk matrices A = (I + L)^{-1}, P = D o Q K^T.
// Per value head, with X^T denoting value-major tiles ([v][c]):
//
//   KS^T = h^T K^T,  QS^T = h^T Q^T                       R = diag(beta)(V - diag(Gam) KS)
//   Dl^T = R^T A^T,  KdS^T = dSe^T K^T,  PdO^T = dO^T P   dDl = scale P^T dO + diag(E) K dSe
//   dR^T = dDl^T A                                        dV = diag(beta) dR
//   [Dl; R] dO^T -> dP^T (rows 0..63),  [Dl; R] dDl^T -> dA^T (rows 64..127)
//   dL = -(A^T dA A^T) strictly lower                     (Z^T = A dA~^T, then dL^T = -Z^T A)
//   dq^T += h (scale Gam o dO)^T + K^T dQK^T               dQK = D o scale dP
//   dk^T += dSe (E o Dl)^T - h (beta Gam o dR)^T + Q^T dQK + K^T (dKK + dKK^T),  dKK = beta D o dL
//   (the two h products run as one N = 128 product over the adjacent dq^T, dk^T accumulators)
//
// and the gate / beta gradients as row sums (dg is the reverse cumsum of dgam
// inside the chunk).  dq and dk accumulate over the group's value heads in
// TMEM.  Every derived operand is split into bf16 hi + lo (3 products when both
// sides are derived); scalings are folded into the operand tiles so that the
// TMEM accumulation is exact in structure.
//
// The kernel is phase-sequential: 512 threads (each TMEM lane quarter is
// served by four warps, one per 16 chunk rows), one of them issues the MMAs of
// a phase and all wait on one mbarrier before the next phase; work that needs
// no result of the running MMAs (dv store-out beside Z = A dA~^T, the (E Dl)^T
// tile beside A^T Z, the dbeta / dg reduction, and the next value head's h:
// copied in and staged in TMEM once the
// h products of the dq / dk accumulation are done, while the rest of it runs)
// proceeds meanwhile.  The k, q, dO and v chunk tiles arrive by TMA, the
// A / P operand images and gate vectors by bulk copy, h and dSe by TMA as
// 128-byte-swizzled fp32 boxes (value-major reads for the TMEM A operands) and
// again by coalesced row loads transposed in shared memory (key-major, for the
// dq / dk products); dv leaves through a shared-memory staging tile in 16-byte
// stores.  Many CTAs (one per chunk and q/k head) keep the GPU busy.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int DK = 128, DV = 128;
constexpr int NT = 512;     // 16 warps: TMEM lane quarter = warp & 3, column quarter = warp >> 2
constexpr int NW = NT / 32;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t S_KQ = 0;         // [kb0: K 8K, Q 8K][kb1: K 8K, Q 8K]
constexpr uint32_t S_DO = 32768;     // dO [r][v] 2 x 8K; later dQK hi / lo [r][i]
constexpr uint32_t S_A = 49152;      // A hi / lo [r][i]
constexpr uint32_t S_P = 65536;      // P hi / lo [r'][r]; later (dKK + dKK^T) hi / lo
constexpr uint32_t S_DR = 81920;     // Dl^T hi | R^T hi | Dl^T lo | R^T lo ([v][i], 16K each); later scale Gam dO, Y
constexpr uint32_t S_DD = 147456;    // V [r][v] (TMA); dDl^T hi / lo [v][r]; dv staging; (E Dl)^T hi / lo [v][i]
constexpr uint32_t S_F = 180224;     // fp32 [64][65]: dA, then dL
constexpr uint32_t S_F2 = S_F + 64 * 65 * 4;   // fp32 [64][65]: dQK staging
constexpr uint32_t S_VEC = S_F2 + 64 * 65 * 4; // gam, Gam, E, beta, beta Gam (64 each); per-warp partial sums
constexpr uint32_t S_BAR = S_VEC + (5 * 64 + 2 * NW * 64 + 2 * NW) * 4;
constexpr uint32_t S_MISC = S_BAR + 40;
constexpr uint32_t S_TOTAL = S_MISC + 16;
constexpr uint32_t SMEM_BYTES = S_TOTAL + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory");
static_assert(S_F + 2048 * NW <= S_VEC, "transpose buffers fit in the fp32 scratch");
static_assert(S_P == S_A + 16384 && S_VEC % 16 == 0, "operand image and vector copies");
static_assert(S_DR % 1024 == 0 && S_F % 1024 == 0 && S_F + 32768 <= S_VEC, "state boxes (128-byte swizzle)");

// TMEM columns
constexpr uint32_t C_DQ = 0, C_DK = 64, C_HT = 128, C_KS = 256, C_QS = 320, C_DL = 384, C_DR = 448;

constexpr uint32_t ID_KK = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_MK = idesc_bf16(128, 64, 1, 0);
constexpr uint32_t ID_MM = idesc_bf16(128, 64, 1, 1);
constexpr uint32_t ID_KM = idesc_bf16(128, 64, 0, 1);
constexpr uint32_t ID_N128 = idesc_bf16(128, 128, 0, 0);
constexpr uint32_t ID_KM128 = idesc_bf16(128, 128, 0, 1);
static_assert(C_QS == C_KS + 64, "KS and QS accumulators must be adjacent");

struct IntraArgs {
    const unsigned char *tiles;  // [chunks][Hv] x 32 KB: A hi / lo, P hi / lo operand images
    const float *vecs;           // [chunks][Hv] x {gam, Gam, E, beta} x 64
    const float *hbuf, *dSe;
    void *dq, *dk, *dv;  // bf16, or fp32 in the checking mode (p.out_f32)
    float *dbeta, *dg;
};

__device__ __forceinline__ uint64_t kdesc(uint32_t a) { return sdesc_sw128(a, 16, 1024); }
__device__ __forceinline__ uint64_t mdesc(uint32_t a, uint32_t lbo) { return sdesc_sw128(a, lbo, 1024); }

// x[j] (16 values) on every lane -> every lane l returns the sum over all 32 lanes of x[l & 15].
__device__ __forceinline__ float warp_transpose_sum16(float (&x)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < o; ++j) {
            const float send = up ? x[j] : x[j + o];
            const float keep = up ? x[j + o] : x[j];
            x[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 16);
}

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// element (row, col) of a 64-wide bf16 swizzled tile
__device__ __forceinline__ float tile_at(const unsigned char *sm, uint32_t off, int row, int col) {
    const uint32_t o = (uint32_t)row * 128u + ((uint32_t)((col >> 3) ^ (row & 7)) << 4) + (uint32_t)(col & 7) * 2u;
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(sm + off + o));
}
// element (row, v) of a [64 rows][128] bf16 tile loaded by two 64-column TMA boxes (8 KB each)
__device__ __forceinline__ float tile128_at(const unsigned char *sm, uint32_t off, int row, int v) {
    return tile_at(sm, off + (uint32_t)(v >> 6) * 8192u, row, v & 63);
}

// dq^T, dk^T accumulation of one value head (issued by one thread), in two groups with a commit to
// bar_h_free between them: the products that read h (TMEM) and the value-major B tiles (S_DR) come
// first, so that the next head's h can be copied in and staged while the rest run.  A separate,
// non-inlined function keeps the issue sequence compact and out of the kernel's register pressure.
__device__ __noinline__ void issue_dq_dk(uint32_t sb, uint32_t tmem, uint32_t acc0, uint32_t bar_h_free) {
        // [dq^T | dk^T] += h [scale Gam dO | Y]^T: one N = 128 product, the two value-major B tiles are
        // adjacent 64-wide blocks (hi at S_DR, lo at S_DR + 32 K)
        mma_chain_ta<8, 128>(tmem + C_DQ, tmem + C_HT, mdesc(sb + S_DR, 16384), ID_KM128, acc0);
        mma_chain_ta<8, 128>(tmem + C_DQ, tmem + C_HT + 64, mdesc(sb + S_DR, 16384), ID_KM128, 1);
        mma_chain_ta<8, 128>(tmem + C_DQ, tmem + C_HT, mdesc(sb + S_DR + 32768, 16384), ID_KM128, 1);
        mma_commit(bar_h_free);
        for (int sp = 0; sp < 2; ++sp)  // dq^T += K^T dQK^T
            mma_chain<4, 128, 2>(tmem + C_DQ, mdesc(sb + S_KQ, 16384), kdesc(sb + S_DO + 8192 * sp), ID_MK, 1);
        // dk^T += dSe (E Dl)^T
        mma_chain_ta<8, 128>(tmem + C_DK, tmem + C_KS, mdesc(sb + S_DD, 8192), ID_KM, 1);
        mma_chain_ta<8, 128>(tmem + C_DK, tmem + C_KS, mdesc(sb + S_DD + 16384, 8192), ID_KM, 1);
        mma_chain_ta<8, 128>(tmem + C_DK, tmem + C_KS + 64, mdesc(sb + S_DD, 8192), ID_KM, 1);
        for (int sp = 0; sp < 2; ++sp) {
            // dk^T += Q^T dQK
            mma_chain<4, 128, 128>(tmem + C_DK, mdesc(sb + S_KQ + 8192, 16384), mdesc(sb + S_DO + 8192 * sp, 8192),
                                   ID_MM, 1);
            // dk^T += K^T (dKK + dKK^T)
            mma_chain<4, 128, 128>(tmem + C_DK, mdesc(sb + S_KQ, 16384), mdesc(sb + S_P + 8192 * sp, 8192),
                                   ID_MM, 1);
        }
        }

// Column v = 32 q + lane of an fp32 state box (32 values x 128 keys, 128-byte rows, 16-byte chunk j of
// row k at j ^ (k & 7)) for keys 32 hh + i: x[i] = state[32 hh + i][v].  Conflict-free: for each key
// the warp reads one whole 128-byte row.
__device__ __forceinline__ void state_col(const unsigned char *box, float (&x)[32]) {
    const int lane = threadIdx.x & 31, hh = (threadIdx.x >> 5) >> 2;
    const unsigned char *b = box + (uint32_t)(32 * hh) * 128u + ((lane & 3) << 2);
#pragma unroll
    for (int i = 0; i < 32; ++i)
        x[i] = *reinterpret_cast<const float *>(b + i * 128 + ((((lane >> 2) ^ (i & 7))) << 4));
}

// Row k = lane of a 32 x 32 fp32 block (row stride 128 floats) into x[32]: coalesced loads of 4 rows
// of 128 bytes per instruction, transposed through the warp's 2 KB swizzled buffer at tb, 16 rows
// at a time.
__device__ __forceinline__ void key_rows(const float *__restrict__ src, uint32_t tb, float (&x)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int rr = 4 * j + (lane >> 3), c = lane & 7;
            const float4 w = __ldg(reinterpret_cast<const float4 *>(src + (size_t)(16 * hf + rr) * 128 + 4 * c));
            st_shared_v4(tb + rr * 128 + ((c ^ (rr & 7)) << 4), __float_as_uint(w.x), __float_as_uint(w.y),
                         __float_as_uint(w.z), __float_as_uint(w.w));
        }
        __syncwarp();
        if ((lane >> 4) == hf) {  // the half-warp whose rows these are reads them (no selects)
            const int rr = lane & 15;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                uint32_t v0, v1, v2, v3;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                             : "r"(tb + rr * 128 + ((c ^ (rr & 7)) << 4)));
                x[4 * c] = __uint_as_float(v0); x[4 * c + 1] = __uint_as_float(v1);
                x[4 * c + 2] = __uint_as_float(v2); x[4 * c + 3] = __uint_as_float(v3);
            }
        }
        __syncwarp();
    }
}

template <bool F32OUT>
__global__ void __launch_bounds__(NT, 1)
k_tc_bwd_intra(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_dse, Plan p,
               IntraArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int lq = warp & 3, hh = warp >> 2;  // TMEM lane quarter; chunk rows 16 hh .. 16 hh + 15
    const int lrow = 32 * lq + lane;          // TMEM lane of this thread (value v, or key)
    const uint32_t trow = (uint32_t)(32 * lq) << 16;
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + S_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *gam = reinterpret_cast<float *>(sm + S_VEC), *Gm = gam + 64, *Ev = gam + 128, *bet = gam + 192,
          *bg = gam + 256;
    // per-warp partial sums (summed in a fixed order, so the result is deterministic):
    // rdb / rdg [16 warps][64 rows] for dbeta / dgam, sH / sF [16] for <h, dSe> and sum F
    float *rdb_all = gam + 320, *rdg_all = rdb_all + NW * 64, *sH = rdg_all + NW * 64, *sF = sH + NW;
    float *rdb = rdb_all + 64 * warp, *rdg = rdg_all + 64 * warp;
    float *Fa = reinterpret_cast<float *>(sm + S_F), *Fb = reinterpret_cast<float *>(sm + S_F2);
    const uint32_t bar_tma = sb + S_BAR, bar_mma = sb + S_BAR + 8;
    // h (4 boxes) and dSe (2 + 2 boxes, two arrivals) of the current head, fp32 with the 128-byte swizzle;
    // bar_hf: the current head's h products are done (S_DR and the h columns of TMEM are free)
    const uint32_t bar_h = sb + S_BAR + 16, bar_d = sb + S_BAR + 24, bar_hf = sb + S_BAR + 32;

    const int gc = blockIdx.x, hq = blockIdx.y;
    const ChunkPos cp = chunk_pos(p, gc);
    const int tok0 = cp.tok0, n = cp.len;

    if (t == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        mbar_init(bar_h, 1);
        mbar_init(bar_d, 2);
        mbar_init(bar_hf, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(sb + S_MISC, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    uint32_t tma_ph = 0, mma_ph = 0, tma_issued = 0, hf_ph = 0;
    // state loads: h phases issued / waited for, dSe arrivals (two per phase) / phases waited for
    uint32_t h_issued = 0, h_waited = 0, d_arrived = 0, d_waited = 0;
    bool ok = true;

    // Waits for the MMAs issued so far by thread 0 (which commits first).  Only warp 0 polls the
    // mbarrier; the other warps block in the CTA barrier, so no polling competes with the tensor
    // core for shared memory while the MMAs run.
    auto mma_sync = [&]() {
        bool w = true;
        if (warp == 0) {
            if (lane == 0) mma_commit(bar_mma);
            __syncwarp();
            w = mbar_wait_warp(bar_mma, mma_ph & 1, abort_flag);
        }
        ++mma_ph;
        ok = __syncthreads_and(w && ok) != 0;
        tc_fence_after();
    };
    // makes generic-proxy smem writes and TMEM stores of all threads visible to the MMA issuer
    auto pre_mma = [&]() {
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
    };
    auto tma_wait = [&]() {
        bool w = true;
        if (warp == 0) w = mbar_wait_warp(bar_tma, tma_ph & 1, abort_flag);
        ++tma_ph;
        ok = __syncthreads_and(w && ok) != 0;
    };

    // h -> S_DR (4 boxes) and dSe boxes 0, 1 -> the fp32 scratch of value head hv_ (thread 0 issues;
    // every thread counts).
    auto issue_state = [&](int hv_) {
        if (t == 0) {
            const size_t unit = (size_t)gc * p.Hv + hv_;
            mbar_arrive_expect_tx(bar_h, 65536);
            for (int b = 0; b < 4; ++b)
                tma_load_2d(sb + S_DR + 16384 * b, &tm_h, bar_h, 32 * b, (int)(unit * DK));
            mbar_arrive_expect_tx(bar_d, 32768);
            for (int b = 0; b < 2; ++b)
                tma_load_2d(sb + S_F + 16384 * b, &tm_dse, bar_d, 32 * b, (int)(unit * DK));
        }
        ++h_issued;
        ++d_arrived;
    };
    // h^T (lane v) from its boxes -> TMEM as the A operand of the KS / QS product: value v = lrow in
    // box lq, keys 32 hh + i.  Returns false if the wait expired.
    auto load_hT = [&]() -> bool {
        bool w = true;
        if (warp == 0) w = mbar_wait_warp(bar_h, h_waited & 1, abort_flag);
        ok = __syncthreads_and(w && ok) != 0;
        if (!ok) return false;
        ++h_waited;
        float xh[32];
        state_col(sm + S_DR + 16384u * (uint32_t)lq, xh);
        uint32_t hi[16], lo[16];
        split_pack16(xh, hi, lo);
        tmem_st16x2(tmem + trow + C_HT + 16 * hh, hi, tmem + trow + C_HT + 64 + 16 * hh, lo);
        return true;
    };

    issue_state(hq * p.G);
    if (t == 0) {
        ++tma_issued;
        mbar_arrive_expect_tx(bar_tma, 32768);
        tma_load_3d(sb + S_KQ, &tm_k, bar_tma, 0, hq, tok0);
        tma_load_3d(sb + S_KQ + 8192, &tm_q, bar_tma, 0, hq, tok0);
        tma_load_3d(sb + S_KQ + 16384, &tm_k, bar_tma, 64, hq, tok0);
        tma_load_3d(sb + S_KQ + 24576, &tm_q, bar_tma, 64, hq, tok0);
    }
    tma_wait();


    for (int g = 0; ok && g < p.G; ++g) {
        const int hv = hq * p.G + g;
        const size_t st_off = ((size_t)gc * p.Hv + hv) * DK * DV;
        // ---------------------------------------------------------------- per-head vectors, dO / V tiles, A / P tiles
        ++tma_issued;
        // (h and dSe boxes 0, 1 of this head were issued before the loop or during the previous
        // head's dq / dk products)
        if (t == 0) {  // dO, V tiles; A / P operand images (S_A, S_P are adjacent); gate vectors
            const size_t unit = (size_t)gc * p.Hv + hv;
            mbar_arrive_expect_tx(bar_tma, 32768 + 32768 + 1024);
            bulk_load(sb + S_VEC, a.vecs + unit * 256, 1024, bar_tma);
            tma_load_3d(sb + S_DO, &tm_do, bar_tma, 0, hv, tok0);
            tma_load_3d(sb + S_DO + 8192, &tm_do, bar_tma, 64, hv, tok0);
            tma_load_3d(sb + S_DD, &tm_v, bar_tma, 0, hv, tok0);
            tma_load_3d(sb + S_DD + 8192, &tm_v, bar_tma, 64, hv, tok0);
            bulk_load(sb + S_A, a.tiles + unit * 32768, 32768, bar_tma);
        }
        for (int o = t; o < 2 * NW * 64 + 2 * NW; o += NT) rdb_all[o] = 0.f;  // rdb, rdg, sH, sF
        // ---------------------------------------------------------------- P1: h^T (lane v) -> TMEM; KS, QS
        // (for the later heads h^T was staged during the previous head's dq / dk products)
        if (g == 0 && !load_hT()) break;
        pre_mma();  // (its barrier also orders the zeroed partial sums before their updates)
        ++d_arrived;
        if (t == 0) {
            // dSe boxes 2, 3 -> S_DR + 0, S_DR + 32 K (h read; the R^T tiles go to S_DR + 16 K, + 48 K)
            const int unit = gc * p.Hv + hv;
            mbar_arrive_expect_tx(bar_d, 32768);
            tma_load_2d(sb + S_DR, &tm_dse, bar_d, 64, unit * DK);
            tma_load_2d(sb + S_DR + 32768, &tm_dse, bar_d, 96, unit * DK);
            // [KS^T | QS^T] = h^T [K; Q]^T: one N = 128 product (K and Q rows are adjacent, as are the
            // two accumulators)
            for (int sp = 0; sp < 2; ++sp)
                for (int blk = 0; blk < 2; ++blk)
                    mma_chain_ta<4, 2>(tmem + C_KS, tmem + C_HT + 64 * sp + 32 * blk, kdesc(sb + S_KQ + 16384 * blk),
                                       ID_N128, (sp | blk) != 0);
        }
        tma_wait();  // dO, V, A, P and the gate vectors of this head
        if (!ok) break;
        // this thread's v and dO values (rows c = 16 hh + i, value lrow), read while K S / Q S run
        float vv[16], dd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = 16 * hh + i;
            vv[i] = c < n ? tile128_at(sm, S_DD, c, lrow) : 0.f;
            dd[i] = c < n ? tile128_at(sm, S_DO, c, lrow) : 0.f;
        }
        mma_sync();
        if (!ok) break;
        if (t < 64) bg[t] = bet[t] * Gm[t];  // read after the next CTA barrier
        // ---------------------------------------------------------------- P2: R^T tile, dgam (scale Gam dO . QS)
        float Xr[16], KSr[16];  // (V - Gam KS) and KS at chunk rows c = 16 hh + i, value lrow
        {
            uint32_t ks[16], qs[16];
            tmem_ld16x2(tmem + trow + C_KS + 16 * hh, ks, tmem + trow + C_QS + 16 * hh, qs);
            float part[16];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float g8[8];
                lds8f(Gm + 16 * hh + 8 * q2, g8);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * q2 + e;
                    KSr[i] = __uint_as_float(ks[i]);
                    Xr[i] = vv[i] - g8[e] * KSr[i];
                    part[i] = p.scale * g8[e] * dd[i] * __uint_as_float(qs[i]);
                }
            }
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float r8[8], b8[8];
                lds8f(bet + 16 * hh + 8 * q2, b8);
#pragma unroll
                for (int e = 0; e < 8; ++e) r8[e] = b8[e] * Xr[8 * q2 + e];
                st_split_chunk(sb + S_DR + 16384, sb + S_DR + 49152, lrow, 2 * hh + q2, r8);
            }
            const float s = warp_transpose_sum16(part);
            if (lane < 16) rdg[16 * hh + lane] += s;
        }
        {  // dSe^T (lane v) from its boxes -> TMEM (h^T no longer needed)
            bool w = true;
            if (warp == 0) w = mbar_wait_warp(bar_d, d_waited & 1, abort_flag);
            ok = __syncthreads_and(w && ok) != 0;
            if (!ok) break;
            ++d_waited;
            const uint32_t box = lq < 2 ? S_F + 16384u * (uint32_t)lq : S_DR + 32768u * (uint32_t)(lq - 2);
            float xd[32];
            state_col(sm + box, xd);
            uint32_t hi[16], lo[16];
            split_pack16(xd, hi, lo);
            tmem_st16x2(tmem + trow + C_HT + 16 * hh, hi, tmem + trow + C_HT + 64 + 16 * hh, lo);
        }
        pre_mma();
        if (t == 0) {
            // Dl^T = R^T A^T (hi hi, hi lo, lo hi)
            mma_chain<4, 2, 2>(tmem + C_DL, kdesc(sb + S_DR + 16384), kdesc(sb + S_A), ID_KK, 0);
            mma_chain<4, 2, 2>(tmem + C_DL, kdesc(sb + S_DR + 16384), kdesc(sb + S_A + 8192), ID_KK, 1);
            mma_chain<4, 2, 2>(tmem + C_DL, kdesc(sb + S_DR + 49152), kdesc(sb + S_A), ID_KK, 1);
            for (int sp = 0; sp < 2; ++sp)  // KdS^T = dSe^T K^T
                for (int blk = 0; blk < 2; ++blk)
                    mma_chain_ta<4, 2>(tmem + C_KS, tmem + C_HT + 64 * sp + 32 * blk, kdesc(sb + S_KQ + 16384 * blk),
                                       ID_KK, (sp | blk) != 0);
            for (int sp = 0; sp < 2; ++sp)  // PdO^T = dO^T P
                mma_chain<4, 128, 128>(tmem + C_QS, mdesc(sb + S_DO, 8192), mdesc(sb + S_P + 8192 * sp, 8192), ID_MM,
                                       sp);
        }
        mma_sync();
        if (!ok) break;
        // ---------------------------------------------------------------- P3: dDl^T and Dl^T tiles; F
        {
            uint32_t dl[16], kd[16], pd[16];
            tmem_ld16x2(tmem + trow + C_DL + 16 * hh, dl, tmem + trow + C_KS + 16 * hh, kd);
            tmem_ld16(tmem + trow + C_QS + 16 * hh, pd);
            float part[16];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float x8[8], d8[8], ev8[8];
                lds8f(Ev + 16 * hh + 8 * q2, ev8);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * q2 + e;
                    x8[e] = fmaf(p.scale, __uint_as_float(pd[i]), ev8[e] * __uint_as_float(kd[i]));
                    d8[e] = __uint_as_float(dl[i]);
                    part[i] = ev8[e] * __uint_as_float(kd[i]) * d8[e];
                }
                st_split_chunk(sb + S_DD, sb + S_DD + 16384, lrow, 2 * hh + q2, x8);
                st_split_chunk(sb + S_DR, sb + S_DR + 32768, lrow, 2 * hh + q2, d8);
            }
            const float f = warp_transpose_sum16(part);  // F of row 16 hh + (lane & 15), partial over 32 values
            if (lane < 16) rdg[16 * hh + lane] -= f;
            float fs = lane < 16 ? f : 0.f;
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) fs += __shfl_xor_sync(0xffffffffu, fs, o);
            if (lane == 0) sF[warp] += fs;
        }
        pre_mma();
        if (t == 0) {
            // dR^T = dDl^T A  (A read MN-major)
            mma_chain<4, 2, 128>(tmem + C_DR, kdesc(sb + S_DD), mdesc(sb + S_A, 8192), ID_KM, 0);
            mma_chain<4, 2, 128>(tmem + C_DR, kdesc(sb + S_DD), mdesc(sb + S_A + 8192, 8192), ID_KM, 1);
            mma_chain<4, 2, 128>(tmem + C_DR, kdesc(sb + S_DD + 16384), mdesc(sb + S_A, 8192), ID_KM, 1);
            for (int sp = 0; sp < 2; ++sp)  // [Dl; R] dO^T  -> dP^T in lanes 0..63
                for (int blk = 0; blk < 2; ++blk)
                    mma_chain<4, 128, 2>(tmem + C_KS, mdesc(sb + S_DR + 32768 * sp + 8192 * blk, 16384),
                                         kdesc(sb + S_DO + 8192 * blk), ID_MK, (sp | blk) != 0);
            // [Dl; R] dDl^T -> dA^T in lanes 64..127
            mma_chain<8, 128, 128>(tmem + C_QS, mdesc(sb + S_DR, 16384), mdesc(sb + S_DD, 8192), ID_MM, 0);
            mma_chain<8, 128, 128>(tmem + C_QS, mdesc(sb + S_DR, 16384), mdesc(sb + S_DD + 16384, 8192), ID_MM, 1);
            mma_chain<8, 128, 128>(tmem + C_QS, mdesc(sb + S_DR + 32768, 16384), mdesc(sb + S_DD, 8192), ID_MM, 1);
        }
        mma_sync();
        if (!ok) break;
        // ---------------------------------------------------------------- P4: dV, dbeta, dgam terms, E Dl / Y tiles
        {
            uint32_t dr[16];
            tmem_ld16(tmem + trow + C_DR + 16 * hh, dr);
            float pb[16], pg[16];
            __nv_bfloat16 *dvs = reinterpret_cast<__nv_bfloat16 *>(sm + S_DD);  // dv staging [r][128]
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float y8[8], s8[8], g8[8], b8[8], bg8[8];
                lds8f(Gm + 16 * hh + 8 * q2, g8);
                lds8f(bet + 16 * hh + 8 * q2, b8);
                lds8f(bg + 16 * hh + 8 * q2, bg8);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * q2 + e, c = 16 * hh + i;
                    const float drv = __uint_as_float(dr[i]);
                    s8[e] = p.scale * g8[e] * tile128_at(sm, S_DO, c, lrow);  // scale Gam dO (Gm = 0 past n)
                    if (!F32OUT)
                        dvs[c * DV + lrow] = __float2bfloat16_rn(b8[e] * drv);
                    else if (c < n)  // checking mode: fp32 dv straight out (one 128-byte row segment per warp)
                        static_cast<float *>(a.dv)[(size_t)(tok0 + c) * p.Hv * DV + (size_t)hv * DV + lrow] =
                            b8[e] * drv;
                    pb[i] = drv * Xr[i];
                    pg[i] = -bg8[e] * drv * KSr[i];
                    y8[e] = -bg8[e] * drv;
                }
                // value-major tiles [v][i]: scale Gam dO and Y = -beta Gam dR side by side (N = 128 B operand)
                st_split_chunk(sb + S_DR, sb + S_DR + 32768, lrow, 2 * hh + q2, s8);
                st_split_chunk(sb + S_DR + 16384, sb + S_DR + 49152, lrow, 2 * hh + q2, y8);
            }
            const float sbt = warp_transpose_sum16(pb);
            const float sgt = warp_transpose_sum16(pg);
            if (lane < 16) {
                rdb[16 * hh + lane] += sbt;
                rdg[16 * hh + lane] += sgt;
            }
        }
        {  // dP (lanes 0..63) and dA (lanes 64..127) -> fp32 staging Fb[r][i] = dP[r][i], Fa[r][i] = dA[r][i]
            uint32_t dd[16];
            tmem_ld16(tmem + trow + (lq < 2 ? C_KS : C_QS) + 16 * hh, dd);
            float *dst = lq < 2 ? Fb : Fa;
            const int i = lrow & 63;
#pragma unroll
            for (int j = 0; j < 16; ++j) dst[(16 * hh + j) * 65 + i] = __uint_as_float(dd[j]);
        }
        __syncthreads();
        // Thread (row r, 8 columns i = 8 c ..): dQK = D o scale dP -> hi / lo tile [r][i] in the dO region;
        // dgam terms of dP o P (row and column sums); dA~ = lower part of dA -> hi / lo tile [k][l] in the P
        // region (each thread overwrites exactly the P chunk it has read).
        {
            const int r = t >> 3, c = t & 7;
            float pv[8], qk[8], da[8], m[8];
            {
                uint32_t ph[4], pl[4];
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(ph[0]), "=r"(ph[1]), "=r"(ph[2]), "=r"(ph[3]) : "r"(sw128_addr(sb + S_P, r, c)));
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(pl[0]), "=r"(pl[1]), "=r"(pl[2]), "=r"(pl[3])
                             : "r"(sw128_addr(sb + S_P + 8192, r, c)));
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pv[2 * e] = bf16_lo_f(ph[e]) + bf16_lo_f(pl[e]);
                    pv[2 * e + 1] = bf16_hi_f(ph[e]) + bf16_hi_f(pl[e]);
                }
            }
            const float gr = gam[r];
            float rs = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = 8 * c + e;
                float mm = 0.f, q = 0.f;
                if (i <= r && r < n) {
                    const float dpv = p.scale * Fb[r * 65 + i];
                    mm = dpv * pv[e];
                    q = __expf(gr - gam[i]) * dpv;
                }
                qk[e] = q;
                m[e] = mm;
                rs += mm;
                da[e] = i <= r ? Fa[r * 65 + i] : 0.f;
            }
            st_split_chunk(sb + S_DO, sb + S_DO + 8192, r, c, qk);
            st_split_chunk(sb + S_P, sb + S_P + 8192, r, c, da);
            rs += __shfl_xor_sync(0xffffffffu, rs, 1);  // row r: the 8 lanes of its columns
            rs += __shfl_xor_sync(0xffffffffu, rs, 2);
            rs += __shfl_xor_sync(0xffffffffu, rs, 4);
#pragma unroll
            for (int e = 0; e < 8; ++e) {  // columns: the warp's 4 rows
                m[e] += __shfl_xor_sync(0xffffffffu, m[e], 8);
                m[e] += __shfl_xor_sync(0xffffffffu, m[e], 16);
            }
            if ((lane & 7) == 0) rdg[r] += rs;
            __syncwarp();
            if (lane < 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) rdg[8 * c + e] -= m[e];
        }
        // ---------------------------------------------------------------- P5: dL = -(A^T dA A^T), strictly lower
        // on the tensor cores: Z^T = A dA~^T (dA~ = lower part of dA), then dL^T = -Z^T A.  Both are
        // M = 128 products whose rows 64..127 read neighbouring tiles and are ignored.
        pre_mma();
        if (t == 0) {  // Z^T[i][k] = sum_l A[i][l] dA~[k][l]
            mma_chain<4, 2, 2>(tmem + C_KS, kdesc(sb + S_A), kdesc(sb + S_P), ID_KK, 0);
            mma_chain<4, 2, 2>(tmem + C_KS, kdesc(sb + S_A), kdesc(sb + S_P + 8192), ID_KK, 1);
            mma_chain<4, 2, 2>(tmem + C_KS, kdesc(sb + S_A + 8192), kdesc(sb + S_P), ID_KK, 1);
        }
        // while Z runs (thread 0 issuing it): dv out by warps 1..15
        if (warp != 0 && !F32OUT) {  // dv out: 64 rows x 256 bytes from the staging tile, 16-byte stores
            const uint4 *src = reinterpret_cast<const uint4 *>(sm + S_DD);
            for (int o = t - 32; o < 64 * 16; o += NT - 32) {
                const int r = o >> 4, c16 = o & 15;
                if (r < n)
                    __stcs(reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.dv) +
                                                     (size_t)(tok0 + r) * p.Hv * DV + (size_t)hv * DV + 8 * c16),
                           src[o]);
            }
        }
        mma_sync();
        if (!ok) break;
        if (lq < 2) {  // Z^T rows (lanes 0..63) -> hi / lo bf16 A operand in TMEM
            uint32_t z[16], hi[8], lo[8];
            tmem_ld16(tmem + trow + C_KS + 16 * hh, z);
#pragma unroll
            for (int i = 0; i < 8; ++i) split_pair(__uint_as_float(z[2 * i]), __uint_as_float(z[2 * i + 1]), hi[i], lo[i]);
            tmem_st8x2(tmem + trow + C_QS + 8 * hh, hi, tmem + trow + C_QS + 32 + 8 * hh, lo);
        }
        pre_mma();
        if (t == 0) {  // (A^T Z)^T[i][r] = sum_k Z^T[i][k] A[k][r]   (A read MN-major)
            mma_chain_ta<4, 128>(tmem + C_KS, tmem + C_QS, mdesc(sb + S_A, 8192), ID_KM, 0);
            mma_chain_ta<4, 128>(tmem + C_KS, tmem + C_QS, mdesc(sb + S_A + 8192, 8192), ID_KM, 1);
            mma_chain_ta<4, 128>(tmem + C_KS, tmem + C_QS + 32, mdesc(sb + S_A, 8192), ID_KM, 1);
        }
        // while A^T Z runs: (E Dl)^T -> value-major hi / lo tile [v][i] in the dDl region (the dv staging
        // has been written out; the tile's readers are the dq / dk products)
        {
            uint32_t dl[16];
            tmem_ld16(tmem + trow + C_DL + 16 * hh, dl);
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float e8[8], ev8[8];
                lds8f(Ev + 16 * hh + 8 * q2, ev8);
#pragma unroll
                for (int e = 0; e < 8; ++e) e8[e] = ev8[e] * __uint_as_float(dl[8 * q2 + e]);
                st_split_chunk(sb + S_DD, sb + S_DD + 16384, lrow, 2 * hh + q2, e8);
            }
        }
        mma_sync();
        if (!ok) break;
        if (lq < 2) {  // Fa[r][i] = dL[r][i] = -(A^T Z)[r][i]
            uint32_t z[16];
            tmem_ld16(tmem + trow + C_KS + 16 * hh, z);
            const int i = lrow;
#pragma unroll
            for (int j = 0; j < 16; ++j) Fa[(16 * hh + j) * 65 + i] = -__uint_as_float(z[j]);
        }
        // K K^T for the beta and gate terms of dL (lanes 0..63 of a [K; Q] K^T product); the barrier in
        // pre_mma orders the dL loads above before it overwrites their columns
        pre_mma();
        if (t == 0)
            for (int blk = 0; blk < 2; ++blk)
                mma_chain<4, 2, 2>(tmem + C_KS, kdesc(sb + S_KQ + 16384 * blk), kdesc(sb + S_KQ + 16384 * blk), ID_KK,
                                   blk);
        mma_sync();
        if (!ok) break;
        if (lq < 2) {  // K K^T (lanes 0..63: row r = lrow, column i = 16 hh + j) -> fp32 staging Fb[r][i]
            uint32_t kk[16];
            tmem_ld16(tmem + trow + C_KS + 16 * hh, kk);
#pragma unroll
            for (int j = 0; j < 16; ++j) Fb[lrow * 65 + 16 * hh + j] = __uint_as_float(kk[j]);
        }
        tc_fence_before();  // every K K^T load is done before the columns are overwritten
        __syncthreads();
        tc_fence_after();
        // Thread (row r, 8 columns i = 8 c ..): dbeta / dgam terms of dL o D o K K^T, and the symmetric tile
        // dKK + dKK^T (dKK_ri = beta_r D_ri dL_ri for i < r) -> hi / lo [r][i] in the P region
        {
            const int r = t >> 3, c = t & 7;
            const float gr = gam[r], br = bet[r];
            float x[8], m[8], sb_ = 0.f, sg = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int i = 8 * c + e;
                float xv = 0.f, mm = 0.f;
                if (i < r && r < n) {
                    const float d = __expf(gr - gam[i]);
                    const float w = Fa[r * 65 + i] * d * Fb[r * 65 + i];
                    sb_ += w;
                    mm = w * br;
                    sg += mm;
                    xv = br * d * Fa[r * 65 + i];
                } else if (r < i && i < n) {
                    xv = bet[i] * __expf(gam[i] - gr) * Fa[i * 65 + r];
                }
                x[e] = xv;
                m[e] = mm;
            }
            st_split_chunk(sb + S_P, sb + S_P + 8192, r, c, x);
#pragma unroll
            for (int o = 1; o <= 4; o <<= 1) {
                sb_ += __shfl_xor_sync(0xffffffffu, sb_, o);
                sg += __shfl_xor_sync(0xffffffffu, sg, o);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                m[e] += __shfl_xor_sync(0xffffffffu, m[e], 8);
                m[e] += __shfl_xor_sync(0xffffffffu, m[e], 16);
            }
            if ((lane & 7) == 0) {
                rdb[r] += sb_;
                rdg[r] += sg;
            }
            __syncwarp();
            if (lane < 8)
#pragma unroll
                for (int e = 0; e < 8; ++e) rdg[8 * c + e] -= m[e];
        }
        __syncthreads();  // the fp32 scratch is read before the transposes below reuse it
        // h and dSe (lane = key) -> TMEM as A operands of the dq / dk products.
        // The warp's 32 x 32 blocks are read with coalesced row loads (4 rows of 128 bytes per
        // instruction) and transposed through a private 2 KB swizzled buffer in the fp32 scratch
        // region (free since the dKK tile), 16 rows at a time.
        {
            const uint32_t tb = sb + S_F + 2048u * (uint32_t)warp;
            {
                float x[32];
                uint32_t hi[16], lo[16];
                key_rows(a.hbuf + st_off + (size_t)(32 * lq) * DV + 32 * hh, tb, x);
                split_pack16(x, hi, lo);
                tmem_st16x2(tmem + trow + C_HT + 16 * hh, hi, tmem + trow + C_HT + 64 + 16 * hh, lo);
                key_rows(a.dSe + st_off + (size_t)(32 * lq) * DV + 32 * hh, tb, x);
                {  // <h, dSe> partial: h read back from its hi / lo TMEM pair (about 16 significant bits)
                    uint32_t h2[16], l2[16];
                    tmem_ld16x2(tmem + trow + C_HT + 16 * hh, h2, tmem + trow + C_HT + 64 + 16 * hh, l2);
                    float hd = 0.f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        hd = fmaf(bf16_lo_f(h2[i]) + bf16_lo_f(l2[i]), x[2 * i], hd);
                        hd = fmaf(bf16_hi_f(h2[i]) + bf16_hi_f(l2[i]), x[2 * i + 1], hd);
                    }
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) hd += __shfl_xor_sync(0xffffffffu, hd, o);
                    if (lane == 0) sH[warp] = hd;
                }
                split_pack16(x, hi, lo);
                tmem_st16x2(tmem + trow + C_KS + 16 * hh, hi, tmem + trow + C_KS + 64 + 16 * hh, lo);
            }
        }
        // ---------------------------------------------------------------- P6: dq^T, dk^T accumulation
        pre_mma();
        if (t == 0) issue_dq_dk(sb, tmem, g != 0, bar_hf);
        // per-row results of this head (warp 1, while thread 0 issues the
        // dq / dk products below; lane holds rows lane and lane + 32): dbeta, and dg as
        // the reverse cumsum of dgam inside the chunk
        if (warp == 1) {
            float hd = 0.f, sf = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                hd += sH[w];
                sf += sF[w];
            }
            float dgv[2], dbv[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = lane + 32 * hf;
                float dgr = 0.f, dbr = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    dgr += rdg_all[64 * w + r];
                    dbr += rdb_all[64 * w + r];
                }
                if (r == n - 1) dgr += Gm[n - 1] * hd + sf;
                dgv[hf] = r < n ? dgr : 0.f;
                dbv[hf] = dbr;
            }
            // suffix sums within each half, then the upper half's total is added to the lower half
#pragma unroll
            for (int hf = 0; hf < 2; ++hf)
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const float y = __shfl_down_sync(0xffffffffu, dgv[hf], o);
                    if (lane + o < 32) dgv[hf] += y;
                }
            dgv[0] += __shfl_sync(0xffffffffu, dgv[1], 0);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int r = lane + 32 * hf;
                if (r < n) {
                    const size_t gi = (size_t)(tok0 + r) * p.Hv + hv;
                    a.dg[gi] = dgv[hf];
                    a.dbeta[gi] = dbv[hf];
                }
            }
        }
        // While the rest of the dq / dk products run: once the h products are done (S_DR and the h^T
        // columns free), the next head's h and dSe boxes 0, 1 are copied in and each warp stages its share
        // of the next h^T as soon as h has landed.  Thread 0 is still issuing, so warps 1..15 wait for the
        // h products (named barrier) and warp 0 joins at the h wait.
        if (g + 1 < p.G) {
            bool w = true;
            if (warp != 0) {
                if (warp == 2) w = mbar_wait_warp(bar_hf, hf_ph & 1, abort_flag);
                w = named_bar_and(1, NT - 32, w);
                if (w && t == 64) {
                    const size_t nu = (size_t)gc * p.Hv + hv + 1;
                    mbar_arrive_expect_tx(bar_h, 65536);
                    for (int b = 0; b < 4; ++b) tma_load_2d(sb + S_DR + 16384 * b, &tm_h, bar_h, 32 * b, (int)(nu * DK));
                    mbar_arrive_expect_tx(bar_d, 32768);
                    for (int b = 0; b < 2; ++b) tma_load_2d(sb + S_F + 16384 * b, &tm_dse, bar_d, 32 * b, (int)(nu * DK));
                }
            }
            ++hf_ph;
            ++h_issued;
            ++d_arrived;
            if (w) w = mbar_wait_warp(bar_h, h_waited & 1, abort_flag);
            if (w) {
                ++h_waited;
                tc_fence_after();
                float xh[32];
                state_col(sm + S_DR + 16384u * (uint32_t)lq, xh);
                uint32_t hi[16], lo[16];
                split_pack16(xh, hi, lo);
                tmem_st16x2(tmem + trow + C_HT + 16 * hh, hi, tmem + trow + C_HT + 64 + 16 * hh, lo);
            }
            ok = ok && w;
            tc_fence_before();
        }
        mma_sync();
    }
    // ---------------------------------------------------------------- dq, dk out (thread: key lrow, rows 16 hh + j)
    if (ok && F32OUT) {  // checking mode: fp32 dq, dk
        uint32_t d[16];
        const size_t rs = (size_t)p.Hq * DK, o0 = (size_t)tok0 * rs + (size_t)hq * DK + lrow;
        float *dqp = static_cast<float *>(a.dq) + o0, *dkp = static_cast<float *>(a.dk) + o0;
        tmem_ld16(tmem + trow + C_DQ + 16 * hh, d);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (16 * hh + j < n) dqp[(size_t)(16 * hh + j) * rs] = __uint_as_float(d[j]);
        tmem_ld16(tmem + trow + C_DK + 16 * hh, d);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (16 * hh + j < n) dkp[(size_t)(16 * hh + j) * rs] = __uint_as_float(d[j]);
    } else if (ok) {
        uint32_t d[16];
        uint16_t *dqp = reinterpret_cast<uint16_t *>(a.dq) + (size_t)hq * DK + lrow;
        uint16_t *dkp = reinterpret_cast<uint16_t *>(a.dk) + (size_t)hq * DK + lrow;
        const size_t rs = (size_t)p.Hq * DK;
        tmem_ld16(tmem + trow + C_DQ + 16 * hh, d);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int r = 16 * hh + j;
            if (r < n) {
                __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(d[j]));
                __stcs(reinterpret_cast<unsigned short *>(dqp + (size_t)(tok0 + r) * rs), *reinterpret_cast<unsigned short *>(&b));
            }
        }
        tmem_ld16(tmem + trow + C_DK + 16 * hh, d);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int r = 16 * hh + j;
            if (r < n) {
                __nv_bfloat16 b = __float2bfloat16_rn(__uint_as_float(d[j]));
                __stcs(reinterpret_cast<unsigned short *>(dkp + (size_t)(tok0 + r) * rs), *reinterpret_cast<unsigned short *>(&b));
            }
        }
    } else if (t == 0) {
        if (atomicCAS(p.err + 1, 0u, 201u) == 0u) {
            p.err[2] = (uint32_t)gc;
            p.err[4] = blockIdx.x + blockIdx.y * gridDim.x;
        }
        atomicOr(p.err, ERR_TIMEOUT);
        // leave nothing in flight: pending TMA loads and every issued MMA
        if (tma_issued > tma_ph) mbar_drain(bar_tma, (tma_issued - 1) & 1);
        if (h_issued > h_waited) mbar_drain(bar_h, (h_issued - 1) & 1);
        if (d_arrived & 1) mbar_arrive(bar_d);  // the second half was never issued
        if ((d_arrived + 1) / 2 > d_waited) mbar_drain(bar_d, ((d_arrived + 1) / 2 - 1) & 1);
        mma_commit(bar_mma);
        mbar_drain(bar_mma, mma_ph & 1);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tc_bwd_intra(const Plan &p, const void *q, const void *k, const void *v, const void *d_o,
                                const unsigned char *tiles, const float *vecs, const float *hbuf, const float *dSe,
                                void *dq, void *dk, void *dv, float *dbeta, float *dg, cudaStream_t st) {
    CUtensorMap tk, tq, tdo, tv;
    if (!make_head_map(&tk, k, p.Hq, p) || !make_head_map(&tq, q, p.Hq, p) || !make_head_map(&tdo, d_o, p.Hv, p) ||
        !make_head_map(&tv, v, p.Hv, p))
        return cudaErrorInvalidValue;
    CUtensorMap th, tdse;
    const size_t units = (size_t)p.total_chunks * p.Hv;
    if (!make_state_map(&th, hbuf, units) || !make_state_map(&tdse, dSe, units)) return cudaErrorInvalidValue;
    auto kern = p.out_f32 ? k_tc_bwd_intra<true> : k_tc_bwd_intra<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    IntraArgs a;
    a.tiles = tiles;
    a.vecs = vecs;
    a.hbuf = hbuf;
    a.dSe = dSe;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dbeta = dbeta;
    a.dg = dg;
    dim3 grid(p.total_chunks, p.Hq);
    kern<<<grid, NT, SMEM_BYTES, st>>>(tk, tq, tdo, tv, th, tdse, p, a);
    return cudaGetLastError();
}

}  // namespace gdn
