// tc_fwd.cu -- fused tensor-core forward of the chunked gated delta rule (bf16 io,
// K = V = 128, chunk 64), one CTA per (sequence, value head), persistent over
// the sequence's chunks.
//
// All contractions run on tcgen05 (kind::f16, fp32 accumulation in TMEM) in the
// value-major form: every MMA has M = 128 = the value dimension, so TMEM lane v
// holds value column v and the thread owning lane v keeps the state row
// S^T[v][:] in registers.  Per chunk (n <= 64 rows, entry state S):
//
//   D1   = [K; Q] K^T                  -> K K^T, Q K^T            (exact bf16 operands)
//   KS^T = S^T K^T,  QS^T = S^T Q^T                               (S split hi + lo, from TMEM)
//   R^T  = (V - diag(Gam) K S)^T diag(beta)                        (CUDA cores)
//   Dl^T = R^T A^T                                                 (R, A split; 3 products)
//   U^T  = (diag(E) Dl)^T K          (K read MN-major)             (E Dl split)
//   O^T  = Dl^T P^T,  P = D o Q K^T                                (Dl, P split; 3 products)
//   S^T <- Gam_last S^T + U^T,   o = scale (diag(Gam) QS + O)
//
// Derived operands (S, R, A, Dl, E Dl, P) enter the tensor cores as hi + lo
// bf16 pairs; q and k are exact bf16 inputs.  Every product then carries about
// 16 significant bits, which the 2e-3 * RMS output bound needs (one bf16
// rounding of any derived operand costs about 1e-2 * RMS).  The pages' step
// list ("computing the A matrix, extracting W and U, V correction, output";
// FlashQLA blog post, section 2) forms the corrected values U - W S; here the
// same Dl is formed as A R, which needs neither W nor U.
//
// Warp roles (448 threads):
//   warp 0      TMA producer: k, q and v chunk tiles (128-byte swizzle), 2 stages
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2-5   prep: gate cumsum, L, A = (I + L)^{-1} (blocked, in place), P;
//               runs one chunk ahead of the state chain; writes g_cum and A
//   warps 6-13  state: S in registers (written to TMEM as the A operand of the
//               KS / QS products), R, E Dl, state update, o epilogue (staged in
//               the consumed v tile, written with 16-byte stores)
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace gdn {
namespace {

using namespace tc;

constexpr int DK = 128, DV = 128;
constexpr int NUM_THREADS = 448;
constexpr int W_TMA = 0, W_MMA = 1, W_PREP0 = 2, W_STATE0 = 6;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t SM_KQ = 0;             // 2 stages x [kb0: K 8K, Q 8K][kb1: K 8K, Q 8K]
constexpr uint32_t KQ_STAGE = 32768;
constexpr uint32_t SM_V = 65536;          // 2 stages x V [64 rows][2 x 64 v] (TMA); then o staging [64][128] bf16
constexpr uint32_t V_STAGE = 16384;
constexpr uint32_t SM_ED = 98304;         // (E Dl)^T hi / lo [128 v][64 c]
constexpr uint32_t SM_RT = 131072;        // R^T hi / lo [128 v][64 c]; later Dl^T hi / lo
constexpr uint32_t SM_AHL = 163840;       // A hi / lo [64][64]
constexpr uint32_t SM_PHL = 180224;       // P hi / lo [64][64]
constexpr uint32_t SM_LM = 196608;        // fp32 [64][65] scratch: L, then A in place
constexpr uint32_t SM_TB = SM_LM + 64 * 65 * 4;       // fp32 3 x [16][17]
constexpr uint32_t SM_VEC = SM_TB + 3 * 16 * 17 * 4;  // 4 x {gam, Gam, E, beta} x 64 fp32
constexpr uint32_t SM_BAR = SM_VEC + 4 * 4 * 64 * 4;  // mbarriers
constexpr uint32_t SM_MISC = SM_BAR + 32 * 8;         // tmem base, abort flag, scan total
constexpr uint32_t SM_TOTAL = SM_MISC + 64;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;

// TMEM columns (512 allocated): S^T hi / lo are bf16 pairs along the keys (A operand)
constexpr uint32_t TM_D1 = 0, TM_KS = 64, TM_DL = 128, TM_U = 64, TM_QS = 192, TM_O = 320, TM_SH = 384,
                   TM_SL = 448;

enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_D1FULL, B_D1FREE, B_SSREADY, B_KSDONE, B_RTREADY, B_AREADY,
    B_DLDONE, B_EDREADY, B_PREADY, B_UPDDONE, B_ODONE, B_EPIFREE0, B_EPIFREE1, B_FINAL, B_VFULL0, B_VFULL1,
    B_VEMPTY0, B_VEMPTY1, B_STAGED0, B_STAGED1, B_COUNT
};

constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_N128_BMN = idesc_bf16(128, 128, 0, 1);

struct FwdArgs {
    const __nv_bfloat16 *v;
    const float *g, *beta, *h0;
    __nv_bfloat16 *o, *A;
    float *g_cum, *h, *ht;
    int g_is_cum;  // g already holds the chunk-local cumsum (backward recompute)
    float *A32, *P32;  // optional fp32 copies of A and P per chunk ([chunk][Hv][64][64])
    // sequence splitting with warmup (see cp.cu): seg_len > 0 enables it
    int seg_len, n_seg, warm, mode;  // mode: CP_WARM or CP_MAIN
    const uint8_t *serial;           // [n_seqs][Hv]: 1 = this head runs unsplit
    float *seg_states;               // [n_seqs][Hv][n_seg][K][V] warmup states
};

// Records the first expired wait: err[1] = barrier + 1, err[2] = chunk,
// err[3] = warp, err[4] = CTA; err[0] |= timeout.
__device__ void record_timeout(const Plan &p, int bar_id, int chunk) {
    if (atomicCAS(p.err + 1, 0u, (uint32_t)(bar_id + 1)) == 0u) {
        p.err[2] = (uint32_t)chunk;
        p.err[3] = threadIdx.x >> 5;
        p.err[4] = blockIdx.x + blockIdx.y * gridDim.x;
    }
    atomicOr(p.err, ERR_TIMEOUT);
}

// Blocked in-place inverse of the unit lower-triangular I + L held in Lm
// ([64][65], strictly lower part = L, rest 0); afterwards Lm = (I + L)^{-1}.
// Column blocks of 16 are processed right to left so that the inverted A_IK
// (K > J) and the untouched L_KJ are both available:
//     A_IJ = -(sum_{K=J+1}^{I} A_IK L_KJ) A_JJ.
// Called by the 128 prep threads (named barrier 1).
__device__ void blocked_inverse(float *Lm, float *Tb, int pt) {
    constexpr int LS = 65, TS = 17;
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
    named_bar(1, 128);
    for (int J = 2; J >= 0; --J) {
        const int nblk = 3 - J;  // blocks I = J+1 .. 3
        for (int o = pt; o < nblk * 256; o += 128) {
            const int I = J + 1 + (o >> 8), r = (o >> 4) & 15, c = o & 15;
            float s = 0.f;
            for (int K = J + 1; K <= I; ++K) {
                const float *arow = Lm + (16 * I + r) * LS + 16 * K;
                const float *lcol = Lm + (16 * K) * LS + 16 * J + c;
#pragma unroll
                for (int k = 0; k < 16; ++k) s = fmaf(arow[k], lcol[k * LS], s);
            }
            Tb[(o >> 8) * 16 * TS + r * TS + c] = s;
        }
        named_bar(1, 128);
        for (int o = pt; o < nblk * 256; o += 128) {
            const int I = J + 1 + (o >> 8), r = (o >> 4) & 15, c = o & 15;
            const float *trow = Tb + (o >> 8) * 16 * TS + r * TS;
            const float *acol = Lm + (16 * J) * LS + 16 * J + c;
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) s = fmaf(trow[k], acol[k * LS], s);
            Lm[(16 * I + r) * LS + 16 * J + c] = -s;
        }
        named_bar(1, 128);
    }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
k_tc_fwd(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
         const __grid_constant__ CUtensorMap tm_v, Plan p, FwdArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + SM_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *vec = reinterpret_cast<float *>(sm + SM_VEC);
    auto bar = [&](int i) { return sb + SM_BAR + 8u * (uint32_t)i; };

    const int hv = blockIdx.y, hq = hv / p.G;
    const int s = a.seg_len > 0 ? (int)blockIdx.x / a.n_seg : (int)blockIdx.x;
    const int pseg = a.seg_len > 0 ? (int)blockIdx.x % a.n_seg : 0;
    SeqRange sr = seq_range(p, s);
    // chunk range of this CTA, its initial / final state and whether it writes the outputs
    const int nseq_ck = sr.c1 - sr.c0;
    int jb = 0, je = nseq_ck;
    const size_t st_base = ((size_t)s * p.Hv + hv) * DK * DV;
    const float *init = a.h0 ? a.h0 + st_base : nullptr;
    float *fin = a.ht ? a.ht + st_base : nullptr;
    bool outs = true;
    if (a.seg_len > 0) {
        const bool serial = a.serial[(size_t)s * p.Hv + hv] != 0;
        const int L = a.seg_len;
        float *segst = a.seg_states + (((size_t)s * p.Hv + hv) * a.n_seg + pseg) * DK * DV;
        if (a.mode == CP_WARM) {  // state after the warmup window that precedes segment pseg, from zero
            outs = false;
            init = nullptr;
            fin = segst;
            if (serial || pseg == 0 || pseg * L >= nseq_ck) jb = je = 0;
            else { jb = max(0, pseg * L - a.warm); je = pseg * L; }
        } else {  // CP_MAIN
            if (serial) {
                if (pseg != 0) jb = je = 0;
            } else {
                jb = min(pseg * L, nseq_ck);
                je = min(nseq_ck, (pseg + 1) * L);
                if (pseg > 0) init = segst;
                if (je < nseq_ck) fin = nullptr;
            }
        }
        if (jb >= je) { jb = je = 0; fin = nullptr; }
    }
    sr.tok0 += jb * C;
    sr.c0 += jb;
    sr.c1 = sr.c0 + (je - jb);
    const int nck = je - jb;
    __nv_bfloat16 *o_out = outs ? a.o : nullptr, *A_out = outs ? a.A : nullptr;
    float *gcum_out = outs ? a.g_cum : nullptr, *h_out = outs ? a.h : nullptr;
    float *A32_out = outs ? a.A32 : nullptr, *P32_out = outs ? a.P32 : nullptr;

    if (threadIdx.x == 0) {
        const uint32_t counts[B_COUNT] = {1, 1, 1, 1, 1, 128, 256, 1, 256, 128, 1, 256, 128, 1, 1, 256, 256, 1,
                                          1, 1, 256, 256, 256, 256};
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), counts[i]);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) tmem_alloc(sb + SM_MISC, 512);
    if (warp == W_TMA && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == W_TMA) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0, vissued = 0;
            for (int j = 0; j < nck; ++j) {
                const int st = j & 1;
                if (j >= 2 && !mbar_wait(bar(B_EMPTY0 + st), ((j >> 1) - 1) & 1, abort_flag)) {
                    record_timeout(p, B_EMPTY0 + st, j);
                    break;
                }
                const int tok0 = sr.tok0 + j * C;
                mbar_arrive_expect_tx(bar(B_FULL0 + st), KQ_STAGE);
                const uint32_t dst = sb + SM_KQ + st * KQ_STAGE;
                tma_load_3d(dst, &tm_k, bar(B_FULL0 + st), 0, hq, tok0);
                tma_load_3d(dst + 8192, &tm_q, bar(B_FULL0 + st), 0, hq, tok0);
                tma_load_3d(dst + 16384, &tm_k, bar(B_FULL0 + st), 64, hq, tok0);
                tma_load_3d(dst + 24576, &tm_q, bar(B_FULL0 + st), 64, hq, tok0);
                issued = j + 1;
                // v tile; its buffer last held the staged o of chunk j - 2
                if (j >= 2 && !mbar_wait(bar(B_VEMPTY0 + st), ((j >> 1) - 1) & 1, abort_flag)) {
                    record_timeout(p, B_VEMPTY0 + st, j);
                    break;
                }
                mbar_arrive_expect_tx(bar(B_VFULL0 + st), V_STAGE);
                tma_load_3d(sb + SM_V + st * V_STAGE, &tm_v, bar(B_VFULL0 + st), 0, hv, tok0);
                tma_load_3d(sb + SM_V + st * V_STAGE + 8192, &tm_v, bar(B_VFULL0 + st), 64, hv, tok0);
                vissued = j + 1;
            }
            // never leave with copies in flight
            for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) mbar_drain(bar(B_FULL0 + (j & 1)), (j >> 1) & 1);
            for (int j = (vissued > 2 ? vissued - 2 : 0); j < vissued; ++j)
                mbar_drain(bar(B_VFULL0 + (j & 1)), (j >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && nck > 0) {
            auto kq = [&](int st) { return sb + SM_KQ + (uint32_t)st * KQ_STAGE; };
            auto d1 = [&](int st) {
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t off = kq(st) + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(tmem + TM_D1, sdesc_sw128(off, 16, 1024), sdesc_sw128(off, 16, 1024), ID_N64, kk);
                }
            };
            int failed = -1, fj = 0;
            auto wait = [&](int id, uint32_t par, int j) {
                if (mbar_wait(bar(id), par, abort_flag)) return true;
                failed = id;
                fj = j;
                return false;
            };
            bool ok = wait(B_FULL0, 0, 0);
            if (ok) {
                tc_fence_after();
                d1(0);
                mma_commit(bar(B_D1FULL));
            }
            for (int j = 0; ok && j < nck; ++j) {
                const int st = j & 1, ph = j & 1;
                if (!(ok = wait(B_SSREADY, ph, j))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // KS^T = S^T K^T (S hi, lo from TMEM)
                    for (int blk = 0; blk < 2; ++blk)
                        mma_chain_ta<4, 2>(tmem + TM_KS, tmem + (sp ? TM_SL : TM_SH) + 32 * blk,
                                           sdesc_sw128(kq(st) + blk * 16384, 16, 1024), ID_N64, (sp | blk) != 0);
                mma_commit(bar(B_KSDONE));
                if (j >= 2 && !(ok = wait(B_EPIFREE0 + st, ((j - 2) >> 1) & 1, j))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // QS^T = S^T Q^T
                    for (int blk = 0; blk < 2; ++blk)
                        mma_chain_ta<4, 2>(tmem + TM_QS + 64 * st, tmem + (sp ? TM_SL : TM_SH) + 32 * blk,
                                           sdesc_sw128(kq(st) + 8192 + blk * 16384, 16, 1024), ID_N64,
                                           (sp | blk) != 0);
                if (j + 1 < nck) {  // next chunk's K K^T / Q K^T for the prep warps
                    if (!(ok = wait(B_FULL0 + (st ^ 1), ((j + 1) >> 1) & 1, j + 1))) break;
                    if (!(ok = wait(B_D1FREE, ph, j))) break;
                    tc_fence_after();
                    d1(st ^ 1);
                    mma_commit(bar(B_D1FULL));
                }
                if (!(ok = wait(B_RTREADY, ph, j))) break;
                if (!(ok = wait(B_AREADY, ph, j))) break;
                tc_fence_after();
                for (int t = 0; t < 3; ++t)  // Dl^T = R^T A^T: (hi,hi) (hi,lo) (lo,hi)
                    mma_chain<4, 2, 2>(tmem + TM_DL, sdesc_sw128(sb + SM_RT + (t == 2 ? 16384 : 0), 16, 1024),
                                       sdesc_sw128(sb + SM_AHL + (t == 1 ? 8192 : 0), 16, 1024), ID_N64, t != 0);
                mma_commit(bar(B_DLDONE));
                if (!(ok = wait(B_EDREADY, ph, j))) break;
                if (!(ok = wait(B_PREADY, ph, j))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // U^T = (E Dl)^T K, K read MN-major
                    mma_chain<4, 2, 128>(tmem + TM_U, sdesc_sw128(sb + SM_ED + sp * 16384, 16, 1024),
                                         sdesc_sw128(kq(st), 16384, 1024), ID_N128_BMN, sp);
                mma_commit(bar(B_UPDDONE));
                // O (one buffer): the epilogue of chunk j - 1 has read it
                if (j >= 1 && !(ok = wait(B_EPIFREE0 + ((j - 1) & 1), ((j - 1) >> 1) & 1, j))) break;
                tc_fence_after();
                for (int t = 0; t < 3; ++t)  // O^T = Dl^T P^T
                    mma_chain<4, 2, 2>(tmem + TM_O, sdesc_sw128(sb + SM_RT + (t == 2 ? 16384 : 0), 16, 1024),
                                       sdesc_sw128(sb + SM_PHL + (t == 1 ? 8192 : 0), 16, 1024), ID_N64, t != 0);
                mma_commit(bar(B_ODONE));
                mma_commit(bar(B_EMPTY0 + st));
            }
            // every issued MMA completes before TMEM is released
            mma_commit(bar(B_FINAL));
            mbar_drain(bar(B_FINAL), 0);
            if (failed >= 0) record_timeout(p, failed, fj);
        }
        __syncwarp();
    } else if (warp < W_STATE0) {
        // ------------------------------------------------------------------ prep warps
        const int row = 32 * (warp & 3) + lane;        // TMEM lane
        const int pt = (warp - W_PREP0) * 32 + lane;   // 0..127
        float *Lm = reinterpret_cast<float *>(sm + SM_LM);
        float *Tb = reinterpret_cast<float *>(sm + SM_TB);
        float *mtot = reinterpret_cast<float *>(misc + 4);
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        int failed = -1, fj = 0;
        auto gwait = [&](int id, uint32_t par, int j) {  // group-uniform bounded wait
            bool w = mbar_wait(bar(id), par, abort_flag);
            if (!w && failed < 0) { failed = id; fj = j; }
            return named_bar_and(1, 128, w);
        };
        for (int j = 0; j < nck; ++j) {
            const int tok0 = sr.tok0 + j * C, n = min(C, sr.tok1 - tok0);
            float *gam = vec + (j & 3) * 256, *Gm = gam + 64, *Ev = gam + 128, *bet = gam + 192;
            // chunk-local inclusive cumsum of g over rows 0..63 (warps holding TMEM lanes 0..63)
            float gv = 0.f, bv = 0.f, x = 0.f;
            if (row < 64 && row < n) {
                const size_t gi = (size_t)(tok0 + row) * p.Hv + hv;
                gv = a.g[gi];
                bv = a.beta[gi];
            }
            if (row < 64 && !a.g_is_cum) {
                x = gv;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                if (row == 31) *mtot = x;
            }
            named_bar(1, 128);
            if (a.g_is_cum) {  // rows past the chunk end repeat the last value, as a cumsum of zeros would
                const int rr = row < n ? row : n - 1;
                x = row < 64 ? a.g[(size_t)(tok0 + rr) * p.Hv + hv] : 0.f;
            } else if (row >= 32 && row < 64) {
                x += *mtot;
            }
            if (row < 64) {
                gam[row] = x;
                bet[row] = bv;
                if (row < n && gcum_out) gcum_out[(size_t)(tok0 + row) * p.Hv + hv] = x;
            }
            named_bar(1, 128);
            const float glast = gam[n - 1];
            if (row < 64) {
                Gm[row] = row < n ? __expf(x) : 0.f;
                Ev[row] = row < n ? __expf(glast - x) : 0.f;
            }
            // K K^T (lanes 0..63) / Q K^T (lanes 64..127) of this chunk
            if (!gwait(B_D1FULL, j & 1, j)) break;
            tc_fence_after();
            uint32_t raw0[32], raw1[32];
            tmem_ld32(trow + TM_D1, raw0);
            tmem_ld32(trow + TM_D1 + 32, raw1);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(B_D1FREE));
            if (row < 64) {  // L = beta D o K K^T, strictly lower
                const int r = row;
                const float gr = gam[r], br = bet[r];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float kk = __uint_as_float(i < 32 ? raw0[i] : raw1[i - 32]);
                    Lm[r * 65 + i] = (i < r && r < n) ? br * __expf(gr - gam[i]) * kk : 0.f;
                }
            } else {  // P = D o Q K^T, lower incl. diagonal, kept in raw0 / raw1
                const int r = row - 64;
                const float gr = gam[r];
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    float qk = __uint_as_float(i < 32 ? raw0[i] : raw1[i - 32]);
                    float pv = (i <= r && r < n) ? __expf(gr - gam[i]) * qk : 0.f;
                    if (i < 32) raw0[i] = __float_as_uint(pv);
                    else raw1[i - 32] = __float_as_uint(pv);
                }
            }
            named_bar(1, 128);
            blocked_inverse(Lm, Tb, pt);
            if (A32_out) {  // fp32 A and P for the backward's gradient kernels
                const size_t mat = ((size_t)(sr.c0 + j) * p.Hv + hv) * C * C;
                const int r = pt >> 1, hh = pt & 1;
                float4 *dst = reinterpret_cast<float4 *>(A32_out + mat + (size_t)r * C + 32 * hh);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    dst[q4] = make_float4(Lm[r * 65 + 32 * hh + 4 * q4], Lm[r * 65 + 32 * hh + 4 * q4 + 1],
                                          Lm[r * 65 + 32 * hh + 4 * q4 + 2], Lm[r * 65 + 32 * hh + 4 * q4 + 3]);
                if (row >= 64) {
                    float4 *pd = reinterpret_cast<float4 *>(P32_out + mat + (size_t)(row - 64) * C);
#pragma unroll
                    for (int q4 = 0; q4 < 16; ++q4) {
                        const uint32_t *src = q4 < 8 ? raw0 + 4 * q4 : raw1 + 4 * (q4 - 8);
                        pd[q4] = make_float4(__uint_as_float(src[0]), __uint_as_float(src[1]),
                                             __uint_as_float(src[2]), __uint_as_float(src[3]));
                    }
                }
            }
            // A -> hi/lo operand tile and the io-dtype output, once Dl of the previous chunk is done
            if (j >= 1 && !gwait(B_DLDONE, (j - 1) & 1, j)) break;
            {
                const int r = pt >> 1, hh = pt & 1;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int ch = 4 * hh + q;
                    float vals[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) vals[e] = Lm[r * 65 + 8 * ch + e];
                    st_split_chunk(sb + SM_AHL, sb + SM_AHL + 8192, r, ch, vals);
                    if (A_out && r < n) {
                        uint4 pk = make_uint4(pack_bf16(vals[0], vals[1]), pack_bf16(vals[2], vals[3]),
                                              pack_bf16(vals[4], vals[5]), pack_bf16(vals[6], vals[7]));
                        *reinterpret_cast<uint4 *>(A_out + ((size_t)(tok0 + r) * p.Hv + hv) * C + 8 * ch) = pk;
                    }
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(B_AREADY));
            // P -> hi/lo operand tile, once O of the previous chunk is done
            if (j >= 1 && !gwait(B_ODONE, (j - 1) & 1, j)) break;
            if (row >= 64) {
                const int r = row - 64;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float pv[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        pv[e] = __uint_as_float(ch < 4 ? raw0[8 * ch + e] : raw1[8 * (ch - 4) + e]);
                    st_split_chunk(sb + SM_PHL, sb + SM_PHL + 8192, r, ch, pv);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(B_PREADY));
        }
        if (failed >= 0) record_timeout(p, failed, fj);
    } else {
        // ------------------------------------------------------------------ state warps
        const int v = 32 * (warp & 3) + lane;          // value column = TMEM lane
        const int hh = (warp - W_STATE0) >> 2;         // key half / chunk-column half
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        int failed = -1, fj = 0;
        auto wwait = [&](int id, uint32_t par, int j) {  // warp-uniform bounded wait
            bool w = mbar_wait_warp(bar(id), par, abort_flag);
            if (!w && failed < 0) { failed = id; fj = j; }
            return w;
        };
        float S[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) S[i] = init ? init[(size_t)(64 * hh + i) * DV + v] : 0.f;

        // o of chunk jj: scale (Gam QS + O) -> bf16, staged as [64 rows][128] in the v buffer of chunk jj
        // (consumed: every state thread has passed R of chunk jj), then written with 16-byte stores
        auto epilogue = [&](int jj) -> bool {
            const int tok0 = sr.tok0 + jj * C, n = min(C, sr.tok1 - tok0), b = jj & 1;
            const float *Gm = vec + (jj & 3) * 256 + 64;
            if (!o_out) {  // nothing to write: release QS / O and the v buffer (this thread is past R of jj)
                mbar_arrive(bar(B_EPIFREE0 + b));
                mbar_arrive(bar(B_VEMPTY0 + b));
                return true;
            }
            if (!wwait(B_ODONE, jj & 1, jj)) return false;
            tc_fence_after();
            __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sm + SM_V + b * V_STAGE);
            uint32_t qs[16], oo[16];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tmem_ld16(trow + TM_QS + 64 * b + 32 * hh + 16 * half, qs);
                tmem_ld16(trow + TM_O + 32 * hh + 16 * half, oo);
                tmem_wait_ld();
                if (half == 1) {
                    tc_fence_before();
                    mbar_arrive(bar(B_EPIFREE0 + b));
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 32 * hh + 16 * half + i;
                    const float ov = p.scale * fmaf(Gm[c], __uint_as_float(qs[i]), __uint_as_float(oo[i]));
                    stg[c * DV + v] = __float2bfloat16_rn(ov);
                }
            }
            mbar_arrive(bar(B_STAGED0 + b));
            if (!wwait(B_STAGED0 + b, (jj >> 1) & 1, jj)) return false;
            {
                const int ts = threadIdx.x - 32 * W_STATE0;
                const uint4 *src = reinterpret_cast<const uint4 *>(stg);
#pragma unroll
                for (int k4 = 0; k4 < 4; ++k4) {
                    const int idx = ts + 256 * k4, r = idx >> 4, c16 = idx & 15;
                    if (r < n)
                        *reinterpret_cast<uint4 *>(o_out + ((size_t)(tok0 + r) * p.Hv + hv) * DV + 8 * c16) = src[idx];
                }
            }
            mbar_arrive(bar(B_VEMPTY0 + b));
            return true;
        };

        bool ok = true;
        for (int j = 0; j < nck && ok; ++j) {
            const int tok0 = sr.tok0 + j * C, n = min(C, sr.tok1 - tok0);
            const float *gam = vec + (j & 3) * 256, *Gm = gam + 64, *Ev = gam + 128, *bet = gam + 192;
            // (a) S^T row -> hi / lo bf16 pairs in TMEM (keys 64hh .. 64hh + 63: columns 32hh ..)
            {
                uint32_t shi[32], slo[32];
                split_pack32(S, shi, slo);
                tmem_st32(trow + TM_SH + 32 * hh, shi);
                tmem_st32(trow + TM_SL + 32 * hh, slo);
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(bar(B_SSREADY));
            if (h_out) {
                const size_t hb = ((size_t)(sr.c0 + j) * p.Hv + hv) * DK * DV;
#pragma unroll
                for (int i = 0; i < 64; ++i) h_out[hb + (size_t)(64 * hh + i) * DV + v] = S[i];
            }
            if (j >= 1 && !(ok = epilogue(j - 1))) break;
            // (c) R^T = beta (V - Gam K S)^T; the gate vectors of chunk j are
            // published by the prep warps together with A (a_ready)
            if (!(ok = wwait(B_AREADY, j & 1, j))) break;
            if (!(ok = wwait(B_KSDONE, j & 1, j))) break;
            if (!(ok = wwait(B_VFULL0 + (j & 1), (j >> 1) & 1, j))) break;
            tc_fence_after();
            uint32_t raw[32];
            tmem_ld32(trow + TM_KS + 32 * hh, raw);
            tmem_wait_ld();
            // v at (row c, column v) of the swizzled tile (two 64-column boxes); rows past the chunk end
            // are finite (next tokens or zero fill) and meet beta = 0
            const unsigned char *vt = sm + SM_V + (j & 1) * V_STAGE + (v >> 6) * 8192;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float R[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 8 * q + e, c = 32 * hh + i;
                    const uint32_t vo = (uint32_t)c * 128u + ((uint32_t)(((v & 63) >> 3) ^ (c & 7)) << 4) + (uint32_t)(v & 7) * 2u;
                    const float vv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(vt + vo));
                    R[e] = bet[c] * (vv - Gm[c] * __uint_as_float(raw[i]));
                }
                st_split_chunk(sb + SM_RT, sb + SM_RT + 16384, v, 4 * hh + q, R);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(bar(B_RTREADY));
            // (e) Dl^T -> (E Dl)^T tile (S region) and Dl^T tile (R region)
            if (!(ok = wwait(B_DLDONE, j & 1, j))) break;
            tc_fence_after();
            tmem_ld32(trow + TM_DL + 32 * hh, raw);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float Dl[8], ED[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    Dl[e] = __uint_as_float(raw[8 * q + e]);
                    ED[e] = Ev[32 * hh + 8 * q + e] * Dl[e];
                }
                st_split_chunk(sb + SM_ED, sb + SM_ED + 16384, v, 4 * hh + q, ED);
                st_split_chunk(sb + SM_RT, sb + SM_RT + 16384, v, 4 * hh + q, Dl);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive(bar(B_EDREADY));
            // (g) S^T <- Gam_last S^T + U^T
            if (!(ok = wwait(B_UPDDONE, j & 1, j))) break;
            tc_fence_after();
            const float gl = Gm[n - 1];
            tmem_ld32(trow + TM_U + 64 * hh, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) S[i] = fmaf(gl, S[i], __uint_as_float(raw[i]));
            tmem_ld32(trow + TM_U + 64 * hh + 32, raw);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) S[32 + i] = fmaf(gl, S[32 + i], __uint_as_float(raw[i]));
            tc_fence_before();
        }
        if (ok && nck > 0) ok = epilogue(nck - 1);
        if (ok && fin) {
#pragma unroll
            for (int i = 0; i < 64; ++i) fin[(size_t)(64 * hh + i) * DV + v] = S[i];
        }
        if (failed >= 0) record_timeout(p, failed, fj);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_MMA) tmem_dealloc(tmem, 512);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

}  // namespace

// [tokens][heads][128] bf16 as a 3-D tensor, boxes of 64 columns x 1 head x 64 tokens, 128-byte swizzle.
bool make_head_map(CUtensorMap *m, const void *ptr, int heads, const Plan &p) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)DK, (cuuint64_t)heads, (cuuint64_t)p.B * (cuuint64_t)p.T};
    cuuint64_t strides[2] = {(cuuint64_t)DK * 2, (cuuint64_t)heads * DK * 2};
    cuuint32_t box[3] = {64, 1, 64};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_fwd_supported(const Plan &p) { return p.io == GDN_BF16 && p.K == DK && p.V == DV && p.B * p.T > 0; }

cudaError_t launch_tc_fwd(const Plan &p, const void *q, const void *k, const void *v, const float *g,
                          const float *beta, const float *h0, void *o, float *g_cum, void *A, float *h,
                          float *ht, cudaStream_t st, bool g_is_cum, float *A32, float *P32, const CpSplit *cp) {
    CUtensorMap tk, tq, tv;
    if (!make_head_map(&tk, k, p.Hq, p) || !make_head_map(&tq, q, p.Hq, p) || !make_head_map(&tv, v, p.Hv, p))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_tc_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    FwdArgs a;
    a.v = static_cast<const __nv_bfloat16 *>(v);
    a.g = g;
    a.beta = beta;
    a.h0 = h0;
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.A = static_cast<__nv_bfloat16 *>(A);
    a.g_cum = g_cum;
    a.h = h;
    a.ht = ht;
    a.g_is_cum = g_is_cum ? 1 : 0;
    a.A32 = A32;
    a.P32 = P32;
    a.seg_len = 0;
    a.n_seg = 1;
    a.warm = 0;
    a.mode = 0;
    a.serial = nullptr;
    a.seg_states = nullptr;
    if (cp) {
        a.seg_len = cp->seg_len;
        a.n_seg = cp->n_seg;
        a.warm = cp->warm;
        a.mode = cp->mode;
        a.serial = cp->serial;
        a.seg_states = cp->seg_states;
    }
    dim3 grid(p.n_seqs * a.n_seg, p.Hv);
    k_tc_fwd<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tk, tq, tv, p, a);
    return cudaGetLastError();
}

}  // namespace gdn
