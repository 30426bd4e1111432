// tc_fwd.cu -- tensor-core state chain of the chunked gated delta rule (bf16
// io, K = V = 128, chunk 64): one CTA per (sequence, value head), persistent
// over the sequence's chunks.  It serves the forward (o, final state) and the
// backward's state recompute (chunk-entry states h).
//
// All contractions run on tcgen05 (kind::f16, fp32 accumulation in TMEM) in the
// value-major form: every MMA has M = 128 = the value dimension, so TMEM lane v
// holds value column v and the four threads owning lane v (one per quarter of
// the keys) keep the state row S^T[v][:] in registers, 32 keys each.  Per chunk (n <= 64 rows, entry state S), with A, P
// and the gate vectors of the chunk precomputed by the prep kernel (tc_prep.cu):
//
//   KS^T = S^T K^T,  QS^T = S^T Q^T                               (S split hi + lo, from TMEM)
//   R^T  = (V - diag(Gam) K S)^T diag(beta)                        (CUDA cores)
//   Dl^T = R^T A^T                                                 (R, A split; 3 products)
//   U^T  = (diag(E) Dl)^T K          (K read MN-major)             (E Dl split, from TMEM)
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
// Warp roles (576 threads):
//   warp 0      producer: k, q (TMA) and the A / P operand image (bulk copy), 2 stages;
//               v (TMA) and the gate vectors (bulk copy), 2 stages
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2-17  state: S in registers (written to TMEM as the A operand of the
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
constexpr int NUM_THREADS = 576;
constexpr int W_TMA = 0, W_MMA = 1, W_STATE0 = 2;
constexpr uint32_t NSTATE = NUM_THREADS - 64;  // state threads: 16 warps, four per TMEM lane quarter
constexpr uint32_t NSW = NSTATE / 32;            // state warps (one barrier arrival each)

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t SM_KQ = 0;             // 2 stages x {[kb0: K 8K, Q 8K][kb1: K 8K, Q 8K], A hi / lo, P hi / lo}
constexpr uint32_t KQ_STAGE = 65536;
constexpr uint32_t KQ_BYTES = 32768, AP_OFF = 32768, AP_BYTES = 32768;
constexpr uint32_t SM_V = 131072;         // 2 stages x {V [64 rows][2 x 64 v] (TMA), gate vectors 1 KB};
constexpr uint32_t V_STAGE = 17408;       // the V part later holds the staged o [64][128] bf16
constexpr uint32_t VEC_OFF = 16384;
constexpr uint32_t SM_RT = SM_V + 2 * V_STAGE;  // R^T hi / lo [128 v][64 c]; later Dl^T hi / lo
constexpr uint32_t SM_BAR = SM_RT + 32768;      // mbarriers
constexpr uint32_t SM_MISC = SM_BAR + 32 * 8;   // tmem base, abort flag
constexpr uint32_t SM_TOTAL = SM_MISC + 64;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;
static_assert(SM_RT % 1024 == 0 && V_STAGE % 1024 == 0, "swizzled tiles need 1024-byte alignment");

// TMEM columns (512 allocated).  A operands held as bf16 pairs: (E Dl)^T hi / lo along the chunk rows,
// S^T hi / lo along the keys.
constexpr uint32_t TM_EDH = 0, TM_EDL = 32, TM_KS = 64, TM_DL = 128, TM_U = 64, TM_QS = 192, TM_O = 320,
                   TM_SH = 384, TM_SL = 448;

enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_SSREADY, B_KSDONE, B_RTREADY, B_DLDONE, B_EDREADY, B_UPDDONE,
    B_ODONE, B_EPIFREE0, B_EPIFREE1, B_FINAL, B_VFULL0, B_VFULL1, B_VEMPTY0, B_VEMPTY1, B_COUNT
};

constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_N128_BMN = idesc_bf16(128, 128, 0, 1);

struct FwdArgs {
    const unsigned char *tiles;  // [chunks][Hv] x 32 KB operand images from the prep kernel
    const float *vecs;           // [chunks][Hv] x {gam, Gam, E, beta} x 64
    const float *h0;
    void *o;  // bf16, or fp32 in the checking mode (p.out_f32)
    float *h, *ht;
    // sequence splitting (see cp.cu and launch.h): seg_len > 0 enables it
    int seg_len, n_seg, warm, mode;  // mode: CP_WARM, CP_MAIN or CP_SEG
    const uint8_t *serial;           // [n_seqs][Hv]: 1 = this head runs unsplit (warmup only; may be null)
    float *seg_states;               // [n_seqs][Hv][n_seg][K][V] segment starting states
    float *seg_h, *seg_M;            // CP_SEG outputs: segment contributions and transitions
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

template <bool F32OUT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
k_tc_fwd(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
         const __grid_constant__ CUtensorMap tm_v, Plan p, FwdArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // (aligned through an integer round trip, so the state warps' shared-memory reads are generic loads:
    // this kernel measured 5 % faster this way than with smem_align1024, unlike the other three)
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                          ~uintptr_t(1023));
    const uint32_t sb = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + SM_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    auto bar = [&](int i) { return sb + SM_BAR + 8u * (uint32_t)i; };

    const int hv = blockIdx.y, hq = hv / p.G;
    // CP_SEG: two CTAs per segment, the second runs the transition (v = 0, identity start)
    const int cps = a.mode == CP_SEG ? 2 : 1;
    const int s = a.seg_len > 0 ? (int)blockIdx.x / (a.n_seg * cps) : (int)blockIdx.x;
    const int pseg = a.seg_len > 0 ? ((int)blockIdx.x / cps) % a.n_seg : 0;
    const bool v_zero = a.mode == CP_SEG && (blockIdx.x & 1);
    SeqRange sr = seq_range(p, s);
    // chunk range of this CTA, its initial / final state and whether it writes the outputs
    const int nseq_ck = sr.c1 - sr.c0;
    int jb = 0, je = nseq_ck;
    const size_t st_base = ((size_t)s * p.Hv + hv) * DK * DV;
    const float *init = a.h0 ? a.h0 + st_base : nullptr;
    float *fin = a.ht ? a.ht + st_base : nullptr;
    bool outs = true;
    bool init_identity = false;
    if (a.seg_len > 0) {
        const bool serial = a.serial && a.serial[(size_t)s * p.Hv + hv] != 0;
        const int L = a.seg_len;
        float *segst = a.seg_states + (((size_t)s * p.Hv + hv) * a.n_seg + pseg) * DK * DV;
        if (a.mode == CP_WARM) {  // state after the warmup window that precedes segment pseg, from zero
            outs = false;
            init = nullptr;
            fin = segst;
            if (serial || pseg == 0 || pseg * L >= nseq_ck) jb = je = 0;
            else { jb = max(0, pseg * L - a.warm); je = pseg * L; }
        } else if (a.mode == CP_SEG) {  // segment pseg alone (not the last one): h_p or M_p
            outs = false;
            init = nullptr;
            init_identity = v_zero;
            const size_t so = (((size_t)s * p.Hv + hv) * a.n_seg + pseg) * DK * DV;
            fin = (v_zero ? a.seg_M : a.seg_h) + so;
            jb = min(pseg * L, nseq_ck);
            je = min(nseq_ck, (pseg + 1) * L);
            if (je >= nseq_ck) jb = je = 0;  // the last segment feeds no other
        } else {  // CP_MAIN: exactly one segment owns the sequence end (segment 0 of an empty sequence)
            if (serial) {
                if (pseg != 0) { jb = je = 0; fin = nullptr; }
            } else {
                jb = min(pseg * L, nseq_ck);
                je = min(nseq_ck, (pseg + 1) * L);
                if (pseg > 0) init = segst;
                const bool owns_end = nseq_ck == 0 ? pseg == 0 : (jb < je && je == nseq_ck);
                if (!owns_end) fin = nullptr;
                if (jb >= je) jb = je = 0;
            }
        }
        if (a.mode != CP_MAIN && jb >= je) { jb = je = 0; fin = nullptr; }
    }
    sr.tok0 += jb * C;
    sr.c0 += jb;
    sr.c1 = sr.c0 + (je - jb);
    const int nck = je - jb;
    void *o_out = outs ? a.o : nullptr;
    float *h_out = outs ? a.h : nullptr;

    if (threadIdx.x == 0) {
        const uint32_t counts[B_COUNT] = {1, 1, 1, 1, NSW, 1, NSW, 1, NSW, 1, 1, NSW, NSW, 1, 1, 1, NSW, NSW};
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
                const size_t unit = (size_t)(sr.c0 + j) * p.Hv + hv;
                if (j >= 2 && !mbar_wait(bar(B_EMPTY0 + st), ((j >> 1) - 1) & 1, abort_flag, p.wait_ns)) {
                    record_timeout(p, B_EMPTY0 + st, j);
                    break;
                }
                const int tok0 = sr.tok0 + j * C;
                if (j != p.drop_load_chunk) {  // (the test aid skips this chunk: its consumer's wait expires)
                    mbar_arrive_expect_tx(bar(B_FULL0 + st), KQ_BYTES + AP_BYTES);
                    const uint32_t dst = sb + SM_KQ + st * KQ_STAGE;
                    tma_load_3d(dst, &tm_k, bar(B_FULL0 + st), 0, hq, tok0);
                    tma_load_3d(dst + 8192, &tm_q, bar(B_FULL0 + st), 0, hq, tok0);
                    tma_load_3d(dst + 16384, &tm_k, bar(B_FULL0 + st), 64, hq, tok0);
                    tma_load_3d(dst + 24576, &tm_q, bar(B_FULL0 + st), 64, hq, tok0);
                    bulk_load(dst + AP_OFF, a.tiles + unit * AP_BYTES, AP_BYTES, bar(B_FULL0 + st));
                }
                issued = j + 1;
                // v tile and gate vectors; the buffer last held the staged o of chunk j - 2
                if (j >= 2 && !mbar_wait(bar(B_VEMPTY0 + st), ((j >> 1) - 1) & 1, abort_flag, p.wait_ns)) {
                    record_timeout(p, B_VEMPTY0 + st, j);
                    break;
                }
                mbar_arrive_expect_tx(bar(B_VFULL0 + st), (v_zero ? 0 : 16384) + 1024);
                if (!v_zero) {
                    tma_load_3d(sb + SM_V + st * V_STAGE, &tm_v, bar(B_VFULL0 + st), 0, hv, tok0);
                    tma_load_3d(sb + SM_V + st * V_STAGE + 8192, &tm_v, bar(B_VFULL0 + st), 64, hv, tok0);
                }
                bulk_load(sb + SM_V + st * V_STAGE + VEC_OFF, a.vecs + unit * 256, 1024, bar(B_VFULL0 + st));
                vissued = j + 1;
            }
            // never leave with copies in flight
            for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j)
                if (j != p.drop_load_chunk) mbar_drain(bar(B_FULL0 + (j & 1)), (j >> 1) & 1, p.wait_ns);
            for (int j = (vissued > 2 ? vissued - 2 : 0); j < vissued; ++j)
                mbar_drain(bar(B_VFULL0 + (j & 1)), (j >> 1) & 1, p.wait_ns);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && nck > 0) {
            auto kq = [&](int st) { return sb + SM_KQ + (uint32_t)st * KQ_STAGE; };
            int failed = -1, fj = 0;
            auto wait = [&](int id, uint32_t par, int j) {
                if (mbar_wait(bar(id), par, abort_flag, p.wait_ns)) return true;
                failed = id;
                fj = j;
                return false;
            };
            bool ok = true;
            for (int j = 0; ok && j < nck; ++j) {
                const int st = j & 1, ph = j & 1;
                if (!(ok = wait(B_FULL0 + st, (j >> 1) & 1, j))) break;
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
                if (!(ok = wait(B_RTREADY, ph, j))) break;
                tc_fence_after();
                for (int t = 0; t < 3; ++t)  // Dl^T = R^T A^T: (hi,hi) (hi,lo) (lo,hi)
                    mma_chain<4, 2, 2>(tmem + TM_DL, sdesc_sw128(sb + SM_RT + (t == 2 ? 16384 : 0), 16, 1024),
                                       sdesc_sw128(kq(st) + AP_OFF + (t == 1 ? 8192 : 0), 16, 1024), ID_N64, t != 0);
                mma_commit(bar(B_DLDONE));
                if (!(ok = wait(B_EDREADY, ph, j))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // U^T = (E Dl)^T K: E Dl hi / lo from TMEM, K read MN-major
                    mma_chain_ta<4, 128>(tmem + TM_U, tmem + (sp ? TM_EDL : TM_EDH), sdesc_sw128(kq(st), 16384, 1024),
                                         ID_N128_BMN, sp);
                mma_commit(bar(B_UPDDONE));
                // O (one buffer): the epilogue of chunk j - 1 has read it
                if (j >= 1 && !(ok = wait(B_EPIFREE0 + ((j - 1) & 1), ((j - 1) >> 1) & 1, j))) break;
                tc_fence_after();
                for (int t = 0; t < 3; ++t)  // O^T = Dl^T P^T
                    mma_chain<4, 2, 2>(tmem + TM_O, sdesc_sw128(sb + SM_RT + (t == 2 ? 16384 : 0), 16, 1024),
                                       sdesc_sw128(kq(st) + AP_OFF + 16384 + (t == 1 ? 8192 : 0), 16, 1024), ID_N64,
                                       t != 0);
                mma_commit(bar(B_ODONE));
                mma_commit(bar(B_EMPTY0 + st));
            }
            // every issued MMA completes before TMEM is released
            mma_commit(bar(B_FINAL));
            mbar_drain(bar(B_FINAL), 0, p.wait_ns);
            if (failed >= 0) record_timeout(p, failed, fj);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ state warps
        // 16 warps: lane quarter warp & 3 holds value columns v; quarter index hh = 0..3 of the warp
        // within its lane quarter picks keys 32 hh .. 32 hh + 31 and chunk rows 16 hh .. 16 hh + 15.
        const int v = 32 * (warp & 3) + lane;          // value column = TMEM lane
        const int hh = (warp - W_STATE0) >> 2;
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        int failed = -1, fj = 0;
        auto wwait = [&](int id, uint32_t par, int j) {  // warp-uniform bounded wait
            bool w = mbar_wait_warp(bar(id), par, abort_flag, p.wait_ns);
            if (!w && failed < 0) { failed = id; fj = j; }
            return w;
        };
        auto vecs = [&](int jj) { return reinterpret_cast<const float *>(sm + SM_V + (jj & 1) * V_STAGE + VEC_OFF); };
        float S[32];  // S^T[v][32 hh + i]
#pragma unroll
        for (int i = 0; i < 32; ++i)
            S[i] = init ? init[(size_t)(32 * hh + i) * DV + v] : (init_identity && 32 * hh + i == v ? 1.f : 0.f);

        // o of chunk jj: scale (Gam QS + O) -> bf16, in two parts of 8 of the warp's 16 rows (part 0 while
        // Dl of the next chunk is computed, part 1 while its U is).  Each warp stages its rows x 32 values in
        // a private 1 KB part of the v buffer of chunk jj (consumed: every state thread is past R of jj) and
        // writes them back as 64-byte row segments with 16-byte stores; no CTA-wide barrier is involved.
        // QS / O and the v buffer are released after part 1.
        auto epilogue = [&](int jj, int part) -> bool {
            const int tok0 = sr.tok0 + jj * C, n = min(C, sr.tok1 - tok0), b = jj & 1;
            const float *Gm = vecs(jj) + 64;
            if (!o_out) {  // nothing to write: release QS / O and the v buffer (this thread is past R of jj)
                if (part == 1) {
                    mbar_arrive_warp(bar(B_EPIFREE0 + b));
                    mbar_arrive_warp(bar(B_VEMPTY0 + b));
                }
                return true;
            }
            if (part == 0) {
                if (!wwait(B_ODONE, jj & 1, jj)) return false;
                tc_fence_after();
            }
            __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(sm + SM_V + b * V_STAGE + 1024 * (warp - W_STATE0));
            uint32_t qs[8], oo[8];
            float gm[8];  // loaded before any store (generic pointers: no reordering across stores)
            lds8f(Gm + 16 * hh + 8 * part, gm);
            tmem_ld8x2(trow + TM_QS + 64 * b + 16 * hh + 8 * part, qs, trow + TM_O + 16 * hh + 8 * part, oo);
            if (part == 1) {
                tc_fence_before();
                mbar_arrive_warp(bar(B_EPIFREE0 + b));
            }
            if (F32OUT) {  // checking mode: the fp32 value, one 128-byte row segment per warp and row
                float *of = static_cast<float *>(o_out) + (size_t)tok0 * p.Hv * DV + (size_t)hv * DV + v;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = 16 * hh + 8 * part + i;
                    if (c < n)
                        of[(size_t)c * p.Hv * DV] =
                            p.scale * fmaf(gm[i], __uint_as_float(qs[i]), __uint_as_float(oo[i]));
                }
                if (part == 1) mbar_arrive_warp(bar(B_VEMPTY0 + b));
                return true;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)  // row 8 part + i of this warp's 16, column lane
                stg[(8 * part + i) * 32 + lane] =
                    __float2bfloat16_rn(p.scale * fmaf(gm[i], __uint_as_float(qs[i]), __uint_as_float(oo[i])));
            __syncwarp();
            {  // lane: row 8 part + lane / 4, 8 values at 8 (lane % 4)
                const uint4 *src = reinterpret_cast<const uint4 *>(stg);
                const int ri = 8 * part + (lane >> 2), c = 16 * hh + ri;
                const uint4 w = src[ri * 4 + (lane & 3)];
                if (c < n)
                    __stcs(reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(o_out) +
                                                     ((size_t)(tok0 + c) * p.Hv + hv) * DV + 32 * (warp & 3) +
                                                     8 * (lane & 3)),
                           w);
            }
            if (part == 1) {
                // the staging writes (generic proxy) are ordered before the next TMA write of this buffer
                fence_proxy_async_smem();
                mbar_arrive_warp(bar(B_VEMPTY0 + b));
            }
            return true;
        };

        bool ok = true;
        for (int j = 0; j < nck && ok; ++j) {
            const int tok0 = sr.tok0 + j * C, n = min(C, sr.tok1 - tok0);
            // (a) S^T row -> hi / lo bf16 pairs in TMEM (keys 32hh .. 32hh + 31: columns 16hh ..)
            {
                uint32_t shi[16], slo[16];
                split_pack16(S, shi, slo);
                tmem_st16x2(trow + TM_SH + 16 * hh, shi, trow + TM_SL + 16 * hh, slo);
            }
            tc_fence_before();
            mbar_arrive_warp(bar(B_SSREADY));
            if (h_out) {  // while KS is computed: the chunk-entry state (backward recompute)
                const size_t hb = ((size_t)(sr.c0 + j) * p.Hv + hv) * DK * DV;
#pragma unroll
                for (int i = 0; i < 32; ++i) __stcs(h_out + hb + (size_t)(32 * hh + i) * DV + v, S[i]);
            }
            // (c) R^T = beta (V - Gam K S)^T
            if (!(ok = wwait(B_VFULL0 + (j & 1), (j >> 1) & 1, j))) break;
            const float *vj = vecs(j), *Gm = vj + 64, *Ev = vj + 128, *bet = vj + 192;
            // the chunk's v values at (row c = 16 hh + i, column v), read while K S is still being computed;
            // rows past the chunk end are finite (next tokens or zero fill) and meet beta = 0
            float vv[16];
            {
                const unsigned char *vt = sm + SM_V + (j & 1) * V_STAGE + (v >> 6) * 8192;  // two 64-column boxes
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 16 * hh + i;
                    const uint32_t vo = (uint32_t)c * 128u + ((uint32_t)(((v & 63) >> 3) ^ (c & 7)) << 4) +
                                        (uint32_t)(v & 7) * 2u;
                    vv[i] = v_zero ? 0.f : __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(vt + vo));
                }
            }
            if (!(ok = wwait(B_KSDONE, j & 1, j))) break;
            tc_fence_after();
            uint32_t raw[32];
            tmem_ld16(trow + TM_KS + 16 * hh, *reinterpret_cast<uint32_t(*)[16]>(raw));
            // every operand is loaded before the first store (the stores are asm with a memory clobber,
            // which would otherwise order each load behind the previous store)
            float R[16], bt[16], gg[16];
            lds16f(bet + 16 * hh, bt);
            lds16f(Gm + 16 * hh, gg);
#pragma unroll
            for (int i = 0; i < 16; ++i) R[i] = bt[i] * (vv[i] - gg[i] * __uint_as_float(raw[i]));
#pragma unroll
            for (int q = 0; q < 2; ++q) st_split_chunk(sb + SM_RT, sb + SM_RT + 16384, v, 2 * hh + q, R + 8 * q);
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive_warp(bar(B_RTREADY));
            // while Dl is computed: o of chunk j - 1
            if (j >= 1 && !(ok = epilogue(j - 1, 0))) break;
            // (e) Dl^T -> Dl^T tile (R region) and (E Dl)^T hi / lo pairs in TMEM
            if (!(ok = wwait(B_DLDONE, j & 1, j))) break;
            tc_fence_after();
            tmem_ld16(trow + TM_DL + 16 * hh, *reinterpret_cast<uint32_t(*)[16]>(raw));
            {
                float ED[16], Dl[16], ev[16];
                lds16f(Ev + 16 * hh, ev);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    Dl[i] = __uint_as_float(raw[i]);
                    ED[i] = ev[i] * Dl[i];
                }
#pragma unroll
                for (int q = 0; q < 2; ++q) st_split_chunk(sb + SM_RT, sb + SM_RT + 16384, v, 2 * hh + q, Dl + 8 * q);
                uint32_t ehi[8], elo[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) split_pair(ED[2 * i], ED[2 * i + 1], ehi[i], elo[i]);
                tmem_st8x2(trow + TM_EDH + 8 * hh, ehi, trow + TM_EDL + 8 * hh, elo);
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive_warp(bar(B_EDREADY));
            // while U is computed: the rest of the o of chunk j - 1
            if (j >= 1 && !(ok = epilogue(j - 1, 1))) break;
            // (g) S^T <- Gam_last S^T + U^T
            if (!(ok = wwait(B_UPDDONE, j & 1, j))) break;
            tc_fence_after();
            const float gl = Gm[n - 1];
            tmem_ld32(trow + TM_U + 32 * hh, raw);
#pragma unroll
            for (int i = 0; i < 32; ++i) S[i] = fmaf(gl, S[i], __uint_as_float(raw[i]));
            tc_fence_before();
        }
        if (ok && nck > 0) ok = epilogue(nck - 1, 0);
        if (ok && nck > 0) ok = epilogue(nck - 1, 1);
        if (ok && fin) {
#pragma unroll
            for (int i = 0; i < 32; ++i) fin[(size_t)(32 * hh + i) * DV + v] = S[i];
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

bool make_state_map(CUtensorMap *m, const float *ptr, size_t units) {
    auto fn = encode_fn();
    if (!fn || units == 0) return false;
    cuuint64_t dims[2] = {(cuuint64_t)DV, (cuuint64_t)units * DK};
    cuuint64_t strides[1] = {(cuuint64_t)DV * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)DK};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool tc_fwd_supported(const Plan &p) { return p.io == GDN_BF16 && p.K == DK && p.V == DV && p.B * p.T > 0; }

cudaError_t launch_tc_fwd(const Plan &p, const void *q, const void *k, const void *v, const unsigned char *tiles,
                          const float *vecs, const float *h0, void *o, float *h, float *ht, cudaStream_t st,
                          const CpSplit *cp) {
    CUtensorMap tk, tq, tv;
    if (!make_head_map(&tk, k, p.Hq, p) || !make_head_map(&tq, q, p.Hq, p) || !make_head_map(&tv, v, p.Hv, p))
        return cudaErrorInvalidValue;
    auto kern = p.out_f32 ? k_tc_fwd<true> : k_tc_fwd<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    FwdArgs a;
    a.tiles = tiles;
    a.vecs = vecs;
    a.h0 = h0;
    a.o = o;
    a.h = h;
    a.ht = ht;
    a.seg_len = 0;
    a.n_seg = 1;
    a.warm = 0;
    a.mode = 0;
    a.serial = nullptr;
    a.seg_states = nullptr;
    a.seg_h = a.seg_M = nullptr;
    if (cp) {
        a.seg_len = cp->seg_len;
        a.n_seg = cp->n_seg;
        a.warm = cp->warm;
        a.mode = cp->mode;
        a.serial = cp->serial;
        a.seg_states = cp->seg_states;
        a.seg_h = cp->seg_h;
        a.seg_M = cp->seg_M;
    }
    dim3 grid(p.n_seqs * a.n_seg * (a.mode == CP_SEG ? 2 : 1), p.Hv);
    kern<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tk, tq, tv, p, a);
    return cudaGetLastError();
}

}  // namespace gdn
