// tc_bwd.cu -- tensor-core reverse scan of the state gradient (bf16 io, K = V = 128).
//
// One CTA per (sequence, value head) walks the sequence's chunks backwards,
// carrying dS = dL/d(state at the chunk end) in registers (value-major: the
// thread owning TMEM lane v holds dS^T[v][:]).  Per chunk (n rows, gates
// gam, Gam = exp(gam), E = exp(gam_last - gam), scale dO' = scale * dO):
//
//   KdS^T   = dS^T K^T                      (dS^T hi / lo from TMEM, K exact)
//   PdO^T   = dO^T P                        (dO exact, P hi / lo)
//   dDl^T   = scale PdO^T + KdS^T diag(E)                       (CUDA cores)
//   dR^T    = dDl^T A                       (dDl, A hi / lo; 3 products)
//   dS^T   <- Gam_last dS^T + dO^T (scale Gam o Q) - (beta Gam o dR)^T K
//
// which is the reverse-mode counterpart of the forward's
// S <- Gam_last S + K^T diag(E) A diag(beta) (V - diag(Gam) K S) plus the
// output's direct dependence on S.  The state gradient at every chunk end is
// written to the workspace for the per-chunk gradient kernel; dh0 is the
// state gradient at the sequence start.
//
// Warp roles (448 threads):
//   warp 0      TMA producer: k and do chunk tiles (128-byte swizzle), 2 stages
//   warp 1      TMEM allocator, single-thread MMA issuer
//   warps 2-5   aux: A and P operand images (bulk copies from the prep kernel's
//               output, double-buffered) and scale Gam o Q operand tiles
//   warps 6-13  state: dS in registers, dDl, beta Gam o dR, state update
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
constexpr int W_TMA = 0, W_MMA = 1, W_AUX0 = 2, W_STATE0 = 6;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t SM_K = 0;          // 2 stages x [kb0 8K][kb1 8K]: K chunk rows x 64 keys
constexpr uint32_t SM_DO = 32768;     // 2 stages x [vb0 8K][vb1 8K]: dO chunk rows x 64 values
constexpr uint32_t SM_DD = 65536;     // dDl^T hi / lo [128 v][64 r] (later beta Gam dR^T)
constexpr uint32_t SM_A = 98304;      // 2 slots x A hi / lo, MN-major rows r x 64 i
constexpr uint32_t SM_P = 131072;     // 2 slots x P hi / lo, MN-major rows r' x 64 r
constexpr uint32_t SM_GQ = 163840;    // scale Gam o Q hi [r][128 keys] (16K), lo (16K), MN-major
constexpr uint32_t SM_VEC = 196608;   // per state warp: E, beta Gam (2 x 32 fp32)
constexpr uint32_t SM_BAR = SM_VEC + 8 * 2 * 32 * 4;
constexpr uint32_t SM_MISC = SM_BAR + 32 * 8;
constexpr uint32_t SM_TOTAL = SM_MISC + 64;
constexpr uint32_t SMEM_BYTES = SM_TOTAL + 1024;

// TMEM columns
constexpr uint32_t TM_KD = 0, TM_PD = 64, TM_DR = 128, TM_U = 192, TM_SH = 320, TM_SL = 384;

enum {
    B_FULL0 = 0, B_FULL1, B_EMPTY0, B_EMPTY1, B_APREADY, B_GQREADY, B_DSREADY, B_KDDONE, B_DDREADY, B_DRDONE,
    B_YREADY, B_UDONE, B_FINAL, B_COUNT
};

constexpr uint32_t ID_N64 = idesc_bf16(128, 64, 0, 0);
constexpr uint32_t ID_N64_AMN_BMN = idesc_bf16(128, 64, 1, 1);
constexpr uint32_t ID_N128_AMN_BMN = idesc_bf16(128, 128, 1, 1);
constexpr uint32_t ID_N128_BMN = idesc_bf16(128, 128, 0, 1);
constexpr uint32_t ID_N64_BMN = idesc_bf16(128, 64, 0, 1);

struct DscanArgs {
    const __nv_bfloat16 *q;
    const float *g_cum, *beta, *dht;
    const unsigned char *tiles;  // [chunks][Hv] x 32 KB: A hi / lo, P hi / lo operand images
    float *dSe, *dh0;
    // sequence splitting (see launch.h), segments counted from the sequence end: seg_len > 0 enables it
    int seg_len, n_seg, mode;
    const float *seg_states;  // [n_seqs][Hv][n_seg][K][V] state gradient entering each segment from the right
    float *seg_h, *seg_M;     // CP_SEG outputs: segment contributions and transitions
};

__device__ void record_timeout(const Plan &p, int bar_id, int chunk) {
    if (atomicCAS(p.err + 1, 0u, (uint32_t)(bar_id + 101)) == 0u) {
        p.err[2] = (uint32_t)chunk;
        p.err[3] = threadIdx.x >> 5;
        p.err[4] = blockIdx.x + blockIdx.y * gridDim.x;
    }
    atomicOr(p.err, ERR_TIMEOUT);
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
k_tc_dscan(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_do, Plan p,
           DscanArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_align1024(smem_raw);
    const uint32_t sb = smem_u32(sm);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + SM_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    auto bar = [&](int i) { return sb + SM_BAR + 8u * (uint32_t)i; };

    const int hv = blockIdx.y, hq = hv / p.G;
    // CP_SEG: two CTAs per segment, the second runs the transition (dO = 0, identity start)
    const int cps = a.mode == CP_SEG ? 2 : 1;
    const int s = a.seg_len > 0 ? (int)blockIdx.x / (a.n_seg * cps) : (int)blockIdx.x;
    const int pr = a.seg_len > 0 ? ((int)blockIdx.x / cps) % a.n_seg : 0;  // segment index from the end
    const bool do_zero = a.mode == CP_SEG && (blockIdx.x & 1);
    SeqRange sr = seq_range(p, s);
    const int nseq_ck = sr.c1 - sr.c0;
    int jb = 0, je = nseq_ck;
    const size_t st_base = ((size_t)s * p.Hv + hv) * DK * DV;
    const float *init = a.dht ? a.dht + st_base : nullptr;
    float *fin = a.dh0 ? a.dh0 + st_base : nullptr;
    bool init_identity = false, outs = true;
    if (a.seg_len > 0) {
        const int L = a.seg_len, P = (nseq_ck + L - 1) / L, ps = P - 1 - pr;  // forward segment index
        const size_t so = (((size_t)s * p.Hv + hv) * a.n_seg + pr) * DK * DV;
        if (pr < P) {
            jb = ps * L;
            je = min(nseq_ck, (ps + 1) * L);
        } else {
            jb = je = 0;
        }
        if (a.mode == CP_SEG) {  // every segment but the sequence's first: contribution or transition
            outs = false;
            init = nullptr;
            init_identity = do_zero;
            fin = (do_zero ? a.seg_M : a.seg_h) + so;
            if (pr >= P || ps == 0) { jb = je = 0; fin = nullptr; }
        } else {  // CP_MAIN: the segment holding the sequence start (segment 0 of an empty one) writes dh0
            if (pr > 0) init = a.seg_states + so;
            const bool owns_start = nseq_ck == 0 ? pr == 0 : (pr < P && ps == 0);
            if (!owns_start) fin = nullptr;
        }
    }
    sr.tok0 += jb * C;
    sr.c0 += jb;
    sr.c1 = sr.c0 + (je - jb);
    const int nck = je - jb;
    float *dSe_out = outs ? a.dSe : nullptr;
    // step t handles chunk j = nck - 1 - t
    auto chunk_tok0 = [&](int t) { return sr.tok0 + (nck - 1 - t) * C; };

    if (threadIdx.x == 0) {
        // GQREADY: the 4 aux warps; DSREADY, DDREADY, YREADY: the 8 state warps (one arrival per warp)
        const uint32_t counts[B_COUNT] = {1, 1, 1, 1, 1, 4, 8, 1, 8, 1, 8, 1, 1};
        for (int i = 0; i < B_COUNT; ++i) mbar_init(bar(i), counts[i]);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) tmem_alloc(sb + SM_MISC, 512);
    if (warp == W_TMA && lane == 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_do);
    }
    if (do_zero) {  // the transition run: both dO stages hold zeros and are never loaded
        for (int i = threadIdx.x; i < 2 * 16384 / 16; i += NUM_THREADS)
            reinterpret_cast<uint4 *>(sm + SM_DO)[i] = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == W_TMA) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < nck; ++t) {
                const int st = t & 1;
                if (t >= 2 && !mbar_wait(bar(B_EMPTY0 + st), ((t >> 1) - 1) & 1, abort_flag)) {
                    record_timeout(p, B_EMPTY0 + st, t);
                    break;
                }
                const int tok0 = chunk_tok0(t);
                mbar_arrive_expect_tx(bar(B_FULL0 + st), do_zero ? 16384 : 32768);
                tma_load_3d(sb + SM_K + st * 16384, &tm_k, bar(B_FULL0 + st), 0, hq, tok0);
                tma_load_3d(sb + SM_K + st * 16384 + 8192, &tm_k, bar(B_FULL0 + st), 64, hq, tok0);
                if (!do_zero) {
                    tma_load_3d(sb + SM_DO + st * 16384, &tm_do, bar(B_FULL0 + st), 0, hv, tok0);
                    tma_load_3d(sb + SM_DO + st * 16384 + 8192, &tm_do, bar(B_FULL0 + st), 64, hv, tok0);
                }
                issued = t + 1;
            }
            for (int t = (issued > 2 ? issued - 2 : 0); t < issued; ++t) mbar_drain(bar(B_FULL0 + (t & 1)), (t >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0 && nck > 0) {
            int failed = -1, fj = 0;
            auto wait = [&](int id, uint32_t par, int t) {
                if (mbar_wait(bar(id), par, abort_flag)) return true;
                failed = id;
                fj = t;
                return false;
            };
            // PdO^T = dO^T P  (A = dO tile MN-major: v blocks at 8K, r' groups at 1K; B = P MN-major)
            auto pdo = [&](int t) {
                const int st = t & 1, sl = t & 1;
                for (int sp = 0; sp < 2; ++sp)
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t ao = sb + SM_DO + st * 16384 + kk * 2048;
                        uint32_t bo = sb + SM_P + sl * 16384 + sp * 8192 + kk * 2048;
                        mma_bf16(tmem + TM_PD, sdesc_sw128(ao, 8192, 1024), sdesc_sw128(bo, 8192, 1024),
                                 ID_N64_AMN_BMN, (sp | kk) != 0);
                    }
            };
            bool ok = wait(B_APREADY, 0, 0) && wait(B_FULL0, 0, 0);
            if (ok) {
                tc_fence_after();
                pdo(0);
            }
            for (int t = 0; ok && t < nck; ++t) {
                const int st = t & 1, ph = t & 1, sl = t & 1;
                if (!(ok = wait(B_DSREADY, ph, t))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // KdS^T = dS^T K^T, dS^T from TMEM
                    for (int kk = 0; kk < 8; ++kk) {
                        uint32_t bo = sb + SM_K + st * 16384 + (kk >> 2) * 8192 + (kk & 3) * 32;
                        mma_bf16_ta(tmem + TM_KD, tmem + (sp ? TM_SL : TM_SH) + kk * 8, sdesc_sw128(bo, 16, 1024),
                                    ID_N64, (sp | kk) != 0);
                    }
                mma_commit(bar(B_KDDONE));
                if (!(ok = wait(B_GQREADY, ph, t))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // U = dO^T (scale Gam o Q): A MN-major, B MN-major (2 key blocks)
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t ao = sb + SM_DO + st * 16384 + kk * 2048;
                        uint32_t bo = sb + SM_GQ + sp * 16384 + kk * 2048;
                        mma_bf16(tmem + TM_U, sdesc_sw128(ao, 8192, 1024), sdesc_sw128(bo, 8192, 1024),
                                 ID_N128_AMN_BMN, (sp | kk) != 0);
                    }
                if (!(ok = wait(B_DDREADY, ph, t))) break;
                tc_fence_after();
                for (int tt = 0; tt < 3; ++tt)  // dR^T = dDl^T A: (hi,hi) (hi,lo) (lo,hi)
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t ao = sb + SM_DD + (tt == 2 ? 16384 : 0) + kk * 32;
                        uint32_t bo = sb + SM_A + sl * 16384 + (tt == 1 ? 8192 : 0) + kk * 2048;
                        mma_bf16(tmem + TM_DR, sdesc_sw128(ao, 16, 1024), sdesc_sw128(bo, 8192, 1024), ID_N64_BMN,
                                 (tt | kk) != 0);
                    }
                mma_commit(bar(B_DRDONE));
                if (!(ok = wait(B_YREADY, ph, t))) break;
                tc_fence_after();
                for (int sp = 0; sp < 2; ++sp)  // U += (beta Gam o dR)^T K   (Y carries the minus sign)
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t ao = sb + SM_DD + sp * 16384 + kk * 32;
                        uint32_t bo = sb + SM_K + st * 16384 + kk * 2048;
                        mma_bf16(tmem + TM_U, sdesc_sw128(ao, 16, 1024), sdesc_sw128(bo, 8192, 1024), ID_N128_BMN,
                                 1);
                    }
                mma_commit(bar(B_UDONE));
                mma_commit(bar(B_EMPTY0 + st));
                if (t + 1 < nck) {
                    if (!(ok = wait(B_APREADY, (t + 1) & 1, t + 1))) break;
                    if (!(ok = wait(B_FULL0 + (st ^ 1), ((t + 1) >> 1) & 1, t + 1))) break;
                    tc_fence_after();
                    pdo(t + 1);
                }
            }
            mma_commit(bar(B_FINAL));
            mbar_drain(bar(B_FINAL), 0);
            if (failed >= 0) record_timeout(p, failed, fj);
        }
        __syncwarp();
    } else if (warp < W_STATE0) {
        // ------------------------------------------------------------------ aux warps
        const int pt = (warp - W_AUX0) * 32 + lane;  // 0..127
        const int r = pt >> 1, hh = pt & 1;          // tile row, column half
        int failed = -1, fj = 0, ap_issued = 0;
        auto gwait = [&](int id, uint32_t par, int t) {
            bool w = mbar_wait(bar(id), par, abort_flag);
            if (!w && failed < 0) { failed = id; fj = t; }
            return named_bar_and(1, 128, w);
        };
        // q row half and gate of tile row r, loaded one chunk ahead (the loads' latency overlaps a step)
        uint4 qn[8];
        float gn = 0.f;
        auto load_q = [&](int t) {
            const int tok0 = chunk_tok0(t), n = min(C, sr.tok1 - tok0);
            if (r < n) {
                gn = a.g_cum[(size_t)(tok0 + r) * p.Hv + hv];
                const uint4 *qrow =
                    reinterpret_cast<const uint4 *>(a.q + ((size_t)(tok0 + r) * p.Hq + hq) * DK + 64 * hh);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) qn[ch] = qrow[ch];
            }
        };
        if (nck > 0) load_q(0);
        for (int t = 0; t < nck; ++t) {
            const int j = nck - 1 - t, gc = sr.c0 + j, tok0 = chunk_tok0(t), n = min(C, sr.tok1 - tok0);
            const int sl = t & 1;
            // the MMA must have taken the previous step's tiles before this slot pair is reused
            if (t >= 1 && !gwait(B_KDDONE, (t - 1) & 1, t)) break;
            if (pt == 0) {  // A and P images of chunk gc into slot sl
                const unsigned char *img = a.tiles + ((size_t)gc * p.Hv + hv) * 32768;
                mbar_arrive_expect_tx(bar(B_APREADY), 32768);
                bulk_load(sb + SM_A + sl * 16384, img, 16384, bar(B_APREADY));
                bulk_load(sb + SM_P + sl * 16384, img + 16384, 16384, bar(B_APREADY));
                ++ap_issued;
            }
            // scale Gam o Q, once the previous step's U (its only reader) is done
            if (t >= 1 && !gwait(B_DRDONE, (t - 1) & 1, t)) break;
            {
                float gsc = 0.f;
                if (r < n) gsc = p.scale * __expf(gn);
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    float x[8];
                    if (r < n) {
                        uint4 w = qn[ch];
                        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            x[2 * e] = gsc * __uint_as_float(u[e] << 16);
                            x[2 * e + 1] = gsc * __uint_as_float(u[e] & 0xFFFF0000u);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] = 0.f;
                    }
                    st_split_chunk(sb + SM_GQ + hh * 8192, sb + SM_GQ + 16384 + hh * 8192, r, ch, x);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive_warp(bar(B_GQREADY));
            if (t + 1 < nck) load_q(t + 1);
        }
        if (pt == 0 && ap_issued > 0) mbar_drain(bar(B_APREADY), (ap_issued - 1) & 1);  // no copy left in flight
        if (failed >= 0) record_timeout(p, failed, fj);
    } else {
        // ------------------------------------------------------------------ state warps
        const int v = 32 * (warp & 3) + lane;
        const int sw = warp - W_STATE0, hh = sw >> 2;
        const uint32_t trow = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        float *wv = reinterpret_cast<float *>(sm + SM_VEC) + sw * 64;  // E[32], beta Gam[32] of this warp's rows
        int failed = -1, fj = 0;
        auto wwait = [&](int id, uint32_t par, int t) {
            bool w = mbar_wait_warp(bar(id), par, abort_flag);
            if (!w && failed < 0) { failed = id; fj = t; }
            return w;
        };
        float S[64];  // dS^T[v][64 hh .. 64 hh + 63]
#pragma unroll
        for (int i = 0; i < 64; ++i)
            S[i] = init ? init[(size_t)(64 * hh + i) * DV + v] : (init_identity && 64 * hh + i == v ? 1.f : 0.f);
        bool ok = true;
        for (int t = 0; t < nck && ok; ++t) {
            const int j = nck - 1 - t, gc = sr.c0 + j, tok0 = chunk_tok0(t), n = min(C, sr.tok1 - tok0);
            // gate values of this warp's chunk row c = 32 hh + lane, loaded first: their latency overlaps the
            // dS split below
            const int cg = 32 * hh + lane;
            const float glast = a.g_cum[(size_t)(tok0 + n - 1) * p.Hv + hv];
            float gcv = 0.f, btv = 0.f;
            if (cg < n) {
                const size_t gi = (size_t)(tok0 + cg) * p.Hv + hv;
                gcv = a.g_cum[gi];
                btv = a.beta[gi];
            }
            // (a) dS^T -> TMEM (hi / lo bf16 pairs) for KdS; dS at this chunk's end -> workspace
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // in halves: dS (64 registers) stays live throughout
                uint32_t hi[16], lo[16];
                split_pack16(S + 32 * hf, hi, lo);
                tmem_st16x2(trow + TM_SH + 32 * hh + 16 * hf, hi, trow + TM_SL + 32 * hh + 16 * hf, lo);
            }
            tc_fence_before();
            mbar_arrive_warp(bar(B_DSREADY));
            // gate vectors of this warp's 32 chunk rows c = 32 hh + lane
            float gl_all;
            {
                float e = 0.f, bg = 0.f;
                if (cg < n) {
                    e = __expf(glast - gcv);
                    bg = -btv * __expf(gcv);
                }
                wv[lane] = e;
                wv[32 + lane] = bg;
                gl_all = __expf(glast);
                __syncwarp();
            }
            // (c) dDl^T = scale PdO^T + KdS^T diag(E)
            if (!(ok = wwait(B_KDDONE, t & 1, t))) break;
            tc_fence_after();
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t kd16[16], pd16[16];
                float ew[16];
                lds16f(wv + 16 * hf, ew);
                tmem_ld16x2(trow + TM_KD + 32 * hh + 16 * hf, kd16, trow + TM_PD + 32 * hh + 16 * hf, pd16);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int i = 8 * q2 + e;
                        x[e] = fmaf(p.scale, __uint_as_float(pd16[i]), ew[i] * __uint_as_float(kd16[i]));
                    }
                    st_split_chunk(sb + SM_DD, sb + SM_DD + 16384, v, 4 * hh + 2 * hf + q2, x);
                }
            }
            uint32_t kd[32];
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive_warp(bar(B_DDREADY));
            if (dSe_out) {  // while dR is computed: dS at this chunk's end -> workspace
                float *dst = dSe_out + ((size_t)gc * p.Hv + hv) * DK * DV + (size_t)(64 * hh) * DV + v;
#pragma unroll
                for (int i = 0; i < 64; ++i) __stcs(dst + (size_t)i * DV, S[i]);
            }
            // (e) Y = -beta Gam o dR
            if (!(ok = wwait(B_DRDONE, t & 1, t))) break;
            tc_fence_after();
            tmem_ld32(trow + TM_DR + 32 * hh, kd);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float bw[16];
                lds16f(wv + 32 + 16 * hf, bw);
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = bw[8 * q2 + e] * __uint_as_float(kd[16 * hf + 8 * q2 + e]);
                    st_split_chunk(sb + SM_DD, sb + SM_DD + 16384, v, 4 * hh + 2 * hf + q2, x);
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();
            mbar_arrive_warp(bar(B_YREADY));
            // (g) dS^T <- Gam_last dS^T + U
            if (!(ok = wwait(B_UDONE, t & 1, t))) break;
            tc_fence_after();
            tmem_ld32(trow + TM_U + 64 * hh, kd);
#pragma unroll
            for (int i = 0; i < 32; ++i) S[i] = fmaf(gl_all, S[i], __uint_as_float(kd[i]));
            tmem_ld32(trow + TM_U + 64 * hh + 32, kd);
#pragma unroll
            for (int i = 0; i < 32; ++i) S[32 + i] = fmaf(gl_all, S[32 + i], __uint_as_float(kd[i]));
            tc_fence_before();
            __syncwarp();
        }
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

}  // namespace

cudaError_t launch_tc_dscan(const Plan &p, const void *q, const void *k, const void *d_o, const float *g_cum,
                            const float *beta, const unsigned char *tiles, const float *dht, float *dSe, float *dh0,
                            cudaStream_t st, const CpSplit *cp) {
    CUtensorMap tk, tdo;
    if (!make_head_map(&tk, k, p.Hq, p) || !make_head_map(&tdo, d_o, p.Hv, p)) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k_tc_dscan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    DscanArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.g_cum = g_cum;
    a.beta = beta;
    a.tiles = tiles;
    a.dht = dht;
    a.dSe = dSe;
    a.dh0 = dh0;
    a.seg_len = 0;
    a.n_seg = 1;
    a.mode = 0;
    a.seg_states = nullptr;
    a.seg_h = a.seg_M = nullptr;
    if (cp) {
        a.seg_len = cp->seg_len;
        a.n_seg = cp->n_seg;
        a.mode = cp->mode;
        a.seg_states = cp->seg_states;
        a.seg_h = cp->seg_h;
        a.seg_M = cp->seg_M;
    }
    dim3 grid(p.n_seqs * a.n_seg * (a.mode == CP_SEG ? 2 : 1), p.Hv);
    k_tc_dscan<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(tk, tdo, p, a);
    return cudaGetLastError();
}

}  // namespace gdn
