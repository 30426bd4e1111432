// simt.cu -- FFMA (CUDA-core) kernels of the chunked gated delta rule.
//
// This is the full-precision path: every product is an fp32 FMA chain and the
// chunk-local gate cumsum is carried in fp64 so that decays exp(gam_r - gam_i)
// of nearby tokens do not lose the low bits of two large cumsums.  It serves
// the fp32 io dtype and every head size the tensor-core path does not cover.
//
// Notation per chunk (n <= 64 rows, r / i row indices, S the entry state):
//   gam   chunk-local inclusive cumsum of g,  Gam_r = exp(gam_r)
//   D_ri  = exp(gam_r - gam_i) for i <= r
//   L     = strict_lower(diag(beta) (D o K K^T)),   A = (I + L)^{-1}
//   R     = diag(beta) (V - diag(Gam) K S)
//   Delta = A R                     (the "V correction" of the pages' step list)
//   O     = scale (diag(Gam) Q S + (D o Q K^T) Delta)
//   S'    = Gam_last S + K^T diag(E) Delta,   E_i = exp(gam_last - gam_i)
// Delta = U - W S with W, U the pages' "W and U variables"; this file never
// forms W or U: Delta = A R needs neither.
#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"

namespace gdn {

constexpr int NT = 256;  // threads per block of every SIMT kernel

// ---------------------------------------------------------------------------
// varlen chunk-offset table: chunk_off[s] = sum_{s' < s} ceil(len_s' / 64)
__global__ void k_chunk_table(const int32_t *cu, int n_seqs, int32_t *chunk_off) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    chunk_off[0] = 0;
    for (int s = 0; s < n_seqs; ++s) {
        int len = cu[s + 1] - cu[s];
        acc += (len + C - 1) / C;
        chunk_off[s + 1] = acc;
    }
}

// ---------------------------------------------------------------------------
// Per (chunk, q/k head): K K^T and Q K^T once, then for each value head of the
// group: gam (fp64), L, A = (I + L)^{-1}, P = D o Q K^T.
// Writes gam64 [tokens][Hv], A32 / P32 [chunks][Hv][64][64] (padded rows:
// A identity, P zero), and optionally g_cum (fp32) and A (io dtype).
template <typename IO, int KD>
__global__ void __launch_bounds__(NT)
k_prep(Plan p, const IO *__restrict__ q, const IO *__restrict__ k, const float *__restrict__ g_in,
       int g_is_cum, const float *__restrict__ beta, float *__restrict__ g_cum_out,
       IO *__restrict__ A_out, double *__restrict__ gam64, float *__restrict__ A32,
       float *__restrict__ P32) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int KS = KD + 1, CS = C + 1;
    double *gam = reinterpret_cast<double *>(smem_raw);   // [C]
    float *bet = reinterpret_cast<float *>(gam + C);       // [C]
    float *ks = bet + C;                                    // [C][KS]
    float *qs = ks + C * KS;                                // [C][KS]
    float *KK = qs + C * KS;                                // [C][CS]
    float *QK = KK + C * CS;                                // [C][CS]
    float *Lm = QK + C * CS;                                // [C][CS]
    float *Am = Lm + C * CS;                                // [C][CS]

    const int gc = blockIdx.x, hq = blockIdx.y, tid = threadIdx.x;
    const ChunkPos cp = chunk_pos(p, gc);
    const int n = cp.len;
    for (int idx = tid; idx < C * KD; idx += NT) {
        int r = idx / KD, d = idx % KD;
        float kv = 0.f, qv = 0.f;
        if (r < n) {
            size_t off = ((size_t)(cp.tok0 + r) * p.Hq + hq) * KD + d;
            kv = to_f(k[off]);
            qv = to_f(q[off]);
        }
        ks[r * KS + d] = kv;
        qs[r * KS + d] = qv;
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += NT) {
        int r = idx / C, i = idx % C;
        float a = 0.f, b = 0.f;
        if (i <= r) {
            for (int d = 0; d < KD; ++d) {
                float kid = ks[i * KS + d];
                a = fmaf(ks[r * KS + d], kid, a);
                b = fmaf(qs[r * KS + d], kid, b);
            }
        }
        KK[r * CS + i] = a;
        QK[r * CS + i] = b;
    }
    for (int gi = 0; gi < p.G; ++gi) {
        const int hv = hq * p.G + gi;
        __syncthreads();
        if (tid == 0) {
            double acc = 0.0;
            for (int r = 0; r < C; ++r) {
                if (r < n) {
                    size_t o = (size_t)(cp.tok0 + r) * p.Hv + hv;
                    acc = g_is_cum ? (double)g_in[o] : acc + (double)g_in[o];
                    bet[r] = beta[o];
                } else {
                    bet[r] = 0.f;
                }
                gam[r] = acc;
            }
        }
        __syncthreads();
        for (int r = tid; r < n; r += NT) {
            size_t o = (size_t)(cp.tok0 + r) * p.Hv + hv;
            gam64[o] = gam[r];
            if (g_cum_out) g_cum_out[o] = (float)gam[r];
        }
        for (int idx = tid; idx < C * C; idx += NT) {
            int r = idx / C, i = idx % C;
            float l = 0.f;
            if (i < r && r < n) l = bet[r] * expf((float)(gam[r] - gam[i])) * KK[r * CS + i];
            Lm[r * CS + i] = l;
        }
        __syncthreads();
        // forward substitution, one column per thread: A[r][j] = -sum_{j<=i<r} L[r][i] A[i][j]
        if (tid < C) {
            const int j = tid;
            for (int r = 0; r < C; ++r) {
                float a;
                if (r < j) a = 0.f;
                else if (r == j) a = 1.f;
                else {
                    float s = 0.f;
                    for (int i = j; i < r; ++i) s = fmaf(Lm[r * CS + i], Am[i * CS + j], s);
                    a = -s;
                }
                Am[r * CS + j] = a;
            }
        }
        __syncthreads();
        const size_t mat = ((size_t)gc * p.Hv + hv) * C * C;
        for (int idx = tid; idx < C * C; idx += NT) {
            int r = idx / C, i = idx % C;
            float a = Am[r * CS + i];
            A32[mat + idx] = a;
            float pv = 0.f;
            if (i <= r && r < n) pv = expf((float)(gam[r] - gam[i])) * QK[r * CS + i];
            P32[mat + idx] = pv;
            if (A_out && r < n) A_out[((size_t)(cp.tok0 + r) * p.Hv + hv) * C + i] = from_f<IO>(a);
        }
    }
}

// ---------------------------------------------------------------------------
// Serial forward scan over the chunks of one (sequence, value head, V block).
// Forward: writes o (and optionally h, final state).  Backward recompute:
// o == nullptr, h = the workspace copy of the chunk-entry states.
template <typename IO, int KD, int VB>
__global__ void __launch_bounds__(NT)
k_scan(Plan p, const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
       const float *__restrict__ beta, const double *__restrict__ gam64,
       const float *__restrict__ A32, const float *__restrict__ P32, const float *__restrict__ h0,
       IO *__restrict__ o, float *__restrict__ h, float *__restrict__ ht) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int RW = NT / VB;  // rows handled in parallel
    double *gam = reinterpret_cast<double *>(smem_raw);
    float *bet = reinterpret_cast<float *>(gam + C);
    float *Gm = bet + C;           // exp(gam)
    float *Ev = Gm + C;            // exp(gam_last - gam)
    float *ks = Ev + C;            // [C][KD]
    float *qs = ks + C * KD;       // [C][KD]
    float *Am = qs + C * KD;       // [C][C]
    float *Pm = Am + C * C;        // [C][C]
    float *S = Pm + C * C;         // [KD][VB]
    float *vs = S + KD * VB;       // [C][VB]
    float *KSb = vs + C * VB;      // [C][VB]  K S, then R, then E o Delta
    float *QSb = KSb + C * VB;     // [C][VB]
    float *Dl = QSb + C * VB;      // [C][VB]

    const int s = blockIdx.x, hv = blockIdx.y, vb = blockIdx.z, hq = hv / p.G;
    const int tid = threadIdx.x, j = tid % VB, w = tid / VB;
    const int VD = p.V;
    const SeqRange sr = seq_range(p, s);
    const size_t st_base = ((size_t)s * p.Hv + hv) * KD * VD + (size_t)vb * VB;

    for (int idx = tid; idx < KD * VB; idx += NT) {
        int d = idx / VB, jj = idx % VB;
        S[idx] = h0 ? h0[st_base + (size_t)d * VD + jj] : 0.f;
    }
    for (int gc = sr.c0; gc < sr.c1; ++gc) {
        const int tok0 = sr.tok0 + (gc - sr.c0) * C;
        const int n = min(C, sr.tok1 - tok0);
        __syncthreads();
        if (h) {
            const size_t hb = ((size_t)gc * p.Hv + hv) * KD * VD + (size_t)vb * VB;
            for (int idx = tid; idx < KD * VB; idx += NT)
                h[hb + (size_t)(idx / VB) * VD + idx % VB] = S[idx];
        }
        for (int idx = tid; idx < C * KD; idx += NT) {
            int r = idx / KD, d = idx % KD;
            float kv = 0.f, qv = 0.f;
            if (r < n) {
                size_t off = ((size_t)(tok0 + r) * p.Hq + hq) * KD + d;
                kv = to_f(k[off]);
                if (o) qv = to_f(q[off]);
            }
            ks[idx] = kv;
            qs[idx] = qv;
        }
        for (int idx = tid; idx < C * VB; idx += NT) {
            int r = idx / VB, jj = idx % VB;
            vs[idx] = r < n ? to_f(v[((size_t)(tok0 + r) * p.Hv + hv) * VD + vb * VB + jj]) : 0.f;
        }
        const size_t mat = ((size_t)gc * p.Hv + hv) * C * C;
        for (int idx = tid; idx < C * C; idx += NT) {
            Am[idx] = A32[mat + idx];
            Pm[idx] = o ? P32[mat + idx] : 0.f;
        }
        if (tid < C) {
            int r = tid;
            if (r < n) {
                size_t gi = (size_t)(tok0 + r) * p.Hv + hv;
                gam[r] = gam64[gi];
                bet[r] = beta[gi];
            } else {
                gam[r] = 0.0;
                bet[r] = 0.f;
            }
        }
        __syncthreads();
        const double glast = gam[n - 1];
        if (tid < C) {
            int r = tid;
            Gm[r] = r < n ? expf((float)gam[r]) : 0.f;
            Ev[r] = r < n ? expf((float)(glast - gam[r])) : 0.f;
        }
        // K S and Q S
        for (int r = w; r < C; r += RW) {
            float a = 0.f, b = 0.f;
            for (int d = 0; d < KD; ++d) {
                float sv = S[d * VB + j];
                a = fmaf(ks[r * KD + d], sv, a);
                b = fmaf(qs[r * KD + d], sv, b);
            }
            KSb[r * VB + j] = a;
            QSb[r * VB + j] = b;
        }
        __syncthreads();
        for (int r = w; r < C; r += RW)  // R = beta (v - Gam K S)
            KSb[r * VB + j] = bet[r] * (vs[r * VB + j] - Gm[r] * KSb[r * VB + j]);
        __syncthreads();
        for (int r = w; r < C; r += RW) {  // Delta = A R
            float a = 0.f;
            for (int i = 0; i <= r; ++i) a = fmaf(Am[r * C + i], KSb[i * VB + j], a);
            Dl[r * VB + j] = a;
        }
        __syncthreads();
        for (int r = w; r < C; r += RW) {
            if (o && r < n) {
                float a = 0.f;
                for (int i = 0; i <= r; ++i) a = fmaf(Pm[r * C + i], Dl[i * VB + j], a);
                float ov = p.scale * fmaf(Gm[r], QSb[r * VB + j], a);
                o[((size_t)(tok0 + r) * p.Hv + hv) * VD + vb * VB + j] = from_f<IO>(ov);
            }
            KSb[r * VB + j] = Ev[r] * Dl[r * VB + j];
        }
        __syncthreads();
        const float gl = Gm[n - 1];
        for (int d = w; d < KD; d += RW) {
            float a = 0.f;
            for (int r = 0; r < n; ++r) a = fmaf(ks[r * KD + d], KSb[r * VB + j], a);
            S[d * VB + j] = fmaf(gl, S[d * VB + j], a);
        }
    }
    __syncthreads();
    if (ht)
        for (int idx = tid; idx < KD * VB; idx += NT)
            ht[st_base + (size_t)(idx / VB) * VD + idx % VB] = S[idx];
}

// ---------------------------------------------------------------------------
// Reverse scan of the state gradient over the chunks of one (sequence, value
// head, V block).  dS enters a chunk as dL/d(state at its end):
//   dDelta = P^T dO' + diag(E) K dS,   dR = A^T dDelta,   dO' = scale dO
//   dS    <- Gam_last dS + Q^T diag(Gam) dO' - K^T diag(beta Gam) dR
// Stores dS_end of every chunk in dSe and the gradient of h0.
template <typename IO, int KD, int VB>
__global__ void __launch_bounds__(NT)
k_dscan(Plan p, const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ d_o,
        const float *__restrict__ beta, const double *__restrict__ gam64,
        const float *__restrict__ A32, const float *__restrict__ P32, const float *__restrict__ dht,
        float *__restrict__ dSe, float *__restrict__ dh0) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    constexpr int RW = NT / VB;
    double *gam = reinterpret_cast<double *>(smem_raw);
    float *bet = reinterpret_cast<float *>(gam + C);
    float *Gm = bet + C;
    float *Ev = Gm + C;
    float *ks = Ev + C;            // [C][KD]
    float *qs = ks + C * KD;       // [C][KD]
    float *Am = qs + C * KD;       // [C][C]
    float *Pm = Am + C * C;        // [C][C]
    float *dS = Pm + C * C;        // [KD][VB]
    float *dOs = dS + KD * VB;     // [C][VB]  scale dO, then Gam o scale dO
    float *KdS = dOs + C * VB;     // [C][VB]
    float *dDl = KdS + C * VB;     // [C][VB]
    float *dR = dDl + C * VB;      // [C][VB]  beta Gam dR

    const int s = blockIdx.x, hv = blockIdx.y, vb = blockIdx.z, hq = hv / p.G;
    const int tid = threadIdx.x, j = tid % VB, w = tid / VB;
    const int VD = p.V;
    const SeqRange sr = seq_range(p, s);
    const size_t st_base = ((size_t)s * p.Hv + hv) * KD * VD + (size_t)vb * VB;

    for (int idx = tid; idx < KD * VB; idx += NT)
        dS[idx] = dht ? dht[st_base + (size_t)(idx / VB) * VD + idx % VB] : 0.f;
    for (int gc = sr.c1 - 1; gc >= sr.c0; --gc) {
        const int tok0 = sr.tok0 + (gc - sr.c0) * C;
        const int n = min(C, sr.tok1 - tok0);
        __syncthreads();
        const size_t hb = ((size_t)gc * p.Hv + hv) * KD * VD + (size_t)vb * VB;
        for (int idx = tid; idx < KD * VB; idx += NT)
            dSe[hb + (size_t)(idx / VB) * VD + idx % VB] = dS[idx];
        for (int idx = tid; idx < C * KD; idx += NT) {
            int r = idx / KD, d = idx % KD;
            float kv = 0.f, qv = 0.f;
            if (r < n) {
                size_t off = ((size_t)(tok0 + r) * p.Hq + hq) * KD + d;
                kv = to_f(k[off]);
                qv = to_f(q[off]);
            }
            ks[idx] = kv;
            qs[idx] = qv;
        }
        for (int idx = tid; idx < C * VB; idx += NT) {
            int r = idx / VB, jj = idx % VB;
            dOs[idx] = r < n ? p.scale * to_f(d_o[((size_t)(tok0 + r) * p.Hv + hv) * VD + vb * VB + jj])
                             : 0.f;
        }
        const size_t mat = ((size_t)gc * p.Hv + hv) * C * C;
        for (int idx = tid; idx < C * C; idx += NT) {
            Am[idx] = A32[mat + idx];
            Pm[idx] = P32[mat + idx];
        }
        if (tid < C) {
            int r = tid;
            if (r < n) {
                size_t gi = (size_t)(tok0 + r) * p.Hv + hv;
                gam[r] = gam64[gi];
                bet[r] = beta[gi];
            } else {
                gam[r] = 0.0;
                bet[r] = 0.f;
            }
        }
        __syncthreads();
        const double glast = gam[n - 1];
        if (tid < C) {
            int r = tid;
            Gm[r] = r < n ? expf((float)gam[r]) : 0.f;
            Ev[r] = r < n ? expf((float)(glast - gam[r])) : 0.f;
        }
        for (int r = w; r < C; r += RW) {  // K dS
            float a = 0.f;
            for (int d = 0; d < KD; ++d) a = fmaf(ks[r * KD + d], dS[d * VB + j], a);
            KdS[r * VB + j] = a;
        }
        __syncthreads();
        for (int r = w; r < C; r += RW) {  // dDelta = P^T dO' + E o K dS
            float a = 0.f;
            for (int rr = r; rr < C; ++rr) a = fmaf(Pm[rr * C + r], dOs[rr * VB + j], a);
            dDl[r * VB + j] = fmaf(Ev[r], KdS[r * VB + j], a);
        }
        __syncthreads();
        for (int i = w; i < C; i += RW) {  // dR = A^T dDelta, stored scaled by beta Gam
            float a = 0.f;
            for (int r = i; r < C; ++r) a = fmaf(Am[r * C + i], dDl[r * VB + j], a);
            dR[i * VB + j] = bet[i] * Gm[i] * a;
            dOs[i * VB + j] *= Gm[i];
        }
        __syncthreads();
        const float gl = Gm[n - 1];
        for (int d = w; d < KD; d += RW) {
            float a = 0.f;
            for (int r = 0; r < n; ++r) {
                a = fmaf(qs[r * KD + d], dOs[r * VB + j], a);
                a = fmaf(-ks[r * KD + d], dR[r * VB + j], a);
            }
            dS[d * VB + j] = fmaf(gl, dS[d * VB + j], a);
        }
    }
    __syncthreads();
    if (dh0)
        for (int idx = tid; idx < KD * VB; idx += NT)
            dh0[st_base + (size_t)(idx / VB) * VD + idx % VB] = dS[idx];
}

// ---------------------------------------------------------------------------
// Per (chunk, q/k head): all parameter gradients of the chunk, looping over the
// value heads of the group (dq / dk accumulate in registers) and over V in
// blocks of VBI columns.  Needs the chunk-entry state h and dS_end.
template <typename IO, int KD>
__global__ void __launch_bounds__(NT)
k_bwd_intra(Plan p, const IO *__restrict__ q, const IO *__restrict__ k, const IO *__restrict__ v,
            const IO *__restrict__ d_o, const float *__restrict__ beta,
            const double *__restrict__ gam64, const float *__restrict__ A32,
            const float *__restrict__ P32, const float *__restrict__ hbuf,
            const float *__restrict__ dSe, IO *__restrict__ dq, IO *__restrict__ dk,
            IO *__restrict__ dv, float *__restrict__ dbeta, float *__restrict__ dg) {
    constexpr int VBI = 16, VBP = VBI + 1, CS = C + 1;
    constexpr int RPT = C * KD / NT;       // rows of dq / dk per thread
    constexpr int RSTEP = NT / KD;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    double *gam = reinterpret_cast<double *>(smem_raw);
    float *bet = reinterpret_cast<float *>(gam + C);
    float *Gm = bet + C;
    float *Ev = Gm + C;
    float *dgam = Ev + C;          // [C]
    float *dbet = dgam + C;        // [C]
    float *Fv = dbet + C;          // [C]
    float *red = Fv + C;           // [NT] scratch for <h, dSe>
    float *ks = red + NT;          // [C][KD]
    float *qs = ks + C * KD;       // [C][KD]
    float *KK = qs + C * KD;       // [C][CS]
    float *Am = KK + C * CS;       // [C][CS]
    float *Pm = Am + C * CS;       // [C][CS]
    float *dP = Pm + C * CS;       // [C][CS]
    float *dA = dP + C * CS;       // [C][CS]
    float *blk = dA + C * CS;      // V-block buffers, reused for M1 / dL afterwards
    float *hb = blk;               // [KD][VBP]
    float *dSb = hb + KD * VBP;    // [KD][VBP]
    float *vs = dSb + KD * VBP;    // [C][VBP]
    float *dOs = vs + C * VBP;     // [C][VBP]
    float *KSb = dOs + C * VBP;    // [C][VBP]
    float *QSb = KSb + C * VBP;    // [C][VBP]
    float *Rb = QSb + C * VBP;     // [C][VBP]
    float *Dl = Rb + C * VBP;      // [C][VBP]
    float *KdS = Dl + C * VBP;     // [C][VBP]
    float *dDl = KdS + C * VBP;    // [C][VBP]
    float *dR = dDl + C * VBP;     // [C][VBP]
    float *M1 = blk;               // [C][CS] (after the V loop)
    float *dL = blk + C * CS;      // [C][CS]

    const int gc = blockIdx.x, hq = blockIdx.y, tid = threadIdx.x;
    const ChunkPos cp = chunk_pos(p, gc);
    const int n = cp.len, tok0 = cp.tok0, VD = p.V;
    const int dcol = tid % KD, r0 = tid / KD;

    for (int idx = tid; idx < C * KD; idx += NT) {
        int r = idx / KD, d = idx % KD;
        float kv = 0.f, qv = 0.f;
        if (r < n) {
            size_t off = ((size_t)(tok0 + r) * p.Hq + hq) * KD + d;
            kv = to_f(k[off]);
            qv = to_f(q[off]);
        }
        ks[idx] = kv;
        qs[idx] = qv;
    }
    __syncthreads();
    for (int idx = tid; idx < C * C; idx += NT) {
        int r = idx / C, i = idx % C;
        float a = 0.f;
        if (i < r)
            for (int d = 0; d < KD; ++d) a = fmaf(ks[r * KD + d], ks[i * KD + d], a);
        KK[r * CS + i] = a;
    }
    float accq[RPT], acck[RPT];
#pragma unroll
    for (int m = 0; m < RPT; ++m) accq[m] = acck[m] = 0.f;

    for (int gi = 0; gi < p.G; ++gi) {
        const int hv = hq * p.G + gi;
        __syncthreads();
        const size_t mat = ((size_t)gc * p.Hv + hv) * C * C;
        for (int idx = tid; idx < C * C; idx += NT) {
            int r = idx / C, i = idx % C;
            Am[r * CS + i] = A32[mat + idx];
            Pm[r * CS + i] = P32[mat + idx];
            dP[r * CS + i] = 0.f;
            dA[r * CS + i] = 0.f;
        }
        if (tid < C) {
            int r = tid;
            if (r < n) {
                size_t gidx = (size_t)(tok0 + r) * p.Hv + hv;
                gam[r] = gam64[gidx];
                bet[r] = beta[gidx];
            } else {
                gam[r] = 0.0;
                bet[r] = 0.f;
            }
            dgam[r] = 0.f;
            dbet[r] = 0.f;
            Fv[r] = 0.f;
        }
        red[tid] = 0.f;
        __syncthreads();
        const double glast = gam[n - 1];
        if (tid < C) {
            int r = tid;
            Gm[r] = r < n ? expf((float)gam[r]) : 0.f;
            Ev[r] = r < n ? expf((float)(glast - gam[r])) : 0.f;
        }
        const size_t st = ((size_t)gc * p.Hv + hv) * KD * VD;
        for (int vb = 0; vb < VD / VBI; ++vb) {
            __syncthreads();
            for (int idx = tid; idx < KD * VBI; idx += NT) {
                int d = idx / VBI, jj = idx % VBI;
                size_t a = st + (size_t)d * VD + vb * VBI + jj;
                float hv_ = hbuf[a], ds_ = dSe[a];
                hb[d * VBP + jj] = hv_;
                dSb[d * VBP + jj] = ds_;
                red[tid] += hv_ * ds_;
            }
            for (int idx = tid; idx < C * VBI; idx += NT) {
                int r = idx / VBI, jj = idx % VBI;
                float vv = 0.f, dd = 0.f;
                if (r < n) {
                    size_t a = ((size_t)(tok0 + r) * p.Hv + hv) * VD + vb * VBI + jj;
                    vv = to_f(v[a]);
                    dd = p.scale * to_f(d_o[a]);
                }
                vs[r * VBP + jj] = vv;
                dOs[r * VBP + jj] = dd;
            }
            __syncthreads();
            // (r, j) products: K h, Q h, K dSe
            for (int idx = tid; idx < C * VBI; idx += NT) {
                int r = idx / VBI, jj = idx % VBI;
                float a = 0.f, b = 0.f, c = 0.f;
                for (int d = 0; d < KD; ++d) {
                    float kr = ks[r * KD + d];
                    a = fmaf(kr, hb[d * VBP + jj], a);
                    b = fmaf(qs[r * KD + d], hb[d * VBP + jj], b);
                    c = fmaf(kr, dSb[d * VBP + jj], c);
                }
                KSb[r * VBP + jj] = a;
                QSb[r * VBP + jj] = b;
                KdS[r * VBP + jj] = c;
                Rb[r * VBP + jj] = bet[r] * (vs[r * VBP + jj] - Gm[r] * a);
            }
            __syncthreads();
            for (int idx = tid; idx < C * VBI; idx += NT) {  // Delta, dDelta
                int r = idx / VBI, jj = idx % VBI;
                float a = 0.f, b = 0.f;
                for (int i = 0; i <= r; ++i) a = fmaf(Am[r * CS + i], Rb[i * VBP + jj], a);
                for (int rr = r; rr < C; ++rr) b = fmaf(Pm[rr * CS + r], dOs[rr * VBP + jj], b);
                Dl[r * VBP + jj] = a;
                dDl[r * VBP + jj] = fmaf(Ev[r], KdS[r * VBP + jj], b);
            }
            __syncthreads();
            for (int idx = tid; idx < C * VBI; idx += NT) {  // dR = A^T dDelta, dV
                int i = idx / VBI, jj = idx % VBI;
                float a = 0.f;
                for (int r = i; r < C; ++r) a = fmaf(Am[r * CS + i], dDl[r * VBP + jj], a);
                dR[i * VBP + jj] = a;
                if (i < n) dv[((size_t)(tok0 + i) * p.Hv + hv) * VD + vb * VBI + jj] = from_f<IO>(bet[i] * a);
            }
            __syncthreads();
            // per-row reductions over the block's columns
            if (tid < C) {
                int r = tid;
                float sb = 0.f, sg = 0.f, sf = 0.f;
                for (int jj = 0; jj < VBI; ++jj) {
                    float drv = dR[r * VBP + jj], ksv = KSb[r * VBP + jj];
                    sb = fmaf(drv, vs[r * VBP + jj] - Gm[r] * ksv, sb);
                    sg = fmaf(Gm[r] * dOs[r * VBP + jj], QSb[r * VBP + jj], sg);
                    sg = fmaf(-bet[r] * Gm[r] * drv, ksv, sg);
                    sf = fmaf(KdS[r * VBP + jj], Dl[r * VBP + jj], sf);
                }
                dbet[r] += sb;
                dgam[r] += sg;
                Fv[r] += Ev[r] * sf;
            }
            // dP += dO' Delta^T, dA += dDelta R^T (lower triangle incl. diagonal)
            for (int idx = tid; idx < C * C; idx += NT) {
                int r = idx / C, i = idx % C;
                if (i <= r) {
                    float a = 0.f, b = 0.f;
                    for (int jj = 0; jj < VBI; ++jj) {
                        a = fmaf(dOs[r * VBP + jj], Dl[i * VBP + jj], a);
                        b = fmaf(dDl[r * VBP + jj], Rb[i * VBP + jj], b);
                    }
                    dP[r * CS + i] += a;
                    dA[r * CS + i] += b;
                }
            }
            // dq += Gam dO' h^T ;  dk += E Delta dSe^T - beta Gam dR h^T
#pragma unroll
            for (int m = 0; m < RPT; ++m) {
                int r = r0 + m * RSTEP;
                float a = 0.f, b = 0.f, c = 0.f;
                for (int jj = 0; jj < VBI; ++jj) {
                    float hv_ = hb[dcol * VBP + jj];
                    a = fmaf(dOs[r * VBP + jj], hv_, a);
                    b = fmaf(Dl[r * VBP + jj], dSb[dcol * VBP + jj], b);
                    c = fmaf(dR[r * VBP + jj], hv_, c);
                }
                accq[m] = fmaf(Gm[r], a, accq[m]);
                acck[m] = fmaf(Ev[r], b, fmaf(-bet[r] * Gm[r], c, acck[m]));
            }
        }
        __syncthreads();
        // dL = -(A^T dA A^T), strict lower: M1 = A^T dA, dL = -M1 A^T
        for (int idx = tid; idx < C * C; idx += NT) {
            int r = idx / C, i = idx % C;
            float a = 0.f;
            for (int kk = max(r, i); kk < C; ++kk) a = fmaf(Am[kk * CS + r], dA[kk * CS + i], a);
            M1[r * CS + i] = a;
        }
        __syncthreads();
        for (int idx = tid; idx < C * C; idx += NT) {
            int r = idx / C, i = idx % C;
            float a = 0.f;
            if (i < r)
                for (int l = 0; l <= i; ++l) a = fmaf(M1[r * CS + l], Am[i * CS + l], a);
            dL[r * CS + i] = -a;
        }
        __syncthreads();
        // convert dP -> dQK = D o dP and dL -> dKK = beta_r D dL in place; gate terms
        for (int idx = tid; idx < C * C; idx += NT) {
            int r = idx / C, i = idx % C;
            float dqk = 0.f, dkk = 0.f;
            if (i <= r && r < n) {
                float D = expf((float)(gam[r] - gam[i]));
                dqk = D * dP[r * CS + i];
                if (i < r) dkk = bet[r] * D * dL[r * CS + i];
            }
            // M_ri = dP o P + dL o L (stored in dA, which is no longer needed)
            float l = (i < r && r < n) ? bet[r] * expf((float)(gam[r] - gam[i])) * KK[r * CS + i] : 0.f;
            dA[r * CS + i] = (i <= r && r < n) ? dP[r * CS + i] * Pm[r * CS + i] + dL[r * CS + i] * l : 0.f;
            dP[r * CS + i] = dqk;
            M1[r * CS + i] = dkk;
        }
        __syncthreads();
        if (tid < C) {
            int r = tid;
            float sb = 0.f, sg = 0.f;
            for (int i = 0; i < r; ++i) {
                float D = expf((float)(gam[r] - gam[i]));
                sb = fmaf(dL[r * CS + i] * D, KK[r * CS + i], sb);
            }
            for (int i = 0; i <= r; ++i) sg += dA[r * CS + i];
            for (int rr = r; rr < C; ++rr) sg -= dA[rr * CS + r];
            dbet[r] += sb;
            dgam[r] += sg - Fv[r];
        }
        if (tid == 0) {
            float hd = 0.f, fs = 0.f;
            for (int t = 0; t < NT; ++t) hd += red[t];
            for (int i = 0; i < n; ++i) fs += Fv[i];
            red[0] = Gm[n - 1] * hd + fs;  // goes to dgam[n-1] below
        }
        __syncthreads();
        if (tid == 0) {
            dgam[n - 1] += red[0];
            float acc = 0.f;  // reverse cumsum: dg_t = sum_{r >= t} dgam_r
            for (int r = n - 1; r >= 0; --r) {
                acc += dgam[r];
                size_t gidx = (size_t)(tok0 + r) * p.Hv + hv;
                dg[gidx] = acc;
                dbeta[gidx] = dbet[r];
            }
        }
        // dq += dQK K ;  dk += dQK^T Q + (dKK + dKK^T) K
#pragma unroll
        for (int m = 0; m < RPT; ++m) {
            int r = r0 + m * RSTEP;
            float a = 0.f, b = 0.f;
            for (int i = 0; i < C; ++i) {
                float ki = ks[i * KD + dcol];
                a = fmaf(dP[r * CS + i], ki, a);                       // dQK[r][i] k_i
                b = fmaf(dP[i * CS + r], qs[i * KD + dcol], b);        // dQK[i][r] q_i
                b = fmaf(M1[r * CS + i] + M1[i * CS + r], ki, b);      // (dKK + dKK^T)[r][i] k_i
            }
            accq[m] += a;
            acck[m] += b;
        }
    }
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        int r = r0 + m * RSTEP;
        if (r < n) {
            size_t off = ((size_t)(tok0 + r) * p.Hq + hq) * KD + dcol;
            dq[off] = from_f<IO>(accq[m]);
            dk[off] = from_f<IO>(acck[m]);
        }
    }
}

// ---------------------------------------------------------------------------
// host launchers
template <typename T>
static size_t smem_prep(int KD) { return (size_t)C * 8 + C * 4 + 2ull * C * (KD + 1) * 4 + 4ull * C * (C + 1) * 4; }
static size_t smem_scan(int KD, int VB) {
    return (size_t)C * 8 + 3ull * C * 4 + 2ull * C * KD * 4 + 2ull * C * C * 4 + (size_t)KD * VB * 4 +
           4ull * C * VB * 4;
}
static size_t smem_dscan(int KD, int VB) { return smem_scan(KD, VB) + (size_t)C * VB * 4; }
static size_t smem_intra(int KD) {
    const int VBP = 17, CS = C + 1;
    size_t blk = 2ull * KD * VBP * 4 + 9ull * C * VBP * 4;
    size_t blk2 = 2ull * C * CS * 4;
    return (size_t)C * 8 + 6ull * C * 4 + NT * 4 + 2ull * C * KD * 4 + 5ull * C * CS * 4 +
           (blk > blk2 ? blk : blk2);
}

template <typename KernelT>
static cudaError_t set_smem(KernelT kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

cudaError_t launch_chunk_table(const Plan &p, cudaStream_t st) {
    if (!p.cu) return cudaSuccess;
    k_chunk_table<<<1, 32, 0, st>>>(p.cu, p.n_seqs, p.chunk_off);
    return cudaGetLastError();
}

template <typename IO, int KD>
static cudaError_t prep_t(const Plan &p, const void *q, const void *k, const float *g, int g_is_cum,
                          const float *beta, float *g_cum, void *A_out, double *gam64, float *A32,
                          float *P32, cudaStream_t st) {
    size_t sm = smem_prep<IO>(KD);
    cudaError_t e = set_smem(k_prep<IO, KD>, sm);
    if (e != cudaSuccess) return e;
    dim3 grid(p.total_chunks, p.Hq);
    if (p.total_chunks == 0) return cudaSuccess;
    k_prep<IO, KD><<<grid, NT, sm, st>>>(p, (const IO *)q, (const IO *)k, g, g_is_cum, beta, g_cum,
                                         (IO *)A_out, gam64, A32, P32);
    return cudaGetLastError();
}

cudaError_t launch_simt_prep(const Plan &p, const void *q, const void *k, const float *g, int g_is_cum,
                             const float *beta, float *g_cum, void *A_out, double *gam64, float *A32,
                             float *P32, cudaStream_t st) {
    if (p.io == GDN_F32)
        return p.K == 64 ? prep_t<float, 64>(p, q, k, g, g_is_cum, beta, g_cum, A_out, gam64, A32, P32, st)
                         : prep_t<float, 128>(p, q, k, g, g_is_cum, beta, g_cum, A_out, gam64, A32, P32, st);
    return p.K == 64
               ? prep_t<__nv_bfloat16, 64>(p, q, k, g, g_is_cum, beta, g_cum, A_out, gam64, A32, P32, st)
               : prep_t<__nv_bfloat16, 128>(p, q, k, g, g_is_cum, beta, g_cum, A_out, gam64, A32, P32, st);
}

template <typename IO, int KD>
static cudaError_t scan_t(const Plan &p, const void *q, const void *k, const void *v, const float *beta,
                          const double *gam64, const float *A32, const float *P32, const float *h0,
                          void *o, float *h, float *ht, cudaStream_t st) {
    constexpr int VB = 32;
    size_t sm = smem_scan(KD, VB);
    cudaError_t e = set_smem(k_scan<IO, KD, VB>, sm);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seqs, p.Hv, p.V / VB);
    k_scan<IO, KD, VB><<<grid, NT, sm, st>>>(p, (const IO *)q, (const IO *)k, (const IO *)v, beta, gam64,
                                             A32, P32, h0, (IO *)o, h, ht);
    return cudaGetLastError();
}

cudaError_t launch_simt_scan(const Plan &p, const void *q, const void *k, const void *v, const float *beta,
                             const double *gam64, const float *A32, const float *P32, const float *h0,
                             void *o, float *h, float *ht, cudaStream_t st) {
    if (p.io == GDN_F32)
        return p.K == 64 ? scan_t<float, 64>(p, q, k, v, beta, gam64, A32, P32, h0, o, h, ht, st)
                         : scan_t<float, 128>(p, q, k, v, beta, gam64, A32, P32, h0, o, h, ht, st);
    return p.K == 64 ? scan_t<__nv_bfloat16, 64>(p, q, k, v, beta, gam64, A32, P32, h0, o, h, ht, st)
                     : scan_t<__nv_bfloat16, 128>(p, q, k, v, beta, gam64, A32, P32, h0, o, h, ht, st);
}

template <typename IO, int KD>
static cudaError_t dscan_t(const Plan &p, const void *q, const void *k, const void *d_o, const float *beta,
                           const double *gam64, const float *A32, const float *P32, const float *dht,
                           float *dSe, float *dh0, cudaStream_t st) {
    constexpr int VB = 32;
    size_t sm = smem_dscan(KD, VB);
    cudaError_t e = set_smem(k_dscan<IO, KD, VB>, sm);
    if (e != cudaSuccess) return e;
    dim3 grid(p.n_seqs, p.Hv, p.V / VB);
    k_dscan<IO, KD, VB><<<grid, NT, sm, st>>>(p, (const IO *)q, (const IO *)k, (const IO *)d_o, beta,
                                              gam64, A32, P32, dht, dSe, dh0);
    return cudaGetLastError();
}

cudaError_t launch_simt_dscan(const Plan &p, const void *q, const void *k, const void *d_o, const float *beta,
                              const double *gam64, const float *A32, const float *P32, const float *dht,
                              float *dSe, float *dh0, cudaStream_t st) {
    if (p.io == GDN_F32)
        return p.K == 64 ? dscan_t<float, 64>(p, q, k, d_o, beta, gam64, A32, P32, dht, dSe, dh0, st)
                         : dscan_t<float, 128>(p, q, k, d_o, beta, gam64, A32, P32, dht, dSe, dh0, st);
    return p.K == 64 ? dscan_t<__nv_bfloat16, 64>(p, q, k, d_o, beta, gam64, A32, P32, dht, dSe, dh0, st)
                     : dscan_t<__nv_bfloat16, 128>(p, q, k, d_o, beta, gam64, A32, P32, dht, dSe, dh0, st);
}

template <typename IO, int KD>
static cudaError_t intra_t(const Plan &p, const void *q, const void *k, const void *v, const void *d_o,
                           const float *beta, const double *gam64, const float *A32, const float *P32,
                           const float *hbuf, const float *dSe, void *dq, void *dk, void *dv, float *dbeta,
                           float *dg, cudaStream_t st) {
    size_t sm = smem_intra(KD);
    cudaError_t e = set_smem(k_bwd_intra<IO, KD>, sm);
    if (e != cudaSuccess) return e;
    if (p.total_chunks == 0) return cudaSuccess;
    dim3 grid(p.total_chunks, p.Hq);
    k_bwd_intra<IO, KD><<<grid, NT, sm, st>>>(p, (const IO *)q, (const IO *)k, (const IO *)v,
                                              (const IO *)d_o, beta, gam64, A32, P32, hbuf, dSe, (IO *)dq,
                                              (IO *)dk, (IO *)dv, dbeta, dg);
    return cudaGetLastError();
}

cudaError_t launch_simt_bwd_intra(const Plan &p, const void *q, const void *k, const void *v, const void *d_o,
                                  const float *beta, const double *gam64, const float *A32,
                                  const float *P32, const float *hbuf, const float *dSe, void *dq, void *dk,
                                  void *dv, float *dbeta, float *dg, cudaStream_t st) {
    if (p.io == GDN_F32)
        return p.K == 64 ? intra_t<float, 64>(p, q, k, v, d_o, beta, gam64, A32, P32, hbuf, dSe, dq, dk, dv,
                                              dbeta, dg, st)
                         : intra_t<float, 128>(p, q, k, v, d_o, beta, gam64, A32, P32, hbuf, dSe, dq, dk, dv,
                                               dbeta, dg, st);
    return p.K == 64 ? intra_t<__nv_bfloat16, 64>(p, q, k, v, d_o, beta, gam64, A32, P32, hbuf, dSe, dq, dk,
                                                  dv, dbeta, dg, st)
                     : intra_t<__nv_bfloat16, 128>(p, q, k, v, d_o, beta, gam64, A32, P32, hbuf, dSe, dq, dk,
                                                   dv, dbeta, dg, st);
}

}  // namespace gdn
