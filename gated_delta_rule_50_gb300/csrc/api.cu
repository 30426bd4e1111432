// api.cu -- the extern "C" entry points of include/gdn.h: host-side validation,
// workspace layout and the launch sequence.  No device memory is allocated and
// the stream is never synchronised (except in gdn_workspace_error, which says so).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "gdn.h"
#include "launch.h"
#include "profile.h"

using namespace gdn;

namespace {

// Test aid of gdn_debug_set_wait: the forward chain's wait limit (0: the default) and dropped load.
std::atomic<long long> g_dbg_wait_ns{0};
std::atomic<int> g_dbg_drop_chunk{-1};
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool ok_ptr(const void *ptr) { return ptr != nullptr && aligned16(ptr); }
bool ok_opt(const void *ptr) { return ptr == nullptr || aligned16(ptr); }

// Validates the problem and fills the host part of the plan.
gdn_status make_plan(const gdn_problem *pr, Plan *pl) {
    if (!pr) return GDN_ERR_INVALID_ARG;
    if (pr->B < 1 || pr->T < 0 || pr->Hq < 1 || pr->Hv < 1 || pr->K < 1 || pr->V < 1)
        return GDN_ERR_INVALID_ARG;
    if (pr->Hv % pr->Hq != 0) return GDN_ERR_INVALID_ARG;
    if (pr->io_dtype != GDN_F32 && pr->io_dtype != GDN_BF16) return GDN_ERR_INVALID_ARG;
    if (pr->cp_mode < GDN_CP_AUTO || pr->cp_mode > GDN_CP_WARMUP) return GDN_ERR_INVALID_ARG;
    if (pr->cp_mode == GDN_CP_WARMUP && (pr->warmup_chunks < 1 || pr->warmup_chunks > 64))
        return GDN_ERR_INVALID_ARG;
    if (pr->out_f32 != 0 && pr->out_f32 != 1) return GDN_ERR_INVALID_ARG;
    if ((pr->K != 64 && pr->K != 128) || (pr->V != 64 && pr->V != 128)) return GDN_ERR_UNSUPPORTED;
    if (pr->B * pr->T > INT32_MAX / 2 || pr->Hv > 65535 || pr->Hq > 65535) return GDN_ERR_UNSUPPORTED;
    std::memset(pl, 0, sizeof(*pl));
    pl->B = (int)pr->B; pl->T = (int)pr->T; pl->Hq = (int)pr->Hq; pl->Hv = (int)pr->Hv;
    pl->K = (int)pr->K; pl->V = (int)pr->V; pl->G = (int)(pr->Hv / pr->Hq);
    pl->io = pr->io_dtype;
    pl->scale = pr->scale;
    pl->out_f32 = pr->io_dtype == GDN_BF16 ? pr->out_f32 : 0;
    const long long wns = g_dbg_wait_ns.load();
    pl->wait_ns = wns > 0 ? (unsigned long long)wns : kDefaultWaitNs;
    pl->drop_load_chunk = g_dbg_drop_chunk.load();
    pl->cp_mode = pr->cp_mode;
    pl->warmup_chunks = pr->warmup_chunks;
    if (pr->cu_seqlens) {
        if (pr->B != 1 || pr->n_seqs < 1 || !pr->cu_seqlens_host) return GDN_ERR_INVALID_ARG;
        if (pr->n_seqs > INT32_MAX / 4) return GDN_ERR_UNSUPPORTED;
        const int32_t *cu = pr->cu_seqlens_host;
        if (cu[0] != 0 || cu[pr->n_seqs] != pr->T) return GDN_ERR_INVALID_ARG;
        int64_t chunks = 0, mx = 0, mxl = 0;
        for (int64_t s = 0; s < pr->n_seqs; ++s) {
            if (cu[s + 1] < cu[s]) return GDN_ERR_INVALID_ARG;
            int64_t c = (cu[s + 1] - cu[s] + C - 1) / C;
            chunks += c;
            mx = c > mx ? c : mx;
            mxl = cu[s + 1] - cu[s] > mxl ? cu[s + 1] - cu[s] : mxl;
        }
        pl->max_seq_len = (int)mxl;
        pl->n_seqs = (int)pr->n_seqs;
        pl->cu = pr->cu_seqlens;
        pl->total_chunks = (int)chunks;
        pl->max_seq_chunks = (int)mx;
        pl->NC = 0;
    } else {
        if (pr->cu_seqlens_host) return GDN_ERR_INVALID_ARG;
        if (pr->n_seqs != pr->B) return GDN_ERR_INVALID_ARG;
        pl->n_seqs = (int)pr->B;
        pl->NC = (int)((pr->T + C - 1) / C);
        pl->total_chunks = pl->NC * pl->B;
        pl->max_seq_chunks = pl->NC;
        pl->max_seq_len = pl->T;
    }
    return GDN_OK;
}

struct FwdWs {
    size_t err, chunk_off, gam64, A32, P32, tiles, vecs, serial, seg_states, seg_h, seg_M, total;
    int seg_len, n_seg;  // n_seg > 1: sequence splitting is planned
    bool exact;          // exact split (transitions) rather than warmup
};
struct BwdWs {
    size_t err, chunk_off, gam64, A32, P32, tiles, vecs, hbuf, dSe, seg_states, seg_h, seg_M, total;
    int seg_len, n_seg;  // n_seg > 1: both backward chains are split exactly
};

// Sequence splitting with warmup runs when asked for, supported and triggered.
bool warmup_split(const Plan &p) {
    if (p.cp_mode != GDN_CP_WARMUP || !tc_fwd_supported(p) || !cp_trigger(p)) return false;
    int L, n;
    cp_geometry(p, &L, &n);
    return n > 1;
}

// Exact sequence splitting (segment transitions, no approximation) in the default mode.
bool exact_split(const Plan &p) {
    if (p.cp_mode != GDN_CP_AUTO || !tc_fwd_supported(p) || !cp_trigger(p) || p.K != p.V) return false;
    int L, n;
    cp_geometry(p, &L, &n);
    return n > 1;
}

FwdWs fwd_layout(const Plan &p) {
    Carve c;
    FwdWs w;
    size_t tokens = (size_t)p.B * p.T;
    size_t mats = (size_t)p.total_chunks * p.Hv * C * C;
    w.err = c.take<uint32_t>(64);
    w.chunk_off = c.take<int32_t>((size_t)p.n_seqs + 1);
    // fp64 gate sums and fp32 A / P scratch serve only the CUDA-core path
    const bool simt = !tc_fwd_supported(p);
    w.gam64 = c.take<double>(simt ? tokens * p.Hv : 0);
    w.A32 = c.take<float>(simt ? mats : 0);
    w.P32 = c.take<float>(simt ? mats : 0);
    // tensor-core path: per (chunk, value head) A / P operand images and gate vectors
    const size_t units = simt ? 0 : (size_t)p.total_chunks * p.Hv;
    w.tiles = c.take<unsigned char>(units * TC_TILE_BYTES);
    w.vecs = c.take<float>(units * TC_VEC_FLOATS);
    w.seg_len = 0;
    w.n_seg = 1;
    w.serial = w.seg_states = w.seg_h = w.seg_M = 0;
    w.exact = exact_split(p);
    if (w.exact || warmup_split(p)) {
        cp_geometry(p, &w.seg_len, &w.n_seg);
        const size_t st = (size_t)p.n_seqs * p.Hv * w.n_seg * p.K * p.V;
        w.seg_states = c.take<float>(st);
        if (w.exact) {
            w.seg_h = c.take<float>(st);
            w.seg_M = c.take<float>(st);
        } else {
            w.serial = c.take<uint8_t>((size_t)p.n_seqs * p.Hv);
        }
    }
    w.total = c.off;
    return w;
}

BwdWs bwd_layout(const Plan &p) {
    Carve c;
    BwdWs w;
    size_t tokens = (size_t)p.B * p.T;
    size_t mats = (size_t)p.total_chunks * p.Hv * C * C;
    size_t states = (size_t)p.total_chunks * p.Hv * p.K * p.V;
    w.err = c.take<uint32_t>(64);
    w.chunk_off = c.take<int32_t>((size_t)p.n_seqs + 1);
    // fp64 gate sums and fp32 A / P serve only the CUDA-core path
    w.gam64 = c.take<double>(tc_fwd_supported(p) ? 0 : tokens * p.Hv);
    w.A32 = c.take<float>(tc_fwd_supported(p) ? 0 : mats);
    w.P32 = c.take<float>(tc_fwd_supported(p) ? 0 : mats);
    const size_t units = tc_fwd_supported(p) ? (size_t)p.total_chunks * p.Hv : 0;
    w.tiles = c.take<unsigned char>(units * TC_TILE_BYTES);
    w.vecs = c.take<float>(units * TC_VEC_FLOATS);
    w.hbuf = c.take<float>(states);
    w.dSe = c.take<float>(states);
    w.seg_len = 0;
    w.n_seg = 1;
    w.seg_states = w.seg_h = w.seg_M = 0;
    if (exact_split(p)) {  // segment buffers, used in turn by the state recompute and the dS scan
        cp_geometry(p, &w.seg_len, &w.n_seg);
        const size_t st = (size_t)p.n_seqs * p.Hv * w.n_seg * p.K * p.V;
        w.seg_states = c.take<float>(st);
        w.seg_h = c.take<float>(st);
        w.seg_M = c.take<float>(st);
    }
    w.total = c.off;
    return w;
}

template <typename T> T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<unsigned char *>(ws) + off);
}

// bf16 problems with a 64-wide head run the 128-wide tensor-core kernels on zero-padded copies (pad.cu)
bool pad_to_tc(const Plan &p) { return p.io == GDN_BF16 && (p.K != 128 || p.V != 128); }
Plan padded_plan(const Plan &p) {
    Plan q = p;
    q.K = 128;
    q.V = 128;
    return q;
}
// Workspace of the padded forward: the 128-wide path's own workspace first (its error record stays at
// offset 0), then the padded inputs and the 128-wide outputs that are sliced back.
// The padded output o comes last, so that what a saved backward reads (the inner workspace and the
// 128-wide states h, ending at saved_end) sits at the same offsets whatever the output dtype.
struct PadFwdWs {
    size_t inner, q, k, v, h0, ht, h, saved_end, o, total;
};
PadFwdWs pad_fwd_layout(const Plan &p) {
    const Plan pp = padded_plan(p);
    const size_t tokens = (size_t)p.B * p.T, state = 128 * 128, nst = (size_t)p.n_seqs * p.Hv;
    Carve c;
    PadFwdWs w;
    w.inner = c.take<unsigned char>(fwd_layout(pp).total);
    w.q = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 : 0);
    w.k = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 : 0);
    w.v = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 : 0);
    w.h0 = c.take<float>(nst * state);
    w.ht = c.take<float>(nst * state);
    w.h = c.take<float>((size_t)p.total_chunks * p.Hv * state);
    w.saved_end = c.off;
    w.o = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.total = c.off;
    return w;
}
struct PadBwdWs {
    size_t inner, q, k, v, d_o, h0, dht, dq, dk, dv, dh0, total;
};
PadBwdWs pad_bwd_layout(const Plan &p) {
    const Plan pp = padded_plan(p);
    const size_t tokens = (size_t)p.B * p.T, state = 128 * 128, nst = (size_t)p.n_seqs * p.Hv;
    Carve c;
    PadBwdWs w;
    w.inner = c.take<unsigned char>(bwd_layout(pp).total);
    w.q = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 : 0);
    w.k = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 : 0);
    w.dq = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.dk = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.v = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 : 0);
    w.d_o = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 : 0);
    w.dv = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.h0 = c.take<float>(nst * state);
    w.dht = c.take<float>(nst * state);
    w.dh0 = c.take<float>(nst * state);
    w.total = c.off;
    return w;
}

#define GDN_TRY(expr)                                  \
    do {                                               \
        cudaError_t e_ = (expr);                       \
        if (e_ != cudaSuccess) return GDN_ERR_CUDA;    \
    } while (0)

// Launch with an optional timing bracket named after the kernel.
#define GDN_LAUNCH(name, expr)                         \
    do {                                               \
        ProfScope ps_(name, st);                       \
        GDN_TRY(expr);                                 \
    } while (0)

// Workspace of gdn_bwd_saved: the backward without its recompute passes.
struct BwdSavedWs {
    size_t err, chunk_off, dSe, seg_states, seg_h, seg_M, total;
    int seg_len, n_seg;
};
BwdSavedWs bwd_saved_layout(const Plan &p) {
    Carve c;
    BwdSavedWs w;
    w.err = c.take<uint32_t>(64);
    w.chunk_off = c.take<int32_t>((size_t)p.n_seqs + 1);
    w.dSe = c.take<float>((size_t)p.total_chunks * p.Hv * p.K * p.V);
    w.seg_len = 0;
    w.n_seg = 1;
    w.seg_states = w.seg_h = w.seg_M = 0;
    if (exact_split(p)) {
        cp_geometry(p, &w.seg_len, &w.n_seg);
        const size_t st = (size_t)p.n_seqs * p.Hv * w.n_seg * p.K * p.V;
        w.seg_states = c.take<float>(st);
        w.seg_h = c.take<float>(st);
        w.seg_M = c.take<float>(st);
    }
    w.total = c.off;
    return w;
}

struct PadBwdSavedWs {
    size_t inner, q, k, v, d_o, dht, dq, dk, dv, dh0, total;
};
PadBwdSavedWs pad_bwd_saved_layout(const Plan &p) {
    const Plan pp = padded_plan(p);
    const size_t tokens = (size_t)p.B * p.T, state = 128 * 128, nst = (size_t)p.n_seqs * p.Hv;
    Carve c;
    PadBwdSavedWs w;
    w.inner = c.take<unsigned char>(bwd_saved_layout(pp).total);
    w.q = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 : 0);
    w.k = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 : 0);
    w.dq = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.dk = c.take<uint16_t>(p.K < 128 ? tokens * p.Hq * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.v = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 : 0);
    w.d_o = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 : 0);
    w.dv = c.take<uint16_t>(p.V < 128 ? tokens * p.Hv * 128 * (p.out_f32 ? 2 : 1) : 0);
    w.dht = c.take<float>(nst * state);
    w.dh0 = c.take<float>(nst * state);
    w.total = c.off;
    return w;
}

// The saved backward's launch sequence (dS scan, per-chunk gradients) for a validated tensor-core plan,
// reading the forward's operand images, gate vectors and chunk-entry states.
gdn_status bwd_saved_impl(Plan pl, const void *q, const void *k, const void *v, const float *g_cum,
                          const float *beta, const void *d_o, const float *dht, const unsigned char *tiles,
                          const float *vecs, const float *h, void *dq, void *dk, void *dv, float *dbeta, float *dg,
                          float *dh0, void *workspace, cudaStream_t st);

}  // namespace

extern "C" {

size_t gdn_fwd_workspace_bytes(const gdn_problem *p) {
    Plan pl;
    if (make_plan(p, &pl) != GDN_OK) return 0;
    return pad_to_tc(pl) ? pad_fwd_layout(pl).total : fwd_layout(pl).total;
}

size_t gdn_bwd_workspace_bytes(const gdn_problem *p) {
    Plan pl;
    if (make_plan(p, &pl) != GDN_OK) return 0;
    return pad_to_tc(pl) ? pad_bwd_layout(pl).total : bwd_layout(pl).total;
}

}  // extern "C"

namespace {

// The forward's launch sequence for a validated plan (arguments checked by gdn_fwd).
gdn_status fwd_impl(Plan pl, const void *q, const void *k, const void *v, const float *g, const float *beta,
                    const float *h0, void *o, float *g_cum, void *A, float *h, float *final_state, void *workspace,
                    cudaStream_t st) {
    FwdWs w = fwd_layout(pl);
    pl.err = at<uint32_t>(workspace, w.err);
    pl.chunk_off = pl.cu ? at<int32_t>(workspace, w.chunk_off) : nullptr;
    GDN_TRY(cudaMemsetAsync(pl.err, 0, 256, st));
    GDN_LAUNCH("chunk_table", launch_chunk_table(pl, st));
    double *gam64 = at<double>(workspace, w.gam64);
    float *A32 = at<float>(workspace, w.A32), *P32 = at<float>(workspace, w.P32);
    unsigned char *tiles = at<unsigned char>(workspace, w.tiles);
    float *vecs = at<float>(workspace, w.vecs);
    if (tc_fwd_supported(pl))  // A, P and the gate vectors of every chunk, in parallel
        GDN_LAUNCH("fwd_prep_tc", launch_tc_prep(pl, q, k, g, false, beta, g_cum, A, nullptr, nullptr, tiles, vecs, st));
    if (w.n_seg > 1) {  // sequence splitting
        CpSplit cs;
        cs.seg_len = w.seg_len;
        cs.n_seg = w.n_seg;
        cs.warm = pl.warmup_chunks;
        cs.serial = nullptr;
        cs.seg_states = at<float>(workspace, w.seg_states);
        cs.seg_h = cs.seg_M = nullptr;
        if (w.exact) {  // segment contributions and transitions, then the scan over segments
            cs.seg_h = at<float>(workspace, w.seg_h);
            cs.seg_M = at<float>(workspace, w.seg_M);
            cs.mode = CP_SEG;
            GDN_LAUNCH("fwd_tc_seg", launch_tc_fwd(pl, q, k, v, tiles, vecs, nullptr, nullptr, nullptr, nullptr, st, &cs));
            GDN_LAUNCH("cp_combine", launch_cp_combine(pl, h0, cs.seg_h, cs.seg_M, cs.seg_len, cs.n_seg, cs.seg_states,
                                                       st));
        } else {  // warmup: each segment after the first starts from a zero-state run over its window
            uint8_t *serial = at<uint8_t>(workspace, w.serial);
            cs.serial = serial;
            GDN_LAUNCH("cp_flags", launch_cp_flags(pl, g, cs.seg_len, cs.n_seg, cs.warm, serial, st));
            cs.mode = CP_WARM;
            GDN_LAUNCH("fwd_tc_warm",
                       launch_tc_fwd(pl, q, k, v, tiles, vecs, nullptr, nullptr, nullptr, nullptr, st, &cs));
        }
        cs.mode = CP_MAIN;
        GDN_LAUNCH("fwd_tc", launch_tc_fwd(pl, q, k, v, tiles, vecs, h0, o, h, final_state, st, &cs));
        return GDN_OK;
    }
    if (tc_fwd_supported(pl)) {
        GDN_LAUNCH("fwd_tc", launch_tc_fwd(pl, q, k, v, tiles, vecs, h0, o, h, final_state, st));
        return GDN_OK;
    }
    if (pl.total_chunks > 0)
        GDN_LAUNCH("fwd_prep", launch_simt_prep(pl, q, k, g, 0, beta, g_cum, A, gam64, A32, P32, st));
    GDN_LAUNCH("fwd_scan", launch_simt_scan(pl, q, k, v, beta, gam64, A32, P32, h0, o, h, final_state, st));
    return GDN_OK;
}

// The backward's launch sequence for a validated plan (arguments checked by gdn_bwd).
gdn_status bwd_impl(Plan pl, const void *q, const void *k, const void *v, const float *g_cum, const float *beta,
                    const void *d_o, const float *dht, const float *h0, void *dq, void *dk, void *dv, float *dbeta,
                    float *dg, float *dh0, void *workspace, cudaStream_t st);

}  // namespace

extern "C" {

gdn_status gdn_fwd(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g,
                   const float *beta, const float *h0, void *o, float *g_cum, void *A, float *h,
                   float *final_state, void *workspace, size_t workspace_bytes, gdn_stream_t stream) {
    Plan pl;
    gdn_status s = make_plan(p, &pl);
    if (s != GDN_OK) return s;
    const bool any_tok = (size_t)pl.B * pl.T > 0;
    if (any_tok && !(ok_ptr(q) && ok_ptr(k) && ok_ptr(v) && ok_ptr(g) && ok_ptr(beta) && ok_ptr(o)))
        return GDN_ERR_INVALID_ARG;
    if (!(ok_opt(h0) && ok_opt(g_cum) && ok_opt(A) && ok_opt(h) && ok_opt(final_state)))
        return GDN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!pad_to_tc(pl)) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < fwd_layout(pl).total)
            return GDN_ERR_WORKSPACE;
        return fwd_impl(pl, q, k, v, g, beta, h0, o, g_cum, A, h, final_state, workspace, st);
    }
    // a 64-wide head: pad to the 128-wide tiles, run, slice the outputs back
    const PadFwdWs w = pad_fwd_layout(pl);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.total)
        return GDN_ERR_WORKSPACE;
    const size_t tokens = (size_t)pl.B * pl.T, nst = (size_t)pl.n_seqs * pl.Hv;
    const void *qp = q, *kp = k, *vp = v;
    void *op = o;
    if (pl.K < 128) {
        qp = at<void>(workspace, w.q);
        kp = at<void>(workspace, w.k);
        GDN_LAUNCH("pad", launch_pad_rows(q, const_cast<void *>(qp), tokens * pl.Hq, pl.K, st));
        GDN_LAUNCH("pad", launch_pad_rows(k, const_cast<void *>(kp), tokens * pl.Hq, pl.K, st));
    }
    if (pl.V < 128) {
        vp = at<void>(workspace, w.v);
        op = at<void>(workspace, w.o);
        GDN_LAUNCH("pad", launch_pad_rows(v, const_cast<void *>(vp), tokens * pl.Hv, pl.V, st));
    }
    float *h0p = h0 ? at<float>(workspace, w.h0) : nullptr;
    if (h0) GDN_LAUNCH("pad", launch_pad_states(h0, h0p, nst, pl.K, pl.V, st));
    float *htp = final_state ? at<float>(workspace, w.ht) : nullptr;
    float *hp = h ? at<float>(workspace, w.h) : nullptr;
    s = fwd_impl(padded_plan(pl), qp, kp, vp, g, beta, h0p, op, g_cum, A, hp, htp, at<void>(workspace, w.inner), st);
    if (s != GDN_OK) return s;
    if (pl.V < 128) GDN_LAUNCH("slice", launch_slice_rows(op, o, tokens * pl.Hv, pl.V, pl.out_f32 ? 4 : 2, st));
    if (final_state) GDN_LAUNCH("slice", launch_slice_states(htp, final_state, nst, pl.K, pl.V, st));
    if (h) GDN_LAUNCH("slice", launch_slice_states(hp, h, (size_t)pl.total_chunks * pl.Hv, pl.K, pl.V, st));
    return GDN_OK;
}

gdn_status gdn_bwd(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g_cum,
                   const float *beta, const void *A, const void *d_o, const float *dht, const float *h0,
                   void *dq, void *dk, void *dv, float *dbeta, float *dg, float *dh0, void *workspace,
                   size_t workspace_bytes, gdn_stream_t stream) {
    (void)A;  // the inverse is recomputed in fp32 (see the header)
    Plan pl;
    gdn_status s = make_plan(p, &pl);
    if (s != GDN_OK) return s;
    const bool any_tok = (size_t)pl.B * pl.T > 0;
    if (any_tok && !(ok_ptr(q) && ok_ptr(k) && ok_ptr(v) && ok_ptr(g_cum) && ok_ptr(beta) && ok_ptr(d_o) &&
                     ok_ptr(dq) && ok_ptr(dk) && ok_ptr(dv) && ok_ptr(dbeta) && ok_ptr(dg)))
        return GDN_ERR_INVALID_ARG;
    if (!(ok_opt(A) && ok_opt(dht) && ok_opt(h0) && ok_opt(dh0))) return GDN_ERR_INVALID_ARG;
    if ((h0 == nullptr) != (dh0 == nullptr)) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!pad_to_tc(pl)) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < bwd_layout(pl).total)
            return GDN_ERR_WORKSPACE;
        return bwd_impl(pl, q, k, v, g_cum, beta, d_o, dht, h0, dq, dk, dv, dbeta, dg, dh0, workspace, st);
    }
    // a 64-wide head: pad to the 128-wide tiles, run, slice the gradients back
    const PadBwdWs w = pad_bwd_layout(pl);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.total)
        return GDN_ERR_WORKSPACE;
    const size_t tokens = (size_t)pl.B * pl.T, nst = (size_t)pl.n_seqs * pl.Hv;
    const void *qp = q, *kp = k, *vp = v, *dop = d_o;
    void *dqp = dq, *dkp = dk, *dvp = dv;
    if (pl.K < 128) {
        qp = at<void>(workspace, w.q);
        kp = at<void>(workspace, w.k);
        dqp = at<void>(workspace, w.dq);
        dkp = at<void>(workspace, w.dk);
        GDN_LAUNCH("pad", launch_pad_rows(q, const_cast<void *>(qp), tokens * pl.Hq, pl.K, st));
        GDN_LAUNCH("pad", launch_pad_rows(k, const_cast<void *>(kp), tokens * pl.Hq, pl.K, st));
    }
    if (pl.V < 128) {
        vp = at<void>(workspace, w.v);
        dop = at<void>(workspace, w.d_o);
        dvp = at<void>(workspace, w.dv);
        GDN_LAUNCH("pad", launch_pad_rows(v, const_cast<void *>(vp), tokens * pl.Hv, pl.V, st));
        GDN_LAUNCH("pad", launch_pad_rows(d_o, const_cast<void *>(dop), tokens * pl.Hv, pl.V, st));
    }
    float *h0p = h0 ? at<float>(workspace, w.h0) : nullptr;
    float *dhtp = dht ? at<float>(workspace, w.dht) : nullptr;
    float *dh0p = dh0 ? at<float>(workspace, w.dh0) : nullptr;
    if (h0) GDN_LAUNCH("pad", launch_pad_states(h0, h0p, nst, pl.K, pl.V, st));
    if (dht) GDN_LAUNCH("pad", launch_pad_states(dht, dhtp, nst, pl.K, pl.V, st));
    s = bwd_impl(padded_plan(pl), qp, kp, vp, g_cum, beta, dop, dhtp, h0p, dqp, dkp, dvp, dbeta, dg, dh0p,
                 at<void>(workspace, w.inner), st);
    if (s != GDN_OK) return s;
    if (pl.K < 128) {
        GDN_LAUNCH("slice", launch_slice_rows(dqp, dq, tokens * pl.Hq, pl.K, pl.out_f32 ? 4 : 2, st));
        GDN_LAUNCH("slice", launch_slice_rows(dkp, dk, tokens * pl.Hq, pl.K, pl.out_f32 ? 4 : 2, st));
    }
    if (pl.V < 128) GDN_LAUNCH("slice", launch_slice_rows(dvp, dv, tokens * pl.Hv, pl.V, pl.out_f32 ? 4 : 2, st));
    if (dh0) GDN_LAUNCH("slice", launch_slice_states(dh0p, dh0, nst, pl.K, pl.V, st));
    return GDN_OK;
}

}  // extern "C"

namespace {

gdn_status bwd_impl(Plan pl, const void *q, const void *k, const void *v, const float *g_cum, const float *beta,
                    const void *d_o, const float *dht, const float *h0, void *dq, void *dk, void *dv, float *dbeta,
                    float *dg, float *dh0, void *workspace, cudaStream_t st) {
    BwdWs w = bwd_layout(pl);
    pl.err = at<uint32_t>(workspace, w.err);
    pl.chunk_off = pl.cu ? at<int32_t>(workspace, w.chunk_off) : nullptr;
    GDN_TRY(cudaMemsetAsync(pl.err, 0, 256, st));
    GDN_LAUNCH("chunk_table", launch_chunk_table(pl, st));
    double *gam64 = at<double>(workspace, w.gam64);
    float *A32 = at<float>(workspace, w.A32), *P32 = at<float>(workspace, w.P32);
    float *hbuf = at<float>(workspace, w.hbuf), *dSe = at<float>(workspace, w.dSe);
    if (pl.total_chunks > 0 && tc_fwd_supported(pl)) {
        // tensor-core path: A, P (fp32 and operand images) of every chunk, then one state recompute pass
        unsigned char *tiles = at<unsigned char>(workspace, w.tiles);
        float *vecs = at<float>(workspace, w.vecs);
        GDN_LAUNCH("bwd_prep_tc", launch_tc_prep(pl, q, k, g_cum, true, beta, nullptr, nullptr, nullptr, nullptr,
                                                 tiles, vecs, st));
        if (w.n_seg > 1) {  // exact split: segment contributions and transitions, scan, then the segments
            CpSplit cs;
            cs.seg_len = w.seg_len;
            cs.n_seg = w.n_seg;
            cs.warm = 0;
            cs.serial = nullptr;
            cs.seg_states = at<float>(workspace, w.seg_states);
            cs.seg_h = at<float>(workspace, w.seg_h);
            cs.seg_M = at<float>(workspace, w.seg_M);
            cs.mode = CP_SEG;
            GDN_LAUNCH("bwd_state_seg", launch_tc_fwd(pl, q, k, v, tiles, vecs, nullptr, nullptr, nullptr, nullptr, st,
                                                      &cs));
            GDN_LAUNCH("cp_combine", launch_cp_combine(pl, h0, cs.seg_h, cs.seg_M, cs.seg_len, cs.n_seg,
                                                       cs.seg_states, st));
            cs.mode = CP_MAIN;
            GDN_LAUNCH("bwd_state_tc", launch_tc_fwd(pl, q, k, v, tiles, vecs, h0, nullptr, hbuf, nullptr, st, &cs));
            cs.mode = CP_SEG;  // the dS scan, segments counted from the sequence end
            GDN_LAUNCH("bwd_dscan_seg", launch_tc_dscan(pl, q, k, d_o, g_cum, beta, tiles, nullptr, nullptr, nullptr,
                                                        st, &cs));
            GDN_LAUNCH("cp_combine", launch_cp_combine(pl, dht, cs.seg_h, cs.seg_M, cs.seg_len, cs.n_seg,
                                                       cs.seg_states, st));
            cs.mode = CP_MAIN;
            GDN_LAUNCH("bwd_dscan_tc", launch_tc_dscan(pl, q, k, d_o, g_cum, beta, tiles, dht, dSe, dh0, st, &cs));
        } else {
            GDN_LAUNCH("bwd_state_tc", launch_tc_fwd(pl, q, k, v, tiles, vecs, h0, nullptr, hbuf, nullptr, st));
        }
    } else if (pl.total_chunks > 0) {
        GDN_LAUNCH("bwd_prep", launch_simt_prep(pl, q, k, g_cum, 1, beta, nullptr, nullptr, gam64, A32, P32, st));
        GDN_LAUNCH("bwd_state", launch_simt_scan(pl, q, k, v, beta, gam64, A32, P32, h0, nullptr, hbuf, nullptr,
                                                 st));
    }
    if (tc_fwd_supported(pl) && w.n_seg > 1) {
        // split dS scan launched above
    } else if (tc_fwd_supported(pl))
        GDN_LAUNCH("bwd_dscan_tc", launch_tc_dscan(pl, q, k, d_o, g_cum, beta, at<unsigned char>(workspace, w.tiles), dht,
                                                   dSe, dh0, st));
    else
        GDN_LAUNCH("bwd_dscan", launch_simt_dscan(pl, q, k, d_o, beta, gam64, A32, P32, dht, dSe, dh0, st));
    if (pl.total_chunks > 0 && tc_fwd_supported(pl))
        GDN_LAUNCH("bwd_intra_tc", launch_tc_bwd_intra(pl, q, k, v, d_o, at<unsigned char>(workspace, w.tiles),
                                                       at<float>(workspace, w.vecs), hbuf, dSe, dq, dk, dv, dbeta,
                                                       dg, st));
    else if (pl.total_chunks > 0)
        GDN_LAUNCH("bwd_intra", launch_simt_bwd_intra(pl, q, k, v, d_o, beta, gam64, A32, P32, hbuf, dSe, dq, dk,
                                                     dv, dbeta, dg, st));
    return GDN_OK;
}

}  // namespace

extern "C" {

size_t gdn_bwd_saved_workspace_bytes(const gdn_problem *p) {
    Plan pl;
    if (make_plan(p, &pl) != GDN_OK) return 0;
    if (tc_fwd_supported(pl)) return bwd_saved_layout(pl).total;
    if (pad_to_tc(pl) && pl.total_chunks > 0) return pad_bwd_saved_layout(pl).total;
    return gdn_bwd_workspace_bytes(p);
}

int gdn_bwd_saved_uses_saved(const gdn_problem *p) {
    Plan pl;
    if (make_plan(p, &pl) != GDN_OK) return -1;
    return (tc_fwd_supported(pl) || pad_to_tc(pl)) && pl.total_chunks > 0 ? 1 : 0;
}

gdn_status gdn_bwd_saved(const gdn_problem *p, const void *q, const void *k, const void *v, const float *g_cum,
                         const float *beta, const void *A, const void *d_o, const float *dht, const float *h0,
                         const float *h, const void *fwd_workspace, size_t fwd_workspace_bytes, void *dq, void *dk,
                         void *dv, float *dbeta, float *dg, float *dh0, void *workspace, size_t workspace_bytes,
                         gdn_stream_t stream) {
    Plan pl;
    gdn_status s = make_plan(p, &pl);
    if (s != GDN_OK) return s;
    const bool pad = pad_to_tc(pl);
    if ((!tc_fwd_supported(pl) && !pad) || pl.total_chunks == 0)  // nothing saved to reuse: recompute
        return gdn_bwd(p, q, k, v, g_cum, beta, A, d_o, dht, h0, dq, dk, dv, dbeta, dg, dh0, workspace,
                       workspace_bytes, stream);
    if (!(ok_ptr(q) && ok_ptr(k) && ok_ptr(v) && ok_ptr(g_cum) && ok_ptr(beta) && ok_ptr(d_o) && ok_ptr(dq) &&
          ok_ptr(dk) && ok_ptr(dv) && ok_ptr(dbeta) && ok_ptr(dg) && ok_ptr(h)))
        return GDN_ERR_INVALID_ARG;
    if (!(ok_opt(A) && ok_opt(dht) && ok_opt(h0) && ok_opt(dh0))) return GDN_ERR_INVALID_ARG;
    if ((h0 == nullptr) != (dh0 == nullptr)) return GDN_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void *fws = const_cast<void *>(fwd_workspace);
    const size_t fwd_need = pad ? pad_fwd_layout(pl).saved_end : fwd_layout(pl).total;
    if (!fws || (reinterpret_cast<uintptr_t>(fws) & 255u) || fwd_workspace_bytes < fwd_need)
        return GDN_ERR_WORKSPACE;
    if (!pad) {
        if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) ||
            workspace_bytes < bwd_saved_layout(pl).total)
            return GDN_ERR_WORKSPACE;
        const FwdWs fw = fwd_layout(pl);
        return bwd_saved_impl(pl, q, k, v, g_cum, beta, d_o, dht, at<unsigned char>(fws, fw.tiles),
                              at<float>(fws, fw.vecs), h, dq, dk, dv, dbeta, dg, dh0, workspace, st);
    }
    // a 64-wide head: the padded forward left its images, vectors and 128-wide chunk-entry states in its
    // workspace; pad the inputs, run, slice the gradients back
    const Plan pp = padded_plan(pl);
    const PadFwdWs pf = pad_fwd_layout(pl);
    const FwdWs fw = fwd_layout(pp);
    void *finner = at<void>(fws, pf.inner);
    const PadBwdSavedWs w = pad_bwd_saved_layout(pl);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < w.total)
        return GDN_ERR_WORKSPACE;
    const size_t tokens = (size_t)pl.B * pl.T, nst = (size_t)pl.n_seqs * pl.Hv;
    const void *qp = q, *kp = k, *vp = v, *dop = d_o;
    void *dqp = dq, *dkp = dk, *dvp = dv;
    if (pl.K < 128) {
        qp = at<void>(workspace, w.q);
        kp = at<void>(workspace, w.k);
        dqp = at<void>(workspace, w.dq);
        dkp = at<void>(workspace, w.dk);
        GDN_LAUNCH("pad", launch_pad_rows(q, const_cast<void *>(qp), tokens * pl.Hq, pl.K, st));
        GDN_LAUNCH("pad", launch_pad_rows(k, const_cast<void *>(kp), tokens * pl.Hq, pl.K, st));
    }
    if (pl.V < 128) {
        vp = at<void>(workspace, w.v);
        dop = at<void>(workspace, w.d_o);
        dvp = at<void>(workspace, w.dv);
        GDN_LAUNCH("pad", launch_pad_rows(v, const_cast<void *>(vp), tokens * pl.Hv, pl.V, st));
        GDN_LAUNCH("pad", launch_pad_rows(d_o, const_cast<void *>(dop), tokens * pl.Hv, pl.V, st));
    }
    float *dhtp = dht ? at<float>(workspace, w.dht) : nullptr;
    float *dh0p = dh0 ? at<float>(workspace, w.dh0) : nullptr;
    if (dht) GDN_LAUNCH("pad", launch_pad_states(dht, dhtp, nst, pl.K, pl.V, st));
    s = bwd_saved_impl(pp, qp, kp, vp, g_cum, beta, dop, dhtp, at<unsigned char>(finner, fw.tiles),
                       at<float>(finner, fw.vecs), at<float>(fws, pf.h), dqp, dkp, dvp, dbeta, dg, dh0p,
                       at<void>(workspace, w.inner), st);
    if (s != GDN_OK) return s;
    if (pl.K < 128) {
        GDN_LAUNCH("slice", launch_slice_rows(dqp, dq, tokens * pl.Hq, pl.K, pl.out_f32 ? 4 : 2, st));
        GDN_LAUNCH("slice", launch_slice_rows(dkp, dk, tokens * pl.Hq, pl.K, pl.out_f32 ? 4 : 2, st));
    }
    if (pl.V < 128) GDN_LAUNCH("slice", launch_slice_rows(dvp, dv, tokens * pl.Hv, pl.V, pl.out_f32 ? 4 : 2, st));
    if (dh0) GDN_LAUNCH("slice", launch_slice_states(dh0p, dh0, nst, pl.K, pl.V, st));
    return GDN_OK;
}

}  // extern "C"

namespace {

gdn_status bwd_saved_impl(Plan pl, const void *q, const void *k, const void *v, const float *g_cum,
                          const float *beta, const void *d_o, const float *dht, const unsigned char *tiles,
                          const float *vecs, const float *h, void *dq, void *dk, void *dv, float *dbeta, float *dg,
                          float *dh0, void *workspace, cudaStream_t st) {
    const BwdSavedWs w = bwd_saved_layout(pl);
    pl.err = at<uint32_t>(workspace, w.err);
    pl.chunk_off = pl.cu ? at<int32_t>(workspace, w.chunk_off) : nullptr;
    GDN_TRY(cudaMemsetAsync(pl.err, 0, 256, st));
    GDN_LAUNCH("chunk_table", launch_chunk_table(pl, st));
    float *dSe = at<float>(workspace, w.dSe);
    if (w.n_seg > 1) {  // exact split of the dS scan (segments counted from the sequence end)
        CpSplit cs;
        cs.seg_len = w.seg_len;
        cs.n_seg = w.n_seg;
        cs.warm = 0;
        cs.serial = nullptr;
        cs.seg_states = at<float>(workspace, w.seg_states);
        cs.seg_h = at<float>(workspace, w.seg_h);
        cs.seg_M = at<float>(workspace, w.seg_M);
        cs.mode = CP_SEG;
        GDN_LAUNCH("bwd_dscan_seg", launch_tc_dscan(pl, q, k, d_o, g_cum, beta, tiles, nullptr, nullptr, nullptr, st,
                                                    &cs));
        GDN_LAUNCH("cp_combine",
                   launch_cp_combine(pl, dht, cs.seg_h, cs.seg_M, cs.seg_len, cs.n_seg, cs.seg_states, st));
        cs.mode = CP_MAIN;
        GDN_LAUNCH("bwd_dscan_tc", launch_tc_dscan(pl, q, k, d_o, g_cum, beta, tiles, dht, dSe, dh0, st, &cs));
    } else {
        GDN_LAUNCH("bwd_dscan_tc", launch_tc_dscan(pl, q, k, d_o, g_cum, beta, tiles, dht, dSe, dh0, st));
    }
    GDN_LAUNCH("bwd_intra_tc", launch_tc_bwd_intra(pl, q, k, v, d_o, tiles, vecs, h, dSe, dq, dk, dv, dbeta, dg, st));
    return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_cp_plan(const gdn_problem *p, int *seg_len, int *n_seg) {
    Plan pl;
    if (make_plan(p, &pl) != GDN_OK) return -1;
    if (pad_to_tc(pl)) pl = padded_plan(pl);
    int L = 0, n = 1;
    const int on = (warmup_split(pl) || exact_split(pl)) ? 1 : 0;
    if (on) cp_geometry(pl, &L, &n);
    if (seg_len) *seg_len = on ? L : 0;
    if (n_seg) *n_seg = on ? n : 1;
    return on;
}

int gdn_cp_trigger(int64_t n_seqs, int64_t n_heads, int64_t seq_len) {
    Plan pl;
    std::memset(&pl, 0, sizeof(pl));
    pl.n_seqs = (int)n_seqs;
    pl.Hv = (int)n_heads;
    pl.max_seq_len = (int)seq_len;
    return cp_trigger(pl) ? 1 : 0;
}

gdn_status gdn_workspace_error(const void *workspace, gdn_stream_t stream) {
    if (!workspace) return GDN_ERR_INVALID_ARG;
    uint32_t word = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    return word == ERR_NONE ? GDN_OK : GDN_ERR_TIMEOUT;
}

const char *gdn_status_str(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported problem";
        case GDN_ERR_WORKSPACE: return "workspace too small or misaligned";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_TIMEOUT: return "device-side wait timed out";
        case GDN_ERR_TOO_LARGE: return "problem exceeds the fixed no-alloc scratch";
    }
    return "unknown status";
}

const char *gdn_version(void) { return "gdn-gb300 0.2 sm_103a"; }

void gdn_debug_set_wait(int64_t wait_ns, int32_t drop_load_chunk) {
    g_dbg_wait_ns.store(wait_ns > 0 ? (long long)wait_ns : 0);
    g_dbg_drop_chunk.store(drop_load_chunk >= 0 ? drop_load_chunk : -1);
}

}  // extern "C"
