/*
 * gdn.h -- C ABI of the GB300 (sm_103a) gated delta rule chunked-prefill library.
 *
 * The operator (Gated DeltaNet, per value head, state S in R^{K x V}):
 *
 *     S_t = exp(g_t) S_{t-1} + k_t (beta_t (v_t - exp(g_t) S_{t-1}^T k_t))^T
 *     o_t = scale * S_t^T q_t
 *
 * computed chunk-parallel with chunk size GDN_CHUNK = 64.  The entry points
 * mirror the two-level API of the flash_qla 0.1.2 README (PyPI METADATA page,
 * sections "Usage / High-level API" and "Usage / Low-level API"):
 *
 *     chunk_gated_delta_rule_fwd(q, k, v, g, beta, scale, initial_state, cu_seqlens)
 *         -> (g, A, o, h, final_state)                          == gdn_fwd
 *     chunk_gated_delta_rule_bwd(q, k, v, g, beta, A, do, dht, scale, initial_state, cu_seqlens)
 *         -> (dq, dk, dv, db, dg, dh0)                          == gdn_bwd
 *
 * General conventions (every entry point):
 *  - All tensor pointers are caller-owned DEVICE memory, row-major and
 *    contiguous, 16-byte aligned.  The library never allocates device memory,
 *    never synchronises the device or the stream, and enqueues all work on
 *    the caller's `stream`.  It keeps no state between calls: concurrent calls
 *    on different streams with different workspaces are safe.
 *  - Arguments are validated on the host before anything is enqueued; a bad
 *    argument returns a status and enqueues nothing.  A failed launch returns
 *    GDN_ERR_CUDA.  Kernels that wait on an mbarrier give up after a bounded
 *    number of polls and record GDN_ERR_TIMEOUT in the workspace's error word;
 *    gdn_workspace_error() reads it back.
 *  - Shapes (B = batch, T = tokens per sequence, Hq = query/key heads,
 *    Hv = value heads, N = number of sequences):
 *        q, k            [B, T, Hq, K]   io dtype
 *        v, o, do, dv    [B, T, Hv, V]   io dtype
 *        dq, dk          [B, T, Hq, K]   io dtype
 *        g, g_cum, dg    [B, T, Hv]      fp32
 *        beta, dbeta     [B, T, Hv]      fp32
 *        A               [B, T, Hv, 64]  io dtype (row r of a chunk's 64x64
 *                                        matrix stored at that chunk's token r)
 *        h               [B, NC, Hv, K, V] fp32 (NC = chunks per sequence;
 *                                        varlen: [total chunks, Hv, K, V])
 *        h0, ht, dht, dh0 [N, Hv, K, V]  fp32
 *  - Grouped value heads: Hv % Hq == 0 and value head hv reads q/k head
 *    hv / (Hv / Hq).
 *  - Varlen: cu_seqlens != NULL requires B == 1; sequence s covers tokens
 *    [cu_seqlens[s], cu_seqlens[s+1]) and has its own h0 / ht; chunks never
 *    cross a sequence boundary.
 *  - Execution paths: bf16 io with K = V = 128 runs the tensor-core kernels.
 *    bf16 io with K or V = 64 runs the same kernels on zero-padded 128-wide
 *    copies that the library makes in its workspace (exact: the padded state
 *    rows and columns stay zero) and slices the outputs back.  fp32 io runs
 *    the CUDA-core kernels.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_CHUNK 64

typedef struct CUstream_st *gdn_stream_t; /* == cudaStream_t; NULL = legacy default stream */

typedef enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad shape, bad enum       */
    GDN_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. K or V not 64 / 128) */
    GDN_ERR_WORKSPACE = 3,   /* workspace too small or misaligned                    */
    GDN_ERR_CUDA = 4,        /* a CUDA launch or async call failed                   */
    GDN_ERR_TIMEOUT = 5,     /* a device-side bounded wait expired (see header)      */
    GDN_ERR_TOO_LARGE = 6    /* gdn_fwd_noalloc: problem exceeds its fixed scratch     */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef enum {
    GDN_CP_AUTO = 0,   /* exact; when the pages' trigger fires, sequences are
                          split and joined through segment transitions (gdn_fwd) */
    GDN_CP_OFF = 1,    /* one serial scan per (sequence, value head)             */
    GDN_CP_WARMUP = 2  /* approximate: segments start from a warmup state, see
                          gdn_fwd; used only when the page's trigger rule fires   */
} gdn_cp_mode;

typedef struct {
    int64_t B, T, Hq, Hv, K, V;      /* K, V in {64, 128}; Hv % Hq == 0              */
    int64_t n_seqs;                  /* = B, or number of sequences when varlen      */
    const int32_t *cu_seqlens;       /* device [n_seqs + 1] or NULL                  */
    const int32_t *cu_seqlens_host;  /* host copy of the same offsets; required iff
                                        cu_seqlens != NULL (used for launch planning) */
    gdn_dtype io_dtype;              /* dtype of q, k, v, o, A, do, dq, dk, dv       */
    float scale;                     /* output scale; K^-0.5 is the usual choice     */
    int32_t cp_mode;                 /* gdn_cp_mode                                  */
    int32_t warmup_chunks;           /* GDN_CP_WARMUP only: chunks of warmup (6..8)  */
    int32_t out_f32;                 /* checking mode, 0 or 1; see below              */
} gdn_problem;

/*
 * out_f32 = 1 with io_dtype GDN_BF16: the same kernels, in the same order,
 * write o and A (gdn_fwd) and dq, dk, dv (gdn_bwd, gdn_bwd_saved) as fp32
 * instead of rounding them to bf16; those buffers are then fp32 tensors of
 * the shapes above.  It exposes the value each kernel holds before its final
 * rounding, so that a test can hold it to an error bound tighter than one
 * bf16 rounding.  Ignored for GDN_F32 (every output is fp32 already).  The
 * forward's saved state for gdn_bwd_saved does not depend on it.
 */

/* Bytes of device workspace gdn_fwd / gdn_bwd need for this problem (0 on a
 * bad problem).  The workspace must be 256-byte aligned. */
size_t gdn_fwd_workspace_bytes(const gdn_problem *p);
size_t gdn_bwd_workspace_bytes(const gdn_problem *p);

/*
 * Forward (the README's chunk_gated_delta_rule_fwd; the high-level
 * chunk_gated_delta_rule returns (o, final_state) of this call).
 *   in : q, k, v (io dtype), g (raw log-decay, fp32, <= 0 expected), beta
 *        (fp32), h0 (nullable: zero initial state).
 *   out: o; g_cum = chunk-local inclusive cumsum of g (the README's returned
 *        `g`); A = (I + L)^{-1} per chunk, L = strict_lower(diag(beta)
 *        (D o K K^T)), D_ri = exp(g_cum_r - g_cum_i) (nullable: not written);
 *        h = state entering every chunk (nullable); final_state (nullable).
 * GDN_CP_WARMUP (the pages' sliding-window warmup, FlashQLA news page,
 * "Technical Principles"): when the trigger fires, each segment after the
 * first starts from the state obtained by running warmup_chunks chunks from a
 * zero state; the result is then approximate: the state error at a segment
 * start is at most exp(sum of g over its warmup window) * |S|_F, S the exact
 * state at the window start.  A value head whose gate sum over some warmup
 * window is above ln(1e-4) runs unsplit (exact) in that sequence.  g_cum, A
 * and h are as in the exact path; final_state comes from the last segment.
 * GDN_CP_AUTO with the trigger on (the pages' AutoCP, news page "FlashQLA's
 * core advantages"; here without approximation): the same segments; each is
 * run from a zero state and, with v = 0, from the identity, which gives its
 * contribution h_p and transition M_p (the recurrence is linear in v and S);
 * the segment starting states S_(p+1) = M_p S_p + h_p are scanned in fp32 and
 * every segment is then run from its own.  The result equals the unsplit one
 * up to rounding.
 */
gdn_status gdn_fwd(const gdn_problem *p,
                   const void *q, const void *k, const void *v,
                   const float *g, const float *beta, const float *h0,
                   void *o, float *g_cum, void *A, float *h, float *final_state,
                   void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * Backward (the README's chunk_gated_delta_rule_bwd).
 *   in : q, k, v, g_cum (the forward's returned g), beta, A (the forward's A;
 *        nullable -- the backward recomputes the inverse in fp32 from k, beta
 *        and g_cum because the stored copy is rounded to the io dtype),
 *        d_o = dL/do, dht = dL/dfinal_state (nullable: zero), h0 (nullable).
 *   out: dq, dk, dv (io dtype), dbeta, dg (fp32; dg is the gradient with
 *        respect to the RAW g given to the forward), dh0 (required iff h0 !=
 *        NULL; must be NULL otherwise).
 */
gdn_status gdn_bwd(const gdn_problem *p,
                   const void *q, const void *k, const void *v,
                   const float *g_cum, const float *beta, const void *A,
                   const void *d_o, const float *dht, const float *h0,
                   void *dq, void *dk, void *dv, float *dbeta, float *dg, float *dh0,
                   void *workspace, size_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_fwd_noalloc -- gdn_fwd for callers that cannot allocate device memory
 * (no counterpart in the FlashQLA pages; this is a deployment convenience).
 * Hosts such as inference runtimes or plugin frameworks that own every device
 * allocation, code replaying a captured CUDA graph with a frozen memory pool,
 * or plain C callers without an allocator cannot provide gdn_fwd's
 * workspace.  This call takes the workspace from a file-scope __device__
 * array of GDN_NOALLOC_SCRATCH_BYTES bytes instead; it calls no cudaMalloc,
 * cudaFree or other allocating routine.  Inputs and outputs are the caller's,
 * exactly as for gdn_fwd.
 *   - Problems with gdn_fwd_workspace_bytes(p) > GDN_NOALLOC_SCRATCH_BYTES
 *     return GDN_ERR_TOO_LARGE and enqueue nothing.
 *   - Every GPU that loads the library holds the array until process exit.
 *   - All calls share the array; it keeps the last call's contents (each call
 *     rewrites what it reads and clears its error word), so calls whose GPU
 *     work overlaps -- on different streams or host threads -- race on it and
 *     must be serialised by the caller.
 *   - The array's address belongs to the CUDA context current at the call.
 *     Outside stream capture each call looks it up afresh, so a device reset
 *     or a caller-made driver context is served with its own address.  During
 *     capture the address cached for the current context by an earlier call
 *     is used: make one call in each context before any stream capture (a
 *     capture in a context never seen before returns GDN_ERR_CUDA).
 *   - What fits: the tensor-core forward needs about 33 KB per (chunk, value
 *     head), so about 1000 chunk x value-head units fit (e.g. B = 1, T = 8192,
 *     Hv = 8: 1024 units, just over; T = 4096, Hv = 8: 512 units plus the
 *     sequence split's segment states, about 30 MB, fits).
 *     gdn_fwd_workspace_bytes(p) is the exact test.
 *   - Invalid or unsupported problems return gdn_fwd's own status.
 */
#define GDN_NOALLOC_SCRATCH_BYTES (32u << 20)
gdn_status gdn_fwd_noalloc(const gdn_problem *p,
                           const void *q, const void *k, const void *v,
                           const float *g, const float *beta, const float *h0,
                           void *o, float *g_cum, void *A, float *h, float *final_state,
                           gdn_stream_t stream);
/* The error word gdn_fwd_noalloc's last call left in the shared array of the
 * current context (synchronises `stream`): GDN_OK, or GDN_ERR_TIMEOUT when a
 * device-side bounded wait of that call expired; GDN_ERR_CUDA if the array
 * cannot be reached. */
gdn_status gdn_fwd_noalloc_error(gdn_stream_t stream);

/*
 * Backward that reuses what the forward saved instead of recomputing it (the
 * save-for-backward form of gdn_bwd; no counterpart in the pages, whose
 * backward recomputes).  The forward must have run on the same problem and
 * inputs with its h output requested; `h` is that output and `fwd_workspace`
 * that call's workspace, both unchanged since.  The backward then skips its
 * A / P preparation and its state recompute (it reads the forward's operand
 * images, gate vectors and chunk-entry states) and runs only the state-
 * gradient scan and the per-chunk gradients.  Results equal gdn_bwd's up to
 * rounding, provided the forward's states were exact (cp_mode AUTO or OFF; a
 * warm-up split forward saves its approximate states, and the gradients then
 * follow those).  Arguments otherwise as gdn_bwd; the workspace must hold
 * gdn_bwd_saved_workspace_bytes(p) bytes.  For 64-wide heads the padded
 * forward's workspace holds the 128-wide states this reads (h must still be
 * passed: it marks that the forward ran with h requested).  fp32 problems
 * run gdn_bwd (h and fwd_workspace unused;
 * the workspace must then hold gdn_bwd_workspace_bytes(p), which this query
 * returns for them).
 */
size_t gdn_bwd_saved_workspace_bytes(const gdn_problem *p);
/* 1 if gdn_bwd_saved reads the forward's h and workspace for this problem
 * (bf16 io with at least one chunk), 0 if it runs gdn_bwd instead (the forward
 * then need not produce h), -1 for an invalid problem. */
int gdn_bwd_saved_uses_saved(const gdn_problem *p);
gdn_status gdn_bwd_saved(const gdn_problem *p,
                         const void *q, const void *k, const void *v,
                         const float *g_cum, const float *beta, const void *A,
                         const void *d_o, const float *dht, const float *h0,
                         const float *h, const void *fwd_workspace,
                         size_t fwd_workspace_bytes,
                         void *dq, void *dk, void *dv, float *dbeta, float *dg,
                         float *dh0, void *workspace, size_t workspace_bytes,
                         gdn_stream_t stream);

/*
 * Sequence splitting with warmup (the "AutoCP" of the FlashQLA pages: news
 * page, "FlashQLA's core advantages"; blog post, section 1).
 * gdn_cp_trigger: 1 iff the pages' rule turns splitting on for n_seqs
 *   sequences of up to seq_len tokens and n_heads value heads
 *   (n_seqs * n_heads <= 40, or <= 56 with seq_len >= 8192).
 * gdn_cp_plan: 1 iff gdn_fwd would split this problem (cp_mode GDN_CP_AUTO
 *   or GDN_CP_WARMUP, bf16 with K = V = 128, trigger on, more than one segment);
 *   then *seg_len = L = round(sqrt(N)) chunks for N chunks of the longest
 *   sequence and *n_seg = ceil(N / L).  Returns 0 otherwise, -1 on a bad problem.
 */
int gdn_cp_trigger(int64_t n_seqs, int64_t n_heads, int64_t seq_len);
int gdn_cp_plan(const gdn_problem *p, int *seg_len, int *n_seg);

/* Reads the device error word a previous gdn_fwd / gdn_bwd left in
 * `workspace` (synchronises `stream`).  Returns GDN_OK or GDN_ERR_TIMEOUT. */
gdn_status gdn_workspace_error(const void *workspace, gdn_stream_t stream);

/* Static description of a status code. */
const char *gdn_status_str(gdn_status s);

/*
 * Kernel timing (tracing; process-wide, off by default, not for concurrent
 * use from several host threads).  While enabled, every kernel the library
 * launches is bracketed by a pair of CUDA events recorded on the caller's
 * stream.  gdn_profile_read() waits for the recorded events, writes up to
 * max_entries rows (kernel name into names + i * name_stride, at most
 * name_stride - 1 characters; launch count; summed device milliseconds) and
 * clears the record.  Returns the number of rows, or -1 on a CUDA error.
 * Events are host-side objects; no device memory is allocated.
 */
void gdn_profile_enable(int on);
int gdn_profile_read(char *names, int name_stride, int *counts, double *ms, int max_entries);

/* Library version string, e.g. "gdn-gb300 0.2 sm_103a". */
const char *gdn_version(void);

/*
 * Test aid for the bounded device-side waits (process-wide; set it only while
 * no other thread calls the library).  Problems planned after this call use
 * wait_ns as the limit of every mbarrier wait of the forward's state-chain
 * kernel (wait_ns <= 0 restores the default of one second) and, when
 * drop_load_chunk >= 0, that kernel's producer skips the k / q / operand-image
 * load of the chunk with this index in every chain.  The consumer's wait on
 * that load then expires: the kernel records GDN_ERR_TIMEOUT in the workspace
 * error word (read by gdn_workspace_error), waits for its own copies and
 * tensor-core operations in flight, frees its tensor memory and returns, and
 * the outputs of that call are incomplete.  Later calls on the same stream
 * run normally.  gdn_debug_set_wait(0, -1) restores the defaults.
 */
void gdn_debug_set_wait(int64_t wait_ns, int32_t drop_load_chunk);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
