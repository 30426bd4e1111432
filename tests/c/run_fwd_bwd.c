/* A plain C99 caller of the library's compute entry points: allocates device
 * buffers with the CUDA runtime, copies raw input files in, runs gdn_fwd and
 * gdn_bwd on a batch-mode problem through include/gdn.h and writes the outputs
 * back as raw files.  tests/test_c_compute.py writes the inputs, compiles this
 * program, runs it and checks the outputs against the fp64 oracle.
 *
 * usage: run_fwd_bwd DIR B T Hq Hv K V
 *   DIR/{q,k,v,g,beta,h0,do,dht,g_cum}.bin in (q, k, v, do bf16; the rest fp32;
 *   g_cum is the backward's gate argument, computed by the caller)
 *   DIR/{o,ht,dq,dk,dv,dbeta,dg,dh0}.bin out
 * Exit status 0 on success; any CUDA or library error prints and exits 1. */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "gdn.h"

static const char *dir;

static void fail(const char *what, const char *detail) {
    fprintf(stderr, "run_fwd_bwd: %s: %s\n", what, detail);
    exit(1);
}

static void check_cuda(cudaError_t e, const char *what) {
    if (e != cudaSuccess) fail(what, cudaGetErrorString(e));
}

static void check_gdn(gdn_status s, const char *what) {
    if (s != GDN_OK) fail(what, gdn_status_str(s));
}

/* Device buffer of `bytes` filled from DIR/name.bin (which must hold exactly that many bytes). */
static void *load(const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s.bin", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) fail("open", path);
    void *host = malloc(bytes ? bytes : 1);
    if (!host) fail("malloc", name);
    if (fread(host, 1, bytes, f) != bytes) fail("short read", path);
    fclose(f);
    void *dev = NULL;
    check_cuda(cudaMalloc(&dev, bytes ? bytes : 16), "cudaMalloc");
    check_cuda(cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice), "copy in");
    free(host);
    return dev;
}

static void *alloc(size_t bytes) {
    void *dev = NULL;
    check_cuda(cudaMalloc(&dev, bytes ? bytes : 16), "cudaMalloc");
    return dev;
}

static void store(const char *name, const void *dev, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s.bin", dir, name);
    void *host = malloc(bytes ? bytes : 1);
    if (!host) fail("malloc", name);
    check_cuda(cudaMemcpy(host, dev, bytes, cudaMemcpyDeviceToHost), "copy out");
    FILE *f = fopen(path, "wb");
    if (!f) fail("open", path);
    if (fwrite(host, 1, bytes, f) != bytes) fail("short write", path);
    fclose(f);
    free(host);
}

int main(int argc, char **argv) {
    if (argc != 8) fail("usage", "run_fwd_bwd DIR B T Hq Hv K V");
    dir = argv[1];
    gdn_problem p;
    memset(&p, 0, sizeof p);
    p.B = atoll(argv[2]);
    p.T = atoll(argv[3]);
    p.Hq = atoll(argv[4]);
    p.Hv = atoll(argv[5]);
    p.K = atoll(argv[6]);
    p.V = atoll(argv[7]);
    p.n_seqs = p.B;
    p.io_dtype = GDN_BF16;
    p.scale = (float)(1.0 / sqrt((double)p.K));
    p.cp_mode = GDN_CP_AUTO;
    p.warmup_chunks = 8;
    p.out_f32 = 0;

    const size_t tok = (size_t)(p.B * p.T);
    const size_t qk = tok * (size_t)(p.Hq * p.K) * 2, vv = tok * (size_t)(p.Hv * p.V) * 2;
    const size_t gate = tok * (size_t)p.Hv * 4, st = (size_t)(p.n_seqs * p.Hv * p.K * p.V) * 4;
    void *q = load("q", qk), *k = load("k", qk), *v = load("v", vv), *d_o = load("do", vv);
    float *g = (float *)load("g", gate), *beta = (float *)load("beta", gate);
    float *g_cum_host = (float *)load("g_cum", gate);
    float *h0 = (float *)load("h0", st), *dht = (float *)load("dht", st);

    cudaStream_t stream;
    check_cuda(cudaStreamCreate(&stream), "cudaStreamCreate");
    /* forward: o and the final state (g_cum, A, h not requested) */
    void *o = alloc(vv);
    float *ht = (float *)alloc(st);
    size_t ws_f = gdn_fwd_workspace_bytes(&p);
    if (ws_f == 0) fail("gdn_fwd_workspace_bytes", "invalid problem");
    void *wsf = alloc(ws_f);
    check_gdn(gdn_fwd(&p, q, k, v, g, beta, h0, o, NULL, NULL, NULL, ht, wsf, ws_f, (gdn_stream_t)stream),
              "gdn_fwd");
    /* backward, from the caller's g_cum */
    void *dq = alloc(qk), *dk = alloc(qk), *dv = alloc(vv);
    float *dbeta = (float *)alloc(gate), *dg = (float *)alloc(gate), *dh0 = (float *)alloc(st);
    size_t ws_b = gdn_bwd_workspace_bytes(&p);
    if (ws_b == 0) fail("gdn_bwd_workspace_bytes", "invalid problem");
    void *wsb = alloc(ws_b);
    check_gdn(gdn_bwd(&p, q, k, v, g_cum_host, beta, NULL, d_o, dht, h0, dq, dk, dv, dbeta, dg, dh0, wsb, ws_b,
                      (gdn_stream_t)stream),
              "gdn_bwd");
    check_cuda(cudaStreamSynchronize(stream), "cudaStreamSynchronize");
    check_gdn(gdn_workspace_error(wsf, (gdn_stream_t)stream), "forward device error word");
    check_gdn(gdn_workspace_error(wsb, (gdn_stream_t)stream), "backward device error word");

    store("o", o, vv);
    store("ht", ht, st);
    store("dq", dq, qk);
    store("dk", dk, qk);
    store("dv", dv, vv);
    store("dbeta", dbeta, gate);
    store("dg", dg, gate);
    store("dh0", dh0, st);

    void *bufs[] = {q, k, v, d_o, g, beta, g_cum_host, h0, dht, o, ht, wsf, dq, dk, dv, dbeta, dg, dh0, wsb};
    for (size_t i = 0; i < sizeof bufs / sizeof bufs[0]; ++i) check_cuda(cudaFree(bufs[i]), "cudaFree");
    check_cuda(cudaStreamDestroy(stream), "cudaStreamDestroy");
    printf("ok\n");
    return 0;
}
