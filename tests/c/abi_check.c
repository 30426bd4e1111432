/* Pure C99 use of the library's C ABI: includes gdn.h, links libgdn.so and calls
 * the host-only entry points (no device needed).  Prints one "name value" line
 * per answer; tests/test_c_abi.py compares them with the Python binding's. */
#include <stdio.h>
#include <string.h>

#include "gdn.h"

static gdn_problem problem(int64_t K, int64_t V, int32_t cp_mode) {
    gdn_problem p;
    memset(&p, 0, sizeof p);
    p.B = 2; p.T = 8192; p.Hq = 16; p.Hv = 64; p.K = K; p.V = V; p.n_seqs = 2;
    p.cu_seqlens = NULL; p.cu_seqlens_host = NULL;
    p.io_dtype = GDN_BF16; p.scale = 0.08838834764831845f; p.cp_mode = cp_mode; p.warmup_chunks = 8;
    return p;
}

int main(void) {
    gdn_problem p = problem(128, 128, GDN_CP_AUTO);
    gdn_problem p64 = problem(64, 64, GDN_CP_AUTO);
    gdn_problem bad = problem(96, 128, GDN_CP_AUTO);
    printf("version %s\n", gdn_version());
    printf("fwd_ws %zu\n", gdn_fwd_workspace_bytes(&p));
    printf("bwd_ws %zu\n", gdn_bwd_workspace_bytes(&p));
    printf("bwd_saved_ws %zu\n", gdn_bwd_saved_workspace_bytes(&p));
    printf("fwd_ws_64 %zu\n", gdn_fwd_workspace_bytes(&p64));
    printf("bad_ws %zu\n", gdn_fwd_workspace_bytes(&bad));
    printf("uses_saved %d\n", gdn_bwd_saved_uses_saved(&p));
    printf("trigger_8 %d\n", gdn_cp_trigger(1, 8, 32768));
    printf("trigger_128 %d\n", gdn_cp_trigger(2, 64, 8192));
    gdn_problem ls = problem(128, 128, GDN_CP_AUTO);
    ls.B = 1; ls.T = 32768; ls.Hq = 4; ls.Hv = 8; ls.n_seqs = 1;
    int L = 0, n = 0;
    int on = gdn_cp_plan(&ls, &L, &n);
    printf("plan %d %d %d\n", on, L, n);
    printf("status_ok %s\n", gdn_status_str(GDN_OK));
    return 0;
}
