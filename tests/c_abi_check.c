/* The C ABI of liblact as a plain C11 program sees it: the header compiles as
 * C, the library links, and the host-only calls answer without a GPU
 * (workspace sizing and argument validation run before any device work). */
#include <stdio.h>
#include <string.h>
#include "lact.h"

int main(void) {
    lact_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.B = 1; cfg.H = 8; cfg.d = 128; cfg.dh = 512;
    cfg.io_dtype = LACT_BF16; cfg.opt = LACT_OPT_MUON; cfg.ns_steps = 5;
    cfg.ns_a = 3.4445; cfg.ns_b = -4.7750; cfg.ns_c = 2.0315; cfg.muon_lr = 0.02;
    cfg.max_chunk = 1 << 20; cfg.momentum = 0.9; cfg.memory = LACT_MEM_SWIGLU;
    size_t ws = lact_workspace_bytes(&cfg);
    if (ws == 0) { fprintf(stderr, "valid config rejected\n"); return 1; }
    lact_config bad = cfg;
    bad.dh = 100;                                   /* not a multiple of 64 */
    if (lact_workspace_bytes(&bad) != 0) { fprintf(stderr, "invalid config accepted\n"); return 2; }
    lact_state* st = NULL;
    /* a null workspace is an argument error, returned before any device call */
    if (lact_init_state(&st, &cfg, NULL, ws, NULL, NULL, NULL, 0) != LACT_ERR_INVALID_ARG) return 3;
    if (lact_sync_status(NULL) != LACT_ERR_INVALID_ARG) return 4;
    if (strlen(lact_status_str(LACT_ERR_TIMEOUT)) == 0) return 5;
    printf("workspace_bytes %zu\n", ws);
    return 0;
}
