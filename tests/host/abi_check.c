/* A plain C11 consumer of the library's C ABI: compiled with gcc against
 * include/arfuse.h alone and linked to libarfuse.so, it drives a dry-run
 * workspace (no GPU needed) through create, validation of a call, the
 * regime-table round trip, the status strings and destroy.  Prints "c abi ok"
 * and exits 0 when every answer is the documented one. */
#include <stdint.h>
#include <stdio.h>

#include "arfuse.h"

static int fails = 0;

static void expect(int cond, const char* what) {
    if (!cond) {
        printf("FAILED: %s\n", what);
        ++fails;
    }
}

/* Distinct, 16-byte aligned fake device addresses: a dry-run workspace only
 * validates them (alignment, no overlap), it never dereferences them. */
static void* fake(int i) { return (void*)(((uintptr_t)1 << 44) + (uintptr_t)i * ((uintptr_t)1 << 28)); }

int main(void) {
    enum { R = 8, K = 8, H = 7168 };
    const int64_t T = 4;
    ar_workspace* ws = NULL;
    ar_status st = ar_workspace_create(0, R, K, H, 64, 1e-6f, AR_WS_DRY_RUN, &ws);
    expect(st == AR_OK && ws != NULL, "create a dry-run workspace");
    if (!ws) return 1;

    const void* E[R];
    const void* S[R];
    for (int r = 0; r < R; ++r) {
        E[r] = fake(r);
        S[r] = fake(R + r);
    }
    const int32_t* perm = (const int32_t*)fake(2 * R);
    const float* w = (const float*)fake(2 * R + 1);
    const void* residual = fake(2 * R + 2);
    const void* gamma = fake(2 * R + 3);
    void* out = fake(2 * R + 4);
    void* residual_out = fake(2 * R + 5);

    st = ar_finalize_rmsnorm(ws, E, T * K, perm, w, S, residual, gamma, 0.0f, 1e-6f, T, R, K, H, out,
                             residual_out, 0, NULL);
    expect(st == AR_VALIDATED, "a valid call validates");
    int ctas = 0;
    const int regime = ar_workspace_last_regime(ws, &ctas);
    expect(regime == AR_REGIME_SPLIT && ctas == 16, "the built-in table's plan for T = 4");
    expect(ar_workspace_last_grid(ws) == (int)(T * 16), "its grid");
    ar_plan_info info;
    expect(ar_workspace_last_plan(ws, &info) == AR_OK && info.regime == AR_REGIME_SPLIT &&
               info.grid == (int)(T * 16) && info.column_groups == 4 && info.copy_rounds == 1,
           "its plan");
    expect(ar_workspace_last_plan(ws, NULL) == AR_ERR_INVALID_ARG, "plan into NULL");

    st = ar_finalize_rmsnorm(ws, E, T * K, perm, w, S, NULL, gamma, 0.0f, 1e-6f, T, R, K, H, out,
                             residual_out, 0, NULL);
    expect(st == AR_ERR_INVALID_ARG, "a missing residual is rejected");
    st = ar_finalize_rmsnorm(ws, E, T * K, perm, w, S, (const char*)residual + 8, gamma, 0.0f, 1e-6f, T, R,
                             K, H, out, residual_out, 0, NULL);
    expect(st == AR_ERR_ALIGNMENT, "a misaligned pointer is rejected");
    st = ar_finalize_rmsnorm(ws, E, 65 * K, perm, w, S, residual, gamma, 0.0f, 1e-6f, 65, R, K, H, out,
                             residual_out, 0, NULL);
    expect(st == AR_ERR_CAPACITY, "T above max_tokens is rejected");

    const ar_regime_rule rules[2] = {{16, AR_REGIME_SPLIT, 16, 0, 0}, {64, AR_REGIME_CLUSTER, 8, 24576, 2}};
    expect(ar_workspace_set_regime_table(ws, rules, 2) == AR_OK, "set a regime table");
    int n = -1;
    expect(ar_workspace_get_regime_table(ws, NULL, 0, &n) == AR_OK && n == 2, "its length");
    ar_regime_rule back[2];
    expect(ar_workspace_get_regime_table(ws, back, 2, &n) == AR_OK && back[1].max_tokens == 64 &&
               back[1].ctas_per_row == 8 && back[1].stage_bytes == 24576 && back[1].producer_warps == 2,
           "the table reads back");
    st = ar_finalize_rmsnorm(ws, E, 32 * K, perm, w, S, residual, gamma, 0.0f, 1e-6f, 32, R, K, H, out,
                             residual_out, 0, NULL);
    expect(st == AR_VALIDATED && ar_workspace_last_regime(ws, &ctas) == AR_REGIME_CLUSTER && ctas == 8,
           "a call follows the table");

    expect(ar_status_string(AR_OK) != NULL && ar_status_string((ar_status)99) != NULL, "status strings");
    expect(ar_workspace_destroy(ws) == AR_OK, "destroy");
    expect(ar_workspace_destroy(NULL) == AR_OK, "destroy NULL");

    if (fails) return 1;
    puts("c abi ok");
    return 0;
}
