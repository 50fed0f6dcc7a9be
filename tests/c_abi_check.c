/* A plain C99 client of the library: compiled against include/ea.h and linked
 * against libea.so by tests/test_c_abi.py.  Exercises only entry points that
 * do not need a GPU: status strings, workspace sizes, host-side argument
 * checks (rejected calls enqueue nothing) and the sparsity ratios. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "ea.h"

static int failures = 0;

#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            ++failures;                                                    \
        }                                                                  \
    } while (0)

int main(void)
{
    int code;
    for (code = 0; code <= 6; ++code) {
        const char *s = ea_status_string((ea_status)code);
        CHECK(s != NULL && strlen(s) > 0);
    }
    CHECK(strcmp(ea_status_string(EA_OK), "ok") == 0);

    /* workspace sizes: d must be 128, Hq a multiple of Hkv */
    CHECK(ea_prefill_workspace_size(1, 4096, 32, 8, 128) > 256);
    CHECK(ea_prefill_workspace_size(1, 4096, 32, 8, 64) == 0);
    CHECK(ea_prefill_workspace_size(1, 4096, 30, 8, 128) == 0);
    CHECK(ea_decode_workspace_size(4, 32, 8, 128, 4096, 0) > 256);
    CHECK(ea_prefill_host_buffer_size(1, 4096, 32, 8, 128, 0) >
          ea_prefill_workspace_size(1, 4096, 32, 8, 128));

    /* host-side rejection: a NULL Q, a misaligned workspace */
    {
        const int64_t qs[4] = {4096 * 32 * 128, 32 * 128, 128, 1};
        const int64_t ks[4] = {4096 * 8 * 128, 8 * 128, 128, 1};
        void *fake = (void *)0x100000;
        CHECK(ea_hybrid_attn_prefill(NULL, fake, fake, fake, NULL, qs, ks, qs, 1, 4096, 32, 8, 128,
                                     0.088f, (const uint8_t *)fake, 64, 256, NULL, 128, fake,
                                     1 << 20, NULL, NULL) == EA_ERR_INVALID_ARG);
        CHECK(ea_hybrid_attn_prefill(fake, fake, fake, fake, NULL, qs, ks, qs, 1, 4096, 32, 8, 128,
                                     0.088f, (const uint8_t *)fake, 64, 256, NULL, 128,
                                     (void *)0x100010, 1 << 20, NULL, NULL) == EA_ERR_WORKSPACE);
        CHECK(ea_check_errors(NULL, NULL) == EA_ERR_WORKSPACE);
    }

    /* sparsity ratios of one layer, S = 256, 2 KV heads: head 0 FA (r = 0),
     * head 1 SSA sink 0 window 128 (r = 1).  Causal pairs 256 * 257 / 2 =
     * 32896; the SSA head keeps sum_i min(i + 1, 128) = 128 * 129 / 2 + 128 *
     * 128 = 24640, so it prunes 8256: Omega_ESR = 8256 / (2 * 32896). */
    {
        const uint8_t r[2] = {0, 1}, m[2] = {EA_FULL, EA_SSA};
        double msr = -1.0, esr = -1.0;
        CHECK(ea_sparsity_ratios(r, m, 1, 2, 256, 0, 128, NULL, 128, &msr, &esr) == EA_OK);
        CHECK(msr == 0.5);
        CHECK(esr == 8256.0 / (2.0 * 32896.0));
        CHECK(ea_sparsity_ratios(r, m, 1, 2, 256, 0, 0, NULL, 128, &msr, &esr) ==
              EA_ERR_INVALID_ARG);
    }

    if (failures == 0)
        printf("c abi: all checks passed\n");
    return failures == 0 ? 0 : 1;
}
