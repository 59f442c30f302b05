/* c_abi_check.c -- a C99 caller of libssmscan, built against
 * include/ssmscan.h alone.  It makes only the calls that answer on the host
 * (the ABI version, status strings and argument validation, which return
 * before any CUDA call), so it runs on a machine without a GPU.  Exits 0 when
 * every answer is the one the header documents. */
#include <stdio.h>
#include <string.h>

#include "ssmscan.h"

/* a 64 KiB-aligned address that validation never dereferences */
#define FAKE ((void *)0x10000)
#define FAKEF ((float *)0x10000)

static int fails = 0;

static void expect(int got, int want, const char *what) {
    if (got != want) {
        printf("FAIL %s: got %d, want %d\n", what, got, want);
        ++fails;
    }
}

static int scan(const void *u, int64_t batch, int64_t N, int dtype) {
    return ssm_scan_fwd(u, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE, NULL, batch, 4, 8, N,
                        dtype, NULL);
}

int main(void) {
    int s;
    expect(ssm_abi_version(), 1, "abi version");
    for (s = SSM_ERR_SCRATCH; s <= SSM_OK; ++s) {
        const char *t = ssm_status_string(s);
        if (!t || !strcmp(t, ssm_status_string(12345))) {
            printf("FAIL status string %d\n", s);
            ++fails;
        }
    }
    expect(scan(FAKE, 0, 16, SSM_BF16), SSM_OK, "scan, no channels");
    expect(scan(NULL, 1, 16, SSM_BF16), SSM_ERR_NULL, "scan, u NULL");
    expect(scan(FAKE, -1, 16, SSM_BF16), SSM_ERR_SIZE, "scan, negative batch");
    expect(scan(FAKE, 0, 0, SSM_BF16), SSM_ERR_SIZE, "scan, N = 0");
    expect(scan(FAKE, 0, SSM_MAX_N + 1, SSM_BF16), SSM_ERR_UNSUPPORTED, "scan, N too large");
    expect(scan(FAKE, 0, 16, 7), SSM_ERR_DTYPE, "scan, dtype");
    expect(scan((const char *)FAKE + 1, 0, 16, SSM_BF16), SSM_ERR_ALIGN, "scan, bf16 alignment");
    expect(ssm_scan_fwd_disc(FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE, NULL, 0, 4, 8,
                             16, SSM_F32, 3, NULL),
           SSM_ERR_UNSUPPORTED, "variant, unknown discretisation");
    expect(ssm_conv_scan_fwd(FAKE, NULL, NULL, 1, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE,
                             NULL, 0, 4, 8, 16, SSM_BF16, NULL),
           SSM_ERR_NULL, "convolution, no filter");
    expect(ssm_scan_bwd(FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, NULL, NULL, FAKE, FAKE,
                        NULL, FAKEF, NULL, NULL, NULL, NULL, 1, 4, 8, 16, SSM_BF16, NULL),
           SSM_ERR_NULL, "backward, dy NULL");
    expect(ssm_scan_fwd_ckpt(FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE, NULL, NULL, 1,
                             64, 8, 16, SSM_BF16, NULL),
           SSM_ERR_NULL, "forward with checkpoints, checkpoints NULL");
    expect(ssm_scan_bwd_ckpt(FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE, NULL, FAKEF,
                             FAKE, FAKE, NULL, FAKEF, NULL, NULL, NULL, NULL, 1, 64, 8, 7,
                             SSM_BF16, NULL),
           SSM_ERR_UNSUPPORTED, "backward with checkpoints, N = 7");
    expect(ssm_ssd_fwd(FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, FAKE, NULL, 0, 4, 2, 0, 64,
                       SSM_BF16, NULL),
           SSM_ERR_SIZE, "SSD, P = 0");
    expect(ssm_step(NULL, FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE, 1, 8, 16,
                    SSM_BF16, NULL),
           SSM_ERR_NULL, "step, state NULL");
    expect(ssm_scan_fwd_noalloc(FAKE, FAKE, NULL, FAKEF, FAKE, FAKE, NULL, NULL, FAKE, NULL, 0, 4,
                                8, 16, SSM_BF16, NULL),
           SSM_OK, "no-alloc, no channels");
    {
        double rates[3];
        expect(ssm_unit_ceilings(NULL, 1, NULL), SSM_ERR_NULL, "ceilings, out NULL");
        expect(ssm_unit_ceilings(rates, 0, NULL), SSM_ERR_SIZE, "ceilings, reps 0");
    }
    printf(fails ? "c abi check: %d failures\n" : "c abi check: ok\n", fails);
    return fails != 0;
}
