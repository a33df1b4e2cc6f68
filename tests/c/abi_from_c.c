/*
 * A plain C caller of libfp8bs.so, built with the system C compiler against
 * include/fp8bs.h.  Only calls that need no GPU: status strings, host-side
 * argument checks and the schedule queries.  Prints "ok" and exits 0 when
 * every check holds.
 */
#include <stdio.h>
#include <string.h>

#include "fp8bs.h"

static int failures = 0;

static void expect(int cond, const char *what)
{
    if (!cond) {
        fprintf(stderr, "FAILED: %s\n", what);
        ++failures;
    }
}

int main(void)
{
    int ctas = 0, npad = 0, tt = 0, split = 0;
    long long units = 0, b = 0, e = 0;

    expect(strcmp(fp8bs_status_string(FP8BS_OK), "ok") == 0, "status string of FP8BS_OK");
    expect(fp8bs_status_string((fp8bs_status)99) != NULL, "status string of an unknown code");

    /* host-side argument checks return before any device work */
    expect(fp8_quant_act(NULL, 8, 512, 512, NULL, NULL, 0, NULL) == FP8BS_ERR_INVALID_ARG, "null input");
    expect(fp8_blockscaled_gemm((const uint8_t *)16, (const float *)16, (const uint8_t *)16, (const float *)16,
                                (void *)16, 513, 256, 512, (void *)256, 1 << 20, 0, NULL) ==
               FP8BS_ERR_UNSUPPORTED_SHAPE,
           "M above 512");

    /* the decode schedule of the 5,120 x 5,120 layer on 152 SMs */
    expect(fp8bs_split_plan(5120, 5120, 0, 152, 0, &ctas, &units, &b, &e) == FP8BS_OK, "split plan");
    expect(ctas == 152 && units == 1600 && b == 0 && e == 10, "split plan values");
    expect(fp8bs_gemm_schedule(512, 5120, 5120, 152, &npad, &tt, &ctas, &units, &split) == FP8BS_OK,
           "schedule query");
    expect(npad == 128 && tt == 4 && ctas == 152 && units == 6400 && split == 1, "schedule values at M = 512");

    /* the fused entry point's route: the separate cast kernel by default; with
       the prologue-cast flag, the prologue for the tiny workload and still the
       separate cast for the square layer at 8 tokens */
    {
        int prologue = -1;
        expect(fp8bs_fused_route(8, 256, 512, 152, 0, &prologue) == FP8BS_OK && prologue == 0, "tiny: separate by default");
        expect(fp8bs_fused_route(8, 256, 512, 152, FP8BS_FLAG_PROLOGUE_CAST, &prologue) == FP8BS_OK && prologue == 1,
               "tiny: prologue with the flag");
        expect(fp8bs_fused_route(8, 5120, 5120, 152, FP8BS_FLAG_PROLOGUE_CAST, &prologue) == FP8BS_OK && prologue == 0,
               "square: separate");
    }

    if (failures == 0)
        printf("ok\n");
    return failures == 0 ? 0 : 1;
}
