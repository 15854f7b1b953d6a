/*
 * A plain C11 caller of the library's C ABI (include/clef.h), built and run
 * by test_c_abi.py on a machine with or without a GPU.  It makes only calls
 * that return before touching a device: version and status strings, and
 * argument errors, which the library reports on the host before it launches
 * anything.  The pointers are fake (16-byte aligned or deliberately not) and
 * never dereferenced.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "clef.h"

static int failures;

#define EXPECT(cond)                                                        \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "c_abi_check.c:%d: %s\n", __LINE__, #cond);     \
            ++failures;                                                     \
        }                                                                   \
    } while (0)

/* an argument error: CLEF_ERR_INVALID_ARG and a message for this thread */
#define EXPECT_ARG(call)                                                    \
    do {                                                                    \
        EXPECT((call) == CLEF_ERR_INVALID_ARG);                             \
        EXPECT(strlen(clef_last_error()) > 0);                              \
    } while (0)

int main(void)
{
    void *fake = (void *)(uintptr_t)0x10000;   /* 16-byte aligned */
    void *odd = (void *)(uintptr_t)0x10008;    /* 8-byte aligned only */
    const int8_t *q8 = (const int8_t *)fake;
    const float *f32 = (const float *)fake;

    EXPECT(clef_abi_version() == 100);
    EXPECT(strcmp(clef_status_string(CLEF_OK), "CLEF_OK") == 0);
    EXPECT(strcmp(clef_status_string(CLEF_ERR_INVALID_ARG), "CLEF_ERR_INVALID_ARG") == 0);

    /* quantizer: null input, rotated mode with a partial 128-block, pitch
     * below K, misaligned input, unknown mode, a non-positive static scale */
    EXPECT_ARG(clef_quant_act(NULL, 4, 128, 128, CLEF_ACT_INT8_H128, fake, (float *)fake, NULL));
    EXPECT_ARG(clef_quant_act(fake, 4, 96, 96, CLEF_ACT_FP8_E4M3_H128, fake, (float *)fake, NULL));
    EXPECT_ARG(clef_quant_act(fake, 4, 128, 120, CLEF_ACT_INT8_H128, fake, (float *)fake, NULL));
    EXPECT_ARG(clef_quant_act(odd, 4, 128, 128, CLEF_ACT_FP8_E4M3, fake, (float *)fake, NULL));
    EXPECT_ARG(clef_quant_act(fake, 4, 128, 128, 7, fake, (float *)fake, NULL));
    EXPECT_ARG(clef_quant_act_static(fake, 4, 128, 128, CLEF_ACT_FP8_E4M3, 0.0f, fake, (float *)fake, NULL));

    /* GEMMs: K not a multiple of 16, N not a multiple of 8, pitch below N */
    EXPECT_ARG(clef_w8a8_linear(q8, f32, q8, f32, NULL, 4, 64, 40, fake, 64, NULL));
    EXPECT_ARG(clef_w8a8_linear(q8, f32, q8, f32, NULL, 4, 60, 64, fake, 64, NULL));
    EXPECT_ARG(clef_w8a8_gateup_swiglu(q8, f32, q8, f32, NULL, 4, 64, 64, fake, 32, NULL));
    EXPECT_ARG(clef_fp8_linear(fake, f32, fake, f32, NULL, 4, 64, 40, fake, 64, NULL));
    EXPECT_ARG(clef_fp8_gateup_swiglu(fake, f32, fake, f32, NULL, 4, 60, 64, fake, 64, NULL));
    EXPECT_ARG(clef_w8a8_gemm_s32(q8, q8, 4, 64, 64, (int32_t *)fake, 32, NULL));

    /* LoRA: rank not a multiple of 8, rank above the limit, null factor */
    EXPECT_ARG(clef_lora_add(fake, 128, fake, fake, 4, 128, 64, 12, fake, fake, 64, NULL));
    EXPECT_ARG(clef_lora_add(fake, 128, fake, fake, 4, 128, 64, 2048, fake, fake, 64, NULL));
    EXPECT_ARG(clef_lora_shrink(fake, 128, NULL, 4, 128, 64, fake, 64, NULL));
    EXPECT_ARG(clef_lora_expand_add(fake, 32, fake, 4, 64, 64, fake, 64, NULL));
    EXPECT_ARG(clef_lora_gateup_swiglu(fake, 128, fake, fake, fake, fake, 4, 128, 64, 12,
                                       fake, fake, 128, fake, 64, NULL));
    EXPECT_ARG(clef_lora_add_noalloc(fake, 128, fake, fake, 4, 128, 64, 12, fake, 64, NULL));
    EXPECT_ARG(clef_swiglu_bf16(fake, 4, 64, 100, fake, 64, NULL));

    /* workspace: null size pointer, misaligned buffer */
    EXPECT_ARG(clef_gemm_workspace_bytes(NULL));
    EXPECT_ARG(clef_bind_workspace(NULL, odd, (int64_t)1 << 26));

    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    puts("ok");
    return 0;
}
