/* A plain C99 client of the C ABI, built by tests/test_c_client.py: it includes only
 * include/vit_attn.h, links against libvitattn.so and makes the calls that need no GPU
 * (version, status strings, workspace sizing, and calls that fail host validation),
 * printing one "name=value" line per result. */
#include <stdio.h>

#include "vit_attn.h"

int main(void)
{
    /* addresses that are never dereferenced: every call below fails a host check first */
    void *p16 = (void *)(uintptr_t)16, *p128 = (void *)(uintptr_t)128, *p256 = (void *)(uintptr_t)256;
    vit_q_rope_t qr = {0};

    printf("version=%s\n", vit_version());
    printf("status_bad_head_dim=%s\n", vit_status_string(VIT_ERR_BAD_HEAD_DIM));
    printf("ws_16x80=%lu\n", (unsigned long)vit_varlen_attn_workspace_size(1024, 16, 1, 80));
    printf("ws_bad_d=%lu\n", (unsigned long)vit_varlen_attn_workspace_size(1024, 16, 1, 81));
    printf("attn_bad_d=%d\n", (int)vit_varlen_attn(p128, p128, p128, 128, 2, 81, 160, 160, 160, p16,
                                                   1, 128, 0.0f, p128, 160, p256, 1u << 20, NULL, NULL));
    printf("attn_neg_max_seqlen=%d\n", (int)vit_varlen_attn(p128, p128, p128, 128, 2, 80, 160, 160, 160,
                                                            p16, 1, -1, 0.0f, p128, 160, p256,
                                                            1u << 20, NULL, NULL));
    printf("prologue_bad_mode=%d\n", (int)vit_qk_norm_rope_ex(p16, p16, p16, p16, 10, 2, 80, 160, 160, 160, 160,
                                                              p16, p16, NULL,
                                                              1e-6f, 2, NULL, NULL));
    qr.pos_hw = p16;
    qr.cos_sin = p16;
    qr.max_pos = 0;                                             /* an empty table */
    qr.eps = 1e-6f;
    qr.rope_mode = VIT_ROPE_ROTATE_HALF;
    printf("fused_empty_table=%d\n", (int)vit_varlen_attn_fused_q(p128, p128, p128, 128, 2, 80, 160, 160, 160, &qr,
                                                                  p16, 1, 128, 0.0f, p128, 160,
                                                                  NULL, p256, 1u << 20, NULL, NULL));
    printf("read_status_null=%d\n", (int)vit_read_status(NULL, NULL));
    return 0;
}
