/* A plain C99 consumer of the library: compiles against include/slimkv.h with a C
 * compiler and calls the entry points that need no GPU (sizes, status strings,
 * argument checks). Exit status 0 when every check holds. */
#include <stdio.h>
#include <stdint.h>

#include "slimkv.h"

#define CHECK(c)                                                   \
    do {                                                           \
        if (!(c)) {                                                \
            fprintf(stderr, "check failed: %s (line %d)\n", #c, __LINE__); \
            return 1;                                              \
        }                                                          \
    } while (0)

int main(void) {
    slimkv_shape s = {8, 32, 8, 128, 8192, 256, 256, 2048, 0.08838834764831845f, 500000.0, SLIMKV_BF16};
    CHECK(slimkv_abi_version() == SLIMKV_ABI_VERSION);
    const size_t ws = slimkv_workspace_bytes(&s, SLIMKV_LATENT);
    CHECK(ws > 0 && ws % 256 == 0);
    CHECK(slimkv_workspace_bytes(&s, SLIMKV_RECONSTRUCT) > ws);
    CHECK(slimkv_status_str(SLIMKV_ERR_SHAPE) != NULL);

    /* invalid sizes are rejected before any launch */
    slimkv_shape bad = s;
    bad.Hq = 30;
    CHECK(slimkv_workspace_bytes(&bad, SLIMKV_LATENT) == 0);
    CHECK(slimkv_kernel_path(&bad, SLIMKV_LATENT) == -1);
    void* p = (void*)(uintptr_t)4096;
    CHECK(slimkv_decode_attn(&bad, p, p, p, p, p, p, p, (const int32_t*)p, (float*)p, p, (size_t)1 << 40, NULL) ==
          SLIMKV_ERR_SHAPE);
    CHECK(slimkv_decode_attn(&s, NULL, p, p, p, p, p, p, (const int32_t*)p, (float*)p, p, ws, NULL) ==
          SLIMKV_ERR_NULL);
    CHECK(slimkv_decode_attn(&s, p, p, p, p, p, p, p, (const int32_t*)p, (float*)p, p, ws - 1, NULL) ==
          SLIMKV_ERR_WORKSPACE);
    CHECK(slimkv_append_kv(&s, p, p, p, p, NULL, NULL) == SLIMKV_ERR_NULL);
    bad = s;
    bad.W = 0;
    CHECK(slimkv_append_kv(&bad, p, p, p, p, (const int32_t*)p, NULL) == SLIMKV_ERR_SHAPE);
    printf("c abi ok (workspace %zu bytes)\n", ws);
    return 0;
}
