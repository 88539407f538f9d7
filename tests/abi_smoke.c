/* A plain C99 client of include/sift.h, built and run by test_abi_c_cpu.py without a
 * GPU: it links against libsift.so and uses only the calls that stay on the host
 * (status names, the workspace size, argument validation before any launch).
 * Prints one "ok" line per check and returns non-zero on the first failure. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "sift.h"

static int failures = 0;

static void check(int cond, const char *what) {
    printf("%s %s\n", cond ? "ok" : "FAIL", what);
    if (!cond) ++failures;
}

int main(void) {
    static const char *names[] = {"SIFT_OK", "SIFT_ERR_INVALID_ARG", "SIFT_ERR_UNSUPPORTED",
                                  "SIFT_ERR_CUDA", "SIFT_ERR_TIMEOUT", "SIFT_ERR_DEVICE_CHECK"};
    int code;
    for (code = 0; code <= 5; ++code) {
        const char *s = sift_status_string((sift_status)code);
        check(s != NULL && strcmp(s, names[code]) == 0, names[code]);
    }
    check(sift_abi_version() == 101, "abi version");

    /* one prompt of 256 tokens, no documents; the device pointers are never touched on
     * the host, so any 16-byte aligned value will do here */
    sift_problem p;
    memset(&p, 0, sizeof p);
    p.num_prompts = 1;
    p.num_layers = 1;
    p.num_q_heads = 4;
    p.num_kv_heads = 2;
    p.head_dim = 128;
    p.tile = 128;
    p.total_tokens = 256;
    p.max_tiles_per_prompt = 2;
    p.cu_seqlens = (const int32_t *)(uintptr_t)256;
    p.doc_cu = (const int32_t *)(uintptr_t)512;
    const size_t ws = sift_workspace_bytes(&p);
    check(ws >= sizeof(int32_t), "workspace bytes of a valid problem");

    void *dev = (void *)(uintptr_t)4096;
    int32_t *status = (int32_t *)(uintptr_t)8192;
    p.num_q_heads = 6;
    p.num_kv_heads = 4; /* Hq is not a multiple of Hkv */
    check(sift_dense_prefill(&p, dev, dev, dev, 0.0f, dev, (float *)dev, dev, ws, status, NULL) ==
              SIFT_ERR_INVALID_ARG,
          "inconsistent head counts rejected on the host");
    check(sift_workspace_bytes(&p) == 0, "no workspace for an invalid problem");
    p.num_q_heads = 4;
    p.num_kv_heads = 2;
    p.total_tokens = 200; /* not a multiple of the tile */
    check(sift_dense_prefill(&p, dev, dev, dev, 0.0f, dev, (float *)dev, dev, ws, status, NULL) ==
              SIFT_ERR_UNSUPPORTED,
          "ragged length rejected by the aligned entry point");
    return failures == 0 ? 0 : 1;
}
