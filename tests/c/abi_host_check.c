/* A plain C consumer of libgva.so: includes only include/gva.h, links the library and
 * exercises the entry points that need no GPU (version, status strings, the RoPE table,
 * argument validation that returns before any CUDA call).  Prints "ok" and exits 0
 * when every check holds; otherwise prints the failed check and exits 1. */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "gva.h"

static int failures = 0;

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            printf("check failed (line %d): %s\n", __LINE__, #cond); \
            ++failures;                                               \
        }                                                             \
    } while (0)

int main(void) {
    CHECK(gva_abi_version() == GVA_ABI_VERSION);
    CHECK(strcmp(gva_status_string(GVA_OK), gva_status_string(GVA_ERR_ARG)) != 0);
    CHECK(strstr(gva_status_string(987654), "unknown") != NULL);

    /* RoPE table: Rot(0) is the identity, and the entry for position 1 of pair 0 is
     * (cos 1, sin 1) rounded to fp32 (theta_0 = 1 for any base). */
    float tab[4 * 8 * 2];
    CHECK(gva_rope_table_fill(tab, 4, 16, 10000.0) == GVA_OK);
    for (int i = 0; i < 8; ++i) {
        CHECK(tab[2 * i] == 1.0f);
        CHECK(tab[2 * i + 1] == 0.0f);
    }
    CHECK(tab[16] == (float)cos(1.0));
    CHECK(tab[17] == (float)sin(1.0));
    CHECK(gva_rope_table_fill(tab, 4, 7, 10000.0) == GVA_ERR_ARG);
    CHECK(gva_rope_table_fill(NULL, 4, 16, 10000.0) == GVA_ERR_ARG);

    /* argument validation before any CUDA call */
    gva_dims d = {2, 16, 4, 64, 64, 16, GVA_BF16, GVA_BF16};
    gva_dims bad = d;
    bad.G = 5; /* H % G != 0 */
    void *fake = (void *)(size_t)0x10000;
    gva_cache cache;
    memset(&cache, 0, sizeof(cache));
    cache.rows.layout = GVA_LAYOUT_CONTIGUOUS;
    cache.rows.num_rows = 2 * 1024;
    cache.rows.T_cap = 1024;
    cache.V = fake;
    cache.K_rope = fake;
    float *ff = (float *)fake;
    CHECK(gva_decode_workspace_size(&bad) == 0);
    CHECK(gva_decode_attention(NULL, &bad, fake, fake, ff, (const int *)fake, &cache, ff, 100,
                               0.1f, ff, NULL, fake, (size_t)1 << 30) == GVA_ERR_ARG);
    CHECK(gva_decode_attention(NULL, &d, fake, fake, ff, (const int *)fake, &cache, ff, 100,
                               0.1f, NULL, NULL, fake, (size_t)1 << 30) == GVA_ERR_ARG);
    CHECK(gva_append_cache(NULL, &bad, ff, ff, (const int *)fake, NULL, &cache, ff, 100) ==
          GVA_ERR_ARG);
    gva_decode_opts o = {GVA_PATH_AUTO, 0, 2 /* unknown flag */, 0.f, NULL};
    CHECK(gva_decode_attention_ex(NULL, &d, fake, fake, ff, (const int *)fake, &cache, ff, 100,
                                  0.1f, ff, NULL, fake, (size_t)1 << 30, &o) == GVA_ERR_ARG);
    /* prefill: ragged caches are not taken by the view paths; an empty chunk is an
       argument error */
    gva_cache rag = cache;
    rag.rows.layout = GVA_LAYOUT_RAGGED;
    rag.rows.offsets = (const int *)fake;
    gva_decode_opts simt = {GVA_PATH_SIMT, 0, 0, 0.f, NULL};
    CHECK(gva_prefill_attention(NULL, &d, 4, fake, fake, ff, (const int *)fake, ff, ff, &rag, ff,
                                100, 0.1f, ff, NULL, fake, (size_t)1 << 30, &simt) ==
          GVA_ERR_UNSUPPORTED);
    CHECK(gva_prefill_attention(NULL, &d, 0, fake, fake, ff, (const int *)fake, ff, ff, &cache,
                                ff, 100, 0.1f, ff, NULL, fake, (size_t)1 << 30, NULL) ==
          GVA_ERR_ARG);
    CHECK(gva_read_probe(NULL, fake, 15, (unsigned *)fake) == GVA_ERR_ARG);

    if (failures) return 1;
    printf("ok\n");
    return 0;
}
