/* Host-only use of the C ABI from a plain C99 program: the header compiles as
 * C, the library links, and the calls that return before touching a device
 * (version, status strings, argument validation, empty problems, workspace
 * sizes) behave as the header documents.  Exit status 0 = every check held;
 * otherwise the number of failed checks. */
#include <stddef.h>
#include <stdio.h>
#include <string.h>

#include "la.h"

static int failures = 0;

#define CHECK(cond)                                                         \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
            ++failures;                                                     \
        }                                                                   \
    } while (0)

/* dense [B, T, H, D] views: batch, token, head strides in elements */
static la_dims dense_dims(int32_t B, int32_t T, int32_t H, int32_t D, int32_t E)
{
    la_dims d;
    memset(&d, 0, sizeof d);
    d.batch = B;
    d.seq_len = T;
    d.heads = H;
    d.dim_qk = D;
    d.dim_v = E;
    d.qk_strides[0] = (int64_t)T * H * D;
    d.qk_strides[1] = (int64_t)H * D;
    d.qk_strides[2] = D;
    d.v_strides[0] = (int64_t)T * H * E;
    d.v_strides[1] = (int64_t)H * E;
    d.v_strides[2] = E;
    return d;
}

/* never dereferenced: every call below fails validation or has nothing to do */
static char fake_buf[16];
#define FAKE ((void *)fake_buf)

static la_status fwd(const la_dims *d, int32_t dtype, const void *q, const void *o,
                     const int32_t *cu, const int32_t *cu_host)
{
    return la_fwd(d, dtype, q, FAKE, FAKE, (const float *)FAKE, 1.0f, NULL, 0, cu, cu_host,
                  (void *)o, NULL, NULL, 0, NULL);
}

int main(void)
{
    la_dims d = dense_dims(2, 16, 2, 64, 64);
    la_dims bad;
    int32_t good_cu[4] = {0, 5, 5, 16};
    int32_t falling_cu[4] = {0, 6, 5, 16};
    int32_t empty_cu[1] = {0};

    /* layout the bindings mirror: no padding */
    CHECK(sizeof(la_dims) == 128);
    CHECK(offsetof(la_dims, qk_strides) == 24);
    CHECK(offsetof(la_dims, kv_heads) == 72);
    CHECK(offsetof(la_dims, k_strides) == 80);

    CHECK(la_version() >= 1);
    CHECK(strcmp(la_strerror(LA_OK), "ok") == 0);
    CHECK(strcmp(la_strerror(99), "unknown status") == 0);

    /* validation: statuses and messages, nothing launched */
    CHECK(fwd(NULL, LA_DTYPE_BF16, FAKE, FAKE, NULL, NULL) == LA_ERR_INVALID_ARG);
    CHECK(strstr(la_last_error(), "dims") != NULL);
    CHECK(fwd(&d, 7, FAKE, FAKE, NULL, NULL) == LA_ERR_INVALID_ARG);
    CHECK(fwd(&d, LA_DTYPE_BF16, NULL, FAKE, NULL, NULL) == LA_ERR_INVALID_ARG);
    CHECK(strstr(la_last_error(), "q is NULL") != NULL);
    bad = dense_dims(2, 16, 2, 64, 300);
    CHECK(fwd(&bad, LA_DTYPE_BF16, FAKE, FAKE, NULL, NULL) == LA_ERR_UNSUPPORTED);
    bad = d;
    bad.kv_heads = 3; /* does not divide 2 heads */
    CHECK(fwd(&bad, LA_DTYPE_BF16, FAKE, FAKE, NULL, NULL) == LA_ERR_INVALID_ARG);
    bad = d;
    bad.reserved = 1;
    CHECK(fwd(&bad, LA_DTYPE_BF16, FAKE, FAKE, NULL, NULL) == LA_ERR_INVALID_ARG);

    /* packed sequences: batch 1, table checked on the host copy */
    bad = dense_dims(1, 16, 2, 64, 64);
    bad.num_seqs = 3;
    CHECK(fwd(&bad, LA_DTYPE_BF16, FAKE, FAKE, good_cu, falling_cu) == LA_ERR_INVALID_ARG);
    CHECK(strstr(la_last_error(), "decreases") != NULL);
    bad.batch = 2;
    CHECK(fwd(&bad, LA_DTYPE_BF16, FAKE, FAKE, good_cu, good_cu) == LA_ERR_INVALID_ARG);

    /* backward entry points validate their own outputs */
    CHECK(la_bwd(&d, LA_DTYPE_BF16, FAKE, FAKE, FAKE, NULL, (const float *)FAKE, 1.0f, NULL, NULL,
                 0, NULL, NULL, FAKE, FAKE, FAKE, NULL, NULL, 0, NULL) == LA_ERR_INVALID_ARG);
    CHECK(strstr(la_last_error(), "d_o") != NULL);

    /* nothing to compute: success without a device */
    bad = dense_dims(0, 16, 2, 64, 64);
    CHECK(fwd(&bad, LA_DTYPE_BF16, NULL, NULL, NULL, NULL) == LA_OK);
    bad = dense_dims(1, 0, 2, 64, 64);
    CHECK(fwd(&bad, LA_DTYPE_BF16, NULL, NULL, empty_cu, empty_cu) == LA_OK);

    /* workspace sizes: the packed schedule in 256-byte blocks */
    CHECK(la_workspace_size(0) == 0);
    CHECK(la_workspace_size(65) == 512);
    bad = dense_dims(1, 16, 2, 64, 64);
    bad.num_seqs = 3;
    CHECK(la_workspace_size_for(&bad, LA_DTYPE_BF16, good_cu) == la_workspace_size(3));

    CHECK(la_kernel_family(&d, LA_DTYPE_BF16) >= 0);
    d.dim_qk = 0;
    CHECK(la_kernel_family(&d, LA_DTYPE_BF16) == -1);

    if (failures == 0)
        printf("all C ABI checks passed\n");
    return failures;
}
