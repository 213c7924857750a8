/*
 * A plain C program against include/gla.h and libgla.so: the boundary compiles as C and
 * links without C++ or torch. Every call here is rejected by argument validation or has
 * no work (a shape with no tokens), so nothing is ever launched and no pointer is ever
 * dereferenced: it runs the same on a machine with or without a GPU.
 * Exit status 0 when every check holds; otherwise the number of the first failed check.
 */
#include <stdio.h>
#include <string.h>

#include "gla.h"

#define CHECK(n, cond)                                       \
    do {                                                     \
        if (!(cond)) {                                       \
            fprintf(stderr, "c_abi_check: check %d failed\n", n); \
            return n;                                        \
        }                                                    \
    } while (0)

int main(void) {
    CHECK(1, gla_version() >= 100);
    CHECK(2, strcmp(gla_status_string(GLA_OK), "GLA_OK") == 0);
    CHECK(3, strcmp(gla_status_string(GLA_ERR_ALIAS), "GLA_ERR_ALIAS") == 0);
    /* NULL inputs with work to do: rejected before any CUDA call */
    CHECK(4, gla_fwd(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, 1, 64, 2, 128, 128, NULL) ==
                 GLA_ERR_NULL_ARG);
    CHECK(5, gla_fwd_f32(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, 1, 64, 2, 128, 128,
                         NULL) == GLA_ERR_NULL_ARG);
    CHECK(6, gdn_fwd(NULL, NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, 1, 64, 2, 128, 128,
                     GLA_IO_BF16, NULL, 0, NULL) == GLA_ERR_NULL_ARG);
    CHECK(7, gla_step(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, 2, 2, 128, 128, GLA_IO_BF16,
                      NULL) == GLA_ERR_NULL_ARG);
    /* bad shapes and options */
    CHECK(8, gla_fwd(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, -1, 64, 2, 128, 128, NULL) ==
                 GLA_ERR_BAD_SHAPE);
    CHECK(9, gdn_fwd(NULL, NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, 1, 64, 2, 130, 128,
                     GLA_IO_BF16, NULL, 0, NULL) == GLA_ERR_UNSUPPORTED_DIM);
    {
        gla_options opt;
        memset(&opt, 0, sizeof(opt));
        opt.seq_splits = -1;
        CHECK(10, gla_fwd_ex(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, 1, 64, 2, 128, 128,
                             GLA_IO_BF16, &opt, NULL) == GLA_ERR_NULL_ARG ||
                      gla_fwd_ex(NULL, NULL, NULL, NULL, 1.0f, NULL, NULL, NULL, 1, 64, 2, 128,
                                 128, GLA_IO_BF16, &opt, NULL) == GLA_ERR_BAD_OPTION);
    }
    /* workspace sizes are pure host arithmetic */
    CHECK(11, gdn_fwd_workspace_size(1, 64, 1, 128, 128) > 0);
    CHECK(12, gdn_fwd_workspace_size(2, 65, 3, 128, 128) == 12 * gdn_fwd_workspace_size(1, 64, 1, 128, 128));
    CHECK(13, gdn_fwd_workspace_size(1, 64, 1, 130, 128) == 0);
    CHECK(14, gla_last_error_detail() != NULL);
    printf("c_abi_check ok\n");
    return 0;
}
