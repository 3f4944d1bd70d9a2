/* A plain C99 client of the library: it includes include/gla.h with a C
 * compiler, links libgla.so, prints the parameter structs' layout as the C
 * compiler sees it and calls two host-only entry points. The ABI tests compare
 * the layout with the Python binding's. No GPU call is made. */
#include <stddef.h>
#include <stdio.h>

#include "gla.h"

int main(void)
{
    printf("fwd %zu %zu %zu %zu %zu\n", sizeof(gla_fwd_params), offsetof(gla_fwd_params, workspace),
           offsetof(gla_fwd_params, path), offsetof(gla_fwd_params, log_b), offsetof(gla_fwd_params, window_chunks));
    printf("bwd %zu %zu %zu %zu %zu\n", sizeof(gla_bwd_params), offsetof(gla_bwd_params, workspace),
           offsetof(gla_bwd_params, path), offsetof(gla_bwd_params, log_b), offsetof(gla_bwd_params, grad_log_b));
    printf("status %s\n", gla_status_string(GLA_ERR_INVALID_ARG));
    printf("version %d\n", gla_version());
    return 0;
}
