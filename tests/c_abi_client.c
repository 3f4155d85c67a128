/* A plain C99 client of libbsa.so: includes the public headers, links the
 * library and makes calls that need no GPU (status strings, the Gather 0
 * sizes, and argument checks that return before any launch).  Prints one
 * line per result for the CPU test that builds and runs it. */
#include <stdint.h>
#include <stdio.h>

#include "bsa.h"
#include "bsa_selftest.h"

int main(void) {
    int32_t n = 0, n_kv = 0, max_kv = 0;
    printf("%s\n", bsa_status_string(BSA_ERR_BOUNDS));
    printf("%d\n", (int)bsa_gather0_sizes(128, 128, 512, 8, &n, &n_kv, &max_kv));
    printf("%d %d %d\n", (int)n, (int)n_kv, (int)max_kv);
    /* D = 96 is unsupported: rejected on the host before anything runs */
    printf("%d\n", (int)bsa_forward(NULL, NULL, NULL, 1, 1, 128, 96, NULL, NULL, 1, NULL, NULL, NULL,
                                     NULL, 0.0f, NULL, NULL, NULL));
    /* an empty row set is a no-op */
    printf("%d\n", (int)bsa_build_index(BSA_IDX_MASK_U8, NULL, 0, 8, 0.0f, NULL, 0, NULL, NULL, 8, NULL));
    return 0;
}
