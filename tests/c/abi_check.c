/* A plain C99 program against the public header: it compiles with
 * -pedantic -Werror, links the library and runs its host-only calls (no GPU
 * needed). Built and run by tests/test_library_cpu.py. */
#include <stdio.h>
#include <string.h>
#include "pagedattn.h"
int main(void) {
    if (pa_version() < 10100) return 1;
    if (strcmp(pa_status_string(PA_OK), "ok") != 0) return 2;
    if (pa_default_partition_size(PA_DTYPE_FP8_E4M3) != 1024) return 3;
    if (pa_decode_workspace_size(0, 8, 128, 100) != 0) return 4;
    if (pa_check_error_word(PA_DEVERR_SLOT) != PA_ERR_DEVICE_BOUNDS) return 5;
    printf("ok\n");
    return 0;
}
