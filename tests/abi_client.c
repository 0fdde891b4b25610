/*
 * A plain C11 client of include/ep.h: it compiles against the header alone
 * and links against libep_gb300.so.  It exercises only calls that finish on
 * the host (sizes, host-side argument checks, empty batches, status text), so
 * it runs with or without a GPU; it prints "abi client ok" and exits 0 when
 * every check holds, else names the failed check and exits 1.
 */
#include <stdio.h>
#include <string.h>

#include "ep.h"

static int failures = 0;

static void check(int cond, const char *what)
{
    if (!cond) {
        printf("FAILED: %s (last error: %s)\n", what, ep_last_error());
        ++failures;
    }
}

int main(void)
{
    ep_shape_t decode = {128, 7168, 256, 8, 32, EP_LAYOUT_CAPACITY, 128};
    ep_shape_t grouped = {16384, 4096, 128, 8, 8, EP_LAYOUT_PACKED, 0};
    ep_shape_t empty = {0, 64, 16, 4, 1, EP_LAYOUT_PACKED, 0};
    ep_shape_t bad_k = {4, 64, 16, 17, 1, EP_LAYOUT_PACKED, 0};
    ep_shape_t too_wide = {300 * 1024 / 8, 8, 1024, 8, 1, EP_LAYOUT_PACKED, 0};
    uint32_t dummy;

    check(ep_abi_version() == 101, "ABI version");
    check(strcmp(ep_status_string(EP_OK), "ok") == 0, "status text");
    check(strcmp(ep_status_str(EP_ERR_CUDA), ep_status_string(EP_ERR_CUDA)) == 0, "status text alias");
    check(ep_recv_rows(&decode) == 256 * 128, "capacity rows");
    check(ep_recv_rows(&grouped) == 16384 * 8, "packed rows");
    check(ep_layout_workspace_bytes(&grouped) == (size_t)128 * 128 * 4, "layout workspace");
    check(ep_combine_src_workspace_bytes(&grouped) == (size_t)2 * 16384 * 8 * 4, "source-map workspace");
    check(ep_recv_rows(&bad_k) == -1, "bad shape has no rows");
    check(ep_get_layout(&bad_k, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL) ==
              EP_ERR_INVALID_ARG, "bad shape rejected");
    check(strlen(ep_last_error()) > 0, "failure text");
    check(ep_get_layout_static(&too_wide, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL) ==
              EP_ERR_UNSUPPORTED, "static layout beyond its scratch");
    /* a misaligned hidden row is refused before anything is enqueued */
    check(ep_dispatch(&decode, (const void *)((char *)&dummy + 2), NULL, (const int32_t *)&dummy,
                      EP_PAYLOAD_BF16, (void *)&dummy, NULL, NULL, NULL, NULL) == EP_ERR_INVALID_ARG,
          "misaligned x rejected");
    /* an empty batch is a no-op for every data-moving call */
    check(ep_dispatch(&empty, NULL, NULL, NULL, EP_PAYLOAD_BF16, NULL, NULL, NULL, NULL, NULL) == EP_OK,
          "empty dispatch");
    check(ep_combine(&empty, NULL, NULL, NULL, NULL, NULL, NULL) == EP_OK, "empty combine");
    check(ep_combine_src(&empty, NULL, NULL, EP_PAYLOAD_BF16, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL) == EP_OK,
          "empty source-map combine");
    if (failures) return 1;
    printf("abi client ok\n");
    return 0;
}
