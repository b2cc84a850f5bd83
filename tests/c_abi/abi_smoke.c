/* Plain-C client of libdg: compiles against include/dg.h alone and calls the
 * host-only entry points (no GPU needed).  Exit code 0 on success. */
#include <stdio.h>
#include <string.h>

#include "dg.h"

int main(void) {
    dg_plan p;
    if (strcmp(dg_status_string(DG_OK), "DG_OK") != 0) return 1;
    if (dg_version() < 100) return 2;
    /* 8192^3 E4M3 on 152 SMs: CTA-pair 256 x 256 tiles, one CTA per SM. */
    if (dg_gemm_plan(8192, 8192, 8192, DG_E4M3, DG_E4M3, 152, &p) != DG_OK) return 3;
    if (p.path != 3 || p.block_m != 256 || p.block_n != 256 || p.grid != 152) return 4;
    /* M = 1 against the decode QKV weights takes the warp-MMA GEMV. */
    if (dg_gemm_plan(1, 12288, 4096, DG_E4M3, DG_BF16, 152, &p) != DG_OK || p.path != 5) return 5;
    /* Argument errors come back before any device access. */
    if (dg_fp8_gemm(0, 0, 0, -1, 1, 16, 0, 0, 0, DG_BF16, 0) != DG_ERR_INVALID_VALUE) return 6;
    if (dg_gemm_plan(4, 4, 16, DG_BF16, DG_BF16, 10, &p) != DG_ERR_INVALID_VALUE) return 7;
    printf("c abi ok\n");
    return 0;
}
