/* c_host.c -- the C-ABI from plain C99, without Python or PyTorch: library version,
 * status strings, the workspace the 4,256-token joint block needs (width 3072, 24 heads
 * of 128, SwiGLU 9216; 4,096 image + 160 text tokens), and argument checks that reject
 * bad calls on the host before anything is launched.  Needs no GPU.
 *
 *   gcc -std=c99 -I include flow_matching_image_flux3_b300/examples/c_host.c \
 *       -L flow_matching_image_flux3_b300 -lflux3 -Wl,-rpath,<dir of libflux3.so> -o c_host
 */
#include <stdio.h>
#include <string.h>
#include "flux3.h"

static int fails = 0;
static void check(int ok, const char *what) {
    printf("%s %s\n", ok ? "ok  " : "FAIL", what);
    if (!ok) ++fails;
}

int main(void) {
    printf("version: %s\n", flux3_version());
    check(strstr(flux3_version(), "sm_103a") != NULL, "library built for sm_103a");
    check(strlen(flux3_status_string(FLUX3_ERR_INVALID_ARG)) > 0, "status strings");

    flux3_dims d = {3072, 24, 128, 9216, 1e-6f, 1e-6f, 10000.f};
    const int32_t n = 4096 + 160;
    const size_t ws = flux3_block_workspace_size(&d, n);
    printf("joint block workspace at %d tokens: %zu bytes\n", n, ws);
    check(ws > (size_t)n * 3072 * 2, "workspace holds at least the modulated input");
    check(flux3_block_bwd_workspace_size(&d, n) > ws, "the backward pass needs more workspace");

    flux3_dims bad = d;
    bad.heads = 23;  /* 23 x 128 != 3072 */
    check(flux3_block_workspace_size(&bad, n) == 0, "inconsistent dims give no workspace size");

    /* an empty sequence is a no-op; a segment table that does not end at N is rejected */
    int32_t off[3] = {0, 4096, n};
    float mod_dummy[1];
    flux3_segments segs = {2, off, mod_dummy};
    flux3_block_weights w;
    memset(&w, 0, sizeof w);
    check(flux3_block_fwd(&d, &w, &segs, NULL, NULL, n + 1, NULL, NULL, 0, NULL) == FLUX3_ERR_INVALID_ARG,
          "segments must end at n_tokens");
    int32_t off0[2] = {0, 0};
    flux3_segments seg0 = {1, off0, mod_dummy};
    check(flux3_rope_build(&d, NULL, 0, NULL, NULL) == FLUX3_OK, "zero tokens: nothing to do");
    check(flux3_block_fwd(&d, &w, &seg0, NULL, NULL, 0, NULL, NULL, 0, NULL) != FLUX3_OK,
          "missing weights are rejected even for an empty sequence");
    printf("%s\n", fails ? "some checks failed" : "all checks passed");
    return fails ? 1 : 0;
}
