/* A plain C99 caller of libflce, compiled and run by tests/test_abi_host.py without a GPU.
 *
 * It shows that include/flce.h is a C header (no C++ or CUDA types in the signatures) and that
 * a C program links against libflce.so and gets the documented answers from the entry points
 * that need no device: the size queries (host arithmetic) and argument validation, which rejects
 * bad calls before any CUDA call. Pointers below are either NULL or never dereferenced: each
 * call fails validation first. Prints "ok" and exits 0 when every check holds.
 */
#include <stdio.h>
#include <string.h>

#include "flce.h"

static int failures = 0;

static void check(int cond, const char* what) {
  if (!cond) {
    printf("FAILED: %s\n", what);
    ++failures;
  }
}

int main(void) {
  const int64_t T = 16384, H = 4096, V = 128256;
  size_t fwd, bwd, both;
  int64_t vc, rows, raster = 0;
  float loss = 0.f;

  check(flce_version() == 10000, "flce_version");
  check(flce_strerror(FLCE_ERR_ARG) != NULL && strlen(flce_strerror(FLCE_ERR_ARG)) > 0,
        "flce_strerror(FLCE_ERR_ARG)");
  check(strcmp(flce_strerror(FLCE_OK), "ok") == 0, "flce_strerror(FLCE_OK)");

  /* size queries: host arithmetic only */
  fwd = flce_forward_workspace_size(T, H, V, FLCE_DTYPE_BF16);
  bwd = flce_backward_workspace_size(T, H, V, FLCE_DTYPE_BF16);
  both = flce_forward_backward_workspace_size(T, H, V, FLCE_DTYPE_BF16);
  check(fwd > 0 && bwd > 0 && both > 0, "workspace sizes of a valid problem");
  /* never the T x V logits in fp32 (8.4 GB here) */
  check(bwd < (size_t)T * (size_t)V * 4u, "backward workspace below the fp32 logits");
  check(flce_forward_workspace_size(0, H, V, FLCE_DTYPE_BF16) == 0, "T = 0 rejected");
  check(flce_backward_workspace_size(T, H, V, 7) == 0, "unknown dtype rejected");
  vc = flce_backward_slab_width(T, H, V, FLCE_DTYPE_BF16);
  check(vc > 0 && vc % 256 == 0 && vc >= V / 8, "slab width");
  rows = flce_forward_backward_chunk_tokens(T, H, V, FLCE_DTYPE_BF16);
  check(rows > 0 && rows <= T && rows % 256 == 0, "single-call chunk rows");

  /* validation before any CUDA call */
  check(flce_forward(NULL, NULL, NULL, T, H, V, FLCE_DTYPE_BF16, FLCE_REDUCTION_MEAN, NULL, NULL,
                     NULL, 0, NULL, NULL) == FLCE_ERR_ARG,
        "flce_forward with null pointers");
  check(flce_backward(NULL, NULL, NULL, NULL, T, H, V, FLCE_DTYPE_BF16, FLCE_REDUCTION_MEAN, NULL,
                      NULL, NULL, NULL, 0, NULL, NULL) == FLCE_ERR_ARG,
        "flce_backward with null pointers");
  check(flce_forward_backward(NULL, NULL, NULL, T, H, V, FLCE_DTYPE_BF16, FLCE_REDUCTION_SUM,
                              NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL) == FLCE_ERR_ARG,
        "flce_forward_backward with null pointers");
  /* the fixed scratch is checked against the problem before any CUDA call: null pointers and
   * T = 0 are invalid, and 32768 tokens at V = 128256 need more than FLCE_STATIC_SCRATCH_BYTES
   * (the stand-in addresses below are never dereferenced) */
  check(flce_forward_static_scratch(NULL, NULL, NULL, T, H, V, FLCE_DTYPE_BF16,
                                    FLCE_REDUCTION_MEAN, &loss, NULL, NULL, NULL) == FLCE_ERR_ARG,
        "flce_forward_static_scratch with null pointers");
  check(flce_forward_static_scratch(&loss, &loss, &raster, 0, H, V, FLCE_DTYPE_BF16,
                                    FLCE_REDUCTION_MEAN, &loss, &loss, &failures, NULL) ==
            FLCE_ERR_ARG,
        "flce_forward_static_scratch with T = 0");
  check(flce_forward_workspace_size(2 * T, H, V, FLCE_DTYPE_BF16) > FLCE_STATIC_SCRATCH_BYTES,
        "forward scratch of 32768 tokens above the static array");
  check(flce_forward_static_scratch(&loss, &loss, &raster, 2 * T, H, V, FLCE_DTYPE_BF16,
                                    FLCE_REDUCTION_MEAN, &loss, &loss, &failures, NULL) ==
            FLCE_ERR_WORKSPACE,
        "flce_forward_static_scratch above its scratch size");

  /* tuning knobs: validation and a value that needs no device */
  check(flce_set_tuning(-12345, 0) == FLCE_ERR_ARG, "unknown tuning key");
  check(flce_set_tuning(FLCE_TUNE_RASTER_ROWS, 100) == FLCE_ERR_ARG, "raster rows not /256");
  check(flce_get_tuning(FLCE_TUNE_RASTER_ROWS, &raster) == FLCE_OK && raster == 2048,
        "default raster rows");
  check(flce_get_tuning(FLCE_TUNE_RASTER_ROWS, NULL) == FLCE_ERR_ARG, "null tuning output");
  check(flce_set_backward_slab_width(100) == FLCE_ERR_ARG, "slab width not /256");

  if (failures == 0) printf("ok\n");
  return failures == 0 ? 0 : 1;
}
