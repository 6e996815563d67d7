/* Plain C99 client of the public header: compiled with gcc -std=c99
 * -pedantic and linked against the built library by tests/test_c_abi.py.
 * Exercises the entry points that need no GPU (version, status strings,
 * argument validation, empty problems) through the C ABI itself, with fake
 * addresses that are never dereferenced.  Prints "ok" on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "skinny_gemm_residual.h"

static int failures = 0;

static void expect(int got, int want, const char* what) {
  if (got != want) {
    printf("FAIL %s: got %d want %d\n", what, got, want);
    ++failures;
  }
}

static const void* fake(uint64_t gib) { return (const void*)(uintptr_t)((uint64_t)1 << 40 | gib << 32); }

int main(void) {
  const int M = 4, N = 7168, K = 3584;
  const void *A = fake(0), *W = fake(1), *R = fake(2), *Y = fake(3), *S = fake(4);

  expect(sgr_abi_version(), SGR_ABI_VERSION, "abi version");
  for (int s = SGR_OK; s <= SGR_ERR_DEVICE; ++s)
    if (!sgr_status_string(s) || strcmp(sgr_status_string(s), "unknown status") == 0) {
      printf("FAIL status string %d\n", s);
      ++failures;
    }

  expect(sgr_validate(A, K, W, R, N, Y, N, M, N, K), SGR_OK, "validate ok");
  expect(sgr_validate(A, K, W, R, N, R, N, M, N, K), SGR_OK, "validate in place");
  expect(sgr_validate(A, K, W, R, N, NULL, N, M, N, K), SGR_ERR_NULL, "validate null Y");
  expect(sgr_validate(A, K, W, R, N, Y, N, M, N + 2, K), SGR_ERR_SHAPE, "validate N % 8");
  expect(sgr_validate((const char*)A + 2, K, W, R, N, Y, N, M, N, K), SGR_ERR_ALIGN, "validate misaligned A");
  expect(sgr_validate(A, K, W, R, N, (const char*)R + 16, N, M, N, K), SGR_ERR_ALIAS, "validate Y inside R");
  expect(sgr_validate(A, K, W, R, N, Y, (int64_t)1 << 40, M, N, K), SGR_ERR_UNSUPPORTED, "validate huge stride");

  expect(sgr_validate_w8(A, K, W, K, (const float*)S, R, N, Y, N, M, N, K), SGR_OK, "validate_w8 ok");
  expect(sgr_validate_w8(A, K, W, K + 8, (const float*)S, R, N, Y, N, M, N, K), SGR_ERR_ALIGN,
         "validate_w8 code stride");
  expect(sgr_validate_w8(A, K, W, K, NULL, R, N, Y, N, M, N, K), SGR_ERR_NULL, "validate_w8 null scale");

  expect(sgr_validate_w4(A, K, W, K / 2, S, K / 16, R, N, Y, N, M, N, K), SGR_OK, "validate_w4 ok");
  expect(sgr_validate_w4(A, K, W, K / 2 + 8, S, K / 16, R, N, Y, N, M, N, K), SGR_ERR_ALIGN,
         "validate_w4 code stride");
  expect(sgr_validate_w4(A, K, W, K / 2, NULL, K / 16, R, N, Y, N, M, N, K), SGR_ERR_NULL,
         "validate_w4 null block scales");
  expect(skinny_gemm_residual_w4(NULL, K, NULL, K / 2, NULL, K / 16, 1.0f, NULL, N, NULL, N, 0, N, K, NULL, 0u,
                                 NULL),
         SGR_OK, "w4 M = 0 no-op");

  /* Empty problems and empty groups return before touching a device. */
  expect(skinny_gemm_residual(NULL, NULL, NULL, NULL, 0, N, K, NULL), SGR_OK, "M = 0 no-op");
  expect(skinny_gemm_residual_grouped(NULL, 0, N, K, NULL, 0u, NULL), SGR_OK, "no groups");
  {
    sgr_group g;
    memset(&g, 0, sizeof g);
    g.M = 0; /* an expert without tokens */
    expect(skinny_gemm_residual_grouped(&g, 1, N, K, NULL, 0u, NULL), SGR_OK, "empty expert");
    g.reserved = 1;
    expect(skinny_gemm_residual_grouped(&g, 1, N, K, NULL, 0u, NULL), SGR_ERR_UNSUPPORTED, "reserved field");
  }

  expect(sgr_select_path(0, N, K) < 0, 1, "select_path rejects M = 0");
  {
    sgr_config c;
    expect(sgr_default_config(0, M, N, K, SGR_PATH_AUTO, NULL), SGR_ERR_NULL, "default_config null");
    expect(sgr_default_config(0, M, N + 2, K, SGR_PATH_AUTO, &c), SGR_ERR_SHAPE, "default_config shape");
  }

  if (failures) return 1;
  printf("ok\n");
  return 0;
}
