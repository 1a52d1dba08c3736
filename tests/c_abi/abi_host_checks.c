/* A plain C client of the q4lin C ABI: compiles against include/q4lin.h alone, links
 * libq4lin.so, and exercises the calls that need no GPU (capacity and route queries,
 * host-side argument checks, status strings).  Prints one line per check and exits
 * non-zero on the first mismatch. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "q4lin.h"

static int fails = 0;

#define CHECK(cond, what)                          \
  do {                                             \
    if (!(cond)) {                                 \
      printf("FAIL %s\n", what);                   \
      ++fails;                                     \
    } else {                                       \
      printf("ok   %s\n", what);                   \
    }                                              \
  } while (0)

int main(void) {
  /* fake, 16-byte aligned addresses: every call below is refused before any use */
  const uint8_t* wq = (const uint8_t*)(uintptr_t)256;
  const uint16_t* sc = (const uint16_t*)(uintptr_t)512;
  const uint16_t* x = (const uint16_t*)(uintptr_t)768;
  uint16_t* y = (uint16_t*)(uintptr_t)1024;

  CHECK(q4lin_workspace_bytes(6144, 5120, 1) == 0, "no workspace on the library's routes");
  CHECK(q4lin_route_workspace_bytes(Q4LIN_ROUTE_TC_FP16, 6144, 5120, 1024) ==
            (size_t)2 * 1024 * 5120 + 4 * 1024 + 4 * 6144,
        "fp16 route workspace: 2TK + 4T + 4N");
  CHECK(q4lin_select_route(6144, 5120, 1) == Q4LIN_ROUTE_GEMV, "one token: the GEMV");
  CHECK(q4lin_linear(wq, sc, x, y, 4, 100, 1, NULL, NULL) == Q4LIN_ERR_UNSUPPORTED_SHAPE, "K % 8 refused");
  CHECK(q4lin_linear(NULL, sc, x, y, 4, 128, 1, NULL, NULL) == Q4LIN_ERR_INVALID_ARG, "null codes refused");
  CHECK(q4lin_linear(wq, sc, x, (uint16_t*)(uintptr_t)1032, 4, 128, 1, NULL, NULL) == Q4LIN_ERR_MISALIGNED,
        "misaligned y refused");
  CHECK(q4lin_linear(NULL, NULL, NULL, NULL, 0, 128, 5, NULL, NULL) == Q4LIN_OK, "empty problem is a no-op");
  CHECK(q4lin_linear_route(Q4LIN_ROUTE_TC_FP16, wq, sc, x, y, 64, 256, 8, NULL, NULL) == Q4LIN_ERR_WORKSPACE,
        "fp16 route without workspace refused");
  CHECK(q4lin_linear_qtype(9, wq, NULL, sc, x, y, 4, 128, 1, NULL, NULL) == Q4LIN_ERR_INVALID_ARG,
        "unknown format refused");
  CHECK(q4lin_linear_fp16_static(wq, sc, x, y, 256, 5120, 2048, NULL) == Q4LIN_ERR_UNSUPPORTED_SHAPE,
        "static-scratch entry refuses a shape beyond its array");
  CHECK(q4lin_linear_add(wq, sc, x, NULL, y, 64, 256, 8, NULL) == Q4LIN_ERR_INVALID_ARG,
        "LinearAdd without a residual refused");
  CHECK(q4lin_host_workspace_bytes(6144, 5120, 1) == (size_t)2 * 5120 + 2 * 6144,
        "host entry workspace: X and Y staging, 256-byte parts");
  CHECK(q4lin_linear_host(wq, sc, x, y, 64, 256, 4, NULL, NULL) == Q4LIN_ERR_WORKSPACE,
        "host entry without workspace refused");
  CHECK(q4lin_qtype_route(Q4LIN_QTYPE_Q5G64, 6144, 5120, 8) == Q4LIN_ROUTE_STREAM_MMA,
        "Q5 at 8 tokens: the warp-MMA route");
  CHECK(q4lin_fused_route(1, 6144, 5120, 8) == Q4LIN_ROUTE_STREAM_MMA &&
            q4lin_fused_route(1, 6144, 5120, 64) == Q4LIN_ROUTE_TC_SPLITK,
        "LinearAdd routes: one-launch warp-MMA form up to 8 tokens, tiles beyond");
  CHECK(strcmp(q4lin_status_string(Q4LIN_ERR_TIMEOUT), "unknown status") != 0, "status strings");
  CHECK(q4lin_version() != NULL && q4lin_version()[0] != 0, "version");
  return fails ? 1 : 0;
}
