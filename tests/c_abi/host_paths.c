/* A plain C caller of the library: links libpa.so through include/pa.h and
 * exercises the calls' host-side paths, which need no GPU (sizes, status
 * strings, partition sizes, and arguments refused before any launch).
 * Prints "ok" and exits 0 when every check holds; otherwise prints the first
 * failed check and exits 1. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "pa.h"

#define CHECK(cond)                                              \
  do {                                                           \
    if (!(cond)) {                                               \
      printf("failed: %s (line %d)\n", #cond, __LINE__);       \
      return 1;                                                  \
    }                                                            \
  } while (0)

int main(void) {
  /* Status strings name their codes. */
  CHECK(strcmp(pa_status_string(PA_OK), "PA_OK") == 0);
  CHECK(strcmp(pa_status_string(PA_ERR_INVALID_ARG), "PA_ERR_INVALID_ARG") == 0);
  CHECK(strcmp(pa_status_string(PA_ERR_TIMEOUT), "PA_ERR_TIMEOUT") == 0);

  /* Partition sizes are positive multiples of 32, and the workspace holds every
   * (sequence, head, partition)'s partial output (D floats) and (m, l) when a
   * context spans several partitions; a context that fits one partition needs
   * no partials. */
  static const int shapes[][4] = {{32, 40, 128, 1024}, {64, 40, 128, 1024}, {32, 40, 128, 4096},
                                  {256, 32, 128, 8192}, {4, 8, 64, 100}};
  for (int i = 0; i < 5; ++i) {
    const int S = shapes[i][0], H = shapes[i][1], D = shapes[i][2], c = shapes[i][3];
    const int p = pa_decode_partition_tokens(S, H, c);
    CHECK(p > 0 && p % 32 == 0);
    const size_t parts = (size_t)(c + p - 1) / p;
    const size_t w = pa_decode_workspace_size(S, H, D, c);
    if (parts > 1) CHECK(w >= (size_t)S * H * parts * ((size_t)D + 2) * 4);
    if (parts == 1) CHECK(w < (size_t)S * H * ((size_t)D + 2) * 4);
  }

  /* Bad arguments are refused before any CUDA call. */
  char buf[64] __attribute__((aligned(16)));
  void* d = buf;
  const int32_t* i32 = (const int32_t*)buf;
  CHECK(pa_decode(d, d, d, d, i32, 4, i32, 2, 2, 96, 16, 8, 0.1f, 64, d, 1 << 20, 0) ==
        PA_ERR_UNSUPPORTED); /* head_dim 96 */
  CHECK(pa_decode(d, d, d, d, i32, 4, i32, 2, 2, 128, 12, 8, 0.1f, 64, d, 1 << 20, 0) ==
        PA_ERR_UNSUPPORTED); /* block size 12 */
  CHECK(pa_decode(0, d, d, d, i32, 4, i32, 2, 2, 128, 16, 8, 0.1f, 64, d, 1 << 20, 0) ==
        PA_ERR_INVALID_ARG); /* null output */
  CHECK(pa_decode(d, d, d, d, i32, 4, i32, 2, 2, 128, 16, 8, 0.1f, 64, d, 16, 0) ==
        PA_ERR_INVALID_ARG); /* workspace too small */
  CHECK(pa_decode_ex(d, d, d, d, i32, 4, i32, 2, 2, 128, 16, 8, 0.1f, 64, d, 1 << 20, 0x4u, 0) ==
        PA_ERR_INVALID_ARG); /* unknown flag */
  CHECK(pa_decode(0, 0, 0, 0, 0, 4, 0, 0, 2, 128, 16, 8, 0.1f, 64, 0, 0, 0) == PA_OK); /* empty */
  CHECK(pa_prefill_ex(d, d, d, d, i32, 4, i32, i32, 2, 10, 2, 128, 16, 8, 0.1f, 8, -1, 0x1u, 0) ==
        PA_ERR_INVALID_ARG); /* unknown flag */
  CHECK(pa_prefill_ex(d, d, d, d, i32, 4, i32, i32, 2, 10, 2, 128, 16, 8, 0.1f, 8, 3, 0u, 0) ==
        PA_ERR_INVALID_ARG); /* more one-token sequences than sequences */
  CHECK(pa_prefill_fp8(d, d, d, d, i32, 4, i32, i32, 2, 10, 2, 128, 16, 8, 0.1f, 0.0f, 1.0f, 8,
                       0) == PA_ERR_INVALID_ARG); /* key scale 0 */
  printf("ok\n");
  return 0;
}
