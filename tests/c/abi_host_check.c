/* A plain C client of include/qgemm.h (no Python, no PyTorch): it links
 * libqgemm.so and exercises the calls that need no GPU -- version, sizes,
 * workspace and launch-count queries, and argument validation, which rejects
 * bad requests on the host before any launch. Prints one line per check and
 * returns the number of failures. Valid C99 and C++. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "qgemm.h"

static int failures = 0;

static void check(int ok, const char* what) {
  printf("%s %s\n", ok ? "ok  " : "FAIL", what);
  if (!ok) ++failures;
}

int main(void) {
  check(qg_version() == 10000, "qg_version");
  check(qg_small_m_max() == 16, "qg_small_m_max");
  check(strncmp(qg_status_string(QG_EINVAL), "QG_EINVAL", 9) == 0, "qg_status_string");

  /* packed sizes: 256-byte multiples holding at least the stream, scales and fp16 copy */
  const size_t b8 = qg_q8_0_packed_bytes(9728, 2560);
  check(b8 % 256 == 0 && b8 >= (size_t)9728 * 2560 * 3, "qg_q8_0_packed_bytes");
  check(qg_q8_0_packed_bytes(16, 48) == 0, "qg_q8_0_packed_bytes rejects K % 32");
  check(qg_q4k_packed_bytes(16, 128) == 0, "qg_q4k_packed_bytes rejects K % 256");

  /* workspace of the layer call: scales + int8 activations (M <= 16) */
  check(qg_linear_workspace_bytes(0, 1, 5120) == 256 + 5120, "qg_linear_workspace_bytes");
  check(qg_gemm_launch_count(0, 40, 5120, 17408, QG_PATH_SMALL) == 3, "qg_gemm_launch_count");

  /* validation happens before any launch: null and misaligned arguments */
  void* fake = (void*)(uintptr_t)0x10000;
  check(qg_gemm_w8a8_q8_0(NULL, NULL, NULL, 4, 256, fake, 16, fake, QG_BF16, 16, NULL) ==
            QG_EINVAL,
        "qg_gemm_w8a8_q8_0 rejects a null scale");
  check(strlen(qg_last_error()) > 0, "qg_last_error holds a reason");
  check(qg_quantize_act(fake, QG_BF16, 4, 64, 68, (int8_t*)fake, (float*)fake, NULL, NULL,
                        NULL) == QG_EALIGN,
        "qg_quantize_act rejects a row stride that is not a multiple of 16 bytes");
  check(qg_linear_w8a8_q8_0(fake, QG_BF16, 4, 256, 256, fake, 16, fake, QG_BF16, 16, NULL,
                            NULL, 0, NULL) == QG_EINVAL,
        "qg_linear_w8a8_q8_0 requires its workspace");
  check(qg_pack_q4k(fake, 4, 128, fake, NULL) == QG_EINVAL, "qg_pack_q4k rejects K % 256");

  printf("%d failure(s)\n", failures);
  return failures;
}
