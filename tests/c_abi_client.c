/* A plain C99 client of include/attn_train.h: built and run by
 * tests/test_abi_cpu.py on the CPU (no GPU needed: it calls only the host-side
 * validation and sizing entry points).  Exit status 0 = every check held. */
#include <stdio.h>
#include <string.h>

#include "attn_train.h"

static int fails = 0;
#define CHECK(cond)                                          \
  do {                                                       \
    if (!(cond)) {                                           \
      fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
      ++fails;                                               \
    }                                                        \
  } while (0)

int main(void) {
  attn_problem p;
  memset(&p, 0, sizeof(p));
  p.B = 1; p.Hq = 32; p.Hkv = 4; p.Sq = 16384; p.Skv = 16384; p.D = 128;
  p.mask = ATTN_MASK_CAUSAL; p.out_dtype = ATTN_OUT_F32;
  CHECK(attn_train_supports(&p) == ATTN_OK);
  {
    char desc[4096];
    size_t need = 0;
    CHECK(attn_train_describe(&p, NULL, 0, &need) == ATTN_ERR_INVALID && need > 1);
    CHECK(attn_train_describe(&p, desc, sizeof(desc), &need) == ATTN_OK);
    CHECK(strlen(desc) + 1 == need && strstr(desc, "\"bwd_dkdv\"") != NULL);
  }

  size_t ws = 0;
  CHECK(attn_train_workspace_size(&p, &ws) == ATTN_OK);
  CHECK(ws == (size_t)32 * 16384 * 4);

  size_t arena = 0;
  CHECK(attn_train_step_host_arena_size(&p, 0, &arena) == ATTN_OK && arena > ws);
  {
    size_t two = 0, four = 0;
    CHECK(attn_train_host_session_arena_size(&p, 0, 2, &two) == ATTN_OK && two == arena);
    CHECK(attn_train_host_session_arena_size(&p, 0, 4, &four) == ATTN_OK && four > two);
    CHECK(attn_train_host_session_arena_size(&p, 0, ATTN_HOST_MAX_SLOTS + 1, &four) ==
          ATTN_ERR_INVALID);
  }

  p.D = 96;  /* unsupported head dim: a status and a message, no fallback */
  CHECK(attn_train_supports(&p) == ATTN_ERR_UNSUPPORTED);
  CHECK(strstr(attn_train_last_error(), "head dim") != NULL);

  p.D = 64; p.mask = ATTN_MASK_TTT; p.ttt_step = 2; p.Skv = 3 * p.Sq;
  CHECK(attn_train_supports(&p) == ATTN_OK);
  p.Skv = 2 * p.Sq;  /* TTT needs Skv == (t + 1) Sq */
  CHECK(attn_train_supports(&p) == ATTN_ERR_INVALID);

  CHECK(attn_train_supports(NULL) == ATTN_ERR_INVALID);
  CHECK(attn_train_logsoftmax_loss_fwd(0, 10, NULL, 10, NULL, 10, NULL, NULL, NULL, NULL, NULL,
                                       NULL) == ATTN_ERR_INVALID);
  if (fails == 0) printf("c abi ok\n");
  return fails == 0 ? 0 : 1;
}
