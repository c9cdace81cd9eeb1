/* A plain C99 consumer of the C ABI: compiled against include/dpp.h and linked with
 * libdpp.so by tests/test_abi.py.  It calls only functions that check their arguments
 * on the host (no GPU is needed) and prints the struct sizes the caller's compiler sees,
 * which the test compares with the Python binding's. */
#include <stdio.h>
#include <string.h>

#include "dpp.h"

static int fails = 0;
#define EXPECT(cond)                                            \
  do {                                                          \
    if (!(cond)) {                                              \
      fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__); \
      ++fails;                                                  \
    }                                                           \
  } while (0)

int main(void) {
  dpp_layer_params p;
  memset(&p, 0, sizeof p);
  p.B = 2; p.H = 64; p.W = 64; p.C = 640; p.P = 4; p.G = 32; p.heads = 10;
  p.head_dim = 64; p.dtype = DPP_BF16; p.refresh = 1; p.eps = 1e-5f;
  EXPECT(dpp_version() >= 100);
  EXPECT(strcmp(dpp_status_string(DPP_OK), "ok") == 0);
  dpp_workspace_layout lo;
  EXPECT(dpp_workspace_query(&p, &lo) == DPP_OK);
  EXPECT(lo.total == dpp_workspace_size(&p) && lo.total > 0);
  EXPECT(lo.y % 256 == 0 && lo.h > lo.y && lo.attn_partial >= lo.o);
  EXPECT(dpp_message_elems(&p) == 2LL * 2 * 4096 * 640 + 2LL * 3 * 2 * 64 * 640);
  EXPECT(dpp_message_blocks(&p) == dpp_message_elems(&p) / 128);
  dpp_layer_params bad = p;
  bad.H = 63;
  EXPECT(dpp_workspace_size(&bad) == 0);
  bad = p;
  bad.gn_mode = 7;
  EXPECT(dpp_workspace_query(&bad, &lo) == DPP_ERR_ARG);
  /* null pointers are refused before any launch */
  dpp_layer_weights w;
  dpp_layer_state st;
  memset(&w, 0, sizeof w);
  memset(&st, 0, sizeof st);
  EXPECT(patch_layer_step(&p, &w, &st, NULL, NULL, DPP_STALE, NULL, NULL) == DPP_ERR_NULL);
  EXPECT(refresh_residual(NULL, NULL, NULL, NULL, 0, DPP_BF16, NULL) == DPP_OK);
  EXPECT(refresh_residual(NULL, NULL, NULL, NULL, 5, DPP_BF16, NULL) == DPP_ERR_NULL);
  printf("sizes %zu %zu %zu %zu\n", sizeof(dpp_layer_params), sizeof(dpp_layer_weights),
         sizeof(dpp_layer_state), sizeof(dpp_workspace_layout));
  return fails ? 1 : 0;
}
