/*
 * A plain C99 client of include/capattn.h, built with gcc and linked against
 * libcapattn.so by tests/test_c_abi.py.  It uses only the host-side calls
 * (no GPU needed): configuration checks, workspace sizing, tile sizes, status
 * strings, and the live-pair bits and visit map of a causal, windowed
 * configuration with a ranker mask.  It prints one line of key=value pairs
 * for the test to check against the oracle, then one status string.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "capattn.h"

static int popcount64(uint64_t x) {
  int n = 0;
  while (x) {
    x &= x - 1;
    ++n;
  }
  return n;
}

int main(int argc, char** argv) {
  if (argc != 5) {
    fprintf(stderr, "usage: %s L window hl,hu cl,cu\n", argv[0]);
    return 2;
  }
  const int L = atoi(argv[1]);
  const int window = atoi(argv[2]);
  int32_t bounds[4];
  if (sscanf(argv[3], "%d,%d", &bounds[0], &bounds[1]) != 2 ||
      sscanf(argv[4], "%d,%d", &bounds[2], &bounds[3]) != 2) {
    fprintf(stderr, "bad bounds\n");
    return 2;
  }

  capattn_config c;
  memset(&c, 0, sizeof c);
  c.struct_size = (uint32_t)sizeof c;
  c.cap_method = CAPATTN_CAP_TANH;
  c.cap = 50.0f;
  c.sm_scale = 0.125f;
  c.causal = 1;
  c.window_len = window;
  c.q_heads_per_kv_head = 2;
  c.B = 1;
  c.L = L;
  c.Hq = 4;
  c.Hkv = 2;
  c.D = 128;
  c.dtype = CAPATTN_BF16;

  const capattn_status ok = capattn_validate_config(&c);
  capattn_config bad = c;
  bad.Hq = 3; /* not a multiple of Hkv */
  const capattn_status st_bad = capattn_validate_config(&bad);
  bad = c;
  bad.D = 96;
  const capattn_status st_d96 = capattn_validate_config(&bad);

  int32_t bq = 0, bk = 0;
  if (capattn_tile_sizes(&c, &bq, &bk) != CAPATTN_OK) return 3;
  const size_t ws_fwd = capattn_workspace_bytes(&c, CAPATTN_PASS_FWD);
  const size_t ws_bwd = capattn_workspace_bytes(&c, CAPATTN_PASS_BWD);

  /* live pairs of batch row 0 */
  const size_t words = (size_t)L * (size_t)((L + 63) / 64);
  uint64_t* bits = (uint64_t*)calloc(words, sizeof(uint64_t));
  if (!bits) return 4;
  if (capattn_mask_bits_host(&c, NULL, bounds, 0, bits, words) != CAPATTN_OK) return 5;
  long live = 0;
  for (size_t w = 0; w < words; ++w) live += popcount64(bits[w]);
  free(bits);

  /* visited tile pairs (query-tile map) */
  size_t n_words = 0;
  const size_t cap_words = 1u << 20;
  uint32_t* map = (uint32_t*)calloc(cap_words, sizeof(uint32_t));
  if (!map) return 4;
  if (capattn_visit_map_host(&c, NULL, bounds, CAPATTN_VISIT_Q_TILES, map, cap_words, &n_words) !=
      CAPATTN_OK)
    return 6;
  long visited = 0;
  for (size_t w = 0; w < n_words; ++w) visited += popcount64(map[w]);
  free(map);

  /* a null workspace is rejected on the host, before any launch */
  const capattn_status st_ws =
      capattn_fwd(&c, (void*)16, (void*)16, (void*)16, NULL, NULL, NULL, (void*)16, (float*)16, NULL,
                  NULL, NULL, 0, (cudaStream_t)0);

  printf("ok=%d bad=%d d96=%d bq=%d bk=%d ws_fwd=%zu ws_bwd=%zu live=%ld visited=%ld ws_null=%d\n",
         (int)ok, (int)st_bad, (int)st_d96, bq, bk, ws_fwd, ws_bwd, live, visited, (int)st_ws);
  printf("%s\n", capattn_status_string(CAPATTN_ERR_WORKSPACE));
  return 0;
}
