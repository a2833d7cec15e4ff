/*
 * c_client.c -- the C ABI used from plain C, without Python or torch.
 *
 * Validates a configuration and prints the buffer sizes a caller has to
 * allocate for one Qwen3-8B-shaped layer (128 requests x 16K tokens, 32 query
 * heads / 8 KV heads, K = 128, fetch ratio 0.05), then checks that a bad
 * configuration is refused with a message.  Needs no GPU: these two calls
 * only do host arithmetic.
 *
 *   cc -I include sparse_kv_block_gb300/examples/c_client.c \
 *      -L sparse_kv_block_gb300 -loasis -Wl,-rpath,sparse_kv_block_gb300 -o c_client
 */
#include <stdio.h>
#include <string.h>

#include "oasis.h"

int main(void) {
  oasis_config cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.num_layers = 1;
  cfg.num_requests = 128;
  cfg.max_blocks = 1024;
  cfg.num_q_heads = 32;
  cfg.num_kv_heads = 8;
  cfg.head_dim = 128;
  cfg.block_size = 16;
  cfg.topk = 128;
  cfg.fetch_ratio = 0.05f;

  const char* err = oasis_config_error(&cfg);
  if (err) {
    printf("config rejected: %s\n", err);
    return 1;
  }
  oasis_sizes s;
  if (oasis_query_sizes(&cfg, &s) != OASIS_OK) return 2;
  printf("fetch_cap %d units_per_head %d\n", s.fetch_cap, s.units_per_head);
  printf("kv_pool_bytes %zu summaries_bytes %zu host_kv_bytes %zu\n", s.kv_pool_bytes,
         s.summaries_bytes, s.host_kv_bytes);
  printf("res_ids_bytes %zu stamps_bytes %zu phys_bytes %zu ctx_len_bytes %zu workspace_bytes %zu\n",
         s.res_ids_bytes, s.stamps_bytes, s.phys_bytes, s.ctx_len_bytes, s.workspace_bytes);

  cfg.head_dim = 64;
  err = oasis_config_error(&cfg);
  if (!err || oasis_query_sizes(&cfg, &s) != OASIS_EINVAL) return 3;
  printf("refused: %s\n", err);
  return 0;
}
