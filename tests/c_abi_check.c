/* The C ABI used from plain C99, with no Python in between.
 *
 * Both headers must compile as strict C.  The program prints the struct
 * layouts so that a test can compare them with the Python binding's ctypes
 * structures.  It then runs the host-only entry points (version, schedule,
 * workspace sizes, status strings) and the argument checks, which refuse
 * bad calls before any CUDA call, so it needs no GPU.
 *
 * Output: one "key value" pair per line.  Exit status 0 on success, else
 * the number of the failed step.
 */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "csbp.h"
#include "csbp_vocab_ce.h"

#define LAYOUT(type, field) \
  printf("offset %s.%s %zu\n", #type, #field, offsetof(type, field))

int main(void) {
  csbp_problem p = {0};
  csbp_schedule_info info;
  csbp_inputs in = {0};
  csbp_ce_problem ce = {0};
  int32_t owner[32];
  int32_t chunk[4];
  void* work;
  csbp_status st;

  printf("version %d\n", (int)csbp_version());
  printf("sizeof csbp_problem %zu\n", sizeof(csbp_problem));
  LAYOUT(csbp_problem, scale);
  LAYOUT(csbp_problem, window);
  LAYOUT(csbp_problem, bwd_chunk);
  LAYOUT(csbp_problem, per_rank);
  LAYOUT(csbp_problem, rank);
  printf("sizeof csbp_inputs %zu\n", sizeof(csbp_inputs));
  LAYOUT(csbp_inputs, v_corr);
  LAYOUT(csbp_inputs, stride_tok);
  LAYOUT(csbp_inputs, stride_batch);
  printf("sizeof csbp_schedule_info %zu\n", sizeof(csbp_schedule_info));
  LAYOUT(csbp_schedule_info, tile_pairs);
  LAYOUT(csbp_schedule_info, bytes);
  LAYOUT(csbp_schedule_info, problem_key);
  printf("sizeof csbp_ce_problem %zu\n", sizeof(csbp_ce_problem));
  LAYOUT(csbp_ce_problem, d_model);
  LAYOUT(csbp_ce_problem, grad_scale);

  /* L = 1024 in blocks of 32 on P = 2 virtual shards: 32 blocks, 4 chunks */
  p.batch = 1;
  p.L = 1024;
  p.M = 32;
  p.Hq = 4;
  p.Hkv = 2;
  p.d = 128;
  p.P = 2;
  p.tile_q = 128;
  p.tile_kv = 128;
  p.has_clean_queries = 1;
  p.scale = 0.08838834764831845f;
  st = csbp_block_schedule(&p, owner, chunk, NULL, 0, &info);
  if (st != CSBP_ERR_CAPACITY) return 1;
  work = malloc((size_t)info.bytes);
  if (!work) return 2;
  st = csbp_block_schedule(&p, owner, chunk, work, info.bytes, &info);
  free(work);
  if (st != CSBP_OK) return 3;
  printf("tile_pairs %lld\n", (long long)info.tile_pairs);
  printf("owner_first_last %d %d\n", (int)owner[0], (int)owner[31]);
  printf("chunk_owner %d %d %d %d\n", (int)chunk[0], (int)chunk[1], (int)chunk[2],
         (int)chunk[3]);
  printf("fwd_workspace %zu\n", csbp_workspace_bytes(&p, 0));
  printf("bwd_workspace %zu\n", csbp_workspace_bytes(&p, 1));
  printf("status_workspace %s\n", csbp_status_string(CSBP_ERR_WORKSPACE));

  /* refused before anything is enqueued: no inputs, then a bad stride */
  st = csbp_attn_fwd(&p, &in, NULL, &info, NULL, NULL, NULL, NULL, 0, NULL);
  printf("fwd_without_inputs %d\n", (int)st);
  in.q_clean = in.k_clean = in.v_clean = (const void*)(uintptr_t)0x10000;
  in.q_corr = in.k_corr = in.v_corr = (const void*)(uintptr_t)0x10000;
  in.stride_tok[1] = 100; /* below Hkv * d and not a multiple of 8 */
  st = csbp_attn_fwd(&p, &in, (const void*)(uintptr_t)0x10000, &info,
                     (void*)(uintptr_t)0x10000, (void*)(uintptr_t)0x10000,
                     (float*)(uintptr_t)0x10000, (void*)(uintptr_t)0x10000, 1 << 30, NULL);
  printf("fwd_bad_stride %d\n", (int)st);
  /* the list was built for L = 1024: a problem of another length refuses it */
  in.stride_tok[1] = 0;
  p.L = 2048;
  st = csbp_attn_fwd(&p, &in, (const void*)(uintptr_t)0x10000, &info,
                     (void*)(uintptr_t)0x10000, (void*)(uintptr_t)0x10000,
                     (float*)(uintptr_t)0x10000, (void*)(uintptr_t)0x10000, 16, NULL);
  printf("fwd_other_problem %d\n", (int)st);
  p.L = 1024;
  st = csbp_attn_fwd(&p, &in, (const void*)(uintptr_t)0x10000, &info,
                     (void*)(uintptr_t)0x10000, (void*)(uintptr_t)0x10000,
                     (float*)(uintptr_t)0x10000, (void*)(uintptr_t)0x10000, 16, NULL);
  printf("fwd_small_workspace %d\n", (int)st);

  ce.rows = 1000;
  ce.d_model = 256;
  ce.vocab = 4096;
  ce.head_grad = 1;
  ce.grad_scale = 0.001f;
  printf("ce_workspace %zu\n", csbp_ce_workspace_bytes(&ce));
  ce.vocab = 100; /* not a multiple of 64 */
  printf("ce_workspace_invalid %zu\n", csbp_ce_workspace_bytes(&ce));

  /* one CSBP rank's rows: needs P > 1 and a rank below P */
  p.per_rank = 1;
  p.rank = 1;
  st = csbp_block_schedule(&p, NULL, NULL, NULL, 0, &info);
  printf("rank_size_query %d\n", (int)st);
  p.rank = 2;
  printf("rank_out_of_range %d\n", (int)csbp_block_schedule(&p, NULL, NULL, NULL, 0, &info));
  p.per_rank = 0;
  p.rank = 0;

  /* fp8 decode: arguments are checked before any CUDA call; n = 0 is a no-op */
  {
    static unsigned char bytes[32] __attribute__((aligned(16)));
    static unsigned short out[32] __attribute__((aligned(16)));
    printf("e4m3_null %d\n", (int)csbp_e4m3_to_bf16(NULL, 1.0f, out, 16, NULL));
    printf("e4m3_zero_scale %d\n", (int)csbp_e4m3_to_bf16(bytes, 0.0f, out, 16, NULL));
    printf("e4m3_misaligned %d\n", (int)csbp_e4m3_to_bf16(bytes + 1, 1.0f, out, 16, NULL));
    printf("e4m3_empty %d\n", (int)csbp_e4m3_to_bf16(bytes, 1.0f, out, 0, NULL));
  }
  return 0;
}
