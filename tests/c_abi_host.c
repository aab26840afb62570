/* Host-side use of the C ABI from plain C (C99, no CUDA headers, no Python): planning for the
 * 32K GQA shape over a bf16 and an FP8 cache, the plan's figures, argument errors caught before
 * anything is enqueued, and the host-only choice of phi. No call here reaches a GPU: the plans
 * are made for an explicit SM count. Prints one "key value" line per figure, then "ok". */
#include <stdio.h>
#include <string.h>

#include "decode_attn.h"

static int fail(const char* what, int rc) {
  printf("FAIL %s: %d %s\n", what, rc, decode_attn_strerror(rc));
  return 1;
}

static da_problem gqa_32k(void) {
  da_problem p;
  memset(&p, 0, sizeof p);
  p.batch = 1;
  p.num_q_heads = 32;
  p.num_kv_heads = 8;
  p.head_dim = 128;
  p.max_seq_len = 32768;
  p.qkv_dtype = DA_BF16;
  p.out_dtype = DA_BF16;
  p.mode = DA_SOFTMAX_UNIFIED;
  p.unified_max = -3.9f;
  p.range_lo = -64.f;
  p.range_hi = 64.f;
  p.num_sms = 152;
  return p;
}

int main(void) {
  if (decode_attn_abi_version() != DECODE_ATTN_ABI_VERSION) return fail("abi version", 0);

  for (int fp8 = 0; fp8 < 2; ++fp8) {
    da_problem p = gqa_32k();
    if (fp8) {
      p.kv_fp8 = 1;
      p.k_scale = 0.0128f;
      p.v_scale = 0.0126f;
    }
    da_plan* plan = NULL;
    size_t ws = 0;
    int rc = decode_attn_plan(&p, 0, &plan, &ws);
    if (rc != DA_OK) return fail("plan", rc);
    da_plan_info info;
    rc = decode_attn_plan_info(plan, &info);
    if (rc != DA_OK) return fail("plan_info", rc);
    if (info.workspace_bytes != ws) return fail("workspace bytes", 0);
    printf("%s grid_ctas %d stages %d stage_tokens %d workspace %zu smem %zu kv_heads %d\n",
           fp8 ? "fp8" : "bf16", info.grid_ctas, info.stages, info.stage_tokens,
           info.workspace_bytes, info.smem_bytes, info.kv_heads_per_group);
    /* a run with null inputs is refused on the host */
    rc = decode_attn_run(plan, NULL, NULL, NULL, NULL, NULL, 0.088f, -1, NULL, NULL, NULL, NULL,
                         0, NULL, NULL);
    if (rc != DA_ERR_INVALID_ARG) return fail("null run", rc);
    decode_attn_destroy(plan);
  }

  /* an FP8 cache with f16 q is not built */
  da_problem bad = gqa_32k();
  bad.kv_fp8 = 1;
  bad.k_scale = bad.v_scale = 1.f;
  bad.qkv_dtype = DA_F16;
  da_plan* plan = NULL;
  size_t ws = 0;
  int rc = decode_attn_plan(&bad, 0, &plan, &ws);
  if (rc != DA_ERR_UNSUPPORTED) return fail("fp8 with f16 q", rc);

  /* phi from a histogram: 4 bins of width 1 over [0, 4); coverage 0.5 keeps [1, 3) */
  const unsigned long long counts[6] = {1, 2, 10, 10, 3, 0};
  float phi = 0.f, x_lo = 0.f, x_hi = 0.f;
  rc = decode_attn_choose_phi(counts, 4, 0.f, 4.f, 0.5, 100.f, &phi, &x_lo, &x_hi);
  if (rc != DA_OK || phi != 1.f || x_lo != 1.f || x_hi != 3.f) return fail("choose_phi", rc);
  printf("phi %g x_lo %g x_hi %g\n", phi, x_lo, x_hi);
  rc = decode_attn_choose_phi(counts, 4, 0.f, 4.f, 0.5, 1.5f, &phi, &x_lo, &x_hi);
  if (rc != DA_ERR_RANGE_TOO_WIDE) return fail("choose_phi width", rc);
  printf("ok\n");
  return 0;
}
