/*
 * A plain C11 client of the C ABI in include/gdn.h: no C++, no CUDA headers, only the shared
 * library.  It sizes workspaces, names every error code and drives the argument checks of the
 * compute entry points with calls that are refused before anything is enqueued (fake, never
 * dereferenced pointers).  Output: one "key value" line per check, read by test_c_client.py.
 */
#include <stdint.h>
#include <stdio.h>

#include "gdn.h"

int main(void) {
  void* fake = (void*)(uintptr_t)0x100000; /* aligned, non-NULL, never dereferenced */
  const int32_t* ifake = (const int32_t*)fake;
  gdn_layer_desc layer = {16, 32, 128, 128, 4, 6, GDN_BF16, 0.0f, GDN_QKV_PACKED, GDN_CONV_ROLLED};
  gdn_layer_params params = {fake, NULL, (const float*)fake, (const float*)fake};
  gdn_pools pools = {fake, (float*)fake, 512};
  gdn_rows spec = {64, 256, ifake, NULL, NULL, NULL, ifake, ifake, 4};
  gdn_rows non_spec = {8, 8, ifake, ifake, ifake, NULL, NULL, NULL, 0};
  gdn_rows prefill = {1, 8192, ifake, NULL, ifake, NULL, NULL, NULL, 0};

  printf("ws_spec %zu\n", gdn_workspace_bytes(&layer, NULL, &spec));
  printf("ws_mixed %zu\n", gdn_workspace_bytes(&layer, &non_spec, &spec));
  printf("ws_prefill %zu\n", gdn_prefill_workspace_bytes(&layer, &prefill, 1));
  for (int code = 0; code >= -8; --code) printf("status%d %s\n", -code, gdn_status_string(code));

  /* refused calls */
  printf("mixed_null %d\n",
         gdn_mixed_batch(NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL, 0, 0, NULL, NULL, NULL, 0, NULL, NULL));
  gdn_rows spec_no_acc = spec;
  spec_no_acc.num_accepted_tokens = NULL;
  printf("conv_spec_pair %d\n",
         gdn_conv_update(&layer, &params, &pools, fake, 256, &spec_no_acc, fake, GDN_F32, NULL, NULL));
  printf("conv_dtype %d\n", gdn_conv_update(&layer, &params, &pools, fake, 256, &spec, fake, (gdn_dtype)9, NULL, NULL));
  printf("recurrent_align %d\n", gdn_recurrent_step(&layer, &params, &pools, (const char*)fake + 4, GDN_F32, fake,
                                                     fake, 256, &spec, fake, NULL, NULL));
  printf("prefill_chunk %d\n", gdn_chunk_prefill(&layer, &params, &pools, fake, GDN_F32, fake, fake, 8192, &prefill,
                                                 32, fake, fake, (size_t)1 << 40, NULL, NULL));
  gdn_layer_desc bad = layer;
  bad.head_k_dim = 48;
  spec.token_indx = ifake;
  non_spec.token_indx = ifake;
  printf("mixed_shape %d\n", gdn_mixed_batch(&bad, &params, &pools, fake, fake, fake, 264, &non_spec, 8, 0, &spec,
                                             fake, fake, (size_t)1 << 40, NULL, NULL));
  printf("mixed_conservation %d\n", gdn_mixed_batch(&layer, &params, &pools, fake, fake, fake, 263, &non_spec, 8, 0,
                                                    &spec, fake, fake, (size_t)1 << 40, NULL, NULL));
  printf("mixed_workspace %d\n", gdn_mixed_batch(&layer, &params, &pools, fake, fake, fake, 264, &non_spec, 8, 0,
                                                 &spec, fake, fake, 16, NULL, NULL));
  return 0;
}
