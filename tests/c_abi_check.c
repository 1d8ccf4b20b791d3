/* The C ABI of libkvq.so used from plain C (C11, no C++): every function the
 * header declares is referenced, and the calls that need no GPU run here --
 * status strings, the version, workspace sizes, and the host-side rejection of
 * invalid arguments before any device work.  Prints one "ok" line per check
 * and exits non-zero at the first failure. */
#include "kvq.h"

#include <stdint.h>
#include <stdio.h>
#include <string.h>

#define CHECK(cond)                                                   \
  do {                                                                \
    if (!(cond)) {                                                    \
      printf("FAIL line %d: %s (%s)\n", __LINE__, #cond, kvq_last_error()); \
      return 1;                                                       \
    }                                                                 \
    printf("ok %s\n", #cond);                                         \
  } while (0)

/* The address of every declared function: a missing export fails the link.
 * (Function pointers convert to one another in ISO C, not to void*.) */
typedef void (*any_fn)(void);
static const any_fn kAll[] = {
    (any_fn)&kv_quant_append,        (any_fn)&attn_decode,
    (any_fn)&attn_decode_append,     (any_fn)&attn_prefill_append,
    (any_fn)&attn_train_donor_forward, (any_fn)&kvq_profile_next_read,
    (any_fn)&attn_decode_workspace_bytes, (any_fn)&attn_prefill_chunk,
    (any_fn)&attn_prefill_workspace_bytes, (any_fn)&attn_mixed,
    (any_fn)&attn_mixed_schedule,
    (any_fn)&attn_decode_static,     (any_fn)&kvq_static_status,
    (any_fn)&kvq_selftest_wait_timeout, (any_fn)&kvq_train_kv_prep,
    (any_fn)&attn_train_forward,     (any_fn)&attn_train_workspace_bytes,
    (any_fn)&kvq_status_string,      (any_fn)&kvq_last_error,
    (any_fn)&kvq_version,
};

int main(void) {
  for (size_t i = 0; i < sizeof kAll / sizeof kAll[0]; ++i) CHECK(kAll[i] != NULL);
  CHECK(kvq_version() >= 100);
  CHECK(strcmp(kvq_status_string(KVQ_OK), "ok") == 0);
  CHECK(strcmp(kvq_status_string(KVQ_EINVAL), kvq_status_string(KVQ_EWORKSPACE)) != 0);

  /* 8 q heads over 2 kv heads, head_dim 256, window 512, full RoPE */
  kvq_layer L;
  memset(&L, 0, sizeof L);
  L.n_q_heads = 8;
  L.n_kv_heads = 2;
  L.head_dim = 256;
  L.group_size = 64;
  L.window = 512;
  L.rope_dims = 256;
  L.rope_theta = 1e4;
  L.rms_eps = 1e-6f;
  L.k_eq_v = 0;
  CHECK(attn_decode_workspace_bytes(&L, 4, 1000) > 0);
  CHECK(attn_decode_workspace_bytes(&L, 4, 1 << 24) == 0);
  CHECK(attn_prefill_workspace_bytes(&L, 2, 64, 32) > 0);

  /* invalid calls are refused on the host; no pointer below is dereferenced */
  CHECK(attn_decode(&L, NULL, 1, NULL, 10, NULL, NULL, NULL, 1, NULL, NULL, 0, NULL) == KVQ_EINVAL);
  CHECK(strlen(kvq_last_error()) > 0);
  CHECK(attn_decode(NULL, NULL, 1, NULL, 10, NULL, NULL, NULL, 1, NULL, NULL, 0, NULL) == KVQ_EINVAL);
  CHECK(attn_decode_append(&L, NULL, 1, NULL, -1, NULL, NULL, NULL, NULL, NULL, NULL, 1, NULL, NULL, NULL, 0,
                           NULL) == KVQ_EINVAL);
  kvq_layer bad = L;
  bad.head_dim = 96;
  CHECK(kv_quant_append(&bad, NULL, 1, NULL, NULL, 1, NULL, NULL, NULL, NULL, NULL) == KVQ_EUNSUPPORTED);
  bad = L;
  bad.group_size = 32;
  /* row_offsets is checked first: give it an aligned address that the failed
   * layer check keeps from being read */
  const int32_t* fake_offsets = (const int32_t*)(uintptr_t)0x100000u;
  CHECK(attn_prefill_chunk(&bad, NULL, 1, fake_offsets, NULL, 4, 4, NULL, NULL, NULL, 1, NULL, NULL, 0, NULL) ==
        KVQ_EUNSUPPORTED);
  CHECK(attn_mixed(&L, NULL, KVQ_MAX_MIXED_GROUPS + 1, NULL, 1, NULL) == KVQ_EINVAL);
  {
    uint32_t mask = 7;
    CHECK(attn_mixed_schedule(&L, NULL, 0, NULL, 1, &mask) == KVQ_OK && mask == 0);
    CHECK(attn_mixed_schedule(&L, NULL, 0, NULL, 1, NULL) == KVQ_EINVAL);
  }
  CHECK(attn_decode_static(&L, NULL, 1, NULL, -1, NULL, NULL, NULL, 1, NULL, NULL) == KVQ_EINVAL);
  CHECK(kvq_selftest_wait_timeout(NULL, 1000000, NULL) == KVQ_EINVAL);
  CHECK(kvq_static_status(NULL, NULL) == KVQ_EINVAL);
  CHECK(kvq_profile_next_read((void*)&L, NULL) == KVQ_EINVAL);
  CHECK(kvq_profile_next_read(NULL, NULL) == KVQ_OK);
  CHECK((KVQ_STATUS_WAIT_TIMEOUT & KVQ_STATUS_SEQ_SKIPPED) == 0);
  CHECK(attn_train_workspace_bytes(&L, 100) == 256 + 100u * 8u * 256u * 2u);
  CHECK(attn_train_forward(&L, 0, fake_offsets, 4, 4, NULL, NULL, NULL, NULL, NULL, 1, NULL, NULL, 0, NULL) ==
        KVQ_EINVAL);
  CHECK(kvq_train_kv_prep(&L, 1, NULL, 4, NULL, NULL, NULL, NULL, NULL, NULL) == KVQ_EINVAL);
  /* nothing to do is not an error */
  CHECK(kvq_train_kv_prep(&L, 1, fake_offsets, 0, NULL, NULL, NULL, NULL, NULL, NULL) == KVQ_OK);
  CHECK(kv_quant_append(&L, NULL, 0, NULL, NULL, 0, NULL, NULL, NULL, NULL, NULL) == KVQ_OK);
  printf("all checks passed\n");
  return 0;
}
