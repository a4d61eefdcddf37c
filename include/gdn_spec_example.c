/*
 * gdn_spec_example.c -- one decode step of one GDN layer through the C ABI of
 * libgdnspec (include/gdn_spec.h): verify the draft window, commit the accepted
 * tokens, fold the rows whose ring is nearly full, and read the device status.
 *
 * Every pointer is caller-owned device memory of the current CUDA device; no
 * call allocates, and the three calls are ordered on `stream`, so the step can
 * be captured in a CUDA graph.  Host-only example: compiles against the header
 * alone (link libgdnspec.so to run it).
 */
#include <stdint.h>
#include <stdio.h>

#include "gdn_spec.h"

int gdn_spec_example_step(int32_t slots, float *ckpt, void *rawv, void *rawk, float *ring_g,
                          float *ring_beta, int32_t *write_pos, int32_t *cache_base,
                          int32_t *is_flush, uint32_t *status, const int32_t *slot_idx, int32_t B,
                          const void *q, const void *k, const void *v, const void *a,
                          const void *b, const float *A_log, const float *dt_bias, void *out,
                          const int32_t *accept_len, void *stream)
{
    /* the Qwen3-Next-shaped layer: 16 q/k heads, 32 v-heads, K = V = 128, a
       window of 4 draft tokens, a ring of 64 records per slot */
    gdn_spec_layer layer = {.H = 16, .HV = 32, .K = 128, .V = 128, .T = 4, .L = 64,
                            .num_slots = slots, .gate_kind = GDN_SPEC_GATE_SCALAR,
                            .io_dtype = GDN_SPEC_DTYPE_BF16, .scale = 1.0f, .l2_eps = 1e-6f,
                            .checkpoint = ckpt, .rawv = rawv, .rawk = rawk,
                            .ring_g = ring_g, .ring_beta = ring_beta};
    gdn_spec_cursors cur = {slots, write_pos, cache_base, is_flush, status};

    /* outputs of the whole draft window; the window's raw records go into the ring */
    int rc = gdn_spec_verify(&layer, &cur, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, stream);
    /* accept_len is produced on the device by the sampler */
    if (!rc) rc = gdn_spec_commit(&cur, layer.T, layer.L, slot_idx, B, accept_len, stream);
    /* folds every layer's flagged rows exactly, then moves the cursors once */
    if (!rc) rc = gdn_spec_fold(&layer, 1, &cur, slot_idx, B, stream);
    if (rc) {
        fprintf(stderr, "%s\n", gdn_spec_strerror(rc));
        return rc;
    }
    /* conditions only the device sees (slot out of range, ring overflow, ...) set
       status bits; reading them synchronises the stream */
    uint32_t st = 0;
    rc = gdn_spec_read_status(&cur, &st, /*clear=*/1, stream);
    if (!rc && st) fprintf(stderr, "device status 0x%x\n", st);
    return rc;
}
