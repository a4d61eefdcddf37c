/*
 * gdn_spec.h -- C ABI of libgdnspec: ReplaySSM ring spec-verify for one
 * Gated DeltaNet (GDN) linear-attention layer, and its KDA variant (one gate
 * per key channel), on a single GB300 GPU (sm_103a).
 *
 * Sources (web pages, cited by title and section):
 *   [blog]    "PR #28695 详解：GDN ReplaySSM Ring Spec-Verify" (yuyanqi.com)
 *   [pr28695] prhub summary of sglang PR #28695 "[GDN] Support ReplaySSM Ring
 *             Spec-Verify"
 *   [pr33102] prhub report of sglang PR #33102 "fused replayssm ring write into
 *             flashinfer gdn mtp verify kernel"
 *   [pr36821] prhub summary of sglang PR #36821 (fused KDA verify with the
 *             ReplaySSM ring write)
 *
 * The layer keeps, per cache slot (one slot per request):
 *   - a frozen fp32 checkpoint state S0                  [num_slots, HV, V, K]
 *   - a ring of L raw records of committed and draft tokens:
 *       rawv [num_slots, HV, L, V], rawk [num_slots, H, L, K] (I/O dtype,
 *       bitwise copies of the inputs, k before its L2 norm), g and beta fp32
 *       ([blog] appendix A.1; [pr36821] ring layout; [pr33102] test anchor 2)
 *   - three cursors shared by all layers of the model ([blog] §4.1, §10.2):
 *       write_pos  committed-but-unfolded records in the ring,
 *       cache_base ring position of the oldest of them,
 *       is_flush   set by commit when the next window might not fit.
 * Record o (0 <= o < write_pos) sits at ring position (cache_base + o) & (L-1);
 * the draft window of a verify is written at (cache_base + write_pos + s) &
 * (L-1), s < T ([blog] §10.1).
 *
 * The recurrence (decay, then delta against the decayed state; [blog] §12.1):
 *   g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b)
 *   k^ = k / sqrt(|k|^2 + l2_eps), q^ likewise
 *   S_t = exp(g_t) S_{t-1} (I - beta_t k^_t k^_t^T) + beta_t v_t k^_t^T
 *         (KDA: S_{t-1} diag(exp(g_t)) in place of exp(g_t) S_{t-1})
 *   o_t = scale * S_t q^_t
 *
 * Calls and their order per decode step: gdn_spec_verify once per layer
 * inside the forward; after sampling, gdn_spec_commit once; then
 * gdn_spec_fold once over all layers (it does work only for slots whose
 * is_flush was set).  gdn_spec_reset at the prefill -> decode handoff.
 *
 * Conventions for every call:
 *   - All tensor pointers are caller-owned DEVICE memory of the current CUDA
 *     device; the library never allocates, frees or copies them, and keeps no
 *     pointer after the call returns.  Descriptor structs are read on the
 *     host during the call only.
 *   - Tensors are dense, row-major in the shapes given, base addresses 16-byte
 *     aligned.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t, passed
 *     as void*; NULL is the legacy default stream).  They do not synchronise
 *     and do not allocate, so they can be captured into a CUDA graph, except
 *     gdn_spec_read_status, which synchronises.
 *   - Slots named in one call must be distinct; `slot_idx[b] < 0` marks a
 *     padding row, which reads and writes nothing (verify writes zeros to
 *     its output rows).
 *   - Return value: 0 on success, a negative GDN_SPEC_E* code for an error
 *     the host can see (nothing is launched then).  Conditions only the
 *     device can see never trap: the kernel ORs a GDN_SPEC_ST_* bit into
 *     *status, skips the row, and verify writes zeros to its outputs.
 */
#ifndef GDN_SPEC_H
#define GDN_SPEC_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_SPEC_ABI_VERSION 4   /* 2: adds gdn_spec_prefill and the snapshot comparison calls;
                                    3: adds gdn_spec_verify_d, gdn_spec_set_wait_limit, commit's
                                       cursor check and the poisoning of rows a fold or prefill
                                       could not finish;
                                    4: adds gdn_spec_prefill_path, the chunk-parallel prefill and
                                       the tensor-core KDA verify ("tc_kda") */

/* host-side error codes (return values) */
#define GDN_SPEC_OK            0
#define GDN_SPEC_EINVAL       -1   /* null pointer, bad size, L not a power of two or L < 2T, H does not divide HV */
#define GDN_SPEC_EDTYPE       -2   /* unknown io_dtype or gate_kind */
#define GDN_SPEC_EALIGN       -3   /* a base pointer not 16-byte aligned, or K / V not a multiple of 8 */
#define GDN_SPEC_ECUDA        -4   /* a CUDA call or launch failed */
#define GDN_SPEC_EUNSUPPORTED -5   /* shape outside what the kernels handle (see gdn_spec_verify) */

/* device-side status bits, ORed into cursors->status */
#define GDN_SPEC_ST_ACCEPT_RANGE   1u  /* commit: accept_len < 0 or > T                  */
#define GDN_SPEC_ST_SLOT_OOR       2u  /* slot_idx[b] >= num_slots                        */
#define GDN_SPEC_ST_RING_OVERFLOW  4u  /* verify: write_pos + T > L (a fold was skipped)  */
#define GDN_SPEC_ST_CURSOR_CORRUPT 8u  /* write_pos < 0, write_pos > L or cache_base outside [0, L) */
#define GDN_SPEC_ST_TIMEOUT       16u  /* a bounded device wait ran out: that call's outputs are invalid.
                                              verify: the CTA that saw it drains its copies and stops, so
                                              rows it had not reached keep whatever `out` held and their
                                              window records may be missing from the ring (do not commit
                                              that step).  fold / prefill: every row with an unfinished
                                              item is poisoned (write_pos = -1, so later calls report
                                              CURSOR_CORRUPT for it); its checkpoint may be partly folded
                                              or partly prefilled, so the slot must be rebuilt:
                                              gdn_spec_reset, then gdn_spec_prefill. */
#define GDN_SPEC_ST_UNFOLDED      32u  /* prefill: continuing from a checkpoint whose ring is not folded */

#define GDN_SPEC_GATE_SCALAR  0    /* GDN: one gate per (token, v-head)            */
#define GDN_SPEC_GATE_PER_KEY 1    /* KDA: one gate per (token, v-head, key channel) */

#define GDN_SPEC_DTYPE_BF16 0
#define GDN_SPEC_DTYPE_FP32 1

/* One GDN layer: dimensions, numerics and its per-slot state. */
typedef struct {
    int32_t H;          /* q/k heads                                               */
    int32_t HV;         /* v heads; H divides HV; v-head hv uses q/k head hv / (HV/H) */
    int32_t K;          /* key dim: 32, 64 or 128                                  */
    int32_t V;          /* value dim (multiple of 8)                               */
    int32_t T;          /* draft window (tokens per row per verify), 1..16         */
    int32_t L;          /* ring length: a power of two, >= 2T ([pr28695] config check) */
    int32_t num_slots;  /* slots in the pool                                       */
    int32_t gate_kind;  /* GDN_SPEC_GATE_SCALAR or GDN_SPEC_GATE_PER_KEY           */
    int32_t io_dtype;   /* dtype of q, k, v, a, b, out, rawv, rawk                 */
    float   scale;      /* output scale (1.0 unless the model scales q)            */
    float   l2_eps;     /* epsilon inside the square root of the q/k L2 norm (1e-6) */
    float  *checkpoint; /* fp32 [num_slots, HV, V, K]                              */
    void   *rawv;       /* io_dtype [num_slots, HV, L, V]                          */
    void   *rawk;       /* io_dtype [num_slots, H, L, K]                           */
    float  *ring_g;     /* fp32 [num_slots, HV, L] (GATE_PER_KEY: [num_slots, HV, L, K]) */
    float  *ring_beta;  /* fp32 [num_slots, HV, L]                                 */
} gdn_spec_layer;

/* Per-slot cursors, shared by every layer of the model, and the status word. */
typedef struct {
    int32_t  num_slots;
    int32_t *write_pos;   /* [num_slots] */
    int32_t *cache_base;  /* [num_slots] */
    int32_t *is_flush;    /* [num_slots] */
    uint32_t *status;     /* [1], device status bits; cleared only by gdn_spec_read_status */
} gdn_spec_cursors;

/*
 * gdn_spec_verify -- output of the whole draft window of every batch row,
 * from the frozen checkpoint plus the ring history, without materialising
 * any per-draft state ([blog] §1.1, §4.1, §5.1; [pr28695] implementation
 * item 3).  Also writes the window's raw records into the ring at
 * (cache_base + write_pos + s) & (L-1) as a side channel: rawv/rawk are
 * bitwise copies of v/k, g/beta the fp32 gate values the kernel computed;
 * the output does not depend on whether the ring positions held anything
 * before ([pr33102] test anchors 1-2; [pr36821] ring write placement).
 * Checkpoint and cursors are only read.
 *
 *   slot_idx  int32 [B]            slot of each row; < 0 marks a padding row
 *   q, k      io_dtype [B, T, H, K]
 *   v         io_dtype [B, T, HV, V]
 *   a         io_dtype [B, T, HV]   (GATE_PER_KEY: [B, T, HV, K])
 *   b         io_dtype [B, T, HV]
 *   A_log     fp32 [HV]
 *   dt_bias   fp32 [HV]             (GATE_PER_KEY: [HV, K])
 *   out       io_dtype [B, T, HV, V]  (written)
 *
 * Device status: SLOT_OOR, CURSOR_CORRUPT, RING_OVERFLOW (the row is skipped
 * and its outputs are zero).  Supported shapes: K in {32, 64, 128}; L <= 128
 * (GATE_SCALAR) or L <= 64 (GATE_PER_KEY); T <= 16; otherwise
 * GDN_SPEC_EUNSUPPORTED.
 */
int gdn_spec_verify(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                    const int32_t *slot_idx, int32_t B,
                    const void *q, const void *k, const void *v, const void *a,
                    const void *b, const float *A_log, const float *dt_bias, void *out,
                    void *stream);

/*
 * gdn_spec_verify_d -- comparison variant of gdn_spec_verify for a ring that
 * also caches every token's corrected delta d_t = beta_t (v_t - S_t^- k^_t)
 * (S_t^- the state after token t's decay): the first design of [blog] §12.1
 * and appendix A.1.  With the history's d cached the verify solves only the
 * window's T x T system; with T = 1 (plain decode) no system at all ([blog]
 * §12.2, §12.9, Part A).  Outputs as gdn_spec_verify; writes the window's raw
 * records into the ring and the window's d into `dring` at the same positions
 * (cache_base + write_pos + s) & (L-1).  The checkpoint and cursors are only
 * read; commit, fold (which replays the raw records, so the cached d never
 * reach the checkpoint) and reset are the ring path's.  A layer that uses it
 * must use it for every verify since its last prefill or reset, so that
 * every committed record's d is in the d ring.
 *   dring  fp32 [num_slots, HV, L, V]   (caller-owned device memory)
 *   other arguments as gdn_spec_verify.
 * Supported shapes: bf16 I/O, GATE_SCALAR, K = 128, V a multiple of 128,
 * L <= 64, T <= 8; otherwise GDN_SPEC_EUNSUPPORTED.
 */
int gdn_spec_verify_d(const gdn_spec_layer *layer, float *dring, const gdn_spec_cursors *cursors,
                      const int32_t *slot_idx, int32_t B, const void *q, const void *k,
                      const void *v, const void *a, const void *b, const float *A_log,
                      const float *dt_bias, void *out, void *stream);

/*
 * gdn_spec_commit -- after sampling: for each row with a slot,
 *   write_pos += accept_len[b];  is_flush = (write_pos + 2T > L)
 * ([blog] §4.2, §8.1-8.2: the early-flush margin keeps one more window in the
 * ring).  Rejected drafts cost nothing: their records stay past write_pos and
 * are overwritten by the next verify ([blog] §4.2-4.3).
 *   accept_len  int32 [B], device; 0 <= accept_len <= T (it counts the bonus
 *               token); outside that the row is skipped with ACCEPT_RANGE.
 * A row whose cursors are out of range (write_pos outside [0, L], cache_base
 * outside [0, L)) is skipped with CURSOR_CORRUPT and left as it is.
 */
int gdn_spec_commit(const gdn_spec_cursors *cursors, int32_t T, int32_t L,
                    const int32_t *slot_idx, int32_t B, const int32_t *accept_len,
                    void *stream);

/*
 * gdn_spec_fold -- exact fold ([pr28695] implementation item 3; [blog] §12.7):
 * for every row whose slot has is_flush set, replay its write_pos committed
 * raw records into the checkpoint of every one of the n_layers layers with the
 * recurrence itself (token by token, fp32), then set
 *   cache_base = (cache_base + write_pos) & (L-1), write_pos = 0, is_flush = 0.
 * Rows without is_flush are left alone, so calling it every step is cheap and
 * calling it twice is harmless.  All layers must have the same dimensions,
 * gate kind and io dtype.  `layers` is a host array of n_layers descriptors.
 */
int gdn_spec_fold(const gdn_spec_layer *layers, int32_t n_layers,
                  const gdn_spec_cursors *cursors, const int32_t *slot_idx, int32_t B,
                  void *stream);

/*
 * gdn_spec_reset -- prefill -> decode handoff ([blog] appendix A.2): for each
 * row with a slot, write_pos = cache_base = 0 and is_flush = 0.  The caller
 * has written that slot's checkpoint.
 */
int gdn_spec_reset(const gdn_spec_cursors *cursors, const int32_t *slot_idx, int32_t B,
                   void *stream);

/*
 * gdn_spec_prefill -- prefill of each row's N prompt tokens into its slot
 * (the step before decode; the reset of the prefill -> decode handoff,
 * [blog] appendix A.2, is part of it): for every v-head the recurrence runs
 * over the tokens from a zero state (from_zero != 0) or from the slot's
 * checkpoint (from_zero == 0, which gives chunked prefill across calls);
 * every token's output is written, the final state becomes the slot's
 * checkpoint, and the slot's cursors are reset (write_pos = cache_base =
 * is_flush = 0).  The ring is not written.  Two kernels (gdn_spec_prefill_path
 * names the one a layer uses): "chunk" -- scalar gate, bf16 I/O, K = 128 and V
 * a multiple of 128 -- the chunk-parallel UT form on the tensor cores, 64
 * tokens per step ([blog] appendix B.1 names chunk_gated_delta_rule as the
 * prefill authority; tf32 operands, the state update split into tf32 high and
 * low parts); "sequential" -- every other shape, token by token in fp32 as
 * the fold does.
 *   q, k      io_dtype [B, N, H, K]
 *   v         io_dtype [B, N, HV, V]
 *   a         io_dtype [B, N, HV]   (GATE_PER_KEY: [B, N, HV, K])
 *   b         io_dtype [B, N, HV]
 *   A_log     fp32 [HV];  dt_bias fp32 [HV] (GATE_PER_KEY: [HV, K])
 *   out       io_dtype [B, N, HV, V]  (written)
 * N >= 0 (N = 0 only zeroes the checkpoints when from_zero, and resets).
 * Device status: SLOT_OOR, CURSOR_CORRUPT, and UNFOLDED when from_zero == 0
 * and the slot's write_pos is not 0 (committed records not yet folded: fold
 * them first); such a row is skipped (its checkpoint and cursors untouched,
 * its outputs zero).
 */
int gdn_spec_prefill(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                     const int32_t *slot_idx, int32_t B, int32_t N,
                     const void *q, const void *k, const void *v, const void *a,
                     const void *b, const float *A_log, const float *dt_bias, void *out,
                     int32_t from_zero, void *stream);

/*
 * Comparison variant, not part of the ring path: the per-draft snapshot
 * design that the ReplaySSM ring replaces ([blog] §0-§1: the intermediate_ssm
 * buffer, one full state per draft position), kept so that its cost can be
 * measured beside the ring on the same machine.
 *
 * gdn_spec_snapshot_verify -- for every row and v-head, from the slot's
 * checkpoint, advance through the T window tokens, write every position's
 * output and store the full state after every position:
 *   snap      fp32 [B, T, HV, V, K]  (written; caller-owned; T V K 4 bytes
 *             per (row, v-head): 256 KiB at the Qwen3-Next shape and T = 4)
 *   q, k, v, a, b, A_log, dt_bias, out: as gdn_spec_verify.
 * The checkpoint is only read; cursors and ring are not used (the status
 * word records SLOT_OOR).
 *
 * gdn_spec_snapshot_commit -- checkpoint[slot_idx[b]] = snap[b, accept_len[b]
 * - 1] for 1 <= accept_len <= T (0 keeps the state; outside [0, T]:
 * ACCEPT_RANGE); accept_len int32 [B], device.
 */
int gdn_spec_snapshot_verify(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                             const int32_t *slot_idx, int32_t B,
                             const void *q, const void *k, const void *v, const void *a,
                             const void *b, const float *A_log, const float *dt_bias, void *out,
                             float *snap, void *stream);
int gdn_spec_snapshot_commit(const gdn_spec_layer *layer, const gdn_spec_cursors *cursors,
                             const int32_t *slot_idx, int32_t B, const int32_t *accept_len,
                             const float *snap, void *stream);

/*
 * gdn_spec_set_wait_limit -- diagnostic: the number of polls after which the
 * first wait on each asynchronous data copy gives up (verify's checkpoint
 * tile on the tensor-core path, the fold's ring records, prefill's prompt
 * chunks).  A wait that gives up sets GDN_SPEC_ST_TIMEOUT; the copy is then
 * drained with the default limit before its buffer is reused, so a small
 * limit exercises the timeout path without leaving anything in flight.
 * Applies to calls made (or graphs captured) afterwards, in every thread of
 * the process.  0xFFFFFFFF restores the default (2^20 polls of at most about
 * 256 ns each: 0.3 s at most).
 * Returns the previous limit.  Not for production use.
 */
uint32_t gdn_spec_set_wait_limit(uint32_t polls);

/*
 * gdn_spec_read_status -- copy the device status word to *host_out after
 * synchronising `stream`; clears it on the device when `clear` is non-zero.
 * Not for use inside a captured graph.
 */
int gdn_spec_read_status(const gdn_spec_cursors *cursors, uint32_t *host_out, int32_t clear,
                         void *stream);

/* Text for a GDN_SPEC_E* code. */
const char *gdn_spec_strerror(int code);

/* GDN_SPEC_ABI_VERSION of the loaded library. */
int gdn_spec_abi_version(void);

/* Name of the verify kernel gdn_spec_verify would launch for this layer
 * ("tc" = TMA + tcgen05 path for the scalar gate, "tc_kda" = TMA + tcgen05
 * path for the per-key gate, "generic" = CUDA-core path), or NULL if the
 * layer is invalid.  Host only; launches nothing. */
const char *gdn_spec_verify_path(const gdn_spec_layer *layer);

/* Name of the prefill kernel gdn_spec_prefill would launch for this layer
 * ("chunk" = chunk-parallel tensor-core path, "sequential" = token-by-token
 * CUDA-core path), or NULL if the layer is invalid.  Host only; launches
 * nothing. */
const char *gdn_spec_prefill_path(const gdn_spec_layer *layer);

#ifdef __cplusplus
}
#endif

#endif /* GDN_SPEC_H */
