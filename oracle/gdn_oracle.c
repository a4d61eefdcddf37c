/*
 * gdn_oracle.c -- fp64 CPU oracle for ReplaySSM ring spec-verify of one
 * Gated DeltaNet (GDN) layer, and of its KDA (per-key-channel gate) variant.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into its own shared
 * library and is called from the tests, from the smoke check and from the
 * CPU-baseline leg of the benchmark.  The CUDA product path never links,
 * loads or calls it, and it shares no code, header or table with that path.
 *
 * Sources (web pages; cited by title and section):
 *   [blog]   "PR #28695 详解：GDN ReplaySSM Ring Spec-Verify" (yuyanqi.com)
 *   [pr28695] prhub summary of sglang PR #28695 "[GDN] Support ReplaySSM Ring
 *            Spec-Verify"
 *   [pr33102] prhub report of sglang PR #33102 "fused replayssm ring write into
 *            flashinfer gdn mtp verify kernel"
 *   [pr36821] prhub summary of sglang PR #36821 (fused KDA verify with the
 *            ReplaySSM ring write)
 *
 * What it computes is the plain definition, in fp64, token by token:
 *   gate:    g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b)
 *   norm:    k^ = k / sqrt(sum k^2 + eps)   (q likewise)
 *   step:    S <- exp(g) S            (KDA: S <- S diag(exp(g)))
 *            d  = beta (v - S k^)      (the corrected delta, [blog] §12.1)
 *            S <- S + d k^T
 *            which equals exp(g) S (I - beta k^ k^T) + beta v k^T
 *   output:  o = scale * S q^
 * Verify replays the committed ring history and then the draft window from
 * the frozen checkpoint; it never changes the checkpoint or the cursors and
 * only writes the draft window's raw records into the ring ([blog] §4.1-4.2,
 * §10.1; [pr33102] test anchors 1-2).  Commit moves write_pos and sets the
 * early-flush flag with margin 2T ([blog] §8.1-8.2).  Fold replays the
 * committed raw records into the checkpoint exactly, then moves cache_base
 * and clears write_pos ([pr28695] implementation item 3; [blog] §12.7).
 *
 * Readings where the pages are silent (each listed in the design notes):
 * softplus threshold 20; eps = l2_eps inside the square root; q scale is a
 * parameter; qk head of v-head hv is hv / (HV/H); any slot < 0 is a padding
 * row; 0 <= accept_len <= T; protocol "B" (fold is its own call between
 * commit and the next verify).
 *
 * Every function here is pinned by tests against something other than
 * itself (dense matrix products, the closed-form UT transform, invariants,
 * exhaustive cursor simulation, the pages' printed cursor examples).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <pthread.h>

/* Status bits; the same meaning as the library's device status word. */
#define ORC_ST_ACCEPT_RANGE   1u
#define ORC_ST_SLOT_OOR       2u
#define ORC_ST_RING_OVERFLOW  4u
#define ORC_ST_CURSOR_CORRUPT 8u
#define ORC_ST_UNFOLDED      32u   /* prefill from the checkpoint with records not yet folded */

typedef struct {
    int H, HV, K, V, T, L, num_slots;
    int per_key_gate;          /* 0: one gate per (token, v-head); 1: one per key channel */
    double scale, l2_eps;
} orc_dims;

/* ------------------------------------------------------------------ */
/* Gating ([pr33102] test anchor 3: fused_gdn_gating and fp32 sigmoid)  */
/* ------------------------------------------------------------------ */

double orc_softplus(double x)
{
    /* softplus with beta = 1 and a linear branch above the threshold 20 */
    return x > 20.0 ? x : log1p(exp(x));
}

double orc_gate_g(double A_log, double a, double dt_bias)
{
    return -exp(A_log) * orc_softplus(a + dt_bias);
}

double orc_gate_beta(double b)
{
    return 1.0 / (1.0 + exp(-b));
}

/* ------------------------------------------------------------------ */
/* One recurrence step on a V x K state (row-major, S[i*K + j])        */
/* ------------------------------------------------------------------ */

void orc_l2norm(int n, const double *x, double eps, double *out)
{
    double ss = 0.0;
    for (int j = 0; j < n; ++j) ss += x[j] * x[j];
    double r = 1.0 / sqrt(ss + eps);
    for (int j = 0; j < n; ++j) out[j] = x[j] * r;
}

/* g points to one value (GDN) or K values (KDA). k_raw is the raw key;
 * it is L2-normalised here, as the kernel does with the in-kernel norm. */
/* One step of the recurrence on S [V][K]; when d_out is not NULL it receives
 * the corrected delta d [V] of the step ([blog] §12.1). */
static void step_impl(int V, int K, int per_key_gate, double *S, const double *v,
                      const double *k_raw, const double *g, double beta, double eps,
                      double *d_out)
{
    double *kh = (double *)malloc(sizeof(double) * (size_t)K);
    orc_l2norm(K, k_raw, eps, kh);
    /* decay first, then the delta against the decayed state ([blog] §12.1) */
    if (per_key_gate) {
        for (int i = 0; i < V; ++i)
            for (int j = 0; j < K; ++j) S[(size_t)i * K + j] *= exp(g[j]);
    } else {
        double alpha = exp(g[0]);
        for (size_t e = 0; e < (size_t)V * K; ++e) S[e] *= alpha;
    }
    for (int i = 0; i < V; ++i) {
        double *row = S + (size_t)i * K;
        double u = 0.0;
        for (int j = 0; j < K; ++j) u += row[j] * kh[j];
        double d = beta * (v[i] - u);
        for (int j = 0; j < K; ++j) row[j] += d * kh[j];
        if (d_out) d_out[i] = d;
    }
    free(kh);
}

void orc_step(int V, int K, int per_key_gate, double *S, const double *v,
              const double *k_raw, const double *g, double beta, double eps)
{
    step_impl(V, K, per_key_gate, S, v, k_raw, g, beta, eps, NULL);
}

/* o = scale * S q^ */
void orc_readout(int V, int K, const double *S, const double *q_raw,
                 double eps, double scale, double *o)
{
    double *qh = (double *)malloc(sizeof(double) * (size_t)K);
    orc_l2norm(K, q_raw, eps, qh);
    for (int i = 0; i < V; ++i) {
        double acc = 0.0;
        for (int j = 0; j < K; ++j) acc += S[(size_t)i * K + j] * qh[j];
        o[i] = scale * acc;
    }
    free(qh);
}

/* ------------------------------------------------------------------ */
/* Layer arrays (all fp64, same index order as the device layout)      */
/* ------------------------------------------------------------------ */

typedef struct {
    double *checkpoint;   /* [num_slots, HV, V, K]                    */
    double *rawv;         /* [num_slots, HV, L, V]                    */
    double *rawk;         /* [num_slots, H,  L, K]                    */
    double *ring_g;       /* [num_slots, HV, L] or [num_slots, HV, L, K] */
    double *ring_beta;    /* [num_slots, HV, L]                       */
} orc_layer;

typedef struct {
    int32_t *write_pos, *cache_base, *is_flush;   /* [num_slots] */
} orc_cursors;

static size_t g_width(const orc_dims *d) { return d->per_key_gate ? (size_t)d->K : 1; }

/* physical ring position of logical offset o ([blog] §10.1) */
static int ring_pos(int base, int o, int L) { return (base + o) & (L - 1); }

/* ------------------------------------------------------------------ */
/* Verify ([blog] §1.1, §4.1-4.2, §5.1; [pr33102] test anchors 1-2)     */
/* ------------------------------------------------------------------ */

typedef struct {
    const orc_dims *d;
    const orc_layer *ly;
    const orc_cursors *cur;
    const int32_t *slot_idx;
    int B;
    const double *q, *k, *v, *a, *b, *A_log, *dt_bias;
    double *out;
    double *dwin;              /* [B, T, HV, V] or NULL: the window's corrected deltas */
    const uint8_t *unit_mask;  /* [B*HV] or NULL: which (row, v-head) units to compute */
    uint32_t *row_status;      /* [B] */
    int next_unit;
    pthread_mutex_t lock;
} verify_job;

/* Window gate for token s of row bb, v-head hv; writes 1 or K values to g. */
static void window_gate(const verify_job *J, int bb, int s, int hv, double *g, double *beta)
{
    const orc_dims *d = J->d;
    size_t tok = (size_t)bb * d->T + s;
    if (d->per_key_gate) {
        for (int j = 0; j < d->K; ++j)
            g[j] = orc_gate_g(J->A_log[hv], J->a[(tok * d->HV + hv) * d->K + j],
                              J->dt_bias[(size_t)hv * d->K + j]);
    } else {
        g[0] = orc_gate_g(J->A_log[hv], J->a[tok * d->HV + hv], J->dt_bias[hv]);
    }
    *beta = orc_gate_beta(J->b[tok * d->HV + hv]);
}

/* Validate a row's slot and cursors; returns 1 if the row is computed. */
static int row_ok(const orc_dims *d, const orc_cursors *cur, int slot, uint32_t *st)
{
    if (slot < 0) return 0;
    if (slot >= d->num_slots) { *st |= ORC_ST_SLOT_OOR; return 0; }
    int wp = cur->write_pos[slot], base = cur->cache_base[slot];
    if (wp < 0 || base < 0 || base >= d->L) { *st |= ORC_ST_CURSOR_CORRUPT; return 0; }
    if (wp + d->T > d->L) { *st |= ORC_ST_RING_OVERFLOW; return 0; }
    return 1;
}

static void verify_unit(verify_job *J, int bb, int hv)
{
    const orc_dims *d = J->d;
    const orc_layer *ly = J->ly;
    const int K = d->K, V = d->V, T = d->T, L = d->L, H = d->H, HV = d->HV;
    const int h = hv / (HV / H);
    double *o_row0 = J->out;  /* out[bb, s, hv, :] */
    int slot = J->slot_idx[bb];
    uint32_t st = 0;
    if (!row_ok(d, J->cur, slot, &st)) {
        for (int s = 0; s < T; ++s) {
            memset(o_row0 + (((size_t)bb * T + s) * HV + hv) * V, 0, sizeof(double) * V);
            if (J->dwin) memset(J->dwin + (((size_t)bb * T + s) * HV + hv) * V, 0, sizeof(double) * V);
        }
        return;
    }
    const int base = J->cur->cache_base[slot];
    const int W = J->cur->write_pos[slot];
    const size_t gw = g_width(d);
    double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
    double *g = (double *)malloc(sizeof(double) * gw);
    memcpy(S, ly->checkpoint + ((size_t)slot * HV + hv) * V * K, sizeof(double) * (size_t)V * K);
    /* committed history: o = 0..W-1 at (base + o) & (L-1) */
    for (int o = 0; o < W; ++o) {
        int p = ring_pos(base, o, L);
        orc_step(V, K, d->per_key_gate, S,
                 ly->rawv + (((size_t)slot * HV + hv) * L + p) * V,
                 ly->rawk + (((size_t)slot * H + h) * L + p) * K,
                 ly->ring_g + (((size_t)slot * HV + hv) * L + p) * gw,
                 ly->ring_beta[((size_t)slot * HV + hv) * L + p], d->l2_eps);
    }
    /* draft window: advance a scratch copy, read out every position */
    for (int s = 0; s < T; ++s) {
        size_t tok = (size_t)bb * T + s;
        double beta;
        window_gate(J, bb, s, hv, g, &beta);
        step_impl(V, K, d->per_key_gate, S, J->v + (tok * HV + hv) * V,
                  J->k + (tok * H + h) * K, g, beta, d->l2_eps,
                  J->dwin ? J->dwin + (tok * HV + hv) * V : NULL);
        orc_readout(V, K, S, J->q + (tok * H + h) * K, d->l2_eps, d->scale,
                    o_row0 + (tok * HV + hv) * V);
    }
    free(g);
    free(S);
}

static void *verify_worker(void *arg)
{
    verify_job *J = (verify_job *)arg;
    const int nunits = J->B * J->d->HV;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= nunits) break;
        if (J->unit_mask && !J->unit_mask[u]) continue;
        verify_unit(J, u / J->d->HV, u % J->d->HV);
    }
    return NULL;
}

/* Ring write of the draft window's raw records (the side channel).
 * Position of window token s: (base + write_pos + s) & (L-1) ([blog] §10.1).
 * Runs after every unit has read its history. */
static void verify_ring_write(verify_job *J)
{
    const orc_dims *d = J->d;
    const orc_layer *ly = J->ly;
    const int K = d->K, V = d->V, T = d->T, L = d->L, H = d->H, HV = d->HV;
    const int G = HV / H;
    const size_t gw = g_width(d);
    double *g = (double *)malloc(sizeof(double) * gw);
    for (int bb = 0; bb < J->B; ++bb) {
        int slot = J->slot_idx[bb];
        uint32_t st = 0;
        if (!row_ok(d, J->cur, slot, &st)) continue;
        int base = J->cur->cache_base[slot], W = J->cur->write_pos[slot];
        for (int hv = 0; hv < HV; ++hv) {
            int want = !J->unit_mask || J->unit_mask[(size_t)bb * HV + hv];
            /* a k-head's raw key is written when any v-head of its group is computed */
            int want_k = 0;
            for (int x = (hv / G) * G; x < (hv / G + 1) * G; ++x)
                want_k |= !J->unit_mask || J->unit_mask[(size_t)bb * HV + x];
            for (int s = 0; s < T; ++s) {
                int p = ring_pos(base, W + s, L);
                size_t tok = (size_t)bb * T + s;
                if (want) {
                    double beta;
                    window_gate(J, bb, s, hv, g, &beta);
                    memcpy(ly->rawv + (((size_t)slot * HV + hv) * L + p) * V,
                           J->v + (tok * HV + hv) * V, sizeof(double) * V);
                    memcpy(ly->ring_g + (((size_t)slot * HV + hv) * L + p) * gw, g, sizeof(double) * gw);
                    ly->ring_beta[((size_t)slot * HV + hv) * L + p] = beta;
                }
                if (want_k && hv % G == 0) {
                    int h = hv / G;
                    memcpy(ly->rawk + (((size_t)slot * H + h) * L + p) * K,
                           J->k + (tok * H + h) * K, sizeof(double) * K);
                }
            }
        }
    }
    free(g);
}

static uint32_t verify_run(const orc_dims *d, orc_layer *ly, const orc_cursors *cur,
                           const int32_t *slot_idx, int B, const double *q, const double *k,
                           const double *v, const double *a, const double *b,
                           const double *A_log, const double *dt_bias, double *out,
                           double *dwin, const uint8_t *unit_mask, int nthreads)
{
    verify_job J;
    memset(&J, 0, sizeof J);
    J.d = d; J.ly = ly; J.cur = cur; J.slot_idx = slot_idx; J.B = B;
    J.q = q; J.k = k; J.v = v; J.a = a; J.b = b; J.A_log = A_log; J.dt_bias = dt_bias;
    J.out = out; J.dwin = dwin; J.unit_mask = unit_mask;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, verify_worker, &J);
    verify_worker(&J);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    verify_ring_write(&J);
    uint32_t st = 0;
    for (int bb = 0; bb < B; ++bb) row_ok(d, cur, slot_idx[bb], &st);
    return st;
}

/* Returns the OR of the status bits of all rows. */
uint32_t orc_verify(const orc_dims *d, orc_layer *ly, const orc_cursors *cur,
                    const int32_t *slot_idx, int B,
                    const double *q, const double *k, const double *v,
                    const double *a, const double *b,
                    const double *A_log, const double *dt_bias,
                    double *out, const uint8_t *unit_mask, int nthreads)
{
    return verify_run(d, ly, cur, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, NULL,
                      unit_mask, nthreads);
}

/* Verify that also returns the corrected delta d [B, T, HV, V] of every window
 * token: d = beta (v - S k^) against the decayed state before the token
 * ([blog] §12.1).  These are the values a ring that caches d (the derived-d
 * design of [blog] appendix A.1) would hold for the window's records; rows
 * that are not computed read zeros. */
uint32_t orc_verify_d(const orc_dims *d, orc_layer *ly, const orc_cursors *cur,
                      const int32_t *slot_idx, int B,
                      const double *q, const double *k, const double *v,
                      const double *a, const double *b,
                      const double *A_log, const double *dt_bias,
                      double *out, double *dwin, int nthreads)
{
    return verify_run(d, ly, cur, slot_idx, B, q, k, v, a, b, A_log, dt_bias, out, dwin, NULL,
                      nthreads);
}

/* ------------------------------------------------------------------ */
/* Commit ([blog] §4.2, §8.1-8.2): write_pos += accept_len, then        */
/* is_flush = (write_pos + 2T > L), strict                               */
/* ------------------------------------------------------------------ */

uint32_t orc_commit(const orc_dims *d, orc_cursors *cur, const int32_t *slot_idx,
                    int B, const int32_t *accept_len)
{
    uint32_t st = 0;
    for (int bb = 0; bb < B; ++bb) {
        int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= d->num_slots) { st |= ORC_ST_SLOT_OOR; continue; }
        int acc = accept_len[bb];
        if (acc < 0 || acc > d->T) { st |= ORC_ST_ACCEPT_RANGE; continue; }
        /* cursors out of range (the same rule verify applies): skip the row */
        int wp0 = cur->write_pos[slot], base = cur->cache_base[slot];
        if (wp0 < 0 || wp0 > d->L || base < 0 || base >= d->L) { st |= ORC_ST_CURSOR_CORRUPT; continue; }
        int wp = wp0 + acc;
        cur->write_pos[slot] = wp;
        cur->is_flush[slot] = (wp + 2 * d->T > d->L) ? 1 : 0;
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* Exact fold ([pr28695] item 3; [blog] §12.7): replay the committed     */
/* raw records into the checkpoint with the recurrence itself, then      */
/* cache_base = (cache_base + write_pos) & (L-1), write_pos = 0,         */
/* is_flush = 0.  Only rows whose is_flush is set are folded.            */
/* ------------------------------------------------------------------ */

typedef struct {
    const orc_dims *d;
    orc_layer *layers;
    int n_layers;
    const orc_cursors *cur;
    const int32_t *slot_idx;
    int B;
    int next_unit;
    pthread_mutex_t lock;
} fold_job;

static void fold_unit(fold_job *J, int li, int bb, int hv)
{
    const orc_dims *d = J->d;
    orc_layer *ly = &J->layers[li];
    const int K = d->K, V = d->V, L = d->L, H = d->H, HV = d->HV;
    const int h = hv / (HV / H);
    int slot = J->slot_idx[bb];
    uint32_t st = 0;
    if (slot < 0 || slot >= d->num_slots) return;
    if (!J->cur->is_flush[slot]) return;
    int wp = J->cur->write_pos[slot], base = J->cur->cache_base[slot];
    if (wp < 0 || wp > L || base < 0 || base >= L) return;
    (void)st;
    const size_t gw = g_width(d);
    double *S = ly->checkpoint + ((size_t)slot * HV + hv) * V * K;
    for (int o = 0; o < wp; ++o) {
        int p = ring_pos(base, o, L);
        orc_step(V, K, d->per_key_gate, S,
                 ly->rawv + (((size_t)slot * HV + hv) * L + p) * V,
                 ly->rawk + (((size_t)slot * H + h) * L + p) * K,
                 ly->ring_g + (((size_t)slot * HV + hv) * L + p) * gw,
                 ly->ring_beta[((size_t)slot * HV + hv) * L + p], d->l2_eps);
    }
}

static void *fold_worker(void *arg)
{
    fold_job *J = (fold_job *)arg;
    const int per_layer = J->B * J->d->HV;
    const int nunits = J->n_layers * per_layer;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= nunits) break;
        int li = u / per_layer, r = u % per_layer;
        fold_unit(J, li, r / J->d->HV, r % J->d->HV);
    }
    return NULL;
}

uint32_t orc_fold(const orc_dims *d, orc_layer *layers, int n_layers, orc_cursors *cur,
                  const int32_t *slot_idx, int B, int nthreads)
{
    fold_job J;
    memset(&J, 0, sizeof J);
    J.d = d; J.layers = layers; J.n_layers = n_layers; J.cur = cur;
    J.slot_idx = slot_idx; J.B = B;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, fold_worker, &J);
    fold_worker(&J);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    /* the cursors move once, after every layer has folded */
    uint32_t st = 0;
    for (int bb = 0; bb < B; ++bb) {
        int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= d->num_slots) { st |= ORC_ST_SLOT_OOR; continue; }
        if (!cur->is_flush[slot]) continue;
        int wp = cur->write_pos[slot], base = cur->cache_base[slot];
        if (wp < 0 || wp > d->L || base < 0 || base >= d->L) { st |= ORC_ST_CURSOR_CORRUPT; continue; }
        cur->cache_base[slot] = ring_pos(base, wp, d->L);
        cur->write_pos[slot] = 0;
        cur->is_flush[slot] = 0;
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* Reset at the prefill -> decode handoff ([blog] appendix A.2):          */
/* write_pos = cache_base = 0, is_flush = 0                              */
/* ------------------------------------------------------------------ */

uint32_t orc_reset(const orc_dims *d, orc_cursors *cur, const int32_t *slot_idx, int B)
{
    uint32_t st = 0;
    for (int bb = 0; bb < B; ++bb) {
        int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= d->num_slots) { st |= ORC_ST_SLOT_OOR; continue; }
        cur->write_pos[slot] = 0;
        cur->cache_base[slot] = 0;
        cur->is_flush[slot] = 0;
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* Plain recurrence from a given state over a token sequence (used to   */
/* build prefix checkpoints and the running committed state).            */
/* ------------------------------------------------------------------ */

/* S: [V,K]; v: [n,V]; k_raw: [n,K]; g: [n,gw]; beta: [n] */
void orc_run(const orc_dims *d, double *S, int n, const double *v, const double *k_raw,
             const double *g, const double *beta)
{
    const size_t gw = g_width(d);
    for (int t = 0; t < n; ++t)
        orc_step(d->V, d->K, d->per_key_gate, S, v + (size_t)t * d->V,
                 k_raw + (size_t)t * d->K, g + (size_t)t * gw, beta[t], d->l2_eps);
}

/* Many independent runs at once (one per unit), spread over threads.
 * S: [nunits, V, K]; v: [nunits, n, V]; k_raw: [nunits, n, K];
 * g: [nunits, n, gw]; beta: [nunits, n]. */
typedef struct {
    const orc_dims *d;
    int nunits, n;
    double *S;
    const double *v, *k_raw, *g, *beta;
    int next;
    pthread_mutex_t lock;
} run_job;

static void *run_worker(void *arg)
{
    run_job *J = (run_job *)arg;
    const orc_dims *d = J->d;
    const size_t gw = g_width(d), VK = (size_t)d->V * d->K;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->nunits) break;
        orc_run(d, J->S + (size_t)u * VK, J->n, J->v + (size_t)u * J->n * d->V,
                J->k_raw + (size_t)u * J->n * d->K, J->g + (size_t)u * J->n * gw,
                J->beta + (size_t)u * J->n);
    }
    return NULL;
}

void orc_run_batch(const orc_dims *d, int nunits, double *S, int n, const double *v,
                   const double *k_raw, const double *g, const double *beta, int nthreads)
{
    run_job J;
    memset(&J, 0, sizeof J);
    J.d = d; J.nunits = nunits; J.n = n; J.S = S; J.v = v; J.k_raw = k_raw; J.g = g; J.beta = beta;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, run_worker, &J);
    run_worker(&J);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
}

/* ------------------------------------------------------------------ */
/* Prefill: the recurrence over the N prompt tokens of every row, with   */
/* the output of every token, from a zero state or from the row's        */
/* checkpoint; the final state becomes the checkpoint and the row's      */
/* cursors are reset for decode (the prefill -> decode handoff, [blog]   */
/* appendix A.2).  Continuing from the checkpoint needs an empty ring    */
/* (write_pos == 0): the committed state is then the checkpoint itself.  */
/* ------------------------------------------------------------------ */

typedef struct {
    const orc_dims *d;
    orc_layer *ly;
    const orc_cursors *cur;
    const int32_t *slot_idx;
    int B, N, from_zero;
    const double *q, *k, *v, *a, *b, *A_log, *dt_bias;
    double *out;
    int next_unit;
    pthread_mutex_t lock;
} prefill_job;

/* Which rows a prefill computes; sets the status bits of the others. */
static int prefill_row_ok(const orc_dims *d, const orc_cursors *cur, int slot, int from_zero,
                          uint32_t *st)
{
    if (slot < 0) return 0;
    if (slot >= d->num_slots) { *st |= ORC_ST_SLOT_OOR; return 0; }
    int wp = cur->write_pos[slot], base = cur->cache_base[slot];
    if (wp < 0 || wp > d->L || base < 0 || base >= d->L) { *st |= ORC_ST_CURSOR_CORRUPT; return 0; }
    if (!from_zero && wp != 0) { *st |= ORC_ST_UNFOLDED; return 0; }
    return 1;
}

static void prefill_unit(prefill_job *J, int bb, int hv)
{
    const orc_dims *d = J->d;
    const int K = d->K, V = d->V, N = J->N, H = d->H, HV = d->HV;
    const int h = hv / (HV / H);
    int slot = J->slot_idx[bb];
    uint32_t st = 0;
    if (!prefill_row_ok(d, J->cur, slot, J->from_zero, &st)) {
        for (int t = 0; t < N; ++t)
            memset(J->out + (((size_t)bb * N + t) * HV + hv) * V, 0, sizeof(double) * V);
        return;
    }
    const size_t gw = g_width(d);
    double *S = J->ly->checkpoint + ((size_t)slot * HV + hv) * V * K;
    double *g = (double *)malloc(sizeof(double) * gw);
    if (J->from_zero) memset(S, 0, sizeof(double) * (size_t)V * K);
    for (int t = 0; t < N; ++t) {
        size_t tok = (size_t)bb * N + t;
        if (d->per_key_gate) {
            for (int j = 0; j < K; ++j)
                g[j] = orc_gate_g(J->A_log[hv], J->a[(tok * HV + hv) * K + j], J->dt_bias[(size_t)hv * K + j]);
        } else {
            g[0] = orc_gate_g(J->A_log[hv], J->a[tok * HV + hv], J->dt_bias[hv]);
        }
        double beta = orc_gate_beta(J->b[tok * HV + hv]);
        orc_step(V, K, d->per_key_gate, S, J->v + (tok * HV + hv) * V, J->k + (tok * H + h) * K, g,
                 beta, d->l2_eps);
        orc_readout(V, K, S, J->q + (tok * H + h) * K, d->l2_eps, d->scale, J->out + (tok * HV + hv) * V);
    }
    free(g);
}

static void *prefill_worker(void *arg)
{
    prefill_job *J = (prefill_job *)arg;
    const int nunits = J->B * J->d->HV;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->lock);
        if (u >= nunits) break;
        prefill_unit(J, u / J->d->HV, u % J->d->HV);
    }
    return NULL;
}

/* q, k: [B, N, H, K]; v: [B, N, HV, V]; a: [B, N, HV] (per-key gate: [B, N, HV, K]);
 * b: [B, N, HV]; out: [B, N, HV, V].  Returns the OR of the rows' status bits. */
uint32_t orc_prefill(const orc_dims *d, orc_layer *ly, orc_cursors *cur, const int32_t *slot_idx,
                     int B, int N, const double *q, const double *k, const double *v,
                     const double *a, const double *b, const double *A_log, const double *dt_bias,
                     double *out, int from_zero, int nthreads)
{
    prefill_job J;
    memset(&J, 0, sizeof J);
    J.d = d; J.ly = ly; J.cur = cur; J.slot_idx = slot_idx; J.B = B; J.N = N; J.from_zero = from_zero;
    J.q = q; J.k = k; J.v = v; J.a = a; J.b = b; J.A_log = A_log; J.dt_bias = dt_bias; J.out = out;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int t = 1; t < nthreads; ++t) pthread_create(&th[t], NULL, prefill_worker, &J);
    prefill_worker(&J);
    for (int t = 1; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    /* the cursors of the rows computed are reset for decode */
    uint32_t st = 0;
    for (int bb = 0; bb < B; ++bb) {
        int slot = slot_idx[bb];
        if (!prefill_row_ok(d, cur, slot, from_zero, &st)) continue;
        cur->write_pos[slot] = 0;
        cur->cache_base[slot] = 0;
        cur->is_flush[slot] = 0;
    }
    return st;
}

/* ------------------------------------------------------------------ */
/* Comparison variant: the per-draft snapshot design that the ring       */
/* replaces ([blog] §0-§1: the intermediate_ssm buffer, one full state   */
/* per draft position).  Verify advances each row's state through the    */
/* window, reads out every position and stores every intermediate state; */
/* commit copies the state after the accepted tokens back.               */
/* ------------------------------------------------------------------ */

/* snap: [B, T, HV, V, K]; q, k: [B, T, H, K]; v: [B, T, HV, V]; a, b: [B, T, HV]
 * (per-key gate: a [B, T, HV, K]); out: [B, T, HV, V].  Rows with slot < 0 or
 * slot >= num_slots read out zeros and store nothing (status SLOT_OOR for
 * the latter).  The checkpoint is only read. */
uint32_t orc_snapshot_verify(const orc_dims *d, const orc_layer *ly, const int32_t *slot_idx, int B,
                             const double *q, const double *k, const double *v, const double *a,
                             const double *b, const double *A_log, const double *dt_bias,
                             double *out, double *snap)
{
    const int K = d->K, V = d->V, T = d->T, H = d->H, HV = d->HV;
    const size_t gw = g_width(d), VK = (size_t)V * K;
    uint32_t st = 0;
    double *S = (double *)malloc(sizeof(double) * VK);
    double *g = (double *)malloc(sizeof(double) * gw);
    for (int bb = 0; bb < B; ++bb) {
        int slot = slot_idx[bb];
        for (int hv = 0; hv < HV; ++hv) {
            const int h = hv / (HV / H);
            if (slot < 0 || slot >= d->num_slots) {
                if (slot >= d->num_slots) st |= ORC_ST_SLOT_OOR;
                for (int s = 0; s < T; ++s)
                    memset(out + (((size_t)bb * T + s) * HV + hv) * V, 0, sizeof(double) * V);
                continue;
            }
            memcpy(S, ly->checkpoint + ((size_t)slot * HV + hv) * VK, sizeof(double) * VK);
            for (int s = 0; s < T; ++s) {
                size_t tok = (size_t)bb * T + s;
                if (d->per_key_gate) {
                    for (int j = 0; j < K; ++j)
                        g[j] = orc_gate_g(A_log[hv], a[(tok * HV + hv) * K + j], dt_bias[(size_t)hv * K + j]);
                } else {
                    g[0] = orc_gate_g(A_log[hv], a[tok * HV + hv], dt_bias[hv]);
                }
                orc_step(V, K, d->per_key_gate, S, v + (tok * HV + hv) * V, k + (tok * H + h) * K, g,
                         orc_gate_beta(b[tok * HV + hv]), d->l2_eps);
                orc_readout(V, K, S, q + (tok * H + h) * K, d->l2_eps, d->scale, out + (tok * HV + hv) * V);
                memcpy(snap + (tok * HV + hv) * VK, S, sizeof(double) * VK);
            }
        }
    }
    free(g);
    free(S);
    return st;
}

/* checkpoint[slot] = snap[b, accept_len - 1] for rows with 1 <= accept_len <= T
 * (accept_len 0 keeps the state; outside [0, T]: status ACCEPT_RANGE). */
uint32_t orc_snapshot_commit(const orc_dims *d, orc_layer *ly, const int32_t *slot_idx, int B,
                             const int32_t *accept_len, const double *snap)
{
    const int T = d->T, HV = d->HV;
    const size_t VK = (size_t)d->V * d->K;
    uint32_t st = 0;
    for (int bb = 0; bb < B; ++bb) {
        int slot = slot_idx[bb];
        if (slot < 0) continue;
        if (slot >= d->num_slots) { st |= ORC_ST_SLOT_OOR; continue; }
        int acc = accept_len[bb];
        if (acc < 0 || acc > T) { st |= ORC_ST_ACCEPT_RANGE; continue; }
        if (acc == 0) continue;
        for (int hv = 0; hv < HV; ++hv)
            memcpy(ly->checkpoint + ((size_t)slot * HV + hv) * VK,
                   snap + (((size_t)bb * T + acc - 1) * HV + hv) * VK, sizeof(double) * VK);
    }
    return st;
}
