/*
 * Plain fp64 CPU oracle for the Key-Value Means (KVM) layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library, and it is deliberately slow: naive loops, no blocking, no fusion,
 * every step in the order the method states it.
 *
 * Sources (page title "Key-Value Means"; the gist.science technical summary is
 * cited as "KVM summary", the chatpaper.ai abstract as "KVM abstract"):
 *   - KVM summary, Core mechanism 1 (block-sliding window with compressed
 *     state): input is processed in chunks; a block that overflows the window
 *     is folded into the state instead of being dropped.
 *   - KVM summary, Core mechanism 2 (state compression and merging): each
 *     overflowed key goes to the single most correlated state key (winner
 *     take all, cosine-like similarity); state keys are LayerNorm'd before
 *     use; state values are rescaled to a read radius rho_i fixed when the
 *     slot is created; a data-dependent scalar gate modulates how much of the
 *     incoming key/value is absorbed.
 *   - KVM summary, lay part "smart merge": slots keep raw sums and counts; the
 *     division happens only when the state is read (just in time).
 *   - KVM summary, Core mechanism 3 (state growth): the most surprising
 *     (least redundant) overflow tokens are appended as new slots, the rest
 *     are merged; fixed-size or sqrt(N) growth.
 *   - KVM summary, Core mechanism 4 (position encoding): the rotary subspace
 *     of state keys is zeroed; unrotated queries read the state, rotated
 *     queries read the window, in one attention pass.
 *   - KVM summary, Core mechanism 5 (sinks): a protected set of initial
 *     state rows is never merged into.
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes): read radius = L2 norm of the founding value; argmax ties go
 * to the lowest slot index; surprise ties to the lower position; sums are
 * gate-weighted, counts are integers; LayerNorm without affine, biased
 * variance; cosine over the full head dimension against the unrotated key;
 * window of chunk c = chunks c-W/C .. c (causal in c); chunk c-W/C-1 is
 * folded just before chunk c; the first S overflowed tokens found the S sink
 * slots; remaining tokens of a chunk merge into the post-append state, all
 * decided against the same state (chunk-parallel); rotate-half RoPE over the
 * first r dims; softmax scale 1/sqrt(d) for state and window alike.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t head_dim;      /* d */
    int32_t rope_dims;     /* r: RoPE rotates dims [0, r) */
    double rope_theta;     /* RoPE base */
    int32_t chunk;         /* C */
    int32_t window;        /* W, a multiple of C */
    int32_t n_sinks;       /* S */
    int32_t sched;         /* 0 = fixed (cap = max_slots), 1 = power law */
    int32_t max_slots;     /* M */
    double coef, expo;     /* power law: cap(t) = S + ceil(coef * t^expo) */
    double ln_eps;         /* LayerNorm epsilon */
    int32_t merge_pre_append;  /* alternative reading: merge targets = pre-append slots only */
    int32_t cos_nope_only;     /* alternative reading: cosine over dims [r, d) only */
    int32_t no_value_norm;     /* ablation: read value = sum_v / count (no value-length norm) */
} kvo_config;

enum { KVO_MERGED = 0, KVO_APPENDED = 1, KVO_SINK = 2 };
enum { KVO_OK = 0, KVO_ERR_CAPACITY = 3, KVO_ERR_ARG = 1 };

/* ---------------------------------------------------------------- helpers */

static double dot(const double* a, const double* b, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

static double norm2(const double* a, int n) { return sqrt(dot(a, a, n)); }

/* cosine similarity; 0 when either vector is zero */
static double cosine(const double* a, const double* b, int n) {
    double na = norm2(a, n), nb = norm2(b, n);
    if (na == 0.0 || nb == 0.0) return 0.0;
    return dot(a, b, n) / (na * nb);
}

/* LayerNorm without affine parameters, biased variance. */
static void layernorm(const double* x, int n, double eps, double* out) {
    double mean = 0.0;
    for (int i = 0; i < n; ++i) mean += x[i];
    mean /= n;
    double var = 0.0;
    for (int i = 0; i < n; ++i) var += (x[i] - mean) * (x[i] - mean);
    var /= n;
    double inv = 1.0 / sqrt(var + eps);
    for (int i = 0; i < n; ++i) out[i] = (x[i] - mean) * inv;
}

/* Rotate-half RoPE on dims [0, r) at absolute position p: pair (i, i + r/2)
 * turns by angle p * theta^(-2i/r).  Dims [r, d) are copied. */
static void rope(const double* x, int64_t p, const kvo_config* cfg, double* out) {
    int d = cfg->head_dim, half = cfg->rope_dims / 2;
    for (int i = 0; i < d; ++i) out[i] = x[i];
    for (int i = 0; i < half; ++i) {
        double freq = pow(cfg->rope_theta, -2.0 * (double)i / (double)cfg->rope_dims);
        double ang = (double)p * freq;
        double c = cos(ang), s = sin(ang);
        out[i] = x[i] * c - x[i + half] * s;
        out[i + half] = x[i + half] * c + x[i] * s;
    }
}

/* Slot capacity after t overflowed tokens (KVM summary, Core mechanism 3:
 * fixed-size or sqrt growth). */
int64_t kvo_capacity(const kvo_config* cfg, int64_t t) {
    if (cfg->sched == 0) return cfg->max_slots;
    if (t <= 0) return cfg->n_sinks;
    return (int64_t)cfg->n_sinks + (int64_t)ceil(cfg->coef * pow((double)t, cfg->expo));
}

/* State key of slot j as read: LayerNorm(sum_k / count) over all d dims. */
static void state_key_full(const kvo_config* cfg, const double* sum_k, const int64_t* count,
                           int64_t j, double* out) {
    int d = cfg->head_dim;
    double* mean_k = (double*)malloc(sizeof(double) * d);
    for (int i = 0; i < d; ++i) mean_k[i] = sum_k[j * d + i] / (double)count[j];
    layernorm(mean_k, d, cfg->ln_eps, out);
    free(mean_k);
}

/* Similarity used by the winner-take-all rule: cosine of the raw key against
 * the LayerNorm'd state key (full head dim unless cos_nope_only). */
static double merge_similarity(const kvo_config* cfg, const double* k, const double* key_hat) {
    int d = cfg->head_dim;
    if (cfg->cos_nope_only) {
        int r = cfg->rope_dims;
        return cosine(k + r, key_hat + r, d - r);
    }
    return cosine(k, key_hat, d);
}

/* ------------------------------------------------------------- fold event */

/*
 * Fold one chunk of C overflowed tokens into the state of one (batch, head).
 * KVM summary, Core mechanisms 1-3 and 5.
 *
 * n_slots, t: in/out slot count and number of overflowed tokens so far.
 * sum_k, sum_v: [max_slots, d] raw gate-weighted sums; count: [max_slots];
 * rho: [max_slots] read radius.
 * first_pos: absolute position of the chunk's first token.
 * k, v: [C, d] unrotated keys and values; g: [C] merge gate.
 * Outputs per token (any may be NULL): assign = slot the token went to;
 * kind = merged / appended / sink; max_sim = surprise score m_t (highest
 * cosine against the mergeable slots before this chunk's appends, -inf when
 * there are none, NaN for sinks); gap = top-2 gap of the final argmax
 * (+inf with fewer than two candidates, NaN for sinks and appended tokens).
 * sel_margin: the gap between the a-th and (a+1)-th smallest surprise score
 * (+inf when the selection is forced).
 */
int kvo_fold_event(const kvo_config* cfg, int64_t* n_slots, int64_t* t,
                   double* sum_k, double* sum_v, int64_t* count, double* rho,
                   int64_t first_pos, const double* k, const double* v, const double* g,
                   int32_t* assign, int32_t* kind, double* max_sim, double* gap,
                   double* sel_margin) {
    const int d = cfg->head_dim, C = cfg->chunk, S = cfg->n_sinks;
    const int64_t M = cfg->max_slots;
    int64_t n = *n_slots;

    /* 1. the first S overflowed tokens found the sink slots, in order */
    int* is_cand = (int*)calloc(C, sizeof(int));
    int ncand = 0;
    for (int i = 0; i < C; ++i) {
        int64_t pos = first_pos + i;
        if (pos < S) {
            if (n != pos || n >= M) { free(is_cand); return KVO_ERR_ARG; }
            for (int x = 0; x < d; ++x) {
                sum_k[n * d + x] = g[i] * k[i * d + x];
                sum_v[n * d + x] = g[i] * v[i * d + x];
            }
            count[n] = 1;
            rho[n] = norm2(v + (int64_t)i * d, d);
            if (assign) assign[i] = (int32_t)n;
            if (kind) kind[i] = KVO_SINK;
            if (max_sim) max_sim[i] = NAN;
            if (gap) gap[i] = NAN;
            n += 1;
        } else {
            is_cand[i] = 1;
            ncand += 1;
        }
    }

    int64_t t_new = *t + C;
    int64_t cap = kvo_capacity(cfg, t_new);
    int64_t n0 = n; /* slots before this chunk's appends */

    /* 2. surprise: highest cosine of each candidate against the mergeable
     *    slots [S, n0) of the state as it stands */
    double* key_hat = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * d);
    for (int64_t j = S; j < n0; ++j) state_key_full(cfg, sum_k, count, j, key_hat + j * d);
    double* m = (double*)malloc(sizeof(double) * C);
    for (int i = 0; i < C; ++i) {
        m[i] = -INFINITY;
        if (!is_cand[i]) continue;
        for (int64_t j = S; j < n0; ++j) {
            double c = merge_similarity(cfg, k + (int64_t)i * d, key_hat + j * d);
            if (c > m[i]) m[i] = c;
        }
        if (max_sim) max_sim[i] = m[i];
    }

    /* 3. number of appends: fill up to the capacity, at most every candidate */
    int64_t a = cap - n0;
    if (a < 0) a = 0;
    if (a > ncand) a = ncand;
    if (n0 + a > M) { free(is_cand); free(key_hat); free(m); return KVO_ERR_CAPACITY; }

    /* pick the a most surprising candidates: smallest m, ties to the lower
     * position (selection by repeated minimum; plain and obviously stable) */
    int* chosen = (int*)calloc(C, sizeof(int));
    int* order = (int*)malloc(sizeof(int) * C);
    int norder = 0;
    for (int step = 0; step < ncand; ++step) {
        int best = -1;
        for (int i = 0; i < C; ++i) {
            if (!is_cand[i] || chosen[i]) continue;
            if (best < 0 || m[i] < m[best]) best = i; /* strict: keeps the lower position on ties */
        }
        chosen[best] = 1;
        order[norder++] = best;
    }
    if (sel_margin) {
        if (a > 0 && a < ncand) *sel_margin = m[order[a]] - m[order[a - 1]];
        else *sel_margin = INFINITY;
    }
    for (int i = 0; i < C; ++i) chosen[i] = 0;
    for (int64_t s = 0; s < a; ++s) chosen[order[s]] = 1;

    /* 4. append the chosen tokens as new slots, in position order */
    for (int i = 0; i < C; ++i) {
        if (!chosen[i]) continue;
        for (int x = 0; x < d; ++x) {
            sum_k[n * d + x] = g[i] * k[(int64_t)i * d + x];
            sum_v[n * d + x] = g[i] * v[(int64_t)i * d + x];
        }
        count[n] = 1;
        rho[n] = norm2(v + (int64_t)i * d, d);
        if (assign) assign[i] = (int32_t)n;
        if (kind) kind[i] = KVO_APPENDED;
        if (gap) gap[i] = NAN;
        n += 1;
    }

    /* 5. every other candidate goes to its argmax over the mergeable slots of
     *    the post-append state (lowest index on ties); all decisions are taken
     *    against the same state, before any merge of this chunk */
    int64_t hi = cfg->merge_pre_append ? n0 : n;
    for (int64_t j = n0; j < hi; ++j) state_key_full(cfg, sum_k, count, j, key_hat + j * d);
    int32_t* target = (int32_t*)malloc(sizeof(int32_t) * C);
    for (int i = 0; i < C; ++i) {
        target[i] = -1;
        if (!is_cand[i] || chosen[i]) continue;
        double best = -INFINITY, second = -INFINITY;
        int64_t arg = -1;
        for (int64_t j = S; j < hi; ++j) {
            double c = merge_similarity(cfg, k + (int64_t)i * d, key_hat + j * d);
            if (c > best) { second = best; best = c; arg = j; }
            else if (c > second) { second = c; }
        }
        if (arg < 0) { free(is_cand); free(key_hat); free(m); free(chosen); free(order); free(target); return KVO_ERR_ARG; }
        target[i] = (int32_t)arg;
        if (assign) assign[i] = (int32_t)arg;
        if (kind) kind[i] = KVO_MERGED;
        if (gap) gap[i] = best - second;
    }

    /* 6. merge: gate-weighted raw sums, integer counts, in position order */
    for (int i = 0; i < C; ++i) {
        if (target[i] < 0) continue;
        int64_t j = target[i];
        for (int x = 0; x < d; ++x) {
            sum_k[j * d + x] += g[i] * k[(int64_t)i * d + x];
            sum_v[j * d + x] += g[i] * v[(int64_t)i * d + x];
        }
        count[j] += 1;
    }

    *n_slots = n;
    *t = t_new;
    free(is_cand); free(key_hat); free(m); free(chosen); free(order); free(target);
    return KVO_OK;
}

/* ------------------------------------------------------------ state read */

/*
 * Just-in-time read view of n slots (KVM summary, Core mechanisms 2 and 4):
 * key_view = LayerNorm(sum_k / count) with dims [0, r) set to zero;
 * val_view = rho * sum_v / ||sum_v||  (zero when sum_v is zero);
 * with the value-length normalisation removed (the pages' ablation, technical
 * summary, Experimental results), val_view = sum_v / count.
 */
void kvo_state_view(const kvo_config* cfg, int64_t n, const double* sum_k, const double* sum_v,
                    const int64_t* count, const double* rho, double* key_view, double* val_view) {
    int d = cfg->head_dim, r = cfg->rope_dims;
    for (int64_t j = 0; j < n; ++j) {
        state_key_full(cfg, sum_k, count, j, key_view + j * d);
        for (int x = 0; x < r; ++x) key_view[j * d + x] = 0.0;
        double nv = norm2(sum_v + j * d, d);
        for (int x = 0; x < d; ++x) {
            if (cfg->no_value_norm)
                val_view[j * d + x] = sum_v[j * d + x] / (double)count[j];
            else
                val_view[j * d + x] = nv == 0.0 ? 0.0 : rho[j] * sum_v[j * d + x] / nv;
        }
    }
}

/* ------------------------------------------------------------- attention */

/* RoPE of nw rows at positions first_pos, first_pos + 1, ... */
void kvo_rope_rows(const kvo_config* cfg, int64_t nw, int64_t first_pos, const double* x,
                   double* out) {
    int d = cfg->head_dim;
    for (int64_t i = 0; i < nw; ++i) rope(x + i * d, first_pos + i, cfg, out + i * d);
}

/*
 * One query at absolute position p over n state rows and nw window tokens,
 * in one softmax (KVM summary, Methodology and Core mechanism 4).  The state
 * is scored with the unrotated query q; the window with the rotated query
 * against wk_rot, the window keys already rotated at their own positions.
 * Both parts use scale 1/sqrt(d).  Two-pass softmax.
 */
void kvo_attend_query(const kvo_config* cfg, int64_t n, const double* key_view,
                      const double* val_view, const double* q, int64_t p,
                      int64_t nw, const double* wk_rot, const double* wv, double* out) {
    int d = cfg->head_dim;
    double scale = 1.0 / sqrt((double)d);
    int64_t nk = n + nw;
    double* s = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double* qr = (double*)malloc(sizeof(double) * d);
    rope(q, p, cfg, qr);
    for (int64_t j = 0; j < n; ++j) s[j] = dot(q, key_view + j * d, d) * scale;
    for (int64_t i = 0; i < nw; ++i) s[n + i] = dot(qr, wk_rot + i * d, d) * scale;
    double mx = -INFINITY;
    for (int64_t j = 0; j < nk; ++j) if (s[j] > mx) mx = s[j];
    double den = 0.0;
    for (int64_t j = 0; j < nk; ++j) { s[j] = exp(s[j] - mx); den += s[j]; }
    for (int x = 0; x < d; ++x) out[x] = 0.0;
    for (int64_t j = 0; j < n; ++j)
        for (int x = 0; x < d; ++x) out[x] += s[j] * val_view[j * d + x];
    for (int64_t i = 0; i < nw; ++i)
        for (int x = 0; x < d; ++x) out[x] += s[n + i] * wv[i * d + x];
    for (int x = 0; x < d; ++x) out[x] /= den;
    free(s); free(qr);
}

/* --------------------------------------------------------------- prefill */

/*
 * Chunked prefill of one (batch, head) from an empty state (KVM summary,
 * Core mechanism 1; KVM abstract, chunk-wise parallel prefill).
 * For chunk c: if c >= W/C + 1, fold chunk c - W/C - 1; then every query of
 * chunk c attends to the state plus tokens (c - W/C)*C .. its own position.
 *
 * q, k, v: [N, d]; g: [N]; out: [N, d].  State arrays hold max_slots rows and
 * are overwritten.  Debug arrays (nullable) hold max_events * C entries;
 * sel_margin holds max_events entries.
 */
int kvo_prefill_head(const kvo_config* cfg, int64_t N, const double* q, const double* k,
                     const double* v, const double* g, double* out,
                     int64_t* n_slots, int64_t* t, double* sum_k, double* sum_v,
                     int64_t* count, double* rho,
                     int64_t max_events, int32_t* assign, int32_t* kind, double* max_sim,
                     double* gap, double* sel_margin) {
    const int d = cfg->head_dim, C = cfg->chunk;
    const int64_t Wc = cfg->window / C, M = cfg->max_slots;
    *n_slots = 0;
    *t = 0;
    memset(sum_k, 0, sizeof(double) * (size_t)M * d);
    memset(sum_v, 0, sizeof(double) * (size_t)M * d);
    memset(count, 0, sizeof(int64_t) * (size_t)M);
    memset(rho, 0, sizeof(double) * (size_t)M);
    double* key_view = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * d);
    double* val_view = (double*)malloc(sizeof(double) * (size_t)(M > 0 ? M : 1) * d);
    double* wk_rot = (double*)malloc(sizeof(double) * (size_t)(cfg->window + C) * d);
    int64_t nchunks = (N + C - 1) / C;
    int rc = KVO_OK;
    for (int64_t c = 0; c < nchunks; ++c) {
        if (c >= Wc + 1) {
            int64_t e = c - Wc - 1;
            int64_t o = e * C;
            int have = e < max_events;
            rc = kvo_fold_event(cfg, n_slots, t, sum_k, sum_v, count, rho, o,
                                k + o * d, v + o * d, g + o,
                                have && assign ? assign + o : NULL, have && kind ? kind + o : NULL,
                                have && max_sim ? max_sim + o : NULL, have && gap ? gap + o : NULL,
                                have && sel_margin ? sel_margin + e : NULL);
            if (rc != KVO_OK) break;
        }
        kvo_state_view(cfg, *n_slots, sum_k, sum_v, count, rho, key_view, val_view);
        int64_t ws = (c - Wc) * C;
        if (ws < 0) ws = 0;
        int64_t pe = (c + 1) * C < N ? (c + 1) * C : N;
        /* every query of the chunk sees the same rotated window keys */
        kvo_rope_rows(cfg, pe - ws, ws, k + ws * d, wk_rot);
        for (int64_t p = c * C; p < pe; ++p)
            kvo_attend_query(cfg, *n_slots, key_view, val_view, q + p * d, p,
                             p - ws + 1, wk_rot, v + ws * d, out + p * d);
    }
    free(key_view); free(val_view); free(wk_rot);
    return rc;
}

/* ------------------------------------------- threaded driver over heads */

typedef struct {
    const kvo_config* cfg;
    int64_t N, n_heads, max_events;
    const double *q, *k, *v, *g;
    double* out;
    int64_t *n_slots, *t;
    double *sum_k, *sum_v, *rho;
    int64_t* count;
    int32_t *assign, *kind;
    double *max_sim, *gap, *sel_margin;
    int64_t next;
    int rc;
    pthread_mutex_t mu;
} prefill_job;

static void* prefill_worker(void* arg) {
    prefill_job* J = (prefill_job*)arg;
    const int64_t N = J->N, d = J->cfg->head_dim, M = J->cfg->max_slots;
    const int64_t E = J->max_events, C = J->cfg->chunk;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t h = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (h >= J->n_heads) break;
        int rc = kvo_prefill_head(J->cfg, N, J->q + h * N * d, J->k + h * N * d, J->v + h * N * d,
                                  J->g + h * N, J->out + h * N * d, J->n_slots + h, J->t + h,
                                  J->sum_k + h * M * d, J->sum_v + h * M * d, J->count + h * M,
                                  J->rho + h * M, E,
                                  J->assign ? J->assign + h * E * C : NULL,
                                  J->kind ? J->kind + h * E * C : NULL,
                                  J->max_sim ? J->max_sim + h * E * C : NULL,
                                  J->gap ? J->gap + h * E * C : NULL,
                                  J->sel_margin ? J->sel_margin + h * E : NULL);
        if (rc != KVO_OK) {
            pthread_mutex_lock(&J->mu);
            J->rc = rc;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

/* Prefill of n_heads independent (batch, head) rows, [n_heads, N, d] each,
 * spread over n_threads POSIX threads (one head at a time per thread). */
int kvo_prefill(const kvo_config* cfg, int64_t n_heads, int64_t N, const double* q,
                const double* k, const double* v, const double* g, double* out,
                int64_t* n_slots, int64_t* t, double* sum_k, double* sum_v, int64_t* count,
                double* rho, int64_t max_events, int32_t* assign, int32_t* kind,
                double* max_sim, double* gap, double* sel_margin, int n_threads) {
    prefill_job J;
    J.cfg = cfg; J.N = N; J.n_heads = n_heads; J.max_events = max_events;
    J.q = q; J.k = k; J.v = v; J.g = g; J.out = out;
    J.n_slots = n_slots; J.t = t; J.sum_k = sum_k; J.sum_v = sum_v; J.count = count; J.rho = rho;
    J.assign = assign; J.kind = kind; J.max_sim = max_sim; J.gap = gap; J.sel_margin = sel_margin;
    J.next = 0; J.rc = KVO_OK;
    pthread_mutex_init(&J.mu, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n_heads) n_threads = (int)(n_heads > 0 ? n_heads : 1);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
    for (int i = 0; i < n_threads; ++i) pthread_create(&th[i], NULL, prefill_worker, &J);
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.rc;
}
