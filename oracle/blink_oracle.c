/*
 * blink_oracle.c -- the plain FP64 CPU oracle for the shared-prefix one-pass decision path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table or helper with the
 * CUDA path; the two meet only through the seeded input generators.
 *
 * Every function states what it follows on the source pages ("blink.py" is the first page,
 * blink-4b/blink.py; "simit engine.py" is the second, simit/backends/mot/engine.py).  The code
 * is the definition written out: no blocking, no fusion, no reordering beyond what the
 * definition states.  Floating point is IEEE double throughout; bf16 inputs are widened
 * exactly (a bf16 value is the upper half of an IEEE single).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_LABEL 5

/* Exact widening of a bf16 bit pattern to double. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------------------------
 * Pack plan.  blink.py, `_batches` (token-budget packing) and `_padded` (right padding), plus
 * the per-slot indices the varlen layout needs.
 *
 * The pages' rule, as read here:
 *   - visit the questions shortest first; equal lengths keep their request order (Python's
 *     `sorted` with a length key is stable);
 *   - a forward that already holds `count` questions and whose longest is `longest` closes
 *     before question i when max(longest, len_i) * (count + 1) > budget, or when a row cap
 *     max_rows > 0 is set and count >= max_rows;
 *   - a question longer than the budget therefore runs alone.
 * Outputs, for slot s (the s-th question visited):
 *   order[s]            question index
 *   fwd_of_slot[s]      forward id
 *   fwd_slot_start[f]   first slot of forward f, for f = 0..n_forwards (the last entry is n);
 *                       entries past n_forwards are set to n
 *   fwd_width[f]        padded width of forward f (its longest length); 0 past n_forwards
 *   cu_seqlens[s]       token offset of slot s in the varlen packing of all slots (n+1 entries)
 *   last_varlen[s]      cu_seqlens[s+1] - 1: the last token of slot s in the varlen packing
 *   last_padded[s]      row * fwd_width[f] + len - 1: the last token in forward f's padded
 *                       [rows, width] batch, row being the slot's position inside the forward
 * Returns the number of forwards (>= 1 for n >= 1), or -1 on a bad argument.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
    int32_t len;
    int32_t idx;
} len_idx;

static int cmp_len_idx(const void *a, const void *b)
{
    const len_idx *x = (const len_idx *)a, *y = (const len_idx *)b;
    if (x->len != y->len) return x->len < y->len ? -1 : 1;
    return x->idx < y->idx ? -1 : (x->idx > y->idx ? 1 : 0);
}

int32_t oracle_pack_plan(const int32_t *lengths, int32_t n, int32_t budget, int32_t max_rows,
                         int32_t *order, int32_t *fwd_of_slot, int32_t *fwd_slot_start,
                         int32_t *fwd_width, int32_t *cu_seqlens, int32_t *last_varlen,
                         int32_t *last_padded)
{
    if (n < 1 || budget < 1 || max_rows < 0) return -1;
    for (int32_t i = 0; i < n; i++)
        if (lengths[i] < 1) return -1;

    /* Stable ascending order by length: a sort on the key (length, request index). */
    len_idx *keys = (len_idx *)malloc(sizeof(len_idx) * (size_t)n);
    if (!keys) return -1;
    for (int32_t i = 0; i < n; i++) {
        keys[i].len = lengths[i];
        keys[i].idx = i;
    }
    qsort(keys, (size_t)n, sizeof(len_idx), cmp_len_idx);
    for (int32_t s = 0; s < n; s++) order[s] = keys[s].idx;
    free(keys);

    /* The greedy walk, one question at a time, exactly as the rule reads. */
    int32_t f = 0, count = 0, longest = 0;
    fwd_slot_start[0] = 0;
    for (int32_t s = 0; s < n; s++) {
        int32_t L = lengths[order[s]];
        int32_t grown = longest > L ? longest : L;
        int close_now = 0;
        if (count > 0) {
            if ((int64_t)grown * (int64_t)(count + 1) > (int64_t)budget) close_now = 1;
            if (max_rows > 0 && count >= max_rows) close_now = 1;
        }
        if (close_now) {
            fwd_width[f] = longest;
            f += 1;
            fwd_slot_start[f] = s;
            count = 0;
            grown = L;
        }
        fwd_of_slot[s] = f;
        count += 1;
        longest = grown;
    }
    fwd_width[f] = longest;
    int32_t n_forwards = f + 1;
    for (int32_t k = n_forwards; k <= n; k++) fwd_slot_start[k] = n;
    for (int32_t k = n_forwards; k < n; k++) fwd_width[k] = 0;

    /* Varlen offsets over all slots, and both last-token indices. */
    cu_seqlens[0] = 0;
    for (int32_t s = 0; s < n; s++) cu_seqlens[s + 1] = cu_seqlens[s] + lengths[order[s]];
    for (int32_t s = 0; s < n; s++) {
        int32_t fw = fwd_of_slot[s];
        int32_t row = s - fwd_slot_start[fw];
        last_varlen[s] = cu_seqlens[s + 1] - 1;
        last_padded[s] = row * fwd_width[fw] + lengths[order[s]] - 1;
    }
    return n_forwards;
}

/* ------------------------------------------------------------------------------------------
 * Prefix-tail attention.  blink.py, the PREFIX_CACHE note ("same tokens, same positions; only
 * floating-point order differs") and `_forward_shared`: every question's tail runs against
 * the one shared prefix cache, so a tail token at tail position i (absolute position P + i)
 * sees all P prefix keys and the tail keys 0..i of its own question.
 *
 * Direct definition per (question b, query head h, tail row i), with kv head h / g (g = Hq/Hkv,
 * consecutive query heads share a kv head):
 *   s_j  = scale * <q, k_j>           over the P prefix keys then the i+1 own-tail keys
 *   m    = max_j s_j
 *   O    = sum_j exp(s_j - m) v_j / sum_j exp(s_j - m)
 *   LSE  = m + log(sum_j exp(s_j - m))          (natural log)
 *
 * Layouts (row-major, bf16 bit patterns):
 *   q      [rows, Hq, d]   token r of question b at row seq_start[b] + r
 *   k_tail [rows, Hkv, d]  same token rows as q
 *   v_tail [rows, Hkv, d]
 *   k_pre  [P, Hkv, d]     prefix key of position p at k_pre + p * pre_row_stride
 *   v_pre  [P, Hkv, d]     (pre_row_stride in elements, >= Hkv * d: a slice of a KV arena)
 * Outputs (double): out [rows, Hq, d], lse [Hq, rows].  Only the (token, head) pairs computed
 * are written.  If `sel_tok`/`sel_head` are given, only those n_sel pairs are computed (each
 * token must belong to some question); otherwise every (token of every question, head).
 * ------------------------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *q, *k_pre, *v_pre, *k_tail, *v_tail;
    int64_t pre_row_stride;
    const int32_t *seq_start, *seq_len;
    int32_t B, P, Hq, Hkv, d;
    double scale;
    double *out, *lse;
    int64_t rows;
    /* work list: (token row, head) pairs, each with its question */
    const int32_t *w_tok, *w_head, *w_q;
    int64_t n_work;
    int64_t next;
    pthread_mutex_t lock;
} attn_job;

static void attention_one(const attn_job *J, int32_t t, int32_t h, int32_t b, double *sc)
{
    const int32_t d = J->d, Hq = J->Hq, Hkv = J->Hkv, P = J->P;
    const int32_t g = Hq / Hkv;
    const int32_t kvh = h / g;
    const int32_t i = t - J->seq_start[b]; /* tail position inside question b */
    const int32_t start = J->seq_start[b];
    const uint16_t *q = J->q + ((int64_t)t * Hq + h) * d;
    const int64_t nk = (int64_t)P + i + 1;

    /* scores */
    for (int64_t j = 0; j < nk; j++) {
        const uint16_t *k;
        if (j < P)
            k = J->k_pre + (int64_t)j * J->pre_row_stride + (int64_t)kvh * d;
        else
            k = J->k_tail + ((int64_t)(start + (j - P)) * Hkv + kvh) * d;
        double acc = 0.0;
        for (int32_t c = 0; c < d; c++) acc += widen_bf16(q[c]) * widen_bf16(k[c]);
        sc[j] = J->scale * acc;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < nk; j++)
        if (sc[j] > m) m = sc[j];
    double denom = 0.0;
    for (int64_t j = 0; j < nk; j++) {
        sc[j] = exp(sc[j] - m);
        denom += sc[j];
    }
    double *o = J->out + ((int64_t)t * Hq + h) * d;
    for (int32_t c = 0; c < d; c++) o[c] = 0.0;
    for (int64_t j = 0; j < nk; j++) {
        const uint16_t *v;
        if (j < P)
            v = J->v_pre + (int64_t)j * J->pre_row_stride + (int64_t)kvh * d;
        else
            v = J->v_tail + ((int64_t)(start + (j - P)) * Hkv + kvh) * d;
        for (int32_t c = 0; c < d; c++) o[c] += sc[j] * widen_bf16(v[c]);
    }
    for (int32_t c = 0; c < d; c++) o[c] /= denom;
    if (J->lse) J->lse[(int64_t)h * J->rows + t] = m + log(denom);
}

static void *attention_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    int32_t max_len = 0;
    for (int32_t b = 0; b < J->B; b++)
        if (J->seq_len[b] > max_len) max_len = J->seq_len[b];
    double *sc = (double *)malloc(sizeof(double) * ((size_t)J->P + (size_t)max_len + 1));
    if (!sc) return NULL;
    for (;;) {
        int64_t w;
        pthread_mutex_lock(&J->lock);
        w = J->next;
        J->next += 64;
        pthread_mutex_unlock(&J->lock);
        if (w >= J->n_work) break;
        int64_t e = w + 64 < J->n_work ? w + 64 : J->n_work;
        for (int64_t k = w; k < e; k++) attention_one(J, J->w_tok[k], J->w_head[k], J->w_q[k], sc);
    }
    free(sc);
    return NULL;
}

/* The question that owns token row t, or -1 (a padding row). */
static int32_t owner_of(const int32_t *seq_start, const int32_t *seq_len, int32_t B, int32_t t)
{
    for (int32_t b = 0; b < B; b++)
        if (t >= seq_start[b] && t < seq_start[b] + seq_len[b]) return b;
    return -1;
}

int oracle_prefix_tail_attention(const uint16_t *q, const uint16_t *k_pre, const uint16_t *v_pre,
                                 int64_t pre_row_stride, const uint16_t *k_tail,
                                 const uint16_t *v_tail, const int32_t *seq_start,
                                 const int32_t *seq_len, int32_t B, int64_t rows, int32_t P,
                                 int32_t Hq, int32_t Hkv, int32_t d, double scale,
                                 const int32_t *sel_tok, const int32_t *sel_head, int64_t n_sel,
                                 double *out, double *lse, int32_t n_threads)
{
    if (B < 1 || P < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || d < 1 || rows < 1)
        return ORACLE_BAD_ARG;
    if (P > 0 && pre_row_stride < (int64_t)Hkv * d) return ORACLE_BAD_ARG;
    for (int32_t b = 0; b < B; b++)
        if (seq_len[b] < 1 || seq_start[b] < 0 || (int64_t)seq_start[b] + seq_len[b] > rows)
            return ORACLE_BAD_ARG;

    attn_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k_pre = k_pre; J.v_pre = v_pre; J.k_tail = k_tail; J.v_tail = v_tail;
    J.pre_row_stride = pre_row_stride;
    J.seq_start = seq_start; J.seq_len = seq_len;
    J.B = B; J.P = P; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.scale = scale > 0.0 ? scale : 1.0 / sqrt((double)d);
    J.out = out; J.lse = lse; J.rows = rows;

    int64_t n_work = 0;
    if (sel_tok) {
        n_work = n_sel;
    } else {
        for (int32_t b = 0; b < B; b++) n_work += (int64_t)seq_len[b] * Hq;
    }
    int32_t *w_tok = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_work ? n_work : 1));
    int32_t *w_head = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_work ? n_work : 1));
    int32_t *w_q = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_work ? n_work : 1));
    if (!w_tok || !w_head || !w_q) {
        free(w_tok); free(w_head); free(w_q);
        return ORACLE_BAD_ARG;
    }
    int status = ORACLE_OK;
    if (sel_tok) {
        for (int64_t k = 0; k < n_sel; k++) {
            int32_t b = owner_of(seq_start, seq_len, B, sel_tok[k]);
            if (b < 0 || sel_head[k] < 0 || sel_head[k] >= Hq) {
                status = ORACLE_BAD_ARG;
                break;
            }
            w_tok[k] = sel_tok[k];
            w_head[k] = sel_head[k];
            w_q[k] = b;
        }
    } else {
        int64_t k = 0;
        for (int32_t b = 0; b < B; b++)
            for (int32_t h = 0; h < Hq; h++)
                for (int32_t r = 0; r < seq_len[b]; r++) {
                    w_tok[k] = seq_start[b] + r;
                    w_head[k] = h;
                    w_q[k] = b;
                    k++;
                }
    }
    if (status == ORACLE_OK) {
        J.w_tok = w_tok; J.w_head = w_head; J.w_q = w_q; J.n_work = n_work; J.next = 0;
        pthread_mutex_init(&J.lock, NULL);
        if (n_threads <= 0) n_threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
        if (n_threads < 1) n_threads = 1;
        if (n_threads > 256) n_threads = 256;
        pthread_t th[256];
        int started = 0;
        for (int32_t k = 0; k < n_threads; k++)
            if (pthread_create(&th[k], NULL, attention_worker, &J) == 0) started++;
            else break;
        if (started == 0) attention_worker(&J);
        for (int k = 0; k < started; k++) pthread_join(th[k], NULL);
        pthread_mutex_destroy(&J.lock);
    }
    free(w_tok); free(w_head); free(w_q);
    return status;
}

/* ------------------------------------------------------------------------------------------
 * Label readout.  blink.py, `_read` / `_read_batched` (the last-token hidden state against the
 * label rows of lm_head only, in FP32 there, FP64 here), `softmax` (temperature softmax:
 * z = v / T, m = max z, p = exp(z - m) / sum) and the positivity of the temperature in
 * `decide`.
 *
 *   hidden   [rows, H] bf16, row r at hidden + r * hidden_row_stride
 *   last_idx [B]       the hidden row read for question b
 *   unembed  [V, H]    bf16, row-major
 *   label_off[B+1], label_ids[sum K]  CSR: question b offers label_ids[label_off[b] ..
 *                                     label_off[b+1]) in request order
 * Outputs (double, CSR like label_ids): logits (may be NULL) and probs.
 * A label id outside [0, V) makes that question's outputs NaN and the call return 5.
 * ------------------------------------------------------------------------------------------ */
int oracle_label_readout(const uint16_t *hidden, int64_t hidden_row_stride,
                         const int32_t *last_idx, const uint16_t *unembed, int32_t V, int32_t H,
                         const int32_t *label_off, const int32_t *label_ids, int32_t B,
                         double temperature, double *logits, double *probs)
{
    if (B < 1 || H < 1 || V < 1 || !(temperature > 0.0) || !isfinite(temperature))
        return ORACLE_BAD_ARG;
    if (label_off[0] != 0) return ORACLE_BAD_ARG;
    for (int32_t b = 0; b < B; b++)
        if (label_off[b + 1] <= label_off[b]) return ORACLE_BAD_ARG;
    int status = ORACLE_OK;
    for (int32_t b = 0; b < B; b++) {
        const uint16_t *h = hidden + (int64_t)last_idx[b] * hidden_row_stride;
        const int32_t lo = label_off[b], hi = label_off[b + 1];
        int bad = 0;
        double m = -INFINITY;
        for (int32_t k = lo; k < hi; k++) {
            int32_t id = label_ids[k];
            double z;
            if (id < 0 || id >= V) {
                bad = 1;
                z = NAN;
            } else {
                const uint16_t *w = unembed + (int64_t)id * H;
                double acc = 0.0;
                for (int32_t j = 0; j < H; j++) acc += widen_bf16(h[j]) * widen_bf16(w[j]);
                z = acc;
            }
            if (logits) logits[k] = z;
            probs[k] = z / temperature; /* z / T held here until the max is known */
            if (probs[k] > m) m = probs[k];
        }
        if (bad) {
            status = ORACLE_BAD_LABEL;
            for (int32_t k = lo; k < hi; k++) probs[k] = NAN;
            continue;
        }
        double s = 0.0;
        for (int32_t k = lo; k < hi; k++) {
            probs[k] = exp(probs[k] - m);
            s += probs[k];
        }
        for (int32_t k = lo; k < hi; k++) probs[k] /= s;
    }
    return status;
}
