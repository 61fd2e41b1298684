/*
 * fp64 CPU oracle for decode attention over a branching, paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this code; the library never does, and it shares no source with the library.
 *
 * What it computes (the exact definition; the GPU method reaches the same result faster):
 *
 *   For branch b, its logical sequence is the concatenation of the tokens of its listed
 *   segments, in list order.  Logical index j of b lives at physical page
 *   page_ids[seg.page_off + (seg.tok_begin + t) / P], slot (seg.tok_begin + t) % P.
 *     - Octopus (zicq.com), "Zero-Copy Radix Forking": forked branches list the same prefix
 *       pages, read-only, so a fork reads exactly the KV a copied context would hold.
 *     - Octopus, "Attention-Only KV Mounting": a mounted sibling block is just more entries
 *       of the branch's sequence, read in place.
 *   Query token i of b (n_q_b query tokens, the last ones of the sequence, AKV "Append")
 *   sits at position p_i = n_b - n_q_b + i and sees V_{b,i} = { j <= p_i : vis_b[j] = 1 }.
 *     - AKV (news.farwalk.ai), "AKV 如何工作？": Drop removes an entry from later attention
 *       but keeps every position, so a dropped entry is only a cleared visibility bit.
 *   For query head h, KV head g = h / (Hq / Hkv) (GQA grouping, Octopus mounting section):
 *     s_j = scale * <q_{b,i,h}, K[slot(j), g]>
 *     LSE = ln sum_{j in V} exp(s_j)
 *     out = sum_{j in V} exp(s_j - LSE) * V[slot(j), g]
 *   An empty visible set gives out = 0 and LSE = -inf.
 *
 * How: for every (branch, KV head) that a requested row needs, copy the visible K and V rows
 * into contiguous fp64 arrays (the "copied context"), then run textbook two-pass softmax
 * attention for each requested (query token, query head).  bf16 inputs are widened exactly.
 * Threads split the (branch, KV head) tasks.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t num_q_heads, num_kv_heads, head_dim, page_size;
    double scale;
    const int32_t *page_ids;
    int64_t num_page_ids;
    const int32_t *segs; /* [num_segs][3] = page_off, tok_begin, len */
    int32_t num_segs;
    const int32_t *branch_seg_off; /* [B+1] */
    const int32_t *branch_segs;
    int32_t num_branches;
    const int32_t *branch_q_off; /* [B+1] */
    const uint32_t *vis_bits;     /* NULL = all visible */
    const int64_t *vis_word_off;  /* [B+1] */
    int64_t num_pages_pool;
    const uint16_t *q; /* bf16 bits [total_q][Hq][D] */
    const uint16_t *k; /* bf16 bits [pool][Hkv][P][D] */
    const uint16_t *v;
} oracle_problem;

static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int branch_of_token(const oracle_problem *pr, int64_t t) {
    int lo = 0, hi = pr->num_branches - 1;
    while (lo < hi) { /* largest b with q_off[b] <= t */
        int mid = (lo + hi + 1) / 2;
        if (pr->branch_q_off[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static int64_t branch_len(const oracle_problem *pr, int b) {
    int64_t n = 0;
    for (int32_t e = pr->branch_seg_off[b]; e < pr->branch_seg_off[b + 1]; ++e)
        n += pr->segs[3 * pr->branch_segs[e] + 2];
    return n;
}

/* One task = one (branch, KV head) and the requested rows that fall in it. */
typedef struct {
    int32_t b, g;
    int64_t first, count; /* range in the sorted request order */
} task_t;

typedef struct {
    const oracle_problem *pr;
    const int64_t *rows;   /* requested rows (query token * Hq + head), NULL = all */
    const int64_t *order;  /* request indices sorted by task */
    const task_t *tasks;
    int64_t n_tasks;
    int64_t next;          /* shared task counter */
    double *out, *lse;
    int failed;
} job_t;

static void run_task(job_t *job, const task_t *tk) {
    const oracle_problem *pr = job->pr;
    const int D = pr->head_dim, P = pr->page_size, Hq = pr->num_q_heads, Hkv = pr->num_kv_heads;
    const int b = tk->b, g = tk->g;
    const int64_t n_b = branch_len(pr, b);
    /* 1. copied context: visible entries of b, in logical order, with their positions */
    double *kc = (double *)malloc(sizeof(double) * (size_t)(n_b > 0 ? n_b : 1) * D);
    double *vc = (double *)malloc(sizeof(double) * (size_t)(n_b > 0 ? n_b : 1) * D);
    int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_b > 0 ? n_b : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_b > 0 ? n_b : 1));
    if (!kc || !vc || !pos || !s) {
        job->failed = 1;
        free(kc); free(vc); free(pos); free(s);
        return;
    }
    int64_t n_vis = 0, j = 0;
    for (int32_t e = pr->branch_seg_off[b]; e < pr->branch_seg_off[b + 1]; ++e) {
        const int32_t *sg = pr->segs + 3 * pr->branch_segs[e];
        for (int32_t t = 0; t < sg[2]; ++t, ++j) {
            int visible = 1;
            if (pr->vis_bits) {
                uint32_t w = pr->vis_bits[pr->vis_word_off[b] + j / 32];
                visible = (int)((w >> (j % 32)) & 1u);
            }
            if (!visible) continue;
            int64_t page = pr->page_ids[sg[0] + (sg[1] + t) / P];
            int64_t slot = (sg[1] + t) % P;
            const uint16_t *kr = pr->k + ((page * Hkv + g) * P + slot) * D;
            const uint16_t *vr = pr->v + ((page * Hkv + g) * P + slot) * D;
            for (int d = 0; d < D; ++d) {
                kc[n_vis * D + d] = widen_bf16(kr[d]);
                vc[n_vis * D + d] = widen_bf16(vr[d]);
            }
            pos[n_vis] = j;
            ++n_vis;
        }
    }
    const int32_t nq = pr->branch_q_off[b + 1] - pr->branch_q_off[b];
    /* 2. textbook softmax attention per requested row */
    for (int64_t r = tk->first; r < tk->first + tk->count; ++r) {
        int64_t req = job->order[r];
        int64_t row = job->rows ? job->rows[req] : req;
        int64_t qt = row / Hq;
        int h = (int)(row % Hq);
        int i = (int)(qt - pr->branch_q_off[b]);
        int64_t p_i = n_b - nq + i;
        double qv[512];
        for (int d = 0; d < D; ++d) qv[d] = widen_bf16(pr->q[(qt * Hq + h) * D + d]);
        double m = -INFINITY;
        int64_t cnt = 0;
        for (int64_t c = 0; c < n_vis; ++c) {
            if (pos[c] > p_i) break; /* positions increase along the copied context */
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qv[d] * kc[c * D + d];
            s[c] = pr->scale * acc;
            if (s[c] > m) m = s[c];
            ++cnt;
        }
        double *o = job->out + req * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (cnt == 0) {
            job->lse[req] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t c = 0; c < cnt; ++c) sum += exp(s[c] - m);
        double L = m + log(sum);
        for (int64_t c = 0; c < cnt; ++c) {
            double wgt = exp(s[c] - L);
            for (int d = 0; d < D; ++d) o[d] += wgt * vc[c * D + d];
        }
        job->lse[req] = L;
    }
    free(kc); free(vc); free(pos); free(s);
}

static void *worker(void *arg) {
    job_t *job = (job_t *)arg;
    for (;;) {
        int64_t t = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (t >= job->n_tasks) break;
        run_task(job, &job->tasks[t]);
    }
    return NULL;
}

static const oracle_problem *g_sort_pr;
static const int64_t *g_sort_rows;
static int64_t task_key(int64_t req) {
    const oracle_problem *pr = g_sort_pr;
    int64_t row = g_sort_rows ? g_sort_rows[req] : req;
    int64_t qt = row / pr->num_q_heads;
    int h = (int)(row % pr->num_q_heads);
    int G = pr->num_q_heads / pr->num_kv_heads;
    return (int64_t)branch_of_token(pr, qt) * pr->num_kv_heads + h / G;
}
static int cmp_req(const void *a, const void *b) {
    int64_t ka = task_key(*(const int64_t *)a), kb = task_key(*(const int64_t *)b);
    if (ka != kb) return ka < kb ? -1 : 1;
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return x < y ? -1 : (x > y);
}

/*
 * Computes the requested rows.  rows[r] = query_token * Hq + q_head; rows == NULL means every
 * row in order (n_rows must then be total_q * Hq).  out: [n_rows][D], lse: [n_rows].
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_fork_attn(const oracle_problem *pr, const int64_t *rows, int64_t n_rows,
                     double *out, double *lse, int n_threads) {
    if (!pr || !out || !lse || n_rows < 0) return -1;
    if (pr->head_dim > 512 || pr->num_kv_heads <= 0 || pr->num_q_heads % pr->num_kv_heads)
        return -1;
    const int64_t total_rows = (int64_t)pr->branch_q_off[pr->num_branches] * pr->num_q_heads;
    for (int64_t r = 0; rows && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= total_rows) return -1;
    if (!rows && n_rows != total_rows) return -1;
    if (n_rows == 0) return 0;
    int64_t *order = (int64_t *)malloc(sizeof(int64_t) * (size_t)n_rows);
    task_t *tasks = (task_t *)malloc(sizeof(task_t) * (size_t)n_rows);
    if (!order || !tasks) { free(order); free(tasks); return -1; }
    for (int64_t r = 0; r < n_rows; ++r) order[r] = r;
    g_sort_pr = pr;
    g_sort_rows = rows;
    qsort(order, (size_t)n_rows, sizeof(int64_t), cmp_req);
    int64_t n_tasks = 0;
    for (int64_t r = 0; r < n_rows;) {
        int64_t key = task_key(order[r]);
        int64_t e = r;
        while (e < n_rows && task_key(order[e]) == key) ++e;
        tasks[n_tasks].b = (int32_t)(key / pr->num_kv_heads);
        tasks[n_tasks].g = (int32_t)(key % pr->num_kv_heads);
        tasks[n_tasks].first = r;
        tasks[n_tasks].count = e - r;
        ++n_tasks;
        r = e;
    }
    job_t job = {pr, rows, order, tasks, n_tasks, 0, out, lse, 0};
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    pthread_t th[256];
    int started = 0;
    for (int t = 1; t < n_threads; ++t)
        if (pthread_create(&th[started], NULL, worker, &job) == 0) ++started;
    worker(&job);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    free(order);
    free(tasks);
    return job.failed ? -1 : 0;
}

/*
 * Counts what the measurement calls unique KV: distinct physical token slots that are visible
 * to at least one query token (a slot read by several branches counts once), and distinct
 * physical pages that hold at least one such slot.  Every visible entry of a branch is at or
 * before its last query token, so causality removes nothing from this union.
 */
int oracle_unique_slots(const oracle_problem *pr, int64_t *n_slots, int64_t *n_pages) {
    if (!pr || !n_slots || !n_pages) return -1;
    const int P = pr->page_size;
    const int64_t n_slot_total = pr->num_pages_pool * P;
    unsigned char *seen = (unsigned char *)calloc((size_t)n_slot_total, 1);
    unsigned char *pseen = (unsigned char *)calloc((size_t)pr->num_pages_pool, 1);
    if (!seen || !pseen) { free(seen); free(pseen); return -1; }
    int64_t slots = 0, pages = 0;
    for (int b = 0; b < pr->num_branches; ++b) {
        int64_t j = 0;
        for (int32_t e = pr->branch_seg_off[b]; e < pr->branch_seg_off[b + 1]; ++e) {
            const int32_t *sg = pr->segs + 3 * pr->branch_segs[e];
            for (int32_t t = 0; t < sg[2]; ++t, ++j) {
                if (pr->vis_bits) {
                    uint32_t w = pr->vis_bits[pr->vis_word_off[b] + j / 32];
                    if (!((w >> (j % 32)) & 1u)) continue;
                }
                int64_t page = pr->page_ids[sg[0] + (sg[1] + t) / P];
                int64_t slot = page * P + (sg[1] + t) % P;
                if (!seen[slot]) { seen[slot] = 1; ++slots; }
                if (!pseen[page]) { pseen[page] = 1; ++pages; }
            }
        }
    }
    free(seen);
    free(pseen);
    *n_slots = slots;
    *n_pages = pages;
    return 0;
}
