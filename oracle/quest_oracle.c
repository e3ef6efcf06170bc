/*
 * quest_oracle.c - plain, slow CPU oracle of Quest's decode-time path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the CUDA
 * library is checked against.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg may load or call it; the library itself never
 * does, and it shares no code, header, table or helper with the CUDA sources.
 *
 * Sources (web pages about Quest, Tang et al., ICML 2024):
 *   [Guide]   "Guide to Quest: Query-Aware KV Cache Sparsity for LLMs"
 *   [Summary] "Quest: Query-Aware Sparsity for Efficient Long-Context LLM Inference"
 *             (Tang 2024 paper summary page)
 *
 * Precision.  Keys, values and queries are fp16 values; this file receives them widened
 * to float (an exact conversion).  Bounding boxes are therefore exact.  Page scores are
 * summed in float in dimension order 0..d-1, because the score decides an integer result
 * (the selected pages) and the CUDA path takes that decision in float as well.  Attention
 * is computed in double.
 *
 * Every function is a straight loop over the definition; nothing is blocked, fused or
 * reordered.  Layouts (row-major):
 *   k_pool, v_pool : [num_phys][Hkv][P][d]
 *   meta           : [num_phys][Hkv][2][d]      (index 0 = per-dim minimum, 1 = maximum)
 *   block_table    : [B][max_pages]             logical page -> physical page
 *   seq_lens       : [B]                        tokens in the cache
 *   q              : [B][Hq][d]
 *   scores         : [B][Hkv][max_pages]        (-inf past the last page)
 *   idx            : [B][Hkv][K] logical pages in rank order, count : [B][Hkv]
 *   out            : [B][Hq][d] (double),   lse : [B][Hq] (double)
 *
 * Return value of the int functions: 0 on success, -1 if a block-table entry, a length
 * or a page index is out of range (nothing further is computed then).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t batch;
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    int32_t max_pages;
    int32_t num_phys;
} oq_dims;

static size_t kv_at(const oq_dims* s, int64_t phys, int g, int slot) {
    return (((size_t)phys * s->num_kv_heads + g) * s->page_size + slot) * s->head_dim;
}

static size_t meta_at(const oq_dims* s, int64_t phys, int g, int which) {
    return (((size_t)phys * s->num_kv_heads + g) * 2 + which) * s->head_dim;
}

static int pages_of(const oq_dims* s, int len) {
    return (len + s->page_size - 1) / s->page_size;
}

/* Physical page of logical page p of sequence b, or -1 if the table entry is unusable. */
static int64_t phys_of(const oq_dims* s, const int32_t* block_table, int b, int p) {
    if (p < 0 || p >= s->max_pages) return -1;
    int64_t phys = block_table[(size_t)b * s->max_pages + p];
    if (phys < 0 || phys >= s->num_phys) return -1;
    return phys;
}

static int len_ok(const oq_dims* s, int len) {
    return len >= 0 && (int64_t)len <= (int64_t)s->max_pages * s->page_size;
}

/* ---------------------------------------------------------------------------------
 * Bounding boxes.  [Guide] Solution, step 1 (min-max key bounding box equations):
 * for page p the per-dimension minimum and maximum over the keys it holds.  Only the
 * tokens t < seq_len exist; a partially filled last page is boxed over its valid tokens.
 * --------------------------------------------------------------------------------- */
int oq_build_meta(const oq_dims* s, const float* k_pool, const int32_t* block_table,
                  const int32_t* seq_lens, float* meta) {
    const int d = s->head_dim, P = s->page_size;
    for (int b = 0; b < s->batch; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L)) return -1;
        const int n_pages = pages_of(s, L);
        for (int p = 0; p < n_pages; ++p) {
            const int64_t phys = phys_of(s, block_table, b, p);
            if (phys < 0) return -1;
            int n_valid = L - p * P;
            if (n_valid > P) n_valid = P;
            for (int g = 0; g < s->num_kv_heads; ++g) {
                float* mn = meta + meta_at(s, phys, g, 0);
                float* mx = meta + meta_at(s, phys, g, 1);
                for (int i = 0; i < d; ++i) {
                    float lo = k_pool[kv_at(s, phys, g, 0) + i];
                    float hi = lo;
                    for (int t = 1; t < n_valid; ++t) {
                        float v = k_pool[kv_at(s, phys, g, t) + i];
                        if (v < lo) lo = v;
                        if (v > hi) hi = v;
                    }
                    mn[i] = lo;
                    mx[i] = hi;
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Decode-time append.  [Guide] Solution, step 1: a page's box is built as the page fills,
 * in generation as in prefill: the new token of sequence b goes
 * to position seq_lens[b] (page seq_len / P, slot seq_len % P); a token that opens a
 * page starts that page's box, any other token widens the existing box.  The length
 * then grows by one.
 * --------------------------------------------------------------------------------- */
int oq_append(const oq_dims* s, float* k_pool, float* v_pool, float* meta,
              const int32_t* block_table, int32_t* seq_lens, const float* k_new,
              const float* v_new) {
    const int d = s->head_dim, P = s->page_size;
    for (int b = 0; b < s->batch; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L + 1)) return -1;
        const int p = L / P, slot = L % P;
        const int64_t phys = phys_of(s, block_table, b, p);
        if (phys < 0) return -1;
        for (int g = 0; g < s->num_kv_heads; ++g) {
            const float* kn = k_new + ((size_t)b * s->num_kv_heads + g) * d;
            const float* vn = v_new + ((size_t)b * s->num_kv_heads + g) * d;
            float* kd = k_pool + kv_at(s, phys, g, slot);
            float* vd = v_pool + kv_at(s, phys, g, slot);
            float* mn = meta + meta_at(s, phys, g, 0);
            float* mx = meta + meta_at(s, phys, g, 1);
            for (int i = 0; i < d; ++i) {
                kd[i] = kn[i];
                vd[i] = vn[i];
                if (slot == 0) {
                    mn[i] = kn[i];
                    mx[i] = kn[i];
                } else {
                    if (kn[i] < mn[i]) mn[i] = kn[i];
                    if (kn[i] > mx[i]) mx[i] = kn[i];
                }
            }
        }
        seq_lens[b] = L + 1;
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Criticality.  [Guide] Solution, step 2, the upper-bound inequality:
 *     U(q, p) = sum_i max(q_i * Kmin_i, q_i * Kmax_i)
 * The page's 1/sqrt(d) factor is left out: it is a positive constant, so it cannot
 * change which pages rank highest.  Each product of two fp16 values is exact in float;
 * the sum is taken in float in dimension order.  Grouped-query attention: the score of a
 * page for a kv head is the largest of the bounds of the query heads that share it.
 * Pages at or past ceil(seq_len / P) get -inf.
 * --------------------------------------------------------------------------------- */
int oq_score(const oq_dims* s, const float* q, const float* meta, const int32_t* block_table,
             const int32_t* seq_lens, float* scores) {
    const int d = s->head_dim;
    const int G = s->num_q_heads / s->num_kv_heads;
    for (int b = 0; b < s->batch; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L)) return -1;
        const int n_pages = pages_of(s, L);
        for (int g = 0; g < s->num_kv_heads; ++g) {
            float* row = scores + ((size_t)b * s->num_kv_heads + g) * s->max_pages;
            for (int p = 0; p < s->max_pages; ++p) {
                if (p >= n_pages) {
                    row[p] = -INFINITY;
                    continue;
                }
                const int64_t phys = phys_of(s, block_table, b, p);
                if (phys < 0) return -1;
                const float* mn = meta + meta_at(s, phys, g, 0);
                const float* mx = meta + meta_at(s, phys, g, 1);
                float best = -INFINITY;
                for (int h = g * G; h < (g + 1) * G; ++h) {
                    const float* qh = q + ((size_t)b * s->num_q_heads + h) * d;
                    float u = 0.0f;
                    for (int i = 0; i < d; ++i) {
                        float a = qh[i] * mn[i];
                        float c = qh[i] * mx[i];
                        u += (a > c) ? a : c;
                    }
                    if (u > best) best = u;
                }
                row[p] = best;
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * The same bound per query head, without the maximum over a group: scores_h is
 * [batch][num_q_heads][max_pages] (-inf past the last page).  Used by the group-level
 * selection below.
 * --------------------------------------------------------------------------------- */
int oq_score_heads(const oq_dims* s, const float* q, const float* meta, const int32_t* block_table,
                   const int32_t* seq_lens, float* scores_h) {
    const int d = s->head_dim;
    const int G = s->num_q_heads / s->num_kv_heads;
    for (int b = 0; b < s->batch; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L)) return -1;
        const int n_pages = pages_of(s, L);
        for (int h = 0; h < s->num_q_heads; ++h) {
            const int g = h / G;
            const float* qh = q + ((size_t)b * s->num_q_heads + h) * d;
            float* row = scores_h + ((size_t)b * s->num_q_heads + h) * s->max_pages;
            for (int p = 0; p < s->max_pages; ++p) {
                if (p >= n_pages) {
                    row[p] = -INFINITY;
                    continue;
                }
                const int64_t phys = phys_of(s, block_table, b, p);
                if (phys < 0) return -1;
                const float* mn = meta + meta_at(s, phys, g, 0);
                const float* mx = meta + meta_at(s, phys, g, 1);
                float u = 0.0f;
                for (int i = 0; i < d; ++i) {
                    float a = qh[i] * mn[i];
                    float c = qh[i] * mx[i];
                    u += (a > c) ? a : c;
                }
                row[p] = u;
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Page selection.  [Guide] Solution, step 3: keep the K pages with the highest bounds
 * ([Summary], Summary: the K best-scoring pages).  Pages are ordered by score, larger
 * first, and equal scores by page index, lower first; the first K_b = min(K, N_b) are
 * kept.  When the sequence has no more than K pages every page is kept ([Guide],
 * Implementation step 2, the short-sequence case).
 *
 * Mandatory pages ([Guide] Solution step 3, third bullet, and Implementation step 2):
 * the first `sink` pages and the last `local` pages of a sequence longer than K pages are
 * kept unconditionally, and only the remaining K - sink - local slots are competed for,
 * by the pages between them, in the order above.  sink = local = 0 is the plain top-K;
 * local = 0 keeps no trailing page.  Requires sink, local >= 0 and sink + local <= K.
 *
 * idx receives the kept pages: for a short sequence all pages in rank order, otherwise the
 * sinks, then the local pages, then the competitive pages in rank order; entries past
 * count are set to -1.
 * --------------------------------------------------------------------------------- */
typedef struct {
    float score;
    int32_t page;
} oq_ranked;

static int oq_rank_cmp(const void* x, const void* y) {
    const oq_ranked* a = (const oq_ranked*)x;
    const oq_ranked* b = (const oq_ranked*)y;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->page < b->page) ? -1 : (a->page > b->page) ? 1 : 0;
}

int oq_topk(const oq_dims* s, const float* scores, const int32_t* seq_lens, int K, int sink,
            int local, int32_t* idx, int32_t* count) {
    if (K < 1 || sink < 0 || local < 0 || sink + local > K) return -1;
    oq_ranked* tmp = (oq_ranked*)malloc(sizeof(oq_ranked) * (size_t)(s->max_pages > 0 ? s->max_pages : 1));
    if (!tmp) return -1;
    for (int b = 0; b < s->batch; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L)) { free(tmp); return -1; }
        const int n_pages = pages_of(s, L);
        for (int g = 0; g < s->num_kv_heads; ++g) {
            const float* row = scores + ((size_t)b * s->num_kv_heads + g) * s->max_pages;
            int32_t* out = idx + ((size_t)b * s->num_kv_heads + g) * K;
            int n_out = 0;
            if (n_pages <= K) {
                for (int p = 0; p < n_pages; ++p) {
                    tmp[p].score = row[p];
                    tmp[p].page = p;
                }
                qsort(tmp, (size_t)n_pages, sizeof(oq_ranked), oq_rank_cmp);
                for (int r = 0; r < n_pages; ++r) out[n_out++] = tmp[r].page;
            } else {
                for (int p = 0; p < sink; ++p) out[n_out++] = p;
                for (int p = n_pages - local; p < n_pages; ++p) out[n_out++] = p;
                int n_cand = 0;
                for (int p = sink; p < n_pages - local; ++p) {
                    tmp[n_cand].score = row[p];
                    tmp[n_cand].page = p;
                    ++n_cand;
                }
                qsort(tmp, (size_t)n_cand, sizeof(oq_ranked), oq_rank_cmp);
                for (int r = 0; r < K - sink - local; ++r) out[n_out++] = tmp[r].page;
            }
            for (int r = n_out; r < K; ++r) out[r] = -1;
            count[(size_t)b * s->num_kv_heads + g] = n_out;
        }
    }
    free(tmp);
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Group-level selection, union form.  [Guide] Best Practices step 2 (GQA): the bounds of
 * every query head of a group are computed and the union of their top-k pages is kept,
 * so the kv head's pages are loaded once for all of its query heads.  Each query head h of
 * kv head g keeps its own K best pages (score larger first, then lower page, as above);
 * the kv head keeps the union, at most G * K pages.  A sequence of at most K pages keeps
 * every page.  idx: [batch][num_kv_heads][cap] with cap >= min(G * K, max_pages), the kept
 * pages in ascending order, -1 after count.
 * --------------------------------------------------------------------------------- */
int oq_topk_union(const oq_dims* s, const float* scores_h, const int32_t* seq_lens, int K, int cap,
                  int32_t* idx, int32_t* count) {
    const int G = s->num_q_heads / s->num_kv_heads;
    if (K < 1 || cap < 1) return -1;
    oq_ranked* tmp = (oq_ranked*)malloc(sizeof(oq_ranked) * (size_t)(s->max_pages > 0 ? s->max_pages : 1));
    unsigned char* kept = (unsigned char*)malloc((size_t)(s->max_pages > 0 ? s->max_pages : 1));
    if (!tmp || !kept) { free(tmp); free(kept); return -1; }
    for (int b = 0; b < s->batch; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L)) { free(tmp); free(kept); return -1; }
        const int n_pages = pages_of(s, L);
        for (int g = 0; g < s->num_kv_heads; ++g) {
            for (int p = 0; p < n_pages; ++p) kept[p] = (unsigned char)(n_pages <= K);
            if (n_pages > K) {
                for (int h = g * G; h < (g + 1) * G; ++h) {
                    const float* row = scores_h + ((size_t)b * s->num_q_heads + h) * s->max_pages;
                    for (int p = 0; p < n_pages; ++p) {
                        tmp[p].score = row[p];
                        tmp[p].page = p;
                    }
                    qsort(tmp, (size_t)n_pages, sizeof(oq_ranked), oq_rank_cmp);
                    for (int r = 0; r < K; ++r) kept[tmp[r].page] = 1;
                }
            }
            int32_t* out = idx + ((size_t)b * s->num_kv_heads + g) * cap;
            int n_out = 0;
            for (int p = 0; p < n_pages; ++p) {
                if (!kept[p]) continue;
                if (n_out >= cap) { free(tmp); free(kept); return -1; }
                out[n_out++] = p;
            }
            for (int r = n_out; r < cap; ++r) out[r] = -1;
            count[(size_t)b * s->num_kv_heads + g] = n_out;
        }
    }
    free(tmp);
    free(kept);
    return 0;
}

/* ---------------------------------------------------------------------------------
 * Attention over the kept pages.  [Summary] Summary: exact attention is computed only
 * over the selected pages; [Guide] Solution step 3 and Implementation step 3: the kept
 * pages' keys and values are gathered and softmax(q k^T / sqrt(d)) v is taken over
 * them.  Query head h reads kv head h / G (grouped-query attention) and that kv head's
 * selection.  Tokens t >= seq_len do not exist and are skipped.  Output and the
 * log-sum-exp lse = m + ln(sum_t exp(z_t - m)) are double.  With no token, out = 0 and
 * lse = -inf.
 * --------------------------------------------------------------------------------- */
int oq_attend(const oq_dims* s, const float* q, const float* k_pool, const float* v_pool,
              const int32_t* block_table, const int32_t* seq_lens, const int32_t* idx,
              const int32_t* count, int K, double* out, double* lse) {
    const int d = s->head_dim, P = s->page_size;
    const int G = s->num_q_heads / s->num_kv_heads;
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double* z = (double*)malloc(sizeof(double) * (size_t)K * P + sizeof(double));
    int64_t* tok_phys = (int64_t*)malloc(sizeof(int64_t) * (size_t)K * P + sizeof(int64_t));
    int* tok_slot = (int*)malloc(sizeof(int) * (size_t)K * P + sizeof(int));
    if (!z || !tok_phys || !tok_slot) { free(z); free(tok_phys); free(tok_slot); return -1; }
    int rc = 0;
    for (int b = 0; b < s->batch && rc == 0; ++b) {
        const int L = seq_lens[b];
        if (!len_ok(s, L)) { rc = -1; break; }
        const int n_pages = pages_of(s, L);
        for (int h = 0; h < s->num_q_heads && rc == 0; ++h) {
            const int g = h / G;
            const float* qh = q + ((size_t)b * s->num_q_heads + h) * d;
            const int32_t* sel = idx + ((size_t)b * s->num_kv_heads + g) * K;
            const int n_sel = count[(size_t)b * s->num_kv_heads + g];
            double* o = out + ((size_t)b * s->num_q_heads + h) * d;
            /* logits of every existing token of every kept page */
            int n_tok = 0;
            for (int r = 0; r < n_sel; ++r) {
                const int p = sel[r];
                if (p < 0 || p >= n_pages) { rc = -1; break; }
                const int64_t phys = phys_of(s, block_table, b, p);
                if (phys < 0) { rc = -1; break; }
                for (int t = 0; t < P; ++t) {
                    if (p * P + t >= L) break;
                    const float* k = k_pool + kv_at(s, phys, g, t);
                    double dot = 0.0;
                    for (int i = 0; i < d; ++i) dot += (double)qh[i] * (double)k[i];
                    z[n_tok] = dot * inv_sqrt_d;
                    tok_phys[n_tok] = phys;
                    tok_slot[n_tok] = t;
                    ++n_tok;
                }
            }
            if (rc) break;
            for (int i = 0; i < d; ++i) o[i] = 0.0;
            if (n_tok == 0) {
                lse[(size_t)b * s->num_q_heads + h] = -INFINITY;
                continue;
            }
            double m = z[0];
            for (int t = 1; t < n_tok; ++t) if (z[t] > m) m = z[t];
            double denom = 0.0;
            for (int t = 0; t < n_tok; ++t) denom += exp(z[t] - m);
            for (int t = 0; t < n_tok; ++t) {
                const double w = exp(z[t] - m) / denom;
                const float* v = v_pool + kv_at(s, tok_phys[t], g, tok_slot[t]);
                for (int i = 0; i < d; ++i) o[i] += w * (double)v[i];
            }
            lse[(size_t)b * s->num_q_heads + h] = m + log(denom);
        }
    }
    free(z);
    free(tok_phys);
    free(tok_slot);
    return rc;
}
