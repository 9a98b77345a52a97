/*
 * Oracle: paged decode attention and tree-verify attention, by definition, in
 * fp64.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the timed
 * CPU baseline of the benchmark call this; the library never does.  It shares
 * no code, header or constant with the CUDA path.
 *
 * Definition followed (for each layer l, query token r, query head h):
 *   1. gather: the query's keys are token positions of its sequence; token t
 *      lives in block table[t / bs], slot t % bs (paged KV of fixed-size
 *      token blocks: "Dendrite", section on memory management; "Trellis",
 *      section "RadixAttention in Trellis": a session holds an ordered list
 *      of block ids into a shared pool).  The kv head is g = h / (Hq / Hkv).
 *   2. scores:  z_t = (q . k_t) * scale          (scale = 1/sqrt(d) by default)
 *   3. softmax: p_t = exp(z_t - max z) / sum exp(z - max z)
 *   4. output:  out = sum_t p_t v_t,  lse = max z + ln sum exp(z - max z)
 * Decode: query r of the batch attends to the first lens[r] tokens of its
 * table ("SGLang RadixAttention", decode step: one new token attends to the
 * cached keys and values).
 * Verify: draft node i of sequence b attends to context tokens t < ctx[b]
 * and to draft tokens ctx[b] + j for j in anc*(i) = {i, parent(i),
 * parent(parent(i)), ...} ("CAST", section 2: the target model verifies the
 * draft tree's tokens in one forward pass; EAGLE-2/3 dynamic draft trees).
 *
 * All storage is bf16 bit patterns (uint16), upcast exactly to double.
 * Layouts: q [L][nq][Hq][d]; pools [L][NB][Hkv][bs][d]; tables [rows][MB].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t L, nq, Hq, Hkv, d, bs, NB, MB;
    double scale;
} oracle_shape;

static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Steps 2-4 for one query vector over an explicit list of key positions. */
static void attend_one(const oracle_shape *s, int l, int g, const uint16_t *q,
                       const uint16_t *kp, const uint16_t *vp, const int32_t *table,
                       const int32_t *pos, int n, double *z, double *out, double *lse)
{
    const int d = s->d;
    for (int i = 0; i < n; ++i) {
        int t = pos[i];
        int blk = table[t / s->bs];
        int slot = t % s->bs;
        const uint16_t *k = kp + ((((size_t)l * s->NB + blk) * s->Hkv + g) * s->bs + slot) * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c)
            acc += bf16_to_double(q[c]) * bf16_to_double(k[c]);
        z[i] = acc * s->scale;
    }
    double zmax = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (z[i] > zmax) zmax = z[i];
    double sum = 0.0;
    for (int i = 0; i < n; ++i) {
        z[i] = exp(z[i] - zmax);
        sum += z[i];
    }
    for (int c = 0; c < d; ++c) out[c] = 0.0;
    for (int i = 0; i < n; ++i) {
        int t = pos[i];
        int blk = table[t / s->bs];
        int slot = t % s->bs;
        const uint16_t *v = vp + ((((size_t)l * s->NB + blk) * s->Hkv + g) * s->bs + slot) * d;
        double p = z[i] / sum;
        for (int c = 0; c < d; ++c)
            out[c] += p * bf16_to_double(v[c]);
    }
    *lse = zmax + log(sum);
}

static int check_table(const oracle_shape *s, const int32_t *table, int len)
{
    if (len <= 0 || (len + s->bs - 1) / s->bs > s->MB) return -1;
    for (int j = 0; j < (len + s->bs - 1) / s->bs; ++j)
        if (table[j] < 0 || table[j] >= s->NB) return -1;
    return 0;
}

/*
 * Decode attention.  If samples != NULL, computes only the n_samples triples
 * (layer, query, head) given there and writes out[n_samples][d], lse[n_samples];
 * otherwise computes everything into out[L][nq][Hq][d], lse[L][nq][Hq].
 * Returns 0, or -1 for an empty sequence or a block id outside the pool.
 */
int oracle_decode(const oracle_shape *s, const uint16_t *q, const uint16_t *kp,
                  const uint16_t *vp, const int32_t *tables, const int32_t *lens,
                  const int32_t *samples, int64_t n_samples, double *out, double *lse,
                  int nthreads)
{
    const int G = s->Hq / s->Hkv;
    for (int r = 0; r < s->nq; ++r)
        if (check_table(s, tables + (size_t)r * s->MB, lens[r])) return -1;
    int64_t total = samples ? n_samples : (int64_t)s->L * s->nq * s->Hq;
    int maxlen = 0;
    for (int r = 0; r < s->nq; ++r)
        if (lens[r] > maxlen) maxlen = lens[r];
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)maxlen);
        int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)maxlen);
#pragma omp for schedule(dynamic, 4)
        for (int64_t i = 0; i < total; ++i) {
            int l, r, h;
            if (samples) {
                l = samples[3 * i]; r = samples[3 * i + 1]; h = samples[3 * i + 2];
            } else {
                l = (int)(i / ((int64_t)s->nq * s->Hq));
                r = (int)((i / s->Hq) % s->nq);
                h = (int)(i % s->Hq);
            }
            int n = lens[r];
            for (int t = 0; t < n; ++t) pos[t] = t;
            const uint16_t *qv = q + (((size_t)l * s->nq + r) * s->Hq + h) * s->d;
            attend_one(s, l, h / G, qv, kp, vp, tables + (size_t)r * s->MB, pos, n, z,
                       out + (size_t)i * s->d, lse + i);
        }
        free(z);
        free(pos);
    }
    return 0;
}

/*
 * Tree-verify attention.  Batch of B sequences (table row b, context length
 * ctx[b]); n draft nodes each, parent[b][i] < i or -1; query row r = b*n + i.
 * Sampling as in oracle_decode.  Returns -1 on a bad parent pointer, an
 * empty context combined with no draft, or a block id outside the pool.
 */
int oracle_verify(const oracle_shape *s, int B, int n, const uint16_t *q, const uint16_t *kp,
                  const uint16_t *vp, const int32_t *tables, const int32_t *ctx,
                  const int32_t *parent, const int32_t *samples, int64_t n_samples,
                  double *out, double *lse, int nthreads)
{
    const int G = s->Hq / s->Hkv;
    int maxlen = 0;
    for (int b = 0; b < B; ++b) {
        if (ctx[b] < 0 || check_table(s, tables + (size_t)b * s->MB, ctx[b] + n)) return -1;
        for (int i = 0; i < n; ++i) {
            int p = parent[(size_t)b * n + i];
            if (p >= i || p < -1) return -1;
        }
        if (ctx[b] + n > maxlen) maxlen = ctx[b] + n;
    }
    int64_t total = samples ? n_samples : (int64_t)s->L * B * n * s->Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)maxlen);
        int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (size_t)maxlen);
#pragma omp for schedule(dynamic, 4)
        for (int64_t it = 0; it < total; ++it) {
            int l, r, h;
            if (samples) {
                l = samples[3 * it]; r = samples[3 * it + 1]; h = samples[3 * it + 2];
            } else {
                l = (int)(it / ((int64_t)B * n * s->Hq));
                r = (int)((it / s->Hq) % ((int64_t)B * n));
                h = (int)(it % s->Hq);
            }
            int b = r / n, i = r % n;
            int cnt = 0;
            for (int t = 0; t < ctx[b]; ++t) pos[cnt++] = t;
            /* ancestors-or-self, walking parent pointers up to a root */
            for (int j = i; j >= 0; j = parent[(size_t)b * n + j]) pos[cnt++] = ctx[b] + j;
            const uint16_t *qv = q + (((size_t)l * s->nq + r) * s->Hq + h) * s->d;
            attend_one(s, l, h / G, qv, kp, vp, tables + (size_t)b * s->MB, pos, cnt, z,
                       out + (size_t)it * s->d, lse + it);
        }
        free(z);
        free(pos);
    }
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
