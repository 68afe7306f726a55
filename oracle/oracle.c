/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged-KV decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark load it.  It shares no header, helper or constant with the
 * CUDA path.
 *
 * Sources (page title, section):
 *   [PA]  "論文解説: PagedAttention — 仮想メモリ着想のKVキャッシュ管理でLLMサービングを高効率化"
 *         (0h-n0.github.io, arXiv 2309.06180 explainer)
 *   [VA]  "論文解説: vAttention - PagedAttentionを使わないLLMサービング向け動的メモリ管理"
 *         (0h-n0.github.io, arXiv 2405.04437 explainer)
 *
 * Data layout of the physical KV pool (the pseudocode's kv_cache, shape
 * (blocks, B, 2, d), widened to several KV heads):
 *     pool[NB][B][2][H_kv][D], index 0 on the third axis is K, 1 is V.
 * Element types are carried as raw 16-bit patterns: dtype 0 = IEEE binary16,
 * dtype 1 = bfloat16.  Every value is widened to double before any arithmetic.
 *
 * Return codes: 0 ok, 1 invalid argument / out-of-range index, 2 allocation failure.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_INVALID 1
#define ORC_NOMEM 2

/* ---------------------------------------------------------------------------
 * 16-bit float decoding, written from the format definitions.
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * bfloat16: the upper half of an IEEE binary32.
 * ------------------------------------------------------------------------- */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0) {
        mag = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 / 2^10 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexp(1.0 + (double)frac / 1024.0, expo - 15);
    }
    return sign ? -mag : mag;
}

double oracle_bf16_to_double(uint16_t b) {
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double widen(uint16_t x, int dtype) {
    return dtype == 0 ? oracle_half_to_double(x) : oracle_bf16_to_double(x);
}

/* ---------------------------------------------------------------------------
 * Sizes.
 * [PA] 技術的詳細 / KVキャッシュのメモリ要件: bytes = 2 (K and V) x element bytes x
 * tokens x layers x heads x head dim.  With fp16 this is the page's 4*t*L*H*D_h.
 * ------------------------------------------------------------------------- */
double oracle_kv_cache_bytes(double tokens, double layers, double heads, double head_dim, double elem_bytes) {
    return 2.0 * elem_bytes * tokens * layers * heads * head_dim;
}

/* [VA] 技術的詳細 / 仮想メモリの事前予約 and the fine-grained page table: one K (or V)
 * buffer of one layer holds H*D*P bytes per token, so a page of page_bytes holds
 * page_bytes / (H*D*P) tokens. */
double oracle_tokens_per_page(double page_bytes, double kv_heads, double head_dim, double elem_bytes) {
    return page_bytes / (kv_heads * head_dim * elem_bytes);
}

/* ---------------------------------------------------------------------------
 * Cache write ([PA] block definition and block table: token t of a sequence
 * lives in logical block t/B at offset t%B; slot = physical block * B + offset).
 * k, v: [T][H_kv][D].  slot < 0 means "no write" (padding).
 * ------------------------------------------------------------------------- */
int oracle_reshape_and_cache(const uint16_t* k, const uint16_t* v, uint16_t* pool, const int64_t* slot_mapping, int T,
                             int NB, int B, int H_kv, int D) {
    if (T < 0 || NB <= 0 || B <= 0 || H_kv <= 0 || D <= 0) return ORC_INVALID;
    const int64_t row = (int64_t)H_kv * D; /* elements of one token's K (or V) */
    for (int i = 0; i < T; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)NB * B) return ORC_INVALID;
        int64_t blk = slot / B, off = slot % B;
        for (int64_t e = 0; e < row; ++e) {
            pool[((blk * B + off) * 2 + 0) * row + e] = k[(int64_t)i * row + e];
            pool[((blk * B + off) * 2 + 1) * row + e] = v[(int64_t)i * row + e];
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Copy-on-write block copy ([PA] 技術的詳細 / Copy-on-Write: a shared block is
 * copied before it is written).  pairs: [n][2] = (src, dst); the whole block
 * (B tokens x K,V x H_kv x D) is copied.  All copies read the pool as it was
 * before the call (the pairs must not chain).
 * ------------------------------------------------------------------------- */
int oracle_copy_blocks(uint16_t* pool, const int64_t* pairs, int n, int NB, int B, int H_kv, int D) {
    if (n < 0) return ORC_INVALID;
    const int64_t blk_elems = (int64_t)B * 2 * H_kv * D;
    for (int i = 0; i < n; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= NB || d < 0 || d >= NB) return ORC_INVALID;
        for (int j = 0; j < n; ++j) /* a destination may not also be read in the same call */
            if (pairs[2 * j] == d || (j != i && pairs[2 * j + 1] == d)) return ORC_INVALID;
    }
    for (int i = 0; i < n; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        memmove(pool + d * blk_elems, pool + s * blk_elems, (size_t)blk_elems * sizeof(uint16_t));
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Swap copy between two pools ([PA] 実装のポイント: a preempted request's KV
 * cache is moved to CPU memory and back).  pairs: [n][2] = (src block in
 * src_pool, dst block in dst_pool); whole blocks of blk_elems elements.
 * ------------------------------------------------------------------------- */
int oracle_swap_blocks(uint16_t* dst_pool, int NB_dst, const uint16_t* src_pool, int NB_src, const int64_t* pairs,
                       int n, int64_t blk_elems) {
    if (n < 0 || blk_elems <= 0) return ORC_INVALID;
    for (int i = 0; i < n; ++i) {
        int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
        if (s < 0 || s >= NB_src || d < 0 || d >= NB_dst) return ORC_INVALID;
        for (int j = 0; j < i; ++j)
            if (pairs[2 * j + 1] == d) return ORC_INVALID; /* destinations are distinct */
    }
    for (int i = 0; i < n; ++i)
        memcpy(dst_pool + pairs[2 * i + 1] * blk_elems, src_pool + pairs[2 * i] * blk_elems,
               (size_t)blk_elems * sizeof(uint16_t));
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Decode attention, plain definition ([PA] 技術的詳細 / PagedAttentionアルゴリズム,
 * decode equation for o_t):  for query q of head h,
 *     x_t = (q . K_t) * scale,   o = sum_t softmax(x)_t V_t,   t = 0 .. ctx-1,
 * where K_t, V_t are fetched through the block table (logical block t/B ->
 * physical block, offset t%B).  The exponentials are taken relative to the
 * maximum score, which leaves the quotient unchanged.  Query head h reads KV
 * head h / (H_q / H_kv).
 *
 * Addressing is delegated to a small fetch function so the paged and the
 * contiguous layouts share the attention definition and nothing else.
 * ------------------------------------------------------------------------- */
typedef struct {
    const uint16_t* pool;
    const int32_t* tables;
    int MB, NB, B;
    const uint16_t* kbuf;
    const uint16_t* vbuf;
    const int32_t* req_ids;
    int S_max, N_max;
    int H_kv, D;
    int paged;
} kv_source;

/* pointer to the D elements of K (which=0) or V (which=1) of token t, sequence s, KV head g; NULL if out of range */
static const uint16_t* fetch_row(const kv_source* src, int s, int t, int g, int which) {
    if (src->paged) {
        int lb = t / src->B, off = t % src->B;
        if (lb >= src->MB) return NULL;
        int32_t pb = src->tables[(int64_t)s * src->MB + lb];
        if (pb < 0 || pb >= src->NB) return NULL;
        int64_t idx = ((((int64_t)pb * src->B + off) * 2 + which) * src->H_kv + g) * src->D;
        return src->pool + idx;
    } else {
        /* [VA] リクエスト単位のKVキャッシュインデキシング: request r occupies the
         * sub-tensor starting at r * S, S = max_context * H * D elements; an
         * identifier outside [0, max_batch) is rejected. */
        int32_t r = src->req_ids[s];
        if (r < 0 || r >= src->N_max || t >= src->S_max) return NULL;
        int64_t idx = (((int64_t)r * src->S_max + t) * src->H_kv + g) * src->D;
        return (which ? src->vbuf : src->kbuf) + idx;
    }
}

/* out receives the row only at the end; it is never used as an accumulator, so a row listed
 * twice and computed by two threads at once still ends up with the right values. */
static int attend_one(double* out, const uint16_t* q, const kv_source* src, int s, int h, int n, int G, double scale,
                      int dtype, double* x, double* acc) {
    const int D = src->D, g = h / G;
    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int t = 0; t < n; ++t) {
        const uint16_t* kr = fetch_row(src, s, t, g, 0);
        if (!kr) return ORC_INVALID;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += widen(q[d], dtype) * widen(kr[d], dtype);
        x[t] = dot * scale;
        if (x[t] > m) m = x[t];
    }
    /* pass 2: normaliser and weighted sum of V */
    double z = 0.0;
    for (int t = 0; t < n; ++t) {
        x[t] = exp(x[t] - m);
        z += x[t];
    }
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int t = 0; t < n; ++t) {
        const uint16_t* vr = fetch_row(src, s, t, g, 1);
        if (!vr) return ORC_INVALID;
        double w = x[t] / z;
        for (int d = 0; d < D; ++d) acc[d] += w * widen(vr[d], dtype);
    }
    for (int d = 0; d < D; ++d) out[d] = acc[d];
    return ORC_OK;
}

/* Runs attend_one over a list of (seq, query head) pairs, or over all of them
 * when pairs == NULL.  out: [N][H_q][D] (only the listed rows are written).
 * The thread count only splits independent rows; each row is summed in order. */
static int attend_rows(double* out, const uint16_t* q, const kv_source* src, const int32_t* ctx, int N, int H_q, int H_kv,
                       int D, double scale, int dtype, const int32_t* pairs, int npairs, int nthreads, int max_n) {
    if (N <= 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || H_q % H_kv) return ORC_INVALID;
    const int G = H_q / H_kv;
    const int64_t rows = pairs ? npairs : (int64_t)N * H_q;
    for (int s = 0; s < N; ++s)
        if (ctx[s] < 1 || ctx[s] > max_n) return ORC_INVALID; /* an empty context has no softmax */
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)((max_n > 0 ? max_n : 1) + D));
        if (!x) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORC_NOMEM;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < rows; ++r) {
                int s, h;
                if (pairs) {
                    s = pairs[2 * r];
                    h = pairs[2 * r + 1];
                } else {
                    s = (int)(r / H_q);
                    h = (int)(r % H_q);
                }
                int rc = ORC_INVALID;
                if (s >= 0 && s < N && h >= 0 && h < H_q)
                    rc = attend_one(out + ((int64_t)s * H_q + h) * D, q + ((int64_t)s * H_q + h) * D, src, s, h, ctx[s], G,
                                    scale, dtype, x, x + (max_n > 0 ? max_n : 1));
                if (rc != ORC_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                    status = rc;
                }
            }
            free(x);
        }
    }
    (void)nthreads;
    return status;
}

/* Paged decode.  q: [N][H_q][D]; pool: [NB][B][2][H_kv][D]; tables: [N][MB];
 * ctx: [N] (each >= 1 and <= MB*B); out: [N][H_q][D] fp64. */
int oracle_paged_decode(double* out, const uint16_t* q, const uint16_t* pool, const int32_t* tables, const int32_t* ctx,
                        int N, int H_q, int H_kv, int D, int B, int MB, int NB, double scale, int dtype,
                        const int32_t* pairs, int npairs, int nthreads) {
    if (B <= 0 || MB <= 0 || NB <= 0) return ORC_INVALID;
    kv_source src;
    memset(&src, 0, sizeof src);
    src.pool = pool;
    src.tables = tables;
    src.MB = MB;
    src.NB = NB;
    src.B = B;
    src.H_kv = H_kv;
    src.D = D;
    src.paged = 1;
    return attend_rows(out, q, &src, ctx, N, H_q, H_kv, D, scale, dtype, pairs, npairs, nthreads, MB * B);
}

/* Contiguous (unpaged) decode over per-request K and V buffers [N_max][S_max][H_kv][D];
 * sequence s reads request req_ids[s]. */
int oracle_contiguous_decode(double* out, const uint16_t* q, const uint16_t* kbuf, const uint16_t* vbuf,
                             const int32_t* req_ids, const int32_t* ctx, int N, int H_q, int H_kv, int D, int S_max,
                             int N_max, double scale, int dtype, const int32_t* pairs, int npairs, int nthreads) {
    if (S_max <= 0 || N_max <= 0) return ORC_INVALID;
    kv_source src;
    memset(&src, 0, sizeof src);
    src.kbuf = kbuf;
    src.vbuf = vbuf;
    src.req_ids = req_ids;
    src.S_max = S_max;
    src.N_max = N_max;
    src.H_kv = H_kv;
    src.D = D;
    src.paged = 0;
    return attend_rows(out, q, &src, ctx, N, H_q, H_kv, D, scale, dtype, pairs, npairs, nthreads, S_max);
}

/* ---------------------------------------------------------------------------
 * Paged prefill attention ([PA] 実装のポイント: the paged kernel serves both the
 * prefill and the decode phase).  Sequence s holds ctx[s] tokens in the pool;
 * its last q_len_s = q_start[s+1] - q_start[s] tokens are the chunk being
 * prefilled, with queries in rows q_start[s] .. q_start[s+1]-1 of q
 * ([T][H_q][D]).  Query i of the chunk sits at position p = ctx - q_len + i and
 * attends causally to positions 0 .. p (the decode equation with the context
 * cut at p).  out: [T][H_q][D].  Two-pass fp64 per row, like the decode oracle.
 * ------------------------------------------------------------------------- */
int oracle_paged_prefill(double* out, const uint16_t* q, const uint16_t* pool, const int32_t* tables,
                         const int32_t* ctx, const int32_t* q_start, int N, int H_q, int H_kv, int D, int B, int MB,
                         int NB, double scale, int dtype, const int32_t* rows, int nrows, int nthreads) {
    if (N <= 0 || H_q <= 0 || H_kv <= 0 || D <= 0 || H_q % H_kv || B <= 0 || MB <= 0 || NB <= 0) return ORC_INVALID;
    for (int s = 0; s < N; ++s) {
        const int ql = q_start[s + 1] - q_start[s];
        if (ql < 0 || ql > ctx[s] || ctx[s] > MB * B || (ql == 0 && ctx[s] < 0)) return ORC_INVALID;
    }
    const int T = q_start[N];
    const int G = H_q / H_kv;
    kv_source src;
    memset(&src, 0, sizeof src);
    src.pool = pool;
    src.tables = tables;
    src.MB = MB;
    src.NB = NB;
    src.B = B;
    src.H_kv = H_kv;
    src.D = D;
    src.paged = 1;
    const int64_t total = rows ? nrows : (int64_t)T * H_q;
    int status = ORC_OK;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* x = (double*)malloc(sizeof(double) * ((size_t)MB * B + D));
        if (!x) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            status = ORC_NOMEM;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < total; ++r) {
                /* row = (query token t, head h) */
                const int64_t row = rows ? rows[r] : r;
                const int t = (int)(row / H_q), h = (int)(row % H_q);
                int s = 0;
                while (s < N && q_start[s + 1] <= t) ++s;
                int rc = ORC_INVALID;
                if (t >= 0 && t < T && s < N) {
                    const int ql = q_start[s + 1] - q_start[s];
                    const int pos = ctx[s] - ql + (t - q_start[s]);
                    rc = attend_one(out + row * D, q + row * D, &src, s, h, pos + 1, G, scale, dtype, x,
                                    x + (size_t)MB * B);
                }
                if (rc != ORC_OK) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
                    status = rc;
                }
            }
            free(x);
        }
    }
    (void)nthreads;
    return status;
}

/* ---------------------------------------------------------------------------
 * Block-streaming decode, following the explainer's paged_attention_decode
 * pseudocode ([PA] アルゴリズムの擬似コード): walk the block table in logical
 * order; for each block compute the block's scores, raise the running maximum,
 * rescale the running output and exponential sum by exp(old max - new max), add
 * the block's exponentials and their V-weighted sum; divide at the end.
 * Only slots t < ctx take part (the pseudocode scores whole blocks; the unused
 * tail of the last block is excluded here).  One (seq, query head) row.
 * ------------------------------------------------------------------------- */
int oracle_paged_decode_online_row(double* out, const uint16_t* q, const uint16_t* pool, const int32_t* table, int ctx,
                                   int H_kv, int D, int B, int NB, int g, double scale, int dtype) {
    if (ctx < 1 || B <= 0 || g < 0 || g >= H_kv) return ORC_INVALID;
    double max_score = -INFINITY, sum_exp = 0.0;
    double* score = (double*)malloc(sizeof(double) * (size_t)B);
    if (!score) return ORC_NOMEM;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    const int nblocks = (ctx + B - 1) / B;
    for (int lb = 0; lb < nblocks; ++lb) {
        int32_t pb = table[lb];
        if (pb < 0 || pb >= NB) {
            free(score);
            return ORC_INVALID;
        }
        int valid = ctx - lb * B < B ? ctx - lb * B : B;
        double block_max = -INFINITY;
        for (int j = 0; j < valid; ++j) {
            const uint16_t* kr = pool + ((((int64_t)pb * B + j) * 2 + 0) * H_kv + g) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += widen(q[d], dtype) * widen(kr[d], dtype);
            score[j] = dot * scale;
            if (score[j] > block_max) block_max = score[j];
        }
        double new_max = block_max > max_score ? block_max : max_score;
        double rescale = exp(max_score - new_max); /* exp(-inf) = 0 on the first block */
        for (int d = 0; d < D; ++d) out[d] *= rescale;
        sum_exp *= rescale;
        for (int j = 0; j < valid; ++j) {
            double e = exp(score[j] - new_max);
            const uint16_t* vr = pool + ((((int64_t)pb * B + j) * 2 + 1) * H_kv + g) * D;
            for (int d = 0; d < D; ++d) out[d] += e * widen(vr[d], dtype);
            sum_exp += e;
        }
        max_score = new_max;
    }
    for (int d = 0; d < D; ++d) out[d] /= sum_exp;
    free(score);
    return ORC_OK;
}

/* ---------------------------------------------------------------------------
 * Split-context partials and their merge.  The context [0, ctx) is cut into
 * consecutive partitions of P tokens; each partition keeps the same three
 * running quantities the block-streaming pseudocode keeps (maximum, exponential
 * sum, unnormalised output).  Maxima are stored in base-2 units
 * (m2 = max_t x_t * log2 e) so that a partition's weights are 2^(x_t log2 e - m2).
 * Merging: M = max_p m2_p, o = sum_p 2^(m2_p - M) acc_p / sum_p 2^(m2_p - M) l_p.
 * ------------------------------------------------------------------------- */
int oracle_paged_partials_row(double* m2, double* l, double* acc /*[P][D]*/, const uint16_t* q, const uint16_t* pool,
                              const int32_t* table, int ctx, int H_kv, int D, int B, int NB, int g, double scale,
                              int dtype, int part_tokens, int nparts) {
    if (ctx < 1 || part_tokens <= 0 || (ctx + part_tokens - 1) / part_tokens > nparts) return ORC_INVALID;
    const double log2e = 1.0 / log(2.0);
    for (int p = 0; p < nparts; ++p) {
        int t0 = p * part_tokens, t1 = t0 + part_tokens < ctx ? t0 + part_tokens : ctx;
        double* a = acc + (int64_t)p * D;
        for (int d = 0; d < D; ++d) a[d] = 0.0;
        m2[p] = -INFINITY;
        l[p] = 0.0;
        if (t0 >= ctx) continue;
        double mx = -INFINITY;
        for (int t = t0; t < t1; ++t) {
            int32_t pb = table[t / B];
            if (pb < 0 || pb >= NB) return ORC_INVALID;
            const uint16_t* kr = pool + ((((int64_t)pb * B + t % B) * 2 + 0) * H_kv + g) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += widen(q[d], dtype) * widen(kr[d], dtype);
            double x = dot * scale * log2e;
            if (x > mx) mx = x;
        }
        for (int t = t0; t < t1; ++t) {
            int32_t pb = table[t / B];
            const uint16_t* kr = pool + ((((int64_t)pb * B + t % B) * 2 + 0) * H_kv + g) * D;
            const uint16_t* vr = pool + ((((int64_t)pb * B + t % B) * 2 + 1) * H_kv + g) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += widen(q[d], dtype) * widen(kr[d], dtype);
            double w = exp2(dot * scale * log2e - mx);
            l[p] += w;
            for (int d = 0; d < D; ++d) a[d] += w * widen(vr[d], dtype);
        }
        m2[p] = mx;
    }
    return ORC_OK;
}

/* rows: R independent (m2, l, acc) sets of nparts[r] partitions each, laid out
 * [R][P] and [R][P][D]; out: [R][D]. */
int oracle_partition_merge(double* out, const double* m2, const double* l, const double* acc, const int32_t* nparts,
                           int R, int P, int D) {
    for (int r = 0; r < R; ++r) {
        int np = nparts[r];
        if (np < 1 || np > P) return ORC_INVALID;
        double M = -INFINITY;
        for (int p = 0; p < np; ++p)
            if (m2[(int64_t)r * P + p] > M) M = m2[(int64_t)r * P + p];
        double den = 0.0;
        double* o = out + (int64_t)r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int p = 0; p < np; ++p) {
            double w = exp2(m2[(int64_t)r * P + p] - M);
            den += w * l[(int64_t)r * P + p];
            for (int d = 0; d < D; ++d) o[d] += w * acc[((int64_t)r * P + p) * D + d];
        }
        for (int d = 0; d < D; ++d) o[d] /= den;
    }
    return ORC_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
