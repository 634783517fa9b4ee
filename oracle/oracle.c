/*
 * fp64 CPU oracle for exact attention, its paged-KV-cache variant and the
 * KV-cache append.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it follows ("Fast Attention Kernels and Operator Fusion"):
 *   - section "FlashAttention-Style Kernels", attention equation:
 *       Attention(Q,K,V) = softmax(Q K^T / sqrt(d) + M) V
 *     computed the plain way the same section describes first: the whole
 *     score matrix of a head is materialised (here in fp64), then each row is
 *     normalised by softmax and multiplied into V.  The scale is passed in
 *     explicitly (1/sqrt(d) in every workload).
 *   - section "Paged Attention Kernels": keys and values live in fixed-size
 *     blocks (16 tokens, the block size of the vLLM example there); a
 *     per-sequence block table maps logical block b to a physical block, and
 *     logical token t is read from physical block table[t / 16], offset
 *     t % 16.  The oracle gathers each sequence into contiguous storage with a
 *     naive loop and then applies the plain definition above.
 *   - section "Operator Fusion", fusion list item "updating the KV cache while
 *     transforming key and value tensors": the append writes each new token's
 *     K/V row into its cache slot (slot = block * 16 + offset), rounding fp32
 *     inputs to bf16; with the list item "applying rotary position embeddings
 *     to queries and keys", the fused variant rotates q and k first (the
 *     rotation itself is a reading, stated at ora_rope_cache_append).
 *
 * Readings where the pages are silent (also listed in the design notes):
 *   - grouped-query attention: query head h reads kv head h / (Hq / Hkv);
 *   - causal masking with Tq <= Tk is bottom-right aligned: query i sits at
 *     position i + Tk - Tq and sees keys j <= i + Tk - Tq;
 *   - a user mask M is float32 [Tq, Tk], broadcast over batch and heads, and
 *     adds to the causal mask when both are given;
 *   - a row whose scores are all -inf yields output 0 and LSE = -inf;
 *   - the LSE is the natural-log log-sum-exp of the row's final scores;
 *   - cache layout [num_blocks, Hkv, 16, d]; a negative slot is skipped;
 *   - fp32 -> bf16 rounding is IEEE round-to-nearest-even.
 *
 * All floating-point inputs reach the arithmetic as bf16 bit patterns decoded
 * exactly to double; accumulation is fp64 throughout.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORA_OK 0
#define ORA_ERR_ARG 1
#define ORA_ERR_BOUNDS 2
#define ORA_ERR_NOMEM 3

/* ---------------------------------------------------------------- bf16 -- */

static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE 754 round-to-nearest-even of a binary32 value to bfloat16 (the top 16
 * bits of binary32).  Adding 0x7FFF plus the lowest kept bit and truncating
 * rounds halfway cases to the even neighbour; NaNs are kept quiet. */
uint16_t ora_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep_lsb = (u >> 16) & 1u;
    u += 0x7FFFu + keep_lsb;
    return (uint16_t)(u >> 16);
}

void ora_bf16_rne_array(const float* x, uint16_t* y, long n)
{
    for (long i = 0; i < n; ++i)
        y[i] = ora_bf16_rne(x[i]);
}

void ora_bf16_to_double_array(const uint16_t* x, double* y, long n)
{
    for (long i = 0; i < n; ++i)
        y[i] = bf16_to_double(x[i]);
}

/* ------------------------------------------------------- one head, rows -- */

/*
 * Attention for one (batch, head): rows [r0, r1) of a Tq x Tk problem.
 *   Q: Tq rows of d doubles (row stride d), K, V: Tk rows of d doubles.
 *   S: scratch of (r1 - r0) * Tk doubles -- the materialised score matrix.
 *   O: (r1 - r0) rows of d doubles; lse: r1 - r0 doubles (may be NULL).
 */
static void attend_rows(const double* Q, const double* K, const double* V,
                        const float* M, int Tq, int Tk, int d, int causal,
                        double scale, int r0, int r1, double* S, double* O,
                        double* lse)
{
    const int off = Tk - Tq;
    /* score matrix S = Q K^T * scale + M (+ causal -inf) */
    for (int i = r0; i < r1; ++i) {
        double* srow = S + (long)(i - r0) * Tk;
        const double* qi = Q + (long)i * d;
        for (int j = 0; j < Tk; ++j) {
            const double* kj = K + (long)j * d;
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += qi[c] * kj[c];
            double s = dot * scale;
            if (M)
                s += (double)M[(long)i * Tk + j];
            if (causal && j > i + off)
                s = -INFINITY;
            srow[j] = s;
        }
    }
    /* row-wise softmax, then P V */
    for (int i = r0; i < r1; ++i) {
        double* srow = S + (long)(i - r0) * Tk;
        double* orow = O + (long)(i - r0) * d;
        double mx = -INFINITY;
        for (int j = 0; j < Tk; ++j)
            if (srow[j] > mx)
                mx = srow[j];
        for (int c = 0; c < d; ++c)
            orow[c] = 0.0;
        if (mx == -INFINITY) {
            if (lse)
                lse[i - r0] = -INFINITY;
            continue;
        }
        double z = 0.0;
        for (int j = 0; j < Tk; ++j) {
            srow[j] = exp(srow[j] - mx);
            z += srow[j];
        }
        for (int j = 0; j < Tk; ++j) {
            double p = srow[j] / z;
            if (p == 0.0)
                continue;
            const double* vj = V + (long)j * d;
            for (int c = 0; c < d; ++c)
                orow[c] += p * vj[c];
        }
        if (lse)
            lse[i - r0] = mx + log(z);
    }
}

/* ------------------------------------------------------ thread helpers -- */

typedef struct {
    pthread_mutex_t lock;
    long next;
    long total;
    int status;
} work_queue;

static long take_unit(work_queue* wq)
{
    pthread_mutex_lock(&wq->lock);
    long u = wq->next < wq->total ? wq->next++ : -1;
    pthread_mutex_unlock(&wq->lock);
    return u;
}

static void set_status(work_queue* wq, int st)
{
    pthread_mutex_lock(&wq->lock);
    if (wq->status == ORA_OK)
        wq->status = st;
    pthread_mutex_unlock(&wq->lock);
}

static int run_threads(void* (*fn)(void*), void* arg, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads == 1) {
        fn(arg);
        return ORA_OK;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th)
        return ORA_ERR_NOMEM;
    int started = 0;
    for (int t = 0; t < nthreads; ++t)
        if (pthread_create(&th[started], NULL, fn, arg) == 0)
            ++started;
    if (started == 0)
        fn(arg);
    for (int t = 0; t < started; ++t)
        pthread_join(th[t], NULL);
    free(th);
    return ORA_OK;
}

/* ------------------------------------------------- contiguous attention -- */

typedef struct {
    work_queue wq;
    const uint16_t *q, *k, *v;
    const float* mask;
    double *out, *lse;
    int B, Tq, Tk, Hq, Hkv, d, causal;
    double scale;
} dense_job;

static void* dense_worker(void* p)
{
    dense_job* J = (dense_job*)p;
    const int d = J->d, Tq = J->Tq, Tk = J->Tk;
    double* Q = (double*)malloc(sizeof(double) * (size_t)Tq * d);
    double* K = (double*)malloc(sizeof(double) * (size_t)Tk * d);
    double* V = (double*)malloc(sizeof(double) * (size_t)Tk * d);
    double* S = (double*)malloc(sizeof(double) * (size_t)Tq * Tk);
    double* O = (double*)malloc(sizeof(double) * (size_t)Tq * d);
    double* L = (double*)malloc(sizeof(double) * (size_t)Tq);
    if (!Q || !K || !V || !S || !O || !L) {
        set_status(&J->wq, ORA_ERR_NOMEM);
        goto done;
    }
    for (long u; (u = take_unit(&J->wq)) >= 0;) {
        const int b = (int)(u / J->Hq), h = (int)(u % J->Hq);
        const int hk = h / (J->Hq / J->Hkv);
        for (int i = 0; i < Tq; ++i)
            for (int c = 0; c < d; ++c)
                Q[(long)i * d + c] = bf16_to_double(J->q[(((long)b * Tq + i) * J->Hq + h) * d + c]);
        for (int j = 0; j < Tk; ++j)
            for (int c = 0; c < d; ++c) {
                long src = (((long)b * Tk + j) * J->Hkv + hk) * d + c;
                K[(long)j * d + c] = bf16_to_double(J->k[src]);
                V[(long)j * d + c] = bf16_to_double(J->v[src]);
            }
        attend_rows(Q, K, V, J->mask, Tq, Tk, d, J->causal, J->scale, 0, Tq, S, O, L);
        for (int i = 0; i < Tq; ++i) {
            memcpy(J->out + (((long)b * Tq + i) * J->Hq + h) * d, O + (long)i * d,
                   sizeof(double) * (size_t)d);
            if (J->lse)
                J->lse[((long)b * J->Hq + h) * Tq + i] = L[i];
        }
    }
done:
    free(Q); free(K); free(V); free(S); free(O); free(L);
    return NULL;
}

/*
 * q: bf16 bits [B, Tq, Hq, d]; k, v: bf16 bits [B, Tk, Hkv, d];
 * mask: float32 [Tq, Tk] or NULL; out: double [B, Tq, Hq, d];
 * lse: double [B, Hq, Tq] or NULL.
 */
int ora_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const float* mask, double* out, double* lse, int B, int Tq,
                  int Tk, int Hq, int Hkv, int d, int causal, double scale,
                  int nthreads)
{
    if (B < 0 || Tq < 0 || Tk < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0)
        return ORA_ERR_ARG;
    if (causal && Tq > Tk)
        return ORA_ERR_ARG;
    if ((long)B * Tq == 0)
        return ORA_OK;
    dense_job J;
    memset(&J, 0, sizeof J);
    pthread_mutex_init(&J.wq.lock, NULL);
    J.wq.total = (long)B * Hq;
    J.q = q; J.k = k; J.v = v; J.mask = mask; J.out = out; J.lse = lse;
    J.B = B; J.Tq = Tq; J.Tk = Tk; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.causal = causal; J.scale = scale;
    int st = run_threads(dense_worker, &J, nthreads);
    pthread_mutex_destroy(&J.wq.lock);
    return st != ORA_OK ? st : J.wq.status;
}

/*
 * Sampled rows of the same problem: rows[3*r .. 3*r+2] = (b, h, i).
 * out: double [nrows, d]; lse: double [nrows] or NULL.
 */
typedef struct {
    work_queue wq;
    const uint16_t *q, *k, *v;
    const float* mask;
    const int32_t* rows;
    double *out, *lse;
    int B, Tq, Tk, Hq, Hkv, d, causal;
    double scale;
} rows_job;

static void* rows_worker(void* p)
{
    rows_job* J = (rows_job*)p;
    const int d = J->d, Tk = J->Tk;
    double* Q = (double*)malloc(sizeof(double) * (size_t)J->Tq * d);
    double* K = (double*)malloc(sizeof(double) * (size_t)Tk * d);
    double* V = (double*)malloc(sizeof(double) * (size_t)Tk * d);
    double* S = (double*)malloc(sizeof(double) * (size_t)Tk);
    if (!Q || !K || !V || !S) {
        set_status(&J->wq, ORA_ERR_NOMEM);
        goto done;
    }
    long loaded_b = -1, loaded_hk = -1;
    for (long r; (r = take_unit(&J->wq)) >= 0;) {
        const int b = J->rows[3 * r], h = J->rows[3 * r + 1], i = J->rows[3 * r + 2];
        if (b < 0 || b >= J->B || h < 0 || h >= J->Hq || i < 0 || i >= J->Tq) {
            set_status(&J->wq, ORA_ERR_BOUNDS);
            continue;
        }
        const int hk = h / (J->Hq / J->Hkv);
        if (b != loaded_b || hk != loaded_hk) {
            for (int j = 0; j < Tk; ++j)
                for (int c = 0; c < d; ++c) {
                    long src = (((long)b * Tk + j) * J->Hkv + hk) * d + c;
                    K[(long)j * d + c] = bf16_to_double(J->k[src]);
                    V[(long)j * d + c] = bf16_to_double(J->v[src]);
                }
            loaded_b = b;
            loaded_hk = hk;
        }
        for (int c = 0; c < d; ++c)
            Q[(long)i * d + c] = bf16_to_double(J->q[(((long)b * J->Tq + i) * J->Hq + h) * d + c]);
        attend_rows(Q, K, V, J->mask, J->Tq, Tk, d, J->causal, J->scale, i, i + 1, S,
                    J->out + r * d, J->lse ? J->lse + r : NULL);
    }
done:
    free(Q); free(K); free(V); free(S);
    return NULL;
}

int ora_attention_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const float* mask, int B, int Tq, int Tk, int Hq, int Hkv,
                       int d, int causal, double scale, const int32_t* rows,
                       long nrows, double* out, double* lse, int nthreads)
{
    if (Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv != 0 || (causal && Tq > Tk))
        return ORA_ERR_ARG;
    rows_job J;
    memset(&J, 0, sizeof J);
    pthread_mutex_init(&J.wq.lock, NULL);
    J.wq.total = nrows;
    J.q = q; J.k = k; J.v = v; J.mask = mask; J.rows = rows; J.out = out; J.lse = lse;
    J.B = B; J.Tq = Tq; J.Tk = Tk; J.Hq = Hq; J.Hkv = Hkv; J.d = d;
    J.causal = causal; J.scale = scale;
    int st = run_threads(rows_worker, &J, nthreads);
    pthread_mutex_destroy(&J.wq.lock);
    return st != ORA_OK ? st : J.wq.status;
}

/* ------------------------------------------------------- paged storage -- */

/*
 * Logical-to-physical translation through the block table, written as a
 * plain loop: token t of sequence `seq` lives in physical block
 * block_table[seq][t / block_size] at offset t % block_size.
 * cache: bf16 bits [num_blocks, Hkv, block_size, d];
 * out:   bf16 bits [ctx_len, Hkv, d].
 */
int ora_gather_kv(const uint16_t* cache, const int32_t* block_table,
                  int max_blocks_per_seq, int num_blocks, int seq, int ctx_len,
                  int Hkv, int d, int block_size, uint16_t* out)
{
    if (ctx_len < 0 || ctx_len > max_blocks_per_seq * block_size)
        return ORA_ERR_BOUNDS;
    for (int t = 0; t < ctx_len; ++t) {
        int logical_block = t / block_size;
        int offset = t % block_size;
        int physical = block_table[(long)seq * max_blocks_per_seq + logical_block];
        if (physical < 0 || physical >= num_blocks)
            return ORA_ERR_BOUNDS;
        for (int h = 0; h < Hkv; ++h)
            for (int c = 0; c < d; ++c)
                out[((long)t * Hkv + h) * d + c] =
                    cache[(((long)physical * Hkv + h) * block_size + offset) * d + c];
    }
    return ORA_OK;
}

/*
 * Cache append: for each new token i with slot_mapping[i] >= 0, write its
 * Hkv x d key and value rows (bf16 bits) into slot slot_mapping[i], i.e.
 * block slot / block_size, offset slot % block_size.
 */
int ora_cache_append(const uint16_t* k, const uint16_t* v, const int32_t* slot_mapping,
                     int N, int Hkv, int d, int num_blocks, int block_size,
                     uint16_t* k_cache, uint16_t* v_cache)
{
    for (int i = 0; i < N; ++i) {
        long slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (long)num_blocks * block_size)
            return ORA_ERR_BOUNDS;
        long blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < Hkv; ++h)
            for (int c = 0; c < d; ++c) {
                long dst = ((blk * Hkv + h) * block_size + off) * d + c;
                long src = ((long)i * Hkv + h) * d + c;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
    }
    return ORA_OK;
}

/* ------------------------------------------------------ rotary + append -- */

/*
 * IEEE round-to-nearest-even of a double straight to bfloat16 (no
 * intermediate binary32 rounding): keep 8 significant bits of the value.
 */
static uint16_t bf16_rne_double(double x)
{
    if (x != x)
        return 0x7FC0u;
    if (x == 0.0)
        return signbit(x) ? 0x8000u : 0x0000u;
    double ax = fabs(x), r;
    if (ax < ldexp(1.0, -126)) {                /* bf16 subnormal range: spacing 2^-133 */
        r = nearbyint(ax * ldexp(1.0, 133)) * ldexp(1.0, -133);
    } else {
        int e;
        double m = frexp(ax, &e);               /* ax = m * 2^e, m in [1/2, 1) */
        r = ldexp(nearbyint(ldexp(m, 8)), e - 8);
    }
    float f = r >= ldexp(1.0, 128) ? INFINITY : (float)r;   /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)((u >> 16) | (x < 0 ? 0x8000u : 0u));
}

/*
 * Rotary position embedding of one d-channel row at table row `pos`.  The
 * pages name the fusion ("Operator Fusion", fusion list: applying rotary
 * position embeddings to queries and keys) but not the rotation; reading:
 * the rotate-half form, channel j paired with channel j + d/2 (j < d/2) and
 * turned by the angle whose cosine and sine sit at columns j and d/2 + j of
 * the caller's table cos_sin [max_pos, d]:
 *   y_j       = x_j cos - x_{j+d/2} sin
 *   y_{j+d/2} = x_{j+d/2} cos + x_j sin        (fp64)
 */
static void rope_row(const double* x, const float* cs, int d, double* y)
{
    int h = d / 2;
    for (int j = 0; j < h; ++j) {
        double c = (double)cs[j], s = (double)cs[h + j];
        y[j] = x[j] * c - x[h + j] * s;
        y[h + j] = x[h + j] * c + x[j] * s;
    }
}

/* rope_row over nrows rows (row i at table row pos[i]), fp64 in and out */
int ora_rope_f64(const double* x, const int32_t* pos, const float* cos_sin, int max_pos, long nrows, int d,
                 double* y)
{
    if (d <= 0 || d % 2)
        return ORA_ERR_ARG;
    for (long i = 0; i < nrows; ++i) {
        if (pos[i] < 0 || pos[i] >= max_pos)
            return ORA_ERR_BOUNDS;
        rope_row(x + i * d, cos_sin + (long)pos[i] * d, d, y + i * d);
    }
    return ORA_OK;
}

/*
 * Rotary embedding fused with the cache append ("Operator Fusion", fusion
 * list: applying rotary position embeddings to queries and keys; updating
 * the KV cache while transforming key and value tensors).  Token i sits at
 * table row positions[i].  Its Hq query rows are rotated into q_out; its Hkv
 * key rows are rotated and, with its unrotated value rows, written to slot
 * slot_mapping[i] exactly as ora_cache_append places them (a negative slot
 * skips the cache write only).  q and k come in as exact fp64 copies of the
 * caller's values (bf16 or fp32), v as bf16 bits; rotated values are rounded
 * once from fp64 to bf16 (RNE).
 */
int ora_rope_cache_append(const double* q, const double* k, const uint16_t* v, const int32_t* positions,
                          const float* cos_sin, int max_pos, const int32_t* slot_mapping, int N, int Hq,
                          int Hkv, int d, int num_blocks, int block_size, uint16_t* q_out,
                          uint16_t* k_cache, uint16_t* v_cache)
{
    double* x = malloc(sizeof(double) * 2 * (size_t)d);
    if (!x)
        return ORA_ERR_NOMEM;
    double* y = x + d;
    int st = ORA_OK;
    for (int i = 0; i < N && st == ORA_OK; ++i) {
        int pos = positions[i];
        if (pos < 0 || pos >= max_pos) {
            st = ORA_ERR_BOUNDS;
            break;
        }
        const float* cs = cos_sin + (long)pos * d;
        for (int h = 0; h < Hq; ++h) {
            long base = ((long)i * Hq + h) * d;
            for (int c = 0; c < d; ++c)
                x[c] = q[base + c];
            rope_row(x, cs, d, y);
            for (int c = 0; c < d; ++c)
                q_out[base + c] = bf16_rne_double(y[c]);
        }
        long slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (long)num_blocks * block_size) {
            st = ORA_ERR_BOUNDS;
            break;
        }
        long blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < Hkv; ++h) {
            long src = ((long)i * Hkv + h) * d;
            long dst = ((blk * Hkv + h) * block_size + off) * d;
            for (int c = 0; c < d; ++c)
                x[c] = k[src + c];
            rope_row(x, cs, d, y);
            for (int c = 0; c < d; ++c) {
                k_cache[dst + c] = bf16_rne_double(y[c]);
                v_cache[dst + c] = v[src + c];
            }
        }
    }
    free(x);
    return st;
}

/* --------------------------------------------------------- fp8 cache ---- */

/*
 * FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448).  Used for the 8-bit KV
 * cache: the pages mention 8-bit matrix arithmetic ("8-bit MMA") without a
 * scale convention; reading: one scale per cache (k_scale, v_scale), stored
 * code = e4m3(x / scale) with the division in binary32 and round to nearest
 * even, saturating at +-448; the value the code stands for is e4m3 * scale.
 */
double ora_e4m3_value(uint8_t code)
{
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                 /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* nearest E4M3 code to y (exact comparison in double), ties to the even
 * code, |y| beyond 448 saturates to +-448, NaN gives the NaN code.  The
 * positive codes 0 .. 0x7E increase with their value, so the two neighbours
 * of |y| are found by bisection and the nearer one is kept. */
uint8_t ora_e4m3_rne(float y)
{
    if (y != y)
        return 0x7F;
    double a = fabs((double)y);
    uint8_t best;
    if (a >= 448.0) {
        best = 0x7E;
    } else {
        int lo = 0, hi = 0x7E;                    /* value(lo) <= a < value(hi) */
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (ora_e4m3_value((uint8_t)mid) <= a)
                lo = mid;
            else
                hi = mid;
        }
        double dl = a - ora_e4m3_value((uint8_t)lo), dh = ora_e4m3_value((uint8_t)hi) - a;
        best = (uint8_t)(dl < dh ? lo : dh < dl ? hi : ((lo & 1) ? hi : lo));
    }
    return (uint8_t)(best | (y < 0 ? 0x80 : 0));
}

/* the same rounding by exhaustive search over all codes (test cross-check) */
uint8_t ora_e4m3_rne_exhaustive(float y)
{
    if (y != y)
        return 0x7F;
    double a = fabs((double)y);
    uint8_t best = 0;
    double berr = a;
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(ora_e4m3_value((uint8_t)c) - a);
        if (err < berr || (err == berr && (c & 1) == 0 && (best & 1))) {
            best = (uint8_t)c;
            berr = err;
        }
    }
    if (a > 448.0)
        best = 0x7E;
    return (uint8_t)(best | (y < 0 ? 0x80 : 0));
}

/* codes of x[i] / scale (x: binary32 values; division in binary32) */
void ora_quant_e4m3(const float* x, long n, float scale, uint8_t* out)
{
    for (long i = 0; i < n; ++i) {
        volatile float y = x[i] / scale;
        out[i] = ora_e4m3_rne(y);
    }
}

/*
 * Append into the 8-bit cache.  k, v: binary32 values [N, Hkv, d] (bf16
 * inputs decoded exactly).  K codes go to k_cache [num_blocks, Hkv, 16, d]
 * like the bf16 append; V codes go to v_cache [num_blocks, Hkv, d, 16], the
 * 16 tokens of a block contiguous for each channel (reading: the layout the
 * decode kernel reads as token pairs).  slot < 0 skips the token.
 */
int ora_cache_append_fp8(const float* k, const float* v, const int32_t* slot_mapping, int N, int Hkv, int d,
                         int num_blocks, float k_scale, float v_scale, uint8_t* k_cache, uint8_t* v_cache)
{
    for (int i = 0; i < N; ++i) {
        long slot = slot_mapping[i];
        if (slot < 0)
            continue;
        if (slot >= (long)num_blocks * 16)
            return ORA_ERR_BOUNDS;
        long blk = slot / 16, off = slot % 16;
        for (int h = 0; h < Hkv; ++h)
            for (int c = 0; c < d; ++c) {
                long src = ((long)i * Hkv + h) * d + c;
                uint8_t kq, vq;
                ora_quant_e4m3(k + src, 1, k_scale, &kq);
                ora_quant_e4m3(v + src, 1, v_scale, &vq);
                k_cache[((blk * Hkv + h) * 16 + off) * d + c] = kq;
                v_cache[((blk * Hkv + h) * d + c) * 16 + off] = vq;
            }
    }
    return ORA_OK;
}

/* ---------------------------------------------------- paged attention -- */

typedef struct {
    work_queue wq;
    const uint16_t *q, *kc, *vc;
    const uint8_t *kc8, *vc8;   /* 8-bit caches (when set, kc / vc are unused) */
    double k_scale, v_scale;
    const int32_t *bt, *ctx_lens, *q_lens;
    const long* q_start;
    const int32_t* rows; /* NULL: every row; else (seq, qi, h) triples */
    double *out, *lse;
    int num_seqs, max_blocks, num_blocks, Hq, Hkv, d, block_size, causal;
    double scale;
    int max_ctx;
} paged_job;

/* gathers sequence s's keys and values for kv head hk into K, V (doubles) */
static int gather_seq_head(const paged_job* J, int s, int hk, uint16_t* tmp,
                           double* K, double* V)
{
    const int ctx = J->ctx_lens[s], d = J->d;
    if (J->kc8) {  /* 8-bit caches: follow the block table, decode, scale */
        for (int t = 0; t < ctx; ++t) {
            long phys = J->bt[(long)s * J->max_blocks + t / 16];
            if (phys < 0 || phys >= J->num_blocks)
                return ORA_ERR_BOUNDS;
            long off = t % 16;
            for (int c = 0; c < d; ++c) {
                K[(long)t * d + c] = ora_e4m3_value(J->kc8[((phys * J->Hkv + hk) * 16 + off) * d + c]) * J->k_scale;
                V[(long)t * d + c] = ora_e4m3_value(J->vc8[((phys * J->Hkv + hk) * d + c) * 16 + off]) * J->v_scale;
            }
        }
        return ORA_OK;
    }
    int st = ora_gather_kv(J->kc, J->bt, J->max_blocks, J->num_blocks, s, ctx, J->Hkv, d,
                           J->block_size, tmp);
    if (st)
        return st;
    for (int t = 0; t < ctx; ++t)
        for (int c = 0; c < d; ++c)
            K[(long)t * d + c] = bf16_to_double(tmp[((long)t * J->Hkv + hk) * d + c]);
    st = ora_gather_kv(J->vc, J->bt, J->max_blocks, J->num_blocks, s, ctx, J->Hkv, d,
                       J->block_size, tmp);
    if (st)
        return st;
    for (int t = 0; t < ctx; ++t)
        for (int c = 0; c < d; ++c)
            V[(long)t * d + c] = bf16_to_double(tmp[((long)t * J->Hkv + hk) * d + c]);
    return ORA_OK;
}

static void* paged_worker(void* p)
{
    paged_job* J = (paged_job*)p;
    const int d = J->d, mc = J->max_ctx > 0 ? J->max_ctx : 1;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)mc * J->Hkv * d);
    double* K = (double*)malloc(sizeof(double) * (size_t)mc * d);
    double* V = (double*)malloc(sizeof(double) * (size_t)mc * d);
    double* Q = (double*)malloc(sizeof(double) * (size_t)mc * d);
    double* S = NULL; /* score matrix, grown to q_len x ctx as needed */
    size_t s_cap = 0;
    double* O = (double*)malloc(sizeof(double) * (size_t)mc * d);
    double* L = (double*)malloc(sizeof(double) * (size_t)mc);
    if (!tmp || !K || !V || !Q || !O || !L) {
        set_status(&J->wq, ORA_ERR_NOMEM);
        goto done;
    }
    int loaded_s = -1, loaded_hk = -1;
    for (long u; (u = take_unit(&J->wq)) >= 0;) {
        int s, h, r0, r1;
        if (J->rows) {
            s = J->rows[3 * u];
            r0 = J->rows[3 * u + 1];
            r1 = r0 + 1;
            h = J->rows[3 * u + 2];
            if (s < 0 || s >= J->num_seqs || h < 0 || h >= J->Hq || r0 < 0 || r0 >= J->q_lens[s]) {
                set_status(&J->wq, ORA_ERR_BOUNDS);
                continue;
            }
        } else {
            s = (int)(u / J->Hq);
            h = (int)(u % J->Hq);
            r0 = 0;
            r1 = J->q_lens[s];
        }
        const int ql = J->q_lens[s], ctx = J->ctx_lens[s];
        if (ql <= 0)
            continue;
        if (ql > ctx || ctx > J->max_blocks * J->block_size) {
            set_status(&J->wq, ORA_ERR_BOUNDS);
            continue;
        }
        const int hk = h / (J->Hq / J->Hkv);
        if (s != loaded_s || hk != loaded_hk) {
            int st = gather_seq_head(J, s, hk, tmp, K, V);
            if (st) {
                set_status(&J->wq, st);
                continue;
            }
            loaded_s = s;
            loaded_hk = hk;
        }
        size_t need = (size_t)(r1 - r0) * (size_t)ctx;
        if (need > s_cap) {
            free(S);
            S = (double*)malloc(sizeof(double) * need);
            s_cap = S ? need : 0;
            if (!S) {
                set_status(&J->wq, ORA_ERR_NOMEM);
                continue;
            }
        }
        for (int i = r0; i < r1; ++i)
            for (int c = 0; c < d; ++c)
                Q[(long)i * d + c] = bf16_to_double(J->q[((J->q_start[s] + i) * J->Hq + h) * d + c]);
        attend_rows(Q, K, V, NULL, ql, ctx, d, J->causal, J->scale, r0, r1, S, O, L);
        for (int i = r0; i < r1; ++i) {
            double* dst = J->rows ? J->out + u * d : J->out + ((J->q_start[s] + i) * J->Hq + h) * d;
            memcpy(dst, O + (long)(i - r0) * d, sizeof(double) * (size_t)d);
            if (J->lse) {
                if (J->rows)
                    J->lse[u] = L[i - r0];
                else
                    J->lse[(J->q_start[s] + i) * J->Hq + h] = L[i - r0];
            }
        }
    }
done:
    free(tmp); free(K); free(V); free(Q); free(S); free(O); free(L);
    return NULL;
}

static int paged_common(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const uint8_t* k_cache8, const uint8_t* v_cache8, double k_scale, double v_scale,
                        const int32_t* block_table, const int32_t* ctx_lens,
                        const int32_t* q_lens, int num_seqs, int max_blocks_per_seq,
                        int num_blocks, int Hq, int Hkv, int d, int block_size, int causal,
                        double scale, const int32_t* rows, long nrows, double* out,
                        double* lse, int nthreads)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || Hq % Hkv || block_size <= 0)
        return ORA_ERR_ARG;
    long* q_start = (long*)malloc(sizeof(long) * (size_t)(num_seqs + 1));
    if (!q_start)
        return ORA_ERR_NOMEM;
    q_start[0] = 0;
    int max_ctx = 1;
    for (int s = 0; s < num_seqs; ++s) {
        q_start[s + 1] = q_start[s] + q_lens[s];
        if (ctx_lens[s] > max_ctx)
            max_ctx = ctx_lens[s];
    }
    if (max_ctx > max_blocks_per_seq * block_size)
        max_ctx = max_blocks_per_seq * block_size;
    paged_job J;
    memset(&J, 0, sizeof J);
    pthread_mutex_init(&J.wq.lock, NULL);
    J.wq.total = rows ? nrows : (long)num_seqs * Hq;
    J.q = q; J.kc = k_cache; J.vc = v_cache; J.bt = block_table;
    J.kc8 = k_cache8; J.vc8 = v_cache8; J.k_scale = k_scale; J.v_scale = v_scale;
    J.ctx_lens = ctx_lens; J.q_lens = q_lens; J.q_start = q_start; J.rows = rows;
    J.out = out; J.lse = lse; J.num_seqs = num_seqs; J.max_blocks = max_blocks_per_seq;
    J.num_blocks = num_blocks; J.Hq = Hq; J.Hkv = Hkv; J.d = d; J.block_size = block_size;
    J.causal = causal; J.scale = scale; J.max_ctx = max_ctx;
    int st = run_threads(paged_worker, &J, nthreads);
    pthread_mutex_destroy(&J.wq.lock);
    free(q_start);
    return st != ORA_OK ? st : J.wq.status;
}

/*
 * Paged attention.  q: bf16 bits [sum(q_lens), Hq, d], packed in sequence
 * order; caches: bf16 bits [num_blocks, Hkv, block_size, d];
 * ctx_lens[s] counts every token of sequence s (the chunk included), so the
 * chunk's queries are positions ctx - q_len .. ctx - 1.
 * out: double [sum(q_lens), Hq, d]; lse: double [sum(q_lens), Hq] or NULL.
 */
int ora_paged_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                        const int32_t* block_table, const int32_t* ctx_lens,
                        const int32_t* q_lens, int num_seqs, int max_blocks_per_seq,
                        int num_blocks, int Hq, int Hkv, int d, int block_size, int causal,
                        double scale, double* out, double* lse, int nthreads)
{
    return paged_common(q, k_cache, v_cache, NULL, NULL, 1.0, 1.0, block_table, ctx_lens, q_lens, num_seqs,
                        max_blocks_per_seq, num_blocks, Hq, Hkv, d, block_size, causal,
                        scale, NULL, 0, out, lse, nthreads);
}

/*
 * Paged attention over the 8-bit caches (layouts and scales as in
 * ora_cache_append_fp8): each cached key / value element is the E4M3 value
 * of its code times k_scale / v_scale; the rest is ora_paged_attention.
 */
int ora_paged_attention_fp8(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache, double k_scale,
                            double v_scale, const int32_t* block_table, const int32_t* ctx_lens,
                            const int32_t* q_lens, int num_seqs, int max_blocks_per_seq, int num_blocks, int Hq,
                            int Hkv, int d, int causal, double scale, const int32_t* rows, long nrows, double* out,
                            double* lse, int nthreads)
{
    return paged_common(q, NULL, NULL, k_cache, v_cache, k_scale, v_scale, block_table, ctx_lens, q_lens,
                        num_seqs, max_blocks_per_seq, num_blocks, Hq, Hkv, d, 16, causal, scale, rows, nrows,
                        out, lse, nthreads);
}

/* Sampled rows: rows[3*r .. 3*r+2] = (seq, query index within the chunk, head). */
int ora_paged_attention_rows(const uint16_t* q, const uint16_t* k_cache,
                             const uint16_t* v_cache, const int32_t* block_table,
                             const int32_t* ctx_lens, const int32_t* q_lens, int num_seqs,
                             int max_blocks_per_seq, int num_blocks, int Hq, int Hkv, int d,
                             int block_size, int causal, double scale, const int32_t* rows,
                             long nrows, double* out, double* lse, int nthreads)
{
    return paged_common(q, k_cache, v_cache, NULL, NULL, 1.0, 1.0, block_table, ctx_lens, q_lens, num_seqs,
                        max_blocks_per_seq, num_blocks, Hq, Hkv, d, block_size, causal,
                        scale, rows, nrows, out, lse, nthreads);
}

/* ----------------------------------------------------- partial merging -- */

/*
 * Combines attention results computed over disjoint parts of the key set.
 * Part p contributes its normalised output O_p (d doubles) and its
 * log-sum-exp lse_p.  The softmax over the union weights part p by
 * exp(lse_p) / sum_q exp(lse_q); the union's LSE is log sum_p exp(lse_p).
 * Parts with lse = -inf (no visible key) carry zero weight.
 */
void ora_lse_merge(int nparts, int d, const double* O_parts, const double* lse_parts,
                   double* O, double* lse)
{
    double mx = -INFINITY;
    for (int p = 0; p < nparts; ++p)
        if (lse_parts[p] > mx)
            mx = lse_parts[p];
    for (int c = 0; c < d; ++c)
        O[c] = 0.0;
    if (mx == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int p = 0; p < nparts; ++p)
        wsum += exp(lse_parts[p] - mx);
    for (int p = 0; p < nparts; ++p) {
        double w = exp(lse_parts[p] - mx) / wsum;
        for (int c = 0; c < d; ++c)
            O[c] += w * O_parts[(long)p * d + c];
    }
    *lse = mx + log(wsum);
}

/* ------------------------------------------------- mask tile classes -- */

/*
 * Class of each bm x bn tile of an additive mask [Tq, Tk] (edge tiles cover
 * only their in-range elements): 0 = every element -inf (the tile contributes
 * nothing), 1 = every element exactly 0 (the mask changes nothing there),
 * 3 = every element is 0 or -inf and, in every row, the columns holding 0 are
 * one contiguous run (possibly empty) -- the tile restricts each row to an
 * interval of keys and adds nothing else -- 2 = anything else.
 * cls: uint8 [ceil(Tq/bm), ceil(Tk/bn)].  iv (may be NULL): uint8
 * [ceil(Tq/bm), ceil(Tk/bn), bm, 2]; for a class-3 tile, row r of the tile
 * gets (lo, hi), the run of zeros being columns [lo, hi) of the tile (lo = hi
 * = 0 for a row of -inf only; rows past Tq get 0, 0); other tiles' entries are
 * left as they are.  Needs bn <= 255.
 */
void ora_mask_tile_classes(const float* M, int Tq, int Tk, int bm, int bn, uint8_t* cls, uint8_t* iv)
{
    int nti = (Tq + bm - 1) / bm, ntj = (Tk + bn - 1) / bn;
    for (int ti = 0; ti < nti; ++ti)
        for (int tj = 0; tj < ntj; ++tj) {
            int all_neg_inf = 1, all_zero = 1, intervals = 1;
            for (int i = ti * bm; i < Tq && i < (ti + 1) * bm; ++i) {
                int first = -1, last = -1, zeros = 0;
                for (int j = tj * bn; j < Tk && j < (tj + 1) * bn; ++j) {
                    float x = M[(long)i * Tk + j];
                    if (!(x == -INFINITY))
                        all_neg_inf = 0;
                    if (!(x == 0.0f))
                        all_zero = 0;
                    if (x == 0.0f) {
                        if (first < 0)
                            first = j - tj * bn;
                        last = j - tj * bn;
                        ++zeros;
                    } else if (!(x == -INFINITY)) {
                        intervals = 0;
                    }
                }
                if (zeros > 0 && zeros != last - first + 1)
                    intervals = 0;
            }
            uint8_t c = (uint8_t)(all_neg_inf ? 0 : (all_zero ? 1 : (intervals ? 3 : 2)));
            cls[(long)ti * ntj + tj] = c;
            if (c == 3 && iv) {
                uint8_t* out = iv + ((long)ti * ntj + tj) * bm * 2;
                for (int r = 0; r < bm; ++r) {
                    int i = ti * bm + r, lo = 0, hi = 0;
                    if (i < Tq)
                        for (int j = tj * bn; j < Tk && j < (tj + 1) * bn; ++j)
                            if (M[(long)i * Tk + j] == 0.0f) {
                                if (hi == 0)
                                    lo = j - tj * bn;
                                hi = j - tj * bn + 1;
                            }
                    out[2 * r] = (uint8_t)lo;
                    out[2 * r + 1] = (uint8_t)hi;
                }
            }
        }
}
