/*
 * pkv_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, scalar CPU oracle for decode-time attention over a block-paged
 * KV cache.  It is the yardstick the CUDA library is checked against, nothing
 * more: only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code, header, table or helper with the CUDA
 * library, and it never calls into it.
 *
 * Every floating-point result is computed in IEEE double (fp64) from inputs
 * that are first widened exactly; the only fp32 arithmetic is the quantiser,
 * whose fixed fp32 operation sequence is part of the cache format and must be
 * reproduced bit for bit.  Build with -ffp-contract=off and without fast-math.
 *
 * Sources (web pages on the paged KV cache; each function cites the section it
 * follows):
 *   [MTPLX-1] "How the Paged KV Cache Works in MTPLX: Architecture and Implementation"
 *   [MTPLX-2] "How MTPLX Manages Memory Using Request-Sized Paged KV Cache"
 *   [MTPLX-3] "How MTPLX Manages Memory with KV Caching Strategies"
 *   [MLXCEL]  mlxcel manual, "KV Cache"
 *   [METAL]   metalworking, "The KV Cache"
 *
 * Pins: every function here is checked by the `-m "not gpu"` tests against
 * closed forms, invariants, independent library routines or brute force (see
 * tests/test_oracle_*.py).  The one deliberately unpinned item is the pages'
 * quoted K8/V4 cache size, which no format in this file can reproduce.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element type codes used by every entry point below */
enum { OT_F16 = 0, OT_BF16 = 1, OT_F32 = 2, OT_F64 = 3 };
/* cache kinds */
enum { OC_F16 = 0, OC_BF16 = 1, OC_K8V4 = 2 };

/* ------------------------------------------------------------------------- */
/* Number formats, written from the IEEE 754 binary16 definition and the     */
/* bfloat16 definition (binary32 with the low 16 fraction bits dropped).     */
/* ------------------------------------------------------------------------- */

double pkvo_f16_to_f64(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                  /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);      /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

double pkvo_bf16_to_f64(uint16_t b)
{
    int sign = b >> 15, e = (b >> 7) & 0xff, m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                 /* subnormal: m * 2^-133 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + m), e - 134);      /* (1 + m/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a binary32 value to binary16, round-to-nearest-even.
 * The value is widened to double (exact), scaled by a power of two so that the
 * 11 significant bits sit left of the binary point, and rounded with
 * nearbyint() (default rounding mode: to nearest, ties to even). */
uint16_t pkvo_f32_to_f16_rne(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isnan(a)) return sign | 0x7e00;
    if (isinf(a)) return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {                       /* zero / subnormal range */
        double q = nearbyint(a * ldexp(1.0, 24));    /* units of 2^-24, q <= 1024 */
        return sign | (uint16_t)q;                   /* q == 1024 is the smallest normal */
    }
    int e;
    double fr = frexp(a, &e);                        /* a = fr * 2^e, fr in [0.5, 1) */
    int E = e - 1;                                   /* a = 1.f * 2^E */
    double q = nearbyint(ldexp(fr, 11));             /* significand in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return sign | 0x7c00;                /* overflow to infinity */
    return sign | (uint16_t)(((E + 15) << 10) | ((int)q - 1024));
}

/* Round a binary32 value to bfloat16, round-to-nearest-even (same method). */
uint16_t pkvo_f32_to_bf16_rne(float x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs((double)x);
    if (isnan(a)) return sign | 0x7fc0;
    if (isinf(a)) return sign | 0x7f80;
    if (a < ldexp(1.0, -126)) {
        double q = nearbyint(a * ldexp(1.0, 133));   /* units of 2^-133, q <= 128 */
        return sign | (uint16_t)q;
    }
    int e;
    double fr = frexp(a, &e);
    int E = e - 1;
    double q = nearbyint(ldexp(fr, 8));              /* significand in [128, 256] */
    if (q == 256.0) { q = 128.0; E += 1; }
    if (E > 127) return sign | 0x7f80;
    return sign | (uint16_t)(((E + 127) << 7) | ((int)q - 128));
}

void pkvo_f32_to_f16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = pkvo_f32_to_f16_rne(x[i]);
}

void pkvo_f32_to_bf16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = pkvo_f32_to_bf16_rne(x[i]);
}

void pkvo_f16_to_f64_array(const uint16_t *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = pkvo_f16_to_f64(x[i]);
}

void pkvo_bf16_to_f64_array(const uint16_t *x, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = pkvo_bf16_to_f64(x[i]);
}

static double load_elem(const void *p, int dtype, size_t i)
{
    switch (dtype) {
    case OT_F16: return pkvo_f16_to_f64(((const uint16_t *)p)[i]);
    case OT_BF16: return pkvo_bf16_to_f64(((const uint16_t *)p)[i]);
    case OT_F32: return (double)((const float *)p)[i];
    default: return ((const double *)p)[i];
    }
}

/* ------------------------------------------------------------------------- */
/* Cache writes and reads                                                    */
/* ------------------------------------------------------------------------- */

/* reshape_and_cache: scatter each new token's K and V rows (all kv heads) into
 * the slot named by slot_mapping.  Slot s lives in physical block s / block_size
 * at offset s % block_size of a cache laid out [num_blocks, block_size,
 * num_kv_heads, head_dim] [MTPLX-1 §"4-D Tensor Structure"; MLXCEL §"Attention
 * Dispatch and In-Place Decode Writes"; METAL §"Layout matters at the kernel
 * level" names reshape_and_cache].  A negative slot is padding and is skipped;
 * a slot past the pool is skipped and counted.  Returns the count. */
int pkvo_reshape_and_cache(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                           const int64_t *slot_mapping, int num_tokens, int num_blocks,
                           int block_size, int num_kv_heads, int head_dim, int elem_bytes)
{
    size_t row = (size_t)num_kv_heads * head_dim * elem_bytes;   /* one token, all kv heads */
    int bad = 0;
    for (int i = 0; i < num_tokens; i++) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { bad++; continue; }
        int64_t blk = slot / block_size, off = slot % block_size;
        size_t dst = ((size_t)blk * block_size + (size_t)off) * row;
        memcpy((char *)k_cache + dst, (const char *)k_new + (size_t)i * row, row);
        memcpy((char *)v_cache + dst, (const char *)v_new + (size_t)i * row, row);
    }
    return bad;
}

/* gather_kv_cache: copy every visible token of every sequence back into a
 * contiguous [sum(ctx), num_kv_heads, head_dim] array, logical token t of
 * sequence s going to row cu_seq_lens[s] + t.  Logical token t sits in physical
 * block block_tables[s][t / block_size] at offset t % block_size
 * [METAL §"Layout matters at the kernel level": fixed-size blocks plus an
 * indirection table, gather_kv_cache].  Returns -1 on an out-of-range block id
 * or a context longer than the table, else 0. */
int pkvo_gather_kv_cache(void *k_out, void *v_out, const int32_t *cu_seq_lens,
                         const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         int num_seqs, int max_blocks, int num_blocks, int block_size,
                         int num_kv_heads, int head_dim, int elem_bytes)
{
    size_t row = (size_t)num_kv_heads * head_dim * elem_bytes;
    for (int s = 0; s < num_seqs; s++) {
        int ctx = context_lens[s];
        if (ctx > max_blocks * block_size) return -1;
        for (int t = 0; t < ctx; t++) {
            int pb = block_tables[(size_t)s * max_blocks + t / block_size];
            if (pb < 0 || pb >= num_blocks) return -1;
            size_t src = ((size_t)pb * block_size + (size_t)(t % block_size)) * row;
            size_t dst = ((size_t)cu_seq_lens[s] + (size_t)t) * row;
            memcpy((char *)k_out + dst, (const char *)k_cache + src, row);
            memcpy((char *)v_out + dst, (const char *)v_cache + src, row);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Mixed-precision K8/V4 cache                                               */
/* ------------------------------------------------------------------------- */

/* The quantised format keeps K more precise than V because K feeds the softmax
 * and V only a weighted average [METAL §"The K/V asymmetry"]; scales and zeros
 * live in their own paged tensors with the same block indices as the codes
 * [MTPLX-2 §"Quantization-Aware Memory Layout"; MTPLX-3 §"Quantization-Aware
 * Allocation": per-block scale and zero tensors].
 *
 * Layout (block_size bs, kv heads H, head_dim D, groups NG = D / v_group):
 *   k_q     int8  [NB, bs, H, D]          code c in [-127, 127]
 *   k_scale fp16  [NB, H, bs]             one scale per (token, kv head)
 *   v_q     uint8 [NB, bs, H, D/2]        two 4-bit codes per byte, even dim in the low nibble
 *   v_scale fp16  [NB, H, bs, NG]         one scale per (token, kv head, group)
 *   v_zero  fp16  [NB, H, bs, NG]         one float offset per (token, kv head, group)
 *
 * Quantiser, as a fixed fp32 operation sequence:
 *   K: a = max_d |k_d|;  s = fp16_rne(a / 127);  c_d = s == 0 ? 0 : clamp(rint(k_d / s), -127, 127)
 *   V: lo = min, hi = max over the group (a zero minimum taken as +0);
 *      s = fp16_rne((hi - lo) / 15);  z = fp16_rne(lo)
 *      c_d = s == 0 ? 0 : clamp(rint((v_d - z) / s), 0, 15)
 * where rint rounds half to even and / is the IEEE-rounded fp32 quotient.
 * Dequantisation: k = c * s,  v = c * s + z. */
static float clampf(float x, float lo, float hi) { return x < lo ? lo : (x > hi ? hi : x); }

int pkvo_quantize_kv(int8_t *k_q, uint16_t *k_scale, uint8_t *v_q, uint16_t *v_scale,
                     uint16_t *v_zero, const void *k_new, const void *v_new, int src_dtype,
                     const int64_t *slot_mapping, int num_tokens, int num_blocks, int block_size,
                     int num_kv_heads, int head_dim, int v_group)
{
    int D = head_dim, NG = head_dim / v_group, bad = 0;
    float *kv = (float *)malloc(sizeof(float) * (size_t)D);
    for (int i = 0; i < num_tokens; i++) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) { bad++; continue; }
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; h++) {
            size_t src = ((size_t)i * num_kv_heads + h) * D;
            size_t row = ((size_t)blk * block_size + (size_t)off) * num_kv_heads + h;
            size_t meta = ((size_t)blk * num_kv_heads + h) * block_size + (size_t)off;
            /* K: symmetric int8 with one fp16 scale */
            float a = 0.0f;
            for (int d = 0; d < D; d++) {
                kv[d] = (float)load_elem(k_new, src_dtype, src + d);   /* exact */
                float m = fabsf(kv[d]);
                if (m > a) a = m;
            }
            uint16_t s16 = pkvo_f32_to_f16_rne(a / 127.0f);
            float s = (float)pkvo_f16_to_f64(s16);
            for (int d = 0; d < D; d++) {
                float c = (s == 0.0f) ? 0.0f : clampf(rintf(kv[d] / s), -127.0f, 127.0f);
                k_q[row * D + d] = (int8_t)c;
            }
            k_scale[meta] = s16;
            /* V: asymmetric 4-bit, one fp16 scale and fp16 zero per group */
            for (int d = 0; d < D; d++) kv[d] = (float)load_elem(v_new, src_dtype, src + d);
            for (int g = 0; g < NG; g++) {
                float lo = kv[g * v_group], hi = lo;
                for (int d = g * v_group; d < (g + 1) * v_group; d++) {
                    if (kv[d] < lo) lo = kv[d];
                    if (kv[d] > hi) hi = kv[d];
                }
                if (lo == 0.0f) lo = 0.0f;            /* a zero minimum is stored as +0 */
                uint16_t vs16 = pkvo_f32_to_f16_rne((hi - lo) / 15.0f);
                uint16_t vz16 = pkvo_f32_to_f16_rne(lo);
                float vs = (float)pkvo_f16_to_f64(vs16), vz = (float)pkvo_f16_to_f64(vz16);
                for (int d = g * v_group; d < (g + 1) * v_group; d++) {
                    float c = (vs == 0.0f) ? 0.0f : clampf(rintf((kv[d] - vz) / vs), 0.0f, 15.0f);
                    uint8_t code = (uint8_t)c;
                    uint8_t *byte = &v_q[row * (size_t)(D / 2) + (size_t)(d / 2)];
                    if (d % 2 == 0) *byte = (uint8_t)((*byte & 0xf0) | code);
                    else *byte = (uint8_t)((*byte & 0x0f) | (code << 4));
                }
                v_scale[meta * NG + g] = vs16;
                v_zero[meta * NG + g] = vz16;
            }
        }
    }
    free(kv);
    return bad;
}

/* ------------------------------------------------------------------------- */
/* Attention                                                                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    /* outputs */
    double *out, *part_o, *part_m, *part_l;
    int partition_size, max_partitions;
    /* query */
    const void *q;
    int q_dtype, num_heads;
    double scale;
    /* cache */
    int cache_kind;
    const void *k_cache, *v_cache, *k_scale, *v_scale, *v_zero;
    int num_blocks, block_size, num_kv_heads, head_dim, v_group;
    /* sequences */
    const int32_t *block_tables, *context_lens;
    int num_seqs, max_blocks, q_len;
    int window;   /* sliding window in tokens, 0 = none */
    /* sparse page indirection (optional): pages of each sequence to attend */
    const int32_t *page_lists, *page_counts;
    int max_pages;
    /* work */
    const int32_t *row_list;
    int n_rows, n_threads, thread_id;
    int error;
} attn_job;

/* The K row of logical token t, kv head kvh, of sequence s, widened to fp64.
 * Scalar gather through the block table [METAL §"Layout matters at the kernel
 * level"; MTPLX-1 §"4-D Tensor Structure"], with the K8/V4 dequantisation
 * k = c * s applied element by element. */
static int load_k_row(const attn_job *J, int s, int t, int kvh, double *k)
{
    int bs = J->block_size, D = J->head_dim, H = J->num_kv_heads;
    int pb = J->block_tables[(size_t)s * J->max_blocks + t / bs];
    if (pb < 0 || pb >= J->num_blocks) return -1;
    size_t row = ((size_t)pb * bs + (size_t)(t % bs)) * H + kvh;
    if (J->cache_kind == OC_K8V4) {
        size_t meta = ((size_t)pb * H + kvh) * bs + (size_t)(t % bs);
        double sc = pkvo_f16_to_f64(((const uint16_t *)J->k_scale)[meta]);
        for (int d = 0; d < D; d++) k[d] = (double)((const int8_t *)J->k_cache)[row * D + d] * sc;
    } else {
        int dt = J->cache_kind == OC_F16 ? OT_F16 : OT_BF16;
        for (int d = 0; d < D; d++) k[d] = load_elem(J->k_cache, dt, row * D + d);
    }
    return 0;
}

/* The V row of logical token t, with v = c * s + z for the K8/V4 cache. */
static int load_v_row(const attn_job *J, int s, int t, int kvh, double *v)
{
    int bs = J->block_size, D = J->head_dim, H = J->num_kv_heads;
    int pb = J->block_tables[(size_t)s * J->max_blocks + t / bs];
    if (pb < 0 || pb >= J->num_blocks) return -1;
    size_t row = ((size_t)pb * bs + (size_t)(t % bs)) * H + kvh;
    if (J->cache_kind == OC_K8V4) {
        int NG = D / J->v_group;
        size_t meta = ((size_t)pb * H + kvh) * bs + (size_t)(t % bs);
        for (int d = 0; d < D; d++) {
            uint8_t byte = ((const uint8_t *)J->v_cache)[row * (size_t)(D / 2) + (size_t)(d / 2)];
            int c = (d % 2 == 0) ? (byte & 0x0f) : (byte >> 4);
            int g = d / J->v_group;
            double sc = pkvo_f16_to_f64(((const uint16_t *)J->v_scale)[meta * NG + g]);
            double z = pkvo_f16_to_f64(((const uint16_t *)J->v_zero)[meta * NG + g]);
            v[d] = (double)c * sc + z;
        }
    } else {
        int dt = J->cache_kind == OC_F16 ? OT_F16 : OT_BF16;
        for (int d = 0; d < D; d++) v[d] = load_elem(J->v_cache, dt, row * D + d);
    }
    return 0;
}

/* Softmax attention of one query row against the logical tokens [t0, t1) of a
 * sequence, straight from the definition:
 *   x_t = scale * sum_d q_d K_t[d];  m = max_t x_t;  w_t = exp(x_t - m);
 *   l = sum_t w_t;  o = sum_t w_t V_t / l.
 * An empty range gives o = 0, m = -inf, l = 0.  The query head's kv head is
 * h / (H / H_kv) [METAL §"GQA": kv_head_idx = tid.y / gqa_factor]. */
static int attend_range(const attn_job *J, int s, int kvh, const double *qd, int t0, int t1,
                        double *o, double *m_out, double *l_out, double *x, double *row)
{
    int D = J->head_dim;
    for (int d = 0; d < D; d++) o[d] = 0.0;
    if (t1 <= t0) { *m_out = -INFINITY; *l_out = 0.0; return 0; }
    double m = -INFINITY;
    for (int t = t0; t < t1; t++) {
        if (load_k_row(J, s, t, kvh, row)) return -1;
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += qd[d] * row[d];
        x[t - t0] = J->scale * dot;
        if (x[t - t0] > m) m = x[t - t0];
    }
    double l = 0.0;
    for (int t = t0; t < t1; t++) {
        double w = exp(x[t - t0] - m);
        l += w;
        if (load_v_row(J, s, t, kvh, row)) return -1;
        for (int d = 0; d < D; d++) o[d] += w * row[d];
    }
    for (int d = 0; d < D; d++) o[d] /= l;
    *m_out = m;
    *l_out = l;
    return 0;
}

/* The same attention over an explicit list of logical tokens tok[0..n) (in
 * increasing order), for sparse page-indirection decode. */
static int attend_list(const attn_job *J, int s, int kvh, const double *qd, const int *tok, int n,
                       double *o, double *m_out, double *l_out, double *x, double *row)
{
    int D = J->head_dim;
    for (int d = 0; d < D; d++) o[d] = 0.0;
    if (n <= 0) { *m_out = -INFINITY; *l_out = 0.0; return 0; }
    double m = -INFINITY;
    for (int i = 0; i < n; i++) {
        if (load_k_row(J, s, tok[i], kvh, row)) return -1;
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += qd[d] * row[d];
        x[i] = J->scale * dot;
        if (x[i] > m) m = x[i];
    }
    double l = 0.0;
    for (int i = 0; i < n; i++) {
        double w = exp(x[i] - m);
        l += w;
        if (load_v_row(J, s, tok[i], kvh, row)) return -1;
        for (int d = 0; d < D; d++) o[d] += w * row[d];
    }
    for (int d = 0; d < D; d++) o[d] /= l;
    *m_out = m;
    *l_out = l;
    return 0;
}

/* Tokens a sparse page list makes visible in [lo, vis) [MLXCEL §"Paged Decode
 * Storage and Kernels": sparse page-indirection decode].  Reading: the list
 * names logical pages (16-token blocks) of the sequence; page p contributes its
 * tokens p*16 .. p*16+15 that lie in [lo, vis).  Entries are taken in order;
 * one that is outside [0, ceil(ctx / 16)) or not above the last page taken is
 * skipped.  Returns the number of tokens written to tok. */
static int sparse_tokens(const attn_job *J, int s, int ctx, int lo, int vis, int *tok)
{
    int bs = J->block_size, n = 0, last = -1;
    int cnt = J->page_counts[s];
    if (cnt > J->max_pages) cnt = J->max_pages;
    int npages = (ctx + bs - 1) / bs;
    for (int i = 0; i < cnt; i++) {
        int p = J->page_lists[(size_t)s * J->max_pages + i];
        if (p < 0 || p >= npages || p <= last) continue;
        last = p;
        for (int o = 0; o < bs; o++) {
            int t = p * bs + o;
            if (t >= lo && t < vis) tok[n++] = t;
        }
    }
    return n;
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    int H = J->num_heads, D = J->head_dim, g = J->num_heads / J->num_kv_heads;
    int R = J->row_list ? J->n_rows : J->num_seqs * J->q_len;
    int cap = J->max_blocks * J->block_size;
    double *qd = (double *)malloc(sizeof(double) * (size_t)D);
    double *row = (double *)malloc(sizeof(double) * (size_t)D);
    double *x = (double *)malloc(sizeof(double) * (size_t)(cap > 0 ? cap : 1));
    int *tok = J->page_lists ? (int *)malloc(sizeof(int) * (size_t)(cap > 0 ? cap : 1)) : NULL;
    double m, l;
    for (long task = J->thread_id; task < (long)R * H; task += J->n_threads) {
        int r = J->row_list ? J->row_list[task / H] : (int)(task / H);
        int h = (int)(task % H);
        int s = r / J->q_len, j = r % J->q_len;
        int ctx = J->context_lens[s];
        if (ctx > cap || ctx < 0) { J->error = -2; break; }
        /* Row j of a multi-token verify block sees the history plus drafts
         * 0..j: the tokens [0, ctx - q_len + j + 1) [MLXCEL §"Matrix-Absorbed MLA
         * Decode" and §"Speculative Rewind": a speculative verify block].  For
         * q_len = 1 this is the whole stored context [MTPLX-2 §"Request-Sized
         * Offset Tracking": kernels read only the tokens stored so far]. */
        int vis = ctx - J->q_len + j + 1;
        if (vis < 0) vis = 0;
        /* Sliding window: the visible part of the cache is trimmed to its last
         * `window` stored tokens; older ones are masked, not freed [MTPLX-2
         * §"Sliding-Window Memory Control" and the FAQ on adjusting the window].
         * The trim is of the stored cache (the last `window` of its ctx tokens),
         * so every draft row of a verify block starts at the same token. */
        int lo = 0;
        if (J->window > 0 && ctx > J->window) lo = ctx - J->window;
        if (lo > vis) lo = vis;
        int kvh = h / g;
        size_t qoff = ((size_t)r * H + h) * D;
        for (int d = 0; d < D; d++) qd[d] = load_elem(J->q, J->q_dtype, qoff + d);
        if (J->out && J->page_lists) {
            int n = sparse_tokens(J, s, ctx, lo, vis, tok);
            if (attend_list(J, s, kvh, qd, tok, n, J->out + qoff, &m, &l, x, row)) { J->error = -1; break; }
        } else if (J->out) {
            if (attend_range(J, s, kvh, qd, lo, vis, J->out + qoff, &m, &l, x, row)) { J->error = -1; break; }
        }
        if (J->part_o) {
            /* Split-KV: partition p covers logical tokens [pP, (p+1)P) of the
             * visible range [MLXCEL §"Paged Decode Storage and Kernels": decode
             * splits; METAL: "split-KV decode kernels"]. */
            int P = J->partition_size;
            for (int p = 0; p < J->max_partitions; p++) {
                int t0 = p * P > lo ? p * P : lo, t1 = (p + 1) * P < vis ? (p + 1) * P : vis;
                size_t pi = ((size_t)r * H + h) * J->max_partitions + p;
                if (attend_range(J, s, kvh, qd, t0, t1, J->part_o + pi * D, &J->part_m[pi],
                                 &J->part_l[pi], x, row)) { J->error = -1; break; }
            }
            if (J->error) break;
        }
    }
    free(qd);
    free(row);
    free(x);
    free(tok);
    return NULL;
}

/* Paged decode attention.  q is [R, H, D] with R = num_seqs * q_len rows
 * (row r = sequence r / q_len, draft r % q_len); out is [R, H, D] fp64.  When
 * part_o is given, the per-partition (o_p, m_p, l_p) of partition_size tokens
 * are written to part_o [R, H, max_partitions, D] and part_m / part_l
 * [R, H, max_partitions] (m_p in the units of scale * q.k, natural log base).
 * row_list (optional) restricts the work to the listed rows; the other rows of
 * out are left untouched.  window > 0 keeps only the last `window` stored tokens
 * of each sequence visible.  page_lists [num_seqs, max_pages] / page_counts
 * [num_seqs] (optional, out only): each row attends only the tokens of its
 * sequence's listed pages (sparse_tokens).  Returns 0, or a negative code on an
 * out-of-range block id (-1) or a context longer than its table (-2). */
int pkvo_paged_attention(double *out, double *part_o, double *part_m, double *part_l,
                         int partition_size, int max_partitions, const void *q, int q_dtype,
                         int num_heads, double scale, int cache_kind, const void *k_cache,
                         const void *v_cache, const void *k_scale, const void *v_scale,
                         const void *v_zero, int num_blocks, int block_size, int num_kv_heads,
                         int head_dim, int v_group, const int32_t *block_tables,
                         const int32_t *context_lens, int num_seqs, int max_blocks, int q_len,
                         const int32_t *row_list, int n_rows, int n_threads, int window,
                         const int32_t *page_lists, const int32_t *page_counts, int max_pages)
{
    if (window < 0) return -3;
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -3;
    if (part_o && partition_size <= 0) return -3;
    if (page_lists && (part_o || !page_counts || max_pages < 0)) return -3;
    if (n_threads < 1) n_threads = 1;
    attn_job base = {out, part_o, part_m, part_l, partition_size, max_partitions, q, q_dtype,
                     num_heads, scale, cache_kind, k_cache, v_cache, k_scale, v_scale, v_zero,
                     num_blocks, block_size, num_kv_heads, head_dim, v_group, block_tables,
                     context_lens, num_seqs, max_blocks, q_len, window, page_lists, page_counts,
                     max_pages, row_list, n_rows, n_threads, 0, 0};
    attn_job *jobs = (attn_job *)malloc(sizeof(attn_job) * (size_t)n_threads);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    for (int i = 0; i < n_threads; i++) {
        jobs[i] = base;
        jobs[i].thread_id = i;
    }
    for (int i = 1; i < n_threads; i++) pthread_create(&th[i], NULL, attn_worker, &jobs[i]);
    attn_worker(&jobs[0]);
    int err = jobs[0].error;
    for (int i = 1; i < n_threads; i++) {
        pthread_join(th[i], NULL);
        if (jobs[i].error) err = jobs[i].error;
    }
    free(jobs);
    free(th);
    return err;
}

/* Cross-partition log-sum-exp combination of split-KV partials:
 *   M = max_p m_p;  w_p = l_p exp(m_p - M);  out = sum_p w_p o_p / sum_p w_p.
 * Partitions with l_p = 0 carry no weight; a row with none gives 0.  The
 * pages name split-KV decode but print no combination formula; this is the
 * exact identity that makes split attention equal single-pass attention. */
void pkvo_lse_reduce(double *out, const double *part_o, const double *part_m,
                     const double *part_l, int num_rows, int num_heads, int num_partitions,
                     int head_dim)
{
    for (long rh = 0; rh < (long)num_rows * num_heads; rh++) {
        const double *m = part_m + rh * num_partitions, *l = part_l + rh * num_partitions;
        double *o = out + rh * head_dim;
        double M = -INFINITY;
        for (int p = 0; p < num_partitions; p++)
            if (l[p] > 0.0 && m[p] > M) M = m[p];
        for (int d = 0; d < head_dim; d++) o[d] = 0.0;
        if (M == -INFINITY) continue;
        double W = 0.0;
        for (int p = 0; p < num_partitions; p++) {
            if (!(l[p] > 0.0)) continue;
            double w = l[p] * exp(m[p] - M);
            W += w;
            for (int d = 0; d < head_dim; d++) o[d] += w * part_o[(rh * num_partitions + p) * head_dim + d];
        }
        for (int d = 0; d < head_dim; d++) o[d] /= W;
    }
}

/* Dequantising gather of a K8/V4 cache: every visible token of every sequence
 * to contiguous [sum(ctx), num_kv_heads, head_dim] rows of out_dtype (OT_F16 or
 * OT_BF16), logical token t of sequence s going to row cu_seq_lens[s] + t, the
 * gather of gather_kv_cache [METAL §"Layout matters at the kernel level"] with
 * the K8/V4 values k = c * s_k and v = c * s_v + z_v [METAL §"The K/V
 * asymmetry"; MTPLX-2 §"Quantization-Aware Memory Layout"].  Each value is
 * formed in fp64 (exact for these operands), rounded once to fp32 and then
 * to out_dtype, both round-to-nearest-even.  Returns -1 on an out-of-range
 * block id or a context longer than the table, else 0. */
int pkvo_gather_kv_cache_dequant(uint16_t *k_out, uint16_t *v_out, int out_dtype,
                                 const int32_t *cu_seq_lens, const int8_t *k_q,
                                 const uint16_t *k_scale, const uint8_t *v_q,
                                 const uint16_t *v_scale, const uint16_t *v_zero,
                                 const int32_t *block_tables, const int32_t *context_lens,
                                 int num_seqs, int max_blocks, int num_blocks, int block_size,
                                 int num_kv_heads, int head_dim, int v_group)
{
    int H = num_kv_heads, D = head_dim, NG = head_dim / v_group;
    for (int s = 0; s < num_seqs; s++) {
        int ctx = context_lens[s];
        if (ctx > max_blocks * block_size) return -1;
        for (int t = 0; t < ctx; t++) {
            int pb = block_tables[(size_t)s * max_blocks + t / block_size];
            if (pb < 0 || pb >= num_blocks) return -1;
            int off = t % block_size;
            for (int h = 0; h < H; h++) {
                size_t src = ((size_t)pb * block_size + (size_t)off) * H + (size_t)h;
                size_t meta = ((size_t)pb * H + (size_t)h) * block_size + (size_t)off;
                size_t dst = (((size_t)cu_seq_lens[s] + (size_t)t) * H + (size_t)h) * D;
                double sk = pkvo_f16_to_f64(k_scale[meta]);
                for (int d = 0; d < D; d++) {
                    double kv = (double)k_q[src * D + d] * sk;
                    uint8_t byte = v_q[src * (size_t)(D / 2) + (size_t)(d / 2)];
                    int c = (d & 1) ? (byte >> 4) : (byte & 0x0f);   /* even dim: low nibble */
                    double sv = pkvo_f16_to_f64(v_scale[meta * NG + d / v_group]);
                    double zv = pkvo_f16_to_f64(v_zero[meta * NG + d / v_group]);
                    double vv = (double)c * sv + zv;
                    float kf = (float)kv, vf = (float)vv;
                    k_out[dst + d] = out_dtype == OT_F16 ? pkvo_f32_to_f16_rne(kf) : pkvo_f32_to_bf16_rne(kf);
                    v_out[dst + d] = out_dtype == OT_F16 ? pkvo_f32_to_f16_rne(vf) : pkvo_f32_to_bf16_rne(vf);
                }
            }
        }
    }
    return 0;
}
