/*
 * CPU oracle for the paged KV cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, obviously correct restatement of what
 * the path computes, used to check the CUDA library.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table or constant
 * with the CUDA library, and the CUDA library never calls it.
 *
 * Sources (web pages on vLLM's paged KV cache):
 *  [P1] "Deep Dive into vLLM Worker-Side GPU KV Cache Initialization" (kongchang.com/en),
 *       sections "PagedAttention and Block Management", "Pinpointing the Token Slot",
 *       "Hybrid Attention Mechanisms", "Summary".
 *  [P2] "vLLM의 KV cache 연결 흐름" (llm-engineer.pages.dev), sections "GPU worker가 하는 일",
 *       "Slot mapping은 왜 필요한가", "Forward 직전의 metadata", "EngineCore가 하는 일".
 *  [P3] "Understanding PageAttention Memory Optimization" (freaks.city), sections
 *       "Handling Softmax Across Blocks" (its formula is missing from the page) and the
 *       block-of-4-tokens example.
 *  [P4] "vLLM Worker侧GPU KV Cache初始化流程深度解析" (kongchang.com), sections "KV Cache技术背景"
 *       (FP8 KV cache), "混合注意力机制" (sliding window), "Worker与ModelRunner的协作"
 *       (layout [num_blocks, block_size, num_heads, head_dim]).
 *
 * Number formats are decoded and encoded from their published definitions: IEEE 754 binary16,
 * bfloat16 (the top half of IEEE binary32), and OCP 8-bit floating point E4M3 ("fn": bias 7,
 * no infinities, S.1111.111 is NaN, largest finite 448).
 *
 * Conventions (readings of the pages, listed in the design notes):
 *  - positions are 0-based; seq_lens include this step's tokens; new tokens sit at positions
 *    L-q_len .. L-1;
 *  - the cache is [num_blocks, block_size, num_kv_heads, head_dim], row-major, K and V apart;
 *  - q head hq uses kv head hq / (Hq / Hkv);
 *  - a window W > 0 keeps keys j with p - W < j <= p (the W most recent, current included);
 *  - speculative tokens are causal among themselves: query at position p sees keys j <= p;
 *  - softmax is the textbook max-subtracted softmax, accumulated in double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_INT4 = 3 };

/* error bits reported by the oracle (own numbering, test-side only) */
enum { ORC_BAD_BLOCK = 1, ORC_BAD_SLOT = 2, ORC_PAST_TABLE = 4, ORC_BAD_LEN = 16 };

/* ------------------------------------------------------------------ number formats */

double orc_f16_to_double(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m/2^10 * 2^-14 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

double orc_bf16_to_double(uint16_t b)
{
    int s = b >> 15, e = (b >> 7) & 0xff, m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);              /* subnormal: m/2^7 * 2^-126 */
    else if (e == 255)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + m / 128.0, e - 127);
    return s ? -v : v;
}

double orc_e4m3_to_double(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* float -> E4M3 with round-to-nearest-even; finite values (and infinities) beyond the largest
 * finite magnitude saturate to +-448; NaN stays NaN. */
uint8_t orc_e4m3_from_float(float xf)
{
    double x = (double)xf;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (isnan(x))
        return (uint8_t)(sign | 0x7f);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: spacing 2^-9; a code of 8 is exactly the smallest normal */
        double q = nearbyint(a * 512.0);         /* default rounding mode: ties to even */
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e;
    frexp(a, &e);                                /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                      /* a in [2^e, 2^(e+1)) */
    double q = nearbyint(ldexp(a, 3 - e));       /* in [8, 16] */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    int code = ((e + 7) << 3) | ((int)q - 8);
    if (code > 0x7e)
        code = 0x7e;
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------ INT4
 * [P4] "KV Cache技术背景": an INT4 KV cache stores half a byte per element (with scales that real
 * deployments calibrate; here they are given).  Reading of the format: a signed 4-bit
 * two's-complement integer q in [-8, 7] per element, value = q * scale, one float32 scale per
 * (kv head, group of group_size consecutive dims); two elements per byte, the even dim in the
 * low nibble.  Encoding: q = x / scale in float32 (correctly rounded division), rounded to the
 * nearest integer with ties to even, clamped to [-8, 7] (so +-inf saturate); NaN, which has no
 * nearest integer, is stored as 0.
 */
uint8_t orc_int4_from_float(float x)
{
    if (isnan(x))                       /* no nearest integer: stored as code 0 */
        return 0;
    double q = nearbyint((double)x);    /* the default rounding mode: ties to even */
    if (q > 7.0)
        q = 7.0;
    if (q < -8.0)
        q = -8.0;
    int iq = (int)q;
    return (uint8_t)(iq & 0xF);
}

double orc_int4_to_double(uint8_t nibble)
{
    int n = nibble & 0xF;
    return (double)(n >= 8 ? n - 16 : n);
}

/* element idx (in elements of the [.., head_dim] row-major layout) of an INT4 cache */
static uint8_t int4_at(const void *base, int64_t idx)
{
    uint8_t byte = ((const uint8_t *)base)[idx >> 1];
    return (idx & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
}

static void int4_put(void *base, int64_t idx, uint8_t nibble)
{
    uint8_t *byte = (uint8_t *)base + (idx >> 1);
    if (idx & 1)
        *byte = (uint8_t)((*byte & 0x0F) | (nibble << 4));
    else
        *byte = (uint8_t)((*byte & 0xF0) | (nibble & 0xF));
}

static double elem_to_double(const void *base, int64_t idx, int dtype)
{
    if (dtype == ORC_INT4)
        return orc_int4_to_double(int4_at(base, idx));
    if (dtype == ORC_F16)
        return orc_f16_to_double(((const uint16_t *)base)[idx]);
    if (dtype == ORC_BF16)
        return orc_bf16_to_double(((const uint16_t *)base)[idx]);
    return orc_e4m3_to_double(((const uint8_t *)base)[idx]);
}

/* ------------------------------------------------------------------ slot mapping
 * [P1] "Pinpointing the Token Slot" and [P2] "Slot mapping은 왜 필요한가": a token at position
 * pos of request row r goes to logical block pos / block_size at offset pos % block_size; the
 * row's block table gives the physical block; the slot is physical * block_size + offset.
 * Tokens whose position is negative, and tokens outside every request's range, get slot -1.
 */
int32_t orc_slot_mapping(const int32_t *block_table, int64_t bt_stride, int32_t num_seqs,
                         int32_t max_blocks_per_seq, const int32_t *query_start_loc,
                         const int32_t *positions, int32_t num_tokens, int32_t block_size,
                         int32_t num_blocks, int64_t *slot_mapping)
{
    int32_t err = 0;
    for (int32_t t = 0; t < num_tokens; ++t)
        slot_mapping[t] = -1;
    for (int32_t r = 0; r < num_seqs; ++r) {
        for (int32_t t = query_start_loc[r]; t < query_start_loc[r + 1]; ++t) {
            if (t < 0 || t >= num_tokens)
                continue;
            int64_t pos = positions[t];
            if (pos < 0)
                continue;
            int64_t logical = pos / block_size;
            int64_t offset = pos % block_size;
            if (logical >= max_blocks_per_seq) {
                err |= ORC_PAST_TABLE;
                continue;
            }
            int64_t physical = block_table[(int64_t)r * bt_stride + logical];
            if (physical < 0 || physical >= num_blocks) {
                err |= ORC_BAD_BLOCK;
                continue;
            }
            slot_mapping[t] = physical * block_size + offset;
        }
    }
    return err;
}

/* ------------------------------------------------------------------ cache write
 * [P2] "Slot mapping은 왜 필요한가": decode stores each new token's K/V at its slot.  The slot
 * names (block, offset) = (slot / block_size, slot % block_size) in the
 * [num_blocks, block_size, num_kv_heads, head_dim] layout of [P4] "Worker与ModelRunner的协作".
 * Same dtype: the bits are copied.  E4M3 cache ([P4] "KV Cache技术背景", FP8 KV cache): the
 * value is divided by the per-tensor scale in float32 and encoded with round-to-nearest-even,
 * saturating to the largest finite value.
 */
int32_t orc_reshape_and_cache(const void *key, const void *value, int32_t src_dtype,
                              int64_t key_row_stride, int64_t value_row_stride,
                              int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                              const int64_t *slot_mapping, void *k_cache, void *v_cache,
                              int32_t cache_dtype, int32_t num_blocks, int32_t block_size,
                              float k_scale, float v_scale)
{
    int32_t err = 0;
    const int64_t row = (int64_t)num_kv_heads * head_dim;   /* elements per slot */
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            err |= ORC_BAD_SLOT;
            continue;
        }
        int64_t block = slot / block_size, offset = slot % block_size;
        int64_t dst = (block * block_size + offset) * row;
        for (int64_t i = 0; i < row; ++i) {
            int64_t ks = (int64_t)t * key_row_stride + i;
            int64_t vs = (int64_t)t * value_row_stride + i;
            if (cache_dtype == src_dtype) {
                ((uint16_t *)k_cache)[dst + i] = ((const uint16_t *)key)[ks];
                ((uint16_t *)v_cache)[dst + i] = ((const uint16_t *)value)[vs];
            } else if (cache_dtype == ORC_E4M3) {
                float kx = (float)elem_to_double(key, ks, src_dtype);
                float vx = (float)elem_to_double(value, vs, src_dtype);
                ((uint8_t *)k_cache)[dst + i] = orc_e4m3_from_float(kx / k_scale);
                ((uint8_t *)v_cache)[dst + i] = orc_e4m3_from_float(vx / v_scale);
            } else {
                return -1;                      /* conversions between 16-bit types: not defined */
            }
        }
    }
    return err;
}

/* INT4 cache write: each element divided by its (head, dim group) scale in float32, encoded as
 * above, stored in its nibble of the [num_blocks, block_size, num_kv_heads, head_dim / 2]-byte
 * cache.  scales: float32 [num_kv_heads, head_dim / group_size]. */
int32_t orc_reshape_and_cache_int4(const void *key, const void *value, int32_t src_dtype,
                                   int64_t key_row_stride, int64_t value_row_stride,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                   const int64_t *slot_mapping, void *k_cache, void *v_cache,
                                   int32_t num_blocks, int32_t block_size, const float *k_scales,
                                   const float *v_scales, int32_t group_size)
{
    if (group_size <= 0 || head_dim % group_size != 0 || head_dim % 2 != 0)
        return -1;
    int32_t err = 0;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    const int32_t groups = head_dim / group_size;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)num_blocks * block_size) {
            err |= ORC_BAD_SLOT;
            continue;
        }
        for (int64_t i = 0; i < row; ++i) {
            int64_t h = i / head_dim, d = i % head_dim;
            float ks = k_scales[h * groups + d / group_size];
            float vs = v_scales[h * groups + d / group_size];
            float kx = (float)elem_to_double(key, (int64_t)t * key_row_stride + i, src_dtype);
            float vx = (float)elem_to_double(value, (int64_t)t * value_row_stride + i, src_dtype);
            int4_put(k_cache, slot * row + i, orc_int4_from_float(kx / ks));
            int4_put(v_cache, slot * row + i, orc_int4_from_float(vx / vs));
        }
    }
    return err;
}

/* ------------------------------------------------------------------ attention
 * [P2] "Forward 직전의 metadata" and "Slot mapping은 왜 필요한가": attention reads past K/V
 * through the block table rather than a contiguous tensor.  The oracle first materialises
 * sequence b's contiguous K_b, V_b (one kv head at a time) by walking block_table[b][j / bs] at
 * offset j % bs, decoding to double (E4M3: decoded value times the per-tensor scale), and then
 * runs textbook softmax attention ([P3] "Handling Softmax Across Blocks" names the problem; its
 * formula is missing, so the plain definition is used):
 *     s_j = scale * sum_d q_d K_j,d          for the keys j the query may see
 *     m = max_j s_j,  e_j = exp(s_j - m),  out = sum_j e_j V_j / sum_j e_j,
 *     lse = m + ln(sum_j e_j).
 * GQA ([P1] "Hybrid Attention Mechanisms"): q head hq reads kv head hq / (Hq/Hkv).
 * Sliding window ([P4] "混合注意力机制"): keys p - W < j <= p when W > 0.
 * Speculative queries ([P2] "EngineCore가 하는 일"): query i of q_len sits at position
 * L - q_len + i and sees keys j <= its position.
 * Chunked prefill ([P2] "EngineCore가 하는 일": each step computes num_new_tokens of a request,
 * its tokens with spec minus those already computed): sequence b's n_b query tokens are the
 * rows query_start_loc[b] .. query_start_loc[b+1]-1, at positions L - n_b + i, with the same
 * causal rule; the uniform case is query_start_loc[b] = b * q_len.
 */
typedef struct {
    const void *q;
    int32_t q_dtype, num_seqs, q_len, num_q_heads;
    const void *k_cache, *v_cache;
    int32_t cache_dtype, num_kv_heads, head_dim, block_size, num_blocks;
    const int32_t *block_table;
    int64_t bt_stride;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    double scale;
    int32_t window;
    double k_scale, v_scale;
    const int32_t *query_start_loc; /* [num_seqs + 1] query rows per sequence, or NULL: q_len each */
    const float *k_gscales, *v_gscales; /* INT4 caches: [num_kv_heads, head_dim / group_size] */
    int32_t group_size;
    const int32_t *seqs;        /* which sequences to compute */
    int32_t num_work;           /* items = len(seqs) * num_kv_heads */
    double *out;                /* [num_seqs * q_len, Hq, D] */
    double *lse;                /* [num_seqs * q_len, Hq] */
    int32_t next;               /* work counter */
    int32_t err;
    pthread_mutex_t lock;
} attn_job;

static int take_work(attn_job *J)
{
    pthread_mutex_lock(&J->lock);
    int w = J->next < J->num_work ? J->next++ : -1;
    pthread_mutex_unlock(&J->lock);
    return w;
}

static void set_err(attn_job *J, int32_t bits)
{
    pthread_mutex_lock(&J->lock);
    J->err |= bits;
    pthread_mutex_unlock(&J->lock);
}

static void attend_one(attn_job *J, int32_t b, int32_t h, double *K, double *V, double *s,
                       double *qv)
{
    const int32_t D = J->head_dim, bs = J->block_size, Hkv = J->num_kv_heads;
    const int32_t Hq = J->num_q_heads, g = Hq / Hkv;
    /* this sequence's query rows: first row and count */
    const int64_t row0 = J->query_start_loc ? J->query_start_loc[b] : (int64_t)b * J->q_len;
    const int64_t ql = J->query_start_loc ? J->query_start_loc[b + 1] - row0 : J->q_len;
    const int64_t L = J->seq_lens[b];
    if (ql < 0 || L < ql || (L + bs - 1) / bs > J->max_blocks_per_seq) {
        set_err(J, ORC_BAD_LEN);
        return;
    }
    /* materialise contiguous K_b, V_b for kv head h over the keys some query can see: with a
       window, blocks wholly before the first query's window have left it and may have been
       returned to the pool, so their table entries are not read */
    const int64_t first_key = J->window > 0 && L - ql - J->window + 1 > 0 ? L - ql - J->window + 1 : 0;
    for (int64_t j = first_key; j < L; ++j) {
        int64_t physical = J->block_table[(int64_t)b * J->bt_stride + j / bs];
        if (physical < 0 || physical >= J->num_blocks) {
            set_err(J, ORC_BAD_BLOCK);
            return;
        }
        int64_t base = ((physical * bs + j % bs) * Hkv + h) * (int64_t)D;
        for (int32_t d = 0; d < D; ++d) {
            double ksc = J->k_scale, vsc = J->v_scale;
            if (J->cache_dtype == ORC_INT4) {
                ksc = J->k_gscales[(int64_t)h * (D / J->group_size) + d / J->group_size];
                vsc = J->v_gscales[(int64_t)h * (D / J->group_size) + d / J->group_size];
            }
            K[j * D + d] = elem_to_double(J->k_cache, base + d, J->cache_dtype) * ksc;
            V[j * D + d] = elem_to_double(J->v_cache, base + d, J->cache_dtype) * vsc;
        }
    }
    for (int64_t i = 0; i < ql; ++i) {
        const int64_t p = L - ql + i;
        const int64_t lo = J->window > 0 ? (p - J->window + 1 > 0 ? p - J->window + 1 : 0) : 0;
        const int64_t tok = row0 + i;
        for (int32_t k = 0; k < g; ++k) {
            const int32_t hq = h * g + k;
            const int64_t qoff = (tok * Hq + hq) * (int64_t)D;
            for (int32_t d = 0; d < D; ++d)
                qv[d] = elem_to_double(J->q, qoff + d, J->q_dtype);
            double m = -INFINITY;
            for (int64_t j = lo; j <= p; ++j) {
                double acc = 0.0;
                for (int32_t d = 0; d < D; ++d)
                    acc += qv[d] * K[j * D + d];
                s[j] = J->scale * acc;
                if (s[j] > m)
                    m = s[j];
            }
            double den = 0.0;
            double *o = J->out + qoff;
            for (int32_t d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int64_t j = lo; j <= p; ++j) {
                double e = exp(s[j] - m);
                den += e;
                for (int32_t d = 0; d < D; ++d)
                    o[d] += e * V[j * D + d];
            }
            for (int32_t d = 0; d < D; ++d)
                o[d] /= den;
            J->lse[tok * Hq + hq] = m + log(den);
        }
    }
}

static void *attn_worker(void *arg)
{
    attn_job *J = (attn_job *)arg;
    int64_t cap = 0;
    for (int32_t i = 0; i < J->num_work / J->num_kv_heads; ++i)
        if (J->seq_lens[J->seqs[i]] > cap)
            cap = J->seq_lens[J->seqs[i]];
    if (cap < 1)
        cap = 1;
    double *K = malloc(sizeof(double) * cap * J->head_dim);
    double *V = malloc(sizeof(double) * cap * J->head_dim);
    double *s = malloc(sizeof(double) * cap);
    double *qv = malloc(sizeof(double) * J->head_dim);
    if (!K || !V || !s || !qv) {
        set_err(J, -1);
    } else {
        for (int w; (w = take_work(J)) >= 0;)
            attend_one(J, J->seqs[w / J->num_kv_heads], w % J->num_kv_heads, K, V, s, qv);
    }
    free(K);
    free(V);
    free(s);
    free(qv);
    return NULL;
}

static int32_t run_attention(attn_job *J, int32_t threads)
{
    pthread_mutex_init(&J->lock, NULL);
    if (threads < 1)
        threads = 1;
    pthread_t *tid = malloc(sizeof(pthread_t) * threads);
    int started = 0;
    for (int i = 0; tid && i < threads; ++i)
        if (pthread_create(&tid[i], NULL, attn_worker, J) == 0)
            ++started;
    if (started == 0)
        attn_worker(J);
    for (int i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    free(tid);
    pthread_mutex_destroy(&J->lock);
    return J->err;
}

int32_t orc_paged_attention(const void *q, int32_t q_dtype, int32_t num_seqs, int32_t q_len,
                            int32_t num_q_heads, const void *k_cache, const void *v_cache,
                            int32_t cache_dtype, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, const int32_t *block_table,
                            int64_t bt_stride, int32_t max_blocks_per_seq,
                            const int32_t *seq_lens, double scale, int32_t window,
                            double k_scale, double v_scale, const int32_t *seqs,
                            int32_t num_selected, double *out, double *lse, int32_t threads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    attn_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.q_dtype = q_dtype; J.num_seqs = num_seqs; J.q_len = q_len;
    J.num_q_heads = num_q_heads; J.k_cache = k_cache; J.v_cache = v_cache;
    J.cache_dtype = cache_dtype; J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
    J.block_size = block_size; J.num_blocks = num_blocks; J.block_table = block_table;
    J.bt_stride = bt_stride; J.max_blocks_per_seq = max_blocks_per_seq;
    J.seq_lens = seq_lens; J.scale = scale; J.window = window;
    J.k_scale = cache_dtype == ORC_E4M3 ? k_scale : 1.0;
    J.v_scale = cache_dtype == ORC_E4M3 ? v_scale : 1.0;
    J.seqs = seqs; J.num_work = num_selected * num_kv_heads;
    J.out = out; J.lse = lse;
    return run_attention(&J, threads);
}

/* The same attention with a different number of query rows per sequence (query_start_loc). */
int32_t orc_paged_attention_varlen(const void *q, int32_t q_dtype, int32_t num_seqs,
                                   const int32_t *query_start_loc, int32_t num_q_heads,
                                   const void *k_cache, const void *v_cache, int32_t cache_dtype,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int32_t num_blocks, const int32_t *block_table,
                                   int64_t bt_stride, int32_t max_blocks_per_seq,
                                   const int32_t *seq_lens, double scale, int32_t window,
                                   double k_scale, double v_scale, const int32_t *seqs,
                                   int32_t num_selected, double *out, double *lse, int32_t threads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return -1;
    attn_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.q_dtype = q_dtype; J.num_seqs = num_seqs; J.q_len = 0;
    J.query_start_loc = query_start_loc;
    J.num_q_heads = num_q_heads; J.k_cache = k_cache; J.v_cache = v_cache;
    J.cache_dtype = cache_dtype; J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
    J.block_size = block_size; J.num_blocks = num_blocks; J.block_table = block_table;
    J.bt_stride = bt_stride; J.max_blocks_per_seq = max_blocks_per_seq;
    J.seq_lens = seq_lens; J.scale = scale; J.window = window;
    J.k_scale = cache_dtype == ORC_E4M3 ? k_scale : 1.0;
    J.v_scale = cache_dtype == ORC_E4M3 ? v_scale : 1.0;
    J.seqs = seqs; J.num_work = num_selected * num_kv_heads;
    J.out = out; J.lse = lse;
    return run_attention(&J, threads);
}

/* The attention over an INT4 cache (uniform q_len), with per (head, dim group) scales. */
int32_t orc_paged_attention_int4(const void *q, int32_t q_dtype, int32_t num_seqs, int32_t q_len,
                                 int32_t num_q_heads, const void *k_cache, const void *v_cache,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t num_blocks, const int32_t *block_table, int64_t bt_stride,
                                 int32_t max_blocks_per_seq, const int32_t *seq_lens, double scale,
                                 int32_t window, const float *k_scales, const float *v_scales,
                                 int32_t group_size, const int32_t *seqs, int32_t num_selected,
                                 double *out, double *lse, int32_t threads)
{
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || group_size <= 0 ||
        head_dim % group_size != 0)
        return -1;
    attn_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.q_dtype = q_dtype; J.num_seqs = num_seqs; J.q_len = q_len;
    J.num_q_heads = num_q_heads; J.k_cache = k_cache; J.v_cache = v_cache;
    J.cache_dtype = ORC_INT4; J.num_kv_heads = num_kv_heads; J.head_dim = head_dim;
    J.block_size = block_size; J.num_blocks = num_blocks; J.block_table = block_table;
    J.bt_stride = bt_stride; J.max_blocks_per_seq = max_blocks_per_seq;
    J.seq_lens = seq_lens; J.scale = scale; J.window = window;
    J.k_scale = 1.0; J.v_scale = 1.0;
    J.k_gscales = k_scales; J.v_gscales = v_scales; J.group_size = group_size;
    J.seqs = seqs; J.num_work = num_selected * num_kv_heads;
    J.out = out; J.lse = lse;
    return run_attention(&J, threads);
}
