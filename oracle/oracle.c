/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the paged KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, calls or
 * includes this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no header, helper, table or constant
 * with the CUDA sources.
 *
 * What it computes, and where the pages define it:
 *
 *  - orc_write_flat: the cache write.  For each new token t whose slot_mapping
 *    entry is non-negative, copy (or quantise) its K/V row to cache row `slot`.
 *    The cache is indexed by the flat slot itself, never split into
 *    (block, offset).  A negative slot means "no destination": nothing is
 *    written.  ("Inside vLLM CUDA Kernels: KV-Cache Writes and Paged
 *    Attention", Part 2, "Decomposing a Slot into Block and Offset";
 *    "How vLLM CUDA Kernels Write and Read the Paged KV Cache", "Writing K and
 *    V into the cache".)
 *
 *  - orc_e4m3_encode / orc_e4m3_decode: the FP8 E4M3 format of the OCP 8-bit
 *    Floating Point specification (OFP8): 1 sign bit, 4 exponent bits with
 *    bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite
 *    magnitude 448, subnormals m * 2^-9.  The write side "applies scaling and
 *    type conversion" (Inside vLLM CUDA Kernels, Part 2, k_op); the reading
 *    taken here is: y = fl32(fl32(x) / fl32(scale)), then y rounded to the
 *    nearest E4M3 value, ties to the even code, magnitudes above 448
 *    saturating to 448, NaN giving the code 0x7F.
 *
 *  - orc_dense_decode: single-query attention for one sequence over its
 *    logically contiguous K/V, in fp64:  z_t = scale * q . k_t,
 *    p = softmax(z), o = sum_t p_t v_t, with the GQA head map
 *    kv_head = q_head / (Hq / Hkv).  ("Inside vLLM CUDA Kernels", Part 3,
 *    "How Each K/V Tile Contributes to the Output"; "vLLM 源码完全拆解（七）",
 *    先明确问题 and GQA 的映射.)  A sequence of length 0 gives a zero output.
 *
 *  - orc_paged_walk_decode: the same attention reached by walking the block
 *    table token by token with the online-softmax recurrence (m, l, acc)
 *    ("Inside vLLM CUDA Kernels", Part 3, online softmax; "PagedAttention
 *    kernel: paged KV cache & block tables", Code).  Used only to check the
 *    oracle itself: paged == dense for any physical permutation.
 *
 *  - orc_write_flat_heads: the write with one FP8 scale per KV head ("Inside
 *    vLLM CUDA Kernels", Part 2, why layout and quantization scale produce two
 *    copy paths: kv_scale_stride == 0 means every head shares one scale,
 *    otherwise head h uses scale[h * kv_scale_stride]).
 *
 *  - orc_attention_causal: n query tokens of one sequence over its L K/V rows.
 *    Query i sits at position L - n + i and sees tokens t <= L - n + i (the
 *    varlen read path of "Inside vLLM CUDA Kernels", Part 3: query_start_loc
 *    packs a request's new tokens, seq_lens bounds the visible history; the
 *    reading taken here is the usual causal mask with the new tokens at the end
 *    of the history).  With ALiBi ("vLLM 源码完全拆解（七）", the QK step: the
 *    kernel adds the head's slope a_h times the token's non-positive distance
 *    from the current position, which has bias 0), the logit is
 *    scale * q_i . k_t + a_h * (t - (L - n + i)).  n = 1 is single-query decode.
 *
 *  - orc_partial_decode / orc_lse_merge: the split-KV form -- the unnormalised
 *    state (m, l, acc) of one token range, and the max/log-sum-exp merge of
 *    several ranges ("Inside vLLM CUDA Kernels", Part 3, "Split-KV changes the
 *    work partition, not the softmax identity"; "vLLM 源码完全拆解（七）",
 *    V1 与 V2).  Used only to check the oracle itself: split == unsplit.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* element codes used by this file only */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_E4M3 = 3 };

/* ---------------------------------------------------------------- helpers */

static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;   /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* IEEE binary16 -> float, written from the format's definition. */
static float f16_bits_to_float(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 31)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (float)(s ? -v : v);
}

static float load_elem(const void *base, int dtype, int64_t i)
{
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * i, 4);
        return f;
    }
    uint16_t b;
    memcpy(&b, (const char *)base + 2 * i, 2);
    return dtype == ORC_BF16 ? bf16_bits_to_float(b) : f16_bits_to_float(b);
}

static int elem_bytes(int dtype)
{
    return dtype == ORC_F32 ? 4 : dtype == ORC_E4M3 ? 1 : 2;
}

/* ------------------------------------------------------------- FP8 E4M3 */

/* Value of an E4M3 code (OFP8): normal (1 + m/8) 2^(e-7), subnormal m 2^-9. */
double orc_e4m3_decode(uint8_t code)
{
    int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);
    else
        mag = ldexp((double)(8 + m), e - 10);
    return s ? -mag : mag;
}

/* Nearest finite E4M3 code to x by exhaustive search over the 127 magnitude
 * codes 0x00..0x7E; on a tie the code with an even last mantissa bit wins.
 * |x| > 448 (and +-inf) saturate to +-448; NaN gives 0x7F; the sign of zero
 * and of values that round to zero is kept. */
uint8_t orc_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    int best = 0;
    double bestd = INFINITY;
    if (a > 448.0)
        return (uint8_t)((neg << 7) | 0x7E);
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(orc_e4m3_decode((uint8_t)c) - a);
        if (d < bestd || (d == bestd && (c & 1) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)((neg << 7) | best);
}

/* The write-side conversion of one element into an E4M3 cache. */
uint8_t orc_quantize_e4m3(float x, float scale)
{
    float y = x / scale;   /* one IEEE fp32 division, rounded to nearest */
    return orc_e4m3_encode(y);
}

/* ------------------------------------------------------------------ write */

/*
 * rows:       [T, Hkv, D] elements of rows_dtype; token t starts at element
 *             t * row_stride, head h at + h * D.
 * slots:      int64 [T]; slot < 0 -> row t is not written.
 * cache_flat: [num_slots, Hkv, D] elements of cache_dtype, indexed by slot.
 * cache_dtype == rows_dtype copies bytes; cache_dtype == ORC_E4M3 quantises.
 * Returns 0, or -1 if a slot is >= num_slots, or -2 for an unsupported pair.
 */
int orc_write_flat(const void *rows, int rows_dtype, int64_t T, int64_t row_stride,
                   int Hkv, int D, const int64_t *slots, int64_t num_slots,
                   void *cache_flat, int cache_dtype, float scale)
{
    int rb = elem_bytes(rows_dtype), cb = elem_bytes(cache_dtype);
    if (cache_dtype != rows_dtype && cache_dtype != ORC_E4M3)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots)
            return -1;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = t * row_stride + (int64_t)h * D + d;
                int64_t dst = (slot * Hkv + h) * (int64_t)D + d;
                if (cache_dtype == rows_dtype) {
                    memcpy((char *)cache_flat + dst * cb, (const char *)rows + src * rb, (size_t)rb);
                } else {
                    uint8_t code = orc_quantize_e4m3(load_elem(rows, rows_dtype, src), scale);
                    ((uint8_t *)cache_flat)[dst] = code;
                }
            }
        }
    }
    return 0;
}

/* ----------------------------------------------------------------- decode */

/*
 * One sequence.  q: [Hq, D]; K, V: [L, Hkv, D] (logical token order);
 * out: [Hq, D].  probs (nullable): [Hq, L] receives the softmax weights.
 * Returns -1 if Hq is not a multiple of Hkv.
 */
int orc_dense_decode(const double *q, const double *K, const double *V, int64_t L,
                     int Hq, int Hkv, int D, double scale, double *out, double *probs)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    int G = Hq / Hkv;
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;                       /* GQA: query head -> KV head */
        double *o = out + (int64_t)h * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        if (L == 0)
            continue;
        double M = -INFINITY;
        for (int64_t t = 0; t < L; ++t) {
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                z += q[(int64_t)h * D + d] * K[(t * Hkv + g) * (int64_t)D + d];
            z *= scale;
            if (z > M)
                M = z;
        }
        double S = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                z += q[(int64_t)h * D + d] * K[(t * Hkv + g) * (int64_t)D + d];
            S += exp(z * scale - M);
        }
        for (int64_t t = 0; t < L; ++t) {
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                z += q[(int64_t)h * D + d] * K[(t * Hkv + g) * (int64_t)D + d];
            double p = exp(z * scale - M) / S;
            if (probs)
                probs[(int64_t)h * L + t] = p;
            for (int d = 0; d < D; ++d)
                o[d] += p * V[(t * Hkv + g) * (int64_t)D + d];
        }
    }
    return 0;
}

/*
 * Split-KV state of one token range [t0, t1) of one sequence, fp64:
 * m[h] = max_t z_t, l[h] = sum_t exp(z_t - m), acc[h][d] = sum_t exp(z_t - m) v_t[d].
 * An empty range gives m = -inf, l = 0, acc = 0.
 */
int orc_partial_decode(const double *q, const double *K, const double *V, int64_t t0, int64_t t1,
                       int Hq, int Hkv, int D, double scale, double *m, double *l, double *acc)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    int G = Hq / Hkv;
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;
        double mh = -INFINITY, lh = 0.0;
        double *a = acc + (int64_t)h * D;
        for (int d = 0; d < D; ++d)
            a[d] = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                z += q[(int64_t)h * D + d] * K[(t * Hkv + g) * (int64_t)D + d];
            z *= scale;
            if (z > mh)
                mh = z;
        }
        for (int64_t t = t0; t < t1; ++t) {
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                z += q[(int64_t)h * D + d] * K[(t * Hkv + g) * (int64_t)D + d];
            double w = exp(z * scale - mh);
            lh += w;
            for (int d = 0; d < D; ++d)
                a[d] += w * V[(t * Hkv + g) * (int64_t)D + d];
        }
        m[h] = mh;
        l[h] = lh;
    }
    return 0;
}

/*
 * Merge P partial states of one (sequence, head): M = max_p m_p,
 * out = sum_p exp(m_p - M) acc_p / sum_p exp(m_p - M) l_p.
 * m, l: [P]; acc: [P, D]; out: [D].  All-empty input gives a zero output.
 */
void orc_lse_merge(const double *m, const double *l, const double *acc, int P, int D, double *out)
{
    double M = -INFINITY, den = 0.0;
    for (int p = 0; p < P; ++p)
        if (m[p] > M)
            M = m[p];
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    if (M == -INFINITY)
        return;
    for (int p = 0; p < P; ++p) {
        double w = exp(m[p] - M);   /* an empty part has m = -inf, w = 0 */
        den += w * l[p];
        for (int d = 0; d < D; ++d)
            out[d] += w * acc[(int64_t)p * D + d];
    }
    for (int d = 0; d < D; ++d)
        out[d] /= den;
}

/*
 * The block-table walk, token by token, with the online-softmax recurrence
 * m_new = max(m, z), alpha = exp(m - m_new), l = alpha l + exp(z - m_new),
 * acc = alpha acc + exp(z - m_new) v, o = acc / l.
 * pool_k, pool_v: [num_slots, Hkv, D] indexed by flat slot; block_table: the
 * sequence's row (int32); logical token t lives at slot
 * block_table[t / block_size] * block_size + t % block_size.
 */
int orc_paged_walk_decode(const double *q, const double *pool_k, const double *pool_v,
                          const int32_t *block_table, int block_size, int64_t L,
                          int Hq, int Hkv, int D, double scale, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0 || block_size <= 0)
        return -1;
    int G = Hq / Hkv;
    for (int h = 0; h < Hq; ++h) {
        int g = h / G;
        double m = -INFINITY, l = 0.0;
        double *o = out + (int64_t)h * D;
        for (int d = 0; d < D; ++d)
            o[d] = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            int64_t logical_block = t / block_size;
            int64_t offset = t % block_size;
            int64_t slot = (int64_t)block_table[logical_block] * block_size + offset;
            const double *k = pool_k + (slot * Hkv + g) * (int64_t)D;
            const double *v = pool_v + (slot * Hkv + g) * (int64_t)D;
            double z = 0.0;
            for (int d = 0; d < D; ++d)
                z += q[(int64_t)h * D + d] * k[d];
            z *= scale;
            double m_new = z > m ? z : m;
            double alpha = exp(m - m_new);   /* exp(-inf) = 0 on the first token */
            double p = exp(z - m_new);
            l = alpha * l + p;
            for (int d = 0; d < D; ++d)
                o[d] = alpha * o[d] + p * v[d];
            m = m_new;
        }
        if (L > 0)
            for (int d = 0; d < D; ++d)
                o[d] /= l;
    }
    return 0;
}

/* ------------------------------------------------- per-head scales, causal */

/*
 * orc_write_flat with one scale per KV head: head h of every row quantises with
 * scales[h].  Same arguments otherwise; scales is [Hkv].
 */
int orc_write_flat_heads(const void *rows, int rows_dtype, int64_t T, int64_t row_stride,
                         int Hkv, int D, const int64_t *slots, int64_t num_slots,
                         void *cache_flat, int cache_dtype, const float *scales)
{
    int rb = elem_bytes(rows_dtype), cb = elem_bytes(cache_dtype);
    if (cache_dtype != rows_dtype && cache_dtype != ORC_E4M3)
        return -2;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots)
            return -1;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                int64_t src = t * row_stride + (int64_t)h * D + d;
                int64_t dst = (slot * Hkv + h) * (int64_t)D + d;
                if (cache_dtype == rows_dtype)
                    memcpy((char *)cache_flat + dst * cb, (const char *)rows + src * rb, (size_t)rb);
                else
                    ((uint8_t *)cache_flat)[dst] = orc_quantize_e4m3(load_elem(rows, rows_dtype, src), scales[h]);
            }
        }
    }
    return 0;
}

/*
 * n query tokens of one sequence, causal, optional ALiBi.  q: [n, Hq, D];
 * K, V: [L, Hkv, D] in logical order; slopes: [Hq] or NULL; out: [n, Hq, D].
 * Query i (position L - n + i) sees tokens 0 .. L - n + i:
 *   z_t = scale * q_i . k_t + slope_h * (t - (L - n + i)),  o = sum_t softmax(z)_t v_t.
 * Returns -1 if Hq is not a multiple of Hkv, -2 if n > L.
 */
int orc_attention_causal(const double *q, const double *K, const double *V, int64_t n, int64_t L,
                         int Hq, int Hkv, int D, double scale, const double *slopes, double *out)
{
    if (Hkv <= 0 || Hq % Hkv != 0)
        return -1;
    if (n > L)
        return -2;
    int G = Hq / Hkv;
    for (int64_t i = 0; i < n; ++i) {
        int64_t pos = L - n + i;             /* this query's position; it sees 0 .. pos */
        for (int h = 0; h < Hq; ++h) {
            int g = h / G;
            const double *qh = q + (i * Hq + h) * (int64_t)D;
            double *o = out + (i * Hq + h) * (int64_t)D;
            double a = slopes ? slopes[h] : 0.0;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            double M = -INFINITY;
            for (int64_t t = 0; t <= pos; ++t) {
                double z = 0.0;
                for (int d = 0; d < D; ++d)
                    z += qh[d] * K[(t * Hkv + g) * (int64_t)D + d];
                z = z * scale + a * (double)(t - pos);
                if (z > M)
                    M = z;
            }
            double S = 0.0;
            for (int64_t t = 0; t <= pos; ++t) {
                double z = 0.0;
                for (int d = 0; d < D; ++d)
                    z += qh[d] * K[(t * Hkv + g) * (int64_t)D + d];
                S += exp(z * scale + a * (double)(t - pos) - M);
            }
            for (int64_t t = 0; t <= pos; ++t) {
                double z = 0.0;
                for (int d = 0; d < D; ++d)
                    z += qh[d] * K[(t * Hkv + g) * (int64_t)D + d];
                double p = exp(z * scale + a * (double)(t - pos) - M) / S;
                for (int d = 0; d < D; ++d)
                    o[d] += p * V[(t * Hkv + g) * (int64_t)D + d];
            }
        }
    }
    return 0;
}
