/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV decode attention and
 * its two companion cache operations.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * checked against.  Only the test suite, the smoke check in __graft_entry__ and
 * the CPU-baseline leg of bench.py may load it.  The product library shares no
 * code, header, table or helper with it, and nothing on the product path may
 * call it.
 *
 * What it computes, and where the pages define it:
 *
 *  - Address translation: token position pos of a sequence lives at offset
 *    pos % B of physical block table[pos / B].  ("PagedAttention: Virtual
 *    Memory for the KV Cache", section "A block table preserves token order";
 *    "Paged Attention and vLLM", section "Block Table and Logical-to-Physical
 *    Mapping", the definition of tau_s.)
 *
 *  - Decode attention for one query per sequence:
 *        o = softmax(scale * q . [K_tau(0) || K_tau(1) || ...]^T) . V
 *    over exactly the ctx_len stored tokens.  ("Paged Attention and vLLM",
 *    "Block Table and Logical-to-Physical Mapping", the a_t equation; the
 *    value product is the usual attention output.)  The oracle is the plain
 *    definition: gather a contiguous K and V, form every logit, subtract the
 *    maximum, exponentiate with libm exp, normalise, multiply by V.  Inputs are
 *    widened exactly to double; every operation is in double.
 *
 *  - The partitioned form: per partition b, m_b = max logit, l_b = sum of
 *    exp(logit - m_b), acc_b = sum of exp(logit - m_b) v_i; then
 *    o = sum_b e^(m_b - m*) acc_b / sum_b e^(m_b - m*) l_b with m* = max_b m_b.
 *    ("Paged Attention and vLLM", section "Paged Attention CUDA Kernel", the
 *    m_b / l_b / v_b^acc equation and the merge equation.)  This is a second,
 *    independent evaluation used to pin the first.
 *
 *  - KV write: each new token's key and value rows are copied to its slot
 *    (slot = physical block * B + offset); negative slots are skipped.
 *    ("PagedAttention: Virtual Memory for the KV Cache", section "Sharing a
 *    prefix and copying a partial block": "... writes the new entry".)
 *
 *  - Block copy: copy-on-write copy of a whole physical block (all KV heads,
 *    all B slots, keys and values).  (Same section; "Paged Attention and vLLM",
 *    "Continuous Batching and Scheduler", the copy-on-write rule.)
 *
 *  - Attention for a chunk of query tokens per sequence (chunked prefill,
 *    verification of drafted tokens): the n_s query tokens of sequence s are
 *    its last n_s positions, len - n_s .. len - 1, and the query at position
 *    pos attends to positions 0 .. pos only -- the cache a one-token-at-a-time
 *    decode would hold at that point ("Paged Attention and vLLM", "KV Cache
 *    Fundamentals": the key cache at length t is the keys of tokens 1..t;
 *    "KV Cache Optimization and Management", "Common misconception": paging
 *    leaves the scores and the softmax unchanged).  Plain definition again,
 *    one query row at a time.
 *
 *  - Block swap: the same whole-block copy between two pools (device blocks to
 *    host blocks and back), for preemption ("Paged Attention and vLLM",
 *    "Continuous Batching and Scheduler": evict a sequence's physical blocks to
 *    CPU and swap them back later).
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - the query-head to KV-head map is consecutive grouping: kv = h / (Hq/Hkv);
 *  - ctx_len == 0 gives an all-zero output;
 *  - the table entries past ceil(ctx_len / B) are never read;
 *  - q is stored in the cache dtype, the output is returned in double.
 *
 * Storage layouts (row-major, element type given by `dtype`):
 *   q        [S, Hq, D]   (chunk attention: [T, Hq, D], T query tokens,
 *                          sequence s owning rows query_start[s] .. query_start[s+1]-1)
 *   k_cache  [N, Hkv, B, D]     v_cache the same
 *   tables   int32 [S, max_blocks]
 *   lens     int32 [S]
 *   out      double [S, Hq, D]
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared pa_oracle.c -lm
 * (no fused multiply-add contraction, so x86 and Arm hosts give the same bits).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* ---- exact widening of the three storage types to double ------------------ */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double mag;
    if (e == 0)
        mag = ldexp((double)f, -24);             /* subnormal: f * 2^-14 * 2^-10 */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexp((double)(f | 0x400), e - 25); /* (1024 + f) * 2^(e-15-10) */
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double load_elem(const void *base, size_t idx, int dtype)
{
    switch (dtype) {
    case ORACLE_F32: return (double)((const float *)base)[idx];
    case ORACLE_F16: return f16_bits_to_double(((const uint16_t *)base)[idx]);
    default:         return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    }
}

static size_t elem_size(int dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

/* ---- address translation ---------------------------------------------------- */

/* Physical block and offset of token `pos` of a sequence whose table row is `row`. */
static int translate(const int32_t *row, int B, int pos, int *phys, int *off)
{
    *phys = row[pos / B];
    *off = pos % B;
    return 0;
}

int pa_oracle_slot(const int32_t *row, int B, int pos, int64_t *slot)
{
    int phys, off;
    if (B <= 0 || pos < 0)
        return -1;
    translate(row, B, pos, &phys, &off);
    *slot = (int64_t)phys * B + off;
    return 0;
}

/* slot of token positions[t] of sequence seq_of[t]; out[t] = -1 where positions[t] < 0. */
int pa_oracle_slot_mapping(int T, const int32_t *tables, int max_blocks, int B,
                           const int32_t *seq_of, const int32_t *positions, int64_t *out)
{
    for (int t = 0; t < T; ++t) {
        if (positions[t] < 0) { out[t] = -1; continue; }
        if (positions[t] / B >= max_blocks)
            return -1;
        if (pa_oracle_slot(tables + (size_t)seq_of[t] * max_blocks, B, positions[t], &out[t]))
            return -1;
    }
    return 0;
}

/* ---- gather: one sequence, one KV head, contiguous K and V in double ------- */

static int gather(const void *k_cache, const void *v_cache, int dtype,
                  int Hkv, int B, int D, int N, const int32_t *row, int len, int kvh,
                  double *Kc, double *Vc)
{
    for (int i = 0; i < len; ++i) {
        int phys, off;
        translate(row, B, i, &phys, &off);
        if (phys < 0 || phys >= N)
            return -1;
        size_t base = (((size_t)phys * Hkv + kvh) * B + off) * (size_t)D;
        for (int d = 0; d < D; ++d) {
            Kc[(size_t)i * D + d] = load_elem(k_cache, base + d, dtype);
            Vc[(size_t)i * D + d] = load_elem(v_cache, base + d, dtype);
        }
    }
    return 0;
}

static int check_dims(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks,
                      int dtype, const int32_t *lens)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || B <= 0 || N <= 0 || max_blocks <= 0)
        return -1;
    if (Hq % Hkv != 0 || dtype < 0 || dtype > 2)
        return -1;
    for (int s = 0; s < S; ++s)
        if (lens[s] < 0 || (int64_t)lens[s] > (int64_t)max_blocks * B)
            return -1;
    return 0;
}

/* ---- decode, plain softmax definition --------------------------------------- */

int pa_oracle_decode(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks, int dtype,
                     const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *tables, const int32_t *lens, double scale, double *out)
{
    if (check_dims(S, Hq, Hkv, D, B, N, max_blocks, dtype, lens))
        return -1;
    const int G = Hq / Hkv;
    int rc = 0;
    for (int s = 0; s < S && rc == 0; ++s) {
        const int len = lens[s];
        const int32_t *row = tables + (size_t)s * max_blocks;
        double *Kc = malloc(sizeof(double) * ((size_t)len * D + 1));
        double *Vc = malloc(sizeof(double) * ((size_t)len * D + 1));
        double *z = malloc(sizeof(double) * ((size_t)len + 1));
        if (!Kc || !Vc || !z) { free(Kc); free(Vc); free(z); return -2; }
        for (int h = 0; h < Hq && rc == 0; ++h) {
            const int kvh = h / G;
            double *o = out + ((size_t)s * Hq + h) * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            if (len == 0)
                continue;
            if (gather(k_cache, v_cache, dtype, Hkv, B, D, N, row, len, kvh, Kc, Vc)) {
                rc = -1;
                break;
            }
            const size_t qbase = ((size_t)s * Hq + h) * D;
            /* logits */
            for (int i = 0; i < len; ++i) {
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += load_elem(q, qbase + d, dtype) * Kc[(size_t)i * D + d];
                z[i] = scale * dot;
            }
            /* softmax */
            double m = z[0];
            for (int i = 1; i < len; ++i)
                if (z[i] > m)
                    m = z[i];
            double den = 0.0;
            for (int i = 0; i < len; ++i) {
                z[i] = exp(z[i] - m);
                den += z[i];
            }
            /* weighted sum of values */
            for (int i = 0; i < len; ++i)
                for (int d = 0; d < D; ++d)
                    o[d] += z[i] * Vc[(size_t)i * D + d];
            for (int d = 0; d < D; ++d)
                o[d] /= den;
        }
        free(Kc);
        free(Vc);
        free(z);
    }
    return rc;
}

/* ---- chunk attention: several query tokens per sequence, causal -------------- */

int pa_oracle_chunk_attention(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks, int dtype,
                              const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *tables, const int32_t *lens, const int32_t *query_start,
                              int T, double scale, double *out)
{
    if (check_dims(S, Hq, Hkv, D, B, N, max_blocks, dtype, lens) || T < 0 || query_start[0] != 0 ||
        query_start[S] != T)
        return -1;
    for (int s = 0; s < S; ++s) {
        const int n = query_start[s + 1] - query_start[s];
        if (n < 0 || n > lens[s])
            return -1;
    }
    const int G = Hq / Hkv;
    int rc = 0;
    for (int s = 0; s < S && rc == 0; ++s) {
        const int len = lens[s];
        const int n = query_start[s + 1] - query_start[s];
        const int32_t *row = tables + (size_t)s * max_blocks;
        double *Kc = malloc(sizeof(double) * ((size_t)len * D + 1));
        double *Vc = malloc(sizeof(double) * ((size_t)len * D + 1));
        double *z = malloc(sizeof(double) * ((size_t)len + 1));
        if (!Kc || !Vc || !z) { free(Kc); free(Vc); free(z); return -2; }
        for (int kvh = 0; kvh < Hkv && rc == 0 && n > 0; ++kvh) {
            if (gather(k_cache, v_cache, dtype, Hkv, B, D, N, row, len, kvh, Kc, Vc)) {
                rc = -1;
                break;
            }
            for (int t = 0; t < n; ++t) {
                const int pos = len - n + t;   /* this query's position; keys 0..pos */
                const size_t tok = (size_t)query_start[s] + t;
                for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
                    const size_t qbase = (tok * Hq + h) * D;
                    double *o = out + qbase;
                    for (int i = 0; i <= pos; ++i) {
                        double dot = 0.0;
                        for (int d = 0; d < D; ++d)
                            dot += load_elem(q, qbase + d, dtype) * Kc[(size_t)i * D + d];
                        z[i] = scale * dot;
                    }
                    double m = z[0];
                    for (int i = 1; i <= pos; ++i)
                        if (z[i] > m)
                            m = z[i];
                    double den = 0.0;
                    for (int i = 0; i <= pos; ++i) {
                        z[i] = exp(z[i] - m);
                        den += z[i];
                    }
                    for (int d = 0; d < D; ++d)
                        o[d] = 0.0;
                    for (int i = 0; i <= pos; ++i)
                        for (int d = 0; d < D; ++d)
                            o[d] += z[i] * Vc[(size_t)i * D + d];
                    for (int d = 0; d < D; ++d)
                        o[d] /= den;
                }
            }
        }
        free(Kc);
        free(Vc);
        free(z);
    }
    return rc;
}

/* ---- decode, partitioned form with the log-sum-exp merge -------------------- */

int pa_oracle_decode_partitioned(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks,
                                 int dtype, const void *q, const void *k_cache,
                                 const void *v_cache, const int32_t *tables,
                                 const int32_t *lens, double scale, int partition_size,
                                 double *out)
{
    if (check_dims(S, Hq, Hkv, D, B, N, max_blocks, dtype, lens) || partition_size <= 0)
        return -1;
    const int G = Hq / Hkv;
    int rc = 0;
    for (int s = 0; s < S && rc == 0; ++s) {
        const int len = lens[s];
        const int nparts = (len + partition_size - 1) / partition_size;
        const int32_t *row = tables + (size_t)s * max_blocks;
        double *Kc = malloc(sizeof(double) * ((size_t)len * D + 1));
        double *Vc = malloc(sizeof(double) * ((size_t)len * D + 1));
        double *mb = malloc(sizeof(double) * ((size_t)nparts + 1));
        double *lb = malloc(sizeof(double) * ((size_t)nparts + 1));
        double *accb = malloc(sizeof(double) * ((size_t)nparts * D + 1));
        if (!Kc || !Vc || !mb || !lb || !accb) {
            free(Kc); free(Vc); free(mb); free(lb); free(accb);
            return -2;
        }
        for (int h = 0; h < Hq && rc == 0; ++h) {
            const int kvh = h / G;
            double *o = out + ((size_t)s * Hq + h) * D;
            for (int d = 0; d < D; ++d)
                o[d] = 0.0;
            if (len == 0)
                continue;
            if (gather(k_cache, v_cache, dtype, Hkv, B, D, N, row, len, kvh, Kc, Vc)) {
                rc = -1;
                break;
            }
            const size_t qbase = ((size_t)s * Hq + h) * D;
            /* per partition: m_b, l_b, acc_b */
            for (int b = 0; b < nparts; ++b) {
                const int i0 = b * partition_size;
                const int i1 = (i0 + partition_size < len) ? i0 + partition_size : len;
                double m = -INFINITY;
                for (int i = i0; i < i1; ++i) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += load_elem(q, qbase + d, dtype) * Kc[(size_t)i * D + d];
                    if (scale * dot > m)
                        m = scale * dot;
                }
                double l = 0.0;
                double *acc = accb + (size_t)b * D;
                for (int d = 0; d < D; ++d)
                    acc[d] = 0.0;
                for (int i = i0; i < i1; ++i) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d)
                        dot += load_elem(q, qbase + d, dtype) * Kc[(size_t)i * D + d];
                    const double w = exp(scale * dot - m);
                    l += w;
                    for (int d = 0; d < D; ++d)
                        acc[d] += w * Vc[(size_t)i * D + d];
                }
                mb[b] = m;
                lb[b] = l;
            }
            /* merge */
            double mstar = mb[0];
            for (int b = 1; b < nparts; ++b)
                if (mb[b] > mstar)
                    mstar = mb[b];
            double den = 0.0;
            for (int b = 0; b < nparts; ++b) {
                const double c = exp(mb[b] - mstar);
                den += c * lb[b];
                for (int d = 0; d < D; ++d)
                    o[d] += c * accb[(size_t)b * D + d];
            }
            for (int d = 0; d < D; ++d)
                o[d] /= den;
        }
        free(Kc); free(Vc); free(mb); free(lb); free(accb);
    }
    return rc;
}

/* ---- KV write: copy each new token's rows to its slot ----------------------- */

int pa_oracle_write_kv(int T, int Hkv, int D, int B, int N, int dtype,
                       const void *k, const void *v, const int64_t *slots,
                       void *k_cache, void *v_cache)
{
    const size_t es = elem_size(dtype);
    const size_t row = (size_t)D * es;
    for (int t = 0; t < T; ++t) {
        const int64_t slot = slots[t];
        if (slot < 0)
            continue;
        if (slot >= (int64_t)N * B)
            return -1;
        const int64_t phys = slot / B;
        const int64_t off = slot % B;
        for (int h = 0; h < Hkv; ++h) {
            const size_t dst = (((size_t)phys * Hkv + h) * B + (size_t)off) * row;
            const size_t src = ((size_t)t * Hkv + h) * row;
            memcpy((char *)k_cache + dst, (const char *)k + src, row);
            memcpy((char *)v_cache + dst, (const char *)v + src, row);
        }
    }
    return 0;
}

/* ---- block copy: whole-block copy for each (src, dst) pair ------------------ */

int pa_oracle_copy_blocks(int Hkv, int D, int B, int N, int dtype,
                          void *k_cache, void *v_cache, const int64_t *pairs, int P)
{
    const size_t blk = (size_t)Hkv * B * D * elem_size(dtype);
    for (int p = 0; p < P; ++p) {
        const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= N || dst < 0 || dst >= N)
            return -1;
        memmove((char *)k_cache + (size_t)dst * blk, (const char *)k_cache + (size_t)src * blk, blk);
        memmove((char *)v_cache + (size_t)dst * blk, (const char *)v_cache + (size_t)src * blk, blk);
    }
    return 0;
}

/* ---- block swap between two pools: whole-block copy for each (src, dst) pair */

int pa_oracle_swap_blocks(int Hkv, int D, int B, int dtype, const void *from_k, const void *from_v, int from_n,
                          void *to_k, void *to_v, int to_n, const int64_t *pairs, int P)
{
    const size_t blk = (size_t)Hkv * B * D * elem_size(dtype);
    for (int p = 0; p < P; ++p) {
        const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
        if (src < 0 || src >= from_n || dst < 0 || dst >= to_n)
            return -1;
        memcpy((char *)to_k + (size_t)dst * blk, (const char *)from_k + (size_t)src * blk, blk);
        memcpy((char *)to_v + (size_t)dst * blk, (const char *)from_v + (size_t)src * blk, blk);
    }
    return 0;
}
