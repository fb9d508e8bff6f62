/*
 * oracle_stress.c -- random small problems through every entry point of the
 * CPU oracle (oracle/pa_oracle.c), for builds with AddressSanitizer and
 * UndefinedBehaviorSanitizer.  Besides memory safety it checks, on each
 * problem:
 *   - the partitioned decode agrees with the plain definition (1e-9);
 *   - the last query of each chunk equals a decode over the whole context;
 *   - a KV write puts each row at its slot and skips negative slots, a block
 *     copy and a block swap move whole blocks;
 *   - out-of-range lengths and bad query ranges are refused (-1).
 * Usage: oracle_stress <seed> <problems>; exit status 0 when every check holds.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

int pa_oracle_slot(const int32_t *row, int B, int pos, int64_t *slot);
int pa_oracle_decode(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks, int dtype, const void *q,
                     const void *k_cache, const void *v_cache, const int32_t *tables, const int32_t *lens,
                     double scale, double *out);
int pa_oracle_decode_partitioned(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks, int dtype,
                                 const void *q, const void *k_cache, const void *v_cache, const int32_t *tables,
                                 const int32_t *lens, double scale, int partition_size, double *out);
int pa_oracle_chunk_attention(int S, int Hq, int Hkv, int D, int B, int N, int max_blocks, int dtype,
                              const void *q, const void *k_cache, const void *v_cache, const int32_t *tables,
                              const int32_t *lens, const int32_t *query_start, int T, double scale, double *out);
int pa_oracle_write_kv(int T, int Hkv, int D, int B, int N, int dtype, const void *k, const void *v,
                       const int64_t *slots, void *k_cache, void *v_cache);
int pa_oracle_copy_blocks(int Hkv, int D, int B, int N, int dtype, void *k_cache, void *v_cache,
                          const int64_t *pairs, int P);
int pa_oracle_swap_blocks(int Hkv, int D, int B, int dtype, const void *from_k, const void *from_v, int from_n,
                          void *to_k, void *to_v, int to_n, const int64_t *pairs, int P);

static uint64_t rng_state;
static uint32_t rnd(void) { /* xorshift64* */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (uint32_t)((rng_state * 0x2545F4914F6CDD1Dull) >> 32);
}
static int below(int n) { return n <= 0 ? 0 : (int)(rnd() % (uint32_t)n); }

static int failures = 0;
#define CHECK(cond, ...)                                              \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "check failed at line %d: ", __LINE__);   \
            fprintf(stderr, __VA_ARGS__);                             \
            fprintf(stderr, "\n");                                    \
            if (++failures > 20) exit(1);                             \
        }                                                             \
    } while (0)

/* A finite value of magnitude about 2^-3 .. 2^3 in the storage type. */
static void fill(void *buf, size_t n, int dtype) {
    for (size_t i = 0; i < n; ++i) {
        const uint32_t sign = rnd() & 1u, mant = rnd();
        if (dtype == 0) {
            const float x = (float)((int)(mant % 2001) - 1000) / 125.0f;
            ((float *)buf)[i] = sign ? -x : x;
        } else if (dtype == 1) { /* f16: exponent 12..18 */
            ((uint16_t *)buf)[i] = (uint16_t)((sign << 15) | ((12u + mant % 7u) << 10) | ((mant >> 8) & 0x3ffu));
        } else { /* bf16: exponent 124..130 */
            ((uint16_t *)buf)[i] = (uint16_t)((sign << 15) | ((124u + mant % 7u) << 7) | ((mant >> 8) & 0x7fu));
        }
    }
}

static size_t esize(int dtype) { return dtype == 0 ? 4 : 2; }

static void one_problem(void) {
    const int dtype = below(3);
    const int Hkv = 1 + below(2), G = 1 << below(3), Hq = Hkv * G;
    const int Ds[3] = {8, 16, 64}, Bs[3] = {1, 4, 16};
    const int D = Ds[below(3)], B = Bs[below(3)];
    const int S = 1 + below(5), max_blocks = 1 + below(6);
    const int N = S * max_blocks + below(4);
    const size_t es = esize(dtype), row = (size_t)D * es, blk = (size_t)Hkv * B * row;
    int32_t *tables = malloc(sizeof(int32_t) * S * max_blocks), *lens = malloc(sizeof(int32_t) * S);
    int32_t *perm = malloc(sizeof(int32_t) * N);
    for (int i = 0; i < N; ++i) perm[i] = i;
    for (int i = N - 1; i > 0; --i) {
        const int j = below(i + 1), t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
    for (int s = 0; s < S; ++s) {
        lens[s] = below(max_blocks * B + 1);
        const int used = (lens[s] + B - 1) / B;
        for (int j = 0; j < max_blocks; ++j) tables[s * max_blocks + j] = j < used ? perm[s * max_blocks + j] : -1;
    }
    void *kc = malloc(blk * N), *vc = malloc(blk * N), *q = malloc((size_t)S * Hq * row);
    fill(kc, (size_t)N * Hkv * B * D, dtype);
    fill(vc, (size_t)N * Hkv * B * D, dtype);
    fill(q, (size_t)S * Hq * D, dtype);
    const double scale = 1.0 / sqrt((double)D);
    double *o1 = malloc(sizeof(double) * S * Hq * D), *o2 = malloc(sizeof(double) * S * Hq * D);
    CHECK(pa_oracle_decode(S, Hq, Hkv, D, B, N, max_blocks, dtype, q, kc, vc, tables, lens, scale, o1) == 0,
          "decode refused");
    const int psize = B * (1 + below(3));
    CHECK(pa_oracle_decode_partitioned(S, Hq, Hkv, D, B, N, max_blocks, dtype, q, kc, vc, tables, lens, scale,
                                       psize, o2) == 0, "partitioned decode refused");
    for (int i = 0; i < S * Hq * D; ++i)
        CHECK(fabs(o1[i] - o2[i]) <= 1e-9 * (1.0 + fabs(o1[i])), "partitioned %g vs plain %g", o2[i], o1[i]);
    for (int s = 0; s < S; ++s)
        if (lens[s] == 0)
            for (int i = 0; i < Hq * D; ++i) CHECK(o1[(size_t)s * Hq * D + i] == 0.0, "empty context not zero");

    /* chunk attention: up to 3 queries per sequence; the last one is a decode */
    int32_t *qs = malloc(sizeof(int32_t) * (S + 1));
    qs[0] = 0;
    for (int s = 0; s < S; ++s) {
        const int n = lens[s] < 3 ? lens[s] : below(4);
        qs[s + 1] = qs[s] + (n <= lens[s] ? n : lens[s]);
    }
    const int T = qs[S];
    void *qc = malloc((size_t)(T > 0 ? T : 1) * Hq * row);
    fill(qc, (size_t)T * Hq * D, dtype);
    double *oc = malloc(sizeof(double) * (T > 0 ? T : 1) * Hq * D);
    CHECK(pa_oracle_chunk_attention(S, Hq, Hkv, D, B, N, max_blocks, dtype, qc, kc, vc, tables, lens, qs, T, scale,
                                    oc) == 0, "chunk attention refused");
    for (int s = 0; s < S; ++s) {
        if (qs[s + 1] == qs[s]) continue;
        const int t = qs[s + 1] - 1; /* its position is lens[s] - 1: the whole context */
        double *od = malloc(sizeof(double) * Hq * D);
        CHECK(pa_oracle_decode(1, Hq, Hkv, D, B, N, max_blocks, dtype, (const char *)qc + (size_t)t * Hq * row, kc,
                               vc, tables + (size_t)s * max_blocks, lens + s, scale, od) == 0, "decode refused");
        for (int i = 0; i < Hq * D; ++i)
            CHECK(fabs(od[i] - oc[(size_t)t * Hq * D + i]) <= 1e-12 * (1.0 + fabs(od[i])), "last chunk query");
        free(od);
    }
    /* bad inputs are refused */
    const int32_t saved = lens[0];
    lens[0] = max_blocks * B + 1;
    CHECK(pa_oracle_decode(S, Hq, Hkv, D, B, N, max_blocks, dtype, q, kc, vc, tables, lens, scale, o1) == -1,
          "overlong context accepted");
    lens[0] = saved;
    if (T > 0) {
        qs[S] = T + 1;
        CHECK(pa_oracle_chunk_attention(S, Hq, Hkv, D, B, N, max_blocks, dtype, qc, kc, vc, tables, lens, qs, T,
                                        scale, oc) == -1, "bad query range accepted");
        qs[S] = T;
    }

    /* slots, KV write */
    const int Tw = 1 + below(4);
    int64_t *slots = malloc(sizeof(int64_t) * Tw);
    for (int t = 0; t < Tw; ++t) {
        const int s = below(S);
        if (lens[s] == 0 || below(4) == 0) {
            slots[t] = -1;
            continue;
        }
        CHECK(pa_oracle_slot(tables + (size_t)s * max_blocks, B, below(lens[s]), &slots[t]) == 0, "slot");
    }
    for (int t = 0; t < Tw; ++t) /* later writes win: keep the first of equal slots only */
        for (int u = 0; u < t; ++u)
            if (slots[u] >= 0 && slots[u] == slots[t]) slots[t] = -1;
    void *kn = malloc((size_t)Tw * Hkv * row), *vn = malloc((size_t)Tw * Hkv * row);
    fill(kn, (size_t)Tw * Hkv * D, dtype);
    fill(vn, (size_t)Tw * Hkv * D, dtype);
    void *kc0 = malloc(blk * N);
    memcpy(kc0, kc, blk * N);
    CHECK(pa_oracle_write_kv(Tw, Hkv, D, B, N, dtype, kn, vn, slots, kc, vc) == 0, "write refused");
    for (int t = 0; t < Tw; ++t)
        for (int h = 0; h < Hkv; ++h) {
            if (slots[t] < 0) continue;
            const int64_t b = slots[t] / B, o = slots[t] % B;
            CHECK(memcmp((const char *)kc + (size_t)b * blk + ((size_t)h * B + o) * row,
                         (const char *)kn + ((size_t)t * Hkv + h) * row, row) == 0, "written key row");
        }
    /* rows no slot names are untouched */
    for (int b = 0; b < N; ++b)
        for (int h = 0; h < Hkv; ++h)
            for (int o = 0; o < B; ++o) {
                int named = 0;
                for (int t = 0; t < Tw; ++t) named |= slots[t] == (int64_t)b * B + o;
                if (named) continue;
                const size_t at = (size_t)b * blk + ((size_t)h * B + o) * row;
                CHECK(memcmp((const char *)kc + at, (const char *)kc0 + at, row) == 0, "unnamed row changed");
            }

    /* block copy and swap */
    if (N >= 2) {
        const int64_t pair[2] = {perm[0], perm[1]};
        CHECK(pa_oracle_copy_blocks(Hkv, D, B, N, dtype, kc, vc, pair, 1) == 0, "copy refused");
        CHECK(memcmp((const char *)kc + (size_t)pair[0] * blk, (const char *)kc + (size_t)pair[1] * blk, blk) == 0,
              "copied block");
        const int hn = 2;
        void *hk = calloc(hn, blk), *hv = calloc(hn, blk);
        const int64_t out_pair[2] = {perm[0], 1};
        CHECK(pa_oracle_swap_blocks(Hkv, D, B, dtype, kc, vc, N, hk, hv, hn, out_pair, 1) == 0, "swap refused");
        CHECK(memcmp((const char *)hk + blk, (const char *)kc + (size_t)perm[0] * blk, blk) == 0, "swapped block");
        free(hk);
        free(hv);
    }
    free(tables), free(lens), free(perm), free(kc), free(vc), free(q), free(o1), free(o2), free(qs), free(qc);
    free(oc), free(slots), free(kn), free(vn), free(kc0);
}

int main(int argc, char **argv) {
    rng_state = (argc > 1 ? strtoull(argv[1], NULL, 10) : 1) * 0x9E3779B97F4A7C15ull + 1;
    const long problems = argc > 2 ? strtol(argv[2], NULL, 10) : 200;
    for (long i = 0; i < problems && failures == 0; ++i) one_problem();
    printf("%ld problems, %d failures\n", problems, failures);
    return failures == 0 ? 0 : 1;
}
