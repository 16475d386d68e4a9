/*
 * pa_oracle.c -- fp64 CPU oracle for single-query paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the CPU-baseline leg of
 * the bench use it.  It shares no code, header or constant with the CUDA
 * library, and it is deliberately slow and plain.
 *
 * Sources (web page, then the section of it that a function follows):
 *   [PA-V2]  "paged_attention_v2_triton.py -- Triton PagedAttention V2 for
 *            BI-V100": the module docstring (Phase 2 combine formula), the
 *            phase-1 kernel `_paged_attn_v2_partition_kernel` (paged K/V
 *            gather, scores, partition bounds, unused-partition sentinels) and
 *            the phase-2 kernel `_paged_attn_v2_reduce_kernel`.
 *   [FA-MTL] "flash_attention.metal -- Flash Attention Metal Shaders",
 *            `flash_attention_forward`, final write (inv_l = 0 when l = 0).
 *
 * Layouts (all row-major, contiguous), from the phase-1 kernel's argument
 * comments in [PA-V2]:
 *   query        [S, H, D]                      16-bit floats (fp16 or bf16)
 *   key_cache    [num_blocks, KH, D/x, BS, x]   x = 16 / sizeof(elem) = 8
 *   value_cache  [num_blocks, KH, D, BS]
 *   block_tables [S, MB] int32, seq_lens [S] int32
 *
 * Parity pins: every exported function is checked against closed forms,
 * brute force, a textbook dense softmax and invariants by the CPU tests.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DTYPE_FP16 0
#define ORACLE_DTYPE_BF16 1

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* zero / subnormal */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1.f) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double: bfloat16 is the top half of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double to_double(uint16_t v, int dtype) {
    return dtype == ORACLE_DTYPE_BF16 ? bf16_to_double(v) : fp16_to_double(v);
}

/* Element (token slot o of physical block b, kv head kh, dim d) of the
 * x-packed key cache: key_cache[b, kh, d / x, o, d % x]  ([PA-V2], phase-1
 * kernel, "Paged K gather"). */
static size_t key_index(long b, int kh, int d, int o, int KH, int D, int BS) {
    const int x = 8;
    return ((((size_t)b * KH + kh) * (D / x) + d / x) * BS + o) * x + d % x;
}

/* value_cache[b, kh, d, o]  ([PA-V2], phase-1 kernel, "Paged V gather"). */
static size_t value_index(long b, int kh, int d, int o, int KH, int D, int BS) {
    return (((size_t)b * KH + kh) * D + d) * BS + o;
}

int pa_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Scores z_t = scale * sum_d q_d * K_t[d] for tokens [t0, t1) of sequence s,
 * query head h, with K_t gathered through the block table: physical block
 * block_tables[s, t / BS], slot t % BS ([PA-V2], phase-1 kernel).  The query
 * head reads kv head h / (H / KH) ([PA-V2], "GQA: map query head -> KV
 * head"). */
static void scores_fp64(double* z, int t0, int t1, int s, int h,
                        const uint16_t* q, const uint16_t* kc, const int32_t* bt,
                        double scale, int H, int KH, int D, int BS, int MB, int dtype) {
    const int kh = h / (H / KH);
    const uint16_t* qv = q + ((size_t)s * H + h) * D;
    for (int t = t0; t < t1; ++t) {
        long b = bt[(size_t)s * MB + t / BS];
        int o = t % BS;
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += to_double(qv[d], dtype) * to_double(kc[key_index(b, kh, d, o, KH, D, BS)], dtype);
        z[t - t0] = scale * acc;
    }
}

/* out[s, h, :] = softmax(z) . V over all seq_lens[s] tokens, no partitioning.
 * This is the result the two-phase method reaches ([PA-V2] module docstring:
 * the partition maxima, rescaled sums and weighted partial outputs combine to
 * the full softmax).  Two passes: max, then exp-sum and weighted V.
 * seq_lens[s] == 0 gives zeros, following [FA-MTL]'s inv_l = 0 when l = 0.
 * Returns 0, or -1 on a bad argument or allocation failure. */
int pa_oracle_decode(double* out, const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                     const int32_t* bt, const int32_t* lens, double scale,
                     int S, int H, int KH, int D, int BS, int MB, int dtype, int nthreads) {
    if (S < 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 8 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long sh = 0; sh < (long)S * H; ++sh) {
        int s = (int)(sh / H), h = (int)(sh % H);
        int L = lens[s];
        double* o_sh = out + (size_t)sh * D;
        for (int d = 0; d < D; ++d) o_sh[d] = 0.0;
        if (L <= 0) continue;
        if (L > MB * BS) { bad = 1; continue; }
        double* z = (double*)malloc(sizeof(double) * (size_t)L);
        if (!z) { bad = 1; continue; }
        scores_fp64(z, 0, L, s, h, q, kc, bt, scale, H, KH, D, BS, MB, dtype);
        double mu = -INFINITY;
        for (int t = 0; t < L; ++t) if (z[t] > mu) mu = z[t];
        double den = 0.0;
        for (int t = 0; t < L; ++t) { z[t] = exp(z[t] - mu); den += z[t]; }
        const int kh = h / (H / KH);
        for (int t = 0; t < L; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            for (int d = 0; d < D; ++d)
                o_sh[d] += z[t] * to_double(vc[value_index(b, kh, d, o, KH, D, BS)], dtype);
        }
        for (int d = 0; d < D; ++d) o_sh[d] /= den;
        free(z);
    }
    return bad ? -1 : 0;
}

/* Phase-1 partition statistics, from their definitions ([PA-V2],
 * `_paged_attn_v2_partition_kernel`): partition p of sequence s covers tokens
 * [p*P, min((p+1)*P, L)).  For a used partition
 *     m_p = max z_t,  l_p = sum exp(z_t - m_p),  o_p = sum exp(z_t - m_p) V_t / l_p
 * (o_p normalised, as the kernel's accumulator update keeps it).  A partition
 * with p*P >= L is unused: m_p = -inf, l_p = 0 ("write sentinel values"), and
 * o_p is written as zeros here (the page leaves it untouched).
 * Arrays m, l are [S, H, Pmax]; o is [S, H, Pmax, D]. */
int pa_oracle_partitions(double* m, double* l, double* o,
                         const uint16_t* q, const uint16_t* kc, const uint16_t* vc,
                         const int32_t* bt, const int32_t* lens, double scale,
                         int S, int H, int KH, int D, int BS, int MB, int P, int Pmax,
                         int dtype, int nthreads) {
    if (S < 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 8 || BS <= 0 || MB < 0 ||
        P <= 0 || Pmax < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long shp = 0; shp < (long)S * H * Pmax; ++shp) {
        int p = (int)(shp % Pmax);
        long sh = shp / Pmax;
        int s = (int)(sh / H), h = (int)(sh % H);
        int L = lens[s];
        double* o_p = o + (size_t)shp * D;
        for (int d = 0; d < D; ++d) o_p[d] = 0.0;
        long start = (long)p * P;
        if (L > MB * BS || (L > 0 && (L + P - 1) / P > Pmax)) { bad = 1; continue; }
        if (start >= L) { m[shp] = -INFINITY; l[shp] = 0.0; continue; }
        int t0 = (int)start;
        int t1 = (int)(start + P < L ? start + P : L);
        double* z = (double*)malloc(sizeof(double) * (size_t)(t1 - t0));
        if (!z) { bad = 1; continue; }
        scores_fp64(z, t0, t1, s, h, q, kc, bt, scale, H, KH, D, BS, MB, dtype);
        double mp = -INFINITY;
        for (int i = 0; i < t1 - t0; ++i) if (z[i] > mp) mp = z[i];
        double lp = 0.0;
        for (int i = 0; i < t1 - t0; ++i) { z[i] = exp(z[i] - mp); lp += z[i]; }
        const int kh = h / (H / KH);
        for (int t = t0; t < t1; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int ot = t % BS;
            for (int d = 0; d < D; ++d)
                o_p[d] += z[t - t0] * to_double(vc[value_index(b, kh, d, ot, KH, D, BS)], dtype);
        }
        for (int d = 0; d < D; ++d) o_p[d] /= lp;
        m[shp] = mp;
        l[shp] = lp;
        free(z);
    }
    return bad ? -1 : 0;
}

/* Phase 2, cross-partition log-sum-exp combine ([PA-V2] module docstring and
 * `_paged_attn_v2_reduce_kernel`), over the NP = ceil(L / P) used partitions:
 *     M = max_p m_p,  total = sum_p exp(m_p - M) l_p,
 *     out = sum_p (exp(m_p - M) l_p / total) o_p.
 * All NP partitions are combined (the page caps them at 1024; this does not).
 * L == 0 gives zeros (the [FA-MTL] inv_l = 0 convention). */
int pa_oracle_combine(double* out, const double* m, const double* l, const double* o,
                      const int32_t* lens, int S, int H, int D, int P, int Pmax) {
    if (S < 0 || H <= 0 || D <= 0 || P <= 0 || Pmax < 0) return -1;
    int bad = 0;
    for (long sh = 0; sh < (long)S * H; ++sh) {
        int s = (int)(sh / H);
        int L = lens[s];
        double* out_sh = out + (size_t)sh * D;
        for (int d = 0; d < D; ++d) out_sh[d] = 0.0;
        if (L <= 0) continue;
        int np = (L + P - 1) / P;
        if (np > Pmax) { bad = 1; continue; }
        const double* m_sh = m + (size_t)sh * Pmax;
        const double* l_sh = l + (size_t)sh * Pmax;
        double M = -INFINITY;
        for (int p = 0; p < np; ++p) if (m_sh[p] > M) M = m_sh[p];
        double total = 0.0;
        for (int p = 0; p < np; ++p) total += exp(m_sh[p] - M) * l_sh[p];
        for (int p = 0; p < np; ++p) {
            double w = exp(m_sh[p] - M) * l_sh[p] / total;
            const double* o_p = o + ((size_t)sh * Pmax + p) * D;
            for (int d = 0; d < D; ++d) out_sh[d] += w * o_p[d];
        }
    }
    return bad ? -1 : 0;
}

/* Log-sum-exp of the scaled scores of each (s, h) over its seq_lens[s] tokens,
 * in natural-log units:  lse = mu + log(sum_t exp(z_t - mu)),  mu = max_t z_t.
 * This is the value the forward kernel of [FA-MTL] stores beside its output
 * (its running maximum plus the log of its running sum, "log-sum-exp for
 * backward pass"); outputs computed over disjoint token sets merge with it.
 * seq_lens[s] == 0 gives -inf (the running maximum never leaves -inf there).
 * lse is [S, H].  Returns 0, or -1 on a bad argument or allocation failure. */
int pa_oracle_lse(double* lse, const uint16_t* q, const uint16_t* kc, const int32_t* bt,
                  const int32_t* lens, double scale, int S, int H, int KH, int D, int BS, int MB,
                  int dtype, int nthreads) {
    if (S < 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 8 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long sh = 0; sh < (long)S * H; ++sh) {
        int s = (int)(sh / H), h = (int)(sh % H);
        int L = lens[s];
        lse[sh] = -INFINITY;
        if (L <= 0) continue;
        if (L > MB * BS) { bad = 1; continue; }
        double* z = (double*)malloc(sizeof(double) * (size_t)L);
        if (!z) { bad = 1; continue; }
        scores_fp64(z, 0, L, s, h, q, kc, bt, scale, H, KH, D, BS, MB, dtype);
        double mu = -INFINITY;
        for (int t = 0; t < L; ++t) if (z[t] > mu) mu = z[t];
        double sum = 0.0;
        for (int t = 0; t < L; ++t) sum += exp(z[t] - mu);
        lse[sh] = mu + log(sum);
        free(z);
    }
    return bad ? -1 : 0;
}

/* The same log-sum-exp from phase-1 states, by the combine of [PA-V2] (module
 * docstring): M = max_p m_p, total = sum_p exp(m_p - M) l_p, lse = M + log(total),
 * over the ceil(L / P) used partitions; L == 0 gives -inf.  lse is [S, H]. */
int pa_oracle_combine_lse(double* lse, const double* m, const double* l, const int32_t* lens,
                          int S, int H, int P, int Pmax) {
    if (S < 0 || H <= 0 || P <= 0 || Pmax < 0) return -1;
    int bad = 0;
    for (long sh = 0; sh < (long)S * H; ++sh) {
        int s = (int)(sh / H);
        int L = lens[s];
        lse[sh] = -INFINITY;
        if (L <= 0) continue;
        int np = (L + P - 1) / P;
        if (np > Pmax) { bad = 1; continue; }
        const double* m_sh = m + (size_t)sh * Pmax;
        const double* l_sh = l + (size_t)sh * Pmax;
        double M = -INFINITY;
        for (int p = 0; p < np; ++p) if (m_sh[p] > M) M = m_sh[p];
        double total = 0.0;
        for (int p = 0; p < np; ++p) total += exp(m_sh[p] - M) * l_sh[p];
        lse[sh] = M + log(total);
    }
    return bad ? -1 : 0;
}

/* Multi-query decode (several new tokens per sequence, e.g. speculative
 * verification): query[s, i, h, :] for i < q_len is the query of the i-th of
 * the sequence's last q_len tokens, which sits at position L - q_len + i of its
 * seq_lens[s] = L cached tokens and attends causally to positions
 * 0 .. L - q_len + i.  This is the decode of [PA-V2] widened from one query
 * row (its module docstring: "For decode (BLOCK_M=1), the Q tile is just one
 * vector") to q_len rows with the causal rule of the prefix-prefill kernel its
 * gather comes from.  out and lse are [S, q_len, H, D] and [S, q_len, H]; lse
 * (may be NULL) is as in pa_oracle_lse.  L < q_len is an error (the new
 * tokens must be in the cache). */
int pa_oracle_decode_mq(double* out, double* lse, const uint16_t* q, const uint16_t* kc,
                        const uint16_t* vc, const int32_t* bt, const int32_t* lens, double scale,
                        int S, int q_len, int H, int KH, int D, int BS, int MB, int dtype,
                        int nthreads) {
    if (S < 0 || q_len <= 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 8 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
    const long rows = (long)S * q_len * H;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long r = 0; r < rows; ++r) {
        const int h = (int)(r % H);
        const int i = (int)((r / H) % q_len);
        const int s = (int)(r / ((long)H * q_len));
        double* o_r = out + (size_t)r * D;
        for (int d = 0; d < D; ++d) o_r[d] = 0.0;
        if (lse) lse[r] = -INFINITY;
        const int L = lens[s];
        if (L < q_len || L > MB * BS) { bad = 1; continue; }
        const int visible = L - q_len + i + 1;          /* positions 0 .. L - q_len + i */
        double* z = (double*)malloc(sizeof(double) * (size_t)visible);
        if (!z) { bad = 1; continue; }
        /* Scores of this query row: its vector is query[s, i, h, :], i.e. row
         * s * q_len + i of a [S * q_len, H, D] array, against sequence s's keys. */
        const int kh = h / (H / KH);
        const uint16_t* qv = q + ((size_t)(s * q_len + i) * H + h) * D;
        for (int t = 0; t < visible; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += to_double(qv[d], dtype) * to_double(kc[key_index(b, kh, d, o, KH, D, BS)], dtype);
            z[t] = scale * acc;
        }
        double mu = -INFINITY;
        for (int t = 0; t < visible; ++t) if (z[t] > mu) mu = z[t];
        double den = 0.0;
        for (int t = 0; t < visible; ++t) { z[t] = exp(z[t] - mu); den += z[t]; }
        for (int t = 0; t < visible; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            for (int d = 0; d < D; ++d)
                o_r[d] += z[t] * to_double(vc[value_index(b, kh, d, o, KH, D, BS)], dtype);
        }
        for (int d = 0; d < D; ++d) o_r[d] /= den;
        if (lse) lse[r] = mu + log(den);
        free(z);
    }
    return bad ? -1 : 0;
}

/* 8-bit float E4M3 (the "e4m3fn" variant: no infinities) -> double, from the
 * format's definition: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits;
 * exponent 0 is subnormal (fraction * 2^-9); exponent 15 with fraction 7 is
 * NaN; every other code is finite, the largest being 1.75 * 2^8 = 448. */
static double e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int expo = (b >> 3) & 0xf;
    int frac = b & 0x7;
    double v;
    if (expo == 15 && frac == 7) {
        v = NAN;
    } else if (expo == 0) {
        v = ldexp((double)frac, -9);                 /* 0.fff * 2^(1-7) */
    } else {
        v = ldexp((double)(8 + frac), expo - 10);    /* 1.fff * 2^(e-7) */
    }
    return sign ? -v : v;
}

int pa_oracle_e4m3_decode(double* out, const uint8_t* codes, int n) {
    if (n < 0) return -1;
    for (int i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
    return 0;
}

/* key_cache[b, kh, d / x, o, d % x] with x = 16 / sizeof(element) = 16 for
 * one-byte elements (the launcher of [PA-V2] takes x from the cache's last
 * dimension). */
static size_t key_index_x16(long b, int kh, int d, int o, int KH, int D, int BS) {
    const int x = 16;
    return ((((size_t)b * KH + kh) * (D / x) + d / x) * BS + o) * x + d % x;
}

/* Decode over an fp8 (E4M3) KV cache with per-tensor scales: the launcher of
 * [PA-V2] takes kv_cache_dtype, k_scale and v_scale (and ignores them); the
 * plain reading is that the cached bytes are E4M3 codes and the real keys and
 * values are k_scale * K and v_scale * V.  query and the result are 16-bit as
 * before (qdtype); key_cache [NB, KH, D/16, BS, 16] and value_cache
 * [NB, KH, D, BS] hold the codes.  out [S, H, D], lse [S, H] (may be NULL);
 * seq_lens[s] == 0 gives zeros and lse -inf. */
int pa_oracle_decode_fp8kv(double* out, double* lse, const uint16_t* q, const uint8_t* kc,
                           const uint8_t* vc, const int32_t* bt, const int32_t* lens, double scale,
                           double k_scale, double v_scale, int S, int H, int KH, int D, int BS,
                           int MB, int qdtype, int nthreads) {
    if (S < 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 16 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long sh = 0; sh < (long)S * H; ++sh) {
        int s = (int)(sh / H), h = (int)(sh % H);
        int L = lens[s];
        double* o_sh = out + (size_t)sh * D;
        for (int d = 0; d < D; ++d) o_sh[d] = 0.0;
        if (lse) lse[sh] = -INFINITY;
        if (L <= 0) continue;
        if (L > MB * BS) { bad = 1; continue; }
        double* z = (double*)malloc(sizeof(double) * (size_t)L);
        if (!z) { bad = 1; continue; }
        const int kh = h / (H / KH);
        const uint16_t* qv = q + (size_t)sh * D;
        for (int t = 0; t < L; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += to_double(qv[d], qdtype) *
                       (k_scale * e4m3_to_double(kc[key_index_x16(b, kh, d, o, KH, D, BS)]));
            z[t] = scale * acc;
        }
        double mu = -INFINITY;
        for (int t = 0; t < L; ++t) if (z[t] > mu) mu = z[t];
        double den = 0.0;
        for (int t = 0; t < L; ++t) { z[t] = exp(z[t] - mu); den += z[t]; }
        for (int t = 0; t < L; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            for (int d = 0; d < D; ++d)
                o_sh[d] += z[t] * (v_scale * e4m3_to_double(vc[value_index(b, kh, d, o, KH, D, BS)]));
        }
        for (int d = 0; d < D; ++d) o_sh[d] /= den;
        if (lse) lse[sh] = mu + log(den);
        free(z);
    }
    return bad ? -1 : 0;
}

/* Multi-query decode over an fp8 (E4M3) KV cache: the q_len causal rows of
 * pa_oracle_decode_mq (row i of a sequence of L tokens sees positions
 * 0 .. L - q_len + i) with the keys and values of pa_oracle_decode_fp8kv
 * (k_scale * E4M3(K), v_scale * E4M3(V), key layout x = 16).  query, out
 * [S, q_len, H, D], lse [S, q_len, H] (may be NULL); L < q_len is an error. */
int pa_oracle_decode_mq_fp8kv(double* out, double* lse, const uint16_t* q, const uint8_t* kc,
                              const uint8_t* vc, const int32_t* bt, const int32_t* lens,
                              double scale, double k_scale, double v_scale, int S, int q_len,
                              int H, int KH, int D, int BS, int MB, int qdtype, int nthreads) {
    if (S < 0 || q_len <= 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 16 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
    const long rows = (long)S * q_len * H;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long r = 0; r < rows; ++r) {
        const int h = (int)(r % H);
        const int i = (int)((r / H) % q_len);
        const int s = (int)(r / ((long)H * q_len));
        double* o_r = out + (size_t)r * D;
        for (int d = 0; d < D; ++d) o_r[d] = 0.0;
        if (lse) lse[r] = -INFINITY;
        const int L = lens[s];
        if (L < q_len || L > MB * BS) { bad = 1; continue; }
        const int seen = L - q_len + i + 1;             /* positions 0 .. L - q_len + i */
        double* z = (double*)malloc(sizeof(double) * (size_t)seen);
        if (!z) { bad = 1; continue; }
        const int kh = h / (H / KH);
        const uint16_t* qrow = q + ((size_t)(s * q_len + i) * H + h) * D;
        for (int t = 0; t < seen; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += to_double(qrow[d], qdtype) *
                       (k_scale * e4m3_to_double(kc[key_index_x16(b, kh, d, o, KH, D, BS)]));
            z[t] = scale * acc;
        }
        double mu = -INFINITY;
        for (int t = 0; t < seen; ++t) if (z[t] > mu) mu = z[t];
        double den = 0.0;
        for (int t = 0; t < seen; ++t) { z[t] = exp(z[t] - mu); den += z[t]; }
        for (int t = 0; t < seen; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            for (int d = 0; d < D; ++d)
                o_r[d] += z[t] * (v_scale * e4m3_to_double(vc[value_index(b, kh, d, o, KH, D, BS)]));
        }
        for (int d = 0; d < D; ++d) o_r[d] /= den;
        if (lse) lse[r] = mu + log(den);
        free(z);
    }
    return bad ? -1 : 0;
}

/* key_cache[b, kh, d / x, o, d % x] with x = 16 / sizeof(element) = 4 for
 * four-byte (fp32) elements ([PA-V2]: the launcher's x = 16 / sizeof(dtype)). */
static size_t key_index_x4(long b, int kh, int d, int o, int KH, int D, int BS) {
    const int x = 4;
    return ((((size_t)b * KH + kh) * (D / x) + d / x) * BS + o) * x + d % x;
}

/* Decode with fp32 query, caches and result ([PA-V2] takes the element type
 * from the query's dtype and sizes the key layout's x from it): the plain
 * definition softmax(scale * q . K^T) . V over all seq_lens[s] tokens, in
 * fp64 from the fp32 values.  key_cache [NB, KH, D/4, BS, 4], value_cache
 * [NB, KH, D, BS]; out [S, H, D], lse [S, H] (may be NULL); seq_lens[s] == 0
 * gives zeros and lse -inf. */
int pa_oracle_decode_fp32(double* out, double* lse, const float* q, const float* kc, const float* vc,
                          const int32_t* bt, const int32_t* lens, double scale, int S, int H, int KH,
                          int D, int BS, int MB, int nthreads) {
    if (S < 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 4 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long sh = 0; sh < (long)S * H; ++sh) {
        int s = (int)(sh / H), h = (int)(sh % H);
        int L = lens[s];
        double* o_sh = out + (size_t)sh * D;
        for (int d = 0; d < D; ++d) o_sh[d] = 0.0;
        if (lse) lse[sh] = -INFINITY;
        if (L <= 0) continue;
        if (L > MB * BS) { bad = 1; continue; }
        double* z = (double*)malloc(sizeof(double) * (size_t)L);
        if (!z) { bad = 1; continue; }
        const int kh = h / (H / KH);
        const float* qv = q + (size_t)sh * D;
        for (int t = 0; t < L; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)qv[d] * (double)kc[key_index_x4(b, kh, d, o, KH, D, BS)];
            z[t] = scale * acc;
        }
        double mu = -INFINITY;
        for (int t = 0; t < L; ++t) if (z[t] > mu) mu = z[t];
        double den = 0.0;
        for (int t = 0; t < L; ++t) { z[t] = exp(z[t] - mu); den += z[t]; }
        for (int t = 0; t < L; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            for (int d = 0; d < D; ++d)
                o_sh[d] += z[t] * (double)vc[value_index(b, kh, d, o, KH, D, BS)];
        }
        for (int d = 0; d < D; ++d) o_sh[d] /= den;
        if (lse) lse[sh] = mu + log(den);
        free(z);
    }
    return bad ? -1 : 0;
}

/* Multi-query decode with fp32 query, caches and result: the q_len causal
 * rows of pa_oracle_decode_mq (row i of a sequence of L tokens sees positions
 * 0 .. L - q_len + i) over the fp32 caches of pa_oracle_decode_fp32 (key
 * layout x = 4).  query, out [S, q_len, H, D], lse [S, q_len, H] (may be
 * NULL); L < q_len is an error. */
int pa_oracle_decode_mq_fp32(double* out, double* lse, const float* q, const float* kc, const float* vc,
                             const int32_t* bt, const int32_t* lens, double scale, int S, int q_len,
                             int H, int KH, int D, int BS, int MB, int nthreads) {
    if (S < 0 || q_len <= 0 || H <= 0 || KH <= 0 || H % KH || D <= 0 || D % 4 || BS <= 0 || MB < 0)
        return -1;
    int bad = 0;
    if (nthreads <= 0) nthreads = pa_oracle_max_threads();
    const long rows = (long)S * q_len * H;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(| : bad)
    for (long r = 0; r < rows; ++r) {
        const int h = (int)(r % H);
        const int i = (int)((r / H) % q_len);
        const int s = (int)(r / ((long)H * q_len));
        double* o_r = out + (size_t)r * D;
        for (int d = 0; d < D; ++d) o_r[d] = 0.0;
        if (lse) lse[r] = -INFINITY;
        const int L = lens[s];
        if (L < q_len || L > MB * BS) { bad = 1; continue; }
        const int upto = L - q_len + i + 1;             /* positions 0 .. L - q_len + i */
        double* z = (double*)malloc(sizeof(double) * (size_t)upto);
        if (!z) { bad = 1; continue; }
        const int kh = h / (H / KH);
        const float* qr = q + ((size_t)(s * q_len + i) * H + h) * D;
        for (int t = 0; t < upto; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += (double)qr[d] * (double)kc[key_index_x4(b, kh, d, o, KH, D, BS)];
            z[t] = scale * acc;
        }
        double mu = -INFINITY;
        for (int t = 0; t < upto; ++t) if (z[t] > mu) mu = z[t];
        double den = 0.0;
        for (int t = 0; t < upto; ++t) { z[t] = exp(z[t] - mu); den += z[t]; }
        for (int t = 0; t < upto; ++t) {
            long b = bt[(size_t)s * MB + t / BS];
            int o = t % BS;
            for (int d = 0; d < D; ++d)
                o_r[d] += z[t] * (double)vc[value_index(b, kh, d, o, KH, D, BS)];
        }
        for (int d = 0; d < D; ++d) o_r[d] /= den;
        if (lse) lse[r] = mu + log(den);
        free(z);
    }
    return bad ? -1 : 0;
}
