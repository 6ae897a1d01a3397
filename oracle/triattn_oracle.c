/*
 * triattn_oracle.c -- plain fp64 CPU definition of the masked, biased
 * triangle-attention forward and of its packed (varlen) block-sparse form.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header or table with the CUDA
 * library.
 *
 * What it computes (cuEquivariance "triangle_attention" API page, formula):
 *   x_k = s * (Q_q . K_k) + B_qk    if key k is valid (M_k = 1)
 *   x_k = -1e9                      otherwise (the logit is replaced, not offset)
 *   O_q = sum_k softmax_k(x) V_k,   lse = log sum_k exp(x_k),   max = max_k x_k
 * Every stored input is widened exactly to double; s is the float scale the
 * caller passed, widened to double.  No tiling, no skipping, no reordering:
 * one query row at a time over all keys, in index order.
 *
 * Validity of key k for row (b,n):
 *   no mask        -> every key valid;
 *   dense mask     -> mask[b,n,0,0,k] != 0 (the page: "cast to bool");
 *   kv_lengths     -> k < clamp(kv_lengths[b,n], 0, K) (the page: prefix mask,
 *                     values above K clamped to K; negative values read as 0).
 *
 * Varlen form (Transformer Engine fused_attn.h: NVTE_NOT_INTERLEAVED layout,
 * cu_seqlens; tensorplay BlockMask: kv_num_blocks / kv_indices with optional
 * full_kv_* lists).  For sequence i and head h, local q < Lq and k < Lk:
 *   - the block-level mask is rebuilt with the BlockMask page's reconstruction
 *     loop (set semantics, entries past the count ignored, out-of-range block
 *     indices ignored);
 *   - a block from the full list is valid everywhere; a block from the partial
 *     list is valid where mask_mod holds, with local indices: causal k <= q;
 *     sliding window q - W < k <= q (the query and the W - 1 keys before it);
 *     prefix LM k <= q or k < P (P: the sequence's prefix length);
 *   - keys outside every listed block get -1e9, as in the triangle formula;
 *   - with no lists at all every block is partial.
 * Keys k >= Lk do not exist and take no part.  An optional post-scale bias
 * (Transformer Engine fused_attn.h, NVTE_POST_SCALE_BIAS), shaped
 * (H, max_seqlen_q, max_seqlen_k) and indexed by local positions, is added to
 * the logit of every valid key: x = s * (Q . K) + bias[h, q, k].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2 };
enum { OR_MASK_NONE = 0, OR_MASK_CAUSAL = 1, OR_MASK_SLIDING_WINDOW = 2, OR_MASK_PREFIX_LM = 3 };

#define OR_MASKED (-1.0e9)

/* IEEE-754 binary16 -> double, exact (sign, 5-bit exponent bias 15, 10-bit fraction). */
static double or_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 1024), e - 25);   /* (1024 + m) * 2^(e-25) */
    return sign ? -v : v;
}

/* bfloat16 -> double, exact: the upper half of a binary32. */
static double or_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double or_load(const void* p, int dt, size_t i) {
    switch (dt) {
    case OR_F32: return (double)((const float*)p)[i];
    case OR_F16: return or_half_to_double(((const uint16_t*)p)[i]);
    default:     return or_bf16_to_double(((const uint16_t*)p)[i]);
    }
}

/* Exposed so the tests can pin the widening against numpy / torch. */
double oracle_widen(const void* p, int dt, long long i) { return or_load(p, dt, (size_t)i); }

/*
 * Softmax-weighted sum for one query row, given its logits x[0..nk).
 * out[d] = sum_k exp(x_k - m) v[k][d] / sum_k exp(x_k - m); *lse = m + log(l); *mx = m.
 * v rows are at v + (v_off + k * v_stride) elements, d contiguous.
 */
static void or_softmax_row(const double* x, int nk, const void* v, int dt, size_t v_off,
                           size_t v_stride, int D, double* out, double* lse, double* mx,
                           double* w) {
    double m = -INFINITY;
    for (int k = 0; k < nk; ++k)
        if (x[k] > m) m = x[k];
    double l = 0.0;
    for (int k = 0; k < nk; ++k) {
        w[k] = exp(x[k] - m);
        l += w[k];
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int k = 0; k < nk; ++k) acc += w[k] * or_load(v, dt, v_off + (size_t)k * v_stride + d);
        out[d] = acc / l;
    }
    *lse = m + log(l);
    *mx = m;
}

/*
 * Triangle form.  Computes the rows listed in rows[0..nrows) (flat index of
 * (b,n,h,q) in the (B,N,H,Q) grid), or every row when rows == NULL (then
 * nrows is ignored).  out is (nrows or B*N*H*Q, D); lse, mx are per row.
 * mask (u8, (B,N,K)) and kv_len (int32, (B,N)) are each optional, not both.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_tri_fwd(const void* q, const void* k, const void* v, int dt,
                   const void* bias, int bias_dt,
                   const uint8_t* mask, const int32_t* kv_len,
                   int B, int N, int H, int Q, int K, int D, double scale,
                   const long long* rows, long long nrows,
                   double* out, double* lse, double* mx, int nthreads) {
    if (mask && kv_len) return -1;
    if (B <= 0 || N <= 0 || H <= 0 || Q <= 0 || K <= 0 || D <= 0) return -1;
    long long total = rows ? nrows : (long long)B * N * H * Q;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
#pragma omp parallel
    {
        double* x = (double*)malloc(sizeof(double) * (size_t)K);
        double* w = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(dynamic, 16)
        for (long long r = 0; r < total; ++r) {
            long long flat = rows ? rows[r] : r;
            int qi = (int)(flat % Q);
            long long t = flat / Q;
            int h = (int)(t % H);
            t /= H;
            int n = (int)(t % N);
            int b = (int)(t / N);
            size_t q_off = (size_t)flat * D;
            size_t kv_base = ((((size_t)b * N + n) * H + h) * (size_t)K) * D;
            size_t bias_off = (((size_t)b * H + h) * (size_t)Q + qi) * (size_t)K;
            int len = K;
            if (kv_len) {
                int L = kv_len[(size_t)b * N + n];
                len = L < 0 ? 0 : (L > K ? K : L);
            }
            for (int kk = 0; kk < K; ++kk) {
                int valid;
                if (mask) valid = mask[((size_t)b * N + n) * K + kk] != 0;
                else valid = kk < len;
                if (!valid) {
                    x[kk] = OR_MASKED;
                    continue;
                }
                double dot = 0.0;
                for (int d = 0; d < D; ++d)
                    dot += or_load(q, dt, q_off + d) * or_load(k, dt, kv_base + (size_t)kk * D + d);
                x[kk] = scale * dot + or_load(bias, bias_dt, bias_off + kk);
            }
            or_softmax_row(x, K, v, dt, kv_base, (size_t)D, D, out + (size_t)r * D, lse + r, mx + r, w);
        }
        free(x);
        free(w);
    }
    return 0;
}

/*
 * Row count of leading valid keys of a dense (B*N, K) u8 mask, and whether the
 * row is a prefix mask (no valid key after the first masked one).  This is the
 * reading of the page's mask_to_kv_lengths helper used by the tests.
 */
void oracle_mask_to_kv_lengths(const uint8_t* mask, long long rows, int K, int32_t* kv_len,
                               uint8_t* is_prefix) {
    for (long long r = 0; r < rows; ++r) {
        int L = 0;
        while (L < K && mask[r * K + L]) ++L;
        int prefix = 1;
        for (int kk = L; kk < K; ++kk)
            if (mask[r * K + kk]) prefix = 0;
        kv_len[r] = L;
        if (is_prefix) is_prefix[r] = (uint8_t)prefix;
    }
}

/* The mask_mod predicate for local query qi and key kk of a partial block. */
static int or_mask_mod(int mask_mod, int qi, int kk, int window, int prefix) {
    switch (mask_mod) {
    case OR_MASK_CAUSAL: return kk <= qi;
    case OR_MASK_SLIDING_WINDOW: return kk <= qi && qi - kk < window;
    case OR_MASK_PREFIX_LM: return kk <= qi || kk < prefix;
    default: return 1;
    }
}

/*
 * Varlen form.  q/out (total_q, H, D); k/v (total_k, H, D); lse/mx (H, total_q).
 * kv_num (S, mask_heads, MQ), kv_idx (S, mask_heads, MQ, MK); full_* the same or NULL.
 * kv_num == NULL: every block is partial.  window: the sliding window's width
 * (mask_mod 2); prefix_len (S,) or NULL, then prefix_all for every sequence
 * (mask_mod 3).  bias (H, max_q, max_k) of bias_dt, or NULL.  Returns 0 or -1.
 */
int oracle_varlen_fwd(const void* q, const void* k, const void* v, int dt,
                      const int32_t* cu_q, const int32_t* cu_k, int num_seqs, int H, int D,
                      double scale,
                      const int32_t* kv_num, const int32_t* kv_idx,
                      const int32_t* full_num, const int32_t* full_idx,
                      int mask_heads, int MQ, int MK, int block, int mask_mod,
                      int window, const int32_t* prefix_len, int prefix_all,
                      const void* bias, int bias_dt, int max_q, int max_k,
                      double* out, double* lse, double* mx, int nthreads) {
    if (num_seqs <= 0 || H <= 0 || D <= 0 || block <= 0) return -1;
    if (mask_mod == OR_MASK_SLIDING_WINDOW && window <= 0) return -1;
    if ((full_num == NULL) != (full_idx == NULL)) return -1;
    long long total_q = cu_q[num_seqs];
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    long long units = (long long)num_seqs * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long u = 0; u < units; ++u) {
        int s = (int)(u / H), h = (int)(u % H);
        int q0 = cu_q[s], Lq = cu_q[s + 1] - cu_q[s];
        int k0 = cu_k[s], Lk = cu_k[s + 1] - cu_k[s];
        if (Lq <= 0) continue;
        int nbq = (Lq + block - 1) / block, nbk = (Lk + block - 1) / block;
        int hm = mask_heads == 1 ? 0 : h;
        /* Block states: 0 unlisted, 1 partial (mask_mod), 2 full. */
        unsigned char* state = (unsigned char*)calloc((size_t)nbq * (nbk > 0 ? nbk : 1), 1);
        for (int qb = 0; qb < nbq; ++qb) {
            if (!kv_num) {
                for (int kb = 0; kb < nbk; ++kb) state[(size_t)qb * nbk + kb] = 1;
                continue;
            }
            if (qb >= MQ) continue;
            size_t row = ((size_t)s * mask_heads + hm) * MQ + qb;
            int cnt = kv_num[row];
            for (int t = 0; t < cnt && t < MK; ++t) {
                int kb = kv_idx[row * MK + t];
                if (kb >= 0 && kb < nbk && state[(size_t)qb * nbk + kb] < 1) state[(size_t)qb * nbk + kb] = 1;
            }
            if (full_num) {
                int fc = full_num[row];
                for (int t = 0; t < fc && t < MK; ++t) {
                    int kb = full_idx[row * MK + t];
                    if (kb >= 0 && kb < nbk) state[(size_t)qb * nbk + kb] = 2;
                }
            }
        }
        double* x = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        double* w = (double*)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        int prefix = prefix_len ? prefix_len[s] : prefix_all;
        for (int qi = 0; qi < Lq; ++qi) {
            size_t q_off = (((size_t)(q0 + qi)) * H + h) * D;
            for (int kk = 0; kk < Lk; ++kk) {
                int st = state[(size_t)(qi / block) * nbk + kk / block];
                int valid = st == 2 || (st == 1 && or_mask_mod(mask_mod, qi, kk, window, prefix));
                if (!valid) {
                    x[kk] = OR_MASKED;
                    continue;
                }
                size_t k_off = (((size_t)(k0 + kk)) * H + h) * D;
                double dot = 0.0;
                for (int d = 0; d < D; ++d) dot += or_load(q, dt, q_off + d) * or_load(k, dt, k_off + d);
                x[kk] = scale * dot;
                if (bias) x[kk] += or_load(bias, bias_dt, ((size_t)h * max_q + qi) * (size_t)max_k + kk);
            }
            size_t row_out = (size_t)(q0 + qi);
            size_t a = (size_t)h * total_q + row_out;
            if (Lk <= 0) {
                /* Empty key sequence: the sum over no keys is 0, so lse = max = -inf
                 * and O is set to 0 (the pages leave this case undefined). */
                for (int d = 0; d < D; ++d) out[(row_out * H + h) * D + d] = 0.0;
                lse[a] = -INFINITY;
                mx[a] = -INFINITY;
                continue;
            }
            or_softmax_row(x, Lk, v, dt, ((size_t)k0 * H + h) * D, (size_t)H * D, D,
                           out + (row_out * H + h) * D, lse + a, mx + a, w);
        }
        free(x);
        free(w);
        free(state);
    }
    return 0;
}
