// simt_fwd.cu -- CUDA-core forward for fp32 inputs (exact fp32 arithmetic, no TF32).
//
// Computes the cuEquivariance triangle_attention formula (and its packed,
// block-sparse form) with an online softmax: for each 32-key tile the running
// row max m and normaliser l are updated and the accumulator rescaled by
// exp(m_old - m_new).  A masked key's logit is replaced by -1e9; a key past
// the end of its sequence takes no part.  A row that sees no valid key has
// every logit equal to -1e9, so its result is the mean of V over all keys of
// its sequence; that case is computed directly.
//
// Layout: one CTA = 32 query rows of one (b,n,h) slab (triangle) or one
// (sequence, head) pair (varlen); 4 warps x 8 rows; each lane owns one key of
// the current tile for the logits and D/32 output columns for the accumulate
// (DPL = 4 columns per lane for D <= 128, 8 for D <= 256).  It also carries
// 16-bit inputs with D in (128, 256], which the tensor-core kernels do not take.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace triattn {
namespace {

constexpr int kQT = 32;
constexpr int kKT = 32;
constexpr int kWarps = 4;
constexpr int kRows = kQT / kWarps;  // rows per warp
constexpr float kMasked = -1.0e9f;

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Key validity modes of one tile.
enum { kKeyAll = 0, kKeyPrefix = 1, kKeyDense = 2, kKeyMod = 3 };

template <typename T, typename BT, int DPL>
struct SimtState {
    const AttnParams* p;
    float* Qs;
    float* Ks;
    float* Vs;
    float* Ps;  // this warp's [kRows][kKT]
    int D, Dp1, warp, lane;
    long long k_off, k_rs, v_off, v_rs;
    int Lk;
    long long bias_row0;  // element offset of the bias row of query q0 (key 0), -1 = none
    int bias_rs;
    int rows;             // query rows of this CTA that exist (Lq - q0, at most kQT)
    int q0;               // first query row of the CTA (local index)
    int prefix_len;
    int prefix_lm;        // packed form, mask_mod prefix LM: the sequence's prefix length
    const uint8_t* dense;
    float m[kRows], l[kRows], acc[kRows][DPL];
    bool seen[kRows];
};

// Process keys [key0, key0 + 32) ∩ [0, Lk) with the given validity mode.
template <typename T, typename BT, int DPL>
__device__ void simt_tile(SimtState<T, BT, DPL>& st, int key0, int mode) {
    const AttnParams& p = *st.p;
    const T* kp = static_cast<const T*>(p.k);
    const T* vp = static_cast<const T*>(p.v);
    const int D = st.D, Dp1 = st.Dp1;
    __syncthreads();
    for (int e = threadIdx.x; e < kKT * D; e += blockDim.x) {
        int j = e / D, d = e - j * D;
        int key = key0 + j;
        float kv = 0.f, vv = 0.f;
        if (key < st.Lk) {
            kv = to_f(kp[st.k_off + (long long)key * st.k_rs + d]);
            vv = to_f(vp[st.v_off + (long long)key * st.v_rs + d]);
        }
        st.Ks[j * Dp1 + d] = kv;
        st.Vs[j * D + d] = vv;
    }
    __syncthreads();

    const int key = key0 + st.lane;
    const bool exists = key < st.Lk;
    float s[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) s[i] = 0.f;
    for (int d = 0; d < D; ++d) {
        float kd = st.Ks[st.lane * Dp1 + d];
#pragma unroll
        for (int i = 0; i < kRows; ++i) s[i] = fmaf(st.Qs[(st.warp * kRows + i) * Dp1 + d], kd, s[i]);
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        const int qrow = st.q0 + st.warp * kRows + i;
        bool valid = exists;
        if (mode == kKeyPrefix) valid = valid && key < st.prefix_len;
        else if (mode == kKeyDense) valid = valid && st.dense[key] != 0;
        else if (mode == kKeyMod) {
            // BlockMask mask_mod on a partial block, local indices
            if (p.mask_mod == TA_MASK_CAUSAL) valid = valid && key <= qrow;
            else if (p.mask_mod == TA_MASK_SLIDING_WINDOW) valid = valid && key <= qrow && qrow - key < p.window;
            else if (p.mask_mod == TA_MASK_PREFIX_LM) valid = valid && (key <= qrow || key < st.prefix_lm);
        }
        float x;
        if (!exists) {
            x = -INFINITY;
        } else if (!valid) {
            x = kMasked;
        } else {
            float b = 0.f;
            // (rows past the end of the queries read no bias: they may lie past the buffer)
            if (st.bias_row0 >= 0 && st.warp * kRows + i < st.rows) {
                const BT* bp = static_cast<const BT*>(p.bias);
                b = to_f(bp[st.bias_row0 + (long long)(st.warp * kRows + i) * st.bias_rs + key]);
            }
            x = fmaf(s[i], p.scale, b);
        }
        st.seen[i] = st.seen[i] || (__ballot_sync(0xffffffffu, valid) != 0);
        float mt = warp_max(x);
        float mn = fmaxf(st.m[i], mt);
        float alpha = (st.m[i] == -INFINITY) ? 0.f : expf(st.m[i] - mn);
        float pr = (x == -INFINITY) ? 0.f : expf(x - mn);
        st.l[i] = st.l[i] * alpha + warp_sum(pr);
        st.m[i] = mn;
        st.Ps[i * kKT + st.lane] = pr;
#pragma unroll
        for (int j = 0; j < DPL; ++j) st.acc[i][j] *= alpha;
    }
    __syncwarp();
    for (int j = 0; j < kKT; ++j) {
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            int d = st.lane + 32 * c;
            if (d < D) {
                float vv = st.Vs[j * D + d];
#pragma unroll
                for (int i = 0; i < kRows; ++i) st.acc[i][c] = fmaf(st.Ps[i * kKT + j], vv, st.acc[i][c]);
            }
        }
    }
    __syncwarp();
}

template <typename T, typename BT, int DPL>
__global__ void __launch_bounds__(kWarps * 32) simt_fwd_kernel(const AttnParams p) {
    extern __shared__ float smem[];
    const int D = p.D, Dp1 = D + 1;
    SimtState<T, BT, DPL> st;
    st.p = &p;
    st.D = D;
    st.Dp1 = Dp1;
    st.warp = threadIdx.x / 32;
    st.lane = threadIdx.x % 32;
    st.Qs = smem;
    st.Ks = st.Qs + kQT * Dp1;
    st.Vs = st.Ks + kKT * Dp1;
    st.Ps = st.Vs + kKT * D + st.warp * kRows * kKT;

    const T* qp = static_cast<const T*>(p.q);
    long long q_off, q_rs, o_off, o_rs, lse_off;
    int Lq, qt;
    st.bias_row0 = -1;
    st.bias_rs = 0;
    st.prefix_len = 0;
    st.dense = nullptr;
    int seq = 0, h = 0;

    if (!p.varlen) {
        const int nqt = (p.Q + kQT - 1) / kQT;
        const long long u = blockIdx.x / nqt;
        qt = blockIdx.x % nqt;
        h = (int)(u % p.H);
        const long long bn = u / p.H;
        const int b = (int)(bn / p.N);
        const long long n = bn - (long long)b * p.N;
        q_off = b * p.qs[0] + n * p.qs[1] + h * p.qs[2];
        q_rs = p.qs[3];
        o_off = u * p.Q * (long long)D;
        o_rs = D;
        st.k_off = b * p.ks[0] + n * p.ks[1] + h * p.ks[2];
        st.k_rs = p.ks[3];
        st.v_off = b * p.vs[0] + n * p.vs[1] + h * p.vs[2];
        st.v_rs = p.vs[3];
        Lq = p.Q;
        st.Lk = p.K;
        st.bias_row0 = (((long long)b * p.H + h) * p.Q + (long long)qt * kQT) * p.K;
        st.bias_rs = p.K;
        lse_off = u * p.Q;
        if (p.kv_len) {
            int L = p.kv_len[bn];
            st.prefix_len = L < 0 ? 0 : (L > p.K ? p.K : L);
        }
        if (p.mask) st.dense = p.mask + bn * p.K;
    } else {
        const int nqt = (p.max_q + kQT - 1) / kQT;
        seq = blockIdx.x / (p.H * nqt);
        h = (blockIdx.x / nqt) % p.H;
        qt = blockIdx.x % nqt;
        const int cq0 = p.cu_q[seq], cq1 = p.cu_q[seq + 1];
        const int ck0 = p.cu_k[seq], ck1 = p.cu_k[seq + 1];
        Lq = cq1 - cq0;
        st.Lk = ck1 - ck0;
        if (Lq > p.max_q || st.Lk > p.max_k || Lq < 0 || st.Lk < 0 || cq0 < 0 || ck0 < 0 || cq1 > p.total_q ||
            ck1 > p.total_k) {
            if (threadIdx.x == 0 && qt == 0 && h == 0) atomicCAS(p.status, 0, kStatusDevice);
            return;
        }
        // Packed rows: q / k / v rows are q_rs / k_rs / v_rs elements apart, out rows H * D.
        q_off = (long long)cq0 * p.q_rs + (long long)h * D;
        q_rs = p.q_rs;
        o_off = (long long)cq0 * p.H * D + (long long)h * D;
        o_rs = (long long)p.H * D;
        st.k_off = (long long)ck0 * p.k_rs + (long long)h * D;
        st.k_rs = p.k_rs;
        st.v_off = (long long)ck0 * p.v_rs + (long long)h * D;
        st.v_rs = p.v_rs;
        lse_off = (long long)h * p.total_q + cq0;  // (H, total_q)
        st.prefix_lm = p.prefix_len ? p.prefix_len[seq] : p.prefix_all;
    }
    st.q0 = qt * kQT;
    if (st.q0 >= Lq) return;
    st.rows = Lq - st.q0;
    if (p.varlen && p.bias) {
        // packed form: post-scale bias (H, max_seqlen_q, max_seqlen_k) at local positions
        st.bias_row0 = ((long long)h * p.max_q + st.q0) * p.max_k;
        st.bias_rs = p.max_k;
    }

    for (int e = threadIdx.x; e < kQT * D; e += blockDim.x) {
        int r = e / D, d = e - r * D;
        int qrow = st.q0 + r;
        st.Qs[r * Dp1 + d] = qrow < Lq ? to_f(qp[q_off + (long long)qrow * q_rs + d]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        st.m[i] = -INFINITY;
        st.l[i] = 0.f;
        st.seen[i] = false;
#pragma unroll
        for (int c = 0; c < DPL; ++c) st.acc[i][c] = 0.f;
    }

    if (!p.varlen) {
        // kv_lengths: only tiles below the prefix length hold valid keys; with
        // length 0 no tile is visited and the all-masked path below applies.
        int mode = p.kv_len ? kKeyPrefix : (p.mask ? kKeyDense : kKeyAll);
        int kend = p.kv_len ? st.prefix_len : p.K;
        for (int key0 = 0; key0 < kend; key0 += kKT) simt_tile(st, key0, mode);
    } else {
        const int nbk = (st.Lk + 127) / 128;
        const int qb = st.q0 / 128;
        if (!p.kv_num) {
            for (int kb = 0; kb < nbk; ++kb)
                for (int t = 0; t < 4; ++t)
                    if (kb * 128 + t * kKT < st.Lk)
                        simt_tile(st, kb * 128 + t * kKT, p.mask_mod != TA_MASK_NONE ? kKeyMod : kKeyAll);
        } else if (qb < p.MQ) {
            const int hm = p.mask_heads == 1 ? 0 : h;
            const long long row = ((long long)seq * p.mask_heads + hm) * p.MQ + qb;
            if (p.full_num) {
                int cnt = min(p.full_num[row], p.MK);
                for (int t = 0; t < cnt; ++t) {
                    int kb = p.full_idx[row * p.MK + t];
                    if (kb < 0 || kb >= nbk) continue;
                    for (int s4 = 0; s4 < 4; ++s4)
                        if (kb * 128 + s4 * kKT < st.Lk) simt_tile(st, kb * 128 + s4 * kKT, kKeyAll);
                }
            }
            int cnt = min(p.kv_num[row], p.MK);
            for (int t = 0; t < cnt; ++t) {
                int kb = p.kv_idx[row * p.MK + t];
                if (kb < 0 || kb >= nbk) continue;
                for (int s4 = 0; s4 < 4; ++s4)
                    if (kb * 128 + s4 * kKT < st.Lk)
                        simt_tile(st, kb * 128 + s4 * kKT, p.mask_mod != TA_MASK_NONE ? kKeyMod : kKeyAll);
            }
        }
    }

    // Rows with no valid key: every logit is -1e9 -> uniform weights over all
    // keys of the sequence.  Their mean of V is shared by the warp's rows.
    bool any_unseen = false;
#pragma unroll
    for (int i = 0; i < kRows; ++i) any_unseen = any_unseen || !st.seen[i];
    float meanv[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) meanv[c] = 0.f;
    if (any_unseen && st.Lk > 0) {
        const T* vp = static_cast<const T*>(p.v);
        for (int key = 0; key < st.Lk; ++key) {
#pragma unroll
            for (int c = 0; c < DPL; ++c) {
                int d = st.lane + 32 * c;
                if (d < D) meanv[c] += to_f(vp[st.v_off + (long long)key * st.v_rs + d]);
            }
        }
#pragma unroll
        for (int c = 0; c < DPL; ++c) meanv[c] /= (float)st.Lk;
    }

    T* op = static_cast<T*>(p.out);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
        const int qrow = st.q0 + st.warp * kRows + i;
        if (qrow >= Lq) continue;
        float lse, mx;
        float o[DPL];
        if (st.Lk == 0) {
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[c] = 0.f;
            lse = -INFINITY;
            mx = -INFINITY;
        } else if (!st.seen[i]) {
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[c] = meanv[c];
            mx = kMasked;
            lse = kMasked + logf((float)st.Lk);
        } else {
            float inv = 1.f / st.l[i];
#pragma unroll
            for (int c = 0; c < DPL; ++c) o[c] = st.acc[i][c] * inv;
            mx = st.m[i];
            lse = st.m[i] + logf(st.l[i]);
        }
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            int d = st.lane + 32 * c;
            if (d < D) op[o_off + (long long)qrow * o_rs + d] = from_f<T>(o[c]);
        }
        if (st.lane == 0) {
            if (p.lse) p.lse[lse_off + qrow] = lse;
            if (p.mx) p.mx[lse_off + qrow] = mx;
        }
    }
}

template <typename T, typename BT>
cudaError_t launch_typed(const AttnParams& p, cudaStream_t stream) {
    const int D = p.D;
    size_t smem = sizeof(float) * ((size_t)kQT * (D + 1) + (size_t)kKT * (D + 1) + (size_t)kKT * D +
                                   (size_t)kWarps * kRows * kKT);
    auto kern = D <= 128 ? simt_fwd_kernel<T, BT, 4> : simt_fwd_kernel<T, BT, 8>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    long long grid;
    if (!p.varlen) grid = (long long)p.B * p.N * p.H * ((p.Q + kQT - 1) / kQT);
    else grid = (long long)p.num_seqs * p.H * ((p.max_q + kQT - 1) / kQT);
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kWarps * 32, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_fwd(const AttnParams& p, cudaStream_t stream) {
    switch (p.dtype) {
    case TA_F32: return launch_typed<float, float>(p, stream);
    case TA_F16: return p.bias_f32 ? launch_typed<__half, float>(p, stream) : launch_typed<__half, __half>(p, stream);
    default:
        return p.bias_f32 ? launch_typed<__nv_bfloat16, float>(p, stream)
                          : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, stream);
    }
}

}  // namespace triattn
