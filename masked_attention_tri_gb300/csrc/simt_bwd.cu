// simt_bwd.cu -- backward of the triangle-attention forward on CUDA cores
// (exact fp32 arithmetic for every input dtype).
//
// The forward (cuEquivariance triangle_attention page) is
//     x = s Q.K + bias at valid keys, -1e9 at masked keys;  P = softmax_k(x);  O = P V
// and its context is saved for backward.  For a loss with dL/dO = dO the chain
// rule gives, per (b, n, h) slab and query row q:
//     dV[k]  = sum_q P[q,k] dO[q]
//     dP     = dO[q] . V[k]
//     dx     = P (dP - sum_k' P[q,k'] dP[q,k'])   at valid keys, 0 at masked keys
//     dQ[q]  = s sum_k dx K[k],   dK[k] = s sum_q dx Q[q]
//     dBias[b,0,h,q,k] = sum_n dx[b,n,h,q,k]
// P is recomputed from the forward's saved lse: P = exp(x - lse).  A row whose
// keys are all masked has every logit at -1e9 and lse = -1e9 + ln K, which is
// -1e9 once stored in fp32; such a row (lse at or below -1e9 + 64, while any
// valid logit lies above -1e9 + 100) takes its exact weights 1/K.
//
// The same kernels serve packed sequences (q / k / v / O / dO (total, H, D),
// lse / delta (H, total_q), the BlockMask lists and mask_mod deciding each
// (query, key) pair, an optional (H, max_seqlen_q, max_seqlen_k) bias whose
// gradient sums over the sequences); there the per-row sums come from O.
//
// Three kernels:
//   delta   one CTA per (slab, 32 query rows): delta[q] = sum_k P dP over every key
//           (the exact definition); zeroes the fp32 dQ accumulator rows and
//           (grid-stride) the dBias accumulator.  When the caller passes the
//           forward's O, delta[q] = dO[q] . O[q] instead (sum_k P dP = dO . O),
//           one pass over two (Q, D) tensors.
//   main    one CTA per (slab, 32 keys), looping over the query tiles: dK and dV
//           of its keys in registers, dQ and dBias added atomically (fp32) into
//           the caller's workspace.  16-bit inputs with D % 16 == 0, D <= 64 and
//           K % 8 == 0 take the tensor-core form of this step (tc_bwd.cu).
//   finish  dQ and dBias accumulators converted to the output dtypes.
// Layout of one CTA: 4 warps; in the score steps warp w owns query rows
// 8w..8w+7 and lane j key j; in the accumulation steps warp w owns keys (dK, dV)
// or rows (dQ) 8w..8w+7 and lane l the columns l + 32c, c < DPL (D <= 32 DPL).

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace triattn {
namespace {

constexpr int kT = 32;      // query rows / keys per tile
constexpr int kBW = 4;      // warps per CTA
constexpr int kBR = kT / kBW;  // rows (or keys) per warp
constexpr float kMaskedLogit = -1.0e9f;

template <typename T>
__device__ __forceinline__ float ld_f(const T* p, long long i);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p, long long i) { return p[i]; }
template <>
__device__ __forceinline__ float ld_f<__half>(const __half* p, long long i) { return __half2float(p[i]); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
    return __bfloat162float(p[i]);
}
template <typename T>
__device__ __forceinline__ T to_t(float x);
template <>
__device__ __forceinline__ float to_t<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half to_t<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 to_t<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Softmax weight of an existing key from its logit x and the row's stored lse.
__device__ __forceinline__ float weight(float x, float lse, float inv_k) {
    return lse <= kMaskedLogit + 64.f ? inv_k : expf(x - lse);
}

// Key `key` of (b, n) row bn takes part (kv_lengths prefix, dense mask or every key).
__device__ __forceinline__ bool key_valid(const BwdParams& p, long long bn, int key) {
    if (p.kv_len) {
        int L = p.kv_len[bn];
        L = L < 0 ? 0 : (L > p.K ? p.K : L);
        return key < L;
    }
    if (p.mask) return p.mask[bn * p.K + key] != 0;
    return true;
}

// Loads rows [r0, r0 + 32) of a (rows x D) slab matrix into smem [32][D + 1] as fp32 (zeros past `rows`).
// Rows `rs` elements apart (D for the triangle form, H * D for packed sequences).
template <typename T>
__device__ __forceinline__ void load_tile(float* dst, const T* src, long long base, int r0, int rows, int D,
                                          long long rs) {
    const int Dp1 = D + 1;
    for (int e = threadIdx.x; e < kT * D; e += blockDim.x) {
        const int r = e / D, d = e - r * D;
        dst[r * Dp1 + d] = (r0 + r < rows) ? ld_f(src, base + (long long)(r0 + r) * rs + d) : 0.f;
    }
}
template <typename T>
__device__ __forceinline__ void load_tile(float* dst, const T* src, long long base, int r0, int rows, int D) {
    load_tile(dst, src, base, r0, rows, D, (long long)D);
}

// Packed sequences: the BlockMask status of q block qb and kv block kb (tensorplay
// BlockMask page, Details 1-2): 2 = full (mask_mod skipped), 1 = partial (mask_mod
// applies; also every block when no lists are given), 0 = not visited (masked).
__device__ __forceinline__ int block_status(const BwdParams& p, int seq, int h, int qb, int kb) {
    if (!p.kv_num) return 1;
    if (qb >= p.MQ) return 0;
    const int hm = p.mask_heads == 1 ? 0 : h;
    const long long row = ((long long)seq * p.mask_heads + hm) * p.MQ + qb;
    if (p.full_num) {
        const int n = min(max(p.full_num[row], 0), p.MK);
        for (int t = 0; t < n; ++t)
            if (p.full_idx[row * p.MK + t] == kb) return 2;
    }
    const int n = min(max(p.kv_num[row], 0), p.MK);
    for (int t = 0; t < n; ++t)
        if (p.kv_idx[row * p.MK + t] == kb) return 1;
    return 0;
}
// mask_mod on a partial block, local indices: causal k <= q; sliding window
// q - window < k <= q; prefix LM k <= q or k < prefix.
__device__ __forceinline__ bool mod_keep(int mod, int q, int k, int window, int prefix) {
    switch (mod) {
    case TA_MASK_CAUSAL: return k <= q;
    case TA_MASK_SLIDING_WINDOW: return k <= q && k > q - window;
    case TA_MASK_PREFIX_LM: return k <= q || k < prefix;
    default: return true;
    }
}

// Scores of the tile pair: for warp rows i (query q0 + 8w + i) and lane key j
// (key k0 + lane) returns x (logit, -1e9 if masked) in x[i] and dP in dp[i].
__device__ __forceinline__ void scores(const float* Qs, const float* Ks, const float* dOs, const float* Vs, int D,
                                       int warp, int lane, float (&qk)[kBR], float (&dp)[kBR]) {
    const int Dp1 = D + 1;
#pragma unroll
    for (int i = 0; i < kBR; ++i) qk[i] = dp[i] = 0.f;
    for (int d = 0; d < D; ++d) {
        const float kd = Ks[lane * Dp1 + d], vd = Vs[lane * Dp1 + d];
#pragma unroll
        for (int i = 0; i < kBR; ++i) {
            qk[i] = fmaf(Qs[(warp * kBR + i) * Dp1 + d], kd, qk[i]);
            dp[i] = fmaf(dOs[(warp * kBR + i) * Dp1 + d], vd, dp[i]);
        }
    }
}

template <typename T, typename BT>
__global__ void __launch_bounds__(kBW * 32) bwd_delta_kernel(const BwdParams p) {
    extern __shared__ float sm[];
    const int D = p.D, Dp1 = D + 1;
    float* Qs = sm;
    float* dOs = Qs + kT * Dp1;
    float* Ks = dOs + kT * Dp1;
    float* Vs = Ks + kT * Dp1;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nqt = (p.Q + kT - 1) / kT;
    const long long unit = blockIdx.x / nqt;  // (b*N + n)*H + h
    const int q0 = (int)(blockIdx.x - unit * nqt) * kT;
    const int h = (int)(unit % p.H);
    const long long bn = unit / p.H;
    const int b = (int)(bn / p.N);

    // dBias accumulator zeroed grid-stride (the main kernel runs after this one).
    if (p.dbias_acc) {
        const long long tot = (long long)p.B * p.H * p.Q * p.K;
        for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < tot; e += (long long)gridDim.x * blockDim.x)
            p.dbias_acc[e] = 0.f;
    }
    const long long qbase = unit * p.Q * D, kbase = unit * (long long)p.K * D;
    for (int e = threadIdx.x; e < kT * D; e += blockDim.x) {
        const int r = e / D;
        if (q0 + r < p.Q) p.dq_acc[qbase + (long long)(q0 + r) * D + (e - r * D)] = 0.f;
    }
    load_tile(Qs, static_cast<const T*>(p.q), qbase, q0, p.Q, D);
    load_tile(dOs, static_cast<const T*>(p.d_out), qbase, q0, p.Q, D);
    float lse[kBR], acc[kBR];
#pragma unroll
    for (int i = 0; i < kBR; ++i) {
        const int q = q0 + warp * kBR + i;
        lse[i] = q < p.Q ? p.lse[unit * p.Q + q] : 0.f;
        acc[i] = 0.f;
    }
    const BT* bias = static_cast<const BT*>(p.bias);
    const long long brow = ((long long)b * p.H + h) * p.Q;
    for (int k0 = 0; k0 < p.K; k0 += kT) {
        __syncthreads();
        load_tile(Ks, static_cast<const T*>(p.k), kbase, k0, p.K, D);
        load_tile(Vs, static_cast<const T*>(p.v), kbase, k0, p.K, D);
        __syncthreads();
        float qk[kBR], dp[kBR];
        scores(Qs, Ks, dOs, Vs, D, warp, lane, qk, dp);
        const int key = k0 + lane;
        const bool exists = key < p.K;
        const bool valid = exists && key_valid(p, bn, key);
#pragma unroll
        for (int i = 0; i < kBR; ++i) {
            const int q = q0 + warp * kBR + i;
            if (!exists || q >= p.Q) continue;
            const float x = valid ? fmaf(p.scale, qk[i], ld_f(bias, (brow + q) * p.K + key)) : kMaskedLogit;
            acc[i] = fmaf(weight(x, lse[i], 1.f / (float)p.K), dp[i], acc[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < kBR; ++i) {
        float v = acc[i];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        const int q = q0 + warp * kBR + i;
        if (lane == 0 && q < p.Q) p.delta[unit * p.Q + q] = v;
    }
}

// delta[row] = sum_d dO[row, d] O[row, d] from the forward's stored O (eight
// lanes per row, 16-byte loads); zeroes the row's fp32 dQ accumulator and,
// grid-stride, the dBias accumulator.
template <typename T>
__global__ void __launch_bounds__(256) bwd_delta_out_kernel(const BwdParams p) {
    constexpr int kE = 16 / (int)sizeof(T);  // elements per 16-byte chunk
    const long long rows = p.delta_rows;  // (b,n,h,q) rows, or (token, head) rows of packed sequences
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) / 8;
    const int g = threadIdx.x % 8;
    if (p.dbias_acc) {
        for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < p.dbias_elems;
             e += (long long)gridDim.x * blockDim.x)
            p.dbias_acc[e] = 0.f;
    }
    float acc = 0.f;
    if (row < rows) {
        const T* o = static_cast<const T*>(p.out) + row * p.D;
        const T* d = static_cast<const T*>(p.d_out) + row * p.D;
        for (int c = g; c * kE < p.D; c += 8) {
            const uint4 ov = reinterpret_cast<const uint4*>(o)[c];
            const uint4 dv = reinterpret_cast<const uint4*>(d)[c];
            const T* oe = reinterpret_cast<const T*>(&ov);
            const T* de = reinterpret_cast<const T*>(&dv);
#pragma unroll
            for (int e = 0; e < kE; ++e) acc = fmaf(ld_f(oe, e), ld_f(de, e), acc);
        }
        float4* dq = reinterpret_cast<float4*>(p.dq_acc + row * p.D);
        for (int c = g; c * 4 < p.D; c += 8) dq[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int o = 4; o; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (g == 0 && row < rows) p.delta[p.varlen ? (row % p.H) * p.total_q + row / p.H : row] = acc;
}

template <typename T, typename BT, int DPL, bool VARLEN>
__global__ void __launch_bounds__(kBW * 32) bwd_main_kernel(const BwdParams p) {
    extern __shared__ float sm[];
    const int D = p.D, Dp1 = D + 1;
    float* Ks = sm;
    float* Vs = Ks + kT * Dp1;
    float* Qs = Vs + kT * Dp1;
    float* dOs = Qs + kT * Dp1;
    float* Ps = dOs + kT * Dp1;       // [32 rows][33]
    float* dSs = Ps + kT * (kT + 1);  // [32 rows][33]
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // The unit's rows: queries q at qbase + q * rs, keys k at kbase + k * rs, lse / delta at
    // lrow0 + q, bias / dBias at brow0 + q * bstride + k.
    long long qbase, kbase, rs, lrow0, brow0, bstride, bn = 0;
    int Lq, Lk, k0, h, seq = 0, prefix = 0;
    if constexpr (!VARLEN) {
        const int nkt = (p.K + kT - 1) / kT;
        const long long unit = blockIdx.x / nkt;
        k0 = (int)(blockIdx.x - unit * nkt) * kT;
        h = (int)(unit % p.H);
        bn = unit / p.H;
        const int b = (int)(bn / p.N);
        qbase = unit * p.Q * D;
        kbase = unit * (long long)p.K * D;
        rs = D;
        Lq = p.Q;
        Lk = p.K;
        lrow0 = unit * p.Q;
        brow0 = ((long long)b * p.H + h) * p.Q * p.K;
        bstride = p.K;
    } else {
        const int nkt = (p.max_k + kT - 1) / kT;
        seq = blockIdx.x / (p.H * nkt);
        h = (blockIdx.x / nkt) % p.H;
        k0 = (blockIdx.x % nkt) * kT;
        const int cq0 = p.cu_q[seq], cq1 = p.cu_q[seq + 1], ck0 = p.cu_k[seq], ck1 = p.cu_k[seq + 1];
        Lq = cq1 - cq0;
        Lk = ck1 - ck0;
        if (Lq > p.max_q || Lk > p.max_k || Lq < 0 || Lk < 0 || cq0 < 0 || ck0 < 0 || cq1 > p.total_q ||
            ck1 > p.total_k) {
            if (threadIdx.x == 0 && k0 == 0 && h == 0) atomicCAS(p.status, 0, kStatusDevice);
            return;
        }
        rs = (long long)p.H * D;
        qbase = (long long)cq0 * rs + (long long)h * D;
        kbase = (long long)ck0 * rs + (long long)h * D;
        lrow0 = (long long)h * p.total_q + cq0;
        brow0 = (long long)h * p.max_q * p.max_k;
        bstride = p.max_k;
        prefix = p.prefix_len ? p.prefix_len[seq] : p.prefix_all;
    }
    if (k0 >= Lk) return;

    load_tile(Ks, static_cast<const T*>(p.k), kbase, k0, Lk, D, rs);
    load_tile(Vs, static_cast<const T*>(p.v), kbase, k0, Lk, D, rs);
    const int key = k0 + lane;  // this lane's key in the score steps
    const bool exists = key < Lk;
    const bool key_ok = !VARLEN ? (exists && key_valid(p, bn, key)) : exists;
    const float inv_k = 1.f / (float)Lk;
    float dk[kBR][DPL], dv[kBR][DPL];
#pragma unroll
    for (int j = 0; j < kBR; ++j)
#pragma unroll
        for (int c = 0; c < DPL; ++c) dk[j][c] = dv[j][c] = 0.f;
    const BT* bias = static_cast<const BT*>(p.bias);

    for (int q0 = 0; q0 < Lq; q0 += kT) {
        __syncthreads();  // the previous tile's Qs, dOs, Ps, dSs are no longer read
        load_tile(Qs, static_cast<const T*>(p.q), qbase, q0, Lq, D, rs);
        load_tile(dOs, static_cast<const T*>(p.d_out), qbase, q0, Lq, D, rs);
        const int bstat = VARLEN ? block_status(p, seq, h, q0 / 128, k0 / 128) : 1;
        __syncthreads();
        float qk[kBR], dp[kBR];
        scores(Qs, Ks, dOs, Vs, D, warp, lane, qk, dp);
#pragma unroll
        for (int i = 0; i < kBR; ++i) {
            const int r = warp * kBR + i, q = q0 + r;
            float P = 0.f, dS = 0.f;
            if (exists && q < Lq) {
                const long long row = lrow0 + q;
                bool valid = key_ok;
                if constexpr (VARLEN)
                    valid = bstat == 2 || (bstat == 1 && mod_keep(p.mask_mod, q, key, p.window, prefix));
                const long long bi = brow0 + (long long)q * bstride + key;
                const float bv = bias ? ld_f(bias, bi) : 0.f;
                const float x = valid ? fmaf(p.scale, qk[i], bv) : kMaskedLogit;
                P = weight(x, p.lse[row], inv_k);
                if (valid) {
                    dS = P * (dp[i] - p.delta[row]);
                    if (p.dbias_acc) atomicAdd(p.dbias_acc + bi, dS);
                }
            }
            Ps[r * (kT + 1) + lane] = P;
            dSs[r * (kT + 1) + lane] = dS;
        }
        __syncthreads();
        // dV[j] += sum_i P[i,j] dO[i],  dK[j] += sum_i dS[i,j] Q[i]   (keys j = 8 warp + jj)
        for (int i = 0; i < kT; ++i) {
            float qv[DPL], ov[DPL];
#pragma unroll
            for (int c = 0; c < DPL; ++c) {
                const int d = lane + 32 * c;
                qv[c] = d < D ? Qs[i * Dp1 + d] : 0.f;
                ov[c] = d < D ? dOs[i * Dp1 + d] : 0.f;
            }
#pragma unroll
            for (int jj = 0; jj < kBR; ++jj) {
                const float pv = Ps[i * (kT + 1) + warp * kBR + jj], sv = dSs[i * (kT + 1) + warp * kBR + jj];
#pragma unroll
                for (int c = 0; c < DPL; ++c) {
                    dv[jj][c] = fmaf(pv, ov[c], dv[jj][c]);
                    dk[jj][c] = fmaf(sv, qv[c], dk[jj][c]);
                }
            }
        }
        // dQ[i] += s sum_j dS[i,j] K[j]   (rows i = 8 warp + ii), added to the fp32 accumulator
        float dq[kBR][DPL];
#pragma unroll
        for (int ii = 0; ii < kBR; ++ii)
#pragma unroll
            for (int c = 0; c < DPL; ++c) dq[ii][c] = 0.f;
        for (int j = 0; j < kT; ++j) {
            float kv[DPL];
#pragma unroll
            for (int c = 0; c < DPL; ++c) {
                const int d = lane + 32 * c;
                kv[c] = d < D ? Ks[j * Dp1 + d] : 0.f;
            }
#pragma unroll
            for (int ii = 0; ii < kBR; ++ii) {
                const float sv = dSs[(warp * kBR + ii) * (kT + 1) + j];
#pragma unroll
                for (int c = 0; c < DPL; ++c) dq[ii][c] = fmaf(sv, kv[c], dq[ii][c]);
            }
        }
#pragma unroll
        for (int ii = 0; ii < kBR; ++ii) {
            const int q = q0 + warp * kBR + ii;
            if (q >= Lq) continue;
#pragma unroll
            for (int c = 0; c < DPL; ++c) {
                const int d = lane + 32 * c;
                if (d < D && dq[ii][c] != 0.f) atomicAdd(p.dq_acc + qbase + (long long)q * rs + d, p.scale * dq[ii][c]);
            }
        }
    }
    T* dkp = static_cast<T*>(p.dk);
    T* dvp = static_cast<T*>(p.dv);
#pragma unroll
    for (int jj = 0; jj < kBR; ++jj) {
        const int kk = k0 + warp * kBR + jj;
        if (kk >= Lk) continue;
#pragma unroll
        for (int c = 0; c < DPL; ++c) {
            const int d = lane + 32 * c;
            if (d < D) {
                dkp[kbase + (long long)kk * rs + d] = to_t<T>(p.scale * dk[jj][c]);
                dvp[kbase + (long long)kk * rs + d] = to_t<T>(dv[jj][c]);
            }
        }
    }
}

__device__ __forceinline__ uint32_t pack_pair(__half, float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_pair(__nv_bfloat16, float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// dst[e] = src[e] in T, e < n, grid-stride.  16-bit outputs with 16-byte aligned
// buffers: eight elements per step (two 16-byte loads, one 16-byte store).
template <typename T>
__device__ __forceinline__ void convert_range(const float* src, void* dstv, long long n, long long tid,
                                              long long stride) {
    T* dst = static_cast<T*>(dstv);
    long long done = 0;
    if constexpr (sizeof(T) == 2) {
        if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0) {
            const long long n8 = n / 8;
            const float4* s4 = reinterpret_cast<const float4*>(src);
            uint4* d8 = reinterpret_cast<uint4*>(dst);
            for (long long i = tid; i < n8; i += stride) {
                const float4 a = s4[2 * i], b = s4[2 * i + 1];
                d8[i] = make_uint4(pack_pair(T(), a.x, a.y), pack_pair(T(), a.z, a.w), pack_pair(T(), b.x, b.y),
                                   pack_pair(T(), b.z, b.w));
            }
            done = n8 * 8;
        }
    }
    for (long long e = done + tid; e < n; e += stride) dst[e] = to_t<T>(src[e]);
}

template <typename T, typename BT>
__global__ void bwd_finish_kernel(const BwdParams p) {
    const long long stride = (long long)gridDim.x * blockDim.x;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    convert_range<T>(p.dq_acc, p.dq, p.dq_elems, tid, stride);
    if (p.dbias) convert_range<BT>(p.dbias_acc, p.dbias, p.dbias_elems, tid, stride);
}

template <typename T, typename BT>
cudaError_t launch_typed(const BwdParams& p, cudaStream_t stream) {
    const int D = p.D;
    const long long units = (long long)p.B * p.N * p.H;
    const size_t sm1 = sizeof(float) * 4 * kT * (size_t)(D + 1);
    const size_t sm2 = sm1 + sizeof(float) * 2 * kT * (kT + 1);
    auto k1 = bwd_delta_kernel<T, BT>;
    auto k2 = p.varlen ? (D <= 128 ? bwd_main_kernel<T, BT, 4, true> : bwd_main_kernel<T, BT, 8, true>)
                       : (D <= 128 ? bwd_main_kernel<T, BT, 4, false> : bwd_main_kernel<T, BT, 8, false>);
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm2)) != cudaSuccess) return e;
    const long long g1 = units * ((p.Q + kT - 1) / kT);
    const long long g2 = p.varlen ? (long long)p.num_seqs * p.H * ((p.max_k + kT - 1) / kT)
                                  : units * ((p.K + kT - 1) / kT);
    if (g1 > 0x7fffffffLL || g2 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (p.varlen && !p.out) return cudaErrorInvalidValue;  // packed sequences: the sums come from O
    if (p.out) {
        const long long gd = (p.delta_rows * 8 + 255) / 256;
        if (gd > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        bwd_delta_out_kernel<T><<<(unsigned)gd, 256, 0, stream>>>(p);
    } else {
        k1<<<(unsigned)g1, kBW * 32, sm1, stream>>>(p);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.tc_main) {
        if ((e = launch_tc_bwd_main(p, stream)) != cudaSuccess) return e;
    } else if (g2 > 0) {
        k2<<<(unsigned)g2, kBW * 32, sm2, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    bwd_finish_kernel<T, BT><<<1024, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_workspace_floats_n(long long dq_elems, long long dbias_elems, long long delta_rows) {
    auto up = [](size_t n) { return (n + 63) & ~(size_t)63; };  // 256-byte pieces
    return up((size_t)dq_elems) + up((size_t)dbias_elems) + up((size_t)delta_rows);
}

size_t bwd_workspace_floats(int B, int N, int H, int Q, int K, int D) {
    const long long units = (long long)B * N * H;
    return bwd_workspace_floats_n(units * Q * D, (long long)B * H * Q * K, units * Q);
}

cudaError_t launch_simt_bwd(const BwdParams& p, cudaStream_t stream) {
    switch (p.dtype) {
    case TA_F32: return launch_typed<float, float>(p, stream);
    case TA_F16: return p.bias_f32 ? launch_typed<__half, float>(p, stream) : launch_typed<__half, __half>(p, stream);
    default:
        return p.bias_f32 ? launch_typed<__nv_bfloat16, float>(p, stream)
                          : launch_typed<__nv_bfloat16, __nv_bfloat16>(p, stream);
    }
}

}  // namespace triattn
