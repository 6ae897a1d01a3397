// host.cu -- the C ABI (include/triattn.h): argument checks, dispatch by
// dtype, and the device status word.
//
// Checks follow the cuEquivariance triangle_attention page (Parameters:
// "Pass either mask or kv_lengths, not both"; Notes 3-4 for the supported
// head dimensions and the K % 8 rule of the Blackwell kernels), the
// Transformer Engine fused_attn.h page (cu_seqlens, max_seqlen) and the
// tensorplay BlockMask page (full_kv_* lists given together, BLOCK_SIZE).

#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

#define TA_EXPORT extern "C" __attribute__((visibility("default")))

namespace triattn {

// The triangle form with 16-bit inputs and D in (128, 256] on tensor cores (tc_wide.cu);
// cudaErrorNotSupported for a case it does not take.
cudaError_t launch_tc_wide(const AttnParams& a, cudaStream_t stream);

// One status word per device, written by kernels that give up.
__device__ int g_status_word = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_status_mu;
int* g_status_ptr[kMaxDevices] = {};
}  // namespace

int* status_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int*>(p);
    }
    return g_status_ptr[dev];
}

}  // namespace triattn

using triattn::AttnParams;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_dtype(int d) { return d == TA_F32 || d == TA_F16 || d == TA_BF16; }

// Head-dimension rules: 16-bit inputs D % 8 == 0 and D <= 256; fp32 D % 4 == 0 and D <= 256.
bool supported_d(int dtype, int D) {
    if (D > 256) return false;
    return dtype == TA_F32 ? (D % 4 == 0) : (D % 8 == 0);
}

// fp32 inputs run on the CUDA-core kernel; 16-bit inputs on the tensor-core kernels:
// D <= 128 on tc_fwd / tc_split, D in (128, 256] on tc_wide (the triangle form with
// contiguous q / k / v; packed sequences and strided views with D > 128 take the
// CUDA-core kernel).
ta_status run(const AttnParams& p, cudaStream_t stream) {
    cudaError_t e;
    if (p.dtype == TA_F32) {
        e = triattn::launch_simt_fwd(p, stream);
    } else if (p.D > 128) {
        e = triattn::launch_tc_wide(p, stream);
        if (e == cudaErrorNotSupported) e = triattn::launch_simt_fwd(p, stream);
    } else {
        e = triattn::launch_tc_fwd(p, stream);
    }
    return e == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}

}  // namespace

// Element strides {b, n, h, row} of a (B, N, H, rows, D) tensor whose D elements are contiguous:
// the given ones (checked) or, for NULL, the contiguous layout.
ta_status triangle_strides(const long long* given, int B, int N, int H, int rows, int D, int esz, long long (&st)[4]) {
    if (!given) {
        st[3] = D;
        st[2] = (long long)rows * D;
        st[1] = st[2] * H;
        st[0] = st[1] * N;
        return TA_OK;
    }
    const long long ext[4] = {B, N, H, rows};
    for (int i = 0; i < 4; ++i) {
        st[i] = given[i];
        if (st[i] < 1) return TA_ERR_INVALID_ARG;
        // tensor-map strides: 16-byte multiples below 2^40 bytes; every offset fits in 62 bits
        if ((st[i] * esz) % 16 != 0 || st[i] * esz >= (1LL << 40)) return TA_ERR_UNSUPPORTED;
        if (ext[i] > 1 && st[i] > ((1LL << 60) / (ext[i] - 1))) return TA_ERR_UNSUPPORTED;
    }
    if (st[3] < D) return TA_ERR_INVALID_ARG;  // the D elements of one row may not overlap the next row
    return TA_OK;
}

TA_EXPORT ta_status tri_attn_fwd(const void* q, const void* k, const void* v, ta_dtype qkv_dtype, const void* bias,
                                 ta_dtype bias_dtype, const uint8_t* mask, const int32_t* kv_lengths, int B, int N,
                                 int H, int Q, int K, int D, float scale, void* out, float* lse, float* max,
                                 void* stream) {
    return tri_attn_fwd_strided(q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B, N, H, Q, K, D, scale,
                                nullptr, nullptr, nullptr, out, lse, max, stream);
}

TA_EXPORT ta_status tri_attn_fwd_strided(const void* q, const void* k, const void* v, ta_dtype qkv_dtype,
                                         const void* bias, ta_dtype bias_dtype, const uint8_t* mask,
                                         const int32_t* kv_lengths, int B, int N, int H, int Q, int K, int D,
                                         float scale, const long long* q_strides, const long long* k_strides,
                                         const long long* v_strides, void* out, float* lse, float* max,
                                         void* stream) {
    if (!q || !k || !v || !bias || !out) return TA_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || H <= 0 || Q <= 0 || K <= 0 || D <= 0) return TA_ERR_INVALID_ARG;
    if (mask && kv_lengths) return TA_ERR_INVALID_ARG;
    if (!valid_dtype(qkv_dtype) || !valid_dtype(bias_dtype)) return TA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(bias, 16) || !aligned(out, 16))
        return TA_ERR_INVALID_ARG;
    if ((lse && !aligned(lse, 4)) || (max && !aligned(max, 4)) || (kv_lengths && !aligned(kv_lengths, 4)))
        return TA_ERR_INVALID_ARG;
    if (bias_dtype != TA_F32 && bias_dtype != qkv_dtype) return TA_ERR_UNSUPPORTED;
    if (!supported_d(qkv_dtype, D)) return TA_ERR_UNSUPPORTED;
    if (qkv_dtype != TA_F32 && K % 8 != 0) return TA_ERR_UNSUPPORTED;
    // Sizes: every flat element index must fit in 63 bits and the grid in 31.
    const long long units = (long long)B * N * H;
    // The bias plane (Q x K elements of up to 4 bytes) is one stride of a tensor map, and tensor-map
    // strides must stay below 2^40 bytes.
    if (units > (1LL << 40) || (long long)Q * K * 4 >= (1LL << 40) || units * ((Q + 31) / 32) > 0x7fffffffLL)
        return TA_ERR_UNSUPPORTED;

    AttnParams p{};
    const int esz = qkv_dtype == TA_F32 ? 4 : 2;
    ta_status sst;
    if ((sst = triangle_strides(q_strides, B, N, H, Q, D, esz, p.qs)) != TA_OK) return sst;
    if ((sst = triangle_strides(k_strides, B, N, H, K, D, esz, p.ks)) != TA_OK) return sst;
    if ((sst = triangle_strides(v_strides, B, N, H, K, D, esz, p.vs)) != TA_OK) return sst;

    int* status = triattn::status_word();
    if (!status) return TA_ERR_CUDA;
    p.q = q;
    p.k = k;
    p.v = v;
    p.bias = bias;
    p.mask = mask;
    p.kv_len = kv_lengths;
    p.out = out;
    p.lse = lse;
    p.mx = max;
    p.status = status;
    p.dtype = qkv_dtype;
    p.bias_f32 = bias_dtype == TA_F32;
    p.scale = scale;
    p.B = B;
    p.N = N;
    p.H = H;
    p.Q = Q;
    p.K = K;
    p.D = D;
    p.varlen = 0;
    return run(p, static_cast<cudaStream_t>(stream));
}

TA_EXPORT ta_status tri_attn_varlen_fwd(const void* q, const void* k, const void* v, ta_dtype dtype,
                                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int D,
                                        float scale,
                                        const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                        const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                        int mask_heads, int max_q_blocks, int max_kv_blocks, int block_q,
                                        int block_k, ta_mask_mod mask_mod, void* out, float* lse, float* max,
                                        void* stream) {
    return tri_attn_varlen_fwd_strided(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                       max_seqlen_q, max_seqlen_k, H, D, scale, kv_num_blocks, kv_indices,
                                       full_kv_num_blocks, full_kv_indices, mask_heads, max_q_blocks, max_kv_blocks,
                                       block_q, block_k, mask_mod, 0, 0, 0, out, lse, max, stream);
}

TA_EXPORT ta_status tri_attn_varlen_fwd_strided(const void* q, const void* k, const void* v, ta_dtype dtype,
                                                const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                                int num_seqs, int total_q, int total_k, int max_seqlen_q,
                                                int max_seqlen_k, int H, int D, float scale,
                                                const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                                const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                                int mask_heads, int max_q_blocks, int max_kv_blocks, int block_q,
                                                int block_k, ta_mask_mod mask_mod, long long q_row_stride,
                                                long long k_row_stride, long long v_row_stride, void* out,
                                                float* lse, float* max, void* stream) {
    // The parameterised mask_mods take their parameter through tri_attn_varlen_fwd_masked.
    if (mask_mod != TA_MASK_NONE && mask_mod != TA_MASK_CAUSAL) return TA_ERR_INVALID_ARG;
    return tri_attn_varlen_fwd_masked(q, k, v, dtype, cu_seqlens_q, cu_seqlens_k, num_seqs, total_q, total_k,
                                      max_seqlen_q, max_seqlen_k, H, D, scale, kv_num_blocks, kv_indices,
                                      full_kv_num_blocks, full_kv_indices, mask_heads, max_q_blocks, max_kv_blocks,
                                      block_q, block_k, mask_mod, 0, nullptr, 0, nullptr, TA_F32, q_row_stride,
                                      k_row_stride, v_row_stride, out, lse, max, stream);
}

TA_EXPORT ta_status tri_attn_varlen_fwd_masked(const void* q, const void* k, const void* v, ta_dtype dtype,
                                               const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                               int num_seqs, int total_q, int total_k, int max_seqlen_q,
                                               int max_seqlen_k, int H, int D, float scale,
                                               const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                               const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                               int mask_heads, int max_q_blocks, int max_kv_blocks, int block_q,
                                               int block_k, ta_mask_mod mask_mod, int window,
                                               const int32_t* prefix_lengths, int prefix_length,
                                               const void* bias, ta_dtype bias_dtype,
                                               long long q_row_stride, long long k_row_stride,
                                               long long v_row_stride, void* out, float* lse, float* max,
                                               void* stream) {
    if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return TA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || H <= 0 || D <= 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return TA_ERR_INVALID_ARG;
    if (total_q < 0 || total_k < 0) return TA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return TA_ERR_INVALID_ARG;
    if (mask_mod < TA_MASK_NONE || mask_mod > TA_MASK_PREFIX_LM) return TA_ERR_INVALID_ARG;
    if (mask_mod == TA_MASK_SLIDING_WINDOW && window <= 0) return TA_ERR_INVALID_ARG;
    if (mask_mod == TA_MASK_PREFIX_LM && !prefix_lengths && prefix_length < 0) return TA_ERR_INVALID_ARG;
    if (prefix_lengths && !aligned(prefix_lengths, 4)) return TA_ERR_INVALID_ARG;
    if (bias) {
        // (H, max_seqlen_q, max_seqlen_k) of bias_dtype, read by the TMA: 16-byte aligned base
        // and a 16-byte multiple for the row of max_seqlen_k elements
        if (!valid_dtype(bias_dtype) || !aligned(bias, 16)) return TA_ERR_INVALID_ARG;
        if (bias_dtype != TA_F32 && bias_dtype != dtype) return TA_ERR_UNSUPPORTED;
        const int ebias = bias_dtype == TA_F32 ? 4 : 2;
        if (((long long)max_seqlen_k * ebias) % 16 != 0) return TA_ERR_UNSUPPORTED;
        if ((long long)max_seqlen_q * max_seqlen_k * 4 >= (1LL << 40)) return TA_ERR_UNSUPPORTED;
    }
    if ((kv_num_blocks == nullptr) != (kv_indices == nullptr)) return TA_ERR_INVALID_ARG;
    if ((full_kv_num_blocks == nullptr) != (full_kv_indices == nullptr)) return TA_ERR_INVALID_ARG;
    if (full_kv_num_blocks && !kv_num_blocks) return TA_ERR_INVALID_ARG;
    if (kv_num_blocks) {
        if (mask_heads != 1 && mask_heads != H) return TA_ERR_INVALID_ARG;
        if (max_q_blocks <= 0 || max_kv_blocks <= 0) return TA_ERR_INVALID_ARG;
    }
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return TA_ERR_INVALID_ARG;
    if ((lse && !aligned(lse, 4)) || (max && !aligned(max, 4))) return TA_ERR_INVALID_ARG;
    if (block_q != 128 || block_k != 128) return TA_ERR_UNSUPPORTED;
    if (!supported_d(dtype, D)) return TA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * H * ((max_seqlen_q + 31) / 32) > 0x7fffffffLL) return TA_ERR_UNSUPPORTED;
    // Packed-row strides (elements): 0 = H * D; at least one row of heads;
    // 16-byte multiples (TMA row pitch, and the same rule for fp32).
    const long long hd = (long long)H * D;
    if (q_row_stride == 0) q_row_stride = hd;
    if (k_row_stride == 0) k_row_stride = hd;
    if (v_row_stride == 0) v_row_stride = hd;
    if (q_row_stride < hd || k_row_stride < hd || v_row_stride < hd) return TA_ERR_INVALID_ARG;
    // Row strides are tensor-map strides in bytes, which must stay below 2^40.
    const long long esz = dtype == TA_F32 ? 4 : 2;
    if (q_row_stride * esz >= (1LL << 40) || k_row_stride * esz >= (1LL << 40) ||
        v_row_stride * esz >= (1LL << 40))
        return TA_ERR_UNSUPPORTED;
    const int per16 = dtype == TA_F32 ? 4 : 8;
    if (q_row_stride % per16 || k_row_stride % per16 || v_row_stride % per16) return TA_ERR_UNSUPPORTED;
    if (max_seqlen_q == 0 || total_q == 0) return TA_OK;

    int* status = triattn::status_word();
    if (!status) return TA_ERR_CUDA;
    AttnParams p{};
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.lse = lse;
    p.mx = max;
    p.status = status;
    p.dtype = dtype;
    p.scale = scale;
    p.H = H;
    p.D = D;
    p.varlen = 1;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.num_seqs = num_seqs;
    p.max_q = max_seqlen_q;
    p.max_k = max_seqlen_k;
    p.kv_num = kv_num_blocks;
    p.kv_idx = kv_indices;
    p.full_num = full_kv_num_blocks;
    p.full_idx = full_kv_indices;
    p.mask_heads = kv_num_blocks ? mask_heads : 1;
    p.MQ = kv_num_blocks ? max_q_blocks : 0;
    p.MK = kv_num_blocks ? max_kv_blocks : 0;
    p.mask_mod = mask_mod;
    p.window = mask_mod == TA_MASK_SLIDING_WINDOW ? window : 0;
    p.prefix_len = mask_mod == TA_MASK_PREFIX_LM ? prefix_lengths : nullptr;
    p.prefix_all = mask_mod == TA_MASK_PREFIX_LM ? prefix_length : 0;
    p.bias = bias;
    p.bias_f32 = bias && bias_dtype == TA_F32;
    p.total_q = total_q;
    p.total_k = total_k;
    p.q_rs = q_row_stride;
    p.k_rs = k_row_stride;
    p.v_rs = v_row_stride;
    return run(p, static_cast<cudaStream_t>(stream));
}

TA_EXPORT ta_status tri_attn_mask_to_kv_lengths(const uint8_t* mask, int B, int N, int K, int32_t* kv_lengths,
                                                int32_t* nonprefix_count, void* stream) {
    if (!mask || !kv_lengths) return TA_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || K <= 0) return TA_ERR_INVALID_ARG;
    if (!aligned(kv_lengths, 4) || (nonprefix_count && !aligned(nonprefix_count, 4))) return TA_ERR_INVALID_ARG;
    cudaError_t e = triattn::launch_mask_to_kv_lengths(mask, (long long)B * N, K, kv_lengths, nonprefix_count,
                                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}

TA_EXPORT size_t tri_attn_bwd_workspace_size(int B, int N, int H, int Q, int K, int D) {
    if (B <= 0 || N <= 0 || H <= 0 || Q <= 0 || K <= 0 || D <= 0) return 0;
    return triattn::bwd_workspace_floats(B, N, H, Q, K, D) * sizeof(float);
}

TA_EXPORT ta_status tri_attn_bwd(const void* q, const void* k, const void* v, ta_dtype qkv_dtype, const void* bias,
                                 ta_dtype bias_dtype, const uint8_t* mask, const int32_t* kv_lengths, int B, int N,
                                 int H, int Q, int K, int D, float scale, const float* lse, const void* out,
                                 const void* d_out, void* dq, void* dk, void* dv, void* dbias, void* workspace,
                                 size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !bias || !lse || !d_out || !dq || !dk || !dv || !workspace) return TA_ERR_INVALID_ARG;
    if (B <= 0 || N <= 0 || H <= 0 || Q <= 0 || K <= 0 || D <= 0) return TA_ERR_INVALID_ARG;
    if (mask && kv_lengths) return TA_ERR_INVALID_ARG;
    if (!valid_dtype(qkv_dtype) || !valid_dtype(bias_dtype)) return TA_ERR_INVALID_ARG;
    const void* ptrs16[] = {q, k, v, bias, d_out, dq, dk, dv};
    for (const void* ptr : ptrs16)
        if (!aligned(ptr, 16)) return TA_ERR_INVALID_ARG;
    if ((dbias && !aligned(dbias, 16)) || (out && !aligned(out, 16)) || !aligned(lse, 4) || !aligned(workspace, 256) ||
        (kv_lengths && !aligned(kv_lengths, 4)))
        return TA_ERR_INVALID_ARG;
    if (bias_dtype != TA_F32 && bias_dtype != qkv_dtype) return TA_ERR_UNSUPPORTED;
    if (!supported_d(qkv_dtype, D)) return TA_ERR_UNSUPPORTED;
    const long long units = (long long)B * N * H;
    if (units > (1LL << 40) || units * ((Q + 31) / 32) > 0x7fffffffLL || units * ((K + 31) / 32) > 0x7fffffffLL ||
        (long long)Q * K >= (1LL << 40))
        return TA_ERR_UNSUPPORTED;
    if (workspace_bytes < tri_attn_bwd_workspace_size(B, N, H, Q, K, D)) return TA_ERR_INVALID_ARG;

    triattn::BwdParams p{};
    float* ws = static_cast<float*>(workspace);
    auto up = [](size_t n) { return (n + 63) & ~(size_t)63; };
    p.dq_acc = ws;
    p.dbias_acc = dbias ? ws + up((size_t)units * Q * D) : nullptr;
    p.delta = ws + up((size_t)units * Q * D) + up((size_t)B * H * Q * K);
    p.q = q;
    p.k = k;
    p.v = v;
    p.bias = bias;
    p.d_out = d_out;
    p.mask = mask;
    p.kv_len = kv_lengths;
    p.lse = lse;
    p.out = out;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dbias = dbias;
    p.dtype = qkv_dtype;
    p.bias_f32 = bias_dtype == TA_F32;
    p.scale = scale;
    p.B = B;
    p.N = N;
    p.H = H;
    p.Q = Q;
    p.K = K;
    p.D = D;
    p.dq_elems = units * Q * D;
    p.dbias_elems = (long long)B * H * Q * K;
    p.delta_rows = units * Q;
    p.status = triattn::status_word();
    if (!p.status) return TA_ERR_CUDA;
    p.tc_main = triattn::tc_bwd_supported(p) ? 1 : 0;
    const cudaError_t e = triattn::launch_simt_bwd(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}

TA_EXPORT size_t tri_attn_varlen_bwd_workspace_size(int total_q, int H, int D, int max_seqlen_q, int max_seqlen_k,
                                                   int with_bias) {
    if (total_q < 0 || H <= 0 || D <= 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return 0;
    const long long rows = (long long)total_q * H;
    const long long nb = with_bias ? (long long)H * max_seqlen_q * max_seqlen_k : 0;
    return triattn::bwd_workspace_floats_n(rows * D, nb, rows) * sizeof(float);
}

TA_EXPORT ta_status tri_attn_varlen_bwd(const void* q, const void* k, const void* v, ta_dtype dtype,
                                        const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                                        int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int D,
                                        float scale, const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                        const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                        int mask_heads, int max_q_blocks, int max_kv_blocks, int block_q,
                                        int block_k, ta_mask_mod mask_mod, int window,
                                        const int32_t* prefix_lengths, int prefix_length, const void* bias,
                                        ta_dtype bias_dtype, const float* lse, const void* out, const void* d_out,
                                        void* dq, void* dk, void* dv, void* dbias, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !cu_seqlens_q || !cu_seqlens_k || !lse || !out || !d_out || !dq || !dk || !dv ||
        !workspace)
        return TA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || H <= 0 || D <= 0 || max_seqlen_q < 0 || max_seqlen_k < 0) return TA_ERR_INVALID_ARG;
    if (total_q < 0 || total_k < 0) return TA_ERR_INVALID_ARG;
    if (!valid_dtype(dtype)) return TA_ERR_INVALID_ARG;
    if (mask_mod < TA_MASK_NONE || mask_mod > TA_MASK_PREFIX_LM) return TA_ERR_INVALID_ARG;
    if (mask_mod == TA_MASK_SLIDING_WINDOW && window <= 0) return TA_ERR_INVALID_ARG;
    if (mask_mod == TA_MASK_PREFIX_LM && !prefix_lengths && prefix_length < 0) return TA_ERR_INVALID_ARG;
    if (prefix_lengths && !aligned(prefix_lengths, 4)) return TA_ERR_INVALID_ARG;
    if ((kv_num_blocks == nullptr) != (kv_indices == nullptr)) return TA_ERR_INVALID_ARG;
    if ((full_kv_num_blocks == nullptr) != (full_kv_indices == nullptr)) return TA_ERR_INVALID_ARG;
    if (full_kv_num_blocks && !kv_num_blocks) return TA_ERR_INVALID_ARG;
    if (kv_num_blocks) {
        if (mask_heads != 1 && mask_heads != H) return TA_ERR_INVALID_ARG;
        if (max_q_blocks <= 0 || max_kv_blocks <= 0) return TA_ERR_INVALID_ARG;
    }
    if (dbias && !bias) return TA_ERR_INVALID_ARG;
    if (bias) {
        if (!valid_dtype(bias_dtype) || !aligned(bias, 16) || (dbias && !aligned(dbias, 16))) return TA_ERR_INVALID_ARG;
        if (bias_dtype != TA_F32 && bias_dtype != dtype) return TA_ERR_UNSUPPORTED;
    }
    const void* ptrs16[] = {q, k, v, out, d_out, dq, dk, dv};
    for (const void* ptr : ptrs16)
        if (!aligned(ptr, 16)) return TA_ERR_INVALID_ARG;
    if (!aligned(lse, 4) || !aligned(workspace, 256)) return TA_ERR_INVALID_ARG;
    if (block_q != 128 || block_k != 128) return TA_ERR_UNSUPPORTED;
    if (!supported_d(dtype, D)) return TA_ERR_UNSUPPORTED;
    if ((long long)num_seqs * H * ((max_seqlen_k + 31) / 32) > 0x7fffffffLL) return TA_ERR_UNSUPPORTED;
    if (workspace_bytes < tri_attn_varlen_bwd_workspace_size(total_q, H, D, max_seqlen_q, max_seqlen_k, dbias != nullptr))
        return TA_ERR_INVALID_ARG;
    if (total_q == 0) return TA_OK;

    triattn::BwdParams p{};
    const long long rows = (long long)total_q * H;
    p.dq_elems = rows * D;
    p.dbias_elems = dbias ? (long long)H * max_seqlen_q * max_seqlen_k : 0;
    p.delta_rows = rows;
    float* ws = static_cast<float*>(workspace);
    auto up = [](long long n) { return (n + 63) & ~63LL; };
    p.dq_acc = ws;
    p.dbias_acc = dbias ? ws + up(p.dq_elems) : nullptr;
    p.delta = ws + up(p.dq_elems) + up(p.dbias_elems);
    p.q = q;
    p.k = k;
    p.v = v;
    p.bias = bias;
    p.d_out = d_out;
    p.lse = lse;
    p.out = out;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.dbias = dbias;
    p.dtype = dtype;
    p.bias_f32 = bias && bias_dtype == TA_F32;
    p.scale = scale;
    p.B = 1;
    p.N = 1;
    p.H = H;
    p.D = D;
    p.Q = 0;
    p.K = 0;
    p.varlen = 1;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.num_seqs = num_seqs;
    p.total_q = total_q;
    p.total_k = total_k;
    p.max_q = max_seqlen_q;
    p.max_k = max_seqlen_k;
    p.kv_num = kv_num_blocks;
    p.kv_idx = kv_indices;
    p.full_num = full_kv_num_blocks;
    p.full_idx = full_kv_indices;
    p.mask_heads = kv_num_blocks ? mask_heads : 1;
    p.MQ = kv_num_blocks ? max_q_blocks : 0;
    p.MK = kv_num_blocks ? max_kv_blocks : 0;
    p.mask_mod = mask_mod;
    p.window = mask_mod == TA_MASK_SLIDING_WINDOW ? window : 0;
    p.prefix_len = mask_mod == TA_MASK_PREFIX_LM ? prefix_lengths : nullptr;
    p.prefix_all = mask_mod == TA_MASK_PREFIX_LM ? prefix_length : 0;
    p.status = triattn::status_word();
    if (!p.status) return TA_ERR_CUDA;
    p.tc_main = triattn::tc_bwd_supported(p) ? 1 : 0;  // 16-bit, D <= 128: tensor cores
    const cudaError_t e = triattn::launch_simt_bwd(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}

// Scratch of tri_attn_bwd_noalloc: a fixed-size array that is part of the
// library's device image (one copy per device, present from module load), so a
// call allocates nothing.  Its address is looked up once per device.
static __device__ __align__(256) float g_bwd_noalloc_scratch[TRI_ATTN_BWD_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

void* bwd_noalloc_scratch() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_bwd_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc_ptr[dev] = ptr;
    }
    return g_noalloc_ptr[dev];
}
}  // namespace

TA_EXPORT ta_status tri_attn_bwd_noalloc(const void* q, const void* k, const void* v, ta_dtype qkv_dtype,
                                         const void* bias, ta_dtype bias_dtype, const uint8_t* mask,
                                         const int32_t* kv_lengths, int B, int N, int H, int Q, int K, int D,
                                         float scale, const float* lse, const void* out, const void* d_out,
                                         void* dq, void* dk,
                                         void* dv, void* dbias, void* stream) {
    // A problem whose workspace exceeds the static scratch is refused before anything runs.
    if (tri_attn_bwd_workspace_size(B, N, H, Q, K, D) > (size_t)TRI_ATTN_BWD_NOALLOC_SCRATCH_BYTES)
        return TA_ERR_UNSUPPORTED;
    void* ws = bwd_noalloc_scratch();
    if (!ws) return TA_ERR_CUDA;
    return tri_attn_bwd(q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B, N, H, Q, K, D, scale, lse, out, d_out,
                        dq, dk, dv, dbias, ws, (size_t)TRI_ATTN_BWD_NOALLOC_SCRATCH_BYTES, stream);
}

TA_EXPORT ta_status tri_attn_get_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TA_ERR_CUDA;
    int* w = triattn::status_word();
    if (!w) return TA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TA_ERR_CUDA;
    if (v != 0 && cudaMemset(w, 0, sizeof(int)) != cudaSuccess) return TA_ERR_CUDA;
    return static_cast<ta_status>(v);
}

TA_EXPORT const char* tri_attn_error_string(ta_status s) {
    switch (s) {
    case TA_OK: return "ok";
    case TA_ERR_INVALID_ARG: return "invalid argument";
    case TA_ERR_UNSUPPORTED: return "unsupported configuration";
    case TA_ERR_CUDA: return "CUDA error";
    case TA_ERR_TIMEOUT: return "kernel pipeline wait timed out";
    case TA_ERR_DEVICE: return "device-side value outside its contract";
    default: return "unknown status";
    }
}

TA_EXPORT int tri_attn_version(void) { return (1 << 16) | 3; }
