// internal.h -- parameter blocks and launchers shared by the host entry points
// and the kernels of the triangle-attention library.  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/triattn.h"

namespace triattn {

// Device-side status codes (match ta_status).  A kernel that gives up writes
// one with atomicCAS(status, 0, code) so the first fault is kept.
enum : int { kStatusOk = 0, kStatusTimeout = TA_ERR_TIMEOUT, kStatusDevice = TA_ERR_DEVICE };

// One attention problem as the kernels see it.  Triangle form: units are
// (b, n, h) slabs with Q query rows and K keys.  Varlen form: units are
// (sequence, h) with lengths read from cu_seqlens.
struct AttnParams {
    const void* q;
    const void* k;
    const void* v;
    const void* bias;       // triangle only, may be NULL in varlen
    const uint8_t* mask;    // triangle dense key mask (B,N,K) or NULL
    const int32_t* kv_len;  // triangle kv_lengths (B,N) or NULL
    void* out;
    float* lse;
    float* mx;
    int* status;            // device status word

    int dtype;              // ta_dtype of q/k/v/out
    int bias_f32;           // 1: bias is fp32, 0: bias has the q/k/v dtype
    float scale;

    // triangle sizes
    int B, N, H, Q, K, D;
    // triangle q, k, v: element strides of the b, n, h and row (q / key) indices; the D elements of
    // a row are contiguous.  Contiguous tensors: {N*H*rows*D, H*rows*D, rows*D, D}.
    long long qs[4], ks[4], vs[4];

    // varlen
    int varlen;
    const int32_t* cu_q;
    const int32_t* cu_k;
    int num_seqs, max_q, max_k;
    const int32_t* kv_num;
    const int32_t* kv_idx;
    const int32_t* full_num;
    const int32_t* full_idx;
    int mask_heads, MQ, MK, mask_mod;
    int window;             // TA_MASK_SLIDING_WINDOW: keys q - window < k <= q
    const int32_t* prefix_len;  // TA_MASK_PREFIX_LM: per-sequence prefix lengths, or NULL:
    int prefix_all;         //   then prefix_all for every sequence
    int total_q;            // rows of q/out (lse/max stride in varlen)
    int total_k;            // rows of k/v
    long long q_rs, k_rs, v_rs;  // varlen: elements between packed rows of q, k, v (out: H * D)
};

// Backward of the triangle form (CUDA cores, exact fp32 arithmetic).
struct BwdParams {
    const void* q;
    const void* k;
    const void* v;
    const void* bias;
    const void* d_out;
    const uint8_t* mask;
    const int32_t* kv_len;
    const float* lse;       // (B, N, H, Q) from the forward
    const void* out;        // the forward's O (q dtype) or NULL: delta = rowsum(dO * O) if given
    void* dq;
    void* dk;
    void* dv;
    void* dbias;            // (B, 1, H, Q, K) or NULL
    float* dq_acc;          // workspace: fp32 dQ (B, N, H, Q, D)
    float* dbias_acc;       // workspace: fp32 dBias (B, H, Q, K), NULL with dbias
    float* delta;           // workspace: sum_k P dP per query row (B, N, H, Q)
    int dtype, bias_f32;
    float scale;
    int B, N, H, Q, K, D;
    int tc_main;            // 1: the per-key-tile gradients on tensor cores (tc_bwd.cu)
    // Element counts of dQ and dBias and the number of per-row sums (either form).
    long long dq_elems, dbias_elems, delta_rows;
    // Packed sequences (varlen = 1): q / k / v / O / dO (total, H, D), lse / delta (H, total_q),
    // the optional bias and dBias (H, max_seqlen_q, max_seqlen_k), the BlockMask lists.
    int varlen;
    const int32_t* cu_q;
    const int32_t* cu_k;
    int num_seqs, total_q, total_k, max_q, max_k;
    const int32_t* kv_num;
    const int32_t* kv_idx;
    const int32_t* full_num;
    const int32_t* full_idx;
    int mask_heads, MQ, MK, mask_mod, window;
    const int32_t* prefix_len;
    int prefix_all;
    int* status;
};
// Workspace of the backward in floats: dQ, dBias and the per-row sums, each rounded up
// to a multiple of 64 floats.
size_t bwd_workspace_floats(int B, int N, int H, int Q, int K, int D);
size_t bwd_workspace_floats_n(long long dq_elems, long long dbias_elems, long long delta_rows);
cudaError_t launch_simt_bwd(const BwdParams& p, cudaStream_t stream);
// The tensor-core form of the backward's per-key-tile kernel (16-bit, D % 16 == 0,
// D <= 64, K % 8 == 0); the caller runs the per-row sums before and the conversion after.
cudaError_t launch_tc_bwd_main(const BwdParams& p, cudaStream_t stream);
bool tc_bwd_supported(const BwdParams& p);

// CUDA-core path: exact fp32 arithmetic, any dtype, both forms.
cudaError_t launch_simt_fwd(const AttnParams& p, cudaStream_t stream);

// tcgen05 / TMA path for fp16 / bf16 (both forms).
cudaError_t launch_tc_fwd(const AttnParams& p, cudaStream_t stream);

// mask -> prefix lengths.
cudaError_t launch_mask_to_kv_lengths(const uint8_t* mask, long long rows, int K, int32_t* kv_len,
                                      int32_t* nonprefix, cudaStream_t stream);

// Device address of the status word on the current device (set up once per device).
int* status_word();

}  // namespace triattn
