/*
 * triattn.h -- C ABI of the GB300 (sm_103a) triangle-attention forward.
 *
 * Operation (cuEquivariance "triangle_attention" API page, formula):
 *
 *   O[b,n,h,q,:] = sum_k softmax_k(x) V[b,n,h,k,:]
 *   x_k = s * (Q[b,n,h,q,:] . K[b,n,h,k,:]) + bias[b,0,h,q,k]   if key k is valid
 *   x_k = -1e9                                                   otherwise
 *   lse[b,n,h,q] = log sum_k exp(x_k),   max[b,n,h,q] = max_k x_k
 *
 * A masked key's logit is REPLACED by -1e9, so a row with no valid key gets a
 * uniform softmax over all K keys: O is the mean of V, max = -1e9 and
 * lse = -1e9 + ln K, which is -1e9 after rounding to fp32.
 *
 * Conventions shared by every entry point:
 *   - All tensors are dense, contiguous, row-major device buffers owned by the
 *     caller.  q, k, v, bias and out must be 16-byte aligned (they are read
 *     and written in 16-byte vectors and by the TMA); lse, max, kv_lengths,
 *     the sequence offsets and the block lists need 4-byte alignment.  A
 *     misaligned pointer returns TA_ERR_INVALID_ARG.  The library allocates
 *     no device memory per call and keeps no state between calls besides one
 *     device-side status word (see tri_attn_get_status).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously on it; results are ready when the stream is.
 *   - Argument checks are made on the host before anything is enqueued, read
 *     no device memory, and return TA_ERR_INVALID_ARG (malformed call) or
 *     TA_ERR_UNSUPPORTED (well-formed but outside what the kernels cover).
 *     A CUDA launch error returns TA_ERR_CUDA.  Nothing throws across the ABI.
 *   - Faults detected inside a kernel (a bounded wait that ran out, a device
 *     value outside its contract) do not trap: the kernel records a code in
 *     the status word and returns.  tri_attn_get_status() reports it.
 *   - Entry points are thread-safe; calls on different streams may overlap.
 */
#ifndef TRIATTN_H
#define TRIATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TA_OK = 0,
    TA_ERR_INVALID_ARG = 1, /* malformed call: NULL required pointer, size <= 0, misaligned pointer, both mask kinds */
    TA_ERR_UNSUPPORTED = 2, /* well-formed but outside the kernels: dtype pair, D, K alignment, block size */
    TA_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed (no device, launch failure, ...) */
    TA_ERR_TIMEOUT = 4,     /* a kernel's bounded pipeline wait ran out (reported by tri_attn_get_status) */
    TA_ERR_DEVICE = 5       /* a kernel saw a device-side value outside its contract (e.g. seqlen > max_seqlen) */
} ta_status;

/* Element types.  Precision follows the input dtype (triangle_attention page, Notes 2). */
typedef enum { TA_F32 = 0, TA_F16 = 1, TA_BF16 = 2 } ta_dtype;

/* Element predicate applied on partial blocks of a BlockMask (tensorplay
 * "BlockMask", Details 2: mask_mod is skipped on full blocks), for query q and
 * key k, both indices local to their sequence:
 *   CAUSAL          k <= q
 *   SLIDING_WINDOW  q - window < k <= q  (the query and the window - 1 keys before it)
 *   PREFIX_LM       k <= q  or  k < prefix  (the sequence's prefix is seen by every query)
 * The last two carry a parameter and are taken by tri_attn_varlen_fwd_masked only. */
typedef enum {
    TA_MASK_NONE = 0,
    TA_MASK_CAUSAL = 1,
    TA_MASK_SLIDING_WINDOW = 2,
    TA_MASK_PREFIX_LM = 3
} ta_mask_mod;

/*
 * tri_attn_fwd -- triangle-attention forward.
 * (cuEquivariance triangle_attention page: formula; Parameters q, k, v, bias,
 *  mask, scale, kv_lengths; Returns.)
 *
 *   q, out      (B, N, H, Q, D) of `qkv_dtype`
 *   k, v        (B, N, H, K, D) of `qkv_dtype`
 *   bias        (B, 1, H, Q, K) of `bias_dtype`; required; shared over N.
 *               bias_dtype is TA_F32 or equal to qkv_dtype; it is read in
 *               its stored type, never cast.
 *   mask        optional (B, N, 1, 1, K) uint8, nonzero = valid key
 *   kv_lengths  optional (B, N) int32 (same memory as (B, N, 1, 1, 1)): keys
 *               j < kv_lengths[b,n] are valid.  Values above K are clamped to
 *               K (the page); negative values are read as 0 (all masked).
 *               At most one of mask / kv_lengths may be given (the page:
 *               "Pass either mask or kv_lengths, not both"); neither = no mask.
 *   scale       s in the formula, used as given (the Python binding applies
 *               the page's default 1/sqrt(D) when scale is None).
 *               Precondition: every valid key's logit s*(Q.K) + bias stays
 *               above -1e9 + 100 (true whenever |bias| and |s*Q.K| are far
 *               below 1e9).  The kernels skip key tiles that hold only masked
 *               keys, which is exact because such a key's weight
 *               exp(-1e9 - max) is 0 in fp32; a row whose valid logits all
 *               lie at or below -1e9 would instead need those masked keys.
 *   lse, max    optional (B, N, H, Q) fp32 outputs (return_aux); NULL skips.
 *
 * Supported: fp16/bf16 q/k/v with D % 8 == 0, D <= 256 and K % 8 == 0 (the
 * page's Notes 3-4 bounds for the half-precision forward: hidden_dim <= 256),
 * on tcgen05 tensor cores for D <= 128 and on the exact-fp32 CUDA-core kernel
 * for D in (128, 256]; fp32 q/k/v with D % 4 == 0, D <= 256 on exact-fp32
 * CUDA-core arithmetic (no TF32).  fp32 bias with 16-bit q/k/v additionally needs
 * K % 4 == 0 (met by K % 8).  Anything else -> TA_ERR_UNSUPPORTED; there is
 * no fallback path.
 */
ta_status tri_attn_fwd(const void* q, const void* k, const void* v, ta_dtype qkv_dtype,
                       const void* bias, ta_dtype bias_dtype,
                       const uint8_t* mask, const int32_t* kv_lengths,
                       int B, int N, int H, int Q, int K, int D, float scale,
                       void* out, float* lse, float* max, void* stream);

/*
 * tri_attn_fwd_strided -- tri_attn_fwd on q / k / v given as strided views.
 * (cuEquivariance triangle_attention page: the same operation on the same
 *  (B, N, H, Q|K, D) tensors; views such as a (B, N, Q, H, D) buffer read as
 *  (B, N, H, Q, D), or rows padded past D, are read in place.)
 *
 *   q_strides, k_strides, v_strides  optional host arrays of 4 element strides
 *                  {b, n, h, row} of q, k, v (row = the q / key index); the D
 *                  elements of a row are contiguous.  NULL = contiguous.  Each
 *                  stride must be >= 1 and the row stride >= D (else
 *                  TA_ERR_INVALID_ARG), and a multiple of 16 bytes below 2^40
 *                  bytes (else TA_ERR_UNSUPPORTED).  The inputs are only read,
 *                  so views may overlap one another.
 *   every other argument, including the contiguous `out`, as in tri_attn_fwd.
 */
ta_status tri_attn_fwd_strided(const void* q, const void* k, const void* v, ta_dtype qkv_dtype,
                               const void* bias, ta_dtype bias_dtype,
                               const uint8_t* mask, const int32_t* kv_lengths,
                               int B, int N, int H, int Q, int K, int D, float scale,
                               const long long* q_strides, const long long* k_strides, const long long* v_strides,
                               void* out, float* lse, float* max, void* stream);

/*
 * tri_attn_bwd -- gradients of tri_attn_fwd: dQ, dK, dV and dBias.
 * (cuEquivariance triangle_attention page, Notes 1: the context is saved for
 *  backward, and its Example reads q.grad, k.grad, v.grad and bias.grad.)
 * For a loss L with dL/dO = d_out, per (b, n, h) slab and query row q:
 *     P = exp(x - lse) (x the forward's logits, -1e9 at masked keys),
 *     dV[k] = sum_q P dO[q],  dP = dO[q] . V[k],
 *     dx = P (dP - sum_k' P dP) at valid keys, 0 at masked keys,
 *     dQ[q] = s sum_k dx K[k],  dK[k] = s sum_q dx Q[q],
 *     dBias[b, 0, h, q, k] = sum over n of dx[b, n, h, q, k].
 * A row whose keys are all masked passes no gradient to q, k or the bias; its
 * uniform weights 1/K still reach dV (such a row is recognised by its stored
 * lse, -1e9 in fp32; any row with a valid key has lse above -1e9 + 100 by the
 * forward's precondition on the logits).
 *
 *   q, k, v, qkv_dtype, bias, bias_dtype, mask, kv_lengths, B..D, scale
 *               as given to tri_attn_fwd (contiguous tensors).
 *   lse         (B, N, H, Q) fp32, the forward's lse output (required).
 *   out         the forward's O (B, N, H, Q, D) in qkv_dtype, or NULL.  Given,
 *               sum_k' P dP is formed as the row sum of dO * O (fp32 from the
 *               stored O, one pass over two (Q, D) tensors); NULL, it is formed
 *               exactly from its definition, a second pass over every key.
 *   d_out       (B, N, H, Q, D) in qkv_dtype: dL/dO.
 *   dq, dk, dv  (B, N, H, Q|K, D) outputs in qkv_dtype.
 *   dbias       (B, 1, H, Q, K) output in bias_dtype, or NULL to skip it.
 *   workspace   device scratch of at least tri_attn_bwd_workspace_size(...)
 *               bytes, 256-byte aligned, owned by the caller; its contents on
 *               entry are ignored and on return are unspecified.  Two calls in
 *               flight must not share a workspace.
 * Arithmetic (three kernels: the per-row sum of P dP, the per-key-tile
 * gradients with dQ and dBias added atomically in fp32, the conversion to the
 * output dtypes): fp16 / bf16 inputs with D in {16, 32, 64}, or a multiple of 16
 * up to 128, and K % 8 == 0 take the per-key-tile gradients on tcgen05 tensor
 * cores (P^T and dS^T in 16 bits,
 * fp32 accumulation); every other case runs exact fp32 on CUDA cores.  The
 * summation order of dQ and dBias varies from run to run within fp32 rounding.
 * Supported: as tri_attn_fwd (D <= 256).  Errors: NULL required pointer,
 * misalignment (16 bytes for tensors, 4 for lse / kv_lengths, 256 for the
 * workspace) or a workspace below the required size -> TA_ERR_INVALID_ARG;
 * unsupported sizes or dtypes -> TA_ERR_UNSUPPORTED; a launch failure ->
 * TA_ERR_CUDA.  Asynchronous on `stream`.
 */
ta_status tri_attn_bwd(const void* q, const void* k, const void* v, ta_dtype qkv_dtype,
                       const void* bias, ta_dtype bias_dtype,
                       const uint8_t* mask, const int32_t* kv_lengths,
                       int B, int N, int H, int Q, int K, int D, float scale,
                       const float* lse, const void* out, const void* d_out,
                       void* dq, void* dk, void* dv, void* dbias,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace tri_attn_bwd needs for these sizes (0 for a non-positive size). */
size_t tri_attn_bwd_workspace_size(int B, int N, int H, int Q, int K, int D);

/* Size of the fixed device scratch tri_attn_bwd_noalloc works in (bytes). */
#define TRI_ATTN_BWD_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * tri_attn_bwd_noalloc -- tri_attn_bwd without a caller workspace and without
 * any allocation.  The source pages have no counterpart of this call: it is a
 * library-side variant of tri_attn_bwd for callers that may not allocate.
 *
 * Arguments, results and errors as tri_attn_bwd, minus workspace and
 * workspace_bytes.  The scratch is a static device array of
 * TRI_ATTN_BWD_NOALLOC_SCRATCH_BYTES bytes inside the library (one per
 * device); its address is looked up once per device.  The call itself
 * allocates no memory of any kind.  It needs no zeroed scratch: the backward's
 * first kernel zeroes the accumulators it uses on every call.
 *   A problem whose tri_attn_bwd_workspace_size exceeds the scratch ->
 *   TA_ERR_UNSUPPORTED (nothing is launched); use tri_attn_bwd then.
 *   Calls in flight at the same time on one device (on any streams, from any
 *   threads) share the scratch and race: the caller must order them, e.g. by
 *   issuing them on one stream.
 */
ta_status tri_attn_bwd_noalloc(const void* q, const void* k, const void* v, ta_dtype qkv_dtype,
                               const void* bias, ta_dtype bias_dtype,
                               const uint8_t* mask, const int32_t* kv_lengths,
                               int B, int N, int H, int Q, int K, int D, float scale,
                               const float* lse, const void* out, const void* d_out,
                               void* dq, void* dk, void* dv, void* dbias, void* stream);

/*
 * tri_attn_varlen_fwd -- packed-sequence forward with a block-sparse mask.
 * (Transformer Engine 0.9 fused_attn.h: NVTE_NOT_INTERLEAVED layout,
 *  cu_seqlens_q / cu_seqlens_kv, max_seqlen_q / max_seqlen_kv; tensorplay
 *  nn.attention "BlockMask": kv_num_blocks / kv_indices, full_kv_* lists,
 *  BLOCK_SIZE, mask_mod.)
 *
 *   q, out        (total_q, H, D) of `dtype`;  k, v (total_k, H, D); total_q and
 *                 total_k are the row counts of those buffers (the packed
 *                 "total_seqs" dimension), so no kernel touches a row past them
 *   cu_seqlens_q  (num_seqs + 1) int32, cu_seqlens_q[0] = 0, non-decreasing;
 *   cu_seqlens_k  likewise for keys.  Sequence i holds rows
 *                 [cu[i], cu[i+1]).  Every length must be <= the matching
 *                 max_seqlen and cu[num_seqs] <= the matching total (else
 *                 TA_ERR_DEVICE is recorded and that sequence is skipped).
 *   kv_num_blocks (num_seqs, mask_heads, max_q_blocks) int32 and
 *   kv_indices    (num_seqs, mask_heads, max_q_blocks, max_kv_blocks) int32:
 *                 partial kv blocks of each 128-row q block, sequence-local
 *                 block indices; entries past the count are never read and
 *                 out-of-range indices are skipped.  NULL (both) = every
 *                 block of the sequence is partial.
 *   full_kv_num_blocks / full_kv_indices: same shapes, optional, both or
 *                 neither (else TA_ERR_INVALID_ARG): blocks where every key
 *                 is valid, visited without mask_mod.  The two lists must be
 *                 disjoint.  Keys outside every listed block have logit -1e9.
 *   mask_heads    1 (one mask for all heads) or H.
 *   block_q, block_k  must both be 128 (else TA_ERR_UNSUPPORTED).
 *   lse, max      optional (H, total_q) fp32.
 *   No bias here (tri_attn_varlen_fwd_masked takes one).  A key row past the end of its sequence takes no part.  A
 *   sequence with no keys gets O = 0 and lse = max = -inf.
 *
 * Supported: fp16/bf16 with D % 8 == 0, D <= 256 (tcgen05 up to 128, the
 * CUDA-core kernel above), fp32 with D % 4 == 0, D <= 256 (CUDA cores).
 */
ta_status tri_attn_varlen_fwd(const void* q, const void* k, const void* v, ta_dtype dtype,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                              int num_seqs, int total_q, int total_k,
                              int max_seqlen_q, int max_seqlen_k, int H, int D,
                              float scale,
                              const int32_t* kv_num_blocks, const int32_t* kv_indices,
                              const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                              int mask_heads, int max_q_blocks, int max_kv_blocks,
                              int block_q, int block_k, ta_mask_mod mask_mod,
                              void* out, float* lse, float* max, void* stream);

/*
 * tri_attn_varlen_fwd_strided -- tri_attn_varlen_fwd on q / k / v whose
 * packed rows are `*_row_stride` elements apart.
 * (Transformer Engine fused_attn.h, NVTE_QKV_Layout: NVTE_NOT_INTERLEAVED is
 *  q, k, v each (total, H, D); NVTE_QKV_INTERLEAVED is one (total, 3, H, D)
 *  buffer, i.e. q, k, v at element offsets 0, H*D, 2*H*D with row stride
 *  3*H*D; NVTE_KV_INTERLEAVED keeps q (total_q, H, D) and packs k, v in one
 *  (total_k, 2, H, D) buffer: offsets 0, H*D, row stride 2*H*D.)
 *
 *   q, k, v        row r, head h, element d at  base[r * row_stride + h * D + d]
 *                  (heads contiguous within a row); every other argument,
 *                  including the contiguous (total_q, H, D) `out`, as in
 *                  tri_attn_varlen_fwd.
 *   *_row_stride   elements between consecutive packed rows; 0 means H * D
 *                  (no interleaving).  Must be >= H * D (else
 *                  TA_ERR_INVALID_ARG) and a multiple of 16 bytes
 *                  (fp16 / bf16: of 8 elements; fp32: of 4), else
 *                  TA_ERR_UNSUPPORTED.  The pointers keep the 16-byte rule.
 *   The buffers are read only; interleaved q / k / v may share memory.
 */
ta_status tri_attn_varlen_fwd_strided(const void* q, const void* k, const void* v, ta_dtype dtype,
                                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                      int num_seqs, int total_q, int total_k,
                                      int max_seqlen_q, int max_seqlen_k, int H, int D,
                                      float scale,
                                      const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                      const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                      int mask_heads, int max_q_blocks, int max_kv_blocks,
                                      int block_q, int block_k, ta_mask_mod mask_mod,
                                      long long q_row_stride, long long k_row_stride, long long v_row_stride,
                                      void* out, float* lse, float* max, void* stream);

/*
 * tri_attn_varlen_fwd_masked -- tri_attn_varlen_fwd_strided with the
 * parameterised mask_mods and an optional post-scale bias.
 * (tensorplay nn.attention "BlockMask": from_kv_blocks(..., mask_mod=...) and
 *  Details 2, mask_mod applied on partial blocks only; the sliding-window and
 *  prefix-LM predicates are the two most common mask_mods besides causal.)
 *
 *   mask_mod        TA_MASK_NONE, TA_MASK_CAUSAL, TA_MASK_SLIDING_WINDOW or
 *                   TA_MASK_PREFIX_LM (else TA_ERR_INVALID_ARG)
 *   window          SLIDING_WINDOW: keys q - window < k <= q are kept; must be
 *                   >= 1 (else TA_ERR_INVALID_ARG); ignored otherwise
 *   prefix_lengths  PREFIX_LM: optional (num_seqs) int32 on the device, the
 *                   prefix of each sequence (values <= 0 keep only causal
 *                   keys); when NULL, `prefix_length` (>= 0, else
 *                   TA_ERR_INVALID_ARG) applies to every sequence
 *   bias            optional post-scale bias (Transformer Engine fused_attn.h,
 *                   NVTE_Bias_Type NVTE_POST_SCALE_BIAS): (H, max_seqlen_q,
 *                   max_seqlen_k) of `bias_dtype` (TA_F32 or `dtype`, else
 *                   TA_ERR_UNSUPPORTED), shared by every sequence and indexed
 *                   by local positions: x = s * (Q . K) + bias[h, q, k] for a
 *                   valid key (a masked key's logit is -1e9 as always).  16-byte
 *                   aligned, and max_seqlen_k * its element size a multiple of
 *                   16 bytes (else TA_ERR_UNSUPPORTED).  NULL = no bias.
 *   every other argument as in tri_attn_varlen_fwd_strided (which takes
 *   TA_MASK_NONE and TA_MASK_CAUSAL only, and no bias).  A row whose visited
 *   keys are all masked gets the mean of V over the sequence's keys (every
 *   logit -1e9), as with any other mask.
 */
ta_status tri_attn_varlen_fwd_masked(const void* q, const void* k, const void* v, ta_dtype dtype,
                                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                                     int num_seqs, int total_q, int total_k,
                                     int max_seqlen_q, int max_seqlen_k, int H, int D,
                                     float scale,
                                     const int32_t* kv_num_blocks, const int32_t* kv_indices,
                                     const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                                     int mask_heads, int max_q_blocks, int max_kv_blocks,
                                     int block_q, int block_k, ta_mask_mod mask_mod,
                                     int window, const int32_t* prefix_lengths, int prefix_length,
                                     const void* bias, ta_dtype bias_dtype,
                                     long long q_row_stride, long long k_row_stride, long long v_row_stride,
                                     void* out, float* lse, float* max, void* stream);

/*
 * tri_attn_varlen_bwd -- gradients of the packed-sequence forward
 * (tri_attn_varlen_fwd_masked with contiguous rows): dQ, dK, dV and, with a
 * bias, dBias.  (cuEquivariance triangle_attention page, Notes 1: context saved
 * for backward; tensorplay BlockMask page, Details 1-4: the block lists decide
 * which (query, key) blocks take part, full blocks skip mask_mod.)
 * Per sequence and head, with P = exp(x - lse) from the forward's lse:
 *     dV = P^T dO,  dx = P (dP - sum_k P dP) at valid keys (0 at masked ones),
 *     dQ = s dx K,  dK = s dx^T Q,  dBias[h, q, k] = sum over sequences of dx.
 * A key is valid for a query when its block is a full block, or a partial
 * block (every block without lists) whose mask_mod keeps it; keys of blocks
 * the lists leave out are masked.
 *   q, k, v, dtype, cu_seqlens_*, num_seqs, total_*, max_seqlen_*, H, D, scale,
 *   the block lists, mask_mod, window, prefix_lengths / prefix_length, bias,
 *   bias_dtype    as given to tri_attn_varlen_fwd_masked; q / k / v contiguous
 *                 (total, H, D).
 *   lse           (H, total_q) fp32 from the forward (required).
 *   out           the forward's O (total_q, H, D) (required: sum_k P dP is the
 *                 row sum of dO * O).
 *   d_out         (total_q, H, D) in dtype.
 *   dq, dk, dv    outputs shaped like q, k, v.
 *   dbias         (H, max_seqlen_q, max_seqlen_k) in bias_dtype, or NULL (needs a bias).
 *   workspace     device scratch of tri_attn_varlen_bwd_workspace_size(...,
 *                 with_bias = dbias != NULL) bytes, 256-byte aligned, owned by
 *                 the caller.
 * Arithmetic: fp16 / bf16 inputs with D a multiple of 16 up to 128 (no bias, or
 * a bias whose max_seqlen_k rows are 16-byte multiples) run on tensor cores (one CTA per sequence, head and 128-key block, over the q
 * blocks whose lists hold that block and those with a row that has no valid
 * key; P and dS rounded to the input type as the MMAs' operands, fp32
 * accumulation); every other case exact fp32 on CUDA cores (one CTA per
 * sequence, head and 32 keys).  dQ and dBias are added in fp32 with atomic
 * reductions, so their summation order varies from run to run.  Errors as tri_attn_bwd; a sequence that
 * breaks the max_seqlen / total contract is skipped and TA_ERR_DEVICE recorded.
 */
ta_status tri_attn_varlen_bwd(const void* q, const void* k, const void* v, ta_dtype dtype,
                              const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs,
                              int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int H, int D,
                              float scale, const int32_t* kv_num_blocks, const int32_t* kv_indices,
                              const int32_t* full_kv_num_blocks, const int32_t* full_kv_indices,
                              int mask_heads, int max_q_blocks, int max_kv_blocks, int block_q, int block_k,
                              ta_mask_mod mask_mod, int window, const int32_t* prefix_lengths, int prefix_length,
                              const void* bias, ta_dtype bias_dtype, const float* lse, const void* out,
                              const void* d_out, void* dq, void* dk, void* dv, void* dbias, void* workspace,
                              size_t workspace_bytes, void* stream);

/* Bytes of workspace tri_attn_varlen_bwd needs (0 for a negative size). */
size_t tri_attn_varlen_bwd_workspace_size(int total_q, int H, int D, int max_seqlen_q, int max_seqlen_k,
                                          int with_bias);

/*
 * tri_attn_mask_to_kv_lengths -- dense key mask -> prefix lengths.
 * (triangle_attention page, Example: mask_to_kv_lengths(mask).)
 *
 *   mask            (B, N, 1, 1, K) uint8, nonzero = valid
 *   kv_lengths      (B, N) int32 output: count of leading valid keys per row
 *   nonprefix_count optional single int32 on the device; the number of rows
 *                   that have a valid key after their first masked key (rows
 *                   a prefix length cannot represent) is ADDED to it.
 */
ta_status tri_attn_mask_to_kv_lengths(const uint8_t* mask, int B, int N, int K, int32_t* kv_lengths,
                                      int32_t* nonprefix_count, void* stream);

/*
 * tri_attn_get_status -- synchronize `stream`, then read and clear the
 * device-side status word of the current device.  Returns TA_OK, or the first
 * TA_ERR_TIMEOUT / TA_ERR_DEVICE recorded by a kernel since the last call, or
 * TA_ERR_CUDA if the synchronization itself failed.
 */
ta_status tri_attn_get_status(void* stream);

/* Static, human-readable name of a status code (never NULL). */
const char* tri_attn_error_string(ta_status status);

/* Library ABI version, (major << 16) | minor. */
int tri_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TRIATTN_H */
