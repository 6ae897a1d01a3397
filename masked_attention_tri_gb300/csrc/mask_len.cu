// mask_len.cu -- dense key mask -> prefix lengths (the triangle_attention
// page's mask_to_kv_lengths helper, Example).
//
// One warp per (b, n) row: scan the K mask bytes in 32-key chunks, find the
// first masked key with a ballot, and note whether any valid key follows it
// (a row that a prefix length cannot represent).

#include "internal.h"

namespace triattn {
namespace {

__global__ void __launch_bounds__(256) mask_len_kernel(const uint8_t* __restrict__ mask, long long rows, int K,
                                                       int32_t* __restrict__ kv_len, int32_t* nonprefix) {
    const long long row = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= rows) return;
    const uint8_t* m = mask + row * K;
    int first_zero = K;
    bool holey = false;
    for (int base = 0; base < K; base += 32) {
        int key = base + lane;
        bool valid = key < K && m[key] != 0;
        bool masked = key < K && !valid;
        unsigned zeros = __ballot_sync(0xffffffffu, masked);
        unsigned ones = __ballot_sync(0xffffffffu, valid);
        if (first_zero == K) {
            if (zeros) {
                int z = __ffs(zeros) - 1;
                first_zero = base + z;
                // valid keys after the first masked key in this chunk
                unsigned after = (z == 31) ? 0u : (ones & (0xffffffffu << (z + 1)));
                if (after) holey = true;
            }
        } else if (ones) {
            holey = true;
        }
        if (holey) break;
    }
    if (lane == 0) {
        kv_len[row] = first_zero;
        if (holey && nonprefix) atomicAdd(nonprefix, 1);
    }
}

}  // namespace

cudaError_t launch_mask_to_kv_lengths(const uint8_t* mask, long long rows, int K, int32_t* kv_len,
                                      int32_t* nonprefix, cudaStream_t stream) {
    if (rows <= 0) return cudaSuccess;
    const int warps = 8;
    long long grid = (rows + warps - 1) / warps;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    mask_len_kernel<<<(unsigned)grid, warps * 32, 0, stream>>>(mask, rows, K, kv_len, nonprefix);
    return cudaGetLastError();
}

}  // namespace triattn
