// tc_fwd.cu -- host side of the tcgen05 forward: TMA descriptors, geometry
// (query tiles per CTA, pipeline depths, tensor-memory columns), the choice
// of the folded softmax for the packed form, and the launch.  Triangle
// problems with D <= 64 and packed sequences (up to kSplitMaxSeqs of them) go
// to the key-split kernel of tc_split.cuh, the rest to tc_kernel.cuh.

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <mutex>

#include "tc_split.cuh"

namespace triattn {
namespace tc {

TRIATTN_TC_VARIANTS(TRIATTN_TC_EXTERN)
TRIATTN_SPLIT_TRI_VARIANTS(TRIATTN_SPLIT_EXTERN)
TRIATTN_SPLIT_VARLEN_VARIANTS(TRIATTN_SPLIT_EXTERN)
TRIATTN_SPLIT_VARLEN_BIAS_VARIANTS(TRIATTN_SPLIT_EXTERN)

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
std::mutex g_sm_mu;
int g_num_sms[64] = {};

bool get_encode() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

int num_sms() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(g_sm_mu);
    if (!g_num_sms[dev]) cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    return g_num_sms[dev];
}

// 3-D tiled map: dims {d0, d1, d2} (d0 innermost), byte strides of d1 and d2,
// box {b0, b1, b2}; 128-byte swizzle unless given, out-of-range elements read
// as zero (and are not written by a store).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
              CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_128B) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 5-D tiled map of a triangle-form q / k / v: dims {D, rows, H, N, B} with the
// element strides st = {b, n, h, row}; boxes of 64 elements x 128 rows.
bool make_map5(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t D, uint64_t rows, const AttnParams& a,
               const long long (&st)[4]) {
    cuuint64_t dims[5] = {D, rows, (cuuint64_t)a.H, (cuuint64_t)a.N, (cuuint64_t)a.B};
    cuuint64_t strides[4] = {(cuuint64_t)st[3] * 2, (cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
    cuuint32_t box[5] = {64, 128, 1, 1, 1};
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(m, dt, 5, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Instruction descriptor of kind::f16: D fp32 at [4,6), A/B type at [7,10) /
// [10,13) (0 f16, 1 bf16), B major at bit 16 (0 K-major, 1 MN-major), N>>3
// at [17,23), M>>4 at [24,29).
uint32_t make_idesc(bool bf16, int M, int N, bool b_mn_major) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

constexpr size_t kSmemLimit = 232448;  // 227 KB: the per-block opt-in maximum

// Pick NQ and the pipeline depths: two query tiles per CTA when they fit,
// then as many Q buffers, K/V stages and bias stages as shared memory allows.
// The MMA issues PV of a tile after waiting for the next tile's K/V, so two
// K/V stages are the minimum.  The packed form always uses two query tiles.
bool choose_geometry(TcParams& P, bool varlen, int& NQ) {
    // (Q buffers, K/V stages, bias stages per query tile), in order of preference
    const int prefs[][3] = {{2, 3, 2}, {2, 3, 1}, {2, 2, 2}, {2, 2, 1}, {1, 3, 2}, {1, 3, 1}, {1, 2, 2}, {1, 2, 1}};
    for (int nq = 2; nq >= (varlen ? 2 : 1); --nq) {
        const uint32_t cols = nq * 128 + nq * P.o_cols;
        if (cols > 512) continue;
        for (const auto& pr : prefs) {
            P.q_bufs = pr[0];
            P.kv_stages = pr[1];
            P.bias_stages = varlen ? 0 : pr[2];
            if (make_layout(nq, P).total + 1024 <= kSmemLimit) {
                NQ = nq;
                P.o_col0 = nq * 128;
                P.tmem_cols = 32;
                while (P.tmem_cols < cols) P.tmem_cols <<= 1;
                return true;
            }
        }
    }
    return false;
}

// The key-split kernel (triangle form with D <= 64, packed form with D <=
// 128): one query tile per item; S buffers (three for the triangle form, two
// for the packed form) and two O accumulator sets when the remaining columns
// hold them (else one), in 512 tensor-memory columns; Q buffers, K/V stages and
// bias stages as shared memory allows.
bool choose_split_geometry(TcParams& P, bool varlen) {
    const int prefs[][3] = {{2, 3, 2}, {2, 3, 1}, {2, 2, 2}, {2, 2, 1}, {1, 2, 2}, {1, 2, 1}, {1, 1, 1}};
    P.s_bufs = varlen ? 2 : 3;
    // The columns after the S buffers hold O: packed form, one O of o_cols per set; triangle
    // form, one per key half (two per set)
    const uint32_t per_set = (varlen ? 1u : 2u) * P.o_cols;
    const uint32_t avail = 512u - 128u * (uint32_t)P.s_bufs;
    P.o_bufs = per_set * 2 <= avail ? 2 : 1;
    if (per_set > avail) return false;
    for (const auto& pr : prefs) {
        P.q_bufs = pr[0];
        P.kv_stages = pr[1];
        P.bias_stages = (varlen && !P.a.bias) ? 0 : pr[2];
        if (make_split_layout(P).total + 1024 <= kSmemLimit) {
            P.o_col0 = 128u * (uint32_t)P.s_bufs;
            P.tmem_cols = 512;
            return true;
        }
    }
    return false;
}

template <bool VARLEN, bool BF16, bool BIAS_F32, bool FOLD>
cudaError_t launch_nq(int NQ, const TcParams& P, int grid, cudaStream_t stream) {
    if constexpr (VARLEN) {
        return NQ == 2 ? launch_kernel<2, true, BF16, false, FOLD>(P, grid, stream) : cudaErrorInvalidConfiguration;
    } else {
        return NQ == 2 ? launch_kernel<2, false, BF16, BIAS_F32, FOLD>(P, grid, stream)
                       : launch_kernel<1, false, BF16, BIAS_F32, FOLD>(P, grid, stream);
    }
}

}  // namespace

// Shared with the backward (tc_bwd.cu): a 3-D tensor map through the driver
// entry point, and the SM count of the current device.
bool encode_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw) {
    return get_encode() && make_map(m, dt, ptr, d0, d1, d2, s1, s2, b0, b1, b2, sw);
}
int device_sm_count() { return num_sms(); }

}  // namespace tc

cudaError_t launch_tc_fwd(const AttnParams& a, cudaStream_t stream) {
    using namespace tc;
    if (!get_encode()) return cudaErrorNotSupported;
    const bool bf16 = a.dtype == TA_BF16;
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    TcParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    const int D = a.D;
    P.nsub = D > 64 ? 2 : 1;
    P.ksteps = (D + 15) / 16;
    P.npv = D > 64 ? 128 : ((D + 15) / 16) * 16;
    P.o_cols = P.npv;
    P.tile_bytes = P.nsub * kBox;
    P.idesc_qk = make_idesc(bf16, 128, 128, false);
    P.idesc_pv = make_idesc(bf16, 128, P.npv, true);
    P.scale_log2e = a.scale * kLog2e;
    const uint64_t rs = (uint64_t)D * 2;
    bool fold;
    if (!a.varlen) {
        const uint64_t eb = a.bias_f32 ? 4 : 2;
        P.bias_box_cols = a.bias_f32 ? 32 : 64;
        P.bias_boxes = kBN / P.bias_box_cols;
        P.bias_bytes = P.bias_boxes * kBox;
        P.mask_kind = a.kv_len ? 1 : (a.mask ? 2 : 0);
        // Contiguous q / k / v (strides {N*H*rows*D, H*rows*D, rows*D, D}) keep 3-D maps over the
        // (b, n, h) slabs; strided views take 5-D maps.
        auto contiguous = [&](const long long (&st)[4], int rows) {
            return st[3] == D && st[2] == (long long)rows * D && st[1] == st[2] * a.H && st[0] == st[1] * a.N;
        };
        P.tri5d = !(contiguous(a.qs, a.Q) && contiguous(a.ks, a.K) && contiguous(a.vs, a.K));
        const uint64_t units = (uint64_t)a.B * a.N * a.H;
        const bool maps_ok =
            P.tri5d ? make_map5(&P.tm_q, dt, a.q, D, a.Q, a, a.qs) && make_map5(&P.tm_k, dt, a.k, D, a.K, a, a.ks) &&
                          make_map5(&P.tm_v, dt, a.v, D, a.K, a, a.vs)
                    : make_map(&P.tm_q, dt, a.q, D, a.Q, units, rs, rs * a.Q, 64, kBM, 1) &&
                          make_map(&P.tm_k, dt, a.k, D, a.K, units, rs, rs * a.K, 64, kBN, 1) &&
                          make_map(&P.tm_v, dt, a.v, D, a.K, units, rs, rs * a.K, 64, kBN, 1);
        if (!maps_ok ||
            !make_map(&P.tm_bias, a.bias_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, a.bias, a.K, a.Q,
                      (uint64_t)a.B * a.H, a.K * eb, a.K * eb * a.Q, P.bias_box_cols, kBM, 1))
            return cudaErrorInvalidValue;
        P.nqt = (a.Q + kBM - 1) / kBM;
        fold = false;  // the bias is added in the softmax
        // O rows of 32, 64 or 128 bytes (D = 16, 32, 64) leave through a TMA store
        // (rows past Q are clipped by the map); other D store rows directly.
        if (D == 16 || D == 32 || D == 64) {
            const CUtensorMapSwizzle sw = D == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                  : (D == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
            P.o_tma = make_map(&P.tm_o, dt, a.out, D, a.Q, units, rs, rs * a.Q, D, 32, 1, sw) ? 1 : 0;
            P.o_rowb = (int)rs;
        }
    } else {
        const uint64_t tk = a.total_k > 0 ? a.total_k : 1;
        // Rows of the packed (total, H, D) views are q_rs / k_rs / v_rs elements apart.
        if (!make_map(&P.tm_q, dt, a.q, D, a.H, a.total_q, rs, 2 * (uint64_t)a.q_rs, 64, 1, kBM) ||
            !make_map(&P.tm_k, dt, a.k, D, a.H, tk, rs, 2 * (uint64_t)a.k_rs, 64, 1, kBN) ||
            !make_map(&P.tm_v, dt, a.v, D, a.H, tk, rs, 2 * (uint64_t)a.v_rs, 64, 1, kBN))
            return cudaErrorInvalidValue;
        P.nqt = (a.max_q + kBM - 1) / kBM;
        fold = a.scale > 0.f && std::isfinite(a.scale) && !a.bias;  // a bias is added after the scale
        if (a.bias) {
            // post-scale bias (H, max_seqlen_q, max_seqlen_k), read as (K, Q, H) boxes
            const uint64_t eb = a.bias_f32 ? 4 : 2;
            P.bias_box_cols = a.bias_f32 ? 32 : 64;
            P.bias_boxes = kBN / P.bias_box_cols;
            P.bias_bytes = P.bias_boxes * kBox;
            if (!make_map(&P.tm_bias, a.bias_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, a.bias, a.max_k, a.max_q,
                          a.H, a.max_k * eb, a.max_k * eb * a.max_q, P.bias_box_cols, kBM, 1))
                return cudaErrorInvalidValue;
        }
    }
    int NQ = 1;
    // Triangle form with D <= 64, and packed sequences whose offsets fit the
    // key-split kernel's schedule, run on the key-split kernel.
    // (a packed problem with a bias always takes the key-split kernel)
    const bool split = a.varlen ? (a.num_seqs <= kSplitMaxSeqs || a.bias) : D <= 64;
    if (a.varlen && a.bias && a.num_seqs > kSplitMaxSeqs) return cudaErrorNotSupported;
    if (split ? !choose_split_geometry(P, a.varlen != 0) : !choose_geometry(P, a.varlen != 0, NQ))
        return cudaErrorInvalidConfiguration;
    P.items_per_unit = (P.nqt + NQ - 1) / NQ;
    const long long units = !a.varlen ? (long long)a.B * a.N * a.H : (long long)a.num_seqs * a.H;
    const long long items = units * P.items_per_unit;  // packed form: an upper bound (empty q blocks included)
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    P.items = (int)items;
    // Divisors of the work-item decode (each at least 1; with no items nothing is launched).
    P.fd_ipu = make_fastdiv((uint32_t)(P.items_per_unit > 0 ? P.items_per_unit : 1));
    P.fd_h = make_fastdiv((uint32_t)(a.H > 0 ? a.H : 1));
    P.fd_n = make_fastdiv((uint32_t)(!a.varlen && a.N > 0 ? a.N : 1));
    P.fd_per = make_fastdiv((uint32_t)(a.varlen && units > 0 ? units : 1));
    const int sms = num_sms();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = P.items < sms ? P.items : sms;
    if (grid <= 0) return cudaSuccess;
    P.fd_2g = make_fastdiv(2u * (uint32_t)grid);

    if (a.varlen && split && a.bias) {
        if (bf16) return a.bias_f32 ? launch_split<true, true, true, false, true>(P, grid, stream)
                                    : launch_split<true, false, true, false, true>(P, grid, stream);
        return a.bias_f32 ? launch_split<false, true, true, false, true>(P, grid, stream)
                          : launch_split<false, false, true, false, true>(P, grid, stream);
    }
    if (a.varlen && split) {
        if (bf16) return fold ? launch_split<true, false, true, true, false>(P, grid, stream)
                              : launch_split<true, false, true, false, false>(P, grid, stream);
        return fold ? launch_split<false, false, true, true, false>(P, grid, stream)
                    : launch_split<false, false, true, false, false>(P, grid, stream);
    }
    if (a.varlen) {
        if (bf16) return fold ? launch_nq<true, true, false, true>(NQ, P, grid, stream)
                              : launch_nq<true, true, false, false>(NQ, P, grid, stream);
        return fold ? launch_nq<true, false, false, true>(NQ, P, grid, stream)
                    : launch_nq<true, false, false, false>(NQ, P, grid, stream);
    }
    (void)fold;
    if (split) {
        if (bf16) return a.bias_f32 ? launch_split<true, true, false, false, true>(P, grid, stream)
                                    : launch_split<true, false, false, false, true>(P, grid, stream);
        return a.bias_f32 ? launch_split<false, true, false, false, true>(P, grid, stream)
                          : launch_split<false, false, false, false, true>(P, grid, stream);
    }
    if (bf16) return a.bias_f32 ? launch_nq<false, true, true, false>(NQ, P, grid, stream)
                                : launch_nq<false, true, false, false>(NQ, P, grid, stream);
    return a.bias_f32 ? launch_nq<false, false, true, false>(NQ, P, grid, stream)
                      : launch_nq<false, false, false, false>(NQ, P, grid, stream);
}

}  // namespace triattn
