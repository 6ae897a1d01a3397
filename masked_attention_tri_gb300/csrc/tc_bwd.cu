// tc_bwd.cu -- the backward's per-key-tile gradients on tcgen05 tensor cores
// (16-bit q/k/v with D in {16, 32, 64}, or D % 16 == 0 in (64, 128];
// K % 8 == 0; triangle form; and packed sequences, D as above, with no bias or one as above).
//
// The forward (cuEquivariance triangle_attention page) has its context saved for
// backward.  With P recomputed from the saved lse and delta[q] = sum_k P dP (the
// per-row sums, formed before this kernel), per (b, n, h) slab:
//     dV = P^T dO,  dP = dO V^T,  dS = P (dP - delta) at valid keys (0 at masked),
//     dK = s dS^T Q,  dQ = s dS K,  dBias[b, h] += dS (summed over n).
// One CTA per (slab, 128-key tile), looping over the slab's 128-row query tiles,
// each taken as two halves of 64 queries.  MMAs, with 128 keys on the TMEM lanes:
//     S^T  = K Q_h^T   (A = K, B = Q rows of half h, both K-major)  TMEM [64 h, +64)
//     dP^T = V dO_h^T  (A = V, B = dO rows of half h)                TMEM [128 + 64 h, +64)
//     dV  += P^T dO_h  (A = P^T from TMEM, over S^T; B = dO read MN-major)  TMEM [256, 256 + D)
//     dK  += dS^T Q_h  (A = dS^T from TMEM, over dP^T; B = Q read MN-major) TMEM [256 + D, 256 + 2D)
//     dQ_j = dS K      (per tile: A = dS from shared memory, M = queries, MN-major;
//                       B = K read MN-major)                          TMEM [256 + 2D, 256 + 3D)
// The two halves use separate S^T / dP^T columns, so the tensor core computes one
// half's S^T / dP^T while the compute warps work on the other.  Warps 0-15 (one thread
// per key row = TMEM lane; the four warps w, w + 4, w + 8, w + 12 of a lane quarter take
// 16 queries each of every half) turn S^T and dP^T into P^T and dS^T (16-bit pairs
// written over the columns just read; dS also into shared memory as the A operand of
// dQ) and add dS to the fp32 dBias accumulator (coalesced over keys); between the
// halves of tile j each reads its 16 columns of dQ_{j-1} (one thread per query row)
// and adds them to the fp32 dQ accumulator with a TMA reduce-add, and at the end
// writes its 16 columns of dK and dV.  Warp 16 loads K and V once and, per query tile,
// Q, dO, the rows' lse / delta and the two bias halves (each as soon as the previous
// tile's half is read); warp 17 issues the MMAs.  Every wait is bounded (TA_ERR_TIMEOUT).
// D in (64, 128] (WIDE): every 128-row tile is two 64-column boxes; dV, dK and dQ_j take
// 128 columns each at TMEM [128, 512), leaving one S^T / dP^T buffer (columns [0, 64) and
// [64, 128)) that the halves of a tile take in turn; each compute warp reads out 32
// columns of dQ / dK / dV (16 at a time through its staging rows); the one Q / dO stage
// is filled per query half.
// Packed sequences (VARLEN; tensorplay BlockMask page, Details 3-4: the backward walks the
// q blocks of each kv block): one CTA per (sequence, head, 128-key block).  One warp first
// lists, in shared memory, the q blocks whose full or partial lists hold the key block,
// plus the q blocks with a row that has no valid key (the forward gave such a row the
// mean of V, so it adds 1 / Lk dO to dV at every key); the tile walk above then runs over
// that list, with mask_mod deciding each (query, key) of a partial block.  Rows of a tile
// past the sequence (the next sequence's rows, read through the same maps) have P = 0.

#include "tc_kernel.cuh"

namespace triattn {
namespace tc {
namespace {

struct BwdTc {
    CUtensorMap tm_q, tm_k, tm_v, tm_do, tm_bias, tm_dq;
    const float* lse;
    const float* delta;
    float* dbias_acc;
    const uint8_t* mask;
    const int32_t* kv_len;
    void* dk;
    void* dv;
    int* status;
    float scale;
    int B, N, H, Q, K, D;
    int nkt, nqt, ksteps;
    int nsub;           // 64-column boxes of D (1, or 2 for D in (64, 128])
    uint32_t idesc_s;   // M 128, N 64: K-major A and B
    uint32_t idesc_g;   // M 128, N D: A from TMEM, B MN-major
    uint32_t idesc_q;   // M 128, N D: A and B MN-major in shared memory
    uint32_t bias_bytes;
    int bias_boxes, bias_box_cols;
    int bias_alias;     // 1: the two bias halves share one slot (an fp32 bias with D > 64)
    int qs;             // stages of (Q, dO, lse, delta): 2 when shared memory allows, else 1
    // Packed sequences (VARLEN): q / k / v / dO (total, H, D) and the fp32 dQ accumulator read
    // through (D, total, H) maps, lse / delta (H, total_q), the BlockMask lists, an optional
    // bias (H, max_q, max_k) at local indices (dBias summed over the sequences).
    const int32_t* cu_q;
    const int32_t* cu_k;
    int num_seqs, total_q, total_k, max_q, max_k;
    const int32_t* kv_num;
    const int32_t* kv_idx;
    const int32_t* full_num;
    const int32_t* full_idx;
    int mask_heads, MQ, MK, mask_mod, window, prefix_all;
    const int32_t* prefix_len;
    int qcap;           // entries of the q-block list in shared memory (0: triangle form)
};

// Shared memory (offsets from a 1024-byte aligned base).
// Stage s of the query-tile ring: Q at q + s * 2 tile, dO after it; lse / delta at lse + s * 1024
// (tile = nsub boxes of 128 rows x 128 bytes).
struct BwdLayout {
    uint32_t k, v, q, ds, bias, dqst, lse, qlist, bars, tmem_slot, abort_flag, qn, total;
};
// kv_full, q_full[2], q_empty[2], lse_full[2], bias_full[2], bias_empty[2], s_full[2], p_full[2],
// dq_full, dq_empty, ds_free, fin, drain
constexpr int kBwdBars = 20;
// nsub: the kernel passes its compile-time box count, so that the offsets fold into constants.
__host__ __device__ inline BwdLayout bwd_layout(const BwdTc& P, int nsub) {
    BwdLayout L;
    const uint32_t tile = (uint32_t)nsub * kBox;  // one 128-row tile of D columns
    L.k = 0;
    L.v = L.k + tile;
    L.q = L.v + tile;
    L.ds = L.q + (uint32_t)P.qs * 2 * tile;  // dS as [key][query]: two 64-query boxes
    L.bias = L.ds + 2 * kBox;
    L.dqst = L.bias + (P.bias_alias ? P.bias_bytes / 2u : P.bias_bytes);  // dQ staging: 16 warps x 32 rows x 16 fp32
    L.lse = L.dqst + 16u * 2048u;
    L.qlist = L.lse + (uint32_t)P.qs * 1024u;  // packed form: the q blocks the key tile visits
    L.bars = L.qlist + (((uint32_t)P.qcap * 4u + 15u) & ~15u);
    L.tmem_slot = L.bars + 8 * kBwdBars;
    L.abort_flag = L.tmem_slot + 4;
    L.qn = L.abort_flag + 4;                   // packed form: entries of the q-block list
    L.total = L.qn + 4;
    return L;
}

// TMA reduce-add (fp32 add into global) of a shared-memory box.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* tm, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}

// fp32 add into global memory with no result.  The global state space is explicit: a generic
// atomic could address shared memory, and the compiler would then keep every later shared
// load of the bias tile behind it.
__device__ __forceinline__ void red_add_global(float* p, float v) {
    asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v));
}

__device__ __forceinline__ float bwd_weight(float x, float lse, float inv_k) {
    // A row with every key masked has lse -1e9 in fp32 (its -1e9 + ln K rounds
    // there); its weights are 1 / K.  Any row with a valid key has lse above -1e9 + 100.
    return lse <= kMasked + 64.f ? inv_k : __expf(x - lse);
}

// Warps 0-15 compute (four per TMEM lane quarter), warp 16 loads, warp 17 issues the MMAs.
constexpr int kComputeWarps = 16;
constexpr int kQuarterWarps = kComputeWarps / 4;  // compute warps per TMEM lane quarter
constexpr int kWarpQ = 64 / kQuarterWarps;        // queries of every 64-query half per warp
constexpr int kProducerWarp = kComputeWarps, kMmaWarp = kComputeWarps + 1;
constexpr int kBwdThreads = (kComputeWarps + 2) * 32;

// mask_mod on a partial block (indices local to the sequence): causal k <= q; sliding window
// q - window < k <= q; prefix LM k <= q or k < prefix (tensorplay BlockMask page, Details 2).
__device__ __forceinline__ bool bwd_mod_keep(int mod, int q, int k, int window, int prefix) {
    switch (mod) {
    case TA_MASK_CAUSAL: return k <= q;
    case TA_MASK_SLIDING_WINDOW: return k <= q && k > q - window;
    case TA_MASK_PREFIX_LM: return k <= q || k < prefix;
    default: return true;
    }
}

// WIDE: D in (64, 128] (two 64-column boxes per tile, one S^T / dP^T buffer that the query
// halves take in turn, 32 columns of dQ / dK / dV per compute warp); otherwise D <= 64.
// VARLEN: packed sequences, one CTA per (sequence, head, 128-key block), visiting the q blocks
// whose lists hold the key block (full: every key valid; partial: mask_mod decides) and the
// q blocks with a row that has no valid key (its weights are 1 / Lk at every key).
// HASB: a bias (always in the triangle form; optional with packed sequences).
template <bool BF16, bool BIAS_F32, bool WIDE, bool VARLEN, bool HASB>
__global__ void __launch_bounds__(kBwdThreads, 1) tc_bwd_kernel(const __grid_constant__ BwdTc P) {
    constexpr int kNsub = WIDE ? 2 : 1;   // 64-column boxes per 128-row tile
    constexpr int kCpw = WIDE ? 32 : 16;  // dQ / dK / dV columns per compute warp
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const BwdLayout L = bwd_layout(P, kNsub);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L.abort_flag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.tmem_slot);
    auto bar = [&](int i) { return base + L.bars + 8u * (uint32_t)i; };
    const uint32_t kv_full = bar(0);
    auto q_full = [&](int st) { return bar(1 + st); };
    auto q_empty = [&](int st) { return bar(3 + st); };
    auto lse_full = [&](int st) { return bar(5 + st); };
    auto bias_full = [&](int hh) { return bar(7 + hh); };
    auto bias_empty = [&](int hh) { return bar(9 + hh); };
    auto s_full = [&](int hh) { return bar(11 + hh); };
    auto p_full = [&](int hh) { return bar(13 + hh); };
    const uint32_t dq_full = bar(15), dq_empty = bar(16), ds_free = bar(17), fin = bar(18), drain = bar(19);
    constexpr uint32_t tileb = (uint32_t)kNsub * kBox;
    auto q_smem = [&](int st) { return base + L.q + (uint32_t)st * 2u * tileb; };
    auto do_smem = [&](int st) { return base + L.q + (uint32_t)st * 2u * tileb + tileb; };
    // bias rows [64 hh, 64 hh + 64) of the tile: boxes of bias_box_cols keys x 64 rows (8 KB each)
    // An fp32 bias with D > 64: both halves in one slot, used in the order (j, 0), (j, 1), (j + 1, 0).
    constexpr bool kAlias = WIDE && BIAS_F32;
    auto bias_half = [&](int hh) { return base + L.bias + (kAlias ? 0u : (uint32_t)hh * (P.bias_bytes / 2u)); };

    // The key tile's unit.  Triangle form: slab unit = (b*N + n)*H + h, Qn x Kn = Q x K.
    // Packed form: sequence seq and head h, Qn x Kn = its lengths.  Rows go through the maps
    // at (x, qrow0 + q, tz) and (x, krow0 + k, tz); lse / delta at lrow0 + q.
    long long unit = 0, bn = 0, lrow0;
    int k0, h, b = 0, Qn, Kn, qrow0 = 0, krow0 = 0, tz, seq = 0, prefix = 0;
    if constexpr (!VARLEN) {
        unit = blockIdx.x / P.nkt;
        k0 = (int)(blockIdx.x - unit * P.nkt) * kBN;
        h = (int)(unit % P.H);
        bn = unit / P.H;
        b = (int)(bn / P.N);
        Qn = P.Q;
        Kn = P.K;
        tz = (int)unit;
        lrow0 = unit * P.Q;
    } else {
        // key block slowest: under causal lists key block kb visits the q blocks kb.. of its
        // sequence, so the CTAs with the most work are issued first
        const unsigned sh = (unsigned)P.num_seqs * (unsigned)P.H;
        k0 = (int)(blockIdx.x / sh) * kBN;
        seq = (int)((blockIdx.x % sh) / (unsigned)P.H);
        h = (int)(blockIdx.x % (unsigned)P.H);
        const int cq0 = P.cu_q[seq], cq1 = P.cu_q[seq + 1], ck0 = P.cu_k[seq], ck1 = P.cu_k[seq + 1];
        Qn = cq1 - cq0;
        Kn = ck1 - ck0;
        if (Qn > P.max_q || Kn > P.max_k || Qn < 0 || Kn < 0 || cq0 < 0 || ck0 < 0 || cq1 > P.total_q ||
            ck1 > P.total_k) {
            if (threadIdx.x == 0 && k0 == 0 && h == 0) atomicCAS(P.status, 0, kStatusDevice);
            return;
        }
        if (k0 >= Kn) return;
        qrow0 = cq0;
        krow0 = ck0;
        tz = h;
        lrow0 = (long long)h * P.total_q + cq0;
        prefix = P.prefix_len ? P.prefix_len[seq] : P.prefix_all;
    }

    // The bias: triangle form (B, 1, H, Q, K), always present; packed form (H, max_q, max_k),
    // optional.  Rows of dBias are bst floats apart.
    constexpr bool hasb = HASB;
    const int bz = VARLEN ? h : b * P.H + h;
    const long long bst = VARLEN ? P.max_k : P.K;

    if (!VARLEN && P.kv_len) {
        // A key tile wholly past a kv_length of at least 1: its keys have weight 0 in every
        // row (each row has a valid key), so dK = dV = 0 there and nothing reaches dQ or
        // dBias.  (With kv_length 0 every key has weight 1 / K and the tile is computed.)
        int Lk = P.kv_len[bn];
        Lk = Lk < 0 ? 0 : (Lk > P.K ? P.K : Lk);
        if (Lk > 0 && k0 >= Lk) {
            const int rows = P.K - k0 < kBN ? P.K - k0 : kBN;
            const long long n16 = (long long)rows * P.D / 8;  // 16-byte pieces of each tensor
            const long long off = (unit * P.K + k0) * (long long)P.D;
            uint4* dkz = reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.dk) + off);
            uint4* dvz = reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.dv) + off);
            for (long long i = threadIdx.x; i < n16; i += blockDim.x) {
                dkz[i] = make_uint4(0u, 0u, 0u, 0u);
                dvz[i] = make_uint4(0u, 0u, 0u, 0u);
            }
            return;
        }
    }

    // Packed form: the q blocks this key tile visits, as (q block | status << 24) in shared
    // memory (status 1 partial, 2 full, 3 every key masked), built by one warp.
    int nqt = P.nqt;
    const uint32_t* qlist = reinterpret_cast<const uint32_t*>(gbase + L.qlist);
    if constexpr (VARLEN) {
        if (warp == kProducerWarp) {
            uint32_t* qw = reinterpret_cast<uint32_t*>(gbase + L.qlist);
            const int kb = k0 / kBN, nqb = (Qn + kBM - 1) / kBM;
            int cnt = 0;
            for (int qb = 0; qb < nqb && qb < P.qcap; ++qb) {
                int st = 1;  // no lists: every block partial
                if (P.kv_num) {
                    int f = 0;
                    if (qb < P.MQ) {
                        const int hm = P.mask_heads == 1 ? 0 : h;
                        const long long row = ((long long)seq * P.mask_heads + hm) * P.MQ + qb;
                        if (P.full_num) {
                            const int n = min(max(P.full_num[row], 0), P.MK);
                            for (int t = lane; t < n; t += 32)
                                if (P.full_idx[row * P.MK + t] == kb) f = 2;
                        }
                        const int n = min(max(P.kv_num[row], 0), P.MK);
                        for (int t = lane; t < n; t += 32)
                            if (P.kv_idx[row * P.MK + t] == kb && f == 0) f = 1;
                    }
                    st = (int)__reduce_max_sync(0xffffffffu, (unsigned)f);  // full before partial
                }
                if (st == 0) {  // not listed: visited only for rows with no valid key
                    bool fm = false;
#pragma unroll
                    for (int t = 0; t < kBM / 32; ++t) {
                        const int q = qb * kBM + lane + 32 * t;
                        if (q < Qn && P.lse[lrow0 + q] <= kMasked + 64.f) fm = true;
                    }
                    if (__any_sync(0xffffffffu, fm)) st = 3;
                }
                if (st != 0) {
                    if (lane == 0) qw[cnt] = (uint32_t)qb | ((uint32_t)st << 24);
                    ++cnt;
                }
            }
            if (lane == 0) *reinterpret_cast<volatile int*>(gbase + L.qn) = cnt;
        }
        __syncthreads();
        nqt = *reinterpret_cast<volatile int*>(gbase + L.qn);
        if (nqt == 0) {  // no row reaches these keys: dK = dV = 0
            const int rows = Kn - k0 < kBN ? Kn - k0 : kBN, per = P.D / 8;  // 16-byte pieces per row
            for (int i = threadIdx.x; i < rows * per; i += blockDim.x) {
                const long long off = (long long)(krow0 + k0 + i / per) * P.H * P.D + (long long)h * P.D + (i % per) * 8;
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.dk) + off) = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(P.dv) + off) = make_uint4(0u, 0u, 0u, 0u);
            }
            return;
        }
    }
    // the first query row (within the unit) and the status of entry j of the tile walk
    auto tile_q0 = [&](int j) -> int {
        if constexpr (VARLEN) return (int)(qlist[j] & 0xffffffu) * kBM;
        else return j * kBM;
    };
    auto tile_st = [&](int j) -> int {
        if constexpr (VARLEN) return (int)(qlist[j] >> 24);
        else return 2;
    };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(kv_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(q_full(i), 1);      // the expect_tx arrival of Q and dO
            mbar_init(q_empty(i), 1);
            mbar_init(lse_full(i), 1);    // the lse / delta rows written
            mbar_init(bias_full(i), 1);
            mbar_init(bias_empty(i), kComputeWarps);  // every compute warp has read the bias half
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), kComputeWarps);
        }
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, 4 * ((P.D + kCpw - 1) / kCpw));  // the warps that read dQ_j (kCpw columns each)
        mbar_init(ds_free, 1);
        mbar_init(fin, 1);
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_slot))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t D = (uint32_t)P.D;
    // S^T of query half hh at tS + 64 hh, dP^T at tDP + 64 hh (P^T and dS^T written over them in
    // place), then dV, dK and dQ_j.
    // D <= 64: S^T and dP^T of both halves (2 x 64 columns each), then dV, dK, dQ_j (D each).
    // D > 64: one S^T / dP^T buffer (64 + 64 columns) that the halves take in turn, then dV,
    // dK, dQ_j (128 columns each).  buf(hh): the S^T / dP^T buffer of half hh.
    const uint32_t tS = tmem, tDP = tmem + (WIDE ? 64u : 128u);
    const uint32_t tDV = tmem + (WIDE ? 128u : 256u), tDK = tDV + (WIDE ? 128u : D), tDQ = tDK + (WIDE ? 128u : D);
    auto buf = [&](int hh) { return WIDE ? 0 : hh; };
    // the phase of buffer buf(hh) that half hh of query tile j fills
    auto sphase = [&](int j, int hh) { return WIDE ? (uint32_t)(2 * j + hh) & 1u : (uint32_t)j & 1u; };

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        bool ok = true;
        if (lane == 0) {
            mbar_expect_tx(kv_full, 2u * tileb);
            for (int bx = 0; bx < kNsub; ++bx) {
                tma_load_3d(base + L.k + (uint32_t)bx * kBox, &P.tm_k, 64 * bx, krow0 + k0, tz, kv_full);
                tma_load_3d(base + L.v + (uint32_t)bx * kBox, &P.tm_v, 64 * bx, krow0 + k0, tz, kv_full);
            }
        }
        for (int j = 0; j < nqt && ok; ++j) {
            const int q0 = tile_q0(j), st = j % P.qs, use = j / P.qs;
            // This tile's Q / dO, bias half 0 (as soon as the compute warps have read half 0 of
            // tile j - 1), the rows' lse / delta, then bias half 1.  One shared slot (kAlias):
            // half 0 once half 1 of tile j - 1 is read, half 1 once half 0 of this tile is.
            auto bias_load = [&](int hh) -> bool {
                if (!hasb) return true;
                if (kAlias) {
                    if (hh == 0 && j > 0 &&
                        !__all_sync(0xffffffffu, wait_bar(bias_empty(1), (uint32_t)(j - 1) & 1u, abort_flag, P.status)))
                        return false;
                    if (hh == 1 &&
                        !__all_sync(0xffffffffu, wait_bar(bias_empty(0), (uint32_t)j & 1u, abort_flag, P.status)))
                        return false;
                } else if (j > 0 && !__all_sync(0xffffffffu, wait_bar(bias_empty(hh), (uint32_t)(j - 1) & 1u,
                                                                      abort_flag, P.status))) {
                    return false;
                }
                if (lane == 0) {
                    mbar_expect_tx(bias_full(hh), P.bias_bytes / 2u);
                    for (int bx = 0; bx < P.bias_boxes; ++bx)
                        tma_load_3d(bias_half(hh) + (uint32_t)bx * 8192u, &P.tm_bias, k0 + bx * P.bias_box_cols,
                                    q0 + 64 * hh, bz, bias_full(hh));
                }
                return true;
            };
            float lv[kBM / 32], dv[kBM / 32];  // the rows' lse / delta
            if constexpr (WIDE) {
                // One Q / dO stage taken as two half stages (q_full / q_empty (hh)): the rows of
                // half hh are read only by that half's MMAs, so they are reloaded as soon as those
                // are done.  The lse / delta loads go first (in flight during the waits); the
                // rows are written after half 1 of tile j - 1 is done (its compute warps have
                // read the previous rows by then).
#pragma unroll
                for (int t = 0; t < kBM / 32; ++t) {
                    const int q = q0 + lane + 32 * t;
                    lv[t] = q < Qn ? P.lse[lrow0 + q] : 0.f;
                    dv[t] = q < Qn ? P.delta[lrow0 + q] : 0.f;
                }
                for (int hh = 0; hh < 2 && ok; ++hh) {
                    if (j > 0) {
                        ok = __all_sync(0xffffffffu,
                                        wait_bar(q_empty(hh), (uint32_t)(j - 1) & 1u, abort_flag, P.status));
                        if (!ok) break;
                    }
                    if (lane == 0) {
                        mbar_expect_tx(q_full(hh), tileb);  // 64 rows x D of Q and of dO
                        for (int bx = 0; bx < kNsub; ++bx) {
                            const uint32_t o = (uint32_t)bx * kBox + (uint32_t)hh * (kBox / 2u);
                            tma_load_3d(q_smem(0) + o, &P.tm_q, 64 * bx, qrow0 + q0 + 64 * hh, tz, q_full(hh));
                            tma_load_3d(do_smem(0) + o, &P.tm_do, 64 * bx, qrow0 + q0 + 64 * hh, tz, q_full(hh));
                        }
                    }
                    if (hh == 0) ok = bias_load(0);
                }
                if (!ok) break;
            } else {
                if (j >= P.qs) {  // stage st held tile j - qs: its MMAs and its compute are done
                    ok = __all_sync(0xffffffffu,
                                    wait_bar(q_empty(st), (uint32_t)(use - 1) & 1u, abort_flag, P.status));
                    if (!ok) break;
                }
                if (lane == 0) {
                    mbar_expect_tx(q_full(st), 2u * tileb);
                    for (int bx = 0; bx < kNsub; ++bx) {
                        tma_load_3d(q_smem(st) + (uint32_t)bx * kBox, &P.tm_q, 64 * bx, qrow0 + q0, tz, q_full(st));
                        tma_load_3d(do_smem(st) + (uint32_t)bx * kBox, &P.tm_do, 64 * bx, qrow0 + q0, tz,
                                    q_full(st));
                    }
                }
                ok = bias_load(0);
                if (!ok) break;
#pragma unroll
                for (int t = 0; t < kBM / 32; ++t) {  // every load in flight before the first store
                    const int q = q0 + lane + 32 * t;
                    lv[t] = q < Qn ? P.lse[lrow0 + q] : 0.f;
                    dv[t] = q < Qn ? P.delta[lrow0 + q] : 0.f;
                }
            }
            float* lse_s = reinterpret_cast<float*>(gbase + L.lse + (uint32_t)st * 1024u);
            float* del_s = lse_s + 128;
#pragma unroll
            for (int t = 0; t < kBM / 32; ++t) {
                lse_s[lane + 32 * t] = lv[t];
                del_s[lane + 32 * t] = dv[t];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(lse_full(st));  // release: the rows are written
            ok = bias_load(1);
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------------- MMA
        // Per query tile j and half hh (64 queries): S^T and dP^T of (j, hh) into buffer hh;
        // once P^T / dS^T of (j, hh) are written, dV and dK take them, then S^T / dP^T of
        // (j + 1, hh) go into the same buffer (the tensor core runs them in order), so the
        // compute warps find the next half ready.  After half 1, dQ_j = dS K.  With one Q / dO
        // stage, tile j + 1's S^T / dP^T wait until tile j's MMAs are all issued.  WIDE: one
        // S^T / dP^T buffer for (j, 0), (j, 1), (j + 1, 0), ... in turn; Q / dO rows per half.
        const bool leader = elect_one();
        bool ok = __all_sync(0xffffffffu, wait_bar(kv_full, 0, abort_flag, P.status));
        const uint64_t kK = sw128_desc(base + L.k, 16, 1024), vK = sw128_desc(base + L.v, 16, 1024);
        const uint64_t kM = sw128_desc(base + L.k, kBox, 1024), dsM = sw128_desc(base + L.ds, kBox, 1024);
        auto mma1 = [&](int j, int hh) -> bool {
            const int st = j % P.qs;
            if (WIDE || hh == 0) {  // WIDE: each half's rows have their own barrier
                const uint32_t qb = WIDE ? q_full(hh) : q_full(st);
                if (!__all_sync(0xffffffffu, wait_bar(qb, (uint32_t)(j / P.qs) & 1u, abort_flag, P.status)))
                    return false;
                tc_fence_after();
            }
            // rows 64 hh .. 64 hh + 63 of the K-major Q / dO tiles: 8 KB on (a whole number of swizzle
            // atoms); k step kk reads D elements [16 kk, 16 kk + 16): box kk / 4, 32 bytes per step.
            const uint64_t qK = sw128_desc(q_smem(st), 16, 1024) + 512u * (uint32_t)hh;
            const uint64_t doK = sw128_desc(do_smem(st), 16, 1024) + 512u * (uint32_t)hh;
            const uint32_t b = (uint32_t)buf(hh);
            if (leader) {
                if constexpr (WIDE) {
#pragma unroll 1
                    for (int kk = 0; kk < P.ksteps; ++kk) {  // S^T = K Q^T (D / 16 <= 8 k steps)
                        const uint64_t ko = (uint64_t)((kk >> 2) * (kBox >> 4) + (kk & 3) * 2);
                        mma_ss(tS + 64u * b, kK + ko, qK + ko, P.idesc_s, kk > 0 ? 1u : 0u);
                    }
#pragma unroll 1
                    for (int kk = 0; kk < P.ksteps; ++kk) {  // dP^T = V dO^T
                        const uint64_t ko = (uint64_t)((kk >> 2) * (kBox >> 4) + (kk & 3) * 2);
                        mma_ss(tDP + 64u * b, vK + ko, doK + ko, P.idesc_s, kk > 0 ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // S^T = K Q^T (D / 16 <= 4 k steps)
                        if (kk < P.ksteps)
                            mma_ss(tS + 64u * b, kK + 2u * (uint32_t)kk, qK + 2u * (uint32_t)kk, P.idesc_s,
                                   kk > 0 ? 1u : 0u);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // dP^T = V dO^T
                        if (kk < P.ksteps)
                            mma_ss(tDP + 64u * b, vK + 2u * (uint32_t)kk, doK + 2u * (uint32_t)kk, P.idesc_s,
                                   kk > 0 ? 1u : 0u);
                }
                mma_commit(s_full((int)b));
            }
            return true;
        };
        if (ok && nqt > 0) ok = WIDE ? mma1(0, 0) : (mma1(0, 0) && mma1(0, 1));
        for (int j = 0; j < nqt && ok; ++j) {
            const int st = j % P.qs;
            const uint64_t qM = sw128_desc(q_smem(st), kBox, 1024), doM = sw128_desc(do_smem(st), kBox, 1024);
            for (int hh = 0; hh < 2 && ok; ++hh) {
                const uint32_t b = (uint32_t)buf(hh);
                ok = __all_sync(0xffffffffu, wait_bar(p_full((int)b), sphase(j, hh), abort_flag, P.status));
                if (!ok) break;
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {  // 16 queries per k step; P^T / dS^T at 16 kk
                        const uint32_t acc = (j > 0 || hh > 0 || kk > 0) ? 1u : 0u;
                        const uint32_t qs16 = (uint32_t)(4 * hh + kk);  // 16-query step within the tile
                        mma_ts(tDV, tS + 64u * b + 16u * (uint32_t)kk, doM + 128u * qs16, P.idesc_g, acc);
                        mma_ts(tDK, tDP + 64u * b + 16u * (uint32_t)kk, qM + 128u * qs16, P.idesc_g, acc);
                    }
                    if constexpr (WIDE) mma_commit(q_empty(hh));  // the rows of half hh are read
                }
                if (hh == 1) {
                    if (j > 0) {  // the compute warps have read dQ of the previous tile
                        ok = __all_sync(0xffffffffu, wait_bar(dq_empty, (uint32_t)(j - 1) & 1u, abort_flag, P.status));
                        if (!ok) break;
                        tc_fence_after();
                    }
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < kBN / 16; ++kk)  // dQ_j = dS K, 16 keys per k step
                            mma_ss(tDQ, dsM + 128u * (uint32_t)kk, kM + 128u * (uint32_t)kk, P.idesc_q,
                                   kk > 0 ? 1u : 0u);
                        mma_commit(dq_full);
                        mma_commit(ds_free);
                        if constexpr (!WIDE) mma_commit(q_empty(st));
                    }
                }
                if constexpr (WIDE) {  // the single buffer: the other half next (the tensor core runs them in order)
                    if (hh == 0) ok = mma1(j, 1);
                    else if (j + 1 < nqt) ok = mma1(j + 1, 0);
                } else if (j + 1 < nqt) {
                    if (P.qs > 1) ok = mma1(j + 1, hh);
                    else if (hh == 1) ok = mma1(j + 1, 0) && mma1(j + 1, 1);
                }
            }
        }
        if (leader) {
            if (ok) mma_commit(fin);
            else *abort_flag = 1;
            mma_commit(drain);
        }
        wait_bar_drain(drain, 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------------- compute
        const int wq = warp & 3;          // TMEM lane quarter: keys (and later query rows) 32 wq ..
        const int hq = warp >> 2;         // within each 64-query half: queries kWarpQ hq .. + kWarpQ - 1
        const int kr = wq * 32 + lane;    // key row of the tile
        const int key = k0 + kr;
        const bool exists = key < Kn;
        bool valid = exists;
        if (!VARLEN && exists) {
            if (P.kv_len) {
                int Lk = P.kv_len[bn];
                Lk = Lk < 0 ? 0 : (Lk > P.K ? P.K : Lk);
                valid = key < Lk;
            } else if (P.mask) {
                valid = P.mask[bn * P.K + key] != 0;
            }
        }
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float inv_k = 1.f / (float)Kn;
        const uint32_t rsw = (uint32_t)(kr & 7);
        // this key's column in the bias halves: boxes of bias_box_cols keys x 64 rows, 128B-swizzled
        const uint32_t bbox_off = (uint32_t)(kr / P.bias_box_cols) * 8192u;
        const uint32_t bcol_b = (uint32_t)(kr % P.bias_box_cols) * (BIAS_F32 ? 4u : 2u);
        // swizzled byte offset of this key's column in query row r, by r % 8 (128B swizzle)
        uint32_t xo[8];
#pragma unroll
        for (int r8 = 0; r8 < 8; ++r8) xo[r8] = ((((bcol_b >> 4) ^ (uint32_t)r8)) << 4) + (bcol_b & 15u);
        float* dbias_row = P.dbias_acc ? P.dbias_acc + (VARLEN ? (long long)h * P.max_q * P.max_k
                                                               : ((long long)b * P.H + h) * P.Q * (long long)P.K) + key
                                       : nullptr;
        // dQ staging of this warp: 32 rows x 16 fp32 (64-byte rows, 64B-swizzled)
        const uint32_t dq_stage = base + L.dqst + (uint32_t)warp * 2048u;
        const uint32_t qsw = (uint32_t)((lane >> 1) & 3);

        // dQ_j read out (thread = query row 128 j + 32 wq + lane; warp hq takes columns
        // [kCpw hq, kCpw hq + kCpw), none past D) and added into the accumulator.
        auto readout = [&](int jr) -> bool {
            const int dc0 = kCpw * hq;
            if (dc0 >= P.D) return true;
            if (!__all_sync(0xffffffffu, wait_bar(dq_full, (uint32_t)jr & 1u, abort_flag, P.status))) return false;
            tc_fence_after();
            if constexpr (!WIDE) {
                uint32_t o[16];
                tmem_ld_x16(tDQ + lane_off + (uint32_t)dc0, o);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(dq_empty);    // the accumulator is read
                    bulk_wait_read_all();     // the previous reduce has read the staging rows
                }
                __syncwarp();
                const uint32_t rowa = dq_stage + (uint32_t)lane * 64u;
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    st_shared_v4(rowa + ((((uint32_t)g) ^ qsw) << 4), __float_as_uint(__uint_as_float(o[4 * g]) * P.scale),
                                 __float_as_uint(__uint_as_float(o[4 * g + 1]) * P.scale),
                                 __float_as_uint(__uint_as_float(o[4 * g + 2]) * P.scale),
                                 __float_as_uint(__uint_as_float(o[4 * g + 3]) * P.scale));
                fence_async_shared();
                __syncwarp();
                if (lane == 0 && tile_q0(jr) + 32 * wq < Qn) {
                    tma_reduce_add_3d(&P.tm_dq, dq_stage, dc0, qrow0 + tile_q0(jr) + 32 * wq, tz);
                    bulk_commit();
                }
            } else {
                const bool rows = tile_q0(jr) + 32 * wq < Qn;
#pragma unroll 1
                for (int pc = 0; pc < kCpw / 16; ++pc) {  // 16 columns at a time through the staging rows
                    const int d0 = dc0 + 16 * pc;
                    if (d0 >= P.D) break;
                    uint32_t o[16];
                    tmem_ld_x16(tDQ + lane_off + (uint32_t)d0, o);
                    if (pc + 1 == kCpw / 16 || d0 + 16 >= P.D) {  // the accumulator is read
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(dq_empty);
                    }
                    if (lane == 0) bulk_wait_read_all();  // the previous reduce has read the staging rows
                    __syncwarp();
                    const uint32_t rowa = dq_stage + (uint32_t)lane * 64u;
#pragma unroll
                    for (int g = 0; g < 4; ++g)
                        st_shared_v4(rowa + ((((uint32_t)g) ^ qsw) << 4), __float_as_uint(__uint_as_float(o[4 * g]) * P.scale),
                                     __float_as_uint(__uint_as_float(o[4 * g + 1]) * P.scale),
                                     __float_as_uint(__uint_as_float(o[4 * g + 2]) * P.scale),
                                     __float_as_uint(__uint_as_float(o[4 * g + 3]) * P.scale));
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0 && rows) {
                        tma_reduce_add_3d(&P.tm_dq, dq_stage, d0, qrow0 + tile_q0(jr) + 32 * wq, tz);
                        bulk_commit();
                    }
                }
            }
            return true;
        };

        bool ok = true;
        for (int j = 0; j < nqt && ok; ++j) {
            const uint32_t ph = (uint32_t)j & 1u;
            const int q0 = tile_q0(j), st = j % P.qs, tst = tile_st(j);
            const float* lse_s = reinterpret_cast<const float*>(gbase + L.lse + (uint32_t)st * 1024u);
            const float* del_s = lse_s + 128;
            ok = __all_sync(0xffffffffu, wait_bar(lse_full(st), (uint32_t)(j / P.qs) & 1u, abort_flag, P.status));
            if (!ok) break;
            for (int hh = 0; hh < 2 && ok; ++hh) {
                if (hasb) {
                    ok = __all_sync(0xffffffffu, wait_bar(bias_full(hh), ph, abort_flag, P.status));
                    if (!ok) break;
                }
                ok = __all_sync(0xffffffffu, wait_bar(s_full(buf(hh)), sphase(j, hh), abort_flag, P.status));
                if (!ok) break;
                tc_fence_after();
                const uint32_t tSh = tS + 64u * (uint32_t)buf(hh), tDPh = tDP + 64u * (uint32_t)buf(hh);
                // Chunks of 16 queries: ql = the query row within the tile, col = the column in
                // the half's buffers.  P^T and dS^T (16-bit pairs) go over the chunk's first 8
                // columns, which this warp has read already.
                constexpr int CW = 16;
#pragma unroll 1
                for (int c = 0; c < kWarpQ / CW; ++c) {
                    const int ql = 64 * hh + kWarpQ * hq + CW * c;
                    const uint32_t col = (uint32_t)(kWarpQ * hq + CW * c);
                    uint32_t sr[CW], dr[CW];
                    tmem_ld_x16(tSh + lane_off + col, sr);
                    tmem_ld_x16(tDPh + lane_off + col, dr);
                    // The chunk's lse and delta (shared-memory broadcasts, four at a time) and this
                    // key's bias column: query row ql + i lives at bcb + 128 i + xo[i % 8].
                    float ls[CW], dl[CW];
#pragma unroll
                    for (int i = 0; i < CW; i += 4) {
                        const float4 l4 = *reinterpret_cast<const float4*>(lse_s + ql + i);
                        const float4 d4 = *reinterpret_cast<const float4*>(del_s + ql + i);
                        ls[i] = l4.x, ls[i + 1] = l4.y, ls[i + 2] = l4.z, ls[i + 3] = l4.w;
                        dl[i] = d4.x, dl[i + 1] = d4.y, dl[i + 2] = d4.z, dl[i + 3] = d4.w;
                    }
                    const uint8_t* bcb = gbase + (bias_half(hh) - base) + bbox_off + (uint32_t)(ql - 64 * hh) * 128u;
                    const int nq = Qn - (q0 + ql);  // queries of the chunk that exist
                    uint32_t pp[CW / 2], dd[CW / 2];
                    // Packed form, partial block: the chunk is wholly kept when mask_mod keeps every
                    // (query, key) of it (warp-uniform: this warp's 32 keys x the chunk's 16 queries).
                    bool whole = tst == 2;
                    if (VARLEN && tst == 1) {
                        const int kmin = k0 + 32 * wq, kmax = kmin + 31, qmin = q0 + ql, qmax = qmin + CW - 1;
                        switch (P.mask_mod) {
                        case TA_MASK_NONE: whole = true; break;
                        case TA_MASK_CAUSAL: whole = kmax <= qmin; break;
                        case TA_MASK_SLIDING_WINDOW: whole = kmax <= qmin && kmin > qmax - P.window; break;
                        case TA_MASK_PREFIX_LM: whole = kmax <= qmin || kmax < prefix; break;
                        default: whole = false;
                        }
                    }
                    if (__all_sync(0xffffffffu, valid) && nq >= CW && whole) {
                        // Every key of the warp valid and every query of the chunk present: each row
                        // has a valid key, so its lse is a plain log-sum-exp and P = 2^(x log2e - lse log2e).
                        const float2 sl2 = make_float2(P.scale * kLog2e, P.scale * kLog2e);
                        const float2 l2e2 = make_float2(kLog2e, kLog2e);
                        float* dbp = dbias_row ? dbias_row + (long long)(q0 + ql) * bst : nullptr;
#pragma unroll
                        for (int i = 0; i < CW; i += 2) {
                            float2 bv;
                            if (!hasb) {
                                bv = make_float2(0.f, 0.f);
                            } else if constexpr (BIAS_F32) {
                                bv = make_float2(*reinterpret_cast<const float*>(bcb + i * 128 + xo[i & 7]),
                                                 *reinterpret_cast<const float*>(bcb + (i + 1) * 128 + xo[(i + 1) & 7]));
                            } else {
                                const uint32_t b0 = *reinterpret_cast<const unsigned short*>(bcb + i * 128 + xo[i & 7]);
                                const uint32_t b1 =
                                    *reinterpret_cast<const unsigned short*>(bcb + (i + 1) * 128 + xo[(i + 1) & 7]);
                                bv = unpack2<BF16>(b0 | (b1 << 16));
                            }
                            // y = s S log2e + b log2e - lse log2e
                            const float2 nl = __fmul2_rn(make_float2(ls[i], ls[i + 1]), make_float2(-kLog2e, -kLog2e));
                            const float2 y = __ffma2_rn(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])),
                                                        sl2, __ffma2_rn(bv, l2e2, nl));
                            const float2 pr = make_float2(ex2(y.x), ex2(y.y));
                            const float2 ds = __fmul2_rn(
                                pr, __fadd2_rn(make_float2(__uint_as_float(dr[i]), __uint_as_float(dr[i + 1])),
                                               make_float2(-dl[i], -dl[i + 1])));
                            pp[i / 2] = pack2<BF16>(pr.x, pr.y);
                            dd[i / 2] = pack2<BF16>(ds.x, ds.y);
                            if (dbp) {
                                red_add_global(dbp + (long long)i * bst, ds.x);
                                red_add_global(dbp + (long long)(i + 1) * bst, ds.y);
                            }
                        }
                    } else {
                        // Logits first (every read of the bias tile before any reduction into dBias).
                        // Packed form: bit ii of vm = query ql + ii and this key valid (the block's
                        // status; mask_mod on a partial block).
                        uint32_t vm = 0;
#pragma unroll
                        for (int ii = 0; ii < CW; ++ii) {
                            float x = kMasked;
                            if constexpr (VARLEN) {
                                const bool ve = valid && (tst == 2 || (tst == 1 && bwd_mod_keep(P.mask_mod, q0 + ql + ii,
                                                                                              key, P.window, prefix)));
                                if (ve) {
                                    float bv = 0.f;
                                    if (hasb) {
                                        const uint8_t* ba = bcb + ii * 128 + xo[ii & 7];
                                        if constexpr (BIAS_F32) bv = *reinterpret_cast<const float*>(ba);
                                        else bv = unpack2<BF16>((uint32_t)*reinterpret_cast<const unsigned short*>(ba)).x;
                                    }
                                    x = fmaf(P.scale, __uint_as_float(sr[ii]), bv);
                                    vm |= 1u << ii;
                                }
                            } else if (valid) {
                                const uint8_t* ba = bcb + ii * 128 + xo[ii & 7];
                                float bv;
                                if constexpr (BIAS_F32) bv = *reinterpret_cast<const float*>(ba);
                                else bv = unpack2<BF16>((uint32_t)*reinterpret_cast<const unsigned short*>(ba)).x;
                                x = fmaf(P.scale, __uint_as_float(sr[ii]), bv);
                            }
                            sr[ii] = __float_as_uint(x);
                        }
                        // P and dS (dS kept in dr for the dBias reduction).
#pragma unroll
                        for (int i = 0; i < CW; i += 2) {
                            float pv[2], sv[2];
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                const int ii = i + u;
                                const bool live = exists && ii < nq;
                                const bool ve = VARLEN ? ((vm >> ii) & 1u) != 0u : valid;
                                const float p = live ? bwd_weight(__uint_as_float(sr[ii]), ls[ii], inv_k) : 0.f;
                                const float ds = (live && ve) ? p * (__uint_as_float(dr[ii]) - dl[ii]) : 0.f;
                                pv[u] = p;
                                sv[u] = ds;
                                dr[ii] = __float_as_uint(ds);
                            }
                            pp[i / 2] = pack2<BF16>(pv[0], pv[1]);
                            dd[i / 2] = pack2<BF16>(sv[0], sv[1]);
                        }
                        if (dbias_row) {
#pragma unroll
                            for (int ii = 0; ii < CW; ++ii)
                                if (__uint_as_float(dr[ii]) != 0.f)
                                    red_add_global(dbias_row + (long long)(q0 + ql + ii) * bst, __uint_as_float(dr[ii]));
                        }
                    }
                    tmem_st_x8(tSh + lane_off + col, pp);
                    tmem_st_x8(tDPh + lane_off + col, dd);
                    // dS as [key][query] in shared memory (box ql / 64, 16-byte chunks of 8 queries),
                    // once dQ of the previous tile has read it.
                    if (j > 0 && hh == 0 && c == 0) {
                        ok = __all_sync(0xffffffffu, wait_bar(ds_free, (uint32_t)(j - 1) & 1u, abort_flag, P.status));
                        if (!ok) break;
                    }
                    const uint32_t drow = base + L.ds + (uint32_t)(ql / 64) * kBox + (uint32_t)kr * 128u;
#pragma unroll
                    for (int g = 0; g < CW / 8; ++g) {
                        const uint32_t ch = (uint32_t)((ql % 64) / 8 + g);
                        st_shared_v4(drow + ((ch ^ rsw) << 4), dd[4 * g], dd[4 * g + 1], dd[4 * g + 2], dd[4 * g + 3]);
                    }
                }
                if (!ok) break;
                __syncwarp();  // every lane has read its bias values
                if (hasb && lane == 0) mbar_arrive(bias_empty(hh));
                tmem_st_wait();
                fence_async_shared();  // dS in shared memory is read by the tensor core
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(buf(hh)));
                // dQ of the previous tile, between this tile's halves (its MMAs ran meanwhile)
                if (hh == 0 && j > 0) ok = readout(j - 1);
            }
        }
        if (ok && nqt > 0) ok = readout(nqt - 1);
        if (ok) ok = __all_sync(0xffffffffu, wait_bar(fin, 0, abort_flag, P.status));
        if (ok && kCpw * hq < P.D) {  // dK and dV columns [kCpw hq, kCpw hq + kCpw)
            tc_fence_after();
            // triangle form: row unit * K + key of (B, N, H, K, D); packed form: (krow0 + key, h) of (total_k, H, D)
            const long long kofs = VARLEN ? ((long long)(krow0 + key) * P.H + h) * P.D : (unit * P.K + key) * (long long)P.D;
            uint16_t* dkp = static_cast<uint16_t*>(P.dk) + kofs;
            uint16_t* dvp = static_cast<uint16_t*>(P.dv) + kofs;
#pragma unroll 1
            for (int pc = 0; pc < kCpw / 16; ++pc) {
                const int d0 = kCpw * hq + 16 * pc;
                if (WIDE && d0 >= P.D) break;
                uint32_t ov[16], ok16[16];
                tmem_ld_x16(tDV + lane_off + (uint32_t)d0, ov);
                tmem_ld_x16(tDK + lane_off + (uint32_t)d0, ok16);
                uint32_t wv[8], wk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    wv[e] = pack2<BF16>(__uint_as_float(ov[2 * e]), __uint_as_float(ov[2 * e + 1]));
                    wk[e] = pack2<BF16>(__uint_as_float(ok16[2 * e]) * P.scale, __uint_as_float(ok16[2 * e + 1]) * P.scale);
                }
                if (exists) {
                    reinterpret_cast<uint4*>(dvp + d0)[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    reinterpret_cast<uint4*>(dvp + d0)[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                    reinterpret_cast<uint4*>(dkp + d0)[0] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                    reinterpret_cast<uint4*>(dkp + d0)[1] = make_uint4(wk[4], wk[5], wk[6], wk[7]);
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // this warp's dQ reduce-adds are done
        if (!ok) *abort_flag = 1;
    }

    // ---------------------------------------------------------------- teardown
    if (warp == kProducerWarp && lane == 0 && *abort_flag) {
#pragma unroll 1
        for (int i = 0; i < 2000; ++i) __nanosleep(1000);  // TMA loads already issued land first
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
    }
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A / B type at [7,10) /
// [10,13) (0 f16, 1 bf16), A major at bit 15 and B major at bit 16 (1 = MN-major),
// N >> 3 at [17,23), M >> 4 at [24,29).
uint32_t bwd_idesc(bool bf16, int M, int N, bool a_mn, bool b_mn) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace
}  // namespace tc

bool tc_bwd_supported(const BwdParams& p) {
    if (p.dtype == TA_F32) return false;
    const bool d_ok = p.D == 16 || p.D == 32 || p.D == 64 || (p.D % 16 == 0 && p.D > 64 && p.D <= 128);
    if (!d_ok) return false;
    tc::BwdTc t;
    memset(&t, 0, sizeof(t));
    t.nsub = (p.D + 63) / 64;
    t.qs = 1;
    t.D = p.D;
    if (p.varlen) {
        // Packed sequences; the q-block list of the longest sequence must fit beside the tiles.
        // A bias (H, max_q, max_k) is read through a tensor map: its rows must be 16-byte multiples.
        t.qcap = (p.max_q + tc::kBM - 1) / tc::kBM;
        if (p.bias) {
            if (p.max_q <= 0 || p.max_k <= 0 || ((long long)p.max_k * (p.bias_f32 ? 4 : 2)) % 16 != 0) return false;
            t.bias_bytes = (uint32_t)(tc::kBN / (p.bias_f32 ? 32 : 64)) * tc::kBox;
            t.bias_alias = p.D > 64 && p.bias_f32 ? 1 : 0;
        }
        return tc::bwd_layout(t, t.nsub).total + 1024 <= 232448;
    }
    if (p.K % 8 != 0) return false;
    if (p.D <= 64) return true;
    // D in (64, 128]: two-box tiles, one Q / dO stage; an fp32 bias tile fits beside them as
    // one half at a time.
    t.bias_bytes = (uint32_t)(tc::kBN / (p.bias_f32 ? 32 : 64)) * tc::kBox;
    t.bias_alias = p.bias_f32 ? 1 : 0;
    return tc::bwd_layout(t, t.nsub).total + 1024 <= 232448;
}

cudaError_t launch_tc_bwd_main(const BwdParams& p, cudaStream_t stream) {
    using namespace tc;
    if (!tc_bwd_supported(p)) return cudaErrorInvalidValue;
    const bool bf16 = p.dtype == TA_BF16;
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    BwdTc P;
    memset(&P, 0, sizeof(P));
    const int D = p.D;
    const uint64_t units = (uint64_t)p.B * p.N * p.H;
    const uint64_t rs = (uint64_t)D * 2;
    const auto sw128 = CU_TENSOR_MAP_SWIZZLE_128B;
    P.bias_box_cols = p.bias_f32 ? 32 : 64;
    P.bias_boxes = kBN / P.bias_box_cols;
    P.bias_bytes = (uint32_t)P.bias_boxes * kBox;
    P.bias_alias = D > 64 && p.bias_f32 ? 1 : 0;
    const uint64_t eb = p.bias_f32 ? 4 : 2;
    const int qbox = D > 64 ? kBM / 2 : kBM;  // D > 64: Q / dO rows loaded per query half
    const bool vl = p.varlen != 0;
    if (vl && (p.total_q == 0 || p.total_k == 0 || p.num_seqs <= 0)) return cudaSuccess;  // no key rows
    // Packed sequences: (D, total, H) maps over the (total, H, D) rows.
    const uint64_t prs = (uint64_t)p.H * D * 2;
    const bool maps_ok = vl ?
        encode_map_3d(&P.tm_q, dt, p.q, D, p.total_q, p.H, prs, rs, 64, qbox, 1, sw128) &&
        encode_map_3d(&P.tm_do, dt, p.d_out, D, p.total_q, p.H, prs, rs, 64, qbox, 1, sw128) &&
        encode_map_3d(&P.tm_k, dt, p.k, D, p.total_k, p.H, prs, rs, 64, kBN, 1, sw128) &&
        encode_map_3d(&P.tm_v, dt, p.v, D, p.total_k, p.H, prs, rs, 64, kBN, 1, sw128) &&
        encode_map_3d(&P.tm_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dq_acc, D, p.total_q, p.H, (uint64_t)p.H * D * 4,
                      (uint64_t)D * 4, 16, 32, 1, CU_TENSOR_MAP_SWIZZLE_64B) &&
        (!p.bias || encode_map_3d(&P.tm_bias, p.bias_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, p.bias, p.max_k,
                                  p.max_q, p.H, p.max_k * eb, p.max_k * eb * p.max_q, P.bias_box_cols, kBM / 2, 1,
                                  sw128)) :
        encode_map_3d(&P.tm_q, dt, p.q, D, p.Q, units, rs, rs * p.Q, 64, qbox, 1, sw128) &&
        encode_map_3d(&P.tm_do, dt, p.d_out, D, p.Q, units, rs, rs * p.Q, 64, qbox, 1, sw128) &&
        encode_map_3d(&P.tm_k, dt, p.k, D, p.K, units, rs, rs * p.K, 64, kBN, 1, sw128) &&
        encode_map_3d(&P.tm_v, dt, p.v, D, p.K, units, rs, rs * p.K, 64, kBN, 1, sw128) &&
        encode_map_3d(&P.tm_bias, p.bias_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, p.bias, p.K, p.Q,
                      (uint64_t)p.B * p.H, p.K * eb, p.K * eb * p.Q, P.bias_box_cols, kBM / 2, 1, sw128) &&
        encode_map_3d(&P.tm_dq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, p.dq_acc, D, p.Q, units, (uint64_t)D * 4,
                      (uint64_t)D * 4 * p.Q, 16, 32, 1, CU_TENSOR_MAP_SWIZZLE_64B);  // 16 fp32 x 32 rows
    if (!maps_ok) return cudaErrorInvalidValue;
    P.lse = p.lse;
    P.delta = p.delta;
    P.dbias_acc = p.dbias_acc;
    P.mask = p.mask;
    P.kv_len = p.kv_len;
    P.dk = p.dk;
    P.dv = p.dv;
    P.status = status_word();
    if (!P.status) return cudaErrorInvalidValue;
    P.scale = p.scale;
    P.B = p.B;
    P.N = p.N;
    P.H = p.H;
    P.Q = p.Q;
    P.K = p.K;
    P.D = D;
    P.nkt = vl ? (p.max_k + kBN - 1) / kBN : (p.K + kBN - 1) / kBN;
    P.nqt = vl ? 0 : (p.Q + kBM - 1) / kBM;  // packed form: per key tile, from its q-block list
    if (vl) {
        P.bias_bytes = p.bias ? (uint32_t)P.bias_boxes * kBox : 0;  // 0: no bias
        P.dbias_acc = p.bias ? p.dbias_acc : nullptr;
        P.cu_q = p.cu_q;
        P.cu_k = p.cu_k;
        P.num_seqs = p.num_seqs;
        P.total_q = p.total_q;
        P.total_k = p.total_k;
        P.max_q = p.max_q;
        P.max_k = p.max_k;
        P.kv_num = p.kv_num;
        P.kv_idx = p.kv_idx;
        P.full_num = p.full_num;
        P.full_idx = p.full_idx;
        P.mask_heads = p.mask_heads;
        P.MQ = p.MQ;
        P.MK = p.MK;
        P.mask_mod = p.mask_mod;
        P.window = p.window;
        P.prefix_len = p.prefix_len;
        P.prefix_all = p.prefix_all;
        P.qcap = (p.max_q + kBM - 1) / kBM;
    }
    P.ksteps = D / 16;
    P.nsub = (D + 63) / 64;
    P.idesc_s = bwd_idesc(bf16, 128, 64, false, false);  // 64 queries (one half of the tile)
    P.idesc_g = bwd_idesc(bf16, 128, D, false, true);
    P.idesc_q = bwd_idesc(bf16, 128, D, true, true);
    const long long grid = vl ? (long long)p.num_seqs * p.H * P.nkt : (long long)units * P.nkt;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    P.qs = D > 64 ? 1 : 2;  // D > 64: one stage, taken per query half
    if (bwd_layout(P, P.nsub).total + 1024 > 232448) P.qs = 1;  // the 227 KB per-block limit
    const size_t smem = bwd_layout(P, P.nsub).total + 1024;
    // <BF16, BIAS_F32, WIDE, VARLEN, HASB>; the triangle form always has a bias
    const bool fb = p.bias_f32 != 0;
    decltype(&tc_bwd_kernel<true, false, false, false, true>) kern;
    if (!vl)
        kern = D > 64 ? (bf16 ? (fb ? tc_bwd_kernel<true, true, true, false, true> : tc_bwd_kernel<true, false, true, false, true>)
                              : (fb ? tc_bwd_kernel<false, true, true, false, true> : tc_bwd_kernel<false, false, true, false, true>))
             : bf16   ? (fb ? tc_bwd_kernel<true, true, false, false, true> : tc_bwd_kernel<true, false, false, false, true>)
                      : (fb ? tc_bwd_kernel<false, true, false, false, true> : tc_bwd_kernel<false, false, false, false, true>);
    else if (!p.bias)
        kern = D > 64 ? (bf16 ? tc_bwd_kernel<true, false, true, true, false> : tc_bwd_kernel<false, false, true, true, false>)
                      : (bf16 ? tc_bwd_kernel<true, false, false, true, false> : tc_bwd_kernel<false, false, false, true, false>);
    else
        kern = D > 64 ? (bf16 ? (fb ? tc_bwd_kernel<true, true, true, true, true> : tc_bwd_kernel<true, false, true, true, true>)
                              : (fb ? tc_bwd_kernel<false, true, true, true, true> : tc_bwd_kernel<false, false, true, true, true>))
             : bf16   ? (fb ? tc_bwd_kernel<true, true, false, true, true> : tc_bwd_kernel<true, false, false, true, true>)
                      : (fb ? tc_bwd_kernel<false, true, false, true, true> : tc_bwd_kernel<false, false, false, true, true>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)grid, kBwdThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace triattn
