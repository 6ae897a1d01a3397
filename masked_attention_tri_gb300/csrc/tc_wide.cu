// tc_wide.cu -- the triangle-form forward for 16-bit q/k/v with D in (128, 256] on
// tcgen05 tensor cores (cuEquivariance triangle_attention page, Notes: the forward
// takes hidden dimensions up to 256).
//
// Same arithmetic as the other forward kernels (x = s Q.K + bias at valid keys, -1e9
// at masked ones, no weight at keys past K; online softmax with a lazy O correction;
// O / l, lse = m + ln l, max), with tiles sized for wide heads: a 128-row Q tile
// (D up to 256: four 64-column boxes, 64 KB) stays in shared memory for the work
// item, and the keys stream in tiles of 64 (K and V tiles of 64 rows x D, two stages
// each), so they fit next to Q and the bias.
//   S  = Q K^T  M = 128 rows, N = 64 keys, K-major A and B           TMEM [64 b, +64), b = tile % 2
//   O += P V    A = P from TMEM (over S), B = V read MN-major, N = D  TMEM [128, 128 + D16)
// Warps 0-3: one thread per query row (TMEM lane): logits, masks, softmax, P, and the
// item's epilogue; warp 4: TMA of Q, K, V, the bias tiles and the dense-mask bits;
// warp 5: the MMAs (one elected lane issues).  One persistent CTA per SM, work items
// (query tile, n, h, b) dealt round-robin with the query tile fastest.  Every wait is
// bounded (TA_ERR_TIMEOUT).

#include "tc_split.cuh"

namespace triattn {
namespace tc {
namespace {

constexpr int kWN = 64;                  // keys per tile
constexpr int kWThreads = 6 * 32;
constexpr uint32_t kQBox = 128u * 128u;  // a Q box: 128 rows x 128 bytes
constexpr uint32_t kKBox = 64u * 128u;   // a K / V box: 64 rows x 128 bytes

struct WideParams {
    CUtensorMap tm_q, tm_k, tm_v, tm_bias;
    AttnParams a;
    int nqt, items;
    int nsub;             // 64-column boxes of D
    int dpad;             // D rounded up to 16 (the PV N and the O columns)
    int ksteps;           // dpad / 16
    int mask_kind;        // 0 none, 1 kv_lengths, 2 dense mask
    int bias_boxes;       // bias boxes per tile: 1 (16-bit, 64 keys) or 2 (fp32, 32 keys each)
    int bias_box_cols;    // keys per bias box
    int bias_stages;      // 1 or 2
    uint32_t bias_bytes;  // one stage: bias_boxes x 128 rows x 128 bytes
    uint32_t idesc_qk, idesc_pv;
    uint32_t tmem_cols;
    FastDiv fd_q, fd_n, fd_h;
};

struct WideLayout {
    uint32_t q, k, v, bias, maskw, bars, tmem_slot, abort_flag, total;
};
// q_full, q_empty, k_full[2], k_empty[2], v_full[2], v_empty[2], b_full[2], b_empty[2],
// s_full[2], p_full[2], pv_done[2], o_free, drain
constexpr int kWideBars = 22;
__host__ __device__ inline WideLayout wide_layout(const WideParams& P) {
    WideLayout L;
    L.q = 0;
    L.k = L.q + (uint32_t)P.nsub * kQBox;
    L.v = L.k + 2u * (uint32_t)P.nsub * kKBox;
    L.bias = L.v + 2u * (uint32_t)P.nsub * kKBox;
    L.maskw = L.bias + (uint32_t)P.bias_stages * P.bias_bytes;  // 64 key bits per bias stage
    L.bars = L.maskw + 16u * (uint32_t)P.bias_stages;
    L.tmem_slot = L.bars + 8u * kWideBars;
    L.abort_flag = L.tmem_slot + 4;
    L.total = L.abort_flag + 4;
    return L;
}

// One work item: the slab (b, n, h), its query tile and the key tiles it visits.
struct WItem {
    long long unit, bn;
    int b, h, qt, nkt, prefix;
};
__device__ __forceinline__ WItem wide_decode(const WideParams& P, int item) {
    const AttnParams& a = P.a;
    WItem it;
    const uint32_t u2 = P.fd_q.div((uint32_t)item);  // (b*H + h)*N + n, the query tile fastest
    it.qt = item - (int)(u2 * P.fd_q.d);
    const uint32_t bh = P.fd_n.div(u2);
    const int n = (int)(u2 - bh * P.fd_n.d);
    it.b = (int)P.fd_h.div(bh);
    it.h = (int)(bh - (uint32_t)it.b * P.fd_h.d);
    it.bn = (long long)it.b * a.N + n;
    it.unit = it.bn * a.H + it.h;
    it.nkt = (a.K + kWN - 1) / kWN;
    it.prefix = a.K;
    if (P.mask_kind == 1) {
        // Key tiles past the prefix are skipped; with no valid key every tile is visited
        // (every logit -1e9: uniform weights over all K keys).
        const int Lk = a.kv_len[it.bn];
        it.prefix = Lk < 0 ? 0 : (Lk > a.K ? a.K : Lk);
        if (it.prefix > 0) it.nkt = (it.prefix + kWN - 1) / kWN;
    }
    return it;
}

template <bool BF16, bool BIAS_F32>
__global__ void __launch_bounds__(kWThreads, 1) tc_wide_kernel(const __grid_constant__ WideParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const WideLayout L = wide_layout(P);
    const AttnParams& a = P.a;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L.abort_flag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.tmem_slot);
    auto bar = [&](int i) { return base + L.bars + 8u * (uint32_t)i; };
    const uint32_t q_full = bar(0), q_empty = bar(1);
    auto k_full = [&](int s) { return bar(2 + s); };
    auto k_empty = [&](int s) { return bar(4 + s); };
    auto v_full = [&](int s) { return bar(6 + s); };
    auto v_empty = [&](int s) { return bar(8 + s); };
    auto b_full = [&](int s) { return bar(10 + s); };
    auto b_empty = [&](int s) { return bar(12 + s); };
    auto s_full = [&](int s) { return bar(14 + s); };
    auto p_full = [&](int s) { return bar(16 + s); };
    auto pv_done = [&](uint32_t g) { return bar(18 + (int)(g & 1u)); };  // PV g: phase g / 2 of barrier g % 2
    const uint32_t o_free = bar(20), drain = bar(21);
    auto k_smem = [&](int s) { return base + L.k + (uint32_t)s * (uint32_t)P.nsub * kKBox; };
    auto v_smem = [&](int s) { return base + L.v + (uint32_t)s * (uint32_t)P.nsub * kKBox; };
    auto b_smem = [&](int s) { return base + L.bias + (uint32_t)s * P.bias_bytes; };
    const int BS = P.bias_stages;

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
            mbar_init(b_full(s), 1);
            mbar_init(b_empty(s), 4);  // one arrival per softmax warp
            mbar_init(s_full(s), 1);
            mbar_init(p_full(s), 4);
            mbar_init(pv_done(s), 1);
        }
        mbar_init(o_free, 4);
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(P.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tO = tmem + 128u;  // O: dpad columns after the two S buffers

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        bool ok = true;
        uint32_t g = 0, bt = 0;  // key tiles so far (K / V stage g % 2), bias tiles so far
        int items_done = 0;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x, ++items_done) {
            const WItem it = wide_decode(P, item);
            if (items_done > 0) {  // every QK^T of the previous item has read Q
                ok = __all_sync(0xffffffffu, wait_bar(q_empty, (uint32_t)(items_done - 1) & 1u, abort_flag, a.status));
                if (!ok) break;
            }
            if (lane == 0) {
                mbar_expect_tx(q_full, (uint32_t)P.nsub * kQBox);
                for (int bx = 0; bx < P.nsub; ++bx)
                    tma_load_3d(base + L.q + (uint32_t)bx * kQBox, &P.tm_q, 64 * bx, it.qt * kBM, (int)it.unit, q_full);
            }
            for (int t = 0; t < it.nkt && ok; ++t, ++g, ++bt) {
                const int st = (int)(g & 1u);
                const int k0 = t * kWN;
                if (g >= 2) {  // stage st held tile g - 2: its QK^T read K, its PV read V
                    ok = __all_sync(0xffffffffu, wait_bar(k_empty(st), ((g >> 1) - 1u) & 1u, abort_flag, a.status));
                    if (!ok) break;
                }
                if (lane == 0) {
                    mbar_expect_tx(k_full(st), (uint32_t)P.nsub * kKBox);
                    for (int bx = 0; bx < P.nsub; ++bx)
                        tma_load_3d(k_smem(st) + (uint32_t)bx * kKBox, &P.tm_k, 64 * bx, k0, (int)it.unit, k_full(st));
                }
                if (g >= 2) {
                    ok = __all_sync(0xffffffffu, wait_bar(v_empty(st), ((g >> 1) - 1u) & 1u, abort_flag, a.status));
                    if (!ok) break;
                }
                if (lane == 0) {
                    mbar_expect_tx(v_full(st), (uint32_t)P.nsub * kKBox);
                    for (int bx = 0; bx < P.nsub; ++bx)
                        tma_load_3d(v_smem(st) + (uint32_t)bx * kKBox, &P.tm_v, 64 * bx, k0, (int)it.unit, v_full(st));
                }
                const int bs = (int)(bt % (uint32_t)BS);
                if (bt >= (uint32_t)BS) {  // the softmax has read bias stage bs
                    ok = __all_sync(0xffffffffu,
                                    wait_bar(b_empty(bs), ((bt / (uint32_t)BS) - 1u) & 1u, abort_flag, a.status));
                    if (!ok) break;
                }
                if (P.mask_kind == 2) {
                    // 64 key-validity bits: word w, bit l <-> key k0 + 32 w + l
                    uint32_t* mw = reinterpret_cast<uint32_t*>(gbase + L.maskw + (uint32_t)bs * 16u);
                    for (int ww = 0; ww < 2; ++ww) {
                        const int key = k0 + 32 * ww + lane;
                        const bool v = key < a.K && a.mask[it.bn * a.K + key] != 0;
                        const uint32_t word = __ballot_sync(0xffffffffu, v);
                        if (lane == ww) mw[ww] = word;
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_expect_tx(b_full(bs), P.bias_bytes);
                    for (int bx = 0; bx < P.bias_boxes; ++bx)
                        tma_load_3d(b_smem(bs) + (uint32_t)bx * kQBox, &P.tm_bias, k0 + bx * P.bias_box_cols,
                                    it.qt * kBM, it.b * a.H + it.h, b_full(bs));
                }
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 5) {
        // ----------------------------------------------------------------- MMA
        // Per item: QK^T of its first two key tiles, then for each tile t: PV of t once
        // P(t) is in TMEM, and QK^T of t + 2 into the S buffer PV(t) read (the tensor core
        // runs them in order).  The item's first PV waits until the previous item's O is
        // read out; Q is released once the item's last QK^T is issued.
        const bool leader = elect_one();
        bool ok = true;
        uint32_t g = 0;  // key tiles so far (S buffer and K / V stage g % 2)
        int items_done = 0;
        // K-major SW128 operands: k step kk reads elements [16 kk, 16 kk + 16) of D, in box
        // kk / 4 (boxes 16 KB apart for Q, 8 KB for K), 32 bytes per step within a box.
        const uint64_t qd = sw128_desc(base + L.q, 16, 1024);
        auto qk = [&](uint32_t gg) -> bool {
            const int st = (int)(gg & 1u);
            if (!__all_sync(0xffffffffu, wait_bar(k_full(st), (gg >> 1) & 1u, abort_flag, a.status))) return false;
            tc_fence_after();
            const uint64_t kd = sw128_desc(k_smem(st), 16, 1024);
            if (leader) {
#pragma unroll 1
                for (int kk = 0; kk < P.ksteps; ++kk)
                    mma_ss(tmem + 64u * (uint32_t)st, qd + (uint64_t)((kk >> 2) * (kQBox >> 4) + (kk & 3) * 2),
                           kd + (uint64_t)((kk >> 2) * (kKBox >> 4) + (kk & 3) * 2), P.idesc_qk, kk > 0 ? 1u : 0u);
                mma_commit(s_full(st));
                mma_commit(k_empty(st));
            }
            return true;
        };
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x, ++items_done) {
            const WItem it = wide_decode(P, item);
            ok = __all_sync(0xffffffffu, wait_bar(q_full, (uint32_t)items_done & 1u, abort_flag, a.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t g0 = g;
            for (int t = 0; t < 2 && t < it.nkt && ok; ++t) ok = qk(g0 + (uint32_t)t);
            if (!ok) break;
            if (it.nkt <= 2 && leader) mma_commit(q_empty);  // every QK^T of the item is issued
            for (int t = 0; t < it.nkt && ok; ++t, ++g) {
                const int st = (int)(g & 1u);
                ok = __all_sync(0xffffffffu, wait_bar(p_full(st), (g >> 1) & 1u, abort_flag, a.status));
                if (!ok) break;
                ok = __all_sync(0xffffffffu, wait_bar(v_full(st), (g >> 1) & 1u, abort_flag, a.status));
                if (!ok) break;
                if (t == 0 && items_done > 0) {  // the previous item's O is read out
                    ok = __all_sync(0xffffffffu, wait_bar(o_free, (uint32_t)(items_done - 1) & 1u, abort_flag,
                                                          a.status));
                    if (!ok) break;
                }
                tc_fence_after();
                // V MN-major: 64-column boxes 8 KB apart (LBO), 8-key groups 1 KB apart (SBO),
                // 16 keys (2 KB) per k step; P of the tile over the first 32 columns of its S buffer.
                const uint64_t vd = sw128_desc(v_smem(st), kKBox, 1024);
                if (leader) {
#pragma unroll 1
                    for (int kk = 0; kk < kWN / 16; ++kk)
                        mma_ts(tO, tmem + 64u * (uint32_t)st + 8u * (uint32_t)kk, vd + (uint64_t)kk * 128u, P.idesc_pv,
                               (t > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(pv_done(g));
                    mma_commit(v_empty(st));
                }
                if (t + 2 < it.nkt) {
                    ok = qk(g + 2u);
                    if (ok && t + 2 == it.nkt - 1 && leader) mma_commit(q_empty);
                }
            }
        }
        if (leader) {
            if (!ok) *abort_flag = 1;
            mma_commit(drain);
        }
        wait_bar_drain(drain, 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------------- softmax
        const int r = threadIdx.x;  // query row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        const uint32_t rsw = (uint32_t)(r & 7);  // 128B swizzle: chunk c of row r sits at chunk c ^ (r % 8)
        const float2 scale2 = make_float2(a.scale, a.scale);
        bool ok = true;
        uint32_t g = 0, bt = 0;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const WItem it = wide_decode(P, item);
            const int qrow = it.qt * kBM + r;
            const bool row_ok = qrow < a.Q;
            float m_true = -INFINITY, m_ref = 0.f, l = 0.f;
            for (int t = 0; t < it.nkt && ok; ++t, ++g, ++bt) {
                const int st = (int)(g & 1u);
                const int bs = (int)(bt % (uint32_t)BS);
                ok = __all_sync(0xffffffffu, wait_bar(b_full(bs), (bt / (uint32_t)BS) & 1u, abort_flag, a.status));
                if (!ok) break;
                ok = __all_sync(0xffffffffu, wait_bar(s_full(st), (g >> 1) & 1u, abort_flag, a.status));
                if (!ok) break;
                tc_fence_after();
                const uint32_t s_taddr = tmem + lane_off + 64u * (uint32_t)st;
                float x[64];
                {
                    uint32_t sr[64];
                    tmem_ld_x64(s_taddr, sr);
                    const uint8_t* brow = gbase + (b_smem(bs) - base) + (uint32_t)r * 128u;
                    if constexpr (!BIAS_F32) {
#pragma unroll
                        for (int c = 0; c < 8; ++c) {  // 8 keys per 16-byte chunk
                            const uint4 wv = *reinterpret_cast<const uint4*>(brow + ((((uint32_t)c) ^ rsw) << 4));
                            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 b2 = unpack2<BF16>(ww[e]);
                                const int j = 8 * c + 2 * e;
                                const float2 r2 = __ffma2_rn(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])),
                                                             scale2, b2);
                                x[j] = r2.x;
                                x[j + 1] = r2.y;
                            }
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 16; ++c) {  // 4 keys per 16-byte chunk; boxes of 32 keys
                            const uint4 wv = *reinterpret_cast<const uint4*>(
                                brow + (uint32_t)(c >> 3) * kQBox + ((((uint32_t)c & 7u) ^ rsw) << 4));
                            const int j = 4 * c;
                            const float2 r0 = __ffma2_rn(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])),
                                                         scale2, make_float2(__uint_as_float(wv.x), __uint_as_float(wv.y)));
                            const float2 r1 = __ffma2_rn(
                                make_float2(__uint_as_float(sr[j + 2]), __uint_as_float(sr[j + 3])), scale2,
                                make_float2(__uint_as_float(wv.z), __uint_as_float(wv.w)));
                            x[j] = r0.x;
                            x[j + 1] = r0.y;
                            x[j + 2] = r1.x;
                            x[j + 3] = r1.y;
                        }
                    }
                }
                // Masking (uniform across the warp): per 32 keys, vm bit j = key valid, em bit j = key exists.
                const int k0 = t * kWN;
                if (P.mask_kind == 2 || k0 + kWN > it.prefix) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int kb = k0 + 32 * hh;
                        const uint32_t em = low_bits(a.K - kb);
                        uint32_t vm = em & low_bits(it.prefix - kb);
                        if (P.mask_kind == 2)
                            vm &= *reinterpret_cast<const uint32_t*>(gbase + L.maskw + 16u * (uint32_t)bs + 4u * (uint32_t)hh);
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            x[32 * hh + j] = ((vm >> j) & 1u) ? x[32 * hh + j] : (((em >> j) & 1u) ? kMasked : -INFINITY);
                    }
                }
                __syncwarp();  // every lane has read its bias row and the mask words
                if (lane == 0) mbar_arrive(b_empty(bs));
                // Tile max, then the online update (a new reference only when the max grows by > 2^8).
                float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; j += 8) {
                    m0 = max3(m0, x[j], x[j + 1]);
                    m1 = max3(m1, x[j + 2], x[j + 3]);
                    m2 = max3(m2, x[j + 4], x[j + 5]);
                    m3 = max3(m3, x[j + 6], x[j + 7]);
                }
                const float tm = fmaxf(max3(m0, m1, m2), m3);
                m_true = fmaxf(m_true, tm);
                float alpha = 1.f;
                bool rescale = false;
                if (t == 0) {
                    m_ref = tm;
                    l = 0.f;
                } else {
                    const float m_new = fmaxf(m_ref, tm);
                    const bool need = (m_new - m_ref) * kLog2e > kRescaleLog2;
                    if (__any_sync(0xffffffffu, need)) {
                        rescale = true;
                        alpha = ex2((m_ref - m_new) * kLog2e);
                        l *= alpha;
                        m_ref = m_new;
                    }
                }
                // P (16-bit pairs) over the first 32 columns of the S buffer.  A row with no real
                // logit yet takes weights of exactly 1 at masked keys and 0 at absent ones.
                const bool live = m_ref > kMasked;
                const float2 ul2 = live ? make_float2(kLog2e, kLog2e) : make_float2(1.f, 1.f);
                const float nb = live ? -m_ref * kLog2e : -kMasked;
                const float2 nb2 = make_float2(nb, nb);
                float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float2 y = __ffma2_rn(make_float2(x[2 * j], x[2 * j + 1]), ul2, nb2);
                    const float2 p = make_float2(ex2(y.x), ex2(y.y));
                    if (j & 1) acc1 = __fadd2_rn(acc1, p);
                    else acc0 = __fadd2_rn(acc0, p);
                    pk[j] = pack2<BF16>(p.x, p.y);
                }
                tmem_st_x32(s_taddr, pk);
                l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                if (rescale) {
                    // O holds PV of the previous tile once it completes (PV g - 2 finished before
                    // S(g) did, and P(g) is not given yet, so the parity wait is exact).
                    ok = __all_sync(0xffffffffu, wait_bar(pv_done(g - 1u), ((g - 1u) >> 1) & 1u, abort_flag, a.status));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < P.dpad; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld_x16(tO + lane_off + (uint32_t)c0, o);
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st_x16(tO + lane_off + (uint32_t)c0, o);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(st));
            }
            if (!ok) break;
            // ---- the item's epilogue, once its last PV is in O
            ok = __all_sync(0xffffffffu, wait_bar(pv_done(g - 1u), ((g - 1u) >> 1) & 1u, abort_flag, a.status));
            if (!ok) break;
            tc_fence_after();
            // A row whose visited keys are all masked while tiles past the prefix were not
            // visited (only with a bias at or below -1e9) gets the mean of V over all keys.
            const bool direct = !(m_true > kMasked) && it.nkt * kWN < a.K;
            const long long row0 = it.unit * a.Q + qrow;
            if (row_ok) {
                const float lse = direct ? kMasked + logf((float)a.K) : m_ref + logf(l);
                if (a.lse) a.lse[row0] = lse;
                if (a.mx) a.mx[row0] = direct ? kMasked : m_true;
            }
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint16_t* orow = static_cast<uint16_t*>(a.out) + row0 * a.D;
#pragma unroll 1
            for (int c0 = 0; c0 < P.dpad; c0 += 16) {
                uint32_t o[16];
                tmem_ld_x16(tO + lane_off + (uint32_t)c0, o);
                uint32_t wv[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    wv[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                if (row_ok && !direct) {
                    if (c0 < a.D) *reinterpret_cast<uint4*>(orow + c0) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    if (c0 + 8 < a.D) *reinterpret_cast<uint4*>(orow + c0 + 8) = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_free);
            if (__any_sync(0xffffffffu, direct && row_ok)) {
                const long long n = it.bn - (long long)it.b * a.N;
                const long long v_base = (long long)it.b * a.vs[0] + n * a.vs[1] + (long long)it.h * a.vs[2];
                split_mean_v<BF16>(a, orow, v_base, a.vs[3], a.K, direct && row_ok);
            }
        }
        if (!ok) *abort_flag = 1;
    }

    // ---------------------------------------------------------------- teardown
    if (warp == 4 && lane == 0 && *abort_flag) {
#pragma unroll 1
        for (int i = 0; i < 2000; ++i) __nanosleep(1000);  // TMA loads already issued land first
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P.tmem_cols) : "memory");
    }
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A / B type at [7,10) /
// [10,13) (0 f16, 1 bf16), A major at bit 15 and B major at bit 16 (1 = MN-major),
// N >> 3 at [17,23), M >> 4 at [24,29).
uint32_t wide_idesc(bool bf16, int M, int N, bool a_mn, bool b_mn) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace
}  // namespace tc

// The triangle form with 16-bit inputs, D in (128, 256], contiguous q / k / v.  Returns
// cudaErrorNotSupported for anything else (the caller then runs the CUDA-core kernel).
cudaError_t launch_tc_wide(const AttnParams& a, cudaStream_t stream) {
    using namespace tc;
    if (a.varlen || a.dtype == TA_F32 || a.D <= 128 || a.D > 256 || a.D % 8 != 0 || a.K % 8 != 0 || !a.bias)
        return cudaErrorNotSupported;
    const int D = a.D;
    auto contiguous = [&](const long long (&st)[4], int rows) {
        return st[3] == D && st[2] == (long long)rows * D && st[1] == st[2] * a.H && st[0] == st[1] * a.N;
    };
    if (!contiguous(a.qs, a.Q) || !contiguous(a.ks, a.K) || !contiguous(a.vs, a.K)) return cudaErrorNotSupported;
    const bool bf16 = a.dtype == TA_BF16;
    const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    WideParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    P.nsub = (D + 63) / 64;
    P.dpad = (D + 15) / 16 * 16;
    P.ksteps = P.dpad / 16;
    P.mask_kind = a.kv_len ? 1 : (a.mask ? 2 : 0);
    P.bias_box_cols = a.bias_f32 ? 32 : 64;
    P.bias_boxes = kWN / P.bias_box_cols;
    P.bias_bytes = (uint32_t)P.bias_boxes * kQBox;
    const uint64_t units = (uint64_t)a.B * a.N * a.H;
    const uint64_t rs = (uint64_t)D * 2, eb = a.bias_f32 ? 4 : 2;
    const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
    if (!encode_map_3d(&P.tm_q, dt, a.q, D, a.Q, units, rs, rs * a.Q, 64, kBM, 1, sw) ||
        !encode_map_3d(&P.tm_k, dt, a.k, D, a.K, units, rs, rs * a.K, 64, kWN, 1, sw) ||
        !encode_map_3d(&P.tm_v, dt, a.v, D, a.K, units, rs, rs * a.K, 64, kWN, 1, sw) ||
        !encode_map_3d(&P.tm_bias, a.bias_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, a.bias, a.K, a.Q,
                       (uint64_t)a.B * a.H, a.K * eb, a.K * eb * a.Q, P.bias_box_cols, kBM, 1, sw))
        return cudaErrorInvalidValue;
    P.idesc_qk = wide_idesc(bf16, 128, kWN, false, false);
    P.idesc_pv = wide_idesc(bf16, 128, P.dpad, false, true);
    P.tmem_cols = 512;  // S buffers 128 + O up to 256 columns
    P.bias_stages = 2;
    if (wide_layout(P).total + 1024 > 232448) P.bias_stages = 1;
    if (wide_layout(P).total + 1024 > 232448) return cudaErrorNotSupported;
    P.nqt = (a.Q + kBM - 1) / kBM;
    const long long items = (long long)units * P.nqt;
    if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    P.items = (int)items;
    P.fd_q = make_fastdiv((uint32_t)P.nqt);
    P.fd_n = make_fastdiv((uint32_t)a.N);
    P.fd_h = make_fastdiv((uint32_t)a.H);
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int grid = P.items < sms ? P.items : sms;
    if (grid <= 0) return cudaSuccess;
    const size_t smem = wide_layout(P).total + 1024;
    auto kern = bf16 ? (a.bias_f32 ? tc_wide_kernel<true, true> : tc_wide_kernel<true, false>)
                     : (a.bias_f32 ? tc_wide_kernel<false, true> : tc_wide_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kWThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

}  // namespace triattn
