// tc_split.cuh -- tcgen05 / TMA forward, triangle form with D <= 64: one
// 128-row query tile per work item, its softmax split over eight warps, S
// triple-buffered and O double-buffered in tensor memory.  Launched from
// tc_fwd.cu, instantiated in tc_inst_split.cu.  Computes the same
// cuEquivariance triangle_attention formula as tc_kernel.cuh (see there for
// masking and the lazy rescale).
//
// Warp roles:
//   warps 0..7   softmax.  Warp w works on the 32 rows of TMEM lane quarter
//                w % 4 and on key half w / 4 (64 of a tile's 128 keys).  The
//                two warps of a lane quarter swap their half-tile row maxima
//                through shared memory once per tile (an mbarrier with two
//                arrivals), so both use the same reference max; each writes
//                P for its 64 keys and, in the epilogue, its half of O's
//                columns after swapping the partial row sums once per item.
//   warp 8       producer: TMA of Q and K;
//   warp 9       MMA (warp-wide loop, one elected lane issues);
//   warp 10      bias producer: TMA of bias tiles and the dense-mask bits;
//   warp 11      producer: TMA of V.
// The MMA warp walks the CTA's key tiles as one stream across work items:
// S of tile n + 3 goes into the buffer of tile n as soon as PV of tile n is
// issued, also when tile n + 3 belongs to the next item, so the softmax
// finds the next S ready at item boundaries too.  Items alternate between
// two O accumulators, and the softmax writes out an item's O after the first
// tile of the next item, when the last PV of the item has long finished.
// Tensor memory: three S buffers at columns [0,384) (P overwrites the first 64
// columns of its buffer), O_0 and O_1 at [384, 384 + 2 o_cols).  K and V
// stages have their own barriers: a K stage is refilled once its QK^T is done,
// a V stage once its PV is.  The softmax waits for a PV only before it
// rescales O and before it reads O.

#pragma once

#include "tc_kernel.cuh"

namespace triattn {
namespace tc {

constexpr int kSplitThreads = 12 * 32;

struct SplitLayout {
    uint32_t q, kv, bias, maskw, xbuf, xl, bars, tmem_slot, abort_flag, total;
    int nbars;
};

__host__ __device__ inline SplitLayout make_split_layout(const TcParams& P) {
    SplitLayout L;
    L.q = 0;
    L.kv = L.q + P.q_bufs * P.tile_bytes;
    L.bias = L.kv + P.kv_stages * 2 * P.tile_bytes;
    L.maskw = L.bias + P.bias_stages * P.bias_bytes;
    L.xbuf = L.maskw + P.bias_stages * 16;   // row maxima: [tile parity][key half][128 rows] fp32
    L.xl = L.xbuf + 2 * 2 * 128 * 4;           // row sums: [key half][128 rows] fp32
    L.bars = L.xl + 2 * 128 * 4;
    // q_full, q_empty (QB each), k_full, k_empty, v_full, v_empty (S each),
    // bias_full, bias_empty (BS each), s_full[3], p_full[3], pv_done[2],
    // xchg[4], drain
    L.nbars = 2 * P.q_bufs + 4 * P.kv_stages + 2 * P.bias_stages + 3 + 3 + 2 + 4 + 1;
    L.tmem_slot = L.bars + 8 * L.nbars;
    L.abort_flag = L.tmem_slot + 4;
    L.total = L.abort_flag + 4;
    return L;
}

// A position in the CTA's stream of key tiles: the current item with work,
// its key-tile count, the next tile in it and the item's number among the
// CTA's items with work.
struct SplitCursor {
    int item;
    int nkt;
    int t;
    uint32_t qi;
};

// Moves c.item forward (by the grid stride) to the next item with work.
__device__ __forceinline__ bool split_seek(const TcParams& P, SplitCursor& c) {
    for (; c.item < P.items; c.item += gridDim.x) {
        const Item<1> it = decode<1, false>(P, c.item);
        if (it.any) {
            c.nkt = it.nkb;
            c.t = 0;
            return true;
        }
    }
    return false;
}

template <bool BF16, bool BIAS_F32>
__global__ void __launch_bounds__(kSplitThreads, 1) tc_split_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const SplitLayout L = make_split_layout(P);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    constexpr int kProducerWarp = 8;
    constexpr int kMmaWarp = 9;
    constexpr int kBiasWarp = 10;
    constexpr int kVWarp = 11;
    const AttnParams& a = P.a;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L.abort_flag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.tmem_slot);

    const int S = P.kv_stages;
    const int BS = P.bias_stages;
    const int QB = P.q_bufs;
    auto bar = [&](int idx) -> uint32_t { return base + L.bars + 8u * (uint32_t)idx; };
    auto q_full = [&](int qb) { return bar(qb); };
    auto q_empty = [&](int qb) { return bar(QB + qb); };
    auto k_full = [&](int s) { return bar(2 * QB + s); };
    auto k_empty = [&](int s) { return bar(2 * QB + S + s); };
    auto v_full = [&](int s) { return bar(2 * QB + 2 * S + s); };
    auto v_empty = [&](int s) { return bar(2 * QB + 3 * S + s); };
    auto bias_full = [&](int s) { return bar(2 * QB + 4 * S + s); };
    auto bias_empty = [&](int s) { return bar(2 * QB + 4 * S + BS + s); };
    const int bx0 = 2 * QB + 4 * S + 2 * BS;
    auto s_full = [&](int b) { return bar(bx0 + b); };
    auto p_full = [&](int b) { return bar(bx0 + 3 + b); };
    auto pv_done = [&](uint32_t n) { return bar(bx0 + 6 + (int)(n & 1u)); };  // PV n: phase n / 2 of barrier n % 2
    auto xchg = [&](int q) { return bar(bx0 + 8 + q); };
    const uint32_t drain = bar(bx0 + 12);

    auto q_smem = [&](int qb) { return base + L.q + (uint32_t)qb * P.tile_bytes; };
    auto k_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes; };
    auto v_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes + P.tile_bytes; };
    auto bias_smem = [&](int s) { return base + L.bias + (uint32_t)s * P.bias_bytes; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
#pragma unroll 1
        for (int qb = 0; qb < QB; ++qb) {
            mbar_init(q_full(qb), 1);
            mbar_init(q_empty(qb), 1);
        }
#pragma unroll 1
        for (int s = 0; s < S; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
#pragma unroll 1
        for (int s = 0; s < BS; ++s) {
            mbar_init(bias_full(s), 1);
            mbar_init(bias_empty(s), 8);  // one arrival per softmax warp
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 8);  // one arrival per softmax warp
        }
        mbar_init(pv_done(0), 1);
        mbar_init(pv_done(1), 1);
        for (int q = 0; q < 4; ++q) mbar_init(xchg(q), 2);  // the two warps of a lane quarter
        mbar_init(drain, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(P.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ---------------------------------------------------- producer: Q, K tiles
        StageRing kr = {0, 0u, false}, qr = {0, 0u, false};
        bool ok = true;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<1> it = decode<1, false>(P, item);
            if (!it.any) continue;
            const int qb = qr.idx;
            if (lane == 0 && qr.wrapped) ok = wait_bar(q_empty(qb), qr.ph ^ 1u, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(q_full(qb), P.tile_bytes);
                for (int sb = 0; sb < P.nsub; ++sb)
                    tma_load_3d(q_smem(qb) + sb * kBox, &P.tm_q, sb * 64, it.qt[0] * kBM, (int)it.unit, q_full(qb));
            }
            qr.next(QB);
            for (int kb = 0; kb < it.nkb && ok; ++kb) {
                const int st = kr.idx;
                if (lane == 0 && kr.wrapped) ok = wait_bar(k_empty(st), kr.ph ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_expect_tx(k_full(st), P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb)
                        tma_load_3d(k_smem(st) + sb * kBox, &P.tm_k, sb * 64, kb * kBN, (int)it.unit, k_full(st));
                }
                kr.next(S);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kVWarp) {
        // ---------------------------------------------------------- producer: V tiles
        StageRing vr = {0, 0u, false};
        bool ok = true;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<1> it = decode<1, false>(P, item);
            if (!it.any) continue;
            for (int kb = 0; kb < it.nkb && ok; ++kb) {
                const int st = vr.idx;
                if (lane == 0 && vr.wrapped) ok = wait_bar(v_empty(st), vr.ph ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_expect_tx(v_full(st), P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb)
                        tma_load_3d(v_smem(st) + sb * kBox, &P.tm_v, sb * 64, kb * kBN, (int)it.unit, v_full(st));
                }
                vr.next(S);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kBiasWarp) {
        // ---------------------------------- producer: bias tiles (+ dense-mask bits)
        StageRing br = {0, 0u, false};
        bool ok = true;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<1> it = decode<1, false>(P, item);
            if (!it.any) continue;
            for (int kb = 0; kb < it.nkb && ok; ++kb) {
                const int bs = br.idx;
                if (lane == 0 && br.wrapped) ok = wait_bar(bias_empty(bs), br.ph ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (P.mask_kind == 2) {
                    // 128 key-validity bits: word w, bit l <-> key kb*128 + 32w + l
                    uint32_t* mw = reinterpret_cast<uint32_t*>(gbase + L.maskw + (uint32_t)bs * 16u);
                    for (int ww = 0; ww < 4; ++ww) {
                        const int key = kb * kBN + 32 * ww + lane;
                        const bool v = key < a.K && a.mask[it.bn * a.K + key] != 0;
                        const uint32_t word = __ballot_sync(0xffffffffu, v);
                        if (lane == ww) mw[ww] = word;
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    mbar_expect_tx(bias_full(bs), P.bias_bytes);
                    for (int bx = 0; bx < P.bias_boxes; ++bx)
                        tma_load_3d(bias_smem(bs) + bx * kBox, &P.tm_bias, kb * kBN + bx * P.bias_box_cols,
                                    it.qt[0] * kBM, it.b * a.H + it.h, bias_full(bs));
                }
                br.next(BS);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        // Two cursors over the CTA's items with work: `qc` for the next QK^T,
        // `pc` for the next PV.  Tile n of the stream (counted over items) has
        // S buffer n % 3 and K/V stage n % S; item number i has Q buffer i % QB
        // and O accumulator i % 2.
        const bool leader = elect_one();
        SplitCursor qc, pc;
        qc.item = blockIdx.x;
        qc.qi = 0;
        bool has_q = split_seek(P, qc);
        pc = qc;
        bool has_p = has_q;
        uint32_t np = 0;                                    // PV issued so far
        StageRing qr = {0, 0u, false};                      // Q buffer of qc's item
        StageRing kq = {0, 0u, false}, sq = {0, 0u, false};  // K stage / S buffer of the next QK^T
        StageRing vp = {0, 0u, false}, sp = {0, 0u, false};  // V stage / S buffer of the next PV
        bool ok = true;
        auto kstep = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4); };
        auto issue_qk = [&]() -> bool {
            if (!has_q) return true;
            const int qb = qr.idx;
            if (qc.t == 0 && !__all_sync(0xffffffffu, wait_bar(q_full(qb), qr.ph, abort_flag, a.status))) return false;
            const int st = kq.idx;
            if (!__all_sync(0xffffffffu, wait_bar(k_full(st), kq.ph, abort_flag, a.status))) return false;
            tc_fence_after();
            const uint64_t qd = sw128_desc(q_smem(qb), 16, 1024);
            const uint64_t kd = sw128_desc(k_smem(st), 16, 1024);
            const int b = sq.idx;
            const uint32_t sd = tmem + 128u * (uint32_t)b;
            if (leader) {
                mma_ss(sd, qd, kd, P.idesc_qk, 0u);
                for (int kk = 1; kk < P.ksteps; ++kk) mma_ss(sd, qd + kstep(kk), kd + kstep(kk), P.idesc_qk, 1u);
                mma_commit(s_full(b));
                mma_commit(k_empty(st));
            }
            kq.next(S);
            sq.next(3);
            if (++qc.t == qc.nkt) {
                if (leader) mma_commit(q_empty(qb));  // every QK^T of the item is issued
                qr.next(QB);
                ++qc.qi;
                qc.item += gridDim.x;
                has_q = split_seek(P, qc);
            }
            return true;
        };
        for (int i = 0; i < 3 && ok; ++i) ok = issue_qk();
        while (ok && has_p) {
            const int b = sp.idx;
            const int st = vp.idx;
            const bool ready = mbar_test(p_full(b), sp.ph) & mbar_test(v_full(st), vp.ph);
            if (!__all_sync(0xffffffffu, ready)) {
                ok = __all_sync(0xffffffffu, wait_bar(p_full(b), sp.ph, abort_flag, a.status));
                if (!ok) break;
                ok = __all_sync(0xffffffffu, wait_bar(v_full(st), vp.ph, abort_flag, a.status));
                if (!ok) break;
            }
            tc_fence_after();
            const uint64_t vd = sw128_desc(v_smem(st), kBox, 1024);
            const uint32_t d = tmem + P.o_col0 + (pc.qi & 1u) * P.o_cols;
            const uint32_t pa = tmem + 128u * (uint32_t)b;
            if (leader) {
#pragma unroll 1
                for (int kk = 0; kk < kBN / 16; ++kk)
                    mma_ts(d, pa + kk * 8, vd + (uint64_t)kk * 128, P.idesc_pv, (pc.t > 0 || kk > 0) ? 1u : 0u);
                mma_commit(pv_done(np));
                mma_commit(v_empty(st));
            }
            ++np;
            sp.next(3);
            vp.next(S);
            if (++pc.t == pc.nkt) {
                ++pc.qi;
                pc.item += gridDim.x;
                has_p = split_seek(P, pc);
            }
            // The buffer just multiplied by V takes the S three tiles on.
            ok = issue_qk();
        }
        if (!ok && leader) *abort_flag = 1;
        if (leader) mma_commit(drain);
        wait_bar_drain(drain, 0);
        __syncwarp();
    } else if (warp < 8) {
        // -------------------------------------------------------------- softmax
        const int wq = warp % 4;               // TMEM lane quarter
        const int h = warp / 4;                // key half: keys [64h, 64h + 64) of each tile
        const int r = wq * 32 + lane;          // row within the q tile
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t half_o = P.o_cols / 2;  // this warp's O columns: [h half_o, (h + 1) half_o)
        const uint32_t o_base = tmem + lane_off + P.o_col0 + (uint32_t)h * half_o;  // + accumulator * o_cols
        const uint32_t rsw = (uint32_t)(r & 7);  // 128B swizzle: chunk c of row r sits at chunk c ^ (r % 8)
        const uint32_t rrow = (uint32_t)r * 128u;
        uint32_t sn = 0, x_it = 0;  // sn: key tiles so far (the PV index)
        int sb = 0, sph = 0;        // sn % 3 and (sn / 3) & 1: S buffer and its phase
        StageRing br = {0, 0u, false};
        const float2 scale2 = make_float2(a.scale, a.scale);
        float* xbuf = reinterpret_cast<float*>(gbase + L.xbuf);
        float* xl = reinterpret_cast<float*>(gbase + L.xl);
        bool ok = true;
        // Swap a value with the partner warp of this lane quarter (bounded wait).
        // The fences order this warp's tensor-memory loads before the partner's
        // later stores (P of key half 1 lands in half 0's logit columns).
        auto swap = [&](float* buf, float v) -> float {
            buf[h * 128 + r] = v;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(xchg(wq));
            const bool w_ok = __all_sync(0xffffffffu, wait_bar(xchg(wq), x_it & 1, abort_flag, a.status));
            ++x_it;
            tc_fence_after();
            if (!w_ok) {
                ok = false;
                return v;
            }
            return buf[(1 - h) * 128 + r];
        };

        // Wait until PV n is in O.  PV k completes phase k / 2 of barrier k % 2,
        // so a parity wait is exact while that barrier is neither a phase ahead
        // (PV n + 2 done) nor behind (PV n - 2 not done).  The callers hold:
        // this warp has not given P of tile n + 2, and PV n - 2 finished
        // before the S it last read (S of tile m is issued after PV m - 3).
        // With `prev`, PV n - 1 is waited for first, which covers a caller
        // that only knows PV n - 3 finished.
        auto wait_pv = [&](uint32_t n, bool prev) -> bool {
            if (prev && n > 0 &&
                !__all_sync(0xffffffffu, wait_bar(pv_done(n - 1u), ((n - 1u) >> 1) & 1, abort_flag, a.status)))
                return false;
            if (!__all_sync(0xffffffffu, wait_bar(pv_done(n), (n >> 1) & 1, abort_flag, a.status))) return false;
            tc_fence_after();
            return true;
        };

        // The epilogue of the previous item, run after the first tile of the
        // next one (or at the end).  A row with no valid key has every logit
        // -1e9; every key tile was then visited with unit weights and O / l is
        // the mean of V.  A row whose valid keys all have logits at or below
        // -1e9 (only with a bias of that size) visited only the prefix tiles:
        // the h == 0 warp forms the mean of V over all keys for it directly.
        struct Pending {
            float m_ref, l, m_true;
            long long orow, unit;
            uint32_t n_last, ob;
            bool row_ok, direct;
        } pe = {};
        bool pend = false;
        auto epilogue = [&](bool at_end) -> bool {
            const float l_all = pe.l + swap(xl, pe.l);
            if (!ok) return false;
            if (pe.row_ok && h == 0) {
                const float lse = pe.direct ? kMasked + logf((float)a.K) : pe.m_ref + logf(l_all);
                if (a.lse) a.lse[pe.orow] = lse;
                if (a.mx) a.mx[pe.orow] = pe.direct ? kMasked : pe.m_true;
            }
            if (!wait_pv(pe.n_last, at_end)) return false;
            const uint32_t oa = o_base + pe.ob * P.o_cols;
            uint16_t* orow_p = static_cast<uint16_t*>(a.out) + pe.orow * a.D;
            uint16_t* op = orow_p + (long long)h * half_o;
            const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
            const int dlim = a.D - h * (int)half_o;  // columns of this half that exist
            if (half_o == 32) {  // D in (48, 64]: this warp's 32 columns in one load
                uint32_t o[32];
                tmem_ld_x32(oa, o);
                uint32_t wv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    wv[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                if (pe.row_ok && !pe.direct) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (8 * i < dlim)
                            reinterpret_cast<uint4*>(op)[i] =
                                make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                }
            } else {
#pragma unroll 1
                for (uint32_t c0 = 0; c0 < half_o; c0 += 8) {
                    uint32_t o[8];
                    tmem_ld_x8(oa + c0, o);
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        wv[e / 2] = pack2<BF16>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                    if (pe.row_ok && !pe.direct && (int)c0 < dlim)
                        *reinterpret_cast<uint4*>(op + c0) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            if (h == 0 && __any_sync(0xffffffffu, pe.direct && pe.row_ok)) {
                // Lane l forms the means of columns l and l + 32; rows take them by shuffles.
#pragma unroll 1
                for (int d0 = 0; d0 < a.D; d0 += 32) {
                    const int d = d0 + lane;
                    float sum[4] = {0.f, 0.f, 0.f, 0.f};
                    if (d < a.D) {
                        const long long vrow0 = pe.unit * a.K;
                        int key = 0;
#pragma unroll 1
                        for (; key + 4 <= a.K; key += 4) {
#pragma unroll
                            for (int u = 0; u < 4; ++u) sum[u] += load16<BF16>(a.v, (vrow0 + key + u) * a.D + d);
                        }
#pragma unroll 1
                        for (; key < a.K; ++key) sum[0] += load16<BF16>(a.v, (vrow0 + key) * a.D + d);
                    }
                    const float mv = ((sum[0] + sum[1]) + (sum[2] + sum[3])) / (float)a.K;
#pragma unroll 1
                    for (int e = 0; e < 32 && d0 + e < a.D; ++e) {
                        const float m = __shfl_sync(0xffffffffu, mv, e);
                        if (pe.row_ok && pe.direct) orow_p[d0 + e] = (uint16_t)(pack2<BF16>(m, 0.f) & 0xffffu);
                    }
                }
            }
            return true;
        };

        uint32_t qi = 0;  // items with work so far: O accumulator qi % 2
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<1> it = decode<1, false>(P, item);
            if (!it.any) continue;
            const uint32_t ob = qi & 1u;
            ++qi;
            const uint32_t o_taddr = o_base + ob * P.o_cols;
            const int qrow = it.qt[0] * kBM + r;
            float m_true = -INFINITY, m_ref = 0.f, l = 0.f;
            int jv = 0;
            for (int kb = 0; kb < it.nkb && ok; ++kb) {
                const int key0 = kb * kBN;
                const int vlim = P.mask_kind == 1 ? it.prefix : a.K;
                const bool all_valid = P.mask_kind != 2 && key0 + kBN <= vlim;
                const int nexist = a.K - key0;
                const int bs = br.idx;
                // Both barriers tested at once; the bounded waits only when one is not ready.
                const bool ready = mbar_test(bias_full(bs), br.ph) & mbar_test(s_full(sb), (uint32_t)sph);
                if (!__all_sync(0xffffffffu, ready)) {
                    ok = __all_sync(0xffffffffu, wait_bar(bias_full(bs), br.ph, abort_flag, a.status));
                    if (!ok) break;
                    ok = __all_sync(0xffffffffu, wait_bar(s_full(sb), (uint32_t)sph, abort_flag, a.status));
                    if (!ok) break;
                }
                const uint32_t boff = bias_smem(bs) - base + rrow;
                const uint32_t mwoff = L.maskw + (uint32_t)bs * 16u;
                const uint32_t s_taddr = tmem + lane_off + 128u * (uint32_t)sb;
                tc_fence_after();

                // ---- x: this warp's 64 values of the row (logits).
                float x[64];
                {
                    uint32_t sr[64];
                    tmem_ld_x64(s_taddr + 64u * (uint32_t)h, sr);
                    if constexpr (!BIAS_F32) {
                        const uint32_t bbox = boff + (uint32_t)h * kBox;  // keys 64h .. 64h+63: box h
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const uint4 wv = *reinterpret_cast<const uint4*>(gbase + bbox + ((((uint32_t)g) ^ rsw) << 4));
                            const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 b2 = unpack2<BF16>(ww[e]);
                                const int j = 8 * g + 2 * e;
                                const float2 r2 = __ffma2_rn(
                                    make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])), scale2, b2);
                                x[j] = r2.x;
                                x[j + 1] = r2.y;
                            }
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < 16; ++g) {  // 4 keys per 16-byte chunk; boxes 2h, 2h+1
                            const uint4 wv = *reinterpret_cast<const uint4*>(
                                gbase + boff + (uint32_t)(2 * h + (g >> 3)) * kBox + ((((uint32_t)g & 7u) ^ rsw) << 4));
                            const int j = 4 * g;
                            const float2 r0 = __ffma2_rn(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])),
                                                         scale2, make_float2(__uint_as_float(wv.x), __uint_as_float(wv.y)));
                            const float2 r1 =
                                __ffma2_rn(make_float2(__uint_as_float(sr[j + 2]), __uint_as_float(sr[j + 3])), scale2,
                                           make_float2(__uint_as_float(wv.z), __uint_as_float(wv.w)));
                            x[j] = r0.x;
                            x[j + 1] = r0.y;
                            x[j + 2] = r1.x;
                            x[j + 3] = r1.y;
                        }
                    }
                }
                // ---- Masking (boundary tiles only; uniform across the warp).
                if (!all_valid) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int k0 = 64 * h + 32 * hh;
                        const uint32_t em = low_bits(nexist - k0);
                        uint32_t vm = em & low_bits(vlim - key0 - k0);
                        if (P.mask_kind == 2)
                            vm &= *reinterpret_cast<const uint32_t*>(gbase + mwoff + 4u * (uint32_t)(2 * h + hh));
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            x[32 * hh + j] =
                                ((vm >> j) & 1u) ? x[32 * hh + j] : (((em >> j) & 1u) ? kMasked : -INFINITY);
                    }
                }
                __syncwarp();  // every lane of the warp has read its bias and the mask words
                if (lane == 0) mbar_arrive(bias_empty(bs));
                br.next(BS);

                // ---- Row max of the tile: this half's, then the partner's.
                float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; j += 8) {
                    m0 = max3(m0, x[j], x[j + 1]);
                    m1 = max3(m1, x[j + 2], x[j + 3]);
                    m2 = max3(m2, x[j + 4], x[j + 5]);
                    m3 = max3(m3, x[j + 6], x[j + 7]);
                }
                const float mh = fmaxf(max3(m0, m1, m2), m3);
                const float tm = fmaxf(mh, swap(xbuf + (sn & 1u) * 256u, mh));
                if (!ok) break;
                m_true = fmaxf(m_true, tm);
                if (jv == 0) {
                    m_ref = tm;
                    l = 0.f;
                } else {
                    const float m_new = fmaxf(m_ref, tm);
                    const bool need = (m_new - m_ref) * kLog2e > kRescaleLog2;
                    if (__any_sync(0xffffffffu, need)) {
                        // Both warps of the lane quarter take this branch for the same
                        // rows (same tm, same m_ref); each scales its O columns once
                        // O holds the previous tile.
                        ok = wait_pv(sn - 1u, false);
                        if (!ok) break;
                        const float alpha = ex2((m_ref - m_new) * kLog2e);
                        l *= alpha;
                        m_ref = m_new;
                        for (uint32_t c0 = 0; c0 < half_o; c0 += 8) {
                            uint32_t o[8];
                            tmem_ld_x8(o_taddr + c0, o);
#pragma unroll
                            for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st_x8(o_taddr + c0, o);
                        }
                    }
                }

                // ---- P for this warp's 64 keys into columns [32h, 32h + 32) of the
                // buffer (after the swap, so the partner has read its logits).
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
                tmem_st_x32(s_taddr + 32u * (uint32_t)h, pk);
                l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(p_full(sb));
                ++sn;
                if (++sb == 3) {
                    sb = 0;
                    sph ^= 1;
                }
                if (++jv == 1 && pend) {
                    pend = false;
                    ok = epilogue(false);
                }
            }
            if (!ok) break;
            pe.m_ref = m_ref;
            pe.l = l;
            pe.m_true = m_true;
            pe.orow = it.unit * a.Q + qrow;
            pe.unit = it.unit;
            pe.n_last = sn - 1u;
            pe.ob = ob;
            pe.row_ok = qrow < it.Lq;
            pe.direct = !(m_true > kMasked) && jv != (a.K + kBN - 1) / kBN;
            pend = true;
        }
        if (ok && pend) ok = epilogue(true);
        if (!ok) *abort_flag = 1;
    }

    // ---------------------------------------------------------------- teardown
    if (warp == kProducerWarp && lane == 0 && *abort_flag) {
#pragma unroll 1
        for (int i = 0; i < 2000; ++i) __nanosleep(1000);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(P.tmem_cols)
                     : "memory");
    }
}

template <bool BF16, bool BIAS_F32>
cudaError_t launch_split(const TcParams& P, int grid, cudaStream_t stream) {
    const SplitLayout L = make_split_layout(P);
    const size_t smem = L.total + 1024;
    auto kern = tc_split_kernel<BF16, BIAS_F32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kSplitThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

#define TRIATTN_SPLIT_VARIANTS(X) X(true, false) X(true, true) X(false, false) X(false, true)
#define TRIATTN_SPLIT_EXTERN(b, f) extern template cudaError_t launch_split<b, f>(const TcParams&, int, cudaStream_t);
#define TRIATTN_SPLIT_INSTANTIATE(b, f) template cudaError_t launch_split<b, f>(const TcParams&, int, cudaStream_t);

}  // namespace tc
}  // namespace triattn
