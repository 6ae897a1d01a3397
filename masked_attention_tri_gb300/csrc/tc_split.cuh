// tc_split.cuh -- tcgen05 / TMA forward with one 128-row query tile per work
// item and its softmax split over eight warps: the triangle form with D <= 64,
// and the packed-sequence (varlen) form with D <= 128.  Launched from
// tc_fwd.cu, instantiated in tc_inst_split*.cu.  Computes the same
// cuEquivariance triangle_attention formula as tc_kernel.cuh (see there for
// masking and the lazy rescale); the packed form visits the kv blocks that a
// tensorplay BlockMask lists for each q block (full blocks skip mask_mod).
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
//   warp 10      bias producer: TMA of bias tiles and the dense-mask bits
//                (triangle form);
//   warp 11      producer: TMA of V.
// The MMA warp walks the CTA's key tiles as one stream across work items:
// when P of tile n is ready, PV of tile n is issued and then QK^T of tile
// n + SB into the S buffer it read (SB = 3 S buffers for the triangle form,
// 2 for the packed form), also when that tile belongs to the next item, so
// the softmax finds S ready at item boundaries too.  Tensor memory: the S
// buffers of 128 columns from column 0 (P overwrites the first 64 columns of
// its buffer) and, after them, two O accumulator sets (items alternate
// between them): triangle form, two halves of up to 64 columns each per set;
// packed form, one O of up to 128 columns per set.  (With one set, an item's
// first PV waits until the softmax has read the previous item's O.)  The softmax writes out an item's O after
// the first tile of the next item, when the last PV of the item has long
// finished.  K and V stages have their own barriers: a K stage is refilled
// once its QK^T is done, a V stage once its PV is.  The softmax waits for a
// PV only before it rescales O and before it reads O.
//
// Work items.  Triangle form: one q tile of one (b, n, h) slab, in index
// order, dealt round-robin over the CTAs (q tiles fastest, then n: the CTAs
// running at once share K / V and bias tiles in L2).  Packed form: one
// 128-row q block of one (sequence, head).  A causal q block visits about as
// many kv blocks as its index + 1, so items are ordered by q block,
// highest first (within one q block by sequence, then head) and dealt
// serpentine (CTA c takes positions c, 2G - 1 - c, 2G + c, ... of G CTAs),
// which balances the CTAs' key-tile counts much like a longest-first
// schedule.  Every CTA reads the sequence offsets into shared memory once and
// walks this order itself; every role walks it the same way.

#pragma once

#include "tc_kernel.cuh"

namespace triattn {
namespace tc {

constexpr int kSplitThreads = 12 * 32;
// Packed form: sequences whose offsets the schedule keeps in shared memory
// (more sequences go to the two-tile kernel).
constexpr int kSplitMaxSeqs = 1024;

// Packed form: decoded work items, handed from the scheduler warp to the
// other roles through a ring in shared memory.
constexpr int kRing = 8;
struct VEntry {
    int seq, h, qb, nkt;       // nkt < 0: no more items
    int q_row0, Lq, k_row0, Lk;
    int nkb, n_part, n_full, lists;
    const int32_t* part_l;
    const int32_t* full_l;
    unsigned long long part0, full0;
};

struct SplitLayout {
    uint32_t q, kv, bias, ostage, maskw, xbuf, xl, sched, ring, bars, tmem_slot, abort_flag, total;
    int nbars;
};

__host__ __device__ inline SplitLayout make_split_layout(const TcParams& P) {
    SplitLayout L;
    L.q = 0;
    L.kv = L.q + P.q_bufs * P.tile_bytes;
    L.bias = L.kv + P.kv_stages * 2 * P.tile_bytes;
    // O staging for the TMA store: 4 lane quarters x 32 rows x o_rowb bytes (1024-aligned:
    // the bias stages are whole 16 KB boxes)
    L.ostage = L.bias + P.bias_stages * P.bias_bytes;
    L.maskw = L.ostage + (P.o_tma ? 4u * 32u * (uint32_t)P.o_rowb : 0u);
    // shared O: row maxima [tile parity][key half][128 rows]; split O: the epilogue's
    // (reference max, sum, max) [item parity][key half][3][128 rows] (fp32)
    L.xbuf = L.maskw + P.bias_stages * 16;
    L.xl = L.xbuf + (P.a.varlen ? 2 * 2 : 2 * 2 * 3) * 128 * 4;  // row sums: [key half][128 rows] fp32
    // packed form: cu_q[S+1], cu_k[S+1], q blocks[S], sequences per q block level[nqt] (int32)
    L.sched = L.xl + 2 * 128 * 4;
    const uint32_t sched_bytes = P.a.varlen ? (uint32_t)(3 * P.a.num_seqs + 2 + P.nqt) * 4u : 0u;
    // ring: ring_full[kRing], ring_empty[kRing] (8-byte mbarriers), then the entries
    L.ring = (L.sched + sched_bytes + 15u) & ~15u;
    L.bars = L.ring + (P.a.varlen ? (uint32_t)(16 * kRing + kRing * sizeof(VEntry)) : 0u);
    // q_full, q_empty (QB each), k_full, k_empty, v_full, v_empty (S each),
    // bias_full, bias_empty (BS each), s_full[s_bufs], p_full[s_bufs],
    // pv_done[2], drain, o_empty
    L.nbars = 2 * P.q_bufs + 4 * P.kv_stages + 2 * P.bias_stages + 2 * P.s_bufs + 2 + 1 + 1;
    L.tmem_slot = L.bars + 8 * L.nbars;
    L.abort_flag = L.tmem_slot + 4;
    L.total = L.abort_flag + 4;
    return L;
}

// One work item of the key-split kernel.
struct SItem {
    int qt;             // q tile (triangle) / q block (packed form)
    long long unit;     // triangle: (b*N+n)*H+h
    long long bn;       // triangle: b*N+n
    int b, h, seq;
    int Lq, Lk;         // query rows / keys of the unit
    int q_row0, k_row0; // packed form: first row of the sequence
    int prefix;         // triangle kv_lengths (clamped)
    int nkb;            // key blocks of the unit
    int nkt;            // key tiles the item visits
    bool lists;         // packed form: BlockMask lists given
    const int32_t* part_l;
    const int32_t* full_l;
    int n_part, n_full;
    uint64_t part0, full0;  // packed form: visited blocks of window 0 (blocks 0..63)
};

// Packed form, blocks [64 w, 64 w + 64) of the item: `part` (mask_mod applies)
// and `full` (mask_mod skipped).  Warp-cooperative (every lane of the warp
// calls it and gets the same masks): lane t reads list entries t, t + 32, ...
// pre_p / pre_f: entries `lane` of the two lists when the caller has loaded them already (else < 0).
__device__ __forceinline__ void split_window(const SItem& it, int w, uint64_t& part, uint64_t& full, int pre_p = -1,
                                             int pre_f = -1) {
    const int lo = 64 * w;
    const int n = min(64, it.nkb - lo);
    if (n <= 0) {
        part = full = 0;
        return;
    }
    const uint64_t range = n >= 64 ? ~0ull : ((1ull << n) - 1ull);
    if (!it.lists) {
        part = range;
        full = 0;
        return;
    }
    const int lane = threadIdx.x % 32;
    uint64_t p = 0, f = 0;
    for (int t = lane; t < it.n_part; t += 32) {
        const int kb = (t == lane && pre_p >= 0 ? pre_p : it.part_l[t]) - lo;
        if (kb >= 0 && kb < n) p |= 1ull << kb;
    }
    for (int t = lane; t < it.n_full; t += 32) {
        const int kb = (t == lane && pre_f >= 0 ? pre_f : it.full_l[t]) - lo;
        if (kb >= 0 && kb < n) f |= 1ull << kb;
    }
    const uint32_t plo = __reduce_or_sync(0xffffffffu, (uint32_t)p), phi = __reduce_or_sync(0xffffffffu, (uint32_t)(p >> 32));
    const uint32_t flo = __reduce_or_sync(0xffffffffu, (uint32_t)f), fhi = __reduce_or_sync(0xffffffffu, (uint32_t)(f >> 32));
    full = ((uint64_t)fhi << 32) | flo;
    part = (((uint64_t)phi << 32) | plo) & ~full;
}

// The packed form's schedule: a cursor over (q block descending, sequence,
// head) and the serpentine deal of those positions over the grid.
struct VCursor {
    int qb, s, hnext;
    uint32_t cnt;  // positions before (qb, s)
};

__device__ __forceinline__ VCursor vcursor_begin(const TcParams& P) { return VCursor{P.nqt - 1, 0, 0, 0u}; }

// Next item of this CTA: (sequence, head, q block).  `snb` holds each
// sequence's q block count (0 for a sequence that breaks its contract) and
// `lvl` the number of sequences with more than qb q blocks, for each qb.  The
// CTA's next position in the deal is fixed by the positions before the
// cursor, so it is found once; q block levels that end before it are skipped
// whole, then the level's (sequence, head) groups are walked.
__device__ __forceinline__ bool vcursor_next(const TcParams& P, const int* snb, const int* lvl, VCursor& c, int& seq,
                                             int& h, int& qb) {
    const int S = P.a.num_seqs, H = P.a.H;
    const uint32_t G2 = P.fd_2g.d;
    const uint32_t lo = blockIdx.x, hi = G2 - 1u - blockIdx.x;
    const uint32_t x = c.cnt + (uint32_t)c.hnext;
    const uint32_t base = P.fd_2g.div(x) * G2;
    const uint32_t r = x - base;
    const uint32_t pos = r <= lo ? base + lo : (r <= hi ? base + hi : base + G2 + lo);
    while (c.qb >= 0) {
        if (c.s == 0) {
            const uint32_t lv = (uint32_t)lvl[c.qb] * (uint32_t)H;  // the level's positions
            if (pos >= c.cnt + lv) {
                c.cnt += lv;
                c.hnext = 0;
                --c.qb;
                continue;
            }
        }
        if (c.s >= S) {
            c.s = 0;
            --c.qb;
            continue;
        }
        if (snb[c.s] > c.qb) {
            if (pos < c.cnt + (uint32_t)H) {
                seq = c.s;
                h = (int)(pos - c.cnt);
                qb = c.qb;
                c.hnext = h + 1;
                return true;
            }
            c.cnt += (uint32_t)H;
        }
        c.hnext = 0;
        ++c.s;
    }
    return false;
}

// Triangle item from its index (kv_lengths resolved), or packed item from
// (sequence, head, q block) with its visited-tile count (warp-cooperative).
template <bool VARLEN>
__device__ __forceinline__ SItem split_decode(const TcParams& P, const int* sched, int item, int seq, int h, int qb,
                                              int pre_len = kNoLen) {
    SItem it;
    const AttnParams& a = P.a;
    it.lists = false;
    it.part_l = it.full_l = nullptr;
    it.n_part = it.n_full = 0;
    it.part0 = it.full0 = 0;
    it.prefix = 0;
    it.q_row0 = it.k_row0 = 0;
    if constexpr (!VARLEN) {
        const Item<1> t = decode<1, false>(P, item, pre_len);
        it.qt = t.qt[0];
        it.unit = t.unit;
        it.bn = t.bn;
        it.b = t.b;
        it.h = t.h;
        it.seq = 0;
        it.Lq = t.Lq;
        it.Lk = t.Lk;
        it.prefix = t.prefix;
        it.nkb = t.nkb;
        it.nkt = t.any ? t.nkb : 0;
    } else {
        const int S = a.num_seqs;
        const int* scq = sched;
        const int* sck = sched + S + 1;
        it.qt = qb;
        it.unit = it.bn = 0;
        it.b = 0;
        it.h = h;
        it.seq = seq;
        it.q_row0 = scq[seq];
        it.Lq = scq[seq + 1] - it.q_row0;
        it.k_row0 = sck[seq];
        it.Lk = sck[seq + 1] - it.k_row0;
        it.nkb = (it.Lk + kBN - 1) / kBN;
        int pre_p = -1, pre_f = -1;
        if (a.kv_num != nullptr) {
            it.lists = true;
            if (qb < a.MQ) {
                const int hm = a.mask_heads == 1 ? 0 : h;
                const long long row = ((long long)seq * a.mask_heads + hm) * a.MQ + qb;
                const int lane = threadIdx.x % 32;
                it.part_l = a.kv_idx + row * a.MK;
                if (a.full_num) it.full_l = a.full_idx + row * a.MK;
                // The row's first 32 list entries are read together with the counts (one
                // memory round trip instead of two); entries past the count are unused.
                if (lane < a.MK) {
                    pre_p = max(it.part_l[lane], -1);
                    if (a.full_num) pre_f = max(it.full_l[lane], -1);
                }
                it.n_part = min(max(a.kv_num[row], 0), a.MK);
                if (a.full_num) it.n_full = min(max(a.full_num[row], 0), a.MK);
            }
        }
        split_window(it, 0, it.part0, it.full0, pre_p, pre_f);
        int nkt = __popcll(it.part0 | it.full0);
        for (int w = 1; 64 * w < it.nkb; ++w) {
            uint64_t pm, fm;
            split_window(it, w, pm, fm);
            nkt += __popcll(pm | fm);
        }
        it.nkt = nkt;
    }
    return it;
}

// The key tiles of one item in ascending order: kb and whether mask_mod is
// skipped on it (a full block).
struct TileWalk {
    int w, t;
    uint64_t rem, full;
};

template <bool VARLEN>
__device__ __forceinline__ TileWalk tiles_begin(const SItem& it) {
    TileWalk tw;
    tw.w = 0;
    tw.t = 0;
    tw.rem = VARLEN ? (it.part0 | it.full0) : 0ull;
    tw.full = VARLEN ? it.full0 : 0ull;
    return tw;
}

template <bool VARLEN>
__device__ __forceinline__ bool tiles_next(const SItem& it, TileWalk& tw, int& kb, bool& is_full) {
    if constexpr (!VARLEN) {
        if (tw.t >= it.nkt) return false;
        kb = tw.t++;
        is_full = false;
        return true;
    } else {
        while (tw.rem == 0) {
            ++tw.w;
            if (64 * tw.w >= it.nkb) return false;
            uint64_t pm, fm;
            split_window(it, tw.w, pm, fm);
            tw.rem = pm | fm;
            tw.full = fm;
        }
        const int bit = __ffsll((long long)tw.rem) - 1;
        tw.rem &= tw.rem - 1;
        kb = 64 * tw.w + bit;
        is_full = (tw.full >> bit) & 1ull;
        ++tw.t;
        return true;
    }
}

// Where the roles of the packed form read their work items: the ring's
// shared-memory address (barriers ring_full[i] at ring + 8 i, ring_empty[i] at
// ring + 8 (kRing + i), entries from ring + 16 kRing) and the CTA's abort flag.
struct RingRef {
    uint32_t ring;
    volatile int* abort_flag;
};

// Consumers of one entry: the Q/K and V producers, the MMA warp's two cursors
// and the eight softmax warps.
constexpr int kRingConsumers = 12;

// A role's walk over this CTA's items (all of them, also those without key
// tiles).  Triangle form: item indices blockIdx.x + k * gridDim.x, decoded by
// every role.  Packed form: the entries the scheduler warp decodes in turn.
template <bool VARLEN>
struct ItemWalk;

template <>
struct ItemWalk<false> {
    int item;
    int len;  // kv_lengths entry of `item`, loaded one item ahead
    __device__ __forceinline__ void begin(const TcParams& P, const RingRef&) {
        item = (int)blockIdx.x;
        len = tri_item_len(P, item);
    }
    __device__ __forceinline__ bool next(const TcParams& P, const RingRef&, SItem& it) {
        if (item >= P.items) return false;
        it = split_decode<false>(P, nullptr, item, 0, 0, 0, len);
        item += gridDim.x;
        len = tri_item_len(P, item);
        return true;
    }
};

template <>
struct ItemWalk<true> {
    StageRing rr;
    __device__ __forceinline__ void begin(const TcParams&, const RingRef&) { rr = {0, 0u, false}; }
    __device__ __forceinline__ bool next(const TcParams& P, const RingRef& r, SItem& it) {
        const int slot = rr.idx;
        // A wait that runs out raises the abort flag; the role then leaves like every other.
        if (!__all_sync(0xffffffffu, wait_bar(r.ring + 8u * (uint32_t)slot, rr.ph, r.abort_flag, P.a.status)))
            return false;
        const VEntry* v = reinterpret_cast<const VEntry*>(
            __cvta_shared_to_generic(r.ring + 16u * kRing + (uint32_t)(slot * sizeof(VEntry))));
        it.nkt = v->nkt;
        it.qt = v->qb;
        it.h = v->h;
        it.seq = v->seq;
        it.q_row0 = v->q_row0;
        it.Lq = v->Lq;
        it.k_row0 = v->k_row0;
        it.Lk = v->Lk;
        it.nkb = v->nkb;
        it.lists = v->lists != 0;
        it.part_l = v->part_l;
        it.full_l = v->full_l;
        it.n_part = v->n_part;
        it.n_full = v->n_full;
        it.part0 = v->part0;
        it.full0 = v->full0;
        it.unit = it.bn = 0;
        it.b = 0;
        it.prefix = 0;
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(r.ring + 8u * (uint32_t)(kRing + slot));
        rr.next(kRing);
        return it.nkt >= 0;
    }
};

// A position in the CTA's stream of key tiles (MMA warp): the current item
// with key tiles, its tile count, the next tile in it and the item's number
// among the CTA's items with key tiles.
template <bool VARLEN>
struct SplitCursor {
    ItemWalk<VARLEN> walk;
    int nkt;
    int t;
    uint32_t qi;
};

// Moves the cursor to the next item with key tiles.
template <bool VARLEN>
__device__ __forceinline__ bool split_seek(const TcParams& P, const RingRef& r, SplitCursor<VARLEN>& c) {
    SItem it;
    while (c.walk.next(P, r, it)) {
        if (it.nkt > 0) {
            c.nkt = it.nkt;
            c.t = 0;
            return true;
        }
    }
    return false;
}

// Rows with no valid key among the visited ones (rare): the mean of V over
// `nkeys` keys (V(key, d) at v[v_base + key * v_stride + d]), or zeros when
// there are no keys, into the rows of this warp for which `mine` holds.  Lane
// l forms the means of columns l, l + 32, ...; rows take them by shuffles.
// Out of line so the per-item epilogue stays small in the instruction cache.
template <bool BF16>
static __device__ __noinline__ void split_mean_v(const AttnParams& a, uint16_t* orow_p, long long v_base,
                                                 long long v_stride, int nkeys, bool mine) {
    const int lane = threadIdx.x % 32;
#pragma unroll 1
    for (int d0 = 0; d0 < a.D; d0 += 32) {
        const int d = d0 + lane;
        float sum[4] = {0.f, 0.f, 0.f, 0.f};
        if (d < a.D) {
            int key = 0;
#pragma unroll 1
            for (; key + 4 <= nkeys; key += 4) {
#pragma unroll
                for (int u = 0; u < 4; ++u) sum[u] += load16<BF16>(a.v, v_base + (key + u) * v_stride + d);
            }
#pragma unroll 1
            for (; key < nkeys; ++key) sum[0] += load16<BF16>(a.v, v_base + key * v_stride + d);
        }
        const float mv = nkeys > 0 ? ((sum[0] + sum[1]) + (sum[2] + sum[3])) / (float)nkeys : 0.f;
#pragma unroll 1
        for (int e = 0; e < 32 && d0 + e < a.D; ++e) {
            const float m = __shfl_sync(0xffffffffu, mv, e);
            if (mine) orow_p[d0 + e] = (uint16_t)(pack2<BF16>(m, 0.f) & 0xffffu);
        }
    }
}

// MMA issue sequences.  The k-step loops stay rolled: issuing the MMAs back to
// back (unrolled, compile-time offsets) measured slower here, as the tensor
// core's bursts then contend with the softmax warps' tensor-memory traffic.
// QK^T k step kk reads D elements [16 kk, 16 kk + 16) of the 128B-swizzled
// Q and K tiles: box kk / 4, 32 bytes per step within the box.
__device__ __forceinline__ uint64_t qk_koff(int kk) { return (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4); }
__device__ __forceinline__ void issue_qk_n(int ks, uint32_t sd, uint64_t qd, uint64_t kd, uint32_t idesc) {
#pragma unroll 1
    for (int kk = 0; kk < ks; ++kk) mma_ss(sd, qd + qk_koff(kk), kd + qk_koff(kk), idesc, kk > 0 ? 1u : 0u);
}
// PV of one tile into one O accumulator d (P from TMEM at pa, 8 columns per 16
// keys; V MN-major, 2 KB per 16 keys).
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t pa, uint64_t vd, uint32_t idesc_pv, bool first) {
#pragma unroll 1
    for (int kk = 0; kk < kBN / 16; ++kk)
        mma_ts(d, pa + kk * 8, vd + (uint64_t)kk * 128, idesc_pv, (!first || kk > 0) ? 1u : 0u);
}
// Split O: keys 0-63 of the tile into O_0 (d0), keys 64-127 into O_1 (d1),
// alternating so the two chains overlap.  P of key half 1 sits in that half's
// own logit columns [64, 96).
__device__ __forceinline__ void issue_pv_split(uint32_t d0, uint32_t d1, uint32_t pa, uint64_t vd, uint32_t idesc_pv,
                                               bool first) {
#pragma unroll 1
    for (int j = 0; j < kBN / 16; ++j) {
        const int kk = (j >> 1) + 4 * (j & 1);
        mma_ts((j & 1) ? d1 : d0, pa + kk * 8 + (kk & 4) * 8, vd + (uint64_t)kk * 128, idesc_pv,
               (!first || (kk & 3) > 0) ? 1u : 0u);
    }
}

template <bool BF16, bool BIAS_F32, bool VARLEN, bool FOLD, bool BIAS>
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
    int* sched = reinterpret_cast<int*>(gbase + L.sched);

    const int S = P.kv_stages;
    const int BS = P.bias_stages;
    const int QB = P.q_bufs;
    constexpr int SB = VARLEN ? 2 : 3;           // S buffers (P.s_bufs)
    const int OB = P.o_bufs;                     // O accumulator sets (items alternate between them)
    // Triangle form: each key half accumulates its own O (P of keys [64h, 64h + 64)
    // times those V rows), so the two softmax warps of a lane quarter need no
    // shared row max per tile; the halves are combined once per item.  Packed
    // form (D up to 128, no room for two halves): one O, shared row max.
    constexpr bool kSplitO = !VARLEN;
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
    auto p_full = [&](int b) { return bar(bx0 + SB + b); };
    auto pv_done = [&](uint32_t n) { return bar(bx0 + 2 * SB + (int)(n & 1u)); };  // PV n: phase n / 2 of barrier n % 2
    const uint32_t drain = bar(bx0 + 2 * SB + 2);
    const uint32_t o_empty = bar(bx0 + 2 * SB + 3);  // one O accumulator: the softmax has read it
    const RingRef ring = {base + L.ring, abort_flag};
    auto ring_full = [&](int i) { return base + L.ring + 8u * (uint32_t)i; };
    auto ring_empty = [&](int i) { return base + L.ring + 8u * (uint32_t)(kRing + i); };

    auto q_smem = [&](int qb) { return base + L.q + (uint32_t)qb * P.tile_bytes; };
    auto k_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes; };
    auto v_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes + P.tile_bytes; };
    auto bias_smem = [&](int s) { return base + L.bias + (uint32_t)s * P.bias_bytes; };

    if constexpr (VARLEN) {
        // Sequence offsets and q block counts, read once.  A sequence that
        // breaks the max_seqlen / total contract gets no q blocks (skipped)
        // and TA_ERR_DEVICE is recorded.
        const int NS = a.num_seqs;
        for (int i = threadIdx.x; i <= NS; i += blockDim.x) {
            sched[i] = a.cu_q[i];
            sched[NS + 1 + i] = a.cu_k[i];
        }
        __syncthreads();
        for (int s = threadIdx.x; s < NS; s += blockDim.x) {
            const int cq0 = sched[s], cq1 = sched[s + 1];
            const int ck0 = sched[NS + 1 + s], ck1 = sched[NS + 2 + s];
            const bool ok = cq0 >= 0 && ck0 >= 0 && cq1 >= cq0 && ck1 >= ck0 && cq1 - cq0 <= a.max_q &&
                            ck1 - ck0 <= a.max_k && cq1 <= a.total_q && ck1 <= a.total_k;
            sched[2 * (NS + 1) + s] = ok ? (cq1 - cq0 + kBM - 1) / kBM : 0;
            if (!ok && blockIdx.x == 0) atomicCAS(a.status, 0, kStatusDevice);
        }
    }
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
#pragma unroll 1
        for (int b = 0; b < SB; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 8);  // one arrival per softmax warp
        }
        mbar_init(pv_done(0), 1);
        mbar_init(pv_done(1), 1);
        mbar_init(drain, 1);
        mbar_init(o_empty, 8);  // one arrival per softmax warp
        if (VARLEN) {
#pragma unroll 1
            for (int i = 0; i < kRing; ++i) {
                mbar_init(ring_full(i), 1);
                mbar_init(ring_empty(i), kRingConsumers);
            }
        }
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
        ItemWalk<VARLEN> walk;
        walk.begin(P, ring);
        SItem it;
        while (ok && walk.next(P, ring, it)) {
            if (it.nkt == 0) continue;
            const int qb = qr.idx;
            if (lane == 0 && qr.wrapped) ok = wait_bar(q_empty(qb), qr.ph ^ 1u, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                mbar_expect_tx(q_full(qb), P.tile_bytes);
                for (int sb = 0; sb < P.nsub; ++sb) {
                    if constexpr (!VARLEN)
                        tma_load_tri(P, q_smem(qb) + sb * kBox, &P.tm_q, sb * 64, it.qt * kBM, it.unit, it.h,
                                     (int)(it.bn - (long long)it.b * a.N), it.b, q_full(qb));
                    else
                        tma_load_3d(q_smem(qb) + sb * kBox, &P.tm_q, sb * 64, it.h, it.q_row0 + it.qt * kBM,
                                    q_full(qb));
                }
            }
            qr.next(QB);
            TileWalk tw = tiles_begin<VARLEN>(it);
            int kb;
            bool fb;
            while (ok && tiles_next<VARLEN>(it, tw, kb, fb)) {
                const int st = kr.idx;
                if (lane == 0 && kr.wrapped) ok = wait_bar(k_empty(st), kr.ph ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_expect_tx(k_full(st), P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb) {
                        if constexpr (!VARLEN)
                            tma_load_tri(P, k_smem(st) + sb * kBox, &P.tm_k, sb * 64, kb * kBN, it.unit, it.h,
                                         (int)(it.bn - (long long)it.b * a.N), it.b, k_full(st));
                        else
                            tma_load_3d(k_smem(st) + sb * kBox, &P.tm_k, sb * 64, it.h, it.k_row0 + kb * kBN,
                                        k_full(st));
                    }
                }
                kr.next(S);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kVWarp) {
        // ---------------------------------------------------------- producer: V tiles
        // (packed form with a bias: also the bias tiles; warp 10 is the scheduler there)
        StageRing vr = {0, 0u, false};
        StageRing br = {0, 0u, false};
        bool ok = true;
        ItemWalk<VARLEN> walk;
        walk.begin(P, ring);
        SItem it;
        while (ok && walk.next(P, ring, it)) {
            TileWalk tw = tiles_begin<VARLEN>(it);
            int kb;
            bool fb;
            while (ok && tiles_next<VARLEN>(it, tw, kb, fb)) {
                if constexpr (VARLEN && BIAS) {
                    const int bs = br.idx;
                    if (lane == 0 && br.wrapped) ok = wait_bar(bias_empty(bs), br.ph ^ 1u, abort_flag, a.status);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (lane == 0) {
                        // bias (H, max_seqlen_q, max_seqlen_k): keys kb*128.., local rows qt*128.., head h
                        mbar_expect_tx(bias_full(bs), P.bias_bytes);
                        for (int bx = 0; bx < P.bias_boxes; ++bx)
                            tma_load_3d(bias_smem(bs) + bx * kBox, &P.tm_bias, kb * kBN + bx * P.bias_box_cols,
                                        it.qt * kBM, it.h, bias_full(bs));
                    }
                    br.next(BS);
                }
                const int st = vr.idx;
                if (lane == 0 && vr.wrapped) ok = wait_bar(v_empty(st), vr.ph ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_expect_tx(v_full(st), P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb) {
                        if constexpr (!VARLEN)
                            tma_load_tri(P, v_smem(st) + sb * kBox, &P.tm_v, sb * 64, kb * kBN, it.unit, it.h,
                                         (int)(it.bn - (long long)it.b * a.N), it.b, v_full(st));
                        else
                            tma_load_3d(v_smem(st) + sb * kBox, &P.tm_v, sb * 64, it.h, it.k_row0 + kb * kBN,
                                        v_full(st));
                    }
                }
                vr.next(S);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kBiasWarp) {
        if constexpr (VARLEN) {
            // ------------------------------------------------------------ scheduler
            // Walks this CTA's (sequence, head, q block) items, decodes each (its
            // lists and visited-tile count, warp-cooperatively) and hands it to
            // the other roles through the ring; an entry with nkt < 0 ends it.
            StageRing rr = {0, 0u, false};
            VCursor vc = vcursor_begin(P);
            VEntry* ents = reinterpret_cast<VEntry*>(gbase + L.ring + 16u * kRing);
            const int* snb = sched + 2 * (a.num_seqs + 1);
            int* lvl = sched + 3 * a.num_seqs + 2;
            for (int qb = lane; qb < P.nqt; qb += 32) lvl[qb] = 0;
            __syncwarp();
            for (int sq = lane; sq < a.num_seqs; sq += 32)
                for (int qb = 0; qb < snb[sq]; ++qb) atomicAdd(&lvl[qb], 1);
            __syncwarp();
            bool ok = true;
            for (;;) {
                int seq = 0, hh = 0, qb = 0;
                const bool more = vcursor_next(P, snb, lvl, vc, seq, hh, qb);
                const int slot = rr.idx;
                if (rr.wrapped) {
                    ok = __all_sync(0xffffffffu, wait_bar(ring_empty(slot), rr.ph ^ 1u, abort_flag, a.status));
                    if (!ok) break;
                }
                SItem it;
                if (more) it = split_decode<true>(P, sched, 0, seq, hh, qb);
                if (lane == 0) {
                    VEntry* e = ents + slot;
                    e->nkt = more ? it.nkt : -1;
                    if (more) {
                        e->seq = seq;
                        e->h = hh;
                        e->qb = qb;
                        e->q_row0 = it.q_row0;
                        e->Lq = it.Lq;
                        e->k_row0 = it.k_row0;
                        e->Lk = it.Lk;
                        e->nkb = it.nkb;
                        e->n_part = it.n_part;
                        e->n_full = it.n_full;
                        e->lists = it.lists ? 1 : 0;
                        e->part_l = it.part_l;
                        e->full_l = it.full_l;
                        e->part0 = it.part0;
                        e->full0 = it.full0;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(ring_full(slot));  // release: the entry is written
                rr.next(kRing);
                if (!more) break;
            }
            if (!ok) *abort_flag = 1;
        } else {
            // ---------------------------------- producer: bias tiles (+ dense-mask bits)
            StageRing br = {0, 0u, false};
            bool ok = true;
            int len = tri_item_len(P, (int)blockIdx.x);  // loaded one item ahead
            for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
                const Item<1> it = decode<1, false>(P, item, len);
                len = tri_item_len(P, item + (int)gridDim.x);
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
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        // Two cursors over the CTA's items with key tiles: `qc` for the next
        // QK^T, `pc` for the next PV.  Tile n of the stream (counted over
        // items) has S buffer n % SB and K/V stage n % S; item number i has Q
        // buffer i % QB and O accumulator set i % o_bufs.  QK^T runs SB tiles
        // ahead: once P of tile n is in TMEM, PV of tile n is issued, then
        // QK^T of tile n + SB into the buffer PV n reads (the tensor core runs
        // them in order).
        const bool leader = elect_one();
        SplitCursor<VARLEN> qc, pc;
        qc.walk.begin(P, ring);
        qc.qi = 0;
        bool has_q = split_seek<VARLEN>(P, ring, qc);
        pc = qc;
        bool has_p = has_q;
        uint32_t np = 0;                                    // PV issued so far
        StageRing qr = {0, 0u, false};                      // Q buffer of qc's item
        StageRing kq = {0, 0u, false}, sq = {0, 0u, false};  // K stage / S buffer of the next QK^T
        StageRing vp = {0, 0u, false}, sp = {0, 0u, false};  // V stage / S buffer of the next PV
        StageRing oe = {0, 0u, false};                      // single O accumulator: its "read" barrier
        bool ok = true;
        // QK^T of the next tile: wait for its Q (first tile of an item) and K stage.
        uint64_t qd = 0, kd = 0;
        uint32_t sd = 0;
        int q_qb = 0, q_st = 0, q_b = 0;
        auto qk_ready = [&]() -> bool {
            q_qb = qr.idx;
            if (qc.t == 0 && !__all_sync(0xffffffffu, wait_bar(q_full(q_qb), qr.ph, abort_flag, a.status)))
                return false;
            q_st = kq.idx;
            if (!__all_sync(0xffffffffu, wait_bar(k_full(q_st), kq.ph, abort_flag, a.status))) return false;
            qd = sw128_desc(q_smem(q_qb), 16, 1024);
            kd = sw128_desc(k_smem(q_st), 16, 1024);
            q_b = sq.idx;
            sd = tmem + 128u * (uint32_t)q_b;
            return true;
        };
        // Commits and cursor moves once the QK^T's MMAs are issued.
        auto qk_done = [&]() {
            if (leader) {
                mma_commit(s_full(q_b));
                mma_commit(k_empty(q_st));
            }
            kq.next(S);
            sq.next(SB);
            if (++qc.t == qc.nkt) {
                if (leader) mma_commit(q_empty(q_qb));  // every QK^T of the item is issued
                qr.next(QB);
                ++qc.qi;
                has_q = split_seek<VARLEN>(P, ring, qc);
            }
        };
        auto qk_alone = [&]() {
            tc_fence_after();
            if (leader) issue_qk_n(P.ksteps, sd, qd, kd, P.idesc_qk);
            qk_done();
        };
        for (int i = 0; i < SB && ok && has_q; ++i) {
            ok = qk_ready();
            if (!ok) break;
            qk_alone();
        }
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
            // With one O accumulator, the first PV of an item waits until the
            // softmax has read out the previous item's O.
            if (OB == 1 && pc.t == 0 && pc.qi > 0) {
                ok = __all_sync(0xffffffffu, wait_bar(o_empty, oe.ph, abort_flag, a.status));
                if (!ok) break;
                oe.next(1);
            }
            tc_fence_after();
            const uint64_t vd = sw128_desc(v_smem(st), kBox, 1024);
            const uint32_t oset = OB == 1 ? 0u : (pc.qi & 1u);
            const uint32_t d = tmem + P.o_col0 + oset * (kSplitO ? 2u : 1u) * P.o_cols;
            const uint32_t pa = tmem + 128u * (uint32_t)b;
            if (leader) {
                if constexpr (kSplitO)
                    issue_pv_split(d, d + P.o_cols, pa, vd, P.idesc_pv, pc.t == 0);
                else
                    issue_pv(d, pa, vd, P.idesc_pv, pc.t == 0);
                mma_commit(pv_done(np));
                mma_commit(v_empty(st));
            }
            ++np;
            sp.next(SB);
            vp.next(S);
            if (++pc.t == pc.nkt) {
                ++pc.qi;
                has_p = split_seek<VARLEN>(P, ring, pc);
            }
            if (has_q) {  // the buffer just multiplied by V takes the S SB tiles on
                ok = qk_ready();
                if (!ok) break;
                qk_alone();
            }
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
        const uint32_t half_o = P.o_cols / 2;  // this warp's output columns: [h half_o, (h + 1) half_o)
        // Split O (triangle): this warp's accumulator O_h of set ob at o_col0 + (2 ob + h) o_cols.
        // Shared O (packed): this warp's columns of set ob at o_col0 + ob o_cols + h half_o.
        const uint32_t o_base = tmem + lane_off + P.o_col0 + (uint32_t)h * (kSplitO ? P.o_cols : half_o);
        const uint32_t o_set = (kSplitO ? 2u : 1u) * P.o_cols;  // columns between accumulator sets
        const uint32_t rsw = (uint32_t)(r & 7);  // 128B swizzle: chunk c of row r sits at chunk c ^ (r % 8)
        const uint32_t rrow = (uint32_t)r * 128u;
        uint32_t sn = 0, x_it = 0;  // sn: key tiles so far (the PV index)
        int sb = 0, sph = 0;        // sn % s_bufs and (sn / s_bufs) & 1: S buffer and its phase
        StageRing br = {0, 0u, false};
        const float2 scale2 = make_float2(a.scale, a.scale);
        // Folded form (packed sequences, scale > 0): values are in units of S
        // (x = s S); a masked key holds -FLT_MAX there (its logit is -1e9).
        constexpr float kMaskVal = FOLD ? -FLT_MAX : kMasked;
        const float unit_l2e = FOLD ? P.scale_log2e : kLog2e;
        float* xbuf = reinterpret_cast<float*>(gbase + L.xbuf);
        float* xl = reinterpret_cast<float*>(gbase + L.xl);
        bool ok = true;
        // Swap a value with the partner warp of this lane quarter (bounded wait).
        // The fences order this warp's tensor-memory loads before the partner's
        // later stores (P of key half 1 lands in half 0's logit columns).
        // Rendezvous of the two warps of this lane quarter on their hardware barrier.  A warp
        // enters it only while the CTA is not aborting, and a warp that leaves on an abort
        // arrives on it once (at the end of this role), so a partner that entered just before
        // the abort is released: this wait without a time limit cannot hang.
        auto pair_sync = [&]() -> bool {
            if (__any_sync(0xffffffffu, *abort_flag != 0)) return false;
            named_barrier(1 + wq, 64);
            return true;
        };
        auto swap = [&](float* buf, float v) -> float {
            buf[h * 128 + r] = v;
            tc_fence_before();
            __syncwarp();
            const bool w_ok = pair_sync();
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
        // before the S it last read (QK^T of tile m is issued after PV m - SB,
        // SB >= 2, and its commit completes only when every MMA issued before
        // it has).  With `prev`, PV n - 1 is
        // waited for first, which covers a caller that only knows PV n - 3
        // finished.
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
        // -1e9; when every key block was visited (with unit weights) O / l is
        // the mean of V.  A row whose visited keys were all masked while some
        // blocks were not visited (packed form: blocks its lists leave out;
        // triangle form: only with a bias at or below -1e9) gets the mean of V
        // over all keys, formed directly by the h == 0 warp.
        // Where a row's outputs go: (out element offset, lse/max index, V's first
        // element, V's key stride, keys).  Triangle form: row0 = the flat
        // (b,n,h,q) row, unit0 = the slab's first V element; packed form: row0 = the
        // packed query row, unit0 = the sequence's first key row, hh = the head,
        // nk = its keys.
        struct RowAddr {
            long long out_off, lse_idx, v_base, v_stride;
            int nkeys;
        };
        auto row_addr = [&](long long row0, long long unit0, int hh, int nk) -> RowAddr {
            RowAddr ra;
            if constexpr (!VARLEN) {
                ra.out_off = row0 * a.D;
                ra.lse_idx = row0;
                ra.v_base = unit0;  // the slab's first V element (the caller passes it)
                ra.v_stride = a.vs[3];
                ra.nkeys = a.K;
            } else {
                ra.out_off = (row0 * a.H + hh) * a.D;
                ra.lse_idx = (long long)hh * a.total_q + row0;
                ra.v_base = unit0 * a.v_rs + (long long)hh * a.D;
                ra.v_stride = a.v_rs;
                ra.nkeys = nk;
            }
            return ra;
        };
        struct Pending {
            float m_ref, l, m_true;
            long long row0, unit0;
            int hh, nk;
            int box_row, box_unit;  // triangle form: the O store box of this lane quarter
            uint32_t n_last, ob;
            bool row_ok, direct;
        } pe = {};
        // O staging rows of this lane quarter: row `lane` holds 16-byte chunk c at
        // chunk c ^ swz (the map's 128 / 64 / 32-byte swizzle of 128 / 64 / 32-byte rows).
        const uint32_t o_stage = base + L.ostage + (uint32_t)(wq * 32 * P.o_rowb) + (uint32_t)(lane * P.o_rowb);
        const uint32_t o_swz = P.o_rowb == 128 ? (uint32_t)(lane & 7)
                                               : (P.o_rowb == 64 ? (uint32_t)((lane >> 1) & 3) : (uint32_t)((lane >> 2) & 1));
        bool pend = false;
        auto epilogue = [&](bool at_end) -> bool {
            // Combine the two key halves' (reference max, row sum, max).  Shared O:
            // one reference max, the sums add.  Split O: each half's O and sum are
            // scaled to the larger reference max (alpha = 2^((m_h - M) log2 e)).
            float l_all, m_ref_all, m_true_all, a_own = 1.f, a_oth = 1.f;
            if constexpr (kSplitO) {
                float* xe = xbuf + (x_it & 1u) * 768u;  // [item parity][half][3][128 rows]
                xe[(h * 3 + 0) * 128 + r] = pe.m_ref;
                xe[(h * 3 + 1) * 128 + r] = pe.l;
                xe[(h * 3 + 2) * 128 + r] = pe.m_true;
                // The partner writes O staging rows only after this arrival, so the previous
                // item's O store must have read them by then.
                if (P.o_tma && h == 0 && lane == 0) bulk_wait_read_all();
                __syncwarp();
                if (!pair_sync()) return ok = false;
                ++x_it;
                const int o3 = (1 - h) * 3;
                const float m_oth = xe[(o3 + 0) * 128 + r], l_oth = xe[(o3 + 1) * 128 + r];
                const float mt_oth = xe[(o3 + 2) * 128 + r];
                m_ref_all = fmaxf(pe.m_ref, m_oth);
                a_own = pe.m_ref == m_ref_all ? 1.f : ex2((pe.m_ref - m_ref_all) * kLog2e);
                a_oth = m_oth == m_ref_all ? 1.f : ex2((m_oth - m_ref_all) * kLog2e);
                l_all = a_own * pe.l + a_oth * l_oth;
                m_true_all = fmaxf(pe.m_true, mt_oth);
            } else {
                l_all = pe.l + swap(xl, pe.l);
                if (!ok) return false;
                m_ref_all = pe.m_ref;
                m_true_all = pe.m_true;
            }
            // (the two item-parity buffers: a warp overwrites a buffer only after the
            // partner's next arrival, which follows its read of that buffer)
            const bool direct = kSplitO ? (!(m_true_all > kMasked) && pe.direct) : pe.direct;
            const RowAddr ra = row_addr(pe.row0, pe.unit0, pe.hh, pe.nk);
            if (pe.row_ok && h == 0) {
                float mr = m_ref_all;
                if constexpr (FOLD) mr = m_ref_all > -FLT_MAX ? m_ref_all * a.scale : kMasked;
                const float lse = direct ? kMasked + logf((float)ra.nkeys) : mr + logf(l_all);
                if (a.lse) a.lse[ra.lse_idx] = lse;
                if (a.mx) a.mx[ra.lse_idx] = direct ? kMasked : m_true_all;
            }
            if (!wait_pv(pe.n_last, at_end)) return false;
            // split O: this warp's output columns of O_0 (oa0) and O_1 (oa0 + o_cols)
            const uint32_t oa = kSplitO ? tmem + lane_off + P.o_col0 + pe.ob * o_set + (uint32_t)h * half_o
                                        : o_base + pe.ob * o_set;
            uint16_t* orow_p = static_cast<uint16_t*>(a.out) + ra.out_off;
            uint16_t* op = orow_p + (long long)h * half_o;
            const float inv = l_all > 0.f ? 1.f / l_all : 0.f;
            // weights of O_0 and O_1 (split O), folded with 1 / l
            const float w0 = (h == 0 ? a_own : a_oth) * inv, w1 = (h == 0 ? a_oth : a_own) * inv;
            const int dlim = a.D - h * (int)half_o;  // columns of this half that exist
            // Triangle form: the lane quarter's 32 rows go to shared memory and leave in one
            // TMA store, unless a row takes the mean of V (then rows are stored directly).
            const bool o_tma = kSplitO && P.o_tma && !__any_sync(0xffffffffu, direct && pe.row_ok);
            auto stage16 = [&](uint32_t c, uint32_t w0_, uint32_t w1_, uint32_t w2_, uint32_t w3_) {
                st_shared_v4(o_stage + ((c ^ o_swz) << 4), w0_, w1_, w2_, w3_);
            };
            if (half_o == 32) {  // D in (48, 64]: this warp's 32 columns in one load
                uint32_t o[32];
                tmem_ld_x32(oa, o);
                if constexpr (kSplitO) {
                    uint32_t o1[32];
                    tmem_ld_x32(oa + P.o_cols, o1);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * w0 + __uint_as_float(o1[e]) * w1);
                }
                const float sc = kSplitO ? 1.f : inv;
                uint32_t wv[16];
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    wv[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * sc, __uint_as_float(o[2 * e + 1]) * sc);
                if (o_tma) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        stage16((uint32_t)(4 * h + i), wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                } else if (pe.row_ok && !direct) {
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (8 * i < dlim)
                            reinterpret_cast<uint4*>(op)[i] =
                                make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                }
            } else if (VARLEN && half_o % 32 == 0) {  // D > 64: 32 of this warp's columns per load
#pragma unroll 1
                for (uint32_t c0 = 0; c0 < half_o; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_x32(oa + c0, o);
                    uint32_t wv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        wv[e] = pack2<BF16>(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    if (pe.row_ok && !direct) {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if ((int)c0 + 8 * i < dlim)
                                reinterpret_cast<uint4*>(op + c0)[i] =
                                    make_uint4(wv[4 * i], wv[4 * i + 1], wv[4 * i + 2], wv[4 * i + 3]);
                    }
                }
            } else {
#pragma unroll 1
                for (uint32_t c0 = 0; c0 < half_o; c0 += 8) {
                    uint32_t o[8];
                    tmem_ld_x8(oa + c0, o);
                    if constexpr (kSplitO) {
                        uint32_t o1[8];
                        tmem_ld_x8(oa + P.o_cols + c0, o1);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * w0 + __uint_as_float(o1[e]) * w1);
                    }
                    const float sc = kSplitO ? 1.f : inv;
                    uint32_t wv[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        wv[e / 2] = pack2<BF16>(__uint_as_float(o[e]) * sc, __uint_as_float(o[e + 1]) * sc);
                    if (o_tma)
                        stage16(((uint32_t)h * half_o + c0) >> 3, wv[0], wv[1], wv[2], wv[3]);
                    else if (pe.row_ok && !direct && (int)c0 < dlim)
                        *reinterpret_cast<uint4*>(op + c0) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
            }
            if (o_tma) {
                // Both warps of the lane quarter have staged their columns: one store of
                // 32 rows x D (rows past Q are not written).
                fence_async_shared();
                if (!pair_sync()) return ok = false;
                if (h == 0 && lane == 0 && pe.box_row < a.Q) {
                    tma_store_3d(&P.tm_o, base + L.ostage + (uint32_t)(wq * 32 * P.o_rowb), 0, pe.box_row,
                                 pe.box_unit);
                    bulk_commit();
                }
            }
            if (OB == 1) {
                // Every load of O has completed (tcgen05.wait::ld in the loads): the
                // accumulator may take the next item's first PV.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_empty);
            }
            if (h == 0 && __any_sync(0xffffffffu, direct && pe.row_ok))
                split_mean_v<BF16>(a, orow_p, ra.v_base, ra.v_stride, ra.nkeys, direct && pe.row_ok);
            return true;
        };

        uint32_t qi = 0;  // items with key tiles so far: O accumulator qi % 2
        ItemWalk<VARLEN> walk;
        walk.begin(P, ring);
        SItem it;
        while (ok && walk.next(P, ring, it)) {
            const int qrow = it.qt * kBM + r;  // local query row
            const bool row_ok = qrow < it.Lq;
            if (VARLEN && it.nkt == 0) {
                // Packed form, a q block that visits no key block: every logit is
                // -1e9 (mean of V over the sequence's keys), or there are no keys
                // (O = 0, lse = max = -inf).
                if (h == 0) {
                    const RowAddr ra = row_addr((long long)it.q_row0 + qrow, it.k_row0, it.h, it.Lk);
                    if (row_ok) {
                        if (a.lse) a.lse[ra.lse_idx] = ra.nkeys > 0 ? kMasked + logf((float)ra.nkeys) : -INFINITY;
                        if (a.mx) a.mx[ra.lse_idx] = ra.nkeys > 0 ? kMasked : -INFINITY;
                    }
                    if (__any_sync(0xffffffffu, row_ok))
                        split_mean_v<BF16>(a, static_cast<uint16_t*>(a.out) + ra.out_off, ra.v_base, ra.v_stride,
                                           ra.nkeys, row_ok);
                }
                continue;
            }
            const uint32_t ob = OB == 1 ? 0u : (qi & 1u);
            ++qi;
            const uint32_t o_taddr = o_base + ob * o_set;
            float m_true = -INFINITY, m_ref = 0.f, l = 0.f;
            // O *= alpha in this warp's columns, once PV of the previous tile is in O.
            auto rescale_o = [&](float alpha) -> bool {
                if (!wait_pv(sn - 1u, false)) return false;
                for (uint32_t c0 = 0; c0 < (kSplitO ? P.o_cols : half_o); c0 += 8) {
                    uint32_t o[8];
                    tmem_ld_x8(o_taddr + c0, o);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_x8(o_taddr + c0, o);
                }
                return true;
            };
            int jv = 0;
            const int prefix_lm = !VARLEN ? 0 : (a.prefix_len ? a.prefix_len[it.seq] : a.prefix_all);
            TileWalk tw = tiles_begin<VARLEN>(it);
            int kb;
            bool is_full;
            while (ok && tiles_next<VARLEN>(it, tw, kb, is_full)) {
                const int key0 = kb * kBN;
                int vlim;
                bool modded = false;  // mask_mod applies (a partial block)
                if constexpr (!VARLEN) {
                    vlim = P.mask_kind == 1 ? it.prefix : a.K;
                } else {
                    vlim = it.Lk;
                    modded = !is_full && a.mask_mod != TA_MASK_NONE;
                }
                const bool all_valid = (VARLEN || P.mask_kind != 2) && key0 + kBN <= vlim &&
                                       (!modded || mod_tile_all(a.mask_mod, it.qt * kBM, key0, a.window, prefix_lm));
                const int nexist = (VARLEN ? it.Lk : a.K) - key0;
                int bs = 0;
                uint32_t boff = 0, mwoff = 0;
                if constexpr (BIAS) {
                    bs = br.idx;
                    // Both barriers tested at once; the bounded waits only when one is not ready.
                    const bool ready = mbar_test(bias_full(bs), br.ph) & mbar_test(s_full(sb), (uint32_t)sph);
                    if (!__all_sync(0xffffffffu, ready)) {
                        ok = __all_sync(0xffffffffu, wait_bar(bias_full(bs), br.ph, abort_flag, a.status));
                        if (!ok) break;
                        ok = __all_sync(0xffffffffu, wait_bar(s_full(sb), (uint32_t)sph, abort_flag, a.status));
                        if (!ok) break;
                    }
                    boff = bias_smem(bs) - base + rrow;
                    mwoff = L.maskw + (uint32_t)bs * 16u;
                } else {
                    ok = __all_sync(0xffffffffu, wait_bar(s_full(sb), (uint32_t)sph, abort_flag, a.status));
                    if (!ok) break;
                }
                const uint32_t s_taddr = tmem + lane_off + 128u * (uint32_t)sb;
                tc_fence_after();

                // ---- x: this warp's 64 values of the row (logits, or raw S in the folded form).
                float x[64];
                {
                    uint32_t sr[64];
                    tmem_ld_x64(s_taddr + 64u * (uint32_t)h, sr);
                    if constexpr (FOLD) {
#pragma unroll
                        for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(sr[j]);
                    } else if constexpr (!BIAS) {
#pragma unroll
                        for (int j = 0; j < 64; j += 2) {
                            const float2 r2 =
                                __fmul2_rn(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])), scale2);
                            x[j] = r2.x;
                            x[j + 1] = r2.y;
                        }
                    } else if constexpr (!BIAS_F32) {
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
                // Per 32 keys: vm bit j = key valid, em bit j = key exists.
                if (!all_valid) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int k0 = 64 * h + 32 * hh;
                        const uint32_t em = low_bits(nexist - k0);
                        uint32_t vm = em & low_bits(vlim - key0 - k0);
                        if constexpr (!VARLEN) {
                            if (P.mask_kind == 2)
                                vm &= *reinterpret_cast<const uint32_t*>(gbase + mwoff + 4u * (uint32_t)(2 * h + hh));
                        } else {
                            if (modded) vm &= mod_bits(a.mask_mod, qrow, key0 + k0, a.window, prefix_lm);
                        }
                        // (em and vm are uniform across the warp: the branches do not diverge)
                        if (em == 0xffffffffu) {  // every key exists: valid, or masked to -1e9
                            if (vm != em) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) x[32 * hh + j] = ((vm >> j) & 1u) ? x[32 * hh + j] : kMaskVal;
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                x[32 * hh + j] =
                                    ((vm >> j) & 1u) ? x[32 * hh + j] : (((em >> j) & 1u) ? kMaskVal : -INFINITY);
                        }
                    }
                }
                if constexpr (BIAS) {
                    __syncwarp();  // every lane of the warp has read its bias and the mask words
                    if (lane == 0) mbar_arrive(bias_empty(bs));
                    br.next(BS);
                }

                // ---- Row max of the tile (units of this form): this half's, then the partner's.
                float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; j += 8) {
                    m0 = max3(m0, x[j], x[j + 1]);
                    m1 = max3(m1, x[j + 2], x[j + 3]);
                    m2 = max3(m2, x[j + 4], x[j + 5]);
                    m3 = max3(m3, x[j + 6], x[j + 7]);
                }
                const float mh = fmaxf(max3(m0, m1, m2), m3);
                const float tm = kSplitO ? mh : fmaxf(mh, swap(xbuf + (sn & 1u) * 256u, mh));
                if (!ok) break;
                float tm_nat;  // the tile max as a logit (natural units)
                if constexpr (FOLD) tm_nat = tm > -FLT_MAX ? tm * a.scale : (tm == -FLT_MAX ? kMasked : -INFINITY);
                else tm_nat = tm;
                m_true = fmaxf(m_true, tm_nat);
                // A new reference max (rows whose max grew by more than 2^8): l and O are
                // scaled by alpha.  Both warps of the lane quarter take this branch for the
                // same rows (same tile max, same reference); each scales its O columns once O
                // holds the previous tile.  Packed form: O after this tile's P is in tensor
                // memory (the logits are no longer live there, which spares registers).
                float alpha = 1.f;
                bool rescale = false;
                if (jv == 0) {
                    m_ref = tm;
                    l = 0.f;
                } else {
                    const float m_new = fmaxf(m_ref, tm);
                    const bool need = (m_new - m_ref) * unit_l2e > kRescaleLog2;
                    if (__any_sync(0xffffffffu, need)) {
                        rescale = true;
                        alpha = ex2((m_ref - m_new) * unit_l2e);
                        l *= alpha;
                        m_ref = m_new;
                        if constexpr (!VARLEN) {
                            ok = rescale_o(alpha);
                            if (!ok) break;
                        }
                    }
                }

                // ---- P for this warp's 64 keys into the S buffer (16-bit pairs).  A row
                // with no real logit yet takes weights of exactly 1 for masked keys
                // and 0 for absent ones: x + (-kMaskVal) is then 0 or -inf.
                const bool live = m_ref > kMaskVal;
                const float2 ul2 = live ? make_float2(unit_l2e, unit_l2e) : make_float2(1.f, 1.f);
                const float nb = live ? -m_ref * unit_l2e : -kMaskVal;
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
                // Split O: each key half writes P into the first 32 of its own 64 logit
                // columns, so no warp overwrites values its partner has yet to read.
                // Shared O: P of both halves in columns [0, 64), after the exchange.
                tmem_st_x32(s_taddr + (kSplitO ? 64u : 32u) * (uint32_t)h, pk);
                l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                if (VARLEN && rescale) {  // (this tile's P is not given yet)
                    ok = rescale_o(alpha);
                    if (!ok) break;
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
#ifdef TRIATTN_TEST_MISSING_ARRIVAL
                // Test builds of the failure path only: softmax warp 0 of CTA 0 withholds
                // its arrival for the first P, so the MMA warp's bounded wait for it runs
                // out and the CTA takes the abort path (status TA_ERR_TIMEOUT).
                const bool give = !(blockIdx.x == 0 && warp == 0 && sn == 0);
#else
                constexpr bool give = true;
#endif
                if (lane == 0 && give) mbar_arrive(p_full(sb));
                ++sn;
                if (++sb == SB) {
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
            if constexpr (!VARLEN) {
                pe.box_row = it.qt * kBM + wq * 32;
                pe.box_unit = (int)it.unit;
                pe.row0 = it.unit * a.Q + qrow;
                pe.unit0 = (long long)it.b * a.vs[0] + (it.bn - (long long)it.b * a.N) * a.vs[1] +
                           (long long)it.h * a.vs[2];
            } else {
                pe.row0 = (long long)it.q_row0 + qrow;
                pe.unit0 = it.k_row0;
                pe.hh = it.h;
                pe.nk = it.Lk;
            }
            pe.n_last = sn - 1u;
            pe.ob = ob;
            pe.row_ok = row_ok;
            // (triangle form: every key block of K; packed form: of the sequence).  Split O:
            // only the "not every block" part here; the epilogue adds the combined max.
            pe.direct = (kSplitO || !(m_true > kMasked)) && jv != (VARLEN ? it.nkb : (a.K + kBN - 1) / kBN);
            pend = true;
        }
        if (ok && pend) ok = epilogue(true);
        if (P.o_tma && h == 0 && lane == 0) bulk_wait_all();  // this lane quarter's O stores are done
        if (!ok) {
            *abort_flag = 1;
            named_barrier_arrive(1 + wq, 64);  // releases a partner inside pair_sync
        }
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

template <bool BF16, bool BIAS_F32, bool VARLEN, bool FOLD, bool BIAS>
cudaError_t launch_split(const TcParams& P, int grid, cudaStream_t stream) {
    const SplitLayout L = make_split_layout(P);
    const size_t smem = L.total + 1024;
    auto kern = tc_split_kernel<BF16, BIAS_F32, VARLEN, FOLD, BIAS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kSplitThreads, smem, stream>>>(P);
    return cudaGetLastError();
}

// Triangle form (bias dtype) and packed form (folded scale or not).
// Triangle form (bias dtype); packed form without a bias (folded scale or not) and
// with a post-scale bias (bias dtype).
#define TRIATTN_SPLIT_TRI_VARIANTS(X) X(true, false, false, false, true) X(true, true, false, false, true) \
    X(false, false, false, false, true) X(false, true, false, false, true)
#define TRIATTN_SPLIT_VARLEN_VARIANTS(X) X(true, false, true, true, false) X(true, false, true, false, false) \
    X(false, false, true, true, false) X(false, false, true, false, false)
#define TRIATTN_SPLIT_VARLEN_BIAS_VARIANTS(X) X(true, false, true, false, true) X(true, true, true, false, true) \
    X(false, false, true, false, true) X(false, true, true, false, true)
#define TRIATTN_SPLIT_EXTERN(b, f, v, fo, bi) \
    extern template cudaError_t launch_split<b, f, v, fo, bi>(const TcParams&, int, cudaStream_t);
#define TRIATTN_SPLIT_INSTANTIATE(b, f, v, fo, bi) \
    template cudaError_t launch_split<b, f, v, fo, bi>(const TcParams&, int, cudaStream_t);

}  // namespace tc
}  // namespace triattn
