// tc_kernel.cuh -- tcgen05 / TMA forward for fp16 and bf16 inputs (sm_103a).
// Instantiated by the tc_inst_*.cu files, launched from tc_fwd.cu.
//
// Computes the cuEquivariance triangle_attention formula
//   O_q = sum_k softmax_k(x) V_k,  x_k = s (Q_q . K_k) + B_qk if key k is valid, else -1e9
// with lse = log sum exp(x) and max = max x per row, and the same for packed
// sequences under a tensorplay BlockMask (full_kv_* blocks skip mask_mod).
//
// One persistent CTA per SM walks a static list of work items.  A work item
// holds NQ (1 or 2) query tiles of 128 rows that share one stream of key /
// value tiles: adjacent q tiles of one (b,n,h) slab (triangle form), or
// adjacent 128-row q blocks of one (sequence, head) (packed form, where each
// q block visits only the kv blocks its lists name).  Warp roles:
//   warps 0 .. 4*NQ-1  softmax: warpgroup i owns query tile i, one thread per
//                      row (= TMEM lane).  A tile's 128 logits of a row are
//                      read from TMEM into registers at once; bias, mask,
//                      row max and the exponentials (packed f32x2 arithmetic)
//                      are formed there, and P goes back to TMEM as 16-bit
//                      pairs; epilogue O / l, lse, max;
//   warp 4*NQ          producer: TMA loads of Q, K and V tiles into a
//                      128B-swizzled shared-memory ring;
//   warp 4*NQ+1        MMA: one thread issues tcgen05.mma
//                      S_i = Q_i K^T (both operands in shared memory, fp32 in
//                      TMEM) and O_i += P_i V (P from TMEM, V from shared);
//   warp 4*NQ+2        bias producer (triangle form): TMA loads of bias tiles
//                      and the dense-mask bits, so that waiting for a free
//                      bias stage never holds back a K/V load;
// Tensor memory: S_i at columns [128 i, 128 i + 128), O_i after all S tiles.
// With NQ = 2 the MMAs of one tile run while the other tile's softmax does:
// the tensor core alternates between the two query tiles.
//
// Masking: a masked key's logit is replaced by -1e9; a key past the end of
// its sequence (ragged tail) gets -inf and takes no part.  With kv_lengths,
// key tiles past the prefix are not visited: they contribute exp(-1e9 - m)
// = 0 exactly when the row has a valid key.  A row with no valid key has
// every logit -1e9: its output is the mean of V over all keys (weights of
// exactly 1 through the tensor core, or formed directly from V when some
// key blocks were not visited).  The running max used for the exponentials
// is only raised when the row max grows by more than 2^8 (in exp2 units), so
// O is rescaled rarely; lse uses the same reference, so the result is
// unchanged.
//
// Every mbarrier wait is bounded: after ~2 s the waiting thread records
// TA_ERR_TIMEOUT in the status word, raises a CTA-wide abort flag and all
// roles leave their loops; the TMEM allocation is always released.

#include <cuda.h>
#include <cfloat>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#pragma once

#include <cstring>

#include "internal.h"
#include "tmem_io.h"

namespace triattn {
namespace tc {

// Host helpers defined in tc_fwd.cu.
bool encode_map_3d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle sw);
int device_sm_count();

constexpr int kBM = 128;                    // query rows per tile
constexpr int kBN = 128;                    // keys per tile
constexpr uint32_t kBox = 128 * 128;        // one [128 rows][128 B] swizzled TMA box
constexpr float kMasked = -1.0e9f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;        // rescale O when the row max grows by > 2^8
// Cycles a bounded wait spins before it gives up (about 2 s).  Test builds of
// the failure path shorten it with -DTRIATTN_WAIT_LIMIT_CYCLES.
#ifndef TRIATTN_WAIT_LIMIT_CYCLES
#define TRIATTN_WAIT_LIMIT_CYCLES 4000000000LL
#endif
constexpr long long kTimeoutCycles = TRIATTN_WAIT_LIMIT_CYCLES;

// Division by a divisor fixed at launch, for 0 <= n < 2^31 (multiply-high
// and shift with a host-computed magic number, Granlund and Montgomery's
// round-up method): a handful of instructions instead of a full division.
struct FastDiv {
    uint32_t d, m, l;
#ifdef __CUDACC__
    __device__ __forceinline__ uint32_t div(uint32_t n) const { return (__umulhi(n, m) + n) >> l; }
#endif
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.l = 0;
    while ((1ull << f.l) < d) ++f.l;
    f.m = (uint32_t)((((1ull << 32) * ((1ull << f.l) - d)) / d) + 1);
    return f;
}

struct TcParams {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    CUtensorMap tm_bias;
    AttnParams a;
    int nsub;           // 64-column boxes covering D (1 or 2)
    int ksteps;         // ceil(D/16): K steps of the QK^T MMA
    int npv;            // N of the PV MMA (multiple of 16)
    int nqt;            // q tiles per unit (triangle) or per longest sequence (varlen)
    int items;          // work items
    int items_per_unit; // ceil(nqt / NQ)
    int q_bufs;         // Q buffers per query tile (2: the next item's Q loads during this one)
    int kv_stages;
    int bias_stages;    // per query tile; 0 for varlen
    int bias_boxes;     // TMA boxes per bias tile
    int bias_box_cols;  // keys per bias box
    uint32_t tile_bytes;
    uint32_t bias_bytes;
    uint32_t idesc_qk;
    uint32_t idesc_pv;
    uint32_t tmem_cols;
    uint32_t o_col0;    // first TMEM column of O_0
    uint32_t o_cols;    // TMEM columns per O tile
    int mask_kind;      // triangle: 0 none, 1 kv_lengths, 2 dense
    FastDiv fd_ipu;     // items_per_unit
    FastDiv fd_n;       // N (triangle)
    FastDiv fd_h;       // H
    FastDiv fd_per;     // num_seqs * H (packed form)
    // Folded softmax (packed form, scale > 0): the softmax reads raw S = Q K^T
    // and applies s inside the exponent.
    float scale_log2e;  // s * log2(e)
    // Key-split kernel only: S buffers (3 with D <= 64, 2 above), O accumulators
    // (2), and the divisor 2 * grid of the packed form's serpentine deal.
    int s_bufs;
    int o_bufs;
    FastDiv fd_2g;
    // Triangle form: q / k / v maps are 5-D {D, rows, H, N, B} (strided views), or
    // 3-D {D, rows, B*N*H} for contiguous tensors.
    int tri5d;
    // Key-split kernel, triangle form: O leaves through shared memory and a TMA
    // tensor store of 32 rows x D per TMEM lane quarter (o_tma = 1; map
    // {D, Q, B*N*H}, rows of o_rowb = 2 D bytes, swizzled by the row width).
    CUtensorMap tm_o;
    int o_tma;
    int o_rowb;
};

// ---------------------------------------------------------------------------
// Shared-memory layout (offsets from a 1024-byte aligned base)
// ---------------------------------------------------------------------------

struct Layout {
    uint32_t q, kv, bias, maskw, bars, tmem_slot, abort_flag, total;
    int nbars;
};

__host__ __device__ inline Layout make_layout(int NQ, const TcParams& P) {
    Layout L;
    L.q = 0;
    L.kv = L.q + NQ * P.q_bufs * P.tile_bytes;
    L.bias = L.kv + P.kv_stages * 2 * P.tile_bytes;
    L.maskw = L.bias + NQ * P.bias_stages * P.bias_bytes;
    L.bars = L.maskw + NQ * (P.bias_stages > 0 ? P.bias_stages : 1) * 16;
    L.nbars = NQ * P.q_bufs + P.q_bufs + 2 * P.kv_stages + 2 * NQ * P.bias_stages + 3 * NQ + 1;
    L.tmem_slot = L.bars + 8 * L.nbars;
    L.abort_flag = L.tmem_slot + 4;
    L.total = L.abort_flag + 4;
    return L;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// A waiting thread is suspended (up to the hint, in ns) instead of spinning,
// so it leaves issue slots to the warps that are computing.
constexpr uint32_t kSuspendHintNs = 1000000;
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns false if the CTA is aborting or the wait ran out.
// The common case (phase already complete) is an inline test; the waiting
// loop is one out-of-line function shared by every call site, which keeps
// the code small.
static __device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  int* status) {
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kTimeoutCycles) {
                *abort_flag = 1;
                atomicCAS(status, 0, kStatusTimeout);
                return false;
            }
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    return mbar_test(bar, parity) || wait_bar_slow(bar, parity, abort_flag, status);
}

// Bounded wait that ignores the abort flag (teardown drains only).
__device__ __forceinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > kTimeoutCycles / 8) return false;
    return true;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

// TMA tensor store of a shared-memory box (bulk-group completion) and the
// bulk-group waits: `.read` waits until the source may be overwritten.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* tm, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(tm)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Generic-proxy shared-memory writes made visible to the async proxy (TMA).
__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Hardware named barrier `id` over `threads` threads (whole warps): wait, or arrive only.
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void named_barrier_arrive(int id, int threads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}

// A triangle-form q / k / v tile: rows [row, row + 128) of slab (b, n, h) from
// the 3-D (contiguous) or 5-D (strided) map.
__device__ __forceinline__ void tma_load_tri(const TcParams& P, uint32_t dst, const CUtensorMap* tm, int c0, int row,
                                             long long unit, int h, int n, int b, uint32_t bar) {
    if (P.tri5d) tma_load_5d(dst, tm, c0, row, h, n, b, bar);
    else tma_load_3d(dst, tm, c0, row, (int)unit, bar);
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 form): start >> 4 at [0,14), leading
// byte offset >> 4 at [16,30), stride byte offset >> 4 at [32,46), fixed 0b001
// at [46,49), swizzle mode at [61,64) (2 = 128-byte swizzle).  Adding n to the
// descriptor moves its start address by 16 n bytes.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// One lane of a converged warp (elect.sync); the same lane every time.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Two 16-bit values of one 32-bit word (low half first) widened to fp32.
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    if constexpr (BF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        return __half22float2(*reinterpret_cast<const __half2*>(&w));
    }
}

template <bool BF16>
__device__ __forceinline__ float load16(const void* base, long long i) {
    const unsigned short u = static_cast<const unsigned short*>(base)[i];
    if constexpr (BF16) return __uint_as_float((uint32_t)u << 16);
    else return __half2float(__ushort_as_half(u));
}

__device__ __forceinline__ uint32_t low_bits(int n) {
    return n >= 32 ? 0xffffffffu : (n <= 0 ? 0u : ((1u << n) - 1u));
}

// BlockMask mask_mod on a partial block (tensorplay BlockMask page, Details 2),
// local indices: bit j of the result says key kg + j is kept for query q.
//   causal          k <= q
//   sliding window  q - window < k <= q
//   prefix LM       k <= q or k < prefix
__device__ __forceinline__ uint32_t mod_bits(int mod, int q, int kg, int window, int prefix) {
    const uint32_t causal = low_bits(q - kg + 1);
    switch (mod) {
    case TA_MASK_CAUSAL: return causal;
    case TA_MASK_SLIDING_WINDOW: return causal & ~low_bits(q - window + 1 - kg);
    case TA_MASK_PREFIX_LM: return causal | low_bits(prefix - kg);
    default: return 0xffffffffu;
    }
}

// True when mask_mod keeps every key of [key0, key0 + 128) for every query of
// [q0, q0 + 128).
__device__ __forceinline__ bool mod_tile_all(int mod, int q0, int key0, int window, int prefix) {
    const bool causal = key0 + 127 <= q0;
    switch (mod) {
    case TA_MASK_CAUSAL: return causal;
    case TA_MASK_SLIDING_WINDOW: return causal && (q0 + 127) - key0 < window;
    case TA_MASK_PREFIX_LM: return causal || key0 + 128 <= prefix;
    default: return true;
    }
}

// Position in a ring of n pipeline stages: the stage, the parity of the
// current pass over the ring, and whether the stage was used before (its
// "empty" barrier then has to complete first, in the previous pass's parity).
// Advanced one use at a time, so the per-tile path has no runtime division.
struct StageRing {
    int idx;
    uint32_t ph;
    bool wrapped;
    __device__ __forceinline__ void next(int n) {
        if (++idx == n) {
            idx = 0;
            ph ^= 1u;
            wrapped = true;
        }
    }
};

// ---------------------------------------------------------------------------
// Work items and their key-tile streams
// ---------------------------------------------------------------------------

template <int NQ>
struct Item {
    bool on[NQ];        // the query tile has rows
    int qt[NQ];         // q tile (triangle) / q block (varlen) index per slot
    long long unit;     // triangle: (b*N+n)*H+h
    long long bn;       // triangle: b*N+n
    int b, h, seq;
    int Lq, Lk;         // query rows / keys of the unit
    int q_row0, k_row0; // varlen: first packed row of the sequence
    int prefix;         // triangle kv_lengths (clamped)
    int nkb;            // key blocks that may be visited
    bool bad;           // varlen: the sequence breaks the max_seqlen / total contract
    bool lists;         // varlen: BlockMask lists given
    bool any;           // something for the producer / MMA to do
    const int32_t* full_l[NQ];
    const int32_t* part_l[NQ];
    int n_full[NQ];
    int n_part[NQ];
};

// The kv_lengths entry of triangle item `item` (0 without kv_lengths or past
// the last item).  The roles that walk items load it one item ahead, so the
// load's latency overlaps the current item instead of stalling the next decode.
__device__ __forceinline__ int tri_item_len(const TcParams& P, int item) {
    if (P.mask_kind != 1 || item >= P.items) return 0;
    const uint32_t u2 = P.fd_ipu.div((uint32_t)item);
    const uint32_t bh = P.fd_n.div(u2);
    const int n = (int)(u2 - bh * P.fd_n.d);
    const int b = (int)P.fd_h.div(bh);
    return __ldg(P.a.kv_len + ((long long)b * P.a.N + n));
}
constexpr int kNoLen = -0x7fffffff - 1;  // decode loads the kv_lengths entry itself

template <int NQ, bool VARLEN>
__device__ Item<NQ> decode(const TcParams& P, int item, int pre_len = kNoLen) {
    Item<NQ> it;
    const AttnParams& a = P.a;
    it.bad = false;
    it.lists = false;
    it.prefix = 0;
    it.seq = 0;
    it.q_row0 = 0;
    it.k_row0 = 0;
    for (int i = 0; i < NQ; ++i) {
        it.full_l[i] = nullptr;
        it.part_l[i] = nullptr;
        it.n_full[i] = 0;
        it.n_part[i] = 0;
    }
    if constexpr (!VARLEN) {
        const uint32_t u2 = P.fd_ipu.div((uint32_t)item);  // ((b*H + h)*N + n): n fastest, so bias tiles are reused from L2
        const int qp = item - (int)(u2 * P.fd_ipu.d);
        const uint32_t bh = P.fd_n.div(u2);
        const int n = (int)(u2 - bh * P.fd_n.d);
        it.b = (int)P.fd_h.div(bh);
        it.h = (int)(bh - (uint32_t)it.b * P.fd_h.d);
        it.bn = (long long)it.b * a.N + n;
        it.unit = it.bn * a.H + it.h;
        it.Lq = a.Q;
        it.Lk = a.K;
        bool any_on = false;
        for (int i = 0; i < NQ; ++i) {
            it.qt[i] = qp * NQ + i;
            it.on[i] = it.qt[i] < P.nqt;
            any_on = any_on || it.on[i];
        }
        it.nkb = (a.K + kBN - 1) / kBN;
        if (P.mask_kind == 1) {
            // Key tiles past the prefix are skipped.  With no valid key at all,
            // every tile is visited with every logit at -1e9 (uniform weights).
            const int L = pre_len != kNoLen ? pre_len : a.kv_len[it.bn];
            it.prefix = L < 0 ? 0 : (L > a.K ? a.K : L);
            if (it.prefix > 0) it.nkb = (it.prefix + kBN - 1) / kBN;
        }
        it.any = any_on && it.nkb > 0;
        return it;
    } else {
        // Heaviest q blocks first (a later q block sees more causal kv blocks).
        const uint32_t qq = P.fd_per.div((uint32_t)item);
        const int qp = P.items_per_unit - 1 - (int)qq;
        const uint32_t sh = (uint32_t)item - qq * P.fd_per.d;
        it.seq = (int)P.fd_h.div(sh);
        it.h = (int)(sh - (uint32_t)it.seq * P.fd_h.d);
        it.b = 0;
        it.bn = 0;
        it.unit = 0;
        const int cq0 = a.cu_q[it.seq], cq1 = a.cu_q[it.seq + 1];
        const int ck0 = a.cu_k[it.seq], ck1 = a.cu_k[it.seq + 1];
        it.q_row0 = cq0;
        it.k_row0 = ck0;
        it.Lq = cq1 - cq0;
        it.Lk = ck1 - ck0;
        const bool ok = it.Lq >= 0 && it.Lk >= 0 && it.Lq <= a.max_q && it.Lk <= a.max_k && cq0 >= 0 && ck0 >= 0 &&
                        cq1 <= a.total_q && ck1 <= a.total_k;
        it.bad = !ok;
        it.nkb = ok ? (it.Lk + kBN - 1) / kBN : 0;
        it.lists = a.kv_num != nullptr;
        bool any_on = false;
        const int hm = a.mask_heads == 1 ? 0 : it.h;
        for (int i = 0; i < NQ; ++i) {
            it.qt[i] = qp * NQ + i;
            it.on[i] = ok && it.qt[i] * kBM < it.Lq;
            any_on = any_on || it.on[i];
            if (it.on[i] && it.lists && it.qt[i] < a.MQ) {
                const long long row = ((long long)it.seq * a.mask_heads + hm) * a.MQ + it.qt[i];
                it.part_l[i] = a.kv_idx + row * a.MK;
                it.n_part[i] = min(max(a.kv_num[row], 0), a.MK);
                if (a.full_num) {
                    it.full_l[i] = a.full_idx + row * a.MK;
                    it.n_full[i] = min(max(a.full_num[row], 0), a.MK);
                }
            }
        }
        it.any = any_on && it.nkb > 0;
        return it;
    }
}

// Which slots visit key blocks [64w, 64w + 64): `full` blocks skip mask_mod,
// `part` blocks apply it (triangle: every block of the prefix is `part`; the
// softmax applies the triangle mask).  Rebuilt from the lists on every window,
// identically in every role.
template <int NQ, bool VARLEN>
__device__ __forceinline__ void window_masks(const Item<NQ>& it, int w, uint64_t (&full)[NQ], uint64_t (&part)[NQ]) {
    const int lo = 64 * w;
    const int n = min(64, it.nkb - lo);
    const uint64_t range = n >= 64 ? ~0ull : ((1ull << n) - 1ull);
    for (int i = 0; i < NQ; ++i) {
        full[i] = 0;
        part[i] = 0;
        if (!it.on[i]) continue;
        if (!VARLEN || !it.lists) {
            part[i] = range;
            continue;
        }
        for (int t = 0; t < it.n_part[i]; ++t) {
            const int kb = it.part_l[i][t] - lo;
            if (kb >= 0 && kb < n) part[i] |= 1ull << kb;
        }
        for (int t = 0; t < it.n_full[i]; ++t) {
            const int kb = it.full_l[i][t] - lo;
            if (kb >= 0 && kb < n) full[i] |= 1ull << kb;
        }
        part[i] &= ~full[i];
    }
}

// Calls f(kb, part_slots, full_slots) for every key block the item visits, in
// ascending order; bit i of part_slots says query tile i takes part in it,
// bit i of full_slots that it does so without mask_mod.  Stops when f
// returns false.  Every role walks the same sequence.
template <int NQ, bool VARLEN, typename F>
__device__ __forceinline__ void for_each_tile(const Item<NQ>& it, F&& f) {
    if constexpr (!VARLEN) {
        uint32_t on = 0;
        for (int i = 0; i < NQ; ++i) on |= it.on[i] ? (1u << i) : 0u;
        for (int kb = 0; kb < it.nkb; ++kb)
            if (!f(kb, on, 0u)) return;
    } else {
        for (int w = 0; w * 64 < it.nkb; ++w) {
            uint64_t fm[NQ], pm[NQ];
            window_masks<NQ, VARLEN>(it, w, fm, pm);
            uint64_t uni = 0;
            for (int i = 0; i < NQ; ++i) uni |= fm[i] | pm[i];
            while (uni) {
                const int bit = __ffsll((long long)uni) - 1;
                uni &= uni - 1;
                uint32_t ps = 0, fs = 0;
                for (int i = 0; i < NQ; ++i) {
                    ps |= (uint32_t)(((fm[i] | pm[i]) >> bit) & 1ull) << i;
                    fs |= (uint32_t)((fm[i] >> bit) & 1ull) << i;
                }
                if (!f(64 * w + bit, ps, fs)) return;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

// Block size: NQ softmax warpgroups + producer, MMA and bias warps.
template <int NQ>
constexpr int kThreads = NQ * 128 + 96;

template <int NQ, bool VARLEN, bool BF16, bool BIAS_F32, bool FOLD>
__global__ void __launch_bounds__(kThreads<NQ>, 1) tc_fwd_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const Layout L = make_layout(NQ, P);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    constexpr int kProducerWarp = NQ * 4;
    constexpr int kMmaWarp = NQ * 4 + 1;
    constexpr int kBiasWarp = NQ * 4 + 2;
    const AttnParams& a = P.a;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L.abort_flag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.tmem_slot);

    const int S = P.kv_stages;
    const int BS = P.bias_stages;
    const int QB = P.q_bufs;
    const int b0 = NQ * QB + QB;  // first K/V barrier
    auto bar = [&](int idx) -> uint32_t { return base + L.bars + 8u * (uint32_t)idx; };
    auto q_full = [&](int i, int qb) { return bar(i * QB + qb); };
    auto q_empty = [&](int qb) { return bar(NQ * QB + qb); };
    auto kv_full = [&](int s) { return bar(b0 + s); };
    auto kv_empty = [&](int s) { return bar(b0 + S + s); };
    auto bias_full = [&](int i, int s) { return bar(b0 + 2 * S + i * BS + s); };
    auto bias_empty = [&](int i, int s) { return bar(b0 + 2 * S + NQ * BS + i * BS + s); };
    auto s_full = [&](int i) { return bar(b0 + 2 * S + 2 * NQ * BS + i); };
    auto p_full = [&](int i) { return bar(b0 + 2 * S + 2 * NQ * BS + NQ + i); };
    auto o_full = [&](int i) { return bar(b0 + 2 * S + 2 * NQ * BS + 2 * NQ + i); };
    const uint32_t drain = bar(b0 + 2 * S + 2 * NQ * BS + 3 * NQ);

    auto q_smem = [&](int i, int qb) { return base + L.q + (uint32_t)(i * QB + qb) * P.tile_bytes; };
    auto k_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes; };
    auto v_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes + P.tile_bytes; };
    auto bias_smem = [&](int i, int s) { return base + L.bias + (uint32_t)(i * BS + s) * P.bias_bytes; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
#pragma unroll 1
        for (int i = 0; i < NQ; ++i) {
#pragma unroll 1
            for (int qb = 0; qb < QB; ++qb) mbar_init(q_full(i, qb), 1);
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), 4);  // one arrival per softmax warp
            mbar_init(o_full(i), 1);
#pragma unroll 1
            for (int s = 0; s < BS; ++s) {
                mbar_init(bias_full(i, s), 1);
                mbar_init(bias_empty(i, s), 4);  // one arrival per softmax warp of the tile
            }
        }
#pragma unroll 1
        for (int qb = 0; qb < QB; ++qb) mbar_init(q_empty(qb), 1);
        mbar_init(drain, 1);
#pragma unroll 1
        for (int s = 0; s < S; ++s) {
            mbar_init(kv_full(s), 1);
            mbar_init(kv_empty(s), 1);
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
        // ------------------------------------------------- producer: Q, K, V tiles
        StageRing kr = {0, 0u, false}, qr = {0, 0u, false};
        bool ok = true;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<NQ> it = decode<NQ, VARLEN>(P, item);
            if (!it.any) continue;
            // Q of every slot goes to buffer set qr.idx (a slot without rows
            // gets an out-of-range, zero-filled box), so each q_full completes
            // once per item with work.
            const int qb = qr.idx;
            if (lane == 0 && qr.wrapped) ok = wait_bar(q_empty(qb), qr.ph ^ 1u, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                for (int i = 0; i < NQ; ++i) {
                    mbar_expect_tx(q_full(i, qb), P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb) {
                        if constexpr (!VARLEN)
                            tma_load_tri(P, q_smem(i, qb) + sb * kBox, &P.tm_q, sb * 64, it.qt[i] * kBM, it.unit,
                                         it.h, (int)(it.bn - (long long)it.b * a.N), it.b, q_full(i, qb));
                        else
                            tma_load_3d(q_smem(i, qb) + sb * kBox, &P.tm_q, sb * 64, it.h, it.q_row0 + it.qt[i] * kBM,
                                        q_full(i, qb));
                    }
                }
            }
            qr.next(QB);
            for_each_tile<NQ, VARLEN>(it, [&](int kb, uint32_t, uint32_t) -> bool {
                const int st = kr.idx;
                if (lane == 0 && kr.wrapped) ok = wait_bar(kv_empty(st), kr.ph ^ 1u, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) return false;
                if (lane == 0) {
                    mbar_expect_tx(kv_full(st), 2 * P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb) {
                        if constexpr (!VARLEN) {
                            const int n = (int)(it.bn - (long long)it.b * a.N);
                            tma_load_tri(P, k_smem(st) + sb * kBox, &P.tm_k, sb * 64, kb * kBN, it.unit, it.h, n, it.b,
                                         kv_full(st));
                            tma_load_tri(P, v_smem(st) + sb * kBox, &P.tm_v, sb * 64, kb * kBN, it.unit, it.h, n, it.b,
                                         kv_full(st));
                        } else {
                            tma_load_3d(k_smem(st) + sb * kBox, &P.tm_k, sb * 64, it.h, it.k_row0 + kb * kBN,
                                        kv_full(st));
                            tma_load_3d(v_smem(st) + sb * kBox, &P.tm_v, sb * 64, it.h, it.k_row0 + kb * kBN,
                                        kv_full(st));
                        }
                    }
                }
                kr.next(S);
                return true;
            });
        }
        if (!ok) *abort_flag = 1;
    } else if (!VARLEN && warp == kBiasWarp) {
        // ---------------------------------- producer: bias tiles (+ dense-mask bits)
        StageRing br[NQ];
#pragma unroll
        for (int i = 0; i < NQ; ++i) br[i] = {0, 0u, false};
        bool ok = true;
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<NQ> it = decode<NQ, VARLEN>(P, item);
            if (!it.any) continue;
            for_each_tile<NQ, VARLEN>(it, [&](int kb, uint32_t ps, uint32_t) -> bool {
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    if (!((ps >> i) & 1u)) continue;
                    const int bs = br[i].idx;
                    if (lane == 0 && br[i].wrapped) ok = wait_bar(bias_empty(i, bs), br[i].ph ^ 1u, abort_flag, a.status);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) return false;
                    if (P.mask_kind == 2) {
                        // 128 key-validity bits: word w, bit l <-> key kb*128 + 32w + l
                        uint32_t* mw = reinterpret_cast<uint32_t*>(gbase + L.maskw + (uint32_t)(i * BS + bs) * 16u);
                        for (int ww = 0; ww < 4; ++ww) {
                            const int key = kb * kBN + 32 * ww + lane;
                            const bool v = key < a.K && a.mask[it.bn * a.K + key] != 0;
                            const uint32_t word = __ballot_sync(0xffffffffu, v);
                            if (lane == ww) mw[ww] = word;
                        }
                        __syncwarp();
                    }
                    if (lane == 0) {
                        mbar_expect_tx(bias_full(i, bs), P.bias_bytes);
                        for (int bx = 0; bx < P.bias_boxes; ++bx)
                            tma_load_3d(bias_smem(i, bs) + bx * kBox, &P.tm_bias, kb * kBN + bx * P.bias_box_cols,
                                        it.qt[i] * kBM, it.b * a.H + it.h, bias_full(i, bs));
                    }
                    br[i].next(BS);
                }
                return true;
            });
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        // The whole warp runs this loop, so descriptors and counters are
        // warp-uniform values; one elected lane issues each tcgen05 instruction.
        const bool leader = elect_one();
        {
            StageRing kr = {0, 0u, false}, qr = {0, 0u, false};
            uint32_t p_it[NQ];
#pragma unroll
            for (int i = 0; i < NQ; ++i) p_it[i] = 0;
            bool ok = true;
            // Descriptor steps (units of 16 B): a K step of 16 inside a 128-byte
            // swizzle row is 32 bytes, the second 64-column box starts kBox
            // bytes later; 16 rows of V are 2048 bytes.
            auto kstep = [](int kk) -> uint64_t { return (uint64_t)(((kk >> 2) * kBox + (kk & 3) * 32) >> 4); };
            for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
                const Item<NQ> it = decode<NQ, VARLEN>(P, item);
                if (!it.any) continue;
                const int qb = qr.idx;
                for (int i = 0; i < NQ && ok; ++i)
                    ok = __all_sync(0xffffffffu, wait_bar(q_full(i, qb), qr.ph, abort_flag, a.status));
                qr.next(QB);
                if (!ok) break;
                uint64_t qd[NQ];
                uint32_t pend = 0;  // bit i: P_i of slot i's last tile is still to be multiplied by V
                int pst[NQ];
                uint32_t npv[NQ];
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    qd[i] = sw128_desc(q_smem(i, qb), 16, 1024);
                    pst[i] = 0;
                    npv[i] = 0;
                }
                int prev = -1;
                // O_i += P_i V, with V from stage `st` and P_i in S_i's columns.
                auto issue_pv = [&](int i, int st) {
                    const uint64_t vd = sw128_desc(v_smem(st), kBox, 1024);
                    const uint32_t d = tmem + P.o_col0 + i * P.o_cols;
                    const uint32_t pa = tmem + i * 128;
#pragma unroll 1
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        if (leader) mma_ts(d, pa + kk * 8, vd + (uint64_t)kk * 128, P.idesc_pv, (npv[i] > 0 || kk > 0) ? 1u : 0u);
                    ++npv[i];
                };
                for_each_tile<NQ, VARLEN>(it, [&](int, uint32_t ps, uint32_t) -> bool {
                    // Per slot: PV of its previous tile (frees S_i; that V is
                    // resident already), then QK of this tile.  Only QK waits for
                    // this tile's K/V, so a late load never holds back a PV.
                    const int st = kr.idx;
                    bool kv_ready = false;
                    auto wait_kv = [&]() -> bool {
                        if (kv_ready) return true;
                        kv_ready = true;
                        if (!__all_sync(0xffffffffu, wait_bar(kv_full(st), kr.ph, abort_flag, a.status)))
                            return false;
                        tc_fence_after();
                        return true;
                    };
                    const uint64_t kd = sw128_desc(k_smem(st), 16, 1024);
#pragma unroll
                    for (int i = 0; i < NQ; ++i) {
                        if ((pend >> i) & 1u) {
                            ok = __all_sync(0xffffffffu, wait_bar(p_full(i), p_it[i]++ & 1, abort_flag, a.status));
                            if (!ok) return false;
                            tc_fence_after();
                            issue_pv(i, pst[i]);
                            pend &= ~(1u << i);
                        }
                        if ((ps >> i) & 1u) {
                            ok = wait_kv();
                            if (!ok) return false;
                            const uint32_t sd = tmem + i * 128;
                            if (leader) {
                                mma_ss(sd, qd[i], kd, P.idesc_qk, 0u);
                                for (int kk = 1; kk < P.ksteps; ++kk)
                                    mma_ss(sd, qd[i] + kstep(kk), kd + kstep(kk), P.idesc_qk, 1u);
                                mma_commit(s_full(i));
                            }
                            pend |= 1u << i;
                            pst[i] = st;
                        }
                    }
                    if (prev >= 0 && leader) mma_commit(kv_empty(prev));  // no pending PV reads stage `prev` any more
                    ok = wait_kv();  // keeps the phases in step if no slot used this tile
                    if (!ok) return false;
                    kr.next(S);
                    prev = st;
                    return true;
                });
                if (!ok) break;
                if (leader) mma_commit(q_empty(qb));  // every QK of the item is issued: its Q buffers may be refilled
#pragma unroll
                for (int i = 0; i < NQ; ++i) {
                    if (!ok) break;
                    if ((pend >> i) & 1u) {
                        ok = __all_sync(0xffffffffu, wait_bar(p_full(i), p_it[i]++ & 1, abort_flag, a.status));
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(i, pst[i]);
                    }
                    if (npv[i] > 0 && leader) mma_commit(o_full(i));
                }
                if (!ok) break;
                if (prev >= 0 && leader) mma_commit(kv_empty(prev));
            }
            if (!ok && leader) *abort_flag = 1;
            // Let every MMA issued so far finish before TMEM is released.
            if (leader) mma_commit(drain);
            wait_bar_drain(drain, 0);
        }
        __syncwarp();
    } else if (warp < 4 * NQ) {
        // -------------------------------------------------------------- softmax
        const int slot = warp / 4;
        const int wq = warp % 4;               // TMEM lane quarter
        const int r = wq * 32 + lane;          // row within the q tile
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t s_taddr = tmem + lane_off + slot * 128;
        const uint32_t o_taddr = tmem + lane_off + P.o_col0 + slot * P.o_cols;
        // 128B swizzle: 16-byte chunk c of row r sits at chunk c ^ (r % 8).
        const uint32_t rsw = (uint32_t)(r & 7);
        const uint32_t rrow = (uint32_t)r * 128u;
        uint32_t s_it = 0, o_it = 0;
        StageRing br = {0, 0u, false};
        const float2 scale2 = make_float2(a.scale, a.scale);
        // Folded form (packed sequences, no bias): values are in units of S
        // (x = s S); a masked key holds -FLT_MAX there (its logit is -1e9).
        constexpr float kMaskVal = FOLD ? -FLT_MAX : kMasked;
        const float unit_l2e = FOLD ? P.scale_log2e : kLog2e;
        bool ok = true;

        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<NQ> it = decode<NQ, VARLEN>(P, item);
            if (VARLEN && it.bad && threadIdx.x == 0) atomicCAS(a.status, 0, kStatusDevice);
            const int prefix_lm = !VARLEN ? 0 : (a.prefix_len ? a.prefix_len[it.seq] : a.prefix_all);
            bool on_s = false;
            int qt_s = 0;
#pragma unroll
            for (int i = 0; i < NQ; ++i) {  // this slot's fields (constant indices keep Item in registers)
                if (i == slot) {
                    on_s = it.on[i];
                    qt_s = it.qt[i];
                }
            }
            if (!on_s) continue;
            const int qrow = qt_s * kBM + r;  // local query row
            float m_true = -INFINITY, m_ref = 0.f, l = 0.f;
            int jv = 0;
            for_each_tile<NQ, VARLEN>(it, [&](int kb, uint32_t ps, uint32_t fs) -> bool {
                if (!((ps >> slot) & 1u)) return true;
                const bool full = (fs >> slot) & 1u;
                const int key0 = kb * kBN;
                int vlim;
                bool modded = false;  // mask_mod applies (a partial block)
                if constexpr (!VARLEN) {
                    vlim = P.mask_kind == 1 ? it.prefix : a.K;
                } else {
                    vlim = it.Lk;
                    modded = !full && a.mask_mod != TA_MASK_NONE;
                }
                const bool all_valid = (VARLEN || P.mask_kind != 2) && key0 + kBN <= vlim &&
                                       (!modded || mod_tile_all(a.mask_mod, qt_s * kBM, key0, a.window, prefix_lm));
                const int nexist = (VARLEN ? it.Lk : a.K) - key0;

                uint32_t boff = 0, mwoff = 0;  // this row's bias / the mask words, from the aligned base
                int bs = 0;
                if constexpr (!VARLEN) {
                    bs = br.idx;
                    ok = __all_sync(0xffffffffu, wait_bar(bias_full(slot, bs), br.ph, abort_flag, a.status));
                    if (!ok) return false;
                    boff = bias_smem(slot, bs) - base + rrow;
                    mwoff = L.maskw + (uint32_t)(slot * BS + bs) * 16u;
                }
                ok = __all_sync(0xffffffffu, wait_bar(s_full(slot), s_it & 1, abort_flag, a.status));
                if (!ok) return false;
                ++s_it;
                tc_fence_after();

                // ---- Two chunks of 64 keys, one pass each: x = s S + bias (or raw S in
                // the folded form), masking at a boundary, the chunk max, then
                // P = 2^((x - m_ref) log2 e) into columns [32c, 32c + 32) as 16-bit
                // pairs (chunk c's values are in registers before any is overwritten).
                // The reference max m_ref follows the running max lazily: it is raised
                // only when the max grows by more than 2^kRescaleLog2, and raising it
                // scales O (complete through this slot's previous tile), l and, within
                // a tile, chunk 0's P.  The loops stay rolled so that the softmax code
                // fits the instruction cache next to the other roles.
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    float x[64];
                    {
                        uint32_t sr[64];
                        tmem_ld_x64(s_taddr + 64 * c, sr);
                        if constexpr (FOLD) {
#pragma unroll
                            for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(sr[j]);
                        } else if constexpr (VARLEN) {
#pragma unroll
                            for (int j = 0; j < 64; j += 2) {
                                const float2 r2 =
                                    __fmul2_rn(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])), scale2);
                                x[j] = r2.x;
                                x[j + 1] = r2.y;
                            }
                        } else if constexpr (!BIAS_F32) {
                            const uint32_t bbox = boff + (uint32_t)c * kBox;  // keys 64c .. 64c+63: box c
#pragma unroll
                            for (int g = 0; g < 8; ++g) {  // 8 keys per 16-byte chunk
                                const uint4 wv =
                                    *reinterpret_cast<const uint4*>(gbase + bbox + ((((uint32_t)g) ^ rsw) << 4));
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
                            for (int g = 0; g < 16; ++g) {  // 4 keys per 16-byte chunk; keys 64c.. in boxes 2c, 2c+1
                                const uint4 wv = *reinterpret_cast<const uint4*>(
                                    gbase + boff + (uint32_t)(2 * c + (g >> 3)) * kBox + ((((uint32_t)g & 7u) ^ rsw) << 4));
                                const int j = 4 * g;
                                const float2 r0 =
                                    __ffma2_rn(make_float2(__uint_as_float(sr[j]), __uint_as_float(sr[j + 1])), scale2,
                                               make_float2(__uint_as_float(wv.x), __uint_as_float(wv.y)));
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
                    // Masking (tiles at a boundary only; the branch is uniform across
                    // the warp).  Per 32 keys: vm bit j = key valid, em bit j = key exists.
                    if (!all_valid) {
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int k0 = 64 * c + 32 * h;
                            const uint32_t em = low_bits(nexist - k0);
                            uint32_t vm = em & low_bits(vlim - key0 - k0);
                            if constexpr (!VARLEN) {
                                if (P.mask_kind == 2)
                                    vm &= *reinterpret_cast<const uint32_t*>(gbase + mwoff + 4u * (uint32_t)(2 * c + h));
                            } else {
                                if (modded) vm &= mod_bits(a.mask_mod, qrow, key0 + k0, a.window, prefix_lm);
                            }
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                x[32 * h + j] =
                                    ((vm >> j) & 1u) ? x[32 * h + j] : (((em >> j) & 1u) ? kMaskVal : -INFINITY);
                        }
                    }
                    if (!VARLEN && c == 1) {
                        __syncwarp();  // every lane of the warp has read its bias row and the mask words
                        if (lane == 0) mbar_arrive(bias_empty(slot, bs));
                        br.next(BS);
                    }
                    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 64; j += 8) {
                        m0 = max3(m0, x[j], x[j + 1]);
                        m1 = max3(m1, x[j + 2], x[j + 3]);
                        m2 = max3(m2, x[j + 4], x[j + 5]);
                        m3 = max3(m3, x[j + 6], x[j + 7]);
                    }
                    // Chunk max (units of this form) and its logit in natural units.
                    const float cm = fmaxf(max3(m0, m1, m2), m3);
                    float cm_nat;
                    if constexpr (FOLD) cm_nat = cm > -FLT_MAX ? cm * a.scale : (cm == -FLT_MAX ? kMasked : -INFINITY);
                    else cm_nat = cm;
                    m_true = fmaxf(m_true, cm_nat);
                    if (jv == 0 && c == 0) {
                        m_ref = cm;
                        l = 0.f;
                    } else {
                        const float m_new = fmaxf(m_ref, cm);
                        const bool need = (m_new - m_ref) * unit_l2e > kRescaleLog2;
                        if (__any_sync(0xffffffffu, need)) {
                            const float alpha = ex2((m_ref - m_new) * unit_l2e);
                            l *= alpha;
                            m_ref = m_new;
                            if (jv > 0) {
                                for (uint32_t c0 = 0; c0 < P.o_cols; c0 += 16) {
                                    uint32_t o[16];
                                    tmem_ld_x16(o_taddr + c0, o);
#pragma unroll
                                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                                    tmem_st_x16(o_taddr + c0, o);
                                }
                            }
                            if (c == 1) {  // chunk 0's P, already in columns [0, 32)
                                tmem_st_wait();
                                uint32_t pr[32];
                                tmem_ld_x32(s_taddr, pr);
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    const float2 pv = unpack2<BF16>(pr[j]);
                                    pr[j] = pack2<BF16>(pv.x * alpha, pv.y * alpha);
                                }
                                tmem_st_x32(s_taddr, pr);
                            }
                        }
                    }
                    // A row with no real logit yet (every value masked or absent) takes
                    // weights of exactly 1 for masked keys and 0 for absent ones:
                    // x + (-kMaskVal) is then 0 or -inf.
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
                    tmem_st_x32(s_taddr + 32 * c, pk);
                    l += (acc0.x + acc0.y) + (acc1.x + acc1.y);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();  // one arrival per warp once all its lanes' P is in TMEM
                if (lane == 0) mbar_arrive(p_full(slot));
                ++jv;
                return true;
            });
            if (!ok) break;
            // ------------------------------------------------------- epilogue
            // A row that saw no valid key has every logit -1e9: uniform weights over
            // all keys, i.e. the mean of V.  If every key block was visited, the
            // tensor-core result O / l is already that mean (P was 1 on every key);
            // otherwise (a packed q block whose lists skip blocks) it is formed
            // here directly from V.  The loops stay rolled: this code runs once
            // per work item and must not crowd the softmax out of the
            // instruction cache.
            const bool seen = jv > 0 && m_true > kMasked;
            const bool covered = jv > 0 && jv == (it.Lk + kBN - 1) / kBN;
            const bool direct = !seen && !covered;
            if (jv > 0) {
                ok = __all_sync(0xffffffffu, wait_bar(o_full(slot), o_it & 1, abort_flag, a.status));
                ++o_it;
                if (!ok) break;
                tc_fence_after();
            }
            const bool row_ok = qrow < it.Lq;
            const long long orow = !VARLEN ? it.unit * a.Q + qrow : (long long)(it.q_row0 + qrow);
            uint16_t* op = static_cast<uint16_t*>(a.out) + (!VARLEN ? orow * a.D : (orow * a.H + it.h) * a.D);
            const float inv = (!direct && l > 0.f) ? 1.f / l : 0.f;
            if (jv > 0) {
#pragma unroll 1
                for (uint32_t c0 = 0; c0 < P.o_cols; c0 += 16) {
                    uint32_t o[16];
                    tmem_ld_x16(o_taddr + c0, o);
                    uint32_t wv[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2)
                        wv[e / 2] = pack2<BF16>(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                    if (row_ok && !direct && (int)c0 < a.D) {
                        uint4* dst = reinterpret_cast<uint4*>(op + c0);
                        dst[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        if ((int)c0 + 8 < a.D) dst[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
                    }
                }
            }
            if (__any_sync(0xffffffffu, direct || (jv == 0 && row_ok))) {
                // Rare: rows with no valid key whose blocks were not all visited,
                // and rows of a sequence with no keys (written as zeros).  Lane
                // l forms the means of columns l, l + 32, ...; each row then
                // takes its values by shuffles.
#pragma unroll 1
                for (int d0 = 0; d0 < a.D; d0 += 32) {
                    float mv = 0.f;
                    const int d = d0 + lane;
                    if (it.Lk > 0 && d < a.D) {
                        // V(key, d) at vcol0 + (vrow0 + key) * vstride + d
                        const long long vrow0 = !VARLEN ? 0 : (long long)it.k_row0;
                        const long long vstride = !VARLEN ? a.vs[3] : a.v_rs;
                        const long long vcol0 = !VARLEN ? (long long)it.b * a.vs[0] +
                                                              (it.bn - (long long)it.b * a.N) * a.vs[1] +
                                                              (long long)it.h * a.vs[2]
                                                        : (long long)it.h * a.D;
                        // Eight independent sums keep eight loads in flight.
                        float sum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                        int key = 0;
#pragma unroll 1
                        for (; key + 8 <= it.Lk; key += 8) {
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                sum[u] += load16<BF16>(a.v, (vrow0 + key + u) * vstride + vcol0 + d);
                        }
#pragma unroll 1
                        for (; key < it.Lk; ++key) sum[0] += load16<BF16>(a.v, (vrow0 + key) * vstride + vcol0 + d);
                        mv = (((sum[0] + sum[1]) + (sum[2] + sum[3])) + ((sum[4] + sum[5]) + (sum[6] + sum[7]))) /
                             (float)it.Lk;
                    }
#pragma unroll 1
                    for (int e = 0; e < 32 && d0 + e < a.D; ++e) {
                        const float m = __shfl_sync(0xffffffffu, mv, e);
                        if (row_ok && (direct || jv == 0)) op[d0 + e] = (uint16_t)(pack2<BF16>(m, 0.f) & 0xffffu);
                    }
                }
            }
            if (row_ok) {
                float lse, mx;
                if (it.Lk == 0) {
                    lse = -INFINITY;
                    mx = -INFINITY;
                } else if (direct) {
                    lse = kMasked + logf((float)it.Lk);
                    mx = kMasked;
                } else {
                    float mr = m_ref;
                    if constexpr (FOLD) mr = m_ref > -FLT_MAX ? m_ref * a.scale : kMasked;
                    lse = mr + logf(l);
                    mx = m_true;
                }
                const long long li = !VARLEN ? orow : (long long)it.h * a.total_q + orow;
                if (a.lse) a.lse[li] = lse;
                if (a.mx) a.mx[li] = mx;
            }
        }
        if (!ok) *abort_flag = 1;
    }

    // ---------------------------------------------------------------- teardown
    if (warp == kProducerWarp && lane == 0 && *abort_flag) {
        // Give TMA loads already issued time to land before the CTA exits.
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



template <int NQ, bool VARLEN, bool BF16, bool BIAS_F32, bool FOLD>
cudaError_t launch_kernel(const TcParams& P, int grid, cudaStream_t stream) {
    const Layout L = make_layout(NQ, P);
    const size_t smem = L.total + 1024;
    auto kern = tc_fwd_kernel<NQ, VARLEN, BF16, BIAS_F32, FOLD>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads<NQ>, smem, stream>>>(P);
    return cudaGetLastError();
}

// The kernel variants the host launches (each instantiated in one tc_inst_*.cu
// file).  The folded softmax is used by the packed form only.
#define TRIATTN_TC_VARIANTS(X)                  \
    X(1, false, true, false, false)             \
    X(1, false, true, true, false)              \
    X(2, false, true, false, false)             \
    X(2, false, true, true, false)              \
    X(1, false, false, false, false)            \
    X(1, false, false, true, false)             \
    X(2, false, false, false, false)            \
    X(2, false, false, true, false)             \
    X(2, true, true, false, false)              \
    X(2, true, true, false, true)               \
    X(2, true, false, false, false)             \
    X(2, true, false, false, true)

#define TRIATTN_TC_EXTERN(nq, v, b, f, fo) \
    extern template cudaError_t launch_kernel<nq, v, b, f, fo>(const TcParams&, int, cudaStream_t);
#define TRIATTN_TC_INSTANTIATE(nq, v, b, f, fo) \
    template cudaError_t launch_kernel<nq, v, b, f, fo>(const TcParams&, int, cudaStream_t);

}  // namespace tc
}  // namespace triattn
