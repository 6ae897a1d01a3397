// tc_fwd.cu -- tcgen05 / TMA forward for fp16 and bf16 inputs (sm_103a).
//
// Computes the cuEquivariance triangle_attention formula
//   O_q = sum_k softmax_k(x) V_k,  x_k = s (Q_q . K_k) + B_qk if key k is valid, else -1e9
// with lse = log sum exp(x) and max = max x per row, and the same for packed
// sequences under a tensorplay BlockMask (full_kv_* blocks skip mask_mod).
//
// One persistent CTA per SM walks a static list of work items.  A work item
// is NQ query tiles of 128 rows that share their key/value tiles (triangle
// form: adjacent q tiles of one (b,n,h) slab).  Warp roles:
//   warps 0 .. 4*NQ-1  softmax: warpgroup i owns query tile i, one thread per
//                      row (= TMEM lane); online softmax in fp32, P written
//                      back to TMEM as 16-bit, epilogue O / l and lse, max;
//   warp 4*NQ          producer: TMA loads of Q, K, V and bias tiles into a
//                      128B-swizzled shared-memory ring (+ dense-mask bits);
//   warp 4*NQ+1        MMA: one thread issues tcgen05.mma
//                      S_i = Q_i K^T (SS, fp32 in TMEM) and O_i += P_i V
//                      (A = P from TMEM, B = V from shared memory).
// Tensor memory: S_i at columns [128 i, 128 i + 128), O_i after all S tiles.
// With NQ = 2 the MMAs of one tile overlap the softmax of the other.
//
// Masking: a masked key's logit is replaced by -1e9; a key past the end of
// its sequence (ragged tail) gets -inf and takes no part.  With kv_lengths,
// key tiles past the prefix are not visited: they contribute exp(-1e9 - m)
// = 0 exactly when the row has a valid key.  A row with no valid key has
// every logit -1e9: its output is the mean of V over all keys, computed
// directly.  The running max used for the exponentials is only raised when
// the row max grows by more than 2^8 (in exp2 units), so O is rescaled
// rarely; lse uses the same reference, so the result is unchanged.
//
// Every mbarrier wait is bounded: after ~2 s the waiting thread records
// TA_ERR_TIMEOUT in the status word, raises a CTA-wide abort flag and all
// roles leave their loops; the TMEM allocation is always released.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "tmem_io.h"

namespace triattn {
namespace {

constexpr int kBM = 128;                    // query rows per tile
constexpr int kBN = 128;                    // keys per tile
constexpr uint32_t kBox = 128 * 128;        // one [128 rows][128 B] swizzled TMA box
constexpr float kMasked = -1.0e9f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;        // rescale O when the row max grows by > 2^8
constexpr long long kTimeoutCycles = 4000000000LL;

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
    int items_per_unit; // triangle: ceil(nqt / NQ)
    int kv_stages;
    int bias_stages;    // 0 for varlen
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
    L.kv = L.q + NQ * P.tile_bytes;
    L.bias = L.kv + P.kv_stages * 2 * P.tile_bytes;
    L.maskw = L.bias + NQ * P.bias_stages * P.bias_bytes;
    L.bars = L.maskw + NQ * (P.bias_stages > 0 ? P.bias_stages : 1) * 16;
    L.nbars = NQ + 1 + 2 * P.kv_stages + 2 * NQ * P.bias_stages + 3 * NQ + 1;
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
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: returns false if the CTA is aborting or the wait ran out.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
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

// Bounded wait that ignores the abort flag (teardown drains only).
__device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 form): start >> 4 at [0,14), leading
// byte offset >> 4 at [16,30), stride byte offset >> 4 at [32,46), fixed 0b001
// at [46,49), swizzle mode at [61,64) (2 = 128-byte swizzle).
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

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
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

template <bool BF16>
__device__ __forceinline__ float load16(const void* base, long long i) {
    const unsigned short u = static_cast<const unsigned short*>(base)[i];
    if constexpr (BF16) return __uint_as_float((uint32_t)u << 16);
    else return __half2float(__ushort_as_half(u));
}

// ---------------------------------------------------------------------------
// Work items
// ---------------------------------------------------------------------------

template <int NQ>
struct Item {
    bool slot_on[NQ];
    int qt[NQ];         // q tile per slot
    long long unit;     // triangle (b*N+n)*H+h
    int b, n, h, seq;
    int Lq, Lk;         // query rows / keys of the unit (local)
    int q_row0, k_row0; // varlen: first packed row of the sequence
    int prefix;         // triangle kv_lengths (clamped)
    long long bn;       // triangle b*N+n
    // key-tile enumeration: raw entries [0, n_raw)
    int n_raw;
    int n_full;         // varlen: leading entries taken from the full list
    const int32_t* full_list;
    const int32_t* part_list;
    bool all_blocks;    // varlen without lists
    bool bad;           // varlen: the sequence breaks the max_seqlen / total contract
    int n_valid;        // entries that name an in-range tile
};

template <int NQ>
__device__ bool tile_at(const Item<NQ>& it, const TcParams& P, int t, int& kb, bool& full) {
    if (!P.a.varlen) {
        kb = t;
        full = false;
        return true;
    }
    const int nbk = (it.Lk + kBN - 1) / kBN;
    if (it.all_blocks) {
        kb = t;
        full = false;
        return t < nbk;
    }
    if (t < it.n_full) {
        kb = it.full_list[t];
        full = true;
    } else {
        kb = it.part_list[t - it.n_full];
        full = false;
    }
    return kb >= 0 && kb < nbk;
}

template <int NQ>
__device__ Item<NQ> decode(const TcParams& P, int item) {
    Item<NQ> it;
    const AttnParams& a = P.a;
    it.bad = false;
    it.full_list = nullptr;
    it.part_list = nullptr;
    it.all_blocks = false;
    it.n_full = 0;
    it.prefix = 0;
    it.seq = 0;
    it.q_row0 = 0;
    it.k_row0 = 0;
    if (!a.varlen) {
        const int qp = item % P.items_per_unit;
        const int u2 = item / P.items_per_unit;  // ((b*H + h)*N + n): n fastest so bias tiles are reused from L2
        it.n = u2 % a.N;
        it.h = (u2 / a.N) % a.H;
        it.b = u2 / (a.N * a.H);
        it.bn = (long long)it.b * a.N + it.n;
        it.unit = it.bn * a.H + it.h;
        it.Lq = a.Q;
        it.Lk = a.K;
        for (int i = 0; i < NQ; ++i) {
            it.qt[i] = qp * NQ + i;
            it.slot_on[i] = it.qt[i] < P.nqt;
        }
        int nkt = (a.K + kBN - 1) / kBN;
        if (P.mask_kind == 1) {
            int L = a.kv_len[it.bn];
            it.prefix = L < 0 ? 0 : (L > a.K ? a.K : L);
            nkt = (it.prefix + kBN - 1) / kBN;  // 0 when every key is masked
        }
        it.n_raw = nkt;
        it.n_valid = nkt;
        return it;
    }
    // varlen: heaviest q tiles first (larger q tile index -> more causal blocks)
    const int per = a.num_seqs * a.H;
    const int qt = P.nqt - 1 - item / per;
    const int sh = item % per;
    it.seq = sh / a.H;
    it.h = sh % a.H;
    it.b = 0;
    it.n = 0;
    it.bn = 0;
    it.unit = 0;
    const int cq0 = a.cu_q[it.seq], cq1 = a.cu_q[it.seq + 1];
    const int ck0 = a.cu_k[it.seq], ck1 = a.cu_k[it.seq + 1];
    it.q_row0 = cq0;
    it.k_row0 = ck0;
    it.Lq = cq1 - cq0;
    it.Lk = ck1 - ck0;
    it.qt[0] = qt;
    bool ok = it.Lq >= 0 && it.Lk >= 0 && it.Lq <= a.max_q && it.Lk <= a.max_k && cq0 >= 0 && ck0 >= 0 &&
              cq1 <= a.total_q && ck1 <= a.total_k;
    it.bad = !ok;
    it.slot_on[0] = ok && qt * kBM < it.Lq;
    for (int i = 1; i < NQ; ++i) it.slot_on[i] = false;
    it.n_raw = 0;
    it.n_valid = 0;
    if (!it.slot_on[0]) return it;
    const int nbk = (it.Lk + kBN - 1) / kBN;
    if (!a.kv_num) {
        it.all_blocks = true;
        it.n_raw = nbk;
        it.n_valid = nbk;
        return it;
    }
    if (qt >= a.MQ) return it;  // q block outside the lists: nothing listed
    const int hm = a.mask_heads == 1 ? 0 : it.h;
    const long long row = ((long long)it.seq * a.mask_heads + hm) * a.MQ + qt;
    if (a.full_num) {
        it.n_full = min(max(a.full_num[row], 0), a.MK);
        it.full_list = a.full_idx + row * a.MK;
    }
    const int np = min(max(a.kv_num[row], 0), a.MK);
    it.part_list = a.kv_idx + row * a.MK;
    it.n_raw = it.n_full + np;
    int nv = 0;
    for (int t = 0; t < it.n_raw; ++t) {
        int kb;
        bool full;
        nv += tile_at(it, P, t, kb, full) ? 1 : 0;
    }
    it.n_valid = nv;
    return it;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <int NQ, bool BF16, bool BIAS_F32>
__global__ void __launch_bounds__(NQ * 128 + 64, 1) tc_fwd_kernel(const __grid_constant__ TcParams P) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const Layout L = make_layout(NQ, P);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    constexpr int kProducerWarp = NQ * 4;
    constexpr int kMmaWarp = NQ * 4 + 1;
    const AttnParams& a = P.a;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L.abort_flag);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L.tmem_slot);

    const int S = P.kv_stages;
    const int BS = P.bias_stages;
    auto bar = [&](int idx) -> uint32_t { return base + L.bars + 8u * (uint32_t)idx; };
    auto q_full = [&](int i) { return bar(i); };
    const uint32_t q_empty = bar(NQ);
    auto kv_full = [&](int s) { return bar(NQ + 1 + s); };
    auto kv_empty = [&](int s) { return bar(NQ + 1 + S + s); };
    auto bias_full = [&](int i, int s) { return bar(NQ + 1 + 2 * S + i * BS + s); };
    auto bias_empty = [&](int i, int s) { return bar(NQ + 1 + 2 * S + NQ * BS + i * BS + s); };
    auto s_full = [&](int i) { return bar(NQ + 1 + 2 * S + 2 * NQ * BS + i); };
    auto p_full = [&](int i) { return bar(NQ + 1 + 2 * S + 2 * NQ * BS + NQ + i); };
    auto o_full = [&](int i) { return bar(NQ + 1 + 2 * S + 2 * NQ * BS + 2 * NQ + i); };
    const uint32_t drain = bar(NQ + 1 + 2 * S + 2 * NQ * BS + 3 * NQ);

    auto q_smem = [&](int i) { return base + L.q + (uint32_t)i * P.tile_bytes; };
    auto k_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes; };
    auto v_smem = [&](int s) { return base + L.kv + (uint32_t)s * 2u * P.tile_bytes + P.tile_bytes; };
    auto bias_smem = [&](int i, int s) { return base + L.bias + (uint32_t)(i * BS + s) * P.bias_bytes; };

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < NQ; ++i) {
            mbar_init(q_full(i), 1);
            mbar_init(s_full(i), 1);
            mbar_init(p_full(i), 128);
            mbar_init(o_full(i), 1);
            for (int s = 0; s < BS; ++s) {
                mbar_init(bias_full(i, s), 1);
                mbar_init(bias_empty(i, s), 128);
            }
        }
        mbar_init(q_empty, 1);
        mbar_init(drain, 1);
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
        // ------------------------------------------------------------- producer
        uint32_t kv_it = 0, q_it = 0;
        uint32_t b_it[NQ];
        for (int i = 0; i < NQ; ++i) b_it[i] = 0;
        bool ok = true;
        // q_empty completes once per item with work; q_full(i) once per item in which slot i is active.
        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<NQ> it = decode<NQ>(P, item);
            bool any = false;
            for (int i = 0; i < NQ; ++i) any = any || it.slot_on[i];
            if (!any || it.n_valid == 0) continue;
            if (lane == 0 && q_it > 0) ok = wait_bar(q_empty, (q_it - 1) & 1, abort_flag, a.status);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                for (int i = 0; i < NQ; ++i) {
                    if (!it.slot_on[i]) continue;
                    mbar_expect_tx(q_full(i), P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb) {
                        if (!a.varlen)
                            tma_load_3d(q_smem(i) + sb * kBox, &P.tm_q, sb * 64, it.qt[i] * kBM, (int)it.unit, q_full(i));
                        else
                            tma_load_3d(q_smem(i) + sb * kBox, &P.tm_q, sb * 64, it.h, it.q_row0 + it.qt[i] * kBM,
                                        q_full(i));
                    }
                }
            }
            ++q_it;
            for (int t = 0; t < it.n_raw && ok; ++t) {
                int kb;
                bool full;
                if (!tile_at(it, P, t, kb, full)) continue;
                const int st = kv_it % S;
                if (lane == 0 && kv_it >= (uint32_t)S) ok = wait_bar(kv_empty(st), ((kv_it / S) - 1) & 1, abort_flag, a.status);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    mbar_expect_tx(kv_full(st), 2 * P.tile_bytes);
                    for (int sb = 0; sb < P.nsub; ++sb) {
                        if (!a.varlen) {
                            tma_load_3d(k_smem(st) + sb * kBox, &P.tm_k, sb * 64, kb * kBN, (int)it.unit, kv_full(st));
                            tma_load_3d(v_smem(st) + sb * kBox, &P.tm_v, sb * 64, kb * kBN, (int)it.unit, kv_full(st));
                        } else {
                            tma_load_3d(k_smem(st) + sb * kBox, &P.tm_k, sb * 64, it.h, it.k_row0 + kb * kBN, kv_full(st));
                            tma_load_3d(v_smem(st) + sb * kBox, &P.tm_v, sb * 64, it.h, it.k_row0 + kb * kBN, kv_full(st));
                        }
                    }
                }
                ++kv_it;
                if (a.varlen) continue;
                for (int i = 0; i < NQ && ok; ++i) {
                    if (!it.slot_on[i]) continue;
                    const int bs = b_it[i] % BS;
                    if (lane == 0 && b_it[i] >= (uint32_t)BS)
                        ok = wait_bar(bias_empty(i, bs), ((b_it[i] / BS) - 1) & 1, abort_flag, a.status);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    if (P.mask_kind == 2) {
                        // 128 key-validity bits of this tile: word w, bit l <-> key kb*128 + 32w + l
                        uint32_t* mw = reinterpret_cast<uint32_t*>(gbase + L.maskw + (uint32_t)(i * BS + bs) * 16u);
                        for (int w = 0; w < 4; ++w) {
                            const int key = kb * kBN + 32 * w + lane;
                            const bool v = key < a.K && a.mask[it.bn * a.K + key] != 0;
                            const uint32_t word = __ballot_sync(0xffffffffu, v);
                            if (lane == w) mw[w] = word;
                        }
                        __syncwarp();
                    }
                    if (lane == 0) {
                        mbar_expect_tx(bias_full(i, bs), P.bias_bytes);
                        for (int bx = 0; bx < P.bias_boxes; ++bx)
                            tma_load_3d(bias_smem(i, bs) + bx * kBox, &P.tm_bias, kb * kBN + bx * P.bias_box_cols,
                                        it.qt[i] * kBM, it.b * a.H + it.h, bias_full(i, bs));
                    }
                    ++b_it[i];
                }
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------------ MMA
        if (lane == 0) {
            uint32_t kv_it = 0;
            uint32_t p_it[NQ], q_it[NQ];
            for (int i = 0; i < NQ; ++i) p_it[i] = q_it[i] = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
                const Item<NQ> it = decode<NQ>(P, item);
                bool any = false;
                for (int i = 0; i < NQ; ++i) any = any || it.slot_on[i];
                if (!any || it.n_valid == 0) continue;
                for (int i = 0; i < NQ && ok; ++i)
                    if (it.slot_on[i]) ok = wait_bar(q_full(i), q_it[i]++ & 1, abort_flag, a.status);
                int jv = 0, prev = 0;
                for (int t = 0; t < it.n_raw && ok; ++t) {
                    int kb;
                    bool full;
                    if (!tile_at(it, P, t, kb, full)) continue;
                    const int st = kv_it % S;
                    ok = wait_bar(kv_full(st), (kv_it / S) & 1, abort_flag, a.status);
                    if (!ok) break;
                    ++kv_it;
                    tc_fence_after();
                    for (int i = 0; i < NQ && ok; ++i) {
                        if (!it.slot_on[i]) continue;
                        if (jv > 0) {
                            ok = wait_bar(p_full(i), p_it[i] & 1, abort_flag, a.status);
                            if (!ok) break;
                            ++p_it[i];
                            tc_fence_after();
                            for (int kk = 0; kk < kBN / 16; ++kk)
                                mma_ts(tmem + P.o_col0 + i * P.o_cols, tmem + i * 128 + kk * 8,
                                       sw128_desc(v_smem(prev) + kk * 16 * 128, kBox, 1024), P.idesc_pv,
                                       (jv > 1 || kk > 0) ? 1u : 0u);
                        }
                        for (int kk = 0; kk < P.ksteps; ++kk) {
                            const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
                            mma_ss(tmem + i * 128, sw128_desc(q_smem(i) + off, 16, 1024),
                                   sw128_desc(k_smem(st) + off, 16, 1024), P.idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(s_full(i));
                    }
                    if (!ok) break;
                    if (jv > 0) mma_commit(kv_empty(prev));
                    prev = st;
                    ++jv;
                }
                for (int i = 0; i < NQ && ok; ++i) {
                    if (!it.slot_on[i]) continue;
                    ok = wait_bar(p_full(i), p_it[i] & 1, abort_flag, a.status);
                    if (!ok) break;
                    ++p_it[i];
                    tc_fence_after();
                    for (int kk = 0; kk < kBN / 16; ++kk)
                        mma_ts(tmem + P.o_col0 + i * P.o_cols, tmem + i * 128 + kk * 8,
                               sw128_desc(v_smem(prev) + kk * 16 * 128, kBox, 1024), P.idesc_pv,
                               (jv > 1 || kk > 0) ? 1u : 0u);
                    mma_commit(o_full(i));
                }
                if (!ok) break;
                mma_commit(kv_empty(prev));
                mma_commit(q_empty);
            }
            if (!ok) *abort_flag = 1;
            // Let every MMA issued so far finish before TMEM is released.
            mma_commit(drain);
            wait_bar_drain(drain, 0);
        }
        __syncwarp();
    } else {
        // -------------------------------------------------------------- softmax
        const int slot = warp / 4;
        const int wq = warp % 4;               // TMEM lane quarter
        const int r = wq * 32 + lane;          // row within the q tile
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t s_taddr = tmem + lane_off + slot * 128;
        const uint32_t o_taddr = tmem + lane_off + P.o_col0 + slot * P.o_cols;
        uint32_t s_it = 0, bias_it = 0, o_it = 0;
        const float scale = a.scale;
        bool ok = true;

        for (int item = blockIdx.x; item < P.items && ok; item += gridDim.x) {
            const Item<NQ> it = decode<NQ>(P, item);
            if (it.bad && threadIdx.x == 0) atomicCAS(a.status, 0, kStatusDevice);
            if (!it.slot_on[slot]) continue;
            const int qrow = it.qt[slot] * kBM + r;  // local query row
            float m_true = -INFINITY, m_ref = 0.f, l = 0.f;
            int jv = 0;
            for (int t = 0; t < it.n_raw && ok; ++t) {
                int kb;
                bool full;
                if (!tile_at(it, P, t, kb, full)) continue;
                ok = __all_sync(0xffffffffu, wait_bar(s_full(slot), s_it & 1, abort_flag, a.status));
                if (!ok) break;
                ++s_it;
                tc_fence_after();
                uint32_t sr[128];
                tmem_ld_x128(s_taddr, sr);
                float x[128];
                const int key0 = kb * kBN;
                // Which keys exist / are valid in this tile.
                bool all_valid;
                int vlim;  // keys < vlim are valid in the prefix / no-mask / full cases
                if (!a.varlen) {
                    vlim = P.mask_kind == 1 ? it.prefix : a.K;
                    all_valid = P.mask_kind != 2 && key0 + kBN <= vlim;
                } else {
                    vlim = it.Lk;
                    const bool causal = !full && a.mask_mod == TA_MASK_CAUSAL;
                    all_valid = key0 + kBN <= it.Lk && (!causal || key0 + kBN - 1 <= it.qt[0] * kBM);
                }
                if (!a.varlen) {
                    const int bs = bias_it % BS;
                    ok = __all_sync(0xffffffffu, wait_bar(bias_full(slot, bs), (bias_it / BS) & 1, abort_flag, a.status));
                    if (!ok) break;
                    const uint8_t* bt = gbase + (bias_smem(slot, bs) - base);
                    const uint32_t sw = (uint32_t)(r & 7);
                    uint32_t mwords[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
                    if (P.mask_kind == 2) {
                        const uint4 mw = *reinterpret_cast<const uint4*>(gbase + L.maskw + (uint32_t)(slot * BS + bs) * 16u);
                        mwords[0] = mw.x;
                        mwords[1] = mw.y;
                        mwords[2] = mw.z;
                        mwords[3] = mw.w;
                    }
                    if constexpr (!BIAS_F32) {
#pragma unroll
                        for (int g = 0; g < 16; ++g) {  // 8 keys per 16-byte chunk
                            const uint32_t sub = g >> 3, ch = g & 7;
                            const uint4 w = *reinterpret_cast<const uint4*>(bt + sub * kBox + r * 128 + ((ch ^ sw) << 4));
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float b0, b1;
                                if constexpr (BF16) {
                                    b0 = __uint_as_float(ww[e] << 16);
                                    b1 = __uint_as_float(ww[e] & 0xffff0000u);
                                } else {
                                    b0 = __half2float(__ushort_as_half((unsigned short)(ww[e] & 0xffffu)));
                                    b1 = __half2float(__ushort_as_half((unsigned short)(ww[e] >> 16)));
                                }
                                x[g * 8 + 2 * e] = fmaf(__uint_as_float(sr[g * 8 + 2 * e]), scale, b0);
                                x[g * 8 + 2 * e + 1] = fmaf(__uint_as_float(sr[g * 8 + 2 * e + 1]), scale, b1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int g = 0; g < 32; ++g) {  // 4 keys per 16-byte chunk
                            const uint32_t sub = g >> 3, ch = g & 7;
                            const float4 w = *reinterpret_cast<const float4*>(bt + sub * kBox + r * 128 + ((ch ^ sw) << 4));
                            x[g * 4 + 0] = fmaf(__uint_as_float(sr[g * 4 + 0]), scale, w.x);
                            x[g * 4 + 1] = fmaf(__uint_as_float(sr[g * 4 + 1]), scale, w.y);
                            x[g * 4 + 2] = fmaf(__uint_as_float(sr[g * 4 + 2]), scale, w.z);
                            x[g * 4 + 3] = fmaf(__uint_as_float(sr[g * 4 + 3]), scale, w.w);
                        }
                    }
                    mbar_arrive(bias_empty(slot, bs));
                    ++bias_it;
                    if (!all_valid) {
#pragma unroll
                        for (int c = 0; c < 128; ++c) {
                            const int key = key0 + c;
                            const bool exists = key < a.K;
                            const bool valid = exists && key < vlim && ((mwords[c >> 5] >> (c & 31)) & 1u);
                            x[c] = valid ? x[c] : (exists ? kMasked : -INFINITY);
                        }
                    }
                } else {
                    const bool causal = !full && a.mask_mod == TA_MASK_CAUSAL;
#pragma unroll
                    for (int c = 0; c < 128; ++c) {
                        const float v = __uint_as_float(sr[c]) * scale;
                        if (all_valid) {
                            x[c] = v;
                        } else {
                            const int key = key0 + c;
                            const bool exists = key < it.Lk;
                            const bool valid = exists && (!causal || key <= qrow);
                            x[c] = valid ? v : (exists ? kMasked : -INFINITY);
                        }
                    }
                }
                // Row max of this tile.
                float mt = x[0];
#pragma unroll
                for (int c = 1; c < 128; ++c) mt = fmaxf(mt, x[c]);
                const float m_new = fmaxf(m_true, mt);
                m_true = m_new;
                if (jv == 0) {
                    m_ref = m_new;
                    l = 0.f;
                } else {
                    const bool need = (m_new - m_ref) * kLog2e > kRescaleLog2;
                    if (__any_sync(0xffffffffu, need)) {
                        // Raise the reference max to the current max; O (complete
                        // through the previous tile) and l scale by 2^((m_ref-m_new) log2 e).
                        const float alpha = ex2((m_ref - m_new) * kLog2e);
                        l *= alpha;
                        m_ref = m_new;
                        for (uint32_t c0 = 0; c0 < P.o_cols; c0 += 16) {
                            uint32_t o[16];
                            tmem_ld_x16(o_taddr + c0, o);
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tmem_st_x16(o_taddr + c0, o);
                        }
                    }
                }
                uint32_t pk[64];
                float lsum = 0.f;
                if (m_ref > kMasked) {
                    const float nb = -m_ref * kLog2e;
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const float p0 = ex2(fmaf(x[c], kLog2e, nb));
                        const float p1 = ex2(fmaf(x[c + 1], kLog2e, nb));
                        lsum += p0 + p1;
                        pk[c / 2] = pack2<BF16>(p0, p1);
                    }
                } else {
                    // No valid key seen yet (every logit so far is -1e9): the
                    // weights are exactly 1 for masked keys and 0 for absent ones.
#pragma unroll
                    for (int c = 0; c < 128; c += 2) {
                        const float p0 = x[c] == kMasked ? 1.f : 0.f;
                        const float p1 = x[c + 1] == kMasked ? 1.f : 0.f;
                        lsum += p0 + p1;
                        pk[c / 2] = pack2<BF16>(p0, p1);
                    }
                }
                l += lsum;
                tmem_st_x64(s_taddr, pk);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(p_full(slot));
                ++jv;
            }
            if (!ok) break;

            // ------------------------------------------------------- epilogue
            bool seen = m_true > kMasked;  // saw a key with a real logit
            if (jv > 0) {
                ok = __all_sync(0xffffffffu, wait_bar(o_full(slot), o_it & 1, abort_flag, a.status));
                ++o_it;
                if (!ok) break;
                tc_fence_after();
            } else {
                seen = false;
            }
            // Rows with no valid key: uniform weights over all keys -> mean of V.
            // Each warp builds the mean once for its rows (lanes split the columns).
            // Lane l holds the means of columns l, l+32, l+64, l+96.
            const bool any_unseen = __any_sync(0xffffffffu, !seen);
            float mv[4] = {0.f, 0.f, 0.f, 0.f};
            if (any_unseen && it.Lk > 0) {
                const long long vrow0 = !a.varlen ? it.unit * a.K : (long long)it.k_row0;
                const long long vstride = !a.varlen ? a.D : (long long)a.H * a.D;
                const long long vcol0 = !a.varlen ? 0 : (long long)it.h * a.D;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int d = lane + 32 * j;
                    if (d >= a.D) continue;
                    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
                    int key = 0;
                    for (; key + 4 <= it.Lk; key += 4) {
                        s0 += load16<BF16>(a.v, (vrow0 + key) * vstride + vcol0 + d);
                        s1 += load16<BF16>(a.v, (vrow0 + key + 1) * vstride + vcol0 + d);
                        s2 += load16<BF16>(a.v, (vrow0 + key + 2) * vstride + vcol0 + d);
                        s3 += load16<BF16>(a.v, (vrow0 + key + 3) * vstride + vcol0 + d);
                    }
                    for (; key < it.Lk; ++key) s0 += load16<BF16>(a.v, (vrow0 + key) * vstride + vcol0 + d);
                    mv[j] = ((s0 + s1) + (s2 + s3)) / (float)it.Lk;
                }
            }
            const bool row_ok = qrow < it.Lq;
            const long long orow = !a.varlen ? it.unit * a.Q + qrow : (long long)(it.q_row0 + qrow);
            uint16_t* op = static_cast<uint16_t*>(a.out);
            const long long obase = !a.varlen ? orow * a.D : (orow * a.H + it.h) * a.D;
            const float inv = (seen && l > 0.f) ? 1.f / l : 0.f;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint32_t c0 = cc * 16;
                if (c0 >= P.o_cols) break;
                uint32_t o[16];
                if (jv > 0) tmem_ld_x16(o_taddr + c0, o);
                float vals[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) vals[e] = __uint_as_float(o[e]) * inv;
                if (any_unseen) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float m = __shfl_sync(0xffffffffu, mv[(cc * 16 + e) >> 5], (cc * 16 + e) & 31);
                        if (!seen) vals[e] = m;
                    }
                }
                if (row_ok && (int)c0 < a.D) {
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 16; e += 2) w[e / 2] = pack2<BF16>(vals[e], vals[e + 1]);
                    uint4* dst = reinterpret_cast<uint4*>(op + obase + c0);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    if ((int)c0 + 8 < a.D) dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
            if (row_ok) {
                float lse, mx;
                if (it.Lk == 0) {
                    lse = -INFINITY;
                    mx = -INFINITY;
                } else if (!seen) {
                    lse = kMasked + logf((float)it.Lk);
                    mx = kMasked;
                } else {
                    lse = m_ref + logf(l);
                    mx = m_true;
                }
                const long long li = !a.varlen ? orow : (long long)it.h * a.total_q + orow;
                if (a.lse) a.lse[li] = lse;
                if (a.mx) a.mx[li] = mx;
            }
        }
        if (!ok) *abort_flag = 1;
    }

    // ---------------------------------------------------------------- teardown
    if (warp == kProducerWarp && lane == 0 && *abort_flag) {
        // Give TMA loads already issued time to land before the CTA exits.
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

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
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

// 3-D tiled map: dims {d0, d1, d2} (d0 innermost), byte strides of d1 and d2, box {b0, b1, b2}.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, dt, 3, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Instruction descriptor of kind::f16: D fp32 at [4,6), A/B type at [7,10)/[10,13)
// (0 f16, 1 bf16), A/B major at bits 15/16 (0 K-major, 1 MN-major), N>>3 at
// [17,23), M>>4 at [24,29).
uint32_t make_idesc(bool bf16, int M, int N, bool b_mn_major) {
    const uint32_t ab = bf16 ? 1u : 0u;
    return (1u << 4) | (ab << 7) | (ab << 10) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

template <int NQ, bool BF16, bool BIAS_F32>
cudaError_t launch_kernel(TcParams& P, cudaStream_t stream) {
    const Layout L = make_layout(NQ, P);
    const size_t smem = L.total + 1024;
    auto kern = tc_fwd_kernel<NQ, BF16, BIAS_F32>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_num_sms[dev]) cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    const int grid = P.items < g_num_sms[dev] ? P.items : g_num_sms[dev];
    if (grid <= 0) return cudaSuccess;
    kern<<<grid, NQ * 128 + 64, smem, stream>>>(P);
    return cudaGetLastError();
}

constexpr size_t kSmemLimit = 232448;  // 227 KB: the per-block opt-in maximum

}  // namespace

cudaError_t launch_tc_fwd(const AttnParams& a, cudaStream_t stream) {
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
    const uint64_t rs = (uint64_t)D * 2;
    int NQ;
    if (!a.varlen) {
        NQ = 1;
        P.nqt = (a.Q + kBM - 1) / kBM;
        P.items_per_unit = (P.nqt + NQ - 1) / NQ;
        const long long items = (long long)a.B * a.N * a.H * P.items_per_unit;
        if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        P.items = (int)items;
        const uint64_t units = (uint64_t)a.B * a.N * a.H;
        if (!make_map(&P.tm_q, dt, a.q, D, a.Q, units, rs, rs * a.Q, 64, kBM, 1) ||
            !make_map(&P.tm_k, dt, a.k, D, a.K, units, rs, rs * a.K, 64, kBN, 1) ||
            !make_map(&P.tm_v, dt, a.v, D, a.K, units, rs, rs * a.K, 64, kBN, 1))
            return cudaErrorInvalidValue;
        const uint64_t eb = a.bias_f32 ? 4 : 2;
        P.bias_box_cols = a.bias_f32 ? 32 : 64;
        P.bias_boxes = kBN / P.bias_box_cols;
        P.bias_bytes = P.bias_boxes * kBox;
        if (!make_map(&P.tm_bias, a.bias_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, a.bias, a.K, a.Q,
                      (uint64_t)a.B * a.H, a.K * eb, a.K * eb * a.Q, P.bias_box_cols, kBM, 1))
            return cudaErrorInvalidValue;
        P.mask_kind = a.kv_len ? 1 : (a.mask ? 2 : 0);
    } else {
        NQ = 1;
        P.nqt = (a.max_q + kBM - 1) / kBM;
        const long long items = (long long)a.num_seqs * a.H * P.nqt;
        if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        P.items = (int)items;
        P.items_per_unit = 1;
        if (!make_map(&P.tm_q, dt, a.q, D, a.H, a.total_q, rs, rs * a.H, 64, 1, kBM) ||
            !make_map(&P.tm_k, dt, a.k, D, a.H, (a.total_k > 0 ? a.total_k : 1), rs, rs * a.H, 64, 1, kBN) ||
            !make_map(&P.tm_v, dt, a.v, D, a.H, (a.total_k > 0 ? a.total_k : 1), rs, rs * a.H, 64, 1, kBN))
            return cudaErrorInvalidValue;
        P.bias_bytes = 0;
        P.bias_boxes = 0;
    }
    // Pipeline depth: as many stages as fit in shared memory.  The MMA issues
    // PV of tile j-1 after waiting for tile j's K/V, so at least two K/V
    // stages are required.
    const int prefs[][2] = {{3, 3}, {3, 2}, {2, 2}, {2, 1}};
    P.kv_stages = 0;
    for (auto& pr : prefs) {
        P.kv_stages = pr[0];
        P.bias_stages = a.varlen ? 0 : pr[1];
        if (make_layout(NQ, P).total + 1024 <= kSmemLimit) break;
        P.kv_stages = 0;
    }
    if (P.kv_stages < 2) return cudaErrorInvalidConfiguration;
    P.o_col0 = NQ * 128;
    uint32_t cols = NQ * 128 + NQ * P.o_cols;
    P.tmem_cols = 32;
    while (P.tmem_cols < cols) P.tmem_cols <<= 1;
    if (P.tmem_cols > 512) return cudaErrorInvalidConfiguration;

    if (bf16) {
        if (a.varlen || !a.bias_f32) return launch_kernel<1, true, false>(P, stream);
        return launch_kernel<1, true, true>(P, stream);
    }
    if (a.varlen || !a.bias_f32) return launch_kernel<1, false, false>(P, stream);
    return launch_kernel<1, false, true>(P, stream);
}

}  // namespace triattn
