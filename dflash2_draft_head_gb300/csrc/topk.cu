// Top-K candidate extraction: for every row of draft logits, the K largest
// entries in descending order of value (equal values by ascending index) and
// the values themselves.
//
// ggml-org/llama.cpp pull request #27342, "spec : add DFlash2 support (local
// convolution + candidate selector)", review thread on the TOP_K kernel: the
// selector consumes the top K candidates of vocabulary-wide rows (a few 1e5
// entries) with small K, swept there up to K = 1024.
//
// The work is one read of every logit, so both kernels keep the per-element
// cost at a load from shared memory and one comparison, and share:
//  - persistent CTAs, one per SM; rows are dealt out to clusters of cs CTAs,
//    each CTA of a cluster taking one contiguous chunk of the row (cs = 1 when
//    there are enough rows to fill the GPU);
//  - one producer lane streaming the chunk's 16-byte-aligned body through a
//    ring of six 16 KB stages with cp.async.bulk (mbarrier completion); the
//    unaligned head and tail (under 16 bytes each) are read directly;
//  - candidates as 64-bit keys: order-preserving value bits above the
//    complemented index, so a larger key is a better candidate and no two
//    keys are equal;
//  - a cluster merge at the end of a row: the other CTAs hand their K best to
//    rank 0 through distributed shared memory (double-buffered mbarrier
//    hand-shake), and rank 0 writes ids and values in rank order.
// topk_async_kernel (K <= 256): eight filter warps test whole stages against
// a threshold key and push survivors into per-warp queues, never waiting for
// one another; a selector warp keeps the exact sorted top-K and raises the
// published threshold (see the section header further down).
// topk_kernel (K <= 1024): 256 consumer threads append survivors to one shared
// candidate buffer and, at stage boundaries, re-select together (rank counting
// or an 8-bit-digit radix select) and tighten the threshold to the K-th value;
// elements tested later have larger indices, so the strict test x > tau is
// exact there.
// topk_rows_kernel (K <= 32, few 16-byte-aligned rows, one cluster per row all
// resident at once, as for one draft block): no streaming; each CTA holds its
// chunk of the row in registers and selects in a few block-wide steps (see the
// section header further down).
// NaN entries never pass a test; rows with fewer than K other entries get
// id -1 and value NaN in the remaining slots.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"
#include "dflash2.h"
#include "ptx.cuh"

namespace df2 {

// Device fault word of the top-K kernel: DF2_FLAG_TIMEOUT when a bounded wait
// gives up, DF2_FLAG_OVERFLOW if the candidate buffer bound were ever hit.
__device__ unsigned int g_topk_fault = 0;

// Row trace of the streaming kernel (compiled in only with -DDF2_TRACE;
// otherwise every trace point is empty): global-timer stamps of CTAs
// 0..1023, 64 slots each: 8 points for each of 8 traced rows of the CTA (its
// rows 0-3 and 10-13), at the points include/dflash2.h lists with
// dflash2_trace_read_topk.
#ifdef DF2_TRACE
__device__ unsigned long long g_trace_topk[1024 * 64];
#define DF2_TK_ROW(r) ((r) < 4 ? (r) : ((r) >= 10 && (r) < 14 ? (r) - 6 : -1))
#define DF2_TK_TRACE(r, k)                                                        \
    do {                                                                          \
        const int tr_ = DF2_TK_ROW(r);                                            \
        if (tr_ >= 0 && blockIdx.x < 1024u)                                       \
            g_trace_topk[blockIdx.x * 64 + tr_ * 8 + (k)] = global_ns();          \
    } while (0)
#else
#define DF2_TK_TRACE(r, k) \
    do {                   \
    } while (0)
#endif

namespace {

constexpr int kNC = 256;                   // consumer threads (8 warps)
constexpr int kThreads = kNC + 32;         // + one producer warp
constexpr uint32_t kSB = 16384;            // bytes per ring stage
constexpr int kNS = 6;                     // ring stages
constexpr int kCap = 12288;                // candidate keys a CTA holds
constexpr int kFillTrigger = kTopkMaxK;    // fill mode: select once more than this many are held
constexpr int kCheckElems = 8192;          // elements between checks (one bf16, two fp32 stages)
// threshold mode re-selects, at a check, once more than K + max(K, 32) keys
// are held, so tau follows the K-th best seen so far
static_assert(2 * kTopkMaxK + kCheckElems <= kCap, "the elements between checks must fit");
static_assert(kFillTrigger + 2 * kNC * 8 <= kCap, "fill-mode sub-blocks must fit");
static_assert(8 * kTopkMaxK <= kCap, "a cluster merge must fit");
static_assert(kNC == 256, "one histogram bin per consumer thread");

constexpr uint32_t kOffBuf = kNS * kSB;
constexpr uint32_t kOffTmp = kOffBuf + kCap * 8;
constexpr uint32_t kOffOut = kOffTmp + kTopkMaxK * 8;
constexpr uint32_t kOffHist = kOffOut + 2 * kTopkMaxK * 8;
constexpr uint32_t kOffCtl = kOffHist + 256 * 4;
constexpr uint32_t kSmem = kOffCtl + 256;
static_assert(kSmem <= 227 * 1024, "shared memory");

struct Ctl {
    uint64_t full[kNS];    // producer -> consumers: stage landed
    uint64_t empty[kNS];   // consumers -> producer: stage free (one arrival per warp)
    uint64_t mfull[2];     // rank r -> rank 0: K best of a row written to out slot
    uint64_t mempty[2];    // rank 0 -> rank r: out slot read
    unsigned long long kmin;
    uint32_t count;
    uint32_t tmp_count;
    uint32_t sel_digit, sel_above, sel_cnt;
    uint32_t out_cnt[2];
    uint32_t abort;
};
static_assert(sizeof(Ctl) <= 256, "control block");

struct TopkParams {
    const void* logits;
    int rows, V, K, cs;
    int32_t* ids;
    float* vals;
};

// Order-preserving key: the value's bits mapped to an unsigned integer that
// sorts like the value (-0 folded onto +0), then the complemented index.
__device__ __forceinline__ uint64_t make_key(float x, uint32_t idx) {
    uint32_t b = __float_as_uint(x);
    if ((b << 1) == 0u) b = 0u;
    const uint32_t o = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((uint64_t)o << 32) | (uint32_t)~idx;
}

__device__ __forceinline__ float key_value(uint64_t k) {
    const uint32_t o = (uint32_t)(k >> 32);
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

__device__ __forceinline__ uint32_t key_index(uint64_t k) { return ~(uint32_t)k; }

template <bool BF16>
__device__ __forceinline__ float load_logit(const void* p, size_t i) {
    if constexpr (BF16)
        return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(p)[i] << 16);
    else
        return reinterpret_cast<const float*>(p)[i];
}

template <bool BF16>
__device__ __forceinline__ void load_vec(uint32_t saddr, float (&x)[BF16 ? 8 : 4]) {
    const uint4 w = lds_v4(saddr);
    if constexpr (BF16) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(q[i] << 16);
            x[2 * i + 1] = __uint_as_float(q[i] & 0xFFFF0000u);
        }
    } else {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    }
}

// Appends this thread's passing elements to the candidate buffer: bit j of m
// selects x[j], element idx0 + (j / G) * stride + j % G of the row (groups of
// G consecutive elements, `stride` apart).  A warp scan of the per-lane counts
// gives each lane its offset; one shared atomic per warp reserves the space.
// Warp-collective.  Returns, on lane 0 of a warp that appended, whether the
// buffer now holds more than `trig` keys.
template <int E, int G = E>
__device__ __forceinline__ bool append(uint32_t m, const float (&x)[E], uint32_t idx0,
                                       uint32_t stride, uint64_t* buf, Ctl* c, int trig) {
    const int lane = threadIdx.x & 31;
    const int n = __popc(m);
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const uint32_t tot = (uint32_t)__shfl_sync(0xffffffffu, incl, 31);
    if (tot == 0) return false;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(&c->count, tot);
    base = __shfl_sync(0xffffffffu, base, 0);
    uint32_t pos = base + (uint32_t)(incl - n);
#pragma unroll
    for (int j = 0; j < E; ++j) {
        if ((m >> j) & 1u) {
            if (pos < (uint32_t)kCap)
                buf[pos] = make_key(x[j], idx0 + (uint32_t)(j / G) * stride + (uint32_t)(j % G));
            else
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
            ++pos;
        }
    }
    return lane == 0 && base + tot > (uint32_t)trig;
}

// Exact selection of a small set (M <= 2 * kNC keys, M > K) by counting: a
// key's rank is the number of larger keys, ranks are distinct, and the K keys
// of rank < K land in rank order.  Same contract as select_top.
__device__ uint64_t select_small(uint64_t* buf, int M, int K, uint64_t* tmp, uint32_t* count) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int i = tid + q * kNC;
        if (i < M) {
            const uint64_t k = buf[i];
            int r = 0;
            for (int j = 0; j < M; ++j) r += buf[j] > k ? 1 : 0;
            if (r < K) tmp[r] = k;
        }
    }
    named_bar_sync(1, kNC);
    for (int i = tid; i < K; i += kNC) buf[i] = tmp[i];
    const uint64_t kth = tmp[K - 1];
    if (tid == 0) *count = (uint32_t)K;
    named_bar_sync(1, kNC);
    return kth;
}

// Exact selection over buf[0, M), M > K: leaves the K largest keys in
// buf[0, K) (unordered), sets the count to K and returns the K-th largest.
// Radix select, most significant 8-bit digit first: each pass histograms the
// keys that share the prefix fixed so far and fixes the next digit of the
// K-th key; a pass whose boundary bin holds exactly the keys still needed
// ends the search (everything at or above the prefix is taken).
__device__ uint64_t select_top(uint64_t* buf, int M, int K, uint64_t* tmp, uint32_t* hist,
                               Ctl* c) {
    const int tid = threadIdx.x;
    uint64_t prefix = 0;
    int need = K;
    for (int shift = 56; shift >= 0; shift -= 8) {
        const uint64_t hm = shift == 56 ? 0ull : (~0ull << (shift + 8));
        hist[tid] = 0u;
        if (tid == 0) {
            c->tmp_count = 0u;
            c->kmin = ~0ull;
        }
        named_bar_sync(1, kNC);
        for (int i = tid; i < M; i += kNC) {
            const uint64_t k = buf[i];
            if ((k & hm) == prefix) atomicAdd(&hist[(uint32_t)(k >> shift) & 255u], 1u);
        }
        named_bar_sync(1, kNC);
        if (tid < 32) {
            // lane l scans bins 255-8l down to 248-8l; lanes run from the top bin down
            uint32_t h[8], local = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                h[j] = hist[255 - 8 * tid - j];
                local += h[j];
            }
            uint32_t incl = local;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const uint32_t excl = incl - local;
            if (excl < (uint32_t)need && (uint32_t)need <= incl) {
                uint32_t acc = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (acc + h[j] >= (uint32_t)need) {
                        c->sel_digit = (uint32_t)(255 - 8 * tid - j);
                        c->sel_above = acc;
                        c->sel_cnt = h[j];
                        break;
                    }
                    acc += h[j];
                }
            }
        }
        named_bar_sync(1, kNC);
        need -= (int)c->sel_above;
        prefix |= (uint64_t)c->sel_digit << shift;
        if (c->sel_cnt == (uint32_t)need) break;
    }
    for (int i = tid; i < M; i += kNC) {
        const uint64_t k = buf[i];
        if (k >= prefix) {
            const uint32_t pos = atomicAdd(&c->tmp_count, 1u);
            if (pos < (uint32_t)K) tmp[pos] = k;
            atomicMin(&c->kmin, (unsigned long long)k);
        }
    }
    named_bar_sync(1, kNC);
    for (int i = tid; i < K; i += kNC) buf[i] = tmp[i];
    const uint64_t kth = c->kmin;
    if (tid == 0) c->count = (uint32_t)K;
    named_bar_sync(1, kNC);
    return kth;
}

constexpr int kVPT = kSB / 16 / kNC;  // 16-byte vectors per thread per stage
constexpr int kWPT = kVPT * 4;        // 32-bit words per thread per stage

// Element e of a thread's staged words (fp32: one per word; bf16: two per
// word, the lower half first).
template <bool BF16>
__device__ __forceinline__ float stage_elem(const uint32_t (&w)[kWPT], int e) {
    if constexpr (BF16)
        return __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
    else
        return __uint_as_float(w[e]);
}

__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));  // NaN yields the other operand
    return d;
}

// Largest non-NaN element of the staged words (NaN if all are NaN), by a
// pairwise tree: fp32 in fp32, bf16 on packed pairs.
template <bool BF16>
__device__ __forceinline__ float stage_max(const uint32_t (&w)[kWPT]) {
    if constexpr (BF16) {
        uint32_t t[kWPT];
#pragma unroll
        for (int i = 0; i < kWPT; ++i) t[i] = w[i];
#pragma unroll
        for (int h = kWPT / 2; h >= 1; h /= 2)
#pragma unroll
            for (int i = 0; i < h; ++i) t[i] = max_bf16x2(t[i], t[i + h]);
        return fmaxf(__uint_as_float(t[0] << 16), __uint_as_float(t[0] & 0xFFFF0000u));
    } else {
        float t[kWPT];
#pragma unroll
        for (int i = 0; i < kWPT; ++i) t[i] = __uint_as_float(w[i]);
#pragma unroll
        for (int h = kWPT / 2; h >= 1; h /= 2)
#pragma unroll
            for (int i = 0; i < h; ++i) t[i] = fmaxf(t[i], t[i + h]);
        return t[0];
    }
}

// Bits e of gt / eq set when staged element e (as stage_elem numbers them) is
// above / equal to t; NaN is neither.  bf16 stages compare packed pairs
// against t as a bf16 pair (exact: every threshold is a bf16 element's value).
template <bool BF16>
__device__ __forceinline__ void stage_cmp_masks(const uint32_t (&w)[kWPT], float t, uint32_t& gt,
                                                uint32_t& eq) {
    gt = 0u;
    eq = 0u;
    if constexpr (BF16) {
        const uint32_t h = __float_as_uint(t) >> 16;
        const uint32_t t2 = h | (h << 16);
        const __nv_bfloat162 tt = *reinterpret_cast<const __nv_bfloat162*>(&t2);
#pragma unroll
        for (int i = 0; i < kWPT; ++i) {
            const __nv_bfloat162 x2 = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
            const uint32_t g = __hgt2_mask(x2, tt);  // low half: element 2i, high: 2i + 1
            const uint32_t q = __heq2_mask(x2, tt);
            gt |= ((g & 1u) | ((g >> 30) & 2u)) << (2 * i);
            eq |= ((q & 1u) | ((q >> 30) & 2u)) << (2 * i);
        }
    } else {
#pragma unroll
        for (int e = 0; e < kWPT; ++e) {
            const float x = __uint_as_float(w[e]);
            gt |= (x > t ? 1u : 0u) << e;
            eq |= (x == t ? 1u : 0u) << e;
        }
    }
}

// Row index of staged element e: vector e / E of the thread's vectors (kNC
// vectors apart), element e % E of it.
template <int E>
__device__ __forceinline__ uint32_t stage_index(uint32_t idx0, int e) {
    return idx0 + (uint32_t)((e / E) * kNC * E + (e % E));
}

// Threshold-mode append, for the rare lanes with a passing element: the lane
// reserves its own slots with one shared atomic (no warp-wide step, so it may
// run divergently).  Returns whether the buffer then holds more than `trig`.
template <bool BF16, int E>
__device__ __forceinline__ bool append_sparse(float t, const uint32_t (&w)[kWPT], uint32_t idx0,
                                              uint64_t* buf, Ctl* c, int trig) {
    constexpr int EPT = kVPT * E;
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < EPT; ++e) m |= (stage_elem<BF16>(w, e) > t ? 1u : 0u) << e;
    if (m == 0) return false;
    const uint32_t n = (uint32_t)__popc(m);
    uint32_t pos = atomicAdd(&c->count, n);
    const bool over = pos + n > (uint32_t)trig;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        if ((m >> e) & 1u) {
            if (pos < (uint32_t)kCap)
                buf[pos] = make_key(stage_elem<BF16>(w, e), stage_index<E>(idx0, e));
            else
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
            ++pos;
        }
    }
    return over;
}

// Fill-mode append of every non-NaN staged element (x >= -inf), or of every
// element above t.  Warp-collective.
template <bool BF16, int E>
__device__ __forceinline__ bool append_dense(float t, bool keep_all, const uint32_t (&w)[kWPT],
                                             uint32_t idx0, uint64_t* buf, Ctl* c, int trig) {
    constexpr int EPT = kVPT * E;
    float x[EPT];
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        x[e] = stage_elem<BF16>(w, e);
        m |= ((keep_all ? x[e] == x[e] : x[e] > t) ? 1u : 0u) << e;
    }
    return append<EPT, E>(m, x, idx0, (uint32_t)(kNC * E), buf, c, trig);
}

// The K best of buf[0, M) (M > K) into buf[0, K); returns the K-th best key.
__device__ __forceinline__ uint64_t select_keep(uint64_t* buf, int M, int K, uint64_t* tmp,
                                                uint32_t* hist, Ctl* c) {
    return M <= 2 * kNC ? select_small(buf, M, K, tmp, &c->count)
                        : select_top(buf, M, K, tmp, hist, c);
}

// Orders buf[0, n) (n <= K, distinct keys) by counting and writes row `row`
// of the outputs; slots n..K-1 get id -1 and value NaN.
template <bool BF16>
__device__ void write_row(const uint64_t* buf, int n, const TopkParams& p, int row) {
    int32_t* ids = p.ids + (size_t)row * p.K;
    float* vals = p.vals + (size_t)row * p.K;
    for (int i = threadIdx.x; i < p.K; i += kNC) {
        int slot = i;
        int32_t id = -1;
        float v = __uint_as_float(0x7FC00000u);
        if (i < n) {
            const uint64_t k = buf[i];
            int r = 0;
            for (int j = 0; j < n; ++j) r += buf[j] > k ? 1 : 0;
            slot = r;
            id = (int32_t)key_index(k);
            v = key_value(k);  // exact, except that the key folded -0 onto +0
            if ((uint32_t)id >= (uint32_t)p.V) {  // not reachable with distinct keys
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
                id = -1;
                v = __uint_as_float(0x7FC00000u);
            } else if (v == 0.f) {
                v = load_logit<BF16>(p.logits, (size_t)row * p.V + (uint32_t)id);
            }
        }
        ids[slot] = id;
        vals[slot] = v;
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1) topk_kernel(TopkParams p) {
    constexpr int E = BF16 ? 8 : 4;  // elements per 16-byte vector
    constexpr int VPT = kVPT;
    constexpr int EPT = VPT * E;     // elements a thread holds per stage
    constexpr uint32_t kNaNWord = BF16 ? 0x7FC07FC0u : 0x7FC00000u;
    constexpr uint32_t esz = BF16 ? 2u : 4u;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t s0 = smem_u32(smem);
    uint64_t* buf = reinterpret_cast<uint64_t*>(smem + kOffBuf);
    uint64_t* tmp = reinterpret_cast<uint64_t*>(smem + kOffTmp);
    uint64_t* outk = reinterpret_cast<uint64_t*>(smem + kOffOut);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
    Ctl* c = reinterpret_cast<Ctl*>(smem + kOffCtl);
    const uint32_t full0 = smem_u32(&c->full[0]);
    const uint32_t empty0 = smem_u32(&c->empty[0]);
    volatile uint32_t* abort_flag = &c->abort;
    const int tid = threadIdx.x;
    const int cs = p.cs;
    const uint32_t rank = cs > 1 ? cluster_ctarank() : 0u;
    const int cid = (int)blockIdx.x / cs;
    const int ncl = (int)gridDim.x / cs;

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kNC / 32);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&c->mfull[i]), cs > 1 ? (uint32_t)(cs - 1) : 1u);
            mbar_init(smem_u32(&c->mempty[i]), 1);
        }
        c->abort = 0;
        fence_mbar_init();
    }
    if (cs > 1)
        cluster_sync();
    else
        __syncthreads();

    // this CTA's chunk [e0, e1) of every row (64-element granules)
    const int L = (((p.V + cs - 1) / cs) + 63) & ~63;
    const int e0 = min(p.V, (int)rank * L);
    const int e1 = min(p.V, e0 + L);
    const uintptr_t lbase = reinterpret_cast<uintptr_t>(p.logits);

    if (tid >= kNC) {
        // ---------------- producer (one lane)
        if (tid == kNC) {
            int it = 0;
            for (int row = cid; row < p.rows && !*abort_flag; row += ncl) {
                const uintptr_t a0 = lbase + ((size_t)row * p.V + e0) * esz;
                const uintptr_t a1 = lbase + ((size_t)row * p.V + e1) * esz;
                const uintptr_t b0 = (a0 + 15) & ~(uintptr_t)15, b1 = a1 & ~(uintptr_t)15;
                for (uintptr_t off = b0; off < b1; off += kSB, ++it) {
                    const int st = it % kNS;
                    const uint32_t ph = (uint32_t)(it / kNS) & 1u;
                    if (*abort_flag) break;
                    if (!mbar_wait_bounded(empty0 + 8 * st, ph ^ 1u, kWaitNs)) {
                        *abort_flag = 1;
                        atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_TIMEOUT);
                        break;
                    }
                    const uint32_t bytes = (uint32_t)min((uintptr_t)kSB, b1 - off);
                    mbar_arrive_expect_tx(full0 + 8 * st, bytes);
                    bulk_g2s(s0 + (uint32_t)st * kSB, reinterpret_cast<const void*>(off), bytes,
                             full0 + 8 * st);
                }
            }
        }
        __syncwarp();
        if (cs > 1) cluster_sync();  // no CTA leaves while a peer may still read it
        return;
    }

    // ---------------- consumers
    const int steady_trig = p.K + max(p.K, 32);
    int it = 0, rit = 0;
    for (int row = cid; row < p.rows; row += ncl, ++rit) {
        const size_t rowoff = (size_t)row * p.V;
        const uintptr_t a0 = lbase + (rowoff + e0) * esz;
        const uintptr_t a1 = lbase + (rowoff + e1) * esz;
        const uintptr_t b0 = (a0 + 15) & ~(uintptr_t)15, b1 = a1 & ~(uintptr_t)15;
        const bool body = b0 < b1;
        const int head = body ? (int)((b0 - a0) / esz) : e1 - e0;
        const int tail = body ? (int)((a1 - b1) / esz) : 0;
        // the unaligned head and tail elements (under 16 bytes each, so one per
        // thread) are loaded now and tested in index order: head first, tail last
        float hx[1] = {0.f}, tx[1] = {0.f};
        if (tid < head) hx[0] = load_logit<BF16>(p.logits, rowoff + e0 + tid);
        if (tid < tail) tx[0] = load_logit<BF16>(p.logits, rowoff + (e1 - tail) + tid);
        named_bar_sync(1, kNC);  // the previous row's readers of buf and count are done
        if (tid == 0) c->count = 0u;
        named_bar_sync(1, kNC);
        // Modes: fill (tau = -inf: every non-NaN element is kept) until a
        // selection; then threshold (x > tau).  tau is either just below a lower
        // bound of the K-th best value (x > tau keeps every x >= the bound) or,
        // after an exact selection, the K-th best value itself.
        float tau = -INFINITY;
        bool fill = true, seeded = false, over = false;
        int ks = 0;  // stages of this row so far
        over |= append<1>(tid < head && hx[0] == hx[0] ? 1u : 0u, hx, (uint32_t)(e0 + tid), 0u,
                          buf, c, kFillTrigger);

        for (uintptr_t off = b0; off < b1; off += kSB, ++it) {
            const int st = it % kNS;
            const uint32_t ph = (uint32_t)(it / kNS) & 1u;
            if (!*abort_flag && !mbar_wait_bounded(full0 + 8 * st, ph, kWaitNs)) {
                *abort_flag = 1;
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_TIMEOUT);
            }
            const uint32_t nvec = (uint32_t)min((uintptr_t)kSB, b1 - off) / 16u;
            const uint32_t ebase = (uint32_t)e0 + (uint32_t)((off - a0) / esz);
            const uint32_t sb = s0 + (uint32_t)st * kSB;
            // the whole stage at once: thread t holds vectors t, t+256, t+512, t+768
            uint32_t w[kWPT];
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
                const uint32_t v = (uint32_t)(q * kNC + tid);
                uint4 u = make_uint4(kNaNWord, kNaNWord, kNaNWord, kNaNWord);  // NaN passes no test
                if (v < nvec) u = lds_v4(sb + v * 16u);
                w[4 * q] = u.x;
                w[4 * q + 1] = u.y;
                w[4 * q + 2] = u.z;
                w[4 * q + 3] = u.w;
            }
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(empty0 + 8 * st);  // the stage is in registers
            const uint32_t idx0 = ebase + (uint32_t)tid * (uint32_t)E;
            const float mx = stage_max<BF16>(w);
            if (!fill) {
                if (mx > tau) over |= append_sparse<BF16, E>(tau, w, idx0, buf, c, steady_trig);
            } else if (!seeded && p.K <= kNC && nvec == (uint32_t)(VPT * kNC)) {
                // First full stage: the K-th largest of the per-thread maxima (and
                // the head) is at most the K-th largest element seen, since those
                // K maxima are distinct elements.  Rebuild the buffer from
                // everything at or above that bound.
                seeded = true;
                int me = -1;
#pragma unroll
                for (int e = 0; e < EPT; ++e)
                    if (me < 0 && stage_elem<BF16>(w, e) == mx) me = e;  // mx is NaN: none
                const float mxa[1] = {mx};
                append<1>(me >= 0 ? 1u : 0u, mxa, stage_index<E>(idx0, max(me, 0)), 0u, buf, c,
                          kCap);
                named_bar_sync(1, kNC);
                const int M = min((int)c->count, kCap);
                float bound = -INFINITY;
                if (M > p.K) bound = key_value(select_keep(buf, M, p.K, tmp, hist, c));
                named_bar_sync(1, kNC);  // count read (and the selection done) everywhere
                if (tid == 0) c->count = 0u;
                named_bar_sync(1, kNC);
                // -inf has no float below it: stay in fill mode then
                const bool use = bound != -INFINITY;
                const float tb = use ? nextafterf(bound, -INFINITY) : -INFINITY;
                over = append<1>(tid < head && (use ? hx[0] > tb : hx[0] == hx[0]) ? 1u : 0u, hx,
                                 (uint32_t)(e0 + tid), 0u, buf, c, kFillTrigger);
                over |= append_dense<BF16, E>(tb, !use, w, idx0, buf, c,
                                              use ? steady_trig : kFillTrigger);
                if (use) {
                    fill = false;
                    tau = tb;
                }
            } else {
                over |= append_dense<BF16, E>(-INFINITY, true, w, idx0, buf, c, kFillTrigger);
            }
            // Check at most every kCheckElems elements (fp32: every other stage).
            // Elements after a check have larger indices than every key held, so
            // after an exact selection x > tau loses nothing.
            ++ks;
            if ((BF16 || (ks & 1) == 0) && bar_red_or(1, kNC, over)) {
                tau = key_value(select_keep(buf, min((int)c->count, kCap), p.K, tmp, hist, c));
                fill = false;
                over = false;
            }
        }

        if (tail > 0) {
            const uint32_t m = tid < tail && (fill ? tx[0] == tx[0] : tx[0] > tau) ? 1u : 0u;
            append<1>(m, tx, (uint32_t)(e1 - tail + tid), 0u, buf, c, kCap);
        }
        named_bar_sync(1, kNC);
        int n = min((int)c->count, kCap);
        if (n > p.K) {
            select_keep(buf, n, p.K, tmp, hist, c);
            n = p.K;
        }

        if (cs == 1) {
            write_row<BF16>(buf, n, p, row);
            continue;
        }
        const int slot = rit & 1;
        const uint32_t par = (uint32_t)(rit >> 1) & 1u;
        if (rank != 0) {
            if (!*abort_flag &&
                !mbar_wait_cluster_bounded(smem_u32(&c->mempty[slot]), par ^ 1u, kWaitNs)) {
                *abort_flag = 1;
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_TIMEOUT);
            }
            uint64_t* o = outk + (size_t)slot * kTopkMaxK;
            for (int i = tid; i < n; i += kNC) o[i] = buf[i];
            if (tid == 0) c->out_cnt[slot] = (uint32_t)n;
            named_bar_sync(1, kNC);
            if (tid == 0) {
                fence_acq_rel_cluster();
                mbar_arrive_remote(map_cluster(smem_u32(&c->mfull[slot]), 0));
            }
        } else {
            if (!*abort_flag &&
                !mbar_wait_cluster_bounded(smem_u32(&c->mfull[slot]), par, kWaitNs)) {
                *abort_flag = 1;
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_TIMEOUT);
            }
            int M = n;
            for (int r = 1; r < cs; ++r) {
                const int cnt = (int)min(
                    ld_cluster_u32(map_cluster(smem_u32(&c->out_cnt[slot]), (uint32_t)r)),
                    (uint32_t)p.K);
                const uint32_t src =
                    map_cluster(smem_u32(outk + (size_t)slot * kTopkMaxK), (uint32_t)r);
                for (int i = tid; i < cnt; i += kNC) buf[M + i] = ld_cluster_u64(src + 8u * i);
                M += cnt;
            }
            named_bar_sync(1, kNC);
            if (tid == 0) {
                fence_acq_rel_cluster();
                for (int r = 1; r < cs; ++r)
                    mbar_arrive_remote(map_cluster(smem_u32(&c->mempty[slot]), (uint32_t)r));
            }
            if (M > p.K) {
                select_keep(buf, M, p.K, tmp, hist, c);
                M = p.K;
            }
            write_row<BF16>(buf, M, p, row);
        }
    }
    // On an abandoned pipeline, give copies still in flight a bounded time to
    // land before the CTA's shared memory is released.
    if (tid == 0 && *abort_flag) {
        for (int i = 0; i < kNS; ++i) mbar_wait_bounded(full0 + 8 * i, 0, kWaitNs / 4);
    }
    if (cs > 1) cluster_sync();  // no CTA leaves while a peer may still read it
}


// ================================================================ K <= 256
//
// For small K the filtering warps never wait for one another.  Eight filter
// warps stream the stages and push the elements that beat the published
// threshold key into their own single-producer queue; a selector warp drains
// the queues into an exact sorted top-K list and raises the threshold key
// (atomic max) as the list improves.  The threshold is a full key (value,
// then index), so the test "key > threshold" is exact in any processing
// order: the threshold is the K-th best key of a subset of the row, so every
// element of the row's top K has a larger key.  Filter warps run at most one
// row ahead of the selector.

constexpr int kAsyncMaxK = 256;
constexpr int kNF = 8;                       // filter warps
constexpr int kAThreads = (kNF + 2) * 32;    // + selector warp + producer warp
constexpr int kQW = 1024;                    // queue slots per filter warp (power of two)
static_assert(kNF * 32 == kNC, "the filter warps are the kNC threads of the seeding step");
static_assert(32 * 8 * kVPT <= kQW, "one stage's pushes must fit a queue");

constexpr uint32_t kAQueue = kNS * kSB;
constexpr uint32_t kASeedLists = kAQueue + kNF * kQW * 8;  // 2 x 256 keys
constexpr uint32_t kAList = kASeedLists + 2 * kNC * 8;
constexpr uint32_t kABatch = kAList + 2 * kAsyncMaxK * 8;
constexpr uint32_t kAOut = kABatch + 32 * 8;
constexpr uint32_t kAMerge = kAOut + 2 * kAsyncMaxK * 8;
constexpr uint32_t kACtl = kAMerge + 8 * kAsyncMaxK * 8;
constexpr uint32_t kASmem = kACtl + 512;
static_assert(kASmem <= 227 * 1024, "shared memory");

struct ACtl {
    uint64_t full[kNS];
    uint64_t empty[kNS];
    uint64_t mfull[2];
    uint64_t mempty[2];
    unsigned long long tau[2];  // published threshold key, by row parity (0: none yet)
    uint32_t qhead[kNF];        // keys pushed by each filter warp (running count)
    uint32_t qtail[kNF];        // keys the selector has taken from each queue
    uint32_t rowend[kNF][2];    // qhead at the end of a row, by row parity
    uint32_t rowtag[kNF][2];    // (row iteration + 1) that rowend belongs to
    unsigned long long seedk[2];       // seeding bound key, by row parity (0: none)
    // best bound any CTA of the cluster has for the row, by row parity:
    // (row iteration + 1) << 32 | ordered value bits; x >= that value passes
    unsigned long long cbound[2];
    uint32_t sel_done;          // rows the selector has finished
    uint32_t out_cnt[2];
    uint32_t abort;
    uint32_t fin_go, fin_s, fin_cur;  // hand-off of a short row's final selection
};
static_assert(sizeof(ACtl) <= 512, "control block");

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_u32(uint32_t* p, uint32_t v) {
    asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.volatile.shared.u64 %0, [%1];" : "=l"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

// Offers the value part of threshold key tk for row iteration rit to every CTA
// of the cluster (lane r of the calling warp writes to rank r; lanes >= cs
// idle).  The word's high half is the row tag, so a late offer for an older
// row never wins over, or passes for, the current row's.
__device__ __forceinline__ void share_bound(unsigned long long* cb, int cs, int rit,
                                            unsigned long long tk) {
    const int lane = threadIdx.x & 31;
    if (lane < cs && (tk >> 32) != 0ull) {
        const unsigned long long word = ((unsigned long long)(uint32_t)(rit + 1) << 32) | (tk >> 32);
        const uint32_t a = map_cluster(smem_u32(cb), (uint32_t)lane);
        asm volatile("red.shared::cluster.max.u64 [%0], %1;" ::"r"(a), "l"(word) : "memory");
    }
}

// Marks the pipeline abandoned (a bounded wait gave up).
__device__ __forceinline__ void set_abort(volatile uint32_t* abort_flag) {
    *abort_flag = 1;
    atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_TIMEOUT);
}

// Bounded wait until *p >= v (a running counter written with release).
__device__ __forceinline__ void wait_counter(const uint32_t* p, uint32_t v,
                                             volatile uint32_t* abort_flag) {
    if (*abort_flag || (int32_t)(ld_acquire_u32(p) - v) >= 0) return;
    const uint64_t t0 = global_ns();
    while ((int32_t)(ld_acquire_u32(p) - v) < 0) {
        if (*abort_flag) return;
        if (global_ns() - t0 > kWaitNs) {
            set_abort(abort_flag);
            return;
        }
        __nanosleep(64);
    }
}

// Element e of thread t's staged vectors, read back from the stage at sb.
template <bool BF16>
__device__ __forceinline__ float stage_elem_smem(uint32_t sb, int t, int e) {
    constexpr int E = BF16 ? 8 : 4;
    const uint32_t a = sb + (uint32_t)((e / E) * kNC + t) * 16u + (uint32_t)(e % E) * (BF16 ? 2u : 4u);
    if constexpr (BF16) {
        uint16_t h;
        asm volatile("ld.shared.u16 %0, [%1];" : "=h"(h) : "r"(a));
        return __uint_as_float((uint32_t)h << 16);
    } else {
        float f;
        asm volatile("ld.shared.f32 %0, [%1];" : "=f"(f) : "r"(a));
        return f;
    }
}

// Pushes this lane's marked staged elements (bit e of m: element e, re-read
// from the stage at sb) into the warp's queue.  Warp-collective.
template <bool BF16, int E>
__device__ __forceinline__ void push_keys(uint32_t m, uint32_t sb, uint32_t idx0, uint64_t* q,
                                          uint32_t& qh, ACtl* c, int fw,
                                          volatile uint32_t* abort_flag) {
    const int lane = threadIdx.x & 31;
    const int n = __popc(m);
    int incl;
    uint32_t tot;
    if (!__any_sync(0xffffffffu, n > 1)) {  // at most one key per lane: offsets from a ballot
        const uint32_t b = __ballot_sync(0xffffffffu, n != 0);
        incl = __popc(b & ((2u << lane) - 1u));
        tot = (uint32_t)__popc(b);
    } else {
        incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        tot = (uint32_t)__shfl_sync(0xffffffffu, incl, 31);
    }
    if (tot == 0) return;
    if (lane == 0) wait_counter(&c->qtail[fw], qh + tot - kQW, abort_flag);  // room for tot keys
    __syncwarp();
    uint32_t pos = qh + (uint32_t)(incl - n);
    for (uint32_t mm = m; mm; mm &= mm - 1u) {
        const int e = __ffs(mm) - 1;
        q[(pos++) & (kQW - 1)] =
            make_key(stage_elem_smem<BF16>(sb, (int)threadIdx.x, e), stage_index<E>(idx0, e));
    }
    __syncwarp();
    qh += tot;
    if (lane == 0) st_release_u32(&c->qhead[fw], qh);
}

// Single-value variant of push_keys (head and tail elements).
__device__ __forceinline__ void push_one(bool pass, float x, uint32_t idx, uint64_t* q,
                                         uint32_t& qh, ACtl* c, int fw,
                                         volatile uint32_t* abort_flag) {
    const int lane = threadIdx.x & 31;
    const uint32_t b = __ballot_sync(0xffffffffu, pass);
    const uint32_t tot = (uint32_t)__popc(b);
    if (tot == 0) return;
    if (lane == 0) wait_counter(&c->qtail[fw], qh + tot - kQW, abort_flag);
    __syncwarp();
    if (pass) q[(qh + (uint32_t)__popc(b & ((1u << lane) - 1u))) & (kQW - 1)] = make_key(x, idx);
    __syncwarp();
    qh += tot;
    if (lane == 0) st_release_u32(&c->qhead[fw], qh);
}

// Inserts key k into the descending list L[0, s) (capacity K), keeping the
// best K.  Precondition: s < K or k > L[K-1].  Selector warp.
__device__ __forceinline__ void list_insert(uint64_t* L, int& s, int K, uint64_t k) {
    const int lane = threadIdx.x & 31;
    int p = 0;
    for (int b = 0; b < s; b += 32) {
        const int i = b + lane;
        p += __popc(__ballot_sync(0xffffffffu, i < s && L[i] > k));
    }
    const int last = min(s, K - 1);  // L[p, last) moves one place down
    uint64_t v[kAsyncMaxK / 32];
#pragma unroll
    for (int t = 0; t < kAsyncMaxK / 32; ++t) {
        const int i = p + lane + 32 * t;
        if (i < last) v[t] = L[i];
    }
    __syncwarp();
#pragma unroll
    for (int t = 0; t < kAsyncMaxK / 32; ++t) {
        const int i = p + lane + 32 * t;
        if (i < last) L[i + 1] = v[t];
    }
    if (lane == 0) L[p] = k;
    __syncwarp();
    s = min(s + 1, K);
}

// Number of keys greater than k in the descending list l[0, n).
__device__ __forceinline__ int count_greater(const uint64_t* l, int n, uint64_t k) {
    int lo = 0, hi = n;  // answer in [lo, hi]
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (l[mid] > k)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Merges up to 32 new keys (one per lane, 0 = none; every real key beats the
// list's K-th when the list is full) into the descending list L[0, s), writing
// the best K of the union to Ln (descending).  The batch is sorted across the
// lanes with a bitonic network, then every key goes to its rank in the union:
// its own position plus the keys above it in the other sorted sequence.
__device__ __forceinline__ void list_merge(const uint64_t* L, uint64_t* Ln, int& s, int K,
                                           uint64_t k, uint64_t* Bs) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, k, j);
            const bool desc = (lane & size) == 0;
            const bool lower = (lane & j) == 0;
            k = (lower == desc) ? (k > o ? k : o) : (k < o ? k : o);
        }
    }
    const int nb = __popc(__ballot_sync(0xffffffffu, k != 0ull));  // real keys come first
    Bs[lane] = k;
    __syncwarp();
    if (lane < nb) {
        const int r = lane + count_greater(L, s, k);
        if (r < K) Ln[r] = k;
    }
    for (int i = lane; i < s; i += 32) {
        const uint64_t v = L[i];
        const int r = i + count_greater(Bs, nb, v);
        if (r < K) Ln[r] = v;
    }
    __syncwarp();
    s = min(s + nb, K);
}

// Sorts one 64-bit key per lane into descending lane order (bitonic network).
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t k) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xffffffffu, k, j);
            const bool desc = (lane & size) == 0;
            const bool lower = (lane & j) == 0;
            k = (lower == desc) ? (k > o ? k : o) : (k < o ? k : o);
        }
    }
    return k;
}

// The 32 largest of two descending lane-sorted sequences a and b, descending:
// max(a[i], b[31-i]) holds the 32 largest and is bitonic; five half-cleaner
// steps sort it.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t a, uint64_t b) {
    const int lane = threadIdx.x & 31;
    const uint64_t br = __shfl_sync(0xffffffffu, b, 31 - lane);
    uint64_t k = a > br ? a : br;
#pragma unroll
    for (int j = 16; j > 0; j >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, k, j);
        k = ((lane & j) == 0) ? (k > o ? k : o) : (k < o ? k : o);
    }
    return k;
}

// Number of keys greater than k in the descending list l[0, 32): a fixed
// binary descent (no data-dependent trip count) so that several can overlap.
__device__ __forceinline__ int count_greater32(const uint64_t* l, uint64_t k) {
    int pos = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1) pos += l[pos + step - 1] > k ? step : 0;
    return pos + (l[pos] > k ? 1 : 0);
}

// Whether every filter warp has published the end of row iteration rit.
__device__ __forceinline__ bool all_rows_ended(ACtl* c, int slot, int rit) {
    bool all = true;
#pragma unroll
    for (int w = 0; w < kNF; ++w)
        all = all && ld_acquire_u32(&c->rowtag[w][slot]) == (uint32_t)(rit + 1);
    return all;
}

// Final selection of a short row by the filter warps and the selector together
// (threads t = 0..kNC+31): the K best of the selector's sorted list L[0, s) and
// every queue's unconsumed range [qtail, rowend), each key ranked by counting
// the larger keys among all of them (keys are distinct), written in rank order.
__device__ void coop_rank(ACtl* c, int slot, const uint64_t* L, int s, const uint64_t* queues,
                          int K, uint64_t* Lout, int t, int nthreads) {
    uint32_t len[kNF + 1], q0[kNF];
    len[0] = (uint32_t)s;
    uint32_t M = (uint32_t)s;
#pragma unroll
    for (int w = 0; w < kNF; ++w) {
        q0[w] = c->qtail[w];
        len[w + 1] = c->rowend[w][slot] - q0[w];
        M += len[w + 1];
    }
    for (uint32_t j = (uint32_t)t; j < M; j += (uint32_t)nthreads) {
        uint32_t off = j;
        int seg = 0;
        while (off >= len[seg]) {
            off -= len[seg];
            ++seg;
        }
        const uint64_t k = seg == 0 ? L[off]
                                    : queues[(size_t)(seg - 1) * kQW + ((q0[seg - 1] + off) & (kQW - 1))];
        int r = 0;
        for (int i = 0; i < s; ++i) r += L[i] > k ? 1 : 0;
#pragma unroll 1
        for (int w = 0; w < kNF; ++w) {
            const uint64_t* q = queues + (size_t)w * kQW;
            for (uint32_t i = 0; i < len[w + 1]; ++i) r += q[(q0[w] + i) & (kQW - 1)] > k ? 1 : 0;
        }
        if (r < K) Lout[r] = k;
    }
}

// Writes one output row from the sorted list (selector warp).
template <bool BF16>
__device__ void write_sorted(const uint64_t* L, int n, const TopkParams& p, int row) {
    int32_t* ids = p.ids + (size_t)row * p.K;
    float* vals = p.vals + (size_t)row * p.K;
    for (int i = threadIdx.x & 31; i < p.K; i += 32) {
        int32_t id = -1;
        float v = __uint_as_float(0x7FC00000u);
        if (i < n) {
            id = (int32_t)key_index(L[i]);
            v = key_value(L[i]);
            if ((uint32_t)id >= (uint32_t)p.V) {  // not reachable with distinct keys
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
                id = -1;
                v = __uint_as_float(0x7FC00000u);
            } else if (v == 0.f) {  // the key folded -0 onto +0
                v = load_logit<BF16>(p.logits, (size_t)row * p.V + (uint32_t)id);
            }
        }
        ids[i] = id;
        vals[i] = v;
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kAThreads, 1) topk_async_kernel(TopkParams p) {
    constexpr int E = BF16 ? 8 : 4;
    constexpr int VPT = kVPT;
    constexpr int EPT = VPT * E;
    constexpr uint32_t esz = BF16 ? 2u : 4u;
    constexpr uint32_t kNaNWord = BF16 ? 0x7FC07FC0u : 0x7FC00000u;
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t s0 = smem_u32(smem);
    uint64_t* queues = reinterpret_cast<uint64_t*>(smem + kAQueue);
    uint64_t* Lbuf = reinterpret_cast<uint64_t*>(smem + kAList);  // two lists of kAsyncMaxK
    uint64_t* slists = reinterpret_cast<uint64_t*>(smem + kASeedLists);
    uint64_t* Bs = reinterpret_cast<uint64_t*>(smem + kABatch);
    uint64_t* outk = reinterpret_cast<uint64_t*>(smem + kAOut);
    uint64_t* merge = reinterpret_cast<uint64_t*>(smem + kAMerge);
    ACtl* c = reinterpret_cast<ACtl*>(smem + kACtl);
    const uint32_t full0 = smem_u32(&c->full[0]);
    const uint32_t empty0 = smem_u32(&c->empty[0]);
    volatile uint32_t* abort_flag = &c->abort;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int cs = p.cs;
    const uint32_t rank = cs > 1 ? cluster_ctarank() : 0u;
    const int cid = (int)blockIdx.x / cs;
    const int ncl = (int)gridDim.x / cs;

    if (tid == 0) {
        for (int i = 0; i < kNS; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, kNF);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&c->mfull[i]), cs > 1 ? (uint32_t)(cs - 1) : 1u);
            mbar_init(smem_u32(&c->mempty[i]), 1);
            c->tau[i] = 0ull;
        }
        for (int w = 0; w < kNF; ++w) {
            c->qhead[w] = 0u;
            c->qtail[w] = 0u;
            c->rowtag[w][0] = c->rowtag[w][1] = 0u;
            c->rowend[w][0] = c->rowend[w][1] = 0u;
        }
        c->sel_done = 0u;
        c->seedk[0] = c->seedk[1] = 0ull;
        c->cbound[0] = c->cbound[1] = 0ull;
        c->abort = 0u;
        fence_mbar_init();
    }
    if (cs > 1)
        cluster_sync();
    else
        __syncthreads();

    const int L_ = (((p.V + cs - 1) / cs) + 63) & ~63;
    const int e0 = min(p.V, (int)rank * L_);
    const int e1 = min(p.V, e0 + L_);
    const uintptr_t lbase = reinterpret_cast<uintptr_t>(p.logits);
    const int warp = tid >> 5;
    // With at most two rows per cluster (latency, not throughput, decides) each
    // row ends with a joint final selection: the selector stops draining once
    // every filter warp has finished the row, and all 288 threads rank what is
    // left (see coop_rank).  With more rows the filter warps run ahead instead.
    const bool shortrow = (p.rows + ncl - 1) / ncl <= 2;

    if (warp == kNF + 1) {
        // ---------------- producer (one lane), as in the general kernel
        if (lane == 0) {
            int it = 0;
            for (int row = cid; row < p.rows && !*abort_flag; row += ncl) {
                const uintptr_t a0 = lbase + ((size_t)row * p.V + e0) * esz;
                const uintptr_t a1 = lbase + ((size_t)row * p.V + e1) * esz;
                const uintptr_t b0 = (a0 + 15) & ~(uintptr_t)15, b1 = a1 & ~(uintptr_t)15;
                for (uintptr_t off = b0; off < b1; off += kSB, ++it) {
                    const int st = it % kNS;
                    const uint32_t ph = (uint32_t)(it / kNS) & 1u;
                    if (*abort_flag) break;
                    if (!mbar_wait_bounded(empty0 + 8 * st, ph ^ 1u, kWaitNs)) {
                        set_abort(abort_flag);
                        break;
                    }
                    const uint32_t bytes = (uint32_t)min((uintptr_t)kSB, b1 - off);
                    mbar_arrive_expect_tx(full0 + 8 * st, bytes);
                    bulk_g2s(s0 + (uint32_t)st * kSB, reinterpret_cast<const void*>(off), bytes,
                             full0 + 8 * st);
                    if (off == b0) DF2_TK_TRACE((row - cid) / ncl, 5);
                    if (off + kSB >= b1) DF2_TK_TRACE((row - cid) / ncl, 6);
                }
            }
        }
        __syncwarp();
        if (cs > 1) cluster_sync();
        return;
    }

    if (warp == kNF) {
        // ---------------- selector warp
        uint32_t qt[kNF];
#pragma unroll
        for (int w = 0; w < kNF; ++w) qt[w] = 0u;
        int rit = 0;
        int cur = 0;
        for (int row = cid; row < p.rows; row += ncl, ++rit) {
            const int slot = rit & 1;
            int s = 0;
            uint64_t* L = Lbuf + cur * kAsyncMaxK;
            uint32_t done = 0u;
            unsigned long long pub = 0ull;
            uint64_t t_idle = 0;
            uint32_t nap = 32u;  // idle back-off (ns)
            int nst = 0;  // keys staged in Bs[0, nst) for the next merge
            bool exited_early = false;
            if (p.K <= 32) {
                // The list lives in registers, lane i holding L[i]: an insertion
                // is one ballot (its place) and one shuffle (the shift), so the
                // threshold can follow every key.
                uint64_t Lr = 0ull, kth = 0ull;  // kth: L[K-1] once the list is full
                while (done != (1u << kNF) - 1u) {
                    if (shortrow && all_rows_ended(c, slot, rit)) {
                        exited_early = true;
                        break;
                    }
                    bool prog = false;
#pragma unroll
                    for (int w = 0; w < kNF; ++w) {
                        if ((done >> w) & 1u) continue;
                        const uint32_t qh = ld_acquire_u32(&c->qhead[w]);
                        const bool ended =
                            ld_acquire_u32(&c->rowtag[w][slot]) == (uint32_t)(rit + 1);
                        const uint32_t lim = ended ? c->rowend[w][slot] : qh;
                        const uint64_t* q = queues + (size_t)w * kQW;
                        while (qt[w] != lim && !*abort_flag) {
                            if (shortrow && all_rows_ended(c, slot, rit)) {
                                exited_early = true;
                                break;
                            }
                            const uint32_t nb = min(32u, lim - qt[w]);
                            const uint64_t k =
                                (uint32_t)lane < nb ? q[(qt[w] + lane) & (kQW - 1)] : 0ull;
                            uint32_t mask = __ballot_sync(0xffffffffu, k > kth);
                            qt[w] += nb;
                            prog = true;
                            __syncwarp();
                            if (lane == 0) st_release_u32(&c->qtail[w], qt[w]);
                            if (__popc(mask) >= 4) {
                                // many at once: sort them and merge with the list
                                const uint64_t kb = warp_sort_desc(k > kth ? k : 0ull);
                                Lr = warp_merge_desc(Lr, kb);
                                if (lane >= p.K) Lr = 0ull;
                                s = min(s + __popc(mask), p.K);
                                if (s == p.K) kth = __shfl_sync(0xffffffffu, Lr, p.K - 1);
                                mask = 0u;
                            }
                            while (mask) {
                                const int b = __ffs(mask) - 1;
                                mask &= mask - 1u;
                                const uint64_t kk = __shfl_sync(0xffffffffu, k, b);
                                if (kk <= kth) continue;
                                const int pos =
                                    __popc(__ballot_sync(0xffffffffu, lane < s && Lr > kk));
                                const uint64_t up = __shfl_up_sync(0xffffffffu, Lr, 1);
                                Lr = lane < pos ? Lr : (lane == pos ? kk : up);
                                if (lane >= p.K) Lr = 0ull;
                                s = min(s + 1, p.K);
                                if (s == p.K) kth = __shfl_sync(0xffffffffu, Lr, p.K - 1);
                            }
                            if (kth > pub) {
                                pub = kth;
                                if (lane == 0) atomicMax(&c->tau[slot], pub);
                                if (cs > 1) share_bound(&c->cbound[slot], cs, rit, pub);
                            }
                        }
                        if (exited_early) break;
                        if (ended && qt[w] == lim) done |= 1u << w;
                        if (*abort_flag) done |= 1u << w;
                    }
                    if (exited_early) break;
                    if (prog) {
                        t_idle = 0;
                        nap = 32u;
                    } else {
                        const uint64_t now = global_ns();
                        if (t_idle == 0) t_idle = now;
                        else if (now - t_idle > kWaitNs) set_abort(abort_flag);
                        __nanosleep(nap);
                        nap = min(2u * nap, 512u);
                    }
                }
                if (lane < s) L[lane] = Lr;
            }
            for (int pass = 0; pass < 2; ++pass) {
            if (pass == 1) {
                if (!shortrow) break;
                // Short row: hand the rest to the whole CTA (when it is small)
                uint32_t M = (uint32_t)s;
#pragma unroll
                for (int w = 0; w < kNF; ++w) M += c->rowend[w][slot] - qt[w];
                const bool go = exited_early && !*abort_flag && M <= 1024u;
                if (lane == 0) {
                    c->fin_go = go ? 1u : 0u;
                    c->fin_s = (uint32_t)s;
                    c->fin_cur = (uint32_t)cur;
                }
                __syncwarp();
                named_bar_sync(2, kNC + 32);
                if (go) coop_rank(c, slot, L, s, queues, p.K, Lbuf + (cur ^ 1) * kAsyncMaxK,
                                  tid, kNC + 32);
                named_bar_sync(2, kNC + 32);
                if (go) {
                    s = (int)min(M, (uint32_t)p.K);
                    cur ^= 1;
                    L = Lbuf + cur * kAsyncMaxK;
#pragma unroll
                    for (int w = 0; w < kNF; ++w) qt[w] = c->rowend[w][slot];
                    if (lane < kNF) st_release_u32(&c->qtail[lane], c->rowend[lane][slot]);
                    done = (1u << kNF) - 1u;
                }
                if (go || !exited_early) break;
                exited_early = false;  // too much left: drain it here after all
            }
            while (!exited_early && done != (1u << kNF) - 1u) {
                if (pass == 0 && shortrow && all_rows_ended(c, slot, rit)) {
                    exited_early = true;
                    break;
                }
                bool prog = false;
#pragma unroll
                for (int w = 0; w < kNF; ++w) {
                    if ((done >> w) & 1u) continue;
                    // qhead before the tag: if the tag is not yet set, every key
                    // below that qhead belongs to this row
                    const uint32_t qh = ld_acquire_u32(&c->qhead[w]);
                    const bool ended = ld_acquire_u32(&c->rowtag[w][slot]) == (uint32_t)(rit + 1);
                    const uint32_t lim = ended ? c->rowend[w][slot] : qh;
                    const uint64_t* q = queues + (size_t)w * kQW;
                    while (qt[w] != lim && !*abort_flag) {
                        if (pass == 0 && shortrow && all_rows_ended(c, slot, rit)) {
                            exited_early = true;
                            break;
                        }
                        // stage the keys that beat the list's K-th (32 at most)
                        const uint32_t nb = min((uint32_t)(32 - nst), lim - qt[w]);
                        const uint64_t k = (uint32_t)lane < nb ? q[(qt[w] + lane) & (kQW - 1)] : 0ull;
                        const bool cand = (uint32_t)lane < nb && (s < p.K || k > L[p.K - 1]);
                        const uint32_t mask = __ballot_sync(0xffffffffu, cand);
                        if (cand) Bs[nst + __popc(mask & ((1u << lane) - 1u))] = k;
                        nst += __popc(mask);
                        qt[w] += nb;
                        prog = true;
                        __syncwarp();
                        if (lane == 0) st_release_u32(&c->qtail[w], qt[w]);
                        if (nst >= 24) {
                            uint64_t* Ln = Lbuf + (cur ^ 1) * kAsyncMaxK;
                            const uint64_t kb = lane < nst ? Bs[lane] : 0ull;
                            __syncwarp();
                            list_merge(L, Ln, s, p.K, kb, Bs);
                            cur ^= 1;
                            L = Ln;
                            nst = 0;
                            if (s == p.K && L[p.K - 1] > pub) {
                                pub = L[p.K - 1];
                                if (lane == 0) atomicMax(&c->tau[slot], pub);
                                if (cs > 1) share_bound(&c->cbound[slot], cs, rit, pub);
                            }
                        }
                    }
                    if (ended && qt[w] == lim) done |= 1u << w;
                    if (*abort_flag) done |= 1u << w;
                }
                // merge what is staged (a few keys: one by one), re-checking each
                // against the K-th, which staging may have raised meanwhile
                if (nst > 3) {
                    uint64_t* Ln = Lbuf + (cur ^ 1) * kAsyncMaxK;
                    uint64_t kb = lane < nst ? Bs[lane] : 0ull;
                    if (s == p.K && kb != 0ull && kb <= L[p.K - 1]) kb = 0ull;
                    __syncwarp();
                    list_merge(L, Ln, s, p.K, kb, Bs);
                    cur ^= 1;
                    L = Ln;
                } else {
                    for (int i = 0; i < nst; ++i) {
                        const uint64_t kk = Bs[i];
                        if (s < p.K || kk > L[p.K - 1]) list_insert(L, s, p.K, kk);
                    }
                }
                nst = 0;
                if (s == p.K && L[p.K - 1] > pub) {
                    pub = L[p.K - 1];
                    if (lane == 0) atomicMax(&c->tau[slot], pub);
                                if (cs > 1) share_bound(&c->cbound[slot], cs, rit, pub);
                }
                if (prog) {
                    t_idle = 0;
                    nap = 32u;
                } else {
                    const uint64_t now = global_ns();
                    if (t_idle == 0) t_idle = now;
                    else if (now - t_idle > kWaitNs) set_abort(abort_flag);
                    __nanosleep(nap);
                    nap = min(2u * nap, 512u);
                }
            }
            }
            __syncwarp();
            if (cs == 1) {
                write_sorted<BF16>(L, s, p, row);
            } else {
                const uint32_t par = (uint32_t)(rit >> 1) & 1u;
                if (rank != 0) {
                    if (!*abort_flag &&
                        !mbar_wait_cluster_bounded(smem_u32(&c->mempty[slot]), par ^ 1u, kWaitNs))
                        set_abort(abort_flag);
                    uint64_t* o = outk + (size_t)slot * kAsyncMaxK;
                    for (int i = lane; i < s; i += 32) o[i] = L[i];
                    if (lane == 0) c->out_cnt[slot] = (uint32_t)s;
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_cluster();
                        mbar_arrive_remote(map_cluster(smem_u32(&c->mfull[slot]), 0));
                    }
                } else {
                    if (!*abort_flag &&
                        !mbar_wait_cluster_bounded(smem_u32(&c->mfull[slot]), par, kWaitNs))
                        set_abort(abort_flag);
                    // the cs sorted lists side by side, K apart: list 0 is ours.  The
                    // counts come in one parallel round of remote loads (lane r reads
                    // rank r's), the keys in batches of 8 loads per lane before any store.
                    const uint32_t myc =
                        (lane >= 1 && lane < cs)
                            ? min(ld_cluster_u32(map_cluster(smem_u32(&c->out_cnt[slot]),
                                                             (uint32_t)lane)),
                                  (uint32_t)p.K)
                            : 0u;
                    for (int i = lane; i < s; i += 32) merge[i] = L[i];
                    int cnt[8];  // every lane holds every rank's count (shuffled, no divergence)
                    cnt[0] = s;
                    int tot_remote = 0;
#pragma unroll
                    for (int r = 1; r < 8; ++r) {
                        cnt[r] = (int)__shfl_sync(0xffffffffu, myc, r);
                        tot_remote += cnt[r];
                    }
                    for (int j0 = 0; j0 < tot_remote; j0 += 32 * 8) {
                        uint64_t v[8];
                        int dst[8];
#pragma unroll
                        for (int m = 0; m < 8; ++m) {
                            int j = j0 + 32 * m + lane;
                            dst[m] = -1;
                            if (j < tot_remote) {
                                int r = 1;
                                while (r < 7 && j >= cnt[r]) {  // the rank whose list holds j
                                    j -= cnt[r];
                                    ++r;
                                }
                                dst[m] = r * kAsyncMaxK + j;
                                v[m] = ld_cluster_u64(map_cluster(
                                    smem_u32(outk + (size_t)slot * kAsyncMaxK + j), (uint32_t)r));
                            }
                        }
#pragma unroll
                        for (int m = 0; m < 8; ++m)
                            if (dst[m] >= 0) merge[dst[m]] = v[m];
                    }
                    __syncwarp();
                    if (lane == 0) {
                        fence_acq_rel_cluster();
                        for (int r = 1; r < cs; ++r)
                            mbar_arrive_remote(
                                map_cluster(smem_u32(&c->mempty[slot]), (uint32_t)r));
                    }
                    // rank of each key in the union: its place in its own list plus
                    // the keys above it in the others (keys are distinct)
                    int total = 0;
                    for (int r = 0; r < cs; ++r) total += cnt[r];
                    int32_t* ids = p.ids + (size_t)row * p.K;
                    float* vals = p.vals + (size_t)row * p.K;
                    for (int r = 0; r < cs; ++r) {
                        for (int i = lane; i < cnt[r]; i += 32) {
                            const uint64_t k = merge[r * kAsyncMaxK + i];
                            int rk = i;
                            for (int r2 = 0; r2 < cs; ++r2)
                                if (r2 != r) rk += count_greater(merge + r2 * kAsyncMaxK, cnt[r2], k);
                            if (rk < p.K) {
                                int32_t id = (int32_t)key_index(k);
                                float v = key_value(k);
                                if ((uint32_t)id >= (uint32_t)p.V) {
                                    atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
                                    id = -1;
                                    v = __uint_as_float(0x7FC00000u);
                                } else if (v == 0.f) {
                                    v = load_logit<BF16>(p.logits, (size_t)row * p.V + (uint32_t)id);
                                }
                                ids[rk] = id;
                                vals[rk] = v;
                            }
                        }
                    }
                    for (int i = total + lane; i < p.K; i += 32) {
                        ids[i] = -1;
                        vals[i] = __uint_as_float(0x7FC00000u);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                c->tau[slot] = 0ull;  // free for row rit + 2
                st_release_u32(&c->sel_done, (uint32_t)(rit + 1));
                DF2_TK_TRACE(rit, 4);
            }
        }
        __syncwarp();
        if (cs > 1) cluster_sync();
        return;
    }

    // ---------------- filter warps
    uint64_t* myq = queues + (size_t)warp * kQW;
    uint32_t qh = 0u;
    int fst = 0, rit = 0;  // ring stage and its phase parity, carried across rows
    uint32_t fph = 0u;
    for (int row = cid; row < p.rows; row += ncl, ++rit) {
        const int slot = rit & 1;
        const size_t rowoff = (size_t)row * p.V;
        const uintptr_t a0 = lbase + (rowoff + e0) * esz;
        const uintptr_t a1 = lbase + (rowoff + e1) * esz;
        const uintptr_t b0 = (a0 + 15) & ~(uintptr_t)15, b1 = a1 & ~(uintptr_t)15;
        const bool body = b0 < b1;
        const int head = body ? (int)((b0 - a0) / esz) : e1 - e0;
        const int tail = body ? (int)((a1 - b1) / esz) : 0;
        // the same for every row of this CTA (the chunk length is), so the
        // filter warps pass the seeding barrier on the same rows
        const bool seedable = p.K <= kAsyncMaxK && (uint32_t)(e1 - e0) * esz >= kSB + 32u;
        unsigned long long seed_key = 0ull;
        float hx = 0.f, tx = 0.f;
        if (tid < head) hx = load_logit<BF16>(p.logits, rowoff + e0 + tid);
        if (tid < tail) tx = load_logit<BF16>(p.logits, rowoff + (e1 - tail) + tid);
        // At most one row ahead of the selector: it has finished the row that
        // last used this threshold slot and reset it to 0 (no threshold).
        if (tid == 0) DF2_TK_TRACE(rit, 0);
        if (lane == 0 && rit >= 2) wait_counter(&c->sel_done, (uint32_t)(rit - 1), abort_flag);
        __syncwarp();
        if (tid == 0) DF2_TK_TRACE(rit, 1);
        if (!seedable && warp == 0)
            push_one(tid < head && hx == hx, hx, (uint32_t)(e0 + tid), myq, qh, c, warp, abort_flag);

        int ks = 0;
        for (uintptr_t off = b0; off < b1; off += kSB, ++ks) {
            const int st = fst;
            const uint32_t ph = fph;
            if (++fst == kNS) {
                fst = 0;
                fph ^= 1u;
            }
            if (!*abort_flag && !mbar_wait_bounded(full0 + 8 * st, ph, kWaitNs)) set_abort(abort_flag);
            const uint32_t nvec = (uint32_t)min((uintptr_t)kSB, b1 - off) / 16u;
            const uint32_t ebase = (uint32_t)e0 + (uint32_t)((off - a0) / esz);
            const uint32_t sb = s0 + (uint32_t)st * kSB;
            uint32_t w[kWPT];
#pragma unroll
            for (int q = 0; q < VPT; ++q) {
                const uint32_t v = (uint32_t)(q * kNC + tid);
                uint4 u = make_uint4(kNaNWord, kNaNWord, kNaNWord, kNaNWord);  // NaN passes no test
                if (v < nvec) u = lds_v4(sb + v * 16u);
                w[4 * q] = u.x;
                w[4 * q + 1] = u.y;
                w[4 * q + 2] = u.z;
                w[4 * q + 3] = u.w;
            }
            const uint32_t idx0 = ebase + (uint32_t)tid * (uint32_t)E;
            const float mx = stage_max<BF16>(w);
            if (seedable && ks == 0) {
                // First (full) stage: the K-th largest of the 256 lane maxima is at
                // most the row's K-th best (those K maxima are distinct elements).
                // Every warp sorts its 32 maxima.  For K <= 32 a tree of pairwise
                // merges (warps w and w+4, then w and w+2, then 0 and 1) leaves the
                // best 32 of all 256 in warp 0, whose lane K-1 is the bound; for
                // larger K a candidate's rank among all 256 is its place in its own
                // list plus the keys above it in the other seven (binary searches),
                // and the one of rank K-1 is the bound.
                int me = -1;
#pragma unroll
                for (int e = 0; e < EPT; ++e)
                    if (me < 0 && stage_elem<BF16>(w, e) == mx) me = e;  // mx is NaN: none
                const uint64_t kk =
                    warp_sort_desc(me >= 0 ? make_key(mx, stage_index<E>(idx0, me)) : 0ull);
                uint64_t* sl = slists + (size_t)slot * kNC;  // 8 sorted lists of 32
                sl[tid] = kk;
                named_bar_sync(1, kNC);
                if (tid == 0) c->seedk[slot ^ 1] = 0ull;  // the other row's readers are done
                if (p.K <= 32) {
                    // each level reads lists the level before wrote and writes only
                    // the reading warps' own slots
                    uint64_t best = kk;
                    if (warp < 4) {
                        best = warp_merge_desc(best, sl[(warp + 4) * 32 + lane]);
                        sl[tid] = best;
                        named_bar_sync(3, 128);
                    }
                    if (warp < 2) {
                        best = warp_merge_desc(best, sl[(warp + 2) * 32 + lane]);
                        sl[tid] = best;
                        named_bar_sync(4, 64);
                    }
                    if (warp == 0) {
                        best = warp_merge_desc(best, sl[32 + lane]);
                        if (lane == p.K - 1) c->seedk[slot] = best;  // 0: fewer than K keys
                    }
                } else if (kk != 0ull && lane < p.K) {
                    int rk = lane;
#pragma unroll
                    for (int v = 0; v < kNF; ++v)
                        if (v != warp) rk += count_greater32(sl + v * 32, kk);
                    if (rk == p.K - 1) c->seedk[slot] = kk;
                }
                named_bar_sync(1, kNC);
                const uint64_t bk = c->seedk[slot];
                // 0: fewer than K lanes held a non-NaN element (no bound); a bound
                // of -inf has no float below it either
                if (bk != 0ull && key_value(bk) != -INFINITY && tid == 0)
                    atomicMax(&c->tau[slot], make_key(key_value(bk), 0xFFFFFFFFu));
                if (warp == 0) {
                    unsigned long long tk = ld_volatile_u64(&c->tau[slot]);
                    if (bk != 0ull && key_value(bk) != -INFINITY)
                        tk = max(tk, (unsigned long long)make_key(key_value(bk), 0xFFFFFFFFu));
                    const bool pass = tid < head && hx == hx && make_key(hx, (uint32_t)(e0 + tid)) > tk;
                    push_one(pass, hx, (uint32_t)(e0 + tid), myq, qh, c, warp, abort_flag);
                }
                seed_key = (bk != 0ull && key_value(bk) != -INFINITY)
                               ? (unsigned long long)make_key(key_value(bk), 0xFFFFFFFFu)
                               : 0ull;
                if (cs > 1 && warp == 0) share_bound(&c->cbound[slot], cs, rit, seed_key);
            }
            unsigned long long tk = max(ld_volatile_u64(&c->tau[slot]), seed_key);
            if (cs > 1) {
                const unsigned long long cw = ld_volatile_u64(&c->cbound[slot]);
                if ((uint32_t)(cw >> 32) == (uint32_t)(rit + 1)) tk = max(tk, (cw & 0xFFFFFFFFull) << 32);
            }
            const float tv = (tk >> 32) == 0ull ? -INFINITY : key_value(tk);
            if (__any_sync(0xffffffffu, mx >= tv)) {
                // key > tk: value above tv, or equal to it (-0 == +0) with an
                // index below the threshold's (complemented in the key)
                uint32_t m, mt;
                stage_cmp_masks<BF16>(w, tv, m, mt);
                const uint32_t ti = ~(uint32_t)tk;
                for (uint32_t mm = mt; mm; mm &= mm - 1u) {
                    const int e = __ffs(mm) - 1;
                    if (stage_index<E>(idx0, e) < ti) m |= 1u << e;
                }
                push_keys<BF16, E>(m, sb, idx0, myq, qh, c, warp, abort_flag);
            }
            __syncwarp();
            if (tid == 0 && ks == 0) DF2_TK_TRACE(rit, 2);
            if (lane == 0) mbar_arrive(empty0 + 8 * st);  // done with the stage
        }
        if (tid == 0) DF2_TK_TRACE(rit, 3);
        if (tid == 224) DF2_TK_TRACE(rit, 7);
        if (warp == 0 && tail > 0) {
            const unsigned long long tk = ld_volatile_u64(&c->tau[slot]);
            const uint32_t ti = (uint32_t)(e1 - tail + tid);
            push_one(tid < tail && tx == tx && make_key(tx, ti) > tk, tx, ti, myq, qh, c, warp,
                     abort_flag);
        }
        __syncwarp();
        if (lane == 0) {
            c->rowend[warp][slot] = qh;
            st_release_u32(&c->rowtag[warp][slot], (uint32_t)(rit + 1));
        }
        if (shortrow) {
            named_bar_sync(2, kNC + 32);
            if (c->fin_go)
                coop_rank(c, slot, Lbuf + c->fin_cur * kAsyncMaxK, (int)c->fin_s, queues, p.K,
                          Lbuf + (c->fin_cur ^ 1) * kAsyncMaxK, tid, kNC + 32);
            named_bar_sync(2, kNC + 32);
        }
    }
    // On an abandoned pipeline, give copies still in flight a bounded time to
    // land before the CTA's shared memory is released.
    if (tid == 0 && *abort_flag) {
        for (int i = 0; i < kNS; ++i) mbar_wait_bounded(full0 + 8 * i, 0, kWaitNs / 4);
    }
    __syncwarp();
    if (cs > 1) cluster_sync();
}

// ---------------------------------------------------------------- few rows
// topk_rows_kernel (K <= 32, rows few enough that one cluster per row fits the
// GPU at once, as for a draft block's 16 rows): the per-row fixed costs of the
// streaming kernels (seeding, queue hand-offs, the joint selection) dominate
// there, so this kernel reads its chunk of the row into registers in one go
// and selects in a few block-wide steps:
//  1. CTA r of the row's cluster owns elements [r*chunk, (r+1)*chunk) (chunk a
//     multiple of one 16-byte vector); thread t holds vectors t, t + 512, ...
//     (at most VPT), all loaded up front with 16-byte read-only loads;
//  2. each thread's best key (NaN skipped); the 512 keys are sorted by warp
//     bitonic sorts and pairwise bitonic merges, and the K-th largest, tau,
//     bounds the chunk's K-th best key from below (the K thread maxima at or
//     above it are K distinct elements);
//  3. every element with key >= tau joins a shared candidate list: only the K
//     threads whose maximum is at or above tau can contribute, so the list
//     holds at most K times a thread's element count; up to 512 candidates
//     are sorted by the same warp sorts and merges, only as many lists as they
//     fill (more, only possible for adversarial chunks, are first cut to the K
//     best by an exact select);
//  4. the other ranks store their sorted lists into rank 0's shared memory
//     (distributed shared memory) before one cluster barrier; rank 0 merges
//     them pairwise and writes the row from the sorted result.
// The cluster size is the largest in 1..8 (not only powers of two) whose
// clusters for all rows are resident at once.
// Keys, ties, NaN and the sign of zero follow the streaming kernels exactly.
constexpr int kRowsMaxK = 32;
constexpr int kRowsThreads = 512;                  // the first kNC run the exact select
constexpr int kRowsVpts[5] = {4, 8, 12, 16, 20};   // 16-byte vectors per thread
constexpr int kRowsMaxVpt = 20;
constexpr int kRowsCap = kRowsMaxK * kRowsMaxVpt * 8;  // candidate keys at most (bf16)

struct RowsSmem {
    uint64_t cand[kRowsCap];
    uint64_t lists[kRowsThreads];          // sorted keys, 16 x 32
    uint64_t merge[8 * 32];                // rank r's sorted top 32 (rank 0's copy)
    uint64_t tmp[kRowsMaxK];
    uint32_t hist[256];
    Ctl ctl;
};

__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

// Pairwise merges of n (<= 16) descending 32-key lists held at
// lists[32*w .. 32*w + 31] into the sorted top 32 at lists[0 .. 31], as a
// binary tree in which a list without a partner waits a round;
// block-collective (every thread calls it).
__device__ __forceinline__ void rows_merge_lists(uint64_t* lists, int n) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
#pragma unroll 1
    for (int step = 1; step < n; step <<= 1) {
        if ((warp & (2 * step - 1)) == 0 && warp + step < n) {
            const uint64_t m = warp_merge_desc(lists[warp * 32 + lane], lists[(warp + step) * 32 + lane]);
            __syncwarp();
            lists[warp * 32 + lane] = m;
        }
        __syncthreads();
    }
}

// Element j (in index order) of a 16-byte vector: fp32 4 per vector, bf16 8.
template <bool BF16>
__device__ __forceinline__ float rows_elem(const uint4& w, int j) {
    const uint32_t q = j < (BF16 ? 2 : 1) ? w.x : j < (BF16 ? 4 : 2) ? w.y : j < (BF16 ? 6 : 3) ? w.z : w.w;
    if constexpr (BF16) return __uint_as_float((j & 1) ? (q & 0xFFFF0000u) : (q << 16));
    return __uint_as_float(q);
}

template <bool BF16, int VPT>
__global__ void __launch_bounds__(kRowsThreads, 1) topk_rows_kernel(const TopkParams p) {
    constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
    extern __shared__ __align__(16) uint8_t rows_smem_raw[];
    RowsSmem& sm = *reinterpret_cast<RowsSmem*>(rows_smem_raw);
    const int tid = threadIdx.x;
    const int P = p.cs;
    const int rank = P > 1 ? (int)cluster_ctarank() : 0;
    const int row = blockIdx.x / P;
    const int K = p.K;
    // chunk: a multiple of EPV elements (the launcher checked that the row
    // starts are 16-byte aligned and that a chunk fits VPT vectors per thread)
    const int chunk = ((p.V + P - 1) / P + EPV - 1) / EPV * EPV;
    const int c0 = min(p.V, rank * chunk);
    const int c1 = min(p.V, c0 + chunk);
    const int nvec = (c1 - c0) / EPV;  // V is a multiple of EPV
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.logits) +
                                                      ((size_t)row * p.V + c0) * (BF16 ? 2 : 4));

    // 1. the thread's vectors (NaN words past the end: never candidates)
    constexpr uint32_t kNaNWord = BF16 ? 0x7FC07FC0u : 0x7FC00000u;
    uint4 w[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        const int v = tid + kRowsThreads * k;
        w[k] = v < nvec ? ldg_nc_v4(src + v) : make_uint4(kNaNWord, kNaNWord, kNaNWord, kNaNWord);
    }
    if (tid == 0) sm.ctl.count = 0u;

    // 2. the thread's best key (0: no non-NaN element), then tau.  Over
    // increasing indices a strict ">" keeps the first of equal values (-0 and
    // +0 compare equal, as the keys order them) and skips NaN; a thread whose
    // non-NaN elements are all -inf sets nothing and takes its first one.
    float mx = -INFINITY;
    int bi = -1, first = -1;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int j = 0; j < EPV; ++j) {
            const float x = rows_elem<BF16>(w[k], j);
            const int idx = c0 + (tid + kRowsThreads * k) * EPV + j;
            if (x > mx) {
                mx = x;
                bi = idx;
            }
            if (first < 0 && x == x) first = idx;
        }
    if (bi < 0) bi = first;  // all -inf (mx stays -inf), or none (bi = -1)
    const uint64_t best = bi < 0 ? 0ull : make_key(mx, (uint32_t)bi);
    sm.lists[tid] = warp_sort_desc(best);
    __syncthreads();
    rows_merge_lists(sm.lists, kRowsThreads / 32);
    // tau = the K-th key; with fewer than K thread maxima (key 0) every non-NaN
    // element passes: the bound (-inf, last index) below every key
    const uint64_t tau = sm.lists[K - 1];
    const float tv = tau == 0 ? -INFINITY : key_value(tau);
    const uint32_t ti = tau == 0 ? 0xFFFFFFFFu : key_index(tau);

    // 3. candidates: key >= tau, i.e. value > tv, or value == tv (-0 == +0)
    // at an index <= ti; a compare per element into a mask, the exact test and
    // the append only for the rare vectors with an element at or above tv
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        uint32_t m = 0;
#pragma unroll
        for (int j = 0; j < EPV; ++j) m |= (rows_elem<BF16>(w[k], j) >= tv ? 1u : 0u) << j;
        if (m != 0) {
#pragma unroll
            for (int j = 0; j < EPV; ++j) {
                if (!((m >> j) & 1u)) continue;
                const float x = rows_elem<BF16>(w[k], j);
                const uint32_t idx = (uint32_t)(c0 + (tid + kRowsThreads * k) * EPV + j);
                if (x > tv || idx <= ti) {
                    const uint32_t pos = atomicAdd(&sm.ctl.count, 1u);
                    if (pos < (uint32_t)kRowsCap)
                        sm.cand[pos] = make_key(x, idx);
                    else
                        atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
                }
            }
        }
    }
    __syncthreads();
    int M = min((int)sm.ctl.count, kRowsCap);
    // the CTA's K best, sorted: at most 512 candidates are sorted directly
    // (one key per thread, missing ones as key 0); more (only for adversarial
    // chunks) are first cut to the K best by the exact radix / counting select
    if (M > kRowsThreads) {
        if (tid < kNC) select_keep(sm.cand, M, K, sm.tmp, sm.hist, &sm.ctl);
        M = K;
        __syncthreads();
    }
    // sorted lists of 32 (the last padded with key 0), merged pairwise
    int nl = 1;
    while (nl * 32 < M) nl <<= 1;
    if ((tid >> 5) < nl) sm.lists[tid] = warp_sort_desc(tid < M ? sm.cand[tid] : 0ull);
    __syncthreads();
    rows_merge_lists(sm.lists, nl);

    // 4. the cluster's sorted lists meet in rank 0, which merges them
    const uint64_t* top = sm.lists;
    if (P > 1) {
        if (rank == 0) {
            if (tid < 32) sm.merge[tid] = sm.lists[tid];
        } else if (tid < 32) {
            const uint32_t a = smem_u32(sm.merge) + (uint32_t)((rank * 32 + tid) * 8);
            st_cluster_u64(map_cluster(a, 0u), sm.lists[tid]);
        }
        cluster_sync();  // release / acquire: the lists are in rank 0
        if (rank != 0) return;
        rows_merge_lists(sm.merge, P);
        top = sm.merge;
    }
    // 5. the row, straight from the sorted list (key 0: fewer than K entries)
    if (tid < K) {
        const uint64_t k = top[tid];
        int32_t id = -1;
        float v = __uint_as_float(0x7FC00000u);
        if (k != 0) {
            id = (int32_t)key_index(k);
            v = key_value(k);  // exact, except that the key folded -0 onto +0
            if ((uint32_t)id >= (uint32_t)p.V) {  // not reachable with distinct keys
                atomicOr(&g_topk_fault, (unsigned)DF2_FLAG_OVERFLOW);
                id = -1;
                v = __uint_as_float(0x7FC00000u);
            } else if (v == 0.f) {
                v = load_logit<BF16>(p.logits, (size_t)row * p.V + (uint32_t)id);
            }
        }
        p.ids[(size_t)row * K + tid] = id;
        p.vals[(size_t)row * K + tid] = v;
    }
}

struct DeviceInfo {
    bool ready = false;
    int max_clusters[2][2][4] = {};  // [async][bf16][log2 cs]: clusters resident at once
    int rows_clusters[2][5][9] = {};  // few-row kernel: [bf16][VPT index][cluster size 1..8]
};

std::mutex g_mu;
DeviceInfo g_info[64];

template <typename Kern>
cudaError_t query_kernel(Kern kern, uint32_t smem_bytes, int threads, int (&out)[4]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes);
    if (e != cudaSuccess) return e;
    for (int l = 0; l < 4; ++l) {
        const int cs = 1 << l;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(cs, 1, 1);
        cfg.blockDim = dim3(threads, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        out[l] = n;
    }
    return cudaSuccess;
}

// Clusters of the few-row kernel resident at once, for every cluster size 1..8
// (its merge takes any size, not only powers of two).
template <typename Kern>
cudaError_t query_rows_kernel(Kern kern, uint32_t smem_bytes, int (&out)[9]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem_bytes);
    if (e != cudaSuccess) return e;
    out[0] = 0;
    for (int cs = 1; cs <= 8; ++cs) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(cs, 1, 1);
        cfg.blockDim = dim3(kRowsThreads, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        out[cs] = n;
    }
    return cudaSuccess;
}

cudaError_t query_device(DeviceInfo& d) {
    cudaError_t e = query_kernel(topk_kernel<false>, kSmem, kThreads, d.max_clusters[0][0]);
    if (e == cudaSuccess) e = query_kernel(topk_kernel<true>, kSmem, kThreads, d.max_clusters[0][1]);
    if (e == cudaSuccess)
        e = query_kernel(topk_async_kernel<false>, kASmem, kAThreads, d.max_clusters[1][0]);
    if (e == cudaSuccess)
        e = query_kernel(topk_async_kernel<true>, kASmem, kAThreads, d.max_clusters[1][1]);
    constexpr uint32_t rs = (uint32_t)sizeof(RowsSmem);
#define DF2_ROWS_Q(BF, I)                                                                         \
    if (e == cudaSuccess)                                                                         \
        e = query_rows_kernel(topk_rows_kernel<BF, kRowsVpts[I]>, rs,                            \
                              d.rows_clusters[BF ? 1 : 0][I]);
    DF2_ROWS_Q(false, 0) DF2_ROWS_Q(false, 1) DF2_ROWS_Q(false, 2) DF2_ROWS_Q(false, 3)
    DF2_ROWS_Q(false, 4) DF2_ROWS_Q(true, 0) DF2_ROWS_Q(true, 1) DF2_ROWS_Q(true, 2)
    DF2_ROWS_Q(true, 3) DF2_ROWS_Q(true, 4)
#undef DF2_ROWS_Q
    return e;
}

template <bool BF16>
cudaError_t launch_rows(const TopkParams& p, int vi, cudaStream_t stream) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(p.rows * p.cs), 1, 1);
    cfg.blockDim = dim3(kRowsThreads, 1, 1);
    cfg.dynamicSmemBytes = sizeof(RowsSmem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = p.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.cs > 1 ? 1 : 0;
    switch (vi) {
        case 0: return cudaLaunchKernelEx(&cfg, topk_rows_kernel<BF16, kRowsVpts[0]>, p);
        case 1: return cudaLaunchKernelEx(&cfg, topk_rows_kernel<BF16, kRowsVpts[1]>, p);
        case 2: return cudaLaunchKernelEx(&cfg, topk_rows_kernel<BF16, kRowsVpts[2]>, p);
        case 3: return cudaLaunchKernelEx(&cfg, topk_rows_kernel<BF16, kRowsVpts[3]>, p);
        default: return cudaLaunchKernelEx(&cfg, topk_rows_kernel<BF16, kRowsVpts[4]>, p);
    }
}

cudaError_t launch_any(const TopkLaunch& a, cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    const bool async = a.K <= kAsyncMaxK;
    int maxc[4];
    int rows_cs = 0, rows_vi = 0;  // the few-row kernel's cluster size and vectors per thread
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DeviceInfo& d = g_info[dev];
        if (!d.ready) {
            e = query_device(d);
            if (e != cudaSuccess) return e;
            d.ready = true;
        }
        for (int l = 0; l < 4; ++l) maxc[l] = d.max_clusters[async ? 1 : 0][a.bf16 ? 1 : 0][l];
        // few rows, small K: one cluster per row if the whole batch fits at once
        // (the largest cluster, for the most parallel reads), each CTA's chunk
        // in its registers, 16-byte aligned
        const int esz = a.bf16 ? 2 : 4;
        if (a.K <= kRowsMaxK && (a.V * esz) % 16 == 0 &&
            reinterpret_cast<uintptr_t>(a.logits) % 16 == 0) {
            for (int P = 8; P >= 1 && rows_cs == 0; --P) {
                const long long vecs = ((long long)(a.V + P - 1) / P * esz + 15) / 16 + 1;
                const long long vpt = (vecs + kRowsThreads - 1) / kRowsThreads;
                int vi = 0;
                while (vi < 5 && kRowsVpts[vi] < vpt) ++vi;
                if (vi == 5) break;  // smaller clusters: longer chunks
                if (a.rows <= d.rows_clusters[a.bf16 ? 1 : 0][vi][P]) {
                    rows_cs = P;
                    rows_vi = vi;
                }
            }
        }
    }
    if (rows_cs > 0) {
        const TopkParams rp{a.logits, a.rows, a.V, a.K, rows_cs, a.ids, a.vals};
        return a.bf16 ? launch_rows<true>(rp, rows_vi, stream) : launch_rows<false>(rp, rows_vi, stream);
    }
    // cluster size: the fewest waves of the longest per-CTA chunk, plus a fixed
    // per-row cost (seeding, selection, merge) worth about 8192 elements
    int best_l = -1;
    long long best_cost = 0;
    for (int l = 0; l < 4; ++l) {
        if (maxc[l] <= 0) continue;
        const int cs = 1 << l;
        const long long waves = (a.rows + maxc[l] - 1) / maxc[l];
        const long long cost = waves * ((a.V + cs - 1) / cs + 8192LL);
        if (best_l < 0 || cost < best_cost) {
            best_l = l;
            best_cost = cost;
        }
    }
    if (best_l < 0) return cudaErrorInvalidConfiguration;
    const int cs = 1 << best_l;
    const int nclusters = a.rows < maxc[best_l] ? a.rows : maxc[best_l];
    TopkParams p{a.logits, a.rows, a.V, a.K, cs, a.ids, a.vals};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(nclusters * cs), 1, 1);
    cfg.blockDim = dim3(async ? kAThreads : kThreads, 1, 1);
    cfg.dynamicSmemBytes = async ? kASmem : kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cs > 1 ? 1 : 0;
    if (async)
        return a.bf16 ? cudaLaunchKernelEx(&cfg, topk_async_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, topk_async_kernel<false>, p);
    return a.bf16 ? cudaLaunchKernelEx(&cfg, topk_kernel<true>, p)
                  : cudaLaunchKernelEx(&cfg, topk_kernel<false>, p);
}

}  // namespace

cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream) { return launch_any(a, stream); }

cudaError_t take_topk_faults(unsigned* flags) {
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_topk_fault, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_topk_fault, &zero, sizeof(zero));
    *flags = v;
    return e;
}

}  // namespace df2

extern "C" int dflash2_trace_read_topk(uint64_t* host, int bytes, int clear) {
#ifdef DF2_TRACE
    if (host == nullptr || bytes < 0 || (size_t)bytes > sizeof(df2::g_trace_topk))
        return DF2_ERR_INVALID_ARG;
    if (cudaMemcpyFromSymbol(host, df2::g_trace_topk, (size_t)bytes) != cudaSuccess)
        return DF2_ERR_CUDA;
    if (clear) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, df2::g_trace_topk) != cudaSuccess ||
            cudaMemset(a, 0, sizeof(df2::g_trace_topk)) != cudaSuccess)
            return DF2_ERR_CUDA;
    }
    return DF2_OK;
#else
    (void)host;
    (void)bytes;
    (void)clear;
    return DF2_ERR_UNSUPPORTED;
#endif
}
