// Grouped dynamic depthwise causal convolution (ggml-org/llama.cpp PR #27342,
// "spec : add DFlash2 support (local convolution + candidate selector)",
// Overview, first formula):
//   out[s,i,c] = sum_{t<T} (base[t,c] + delta[s,i,t,g(c)]) * xh[s,i-t,c]
// xh reads the (T-1)-row history window for positions before the block.
//
// Design (HBM-streaming, one pass):
//  - a thread owns 8 consecutive channels (one 16-byte bf16 vector) of L
//    consecutive positions; a warp covers 256 contiguous channels, so every
//    row load and store is a fully coalesced 512-byte transaction;
//  - the thread issues all T-1+L row loads of its window (halo included) up
//    front, which keeps ~(T-1+L)*16 bytes per thread in flight;
//  - the block stages the delta taps of its L positions and of the channel
//    groups it spans into shared memory as fp32 [l][g][t], so each thread
//    reads its group's T taps as broadcast vector loads;
//  - the static taps base[t, c..c+7] live in registers for the whole tile;
//  - the arithmetic is fp32, two channels per packed FFMA2 instruction.
#include <cuda_bf16.h>

#include <algorithm>

#include "dflash2.h"
#include "common.cuh"
#include "ptx.cuh"

namespace df2 {
namespace {

struct DynParams {
    const void* x;
    const void* hist;
    const void* base;
    const void* delta;
    void* out;
    int S, n, C, G, cg;
    int n_cblk, n_ptile, ng_max;
};

template <typename TIn>
struct Row8;
template <>
struct Row8<__nv_bfloat16> {
    uint4 v;
};
template <>
struct Row8<float> {
    uint4 a, b;
};

__device__ __forceinline__ void load_row(Row8<__nv_bfloat16>& r, const __nv_bfloat16* p) {
    r.v = ldg_nc_v4(p);
}
__device__ __forceinline__ void load_row(Row8<float>& r, const float* p) {
    r.a = ldg_nc_v4(p);
    r.b = ldg_nc_v4(p + 4);
}
__device__ __forceinline__ void zero_row(Row8<__nv_bfloat16>& r) { r.v = make_uint4(0, 0, 0, 0); }
__device__ __forceinline__ void zero_row(Row8<float>& r) {
    r.a = make_uint4(0, 0, 0, 0);
    r.b = r.a;
}

// bf16 -> fp32 is exact: a bf16 is the upper half of an fp32 bit pattern.
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void to_f2x4(const Row8<__nv_bfloat16>& r, float2 (&f)[4]) {
    f[0] = bf16x2_to_f2(r.v.x);
    f[1] = bf16x2_to_f2(r.v.y);
    f[2] = bf16x2_to_f2(r.v.z);
    f[3] = bf16x2_to_f2(r.v.w);
}
__device__ __forceinline__ void to_f2x4(const Row8<float>& r, float2 (&f)[4]) {
    f[0] = make_float2(__uint_as_float(r.a.x), __uint_as_float(r.a.y));
    f[1] = make_float2(__uint_as_float(r.a.z), __uint_as_float(r.a.w));
    f[2] = make_float2(__uint_as_float(r.b.x), __uint_as_float(r.b.y));
    f[3] = make_float2(__uint_as_float(r.b.z), __uint_as_float(r.b.w));
}

__device__ __forceinline__ float load_scalar(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ float load_scalar(const float* p) { return *p; }

__device__ __forceinline__ void store_row(__nv_bfloat16* p, const float2 (&acc)[4]) {
    uint4 v;
    __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0].x, acc[0].y);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[1].x, acc[1].y);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2].x, acc[2].y);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[3].x, acc[3].y);
    v.x = *reinterpret_cast<uint32_t*>(&b0);
    v.y = *reinterpret_cast<uint32_t*>(&b1);
    v.z = *reinterpret_cast<uint32_t*>(&b2);
    v.w = *reinterpret_cast<uint32_t*>(&b3);
    *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ void store_row(float* p, const float2 (&acc)[4]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
    reinterpret_cast<float4*>(p)[1] = make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
}

template <int T, int L, typename TIn, typename TOut>
__global__ void __launch_bounds__(256) dynconv_kernel(const DynParams p) {
    extern __shared__ float dsm[];  // [L][ng][T] fp32 delta taps of this block
    const TIn* __restrict__ x = static_cast<const TIn*>(p.x);
    const TIn* __restrict__ hist = static_cast<const TIn*>(p.hist);
    const TIn* __restrict__ base = static_cast<const TIn*>(p.base);
    const TIn* __restrict__ delta = static_cast<const TIn*>(p.delta);
    TOut* __restrict__ out = static_cast<TOut*>(p.out);

    const int tid = threadIdx.x;
    const int nthr = blockDim.x;
    int b = blockIdx.x;
    const int cblk = b % p.n_cblk;
    b /= p.n_cblk;
    const int ptile = b % p.n_ptile;
    const int s = b / p.n_ptile;
    const int i0 = ptile * L;
    const int blk_c0 = cblk * nthr * 8;
    const int c0 = blk_c0 + tid * 8;
    const bool active = c0 < p.C;
    const int blk_c1 = min(p.C, blk_c0 + nthr * 8);
    const int g_lo = blk_c0 / p.cg;
    const int ng = (blk_c1 - 1) / p.cg - g_lo + 1;
    const size_t C = (size_t)p.C;

    // 1. window rows i0-(T-1) .. i0+L-1 (rows at or past n feed no output)
    Row8<TIn> win[T - 1 + L];
#pragma unroll
    for (int r = 0; r < T - 1 + L; ++r) {
        const int j = i0 - (T - 1) + r;
        if (active && j < p.n) {
            if (j >= 0)
                load_row(win[r], x + ((size_t)s * p.n + j) * C + c0);
            else if (hist != nullptr)
                load_row(win[r], hist + ((size_t)s * (T - 1) + (T - 1 + j)) * C + c0);
            else
                zero_row(win[r]);
        } else {
            zero_row(win[r]);
        }
    }

    // 2. stage delta[s, i0+l, t, g_lo+gg] -> dsm[(l*ng + gg)*T + t]
    const int nstage = L * T * ng;
    for (int q = tid; q < nstage; q += nthr) {
        const int gg = q % ng;
        const int t = (q / ng) % T;
        const int l = q / (ng * T);
        const int i = i0 + l;
        float v = 0.f;
        if (i < p.n) v = load_scalar(delta + (((size_t)s * p.n + i) * T + t) * p.G + g_lo + gg);
        dsm[(l * ng + gg) * T + t] = v;
    }

    // 3. static taps for this thread's 8 channels
    float2 bw[T][4];
#pragma unroll
    for (int t = 0; t < T; ++t) {
        Row8<TIn> br;
        if (active)
            load_row(br, base + (size_t)t * C + c0);
        else
            zero_row(br);
        to_f2x4(br, bw[t]);
    }
    __syncthreads();
    if (!active) return;

    const int gl = c0 / p.cg - g_lo;
#pragma unroll
    for (int l = 0; l < L; ++l) {
        const int i = i0 + l;
        const float* dl = dsm + (l * ng + gl) * T;
        float2 acc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc[k] = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < T; ++t) {
            const float dv = dl[t];
            const float2 d2 = make_float2(dv, dv);
            float2 xf[4];
            to_f2x4(win[l + T - 1 - t], xf);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 w = __fadd2_rn(bw[t][k], d2);
                acc[k] = __ffma2_rn(w, xf[k], acc[k]);
            }
        }
        if (i < p.n) store_row(out + ((size_t)s * p.n + i) * C + c0, acc);
    }
}

// ------------------------------------------------------------------ pipelined path
//
// Persistent CTAs: `nthr` compute threads (8 channels each, the CTA's channel
// block) plus one producer warp.  Work items are (sequence, 8-position tile,
// channel block), channel block fastest.  For every item one producer lane
// stages into a ring of shared-memory buffers, with non-tensor bulk copies
// completing on an mbarrier:
//   - the T-1 halo rows (from x, or from the history window for the first tile
//     of a sequence) and the tile's rows of x, each the CTA's channel segment;
//   - the tile's whole delta block [l][t][G] (contiguous in HBM): one copy, or,
//     when a (l, t) row of G values is a multiple of 128 bytes (every row then
//     starts in the same shared-memory bank), one copy per position with the
//     positions 16 bytes further apart than in HBM.
// Compute threads consume a buffer (16-byte shared loads, a register sliding
// window of T converted rows, packed FFMA2), store 16-byte outputs straight to
// HBM and release the buffer with an mbarrier arrive.  The ring keeps several
// tiles of loads in flight per SM without holding them in registers.


// Device fault word of the convolution kernels: DF2_FLAG_TIMEOUT when a
// bounded wait gives up.
__device__ unsigned int g_dyn_fault = 0;

struct PipeParams {
    const __nv_bfloat16* x;
    const __nv_bfloat16* hist;
    const __nv_bfloat16* base;
    const __nv_bfloat16* delta;
    void* out;
    int S, n, C, G, cg;
    int nthr, n_cblk, n_ptile;
    int n_items;
    int ng_max;            // groups a channel block can span
    int stages;
    uint32_t row_bytes;    // nthr * 16: one staged row segment
    uint32_t dpos_bytes;   // staged delta bytes from one position to the next
    uint32_t stage_bytes;  // (T-1+PL) rows + PL positions of delta, 128-byte rounded
};


// A thread's staged row segment: NP = 4 packed bf16 pairs (8 channels in 16
// bytes), converted to fp32 pairs.
template <int NP>
__device__ __forceinline__ void load_row_f2(uint32_t addr, float2 (&f)[NP]) {
    static_assert(NP == 4, "8-channel threads");
    const uint4 v = lds_v4(addr);
    f[0] = bf16x2_to_f2(v.x);
    f[1] = bf16x2_to_f2(v.y);
    f[2] = bf16x2_to_f2(v.z);
    f[3] = bf16x2_to_f2(v.w);
}

template <int NP>
__device__ __forceinline__ void load_base_f2(const __nv_bfloat16* p, bool active, float2 (&f)[NP]) {
    static_assert(NP == 4, "8-channel threads");
    const uint4 v = active ? ldg_nc_v4(p) : make_uint4(0, 0, 0, 0);
    f[0] = bf16x2_to_f2(v.x);
    f[1] = bf16x2_to_f2(v.y);
    f[2] = bf16x2_to_f2(v.z);
    f[3] = bf16x2_to_f2(v.w);
}

__device__ __forceinline__ void store_pairs(__nv_bfloat16* p, const float2 (&acc)[4]) {
    store_row(p, acc);
}
__device__ __forceinline__ void store_pairs(float* p, const float2 (&acc)[4]) { store_row(p, acc); }

// One output position: acc = sum_t (base_t + delta_t) * x_{i-t}; xw[t] holds
// x_{i-t}; dtl[t] is delta_t of this thread's group (fp32, contiguous).
// Tuning switches of the pipelined kernel, chosen by measurement on GB300
// (long streams and the 256 x 16 batch, T = 4 and T = 8):
//   kSplitTaps:  for T <= 4, even and odd taps accumulate separately (two FMA
//                chains; 3 % faster at T = 4, slower at T = 8);
//   kLanesOverGroups: the delta transpose maps lanes to groups (contiguous
//                reads; measured slower, so off).
constexpr bool kSplitTaps = true;
constexpr bool kLanesOverGroups = false;

// Even and odd taps may accumulate separately (two independent FMA chains per
// channel pair), then add.
template <int T, int NP>
__device__ __forceinline__ void conv_point(const float2 (&bw)[T][NP], const float2 (&xw)[T][NP],
                                           const float* dtl, float2 (&acc)[NP]) {
    float2 odd[NP];
#pragma unroll
    for (int q = 0; q < NP; ++q) {
        acc[q] = make_float2(0.f, 0.f);
        odd[q] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const float dv = dtl[t];
        const float2 d2 = make_float2(dv, dv);
#pragma unroll
        for (int q = 0; q < NP; ++q) {
            if (kSplitTaps && T <= 4 && (t & 1))
                odd[q] = __ffma2_rn(__fadd2_rn(bw[t][q], d2), xw[t][q], odd[q]);
            else
                acc[q] = __ffma2_rn(__fadd2_rn(bw[t][q], d2), xw[t][q], acc[q]);
        }
    }
    if constexpr (kSplitTaps && T > 1 && T <= 4) {
#pragma unroll
        for (int q = 0; q < NP; ++q) acc[q] = __fadd2_rn(acc[q], odd[q]);
    }
}

// A full tile of NL positions from a staged buffer: rows 0..T-2 are the halo
// (all zero for the first tile of a block that has no history), row T-1+l
// holds position l; dt[l*T + t] is delta of this thread's group (fp32).
// Straight-line code: the window shifts are renames, tap offsets immediates.
template <int T, int NP, typename TOut, int NL>
__device__ __forceinline__ void conv_tile(uint32_t sb, uint32_t row_bytes, const float* dt,
                                          bool zero_halo, const float2 (&bw)[T][NP], TOut* op,
                                          int C) {
    float2 xw[T][NP];
#pragma unroll
    for (int k = 0; k < T; ++k)
#pragma unroll
        for (int q = 0; q < NP; ++q) xw[k][q] = make_float2(0.f, 0.f);
    if (!zero_halo) {
#pragma unroll
        for (int r = 0; r < T - 1; ++r) load_row_f2<NP>(sb + (uint32_t)r * row_bytes, xw[T - 2 - r]);
    }
#pragma unroll
    for (int l = 0; l < NL; ++l) {
#pragma unroll
        for (int k = T - 1; k > 0; --k)
#pragma unroll
            for (int q = 0; q < NP; ++q) xw[k][q] = xw[k - 1][q];
        load_row_f2<NP>(sb + (uint32_t)(T - 1 + l) * row_bytes, xw[0]);
        float2 acc[NP];
        conv_point<T, NP>(bw, xw, dt + l * T, acc);
        store_pairs(op + (size_t)l * C, acc);
    }
}

// The last, partial tile of a sequence (nl < PL positions).
template <int T, int NP, typename TOut>
__device__ __forceinline__ void conv_tile_ragged(uint32_t sb, uint32_t row_bytes, const float* dt,
                                                 bool zero_halo, const float2 (&bw)[T][NP],
                                                 TOut* op, int C, int nl) {
    float2 xw[T][NP];
#pragma unroll
    for (int k = 0; k < T; ++k)
#pragma unroll
        for (int q = 0; q < NP; ++q) xw[k][q] = make_float2(0.f, 0.f);
    if (!zero_halo) {
#pragma unroll
        for (int r = 0; r < T - 1; ++r) load_row_f2<NP>(sb + (uint32_t)r * row_bytes, xw[T - 2 - r]);
    }
    for (int l = 0; l < nl; ++l) {
#pragma unroll
        for (int k = T - 1; k > 0; --k)
#pragma unroll
            for (int q = 0; q < NP; ++q) xw[k][q] = xw[k - 1][q];
        load_row_f2<NP>(sb + (uint32_t)(T - 1 + l) * row_bytes, xw[0]);
        float2 acc[NP];
        conv_point<T, NP>(bw, xw, dt + l * T, acc);
        store_pairs(op + (size_t)l * C, acc);
    }
}

// Register budget: 4 CTAs of 160 threads per SM up to T = 4; 2 for longer
// filters, whose window and taps need about 170 registers (8 channels per
// thread either way: on the 8 x 32768 stream at T = 8 that measured 1.287 ms
// against 1.297 ms for twice the threads with 4 channels each).
template <int T, int PL, int NP, typename TOut>
__global__ void __launch_bounds__(160, T <= 4 ? 4 : 2)
    dynconv_pipe_kernel(const PipeParams p) {
    constexpr int VEC = 2 * NP;  // channels per compute thread
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x;
    const int nthr = p.nthr;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)p.stages * p.stage_bytes);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + p.stages);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * p.stages);
    const uint32_t smem0 = smem_u32(smem);
    const int TG = T * p.G;

    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, (uint32_t)nthr);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Launched as a programmatic dependent: everything above overlapped the
    // previous kernel; no input is read before it has completed.
    griddep_wait();
    griddep_launch_dependents();

    // Each CTA keeps one channel block (its base taps stay in registers) and
    // walks the (sequence, tile) pairs pt = blockIdx.x / n_cblk + k * step.
    const int cblk = blockIdx.x % p.n_cblk;
    const int step = gridDim.x / p.n_cblk;
    const int n_pt = p.S * p.n_ptile;
    const int c0 = cblk * nthr * VEC;

    if (tid >= nthr) {
        // ---------------- producer (one lane)
        if (tid != nthr) return;
        const uint32_t seg = (uint32_t)min(nthr * VEC, p.C - c0) * 2u;
        int it = 0;
        for (int pt = blockIdx.x / p.n_cblk; pt < n_pt; pt += step, ++it) {
            const int st = it % p.stages;
            const uint32_t ph = (uint32_t)(it / p.stages) & 1u;
            if (*abort_flag) break;
            if (!mbar_wait_bounded(empty0 + 8 * st, ph ^ 1u, kWaitNs)) {
                *abort_flag = 1;
                atomicOr(&g_dyn_fault, (unsigned)DF2_FLAG_TIMEOUT);
                break;
            }
            const int s = pt / p.n_ptile;
            const int i0 = (pt - s * p.n_ptile) * PL;
            const int nl = min(PL, p.n - i0);
            // halo row r holds position j = i0-(T-1)+r: from x when j >= 0, else from
            // the history window (or nothing: zeros when there is no history)
            const int nneg = max(0, (T - 1) - i0);  // halo rows before the block
            const int nhalo = p.hist == nullptr ? (T - 1) - nneg : T - 1;
            const uint32_t fb = full0 + 8 * st;
            const uint32_t bytes = (uint32_t)(nhalo + nl) * seg + (uint32_t)(nl * TG) * 2u;
            mbar_arrive_expect_tx(fb, bytes);
            const uint32_t dst = smem0 + (uint32_t)st * p.stage_bytes;
            for (int r = 0; r < T - 1; ++r) {
                const int j = i0 - (T - 1) + r;
                const __nv_bfloat16* src;
                if (j >= 0)
                    src = p.x + ((size_t)s * p.n + j) * p.C + c0;
                else if (p.hist != nullptr)
                    src = p.hist + ((size_t)s * (T - 1) + (T - 1 + j)) * p.C + c0;
                else
                    continue;
                bulk_g2s(dst + (uint32_t)r * p.row_bytes, src, seg, fb);
            }
            for (int l = 0; l < nl; ++l)
                bulk_g2s(dst + (uint32_t)(T - 1 + l) * p.row_bytes,
                         p.x + ((size_t)s * p.n + i0 + l) * p.C + c0, seg, fb);
            const uint32_t ddst = dst + (uint32_t)(T - 1 + PL) * p.row_bytes;
            const __nv_bfloat16* dsrc = p.delta + ((size_t)s * p.n + i0) * TG;
            if (p.dpos_bytes == (uint32_t)TG * 2u)
                bulk_g2s(ddst, dsrc, (uint32_t)(nl * TG) * 2u, fb);
            else
                for (int l = 0; l < nl; ++l)
                    bulk_g2s(ddst + (uint32_t)l * p.dpos_bytes, dsrc + (size_t)l * TG,
                             (uint32_t)TG * 2u, fb);
        }
        return;
    }

    // ---------------- compute threads
    const int c = c0 + tid * VEC;
    const bool active = c < p.C;
    const int c_end = min(c0 + nthr * VEC, p.C);
    const int g_lo = c0 / p.cg;
    const int ng = (c_end - 1) / p.cg - g_lo + 1;  // groups of this channel block
    const int gl = active ? c / p.cg - g_lo : 0;
    float* dt0 = reinterpret_cast<float*>(smem + (size_t)p.stages * p.stage_bytes + 256);
    float2 bw[T][NP];
#pragma unroll
    for (int t = 0; t < T; ++t) load_base_f2<NP>(p.base + (size_t)t * p.C + c, active, bw[t]);
    static_assert(PL >= T - 1, "a tile's halo must lie entirely before or inside the block");
    int it = 0;
    for (int pt = blockIdx.x / p.n_cblk; pt < n_pt; pt += step, ++it) {
        const int st = it % p.stages;
        const uint32_t ph = (uint32_t)(it / p.stages) & 1u;
        const int s = pt / p.n_ptile;
        const int i0 = (pt - s * p.n_ptile) * PL;
        const int nl = min(PL, p.n - i0);
        if (!*abort_flag && !mbar_wait_bounded(full0 + 8 * st, ph, kWaitNs)) {
            *abort_flag = 1;
            atomicOr(&g_dyn_fault, (unsigned)DF2_FLAG_TIMEOUT);
        }
        // delta of this block's groups -> fp32 [group][l][t], groups DSTR floats
        // apart (padded so the groups a warp reads fall in different banks),
        // double-buffered by item
        constexpr int DSTR = PL * T + 4;
        float* dt = dt0 + (size_t)(it & 1) * p.ng_max * DSTR;
        {
            const __nv_bfloat16* dsrc = reinterpret_cast<const __nv_bfloat16*>(
                smem + (size_t)st * p.stage_bytes + (size_t)(T - 1 + PL) * p.row_bytes);
            if (p.G % 8 == 0) {
                // 16-byte reads of 8 consecutive groups of one (l, t) row of the
                // staged [l][t][G] block (G % 8 == 0 keeps them aligned), lanes over
                // (l, t) so each of the 8 scattered stores hits nearby words: t
                // fastest, or l fastest when the positions are staggered (rows of
                // one position share banks, rows of 8 positions do not)
                const int g8_lo = g_lo & ~7;
                const int n8 = (g_lo + ng - g8_lo + 7) >> 3;
                const uint32_t src0 = smem_u32(dsrc);
                const bool stagger = p.dpos_bytes != (uint32_t)TG * 2u;
                for (int q = tid; q < PL * T * n8; q += nthr) {
                    const int r = q % (PL * T);
                    const int l = stagger ? r % PL : r / T;
                    const int t = stagger ? r / PL : r % T;
                    const int lt = l * T + t;
                    const int gb = g8_lo + (q / (PL * T)) * 8;
                    const uint4 raw = l < nl ? lds_v4(src0 + (uint32_t)l * p.dpos_bytes +
                                                      (uint32_t)(t * p.G + gb) * 2u)
                                             : make_uint4(0, 0, 0, 0);
                    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int gg = gb + k - g_lo;
                        if (gg >= 0 && gg < ng)
                            dt[gg * DSTR + lt] = __uint_as_float((k & 1) ? (w[k >> 1] & 0xFFFF0000u)
                                                                         : (w[k >> 1] << 16));
                    }
                }
            } else if constexpr (kLanesOverGroups) {
                // lanes walk groups (contiguous in the staged [l][t][G] block),
                // warps walk (l, t)
                const int lane = tid & 31;
                for (int lt = tid >> 5; lt < PL * T; lt += nthr >> 5) {
                    const bool in = (lt / T) < nl;
                    for (int gg = lane; gg < ng; gg += 32)
                        dt[gg * DSTR + lt] =
                            in ? __bfloat162float(dsrc[lt * p.G + g_lo + gg]) : 0.f;
                }
            } else {
                for (int q = tid; q < ng * PL * T; q += nthr) {
                    const int lt = q % (PL * T);
                    const int gg = q / (PL * T);
                    dt[gg * DSTR + lt] =
                        (lt / T) < nl ? __bfloat162float(dsrc[lt * p.G + g_lo + gg]) : 0.f;
                }
            }
        }
        named_bar_sync(1, (uint32_t)nthr);
        if (active && !*abort_flag) {
            const uint32_t sb = smem0 + (uint32_t)st * p.stage_bytes + (uint32_t)tid * (2u * VEC);
            const float* dtg = dt + (size_t)gl * DSTR;
            const bool zero_halo = (i0 == 0 && p.hist == nullptr);
            TOut* op = static_cast<TOut*>(p.out) + ((size_t)s * p.n + i0) * p.C + c;
            if (nl == PL)
                conv_tile<T, NP, TOut, PL>(sb, p.row_bytes, dtg, zero_halo, bw, op, p.C);
            else
                conv_tile_ragged<T, NP, TOut>(sb, p.row_bytes, dtg, zero_halo, bw, op, p.C, nl);
        }
        mbar_arrive(empty0 + 8 * st);
    }
    // On an abandoned pipeline, give copies still in flight a bounded time to
    // land before the CTA's shared memory is released.
    if (tid == 0 && *abort_flag) {
        for (int i = 0; i < p.stages; ++i) mbar_wait_bounded(full0 + 8 * i, 0, kWaitNs / 4);
    }
}

template <int T, int PL, typename TOut>
cudaError_t launch_pipe_t(PipeParams p, cudaStream_t stream) {
    constexpr int NP = 4;      // 8 channels per thread
    p.nthr = p.nthr * 4 / NP;  // nthr arrives as the 8-channel thread count
    p.row_bytes = (uint32_t)p.nthr * (4u * NP);
    auto kern = dynconv_pipe_kernel<T, PL, NP, TOut>;
    p.ng_max = (p.nthr * 2 * NP - 1) / p.cg + 2;
    // stages, then the mbarriers (<= 256 bytes), then two transposed delta buffers
    const size_t smem = (size_t)p.stages * p.stage_bytes + 256 +
                        2 * (size_t)p.ng_max * (PL * T + 4) * sizeof(float);
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, p.nthr + 32, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    // a multiple of n_cblk: every CTA keeps one channel block
    const long long n_pt = (long long)p.S * p.n_ptile;
    const long long per_cblk = std::max<long long>(
        1, std::min<long long>((long long)sms * per_sm / p.n_cblk, n_pt));
    const long long grid = per_cblk * p.n_cblk;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)(p.nthr + 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <int PL, typename TOut>
cudaError_t launch_pipe(const PipeParams& p, int T, cudaStream_t stream) {
    switch (T) {
#define DF2_CASE(TT) \
    case TT:         \
        return launch_pipe_t<TT, PL, TOut>(p, stream);
        DF2_CASE(1) DF2_CASE(2) DF2_CASE(3) DF2_CASE(4) DF2_CASE(5) DF2_CASE(6) DF2_CASE(7)
        DF2_CASE(8)
#undef DF2_CASE
        default:
            return cudaErrorInvalidValue;
    }
}

template <typename TIn>
constexpr int tile_len(int T) {
    return sizeof(TIn) == 4 ? (T <= 8 ? 4 : 2) : (T <= 8 ? 8 : (T <= 12 ? 4 : 2));
}

template <int T, typename TIn, typename TOut>
cudaError_t launch_t(DynParams p, int nthr, cudaStream_t stream) {
    constexpr int L = tile_len<TIn>(T);
    p.n_ptile = (p.n + L - 1) / L;
    const size_t smem = (size_t)L * p.ng_max * T * sizeof(float);
    auto kern = dynconv_kernel<T, L, TIn, TOut>;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const long long blocks = (long long)p.S * p.n_ptile * p.n_cblk;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)blocks, nthr, smem, stream>>>(p);
    return cudaGetLastError();
}

template <typename TIn, typename TOut>
cudaError_t launch_dtype(const DynParams& p, int T, int nthr, cudaStream_t stream) {
    switch (T) {
#define DF2_CASE(TT) \
    case TT:         \
        return launch_t<TT, TIn, TOut>(p, nthr, stream);
        DF2_CASE(1) DF2_CASE(2) DF2_CASE(3) DF2_CASE(4) DF2_CASE(5) DF2_CASE(6) DF2_CASE(7)
        DF2_CASE(8) DF2_CASE(9) DF2_CASE(10) DF2_CASE(11) DF2_CASE(12) DF2_CASE(13)
        DF2_CASE(14) DF2_CASE(15) DF2_CASE(16)
#undef DF2_CASE
        default:
            return cudaErrorInvalidValue;
    }
}

// Threads per block: a warp multiple that divides C/8 when one exists, so no
// block is left partly idle.
int pick_threads(int C) {
    const int nv = C / 8;
    const int cand[] = {128, 160, 192, 224, 96, 256, 64};
    for (int t : cand)
        if (nv % t == 0) return t;
    return nv < 128 ? ((nv + 31) / 32) * 32 : 128;
}

}  // namespace

cudaError_t take_dynconv_faults(unsigned* flags) {
    unsigned v = 0;
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dyn_fault, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_dyn_fault, &zero, sizeof(zero));
    *flags = v;
    return e;
}

cudaError_t launch_dynconv(const DynconvArgs& a, cudaStream_t stream) {
    DynParams p{};
    p.x = a.x;
    p.hist = a.hist;
    p.base = a.base;
    p.delta = a.delta;
    p.out = a.out;
    p.S = a.S;
    p.n = a.n;
    p.C = a.C;
    p.G = a.G;
    p.cg = a.C / a.G;
    const int nthr = pick_threads(a.C);
    p.n_cblk = (a.C / 8 + nthr - 1) / nthr;
    // groups a window of nthr*8 consecutive channels can touch
    p.ng_max = (nthr * 8 - 1) / p.cg + 2;
    if (p.ng_max > a.G) p.ng_max = a.G;
    if (a.in_bf16 && a.T <= 8 && (a.T * a.G) % 8 == 0 && nthr <= 128) {
        PipeParams q{};
        q.x = static_cast<const __nv_bfloat16*>(a.x);
        q.hist = static_cast<const __nv_bfloat16*>(a.hist);
        q.base = static_cast<const __nv_bfloat16*>(a.base);
        q.delta = static_cast<const __nv_bfloat16*>(a.delta);
        q.out = a.out;
        q.S = a.S;
        q.n = a.n;
        q.C = a.C;
        q.G = a.G;
        q.cg = p.cg;
        q.nthr = nthr;
        q.n_cblk = p.n_cblk;
        // Tiles of 8 positions (>= T-1, so a tile's halo is either all history
        // or all x).  Shorter tiles balance the last round better but cost more
        // in halo copies and conversions than they gain (measured).
        constexpr int PLsel = 8;
        q.n_ptile = (a.n + PLsel - 1) / PLsel;
        const long long items = (long long)a.S * q.n_ptile * q.n_cblk;
        if (items <= 0x7FFFFFFFLL) {
            q.n_items = (int)items;
            q.row_bytes = (uint32_t)nthr * 16u;
            // rows of G bf16 that are whole 128-byte lines would all start in
            // one bank: stagger the staged positions by 16 bytes
            q.dpos_bytes = (uint32_t)(a.T * a.G) * 2u + ((a.G * 2) % 128 == 0 ? 16u : 0u);
            const uint32_t raw = (uint32_t)(a.T - 1 + PLsel) * q.row_bytes +
                                 (uint32_t)PLsel * q.dpos_bytes;
            q.stage_bytes = (raw + 127u) & ~127u;
            q.stages = 2;
            return a.out_bf16 ? launch_pipe<PLsel, __nv_bfloat16>(q, a.T, stream)
                              : launch_pipe<PLsel, float>(q, a.T, stream);
        }
    }
    if (a.in_bf16 && a.out_bf16)
        return launch_dtype<__nv_bfloat16, __nv_bfloat16>(p, a.T, nthr, stream);
    if (a.in_bf16)
        return launch_dtype<__nv_bfloat16, float>(p, a.T, nthr, stream);
    return launch_dtype<float, float>(p, a.T, nthr, stream);
}

}  // namespace df2
