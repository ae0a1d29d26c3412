// The DFlash2 convolution with its dynamic taps predicted from its own input,
// in one kernel (ggml-org/llama.cpp PR #27342, "spec : add DFlash2 support
// (local convolution + candidate selector)", Overview: the per-position tap
// offsets are "predicted from the input"; the weight tensor is *_conv_proj):
//
//   delta[p, t*G+g] = bf16( sum_c Wc[t*G+g, c] * x[p, c] )
//   out[p, c]       = sum_t (base[t,c] + delta[p, t, g(c)]) * x[p-t, c]
//
// with x[p-t] taken from the (T-1)-row history window (or zero) where p-t falls
// before the start of p's sequence.  delta is rounded to bf16 between the two
// steps, as when it is stored by the predictor and read back by the conv, so
// the result matches that pair; it never leaves the chip.
//
// Work unit: a tile of 128 consecutive positions (rows of x flattened over
// sequences), handled by one thread-block cluster of `split` CTAs, each owning
// a contiguous slice of the channels (whole 64-channel blocks):
//   1. delta, split-K over the cluster: every CTA streams its channel slice of
//      the tile's x rows and of Wc through a TMA ring (128-byte swizzle,
//      K-major) into tcgen05.mma (M = 128 positions, N = T*G rounded up to 16,
//      fp32 accumulation in tensor memory); two producer threads issue the
//      loads of the even and the odd k-blocks and two threads their MMAs, into
//      two accumulators summed when drained (one thread issuing every load or
//      every MMA is slower per k-block than the ring);
//   2. the partial tiles go to shared memory, column-major (tcgen05.ld by all
//      warps); after a cluster barrier each CTA sums, in rank order
//      (deterministic), the columns its own channel slice needs -- taps t*G+g
//      for the groups g its channels fall in -- with 16-byte loads of the other
//      CTAs' partials through distributed shared memory, and keeps them as bf16;
//   3. each CTA convolves its channel slice over the tile's 128 positions, in
//      pieces of at most 8 positions of one sequence; every thread stages the
//      window rows of its next items into its own slots of the freed TMA ring
//      with 16-byte cp.async copies (zero-fill for a missing history) and
//      slides a window of converted rows over each piece.  x is read again,
//      but the tile's rows were just streamed through L2 by the TMA loads of
//      step 1, so this second read costs L2 bandwidth, not HBM.
// HBM traffic is therefore x once, Wc (shared by every tile, L2-resident) and
// the output: the delta round trip and the second HBM pass over x of the
// unfused predictor + conv pair are gone.  The single wave of CTAs runs step 1
// (HBM-bound) and step 3 (FP32-issue-bound) one after the other, so on a
// one-wave problem the time is close to that of the pair; what it saves is
// bytes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "dflash2.h"
#include "ptx.cuh"

namespace df2 {

// Device fault word of the fused kernel: DF2_FLAG_TIMEOUT when a bounded wait
// gives up.
__device__ unsigned int g_fused_fault = 0;

namespace {

constexpr int kBM = 128;                  // positions per tile (MMA M)
constexpr int kBK = 64;                   // channels per k-block (one 128-byte swizzle row)
// Threads per CTA: 512 (16 warps) for T <= 4, where the conv phase's
// registers allow it, else 256; more warps hide the conv's dependent FMAs.
__host__ __device__ constexpr int threads_for(int T) { return T <= 4 ? 512 : 256; }
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr int kPL = 8;                    // positions per conv strip
constexpr int kMaxStages = 6;

struct FusedParams {
    const __nv_bfloat16* x;     // [P, C]
    const __nv_bfloat16* hist;  // [S, T-1, C] or nullptr (zeros before each sequence)
    const __nv_bfloat16* base;  // [T, C]
    void* out;                  // [P, C] bf16 or fp32
    int P, n, C, G, TG, NP, cg;
    int kblocks, split, stages;
    uint32_t stage_bytes;       // kABytes + NP * 128
    uint32_t ring_bytes;        // TMA ring, reused for the partial tile
    uint32_t ds_bytes;          // bf16 delta of the CTA's groups, largest over the ranks
    uint32_t tmem_cols;         // power of two >= max(NP, 32)
    int cdepth;                 // conv pieces in flight per thread (1..4)
};

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Waits until at most `pending` of this thread's committed groups are in flight.
__device__ __forceinline__ void cp_wait_pending(int pending) {
    switch (pending) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    }
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void row_to_f2(uint4 v, float2 (&f)[4]) {
    f[0] = bf2_to_f2(v.x);
    f[1] = bf2_to_f2(v.y);
    f[2] = bf2_to_f2(v.z);
    f[3] = bf2_to_f2(v.w);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float2 (&a)[4]) {
    uint4 v;
    __nv_bfloat162 b0 = __floats2bfloat162_rn(a[0].x, a[0].y);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(a[1].x, a[1].y);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(a[2].x, a[2].y);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(a[3].x, a[3].y);
    v.x = *reinterpret_cast<uint32_t*>(&b0);
    v.y = *reinterpret_cast<uint32_t*>(&b1);
    v.z = *reinterpret_cast<uint32_t*>(&b2);
    v.w = *reinterpret_cast<uint32_t*>(&b3);
    *reinterpret_cast<uint4*>(p) = v;
}
__device__ __forceinline__ void store8(float* p, const float2 (&a)[4]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(a[0].x, a[0].y, a[1].x, a[1].y);
    reinterpret_cast<float4*>(p)[1] = make_float4(a[2].x, a[2].y, a[3].x, a[3].y);
}

// One output position from its T taps: xw[t] holds x[p-t] (8 channels as 4
// pairs), dt[t] is delta[p, t, g] of these channels' group.  Even and odd taps
// accumulate in separate chains for T <= 4 (as the unfused conv does).
template <int T>
__device__ __forceinline__ void conv8(const float2 (&bw)[T][4], const float2 (&xw)[T][4],
                                      const float (&dt)[T], float2 (&acc)[4]) {
    float2 odd[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        acc[q] = make_float2(0.f, 0.f);
        odd[q] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < T; ++t) {
        const float2 d2 = make_float2(dt[t], dt[t]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (T <= 4 && (t & 1))
                odd[q] = __ffma2_rn(__fadd2_rn(bw[t][q], d2), xw[t][q], odd[q]);
            else
                acc[q] = __ffma2_rn(__fadd2_rn(bw[t][q], d2), xw[t][q], acc[q]);
        }
    }
    if constexpr (T > 1 && T <= 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = __fadd2_rn(acc[q], odd[q]);
    }
}

template <int T, typename TOut, int NT = threads_for(T)>
__global__ void __launch_bounds__(NT, 1)
    dynconv_pred_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                        const FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* ring = smem;
    uint16_t* ds = reinterpret_cast<uint16_t*>(smem + p.ring_bytes);  // [T*ngl][128] bf16 bits
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const int m_tile = blockIdx.x / p.split;
    const int kb0 = (int)((long long)rank * p.kblocks / p.split);
    const int kb1 = (int)((long long)(rank + 1) * p.kblocks / p.split);
    const int nkb = kb1 - kb0;
    const int c_lo = kb0 * kBK;
    const int c_hi = min(kb1 * kBK, p.C);
    const int g_lo = c_lo / p.cg;
    const int ngl = (c_hi - 1) / p.cg - g_lo + 1;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.ring_bytes + p.ds_bytes);
    // barrier block: full[kMaxStages], empty[kMaxStages], accum; then the TMEM
    // slot, the piece count and the piece table of the conv phase
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 1);
    int* n_pieces = reinterpret_cast<int*>(tmem_slot + 1);
    uint8_t* piece_start = reinterpret_cast<uint8_t*>(tmem_slot + 4);  // [kBM + 1]
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + kMaxStages);
    const uint32_t accum = smem_u32(bars + 2 * kMaxStages);

    if (tid == 0) {
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum, 2);  // one commit from each MMA issuer
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    // Launched as a programmatic dependent: the set-up above overlapped the
    // previous kernel; nothing is read or written before it has completed.
    griddep_wait();
    griddep_launch_dependents();

    // ---------------------------------------------------------------- 1. delta on the tensor cores
    // producers: warp 0 the even k-blocks, warp 2 the odd ones; issuers: warp 1 the
    // even ones into columns [0, NP), warp 3 the odd ones into [NP, 2 NP).  The
    // ring stage and its phase advance by two k-blocks per step.
    if ((warp == 0 || warp == 2) && lane == 0) {
        int s = warp >> 1;  // stages >= 2
        uint32_t ph = 0;
        for (int it = warp >> 1; it < nkb; it += 2) {
            if (it >= 2) {
                s += 2;
                while (s >= p.stages) {
                    s -= p.stages;
                    ph ^= 1u;
                }
            }
            if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, kWaitNs)) {
                ok = false;
                break;
            }
            const uint32_t fb = full0 + 8 * s;
            mbar_arrive_expect_tx(fb, p.stage_bytes);
            const uint32_t dst = smem_u32(ring + (size_t)s * p.stage_bytes);
            const int kx = (kb0 + it) * kBK;
            tma_load_2d(dst, &tmX, fb, kx, m_tile * kBM);
            tma_load_2d(dst + kABytes, &tmW, fb, kx, 0);
        }
    } else if ((warp == 1 || warp == 3) && lane == 0) {
        const uint32_t idesc = idesc_bf16_f32(kBM, p.NP);
        const int q = warp >> 1;
        const uint32_t dq = tmem + (uint32_t)(q * p.NP);
        int s = q;
        uint32_t ph = 0;
        for (int it = q; it < nkb; it += 2) {
            if (it >= 2) {
                s += 2;
                while (s >= p.stages) {
                    s -= p.stages;
                    ph ^= 1u;
                }
            }
            if (!mbar_wait_bounded(full0 + 8 * s, ph, kWaitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(ring + (size_t)s * p.stage_bytes);
            const uint32_t b0 = a0 + kABytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
                tc_mma_bf16(dq, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k), idesc,
                            (it > q || k > 0) ? 1u : 0u);
            tc_commit(empty0 + 8 * s);
        }
        tc_commit(accum);  // arrives even when this issuer had no k-block
    }
    __syncwarp();

    // ---------------------------------------------------------------- 2. partial tile -> cluster sum
    // The accumulator barrier fires once every MMA (hence every load) is done,
    // so the ring is free to hold the partial tile, column-major [TG][128]:
    // each delta column's 128 positions are contiguous.
    if (!mbar_wait_bounded(accum, 0, kWaitNs)) ok = false;
    tc_fence_after();
    float* red = reinterpret_cast<float*>(ring);
    {
        // warp w reads TMEM lanes 32*(w%4).. (its quadrant), column chunks
        // (w/4)*32, stepping over the warp groups
        const int row = (warp & 3) * 32 + lane;
#pragma unroll 1
        for (int c0 = (warp >> 2) * 32; c0 < p.TG; c0 += (NT / 128) * 32) {
            const uint32_t ta = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)c0;
            uint32_t v[32];
            float f[32];
            tmem_ld_32x32b_x32(ta, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
            if (nkb > 1) {  // plus the odd k-blocks' accumulator
                tmem_ld_32x32b_x32(ta + (uint32_t)p.NP, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] += __uint_as_float(v[j]);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (c0 + j < p.TG) red[(size_t)(c0 + j) * kBM + row] = f[j];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
    cluster_sync();  // every CTA's partial tile is in its shared memory

    {
        // Each task: 4 positions of one needed column (tap t, group g_lo+gl),
        // summed over the cluster's partial tiles in rank order (deterministic)
        // from 16-byte distributed-shared-memory loads; two tasks per round,
        // all their loads issued before the first sum.
        const uint32_t red_s = smem_u32(red);
        uint32_t src_base[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) src_base[r] = r < p.split ? map_cluster(red_s, (uint32_t)r) : 0u;
        const int tot = T * ngl * (kBM / 4);
#pragma unroll 1
        for (int q0 = tid; q0 < tot; q0 += 2 * NT) {
            float4 v[2][8];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q = min(q0 + e * NT, tot - 1);
                const int cj = q / (kBM / 4);
                const int rq = q - cj * (kBM / 4);
                const int t = cj / ngl;
                const int col = t * p.G + g_lo + (cj - t * ngl);
                const uint32_t off = (uint32_t)(col * kBM + 4 * rq) * 4u;
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < p.split) v[e][r] = ld_cluster_f4(src_base[r] + off);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q = q0 + e * NT;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int r = 0; r < 8; ++r)
                    if (r < p.split) {
                        a.x += v[e][r].x;
                        a.y += v[e][r].y;
                        a.z += v[e][r].z;
                        a.w += v[e][r].w;
                    }
                const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
                uint2 w2;
                w2.x = *reinterpret_cast<const uint32_t*>(&lo);
                w2.y = *reinterpret_cast<const uint32_t*>(&hi);
                if (q < tot) *reinterpret_cast<uint2*>(ds + (size_t)q * 4) = w2;
            }
        }
    }
    // The conv phase's pieces: runs of positions of the tile cut at every
    // 8-position strip and at every sequence start.
    if (tid < kBM) {
        const int pos = m_tile * kBM + tid;
        const bool starts = pos < p.P && ((tid % kPL) == 0 || pos % p.n == 0);
        const unsigned bal = __ballot_sync(0xffffffffu, starts);
        const int below = __popc(bal & ((1u << lane) - 1u));
        // warp totals through the piece table's tail bytes (4 warps)
        int* wsum = reinterpret_cast<int*>(piece_start + kBM + 4);
        if (lane == 0) wsum[warp] = __popc(bal);
        named_bar_sync(2, kBM);
        int off = 0;
        for (int w = 0; w < warp; ++w) off += wsum[w];
        if (starts) piece_start[off + below] = (uint8_t)tid;
        if (tid == kBM - 1) {
            const int total = wsum[0] + wsum[1] + wsum[2] + wsum[3];
            *n_pieces = total;
            piece_start[total] = (uint8_t)min(kBM, p.P - m_tile * kBM);
        }
    }
    cluster_sync();  // no CTA reads another's partial tile after this; delta is complete

    // ---------------------------------------------------------------- 3. the conv on this slice
    // Items: (piece, 8-channel vector), vector fastest so a warp reads 512
    // contiguous bytes of a row.  A piece (at most 8 positions of one sequence)
    // is one sliding window of RW = 8 + T - 1 rows: its T-1 halo rows come
    // from x, or from the history window (or zero) before the sequence start.
    // Every thread stages the rows of its next `cdepth` items into its own
    // slots of the (now free) ring with 16-byte cp.async copies, so several
    // items' loads are in flight while it computes one.
    constexpr int RW = kPL + T - 1;
    const int C = p.C, n = p.n;
    const int nvec = (c_hi - c_lo) / 8;
    const int p0 = m_tile * kBM;
    const int items = *n_pieces * nvec;
    const int my_n = tid < items ? (items - tid + NT - 1) / NT : 0;
    const int depth = p.cdepth;
    const uint32_t ring_s = smem_u32(ring);
    TOut* out = static_cast<TOut*>(p.out);
    auto slot_row = [&](int slot, int r) -> uint32_t {
        return ring_s + (uint32_t)(((slot * RW + r) * NT + tid) * 16);
    };
    auto issue = [&](int k) {
        if (k < my_n) {
            const int item = tid + k * NT;
            const int pc = item / nvec;
            const int c = c_lo + (item - pc * nvec) * 8;
            const int ps = p0 + piece_start[pc];
            const int nl = piece_start[pc + 1] - piece_start[pc];
            const int sq = ps / n;
            const int ia = ps - sq * n;
            const int slot = k % depth;
#pragma unroll
            for (int r = 0; r < RW; ++r) {
                if (r < nl + T - 1) {
                    const int ir = ia + r - (T - 1);  // in-sequence index of window row r
                    const void* src = p.x;
                    uint32_t bytes = 0;
                    if (ir >= 0) {
                        src = p.x + ((size_t)sq * n + ir) * C + c;
                        bytes = 16;
                    } else if (p.hist != nullptr) {
                        src = p.hist + ((size_t)sq * (T - 1) + (T - 1 + ir)) * C + c;
                        bytes = 16;
                    }
                    cp16_zfill(slot_row(slot, r), src, bytes);
                }
            }
        }
        cp_commit();  // one group per item slot, empty or not: uniform counting
    };
    for (int k = 0; k < depth; ++k) issue(k);
#pragma unroll 1
    for (int k = 0; k < my_n; ++k) {
        cp_wait_pending(depth - 1);  // this thread's copies of item k have landed
        const int item = tid + k * NT;
        const int pc = item / nvec;
        const int c = c_lo + (item - pc * nvec) * 8;
        const int row0 = piece_start[pc];
        const int nl = piece_start[pc + 1] - row0;
        const int gl = c / p.cg - g_lo;
        const int slot = k % depth;
        float2 bw[T][4];
#pragma unroll
        for (int t = 0; t < T; ++t) row_to_f2(ldg_nc_v4(p.base + (size_t)t * C + c), bw[t]);
        // xw[t] = x[position - t], converted once per row and slid along: each
        // position first shifts the window by one tap, then loads its own row
        // into xw[0]; before position 0, xw[t] holds window row T-2-t.
        float2 xw[T][4];
#pragma unroll
        for (int t = 0; t < T - 1; ++t) row_to_f2(lds_v4(slot_row(slot, T - 2 - t)), xw[t]);
        const uint16_t* dsr = ds + (size_t)gl * kBM + row0;
        if (nl == kPL && (row0 & (kPL - 1)) == 0) {
            // a full, aligned piece (every piece when n is a multiple of 8): no
            // per-position guard, and each tap's delta for two positions in one
            // 4-byte load
            const uint32_t* dsw = reinterpret_cast<const uint32_t*>(dsr);
            const int wstride = ngl * kBM / 2;  // tap t+1's column, in 4-byte words
            uint32_t dw[T];
#pragma unroll
            for (int l = 0; l < kPL; ++l) {
                if ((l & 1) == 0) {
#pragma unroll
                    for (int t = 0; t < T; ++t) dw[t] = dsw[t * wstride + (l >> 1)];
                }
#pragma unroll
                for (int t = T - 1; t > 0; --t)
#pragma unroll
                    for (int q = 0; q < 4; ++q) xw[t][q] = xw[t - 1][q];
                row_to_f2(lds_v4(slot_row(slot, l + T - 1)), xw[0]);
                float dt[T];
#pragma unroll
                for (int t = 0; t < T; ++t)
                    dt[t] = __uint_as_float((l & 1) ? (dw[t] & 0xFFFF0000u) : (dw[t] << 16));
                float2 acc[4];
                conv8<T>(bw, xw, dt, acc);
                store8(out + (size_t)(p0 + row0 + l) * C + c, acc);
            }
            issue(k + depth);
            continue;
        }
#pragma unroll
        for (int l = 0; l < kPL; ++l) {
            if (l < nl) {
#pragma unroll
                for (int t = T - 1; t > 0; --t)
#pragma unroll
                    for (int q = 0; q < 4; ++q) xw[t][q] = xw[t - 1][q];
                row_to_f2(lds_v4(slot_row(slot, l + T - 1)), xw[0]);
                float dt[T];
#pragma unroll
                for (int t = 0; t < T; ++t)
                    dt[t] = __uint_as_float((uint32_t)dsr[(size_t)t * ngl * kBM + l] << 16);
                float2 acc[4];
                conv8<T>(bw, xw, dt, acc);
                store8(out + (size_t)(p0 + row0 + l) * C + c, acc);
            }
        }
        issue(k + depth);  // the slot's rows have been read: refill it
    }
    cp_wait_pending(0);
    if (!ok) atomicOr(&g_fused_fault, (unsigned)DF2_FLAG_TIMEOUT);
}

unsigned pow2_at_least(unsigned v) {
    unsigned r = 32;
    while (r < v) r <<= 1;
    return r;
}

template <int T, typename TOut>
cudaError_t launch_t(const CUtensorMap& tmX, const CUtensorMap& tmW, const FusedParams& q,
                     size_t smem, int grid, cudaStream_t stream) {
    auto kern = dynconv_pred_kernel<T, TOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(threads_for(T), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)q.split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, tmX, tmW, q);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename TOut>
cudaError_t launch_out(int T, const CUtensorMap& tmX, const CUtensorMap& tmW, const FusedParams& q,
                       size_t smem, int grid, cudaStream_t stream) {
    switch (T) {
        case 1: return launch_t<1, TOut>(tmX, tmW, q, smem, grid, stream);
        case 2: return launch_t<2, TOut>(tmX, tmW, q, smem, grid, stream);
        case 3: return launch_t<3, TOut>(tmX, tmW, q, smem, grid, stream);
        case 4: return launch_t<4, TOut>(tmX, tmW, q, smem, grid, stream);
        case 5: return launch_t<5, TOut>(tmX, tmW, q, smem, grid, stream);
        case 6: return launch_t<6, TOut>(tmX, tmW, q, smem, grid, stream);
        case 7: return launch_t<7, TOut>(tmX, tmW, q, smem, grid, stream);
        case 8: return launch_t<8, TOut>(tmX, tmW, q, smem, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}


// ---------------------------------------------------------------- all-fp32 mode
//
// The same operation with fp32 inputs, delta in exact fp32 (FFMA, no TF32, no
// rounding between the steps): a CTA per 16 positions computes their delta tile
// [16][T*G] from 32-channel chunks of x and Wc staged in shared memory, then
// convolves the 16 positions over all channels from that tile.  Meant for the
// small fp32 shapes; the bf16 kernel above is the fast path.
constexpr int kFP = 16;     // positions per CTA
constexpr int kFK = 32;     // channels per staged chunk
constexpr int kFThreads = 256;

struct F32Params {
    const float* x;
    const float* hist;
    const float* base;
    const float* Wc;
    float* out;
    int P, n, C, T, G, TG, cg;
};

__global__ void __launch_bounds__(kFThreads) dynconv_pred_f32_kernel(const F32Params p) {
    extern __shared__ float fsm[];
    float* xs = fsm;                         // [kFP][kFK + 1]
    float* ws = xs + kFP * (kFK + 1);        // [TG][kFK + 1]
    float* dsm = ws + p.TG * (kFK + 1);      // [kFP][TG]
    const int tid = threadIdx.x;
    const int p0 = blockIdx.x * kFP;
    const int nout = kFP * p.TG;             // <= 16 * 256: at most 16 per thread
    float acc[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) acc[k] = 0.f;
    for (int j0 = 0; j0 < p.C; j0 += kFK) {
        for (int q = tid; q < kFP * kFK; q += kFThreads) {
            const int r = q / kFK, jj = q % kFK, j = j0 + jj;
            xs[r * (kFK + 1) + jj] = (p0 + r < p.P && j < p.C) ? p.x[(size_t)(p0 + r) * p.C + j] : 0.f;
        }
        for (int q = tid; q < p.TG * kFK; q += kFThreads) {
            const int r = q / kFK, jj = q % kFK, j = j0 + jj;
            ws[r * (kFK + 1) + jj] = j < p.C ? p.Wc[(size_t)r * p.C + j] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int q = tid + k * kFThreads;
            if (q < nout) {
                const int r = q / p.TG, col = q - r * p.TG;
                float a = acc[k];
#pragma unroll 8
                for (int jj = 0; jj < kFK; ++jj)
                    a = fmaf(xs[r * (kFK + 1) + jj], ws[col * (kFK + 1) + jj], a);
                acc[k] = a;
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int q = tid + k * kFThreads;
        if (q < nout) dsm[q] = acc[k];
    }
    __syncthreads();
    const int T = p.T;
    for (int q = tid; q < kFP * p.C; q += kFThreads) {
        const int r = q / p.C, c = q - r * p.C;
        const int pos = p0 + r;
        if (pos >= p.P) continue;
        const int s = pos / p.n, i = pos - s * p.n;
        const int g = c / p.cg;
        float a = 0.f;
        for (int t = 0; t < T; ++t) {
            float xv = 0.f;
            if (i - t >= 0)
                xv = p.x[(size_t)(pos - t) * p.C + c];
            else if (p.hist != nullptr)
                xv = p.hist[((size_t)s * (T - 1) + (T - 1 + i - t)) * p.C + c];
            a = fmaf(p.base[(size_t)t * p.C + c] + dsm[r * p.TG + t * p.G + g], xv, a);
        }
        p.out[(size_t)pos * p.C + c] = a;
    }
}

}  // namespace

bool plan_dynconv_pred(const DynconvPredArgs& a, int num_sms, size_t max_smem, DynconvPredPlan* plan) {
    if (a.T < 1 || a.T > kMaxPredT || a.G <= 0 || a.C <= 0 || a.C % a.G != 0) return false;
    const int TG = a.T * a.G;
    if (TG % 8 != 0 || TG > 256 || a.C % 8 != 0 || (a.C / a.G) % 8 != 0) return false;
    const long long P = (long long)a.S * a.n;
    if (P <= 0 || P > 0x7FFFFFFFLL) return false;
    DynconvPredPlan r{};
    r.NP = (TG + 15) & ~15;
    r.kblocks = (a.C + kBK - 1) / kBK;
    r.m_tiles = (int)((P + kBM - 1) / kBM);
    // Cluster size: doubled (up to 8, the portable limit) while the doubled
    // grid still fits the SMs in one wave and every CTA keeps at least two
    // 64-channel blocks.
    r.split = 1;
    while (r.split < 8 && (long long)r.m_tiles * r.split * 2 <= num_sms &&
           r.kblocks >= r.split * 4)
        r.split *= 2;
    if ((long long)r.m_tiles * r.split > 0x7FFFFFFFLL) return false;
    int ngl_max = 0;
    for (int rk = 0; rk < r.split; ++rk) {
        const int kb0 = (int)((long long)rk * r.kblocks / r.split);
        const int kb1 = (int)((long long)(rk + 1) * r.kblocks / r.split);
        const int c_lo = kb0 * kBK, c_hi = kb1 * kBK < a.C ? kb1 * kBK : a.C;
        const int ngl = (c_hi - 1) / (a.C / a.G) - c_lo / (a.C / a.G) + 1;
        if (ngl > ngl_max) ngl_max = ngl;
    }
    r.stage_bytes = kABytes + (uint32_t)r.NP * 128u;
    const size_t red_bytes = (size_t)kBM * TG * 4;
    const size_t conv_row_bytes = (size_t)(kPL + a.T - 1) * threads_for(a.T) * 16;  // one item slot
    const size_t ds_bytes = ((size_t)kBM * a.T * ngl_max * 2 + 15) & ~(size_t)15;
    // barriers, TMEM slot, piece count, piece table [129] and 4 warp counts
    const size_t tail = (2 * kMaxStages + 1) * 8 + 320;
    for (int st = kMaxStages; st >= 2; --st) {
        size_t ring = (size_t)st * r.stage_bytes;
        if (ring < red_bytes) ring = red_bytes;
        ring = (ring + 1023) & ~(size_t)1023;
        if (1024 + ring + ds_bytes + tail > max_smem) continue;
        // conv pieces in flight per thread: as many (up to 4) as fit, the ring
        // growing past the TMA stages if need be
        const size_t room = max_smem - 1024 - ds_bytes - tail;
        int depth = (int)(room / conv_row_bytes);
        if (depth > 4) depth = 4;
        if (depth < 1) continue;
        if ((size_t)depth * conv_row_bytes > ring)
            ring = (((size_t)depth * conv_row_bytes) + 1023) & ~(size_t)1023;
        const size_t total = 1024 + ring + ds_bytes + tail;
        if (total <= max_smem) {
            r.cdepth = depth;
            r.stages = st;
            r.ring_bytes = (uint32_t)ring;
            r.ds_bytes = (uint32_t)ds_bytes;
            r.smem_bytes = total;
            r.tmem_cols = pow2_at_least(2u * (unsigned)r.NP);  // two accumulators
            *plan = r;
            return true;
        }
    }
    return false;
}

cudaError_t launch_dynconv_pred(const DynconvPredArgs& a, const DynconvPredPlan& r,
                                cudaStream_t stream) {
    const int P = a.S * a.n;
    const int TG = a.T * a.G;
    CUtensorMap tmX, tmW;
    if (!make_tmap_rows_bf16(&tmX, a.x, P, a.C, kBM) ||
        !make_tmap_rows_bf16(&tmW, a.Wc, TG, a.C, r.NP))
        return cudaErrorInvalidValue;
    FusedParams q{};
    q.x = static_cast<const __nv_bfloat16*>(a.x);
    q.hist = static_cast<const __nv_bfloat16*>(a.hist);
    q.base = static_cast<const __nv_bfloat16*>(a.base);
    q.out = a.out;
    q.P = P;
    q.n = a.n;
    q.C = a.C;
    q.G = a.G;
    q.TG = TG;
    q.NP = r.NP;
    q.cg = a.C / a.G;
    q.kblocks = r.kblocks;
    q.split = r.split;
    q.stages = r.stages;
    q.stage_bytes = r.stage_bytes;
    q.ring_bytes = r.ring_bytes;
    q.ds_bytes = r.ds_bytes;
    q.tmem_cols = r.tmem_cols;
    q.cdepth = r.cdepth;
    const int grid = r.m_tiles * r.split;
    return a.out_bf16 ? launch_out<__nv_bfloat16>(a.T, tmX, tmW, q, r.smem_bytes, grid, stream)
                      : launch_out<float>(a.T, tmX, tmW, q, r.smem_bytes, grid, stream);
}

cudaError_t launch_dynconv_pred_f32(const DynconvPredArgs& a, cudaStream_t stream) {
    F32Params q{};
    q.x = static_cast<const float*>(a.x);
    q.hist = static_cast<const float*>(a.hist);
    q.base = static_cast<const float*>(a.base);
    q.Wc = static_cast<const float*>(a.Wc);
    q.out = static_cast<float*>(a.out);
    q.P = a.S * a.n;
    q.n = a.n;
    q.C = a.C;
    q.T = a.T;
    q.G = a.G;
    q.TG = a.T * a.G;
    q.cg = a.C / a.G;
    if (q.TG > 256) return cudaErrorInvalidValue;
    const size_t smem = ((size_t)kFP * (kFK + 1) + (size_t)q.TG * (kFK + 1) + (size_t)kFP * q.TG) *
                        sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(dynconv_pred_f32_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((q.P + kFP - 1) / kFP);
    dynconv_pred_f32_kernel<<<grid, kFThreads, smem, stream>>>(q);
    return cudaGetLastError();
}

cudaError_t take_fused_faults(unsigned* flags) {
    unsigned v = 0, zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fused_fault, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fused_fault, &zero, sizeof(zero));
    *flags = v;
    return e;
}

}  // namespace df2
