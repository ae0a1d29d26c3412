// Edge scores and per-predecessor argmax of the DFlash2 candidate selector
// (ggml-org/llama.cpp PR #27342, "spec : add DFlash2 support (local
// convolution + candidate selector)", Overview, second formula):
//   edge(p -> c) = < A[p] (.) project(h), B[c] > + unary[c]
// For every transition into position i (predecessors = candidates of i-1):
//   e[p,c] = sum_r A[id_p,r] u[i,r] B[id_c,r] + unary[i,c],  readout argmax_c.
//
// Paths, by codebook dtype and K:
//  - edges_pipe_kernel (bf16, K a power of two in [4, 128], R <= 512): one
//    persistent CTA per SM, warp-specialised.  Tiles of 128/K transitions
//    (128 predecessor rows and 128 candidate rows) round-robin over the CTAs;
//    16 gather warps copy the codebook rows by token id with 16-byte cp.async
//    straight into the 128-byte-swizzle K-major layout of the tensor core, 4
//    gate warps form A[id_p] (.) u in place (fp32 product, bf16 rounding), one
//    warp issues tcgen05.mma (M = N = 128) into one of two TMEM accumulators,
//    and 4 epilogue warps read back only each transition's K x K diagonal
//    block (+ unary, running argmax, lowest slot on ties).  The off-diagonal
//    blocks are free work on an otherwise idle unit.
//  - edges_tc_kernel (bf16, K in {1, 2}, R <= 384): the same contraction, one
//    tile per CTA, no pipeline.
//  - edges_warp_kernel (any K <= 256, R <= 512, fp32 or bf16 codebooks): one
//    warp per (transition, predecessor); lanes split R, the gate stays in
//    registers, and each candidate's dot product is reduced with warp
//    shuffles.  This is the exact-fp32 path.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>

#include "dflash2.h"
#include "common.cuh"
#include "ptx.cuh"

namespace df2 {
namespace {

struct EParams {
    const int32_t* cand_ids;
    const float* u;
    const void* A;
    const void* B;
    const float* unary;
    int S, n, K, R, V;
    int E;  // transitions = S * (n - 1)
    uint32_t nm1_magic;  // floor((2^32 - 1) / (n - 1)) (1 when n = 1: no transitions)
    float* edges_out;
    int32_t* best_slot;
    float* best_score;
    int32_t* err_flag;
};

// floor(e / d) for 0 <= e < 2^31, d >= 1, with m = floor((2^32 - 1) / d): the
// high half of e * m is the quotient or one less (one correction step), so the
// per-row index math needs no integer divide (which the hardware lacks).
__device__ __forceinline__ int div_by(int e, int d, uint32_t m) {
    int q = (int)__umulhi((uint32_t)e, m);
    if (e - q * d >= d) ++q;
    return q;
}

__device__ __forceinline__ int checked_id(int id, int V, bool& bad) {
    if (id < 0 || id >= V) {
        bad = true;
        return id < 0 ? 0 : V - 1;
    }
    return id;
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t f2_to_bf16x2(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
}

// ------------------------------------------------------------------ tile path

constexpr int TROWS = 128;
constexpr int KB_BYTES = TROWS * 128;  // one 64-element k-block of 128 rows

// Shared memory of the tile kernel: two operand tiles (KB k-blocks of 128
// rows x 128 bytes each), the tile's u rows when they fit, ids and offsets.
template <int KB>
struct TileSmem {
    static constexpr size_t op_bytes = (size_t)KB * KB_BYTES;
    static constexpr size_t fixed = 1024 /*align*/ + 2 * op_bytes + TROWS * 4 * 2 /*ids*/ +
                                    TROWS * 4 /*u row offsets*/ + 64;
    static constexpr size_t max_u = 32768;
    static size_t total(size_t u_bytes) {
        size_t t = fixed + u_bytes;
        // Never fewer than ~60 KB per CTA: at most 3 CTAs share an SM, so their
        // 3 x 128 TMEM columns always fit in the SM's 512.
        return t < 61440 ? 61440 : t;
    }
};

template <int KB>
__global__ void __launch_bounds__(128) edges_tc_kernel(const EParams p, const int log2K,
                                                       const int stage_u) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int K = p.K;
    const int R = p.R;
    const int TP = TROWS >> log2K;
    uint8_t* opA = smem;
    uint8_t* opB = smem + TileSmem<KB>::op_bytes;
    int32_t* ids_p = reinterpret_cast<int32_t*>(opB + TileSmem<KB>::op_bytes);
    int32_t* ids_c = ids_p + TROWS;
    int32_t* urow = ids_c + TROWS;                             // [TP] row index of u
    float* us = reinterpret_cast<float*>(urow + TROWS);        // [TP][R] when staged
    uint64_t* mbar = reinterpret_cast<uint64_t*>(us + (stage_u ? (size_t)TP * R : 0));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int e0 = blockIdx.x * TP;
    const int nm1 = p.n - 1;
    bool bad = false;

    // 1. ids of this tile's 128 predecessor rows and 128 candidate rows, and
    //    the u row of each of its transitions
    {
        const int e = e0 + (tid >> log2K);
        const int slot = tid & (K - 1);
        int idp = 0, idc = 0;
        if (e < p.E) {
            const int s = e / nm1;
            const int i = e % nm1 + 1;
            idp = checked_id(p.cand_ids[((size_t)s * p.n + i - 1) * K + slot], p.V, bad);
            idc = checked_id(p.cand_ids[((size_t)s * p.n + i) * K + slot], p.V, bad);
            if (slot == 0) urow[tid >> log2K] = s * p.n + i;
        } else if (slot == 0) {
            urow[tid >> log2K] = -1;
        }
        ids_p[tid] = idp;
        ids_c[tid] = idc;
    }
    if (tid == 0) {
        mbar_init(smem_u32(mbar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // 2. asynchronous gathers: raw rows of A and B straight into the
    //    128-byte-swizzle K-major operand layout, and the u rows
    constexpr int CPR = KB * 8;  // 16-byte chunks per (padded) row
    const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(p.A);
    const __nv_bfloat16* B = static_cast<const __nv_bfloat16*>(p.B);
    const uint32_t sA = smem_u32(opA);
    const uint32_t sB = smem_u32(opB);
#pragma unroll 4
    for (int j = 0; j < CPR; ++j) {
        const int slot = j * 128 + tid;
        const int row = slot / CPR;
        const int ch = slot % CPR;
        const uint32_t off =
            (uint32_t)((ch >> 3) * KB_BYTES + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
        if (ch * 8 < R) {
            cp_async16(sA + off, A + (size_t)ids_p[row] * R + ch * 8);
            cp_async16(sB + off, B + (size_t)ids_c[row] * R + ch * 8);
        } else {
            st_shared_v4(sA + off, make_uint4(0, 0, 0, 0));
            st_shared_v4(sB + off, make_uint4(0, 0, 0, 0));
        }
    }
    if (stage_u) {
        const uint32_t su = smem_u32(us);
        const int c4 = R >> 2;
        for (int q = tid; q < TP * c4; q += 128) {
            const int tt = q / c4;
            const int r4 = q - tt * c4;
            const int ur = urow[tt];
            if (ur >= 0)
                cp_async16(su + (uint32_t)q * 16u, p.u + (size_t)ur * R + r4 * 4);
            else
                st_shared_v4(su + (uint32_t)q * 16u, make_uint4(0, 0, 0, 0));
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // 3. gate in place: A chunk (.) u, rounded to bf16
#pragma unroll 4
    for (int j = 0; j < CPR; ++j) {
        const int slot = j * 128 + tid;
        const int row = slot / CPR;
        const int ch = slot % CPR;
        if (ch * 8 < R) {
            const uint32_t off =
                (uint32_t)((ch >> 3) * KB_BYTES + row * 128 + (((ch & 7) ^ (row & 7)) << 4));
            const int tt = row >> log2K;
            float4 u0, u1;
            if (stage_u) {
                const float4* ur = reinterpret_cast<const float4*>(us + (size_t)tt * R + ch * 8);
                u0 = ur[0];
                u1 = ur[1];
            } else if (urow[tt] >= 0) {
                const float4* ur =
                    reinterpret_cast<const float4*>(p.u + (size_t)urow[tt] * R + ch * 8);
                u0 = __ldg(ur);
                u1 = __ldg(ur + 1);
            } else {
                u0 = make_float4(0.f, 0.f, 0.f, 0.f);
                u1 = u0;
            }
            const uint4 a = lds_v4(sA + off);
            const float2 a0 = bf16x2_to_f2(a.x), a1 = bf16x2_to_f2(a.y);
            const float2 a2 = bf16x2_to_f2(a.z), a3 = bf16x2_to_f2(a.w);
            uint4 g;
            g.x = f2_to_bf16x2(a0.x * u0.x, a0.y * u0.y);
            g.y = f2_to_bf16x2(a1.x * u0.z, a1.y * u0.w);
            g.z = f2_to_bf16x2(a2.x * u1.x, a2.y * u1.y);
            g.w = f2_to_bf16x2(a3.x * u1.z, a3.y * u1.w);
            st_shared_v4(sA + off, g);
        }
    }
    fence_proxy_async_smem();
    __syncthreads();

    // 3. one thread issues the contraction over R
    if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
        const int ksteps = (R + 15) / 16;
        for (int ks = 0; ks < ksteps; ++ks) {
            const uint32_t koff = (uint32_t)((ks >> 2) * KB_BYTES + (ks & 3) * 32);
            tc_mma_bf16(tmem, sw128_desc(sA + koff), sw128_desc(sB + koff), idesc,
                        ks > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(mbar));
    }
    __syncwarp();
    const bool ok = mbar_wait_bounded(smem_u32(mbar), 0, kWaitNs);
    tc_fence_after();

    // 4. epilogue: this thread's predecessor row, its transition's K columns
    const int r = tid;
    const int e = e0 + (r >> log2K);
    const int pslot = r & (K - 1);
    const int blk0 = r & ~(K - 1);                      // first column of the block
    const int colbase = K >= 32 ? blk0 : 32 * warp;     // warp-uniform
    const int width = K >= 32 ? K : 32;
    int s = 0, i = 1;
    if (e < p.E) {
        s = e / nm1;
        i = e % nm1 + 1;
    }
    const float* un = p.unary + ((size_t)s * p.n + i) * K;
    float* erow = p.edges_out != nullptr ? p.edges_out + ((size_t)e * K + pslot) * K : nullptr;
    float best = 0.f;
    int arg = 0;
#pragma unroll 1
    for (int cc = 0; cc < width; cc += 32) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(colbase + cc), v);
        tmem_ld_wait();
        if (e < p.E) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int c = colbase + cc + j - blk0;
                if (c >= 0 && c < K) {
                    const float ev = __uint_as_float(v[j]) + un[c];
                    if (erow != nullptr) erow[c] = ev;
                    if (c == 0 || ev > best) {
                        best = ev;
                        arg = c;
                    }
                }
            }
        }
    }
    if (e < p.E) {
        p.best_slot[(size_t)e * K + pslot] = arg;
        p.best_score[(size_t)e * K + pslot] = best;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
    if (p.err_flag != nullptr) {
        int flags = (bad ? DF2_FLAG_BAD_ID : 0) | (ok ? 0 : DF2_FLAG_TIMEOUT);
        if (flags) atomicOr(p.err_flag, flags);
    }
}

// ------------------------------------------------------------------ pipelined tile path
//
// Persistent CTAs (at most one per SM), warp-specialised, for K a power of two
// in [4, 128].  Work is a list of tiles of up to TP = 128/K transitions: whole
// tiles round-robin over the CTAs, then the leftover transitions cut into
// equal small pieces, one more per CTA, so the last round is not a partial
// wave of whole tiles.  Per tile and 64-rank k-block:
//   warps 9+    gather:   the tile's 256 candidate ids into shared memory, then
//                         16-byte cp.async copies of the 128 A rows and 128 B
//                         rows (128 bytes of each) straight into the
//                         128-byte-swizzle K-major operand layout, and of the u
//                         slice, completion tracked on full[stage].  Sixteen
//                         warps spread the outstanding requests over all four
//                         SM sub-partitions;
//   warps 4-7   gate:     A (.) u in place (fp32 product, bf16 rounding), proxy
//                         fence, arrive on gated[stage];
//   warp 8      MMA:      tcgen05.mma M=N=128 over the k-block into one of two
//                         TMEM accumulators; commit frees the stage and, after
//                         the last k-block, signals tmem_full;
//   warps 0-3   epilogue: one thread per predecessor row: unary prefetched,
//                         tcgen05.ld of its own transition's K columns, running
//                         argmax, stores; then releases the accumulator.

constexpr int EP_STAGES = 5;
constexpr int EP_OP = TROWS * 128;               // one operand k-block: 16 KB
constexpr int EP_U = 32 * 64 * 4;                // u slice: TP <= 32 rows x 64 ranks fp32
constexpr int EP_STAGE = 2 * EP_OP + EP_U;       // 40 KB
constexpr int EP_GWARPS = 16;                    // gather warps (four per SM sub-partition)
constexpr int EP_GTHREADS = EP_GWARPS * 32;
constexpr int EP_THREADS = (9 + EP_GWARPS) * 32;  // 4 epilogue, 4 gate, 1 MMA, gather warps
constexpr size_t EP_SMEM = 1024 + (size_t)EP_STAGES * EP_STAGE + 6 * TROWS * 4 +
                           (3 * EP_STAGES + 4) * 8 + 16;

struct TileList {
    int TP, rounds_tiles, piece, n_items, E;
    // item -> first transition and transition count
    __device__ __forceinline__ void at(int idx, int& e0, int& cnt) const {
        if (idx < rounds_tiles) {
            e0 = idx * TP;
            cnt = TP;
        } else {
            e0 = rounds_tiles * TP + (idx - rounds_tiles) * piece;
            cnt = min(piece, E - e0);
        }
    }
};

__global__ void __launch_bounds__(EP_THREADS, 1)
    edges_pipe_kernel(const EParams p, const int log2K, const TileList tl_list, const int nkb,
                      const int zero_pad, const int u_only_dependency) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int K = p.K;
    const int R = p.R;
    const int nm1 = p.n - 1;
    int32_t* ids_p = reinterpret_cast<int32_t*>(smem + (size_t)EP_STAGES * EP_STAGE);  // [2][256]
    int32_t* urow = ids_p + 4 * TROWS;                                                 // [2][128]
    uint64_t* bars = reinterpret_cast<uint64_t*>(urow + 2 * TROWS);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t gated0 = full0 + 8 * EP_STAGES;
    const uint32_t empty0 = gated0 + 8 * EP_STAGES;
    const uint32_t tfull0 = empty0 + 8 * EP_STAGES;
    const uint32_t tempty0 = tfull0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * EP_STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t st0 = smem_u32(smem);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (zero_pad) {  // k-block columns past R stay zero for the whole kernel
        for (int q = tid; q < EP_STAGES * EP_STAGE / 16; q += EP_THREADS)
            st_shared_v4(st0 + (uint32_t)q * 16u, make_uint4(0, 0, 0, 0));
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int i = 0; i < EP_STAGES; ++i) {
            mbar_init(full0 + 8 * i, EP_GTHREADS);
            mbar_init(gated0 + 8 * i, 128);
            mbar_init(empty0 + 8 * i, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, 128);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(tmem_slot), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent.  When the previous grid only
    // produces u (the projection of the composite selector, which itself waited
    // for everything before it), ids, codebooks and unary may be read at once
    // and only the u copies wait; otherwise every thread waits here.
    if (!u_only_dependency) griddep_wait();
    griddep_launch_dependents();

    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (*abort_flag) return;
        if (!mbar_wait_bounded(bar, parity, kWaitNs)) *abort_flag = 1;
    };

    if (warp >= 9) {
        // ------------------------------------------------ gather (EP_GWARPS warps)
        // ids and u-row indices are double-buffered by tile parity; the next
        // tile's raw ids are loaded into registers after this tile's copies are
        // issued and range-checked only where they are stored, one tile later,
        // so no copy waits on an id round trip.
        const int gtid = tid - 9 * 32;
        const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(p.A);
        const __nv_bfloat16* B = static_cast<const __nv_bfloat16*>(p.B);
        bool bad = false;
        auto load_id = [&](int idx, int& id, int& ur) {  // thread gtid < 256: one raw id
            id = 0;
            ur = 0;
            if (idx >= tl_list.n_items || gtid >= 2 * TROWS) return;
            int e0, cnt;
            tl_list.at(idx, e0, cnt);
            const int r = gtid & (TROWS - 1);
            const int tt = r >> log2K;
            if (tt < cnt) {
                const int e = e0 + tt;
                const int s = div_by(e, nm1, p.nm1_magic);
                const int i = e - s * nm1 + 1;
                const int pos = s * p.n + i - (gtid < TROWS ? 1 : 0);
                id = p.cand_ids[(size_t)pos * K + (r & (K - 1))];
                ur = s * p.n + i;
            }
        };
        int id_next, ur_next;
        load_id(blockIdx.x, id_next, ur_next);
        int it = 0, tl = 0;
        for (int idx = blockIdx.x; idx < tl_list.n_items; idx += gridDim.x, ++tl) {
            int e0, cnt;
            tl_list.at(idx, e0, cnt);
            const int rows = cnt << log2K;
            int32_t* idp = ids_p + (tl & 1) * 2 * TROWS;  // [pred 128 | cand 128] per parity
            int32_t* idc = idp + TROWS;
            int32_t* urw = urow + (tl & 1) * TROWS;
            // slot tl&1 was last read while issuing tile tl-2; every gather warp
            // finished that before the barrier of tile tl-1 below, which this
            // warp has passed, so the slot is free without another barrier
            if (gtid < TROWS) {
                idp[gtid] = checked_id(id_next, p.V, bad);
                if ((gtid & (K - 1)) == 0) urw[gtid >> log2K] = ur_next;
            } else if (gtid < 2 * TROWS) {
                idc[gtid - TROWS] = checked_id(id_next, p.V, bad);
            }
            named_bar_sync(1, EP_GTHREADS);
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int st = it % EP_STAGES;
                wait(empty0 + 8 * st, (((uint32_t)(it / EP_STAGES)) & 1u) ^ 1u);
                const uint32_t sA = st0 + (uint32_t)st * EP_STAGE;
                const uint32_t sB = sA + EP_OP;
                const uint32_t sU = sB + EP_OP;
                if (!*abort_flag) {
#pragma unroll
                    for (int j = 0; j < (TROWS * 8) / EP_GTHREADS; ++j) {
                        const int q = j * EP_GTHREADS + gtid;
                        const int row = q >> 3;
                        const int ch = q & 7;
                        const int col = kb * 64 + ch * 8;
                        if (row < rows && col < R) {
                            const uint32_t off =
                                (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
                            cp_async16(sA + off, A + (size_t)idp[row] * R + col);
                            cp_async16(sB + off, B + (size_t)idc[row] * R + col);
                        }
                    }
                    if (u_only_dependency && it == 0) griddep_wait();
                    for (int q = gtid; q < cnt * 16; q += EP_GTHREADS) {
                        const int col = kb * 64 + (q & 15) * 4;
                        if (col < R)
                            cp_async16(sU + (uint32_t)q * 16u, p.u + (size_t)urw[q >> 4] * R + col);
                    }
                }
                cp_async_mbar_arrive_noinc(full0 + 8 * st);
            }
            load_id(idx + gridDim.x, id_next, ur_next);  // the next tile's raw ids
        }
        if (bad && p.err_flag != nullptr) atomicOr(p.err_flag, DF2_FLAG_BAD_ID);
    } else if (warp >= 4 && warp < 8) {
        // ------------------------------------------------ gate
        const int gt = tid - 128;
        int it = 0;
        for (int idx = blockIdx.x; idx < tl_list.n_items; idx += gridDim.x) {
            int e0, cnt;
            tl_list.at(idx, e0, cnt);
            const int rows = cnt << log2K;
            for (int kb = 0; kb < nkb; ++kb, ++it) {
                const int st = it % EP_STAGES;
                wait(full0 + 8 * st, ((uint32_t)(it / EP_STAGES)) & 1u);
                const uint32_t sA = st0 + (uint32_t)st * EP_STAGE;
                const float* us = reinterpret_cast<const float*>(smem + (size_t)st * EP_STAGE +
                                                                 2 * EP_OP);
                if (!*abort_flag) {
#pragma unroll 4
                    for (int q = gt; q < TROWS * 8; q += 128) {
                        const int row = q >> 3;
                        const int ch = q & 7;
                        if (row < rows && kb * 64 + ch * 8 < R) {
                            const uint32_t off =
                                (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
                            const float4* ur = reinterpret_cast<const float4*>(
                                us + (row >> log2K) * 64 + ch * 8);
                            const float4 u0 = ur[0];
                            const float4 u1 = ur[1];
                            const uint4 a = lds_v4(sA + off);
                            const float2 a0 = bf16x2_to_f2(a.x), a1 = bf16x2_to_f2(a.y);
                            const float2 a2 = bf16x2_to_f2(a.z), a3 = bf16x2_to_f2(a.w);
                            uint4 g;
                            g.x = f2_to_bf16x2(a0.x * u0.x, a0.y * u0.y);
                            g.y = f2_to_bf16x2(a1.x * u0.z, a1.y * u0.w);
                            g.z = f2_to_bf16x2(a2.x * u1.x, a2.y * u1.y);
                            g.w = f2_to_bf16x2(a3.x * u1.z, a3.y * u1.w);
                            st_shared_v4(sA + off, g);
                        }
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(gated0 + 8 * st);
            }
        }
    } else if (warp == 8) {
        // ------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            int it = 0, tl = 0;
            for (int idx = blockIdx.x; idx < tl_list.n_items; idx += gridDim.x, ++tl) {
                const int buf = tl & 1;
                wait(tempty0 + 8 * buf, (((uint32_t)(tl >> 1)) & 1u) ^ 1u);
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(buf * 128);
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int st = it % EP_STAGES;
                    wait(gated0 + 8 * st, ((uint32_t)(it / EP_STAGES)) & 1u);
                    tc_fence_after();
                    const uint32_t sA = st0 + (uint32_t)st * EP_STAGE;
                    const uint32_t sB = sA + EP_OP;
                    const int kst = min(4, (R - kb * 64 + 15) / 16);
                    for (int k = 0; k < kst; ++k)
                        tc_mma_bf16(d, sw128_desc(sA + 32 * k), sw128_desc(sB + 32 * k), idesc,
                                    (kb > 0 || k > 0) ? 1u : 0u);
                    tc_commit(empty0 + 8 * st);
                }
                tc_commit(tfull0 + 8 * buf);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 0-3)
        const int r = tid;
        const int pslot = r & (K - 1);
        const int blk0 = r & ~(K - 1);
        const int colbase = K >= 32 ? blk0 : 32 * warp;  // warp-uniform
        const int width = K >= 32 ? K : 32;
        int tl = 0;
        for (int idx = blockIdx.x; idx < tl_list.n_items; idx += gridDim.x, ++tl) {
            int e0, cnt;
            tl_list.at(idx, e0, cnt);
            const int buf = tl & 1;
            const bool valid = (r >> log2K) < cnt;
            const int e = e0 + (r >> log2K);
            int s = 0, i = 1;
            if (valid) {
                s = div_by(e, nm1, p.nm1_magic);
                i = e - s * nm1 + 1;
            }
            const float* un = p.unary + ((size_t)s * p.n + i) * K;
            float* erow =
                (p.edges_out != nullptr && valid) ? p.edges_out + ((size_t)e * K + pslot) * K : nullptr;
            float best = 0.f;
            int arg = 0;
            float ua[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) {  // first column chunk's unary, before the wait
                const int c = colbase + j - blk0;
                ua[j] = (valid && c >= 0 && c < K) ? __ldg(un + c) : 0.f;
            }
            wait(tfull0 + 8 * buf, ((uint32_t)(tl >> 1)) & 1u);
            tc_fence_after();
#pragma unroll 1
            for (int cc = 0; cc < width; cc += 32) {
                if (cc > 0) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int c = colbase + cc + j - blk0;
                        ua[j] = (valid && c >= 0 && c < K) ? __ldg(un + c) : 0.f;
                    }
                }
                uint32_t v[32];
                tmem_ld_32x32b_x32(
                    tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * 128 + colbase + cc), v);
                tmem_ld_wait();
                if (valid) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int c = colbase + cc + j - blk0;
                        if (c >= 0 && c < K) {
                            const float ev = __uint_as_float(v[j]) + ua[j];
                            if (erow != nullptr) erow[c] = ev;
                            if (c == 0 || ev > best) {
                                best = ev;
                                arg = c;
                            }
                        }
                    }
                }
            }
            if (valid) {
                p.best_slot[(size_t)e * K + pslot] = arg;
                p.best_score[(size_t)e * K + pslot] = best;
            }
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * buf);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
    if (tid == 0 && *abort_flag && p.err_flag != nullptr) atomicOr(p.err_flag, DF2_FLAG_TIMEOUT);
}

// ------------------------------------------------------------------ warp path

template <typename TCB>
__device__ __forceinline__ float cb_load(const TCB* p);
template <>
__device__ __forceinline__ float cb_load<float>(const float* p) {
    return __ldg(p);
}
template <>
__device__ __forceinline__ float cb_load<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

constexpr int WARP_MAXJ = 16;  // R <= 512

template <typename TCB>
__global__ void __launch_bounds__(256) edges_warp_kernel(const EParams p) {
    const int lane = threadIdx.x & 31;
    const long long gw = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (gw >= (long long)p.E * p.K) return;
    const int K = p.K;
    const int R = p.R;
    const int e = (int)(gw / K);
    const int pslot = (int)(gw % K);
    const int nm1 = p.n - 1;
    const int s = e / nm1;
    const int i = e % nm1 + 1;
    const TCB* A = static_cast<const TCB*>(p.A);
    const TCB* B = static_cast<const TCB*>(p.B);
    bool bad = false;
    const int idp = checked_id(p.cand_ids[((size_t)s * p.n + i - 1) * K + pslot], p.V, bad);
    const float* urow = p.u + ((size_t)s * p.n + i) * R;
    float g[WARP_MAXJ];
#pragma unroll
    for (int j = 0; j < WARP_MAXJ; ++j) {
        const int r = lane + 32 * j;
        g[j] = r < R ? cb_load(A + (size_t)idp * R + r) * urow[r] : 0.f;
    }
    const int32_t* cands = p.cand_ids + ((size_t)s * p.n + i) * K;
    const float* un = p.unary + ((size_t)s * p.n + i) * K;
    float* erow = p.edges_out != nullptr ? p.edges_out + ((size_t)e * K + pslot) * K : nullptr;
    float best = 0.f;
    int arg = 0;
    for (int c = 0; c < K; ++c) {
        const int idc = checked_id(cands[c], p.V, bad);
        const TCB* brow = B + (size_t)idc * R;
        float part = 0.f;
#pragma unroll
        for (int j = 0; j < WARP_MAXJ; ++j) {
            const int r = lane + 32 * j;
            if (r < R) part = fmaf(g[j], cb_load(brow + r), part);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
        const float ev = part + un[c];
        if (erow != nullptr && lane == 0) erow[c] = ev;
        if (c == 0 || ev > best) {
            best = ev;
            arg = c;
        }
    }
    if (lane == 0) {
        p.best_slot[(size_t)e * K + pslot] = arg;
        p.best_score[(size_t)e * K + pslot] = best;
        if (bad && p.err_flag != nullptr) atomicOr(p.err_flag, DF2_FLAG_BAD_ID);
    }
}

EParams make_params(const EdgesArgs& a) {
    EParams p{};
    p.cand_ids = a.cand_ids;
    p.u = a.u;
    p.A = a.A;
    p.B = a.B;
    p.unary = a.unary;
    p.S = a.S;
    p.n = a.n;
    p.K = a.K;
    p.R = a.R;
    p.V = a.V;
    p.E = a.S * (a.n - 1);
    p.nm1_magic = a.n > 1 ? 0xFFFFFFFFu / (uint32_t)(a.n - 1) : 1u;
    p.edges_out = a.edges_out;
    p.best_slot = a.best_slot;
    p.best_score = a.best_score;
    p.err_flag = a.err_flag;
    return p;
}

template <int KB>
cudaError_t launch_tc(const EParams& p, cudaStream_t stream) {
    int log2K = 0;
    while ((1 << log2K) < p.K) ++log2K;
    const int TP = TROWS >> log2K;
    const size_t u_bytes = (size_t)TP * p.R * 4;
    const int stage_u = u_bytes <= TileSmem<KB>::max_u &&
                        TileSmem<KB>::fixed + u_bytes <= 220 * 1024;
    const size_t smem = TileSmem<KB>::total(stage_u ? u_bytes : 0);
    cudaError_t e = cudaFuncSetAttribute(edges_tc_kernel<KB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int tiles = (p.E + TP - 1) / TP;
    edges_tc_kernel<KB><<<tiles, 128, smem, stream>>>(p, log2K, stage_u);
    return cudaGetLastError();
}

}  // namespace

bool edges_tc_supported(int K, int R) {
    if (K < 1 || K > 128 || (K & (K - 1)) != 0 || R % 8 != 0) return false;
    return K >= 4 ? R <= 512 : R <= 384;
}

cudaError_t launch_edges_pipe(const EParams& p, int u_only_dependency, cudaStream_t stream) {
    int log2K = 0;
    while ((1 << log2K) < p.K) ++log2K;
    const int TP = TROWS >> log2K;
    const int nkb = (p.R + 63) / 64;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(edges_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)EP_SMEM);
    if (e != cudaSuccess) return e;
    // whole tiles round-robin, then the leftover transitions in equal pieces
    const int G = p.E < sms ? p.E : sms;
    TileList tl{};
    tl.TP = TP;
    tl.E = p.E;
    tl.rounds_tiles = (p.E / TP / G) * G;
    const int rem = p.E - tl.rounds_tiles * TP;
    tl.piece = rem > 0 ? std::min(TP, (rem + G - 1) / G) : TP;
    const int n_pieces = rem > 0 ? (rem + tl.piece - 1) / tl.piece : 0;
    tl.n_items = tl.rounds_tiles + n_pieces;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(EP_THREADS);
    cfg.dynamicSmemBytes = EP_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, edges_pipe_kernel, p, log2K, tl, nkb, (int)(p.R % 64 != 0),
                           u_only_dependency);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_edges_bf16_tc(const EdgesArgs& a, int u_only_dependency, cudaStream_t stream) {
    const EParams p = make_params(a);
    if (p.E <= 0) return cudaSuccess;
    if (p.K >= 4 && p.K <= 128) return launch_edges_pipe(p, u_only_dependency, stream);
    switch ((a.R + 63) / 64) {
        case 1:
            return launch_tc<1>(p, stream);
        case 2:
            return launch_tc<2>(p, stream);
        case 3:
            return launch_tc<3>(p, stream);
        case 4:
            return launch_tc<4>(p, stream);
        case 5:
            return launch_tc<5>(p, stream);
        case 6:
            return launch_tc<6>(p, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_edges_warp(const EdgesArgs& a, int cb_bf16, cudaStream_t stream) {
    const EParams p = make_params(a);
    if (p.E <= 0) return cudaSuccess;
    const long long warps = (long long)p.E * p.K;
    const long long blocks = (warps + 7) / 8;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    if (cb_bf16)
        edges_warp_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(p);
    else
        edges_warp_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace df2
