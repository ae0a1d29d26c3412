// The composite candidate selector in one kernel: project(h) and the edge
// scores with the per-predecessor argmax (ggml-org/llama.cpp PR #27342,
// "spec : add DFlash2 support (local convolution + candidate selector)",
// Overview, second formula):
//   u      = h W^T                                  (each position's hidden, d -> R)
//   e[p,c] = < A[id_p] (.) u[i], B[id_c] > + unary[i,c]   (p -> c into position i)
//   best_slot / best_score = lowest slot reaching max_c e[p,c], and that max.
//
// Why one kernel: the projection streams h from HBM and the edge scores gather
// codebook rows at random token ids; both are memory-bound, and the gathers do
// not depend on u (only the gate A (.) u does).  Fused, the first edge tile's
// gathers are in flight while h streams, u never goes back to HBM before the
// gate, and the whole selector pays one launch.
//
// Decomposition (bf16; K a power of two in [4, 128]; R = 64, 128 or 256):
//  - Positions are cut into row blocks of MR <= 128 consecutive rows, one per
//    thread-block cluster of CS CTAs (one CTA per SM).  The cluster splits d:
//    CTA r streams k-blocks [r*kb/CS, (r+1)*kb/CS) of its row block of h and
//    of W through a TMA ring (128-byte swizzle) into tcgen05.mma (M = 128,
//    N = R) with the fp32 partial in tensor memory.  Up to three warps issue
//    the MMAs, taking the k-blocks in turn, each into its own accumulator; the
//    accumulators are summed in issuer order when the partial is drained.
//  - The partial tiles are reduced through distributed shared memory: CTA r
//    owns rows [r*MR/CS, (r+1)*MR/CS) of the block; after one cluster barrier
//    every CTA pushes each owner's rows of its partial with one bulk
//    shared-to-shared copy, the owner sums the CS partials in rank order
//    (deterministic), writes its u rows to HBM (the caller's u_out) and keeps
//    them in shared memory, and tells each sender that its buffer has been
//    read (a remote mbarrier arrive the sender waits for only before it
//    reuses that buffer).
//  - CTA r then scores every transition INTO its own positions (transitions
//    are numbered e = s*(n-1) + i-1, so a contiguous run of positions owns a
//    contiguous run of transitions).  Tiles of 128/K transitions hold 128
//    predecessor rows of A and 128 candidate rows of B (one edge stage per 128
//    ranks).  8 gather warps copy the rows by token id with 16-byte cp.async
//    straight into the tensor core's 128-byte-swizzle K-major layout and only
//    issue copies (completion is counted on the stage's mbarrier by
//    cp.async.mbarrier.arrive.noinc): a warp that also read back what it
//    copied would stall its own next copies.  The projection's TMA ring spans
//    the edge stages' memory; the first stage's copies are issued as soon as
//    the projection's MMAs are done, under the exchange of partials.  4 gate
//    warps form A (.) u in place (fp32 product, rounded to bf16) once a stage
//    has landed, fence the async proxy and meet at a named barrier, after
//    which one of their threads issues tcgen05.mma (M = N = 128) into one of
//    two tensor-memory accumulators; 4 epilogue warps read back only each transition's K x K
//    diagonal block, add unary, keep the running argmax (lowest slot on ties)
//    and store.
// Every wait on an mbarrier is bounded by the global timer; on a timeout the
// kernel sets DF2_FLAG_TIMEOUT and runs to completion without hanging.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "dflash2.h"
#include "common.cuh"
#include "ptx.cuh"

namespace df2 {

// Device-side fault word of the fused selector (read by dflash2_take_device_faults).
__device__ unsigned int g_select_fault = 0;

// Phase trace (compiled in only with -DDF2_TRACE; otherwise every trace point
// is empty): global-timer stamps of CTAs 0..kTraceCTAs-1, kTraceSlots per CTA,
// at the points include/dflash2.h lists with dflash2_trace_read.  DF2_TRACE_RB
// records only during a CTA's first row block.
#ifdef DF2_TRACE
constexpr int kTraceCTAs = 512;
constexpr int kTraceSlots = 64;
__device__ unsigned long long g_trace[kTraceCTAs * kTraceSlots];
#define DF2_TRACE_AT(k)                                                                   \
    do {                                                                                  \
        if (blockIdx.x < (unsigned)kTraceCTAs) g_trace[blockIdx.x * kTraceSlots + (k)] = global_ns(); \
    } while (0)
#else
#define DF2_TRACE_AT(k) \
    do {                \
    } while (0)
#endif
#define DF2_TRACE_RB(k)                \
    do {                               \
        if (rbi == 0) DF2_TRACE_AT(k); \
    } while (0)

namespace {

constexpr int SEL_THREADS = 512;   // 16 warps
constexpr int SEL_GTHREADS = 256;  // warps 8..15: gather + gate
constexpr int EROWS = 128;         // rows of an edge operand tile
constexpr int KB_OP = EROWS * 128; // one 64-rank k-block of one edge operand (16 KB)
constexpr int HTILE = 128 * 128;   // one 64-column k-block of 128 rows of h (16 KB)
constexpr int EACC = 256;          // first tensor-memory column of the edge accumulators

struct SelParams {
    const int32_t* cand_ids;
    const float* unary;
    const __nv_bfloat16* A;
    const __nv_bfloat16* B;
    float* u;
    float* edges_out;
    int32_t* best_slot;
    float* best_score;
    int32_t* err_flag;
    int S, n, K, R, V, P;
    int log2K;
    int log2R;
    uint32_t nm1_magic;  // floor((2^32 - 1) / (n - 1)): e / (n - 1) without a divide
    uint32_t ps_magic;   // the same for pstages
    uint32_t es_magic;   // the same for estages
    int CS;            // CTAs per cluster (split of d)
    int MR;            // rows per row block
    int nrb;           // row blocks
    int kblocks;       // 64-column k-blocks of d
    int own_max;       // most rows a CTA owns after the reduction
    int pstages;       // projection TMA stages
    int nmma;          // projection MMA issuers (warps 1..nmma), one accumulator each
    int estages;       // edge stages: stage 0 is region E, the others live in region P
    int nkb_e;         // 64-rank k-blocks per edge stage (1 or 2)
    int nhalf;         // edge stages per tile (R / (64 * nkb_e))
    int n_early;       // edge units gathered while the partials are exchanged
    int sorder;        // physical edge stage of ring slot i: bits [4i, 4i+4)
    uint32_t pstage_bytes;  // HTILE + R * 128
    uint32_t estage_bytes;  // 2 * nkb_e * KB_OP
    uint32_t off_P, off_U, off_un, off_ids, off_bar;
    uint32_t red_stride;    // floats per row of the partial buffers (R + 4)
};

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

// One 16-byte chunk of a gathered A row (8 bf16) times 8 fp32 gate values:
// products in fp32 (round to nearest), each rounded once to bf16.
__device__ __forceinline__ uint4 gate_chunk(uint4 a, float4 u0, float4 u1) {
    const float2 p0 = __fmul2_rn(bf16x2_to_f2(a.x), make_float2(u0.x, u0.y));
    const float2 p1 = __fmul2_rn(bf16x2_to_f2(a.y), make_float2(u0.z, u0.w));
    const float2 p2 = __fmul2_rn(bf16x2_to_f2(a.z), make_float2(u1.x, u1.y));
    const float2 p3 = __fmul2_rn(bf16x2_to_f2(a.w), make_float2(u1.z, u1.w));
    uint4 g;
    g.x = f2_to_bf16x2(p0.x, p0.y);
    g.y = f2_to_bf16x2(p1.x, p1.y);
    g.z = f2_to_bf16x2(p2.x, p2.y);
    g.w = f2_to_bf16x2(p3.x, p3.y);
    return g;
}

__device__ __forceinline__ void mbar_inval(uint32_t bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// floor(e / d) for 0 <= e < 2^31, d >= 1, with m = floor((2^32 - 1) / d): the
// high half of e * m is the quotient or one less (one correction step).  The
// hardware has no integer divide; the compiler's division sequence sat on the
// critical path of the per-row loops below.
__device__ __forceinline__ int div_by(int e, int d, uint32_t m) {
    int q = (int)__umulhi((uint32_t)e, m);
    if (e - q * d >= d) ++q;
    return q;
}

// Number of transitions (s, i >= 1) whose target position lies before position q.
__device__ __forceinline__ int trans_before(int q, int n) {
    const int s = q / n;
    const int i = q - s * n;
    return s * (n - 1) + (i > 0 ? i - 1 : 0);
}

// EDGES_ONLY: u is an input; no projection and no exchange (clusters of one),
// every edge stage free from the start.
template <bool EDGES_ONLY>
__global__ void __launch_bounds__(SEL_THREADS, 1)
    select_fused_kernel(const __grid_constant__ CUtensorMap tmH,
                        const __grid_constant__ CUtensorMap tmW, const SelParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sE = smem_u32(smem);
    const uint32_t sP = sE + p.off_P;
    // receive area (region P from offset 0): [CS][own_max][R+4] fp32, slot src holds
    // CTA src's partial of this CTA's rows (its own partial at slot rank)
    float* uslice = reinterpret_cast<float*>(smem + p.off_U);                   // [own][R]
    float* unslice = reinterpret_cast<float*>(smem + p.off_un);                 // [own][K]
    int* id_ring = reinterpret_cast<int*>(smem + p.off_ids);                    // [2][256]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = full0 + 8 * p.pstages;
    const uint32_t accum = empty0 + 8 * p.pstages;
    const uint32_t recv = accum + 8;
    const uint32_t landed0 = recv + 8;  // [estages]: a unit's copies have landed
    const uint32_t sfree0 = landed0 + 8 * p.estages;
    const uint32_t tfull0 = sfree0 + 8 * p.estages;
    const uint32_t tempty0 = tfull0 + 16;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * p.pstages + 2 + 2 * p.estages + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int CS = p.CS;
    const int rank = (int)cluster_ctarank();
    const int cluster_id = blockIdx.x / CS;
    const int nclusters = gridDim.x / CS;
    const int K = p.K;
    const int R = p.R;
    const int TP = EROWS >> p.log2K;  // transitions per tile
    const int nm1 = p.n - 1;
    const int gtid = tid - 8 * 32;    // gather thread index (>= 0 in warps 8..15)
    const uint32_t row_bytes = p.red_stride * 4u;
    if (tid == 0) DF2_TRACE_AT(0);

    auto init_edge_bars = [&]() {
        for (int i = 0; i < p.estages; ++i) {
            mbar_init(landed0 + 8 * i, SEL_GTHREADS);
            mbar_init(sfree0 + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull0 + 8 * i, 1);
            mbar_init(tempty0 + 8 * i, 128);
        }
    };
    if (tid == 0) {
        if constexpr (!EDGES_ONLY) {
            prefetch_tmap(&tmH);
            prefetch_tmap(&tmW);
        }
        for (int i = 0; i < p.pstages; ++i) {
            mbar_init(full0 + 8 * i, 1);
            mbar_init(empty0 + 8 * i, 1);
        }
        mbar_init(accum, (uint32_t)p.nmma);
        mbar_init(recv, 1);
        init_edge_bars();
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent: the set-up above overlapped the
    // previous kernel; no input is read before it has completed.
    griddep_wait();
    griddep_launch_dependents();
    if (tid == 0) DF2_TRACE_AT(1);

    auto wait = [&](uint32_t bar, uint32_t parity) {
        if (*abort_flag) return;
        if (!mbar_wait_bounded(bar, parity, kWaitNs)) *abort_flag = 1;
    };
    auto estage_base = [&](int st) -> uint32_t {
        return st == 0 ? sE : sP + (uint32_t)(st - 1) * p.estage_bytes;
    };
    // ring slot i of the edge units -> physical stage (the stages clear of the
    // receive area come first, so they can be filled during the exchange)
    auto phys = [&](int i) -> int { return (p.sorder >> (4 * i)) & 15; };

    // A gather thread's place in an edge stage never changes: chunk ch (16 bytes)
    // of k-block kb of rows r0, r0 + row_step, ...; so the 128-byte swizzle of
    // its chunks is one constant (row_step is a multiple of 8).
    const int log2cpr = p.nkb_e == 2 ? 4 : 3;          // 16-byte chunks per row: 16 or 8
    const int g_r0 = gtid >> log2cpr;
    const int g_kb = (gtid >> 3) & (p.nkb_e - 1);
    const int g_ch = gtid & 7;
    const int row_step = SEL_GTHREADS >> log2cpr;      // 16 or 32
    const int g_col = g_kb * 64 + g_ch * 8;            // rank offset within the stage's ranks
    const uint32_t g_off = (uint32_t)(g_kb * KB_OP + g_r0 * 128 + ((g_ch ^ (g_r0 & 7)) << 4));

    bool bad = false;
    int pit = 0;  // projection k-block iterations so far (ring phase)
    int rbi = 0;  // row blocks so far (accumulator / receive phase)
    for (int rb = cluster_id; rb < p.nrb; rb += nclusters, ++rbi) {
        const int row0 = rb * p.MR;
        const int rows = min(p.MR, p.P - row0);
        const int kb0 = (int)((long long)rank * p.kblocks / CS);
        const int kb1 = (int)((long long)(rank + 1) * p.kblocks / CS);
        const int o_lo = rank * rows / CS;
        const int o_hi = (rank + 1) * rows / CS;
        const int pa = row0 + o_lo;  // this CTA's positions [pa, pb)
        const int pb = row0 + o_hi;
        const int e_lo = trans_before(pa, p.n);
        const int e_hi = trans_before(pb, p.n);
        const int ntile = (e_hi - e_lo + TP - 1) / TP;
        const int nunits = ntile * p.nhalf;

        // ---- raw id of tile t for this gather thread's slot g = gtid: g < 128 the
        //      predecessor id of row g (from position i-1), else the candidate id
        //      of row g-128; 0 for rows past the tile.  It is range-checked only
        //      where it is stored (checked_id), one tile later, so the load's
        //      latency never holds up a unit's copies.
        auto raw_id = [&](int t) -> int {
            if (t >= ntile) return 0;
            const int r = gtid & (EROWS - 1);
            const int e0 = e_lo + t * TP;
            if ((r >> p.log2K) >= min(TP, e_hi - e0)) return 0;
            const int e = e0 + (r >> p.log2K);
            const int s = div_by(e, nm1, p.nm1_magic);
            const int i = e - s * nm1 + 1 - (gtid < EROWS ? 1 : 0);
            return p.cand_ids[((size_t)s * p.n + i) * K + (r & (K - 1))];
        };
        int id_next = warp >= 8 ? raw_id(0) : 0;

        // ---- gather issue of edge unit j (tile j / nhalf, rank half j % nhalf).
        //      A new tile's ids go to slot t & 1 of the id ring; the named barrier
        //      makes them visible to all gather threads (and shows that the slot
        //      being overwritten, last read while issuing tile t - 2, has been
        //      read by all of them); the next tile's id is loaded after this
        //      unit's copies are issued.  The thread's arrive on landed[stage]
        //      fires once all its copies so far have completed.
        auto issue_unit = [&](int j) {
            const int use = div_by(j, p.estages, p.es_magic);  // uses of the stage so far
            const int st = phys(j - use * p.estages);
            const int t = j >> (p.nhalf - 1);                  // nhalf is 1 or 2
            const int half = j - t * p.nhalf;
            const int cnt = min(TP, e_hi - (e_lo + t * TP));
            int* ids = id_ring + (t & 1) * 2 * EROWS;
            if (half == 0) {
                ids[gtid] = checked_id(id_next, p.V, bad);
                named_bar_sync(1, SEL_GTHREADS);
            }
            if (j >= p.estages)  // the stage's previous unit has been consumed by the MMA
                wait(sfree0 + 8 * st, (uint32_t)(use - 1) & 1u);
            const int rows_valid = cnt << p.log2K;
            const uint32_t sb = estage_base(st) + g_off;
            const uint32_t sbB = sb + (uint32_t)(p.nkb_e * KB_OP);
            const int col = half * 64 * p.nkb_e + g_col;
            if (!*abort_flag) {
                // the unit's ids first (at most 8 rows per thread), then its copies
                int ia[8], ib[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int row = g_r0 + k * row_step;
                    ia[k] = row < rows_valid ? ids[row] : 0;
                    ib[k] = row < rows_valid ? ids[EROWS + row] : 0;
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int row = g_r0 + k * row_step;
                    if (row < rows_valid) {
                        const uint32_t o = (uint32_t)(k * row_step * 128);
                        cp_async16(sb + o, p.A + (size_t)ia[k] * R + col);
                        cp_async16(sbB + o, p.B + (size_t)ib[k] * R + col);
                    }
                }
            }
            if (gtid == 0 && j < 6) DF2_TRACE_RB(9 + j);
            cp_async_mbar_arrive_noinc(landed0 + 8 * st);
            if (half == p.nhalf - 1) id_next = raw_id(t + 1);
        };

        // ================= phase A: projection of the row block (+ early gathers)
        if constexpr (!EDGES_ONLY) {
            if (warp == 0 || warp == 8) {
                // TMA producers: warp 0 takes the even k-blocks, warp 8 (idle until the
                // gathers) the odd ones; each load instruction holds its issuing thread
                // for a while, so one thread alone falls behind the ring
                if (lane == 0) {
                    const uint32_t tx = (uint32_t)p.MR * 128u + (uint32_t)R * 128u;
                    for (int kb = kb0 + (warp == 8 ? 1 : 0); kb < kb1; kb += 2) {
                        const int it = pit + (kb - kb0);
                        const int use = div_by(it, p.pstages, p.ps_magic);
                        const int st = it - use * p.pstages;
                        wait(empty0 + 8 * st, ((uint32_t)use & 1u) ^ 1u);
                        if (*abort_flag) continue;
                        const uint32_t fb = full0 + 8 * st;
                        const uint32_t dst = sE + (uint32_t)st * p.pstage_bytes;
                        mbar_arrive_expect_tx(fb, tx);
                        tma_load_2d(dst, &tmH, fb, kb * 64, row0);
                        tma_load_2d(dst + HTILE, &tmW, fb, kb * 64, 0);
                    }
                }
                __syncwarp();
            } else if (warp <= p.nmma) {
                // MMA issuers: warp q + 1 takes k-blocks kb0 + q, kb0 + q + nmma, ... into
                // its own accumulator (columns q*R ..); one issuing thread alone spends
                // longer per k-block (waits, four MMAs, a commit) than the ring needs
                if (lane == 0) {
                    const int q = warp - 1;
                    const uint32_t idesc = idesc_bf16_f32(128, R);
                    const uint32_t dq = tmem + (uint32_t)(q * R);
                    for (int kb = kb0 + q; kb < kb1; kb += p.nmma) {
                        const int it = pit + (kb - kb0);
                        const int use = div_by(it, p.pstages, p.ps_magic);
                        const int st = it - use * p.pstages;
                        wait(full0 + 8 * st, (uint32_t)use & 1u);
                        tc_fence_after();
                        if (kb == kb0) DF2_TRACE_RB(2);
                        const uint32_t a0 = sE + (uint32_t)st * p.pstage_bytes;
                        const uint32_t b0 = a0 + HTILE;
                        if (!*abort_flag) {
    #pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc_mma_bf16(dq, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k),
                                            idesc, (kb > kb0 + q || k > 0) ? 1u : 0u);
                        }
                        tc_commit(empty0 + 8 * st);
                    }
                    tc_commit(accum); DF2_TRACE_RB(3 + 0 * q);  // every issuer arrives once, with or without k-blocks
                }
                __syncwarp();
            } else if (warp >= 8) {
            }
        }
        pit += kb1 - kb0;
        // the epilogue warps, idle until the partial is ready, stage the unary
        // scores of this CTA's own positions (read again per tile in phase D)
        if (warp >= 4 && warp < 8) {
            const int n4 = (o_hi - o_lo) * K / 4;
            const float4* src = reinterpret_cast<const float4*>(p.unary + (size_t)pa * K);
            for (int qd = tid - 128; qd < n4; qd += 128)
                reinterpret_cast<float4*>(unslice)[qd] = __ldg(src + qd);
        }

        if constexpr (EDGES_ONLY) {
            // u is the caller's: warps 0-7 copy this CTA's rows of it on chip while
            // the gather warps issue the first units (every edge stage is free)
            if (warp < 8) {
                const int l2c4 = p.log2R - 2;
                const int nq = (o_hi - o_lo) << l2c4;
                const uint32_t us_a = smem_u32(uslice);
                const float4* ug = reinterpret_cast<const float4*>(p.u + (size_t)pa * R);
                for (int qd = tid; qd < nq; qd += 256) {
                    const float4 v = __ldg(ug + qd);
                    st_shared_v4(us_a + (uint32_t)qd * 16u,
                                 make_uint4(__float_as_uint(v.x), __float_as_uint(v.y),
                                            __float_as_uint(v.z), __float_as_uint(v.w)));
                }
            } else {
                for (int jj = 0; jj < p.n_early && jj < nunits; ++jj) issue_unit(jj);
            }
        } else {
            // ================= phase B: one cluster barrier, then the split-d partials
            // The barrier shows every CTA of the cluster done with its projection
            // (its ring drained, so its receive area is free).  Warps 0-7 then move
            // the accumulators (summed in issuer order: deterministic) straight from
            // tensor memory to the owners of the rows: warp w takes lane quadrant
            // w % 4 and half of the columns; a row another CTA owns goes into that
            // CTA's receive slot with asynchronous remote stores (st.async) that
            // complete on its receive barrier, an own row into the own slot.  No
            // outgoing copy of the partial is kept, so the receive area is the only
            // exchange memory and the edge stages clear of it take the first units'
            // gathers meanwhile (warps 8-15).
            if (tid == 0 && CS > 1)
                mbar_arrive_expect_tx(recv, (uint32_t)(CS - 1) * (uint32_t)(o_hi - o_lo) * (uint32_t)R * 4u);
            wait(accum, (uint32_t)rbi & 1u);
        if (tid == 0) DF2_TRACE_RB(4);
            tc_fence_before();
            // the gather warps only arrive: their first units need this CTA's ring
            // drained (the accumulator barrier), not the rest of the cluster, so
            // they wait for the barrier after issuing them
            if (CS > 1) {
                if (warp < 8)
                    cluster_sync();
                else
                    cluster_arrive();
            } else {
                __syncthreads();
            }
            tc_fence_after();
        if (tid == 0) DF2_TRACE_RB(5);
            if (warp < 8) {
                const int q = warp & 3;
                const int cw = R >> 1;
                const int c_lo = (warp >> 2) * cw;
                const int row = q * 32 + lane;
                const int nacc = min(p.nmma, kb1 - kb0);  // accumulators that received MMAs
                // owner X of the row: X*rows/CS <= row < (X+1)*rows/CS
                int X = 0;
                while (X + 1 < CS && (X + 1) * rows < (row + 1) * CS) ++X;
                const int lr = row - X * rows / CS;
                const uint32_t dst = sP + ((uint32_t)(rank * p.own_max + lr)) * row_bytes;
                const uint32_t rdst = X == rank ? dst : map_cluster(dst, (uint32_t)X);
                const uint32_t rbar = map_cluster(recv, (uint32_t)X);
                for (int c0 = c_lo; c0 < c_lo + cw; c0 += 16) {
                    const uint32_t ta = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)c0;
                    float f[16];
                    {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(ta, v);
                        tmem_ld_wait();
    #pragma unroll
                        for (int jj = 0; jj < 16; ++jj) f[jj] = __uint_as_float(v[jj]);
                    }
                    for (int a = 1; a < nacc; ++a) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(ta + (uint32_t)(a * R), v);
                        tmem_ld_wait();
    #pragma unroll
                        for (int jj = 0; jj < 16; ++jj) f[jj] += __uint_as_float(v[jj]);
                    }
                    if (row < rows) {
    #pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const uint4 w4 = make_uint4(__float_as_uint(f[4 * jj]), __float_as_uint(f[4 * jj + 1]),
                                                        __float_as_uint(f[4 * jj + 2]), __float_as_uint(f[4 * jj + 3]));
                            const uint32_t off = (uint32_t)(c0 + 4 * jj) * 4u;
                            if (X == rank)
                                st_shared_v4(dst + off, w4);
                            else
                                st_async_v4(rdst + off, w4, rbar);
                        }
                    }
                }
                tc_fence_before();       // the accumulators are read before any later MMA
                named_bar_sync(3, 256);  // own rows in place
                // ================= phase C: the owner sums its rows' partials
                if (CS > 1) wait(recv, (uint32_t)rbi & 1u);
            if (tid == 0) DF2_TRACE_RB(6);
                // (row, 4-column group) items; R is a power of two, so no divides
                const int own = o_hi - o_lo;
                const int l2c4 = p.log2R - 2;
                const int nq = own << l2c4;
                const uint32_t us_a = smem_u32(uslice);
                for (int qd = tid; qd < nq; qd += 256) {
                    const int l = qd >> l2c4;
                    const uint32_t cb = (uint32_t)(qd & ((1 << l2c4) - 1)) * 16u;  // byte column
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    #pragma unroll 4
                    for (int src = 0; src < CS; ++src) {  // rank order: deterministic
                        const uint4 v = lds_v4(sP + (uint32_t)(src * p.own_max + l) * row_bytes + cb);
                        acc.x += __uint_as_float(v.x);
                        acc.y += __uint_as_float(v.y);
                        acc.z += __uint_as_float(v.z);
                        acc.w += __uint_as_float(v.w);
                    }
                    st_shared_v4(us_a + ((uint32_t)(l * R) << 2) + cb,
                                 make_uint4(__float_as_uint(acc.x), __float_as_uint(acc.y),
                                            __float_as_uint(acc.z), __float_as_uint(acc.w)));
                    *reinterpret_cast<float4*>(p.u + (size_t)(pa + l) * R + (cb >> 2)) = acc;
                }
            } else {
                // every MMA has read its stage: the edge stages clear of the receive
                // area are free, and the first units' rows are gathered meanwhile
                for (int jj = 0; jj < p.n_early && jj < nunits; ++jj) issue_unit(jj);
                if (CS > 1) cluster_wait();
            }
        }
        __syncthreads();  // u slice complete; the receive slots are free
        if (tid == 0) DF2_TRACE_RB(7);

        // ================= phase D: the edge tiles of this CTA's positions
        if (warp >= 8) {
            // gather: issue only; a stage is refilled once the MMA has consumed its
            // previous unit (the first n_early units were issued in phase B)
            for (int j = p.n_early; j < nunits; ++j) issue_unit(j);
            cp_async_wait_all();
            if (gtid == 0) DF2_TRACE_RB(8);
        } else if (warp < 4) {
            // gate: thread tid owns chunk column c of some of the unit's 32 four-row
            // groups (a row slot of cpr threads takes groups g_first, g_first +
            // g_step, ...); A (.) u in fp32, rounded to bf16, in place; proxy
            // fence; the named barrier shows the whole unit gated, and one thread
            // of warp 1 issues its MMAs.  Warp 1 gates one group per slot (the
            // last ones), so that it issues unit j's MMAs while warps 0, 2 and 3
            // gate unit j + 1 (wide workload 25.6 -> 24.1 us per call).
            const int cpr = 8 * p.nkb_e;
            const int c = tid & (cpr - 1);
            const int slot = tid >> log2cpr;
            const int S = 32 >> log2cpr;
            const int g_first = warp == 1 ? 32 - S + (slot - S) : (warp == 0 ? slot : slot - S);
            const int g_end = warp == 1 ? g_first + 1 : 32 - S;
            const int g_step = 3 * S;
            const int ch = c & 7;
            const uint32_t c_off = (uint32_t)((c >> 3) * KB_OP);
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            for (int j = 0; j < nunits; ++j) {
                const int use = div_by(j, p.estages, p.es_magic);
                const int st = phys(j - use * p.estages);
                const int t = j >> (p.nhalf - 1);
                const int half = j - t * p.nhalf;
                const int e0 = e_lo + t * TP;
                const int rows_valid = min(TP, e_hi - e0) << p.log2K;
                wait(landed0 + 8 * st, (uint32_t)use & 1u);
                if (tid == 0 && j < 6) DF2_TRACE_RB(15 + j);
                if (tid == 64 && j < 4) DF2_TRACE_RB(56 + j);
                const uint32_t sb = estage_base(st) + c_off;
                const int col = half * 64 * p.nkb_e + c * 8;
                if (!*abort_flag) {
                    // four rows at a time (independent chains, so the loads and the
                    // arithmetic of the four overlap); rows_valid is a multiple of
                    // K >= 4, so a group is either wholly valid or wholly past the
                    // end, and it lies within one transition
                    int tr_cur = -1;
                    float4 u0 = make_float4(0.f, 0.f, 0.f, 0.f);
                    float4 u1 = u0;
                    for (int g = g_first; g < g_end; g += g_step) {
                        const int row0 = 4 * g;
                        if (row0 >= rows_valid) break;
                        const int tr = row0 >> p.log2K;
                        if (tr != tr_cur) {  // this transition's u row (local to the CTA)
                            tr_cur = tr;
                            // transition e = s*(n-1) + i-1 scores position s*n + i = e + s + 1
                            const int e = e0 + tr;
                            const int lr = e + div_by(e, nm1, p.nm1_magic) + 1 - pa;
                            const uint32_t ua = smem_u32(uslice) + ((uint32_t)(lr * R + col) << 2);
                            const uint4 w0 = lds_v4(ua), w1 = lds_v4(ua + 16);
                            u0 = make_float4(__uint_as_float(w0.x), __uint_as_float(w0.y),
                                             __uint_as_float(w0.z), __uint_as_float(w0.w));
                            u1 = make_float4(__uint_as_float(w1.x), __uint_as_float(w1.y),
                                             __uint_as_float(w1.z), __uint_as_float(w1.w));
                        }
                        uint32_t off[4];
                        uint4 a[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int row = row0 + q;
                            off[q] = sb + (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) a[q] = lds_v4(off[q]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) st_shared_v4(off[q], gate_chunk(a[q], u0, u1));
                    }
                }
                fence_proxy_async_smem();
                named_bar_sync(2, 128);
                if (warp == 1) {
                    if (lane == 0) {  // MMA issue for unit j
                        const int bb = t & 1;
                        if (half == 0 && t >= 2) wait(tempty0 + 8 * bb, (((uint32_t)(t >> 1)) - 1u) & 1u);
                        tc_fence_after();
                        const uint32_t d = tmem + (uint32_t)(EACC + bb * 128);
                        const uint32_t sa = estage_base(st);
                        // the start-address field holds address / 16 and never
                        // carries (shared addresses < 2^18), so a descriptor for
                        // sa + off is the one for sa plus off / 16
                        const uint64_t da = sw128_desc(sa);
                        const uint64_t db = sw128_desc(sa + (uint32_t)(p.nkb_e * KB_OP));
                        if (!*abort_flag) {
                            for (int kb = 0; kb < p.nkb_e; ++kb)
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    const uint64_t step = (uint64_t)((kb * KB_OP + 32 * k) >> 4);
                                    tc_mma_bf16(d, da + step, db + step, idesc,
                                                (half > 0 || kb > 0 || k > 0) ? 1u : 0u);
                                }
                        }
                        tc_commit(sfree0 + 8 * st);
                        if (half == p.nhalf - 1) tc_commit(tfull0 + 8 * bb);
                        if (j < 6) DF2_TRACE_RB(21 + j);
                    }
                    __syncwarp();
                }
            }
        } else {
            // epilogue (warps 4-7): one thread per predecessor row of the tile; its
            // unary scores come from the staged slice
            const int ew = warp - 4;  // tensor-memory lane quadrant
            const int r = ew * 32 + lane;
            const int pslot = r & (K - 1);
            const int blk0 = r & ~(K - 1);
            const uint32_t lane_base = tmem + ((uint32_t)(ew * 32) << 16) + (uint32_t)EACC;
            for (int t = 0; t < ntile; ++t) {
                const int bb = t & 1;
                const int e0 = e_lo + t * TP;
                const int cnt = min(TP, e_hi - e0);
                const bool valid = (r >> p.log2K) < cnt;
                const int e = e0 + (r >> p.log2K);
                int s = 0, i = 1;
                if (valid) {
                    s = div_by(e, nm1, p.nm1_magic);
                    i = e - s * nm1 + 1;
                }
                // unary row of this transition's position (staged in phase A)
                const float* un = unslice + (size_t)(valid ? (s * p.n + i - pa) : 0) * K;
                float* erow = (p.edges_out != nullptr && valid)
                                  ? p.edges_out + ((size_t)e * K + pslot) * K
                                  : nullptr;
                const uint32_t acc_base = lane_base + (uint32_t)(bb * 128);
                float best = 0.f;
                int arg = -1;
                if (K >= 16) {
                    // the lane's own block in chunks of 16 slots (columns blk0 + 16 ch):
                    // no masking; for K = 16 the warp's two blocks come from one
                    // 32-column load and each lane keeps its half
                    const float4* un4 = reinterpret_cast<const float4*>(un);
                    float4 uq[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) uq[q] = un4[q];  // before the accumulator is ready
                    wait(tfull0 + 8 * bb, ((uint32_t)(t >> 1)) & 1u);
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < (K >> 4); ++ch) {
                        if (ch > 0) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) uq[q] = un4[4 * ch + q];
                        }
                        float ev[16];
                        if (K == 16) {
                            uint32_t v[32];
                            tmem_ld_32x32b_x32(acc_base + (uint32_t)(32 * ew), v);
                            tmem_ld_wait();
                            const bool hi = (lane & 16) != 0;
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                ev[jj] = __uint_as_float(hi ? v[16 + jj] : v[jj]);
                        } else {
                            uint32_t v[16];
                            tmem_ld_32x32b_x16(acc_base + (uint32_t)(blk0 + 16 * ch), v);
                            tmem_ld_wait();
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) ev[jj] = __uint_as_float(v[jj]);
                        }
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            ev[4 * q] += uq[q].x;
                            ev[4 * q + 1] += uq[q].y;
                            ev[4 * q + 2] += uq[q].z;
                            ev[4 * q + 3] += uq[q].w;
                        }
                        if (erow != nullptr) {  // the caller's buffer: no alignment assumed
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) erow[16 * ch + jj] = ev[jj];
                        }
                        // argmax by a tree over slot order: on equal values the left
                        // (lower) slot is kept, as in a scan with a strict ">"
                        int bi[16];
#pragma unroll
                        for (int jj = 0; jj < 16; ++jj) bi[jj] = 16 * ch + jj;
#pragma unroll
                        for (int w = 1; w < 16; w <<= 1)
#pragma unroll
                            for (int jj = 0; jj < 16; jj += 2 * w)
                                if (ev[jj + w] > ev[jj]) {
                                    ev[jj] = ev[jj + w];
                                    bi[jj] = bi[jj + w];
                                }
                        if (arg < 0 || ev[0] > best) {  // chunks come in slot order
                            best = ev[0];
                            arg = bi[0];
                        }
                    }
                } else {
                    // K = 4 or 8: a warp's 32 columns hold several blocks; each lane
                    // masks the slots outside its own
                    wait(tfull0 + 8 * bb, ((uint32_t)(t >> 1)) & 1u);
                    tc_fence_after();
#pragma unroll 1
                    for (int ch = 0; ch < 2; ++ch) {
                        uint32_t v[16];
                        tmem_ld_32x32b_x16(acc_base + (uint32_t)(32 * ew + ch * 16), v);
                        tmem_ld_wait();
                        const int c0 = 32 * ew + ch * 16 - blk0;  // slot of column jj = 0
                        if (valid && c0 + 16 > 0 && c0 < K) {
                            // every read in bounds (slot masked into the row), so the 16
                            // shared loads issue together; slots outside this lane's
                            // block are masked out of the argmax
                            float ev[16];
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj)
                                ev[jj] = __uint_as_float(v[jj]) + un[(c0 + jj) & (K - 1)];
                            if (erow != nullptr) {
#pragma unroll
                                for (int jj = 0; jj < 16; ++jj)
                                    if (c0 + jj >= 0 && c0 + jj < K) erow[c0 + jj] = ev[jj];
                            }
                            float bv[16];
                            int bi[16];
#pragma unroll
                            for (int jj = 0; jj < 16; ++jj) {
                                const bool in = c0 + jj >= 0 && c0 + jj < K;
                                bv[jj] = in ? ev[jj] : -INFINITY;
                                bi[jj] = in ? c0 + jj : K;
                            }
#pragma unroll
                            for (int w = 1; w < 16; w <<= 1)
#pragma unroll
                                for (int jj = 0; jj < 16; jj += 2 * w)
                                    if (bv[jj + w] > bv[jj] || (bi[jj] == K && bi[jj + w] < K)) {
                                        bv[jj] = bv[jj + w];
                                        bi[jj] = bi[jj + w];
                                    }
                            if (arg < 0 || bv[0] > best) {  // chunks come in slot order
                                best = bv[0];
                                arg = bi[0];
                            }
                        }
                    }
                }
                if (valid) {
                    p.best_slot[(size_t)e * K + pslot] = arg;
                    p.best_score[(size_t)e * K + pslot] = best;
                }
                tc_fence_before();
                if (tid == 128 && t < 4) DF2_TRACE_RB(27 + t);
                mbar_arrive(tempty0 + 8 * bb);
            }
        }
        // End of the row block: every edge MMA has completed (the epilogue saw
        // its last accumulator), every copy into region E / P has landed and the
        // outgoing partial has been read by its owners, so the next row block may
        // reuse all of shared memory.  The edge barriers restart from phase 0.
        tc_fence_before();
        __syncthreads();
        if (rb + nclusters < p.nrb) {
            if (tid == 0) {
                for (int i = 0; i < p.estages; ++i) {
                    mbar_inval(landed0 + 8 * i);
                    mbar_inval(sfree0 + 8 * i);
                }
                for (int i = 0; i < 2; ++i) {
                    mbar_inval(tfull0 + 8 * i);
                    mbar_inval(tempty0 + 8 * i);
                }
                init_edge_bars();
                fence_mbar_init();
            }
            __syncthreads();
        }
        tc_fence_after();
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0) DF2_TRACE_AT(31);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (bad && p.err_flag != nullptr) atomicOr(p.err_flag, DF2_FLAG_BAD_ID);
    if (tid == 0 && *abort_flag) {
        if (p.err_flag != nullptr) atomicOr(p.err_flag, DF2_FLAG_TIMEOUT);
        atomicOr(&g_select_fault, (unsigned)DF2_FLAG_TIMEOUT);
    }
}

// ---------------------------------------------------------------- planning

struct PlanKey {
    int P, d, R, K, n, sms;
    bool operator==(const PlanKey& o) const { return std::memcmp(this, &o, sizeof(*this)) == 0; }
};

struct Plan {
    bool ok = false;
    int CS = 0, NC = 0, MR = 0, nrb = 0, own_max = 0, pstages = 0, estages = 0, nkb_e = 0, nhalf = 0;
    int n_early = 0, sorder = 0;
    uint32_t pstage_bytes = 0, estage_bytes = 0, off_P = 0, off_U = 0, off_un = 0;
    uint32_t off_ids = 0, off_bar = 0, red_stride = 0;
    size_t smem = 0;
};

std::mutex g_plan_mu;
constexpr int kPlanCache = 16;
PlanKey g_plan_keys[kPlanCache];
Plan g_plans[kPlanCache];
int g_plan_count = 0;
int g_plan_next = 0;

// Shared-memory layout for a cluster size and row-block height; false when it
// does not fit.  Region E = edge stage 0.  Region P = the receive area
// [CS][own_max] (rows of R + 4 floats) from offset 0, and edge stages
// 1..estages-1.  The projection's TMA ring spans regions E and P (it is drained
// before either is used).  Then the u slice, the unary slice, the id ring and
// the barriers.  The edge ring visits stage 0 and the region-P stages clear of
// the receive area first: those take units while the partials are exchanged.
bool layout(int R, int K, int CS, int MR, size_t max_smem, Plan* q) {
    q->nkb_e = R >= 128 ? 2 : 1;
    q->nhalf = R / (64 * q->nkb_e);
    q->estage_bytes = 2u * (uint32_t)q->nkb_e * KB_OP;
    q->pstage_bytes = (uint32_t)HTILE + (uint32_t)R * 128u;
    q->red_stride = (uint32_t)R + 4u;
    q->own_max = (MR + CS - 1) / CS;
    const size_t row_bytes = (size_t)q->red_stride * 4;
    const size_t recv_bytes = (size_t)CS * q->own_max * row_bytes;
    const size_t u_bytes = (size_t)q->own_max * R * 4;
    const size_t un_bytes = (size_t)q->own_max * K * 4;
    const size_t bar_bytes = 8 * (2 * 8 + 2 + 2 * 4 + 4) + 16;
    // Region P holds the receive area, then edge stages 1 .. es-1; the
    // projection's TMA ring (phase A only) spans regions E and P from offset 0.
    for (int es = 4; es >= 2; --es) {
        const size_t regionP =
            std::max((recv_bytes + 1023) & ~(size_t)1023, (size_t)(es - 1) * q->estage_bytes);
        const size_t off_U = q->estage_bytes + regionP;
        const int ps = (int)std::min<size_t>(6, off_U / q->pstage_bytes);
        const size_t off_un = off_U + ((u_bytes + 15) & ~(size_t)15);
        const size_t off_ids = off_un + ((un_bytes + 15) & ~(size_t)15);
        const size_t off_bar = off_ids + 2 * 2 * EROWS * 4;
        const size_t total = 1024 + off_bar + bar_bytes;
        if (total <= max_smem && ps >= 2) {
            q->pstages = ps;
            q->estages = es;
            q->off_P = q->estage_bytes;
            q->off_U = (uint32_t)off_U;
            q->off_un = (uint32_t)off_un;
            q->off_ids = (uint32_t)off_ids;
            q->off_bar = (uint32_t)off_bar;
            // ring order: stage 0, the region-P stages that start at or past the end
            // of the receive area, then the others
            int order[4], n = 0;
            order[n++] = 0;
            for (int st = 1; st < es; ++st)
                if ((size_t)(st - 1) * q->estage_bytes >= recv_bytes) order[n++] = st;
            q->n_early = n;
            for (int st = 1; st < es; ++st)
                if ((size_t)(st - 1) * q->estage_bytes < recv_bytes) order[n++] = st;
            q->sorder = 0;
            for (int i = 0; i < es; ++i) q->sorder |= order[i] << (4 * i);
            q->smem = total;
            return true;
        }
    }
    return false;
}

int max_active_clusters(int CS, size_t smem) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)CS);
    cfg.blockDim = dim3(SEL_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    bool ok = cudaFuncSetAttribute(select_fused_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)smem) == cudaSuccess;
    if (ok && CS > 8)
        ok = cudaFuncSetAttribute(select_fused_kernel<false>,
                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    if (ok) ok = cudaOccupancyMaxActiveClusters(&n, select_fused_kernel<false>, &cfg) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();  // an unsupported cluster size is not an error of the call
        return 0;
    }
    return n;
}

// Dynamic shared memory every launch requests at least: more than half of an
// SM's, so that no two CTAs share an SM.  Each CTA takes all 512 tensor-memory
// columns; two CTAs of one cluster on one SM would otherwise wait for each
// other (one in tcgen05.alloc, the other at the cluster barrier).
constexpr size_t kMinSmem = 120 * 1024;

// Picks the cluster size and row-block height with the least modelled time per
// CTA, times the number of waves of row blocks: the HBM bytes of h and of the
// gathered rows; the L2-served slice of W at half their weight; and the
// partials the CTA receives through distributed shared memory at 2.7 times
// their weight (its remote stores run at about 15 GB/s per SM against about
// 41 GB/s for the gathers).  Weights fitted to cluster-size sweeps on GB300:
// batched 256 x 16 (CS 4 best), wide 64 x 8 with R = 256 (CS 6-8 best, 16
// 15 % slower), one draft block (CS 16 best).
Plan make_plan(int P, int d, int R, int K, int n, int sms, size_t max_smem) {
    Plan best;
    double best_cost = 0;
    const int kblocks = (d + 63) / 64;
    const double E_per_pos = (double)(n - 1) / n;
    for (int CS = 1; CS <= 16; ++CS) {
        if (CS > 8 && CS != 16) continue;
        if (kblocks < CS) break;
        const int ncmax = std::min(sms / CS, max_active_clusters(CS, std::max(kMinSmem, (size_t)160 * 1024)));
        if (ncmax < 1) continue;
        // the largest row block whose layout fits (owned rows <= 32)
        int mr_fit = std::min(128, 32 * CS);
        Plan probe;
        while (mr_fit > 0 && !layout(R, K, CS, mr_fit, max_smem, &probe)) --mr_fit;
        if (mr_fit == 0) continue;
        // a row block per cluster when the rows allow it, else waves of full blocks
        const int MR = std::min(mr_fit, (P + ncmax - 1) / ncmax);
        const int nrb = (P + MR - 1) / MR;
        const int NC = std::min(ncmax, nrb);
        const int waves = (nrb + NC - 1) / NC;
        Plan q;
        if (!layout(R, K, CS, MR, max_smem, &q)) continue;
        const double kpc = (double)kblocks / CS;
        const double h_b = MR * kpc * 128.0;
        const double w_b = R * kpc * 128.0;
        const double g_b = (double)q.own_max * E_per_pos * 2.0 * K * R * 2.0;
        const double x_b = (double)(CS - 1) * q.own_max * R * 4.0;
        const double cost = waves * (h_b + g_b + 0.5 * w_b + 2.7 * x_b) + 1e-3 * NC * CS;
        if (!best.ok || cost < best_cost) {
            best = q;
            best.ok = true;
            best.CS = CS;
            best.NC = NC;
            best.MR = MR;
            best.nrb = nrb;
            best_cost = cost;
        }
    }
    if (best.ok && best.smem < kMinSmem) best.smem = kMinSmem;
    return best;
}

// Edges only (u given): one CTA per cluster, rows cut so that every SM gets a
// row block (at most 128 rows, fewer if the layout needs it), every edge stage
// free from the start.
Plan make_edges_plan(int P, int R, int K, int sms, size_t max_smem) {
    Plan best;
    int MR = std::min(128, (P + sms - 1) / sms);
    Plan q;
    while (MR > 0 && !layout(R, K, 1, MR, max_smem, &q)) --MR;
    if (MR == 0) return best;
    best = q;
    best.ok = true;
    best.CS = 1;
    best.MR = MR;
    best.nrb = (P + MR - 1) / MR;
    best.NC = std::min(best.nrb, sms);
    best.n_early = best.estages;
    best.sorder = 0;
    for (int i = 0; i < best.estages; ++i) best.sorder |= i << (4 * i);
    if (best.smem < kMinSmem) best.smem = kMinSmem;
    return best;
}

// d = 0 keys the edges-only plans (a projection always has d > 0).
Plan get_plan(int P, int d, int R, int K, int n, int sms, size_t max_smem) {
    const PlanKey key{P, d, R, K, n, sms};
    std::lock_guard<std::mutex> lk(g_plan_mu);
    for (int i = 0; i < g_plan_count; ++i)
        if (g_plan_keys[i] == key) return g_plans[i];
    const Plan pl = d == 0 ? make_edges_plan(P, R, K, sms, max_smem)
                           : make_plan(P, d, R, K, n, sms, max_smem);
    const int slot = g_plan_count < kPlanCache ? g_plan_count++ : (g_plan_next++ % kPlanCache);
    g_plan_keys[slot] = key;
    g_plans[slot] = pl;
    return pl;
}

}  // namespace

bool select_fused_supported(int K, int R, int d, int n) {
    return K >= 4 && K <= 128 && (K & (K - 1)) == 0 && (R == 64 || R == 128 || R == 256) &&
           d % 8 == 0 && n >= 2;
}

namespace {

// Launches the kernel for a plan: the fused selector (tensor maps of h and W),
// or with edges_only the edge phase alone on the caller's u (maps unused).
cudaError_t launch_plan(const SelectArgs& a, const Plan& pl, const CUtensorMap& tmH,
                        const CUtensorMap& tmW, int edges_only, cudaStream_t stream) {
    const int P = a.S * a.n;
    SelParams p{};
    p.cand_ids = a.cand_ids;
    p.unary = a.unary;
    p.A = static_cast<const __nv_bfloat16*>(a.A);
    p.B = static_cast<const __nv_bfloat16*>(a.B);
    p.u = a.u;
    p.edges_out = a.edges_out;
    p.best_slot = a.best_slot;
    p.best_score = a.best_score;
    p.err_flag = a.err_flag;
    p.S = a.S;
    p.n = a.n;
    p.K = a.K;
    p.R = a.R;
    p.V = a.V;
    p.P = P;
    int l2 = 0;
    while ((1 << l2) < a.K) ++l2;
    p.log2K = l2;
    int lr2 = 0;
    while ((1 << lr2) < a.R) ++lr2;
    p.log2R = lr2;
    p.nm1_magic = 0xFFFFFFFFu / (uint32_t)(a.n - 1);  // n >= 2 on this path
    p.ps_magic = 0xFFFFFFFFu / (uint32_t)pl.pstages;
    p.es_magic = 0xFFFFFFFFu / (uint32_t)pl.estages;
    p.CS = pl.CS;
    p.MR = pl.MR;
    p.nrb = pl.nrb;
    p.kblocks = (a.d + 63) / 64;
    p.own_max = pl.own_max;
    p.pstages = pl.pstages;
    // three issuers where their accumulators fit in the 512 tensor-memory columns
    // (R = 64, 128: three; R = 256: two); the projection's accumulators are drained
    // before the edge accumulators (columns EACC ..) are first written
    p.nmma = std::min(3, 512 / a.R);
    p.estages = pl.estages;
    p.nkb_e = pl.nkb_e;
    p.nhalf = pl.nhalf;
    p.pstage_bytes = pl.pstage_bytes;
    p.estage_bytes = pl.estage_bytes;
    p.off_P = pl.off_P;
    p.off_U = pl.off_U;
    p.off_un = pl.off_un;
    p.off_ids = pl.off_ids;
    p.off_bar = pl.off_bar;
    p.n_early = pl.n_early;
    p.sorder = pl.sorder;
    p.red_stride = pl.red_stride;
    auto kern = edges_only ? select_fused_kernel<true> : select_fused_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem);
    if (e != cudaSuccess) return e;
    if (pl.CS > 8) {
        e = cudaFuncSetAttribute(kern,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(pl.NC * pl.CS));
    cfg.blockDim = dim3(SEL_THREADS);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pl.CS > 1 ? attr : attr + 1;  // no cluster attribute for clusters of one
    cfg.numAttrs = pl.CS > 1 ? 2 : 1;
    e = cudaLaunchKernelEx(&cfg, kern, tmH, tmW, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select_fused(const SelectArgs& a, cudaStream_t stream, int num_sms,
                                size_t max_smem, bool* launched) {
    *launched = false;
    const int P = a.S * a.n;
    const Plan pl = get_plan(P, a.d, a.R, a.K, a.n, num_sms, max_smem);
    if (!pl.ok) return cudaSuccess;  // the caller falls back to the two-kernel path
    CUtensorMap tmH, tmW;
    if (!make_tmap_rows_bf16(&tmH, a.h, P, a.d, pl.MR) ||
        !make_tmap_rows_bf16(&tmW, a.W, a.R, a.d, a.R))
        return cudaErrorInvalidValue;
    const cudaError_t e = launch_plan(a, pl, tmH, tmW, 0, stream);
    if (e == cudaSuccess) *launched = true;
    return e;
}

cudaError_t launch_select_edges(const EdgesArgs& ea, cudaStream_t stream, int num_sms,
                                size_t max_smem, bool* launched) {
    *launched = false;
    if (!select_fused_supported(ea.K, ea.R, 8, ea.n)) return cudaSuccess;
    const int P = ea.S * ea.n;
    const Plan pl = get_plan(P, 0, ea.R, ea.K, ea.n, num_sms, max_smem);
    if (!pl.ok) return cudaSuccess;
    SelectArgs a{nullptr, nullptr, ea.cand_ids, ea.A, ea.B, ea.unary, ea.S, ea.n, 0, ea.K,
                 ea.R, ea.V, const_cast<float*>(ea.u), ea.edges_out, ea.best_slot,
                 ea.best_score, ea.err_flag};
    const CUtensorMap none{};  // never read in edges-only mode
    const cudaError_t e = launch_plan(a, pl, none, none, 1, stream);
    if (e == cudaSuccess) *launched = true;
    return e;
}

bool select_fused_plan(int S, int n, int d, int K, int R, int num_sms, size_t max_smem,
                       int* cluster_size, int* clusters, int* rows_per_block) {
    if (!select_fused_supported(K, R, d, n)) return false;
    const Plan pl = get_plan(S * n, d, R, K, n, num_sms, max_smem);
    if (!pl.ok) return false;
    *cluster_size = pl.CS;
    *clusters = pl.NC;
    *rows_per_block = pl.MR;
    return true;
}

cudaError_t take_select_faults(unsigned* flags) {
    unsigned v = 0;
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_select_fault, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_select_fault, &zero, sizeof(zero));
    *flags = v;
    return e;
}

}  // namespace df2

extern "C" int dflash2_trace_read(uint64_t* host, int bytes, int clear) {
#ifdef DF2_TRACE
    if (host == nullptr || bytes < 0 || (size_t)bytes > sizeof(df2::g_trace))
        return DF2_ERR_INVALID_ARG;
    if (cudaMemcpyFromSymbol(host, df2::g_trace, (size_t)bytes) != cudaSuccess) return DF2_ERR_CUDA;
    if (clear) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, df2::g_trace) != cudaSuccess ||
            cudaMemset(a, 0, sizeof(df2::g_trace)) != cudaSuccess)
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
