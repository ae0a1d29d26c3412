// project(h): u = h W^T, the dense d -> R projection of each position's hidden
// state (ggml-org/llama.cpp PR #27342, "spec : add DFlash2 support (local
// convolution + candidate selector)", Overview: the position's hidden state is
// projected to the codebook rank; weight tensor "selector_hidden").
//
// bf16 path (tcgen05, one GB300 SM per CTA):
//  - output tile 128 (rows of h) x 128 (columns of u) accumulated in fp32 in
//    tensor memory (128 TMEM columns);
//  - K (= d) is split across the CTAs of a thread-block cluster (split-K);
//    every CTA streams its K range through a 6-stage TMA pipeline of
//    128x64 bf16 tiles of h and W, stored in the 128-byte-swizzle K-major
//    layout that the tensor core reads directly;
//  - two producer threads (warps 0 and 2) drive TMA for the even and the odd
//    k-blocks, and two issuing threads (warps 1 and 3) issue tcgen05.mma
//    (M=128, N=128, K=16) for them into two accumulators, freeing each stage
//    with tcgen05.commit; a single thread issuing loads or MMAs for every
//    k-block is slower per k-block than the TMA ring;
//  - epilogue: tcgen05.ld of both accumulators (summed, even + odd) and of the
//    partial tile into the CTA's shared memory,
//    a cluster barrier, then CTA r sums rows [r*128/split, (r+1)*128/split)
//    over all CTAs of the cluster through distributed shared memory in a
//    fixed order (deterministic) and writes fp32 u.  No global workspace.
// The thin-N GEMM (R = 128..256) is HBM-bound on h when h is cold, so the
// pipeline is sized for bandwidth, not for tensor throughput.
//
// fp32 path: a shared-memory tiled FFMA kernel (exact fp32, no TF32).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cuda_bf16.h>

#include "dflash2.h"
#include "common.cuh"
#include "ptx.cuh"

namespace df2 {

// Device-side fault word of the projection kernel (one per device): DF2_FLAG_*
// bits are ORed here when a bounded wait gives up.
__device__ unsigned int g_fault_word = 0;

namespace {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 64;  // 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int RED_STRIDE = BN + 4;  // padded fp32 row of the reduction buffer
constexpr int NTHREADS = 128;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
// partial tile plus up to 7 receive slots of 16 rows (split 8) or 1 slot of 64 rows (split 2)
static_assert((size_t)BM * RED_STRIDE * 4 * 2 <= (size_t)STAGES * STAGE_BYTES, "reduction buffer");

struct ProjParams {
    float* u;
    __nv_bfloat16* ub;  // when set, the output is written here in bf16 (round to nearest even)
    int P, R;
    int kblocks;
    int splitk;
    // Optional split-K workspace [tiles][SPLIT][128][BN] fp32; nullptr selects the
    // reduction through distributed shared memory.
    float* ws;
};

// Stores four consecutive outputs (fp32, or bf16 when the bf16 output is set).
__device__ __forceinline__ void store_out4(const ProjParams& p, size_t off, float4 v) {
    if (p.ub != nullptr) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&lo);
        w.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(p.ub + off) = w;
    } else {
        *reinterpret_cast<float4*>(p.u + off) = v;
    }
}

// SMEM_BYTES of a kernel instance with N tile BNT (4 stages for 256 columns).
constexpr size_t smem_bytes_for(int BNT) {
    return 1024 + (size_t)(BNT == 256 ? 4 : STAGES) * (A_BYTES + BNT * BK * 2) + 256;
}

// BNT = 256 (one instruction of N = 256, 4 stages) only with SPLIT = 1: for
// outputs wider than 128 columns on grids that fill the GPU without split-K,
// where it halves how often each tile of h is read from L2.
template <int SPLIT, int BNT = 128>
__global__ void __launch_bounds__(NTHREADS, 1)
    project_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const ProjParams p) {
    static_assert(BNT == 128 || (BNT == 256 && SPLIT == 1), "256-column tiles without split-K only");
    constexpr int BN = BNT;
    constexpr int STAGES = BNT == 256 ? 4 : ::df2::STAGES;
    constexpr int STAGE_BYTES = A_BYTES + BN * BK * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* stages = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)STAGES * STAGE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2);
    const uint32_t full0 = smem_u32(bars);
    const uint32_t empty0 = smem_u32(bars + STAGES);
    const uint32_t accum = smem_u32(bars + 2 * STAGES);
    const uint32_t recv = smem_u32(bars + 2 * STAGES + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int m_tile = blockIdx.y;
    const int n_tile = blockIdx.z;
    const int kb0 = (int)((long long)rank * p.kblocks / SPLIT);
    const int kb1 = (int)((long long)(rank + 1) * p.kblocks / SPLIT);
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        mbar_init(accum, 2);  // one commit from each MMA issuer
        mbar_init(recv, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 2 * BN);  // even and odd k-block accumulators
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    // Launched as a programmatic dependent: the set-up above overlapped the
    // previous kernel; h and W are read only after it has completed.
    griddep_wait();
    griddep_launch_dependents();

    if ((warp == 0 || warp == 2) && lane == 0) {
        // TMA producers: warp 0 loads the even k-blocks, warp 2 the odd ones
        for (int it = warp >> 1; it < nkb; it += 2) {
            const int s = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            if (!mbar_wait_bounded(empty0 + 8 * s, ph ^ 1u, kWaitNs)) {
                ok = false;
                break;
            }
            const uint32_t fb = full0 + 8 * s;
            mbar_arrive_expect_tx(fb, STAGE_BYTES);
            const uint32_t dst = smem_u32(stages + (size_t)s * STAGE_BYTES);
            const int kx = (kb0 + it) * BK;
            tma_load_2d(dst, &tmA, fb, kx, m_tile * BM);
            tma_load_2d(dst + A_BYTES, &tmB, fb, kx, n_tile * BN);
        }
    } else if ((warp == 1 || warp == 3) && lane == 0) {
        // MMA issuers: warp 1 the even k-blocks into columns [0, BN), warp 3 the
        // odd ones into [BN, 2 BN)
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
        const int q = warp >> 1;
        const uint32_t dq = tmem + (uint32_t)(q * BN);
        for (int it = q; it < nkb; it += 2) {
            const int s = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            if (!mbar_wait_bounded(full0 + 8 * s, ph, kWaitNs)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(stages + (size_t)s * STAGE_BYTES);
            const uint32_t b0 = a0 + A_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
                tc_mma_bf16(dq, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k), idesc,
                            (it > q || k > 0) ? 1u : 0u);
            tc_commit(empty0 + 8 * s);
        }
        tc_commit(accum);  // arrives even when this issuer had no k-block
    }
    __syncwarp();

    // Epilogue.  The accumulator barrier fires once every issued load has been
    // consumed by an MMA, so the stage buffers are free for the reduction.
    if (!mbar_wait_bounded(accum, 0, kWaitNs)) ok = false;
    tc_fence_after();
    const int row = warp * 32 + lane;
    // 32 columns of this thread's row: the even accumulator plus the odd one (in
    // that order; the odd one is empty when there is a single k-block)
    auto load_acc = [&](int c0, float (&f)[32]) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
        if (nkb > 1) {
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(BN + c0), v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] += __uint_as_float(v[j]);
        }
    };
    if constexpr (SPLIT == 1) {
        // no split: each thread writes its own row straight from TMEM
        const int grow = m_tile * BM + row;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float f[32];
            load_acc(c0, f);
            const int gcol = n_tile * BN + c0;
            if (grow < p.P) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (gcol + 4 * j < p.R)
                        store_out4(p, (size_t)grow * p.R + gcol + 4 * j,
                                   make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]));
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 2 * BN);
        }
    } else if (p.ws != nullptr) {
        // Split-K reduction through an L2-resident workspace.  CTA r of the
        // cluster owns rows [r*RP, (r+1)*RP).  Every CTA stages its partial tile
        // in shared memory, writes the slices the other CTAs own to its slot of
        // the workspace, and after one cluster barrier each owner sums the SPLIT
        // slices in rank order (deterministic): its own from shared memory, the
        // others from the workspace.
        constexpr int RP = BM / SPLIT;
        float* red = reinterpret_cast<float*>(stages);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float f[32];
            load_acc(c0, f);
            float4* dst = reinterpret_cast<float4*>(red + (size_t)row * RED_STRIDE + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
        }
        __syncthreads();
        const size_t tile = (size_t)m_tile * gridDim.z + n_tile;
        float* wsl = p.ws + (tile * SPLIT + rank) * (size_t)BM * BN;  // this CTA's slot
        for (int q = threadIdx.x; q < BM * (BN / 4); q += NTHREADS) {
            const int rr = q / (BN / 4);
            if (rr / RP == (int)rank) continue;  // own rows stay in shared memory
            const int cc = (q % (BN / 4)) * 4;
            *reinterpret_cast<float4*>(wsl + (size_t)rr * BN + cc) =
                *reinterpret_cast<const float4*>(red + (size_t)rr * RED_STRIDE + cc);
        }
        tc_fence_before();
        cluster_sync();  // every slice is written (release/acquire across the cluster)
        const int r_base = (int)rank * RP;
        for (int q = threadIdx.x; q < RP * (BN / 4); q += NTHREADS) {
            const int rr = r_base + q / (BN / 4);
            const int cc = (q % (BN / 4)) * 4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int src = 0; src < SPLIT; ++src) {
                const float4 v =
                    src == (int)rank
                        ? *reinterpret_cast<const float4*>(red + (size_t)rr * RED_STRIDE + cc)
                        : __ldcg(reinterpret_cast<const float4*>(
                              p.ws + ((tile * SPLIT + src) * BM + rr) * (size_t)BN + cc));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int grow = m_tile * BM + rr;
            const int gcol = n_tile * BN + cc;
            if (grow < p.P && gcol < p.R)
                store_out4(p, (size_t)grow * p.R + gcol, acc);
        }
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 2 * BN);
        }
    } else {
        // Split-K reduction through distributed shared memory.  CTA r of the
        // cluster owns rows [r*RP, (r+1)*RP), RP = 128/SPLIT.  Every CTA writes
        // its partial tile (padded rows) to its own shared memory, then pushes
        // each owner's row slice into that owner's receive slot with one bulk
        // shared-to-shared copy; each owner sums the SPLIT slices in rank order
        // (deterministic) and stores its rows of u.
        constexpr int RP = BM / SPLIT;
        constexpr uint32_t SLICE = (uint32_t)RP * RED_STRIDE * 4;
        float* red = reinterpret_cast<float*>(stages);
        const uint32_t red_s = smem_u32(red);
        const uint32_t recv_s = red_s + (uint32_t)BM * RED_STRIDE * 4;  // SPLIT-1 slots
        if (threadIdx.x == 0) mbar_arrive_expect_tx(recv, (SPLIT - 1) * SLICE);
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
            float f[32];
            load_acc(c0, f);
            float4* dst = reinterpret_cast<float4*>(red + (size_t)row * RED_STRIDE + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(f[4 * j], f[4 * j + 1], f[4 * j + 2], f[4 * j + 3]);
        }
        fence_proxy_async_smem();  // partial tile -> visible to the copy engine
        tc_fence_before();
        cluster_sync();            // every CTA's mainloop is done: receive slots are free
        if (threadIdx.x < SPLIT && threadIdx.x != rank) {
            const uint32_t dst_rank = threadIdx.x;
            const uint32_t slot = rank < dst_rank ? rank : rank - 1;
            bulk_s2cluster(map_cluster(recv_s + slot * SLICE, dst_rank),
                           red_s + dst_rank * SLICE, SLICE, map_cluster(recv, dst_rank));
        }
        if (!mbar_wait_bounded(recv, 0, kWaitNs)) ok = false;

        const int r_base = (int)rank * RP;
        for (int q = threadIdx.x; q < RP * (BN / 4); q += NTHREADS) {
            const int rr = q / (BN / 4);
            const int cc = (q % (BN / 4)) * 4;
            const uint32_t eoff = (uint32_t)((rr * RED_STRIDE + cc) * 4);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int src = 0; src < SPLIT; ++src) {
                const uint32_t a = src == (int)rank
                                       ? red_s + (uint32_t)r_base * RED_STRIDE * 4 + eoff
                                       : recv_s + (uint32_t)(src < (int)rank ? src : src - 1) * SLICE + eoff;
                float4 v;
                asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                             : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                             : "r"(a));
                acc.x += v.x;
                acc.y += v.y;
                acc.z += v.z;
                acc.w += v.w;
            }
            const int grow = m_tile * BM + r_base + rr;
            const int gcol = n_tile * BN + cc;
            if (grow < p.P && gcol < p.R)
                store_out4(p, (size_t)grow * p.R + gcol, acc);
        }
        cluster_sync();  // the slices this CTA sent have all been received
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 2 * BN);
        }
    }
    if (!ok) atomicOr(&g_fault_word, (unsigned)DF2_FLAG_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

}  // namespace

// 2-D bf16 tensor [rows, cols] (cols contiguous), box [box_rows, 64], 128 B swizzle.
bool make_tmap_rows_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

// ---------------------------------------------------------------- fp32 path

constexpr int FT = 16;  // 16x16 outputs per block, K chunks of 32

__global__ void __launch_bounds__(256) project_f32_kernel(const float* __restrict__ h,
                                                          const float* __restrict__ W,
                                                          float* __restrict__ u, int P, int d,
                                                          int R) {
    __shared__ float hs[FT][33];
    __shared__ float ws[FT][33];
    const int tx = threadIdx.x % FT;  // output column within the tile
    const int ty = threadIdx.x / FT;  // output row within the tile
    const int r0 = blockIdx.y * FT;
    const int k0 = blockIdx.x * FT;
    float acc = 0.f;
    for (int j0 = 0; j0 < d; j0 += 32) {
        for (int q = threadIdx.x; q < FT * 32; q += 256) {
            const int rr = q / 32, jj = q % 32;
            const int j = j0 + jj;
            hs[rr][jj] = (r0 + rr < P && j < d) ? h[(size_t)(r0 + rr) * d + j] : 0.f;
            ws[rr][jj] = (k0 + rr < R && j < d) ? W[(size_t)(k0 + rr) * d + j] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) acc = fmaf(hs[ty][jj], ws[tx][jj], acc);
        __syncthreads();
    }
    if (r0 + ty < P && k0 + tx < R) u[(size_t)(r0 + ty) * R + k0 + tx] = acc;
}

}  // namespace

size_t project_workspace_bytes(int P, int d, int R, int num_sms) {
    const int kblocks = (d + BK - 1) / BK;
    const int m_tiles = (P + BM - 1) / BM;
    const int n_tiles = (R + BN - 1) / BN;
    const int tiles = m_tiles * n_tiles;
    int split = 1;
    while (split < 8 && tiles * split * 2 <= num_sms && kblocks >= split * 4) split *= 2;
    return split == 1 ? 0 : (size_t)tiles * split * BM * BN * sizeof(float);
}

cudaError_t launch_project_bf16_tc(const ProjectArgs& a, cudaStream_t stream, int num_sms) {
    CUtensorMap tmA, tmB;
    if (!make_tmap_rows_bf16(&tmA, a.h, a.P, a.d, BM) || !make_tmap_rows_bf16(&tmB, a.W, a.R, a.d, BN))
        return cudaErrorInvalidValue;
    const int kblocks = (a.d + BK - 1) / BK;
    const int m_tiles = (a.P + BM - 1) / BM;
    const int n_tiles = (a.R + BN - 1) / BN;
    const int tiles = m_tiles * n_tiles;
    // split-K factor: a power of two <= 8 (portable cluster size) that fills
    // the SMs without exceeding them and leaves every CTA at least 2 k-blocks.
    int split = 1;
    while (split < 8 && tiles * split * 2 <= num_sms && kblocks >= split * 4) split *= 2;
    if (split == 1 && a.R > BN) {
        // 256-column tiles when they still give every SM at least one tile
        const int n_wide = (a.R + 255) / 256;
        if ((long long)m_tiles * n_wide >= num_sms) {
            CUtensorMap tmW;
            if (!make_tmap_rows_bf16(&tmW, a.W, a.R, a.d, 256)) return cudaErrorInvalidValue;
            auto wk = project_tc_kernel<1, 256>;
            const size_t smem = smem_bytes_for(256);
            cudaError_t ew = cudaFuncSetAttribute(wk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  (int)smem);
            if (ew != cudaSuccess) return ew;
            ProjParams pw{a.u, static_cast<__nv_bfloat16*>(a.out_bf16), a.P, a.R, kblocks, 1, a.ws};
            cudaLaunchConfig_t cw{};
            cw.gridDim = dim3(1u, (unsigned)m_tiles, (unsigned)n_wide);
            cw.blockDim = dim3(NTHREADS, 1, 1);
            cw.dynamicSmemBytes = smem;
            cw.stream = stream;
            cudaLaunchAttribute aw[1];
            aw[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            aw[0].val.programmaticStreamSerializationAllowed = 1;
            cw.attrs = aw;
            cw.numAttrs = 1;
            ew = cudaLaunchKernelEx(&cw, wk, tmA, tmW, pw);
            if (ew != cudaSuccess) return ew;
            return cudaGetLastError();
        }
    }

    auto kern = split == 1 ? project_tc_kernel<1>
                : split == 2 ? project_tc_kernel<2>
                : split == 4 ? project_tc_kernel<4>
                             : project_tc_kernel<8>;
    cudaError_t e0 = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)SMEM_BYTES);
    if (e0 != cudaSuccess) return e0;
    ProjParams p{a.u, static_cast<__nv_bfloat16*>(a.out_bf16), a.P, a.R, kblocks, split, a.ws};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)split, (unsigned)m_tiles, (unsigned)n_tiles);
    cfg.blockDim = dim3(NTHREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)split;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// ---------------------------------------------------------------- fixed workspace
//
// A split-K workspace that lives in the library itself, for callers that are
// not allowed to allocate device memory.  Every GPU that loads the library
// holds it until the process exits.  All calls share it: calls that overlap on
// the GPU race on it.  Nothing in it has to start at zero (each call writes
// every slot it reads), so it is never cleared.
static __device__ __align__(256) float g_fixed_ws[kFixedProjectWorkspaceBytes / sizeof(float)];

// Device address of g_fixed_ws in the current context.  Looked up on every
// call (cudaGetSymbolAddress, with the device current) and never cached: after
// cudaDeviceReset, or in another context on the same device, the array lives
// at a new address, and a cached one would be stale.  The name itself is only
// a host-side stand-in, never a device address.
cudaError_t fixed_project_workspace(float** ptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fixed_ws);
    if (e != cudaSuccess) return e;
    *ptr = static_cast<float*>(p);
    return cudaSuccess;
}

cudaError_t take_project_faults(unsigned* flags) {
    unsigned v = 0;
    const unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_fault_word, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(zero));
    *flags = v;
    return e;
}

cudaError_t launch_project_f32(const ProjectArgs& a, cudaStream_t stream) {
    dim3 grid((unsigned)((a.R + FT - 1) / FT), (unsigned)((a.P + FT - 1) / FT));
    project_f32_kernel<<<grid, 256, 0, stream>>>(static_cast<const float*>(a.h),
                                                 static_cast<const float*>(a.W), a.u, a.P, a.d,
                                                 a.R);
    return cudaGetLastError();
}

}  // namespace df2
