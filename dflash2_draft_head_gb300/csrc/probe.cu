// Measurement aid: how fast this GPU gathers random rows of a table.
//
// The edge kernels of the candidate selector read, for every transition, 2K
// codebook rows at token ids that are, to the memory system, random.  Their
// bound is therefore not the streaming bandwidth of HBM but the rate at which
// random rows of a given size can be fetched.  This kernel measures that rate
// the way the edge kernels fetch rows: one CTA per SM stages a block of ids in
// shared memory, then 16 warps issue 16-byte cp.async copies of the rows into
// a 4-stage shared-memory ring (so no copy waits for an id load), and each
// thread folds the chunks it copied into a 32-bit XOR of the row once they
// have landed.  For every id it writes that XOR (1/64 of a 256-byte row), so
// nearly all of its traffic is the gathered reads.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace df2 {
namespace {

constexpr int PROBE_THREADS = 512;
constexpr int PROBE_CH = 4;                                     // chunks per thread per stage
constexpr int PROBE_NST = 4;                                    // ring stages
constexpr int PROBE_STAGE = PROBE_THREADS * PROBE_CH * 16;      // 32 KB
constexpr int PROBE_IDS = 4096;                                 // ids staged at a time
constexpr size_t PROBE_SMEM = (size_t)PROBE_NST * PROBE_STAGE + PROBE_IDS * 4;

__device__ __forceinline__ void probe_wait(int pending) {
    switch (pending) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    }
}

// CPR: 16-byte chunks per row (1..32, a power of two).  The CPR lanes that copy
// one row are consecutive lanes of one warp, so the row's XOR is a shuffle
// reduction.
template <int CPR>
__global__ void __launch_bounds__(PROBE_THREADS, 1) probe_gather_kernel(
    const uint8_t* __restrict__ table, long long rows, const int32_t* __restrict__ ids, int n_ids,
    uint32_t* __restrict__ out) {
    extern __shared__ __align__(16) uint8_t psm[];
    int32_t* sid = reinterpret_cast<int32_t*>(psm + (size_t)PROBE_NST * PROBE_STAGE);
    const int t = threadIdx.x;
    const int lane = t & 31;
    const long long lo = (long long)blockIdx.x * n_ids / gridDim.x;
    const long long hi = (long long)(blockIdx.x + 1) * n_ids / gridDim.x;
    constexpr int ROW_BYTES = CPR * 16;
    constexpr int ROWS_PER_STAGE = PROBE_THREADS * PROBE_CH / CPR;
    for (long long b0 = lo; b0 < hi; b0 += PROBE_IDS) {
        const int nb = (int)min((long long)PROBE_IDS, hi - b0);
        __syncthreads();  // the previous block's ids are no longer read
        for (int i = t; i < nb; i += PROBE_THREADS) {
            long long v = ids[b0 + i];
            sid[i] = (int32_t)(v < 0 ? 0 : (v >= rows ? rows - 1 : v));
        }
        __syncthreads();
        const int nst = (nb + ROWS_PER_STAGE - 1) / ROWS_PER_STAGE;
        // fold the chunks this thread copied for stage s and write the rows' XOR
        auto consume = [&](int s) {
            const uint8_t* st = psm + (size_t)(s % PROBE_NST) * PROBE_STAGE;
#pragma unroll
            for (int k = 0; k < PROBE_CH; ++k) {
                const int q = s * PROBE_THREADS * PROBE_CH + k * PROBE_THREADS + t;
                const int row = q / CPR;
                uint32_t x = 0;
                if (row < nb) {
                    const uint4 v = *reinterpret_cast<const uint4*>(st + (size_t)(k * PROBE_THREADS + t) * 16);
                    x = v.x ^ v.y ^ v.z ^ v.w;
                }
#pragma unroll
                for (int off = CPR / 2; off > 0; off >>= 1) x ^= __shfl_xor_sync(0xFFFFFFFFu, x, off);
                if ((lane & (CPR - 1)) == 0 && row < nb) out[b0 + row] = x;
            }
        };
        for (int s = 0; s < nst; ++s) {
            if (s >= PROBE_NST) {
                probe_wait(PROBE_NST - 1);
                consume(s - PROBE_NST);
            }
            const uint32_t st = smem_u32(psm + (size_t)(s % PROBE_NST) * PROBE_STAGE);
#pragma unroll
            for (int k = 0; k < PROBE_CH; ++k) {
                const int q = s * PROBE_THREADS * PROBE_CH + k * PROBE_THREADS + t;
                const int row = q / CPR;
                if (row < nb)
                    cp_async16(st + (uint32_t)(k * PROBE_THREADS + t) * 16u,
                               table + (long long)sid[row] * ROW_BYTES + (q % CPR) * 16);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        }
        cp_async_wait_all();
        for (int s = nst > PROBE_NST ? nst - PROBE_NST : 0; s < nst; ++s) consume(s);
    }
}

template <int CPR>
cudaError_t launch_probe(const ProbeGatherArgs& a, cudaStream_t stream, int blocks) {
    cudaError_t e = cudaFuncSetAttribute(probe_gather_kernel<CPR>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)PROBE_SMEM);
    if (e != cudaSuccess) return e;
    probe_gather_kernel<CPR><<<blocks, PROBE_THREADS, PROBE_SMEM, stream>>>(
        static_cast<const uint8_t*>(a.table), a.rows, a.ids, a.n_ids, a.out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_probe_gather(const ProbeGatherArgs& a, cudaStream_t stream, int num_sms) {
    if (a.n_ids <= 0) return cudaSuccess;
    switch (a.row_bytes) {  // one CTA per SM
        case 16: return launch_probe<1>(a, stream, num_sms);
        case 32: return launch_probe<2>(a, stream, num_sms);
        case 64: return launch_probe<4>(a, stream, num_sms);
        case 128: return launch_probe<8>(a, stream, num_sms);
        case 256: return launch_probe<16>(a, stream, num_sms);
        case 512: return launch_probe<32>(a, stream, num_sms);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace df2
