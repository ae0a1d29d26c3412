// Measurement aid: how fast this GPU gathers random rows of a table.
//
// The edge kernel of the candidate selector reads, for every transition, 2K
// codebook rows at token ids that are, to the memory system, random.  Its
// bound is therefore not the streaming bandwidth of HBM but the rate at which
// random rows of a given size can be fetched.  This kernel measures that rate
// on its own: for every id it reads the whole row and writes one 32-bit XOR
// of the row's words (1/64 of a 256-byte row), so nearly all of its traffic
// is the gathered reads.
//
// Layout: groups of CPR lanes (16 bytes per lane per chunk, CPL chunks per
// lane) read one row; every warp keeps U rows per group in flight, and the
// grid fills every SM to full occupancy, so the number of outstanding
// requests, not the issue rate, sets the speed.
#include <cuda_runtime.h>

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace df2 {
namespace {

constexpr int PROBE_THREADS = 256;
constexpr int PROBE_U = 4;  // rows in flight per lane group

template <int CPR, int CPL>
__global__ void __launch_bounds__(PROBE_THREADS) probe_gather_kernel(
    const uint8_t* __restrict__ table, long long rows, const int32_t* __restrict__ ids, int n_ids,
    uint32_t* __restrict__ out) {
    constexpr int RPW = 32 / CPR;  // rows per warp per slot
    constexpr int ROW_BYTES = CPR * CPL * 16;
    const int lane = threadIdx.x & 31;
    const int sub = lane % CPR;
    const long long warp = ((long long)blockIdx.x * PROBE_THREADS + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * PROBE_THREADS) >> 5;
    const long long per_iter = (long long)RPW * PROBE_U;
    const long long iters = (n_ids + per_iter - 1) / per_iter;
    for (long long it = warp; it < iters; it += nwarps) {  // warp-uniform loop
        long long r[PROBE_U];
        long long id[PROBE_U];
#pragma unroll
        for (int u = 0; u < PROBE_U; ++u) {
            r[u] = it * per_iter + (long long)u * RPW + lane / CPR;
            long long v = r[u] < n_ids ? (long long)__ldg(ids + r[u]) : 0;
            id[u] = v < 0 ? 0 : (v >= rows ? rows - 1 : v);
        }
        uint4 v[PROBE_U][CPL];
#pragma unroll
        for (int u = 0; u < PROBE_U; ++u)
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                v[u][c] = r[u] < n_ids ? ldg_nc_v4(table + id[u] * ROW_BYTES + (c * CPR + sub) * 16)
                                       : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < PROBE_U; ++u) {
            uint32_t x = 0;
#pragma unroll
            for (int c = 0; c < CPL; ++c) x ^= v[u][c].x ^ v[u][c].y ^ v[u][c].z ^ v[u][c].w;
#pragma unroll
            for (int off = CPR / 2; off > 0; off >>= 1) x ^= __shfl_xor_sync(0xFFFFFFFFu, x, off);
            if (sub == 0 && r[u] < n_ids) out[r[u]] = x;
        }
    }
}

template <int CPR, int CPL>
cudaError_t launch_probe(const ProbeGatherArgs& a, cudaStream_t stream, int blocks) {
    probe_gather_kernel<CPR, CPL><<<blocks, PROBE_THREADS, 0, stream>>>(
        static_cast<const uint8_t*>(a.table), a.rows, a.ids, a.n_ids, a.out);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_probe_gather(const ProbeGatherArgs& a, cudaStream_t stream, int num_sms) {
    if (a.n_ids <= 0) return cudaSuccess;
    // full occupancy: 8 CTAs of 256 threads per SM, grid-stride over the rows
    const int blocks = num_sms * (2048 / PROBE_THREADS);
    switch (a.row_bytes) {
        case 16: return launch_probe<1, 1>(a, stream, blocks);
        case 32: return launch_probe<2, 1>(a, stream, blocks);
        case 64: return launch_probe<4, 1>(a, stream, blocks);
        case 128: return launch_probe<8, 1>(a, stream, blocks);
        case 256: return launch_probe<16, 1>(a, stream, blocks);
        case 512: return launch_probe<32, 1>(a, stream, blocks);
        case 1024: return launch_probe<32, 2>(a, stream, blocks);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace df2
