// Greedy chain readout with a p_min cut: the draft tokens of each sequence,
// read from the selector's per-predecessor argmax table.
//
// ggml-org/llama.cpp pull request #27342, "spec : add DFlash2 support (local
// convolution + candidate selector)": the Overview's readout is each
// predecessor's argmax candidate, and the merged tree names the DFlash2 draft
// path "selector + p_min".  Per sequence s (readings where the text is silent):
//   slot_0 = start_slot[s] (if given, >= 0) else argmax_k unary[s,0,k];
//   slot_i = best_slot[s,i-1,slot_{i-1}];
//   p_0 = softmax(unary[s,0,:])[slot_0];
//   p_i = softmax(edges[s,i-1,slot_{i-1},:])[slot_i];
//   tokens[s,i] = cand_ids[s,i,slot_i];
//   length[s] = the number of leading positions with p_i >= p_min.
//
// One CTA per sequence.  The walk itself is a chain of dependent lookups, so
// the kernel stages the sequence's argmax table in shared memory first (one
// coalesced read), walks it there with one thread, and then scores only the
// n-1 edge rows on the chain, in parallel (one warp per row).  Latency-bound
// by design: the bytes are the table, n rows of K scores and the outputs.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "dflash2.h"

namespace df2 {
namespace {

constexpr int kChainThreads = 256;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Clamps a slot read from an input into [0, K), flagging a bad one.
__device__ __forceinline__ int checked_slot(int v, int K, int32_t* err_flag) {
    if (v < 0 || v >= K) {
        if (err_flag != nullptr) atomicOr(err_flag, DF2_FLAG_BAD_ID);
        return v < 0 ? 0 : K - 1;
    }
    return v;
}

__global__ void __launch_bounds__(kChainThreads) chain_kernel(ChainArgs a) {
    extern __shared__ int32_t sm[];
    const int s = blockIdx.x;
    const int n = a.n, K = a.K, E = n - 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t* bs = sm;                                       // best_slot of this sequence [E][K]
    int32_t* slots = bs + (size_t)E * K;                    // [n]
    float* pr = reinterpret_cast<float*>(slots + n);        // [n]

    const int32_t* bsg = a.best_slot + (size_t)s * E * K;
    for (int i = tid; i < E * K; i += kChainThreads) bs[i] = bsg[i];

    if (warp == 0) {
        // position 0: argmax of the unary scores (lowest slot on ties) and its share
        const float* u0 = a.unary + (size_t)s * n * K;
        float bv = -INFINITY;
        int bi = K;
        for (int k = lane; k < K; k += 32) {
            const float v = u0[k];
            if (v > bv || (v == bv && k < bi)) {
                bv = v;
                bi = k;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
            const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
            if (v2 > bv || (v2 == bv && i2 < bi)) {
                bv = v2;
                bi = i2;
            }
        }
        int slot0 = bi < K ? bi : 0;  // all NaN (unsupported input): never read past the row
        if (a.start_slot != nullptr) {
            const int g = a.start_slot[s];
            if (g >= 0) slot0 = checked_slot(g, K, a.err_flag);
        }
        float z = 0.f;
        for (int k = lane; k < K; k += 32) z += expf(u0[k] - bv);
        z = warp_sum(z);
        if (lane == 0) {
            slots[0] = slot0;
            pr[0] = expf(u0[slot0] - bv) / z;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int slot = slots[0];
        for (int i = 1; i < n; ++i) {
            slot = checked_slot(bs[(i - 1) * K + slot], K, a.err_flag);
            slots[i] = slot;
        }
    }
    __syncthreads();
    // the chosen candidate's share among the scores leaving the chosen predecessor
    for (int i = 1 + warp; i < n; i += kChainThreads / 32) {
        const float* row = a.edges + (((size_t)s * E + (i - 1)) * K + slots[i - 1]) * K;
        float m = -INFINITY;
        for (int c = lane; c < K; c += 32) m = fmaxf(m, row[c]);
        m = warp_max(m);
        float z = 0.f;
        for (int c = lane; c < K; c += 32) z += expf(row[c] - m);
        z = warp_sum(z);
        if (lane == 0) pr[i] = expf(row[slots[i]] - m) / z;
    }
    __syncthreads();
    for (int i = tid; i < n; i += kChainThreads) {
        a.tokens[(size_t)s * n + i] = a.cand_ids[((size_t)s * n + i) * K + slots[i]];
        a.probs[(size_t)s * n + i] = pr[i];
    }
    if (tid == 0) {
        int len = 0;
        while (len < n && pr[len] >= a.p_min) ++len;
        a.length[s] = len;
    }
}

}  // namespace

size_t chain_smem_bytes(int n, int K) {
    return (size_t)(n - 1) * K * 4 + (size_t)n * 8;
}

cudaError_t launch_chain(const ChainArgs& a, cudaStream_t stream) {
    const size_t smem = chain_smem_bytes(a.n, a.K);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(
            chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    chain_kernel<<<a.S, kChainThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace df2
