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
    if (a.in_bf16 && a.out_bf16)
        return launch_dtype<__nv_bfloat16, __nv_bfloat16>(p, a.T, nthr, stream);
    if (a.in_bf16)
        return launch_dtype<__nv_bfloat16, float>(p, a.T, nthr, stream);
    return launch_dtype<float, float>(p, a.T, nthr, stream);
}

}  // namespace df2
