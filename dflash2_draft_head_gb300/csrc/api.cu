// C ABI of the DFlash2 draft-head library: argument validation on the host,
// then dispatch to the kernels.  Nothing here allocates device memory or
// synchronises the host (except dflash2_take_device_faults, by contract).
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "dflash2.h"

namespace {

thread_local char g_err[512] = {0};

int fail(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(DF2_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Buf {
    const void* p;
    size_t bytes;
    const char* name;
};

bool overlap(const Buf& a, const Buf& b) {
    if (a.p == nullptr || b.p == nullptr || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a.p), b0 = reinterpret_cast<uintptr_t>(b.p);
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Every output must be disjoint from every other buffer.
int check_disjoint(const Buf* outs, int nout, const Buf* ins, int nin) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlap(outs[i], ins[j]))
                return fail(DF2_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, ins[j].name);
        for (int j = i + 1; j < nout; ++j)
            if (overlap(outs[i], outs[j]))
                return fail(DF2_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
    }
    return DF2_OK;
}

int check_aligned(const Buf* bufs, int nb) {
    for (int i = 0; i < nb; ++i)
        if (bufs[i].p != nullptr && !aligned16(bufs[i].p))
            return fail(DF2_ERR_INVALID_ARG, "%s is not 16-byte aligned", bufs[i].name);
    return DF2_OK;
}

bool valid_dtype(int d) { return d == DF2_F32 || d == DF2_BF16; }
size_t esize(int d) { return d == DF2_BF16 ? 2 : 4; }

// Per-device attribute caches.  Host threads may call in concurrently, so the
// slots are atomics (a race only ever stores the same value twice).
std::atomic<int> g_num_sms[64];
std::atomic<int> g_max_smem[64];

int num_sms_of_current_device() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    const bool slot = dev >= 0 && dev < 64;
    if (slot) {
        const int c = g_num_sms[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
    if (slot) g_num_sms[dev].store(sms, std::memory_order_relaxed);
    return sms;
}

size_t max_smem_optin_of_current_device() {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 227 * 1024;
    const bool slot = dev >= 0 && dev < 64;
    if (slot) {
        const int c = g_max_smem[dev].load(std::memory_order_relaxed);
        if (c > 0) return (size_t)c;
    }
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return 227 * 1024;
    if (slot) g_max_smem[dev].store(v, std::memory_order_relaxed);
    return (size_t)v;
}

int validate_project(const void* h, const void* W, const float* u, int P, int d, int R,
                     int dtype) {
    if (h == nullptr || W == nullptr || u == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "project: NULL h, W or u");
    if (P <= 0 || d <= 0 || R <= 0)
        return fail(DF2_ERR_INVALID_ARG, "project: P=%d d=%d R=%d must be positive", P, d, R);
    if (!valid_dtype(dtype)) return fail(DF2_ERR_INVALID_ARG, "project: bad dtype %d", dtype);
    const size_t b = esize(dtype);
    const Buf ins[2] = {{h, (size_t)P * d * b, "h"}, {W, (size_t)R * d * b, "W"}};
    const Buf outs[1] = {{u, (size_t)P * R * 4, "u"}};
    int st = check_aligned(ins, 2);
    if (st == DF2_OK) st = check_aligned(outs, 1);
    if (st == DF2_OK) st = check_disjoint(outs, 1, ins, 2);
    if (st != DF2_OK) return st;
    if (R % 8 != 0 || R > 512)
        return fail(DF2_ERR_UNSUPPORTED, "project: R=%d must be a multiple of 8 and <= 512", R);
    if (dtype == DF2_BF16 && d % 8 != 0)
        return fail(DF2_ERR_UNSUPPORTED, "project: bf16 needs d %% 8 == 0 (d=%d)", d);
    if ((long long)P > 65535LL * 128)
        return fail(DF2_ERR_UNSUPPORTED, "project: P=%d exceeds %d rows", P, 65535 * 128);
    return DF2_OK;
}

int validate_edges(const int32_t* cand_ids, const float* u, const void* A, const void* B,
                   const float* unary, int S, int n, int K, int R, int V, int dtype,
                   const float* edges_out, const int32_t* best_slot, const float* best_score,
                   const int32_t* err_flag) {
    if (cand_ids == nullptr || u == nullptr || A == nullptr || B == nullptr || unary == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "edges: NULL required pointer");
    // with a single position there are no transitions, so the outputs are empty
    if (n > 1 && (best_slot == nullptr || best_score == nullptr))
        return fail(DF2_ERR_INVALID_ARG, "edges: NULL best_slot or best_score");
    if (S <= 0 || n <= 0 || K <= 0 || R <= 0 || V <= 0)
        return fail(DF2_ERR_INVALID_ARG, "edges: S=%d n=%d K=%d R=%d V=%d must be positive", S, n,
                    K, R, V);
    if (!valid_dtype(dtype)) return fail(DF2_ERR_INVALID_ARG, "edges: bad dtype %d", dtype);
    const size_t b = esize(dtype);
    const size_t SnK = (size_t)S * n * K;
    const size_t EK = (size_t)S * (n - 1) * K;
    const Buf ins[5] = {{cand_ids, SnK * 4, "cand_ids"},
                        {u, (size_t)S * n * R * 4, "u"},
                        {A, (size_t)V * R * b, "A"},
                        {B, (size_t)V * R * b, "B"},
                        {unary, SnK * 4, "unary"}};
    const Buf outs[4] = {{edges_out, EK * K * 4, "edges_out"},
                         {best_slot, EK * 4, "best_slot"},
                         {best_score, EK * 4, "best_score"},
                         {err_flag, 4, "err_flag"}};
    int st = check_aligned(ins, 5);
    if (st == DF2_OK) st = check_aligned(outs, 3);
    if (st == DF2_OK && err_flag != nullptr && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
        st = fail(DF2_ERR_INVALID_ARG, "err_flag is not 4-byte aligned");
    if (st == DF2_OK) st = check_disjoint(outs, 4, ins, 5);
    if (st != DF2_OK) return st;
    if (K > 256) return fail(DF2_ERR_UNSUPPORTED, "edges: K=%d > 256", K);
    if (R % 8 != 0 || R > 512)
        return fail(DF2_ERR_UNSUPPORTED, "edges: R=%d must be a multiple of 8 and <= 512", R);
    if ((long long)S * (n - 1) > 0x7FFFFFFFLL)
        return fail(DF2_ERR_UNSUPPORTED, "edges: too many transitions");
    return DF2_OK;
}

int run_edges(const int32_t* cand_ids, const float* u, const void* A, const void* B,
              const float* unary, int S, int n, int K, int R, int V, int dtype, float* edges_out,
              int32_t* best_slot, float* best_score, int32_t* err_flag, cudaStream_t stream,
              int u_only_dependency) {
    if (n == 1) return DF2_OK;
    df2::EdgesArgs a{cand_ids, u, A, B, unary, S, n, K, R, V, edges_out, best_slot, best_score,
                     err_flag};
    cudaError_t e;
    if (dtype == DF2_BF16) {
        // the one-kernel selector's edge phase where it covers the shapes
        bool launched = false;
        e = df2::launch_select_edges(a, stream, num_sms_of_current_device(),
                                     max_smem_optin_of_current_device(), &launched);
        if (e != cudaSuccess) return cuda_fail(e, "edges launch");
        if (launched) return DF2_OK;
    }
    if (dtype == DF2_BF16 && df2::edges_tc_supported(K, R))
        e = df2::launch_edges_bf16_tc(a, u_only_dependency, stream);
    else
        e = df2::launch_edges_warp(a, dtype == DF2_BF16, stream);
    if (e != cudaSuccess) return cuda_fail(e, "edges launch");
    return DF2_OK;
}

int run_project(const void* h, const void* W, float* u, int P, int d, int R, int dtype,
                cudaStream_t stream, float* ws = nullptr) {
    df2::ProjectArgs a{h, W, u, P, d, R};
    a.ws = ws;
    cudaError_t e = dtype == DF2_BF16
                        ? df2::launch_project_bf16_tc(a, stream, num_sms_of_current_device())
                        : df2::launch_project_f32(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "project launch");
    return DF2_OK;
}

}  // namespace

extern "C" {

int dflash2_version(void) { return 200; }

const char* dflash2_status_string(int status) {
    switch (status) {
        case DF2_OK:
            return "DF2_OK";
        case DF2_ERR_INVALID_ARG:
            return "DF2_ERR_INVALID_ARG";
        case DF2_ERR_UNSUPPORTED:
            return "DF2_ERR_UNSUPPORTED";
        case DF2_ERR_CUDA:
            return "DF2_ERR_CUDA";
        default:
            return "DF2_UNKNOWN_STATUS";
    }
}

const char* dflash2_last_error(void) { return g_err; }

int dflash2_dynconv(const void* x, const void* hist, const void* base, const void* delta,
                    void* out, int S, int n, int C, int T, int G, int in_dtype, int out_dtype,
                    void* stream) {
    g_err[0] = 0;
    if (x == nullptr || base == nullptr || delta == nullptr || out == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "dynconv: NULL x, base, delta or out");
    if (S <= 0 || n <= 0 || C <= 0 || T <= 0 || G <= 0)
        return fail(DF2_ERR_INVALID_ARG, "dynconv: S=%d n=%d C=%d T=%d G=%d must be positive", S,
                    n, C, T, G);
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
        return fail(DF2_ERR_INVALID_ARG, "dynconv: bad dtype");
    if (C % G != 0) return fail(DF2_ERR_INVALID_ARG, "dynconv: C=%d not a multiple of G=%d", C, G);
    const size_t bi = esize(in_dtype), bo = esize(out_dtype);
    const Buf ins[4] = {{x, (size_t)S * n * C * bi, "x"},
                        {hist, (size_t)S * (T - 1) * C * bi, "hist"},
                        {base, (size_t)T * C * bi, "base"},
                        {delta, (size_t)S * n * T * G * bi, "delta"}};
    const Buf outs[1] = {{out, (size_t)S * n * C * bo, "out"}};
    int st = check_aligned(ins, 4);
    if (st == DF2_OK) st = check_aligned(outs, 1);
    if (st == DF2_OK) st = check_disjoint(outs, 1, ins, 4);
    if (st != DF2_OK) return st;
    if (C % 8 != 0 || (C / G) % 8 != 0)
        return fail(DF2_ERR_UNSUPPORTED, "dynconv: needs C %% 8 == 0 and (C/G) %% 8 == 0");
    if (T > 16) return fail(DF2_ERR_UNSUPPORTED, "dynconv: T=%d > 16", T);
    if (in_dtype == DF2_F32 && out_dtype == DF2_BF16)
        return fail(DF2_ERR_UNSUPPORTED, "dynconv: fp32 input with bf16 output");
    df2::DynconvArgs a{x, T > 1 ? hist : nullptr, base, delta, out, S, n, C, T, G,
                       in_dtype == DF2_BF16, out_dtype == DF2_BF16};
    cudaError_t e = df2::launch_dynconv(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dynconv launch");
    return DF2_OK;
}

int dflash2_project(const void* h, const void* W, float* u, int P, int d, int R, int in_dtype,
                    void* stream) {
    g_err[0] = 0;
    int st = validate_project(h, W, u, P, d, R, in_dtype);
    if (st != DF2_OK) return st;
    return run_project(h, W, u, P, d, R, in_dtype, static_cast<cudaStream_t>(stream));
}

size_t dflash2_project_workspace_bytes(int P, int d, int R) {
    if (P <= 0 || d <= 0 || R <= 0) return 0;
    return df2::project_workspace_bytes(P, d, R, num_sms_of_current_device());
}

int dflash2_project_ws(const void* h, const void* W, float* u, int P, int d, int R, int in_dtype,
                       void* workspace, size_t workspace_bytes, void* stream) {
    g_err[0] = 0;
    int st = validate_project(h, W, u, P, d, R, in_dtype);
    if (st != DF2_OK) return st;
    if (in_dtype != DF2_BF16)  // the fp32 path has no split-K reduction
        return run_project(h, W, u, P, d, R, in_dtype, static_cast<cudaStream_t>(stream));
    const size_t need = df2::project_workspace_bytes(P, d, R, num_sms_of_current_device());
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need)
            return fail(DF2_ERR_INVALID_ARG, "project_ws: workspace of %zu bytes needed, got %zu",
                        need, workspace == nullptr ? (size_t)0 : workspace_bytes);
        if (!aligned16(workspace))
            return fail(DF2_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
        const size_t b = esize(in_dtype);
        const Buf ws[1] = {{workspace, need, "workspace"}};
        const Buf others[3] = {{h, (size_t)P * d * b, "h"}, {W, (size_t)R * d * b, "W"},
                               {u, (size_t)P * R * 4, "u"}};
        st = check_disjoint(ws, 1, others, 3);
        if (st != DF2_OK) return st;
    }
    return run_project(h, W, u, P, d, R, in_dtype, static_cast<cudaStream_t>(stream),
                       need > 0 ? static_cast<float*>(workspace) : nullptr);
}

int dflash2_edges(const int32_t* cand_ids, const float* u, const void* A, const void* B,
                  const float* unary, int S, int n, int K, int R, int V, int cb_dtype,
                  float* edges_out, int32_t* best_slot, float* best_score, int32_t* err_flag,
                  void* stream) {
    g_err[0] = 0;
    int st = validate_edges(cand_ids, u, A, B, unary, S, n, K, R, V, cb_dtype, edges_out,
                            best_slot, best_score, err_flag);
    if (st != DF2_OK) return st;
    return run_edges(cand_ids, u, A, B, unary, S, n, K, R, V, cb_dtype, edges_out, best_slot,
                     best_score, err_flag, static_cast<cudaStream_t>(stream), 0);
}

int dflash2_select(const void* h, const void* W, const int32_t* cand_ids, const void* A,
                   const void* B, const float* unary, int S, int n, int d, int K, int R, int V,
                   int dtype, float* u_out, float* edges_out, int32_t* best_slot,
                   float* best_score, int32_t* err_flag, void* stream) {
    g_err[0] = 0;
    if (S <= 0 || n <= 0)
        return fail(DF2_ERR_INVALID_ARG, "select: S=%d n=%d must be positive", S, n);
    if ((long long)S * n > 0x7FFFFFFFLL) return fail(DF2_ERR_UNSUPPORTED, "select: S*n too large");
    int st = validate_project(h, W, u_out, S * n, d, R, dtype);
    if (st == DF2_OK)
        st = validate_edges(cand_ids, u_out, A, B, unary, S, n, K, R, V, dtype, edges_out,
                            best_slot, best_score, err_flag);
    if (st != DF2_OK) return st;
    // the projection output must not alias anything the selector reads or writes
    const size_t b = esize(dtype);
    const Buf uo[1] = {{u_out, (size_t)S * n * R * 4, "u_out"}};
    const Buf others[8] = {{cand_ids, (size_t)S * n * K * 4, "cand_ids"},
                           {A, (size_t)V * R * b, "A"},
                           {B, (size_t)V * R * b, "B"},
                           {unary, (size_t)S * n * K * 4, "unary"},
                           {edges_out, (size_t)S * (n - 1) * K * K * 4, "edges_out"},
                           {best_slot, (size_t)S * (n - 1) * K * 4, "best_slot"},
                           {best_score, (size_t)S * (n - 1) * K * 4, "best_score"},
                           {err_flag, 4, "err_flag"}};
    st = check_disjoint(uo, 1, others, 8);
    if (st != DF2_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == DF2_BF16 && df2::select_fused_supported(K, R, d, n)) {
        df2::SelectArgs sa{h, W, cand_ids, A, B, unary, S, n, d, K, R, V, u_out, edges_out,
                           best_slot, best_score, err_flag};
        bool launched = false;
        cudaError_t e = df2::launch_select_fused(sa, s, num_sms_of_current_device(),
                                                 max_smem_optin_of_current_device(), &launched);
        if (e != cudaSuccess) return cuda_fail(e, "select launch");
        if (launched) return DF2_OK;
    }
    st = run_project(h, W, u_out, S * n, d, R, dtype, s);
    if (st != DF2_OK) return st;
    // the projection only produces u_out and waited for everything before it
    return run_edges(cand_ids, u_out, A, B, unary, S, n, K, R, V, dtype, edges_out, best_slot,
                     best_score, err_flag, s, dtype == DF2_BF16 ? 1 : 0);
}

int dflash2_select_plan(int S, int n, int d, int K, int R, int dtype, int* plan_out) {
    g_err[0] = 0;
    if (plan_out == nullptr) return fail(DF2_ERR_INVALID_ARG, "select_plan: NULL plan_out");
    if (S <= 0 || n <= 0 || d <= 0 || K <= 0 || R <= 0)
        return fail(DF2_ERR_INVALID_ARG, "select_plan: S=%d n=%d d=%d K=%d R=%d must be positive",
                    S, n, d, K, R);
    if (!valid_dtype(dtype)) return fail(DF2_ERR_INVALID_ARG, "select_plan: bad dtype %d", dtype);
    if ((long long)S * n > 0x7FFFFFFFLL)
        return fail(DF2_ERR_UNSUPPORTED, "select_plan: S*n too large");
    plan_out[0] = plan_out[1] = plan_out[2] = plan_out[3] = 0;
    int cs = 0, nc = 0, mr = 0;
    if (dtype == DF2_BF16 &&
        df2::select_fused_plan(S, n, d, K, R, num_sms_of_current_device(),
                               max_smem_optin_of_current_device(), &cs, &nc, &mr)) {
        plan_out[0] = 1;
        plan_out[1] = cs;
        plan_out[2] = nc;
        plan_out[3] = mr;
    }
    cudaGetLastError();  // planning queries leave no error behind
    return DF2_OK;
}

int dflash2_project_noalloc(const void* h, const void* W, float* u, int P, int d, int R,
                            int in_dtype, void* stream) {
    g_err[0] = 0;
    int st = validate_project(h, W, u, P, d, R, in_dtype);
    if (st != DF2_OK) return st;
    if (in_dtype != DF2_BF16)  // the fp32 path uses no workspace
        return run_project(h, W, u, P, d, R, in_dtype, static_cast<cudaStream_t>(stream));
    const size_t need = df2::project_workspace_bytes(P, d, R, num_sms_of_current_device());
    if (need > df2::kFixedProjectWorkspaceBytes)
        return fail(DF2_ERR_UNSUPPORTED,
                    "project_noalloc: these shapes need %zu bytes of workspace, more than the "
                    "library's fixed %zu; use dflash2_project_ws with your own workspace",
                    need, df2::kFixedProjectWorkspaceBytes);
    float* ws = nullptr;
    if (need > 0) {
        cudaError_t e = df2::fixed_project_workspace(&ws);
        if (e != cudaSuccess) return cuda_fail(e, "project_noalloc workspace address");
    }
    return run_project(h, W, u, P, d, R, in_dtype, static_cast<cudaStream_t>(stream), ws);
}

int dflash2_topk(const void* logits, int rows, int V, int K, int in_dtype, int32_t* cand_ids,
                 float* values, void* stream) {
    g_err[0] = 0;
    if (logits == nullptr || cand_ids == nullptr || values == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "topk: NULL logits, cand_ids or values");
    if (rows <= 0 || V <= 0)
        return fail(DF2_ERR_INVALID_ARG, "topk: rows=%d V=%d must be positive", rows, V);
    if (K < 1 || K > V) return fail(DF2_ERR_INVALID_ARG, "topk: K=%d outside [1, V=%d]", K, V);
    if (!valid_dtype(in_dtype)) return fail(DF2_ERR_INVALID_ARG, "topk: bad dtype %d", in_dtype);
    const Buf ins[1] = {{logits, (size_t)rows * V * esize(in_dtype), "logits"}};
    const Buf outs[2] = {{cand_ids, (size_t)rows * K * 4, "cand_ids"},
                         {values, (size_t)rows * K * 4, "values"}};
    int st = check_aligned(ins, 1);
    if (st == DF2_OK) st = check_aligned(outs, 2);
    if (st == DF2_OK) st = check_disjoint(outs, 2, ins, 1);
    if (st != DF2_OK) return st;
    if (K > df2::kTopkMaxK)
        return fail(DF2_ERR_UNSUPPORTED, "topk: K=%d > %d", K, df2::kTopkMaxK);
    df2::TopkLaunch a{logits, rows, V, K, in_dtype == DF2_BF16, cand_ids, values};
    cudaError_t e = df2::launch_topk(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "topk launch");
    return DF2_OK;
}

int dflash2_predict_delta(const void* x, const void* Wc, void* delta, int P, int C, int TG,
                          int dtype, void* stream) {
    g_err[0] = 0;
    if (x == nullptr || Wc == nullptr || delta == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "predict_delta: NULL x, Wc or delta");
    if (P <= 0 || C <= 0 || TG <= 0)
        return fail(DF2_ERR_INVALID_ARG, "predict_delta: P=%d C=%d TG=%d must be positive", P, C,
                    TG);
    if (!valid_dtype(dtype)) return fail(DF2_ERR_INVALID_ARG, "predict_delta: bad dtype %d", dtype);
    const size_t b = esize(dtype);
    const Buf ins[2] = {{x, (size_t)P * C * b, "x"}, {Wc, (size_t)TG * C * b, "Wc"}};
    const Buf outs[1] = {{delta, (size_t)P * TG * b, "delta"}};
    int st = check_aligned(ins, 2);
    if (st == DF2_OK) st = check_aligned(outs, 1);
    if (st == DF2_OK) st = check_disjoint(outs, 1, ins, 2);
    if (st != DF2_OK) return st;
    if (TG % 8 != 0 || TG > 512)
        return fail(DF2_ERR_UNSUPPORTED, "predict_delta: T*G=%d must be a multiple of 8 and <= 512",
                    TG);
    if (dtype == DF2_BF16 && C % 8 != 0)
        return fail(DF2_ERR_UNSUPPORTED, "predict_delta: bf16 needs C %% 8 == 0 (C=%d)", C);
    if ((long long)P > 65535LL * 128)
        return fail(DF2_ERR_UNSUPPORTED, "predict_delta: P=%d exceeds %d rows", P, 65535 * 128);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == DF2_F32) {
        df2::ProjectArgs a{x, Wc, static_cast<float*>(delta), P, C, TG};
        e = df2::launch_project_f32(a, s);
    } else {
        df2::ProjectArgs a{x, Wc, nullptr, P, C, TG};
        a.out_bf16 = delta;
        e = df2::launch_project_bf16_tc(a, s, num_sms_of_current_device());
    }
    if (e != cudaSuccess) return cuda_fail(e, "predict_delta launch");
    return DF2_OK;
}

int dflash2_dynconv_predicted(const void* x, const void* hist, const void* base, const void* Wc,
                              void* out, int S, int n, int C, int T, int G, int in_dtype,
                              int out_dtype, void* stream) {
    g_err[0] = 0;
    if (x == nullptr || base == nullptr || Wc == nullptr || out == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "dynconv_predicted: NULL x, base, Wc or out");
    if (S <= 0 || n <= 0 || C <= 0 || T <= 0 || G <= 0)
        return fail(DF2_ERR_INVALID_ARG,
                    "dynconv_predicted: S=%d n=%d C=%d T=%d G=%d must be positive", S, n, C, T, G);
    if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype))
        return fail(DF2_ERR_INVALID_ARG, "dynconv_predicted: bad dtype");
    if (C % G != 0)
        return fail(DF2_ERR_INVALID_ARG, "dynconv_predicted: C=%d not a multiple of G=%d", C, G);
    const size_t bi = esize(in_dtype), bo = esize(out_dtype);
    const Buf ins[4] = {{x, (size_t)S * n * C * bi, "x"},
                        {hist, (size_t)S * (T - 1) * C * bi, "hist"},
                        {base, (size_t)T * C * bi, "base"},
                        {Wc, (size_t)T * G * C * bi, "Wc"}};
    const Buf outs[1] = {{out, (size_t)S * n * C * bo, "out"}};
    int st = check_aligned(ins, 4);
    if (st == DF2_OK) st = check_aligned(outs, 1);
    if (st == DF2_OK) st = check_disjoint(outs, 1, ins, 4);
    if (st != DF2_OK) return st;
    if (in_dtype == DF2_F32 && out_dtype == DF2_BF16)
        return fail(DF2_ERR_UNSUPPORTED, "dynconv_predicted: fp32 input with bf16 output");
    if (T > df2::kMaxPredT)
        return fail(DF2_ERR_UNSUPPORTED, "dynconv_predicted: T=%d > %d", T, df2::kMaxPredT);
    const long long TG = (long long)T * G;
    if (C % 8 != 0 || (C / G) % 8 != 0 || TG % 8 != 0 || TG > 256)
        return fail(DF2_ERR_UNSUPPORTED,
                    "dynconv_predicted: needs C %% 8 == 0, (C/G) %% 8 == 0, (T*G) %% 8 == 0 and "
                    "T*G <= 256 (C=%d T=%d G=%d)", C, T, G);
    if ((long long)S * n > 0x7FFFFFFFLL)
        return fail(DF2_ERR_UNSUPPORTED, "dynconv_predicted: S*n above 2^31-1");
    df2::DynconvPredArgs a{x, T > 1 ? hist : nullptr, base, Wc, out, S, n, C, T, G,
                           out_dtype == DF2_BF16};
    if (in_dtype == DF2_F32) {
        cudaError_t e = df2::launch_dynconv_pred_f32(a, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "dynconv_predicted launch");
        return DF2_OK;
    }
    df2::DynconvPredPlan plan{};
    if (!df2::plan_dynconv_pred(a, num_sms_of_current_device(), max_smem_optin_of_current_device(),
                                &plan))
        return fail(DF2_ERR_UNSUPPORTED, "dynconv_predicted: shapes do not fit shared memory");
    cudaError_t e = df2::launch_dynconv_pred(a, plan, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dynconv_predicted launch");
    return DF2_OK;
}

int dflash2_chain(const int32_t* cand_ids, const float* unary, const float* edges,
                  const int32_t* best_slot, const int32_t* start_slot, int S, int n, int K,
                  float p_min, int32_t* tokens, float* probs, int32_t* length, int32_t* err_flag,
                  void* stream) {
    g_err[0] = 0;
    if (cand_ids == nullptr || unary == nullptr || tokens == nullptr || probs == nullptr ||
        length == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "chain: NULL cand_ids, unary, tokens, probs or length");
    if (S <= 0 || n <= 0 || K <= 0)
        return fail(DF2_ERR_INVALID_ARG, "chain: S=%d n=%d K=%d must be positive", S, n, K);
    if (n > 1 && (edges == nullptr || best_slot == nullptr))
        return fail(DF2_ERR_INVALID_ARG, "chain: NULL edges or best_slot with n > 1");
    const size_t SnK = (size_t)S * n * K, EK = (size_t)S * (n - 1) * K;
    const Buf ins[5] = {{cand_ids, SnK * 4, "cand_ids"},
                        {unary, SnK * 4, "unary"},
                        {edges, EK * K * 4, "edges"},
                        {best_slot, EK * 4, "best_slot"},
                        {start_slot, (size_t)S * 4, "start_slot"}};
    const Buf outs[4] = {{tokens, (size_t)S * n * 4, "tokens"},
                         {probs, (size_t)S * n * 4, "probs"},
                         {length, (size_t)S * 4, "length"},
                         {err_flag, 4, "err_flag"}};
    int st = check_aligned(ins, 5);
    if (st == DF2_OK) st = check_aligned(outs, 3);
    if (st == DF2_OK && err_flag != nullptr && (reinterpret_cast<uintptr_t>(err_flag) & 3u))
        st = fail(DF2_ERR_INVALID_ARG, "err_flag is not 4-byte aligned");
    if (st == DF2_OK) st = check_disjoint(outs, 4, ins, 5);
    if (st != DF2_OK) return st;
    if (df2::chain_smem_bytes(n, K) > 200 * 1024)
        return fail(DF2_ERR_UNSUPPORTED, "chain: argmax table of n=%d, K=%d exceeds 200 KB", n, K);
    df2::ChainArgs a{cand_ids, unary, edges, best_slot, start_slot, S, n, K, p_min,
                     tokens, probs, length, err_flag};
    cudaError_t e = df2::launch_chain(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "chain launch");
    return DF2_OK;
}

int dflash2_probe_gather(const void* table, long long rows, int row_bytes, const int32_t* ids,
                         int n_ids, uint32_t* out, void* stream) {
    g_err[0] = 0;
    if (table == nullptr || ids == nullptr || out == nullptr)
        return fail(DF2_ERR_INVALID_ARG, "probe_gather: NULL table, ids or out");
    if (rows <= 0 || n_ids < 0)
        return fail(DF2_ERR_INVALID_ARG, "probe_gather: rows=%lld n_ids=%d", rows, n_ids);
    if (row_bytes < 16 || row_bytes > 512 || (row_bytes & (row_bytes - 1)) != 0)
        return fail(DF2_ERR_INVALID_ARG,
                    "probe_gather: row_bytes=%d must be a power of two in [16, 512]", row_bytes);
    const Buf ins[2] = {{table, (size_t)rows * (size_t)row_bytes, "table"},
                        {ids, (size_t)n_ids * 4, "ids"}};
    const Buf outs[1] = {{out, (size_t)n_ids * 4, "out"}};
    int st = check_aligned(ins, 2);
    if (st == DF2_OK) st = check_aligned(outs, 1);
    if (st == DF2_OK) st = check_disjoint(outs, 1, ins, 2);
    if (st != DF2_OK) return st;
    df2::ProbeGatherArgs a{table, rows, row_bytes, ids, n_ids, out};
    cudaError_t e = df2::launch_probe_gather(a, static_cast<cudaStream_t>(stream),
                                             num_sms_of_current_device());
    if (e != cudaSuccess) return cuda_fail(e, "probe_gather launch");
    return DF2_OK;
}

int dflash2_take_device_faults(int32_t* flags_out) {
    g_err[0] = 0;
    if (flags_out == nullptr) return fail(DF2_ERR_INVALID_ARG, "flags_out is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    unsigned v = 0;
    unsigned v2 = 0;
    if (e == cudaSuccess) e = df2::take_project_faults(&v);
    if (e == cudaSuccess) e = df2::take_dynconv_faults(&v2);
    v |= v2;
    if (e == cudaSuccess) e = df2::take_topk_faults(&v2);
    v |= v2;
    if (e == cudaSuccess) e = df2::take_fused_faults(&v2);
    v |= v2;
    if (e == cudaSuccess) e = df2::take_select_faults(&v2);
    v |= v2;
    if (e != cudaSuccess) return cuda_fail(e, "take_device_faults");
    *flags_out = (int32_t)v;
    return DF2_OK;
}

}  // extern "C"
