// Internal declarations shared by the kernel translation units and the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace df2 {

// Longest time one on-chip wait may take before a kernel gives up (200 ms).
constexpr uint64_t kWaitNs = 200ull * 1000 * 1000;

struct DynconvArgs {
    const void* x;
    const void* hist;
    const void* base;
    const void* delta;
    void* out;
    int S, n, C, T, G;
    int in_bf16, out_bf16;
};

struct ProjectArgs {
    const void* h;
    const void* W;
    float* u;
    int P, d, R;
    float* ws = nullptr;  // optional split-K workspace (project_workspace_bytes)
    void* out_bf16 = nullptr;  // bf16 path only: write the output here in bf16 instead of u
};

struct EdgesArgs {
    const int32_t* cand_ids;
    const float* u;
    const void* A;
    const void* B;
    const float* unary;
    int S, n, K, R, V;
    float* edges_out;
    int32_t* best_slot;
    float* best_score;
    int32_t* err_flag;
};

struct ChainArgs {
    const int32_t* cand_ids;
    const float* unary;
    const float* edges;
    const int32_t* best_slot;
    const int32_t* start_slot;
    int S, n, K;
    float p_min;
    int32_t* tokens;
    float* probs;
    int32_t* length;
    int32_t* err_flag;
};

// Largest K the top-K kernel takes.
constexpr int kTopkMaxK = 1024;

struct TopkLaunch {
    const void* logits;
    int rows, V, K;
    int bf16;
    int32_t* ids;
    float* vals;
};

// 2-D bf16 tensor map over a row-major [rows, cols] array with a box of
// box_rows x 64 columns and 128-byte swizzle (out-of-range elements read as 0).
bool make_tmap_rows_bf16(CUtensorMap* m, const void* base, int rows, int cols, int box_rows);

// Each launcher enqueues on `stream` and returns the launch's cudaError_t.
cudaError_t launch_dynconv(const DynconvArgs& a, cudaStream_t stream);
// Reads and clears the convolution kernels' device fault word (synchronous).
cudaError_t take_dynconv_faults(unsigned* flags);

// The conv with its taps predicted from its input, fused (dynconv_pred.cu).
constexpr int kMaxPredT = 8;
struct DynconvPredArgs {
    const void* x;     // [S*n, C] bf16
    const void* hist;  // [S, T-1, C] bf16 or nullptr
    const void* base;  // [T, C] bf16
    const void* Wc;    // [T*G, C] bf16
    void* out;         // [S*n, C] bf16 or fp32
    int S, n, C, T, G;
    int out_bf16;
};
struct DynconvPredPlan {
    int NP, kblocks, m_tiles, split, stages, cdepth;
    uint32_t stage_bytes, ring_bytes, ds_bytes, tmem_cols;
    size_t smem_bytes;
};
// False when the shapes are outside what the fused kernel supports.
bool plan_dynconv_pred(const DynconvPredArgs& a, int num_sms, size_t max_smem, DynconvPredPlan* plan);
cudaError_t launch_dynconv_pred(const DynconvPredArgs& a, const DynconvPredPlan& plan,
                                cudaStream_t stream);
// fp32 inputs and output (T*G <= 256): delta in exact fp32, no tensor cores.
cudaError_t launch_dynconv_pred_f32(const DynconvPredArgs& a, cudaStream_t stream);
cudaError_t take_fused_faults(unsigned* flags);
cudaError_t launch_project_bf16_tc(const ProjectArgs& a, cudaStream_t stream, int num_sms);
// Bytes of split-K workspace the bf16 projection uses for these shapes (0: none).
size_t project_workspace_bytes(int P, int d, int R, int num_sms);
// Size of the library's own fixed projection workspace (8 MiB).
constexpr size_t kFixedProjectWorkspaceBytes = size_t(8) << 20;
// Device address of that workspace in the current context (looked up on every call).
cudaError_t fixed_project_workspace(float** ptr);
cudaError_t launch_project_f32(const ProjectArgs& a, cudaStream_t stream);
// Reads and clears the projection kernel's device fault word (synchronous).
cudaError_t take_project_faults(unsigned* flags);
// Tensor-core tile path: bf16 codebooks, K a power of two <= 128, R <= 384.
bool edges_tc_supported(int K, int R);
// u_only_dependency: the preceding kernel in the stream only produces u (and
// has itself waited for everything before it), so the kernel may read ids,
// codebooks and unary before that kernel completes.
cudaError_t launch_edges_bf16_tc(const EdgesArgs& a, int u_only_dependency, cudaStream_t stream);
// Warp-per-predecessor path (any K <= 256, R <= 512; fp32 or bf16 codebooks).
cudaError_t launch_edges_warp(const EdgesArgs& a, int cb_bf16, cudaStream_t stream);

// Greedy chain readout (one CTA per sequence; shared memory per CTA below).
size_t chain_smem_bytes(int n, int K);
cudaError_t launch_chain(const ChainArgs& a, cudaStream_t stream);

// Top-K candidate extraction (1 <= K <= min(V, kTopkMaxK)).
cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t stream);
// Reads and clears the top-K kernel's device fault word (synchronous).
cudaError_t take_topk_faults(unsigned* flags);

// The composite selector in one kernel (select.cu): bf16, K a power of two in
// [4, 128], R in {64, 128, 256}, d % 8 == 0, n >= 2.
struct SelectArgs {
    const void* h;
    const void* W;
    const int32_t* cand_ids;
    const void* A;
    const void* B;
    const float* unary;
    int S, n, d, K, R, V;
    float* u;
    float* edges_out;
    int32_t* best_slot;
    float* best_score;
    int32_t* err_flag;
};
bool select_fused_supported(int K, int R, int d, int n);
// Sets *launched = false (and launches nothing) when no cluster layout fits the
// shapes; the caller then runs the projection and the edge kernel separately.
cudaError_t launch_select_fused(const SelectArgs& a, cudaStream_t stream, int num_sms,
                                size_t max_smem, bool* launched);
// The edge scores and argmax alone with the one-kernel selector's edge phase (u
// given; the same shapes as launch_select_fused with any d).  Sets *launched =
// false when the shapes are not covered; the caller then runs an edge kernel.
cudaError_t launch_select_edges(const EdgesArgs& a, cudaStream_t stream, int num_sms,
                                size_t max_smem, bool* launched);
// Whether launch_select_fused runs for these shapes, and its cluster layout.
bool select_fused_plan(int S, int n, int d, int K, int R, int num_sms, size_t max_smem,
                       int* cluster_size, int* clusters, int* rows_per_block);
// Reads and clears the fused selector's device fault word (synchronous).
cudaError_t take_select_faults(unsigned* flags);

// Measurement aid: random-row gather (probe.cu).  out[i] = XOR of the 32-bit
// words of row ids[i] (ids clamped into [0, rows)); row_bytes a power of two
// in [16, 512].
struct ProbeGatherArgs {
    const void* table;
    long long rows;
    int row_bytes;
    const int32_t* ids;
    int n_ids;
    uint32_t* out;
};
cudaError_t launch_probe_gather(const ProbeGatherArgs& a, cudaStream_t stream, int num_sms);

}  // namespace df2
