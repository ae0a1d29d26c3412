/*
 * dflash2.h: C ABI of the DFlash2 draft-head hot path on NVIDIA GB300 (sm_103a).
 *
 * The operations are the two formulas of ggml-org/llama.cpp pull request
 * #27342, "spec : add DFlash2 support (local convolution + candidate
 * selector)", section "Overview":
 *
 *   grouped dynamic depthwise causal convolution
 *     out[i,c] = sum_t (base[t,c] + delta[i,t,g(c)]) * x[i-t,c]
 *   candidate-selector edge score
 *     edge(p->c) = < A[p] (.) project(h), B[c] > + unary[c]
 *
 * with the codebooks A ("selector_predecessor"), B ("selector_successor") and
 * the projection weight ("selector_hidden") named in that thread's review.
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers to contiguous row-major arrays,
 *     16-byte aligned.  The caller allocates and owns them; the library never
 *     allocates, frees or keeps a pointer past the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call only enqueues work on that stream and returns; it never
 *     synchronises the host.
 *   - Return value: a df2_status.  DF2_ERR_INVALID_ARG / DF2_ERR_UNSUPPORTED are
 *     detected on the host before anything is enqueued (nothing is launched).
 *     DF2_ERR_CUDA reports a launch error (cudaGetLastError); a fault inside a
 *     kernel surfaces at the caller's next synchronisation as usual.
 *   - dflash2_last_error() returns a thread-local text for the last non-OK
 *     status of the calling thread.
 *   - dtype codes: DF2_F32 (every float input fp32, fp32 accumulation and
 *     output, no TF32 anywhere) or DF2_BF16 (bf16 inputs, fp32 accumulation).
 */
#ifndef DFLASH2_H_
#define DFLASH2_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DF2_OK = 0,
    DF2_ERR_INVALID_ARG = 1,  /* bad size, NULL required pointer, misalignment, aliasing */
    DF2_ERR_UNSUPPORTED = 2,  /* legal arguments outside what the kernels implement */
    DF2_ERR_CUDA = 3          /* a CUDA runtime error at launch */
} df2_status;

typedef enum { DF2_F32 = 0, DF2_BF16 = 1 } df2_dtype;

/* Bits a kernel ORs into a caller-provided device err_flag (int32). */
#define DF2_FLAG_BAD_ID 1    /* a candidate id outside [0, V): it was clamped for the load */
#define DF2_FLAG_TIMEOUT 2   /* a bounded on-chip wait gave up; outputs of that tile are undefined */
#define DF2_FLAG_OVERFLOW 4  /* an internal buffer bound was reached (not expected for any input);
                                that call's outputs are undefined */

/* Library version (major*10000 + minor*100 + patch). */
int dflash2_version(void);

/* Human-readable name of a status code.  Never NULL. */
const char* dflash2_status_string(int status);

/* Detail text for the calling thread's last non-OK status ("" if none). */
const char* dflash2_last_error(void);

/*
 * Grouped dynamic depthwise causal convolution (PR #27342, Overview, first
 * formula).  For s < S, i < n, c < C:
 *   out[s,i,c] = sum_{t=0}^{T-1} (base[t,c] + delta[s,i,t,g(c)]) * xh[s,i-t,c]
 * where g(c) = c / (C/G) (contiguous groups) and xh[s,j,c] = x[s,j,c] for
 * j >= 0, hist[s,T-1+j,c] for -(T-1) <= j < 0 (oldest history row first; row
 * T-2 is the position just before the block).
 *
 *   x      [S,n,C]    in_dtype
 *   hist   [S,T-1,C]  in_dtype, or NULL for an all-zero history
 *   base   [T,C]      in_dtype
 *   delta  [S,n,T,G]  in_dtype
 *   out    [S,n,C]    out_dtype; must not overlap x, hist, base or delta
 *
 * Accumulation is fp32; a bf16 output is rounded to nearest even once.
 * INVALID_ARG: S,n,C,T,G <= 0; C % G != 0; NULL x/base/delta/out; pointer not
 * 16-byte aligned; out overlapping an input.
 * UNSUPPORTED: C % 8 != 0 or (C/G) % 8 != 0 (8-channel vectors); T > 16;
 * in_dtype F32 with out_dtype BF16.
 */
int dflash2_dynconv(const void* x, const void* hist, const void* base, const void* delta,
                    void* out, int S, int n, int C, int T, int G,
                    int in_dtype, int out_dtype, void* stream);

/*
 * project(h): the dense d -> R map of each position's hidden state (PR
 * #27342, Overview: the hidden state is projected to the codebook rank; its
 * weight tensor is "selector_hidden").
 *   u[r,k] = sum_j h[r,j] * W[k,j]          (u = h W^T)
 *
 *   h  [P,d]  in_dtype
 *   W  [R,d]  in_dtype (K-major: each output column's weights are contiguous)
 *   u  [P,R]  fp32
 *
 * BF16 runs on the tcgen05 tensor cores (TMA-fed, fp32 accumulation in tensor
 * memory, split-K reduced deterministically through distributed shared memory
 * within a thread-block cluster).  F32 runs on the FP32 pipes.
 * INVALID_ARG: P,d,R <= 0; NULL pointer; misalignment.
 * UNSUPPORTED: d % 8 != 0; R % 8 != 0 or R > 512.
 */
int dflash2_project(const void* h, const void* W, float* u, int P, int d, int R,
                    int in_dtype, void* stream);

/*
 * Bytes of workspace dflash2_project_ws needs for these shapes on the current
 * device (0 when the projection is not split along d, or for bad sizes).
 */
size_t dflash2_project_workspace_bytes(int P, int d, int R);

/*
 * dflash2_project with a caller-provided split-K workspace (same operation and
 * result, bit for bit).  When the projection is split along d across the CTAs
 * of a cluster, the partial tiles are exchanged through this L2-resident
 * workspace (one cluster barrier) instead of through distributed shared
 * memory; this is faster for the few-row, deeply split shapes of a single
 * draft step.  workspace: device memory of at least
 * dflash2_project_workspace_bytes(P, d, R) bytes, 16-byte aligned, disjoint
 * from h, W and u, unused by anything else while the call runs (calls that
 * share one workspace must not overlap on the GPU); its contents on entry
 * are irrelevant and on exit undefined.  May be NULL when that size is 0.
 * F32 input ignores the workspace.  Errors as dflash2_project, plus
 * INVALID_ARG for a missing, short, misaligned or overlapping workspace.
 */
int dflash2_project_ws(const void* h, const void* W, float* u, int P, int d, int R,
                       int in_dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Edge scores with the fused per-predecessor argmax (PR #27342, Overview,
 * second formula).  For s < S, position i in 1..n-1 (the candidates of
 * position i-1 are the predecessors), slots p, c < K:
 *   e[s,i-1,p,c] = sum_r A[id_p,r] * u[s*n+i,r] * B[id_c,r] + unary[s,i,c]
 *   id_p = cand_ids[s,i-1,p],  id_c = cand_ids[s,i,c]
 *   best_slot[s,i-1,p]  = lowest c reaching max_c e[s,i-1,p,c]
 *   best_score[s,i-1,p] = that maximum
 *
 *   cand_ids   [S,n,K]        int32 token ids in [0,V)
 *   u          [S*n,R]        fp32 (the output of dflash2_project)
 *   A, B       [V,R]          cb_dtype codebooks
 *   unary      [S,n,K]        fp32
 *   edges_out  [S,n-1,K,K]    fp32, or NULL to skip writing the edge matrix
 *   best_slot  [S,n-1,K]      int32
 *   best_score [S,n-1,K]      fp32
 *   err_flag   one device int32 or NULL; DF2_FLAG_* bits are ORed into it
 *              (the caller zeroes it and reads it after its own sync).
 *
 * n == 1 has no transitions: returns DF2_OK having launched nothing (the three
 * outputs are empty and may be NULL).
 * An id outside [0,V) is clamped into range for the load and flagged
 * (DF2_FLAG_BAD_ID); the kernel never traps.  In BF16 mode the gate
 * A[id_p] (.) u is rounded to bf16 before the tensor-core contraction.
 * INVALID_ARG: S,n,K,R,V <= 0; NULL required pointer; misalignment.
 * UNSUPPORTED: K > 256; R % 8 != 0 or R > 512.
 */
int dflash2_edges(const int32_t* cand_ids, const float* u, const void* A, const void* B,
                  const float* unary, int S, int n, int K, int R, int V, int cb_dtype,
                  float* edges_out, int32_t* best_slot, float* best_score,
                  int32_t* err_flag, void* stream);

/*
 * The composite selector: the projection of every position's hidden state
 * (as dflash2_project, written to u_out) and the edge scores with the
 * per-predecessor argmax (as dflash2_edges, reading that projection).
 *   h [S*n,d], W [R,d] in `dtype`; A, B [V,R] in `dtype`; u_out [S*n,R] fp32
 *   (caller-owned; it receives u).
 * bf16 with K a power of two in [4,128], R = 64, 128 or 256, d % 8 == 0 and
 * n >= 2 runs as ONE kernel (see dflash2_select_plan): thread-block clusters
 * split d of a block of positions, reduce u through distributed shared memory,
 * and score the transitions into those positions from u held on chip, with the
 * first codebook gathers issued while h streams.  Other shapes run
 * dflash2_project then dflash2_edges on `stream`.  Same results either way
 * (within the bf16 tolerance: the d-sums are split differently).
 * Other arguments and errors as for those two calls.
 */
int dflash2_select(const void* h, const void* W, const int32_t* cand_ids, const void* A,
                   const void* B, const float* unary, int S, int n, int d, int K, int R,
                   int V, int dtype, float* u_out, float* edges_out, int32_t* best_slot,
                   float* best_score, int32_t* err_flag, void* stream);

/*
 * How dflash2_select runs these shapes on the current device (a query; nothing
 * is launched).  plan_out[4] receives:
 *   [0] 1 when the one-kernel selector runs (bf16; K a power of two in [4,128];
 *       R = 64, 128 or 256; d % 8 == 0; n >= 2; a cluster layout that fits),
 *       0 when the call runs dflash2_project and then dflash2_edges;
 *   [1] CTAs per thread-block cluster (the split of d), [2] clusters launched,
 *   [3] positions per cluster row block (0 when [0] is 0).
 * The first query for a shape measures cluster occupancy (CUDA runtime calls,
 * no launch) and caches the layout.
 * INVALID_ARG: NULL plan_out; S, n, d, K, R <= 0; bad dtype.
 */
int dflash2_select_plan(int S, int n, int d, int K, int R, int dtype, int* plan_out);

/*
 * dflash2_project for callers that cannot allocate device memory: plugins and
 * custom operators inside an inference runtime that owns the whole device pool
 * and hands them only their input and output tensors, or decode loops where an
 * allocation call (which may synchronise the device) is not allowed.  (No
 * counterpart in the DFlash2 pull request: this is a deployment convenience of
 * this library.)  Same operation and result as dflash2_project_ws, but the
 * split-K workspace is the library's own fixed 8 MiB device array, so nothing
 * is allocated.  The caller still passes h, W and u.
 *   - Shapes that need more than 8 MiB of workspace (see
 *     dflash2_project_workspace_bytes; e.g. more than 4096 rows at R = 128 on
 *     152 SMs) return DF2_ERR_UNSUPPORTED and launch nothing.
 *   - Every call looks up the array's device address in the current context
 *     (cudaGetSymbolAddress, with the device current); nothing is cached, so
 *     the address stays right after cudaDeviceReset or in another context.
 *     The first call on a device may load the library's device code: make it
 *     before any stream capture.
 *   - Every call on a device uses the same array, so calls that overlap on the
 *     GPU (different streams, or different host threads) race and give wrong
 *     results; serialise them.  The array keeps the last call's contents;
 *     nothing needs to start at zero.
 *   - F32 input uses no workspace.
 * Errors as dflash2_project, plus DF2_ERR_UNSUPPORTED for oversized shapes.
 */
int dflash2_project_noalloc(const void* h, const void* W, float* u, int P, int d, int R,
                            int in_dtype, void* stream);

/*
 * Top-K candidate extraction, the step that makes the selector's cand_ids and
 * unary from the draft's logits (ggml-org/llama.cpp pull request #27342, "spec
 * : add DFlash2 support (local convolution + candidate selector)", review
 * thread on the TOP_K kernel: the selector works on the top K candidates of
 * vocabulary-wide rows, with K small).
 *   logits   [rows,V] in `in_dtype` (DF2_F32 or DF2_BF16)
 *   cand_ids [rows,K] int32 out: the indices of the K largest entries of each
 *            row in descending order of value, equal values in ascending
 *            order of index (-0 and +0 are equal)
 *   values   [rows,K] fp32 out: logits[row, cand_ids[row,k]], exactly
 * A NaN entry is never selected; when a row holds fewer than K entries that
 * are not NaN, its remaining slots get id -1 and value NaN.  All three
 * buffers are caller-owned device memory; nothing is allocated.
 * INVALID_ARG: rows or V <= 0; K < 1 or K > V; NULL pointer; misalignment;
 * an output overlapping the logits or the other output.
 * UNSUPPORTED: K > 1024.
 */
int dflash2_topk(const void* logits, int rows, int V, int K, int in_dtype, int32_t* cand_ids,
                 float* values, void* stream);

/*
 * The convolution's dynamic taps predicted from its input (the pull request's
 * "predicted from the input" delta, tensor "*_conv_proj"; the pages give no
 * formula, so the reading is stated here): for every position p,
 *   delta[p, t*G + g] = sum_c Wc[t*G + g, c] * x[p, c]
 * i.e. delta [P, T*G] = x [P, C] . Wc [T*G, C]^T, written in `dtype` (bf16:
 * fp32 accumulation on the tensor cores, rounded to nearest even; fp32: fp32
 * throughout).  With P = S*n the output is the [S,n,T,G] delta that
 * dflash2_dynconv takes; this call is the unfused first half of that pair.
 * INVALID_ARG: P, C, TG <= 0; NULL pointer; misalignment; delta overlapping x
 * or Wc.  UNSUPPORTED: TG % 8 != 0 or TG > 512; bf16 with C % 8 != 0.
 */
int dflash2_predict_delta(const void* x, const void* Wc, void* delta, int P, int C, int TG,
                          int dtype, void* stream);

/*
 * The convolution with its taps predicted from its own input, in one kernel:
 * dflash2_predict_delta followed by dflash2_dynconv, without delta leaving the
 * chip and with x read from HBM once (same pull request, Overview: the conv's
 * per-position offsets are predicted from the input):
 *   delta[p, t, g] = rnd( sum_c Wc[t*G + g, c] * x[p, c] )       (p = s*n + i)
 *   out[s,i,c]     = sum_{t<T} (base[t,c] + delta[s*n+i, t, c/(C/G)]) * xh[s, i-t, c]
 * with xh as in dflash2_dynconv (x, else the history row, else zero); rnd
 * rounds to the input dtype (bf16: nearest even), as the unfused pair stores
 * delta between its two steps.
 *   x [S,n,C], hist [S,T-1,C] or NULL, base [T,C], Wc [T*G,C]: in_dtype;
 *   out [S,n,C]: out_dtype.  All caller-owned device memory.
 * bf16 input (bf16 or fp32 out): tcgen05 tensor cores for delta, fp32 FMA for
 * the conv.  fp32 input (fp32 out): delta in exact fp32 (no TF32) and no
 * rounding between the steps.
 * INVALID_ARG: S, n, C, T, G <= 0; C % G != 0; bad dtype; NULL pointer;
 * misalignment; out overlapping an input.
 * UNSUPPORTED: fp32 input with bf16 output; T > 8; C % 8 != 0 or (C/G) % 8 != 0;
 * (T*G) % 8 != 0 or T*G > 256; S*n >= 2^31; shapes whose working set does not
 * fit one CTA's shared memory.
 */
int dflash2_dynconv_predicted(const void* x, const void* hist, const void* base, const void* Wc,
                              void* out, int S, int n, int C, int T, int G, int in_dtype,
                              int out_dtype, void* stream);

/*
 * Greedy chain readout with a p_min cut: the draft tokens of each sequence,
 * read from the selector's per-predecessor argmax table (ggml-org/llama.cpp
 * pull request #27342: the Overview's readout is each predecessor's argmax
 * candidate; the merged tree names the DFlash2 draft path "selector + p_min";
 * the pages give no formula, so the readings are stated here):
 *   slot_0 = start_slot[s] if start_slot != NULL and start_slot[s] >= 0,
 *            else the argmax over k of unary[s,0,k] (lowest k on ties);
 *   slot_i = best_slot[s,i-1,slot_{i-1}]              (i = 1..n-1)
 *   p_0    = softmax_k(unary[s,0,:])[slot_0]
 *   p_i    = softmax_c(edges[s,i-1,slot_{i-1},:])[slot_i]
 *   tokens[s,i] = cand_ids[s,i,slot_i];  probs[s,i] = p_i (fp32)
 *   length[s]   = number of leading positions with p_i >= p_min.
 *   cand_ids, unary [S,n,K] (int32, fp32); edges [S,n-1,K,K] fp32 and
 *   best_slot [S,n-1,K] int32 as written by dflash2_edges / dflash2_select
 *   (edges_out must have been requested); both may be NULL when n == 1;
 *   start_slot [S] int32 or NULL; tokens, probs [S,n]; length [S] int32.
 * A slot outside [0,K) (from best_slot or start_slot) is clamped and flagged
 * in err_flag (DF2_FLAG_BAD_ID) when err_flag is not NULL.  Non-finite scores
 * are not supported.
 * INVALID_ARG: S, n, K <= 0; NULL required pointer; misalignment; an output
 * overlapping an input or another output.
 * UNSUPPORTED: (n-1)*K*4 + 8*n bytes of argmax table above 200 KB.
 */
int dflash2_chain(const int32_t* cand_ids, const float* unary, const float* edges,
                  const int32_t* best_slot, const int32_t* start_slot, int S, int n, int K,
                  float p_min, int32_t* tokens, float* probs, int32_t* length, int32_t* err_flag,
                  void* stream);

/*
 * Measurement aid (no counterpart in the DFlash2 pull request): the rate at
 * which this GPU gathers random rows, the bound the edge kernel's codebook
 * gathers work against.  For i < n_ids:
 *   out[i] = XOR of the 32-bit words of row ids[i] of table
 * where table is [rows, row_bytes] bytes and an id outside [0, rows) is
 * clamped into range.  Reads every gathered byte once; writes 4 bytes per id.
 * The rows are fetched as the edge kernels fetch codebook rows: one CTA per
 * SM with its ids staged in shared memory, 16-byte cp.async copies into a
 * shared-memory ring.
 *   table  device memory, rows * row_bytes bytes, 16-byte aligned
 *   ids    [n_ids] int32 device;  out [n_ids] uint32 device, disjoint from both
 * n_ids == 0 launches nothing.
 * INVALID_ARG: NULL pointer; rows <= 0; n_ids < 0; row_bytes not a power of
 * two in [16, 512]; misalignment; out overlapping table or ids.
 */
int dflash2_probe_gather(const void* table, long long rows, int row_bytes, const int32_t* ids,
                         int n_ids, uint32_t* out, void* stream);

/*
 * Phase trace of dflash2_select's one-kernel path, for a library built with
 * tracing (build.build_traced(): the selector compiled with -DDF2_TRACE; the
 * normal build returns DF2_ERR_UNSUPPORTED and records nothing).  Copies the
 * first `bytes` bytes of the trace table to host memory `host`, then zeroes the
 * table when `clear` is nonzero.  The table is 512 CTAs x 64 slots of uint64
 * global-timer readings (ns; 0 = not reached), written during each CTA's first
 * row block (slots 0, 1 and 31: every launch), so after one launch slot k of
 * CTA b is host[64*b + k]:
 *   0 entry, set-up done      1 previous grid complete (griddep wait)
 *   2 first TMA stage of h and W landed (MMA issuers)   3 last projection MMAs committed
 *   4 accumulators complete   5 cluster barrier passed (every projection of the cluster done)
 *   6 the CTA's partials received   7 partials summed, u slice written
 *   8 every edge unit's gathers issued
 *   9..14  edge units 0..5 issued (first gather warp)
 *   15..20 edge units 0..5 landed (gate warp)   21..26 units 0..5 MMAs committed
 *   27..30 units 0..3 scored (epilogue)   31 CTA exit
 *   56..59 units 0..3 landed, as seen by the second gate warp
 * Synchronises with nothing: call after the launch has completed.  Returns
 * DF2_OK, DF2_ERR_INVALID_ARG (NULL host, bytes < 0 or larger than the
 * table), DF2_ERR_UNSUPPORTED or DF2_ERR_CUDA.
 */
int dflash2_trace_read(uint64_t* host, int bytes, int clear);

/*
 * Row trace of dflash2_topk's streaming kernel (K <= 256, more rows than the
 * few-row kernel takes), for a library built with tracing as above; the normal
 * build returns DF2_ERR_UNSUPPORTED.  Same copy / clear / return conventions as
 * dflash2_trace_read.  The table is 1024 CTAs x 64 slots of uint64 global-timer
 * readings (ns; 0 = not reached): slot 8*j + k of CTA b is point k of the CTA's
 * j-th traced row, the traced rows being the CTA's rows 0, 1, 2, 3, 10, 11, 12
 * and 13 (its row iterations, in order):
 *   0 filter warp 0 reaches the row   1 ... after waiting for the selector
 *                                       (the filters run at most one row ahead)
 *   2 the row's first stage (the threshold seeding) processed
 *   3 filter warp 0 done with the row   7 filter warp 7 done with the row
 *   4 the selector done with the row
 *   5 the producer issued the row's first stage   6 ... its last stage
 */
int dflash2_trace_read_topk(uint64_t* host, int bytes, int clear);

/*
 * Reads and clears the library's device-side fault word for the current
 * device (DF2_FLAG_TIMEOUT when a bounded wait inside dflash2_dynconv,
 * dflash2_dynconv_predicted, dflash2_project or dflash2_topk gave up; DF2_FLAG_OVERFLOW from
 * dflash2_topk).  Synchronises the current device.  Returns DF2_OK or
 * DF2_ERR_CUDA.
 */
int dflash2_take_device_faults(int32_t* flags_out);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H_ */
