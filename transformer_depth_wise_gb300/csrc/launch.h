// launch.h -- internal launchers behind the C ABI.  Arguments reaching these
// functions have already been validated by the entry points in abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace attnres {

// Streaming-multiprocessor count of the current device (cached per device).
int sm_count();

// SM clock cycles an in-kernel wait of a launch's work loop may take before
// it gives up (attnres_set_wait_limit; about 2 s by default).
long long wait_limit_cycles();

struct AggregateArgs {
  const void *const *sources;  // host array of n device pointers
  int n;
  int64_t rows;                // B * T
  int D;
  int dtype;
  const float *query;          // [D]
  const float *gain;           // [D] or nullptr
  const float *u;              // [D]: apply f(h) = 0.5 tanh(u h) before storing, or nullptr
  float eps;
  void *out;                   // [rows, D]
  float *out_max;              // [rows] or nullptr
  float *out_lse;              // [rows] or nullptr
  cudaStream_t stream;
  // Start every row from the normalised state (lse, o, 1) of an earlier
  // partial softmax (then n may be 0): the merge of further sources into it.
  const void *prior_o = nullptr;     // [rows, D]
  const float *prior_lse = nullptr;  // [rows]
};
// Returns false when D is beyond what the kernel family covers.
bool aggregate_supported(int D, int dtype);
cudaError_t launch_aggregate(const AggregateArgs &a);

struct AggregateBackwardArgs {
  const void *const *sources;  // n device pointers [rows, D]
  int n;
  int64_t rows;
  int D;
  int dtype;
  const float *query;
  const float *gain;           // or nullptr
  float eps;
  const void *grad_out;        // [rows, D] dh
  void *const *grad_sources;   // n device pointers [rows, D]
  bool accumulate;             // grad_sources[i] += (else =)
  float *grad_query;           // [D] or nullptr
  float *grad_gain;            // [D] or nullptr
  float *workspace;            // [workspace_rows, D] fp32 partials (needed with grad_query / grad_gain)
  int64_t workspace_rows;
  cudaStream_t stream;
};
bool aggregate_backward_supported(int D, int dtype);
int aggregate_backward_rows_per_partial(int D, int dtype);
cudaError_t aggregate_backward_workspace_rows(int D, int dtype, int64_t &rows);
cudaError_t launch_aggregate_backward(const AggregateBackwardArgs &a);
int64_t noalloc_scratch_floats();
cudaError_t noalloc_scratch(float *&ptr);  // fixed scratch of the current device

struct MergeArgs {
  const void *inter_out;       // [rows, D]
  const float *inter_lse;      // [rows]
  const void *partial;         // [rows, D] or nullptr
  int64_t rows;
  int D;
  int dtype;
  const float *query;
  const float *gain;
  float eps;
  void *h_out;
  float *out_lse;
  cudaStream_t stream;
};
bool merge_supported(int D, int dtype);
cudaError_t launch_merge(const MergeArgs &a);

struct MergeUpdateArgs {
  const void *inter_out;       // [rows, D]: phase-1 output o_k
  const float *inter_lse;      // [rows]
  const void *partial_in;      // [rows, D] p_{k-2} or nullptr
  const void *sub_out;         // [rows, D] sublayer output (or input, with u)
  const float *u;              // [D] synthetic sublayer, or nullptr
  int64_t rows;
  int D;
  int dtype;
  const float *query;
  const float *gain;
  float eps;
  void *partial_out;           // [rows, D] p_{k-1}
  void *h_out;                 // [rows, D] h_k, or nullptr
  float *out_lse;
  const float *norm_weight;    // [D] pre-norm weight, or nullptr
  float norm_eps;
  void *normed_out;            // [rows, D] RMSNorm(h_k) (.) norm_weight, or nullptr
  cudaStream_t stream;
};
cudaError_t launch_merge_update(const MergeUpdateArgs &a);

struct RmsNormArgs {
  const void *x;               // [rows, D]
  int64_t rows;
  int D;
  int dtype;
  const float *weight;         // [D]
  float eps;
  void *y;                     // [rows, D], may alias x
  cudaStream_t stream;
};
cudaError_t launch_rms_norm(const RmsNormArgs &a);

struct PartialUpdateArgs {
  const void *h;
  const void *partial_in;      // or nullptr
  const float *u;
  int64_t rows;
  int D;
  int dtype;
  void *partial_out;
  cudaStream_t stream;
};
cudaError_t launch_partial_update(const PartialUpdateArgs &a);

struct Phase1Args {
  const void *const *blocks;   // host array of n device pointers
  int n;
  int64_t rows;
  int D;
  int dtype;
  const float *queries;        // [S, D]
  const float *gains;          // [S, D] or nullptr
  int S;
  float eps;
  void *out;                   // [S, rows, D]
  float *out_max;              // [S, rows] or nullptr
  float *out_lse;              // [S, rows]
  cudaStream_t stream;
};
// Returns ATTNRES_OK or a (negative) status for shapes the kernels cannot take.
int phase1_check(int n, int D, int dtype, int S);
cudaError_t launch_phase1(const Phase1Args &a);
// Tensor-core phase 1 (bf16, D a multiple of 64 up to 8192, n <= 10, S <= 24).
bool phase1_tc_supported(int n, int D, int dtype, int S);
cudaError_t launch_phase1_tc(const Phase1Args &a);
// Feature slices the tensor-core path splits the scores into for few token
// rows (partial sums in the tokens' o[1] rows), or 1 when it does not.
int split_parts(const Phase1Args &a);

// Phase 1 over any number of summaries (bf16): tensor-core scores, five
// summaries per work item, into a raw-score buffer, a softmax over all of
// them, then the outputs.  scores: [rows][n][S] fp32 scratch, left holding
// alpha.
// Most summaries the fused phase-1 path takes in one pass (its TMEM holds
// ten sources' scores); wider blocks go through the raw-score path below.
constexpr int kP1TcMaxSources = 10;

struct Phase1ManyArgs {
  const void *const *blocks;
  int n;
  int64_t rows;
  int D;
  const float *queries;        // [S, D]
  const float *gains;          // [S, D] or nullptr
  int S;
  float eps;
  void *out;                   // [S, rows, D] bf16
  float *out_max;              // [S, rows] or nullptr
  float *out_lse;              // [S, rows]
  float *scores;               // [rows, n, S]
  cudaStream_t stream;
};
bool phase1_many_supported(int n, int D, int dtype, int S, int64_t rows);
cudaError_t launch_phase1_many(const Phase1ManyArgs &a);

// Read and clear the per-file flag that records a kernel wait that ran out
// (non-zero: at least one wait gave up).
unsigned int take_error_aggregate();
unsigned int take_error_merge();
unsigned int take_error_phase1();
unsigned int take_error_phase1_tc();

}  // namespace attnres
