// abi.cu -- the extern "C" entry points of libattnres.so (declared in
// include/attnres.h): argument checks, then dispatch to the kernels.
// Nothing here allocates device memory, synchronises, prints or aborts.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "common.cuh"
#include "launch.h"

namespace attnres {

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  int &c = cache[dev & 63];
  if (c == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) v = 1;
    c = v;
  }
  return c;
}

namespace {
std::atomic<long long> g_wait_limit{0};   // 0: the default
}  // namespace

long long wait_limit_cycles() {
  const long long v = g_wait_limit.load(std::memory_order_relaxed);
  return v > 0 ? v : kDrainLimitCycles;
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int vec_elems(int dtype) { return dtype == ATTNRES_BF16 ? 8 : 4; }

// Common checks for a [B,T,D] problem; rows receives B*T.
int check_rows(int64_t B, int64_t T, int64_t D, int dtype, int64_t &rows) {
  if (dtype != ATTNRES_F32 && dtype != ATTNRES_BF16) return ATTNRES_ERR_DTYPE;
  if (B < 0 || T < 0 || D < 1 || D > (int64_t)1 << 20) return ATTNRES_ERR_SHAPE;
  if (T != 0 && B > INT64_MAX / T) return ATTNRES_ERR_SHAPE;
  if (D % vec_elems(dtype) != 0) return ATTNRES_ERR_ALIGNMENT;
  rows = B * T;
  return ATTNRES_OK;
}

int check_eps(float eps) {
  return (std::isfinite(eps) && eps >= 0.f) ? ATTNRES_OK : ATTNRES_ERR_VALUE;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTNRES_OK : ATTNRES_ERR_CUDA; }

// The checks both backward entry points make on everything but the workspace;
// rows receives B*T.  With no token rows, only the query and the parameter
// gradients must be valid (the data pointers of empty tensors may be NULL).
int backward_checks(const void *const *sources, int n, int64_t B, int64_t T, int64_t D, int dtype,
                    const float *query, const float *gain, float eps, const void *grad_out,
                    void *const *grad_sources, int accumulate, const float *grad_query, const float *grad_gain,
                    int64_t &rows) {
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (n < 1) return ATTNRES_ERR_SHAPE;
  if (n > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_TOO_MANY_SOURCES;
  if ((st = check_eps(eps))) return st;
  if (accumulate != 0 && accumulate != 1) return ATTNRES_ERR_VALUE;
  if (!aggregate_backward_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  if (!query) return ATTNRES_ERR_NULL;
  if ((grad_query && !aligned16(grad_query)) || (grad_gain && !aligned16(grad_gain)) || !aligned16(query) ||
      (gain && !aligned16(gain)))
    return ATTNRES_ERR_ALIGNMENT;
  if (rows == 0) return ATTNRES_OK;
  if (!sources || !grad_out || !grad_sources) return ATTNRES_ERR_NULL;
  for (int i = 0; i < n; ++i) {
    if (!sources[i] || !grad_sources[i]) return ATTNRES_ERR_NULL;
    if (!aligned16(sources[i]) || !aligned16(grad_sources[i])) return ATTNRES_ERR_ALIGNMENT;
  }
  if (!aligned16(grad_out)) return ATTNRES_ERR_ALIGNMENT;
  return ATTNRES_OK;
}

}  // namespace
}  // namespace attnres

using namespace attnres;

extern "C" {

const char *attnres_status_string(int status) {
  switch (status) {
    case ATTNRES_OK: return "ok";
    case ATTNRES_ERR_NULL: return "a required pointer is NULL";
    case ATTNRES_ERR_SHAPE: return "a size (n, S, L, B, T or D) is out of range";
    case ATTNRES_ERR_DTYPE: return "dtype must be ATTNRES_F32 or ATTNRES_BF16";
    case ATTNRES_ERR_ALIGNMENT: return "pointers must be 16-byte aligned and D a multiple of the vector width";
    case ATTNRES_ERR_TOO_MANY_SOURCES: return "too many sources for one call";
    case ATTNRES_ERR_CUDA: return "a CUDA launch failed";
    case ATTNRES_ERR_CAPACITY: return "a host output buffer is too small";
    case ATTNRES_ERR_VALUE: return "a value is invalid (eps negative or not finite, block size 0)";
    case ATTNRES_ERR_TIMEOUT: return "a kernel wait ran out of time and gave up (results invalid)";
    case ATTNRES_ERR_SCRATCH: return "the request needs more than the library's fixed scratch";
    default: return "unknown status";
  }
}

int attnres_depth_aggregate(const void *const *sources, int n, int64_t B, int64_t T, int64_t D,
                            int dtype, const float *query, const float *gain, float eps, void *out,
                            float *out_max, float *out_lse, void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (n < 1) return ATTNRES_ERR_SHAPE;
  if (n > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_TOO_MANY_SOURCES;
  if ((st = check_eps(eps))) return st;
  if (!aggregate_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  if (rows == 0) return ATTNRES_OK;  // empty tensors may carry NULL data pointers
  if (!sources || !query || !out) return ATTNRES_ERR_NULL;
  for (int i = 0; i < n; ++i) {
    if (!sources[i]) return ATTNRES_ERR_NULL;
    if (!aligned16(sources[i])) return ATTNRES_ERR_ALIGNMENT;
  }
  if (!aligned16(query) || (gain && !aligned16(gain)) || !aligned16(out)) return ATTNRES_ERR_ALIGNMENT;
  AggregateArgs a{sources, n, rows, (int)D, dtype, query, gain, nullptr, eps, out, out_max, out_lse,
                  static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_aggregate(a));
}

int attnres_block_phase1(const void *const *blocks, int n_blocks, int64_t B, int64_t T, int64_t D,
                         int dtype, const float *queries, const float *gains, int S, float eps,
                         void *out, float *out_max, float *out_lse, void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (n_blocks < 1 || S < 1 || S > ATTNRES_MAX_QUERIES) return ATTNRES_ERR_SHAPE;
  if (n_blocks > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_TOO_MANY_SOURCES;
  if ((st = check_eps(eps))) return st;
  if ((st = phase1_check(n_blocks, (int)D, dtype, S))) return st;
  if (rows == 0) return ATTNRES_OK;
  if (!blocks || !queries || !out || !out_lse) return ATTNRES_ERR_NULL;
  for (int i = 0; i < n_blocks; ++i) {
    if (!blocks[i]) return ATTNRES_ERR_NULL;
    if (!aligned16(blocks[i])) return ATTNRES_ERR_ALIGNMENT;
  }
  if (!aligned16(queries) || (gains && !aligned16(gains)) || !aligned16(out)) return ATTNRES_ERR_ALIGNMENT;
  Phase1Args a{blocks, n_blocks, rows, (int)D, dtype, queries, gains, S, eps, out, out_max, out_lse,
               static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_phase1(a));
}

int attnres_block_phase2_merge(const void *inter_out, const float *inter_lse, const void *partial,
                               int64_t B, int64_t T, int64_t D, int dtype, const float *query,
                               const float *gain, float eps, void *h_out, float *out_lse,
                               void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if ((st = check_eps(eps))) return st;
  if (!merge_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  if (rows == 0) return ATTNRES_OK;
  if (!inter_out || !inter_lse || !query || !h_out) return ATTNRES_ERR_NULL;
  if (!aligned16(inter_out) || (partial && !aligned16(partial)) || !aligned16(query) ||
      (gain && !aligned16(gain)) || !aligned16(h_out))
    return ATTNRES_ERR_ALIGNMENT;
  MergeArgs a{inter_out, inter_lse, partial, rows, (int)D, dtype, query, gain, eps, h_out, out_lse,
              static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_merge(a));
}

int attnres_block_merge_update(const void *inter_out, const float *inter_lse, const void *partial_in,
                               const void *sub_out, const float *u, int64_t B, int64_t T, int64_t D,
                               int dtype, const float *query, const float *gain, float eps,
                               void *partial_out, void *h_out, float *out_lse,
                               const float *norm_weight, float norm_eps, void *normed_out,
                               void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if ((st = check_eps(eps))) return st;
  if (norm_weight && (st = check_eps(norm_eps))) return st;
  if (!merge_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  if (rows == 0) return ATTNRES_OK;
  if (!inter_out || !inter_lse || !sub_out || !query || !partial_out) return ATTNRES_ERR_NULL;
  if (!norm_weight != !normed_out) return ATTNRES_ERR_NULL;   // both or neither
  if (!h_out && !normed_out) return ATTNRES_ERR_NULL;         // something must be written
  if (!aligned16(inter_out) || (partial_in && !aligned16(partial_in)) || !aligned16(sub_out) ||
      (u && !aligned16(u)) || !aligned16(query) || (gain && !aligned16(gain)) ||
      !aligned16(partial_out) || (h_out && !aligned16(h_out)) ||
      (norm_weight && (!aligned16(norm_weight) || !aligned16(normed_out))))
    return ATTNRES_ERR_ALIGNMENT;
  MergeUpdateArgs m{inter_out, inter_lse, partial_in, sub_out, u, rows, (int)D, dtype, query, gain, eps,
                    partial_out, h_out, out_lse, norm_weight, norm_eps, normed_out,
                    static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_merge_update(m));
}

int attnres_rms_norm(const void *x, int64_t B, int64_t T, int64_t D, int dtype, const float *weight,
                     float eps, void *y, void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if ((st = check_eps(eps))) return st;
  if (!merge_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  if (rows == 0) return ATTNRES_OK;
  if (!x || !weight || !y) return ATTNRES_ERR_NULL;
  if (!aligned16(x) || !aligned16(weight) || !aligned16(y)) return ATTNRES_ERR_ALIGNMENT;
  RmsNormArgs a{x, rows, (int)D, dtype, weight, eps, y, static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_rms_norm(a));
}

int attnres_depth_aggregate_backward(const void *const *sources, int n, int64_t B, int64_t T, int64_t D,
                                     int dtype, const float *query, const float *gain, float eps,
                                     const void *grad_out, void *const *grad_sources, int accumulate,
                                     float *grad_query, float *grad_gain, float *workspace,
                                     int64_t workspace_rows, void *stream) {
  int64_t rows = 0;
  int st = backward_checks(sources, n, B, T, D, dtype, query, gain, eps, grad_out, grad_sources, accumulate,
                           grad_query, grad_gain, rows);
  if (st) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rows == 0) {  // no token rows: the parameter gradients are zero, nothing else is touched
    if (grad_query && cudaMemsetAsync(grad_query, 0, (size_t)D * sizeof(float), s) != cudaSuccess)
      return ATTNRES_ERR_CUDA;
    if (grad_gain && cudaMemsetAsync(grad_gain, 0, (size_t)D * sizeof(float), s) != cudaSuccess)
      return ATTNRES_ERR_CUDA;
    return ATTNRES_OK;
  }
  if (grad_query || grad_gain) {
    if (!workspace) return ATTNRES_ERR_NULL;
    if (!aligned16(workspace)) return ATTNRES_ERR_ALIGNMENT;
    if (workspace_rows < aggregate_backward_rows_per_partial((int)D, dtype)) return ATTNRES_ERR_CAPACITY;
  }
  AggregateBackwardArgs a{sources, n, rows, (int)D, dtype, query, gain, eps, grad_out, grad_sources,
                          accumulate != 0, grad_query, grad_gain, workspace, workspace_rows, s};
  return cuda_status(launch_aggregate_backward(a));
}

int attnres_depth_aggregate_backward_noalloc(const void *const *sources, int n, int64_t B, int64_t T,
                                             int64_t D, int dtype, const float *query, const float *gain,
                                             float eps, const void *grad_out, void *const *grad_sources,
                                             int accumulate, float *grad_query, float *grad_gain,
                                             void *stream) {
  // Every argument is checked before the scratch is looked up, so a bad
  // argument reports its own status; empty inputs and calls without a
  // parameter gradient need no scratch at all.
  int64_t rows = 0;
  int st = backward_checks(sources, n, B, T, D, dtype, query, gain, eps, grad_out, grad_sources, accumulate,
                           grad_query, grad_gain, rows);
  if (st) return st;
  float *scratch = nullptr;
  int64_t scratch_rows = 0;
  if (rows > 0 && (grad_query || grad_gain)) {
    scratch_rows = noalloc_scratch_floats() / D;
    if (scratch_rows < aggregate_backward_rows_per_partial((int)D, dtype)) return ATTNRES_ERR_SCRATCH;
    if (noalloc_scratch(scratch) != cudaSuccess) return ATTNRES_ERR_CUDA;
  }
  return attnres_depth_aggregate_backward(sources, n, B, T, D, dtype, query, gain, eps, grad_out, grad_sources,
                                          accumulate, grad_query, grad_gain, scratch, scratch_rows, stream);
}

int64_t attnres_depth_aggregate_backward_workspace_rows(int64_t D, int dtype) {
  int64_t rows = 0;
  int st = check_rows(1, 1, D, dtype, rows);
  if (st) return st;
  if (!aggregate_backward_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  int64_t p = 0;
  if (aggregate_backward_workspace_rows((int)D, dtype, p) != cudaSuccess) return ATTNRES_ERR_CUDA;
  return p;
}

int attnres_partial_update(const void *h, const void *partial_in, const float *u, int64_t B,
                           int64_t T, int64_t D, int dtype, void *partial_out, void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (rows == 0) return ATTNRES_OK;
  if (!h || !u || !partial_out) return ATTNRES_ERR_NULL;
  if (!aligned16(h) || (partial_in && !aligned16(partial_in)) || !aligned16(u) ||
      !aligned16(partial_out))
    return ATTNRES_ERR_ALIGNMENT;
  PartialUpdateArgs a{h, partial_in, u, rows, (int)D, dtype, partial_out,
                      static_cast<cudaStream_t>(stream)};
  return cuda_status(launch_partial_update(a));
}

int attnres_full_stack_forward(void *const *sources, int L, int64_t B, int64_t T, int64_t D,
                               int dtype, const float *queries, const float *gains, const float *u,
                               float eps, void *y_out, void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (L < 1) return ATTNRES_ERR_SHAPE;
  if (L + 1 > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_TOO_MANY_SOURCES;
  if ((st = check_eps(eps))) return st;
  if (!aggregate_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  if (rows == 0) return ATTNRES_OK;
  if (!sources || !queries || !u || !y_out) return ATTNRES_ERR_NULL;
  for (int l = 0; l <= L; ++l) {
    if (!sources[l]) return ATTNRES_ERR_NULL;
    if (!aligned16(sources[l])) return ATTNRES_ERR_ALIGNMENT;
  }
  if (!aligned16(queries) || (gains && !aligned16(gains)) || !aligned16(u) || !aligned16(y_out))
    return ATTNRES_ERR_ALIGNMENT;
  // Rows of queries / gains / u stay 16-byte aligned: D % 4 == 0 holds for
  // both dtypes after check_rows.
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void *const *srcs = const_cast<const void *const *>(sources);
  for (int l = 1; l <= L; ++l) {
    AggregateArgs a{srcs, l, rows, (int)D, dtype, queries + (size_t)(l - 1) * D,
                    gains ? gains + (size_t)(l - 1) * D : nullptr, u + (size_t)(l - 1) * D, eps,
                    sources[l], nullptr, nullptr, s};
    if ((st = cuda_status(launch_aggregate(a)))) return st;
  }
  AggregateArgs fin{srcs, L + 1, rows, (int)D, dtype, queries + (size_t)L * D,
                    gains ? gains + (size_t)L * D : nullptr, nullptr, eps, y_out, nullptr, nullptr, s};
  return cuda_status(launch_aggregate(fin));
}

namespace {

// Workspace layout of attnres_full_stack_two_phase: the phase-1 outputs of
// one block [S, rows, D], their lse [S, rows] fp32, and the raw-score /
// alpha buffer [rows, n, S] fp32 of the widest block (when it has more than
// ten sources); each part 256-byte aligned.
struct TwoPhaseLayout {
  size_t o, lse, scores, total;
};

int64_t full_two_phase_widest(int L, int S) { return (int64_t)((L - 1) / S) * S + 1; }

TwoPhaseLayout full_two_phase_layout(int L, int S, int64_t rows, int64_t D, int dtype) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  TwoPhaseLayout w;
  const size_t elt = dtype == ATTNRES_BF16 ? 2 : 4;
  w.o = 0;
  w.lse = up((size_t)S * rows * D * elt);
  w.scores = w.lse + up((size_t)S * rows * sizeof(float));
  const int64_t n_max = full_two_phase_widest(L, S);
  w.total = w.scores + (n_max > kP1TcMaxSources ? up((size_t)rows * n_max * S * sizeof(float)) : 0);
  return w;
}

// Phase 1 of a block with n sources and Sb queries: which kernel family takes it.
int full_two_phase_block_check(int n, int Sb, int64_t D, int dtype, int64_t rows) {
  if (n <= kP1TcMaxSources) return phase1_check(n, (int)D, dtype, Sb);
  return phase1_many_supported(n, (int)D, dtype, Sb, rows) ? ATTNRES_OK : ATTNRES_ERR_SHAPE;
}

}  // namespace

int64_t attnres_full_stack_two_phase_workspace_bytes(int L, int S, int64_t B, int64_t T, int64_t D, int dtype) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (L < 1 || S < 1) return ATTNRES_ERR_SHAPE;
  return (int64_t)full_two_phase_layout(L, S, rows, D, dtype).total;
}

int attnres_full_stack_two_phase(void *const *sources, int L, int S, int64_t B, int64_t T, int64_t D,
                                 int dtype, const float *queries, const float *gains, const float *u,
                                 float eps, void *y_out, void *workspace, int64_t workspace_bytes,
                                 void *stream) {
  int64_t rows = 0;
  int st = check_rows(B, T, D, dtype, rows);
  if (st) return st;
  if (L < 1 || S < 1 || S > ATTNRES_MAX_QUERIES) return ATTNRES_ERR_SHAPE;
  if (L + 1 > ATTNRES_MAX_SOURCES) return ATTNRES_ERR_TOO_MANY_SOURCES;
  if ((st = check_eps(eps))) return st;
  if (!aggregate_supported((int)D, dtype)) return ATTNRES_ERR_SHAPE;
  for (int start = 0; start < L; start += S) {
    const int Sb = start + S < L ? S : L - start;
    if ((st = full_two_phase_block_check(start + 1, Sb, D, dtype, rows))) return st;
  }
  if (rows == 0) return ATTNRES_OK;
  if (!sources || !queries || !u || !y_out || !workspace) return ATTNRES_ERR_NULL;
  for (int l = 0; l <= L; ++l) {
    if (!sources[l]) return ATTNRES_ERR_NULL;
    if (!aligned16(sources[l])) return ATTNRES_ERR_ALIGNMENT;
  }
  if (!aligned16(queries) || (gains && !aligned16(gains)) || !aligned16(u) || !aligned16(y_out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTNRES_ERR_ALIGNMENT;
  const TwoPhaseLayout w = full_two_phase_layout(L, S, rows, D, dtype);
  if (workspace_bytes < (int64_t)w.total) return ATTNRES_ERR_CAPACITY;
  char *ws = static_cast<char *>(workspace);
  void *o = ws + w.o;
  float *lse = reinterpret_cast<float *>(ws + w.lse);
  float *scores = reinterpret_cast<float *>(ws + w.scores);
  const size_t o_step = (size_t)rows * D * (dtype == ATTNRES_BF16 ? 2 : 4);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const void *const *srcs = const_cast<const void *const *>(sources);
  for (int start = 0; start < L; start += S) {
    const int Sb = start + S < L ? S : L - start;   // sublayers start+1 .. start+Sb
    const int n = start + 1;                         // sources completed before the block
    const float *qb = queries + (size_t)start * D;
    const float *gb = gains ? gains + (size_t)start * D : nullptr;
    // phase 1: the block's Sb queries over v_0 .. v_start, one pass
    if (n <= kP1TcMaxSources) {
      Phase1Args a{srcs, n, rows, (int)D, dtype, qb, gb, Sb, eps, o, nullptr, lse, s};
      if ((st = cuda_status(launch_phase1(a)))) return st;
    } else {
      Phase1ManyArgs a{srcs, n, rows, (int)D, qb, gb, Sb, eps, o, nullptr, lse, scores, s};
      if ((st = cuda_status(launch_phase1_many(a)))) return st;
    }
    // phase 2: each sublayer merges its intra-block sources into its phase-1
    // state, then applies f (fused) and stores v_l
    for (int j = 0; j < Sb; ++j) {
      const int l = start + 1 + j;
      AggregateArgs a{srcs + start + 1, j, rows, (int)D, dtype, queries + (size_t)(l - 1) * D,
                      gains ? gains + (size_t)(l - 1) * D : nullptr, u + (size_t)(l - 1) * D, eps,
                      sources[l], nullptr, nullptr, s};
      a.prior_o = static_cast<const char *>(o) + (size_t)j * o_step;
      a.prior_lse = lse + (size_t)j * rows;
      if ((st = cuda_status(launch_aggregate(a)))) return st;
    }
  }
  AggregateArgs fin{srcs, L + 1, rows, (int)D, dtype, queries + (size_t)L * D,
                    gains ? gains + (size_t)L * D : nullptr, nullptr, eps, y_out, nullptr, nullptr, s};
  return cuda_status(launch_aggregate(fin));
}

int attnres_set_wait_limit(int64_t cycles) {
  if (cycles < 0) return ATTNRES_ERR_VALUE;
  g_wait_limit.store((long long)cycles, std::memory_order_relaxed);
  return ATTNRES_OK;
}

int attnres_take_device_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTNRES_ERR_CUDA;
  const unsigned int f = take_error_aggregate() | take_error_merge() | take_error_phase1() |
                           take_error_phase1_tc();
  if (f & 2u) return ATTNRES_ERR_CUDA;
  return f ? ATTNRES_ERR_TIMEOUT : ATTNRES_OK;
}

int attnres_block_schedule(int num_atomic, int block_size, int *n_sources_per_layer,
                           int *source_ids, int capacity) {
  if (num_atomic < 1) return ATTNRES_ERR_SHAPE;
  if (block_size < 1) return ATTNRES_ERR_VALUE;
  if (!n_sources_per_layer || !source_ids) return ATTNRES_ERR_NULL;
  if (capacity < 0) return ATTNRES_ERR_CAPACITY;
  // Completed blocks so far (block 0 = embedding) and whether a running
  // partial exists.  Sublayer idx closes its block when idx % block_size == 0
  // or it is the last sublayer.
  int completed = 1;
  bool partial = false;
  int written = 0;
  for (int idx = 1; idx <= num_atomic; ++idx) {
    const int count = completed + (partial ? 1 : 0);
    if (written + count > capacity) return ATTNRES_ERR_CAPACITY;
    for (int b = 0; b < completed; ++b) source_ids[written++] = b;
    if (partial) source_ids[written++] = -1;
    n_sources_per_layer[idx - 1] = count;
    partial = true;
    if (idx % block_size == 0 || idx == num_atomic) {
      ++completed;
      partial = false;
    }
  }
  if (written + completed > capacity) return ATTNRES_ERR_CAPACITY;
  for (int b = 0; b < completed; ++b) source_ids[written++] = b;
  n_sources_per_layer[num_atomic] = completed;
  return written;
}

int attnres_atomic_block_size(int num_hidden_layers, int attnres_block_size) {
  if (num_hidden_layers < 1) return ATTNRES_ERR_SHAPE;
  if (attnres_block_size == 0) return ATTNRES_ERR_VALUE;
  int decoder_blocks = attnres_block_size > 0 ? attnres_block_size : (num_hidden_layers + 7) / 8;
  if (decoder_blocks < 1) decoder_blocks = 1;
  return 2 * decoder_blocks;
}

}  // extern "C"
