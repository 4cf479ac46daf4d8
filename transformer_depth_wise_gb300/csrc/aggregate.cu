// aggregate.cu -- depth aggregation kernel (eq. A1-A3 of "Attention Residual
// 深度残差", "DepthResidual.forward"), one pass over the sources.
//
// A "team" of threads owns one token row; each thread owns VPT 16-byte
// vectors of the row (vector j = lane + k * team_size, so the team's loads
// are contiguous).  Sources are streamed in groups of G: the team loads G
// rows, reduces the G dot products w~.v and sums of squares v.v, turns them
// into scores s = (w~.v) * rsqrt(v.v / D + eps) (the RMS factored out of the
// dot), and folds the group into a running online-softmax state (m, denom,
// acc[]) held in registers (eq. OS1 / OS2).  No [n, B, T] score tensor ever
// exists; each source byte is read from HBM once.
//
// The same kernel, with u != nullptr, applies the synthetic sublayer
// v = 0.5 tanh(u (.) h) to the fp32 h before the single rounding store: the
// Full stack uses it so h_l never round-trips through memory.
#include "common.cuh"
#include "launch.h"

ATTNRES_DEFINE_ERROR_FLAG(take_error_aggregate)

namespace attnres {

struct AggParams {
  const void *src[kMaxSources];
  int n;
  int nvec;      // 16-byte vectors per row
  int D;
  float inv_D;
  float eps;
  int64_t rows;
  const float *q;
  const float *g;
  const float *u;
  void *out;
  float *out_max;
  float *out_lse;
  const void *prior_o;     // [rows, D] normalised prior state (o, lse), or nullptr
  const float *prior_lse;  // [rows]
};

constexpr int kGroup = 4;  // sources per reduction step

// TEAM > 0: TEAM lanes of a warp own a row (several rows per CTA).
// TEAM == 0: the whole CTA owns a row.
template <typename T, int VPT, int TEAM, bool FUSED_F>
__global__ void __launch_bounds__(TEAM ? 256 : 512)
aggregate_kernel(const __grid_constant__ AggParams p) {
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  constexpr int NE = VPT * EPV;
  constexpr int G = kGroup;
  __shared__ float red[TEAM ? 1 : 2 * 32 * 2 * G];

  const int tpr = TEAM ? TEAM : blockDim.x;
  const int lt = TEAM ? (threadIdx.x % TEAM) : threadIdx.x;
  const int teams_per_cta = TEAM ? blockDim.x / TEAM : 1;
  const int team = TEAM ? threadIdx.x / TEAM : 0;

  // Folded query w~ = w (.) gamma for this thread's elements, as packed
  // pairs (and u).
  using PR = Pairs<T>;
  constexpr int NP = PR::NP;
  float qe[NE];
  float ue[FUSED_F ? NE : 1];
  bool valid[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int j = lt + k * tpr;
    valid[k] = j < p.nvec;
#pragma unroll
    for (int e4 = 0; e4 < EPV; e4 += 4) {
      float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f), g4 = make_float4(1.f, 1.f, 1.f, 1.f);
      float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (valid[k]) {
        w4 = ld_f4(p.q + j * EPV + e4);
        if (p.g) g4 = ld_f4(p.g + j * EPV + e4);
        if (FUSED_F) u4 = ld_f4(p.u + j * EPV + e4);
      }
      qe[k * EPV + e4 + 0] = w4.x * g4.x;
      qe[k * EPV + e4 + 1] = w4.y * g4.y;
      qe[k * EPV + e4 + 2] = w4.z * g4.z;
      qe[k * EPV + e4 + 3] = w4.w * g4.w;
      if (FUSED_F) {
        ue[k * EPV + e4 + 0] = u4.x; ue[k * EPV + e4 + 1] = u4.y;
        ue[k * EPV + e4 + 2] = u4.z; ue[k * EPV + e4 + 3] = u4.w;
      }
    }
  }

  uint64_t qp[VPT * NP];
#pragma unroll
  for (int j = 0; j < VPT * NP; ++j) qp[j] = pair(qe[2 * j], qe[2 * j + 1]);

  const size_t row_bytes = (size_t)p.D * sizeof(T);
  const int64_t groups = (p.rows + teams_per_cta - 1) / teams_per_cta;
  int parity = 0;
  // Every team of the CTA runs the same number of iterations (rows past the
  // end are masked), so warp shuffles and barriers stay uniform.
  // L2 lookahead: the team walks (row, source) in order; before loading a
  // group it asks L2 for the source rows kAhead positions further on
  // (crossing into the team's next rows), one bulk prefetch per source row,
  // lanes in turn.  No registers are held for them, the L2 footprint is
  // kAhead rows per team, and the group loads then hit L2.
  constexpr int kAhead = 2 * G;
  auto prefetch_src = [&](int64_t rgp, int i) {   // source i of the team's row group rgp (n >= 1)
    const int64_t r = rgp * teams_per_cta + team;
    if (rgp < groups && r < p.rows && i < p.n)
      prefetch_l2_bulk(static_cast<const char *>(p.src[i]) + (size_t)r * row_bytes, (uint32_t)row_bytes);
  };
  if (p.n > 0)
    for (int pos = lt; pos < kAhead; pos += tpr)
      prefetch_src(blockIdx.x + (int64_t)(pos / p.n) * gridDim.x, pos % p.n);
  for (int64_t rg = blockIdx.x; rg < groups; rg += gridDim.x) {
    const int64_t row = rg * teams_per_cta + team;
    const bool row_ok = row < p.rows;
    const size_t row_off = (size_t)row * row_bytes;
    uint64_t acc[VPT * NP];
#pragma unroll
    for (int j = 0; j < VPT * NP; ++j) acc[j] = 0ull;
    float m = -INFINITY, den = 0.f;
    if (p.prior_o) {  // start from the state (lse, o, 1): an earlier partial softmax
      if (row_ok) m = p.prior_lse[row];
      den = 1.f;
#pragma unroll
      for (int k = 0; k < VPT; ++k)
        if (row_ok && valid[k])
          PR::split(ld_stream(static_cast<const char *>(p.prior_o) + row_off + (size_t)(lt + k * tpr) * 16),
                    acc + k * NP);
    }

    for (int i0 = 0; i0 < p.n; i0 += G) {
      for (int g = lt; g < G; g += tpr) {  // kAhead sources past this group's g-th
        const int pos = i0 + kAhead + g;     // counted from the start of this row
        prefetch_src(rg + (int64_t)(pos / p.n) * gridDim.x, pos % p.n);
      }
      uint4 buf[G][VPT];
#pragma unroll
      for (int g = 0; g < G; ++g) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          buf[g][k] = make_uint4(0u, 0u, 0u, 0u);
          if (i0 + g < p.n && row_ok && valid[k])
            buf[g][k] = ld_stream(static_cast<const char *>(p.src[i0 + g]) + row_off +
                                  (size_t)(lt + k * tpr) * 16);
        }
      }
      float part[2 * G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint64_t dot = 0ull, ss = 0ull;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          uint64_t x[NP];
          PR::split(buf[g][k], x);
#pragma unroll
          for (int j = 0; j < NP; ++j) {
            fma_pair(dot, qp[k * NP + j], x[j]);
            fma_pair(ss, x[j], x[j]);
          }
        }
        part[2 * g] = pair_sum(dot);
        part[2 * g + 1] = pair_sum(ss);
      }
      if (TEAM) {
#pragma unroll
        for (int t = 0; t < 2 * G; ++t) part[t] = team_sum_shfl<TEAM ? TEAM : 1>(part[t]);
      } else {
        cta_sum_rs<2 * G>(part, red, parity);
        parity ^= 1;
      }
      float s[G];
      float gmax = -INFINITY;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        s[g] = -INFINITY;
        if (i0 + g < p.n) {
          s[g] = part[2 * g] * rsqrtf(fmaf(part[2 * g + 1], p.inv_D, p.eps));
          gmax = fmaxf(gmax, s[g]);
        }
      }
      const float m_new = fmaxf(m, gmax);
      const float scale = expf(m - m_new);  // 0 on the first group (m = -inf)
      den *= scale;
      const uint64_t scale2 = pair(scale, scale);
#pragma unroll
      for (int j = 0; j < VPT * NP; ++j) scale_pair(acc[j], scale2);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        if (i0 + g < p.n) {
          const float w = expf(s[g] - m_new);
          den += w;
          const uint64_t w2 = pair(w, w);
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            uint64_t x[NP];
            PR::split(buf[g][k], x);
#pragma unroll
            for (int j = 0; j < NP; ++j) fma_pair(acc[k * NP + j], w2, x[j]);
          }
        }
      }
      m = m_new;
    }

    if (row_ok) {
      const float inv = 1.f / den;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        float h[EPV];
#pragma unroll
        for (int j = 0; j < NP; ++j) unpair(acc[k * NP + j], h[2 * j], h[2 * j + 1]);
#pragma unroll
        for (int e = 0; e < EPV; ++e) {
          h[e] = h[e] * inv;
          if (FUSED_F) h[e] = half_tanh(ue[k * EPV + e] * h[e]);
        }
        st_vec(static_cast<char *>(p.out) + row_off + (size_t)(lt + k * tpr) * 16, E::pack(h));
      }
      if (lt == 0) {
        if (p.out_lse) p.out_lse[row] = m + logf(den);
        if (p.out_max) p.out_max[row] = m;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Launch configuration
// ---------------------------------------------------------------------------
namespace {

struct Cfg {
  int vpt;      // vectors per thread
  int team;     // 0 = CTA team, else lanes per row
  int threads;  // CTA size
};

int epv_of(int dtype) { return dtype == ATTNRES_BF16 ? 8 : 4; }

bool choose(int D, int dtype, Cfg &c) {
  const int nvec = D / epv_of(dtype);
  if (nvec <= 64) {
    int need = (nvec + 1) / 2, team = 4;
    while (team < need) team *= 2;
    c = {2, team, 256};
    return true;
  }
  if (nvec <= 1024) {
    c = {2, 0, ((nvec + 1) / 2 + 31) / 32 * 32};
    return true;
  }
  return false;  // D > 1024 vectors (8192 bf16 / 4096 fp32 elements)
}

template <typename T, int VPT, int TEAM, bool F>
cudaError_t run(const AggParams &p, const Cfg &c, cudaStream_t st) {
  auto kern = aggregate_kernel<T, VPT, TEAM, F>;
  static int occ[16] = {0};  // resident CTAs per SM, per device
  int dev = 0;
  cudaGetDevice(&dev);
  int &o = occ[dev & 15];
  if (o == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, c.threads, 0);
    if (e != cudaSuccess) return e;
    if (o < 1) o = 1;
  }
  const int per_cta = TEAM ? c.threads / TEAM : 1;
  const int64_t groups = (p.rows + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)o * sm_count();
  const int grid = (int)(groups < cap ? groups : cap);
  kern<<<grid, c.threads, 0, st>>>(p);
  return cudaGetLastError();
}

template <typename T, bool F>
cudaError_t dispatch(const AggParams &p, const Cfg &c, cudaStream_t st) {
  if (c.team == 0) return run<T, 2, 0, F>(p, c, st);
  switch (c.team) {
    case 4: return run<T, 2, 4, F>(p, c, st);
    case 8: return run<T, 2, 8, F>(p, c, st);
    case 16: return run<T, 2, 16, F>(p, c, st);
    default: return run<T, 2, 32, F>(p, c, st);
  }
}

}  // namespace

bool aggregate_supported(int D, int dtype) {
  Cfg c;
  return choose(D, dtype, c);
}

cudaError_t launch_aggregate(const AggregateArgs &a) {
  Cfg c;
  if (!choose(a.D, a.dtype, c)) return cudaErrorInvalidValue;
  AggParams p;
  for (int i = 0; i < a.n; ++i) p.src[i] = a.sources[i];
  p.n = a.n;
  p.nvec = a.D / epv_of(a.dtype);
  p.D = a.D;
  p.inv_D = 1.f / (float)a.D;
  p.eps = a.eps;
  p.rows = a.rows;
  p.q = a.query;
  p.g = a.gain;
  p.u = a.u;
  p.out = a.out;
  p.out_max = a.out_max;
  p.out_lse = a.out_lse;
  p.prior_o = a.prior_o;
  p.prior_lse = a.prior_lse;
  const bool fused = a.u != nullptr;
  if (a.dtype == ATTNRES_BF16)
    return fused ? dispatch<__nv_bfloat16, true>(p, c, a.stream)
                 : dispatch<__nv_bfloat16, false>(p, c, a.stream);
  return fused ? dispatch<float, true>(p, c, a.stream) : dispatch<float, false>(p, c, a.stream);
}

}  // namespace attnres
