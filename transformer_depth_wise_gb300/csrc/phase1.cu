// phase1.cu -- phase 1 of the two-phase Block scheme ("Attention Residual
// 深度残差", "两阶段算法（inter / intra）", inter step / attn_with_stats):
// the S pseudo-queries of a block score the same n completed block
// summaries, and each query's normalised output o_s plus its statistics
// (m_s, lse_s) are written.
//
// This file holds the general kernel (any D up to 8192 bf16, n <= 16, S <= 64);
// the tensor-core kernel in phase1_tc.cu takes the shapes it supports.
// One CTA owns one token row at a time.  The row's n summaries are read
// from HBM once, into a thread-private shared-memory stage, together with
// their sums of squares; then every query reuses the staged row: the CTA
// reduces the n dot products w~_s . v_i, forms the scores
// s_i = (w~_s . v_i) * rsqrt(v_i.v_i / D + eps), takes the softmax over the
// n summaries and writes o_s = sum_i alpha_i v_i.
#include "common.cuh"
#include "launch.h"

ATTNRES_DEFINE_ERROR_FLAG(take_error_phase1)

namespace attnres {

constexpr int kP1MaxN = 16;  // summaries per phase-1 call (this kernel)
constexpr int64_t kSplitMinRows = 64;   // token rows from which the split tensor-core path is taken

struct P1Params {
  const void *src[kP1MaxN];
  int n;
  int nvec;
  int D;
  float inv_D;
  float eps;
  int64_t rows;
  int S;
  const float *q;  // [S, D]
  const float *g;  // [S, D] or nullptr
  void *out;       // [S, rows, D]
  float *out_max;  // [S, rows] or nullptr
  float *out_lse;  // [S, rows]
};

// NS > 0: the number of summaries built in (the per-summary guards fold
// away); 0: taken from the parameters.
template <typename T, int VPT, int NS>
__global__ void __launch_bounds__(512, 1)
phase1_kernel(const __grid_constant__ P1Params p) {
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  constexpr int NM = kP1MaxN;
  static_assert(NS <= NM, "built-in summary count within the kernel's limit");
  const int n = NS ? NS : p.n;
  extern __shared__ uint4 stage[];  // [n][VPT][blockDim.x], thread-private slots
  __shared__ float red[2 * 32 * NM];

  const int tid = threadIdx.x, nt = blockDim.x;
  bool valid[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) valid[k] = tid + k * nt < p.nvec;

  const size_t row_bytes = (size_t)p.D * sizeof(T);
  int parity = 0;
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const size_t row_off = (size_t)row * row_bytes;
    float rinv[NM];
#pragma unroll
    for (int i = 0; i < NM; ++i) {
      rinv[i] = 0.f;
      if (i < n) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (valid[k])
            v = ld_stream(static_cast<const char *>(p.src[i]) + row_off + (size_t)(tid + k * nt) * 16);
          stage[(i * VPT + k) * nt + tid] = v;
          float x[EPV];
          E::unpack(v, x);
#pragma unroll
          for (int e = 0; e < EPV; ++e) rinv[i] = fmaf(x[e], x[e], rinv[i]);
        }
      }
    }
    cta_sum_rs<NM>(rinv, red, parity);
    parity ^= 1;
#pragma unroll
    for (int i = 0; i < NM; ++i) rinv[i] = rsqrtf(fmaf(rinv[i], p.inv_D, p.eps));

    // The folded query of query s, as packed pairs; the next query's is
    // loaded while the current one is formed (its latency is hidden).
    using PR = Pairs<T>;
    constexpr int NP = PR::NP;
    auto load_q = [&](int s, uint64_t (&qp)[VPT * NP]) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int j = tid + k * nt;
#pragma unroll
        for (int e4 = 0; e4 < EPV; e4 += 4) {
          float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f), g4 = make_float4(1.f, 1.f, 1.f, 1.f);
          if (valid[k] && s < p.S) {
            w4 = ld_f4(p.q + (size_t)s * p.D + j * EPV + e4);
            if (p.g) g4 = ld_f4(p.g + (size_t)s * p.D + j * EPV + e4);
          }
          qp[k * NP + e4 / 2] = pair(w4.x * g4.x, w4.y * g4.y);
          qp[k * NP + e4 / 2 + 1] = pair(w4.z * g4.z, w4.w * g4.w);
        }
      }
    };
    uint64_t qcur[VPT * NP], qnext[VPT * NP];
    load_q(0, qcur);
    for (int s = 0; s < p.S; ++s) {
      load_q(s + 1, qnext);
      float dots[NM];
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        dots[i] = 0.f;
        if (i < n) {
          uint64_t d2 = 0ull;
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            uint64_t x[NP];
            PR::split(stage[(i * VPT + k) * nt + tid], x);
#pragma unroll
            for (int m = 0; m < NP; ++m) fma_pair(d2, qcur[k * NP + m], x[m]);
          }
          dots[i] = pair_sum(d2);
        }
      }
      cta_sum_rs<NM>(dots, red, parity);
      parity ^= 1;
      float m = -INFINITY;
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        dots[i] = i < n ? dots[i] * rinv[i] : -INFINITY;
        m = fmaxf(m, dots[i]);
      }
      float den = 0.f;
#pragma unroll
      for (int i = 0; i < NM; ++i) {
        dots[i] = i < n ? expf(dots[i] - m) : 0.f;
        den += dots[i];
      }
      const float inv = 1.f / den;
      char *orow = static_cast<char *>(p.out) + ((size_t)s * p.rows + row) * row_bytes;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        uint64_t h2[NP];
#pragma unroll
        for (int m2 = 0; m2 < NP; ++m2) h2[m2] = 0ull;
#pragma unroll
        for (int i = 0; i < NM; ++i) {
          if (i < n) {
            uint64_t x[NP];
            PR::split(stage[(i * VPT + k) * nt + tid], x);
            const float a = dots[i] * inv;
            const uint64_t a2 = pair(a, a);
#pragma unroll
            for (int m2 = 0; m2 < NP; ++m2) fma_pair(h2[m2], a2, x[m2]);
          }
        }
        float h[EPV];
#pragma unroll
        for (int m2 = 0; m2 < NP; ++m2) unpair(h2[m2], h[2 * m2], h[2 * m2 + 1]);
        st_stream(orow + (size_t)(tid + k * nt) * 16, E::pack(h));
      }
      if (tid == 0) {
        p.out_lse[(size_t)s * p.rows + row] = m + logf(den);
        if (p.out_max) p.out_max[(size_t)s * p.rows + row] = m;
      }
#pragma unroll
      for (int j = 0; j < VPT * NP; ++j) qcur[j] = qnext[j];
    }
  }
}

namespace {

int epv_of(int dtype) { return dtype == ATTNRES_BF16 ? 8 : 4; }

struct Cfg {
  int vpt, threads;
  size_t smem;
};

bool choose(int n, int D, int dtype, Cfg &c) {
  const int nvec = D / epv_of(dtype);
  if (nvec <= 1024) {
    c.vpt = 2;
    c.threads = ((nvec + 1) / 2 + 31) / 32 * 32;
  } else if (nvec <= 2048) {
    c.vpt = 4;
    c.threads = ((nvec + 3) / 4 + 31) / 32 * 32;
  } else {
    return false;
  }
  c.smem = (size_t)n * c.vpt * c.threads * 16;
  // dynamic stage + the static reduction buffer must fit the 227 KB per-CTA limit
  return c.smem + sizeof(float) * 2 * 32 * kP1MaxN <= 227 * 1024;
}

template <typename T, int VPT, int NS = 0>
cudaError_t run(const P1Params &p, const Cfg &c, cudaStream_t st) {
  auto kern = phase1_kernel<T, VPT, NS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)c.smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, c.threads, c.smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t cap = (int64_t)occ * sm_count();
  const int grid = (int)(p.rows < cap ? p.rows : cap);
  if (cudaError_t le = launch_dependent(kern, dim3((unsigned)(grid)), dim3(c.threads), c.smem, st,
                                        p); le != cudaSuccess)
    return le;
  return cudaGetLastError();
}

}  // namespace

int phase1_check(int n, int D, int dtype, int S) {
  if (S < 1 || S > kMaxQueries) return ATTNRES_ERR_SHAPE;
  if (n > kP1MaxN) return ATTNRES_ERR_TOO_MANY_SOURCES;
  Cfg c;
  if (!choose(n, D, dtype, c)) return ATTNRES_ERR_SHAPE;
  return ATTNRES_OK;
}

cudaError_t launch_phase1(const Phase1Args &a) {
  // The tensor-core path parks the split queries in the last 48 D-rows of
  // `out`, which must not overlap out[0] (where it parks alpha).  Its scores
  // kernel works on 128-row tiles; from 512 rows its work items (tile, five
  // summaries) fill the GPU.  With fewer rows (from kSplitMinRows) it splits
  // the scores over slices of the features instead (split_parts), so that a
  // decode batch still fills it; below that the one-CTA-per-row kernel.
  if (phase1_tc_supported(a.n, a.D, a.dtype, a.S) && (int64_t)(a.S - 1) * a.rows >= 48 &&
      (a.rows >= 512 || (a.rows >= kSplitMinRows && split_parts(a) > 1)))
    return launch_phase1_tc(a);
  Cfg c;
  if (!choose(a.n, a.D, a.dtype, c)) return cudaErrorInvalidValue;
  P1Params p;
  for (int i = 0; i < a.n; ++i) p.src[i] = a.blocks[i];
  p.n = a.n;
  p.nvec = a.D / epv_of(a.dtype);
  p.D = a.D;
  p.inv_D = 1.f / (float)a.D;
  p.eps = a.eps;
  p.rows = a.rows;
  p.S = a.S;
  p.q = a.queries;
  p.g = a.gains;
  p.out = a.out;
  p.out_max = a.out_max;
  p.out_lse = a.out_lse;
  if (a.dtype == ATTNRES_BF16) {
    // The Block shape of the pages (nine completed blocks) has its count built
    // in: decode's phase 1 (256 rows, D = 7168) 0.226 -> 0.141 ms on a GB300.
    if (a.n == 9 && c.vpt == 2)
      return run<__nv_bfloat16, 2, 9>(p, c, a.stream);
    return c.vpt == 2 ? run<__nv_bfloat16, 2>(p, c, a.stream) : run<__nv_bfloat16, 4>(p, c, a.stream);
  }
  return c.vpt == 2 ? run<float, 2>(p, c, a.stream) : run<float, 4>(p, c, a.stream);
}

}  // namespace attnres
