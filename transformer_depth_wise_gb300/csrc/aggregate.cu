// aggregate.cu -- depth aggregation kernels (eq. A1-A3 of "Attention Residual
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
// aggregate_pipe_kernel takes rows of more than 64 vectors with at least one
// source (the CTA is the team, the next group's loads in flight while the
// current one is folded in); aggregate_kernel takes short rows (lane teams of
// a warp) and a prior state with no further source.
//
// aggregate_short_kernel takes bf16 rows of 2048 (256 vectors) merged into a
// prior state, with few sources and few rows (the Full two-phase schedule's
// intra-block steps):
// the row's prior state and sources are held in shared memory and read
// twice, once for the scores and once for the weighted sum, with one
// reduction and one exact softmax per row instead of one per group.
//
// All, with u != nullptr, apply the synthetic sublayer v = 0.5 tanh(u (.) h)
// to the fp32 h before the single rounding store: the Full stack uses it so
// h_l never round-trips through memory.
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
  grid_dependency_wait();
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
// Pipelined variant: rows of more than 64 vectors, n >= 1.
// ---------------------------------------------------------------------------
// A CTA owns one token row at a time and each thread VPT 16-byte vectors of
// it.  Sources go in groups of G (2 or 4); the thread's slices of the next
// group are loaded into a second register set while the current group is
// reduced and folded in, so loads stay in flight through the arithmetic.  The
// folded query lives in shared memory (read once per vector for all sources
// of a group), which leaves the registers to the loads in flight and the
// accumulator.  The arithmetic is that of aggregate_kernel.
// TPR > 0: rows that exactly fill a CTA of TPR threads (nvec == TPR * VPT),
// so the per-vector offsets are constants and every vector is valid.
template <typename T, bool FUSED_F, int G, int VPT, int TPR>
__global__ void __launch_bounds__(TPR ? TPR : 256, TPR ? 512 / (TPR ? TPR : 512) : 2)
aggregate_pipe_kernel(const __grid_constant__ AggParams p) {
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  static_assert(VPT >= 1 && VPT <= 4, "VPT: 1..4 vectors per thread");
  using PR = Pairs<T>;
  constexpr int NP = PR::NP;
  constexpr int Q4 = EPV / 4;               // float4 of w~ per vector
  extern __shared__ float4 qs[];            // [Q4][nvec]: w~ = w (.) gamma
  __shared__ float red[2 * 32 * 2 * G];

  const int tid = threadIdx.x, tpr = TPR ? TPR : blockDim.x;
  const int nvec = TPR ? TPR * VPT : p.nvec;
  for (int idx = tid; idx < nvec * Q4; idx += tpr) {
    const int j = idx / Q4, e4 = (idx % Q4) * 4;
    const float4 w4 = ld_f4(p.q + j * EPV + e4);
    const float4 g4 = p.g ? ld_f4(p.g + j * EPV + e4) : make_float4(1.f, 1.f, 1.f, 1.f);
    qs[(e4 / 4) * nvec + j] = make_float4(w4.x * g4.x, w4.y * g4.y, w4.z * g4.z, w4.w * g4.w);
  }
  __syncthreads();
  bool valid[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) valid[k] = TPR ? true : tid + k * tpr < nvec;
  const float4 *qt = qs + tid;  // this thread's vectors of w~: qt[c * nvec + k * tpr]

  const size_t row_bytes = (size_t)p.D * sizeof(T);
  const int ngr = (p.n + G - 1) / G;  // groups per row
  const int64_t my_rows = p.rows > (int64_t)blockIdx.x ? (p.rows - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t total = my_rows * ngr;

  // Loader cursor: the group whose slices are loaded next.
  int lgi = 0;
  int64_t lrow = blockIdx.x;
  auto load_next = [&](uint4 (&buf)[G][VPT]) {
    const size_t off = (size_t)lrow * row_bytes + (size_t)tid * 16;
    // The shape for many rows (G = 2) also asks L2 for the group after this
    // one, so its rows arrive while this one is processed: block_single 0.134
    // -> 0.126 ms on a GB300.  The G = 4 shape (fewer rows, e.g. the Full
    // stack's 2048) measured slower with it (27.2 -> 30.1 ms) and goes without.
    if (G == 2 && tid < G) {
      const bool wrap = lgi + 1 == ngr;
      const int64_t frow = wrap ? lrow + gridDim.x : lrow;
      const int fi = (wrap ? 0 : (lgi + 1) * G) + tid;
      if (frow < p.rows && fi < p.n)
        prefetch_l2_bulk(static_cast<const char *>(p.src[fi]) + (size_t)frow * row_bytes, (uint32_t)row_bytes);
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const int i = lgi * G + g;
      const char *base = static_cast<const char *>(p.src[i < p.n ? i : 0]) + off;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        buf[g][k] = make_uint4(0u, 0u, 0u, 0u);
        if (i < p.n && valid[k]) buf[g][k] = ld_stream_vec<TPR>(base, k, tpr);
      }
    }
    if (++lgi == ngr) { lgi = 0; lrow += gridDim.x; }
  };

  // Processing cursor and the row's online-softmax state.
  int cgi = 0, parity = 0;
  int64_t crow = blockIdx.x;
  float m = -INFINITY, den = 0.f;
  uint64_t acc[VPT * NP];
  auto process = [&](const uint4 (&buf)[G][VPT]) {
    const size_t row_off = (size_t)crow * row_bytes;
    if (cgi == 0) {  // a new row: empty state, or the prior state (lse, o, 1)
      m = -INFINITY;
      den = 0.f;
#pragma unroll
      for (int j = 0; j < VPT * NP; ++j) acc[j] = 0ull;
      if (p.prior_o) {
        m = p.prior_lse[crow];
        den = 1.f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
          if (valid[k])
            PR::split(ld_stream(static_cast<const char *>(p.prior_o) + row_off + (size_t)(tid + k * tpr) * 16),
                      acc + k * NP);
      }
    }
    const int i0 = cgi * G;
    uint64_t dot[G], ss[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = ss[g] = 0ull;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (!valid[k]) continue;
      uint64_t qp[NP];
#pragma unroll
      for (int c = 0; c < Q4; ++c) {
        const float4 q4 = qt[c * nvec + k * tpr];
        qp[2 * c] = pair(q4.x, q4.y);
        qp[2 * c + 1] = pair(q4.z, q4.w);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        uint64_t x[NP];
        PR::split(buf[g][k], x);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          fma_pair(dot[g], qp[j], x[j]);
          fma_pair(ss[g], x[j], x[j]);
        }
      }
    }
    float part[2 * G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      part[2 * g] = pair_sum(dot[g]);
      part[2 * g + 1] = pair_sum(ss[g]);
    }
    cta_sum_rs<2 * G>(part, red, parity);
    parity ^= 1;
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
    const float scale = expf(m - m_new);  // 0 on a row's first group without a prior (m = -inf)
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
    if (cgi == ngr - 1) {  // the row's last group: normalise and store
      const float inv = 1.f / den;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        if (!valid[k]) continue;
        const int j = tid + k * tpr;
        float h[EPV];
#pragma unroll
        for (int jj = 0; jj < NP; ++jj) unpair(acc[k * NP + jj], h[2 * jj], h[2 * jj + 1]);
#pragma unroll
        for (int e4 = 0; e4 < EPV; e4 += 4) {
          float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
          if (FUSED_F) u4 = ld_f4(p.u + j * EPV + e4);
          const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            h[e4 + e] *= inv;
            if (FUSED_F) h[e4 + e] = half_tanh(uu[e] * h[e4 + e]);
          }
        }
        st_vec(static_cast<char *>(p.out) + row_off + (size_t)j * 16, E::pack(h));
      }
      if (tid == 0) {
        if (p.out_lse) p.out_lse[crow] = m + logf(den);
        if (p.out_max) p.out_max[crow] = m;
      }
    }
    if (++cgi == ngr) { cgi = 0; crow += gridDim.x; }
  };

  // Two register sets in turn: group q + 1 loads while group q is processed.
  uint4 ba[G][VPT], bb[G][VPT];
  if (total > 0) load_next(ba);
  for (int64_t q = 0; q < total; q += 2) {
    if (q + 1 < total) load_next(bb);
    process(ba);
    if (q + 1 >= total) break;
    if (q + 2 < total) load_next(ba);
    process(bb);
  }
}

// ---------------------------------------------------------------------------
// Few sources, few rows (bf16, rows of 256 16-byte vectors): a row of the
// pipelined kernel costs one CTA-wide reduction, an exponential rescale and
// a second unpacking of the group per group of sources, and with few rows a
// CTA a chain of group steps each waiting on its copies.  Here a thread
// copies its two vectors of the row's prior o and of each source into shared
// memory (cp.async; each thread reads back only what it copied, so the
// copies need no barrier), the scores of all sources are reduced at once,
// the softmax is taken exactly (M = max of the prior's lse and the scores),
// and the weighted sum reads the same vectors again.  The buffer holds up
// to 16 row units (11 up to eight sources), so R = units / (1 + n) rows (at
// most seven) are in flight, and a row's slot is refilled R rows later as
// soon as it has been read.  Same
// arithmetic as the online form up to the order of the rescaling (eq. OS1 /
// OS2 collapse to one step when every score is known).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ring_copy16(void *smem, const void *gmem, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void ring_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void ring_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// wait_group takes an immediate: the pending count 0..6 by cases
__device__ __forceinline__ void ring_wait_upto(int pending) {
  switch (pending) {
    case 0: ring_wait<0>(); break;
    case 1: ring_wait<1>(); break;
    case 2: ring_wait<2>(); break;
    case 3: ring_wait<3>(); break;
    case 4: ring_wait<4>(); break;
    case 5: ring_wait<5>(); break;
    default: ring_wait<6>(); break;
  }
}

constexpr int kShortUnits = 16;                 // prior + sources of a row held at once (64 KB: three CTAs an SM)
constexpr int kShortThreads = 128;              // two vectors a thread
constexpr int kShortVectors = 2 * kShortThreads;
// Rows in flight for n sources: as many rows of 1 + n units as the buffer
// holds, at most seven, and the launch sizes the buffer to R (1 + n) units.
// Up to eight sources the buffer is held to 11 units (44 KB), so that five
// CTAs share an SM (their register limit) instead of three with 16 units:
// the Full two-phase schedule at S = 16 went 7.55 -> 7.48 ms on a GB300.
__host__ __device__ constexpr int short_units(int n) { return n <= 8 ? 11 : kShortUnits; }
__host__ __device__ constexpr int short_rows_in_flight(int n) {
  return short_units(n) / (1 + n) < 7 ? short_units(n) / (1 + n) : 7;
}
__host__ __device__ constexpr size_t short_smem(int n) {
  return (size_t)short_rows_in_flight(n) * (1 + n) * kShortVectors * 16;
}

// Five CTAs an SM by registers (96 and 89 a thread, no spills), as shared
// memory allows: up to 10 row units.
template <bool FUSED_F, int K>
__global__ void __launch_bounds__(kShortThreads, 5)
aggregate_short_kernel(const __grid_constant__ AggParams p) {
  grid_dependency_wait();
  using T = __nv_bfloat16;
  using E = Elt<T>;
  using PR = Pairs<T>;
  constexpr int NP = PR::NP, VPT = 2, TPR = kShortThreads, EPV = E::EPV;
  // K: the most sources this instance takes (n <= K); two sums a source in one reduction
  static_assert(K == 8 || K == 16, "K: 8 or 16 sources");
  extern __shared__ uint4 units[];              // [R][1 + n][VPT][TPR]: unit 0 of a slot the prior's o, 1 + i source i
  constexpr int kWarps = kShortThreads / 32;
  __shared__ float red[2 * kWarps * (2 * K)];    // cta_sum_rs<2 K, 4 warps>: [parity][warp][value]
  const int tid = threadIdx.x, n = p.n;
  const bool prior = p.prior_o != nullptr;
  const size_t row_bytes = (size_t)kShortVectors * 16;

  uint64_t qp[VPT][NP];                         // this thread's w~ = w (.) gamma, as pairs
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int j = tid + k * TPR;
#pragma unroll
    for (int c = 0; c < EPV / 4; ++c) {
      const float4 w4 = ld_f4(p.q + j * EPV + c * 4);
      const float4 g4 = p.g ? ld_f4(p.g + j * EPV + c * 4) : make_float4(1.f, 1.f, 1.f, 1.f);
      qp[k][2 * c] = pair(w4.x * g4.x, w4.y * g4.y);
      qp[k][2 * c + 1] = pair(w4.z * g4.z, w4.w * g4.w);
    }
  }
  // A row takes U = 1 + n units (unit 0 the prior's); R rows fit the
  // buffer and are in flight at once (R = 1 from eight sources).
  const int U = 1 + n, R = short_rows_in_flight(n);
  int ub = 0;                                   // first unit of the row being reduced
  auto unit = [&](int u, int k) -> uint4 & { return units[((ub + u) * VPT + k) * TPR + tid]; };
  auto issue = [&](int64_t row, int slot) {     // one commit group per row (empty past the end)
    if (row < p.rows) {
      const size_t off = (size_t)row * row_bytes + (size_t)tid * 16;
      uint4 *base = units + (size_t)slot * U * VPT * TPR + tid;
      if (prior) {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
          ring_copy16(base + k * TPR, static_cast<const char *>(p.prior_o) + off + (size_t)k * TPR * 16, 16u);
      }
      for (int i = 0; i < n; ++i) {
        const char *src = static_cast<const char *>(p.src[i]) + off;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
          ring_copy16(base + ((1 + i) * VPT + k) * TPR, src + (size_t)k * TPR * 16, 16u);
      }
    }
    ring_commit();
  };

  int parity = 0, slot = 0;
  for (int r = 0; r < R; ++r) issue((int64_t)blockIdx.x + (int64_t)r * gridDim.x, r);
  for (int64_t row = blockIdx.x; row < p.rows; row += gridDim.x) {
    const float lse_p = prior ? p.prior_lse[row] : -INFINITY;
    ring_wait_upto(R - 1);                      // this thread's vectors of the row have landed
    ub = slot * U;
    // The source loops are unrolled to K and left at n (uniform): no
    // predicated-off work for the sources past n.
    float part[2 * K];                          // w~.v_i and v_i.v_i
#pragma unroll
    for (int i = 0; i < 2 * K; ++i) part[i] = 0.f;
#pragma unroll
    for (int i = 0; i < K; ++i) {
      if (i >= n) break;
      uint64_t dot = 0ull, ss = 0ull;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        uint64_t x[NP];
        PR::split(unit(1 + i, k), x);
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          fma_pair(dot, qp[k][j], x[j]);
          fma_pair(ss, x[j], x[j]);
        }
      }
      part[2 * i] = pair_sum(dot);
      part[2 * i + 1] = pair_sum(ss);
    }
    cta_sum_rs<2 * K, kWarps>(part, red, parity);
    parity ^= 1;
    float sc[K];
    float M = lse_p;
#pragma unroll
    for (int i = 0; i < K; ++i) sc[i] = -INFINITY;
#pragma unroll
    for (int i = 0; i < K; ++i) {
      if (i >= n) break;
      sc[i] = part[2 * i] * rsqrtf(fmaf(part[2 * i + 1], p.inv_D, p.eps));
      M = fmaxf(M, sc[i]);
    }
    uint64_t acc[VPT][NP];
    float den = 0.f;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int j = 0; j < NP; ++j) acc[k][j] = 0ull;
    if (prior) {                                // the prior state (lse, o, 1) as the first term
      const float wpr = expf(lse_p - M);
      den = wpr;
      const uint64_t w2 = pair(wpr, wpr);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        uint64_t x[NP];
        PR::split(unit(0, k), x);
#pragma unroll
        for (int j = 0; j < NP; ++j) fma_pair(acc[k][j], w2, x[j]);
      }
    }
#pragma unroll
    for (int i = 0; i < K; ++i) {
      if (i >= n) break;
      {
        const float w = expf(sc[i] - M);
        den += w;
        const uint64_t w2 = pair(w, w);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          uint64_t x[NP];
          PR::split(unit(1 + i, k), x);
#pragma unroll
          for (int j = 0; j < NP; ++j) fma_pair(acc[k][j], w2, x[j]);
        }
      }
    }
    // every vector of this row has been read into the sums above: the row R
    // rounds later may overwrite them
    issue(row + (int64_t)R * gridDim.x, slot);
    if (++slot == R) slot = 0;
    const float inv = 1.f / den;
    const size_t row_off = (size_t)row * row_bytes;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int j = tid + k * TPR;
      float h[EPV];
#pragma unroll
      for (int jj = 0; jj < NP; ++jj) unpair(acc[k][jj], h[2 * jj], h[2 * jj + 1]);
#pragma unroll
      for (int e4 = 0; e4 < EPV; e4 += 4) {
        float4 u4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (FUSED_F) u4 = ld_f4(p.u + j * EPV + e4);
        const float uu[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          h[e4 + e] *= inv;
          if (FUSED_F) h[e4 + e] = half_tanh(uu[e] * h[e4 + e]);
        }
      }
      st_vec(static_cast<char *>(p.out) + row_off + (size_t)j * 16, E::pack(h));
    }
    if (tid == 0) {
      if (p.out_lse) p.out_lse[row] = M + logf(den);
      if (p.out_max) p.out_max[row] = M;
    }
  }
  ring_wait<0>();
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
  if (cudaError_t le = launch_dependent(kern, dim3((unsigned)(grid)), dim3(c.threads), 0, st, p); le != cudaSuccess)
    return le;
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

// The pipelined kernel: n >= 1 sources and rows of more than 64 vectors (the
// lane-team kernel takes shorter rows; a prior state with no further source
// goes to aggregate_kernel).  Two shapes, measured on a GB300 for D = 2048:
// groups of 2 sources with 4 vectors per thread (64-thread CTAs for D =
// 2048) win once there are rows enough for every CTA of the grid to take
// several (from 32 rows per SM; e.g. 5.5 against 5.1 TB/s at 16384 rows and
// n = 10), groups of 4 with 2 vectors per thread (twice the threads per row)
// below that (e.g. 4.2 against 4.0 TB/s at 2048 rows and n = 187).  A CTA
// of ceil(nvec / vpt) threads, rounded up to whole warps, per row; rows that
// fill it exactly take the kernel with that thread count built in.
struct PipeCfg {
  int g, vpt, threads;
  int tpr;  // the built-in thread count, or 0 (general kernel)
};

bool choose_pipe(int n, int64_t rows, int D, int dtype, PipeCfg &c) {
  const int nvec = D / epv_of(dtype);
  if (n < 1 || nvec <= 64) return false;
  auto threads_for = [&](int vpt) { return ((nvec + vpt - 1) / vpt + 31) / 32 * 32; };
  const bool many_rows = rows >= 32 * (int64_t)sm_count();
  if (!many_rows && threads_for(2) <= 256) {
    c.g = 4;
    c.vpt = 2;
  } else {
    c.g = 2;
    c.vpt = 4;
  }
  c.threads = threads_for(c.vpt);
  if (c.threads > 256) return false;
  const bool exact = nvec == c.threads * c.vpt;
  c.tpr = 0;
  if (exact) {
    const int built[] = {64, 128, 224, 256};   // 224: D = 7168 bf16 at four vectors a thread
    for (int b : built)
      if (b == c.threads) c.tpr = b;
  }
  return true;
}

template <typename T, bool F, int G, int VPT, int TPR>
cudaError_t run_pipe(const AggParams &p, int threads, cudaStream_t st) {
  auto kern = aggregate_pipe_kernel<T, F, G, VPT, TPR>;
  const size_t smem = (size_t)p.D * sizeof(float);  // w~
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  int occ = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t cap = (int64_t)occ * sm_count();
  const int grid = (int)(p.rows < cap ? p.rows : cap);
  if (cudaError_t le = launch_dependent(kern, dim3((unsigned)(grid)), dim3(threads), smem, st,
                                        p); le != cudaSuccess)
    return le;
  return cudaGetLastError();
}

// The short-row kernel: bf16 rows of 2048 merged into a prior state with the
// sublayer fused (the Full two-phase schedule's intra-block steps, the only
// caller that passes a prior), 1..15 sources (unit 0 of the
// shared-memory row is the prior's, sources take units 1..n), and fewer rows
// than the many-rows shape of the pipelined kernel takes.  Measured on a
// GB300 over the schedule at S = 14: 8.45 -> 7.98-8.07 ms.  Without a prior
// neither kernel wins throughout (2048 rows: 8.3 us for one source either
// way, 13.7 against 15.1 us for five, 20.2 against 17.4 us for eight, 28.7
// against 27.8 us for 13; both pay about 5 us a launch of ramp and tail),
// so plain calls keep the pipelined kernel.
bool short_fits(const AggregateArgs &a) {
  return a.dtype == ATTNRES_BF16 && a.prior_o != nullptr && a.u != nullptr && a.D == 8 * kShortVectors &&
         a.n >= 1 && 1 + a.n <= kShortUnits && a.rows < 32 * (int64_t)sm_count();
}

template <bool F, int K>
cudaError_t run_short(const AggParams &p, cudaStream_t st) {
  auto kern = aggregate_short_kernel<F, K>;
  const size_t smem = short_smem(p.n);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)short_smem(15));
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kShortThreads, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t cap = (int64_t)occ * sm_count();
  const int grid = (int)(p.rows < cap ? p.rows : cap);
  if (cudaError_t le = launch_dependent(kern, dim3((unsigned)grid), dim3(kShortThreads), smem, st, p);
      le != cudaSuccess)
    return le;
  return cudaGetLastError();
}

template <typename T, bool F>
cudaError_t dispatch_pipe(const AggParams &p, const PipeCfg &c, cudaStream_t st) {
  if (c.g == 4) {
    switch (c.tpr) {
      case 64: return run_pipe<T, F, 4, 2, 64>(p, c.threads, st);
      case 128: return run_pipe<T, F, 4, 2, 128>(p, c.threads, st);
      case 256: return run_pipe<T, F, 4, 2, 256>(p, c.threads, st);
      default: return run_pipe<T, F, 4, 2, 0>(p, c.threads, st);
    }
  }
  switch (c.tpr) {
    case 64: return run_pipe<T, F, 2, 4, 64>(p, c.threads, st);
    case 128: return run_pipe<T, F, 2, 4, 128>(p, c.threads, st);
    case 224: return run_pipe<T, F, 2, 4, 224>(p, c.threads, st);
    case 256: return run_pipe<T, F, 2, 4, 256>(p, c.threads, st);
    default: return run_pipe<T, F, 2, 4, 0>(p, c.threads, st);
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
  if (short_fits(a)) return a.n <= 8 ? run_short<true, 8>(p, a.stream) : run_short<true, 16>(p, a.stream);
  PipeCfg pc;
  if (choose_pipe(a.n, a.rows, a.D, a.dtype, pc)) {
    if (a.dtype == ATTNRES_BF16)
      return fused ? dispatch_pipe<__nv_bfloat16, true>(p, pc, a.stream)
                   : dispatch_pipe<__nv_bfloat16, false>(p, pc, a.stream);
    return fused ? dispatch_pipe<float, true>(p, pc, a.stream) : dispatch_pipe<float, false>(p, pc, a.stream);
  }
  if (a.dtype == ATTNRES_BF16)
    return fused ? dispatch<__nv_bfloat16, true>(p, c, a.stream)
                 : dispatch<__nv_bfloat16, false>(p, c, a.stream);
  return fused ? dispatch<float, true>(p, c, a.stream) : dispatch<float, false>(p, c, a.stream);
}

}  // namespace attnres
