// merge.cu -- phase 2 of the two-phase Block scheme and the running partial
// update ("Attention Residual 深度残差", "两阶段算法（inter / intra）",
// eq. OS2 and single_source_stats; "forward_naive" partial = partial + out).
//
// Phase-2 merge, per token row: the partial p is a single source with state
// (s_p, p, 1); the phase-1 state of the same query is (lse, o, 1).  OS2 with
// M = max(lse, s_p) gives
//   h = (e^{lse-M} o + e^{s_p-M} p) / (e^{lse-M} + e^{s_p-M}).
// Three rows move per token (read o, read p, write h): a pure HBM stream.
#include "common.cuh"
#include "launch.h"

ATTNRES_DEFINE_ERROR_FLAG(take_error_merge)

namespace attnres {

struct MergeParams {
  const void *o;
  const float *lse;
  const void *p;
  int nvec;
  int D;
  float inv_D;
  float eps;
  int64_t rows;
  const float *q;
  const float *g;
  void *h;
  float *lse_out;
};

template <typename T, int VPT, int TEAM>
__global__ void __launch_bounds__(TEAM ? 256 : 512)
merge_kernel(const __grid_constant__ MergeParams p) {
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  constexpr int NE = VPT * EPV;
  __shared__ float red[TEAM ? 1 : 2 * 32 * 2];

  const int tpr = TEAM ? TEAM : blockDim.x;
  const int lt = TEAM ? (threadIdx.x % TEAM) : threadIdx.x;
  const int teams_per_cta = TEAM ? blockDim.x / TEAM : 1;
  const int team = TEAM ? threadIdx.x / TEAM : 0;
  const bool has_p = p.p != nullptr;

  float qe[NE];
  bool valid[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int j = lt + k * tpr;
    valid[k] = j < p.nvec;
#pragma unroll
    for (int e4 = 0; e4 < EPV; e4 += 4) {
      float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f), g4 = make_float4(1.f, 1.f, 1.f, 1.f);
      if (valid[k] && has_p) {
        w4 = ld_f4(p.q + j * EPV + e4);
        if (p.g) g4 = ld_f4(p.g + j * EPV + e4);
      }
      qe[k * EPV + e4 + 0] = w4.x * g4.x;
      qe[k * EPV + e4 + 1] = w4.y * g4.y;
      qe[k * EPV + e4 + 2] = w4.z * g4.z;
      qe[k * EPV + e4 + 3] = w4.w * g4.w;
    }
  }

  const size_t row_bytes = (size_t)p.D * sizeof(T);
  const int64_t groups = (p.rows + teams_per_cta - 1) / teams_per_cta;
  int parity = 0;
  for (int64_t rg = blockIdx.x; rg < groups; rg += gridDim.x) {
    const int64_t row = rg * teams_per_cta + team;
    const bool row_ok = row < p.rows;
    const size_t row_off = (size_t)row * row_bytes;
    uint4 ov[VPT], pv[VPT];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      ov[k] = make_uint4(0u, 0u, 0u, 0u);
      pv[k] = make_uint4(0u, 0u, 0u, 0u);
      const size_t off = row_off + (size_t)(lt + k * tpr) * 16;
      if (row_ok && valid[k]) {
        ov[k] = ld_stream(static_cast<const char *>(p.o) + off);
        if (has_p) pv[k] = ld_stream(static_cast<const char *>(p.p) + off);
      }
    }
    if (!has_p) {  // first sublayer of a block: h = o
      if (row_ok) {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
          if (valid[k]) st_vec(static_cast<char *>(p.h) + row_off + (size_t)(lt + k * tpr) * 16, ov[k]);
        if (lt == 0 && p.lse_out) p.lse_out[row] = p.lse[row];
      }
      continue;
    }
    float part[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      float x[EPV];
      E::unpack(pv[k], x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        part[0] = fmaf(qe[k * EPV + e], x[e], part[0]);
        part[1] = fmaf(x[e], x[e], part[1]);
      }
    }
    if (TEAM) {
      part[0] = team_sum_shfl<TEAM ? TEAM : 1>(part[0]);
      part[1] = team_sum_shfl<TEAM ? TEAM : 1>(part[1]);
    } else {
      cta_sum<2>(part, red, parity);
      parity ^= 1;
    }
    if (!row_ok) continue;
    const float sp = part[0] * rsqrtf(fmaf(part[1], p.inv_D, p.eps));
    const float l = p.lse[row];
    const float M = fmaxf(l, sp);
    const float a = expf(l - M), c = expf(sp - M);
    const float inv = 1.f / (a + c);
    const float wa = a * inv, wc = c * inv;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (!valid[k]) continue;
      float xo[EPV], xp[EPV], h[EPV];
      E::unpack(ov[k], xo);
      E::unpack(pv[k], xp);
#pragma unroll
      for (int e = 0; e < EPV; ++e) h[e] = fmaf(wa, xo[e], wc * xp[e]);
      st_vec(static_cast<char *>(p.h) + row_off + (size_t)(lt + k * tpr) * 16, E::pack(h));
    }
    if (lt == 0 && p.lse_out) p.lse_out[row] = M + logf(a + c);
  }
}

// ---------------------------------------------------------------------------
// Fused partial update + phase-2 merge (the intra-block fusion of the K3
// decode path: "intra-block merge + partial-sum update"), per token row:
//   out     = sub_out                      (u == nullptr: the sublayer output)
//           = 0.5 tanh(u (.) sub_out)      (u != nullptr: sub_out is the
//                                           sublayer input, synthetic f)
//   p_new   = (p_in or 0) + out            rounded once, stored
//   h       = merge(o, lse; p_new)         eq. OS2 with the stored p_new
// Three rows are read (o, p_in, sub_out) and two written (p_new, h), against
// six for the separate update and merge.  p_out may alias p_in, and h_out
// may alias sub_out (every element is read before it is written, by the
// thread that writes it, and the rows are reduced in between).
// ---------------------------------------------------------------------------
struct MergeUpdateParams {
  MergeParams m;       // o, lse, (p unused), q, g, h, lse_out, sizes
  const void *p_in;    // or nullptr
  const void *sub;     // sublayer output, or its input when u != nullptr
  const float *u;      // or nullptr
  void *p_out;
  const float *nw;     // pre-norm weight [D] (NORM)
  float neps;          // pre-norm eps (NORM)
  void *y;             // RMSNorm(h) (.) nw, [rows, D] (NORM)
};

// TPR > 0 (CTA teams): rows that exactly fill a CTA of TPR threads (nvec ==
// TPR * VPT), so the per-vector offsets are constants and every vector is
// valid.
template <typename T, int VPT, int TEAM, bool SYNTH, bool NORM, int TPR>
__global__ void __launch_bounds__(TEAM ? 256 : 512)
merge_update_kernel(const __grid_constant__ MergeUpdateParams P) {
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  __shared__ float red[TEAM ? 1 : 2 * 32 * 2];
  __shared__ float red_n[(TEAM || !NORM) ? 1 : 2 * 32];
  const MergeParams &p = P.m;
  static_assert(TPR == 0 || TEAM == 0, "a built-in thread count is for CTA teams");
  const int tpr = TPR ? TPR : (TEAM ? TEAM : blockDim.x);
  // 16-byte vectors per row (read from the parameters where not built in)
  auto nvec = [&]() { return TPR ? TPR * VPT : p.nvec; };
  const int lt = TEAM ? (threadIdx.x % TEAM) : threadIdx.x;
  const int teams_per_cta = TEAM ? blockDim.x / TEAM : 1;
  const int team = TEAM ? threadIdx.x / TEAM : 0;
  const bool has_pin = P.p_in != nullptr;

  // The folded query w~ = w (.) gamma, u and the pre-norm weight live in
  // shared memory (loaded once per CTA), not in registers: fewer registers,
  // more rows in flight.  Layout [quarter e4 / 4][vector j] of float4, so
  // consecutive lanes read consecutive 16 bytes.
  extern __shared__ float4 qu[];   // [EPV/4][nvec] q~, then u (SYNTH), then the norm weight (NORM)
  constexpr int Q4 = EPV / 4;
  constexpr int NW_AT = SYNTH ? 2 * Q4 : Q4;
  for (int idx = threadIdx.x; idx < nvec() * Q4; idx += blockDim.x) {
    const int j = idx / Q4, e4 = (idx % Q4) * 4;
    const float4 w4 = ld_f4(p.q + j * EPV + e4);
    const float4 g4 = p.g ? ld_f4(p.g + j * EPV + e4) : make_float4(1.f, 1.f, 1.f, 1.f);
    qu[(e4 / 4) * nvec() + j] = make_float4(w4.x * g4.x, w4.y * g4.y, w4.z * g4.z, w4.w * g4.w);
    if (SYNTH) qu[(Q4 + e4 / 4) * nvec() + j] = ld_f4(P.u + j * EPV + e4);
    if (NORM) qu[(NW_AT + e4 / 4) * nvec() + j] = ld_f4(P.nw + j * EPV + e4);
  }
  __syncthreads();
  bool valid[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) valid[k] = TPR ? true : lt + k * tpr < nvec();

  const size_t row_bytes = (size_t)p.D * sizeof(T);
  const int64_t groups = (p.rows + teams_per_cta - 1) / teams_per_cta;
  const int64_t my_groups = groups > (int64_t)blockIdx.x
                                ? (groups - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  auto load_row = [&](int64_t k, uint4 (&ov)[VPT], uint4 (&pv)[VPT], uint4 (&sv)[VPT]) {
    const int64_t row = ((int64_t)blockIdx.x + k * gridDim.x) * teams_per_cta + team;
    const bool row_ok = row < p.rows;
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
      ov[kk] = pv[kk] = sv[kk] = make_uint4(0u, 0u, 0u, 0u);
      const size_t off = (size_t)row * row_bytes + (size_t)(lt + kk * tpr) * 16;
      if (row_ok && valid[kk]) {
        ov[kk] = TPR ? ld_stream_vec<TPR>(static_cast<const char *>(p.o) + (size_t)row * row_bytes + (size_t)lt * 16, kk, tpr)
                     : ld_stream(static_cast<const char *>(p.o) + off);
        // p_in and sub may be overwritten by this kernel: coherent loads
        if (has_pin) pv[kk] = *reinterpret_cast<const uint4 *>(static_cast<const char *>(P.p_in) + off);
        sv[kk] = *reinterpret_cast<const uint4 *>(static_cast<const char *>(P.sub) + off);
      }
    }
  };
  int parity = 0, parity_n = 0;
  auto process = [&](int64_t k, const uint4 (&ov)[VPT], const uint4 (&pv)[VPT], const uint4 (&sv)[VPT]) {
    const int64_t row = ((int64_t)blockIdx.x + k * gridDim.x) * teams_per_cta + team;
    const bool row_ok = row < p.rows;
    const size_t row_off = (size_t)row * row_bytes;
    uint4 pn[VPT];
    float part[2] = {0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
      float xp[EPV], xs[EPV], y[EPV];
      E::unpack(pv[kk], xp);
      E::unpack(sv[kk], xs);
      float uu[EPV];
      if (SYNTH && valid[kk]) {
#pragma unroll
        for (int e4 = 0; e4 < EPV; e4 += 4) {
          const float4 v = qu[(Q4 + e4 / 4) * nvec() + lt + kk * tpr];
          uu[e4] = v.x; uu[e4 + 1] = v.y; uu[e4 + 2] = v.z; uu[e4 + 3] = v.w;
        }
      }
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float out = SYNTH ? half_tanh((valid[kk] ? uu[e] : 0.f) * xs[e]) : xs[e];
        y[e] = xp[e] + out;
      }
      pn[kk] = E::pack(y);              // the stored (rounded) partial
      if (!valid[kk]) continue;
      float x[EPV];
      E::unpack_again(pn[kk], x);
#pragma unroll
      for (int e4 = 0; e4 < EPV; e4 += 4) {
        const float4 q4 = qu[(e4 / 4) * nvec() + lt + kk * tpr];
        part[0] = fmaf(q4.x, x[e4], part[0]);
        part[0] = fmaf(q4.y, x[e4 + 1], part[0]);
        part[0] = fmaf(q4.z, x[e4 + 2], part[0]);
        part[0] = fmaf(q4.w, x[e4 + 3], part[0]);
      }
#pragma unroll
      for (int e = 0; e < EPV; ++e) part[1] = fmaf(x[e], x[e], part[1]);
    }
    if (TEAM) {
      part[0] = team_sum_shfl<TEAM ? TEAM : 1>(part[0]);
      part[1] = team_sum_shfl<TEAM ? TEAM : 1>(part[1]);
    } else {
      cta_sum<2>(part, red, parity);
      parity ^= 1;
    }
    if (!NORM) {
      // No pre-norm: h is always stored (the entry point requires h_out then).
      if (!row_ok) return;
      const float sp = part[0] * rsqrtf(fmaf(part[1], p.inv_D, p.eps));
      const float l = p.lse[row];
      const float M = fmaxf(l, sp);
      const float a = expf(l - M), c = expf(sp - M);
      const float inv = 1.f / (a + c);
      const float wa = a * inv, wc = c * inv;
#pragma unroll
      for (int kk = 0; kk < VPT; ++kk) {
        if (!valid[kk]) continue;
        const size_t off = row_off + (size_t)(lt + kk * tpr) * 16;
        st_vec(static_cast<char *>(P.p_out) + off, pn[kk]);
        float xo[EPV], xp[EPV], h[EPV];
        E::unpack(ov[kk], xo);
        E::unpack_again(pn[kk], xp);
#pragma unroll
        for (int e = 0; e < EPV; ++e) h[e] = fmaf(wa, xo[e], wc * xp[e]);
        st_vec(static_cast<char *>(p.h) + off, E::pack(h));
      }
      if (lt == 0 && p.lse_out) p.lse_out[row] = M + logf(a + c);
      return;
    }
    // With the pre-norm every lane of a team takes part in its second
    // reduction, so rows past the end run through with zero weights.
    float wa = 0.f, wc = 0.f, M = 0.f, a = 0.f, c = 0.f;
    if (row_ok) {
      const float sp = part[0] * rsqrtf(fmaf(part[1], p.inv_D, p.eps));
      const float l = p.lse[row];
      M = fmaxf(l, sp);
      a = expf(l - M);
      c = expf(sp - M);
      const float inv = 1.f / (a + c);
      wa = a * inv;
      wc = c * inv;
    }
    float hs = 0.f;                     // NORM: sum of h^2 over the row
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
      if (!valid[kk] || !row_ok) continue;
      const size_t off = row_off + (size_t)(lt + kk * tpr) * 16;
      st_vec(static_cast<char *>(P.p_out) + off, pn[kk]);
      float xo[EPV], xp[EPV], h[EPV];
      E::unpack(ov[kk], xo);
      E::unpack_again(pn[kk], xp);
#pragma unroll
      for (int e = 0; e < EPV; ++e) h[e] = fmaf(wa, xo[e], wc * xp[e]);
      if (p.h) st_vec(static_cast<char *>(p.h) + off, E::pack(h));
#pragma unroll
      for (int e = 0; e < EPV; ++e) hs = fmaf(h[e], h[e], hs);
    }
    {
      // The next sublayer's pre-norm on the unrounded h: y = h / sqrt(mean h^2 + eps) (.) w_n.
      if (TEAM) {
        hs = team_sum_shfl<TEAM ? TEAM : 1>(hs);
      } else {
        float v1[1] = {hs};
        cta_sum<1>(v1, red_n, parity_n);
        parity_n ^= 1;
        hs = v1[0];
      }
      if (row_ok) {
        const float rn = rsqrtf(fmaf(hs, p.inv_D, P.neps));
#pragma unroll
        for (int kk = 0; kk < VPT; ++kk) {
          if (!valid[kk]) continue;
          float xo[EPV], xp[EPV], y[EPV];
          E::unpack(ov[kk], xo);
          E::unpack_again(pn[kk], xp);
#pragma unroll
          for (int e4 = 0; e4 < EPV; e4 += 4) {
            const float4 w4 = qu[(NW_AT + e4 / 4) * nvec() + lt + kk * tpr];
            y[e4 + 0] = fmaf(wa, xo[e4 + 0], wc * xp[e4 + 0]) * rn * w4.x;
            y[e4 + 1] = fmaf(wa, xo[e4 + 1], wc * xp[e4 + 1]) * rn * w4.y;
            y[e4 + 2] = fmaf(wa, xo[e4 + 2], wc * xp[e4 + 2]) * rn * w4.z;
            y[e4 + 3] = fmaf(wa, xo[e4 + 3], wc * xp[e4 + 3]) * rn * w4.w;
          }
          st_vec(static_cast<char *>(P.y) + row_off + (size_t)(lt + kk * tpr) * 16, E::pack(y));
        }
      }
    }
    if (row_ok && lt == 0 && p.lse_out) p.lse_out[row] = M + logf(a + c);
  };

  // One row ahead, three threads of the team ask L2 for the next row's o,
  // p_in and sub (one bulk prefetch each): its loads then find it in L2.
  auto prefetch_row = [&](int64_t k) {
    const int64_t row = ((int64_t)blockIdx.x + k * gridDim.x) * teams_per_cta + team;
    if (k >= my_groups || row >= p.rows || lt >= 3) return;
    const void *base = lt == 0 ? p.o : (lt == 1 ? P.p_in : P.sub);
    if (base) prefetch_l2_bulk(static_cast<const char *>(base) + (size_t)row * row_bytes, (uint32_t)row_bytes);
  };
  prefetch_row(0);
  for (int64_t k = 0; k < my_groups; ++k) {
    uint4 ov[VPT], pv[VPT], sv[VPT];
    prefetch_row(k + 1);
    load_row(k, ov, pv, sv);
    process(k, ov, pv, sv);
  }
}

// Few rows (decode: about one row per SM or fewer).  A CTA takes two rows,
// and each thread the same two 16-byte vectors of both, holding its vectors
// of w~ = w (.) gamma, u and the norm weight in registers: they are read
// once for two rows, with no shared-memory staging and no barrier before the
// rows, and all loads are issued together.  The arithmetic is the fused step
// above, element by element and reduction by reduction.
template <typename T, bool SYNTH, bool NORM>
__global__ void __launch_bounds__(512, 1)
merge_update_few_kernel(const __grid_constant__ MergeUpdateParams P) {
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  constexpr int R = 2, V = 2;          // rows per CTA, vectors per thread
  __shared__ float red[2 * 32 * 2 * R];
  __shared__ float red_n[NORM ? 2 * 32 * R : 1];
  const MergeParams &p = P.m;
  const int lt = threadIdx.x, tpr = blockDim.x;
  const size_t row_bytes = (size_t)p.D * sizeof(T);
  bool valid[V], ok[R];
  int64_t row[R];
#pragma unroll
  for (int k = 0; k < V; ++k) valid[k] = lt + k * tpr < p.nvec;
#pragma unroll
  for (int r = 0; r < R; ++r) {
    row[r] = (int64_t)blockIdx.x * R + r;
    ok[r] = row[r] < p.rows;
  }
  auto off_of = [&](int r, int k) { return (size_t)row[r] * row_bytes + (size_t)(lt + k * tpr) * 16; };

  uint4 ov[R][V], pv[R][V], sv[R][V];
  float lse[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    lse[r] = ok[r] ? p.lse[row[r]] : 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      ov[r][k] = pv[r][k] = sv[r][k] = make_uint4(0u, 0u, 0u, 0u);
      if (!ok[r] || !valid[k]) continue;
      ov[r][k] = ld_stream(static_cast<const char *>(p.o) + off_of(r, k));
      // p_in and sub may be overwritten by this kernel: coherent loads
      if (P.p_in) pv[r][k] = *reinterpret_cast<const uint4 *>(static_cast<const char *>(P.p_in) + off_of(r, k));
      sv[r][k] = *reinterpret_cast<const uint4 *>(static_cast<const char *>(P.sub) + off_of(r, k));
    }
  }
  float q[V][EPV], uu[V][EPV], nw[V][EPV];
#pragma unroll
  for (int k = 0; k < V; ++k)
#pragma unroll
    for (int e4 = 0; e4 < EPV; e4 += 4) {
      float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f), g4 = make_float4(1.f, 1.f, 1.f, 1.f), u4 = w4, n4 = w4;
      const int j = lt + k * tpr;
      if (valid[k]) {
        w4 = ld_f4(p.q + j * EPV + e4);
        if (p.g) g4 = ld_f4(p.g + j * EPV + e4);
        if (SYNTH) u4 = ld_f4(P.u + j * EPV + e4);
        if (NORM) n4 = ld_f4(P.nw + j * EPV + e4);
      }
      q[k][e4] = w4.x * g4.x; q[k][e4 + 1] = w4.y * g4.y; q[k][e4 + 2] = w4.z * g4.z; q[k][e4 + 3] = w4.w * g4.w;
      uu[k][e4] = u4.x; uu[k][e4 + 1] = u4.y; uu[k][e4 + 2] = u4.z; uu[k][e4 + 3] = u4.w;
      nw[k][e4] = n4.x; nw[k][e4 + 1] = n4.y; nw[k][e4 + 2] = n4.z; nw[k][e4 + 3] = n4.w;
    }

  // p_new = p_in + out, rounded as stored; s_p's dot and sum of squares.
  uint4 pn[R][V];
  float part[2 * R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    part[2 * r] = part[2 * r + 1] = 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      float xp[EPV], xs[EPV], y[EPV];
      E::unpack(pv[r][k], xp);
      E::unpack(sv[r][k], xs);
#pragma unroll
      for (int e = 0; e < EPV; ++e) y[e] = xp[e] + (SYNTH ? half_tanh(uu[k][e] * xs[e]) : xs[e]);
      pn[r][k] = E::pack(y);
      if (!valid[k]) continue;
      float x[EPV];
      E::unpack_again(pn[r][k], x);
#pragma unroll
      for (int e = 0; e < EPV; ++e) part[2 * r] = fmaf(q[k][e], x[e], part[2 * r]);
#pragma unroll
      for (int e = 0; e < EPV; ++e) part[2 * r + 1] = fmaf(x[e], x[e], part[2 * r + 1]);
    }
  }
  cta_sum<2 * R>(part, red, 0);

  float wa[R], wc[R], M[R], a[R], c[R], hs[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    wa[r] = wc[r] = M[r] = a[r] = c[r] = hs[r] = 0.f;
    if (!ok[r]) continue;
    const float sp = part[2 * r] * rsqrtf(fmaf(part[2 * r + 1], p.inv_D, p.eps));
    M[r] = fmaxf(lse[r], sp);
    a[r] = expf(lse[r] - M[r]);
    c[r] = expf(sp - M[r]);
    const float inv = 1.f / (a[r] + c[r]);
    wa[r] = a[r] * inv;
    wc[r] = c[r] * inv;
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int k = 0; k < V; ++k) {
      if (!ok[r] || !valid[k]) continue;
      st_vec(static_cast<char *>(P.p_out) + off_of(r, k), pn[r][k]);
      float xo[EPV], xp[EPV], h[EPV];
      E::unpack(ov[r][k], xo);
      E::unpack_again(pn[r][k], xp);
#pragma unroll
      for (int e = 0; e < EPV; ++e) h[e] = fmaf(wa[r], xo[e], wc[r] * xp[e]);
      if (p.h) st_vec(static_cast<char *>(p.h) + off_of(r, k), E::pack(h));
      if (NORM) {
#pragma unroll
        for (int e = 0; e < EPV; ++e) hs[r] = fmaf(h[e], h[e], hs[r]);
      }
    }
  if (NORM) {
    // The next sublayer's pre-norm on the unrounded h: y = h / sqrt(mean h^2 + eps) (.) w_n.
    cta_sum<R>(hs, red_n, 0);
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (!ok[r]) continue;
      const float rn = rsqrtf(fmaf(hs[r], p.inv_D, P.neps));
#pragma unroll
      for (int k = 0; k < V; ++k) {
        if (!valid[k]) continue;
        float xo[EPV], xp[EPV], y[EPV];
        E::unpack(ov[r][k], xo);
        E::unpack_again(pn[r][k], xp);
#pragma unroll
        for (int e = 0; e < EPV; ++e) y[e] = fmaf(wa[r], xo[e], wc[r] * xp[e]) * rn * nw[k][e];
        st_vec(static_cast<char *>(P.y) + off_of(r, k), E::pack(y));
      }
    }
  }
  if (lt == 0 && p.lse_out) {
#pragma unroll
    for (int r = 0; r < R; ++r)
      if (ok[r]) p.lse_out[row[r]] = M[r] + logf(a[r] + c[r]);
  }
}

// The next sublayer's pre-norm as a pass of its own, for the first sublayer
// of a block, whose input is the phase-1 output itself:
//   y = x / sqrt(mean_d x^2 + eps) (.) w,   row by row.
// y may alias x: each thread reads its elements, the row is reduced, and the
// same thread writes the same elements.
template <typename T, int VPT, int TEAM>
__global__ void __launch_bounds__(TEAM ? 256 : 512)
rms_norm_kernel(const void *x, const float *__restrict__ w, void *y, int64_t rows, int nvec,
                float inv_D, float eps) {
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  __shared__ float red[TEAM ? 1 : 2 * 32];
  const int tpr = TEAM ? TEAM : blockDim.x;
  const int lt = TEAM ? (threadIdx.x % TEAM) : threadIdx.x;
  const int teams_per_cta = TEAM ? blockDim.x / TEAM : 1;
  const int team = TEAM ? threadIdx.x / TEAM : 0;
  const size_t row_bytes = (size_t)nvec * 16;
  const int64_t groups = (rows + teams_per_cta - 1) / teams_per_cta;
  int parity = 0;
  for (int64_t rg = blockIdx.x; rg < groups; rg += gridDim.x) {
    const int64_t row = rg * teams_per_cta + team;
    const bool row_ok = row < rows;
    const size_t row_off = (size_t)row * row_bytes;
    uint4 xv[VPT];
    float ss = 0.f;
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
      xv[kk] = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok && lt + kk * tpr < nvec)
        xv[kk] = *reinterpret_cast<const uint4 *>(static_cast<const char *>(x) + row_off +
                                                  (size_t)(lt + kk * tpr) * 16);
      float v[EPV];
      E::unpack(xv[kk], v);
#pragma unroll
      for (int e = 0; e < EPV; ++e) ss = fmaf(v[e], v[e], ss);
    }
    if (TEAM) {
      ss = team_sum_shfl<TEAM ? TEAM : 1>(ss);
    } else {
      float v1[1] = {ss};
      cta_sum<1>(v1, red, parity);
      parity ^= 1;
      ss = v1[0];
    }
    if (!row_ok) continue;
    const float rn = rsqrtf(fmaf(ss, inv_D, eps));
#pragma unroll
    for (int kk = 0; kk < VPT; ++kk) {
      const int j = lt + kk * tpr;
      if (j >= nvec) continue;
      float v[EPV], o[EPV];
      E::unpack(xv[kk], v);
#pragma unroll
      for (int e4 = 0; e4 < EPV; e4 += 4) {
        const float4 w4 = ld_f4(w + j * EPV + e4);
        o[e4 + 0] = v[e4 + 0] * rn * w4.x;
        o[e4 + 1] = v[e4 + 1] * rn * w4.y;
        o[e4 + 2] = v[e4 + 2] * rn * w4.z;
        o[e4 + 3] = v[e4 + 3] * rn * w4.w;
      }
      st_vec(static_cast<char *>(y) + row_off + (size_t)j * 16, E::pack(o));
    }
  }
}

// partial_out = (partial_in or 0) + 0.5 tanh(u (.) h), elementwise.
template <typename T>
__global__ void __launch_bounds__(256)
partial_update_kernel(const void *__restrict__ h, const void *pin, const float *__restrict__ u,
                      void *pout, int64_t total_vec, int nvec) {
  // pin may alias pout (in-place update): every vector is read, then written,
  // by the same thread, and pin is read through the coherent path.
  grid_dependency_wait();
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  constexpr int U = 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; base < total_vec;
       base += stride * U) {
    uint4 hv[U], pv[U];
#pragma unroll
    for (int t = 0; t < U; ++t) {
      const int64_t v = base + t * stride;
      hv[t] = make_uint4(0u, 0u, 0u, 0u);
      pv[t] = make_uint4(0u, 0u, 0u, 0u);
      if (v < total_vec) {
        hv[t] = ld_stream(static_cast<const uint4 *>(h) + v);
        if (pin) pv[t] = static_cast<const uint4 *>(pin)[v];
      }
    }
#pragma unroll
    for (int t = 0; t < U; ++t) {
      const int64_t v = base + t * stride;
      if (v >= total_vec) continue;
      const int j = (int)(v % nvec);
      float xh[EPV], xp[EPV], y[EPV];
      E::unpack(hv[t], xh);
      E::unpack(pv[t], xp);
#pragma unroll
      for (int e4 = 0; e4 < EPV; e4 += 4) {
        const float4 u4 = ld_f4(u + j * EPV + e4);
        y[e4 + 0] = xp[e4 + 0] + half_tanh(u4.x * xh[e4 + 0]);
        y[e4 + 1] = xp[e4 + 1] + half_tanh(u4.y * xh[e4 + 1]);
        y[e4 + 2] = xp[e4 + 2] + half_tanh(u4.z * xh[e4 + 2]);
        y[e4 + 3] = xp[e4 + 3] + half_tanh(u4.w * xh[e4 + 3]);
      }
      st_vec(static_cast<uint4 *>(pout) + v, E::pack(y));
    }
  }
}

namespace {

int epv_of(int dtype) { return dtype == ATTNRES_BF16 ? 8 : 4; }

struct Cfg {
  int vpt, team, threads;
  bool few = false;    // fused update+merge: two rows a CTA, query data in registers
};

bool choose(int D, int dtype, Cfg &c) {
  const int nvec = D / epv_of(dtype);
  if (nvec <= 64) {
    int need = (nvec + 1) / 2, team = 4;
    while (team < need) team *= 2;
    c = {2, team, 256};
    return true;
  }
  if (nvec <= 2048) {
    c = {4, 0, ((nvec + 3) / 4 + 31) / 32 * 32};
    return true;
  }
  return false;
}

template <typename T, int VPT, int TEAM>
cudaError_t run(const MergeParams &p, const Cfg &c, cudaStream_t st) {
  auto kern = merge_kernel<T, VPT, TEAM>;
  static int occ[16] = {0};
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
  return launch_dependent(kern, dim3(grid), dim3(c.threads), 0, st, p);
}

template <typename T>
cudaError_t dispatch(const MergeParams &p, const Cfg &c, cudaStream_t st) {
  switch (c.team) {
    case 0: return c.vpt == 2 ? run<T, 2, 0>(p, c, st) : run<T, 4, 0>(p, c, st);
    case 4: return run<T, 2, 4>(p, c, st);
    case 8: return run<T, 2, 8>(p, c, st);
    case 16: return run<T, 2, 16>(p, c, st);
    default: return run<T, 2, 32>(p, c, st);
  }
}


// Largest dynamic shared memory a fused update+merge launch asks for: the
// query and u (and the norm weight with the pre-norm) at the widest
// supported row (2048 vectors).
constexpr int mu_max_smem(bool norm) { return (norm ? 3 : 2) * 2048 * 8 * (int)sizeof(float); }

template <typename T, int VPT, int TEAM, bool SYNTH, bool NORM, int TPR = 0>
cudaError_t run_mu(const MergeUpdateParams &P, const Cfg &c, cudaStream_t st) {
  auto kern = merge_update_kernel<T, VPT, TEAM, SYNTH, NORM, TPR>;
  const size_t smem = (size_t)P.m.D * sizeof(float) * (1 + (SYNTH ? 1 : 0) + (NORM ? 1 : 0));
  struct Entry { int dev; size_t smem; int occ; };
  static Entry cache[16];
  static int used = 0;
  int dev = 0, o = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].smem == smem) o = cache[i].occ;
  if (o == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, mu_max_smem(NORM));
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, c.threads, smem);
    if (e != cudaSuccess) return e;
    if (o < 1) o = 1;
    if (used < 16) cache[used++] = {dev, smem, o};
  }
  const int per_cta = TEAM ? c.threads / TEAM : 1;
  const int64_t groups = (P.m.rows + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)o * sm_count();
  const int grid = (int)(groups < cap ? groups : cap);
  return launch_dependent(kern, dim3(grid), dim3(c.threads), smem, st, P);
}

template <typename T, bool SYNTH, bool NORM>
cudaError_t run_mu_few(const MergeUpdateParams &P, const Cfg &c, cudaStream_t st) {
  const int64_t grid = (P.m.rows + 1) / 2;
  return launch_dependent(merge_update_few_kernel<T, SYNTH, NORM>, dim3((unsigned)grid), dim3(c.threads), 0, st, P);
}

template <typename T, bool SYNTH, bool NORM>
cudaError_t dispatch_mu(const MergeUpdateParams &P, const Cfg &c, cudaStream_t st) {
  if (c.few) return run_mu_few<T, SYNTH, NORM>(P, c, st);
  // Rows that fill the CTA exactly run with its width built in, except the
  // plain step on 128 threads (D = 4096 bf16), where measured on a GB300 it
  // was slower (0.238 against 0.211 ms); with the pre-norm on the same rows
  // it is faster (0.232 against 0.266 ms), and so on 224 threads (D = 7168:
  // 0.736 against 0.776 ms).
  const bool exact = c.team == 0 && P.m.nvec == c.threads * c.vpt && (NORM || c.threads != 128);
  if (exact && c.vpt == 4) {
    switch (c.threads) {
      case 128: return run_mu<T, 4, 0, SYNTH, NORM, 128>(P, c, st);
      case 224: return run_mu<T, 4, 0, SYNTH, NORM, 224>(P, c, st);
      case 256: return run_mu<T, 4, 0, SYNTH, NORM, 256>(P, c, st);
      default: break;
    }
  }
  switch (c.team) {
    case 0: return c.vpt == 2 ? run_mu<T, 2, 0, SYNTH, NORM>(P, c, st) : run_mu<T, 4, 0, SYNTH, NORM>(P, c, st);
    case 4: return run_mu<T, 2, 4, SYNTH, NORM>(P, c, st);
    case 8: return run_mu<T, 2, 8, SYNTH, NORM>(P, c, st);
    case 16: return run_mu<T, 2, 16, SYNTH, NORM>(P, c, st);
    default: return run_mu<T, 2, 32, SYNTH, NORM>(P, c, st);
  }
}

template <typename T>
cudaError_t dispatch_mu_t(const MergeUpdateParams &P, const Cfg &c, cudaStream_t st) {
  const bool synth = P.u != nullptr, norm = P.nw != nullptr;
  if (synth) return norm ? dispatch_mu<T, true, true>(P, c, st) : dispatch_mu<T, true, false>(P, c, st);
  return norm ? dispatch_mu<T, false, true>(P, c, st) : dispatch_mu<T, false, false>(P, c, st);
}

template <typename T, int VPT, int TEAM>
cudaError_t run_norm(const RmsNormArgs &a, const Cfg &c) {
  auto kern = rms_norm_kernel<T, VPT, TEAM>;
  static int occ[16] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int &o = occ[dev & 15];
  if (o == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, c.threads, 0);
    if (e != cudaSuccess) return e;
    if (o < 1) o = 1;
  }
  const int per_cta = TEAM ? c.threads / TEAM : 1;
  const int64_t groups = (a.rows + per_cta - 1) / per_cta;
  const int64_t cap = (int64_t)o * sm_count();
  const int grid = (int)(groups < cap ? groups : cap);
  return launch_dependent(kern, dim3(grid), dim3(c.threads), 0, a.stream, a.x, a.weight, a.y, a.rows,
                          a.D / epv_of(a.dtype), 1.f / (float)a.D, a.eps);
}

template <typename T>
cudaError_t dispatch_norm(const RmsNormArgs &a, const Cfg &c) {
  switch (c.team) {
    case 0: return c.vpt == 2 ? run_norm<T, 2, 0>(a, c) : run_norm<T, 4, 0>(a, c);
    case 4: return run_norm<T, 2, 4>(a, c);
    case 8: return run_norm<T, 2, 8>(a, c);
    case 16: return run_norm<T, 2, 16>(a, c);
    default: return run_norm<T, 2, 32>(a, c);
  }
}

}  // namespace

cudaError_t launch_merge_update(const MergeUpdateArgs &a) {
  Cfg c;
  if (!choose(a.D, a.dtype, c)) return cudaErrorInvalidValue;
  // Few rows (decode): two vectors per thread, twice the threads on each
  // row, two rows a CTA with the query data in registers.
  if (c.team == 0 && a.rows <= 4 * sm_count() && (a.D / epv_of(a.dtype) + 1) / 2 <= 512)
    c = {2, 0, ((a.D / epv_of(a.dtype) + 1) / 2 + 31) / 32 * 32, true};
  MergeUpdateParams P;
  P.m.o = a.inter_out;
  P.m.lse = a.inter_lse;
  P.m.p = nullptr;
  P.m.nvec = a.D / epv_of(a.dtype);
  P.m.D = a.D;
  P.m.inv_D = 1.f / (float)a.D;
  P.m.eps = a.eps;
  P.m.rows = a.rows;
  P.m.q = a.query;
  P.m.g = a.gain;
  P.m.h = a.h_out;
  P.m.lse_out = a.out_lse;
  P.p_in = a.partial_in;
  P.sub = a.sub_out;
  P.u = a.u;
  P.p_out = a.partial_out;
  P.nw = a.norm_weight;
  P.neps = a.norm_eps;
  P.y = a.normed_out;
  if (a.dtype == ATTNRES_BF16) return dispatch_mu_t<__nv_bfloat16>(P, c, a.stream);
  return dispatch_mu_t<float>(P, c, a.stream);
}

cudaError_t launch_rms_norm(const RmsNormArgs &a) {
  Cfg c;
  if (!choose(a.D, a.dtype, c)) return cudaErrorInvalidValue;
  if (a.dtype == ATTNRES_BF16) return dispatch_norm<__nv_bfloat16>(a, c);
  return dispatch_norm<float>(a, c);
}

namespace {
}  // namespace

bool merge_supported(int D, int dtype) {
  Cfg c;
  return choose(D, dtype, c);
}

cudaError_t launch_merge(const MergeArgs &a) {
  Cfg c;
  if (!choose(a.D, a.dtype, c)) return cudaErrorInvalidValue;
  MergeParams p;
  p.o = a.inter_out;
  p.lse = a.inter_lse;
  p.p = a.partial;
  p.nvec = a.D / epv_of(a.dtype);
  p.D = a.D;
  p.inv_D = 1.f / (float)a.D;
  p.eps = a.eps;
  p.rows = a.rows;
  p.q = a.query;
  p.g = a.gain;
  p.h = a.h_out;
  p.lse_out = a.out_lse;
  return a.dtype == ATTNRES_BF16 ? dispatch<__nv_bfloat16>(p, c, a.stream)
                                 : dispatch<float>(p, c, a.stream);
}

cudaError_t launch_partial_update(const PartialUpdateArgs &a) {
  const int nvec = a.D / epv_of(a.dtype);
  const int64_t total = a.rows * nvec;
  const int threads = 256;
  int64_t blocks = (total + threads * 4 - 1) / (threads * 4);
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (a.dtype == ATTNRES_BF16)
    return launch_dependent(partial_update_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(threads), 0, a.stream,
                            a.h, a.partial_in, a.u, a.partial_out, total, nvec);
  return launch_dependent(partial_update_kernel<float>, dim3((unsigned)blocks), dim3(threads), 0, a.stream, a.h,
                          a.partial_in, a.u, a.partial_out, total, nvec);
}

}  // namespace attnres
