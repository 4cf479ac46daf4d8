// backward.cu -- backward of the depth aggregation (eq. A1-A3 of "Attention
// Residual 深度残差" taken in reverse; the fused forward/backward with
// recomputation named in "Attention Residuals：当网络深度也拥有寻址能力",
// sections "Depth attention 与 online merge reference" and "公开实现边界").
//
// For one token row with sources v_i, folded query w~ = w (.) gamma and the
// upstream gradient dh of h = sum_i alpha_i v_i:
//   r_i  = (mean_d v_i^2 + eps)^(-1/2),  s_i = r_i (w~ . v_i),  alpha = softmax(s)
//   da_i = dh . v_i,                      ds_i = alpha_i (da_i - sum_j alpha_j da_j)
//   dv_i = alpha_i dh + (ds_i r_i) w~ - (ds_i s_i r_i^2 / D) v_i
//   dw~ += (ds_i r_i) v_i                 (summed over every row)
// and dw = dw~ (.) gamma, dgamma = dw~ (.) w.
//
// A team of threads owns a row, each thread the same 16-byte vectors of
// every source (as in the forward kernel).  Pass A streams the n sources
// once with dh resident in registers and reduces the three dots per source;
// one warp of the team turns them into the softmax and the three per-source
// coefficients (kept in shared memory); pass B reads each source again --
// the row's sources were just read, so this is an L2 hit -- and writes dv_i.
// Nothing of size n x rows is stored.  dw~ accumulates in registers across
// the rows a team processes; each team writes its partial row [D] to the
// caller's workspace and a second kernel sums the partials in a fixed order
// (deterministic, no atomics).
#include <atomic>

#include "common.cuh"
#include "launch.h"

namespace attnres {

constexpr int kBwdTeams = 8;    // rows per CTA when TEAM lanes of a warp own a row
constexpr int kBwdGroupA = 4;   // sources per load + reduction step in pass A
constexpr int kBwdGroupB = 2;   // sources per load step in pass B

struct BwdParams {
  const void *src[kMaxSources];
  void *dsrc[kMaxSources];
  int n;
  int nvec;
  int D;
  float inv_D;
  float eps;
  int64_t rows;
  const float *q;
  const float *g;
  const void *dh;
  int accumulate;
  float *ws;       // [gridDim.x * teams per CTA][D] partial dw~ rows, or nullptr
};

template <int W>
__device__ __forceinline__ float lanes_max(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// TEAM > 0: TEAM lanes of a warp own a row (kBwdTeams rows per CTA).
// TEAM == 0: the whole CTA owns a row; with TPR > 0 rows that exactly fill a
// CTA of TPR threads (nvec == TPR * VPT), so the per-vector offsets are
// constants and every vector is valid.
template <typename T, int VPT, int TEAM, int TPR>
__global__ void __launch_bounds__(TEAM ? kBwdTeams * TEAM : (TPR ? TPR : 512), TPR ? 512 / (TPR ? TPR : 512) : 1)
aggregate_backward_kernel(const __grid_constant__ BwdParams p) {
  using E = Elt<T>;
  constexpr int EPV = E::EPV;
  constexpr int NE = VPT * EPV;
  constexpr int GA = kBwdGroupA, GB = kBwdGroupB;
  constexpr int TPC = TEAM ? kBwdTeams : 1;
  constexpr int W = TEAM ? TEAM : 32;     // lanes that run the per-row softmax
  constexpr int KR = 4 * GA;               // per-source sums, padded to a power of two (3 used of 4)
  __shared__ float red[TEAM ? 1 : 2 * 32 * KR];
  __shared__ float coef[TPC][kMaxSources][3];

  static_assert(TPR == 0 || TEAM == 0, "a built-in thread count is for CTA teams");
  const int tpr = TPR ? TPR : (TEAM ? TEAM : blockDim.x);
  const int lt = TEAM ? (threadIdx.x % TEAM) : threadIdx.x;
  const int team = TEAM ? threadIdx.x / TEAM : 0;
  float(*cf)[3] = coef[team];

  float qe[NE];
  bool valid[VPT];
#pragma unroll
  for (int k = 0; k < VPT; ++k) {
    const int j = lt + k * tpr;
    valid[k] = TPR ? true : j < p.nvec;
#pragma unroll
    for (int e4 = 0; e4 < EPV; e4 += 4) {
      float4 w4 = make_float4(0.f, 0.f, 0.f, 0.f), g4 = make_float4(1.f, 1.f, 1.f, 1.f);
      if (valid[k]) {
        w4 = ld_f4(p.q + j * EPV + e4);
        if (p.g) g4 = ld_f4(p.g + j * EPV + e4);
      }
      qe[k * EPV + e4 + 0] = w4.x * g4.x;
      qe[k * EPV + e4 + 1] = w4.y * g4.y;
      qe[k * EPV + e4 + 2] = w4.z * g4.z;
      qe[k * EPV + e4 + 3] = w4.w * g4.w;
    }
  }
  // As packed fp32 pairs (two FMAs per instruction): the folded query and
  // the query-gradient accumulator.
  using PR = Pairs<T>;
  constexpr int NP = PR::NP;
  uint64_t qp[VPT * NP], accp[VPT * NP];
#pragma unroll
  for (int j = 0; j < VPT * NP; ++j) {
    qp[j] = pair(qe[2 * j], qe[2 * j + 1]);
    accp[j] = 0ull;
  }

  const size_t row_bytes = (size_t)p.nvec * 16;
  const int64_t groups = (p.rows + TPC - 1) / TPC;
  int parity = 0;
  // Pass A's reads of the sources are read again by pass B a few
  // microseconds later: they stay in L2 (evict_last); pass B's reads and the
  // gradients it writes are last uses (evict_first).
  const uint64_t keep = l2_policy_keep(), drop = l2_policy_drop();
  for (int64_t rg = blockIdx.x; rg < groups; rg += gridDim.x) {
    const int64_t row = rg * TPC + team;
    const bool row_ok = row < p.rows;
    const size_t row_off = (size_t)row * row_bytes;

    const size_t thr_off = row_off + (size_t)lt * 16;  // this thread's first vector of the row
    uint64_t gp[VPT * NP];  // dh of this row, as pairs
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok && valid[k]) x = ld_stream_vec<TPR>(static_cast<const char *>(p.dh) + thr_off, k, tpr);
      PR::split(x, gp + k * NP);
    }

    // Pass A: sum v^2, w~ . v and dh . v for every source.  With a whole
    // CTA on the row, a few threads first ask L2 for the next group's rows
    // (one bulk prefetch per row), so its loads find them there after this
    // group's reduction.
    for (int i0 = 0; i0 < p.n; i0 += GA) {
      if (!TEAM && row_ok && threadIdx.x < GA && i0 + GA + (int)threadIdx.x < p.n)
        prefetch_l2_bulk(static_cast<const char *>(p.src[i0 + GA + threadIdx.x]) + row_off, (uint32_t)row_bytes);
      uint4 v[GA][VPT];
#pragma unroll
      for (int j = 0; j < GA; ++j)
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          v[j][k] = make_uint4(0u, 0u, 0u, 0u);
          if (i0 + j < p.n && row_ok && valid[k])
            v[j][k] = ld_hint_vec<TPR>(static_cast<const char *>(p.src[i0 + j]) + thr_off, k, tpr, keep);
        }
      float part[KR];
#pragma unroll
      for (int j = 0; j < KR; ++j) part[j] = 0.f;
#pragma unroll
      for (int j = 0; j < GA; ++j) {
        if (i0 + j >= p.n) break;   // the last group's sources past n (the same for every thread)
        uint64_t ss = 0ull, dq = 0ull, dg = 0ull;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          uint64_t x[NP];
          PR::split(v[j][k], x);
#pragma unroll
          for (int m = 0; m < NP; ++m) {
            fma_pair(ss, x[m], x[m]);
            fma_pair(dq, qp[k * NP + m], x[m]);
            fma_pair(dg, gp[k * NP + m], x[m]);
          }
        }
        part[4 * j + 0] = pair_sum(ss);
        part[4 * j + 1] = pair_sum(dq);
        part[4 * j + 2] = pair_sum(dg);
        part[4 * j + 3] = 0.f;
      }
      if (TEAM) {
#pragma unroll
        for (int j = 0; j < GA; ++j)
#pragma unroll
          for (int m = 0; m < 3; ++m) part[4 * j + m] = team_sum_shfl<TEAM ? TEAM : 1>(part[4 * j + m]);
      } else {
        cta_sum_rs<KR>(part, red, parity);
        parity ^= 1;
      }
      if (lt == 0) {
#pragma unroll
        for (int j = 0; j < GA; ++j)
          if (i0 + j < p.n) {
            cf[i0 + j][0] = part[4 * j + 0];
            cf[i0 + j][1] = part[4 * j + 1];
            cf[i0 + j][2] = part[4 * j + 2];
          }
      }
    }
    if (TEAM) __syncwarp(); else __syncthreads();

    // Softmax over the sources and the backward coefficients, by W lanes:
    // cf[i] = (alpha_i, ds_i r_i, ds_i s_i r_i^2 / D).
    if (TEAM || threadIdx.x < 32) {
      float mx = -INFINITY;
      for (int i = lt; i < p.n; i += W) {
        const float r = rsqrtf(fmaf(cf[i][0], p.inv_D, p.eps));
        mx = fmaxf(mx, cf[i][1] * r);
      }
      mx = lanes_max<W>(mx);
      float z = 0.f, zg = 0.f;
      for (int i = lt; i < p.n; i += W) {
        const float r = rsqrtf(fmaf(cf[i][0], p.inv_D, p.eps));
        const float e = expf(cf[i][1] * r - mx);
        z += e;
        zg = fmaf(e, cf[i][2], zg);
      }
      z = team_sum_shfl<W>(z);
      zg = team_sum_shfl<W>(zg);
      const float inv_z = 1.f / z;
      const float mean_da = zg * inv_z;
      for (int i = lt; i < p.n; i += W) {
        const float r = rsqrtf(fmaf(cf[i][0], p.inv_D, p.eps));
        const float s = cf[i][1] * r;
        const float a = expf(s - mx) * inv_z;
        const float ds = a * (cf[i][2] - mean_da);
        cf[i][0] = a;
        cf[i][1] = ds * r;
        cf[i][2] = ds * s * r * r * p.inv_D;
      }
    }
    if (TEAM) __syncwarp(); else __syncthreads();

    // Pass B: dv_i = alpha_i dh + (ds_i r_i) w~ - (ds_i s_i r_i^2 / D) v_i.
    // Meanwhile L2 is asked for the next row's dh and first group of sources.
    if (!TEAM && threadIdx.x <= GA) {
      const int64_t nrow = (rg + gridDim.x) * TPC;
      if (nrow < p.rows) {
        const void *base = threadIdx.x == GA ? p.dh : (threadIdx.x < p.n ? p.src[threadIdx.x] : nullptr);
        if (base) prefetch_l2_bulk(static_cast<const char *>(base) + (size_t)nrow * row_bytes, (uint32_t)row_bytes);
      }
    }
    for (int i0 = 0; i0 < p.n; i0 += GB) {
      uint4 v[GB][VPT], din[GB][VPT];
#pragma unroll
      for (int j = 0; j < GB; ++j)
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          v[j][k] = din[j][k] = make_uint4(0u, 0u, 0u, 0u);
          if (i0 + j < p.n && row_ok && valid[k]) {
            v[j][k] = ld_hint_vec<TPR>(static_cast<const char *>(p.src[i0 + j]) + thr_off, k, tpr, drop);
            if (p.accumulate)
              din[j][k] = *reinterpret_cast<const uint4 *>(static_cast<const char *>(p.dsrc[i0 + j]) + thr_off +
                                                           (size_t)k * tpr * 16);
          }
        }
#pragma unroll
      for (int j = 0; j < GB; ++j) {
        if (i0 + j >= p.n || !row_ok) continue;
        const float a = cf[i0 + j][0], b = cf[i0 + j][1], c = cf[i0 + j][2];
        const uint64_t a2 = pair(a, a), b2 = pair(b, b), nc2 = pair(-c, -c);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          if (!valid[k]) continue;
          uint64_t x[NP], d[NP];
          PR::split(v[j][k], x);
#pragma unroll
          for (int m = 0; m < NP; ++m) {
            d[m] = 0ull;
            fma_pair(d[m], nc2, x[m]);               // -c v
            fma_pair(d[m], b2, qp[k * NP + m]);      // + (ds r) w~
            fma_pair(d[m], a2, gp[k * NP + m]);      // + alpha dh
            fma_pair(accp[k * NP + m], b2, x[m]);    // dw~ += (ds r) v
          }
          float o[EPV];
#pragma unroll
          for (int m = 0; m < NP; ++m) unpair(d[m], o[2 * m], o[2 * m + 1]);
          if (p.accumulate) {
            float w[EPV];
            E::unpack(din[j][k], w);
#pragma unroll
            for (int e = 0; e < EPV; ++e) o[e] += w[e];
          }
          st_hint(static_cast<char *>(p.dsrc[i0 + j]) + thr_off + (size_t)k * tpr * 16, E::pack(o), drop);
        }
      }
    }
    if (TEAM) __syncwarp(); else __syncthreads();  // cf is rewritten by the next row
  }

  if (p.ws) {
    float *dst = p.ws + ((int64_t)blockIdx.x * TPC + team) * p.D;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      if (!valid[k]) continue;
      float *d = dst + (lt + k * tpr) * EPV;
      float w[EPV];
#pragma unroll
      for (int m = 0; m < NP; ++m) unpair(accp[k * NP + m], w[2 * m], w[2 * m + 1]);
#pragma unroll
      for (int e4 = 0; e4 < EPV; e4 += 4)
        *reinterpret_cast<float4 *>(d + e4) = make_float4(w[e4], w[e4 + 1], w[e4 + 2], w[e4 + 3]);
    }
  }
}

// dw~[d] = sum over the P partial rows, in row order; then dw = dw~ (.) gamma
// and dgamma = dw~ (.) w.  A CTA owns 32 columns; its 8 warps each sum every
// 8th partial row (coalesced 128-byte rows), then warp 0 adds the 8 sums.
__global__ void __launch_bounds__(256)
aggregate_backward_reduce_kernel(const float *__restrict__ ws, int P, int D, const float *__restrict__ w,
                                 const float *__restrict__ g, float *dw, float *dg) {
  __shared__ float part[8][33];
  const int lane = threadIdx.x & 31, slice = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (col < D)
    for (int r = slice; r < P; r += 8) s += ws[(size_t)r * D + col];
  part[slice][lane] = s;
  __syncthreads();
  if (slice == 0 && col < D) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += part[k][lane];
    if (dw) dw[col] = t * (g ? g[col] : 1.f);
    if (dg) dg[col] = t * w[col];
  }
}

namespace {

int epv_of(int dtype) { return dtype == ATTNRES_BF16 ? 8 : 4; }

struct Cfg {
  int team, threads;
  int tpr;  // CTA teams: the built-in thread count (rows that fill the CTA exactly), or 0
};

bool choose(int D, int dtype, Cfg &c) {
  const int nvec = D / epv_of(dtype);
  if (nvec <= 64) {
    int need = (nvec + 1) / 2, team = 4;
    while (team < need) team *= 2;
    c = {team, kBwdTeams * team, 0};
    return true;
  }
  if (nvec <= 1024) {
    const int threads = ((nvec + 1) / 2 + 31) / 32 * 32;
    const bool exact = nvec == 2 * threads;
    c = {0, threads, exact && (threads == 64 || threads == 128 || threads == 256) ? threads : 0};
    return true;
  }
  return false;
}

// Resident CTAs per SM of one instantiation on the current device.
template <typename T, int TEAM, int TPR>
cudaError_t occupancy(const Cfg &c, int &o) {
  static int occ[16] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  int &slot = occ[dev & 15];
  if (slot == 0) {
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&slot, aggregate_backward_kernel<T, 2, TEAM, TPR>,
                                                                  c.threads, 0);
    if (e != cudaSuccess) return e;
    if (slot < 1) slot = 1;
  }
  o = slot;
  return cudaSuccess;
}

template <typename T, int TEAM, int TPR>
cudaError_t run(const BwdParams &p0, const AggregateBackwardArgs &a, const Cfg &c) {
  constexpr int TPC = TEAM ? kBwdTeams : 1;
  int o = 0;
  cudaError_t e = occupancy<T, TEAM, TPR>(c, o);
  if (e != cudaSuccess) return e;
  BwdParams p = p0;
  const int64_t groups = (a.rows + TPC - 1) / TPC;
  int64_t grid = (int64_t)o * sm_count();
  if (groups < grid) grid = groups;
  if (p.ws && a.workspace_rows / TPC < grid) grid = a.workspace_rows / TPC;
  if (grid < 1) return cudaErrorInvalidValue;
  aggregate_backward_kernel<T, 2, TEAM, TPR><<<(int)grid, c.threads, 0, a.stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || !p.ws) return e;
  aggregate_backward_reduce_kernel<<<(a.D + 31) / 32, 256, 0, a.stream>>>(
      p.ws, (int)(grid * TPC), a.D, a.query, a.gain, a.grad_query, a.grad_gain);
  return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const BwdParams &p, const AggregateBackwardArgs &a, const Cfg &c) {
  switch (c.team) {
    case 0:
      switch (c.tpr) {
        case 64: return run<T, 0, 64>(p, a, c);
        case 128: return run<T, 0, 128>(p, a, c);
        case 256: return run<T, 0, 256>(p, a, c);
        default: return run<T, 0, 0>(p, a, c);
      }
    case 4: return run<T, 4, 0>(p, a, c);
    case 8: return run<T, 8, 0>(p, a, c);
    case 16: return run<T, 16, 0>(p, a, c);
    default: return run<T, 32, 0>(p, a, c);
  }
}

template <typename T>
cudaError_t rows_for(const Cfg &c, int64_t &rows) {
  int o = 0;
  cudaError_t e = cudaSuccess;
  switch (c.team) {
    case 0:
      switch (c.tpr) {
        case 64: e = occupancy<T, 0, 64>(c, o); break;
        case 128: e = occupancy<T, 0, 128>(c, o); break;
        case 256: e = occupancy<T, 0, 256>(c, o); break;
        default: e = occupancy<T, 0, 0>(c, o); break;
      }
      break;
    case 4: e = occupancy<T, 4, 0>(c, o); break;
    case 8: e = occupancy<T, 8, 0>(c, o); break;
    case 16: e = occupancy<T, 16, 0>(c, o); break;
    default: e = occupancy<T, 32, 0>(c, o); break;
  }
  rows = (int64_t)o * sm_count() * (c.team ? kBwdTeams : 1);
  return e;
}

}  // namespace

// ---------------------------------------------------------------------------
// Fixed scratch for the allocation-free entry point: room for the partial
// rows of the query gradient, shared by every call of that entry point.
// ---------------------------------------------------------------------------
constexpr int64_t kNoAllocScratchFloats = (int64_t)1 << 21;   // 8 MiB
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

int64_t noalloc_scratch_floats() { return kNoAllocScratchFloats; }

// Device address of the scratch array on the current device.  Host code
// cannot use the symbol itself as a device pointer; the address is looked
// up once per device (with that device current) and cached.  The slots are
// atomic: two host threads making their first call on a device at the same
// time may both look the address up, and both store the same value.  A
// cudaDeviceReset unloads the library's device code, so the cached address
// is stale afterwards (the header says so).
cudaError_t noalloc_scratch(float *&ptr) {
  static std::atomic<float *> cache[64];
  ptr = nullptr;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  float *p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    p = static_cast<float *>(addr);
    cache[dev].store(p, std::memory_order_release);
  }
  ptr = p;
  return cudaSuccess;
}

bool aggregate_backward_supported(int D, int dtype) {
  Cfg c;
  return choose(D, dtype, c);
}

int aggregate_backward_rows_per_partial(int D, int dtype) {
  Cfg c;
  if (!choose(D, dtype, c)) return 0;
  return c.team ? kBwdTeams : 1;
}

cudaError_t aggregate_backward_workspace_rows(int D, int dtype, int64_t &rows) {
  Cfg c;
  rows = 0;
  if (!choose(D, dtype, c)) return cudaErrorInvalidValue;
  return dtype == ATTNRES_BF16 ? rows_for<__nv_bfloat16>(c, rows) : rows_for<float>(c, rows);
}

cudaError_t launch_aggregate_backward(const AggregateBackwardArgs &a) {
  Cfg c;
  if (!choose(a.D, a.dtype, c)) return cudaErrorInvalidValue;
  BwdParams p;
  for (int i = 0; i < a.n; ++i) {
    p.src[i] = a.sources[i];
    p.dsrc[i] = a.grad_sources[i];
  }
  p.n = a.n;
  p.nvec = a.D / epv_of(a.dtype);
  p.D = a.D;
  p.inv_D = 1.f / (float)a.D;
  p.eps = a.eps;
  p.rows = a.rows;
  p.q = a.query;
  p.g = a.gain;
  p.dh = a.grad_out;
  p.accumulate = a.accumulate ? 1 : 0;
  p.ws = (a.grad_query || a.grad_gain) ? a.workspace : nullptr;
  if (a.dtype == ATTNRES_BF16) return dispatch<__nv_bfloat16>(p, a, c);
  return dispatch<float>(p, a, c);
}

}  // namespace attnres
