// phase1_tc.cu -- phase 1 of the two-phase Block scheme ("Attention Residual
// 深度残差", "两阶段算法（inter / intra）", inter step / attn_with_stats;
// eq. A1-A3 for S queries at once) for bf16 sources, in two kernels.
//
// Per token, phase 1 is two contractions over the n completed block
// summaries v_i: the S x n scores s_{q,i} = w~_q . v_i / rms(v_i), a dense
// contraction over D whose queries are shared by every token, and the S
// outputs o_q = sum_i alpha_{q,i} v_i (n terms per element, different for
// every token).
//
// Query split.  A small kernel folds w~ = w (.) gamma once per call and
// splits it into bf16 hi + lo parts (w~ ~= hi + lo to ~16 bits), 48 rows of
// D (hi at 0..S-1, lo at 24..24+S-1, unused rows zero), parked in the last
// 48 * D elements of the output buffer -- rows that kernel B overwrites
// after kernel A is done with them (so no scratch memory is needed).
//
// Kernel A (scores, tensor cores).  A CTA owns a tile of 128 token rows.
// TMA streams each summary of the tile in 64-feature chunks (box 64 x 128,
// 128-byte swizzle), one summary after the other, through a ring of
// shared-memory stages, each with a producer lane of its own; each stage
// also carries the parked query parts for the same 64 features (box 64 x
// 48), the MMA's B operand (N = 48).  tcgen05.mma accumulates, per summary
// i, the 128 x 48 partial scores in its own TMEM columns [48 i, 48 i + 48).
// Four warps (one thread per token row) read the same stages to accumulate
// each row's sum of squares, then run the epilogue: scores = (hi + lo) *
// rsqrt(ss / D + eps), the softmax over the n summaries, m and lse to their
// outputs, and alpha (fp32, [n][Sp][2] with Sp = S rounded up to even, each
// value twice) into the first S*n*4 bytes of the token's own o[0] row -- a
// region kernel B reads before it overwrites that row with o_0, so no
// scratch memory is needed.
//
// Kernel B (outputs).  A CTA owns one token at a time, one thread per 16-byte
// chunk of the row (rows wider than 4096 features in two pieces); a 3-stage
// cp.async pipeline brings in the next tokens' n summary chunks and alpha
// while the current token's S outputs are formed, two queries at a time,
// with packed fp32x2 FMAs, and stored.  The pages' shape (9 summaries, 24
// queries) has an instantiation with both counts built in.
//
// Raw-score mode.  With S >= 3 (and room in the token's o[1] row), and for
// more than ten summaries (the Full two-phase schedule), kernel A runs over
// work items (tile, five summaries) at two CTAs per SM and writes raw scores
// only; a softmax kernel then turns them into alpha, m and lse.  Beyond ten
// summaries the outputs come from a tensor-core kernel (mma.sync, K = 16
// summaries per step) or, for S > 16, a packed-FMA kernel.
//
// Each summary byte is read twice (once per kernel); there is no cluster or
// cross-CTA exchange.  Every in-kernel wait is bounded: one that runs out
// records a flag, its role stops issuing work, and the CTA drains what it
// has in flight before it ends.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

ATTNRES_DEFINE_ERROR_FLAG(take_error_phase1_tc)

namespace attnres {
namespace tc {

constexpr int kRows = 128;            // token rows per tile of kernel A (MMA M)
constexpr int kKc = 64;               // features per chunk (one 128-byte swizzle row)
constexpr int kMaxN = 10;             // summaries: TMEM columns n * 48 <= 480
static_assert(kMaxN == kP1TcMaxSources, "one pass of the fused phase 1 takes ten summaries");
constexpr int kMaxS = 24;             // queries
constexpr int kNQ = 2 * kMaxS;        // B rows: hi parts at 0..S-1, lo parts at 24..24+S-1
constexpr int kStages = 9;            // ring of (summary chunk 16 KB + query chunk 6 KB) stages
constexpr uint32_t kVBytes = kRows * kKc * 2;
constexpr uint32_t kQBytes = kNQ * kKc * 2;
constexpr uint32_t kStageBytes = kVBytes + kQBytes;   // both parts 1024-byte aligned
constexpr int kBStages = 3;           // kernel B: tokens in flight (cp.async stages)
constexpr int kWarpsA = 6;            // 0-3: sums of squares + epilogue, 4: TMA, 5: MMA
constexpr int kThreadsA = kWarpsA * 32;
constexpr uint32_t kOffBar = kStages * kStageBytes;
constexpr uint32_t kSmemA = kOffBar + 64 * 8 + 1024;     // barriers + alignment slack
// Work items of CH summaries (10, or 5 in raw-score mode): the stage ring and
// the TMEM columns of a CTA.  With five, a CTA takes 256 TMEM columns and
// about 93 KB of shared memory, so two CTAs share an SM: the tensor-map
// loads one CTA issues are served one box at a time (16 KB boxes stream at
// 4.2 TB/s with one CTA per SM on GB300, 6.2 TB/s with two).
__host__ __device__ constexpr int stages_a(int CH) { return CH == kMaxN ? kStages : 4; }
__host__ __device__ constexpr uint32_t tmem_cols_a(int CH) { return CH * kNQ <= 256 ? 256u : 512u; }
__host__ __device__ constexpr uint32_t smem_a(int CH) { return (uint32_t)stages_a(CH) * kStageBytes + 64 * 8 + 1024; }

template <int NM>
struct ParamsAT {
  CUtensorMap tmap[NM];               // one per summary: [rows, D] bf16, box 64 x 128
  CUtensorMap qmap;                   // parked query parts: [48, D] bf16, box 64 x 48
  void *out;                          // [S, rows, D] bf16 (alpha parked in o[0])
  float *out_max;                     // [S, rows] or nullptr
  float *out_lse;                     // [S, rows]
  int64_t rows;
  int n, S, D;
  float eps, inv_D;
  // Raw-score mode (any number of summaries): the work items are (tile,
  // chunk of CH summaries); each writes the scores s[row][i][q] of its
  // chunk to raw ([rows][n][S] fp32) and nothing else; the softmax over all
  // of them runs afterwards.  Without raw, n <= 10 and there is one chunk.
  float *raw;
  int raw_n, raw_off;                 // raw's summary count and this launch's first summary
  int64_t raw_stride;                 // floats from one row's scores to the next (raw_n * S when packed)
  // Split mode (few token rows, raw set): the work items are (tile, chunk
  // of CH summaries, part kp of kparts slices of the features); each writes
  // its partial dot products and partial sums of squares, unnormalised, to
  // slot kp of the row's raw area: [kp][n S dots, then n sums of squares].
  int kparts;                         // 1: every item covers all of D
  int chunk;                          // summaries per work item, 1..CH (the template's bound)
  long long wait_limit;               // SM clock cycles any wait of the work loop may take
};
// The fused path (up to ten summaries) and the raw-score path, which takes
// up to kManyMaps summaries per launch (the tensor maps ride in the kernel
// parameters: 128 bytes each, within the 32 KB parameter limit).
constexpr int kManyMaps = 200;
using ParamsA = ParamsAT<kMaxN>;
using ParamsAMany = ParamsAT<kManyMaps>;
static_assert(sizeof(ParamsAMany) <= 32764, "kernel parameters are limited to 32764 bytes");

struct ParamsB {
  const void *src[kMaxN];
  void *out;
  int64_t rows;
  int n, S, D, nvec;
  int parts, nvp;   // a row is formed in `parts` pieces of nvp 16-byte chunks (D > 4096: two)
};

// --- small PTX wrappers ------------------------------------------------------
// Bounded waits.  A wait of the work loop that runs out raises the error flag
// and returns false; the role that waited then stops issuing work (it never
// signals a stage it did not consume, so no producer refills a stage that is
// still being read), and every role that issued asynchronous work drains it
// before the CTA ends (drain_wait, with the fixed drain limit): the TMA
// producer lanes wait for their last copies to land, the MMA thread for its
// last tensor-core operations to complete.  Only then is TMEM freed.
__device__ __forceinline__ bool wait_local(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_wait_for(bar, parity, limit)) return true;
  raise_timeout();
  return false;
}
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (!mbar_wait_for(bar, parity, kDrainLimitCycles)) raise_timeout();
}
// The error flag as a launch finds it: set means a wait of an earlier launch
// ran out and the host has not taken the error yet; such a launch issues
// nothing (its results would be invalid as well).
__device__ __forceinline__ bool error_pending() {
  return *reinterpret_cast<volatile unsigned int *>(&g_error_flag) != 0;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Byte offset of 16-byte chunk `j` of row `r` inside a 1024-byte, 8-row atom
// written by TMA (or by hand) with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t j) { return r * 128u + ((j ^ (r & 7u)) << 4); }


// -----------------------------------------------------------------------------
// Query split: parts[row][d], row < 24: bf16(w~), row >= 24: bf16(w~ - hi)
// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) p1_qsplit_kernel(const float *__restrict__ q,
                                                        const float *__restrict__ g, int S, int D,
                                                        __nv_bfloat16 *__restrict__ parts) {
  grid_dependency_wait();
  const int64_t total = (int64_t)kMaxS * D;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int row = (int)(idx / D), d = (int)(idx % D);
    float hi = 0.f, lo = 0.f;
    if (row < S) {
      const float qe = q[(size_t)row * D + d] * (g ? g[(size_t)row * D + d] : 1.f);
      hi = __bfloat162float(__float2bfloat16_rn(qe));
      lo = qe - hi;
    }
    parts[(size_t)row * D + d] = __float2bfloat16_rn(hi);
    parts[(size_t)(kMaxS + row) * D + d] = __float2bfloat16_rn(lo);
  }
}

// -----------------------------------------------------------------------------
// Kernel A: scores on tcgen05, softmax, alpha / m / lse
// -----------------------------------------------------------------------------
template <int NM, int CH = kMaxN>
__global__ void __launch_bounds__(kThreadsA, CH == kMaxN ? 1 : 2) p1_scores_kernel(const __grid_constant__ ParamsAT<NM> p) {
  grid_dependency_wait();
  static_assert(CH >= 1 && CH <= CH, "summaries per work item");
  constexpr int ST = stages_a(CH);                 // stage ring
  constexpr uint32_t TC = tmem_cols_a(CH);         // TMEM columns of this CTA
  constexpr uint32_t OFF_BAR = (uint32_t)ST * kStageBytes;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.n, S = p.S;
  const uint32_t b0 = base + OFF_BAR;
  auto VFULL = [&](int s) { return b0 + 8u * s; };
  auto VEMPTY = [&](int s) { return b0 + 8u * (ST + s); };
  const uint32_t TDONE = b0 + 8u * (2 * ST);
  const uint32_t TFREE = TDONE + 8u;
  const uint32_t MDRAIN = TFREE + 8u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_BAR + 8 * (2 * ST + 3));
  uint32_t *skip = tmem_slot + 1;
  const long long lim = p.wait_limit;

  if (threadIdx.x == 0) {
    *skip = error_pending() ? 1u : 0u;
    for (int s = 0; s < ST; ++s) {
      mbar_init(VFULL(s), 1);
      mbar_init(VEMPTY(s), 1 + 4);    // the MMA's commit + the four row warps
    }
    mbar_init(TDONE, 1);
    mbar_init(TFREE, 4);
    mbar_init(MDRAIN, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (*skip) return;                  // nothing issued yet: no copy, no TMEM
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), TC);
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Work items: (tile of 128 rows, chunk of up to p.chunk <= CH summaries),
  // tile-minor.
  const int64_t tiles = (p.rows + kRows - 1) / kRows;
  const int kparts = p.kparts;
  const int ch = p.chunk;
  const int64_t items = tiles * ((n + ch - 1) / ch) * kparts;
  const int64_t my_tiles = items > (int64_t)blockIdx.x ? (items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int KCP = p.D / kKc / kparts;                 // 64-feature chunks per item
  // item -> (tile, first summary i0 and count nc, feature chunks [kc0, kc0 + KCP))
  auto item_of = [&](int64_t tl, int64_t &tile, int &i0, int &nc, int &kc0) {
    const int64_t item = (int64_t)blockIdx.x + tl * gridDim.x;
    tile = item % tiles;
    const int64_t rest = item / tiles;
    kc0 = (int)(rest % kparts) * KCP;
    i0 = (int)(rest / kparts) * ch;
    nc = n - i0 < ch ? n - i0 : ch;
  };

  if (warp == 4) {
    // ---------------- TMA producers: (tile, summary, chunk) stages ----------------
    // Each stage carries 64 features of one summary for the tile's 128 rows
    // and the same 64 features of the query parts.  Walking the features of
    // one summary in order keeps consecutive stages on neighbouring bytes.
    // The bulk copies one thread issues complete one after another (about
    // 0.4 us each on GB300, whatever their size), so every stage has a
    // producer lane of its own: lane s issues each use of stage s.  All lanes
    // walk the same sequence; the stage's empty barrier orders its uses.
    if (lane < ST) {
      int64_t g = 0, last = -1;
      int s = 0;  // g % ST
      bool ok = true;
      for (int64_t tl = 0; tl < my_tiles && ok; ++tl) {
        int64_t tile;
        int i0, nc, kc0;
        item_of(tl, tile, i0, nc, kc0);
        for (int i = 0; i < nc && ok; ++i)
          for (int kc = kc0; kc < kc0 + KCP; ++kc, ++g) {
            if (s == lane) {
              // a stage is refilled only once every consumer is done with it
              // (which they signal only after its copy has landed)
              if (g >= ST && !wait_local(VEMPTY(s), (uint32_t)((g / ST - 1) & 1), lim)) { ok = false; break; }
              mbar_expect_tx(VFULL(s), kStageBytes);
              const uint32_t st = base + (uint32_t)s * kStageBytes;
              tma_load_2d(st, &p.tmap[i0 + i], kc * kKc, (int)(tile * kRows), VFULL(s));
              tma_load_2d(st + kVBytes, &p.qmap, kc * kKc, 0, VFULL(s));
              last = g;
            }
            if (++s == ST) s = 0;
          }
      }
      // drain: this lane's last copies have landed before the CTA may exit
      // (its earlier uses of the stage landed before the stage was refilled)
      if (last >= 0) drain_wait(VFULL(lane), (uint32_t)((last / ST) & 1));
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kRows, kNQ);
      int64_t g = 0;
      bool ok = true;
      for (int64_t tl = 0; tl < my_tiles && ok; ++tl) {
        // the epilogue has read the last tile's accumulators
        if (tl >= 1 && !wait_local(TFREE, (uint32_t)((tl - 1) & 1), lim)) break;
        tc_fence_after();
        int64_t tile;
        int i0, nc, kc0;
        item_of(tl, tile, i0, nc, kc0);
        for (int i = 0; i < nc && ok; ++i)
          for (int kc = kc0; kc < kc0 + KCP; ++kc, ++g) {
            const int s = (int)(g % ST);
            if (!wait_local(VFULL(s), (uint32_t)((g / ST) & 1), lim)) { ok = false; break; }
            tc_fence_after();
            const uint32_t st = base + (uint32_t)s * kStageBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = sw128_desc(st + kk * 32u, 1024u);
              const uint64_t b = sw128_desc(st + kVBytes + kk * 32u, 1024u);
              mma_bf16(tmem_base + (uint32_t)(i * kNQ), a, b, idesc, (kc > kc0 || kk != 0) ? 1u : 0u);
            }
            mma_commit(VEMPTY(s));
          }
        if (ok) mma_commit(TDONE);
      }
      // drain: every MMA this thread issued has completed
      mma_commit(MDRAIN);
      drain_wait(MDRAIN, 0);
    }
  } else {
    // ---------------- warps 0-3: row sums of squares, then the epilogue ----------------
    const int r = threadIdx.x;                                   // token row in the tile = TMEM lane
    const uint32_t taddr = tmem_base + ((uint32_t)(warp * 32) << 16);
    int64_t g = 0;
    bool ok = true;
    for (int64_t tl = 0; tl < my_tiles && ok; ++tl) {
      int64_t tile;
      int i0, nc, kc0;
      item_of(tl, tile, i0, nc, kc0);
      float ss[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) ss[i] = 0.f;
#pragma unroll
      for (int i = 0; i < CH; ++i) {
        if (i >= nc || !ok) continue;
        for (int kc = kc0; kc < kc0 + KCP; ++kc, ++g) {
          const int s = (int)(g % ST);
          // every lane waits; the warp goes on only if all of them saw the
          // stage land (the code below syncs the warp)
          if (!__all_sync(0xffffffffu, wait_local(VFULL(s), (uint32_t)((g / ST) & 1), lim))) { ok = false; break; }
          const unsigned char *row = sm + (uint32_t)s * kStageBytes;
          uint4 v[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const uint4 *>(row + swz((uint32_t)r, (uint32_t)j));
          float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // eight independent chains
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float x[8];
            Elt<__nv_bfloat16>::unpack(v[j], x);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(x[e], x[e], acc[e]);
          }
          ss[i] += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
          __syncwarp();
          if (lane == 0) mbar_arrive(VEMPTY(s));
        }
      }
      // epilogue: scores -> softmax over the n summaries -> alpha, m, lse
      if (!ok || !__all_sync(0xffffffffu, wait_local(TDONE, (uint32_t)(tl & 1), lim))) { ok = false; break; }
      tc_fence_after();
      float rinv[CH];
#pragma unroll
      for (int i = 0; i < CH; ++i) rinv[i] = rsqrtf(fmaf(ss[i], p.inv_D, p.eps));
      if (kparts > 1) {                                          // split mode: partials
        const int64_t row = tile * kRows + r;
        float c[kNQ];
        float *slot = p.raw + (size_t)row * p.raw_stride + (size_t)(kc0 / KCP) * (size_t)(n * S + n);
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          if (i >= nc) continue;
          tmem_ld16(taddr + i * kNQ, c);
          tmem_ld16(taddr + i * kNQ + 16, c + 16);
          tmem_ld16(taddr + i * kNQ + 32, c + 32);
          tmem_wait_ld();
          if (row < p.rows) {
#pragma unroll
            for (int q = 0; q < kMaxS; ++q)
              if (q < S) slot[(size_t)(i0 + i) * S + q] = c[q] + c[kMaxS + q];
            slot[(size_t)n * S + i0 + i] = ss[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(TFREE);
        continue;
      }
      if (p.raw) {                                               // raw-score mode
        const int64_t row = tile * kRows + r;
        float c[kNQ];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          if (i >= nc) continue;
          tmem_ld16(taddr + i * kNQ, c);
          tmem_ld16(taddr + i * kNQ + 16, c + 16);
          tmem_ld16(taddr + i * kNQ + 32, c + 32);
          tmem_wait_ld();
          if (row < p.rows) {
            float *dst = p.raw + (size_t)row * p.raw_stride + (size_t)(p.raw_off + i0 + i) * S;
#pragma unroll
            for (int q = 0; q < kMaxS; ++q)
              if (q < S) dst[q] = (c[q] + c[kMaxS + q]) * rinv[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(TFREE);
        continue;
      }
      float m[kMaxS], den[kMaxS];
#pragma unroll
      for (int q = 0; q < kMaxS; ++q) { m[q] = -INFINITY; den[q] = 0.f; }
      float c[kNQ];
#pragma unroll
      for (int i = 0; i < CH; ++i) {                          // pass 1: max
        if (i >= nc) continue;
        tmem_ld16(taddr + i * kNQ, c);
        tmem_ld16(taddr + i * kNQ + 16, c + 16);
        tmem_ld16(taddr + i * kNQ + 32, c + 32);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kMaxS; ++q) m[q] = fmaxf(m[q], (c[q] + c[kMaxS + q]) * rinv[i]);
      }
#pragma unroll
      for (int i = 0; i < CH; ++i) {                          // pass 2: denominators
        if (i >= nc) continue;
        tmem_ld16(taddr + i * kNQ, c);
        tmem_ld16(taddr + i * kNQ + 16, c + 16);
        tmem_ld16(taddr + i * kNQ + 32, c + 32);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < kMaxS; ++q) den[q] += expf((c[q] + c[kMaxS + q]) * rinv[i] - m[q]);
      }
      const int64_t row = tile * kRows + r;
      const bool row_ok = row < p.rows;
      float *alpha = reinterpret_cast<float *>(static_cast<char *>(p.out) + (size_t)row * p.D * 2);
#pragma unroll
      for (int i = 0; i < CH; ++i) {                          // pass 3: alpha [n][S]
        if (i >= nc) continue;
        tmem_ld16(taddr + i * kNQ, c);
        tmem_ld16(taddr + i * kNQ + 16, c + 16);
        tmem_ld16(taddr + i * kNQ + 32, c + 32);
        tmem_wait_ld();
        float a[kMaxS];
#pragma unroll
        for (int q = 0; q < kMaxS; ++q) a[q] = expf((c[q] + c[kMaxS + q]) * rinv[i] - m[q]) / den[q];
        if (row_ok) {
          const int Sp = S + (S & 1);
#pragma unroll
          for (int q = 0; q < kMaxS; q += 2)
            if (q < S)
              *reinterpret_cast<float4 *>(alpha + 2 * (i * Sp + q)) = make_float4(a[q], a[q], a[q + 1], a[q + 1]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(TFREE);
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < kMaxS; ++q) {
          if (q < S) {
            p.out_lse[(size_t)q * p.rows + row] = m[q] + logf(den[q]);
            if (p.out_max) p.out_max[(size_t)q * p.rows + row] = m[q];
          }
        }
      }
    }
  }
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TC);
  }
}

// -----------------------------------------------------------------------------
// Kernel B: outputs o_q = sum_i alpha_{q,i} v_i
// -----------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// NS, SQ > 0: the number of summaries and of queries built in (the loops
// over them unroll fully and every alpha load has a constant offset);
// 0: taken from the parameters.
template <int PARTS, int NS, int SQ>
__global__ void __launch_bounds__(512, 1) p1_outputs_kernel(const __grid_constant__ ParamsB p) {
  grid_dependency_wait();
  extern __shared__ uint4 vbuf[];                     // [kBStages][n][nvp] 16-byte chunks
  __shared__ __align__(16) float alpha[kBStages][2 * kMaxN * kMaxS];   // [n][Sp][2]
  static_assert(NS <= kMaxN && SQ <= kMaxS, "built-in shape within the kernel's limits");
  constexpr int kQUnroll = 1;  // unrolling the query pairs spills at 128 registers
  const int tid = threadIdx.x;
  const int n = NS ? NS : p.n, S = SQ ? SQ : p.S, nvp = p.nvp;
  constexpr int parts = PARTS;
  const size_t row_bytes = (size_t)p.D * 2;
  // Items are (token, piece), the pieces of a token consecutive on the same
  // CTA: the first piece brings in alpha (parked in o[0][t], which that piece
  // then overwrites), the next one reads it from the first piece's stage.
  const int64_t my = (p.rows > (int64_t)blockIdx.x ? (p.rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0) * parts;
  const int Sp = S + (S & 1);                          // queries per alpha row (even)
  const int alpha_vecs = (2 * n * Sp) / 4;

  auto prefetch = [&](int64_t k, int buf) {
    const int64_t t = blockIdx.x + (k / parts) * gridDim.x;
    const int part = (int)(k % parts);
    if (tid < nvp) {
      for (int i = 0; i < n; ++i)
        cp_async16(&vbuf[(size_t)(buf * n + i) * nvp + tid],
                   static_cast<const char *>(p.src[i]) + (size_t)t * row_bytes + (size_t)(part * nvp + tid) * 16);
    }
    if (part == 0 && tid < alpha_vecs)
      cp_async16(&alpha[buf][tid * 4], static_cast<const char *>(p.out) + (size_t)t * row_bytes + (size_t)tid * 16);
    cp_async_commit();
  };

  // Tokens k + 1 and k + 2 are in flight while token k is formed.
  for (int64_t k = 0; k < kBStages - 1; ++k) {
    if (k < my) prefetch(k, (int)k);
    else cp_async_commit();                           // keep one group per token
  }
  for (int64_t k = 0; k < my; ++k) {
    const int buf = (int)(k % kBStages);
    const int64_t t = blockIdx.x + (k / parts) * gridDim.x;
    const int part = (int)(k % parts);
    if (k + kBStages - 1 < my) prefetch(k + kBStages - 1, (int)((k + kBStages - 1) % kBStages));
    else cp_async_commit();
    cp_async_wait<kBStages - 1>();
    __syncthreads();    // stage `buf` complete for every thread; alpha of t read before o[0][t] is written
    if (tid < nvp) {
      uint64_t xp[kMaxN][4];                        // the row chunk of every summary, as fp32 pairs
#pragma unroll
      for (int i = 0; i < kMaxN; ++i)
        if (i < n) Pairs<__nv_bfloat16>::split(vbuf[(size_t)(buf * n + i) * nvp + tid], xp[i]);
      char *dst = static_cast<char *>(p.out) + (size_t)t * row_bytes + (size_t)(part * nvp + tid) * 16;
      const size_t qstride = (size_t)p.rows * row_bytes;
      // alpha came with the token's first piece (k - part); the stages in
      // between carry no alpha, so its buffer is intact
      const float *al = alpha[(k - part) % kBStages];
#pragma unroll kQUnroll
      for (int q = 0; q < S; q += 2) {              // queries in pairs
        uint64_t acc0[4] = {0, 0, 0, 0}, acc1[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < kMaxN; ++i) {
          if (i < n) {
            // alpha of queries q and q + 1, each already a duplicated pair
            const ulonglong2 a = *reinterpret_cast<const ulonglong2 *>(al + 2 * (i * Sp + q));
            const uint64_t a0 = a.x, a1 = a.y;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              fma_pair(acc0[m], a0, xp[i][m]);
              fma_pair(acc1[m], a1, xp[i][m]);
            }
          }
        }
        float h0[8], h1[8];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          unpair(acc0[m], h0[2 * m], h0[2 * m + 1]);
          unpair(acc1[m], h1[2 * m], h1[2 * m + 1]);
        }
        st_stream(dst + (size_t)q * qstride, Elt<__nv_bfloat16>::pack(h0));
        if (q + 1 < S) st_stream(dst + (size_t)(q + 1) * qstride, Elt<__nv_bfloat16>::pack(h1));
      }
    }
    __syncthreads();    // every thread is done with stage `buf` before it is refilled
  }
}

// -----------------------------------------------------------------------------
// Up to ten summaries with the scores computed in raw mode: each token's raw
// scores [n][S] sit in its o[1] row; one thread per (row, query) takes their
// softmax, writes m and lse, and writes alpha into the token's o[0] row in
// the layout the outputs kernel reads ([n][Sp][2], each value twice; the
// pad query of an odd S gets zeros).  The outputs kernel then overwrites
// both rows.
// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
p1_park_softmax_kernel(const float *raw, float *alpha, int64_t row_floats, int64_t rows, int n, int S,
                       float *out_max, float *out_lse) {
  grid_dependency_wait();
  const int Sp = S + (S & 1);
  const int64_t total = rows * Sp;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = g / Sp;
    const int q = (int)(g % Sp);
    float *al = alpha + (size_t)row * row_floats;
    if (q >= S) {                                   // the pad query of an odd S
      for (int i = 0; i < n; ++i) *reinterpret_cast<float2 *>(al + 2 * (i * Sp + q)) = make_float2(0.f, 0.f);
      continue;
    }
    const float *s = raw + (size_t)row * row_floats + q;
    float m = -INFINITY;
    for (int i = 0; i < n; ++i) m = fmaxf(m, s[(size_t)i * S]);
    float den = 0.f;
    for (int i = 0; i < n; ++i) den += expf(s[(size_t)i * S] - m);
    const float inv = 1.f / den;
    for (int i = 0; i < n; ++i) {
      const float a = expf(s[(size_t)i * S] - m) * inv;
      *reinterpret_cast<float2 *>(al + 2 * (i * Sp + q)) = make_float2(a, a);
    }
    out_lse[(size_t)q * rows + row] = m + logf(den);
    if (out_max) out_max[(size_t)q * rows + row] = m;
  }
}

// -----------------------------------------------------------------------------
// Split mode: each token's o[1] row holds kparts slots of partial dot
// products [n][S] and partial sums of squares [n] over slices of the
// features.  One CTA per token: thread (i, q) adds up its kparts partials in
// slot order (consecutive threads read consecutive queries), the first n
// threads the sums of squares; then thread q takes the softmax over the n
// scores, writes m and lse, and writes alpha into the token's o[0] row in
// the layout the outputs kernel reads.
// -----------------------------------------------------------------------------
constexpr int kSplitThreads = 256;
static_assert(kSplitThreads >= kMaxN * kMaxS, "one thread per (summary, query)");

__global__ void __launch_bounds__(kSplitThreads)
p1_split_softmax_kernel(const float *raw, float *alpha, int64_t row_floats, int64_t rows, int n, int S, int kparts,
                        float inv_D, float eps, float *out_max, float *out_lse) {
  grid_dependency_wait();
  __shared__ float dots[kMaxN * kMaxS];
  __shared__ float rn[kMaxN];
  const int tid = threadIdx.x;
  const int Sp = S + (S & 1);
  const int slot = n * S + n;
  for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    const float *pr = raw + (size_t)row * row_floats;
    if (tid < n * S) {
      float d = 0.f;
      for (int kp = 0; kp < kparts; ++kp) d += pr[(size_t)kp * slot + tid];
      dots[tid] = d;
    }
    if (tid < n) {
      float ss = 0.f;
      for (int kp = 0; kp < kparts; ++kp) ss += pr[(size_t)kp * slot + (size_t)n * S + tid];
      rn[tid] = rsqrtf(fmaf(ss, inv_D, eps));
    }
    __syncthreads();
    if (tid < Sp) {
      const int q = tid;
      float *al = alpha + (size_t)row * row_floats;
      if (q >= S) {                                   // the pad query of an odd S
        for (int i = 0; i < n; ++i) *reinterpret_cast<float2 *>(al + 2 * (i * Sp + q)) = make_float2(0.f, 0.f);
      } else {
        float sc[kMaxN];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxN; ++i) {
          sc[i] = -INFINITY;
          if (i < n) {
            sc[i] = dots[i * S + q] * rn[i];
            m = fmaxf(m, sc[i]);
          }
        }
        float den = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxN; ++i)
          if (i < n) den += expf(sc[i] - m);
        const float inv = 1.f / den;
#pragma unroll
        for (int i = 0; i < kMaxN; ++i)
          if (i < n) {
            const float a = expf(sc[i] - m) * inv;
            *reinterpret_cast<float2 *>(al + 2 * (i * Sp + q)) = make_float2(a, a);
          }
        out_lse[(size_t)q * rows + row] = m + logf(den);
        if (out_max) out_max[(size_t)q * rows + row] = m;
      }
    }
    __syncthreads();                                  // the next token's partials reuse the buffers
  }
}

// -----------------------------------------------------------------------------
// More than ten summaries: softmax over the raw scores, then the outputs
// -----------------------------------------------------------------------------
// One thread per (row, query): max, sum and normalisation over the n raw
// scores (consecutive threads read consecutive queries), alpha written in
// place; m and lse to their [S, rows] outputs.
__global__ void __launch_bounds__(256)
p1_many_softmax_kernel(float *scores, int64_t rows, int n, int S, float *out_max, float *out_lse) {
  grid_dependency_wait();
  const int64_t total = rows * S;
  for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = g / S;
    const int q = (int)(g % S);
    float *s = scores + (size_t)row * n * S + q;
    float m = -INFINITY;
    for (int i = 0; i < n; ++i) m = fmaxf(m, s[(size_t)i * S]);
    float den = 0.f;
    for (int i = 0; i < n; ++i) den += expf(s[(size_t)i * S] - m);
    const float inv = 1.f / den;
    for (int i = 0; i < n; ++i) s[(size_t)i * S] = expf(s[(size_t)i * S] - m) * inv;
    out_lse[(size_t)q * rows + row] = m + logf(den);
    if (out_max) out_max[(size_t)q * rows + row] = m;
  }
}

struct ParamsB2 {
  const void *src[kMaxSources];
  const float *alpha;   // [rows][n][S]
  void *out;            // [S, rows, D] bf16
  int64_t rows;
  int n, S, D;
};

// o_q = sum_i alpha_{q,i} v_i for any number of summaries: a CTA per token at
// a time, each thread four features (8 bytes of every summary row) and the
// S outputs' accumulators as packed pairs.  The token's alpha is staged in
// shared memory as duplicated pairs (two queries per 16-byte read, feeding
// four packed FMAs); its summary rows are asked into L2 32 ahead and loaded
// four at a time.
constexpr int kB2Ahead = 32;

__global__ void __launch_bounds__(512)
p1_many_outputs_kernel(const __grid_constant__ ParamsB2 p) {
  grid_dependency_wait();
  extern __shared__ uint64_t adup[];  // [n][Sp]
  const int tid = threadIdx.x;
  const int n = p.n, S = p.S, Sp = S + (S & 1);
  const bool valid = tid * 4 < p.D;
  const size_t row_bytes = (size_t)p.D * 2;
  if (S & 1)
    for (int i = tid; i < n; i += blockDim.x) adup[(size_t)i * Sp + S] = 0ull;
  for (int64_t t = blockIdx.x; t < p.rows; t += gridDim.x) {
    __syncthreads();                                   // the previous token's readers are done
    if (tid < n && tid < kB2Ahead)
      prefetch_l2_bulk(static_cast<const char *>(p.src[tid]) + (size_t)t * row_bytes, (uint32_t)row_bytes);
    const float *at = p.alpha + (size_t)t * n * S;
    for (int idx = tid; idx < n * S; idx += blockDim.x) {
      const float a = at[idx];
      adup[(size_t)(idx / S) * Sp + idx % S] = pair(a, a);
    }
    __syncthreads();
    uint64_t acc[kMaxS][2];
#pragma unroll
    for (int q = 0; q < kMaxS; ++q) acc[q][0] = acc[q][1] = 0ull;
    constexpr int U = 4;  // summaries whose loads are in flight together
    for (int i = 0; i < n; i += U) {
      if (tid < U && i + kB2Ahead + tid < n)
        prefetch_l2_bulk(static_cast<const char *>(p.src[i + kB2Ahead + tid]) + (size_t)t * row_bytes,
                         (uint32_t)row_bytes);
      uint2 w[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        w[u] = make_uint2(0u, 0u);
        if (valid && i + u < n)
          w[u] = *reinterpret_cast<const uint2 *>(static_cast<const char *>(p.src[i + u]) + (size_t)t * row_bytes +
                                                  (size_t)tid * 8);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (i + u >= n) break;
        const uint64_t x0 = ((uint64_t)(w[u].x & 0xffff0000u) << 32) | (uint64_t)(w[u].x << 16);
        const uint64_t x1 = ((uint64_t)(w[u].y & 0xffff0000u) << 32) | (uint64_t)(w[u].y << 16);
        const uint4 *ad = reinterpret_cast<const uint4 *>(adup + (size_t)(i + u) * Sp);
#pragma unroll
        for (int qq = 0; qq < kMaxS / 2; ++qq) {
          if (2 * qq >= S) continue;
          const uint4 a = ad[qq];
          const uint64_t a0 = ((uint64_t)a.y << 32) | a.x, a1 = ((uint64_t)a.w << 32) | a.z;
          fma_pair(acc[2 * qq][0], a0, x0);
          fma_pair(acc[2 * qq][1], a0, x1);
          fma_pair(acc[2 * qq + 1][0], a1, x0);
          fma_pair(acc[2 * qq + 1][1], a1, x1);
        }
      }
    }
    if (valid) {
#pragma unroll
      for (int q = 0; q < kMaxS; ++q) {
        if (q >= S) continue;
        float y[4];
        unpair(acc[q][0], y[0], y[1]);
        unpair(acc[q][1], y[2], y[3]);
        const uint2 v = make_uint2(Elt<__nv_bfloat16>::pack_word(y[0], y[1]), Elt<__nv_bfloat16>::pack_word(y[2], y[3]));
        __stcs(reinterpret_cast<uint2 *>(static_cast<char *>(p.out) + ((size_t)q * p.rows + t) * row_bytes + (size_t)tid * 8), v);
      }
    }
  }
}

// -----------------------------------------------------------------------------
// Outputs for many summaries on tensor cores (S <= 16, D a multiple of 256 up
// to 2048).  Per token, O[q][d] = sum_i alpha[q][i] v_i[d] is a dense
// contraction with K = n: warp-level mma.m16n8k16 (bf16 in, fp32 accumulate),
// M = 16 queries, N = 8 features per tile, K = 16 summaries per step.  The
// summary rows are N-major (contiguous along d), which ldmatrix.trans turns
// into the B fragments; alpha (fp32) is split into bf16 hi + lo, two MMAs per
// tile, so it keeps about 16 significant bits.  The summary rows stream
// through a cp.async ring of NS slots, 16 rows per step (rows past n
// zero-filled), with NS - 1 steps in flight while one is multiplied; each
// warp holds the accumulators of its 128 features across the steps.  A work
// item is one of a token's `parts` pieces of WARPS x 128 features, so two
// CTAs of 8 warps can share an SM at D = 2048.
// -----------------------------------------------------------------------------
constexpr int kTcK = 16;           // summaries per step (mma K)
static_assert(kTcK == 16, "alpha staging indexes queries with & 15 and summaries with >> 4");
constexpr int kTcWarps = 16;       // 512 threads

struct ParamsB3 {
  const void *src[kMaxSources];
  const float *alpha;   // [rows][n][S]
  void *out;            // [S, rows, D] bf16
  int64_t rows;
  int n, S, D;
  int parts;            // a token's features in `parts` pieces, each a work item of its own
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
               "{%8, %9}, {%0, %1, %2, %3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// 16-byte cp.async that reads `bytes` (16 or 0) and zero-fills the rest.
__device__ __forceinline__ void cp_async16_zfill(void *smem, const void *gmem, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem)), "l"(gmem), "r"(bytes)
               : "memory");
}

__host__ __device__ constexpr size_t tc_row_v(int D) { return (size_t)D * 2 + 16; }   // padded: no bank conflicts
__host__ __device__ constexpr size_t tc_row_a(int n) { return (size_t)((n + kTcK - 1) / kTcK * kTcK) * 2 + 16; }
// NS ring slots of 16 summary rows; alpha in two item buffers with two
// slots, in one with three (staged between items behind a barrier).
__host__ __device__ constexpr size_t tc_smem(int n, int D, int NS = 2) {
  return (size_t)NS * kTcK * tc_row_v(D) + (NS == 2 ? 2 : 1) * 2 * (size_t)kTcK * tc_row_a(n);
}

template <int WARPS, int NS = 2>
__global__ void __launch_bounds__(WARPS * 32, 16 / WARPS)
p1_many_outputs_tc_kernel(const __grid_constant__ ParamsB3 p) {
  static_assert(NS == 2 || NS == 3, "two or three ring slots");
  constexpr int AB = NS == 2 ? 2 : 1;                            // alpha item buffers
  grid_dependency_wait();
  extern __shared__ __align__(16) unsigned char sm3[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = p.n, S = p.S, D = p.D, parts = p.parts;
  const int DF = D / parts;                                      // features per work item
  const int KS = (n + kTcK - 1) / kTcK, KP = KS * kTcK;
  const size_t RV = tc_row_v(DF), RA = tc_row_a(n);
  unsigned char *vring = sm3;                                    // [NS][16][RV]
  unsigned char *abuf = sm3 + NS * kTcK * RV;                    // [AB items][hi, lo][16][RA]
  const size_t row_bytes = (size_t)D * 2;
  const int chunks = DF / 8;                                     // 16-byte chunks per item row
  const int ntw = DF / 8 / WARPS;                                // n-tiles per warp (even, <= 16)
  const int64_t items = p.rows * parts;
  const int64_t my_tokens = items > (int64_t)blockIdx.x ? (items - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int64_t total = my_tokens * KS;

  // work item j of this CTA: (token, piece of the features), pieces of a
  // token on different CTAs.  Taken once per item: the steps walk items with
  // counters, no division per step.
  auto item_at = [&](int64_t j, int64_t &t, int &fo) {
    const int64_t it = (int64_t)blockIdx.x + j * gridDim.x;
    t = it / parts;
    fo = (int)(it - t * parts) * DF;
  };
  // When the CTA width is a multiple of the chunks per row, a thread's chunk
  // column is fixed and its rows step by a constant (no division per copy).
  const bool whole_rows = blockDim.x % chunks == 0;
  const int rstep = whole_rows ? blockDim.x / chunks : 0, r0 = tid / chunks, ch0 = tid % chunks;
  // step kk of the item (token t, first feature f0): 16 summary rows -> slot sl
  auto issue = [&](int64_t t, int f0, int kk, int sl) {
    const size_t fo = (size_t)f0 * 2;
    unsigned char *slot = vring + (size_t)sl * kTcK * RV;
    if (whole_rows) {
      const size_t goff = (size_t)t * row_bytes + fo + (size_t)ch0 * 16;
      for (int r = r0; r < kTcK; r += rstep) {
        const int i = kk * kTcK + r;
        const char *gp = static_cast<const char *>(p.src[i < n ? i : 0]) + goff;
        cp_async16_zfill(slot + (size_t)r * RV + (size_t)ch0 * 16, gp, i < n ? 16u : 0u);
      }
    } else {
      for (int c = tid; c < kTcK * chunks; c += blockDim.x) {
        const int r = c / chunks, ch = c % chunks, i = kk * kTcK + r;
        const char *gp = static_cast<const char *>(p.src[i < n ? i : 0]) + (size_t)t * row_bytes + fo + (size_t)ch * 16;
        cp_async16_zfill(slot + (size_t)r * RV + (size_t)ch * 16, gp, i < n ? 16u : 0u);
      }
    }
    cp_async_commit();
  };
  // alpha of item j (token t) -> bf16 hi / lo [q][i]; consecutive threads
  // take consecutive queries of one summary (alpha is [n][S] per token)
  auto stage_alpha = [&](int64_t j, int64_t t) {
    unsigned char *ab = abuf + (size_t)(j % AB) * 2 * kTcK * RA;
    const float *at = p.alpha + (size_t)t * n * S;
    for (int idx = tid; idx < kTcK * KP; idx += blockDim.x) {
      const int q = idx & (kTcK - 1), i = idx >> 4;
      const float a = (q < S && i < n) ? at[(size_t)i * S + q] : 0.f;
      const __nv_bfloat16 hi = __float2bfloat16_rn(a);
      const __nv_bfloat16 lo = __float2bfloat16_rn(a - __bfloat162float(hi));
      *reinterpret_cast<__nv_bfloat16 *>(ab + (size_t)q * RA + (size_t)i * 2) = hi;
      *reinterpret_cast<__nv_bfloat16 *>(ab + (size_t)(kTcK + q) * RA + (size_t)i * 2) = lo;
    }
  };

  float c[16][4];
  // step g = j * KS + kk computes; step g + 1 = jn * KS + kn is issued
  int64_t j = 0, t = 0, jn = 0, tn = 0;
  int kk = 0, fo = 0, kn = 0, fon = 0;
  if (total > 0) {
    item_at(0, t, fo);
    tn = t;
    fon = fo;
    if (NS == 2) stage_alpha(0, t);
    issue(t, fo, 0, 0);
    for (int s = 1; s < NS - 1; ++s) {                       // steps 1 .. NS - 2, one commit group each
      if (s < total) {
        if (++kn == KS) {
          kn = 0;
          item_at(++jn, tn, fon);
        }
        issue(tn, fon, kn, s);
      } else {
        cp_async_commit();
      }
    }
  }
  int slot_c = 0;                // slot of step g
  for (int64_t g = 0; g < total; ++g) {
    cp_async_wait<NS - 2>();     // step g has landed (one commit group per step)
    __syncthreads();             // step g's rows are visible; the slot of step g - 1 is free
    if (NS == 3 && kk == 0) {    // a new item: its alpha into the single buffer (every warp is past the last item)
      stage_alpha(j, t);
      __syncthreads();
    }
    if (g + NS - 1 < total) {
      if (++kn == KS) {
        kn = 0;
        item_at(++jn, tn, fon);
      }
      issue(tn, fon, kn, slot_c == 0 ? NS - 1 : slot_c - 1);
    } else if (NS > 2) {
      cp_async_commit();
    }
    if (NS == 2 && kk == 0 && j + 1 < my_tokens) {           // the other alpha buffer (last read by token j - 1)
      int64_t t1;
      int f1;
      item_at(j + 1, t1, f1);
      stage_alpha(j + 1, t1);
    }
    if (kk == 0) {
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) c[nt][0] = c[nt][1] = c[nt][2] = c[nt][3] = 0.f;
    }
    // A fragments (hi, lo) of this step: rows q, columns kk*16 .. +15
    const unsigned char *ab = abuf + (size_t)(j % AB) * 2 * kTcK * RA;
    const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = kk * kTcK + (lane >> 4) * 8;
    uint32_t ahi[4], alo[4];
    ldsm_x4(smem_u32(ab + (size_t)mrow * RA + (size_t)mcol * 2), ahi);
    ldsm_x4(smem_u32(ab + (size_t)(kTcK + mrow) * RA + (size_t)mcol * 2), alo);
    // B fragments from the slot: rows k (summaries), 8 features per tile; two tiles per ldmatrix
    const unsigned char *slot = vring + (size_t)slot_c * kTcK * RV;
    const int krow = (lane & 7) + ((lane >> 3) & 1) * 8, kcol = (lane >> 4) * 8;
#pragma unroll
    for (int pr = 0; pr < 8; ++pr) {
      if (2 * pr >= ntw) break;
      const int f0 = (warp * ntw + 2 * pr) * 8;
      uint32_t b[4];
      ldsm_x4_trans(smem_u32(slot + (size_t)krow * RV + (size_t)(f0 + kcol) * 2), b);
      mma_16816(c[2 * pr], ahi, b[0], b[1]);
      mma_16816(c[2 * pr], alo, b[0], b[1]);
      mma_16816(c[2 * pr + 1], ahi, b[2], b[3]);
      mma_16816(c[2 * pr + 1], alo, b[2], b[3]);
    }
    if (kk == KS - 1) {          // token done: rows q = lane/4 and lane/4 + 8, two features per tile
      const int q0 = lane >> 2, fc = (lane & 3) * 2;
#pragma unroll
      for (int nt = 0; nt < 16; ++nt) {
        if (nt >= ntw) break;
        const int f = fo + (warp * ntw + nt) * 8 + fc;
        if (q0 < S)
          __stcs(reinterpret_cast<uint32_t *>(static_cast<char *>(p.out) + ((size_t)q0 * p.rows + t) * row_bytes + (size_t)f * 2),
                 Elt<__nv_bfloat16>::pack_word(c[nt][0], c[nt][1]));
        if (q0 + 8 < S)
          __stcs(reinterpret_cast<uint32_t *>(static_cast<char *>(p.out) + ((size_t)(q0 + 8) * p.rows + t) * row_bytes + (size_t)f * 2),
                 Elt<__nv_bfloat16>::pack_word(c[nt][2], c[nt][3]));
      }
    }
    if (++kk == KS) {
      kk = 0;
      if (++j < my_tokens) item_at(j, t, fo);
    }
    if (++slot_c == NS) slot_c = 0;
  }
  cp_async_wait<0>();
}

// -----------------------------------------------------------------------------
// Host side
// -----------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

size_t smem_b(int n, int D) { return (size_t)kBStages * n * (D / 8) * 16; }

}  // namespace tc

bool phase1_tc_supported(int n, int D, int dtype, int S) {
  if (dtype != ATTNRES_BF16 || n < 1 || n > tc::kMaxN || S < 1 || S > tc::kMaxS) return false;
  if (D % tc::kKc != 0 || D > 8192) return false;            // kernel B: a thread per 16 bytes of a row piece
  const int parts = D > 4096 ? 2 : 1;
  // alpha fits in o[0]'s row, inside the first piece of it
  if ((size_t)(S + (S & 1)) * n * 8 > (size_t)D * 2 / parts) return false;
  if (tc::smem_b(n, D / parts) + sizeof(float) * tc::kBStages * 2 * tc::kMaxN * tc::kMaxS > 227 * 1024)
    return false;
  return tc::encode_fn() != nullptr;
}

// Feature slices for split mode, or 1 when it does not apply: only when the
// normal work items (128-row tiles x five summaries) would leave most SMs
// idle, and only with room in o[1] for the partials of every slice (o[1]
// must lie before the parked query parts).  The largest divisor of the
// 64-feature chunk count that keeps the items within two per SM.
int split_parts(const Phase1Args &a) {
  using namespace tc;
  const int64_t tiles = (a.rows + kRows - 1) / kRows;
  if (a.S < 3 || (int64_t)(a.S - 2) * a.rows < kNQ) return 1;
  if (tiles * ((a.n + 4) / 5) >= sm_count()) return 1;
  const int KC = a.D / kKc;
  const int64_t slots = 2 * (int64_t)sm_count();
  const size_t per_part = (size_t)(a.n * a.S + a.n) * 4;
  for (int kp = KC; kp >= 2; --kp)
    if (KC % kp == 0 && tiles * a.n * kp <= slots && (size_t)kp * per_part <= (size_t)a.D * 2) return kp;
  return 1;
}

// Summaries per raw-mode work item, 1..max: each CTA streams its
// tensor-map boxes at about the same rate however many it has in flight, so
// a launch takes about (waves of items) x (summaries per item); few
// summaries leave SMs idle with five per item, and a nearly empty last wave
// doubles the time.  The chunk with the least waves x (chunk + 1/4), the
// quarter standing for an item's fixed cost (ramp and epilogue).
static int many_chunk(int64_t tiles, int n, int max_chunk) {
  const int64_t slots = 2 * (int64_t)sm_count();   // resident CTAs
  int best = max_chunk;
  double best_cost = 1e30;
  for (int c = 1; c <= max_chunk; ++c) {
    const int64_t it = tiles * ((n + c - 1) / c);
    const double cost = (double)((it + slots - 1) / slots) * (c + 0.25);
    if (cost < best_cost) {
      best_cost = cost;
      best = c;
    }
  }
  return best;
}

cudaError_t launch_phase1_tc(const Phase1Args &a) {
  using namespace tc;
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  // Kernel A
  ParamsA pa;
  memset(&pa, 0, sizeof(pa));
  for (int i = 0; i < a.n; ++i) {
    cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.rows};
    cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
    cuuint32_t box[2] = {kKc, kRows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&pa.tmap[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.blocks[i]),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // park the query parts in the last 48 rows (of D) of the output buffer
  __nv_bfloat16 *parts = static_cast<__nv_bfloat16 *>(a.out) + ((size_t)a.S * a.rows - kNQ) * a.D;
  {
    const int64_t total = (int64_t)kMaxS * a.D;
    const int blocks = (int)((total + 255) / 256 < 4 * sm_count() ? (total + 255) / 256 : 4 * sm_count());
    if (cudaError_t le = launch_dependent(p1_qsplit_kernel, dim3((unsigned)(blocks)), dim3(256), 0, a.stream,
                                          a.queries, a.gains, a.S, a.D, parts); le != cudaSuccess)
      return le;
    cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)kNQ};
    cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
    cuuint32_t box[2] = {kKc, kNQ};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&pa.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, parts, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  pa.out = a.out;
  pa.out_max = a.out_max;
  pa.out_lse = a.out_lse;
  pa.rows = a.rows;
  pa.n = a.n;
  pa.S = a.S;
  pa.D = a.D;
  pa.eps = a.eps;
  pa.inv_D = 1.f / (float)a.D;
  pa.kparts = 1;
  pa.chunk = kMaxN;
  pa.wait_limit = wait_limit_cycles();
  cudaError_t e = cudaSuccess;
  const int64_t tiles = (a.rows + kRows - 1) / kRows;
  const size_t row_bytes = (size_t)a.D * 2;
  const int kparts = split_parts(a);
  if (kparts > 1) {
    // Split mode: items (tile, one summary, 1/kparts of the features) fill
    // the GPU where (tile, five summaries) would leave it idle; partials in
    // o[1], then their sum and softmax, then the outputs kernel below.
    constexpr int kCh = 1;
    float *raw = reinterpret_cast<float *>(static_cast<char *>(a.out) + (size_t)a.rows * row_bytes);  // o[1]
    pa.raw = raw;
    pa.raw_n = a.n;
    pa.raw_off = 0;
    pa.raw_stride = (int64_t)(row_bytes / 4);
    pa.kparts = kparts;
    pa.chunk = kCh;
    e = cudaFuncSetAttribute(p1_scores_kernel<kMaxN, kCh>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_a(kCh));
    if (e != cudaSuccess) return e;
    const int64_t items = tiles * a.n * kparts;
    const int64_t slots = 2 * (int64_t)sm_count();
    const int64_t waves = (items + slots - 1) / slots;
    const int64_t ga = (items + waves - 1) / waves;
    if (cudaError_t le = launch_dependent((p1_scores_kernel<kMaxN, kCh>), dim3((unsigned)(ga)), dim3(kThreadsA),
                                          smem_a(kCh), a.stream, pa); le != cudaSuccess)
      return le;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t blocks = a.rows < 8 * (int64_t)sm_count() ? a.rows : 8 * (int64_t)sm_count();
    e = launch_dependent(p1_split_softmax_kernel, dim3((unsigned)blocks), dim3(kSplitThreads), 0, a.stream,
                         (const float *)raw, static_cast<float *>(a.out), (int64_t)(row_bytes / 4), a.rows, a.n, a.S,
                         kparts, pa.inv_D, a.eps, a.out_max, a.out_lse);
    if (e != cudaSuccess) return e;
  } else
  // Raw scores with five-summary items, two CTAs per SM (tensor-map loads
  // are served one box at a time per CTA), when each token's o[1] row can
  // hold its raw scores and lies before the parked query parts; then a
  // softmax kernel writes alpha into o[0].  Otherwise the fused kernel: one
  // CTA per SM, the softmax in its epilogue.
  if (a.S >= 3 && (int64_t)(a.S - 2) * a.rows >= kNQ && (size_t)a.n * a.S * 4 <= row_bytes) {
    constexpr int kCh = 5;
    float *raw = reinterpret_cast<float *>(static_cast<char *>(a.out) + (size_t)a.rows * row_bytes);  // o[1]
    pa.chunk = many_chunk(tiles, a.n, kCh);
    pa.raw = raw;
    pa.raw_n = a.n;
    pa.raw_off = 0;
    pa.raw_stride = (int64_t)(row_bytes / 4);
    e = cudaFuncSetAttribute(p1_scores_kernel<kMaxN, kCh>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_a(kCh));
    if (e != cudaSuccess) return e;
    const int64_t items = tiles * ((a.n + pa.chunk - 1) / pa.chunk);
    const int64_t slots = 2 * (int64_t)sm_count();
    const int64_t waves = (items + slots - 1) / slots;
    const int64_t ga = (items + waves - 1) / waves;
    if (cudaError_t le = launch_dependent((p1_scores_kernel<kMaxN, kCh>), dim3((unsigned)(ga)), dim3(kThreadsA),
                                          smem_a(kCh), a.stream, pa); le != cudaSuccess)
      return le;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int64_t total = a.rows * (a.S + (a.S & 1));
    const int64_t blocks = (total + 255) / 256 < 8 * sm_count() ? (total + 255) / 256 : 8 * sm_count();
    e = launch_dependent(p1_park_softmax_kernel, dim3((unsigned)blocks), dim3(256), 0, a.stream, (const float *)raw,
                         static_cast<float *>(a.out), (int64_t)(row_bytes / 4), a.rows, a.n, a.S, a.out_max,
                         a.out_lse);
    if (e != cudaSuccess) return e;
  } else {
    e = cudaFuncSetAttribute(p1_scores_kernel<kMaxN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemA);
    if (e != cudaSuccess) return e;
    // Every CTA gets the same number of tiles (no partly empty last wave).
    const int64_t waves = (tiles + sm_count() - 1) / sm_count();
    const int64_t ga = (tiles + waves - 1) / waves;
    if (cudaError_t le = launch_dependent(p1_scores_kernel<kMaxN>, dim3((unsigned)(ga)), dim3(kThreadsA), kSmemA,
                                          a.stream, pa); le != cudaSuccess)
      return le;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Kernel B
  ParamsB pb;
  for (int i = 0; i < a.n; ++i) pb.src[i] = a.blocks[i];
  pb.out = a.out;
  pb.rows = a.rows;
  pb.n = a.n;
  pb.S = a.S;
  pb.D = a.D;
  pb.nvec = a.D / 8;
  pb.parts = a.D > 4096 ? 2 : 1;
  pb.nvp = pb.nvec / pb.parts;
  const int threads = (pb.nvp + 31) / 32 * 32;
  const size_t smem = smem_b(a.n, a.D / pb.parts);
  // The two-phase Block shape of the pages (9 summaries, 24 queries) has
  // its instantiation with both built in.
  const bool built = a.n == 9 && a.S == 24;
  auto kern = pb.parts == 2 ? (built ? p1_outputs_kernel<2, 9, 24> : p1_outputs_kernel<2, 0, 0>)
                            : (built ? p1_outputs_kernel<1, 9, 24> : p1_outputs_kernel<1, 0, 0>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t cap = (int64_t)occ * sm_count();
  const int64_t gb = a.rows < cap ? a.rows : cap;
  return launch_dependent(kern, dim3((unsigned)gb), dim3(threads), smem, a.stream, pb);
}

bool phase1_many_supported(int n, int D, int dtype, int S, int64_t rows) {
  if (dtype != ATTNRES_BF16 || n < 1 || n > kMaxSources || S < 1 || S > tc::kMaxS) return false;
  if (D % tc::kKc != 0 || D / 4 > 512) return false;           // the outputs kernel: 4 features per thread
  if ((int64_t)S * rows < tc::kNQ) return false;               // room to park the query parts
  if ((size_t)n * (S + (S & 1)) * 8 > 200 * 1024) return false;  // the token's alpha in shared memory
  return tc::encode_fn() != nullptr;
}

cudaError_t launch_phase1_many(const Phase1ManyArgs &a) {
  using namespace tc;
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  // the query parts, parked in the last 48 rows (of D) of the output buffer
  __nv_bfloat16 *parts = static_cast<__nv_bfloat16 *>(a.out) + ((size_t)a.S * a.rows - kNQ) * a.D;
  {
    const int64_t total = (int64_t)kMaxS * a.D;
    const int blocks = (int)((total + 255) / 256 < 4 * sm_count() ? (total + 255) / 256 : 4 * sm_count());
    if (cudaError_t le = launch_dependent(p1_qsplit_kernel, dim3((unsigned)(blocks)), dim3(256), 0, a.stream,
                                          a.queries, a.gains, a.S, a.D, parts); le != cudaSuccess)
      return le;
    cudaError_t e0 = cudaGetLastError();
    if (e0 != cudaSuccess) return e0;
  }
  ParamsAMany pa;
  memset(&pa, 0, sizeof(pa));
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)kNQ};
    cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
    cuuint32_t box[2] = {kKc, kNQ};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&pa.qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, parts, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  pa.out = a.out;
  pa.rows = a.rows;
  pa.S = a.S;
  pa.D = a.D;
  pa.eps = a.eps;
  pa.inv_D = 1.f / (float)a.D;
  pa.raw = a.scores;
  pa.raw_n = a.n;
  pa.raw_stride = (int64_t)a.n * a.S;
  pa.kparts = 1;
  pa.wait_limit = wait_limit_cycles();
  constexpr int kManyCh = 5;   // at most five summaries per work item: two CTAs per SM
  cudaError_t e = cudaFuncSetAttribute(p1_scores_kernel<kManyMaps, kManyCh>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_a(kManyCh));
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.rows + kRows - 1) / kRows;
  // Raw scores: one launch per kManyMaps summaries, its work items (tile,
  // chunk of five) spread evenly over the SMs.
  for (int off = 0; off < a.n; off += kManyMaps) {
    const int nl = a.n - off < kManyMaps ? a.n - off : kManyMaps;
    for (int i = 0; i < nl; ++i) {
      cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.rows};
      cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
      cuuint32_t box[2] = {kKc, kRows};
      cuuint32_t estr[2] = {1, 1};
      CUresult r = encode(&pa.tmap[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.blocks[off + i]),
                          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    pa.n = nl;
    pa.raw_off = off;
    const int64_t slots = 2 * (int64_t)sm_count();   // resident CTAs
    pa.chunk = many_chunk(tiles, nl, kManyCh);
    const int64_t items = tiles * ((nl + pa.chunk - 1) / pa.chunk);
    const int64_t waves = (items + slots - 1) / slots;
    const int64_t ga = (items + waves - 1) / waves;
    if (cudaError_t le = launch_dependent((p1_scores_kernel<kManyMaps, kManyCh>), dim3((unsigned)(ga)),
                                          dim3(kThreadsA), smem_a(kManyCh), a.stream, pa); le != cudaSuccess)
      return le;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const int64_t total = a.rows * a.S;
    const int64_t blocks = (total + 255) / 256 < 8 * sm_count() ? (total + 255) / 256 : 8 * sm_count();
    if (cudaError_t le = launch_dependent(p1_many_softmax_kernel, dim3((unsigned)(blocks)), dim3(256), 0, a.stream,
                                          a.scores, a.rows, a.n, a.S, a.out_max, a.out_lse); le != cudaSuccess)
      return le;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // Two CTAs share an SM, each taking a piece of 1024 features of a token
  // with 8 warps: per-thread row copies stream at a limited rate per CTA, so
  // two CTAs per SM keep more copies in flight (the Full two-phase schedule
  // at D = 2048: 8.8 -> 8.57 ms; pieces of 512 on 4-warp CTAs, three per SM,
  // measured 8.80 ms).  A ring of three slots, with alpha in one buffer,
  // keeps two steps in flight through each step's MMAs and still fits two
  // CTAs (8.58 -> 8.40 ms); two slots where it does not.  Otherwise one CTA
  // of 16 warps takes the whole row.
  for (int warps : {8}) {
    const int DF = 8 * warps * 16;                // features per piece: 16 n-tiles per warp
    if (a.S > kTcK || a.D % DF != 0 || a.D / DF < 2) continue;
    int occ = 0, ns = 3;
    size_t smem3 = 0;
    auto kern = p1_many_outputs_tc_kernel<8, 3>;
    for (; ns >= 2; --ns) {
      kern = ns == 3 ? p1_many_outputs_tc_kernel<8, 3> : p1_many_outputs_tc_kernel<8, 2>;
      smem3 = tc_smem(a.n, DF, ns);
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3);
      if (e != cudaSuccess) return e;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, warps * 32, smem3);
      if (e != cudaSuccess) return e;
      if (occ >= 2) break;
    }
    if (occ < 2) continue;
    ParamsB3 pc;
    for (int i = 0; i < a.n; ++i) pc.src[i] = a.blocks[i];
    pc.alpha = a.scores;
    pc.out = a.out;
    pc.rows = a.rows;
    pc.n = a.n;
    pc.S = a.S;
    pc.D = a.D;
    pc.parts = a.D / DF;
    const int64_t items = a.rows * pc.parts, cap = (int64_t)occ * sm_count();
    const int64_t g3 = items < cap ? items : cap;
    if (cudaError_t le = launch_dependent(kern, dim3((unsigned)(g3)), dim3(warps * 32), smem3, a.stream, pc);
        le != cudaSuccess)
      return le;
    return cudaGetLastError();
  }
  if (a.S <= kTcK && a.D % (8 * kTcWarps * 2) == 0 && a.D <= 8 * kTcWarps * 16 &&
      tc_smem(a.n, a.D) <= 227 * 1024) {
    ParamsB3 pc;
    for (int i = 0; i < a.n; ++i) pc.src[i] = a.blocks[i];
    pc.alpha = a.scores;
    pc.out = a.out;
    pc.rows = a.rows;
    pc.n = a.n;
    pc.S = a.S;
    pc.D = a.D;
    pc.parts = 1;
    const size_t smem3 = tc_smem(a.n, a.D);
    e = cudaFuncSetAttribute(p1_many_outputs_tc_kernel<kTcWarps>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem3);
    if (e != cudaSuccess) return e;
    const int64_t g3 = a.rows < sm_count() ? a.rows : sm_count();
    if (cudaError_t le = launch_dependent(p1_many_outputs_tc_kernel<kTcWarps>, dim3((unsigned)(g3)),
                                          dim3(kTcWarps * 32), smem3, a.stream, pc); le != cudaSuccess)
      return le;
    return cudaGetLastError();
  }
  ParamsB2 pb;
  for (int i = 0; i < a.n; ++i) pb.src[i] = a.blocks[i];
  pb.alpha = a.scores;
  pb.out = a.out;
  pb.rows = a.rows;
  pb.n = a.n;
  pb.S = a.S;
  pb.D = a.D;
  const int threads = (a.D / 4 + 31) / 32 * 32;
  const size_t smem = (size_t)a.n * (a.S + (a.S & 1)) * 8;
  e = cudaFuncSetAttribute(p1_many_outputs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, p1_many_outputs_kernel, threads, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) occ = 1;
  const int64_t cap = (int64_t)occ * sm_count();
  const int64_t gb = a.rows < cap ? a.rows : cap;
  if (cudaError_t le = launch_dependent(p1_many_outputs_kernel, dim3((unsigned)(gb)), dim3(threads), smem,
                                        a.stream, pb); le != cudaSuccess)
    return le;
  return cudaGetLastError();
}

}  // namespace attnres
