// phase1_tc.cu -- phase 1 of the two-phase Block scheme on the 5th-generation
// tensor cores ("Attention Residual 深度残差", "两阶段算法（inter / intra）",
// inter step / attn_with_stats; eq. A1-A3 for S queries at once).
//
// Per token, phase 1 is two contractions over the n completed block
// summaries v_i: the S x n scores s_{q,i} = w~_q . v_i / rms(v_i) (a dense
// contraction over D with the queries shared by every token) and the S
// outputs o_q = sum_i alpha_{q,i} v_i.  The scores run on tcgen05.mma; the
// outputs (n = 9 terms per element) run as packed fp32x2 FMAs.
//
// Work split.  A thread-block cluster of CL = D / 512 CTAs owns a tile of 8
// tokens; CTA c owns the feature slice [512 c, 512 c + 512).
//   * Its slice of the folded queries w~ = w (.) gamma stays in shared memory
//     for the whole kernel, as bf16 hi + lo parts (w~ ~= hi + lo to ~16 bits),
//     K-major with the 128-byte swizzle: the MMA's B operand (N = 2S rows).
//   * The tile's summary rows arrive by TMA (box 64 features x 8 tokens,
//     128-byte swizzle) into a double-buffered stage laid out as the MMA's A
//     operand: M = 128 rows = (source i, token t) pairs, 72 of them used.
//   * tcgen05.mma accumulates the partial scores over the slice in TMEM
//     (128 lanes x 2S fp32 columns); three epilogue warps read them back,
//     add hi + lo, and compute each row's partial sum of squares from the
//     staged tile.
//   * The partial scores and sums of squares of all CL CTAs are combined
//     through distributed shared memory: every CTA pushes (remote stores)
//     its partials of token t into the inbox of CTA t % CL, which reduces
//     them locally, takes the softmax over the n summaries, writes m and
//     lse, and stores alpha into every CTA of the cluster.
//   * Eight output warps (one token each) form o_q for the CTA's slice from
//     the staged tile and alpha, and store it.
// Every summary byte is read from HBM once; the queries never leave the SM.
//
// Synchronisation is by mbarriers only (TMA completion, MMA completion,
// buffer release, cluster-wide "partials ready" / "alpha ready" with remote
// arrivals).  Every wait is bounded; one that runs out records a flag and
// the kernel runs to its end.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

ATTNRES_DEFINE_ERROR_FLAG(take_error_phase1_tc)

namespace attnres {
namespace tc {

constexpr int kTile = 8;            // tokens per tile (rows of one swizzle atom)
constexpr int kDc = 512;            // feature slice per CTA
constexpr int kKB = kDc / 64;       // 64-feature K-atoms per slice
constexpr int kMaxN = 9;            // summaries (72 of the 128 MMA rows)
constexpr int kMaxS = 24;           // queries (2S <= 48 B-operand rows)
constexpr int kPs = kMaxS + 1;      // floats per inbox row: S partial scores + sum of squares
constexpr int kAl = 12;             // floats per (token, query) alpha row
constexpr int kWarps = 13;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiWarp0 = 4;        // warps 4, 5, 6 read TMEM lanes 0-95
constexpr int kNQ = 2 * kMaxS;      // B rows: hi parts at 0..S-1, lo parts at 24..24+S-1
constexpr int kTmemCols = 128;      // two accumulators of kNQ (<= 64) columns

struct Params {
  CUtensorMap tmap[kMaxN];          // one per summary: [rows, D] bf16, box 64 x 8
  const float *q;                   // [S, D]
  const float *g;                   // [S, D] or nullptr
  void *out;                        // [S, rows, D] bf16
  float *out_max;                   // [S, rows] or nullptr
  float *out_lse;                   // [S, rows]
  int64_t rows;
  int n, S, D, CL;
  float eps, inv_D;
  uint32_t off_v1, off_q, off_ps, off_al, off_bar, vbytes;
};

// --- small PTX wrappers ------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void arrive_remote(uint32_t addr_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(addr_cluster) : "memory");
}
__device__ __forceinline__ bool try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}
// After any wait in the process has run out, every later wait gives up at
// once, so a broken run ends quickly instead of spending the limit per wait.
__device__ __forceinline__ bool aborted() {
  return *reinterpret_cast<volatile unsigned int *>(&g_error_flag) != 0;
}
// Wait with cluster-scope acquire (the phase was completed by remote arrivals).
__device__ __forceinline__ void wait_cluster(uint32_t bar, uint32_t parity) {
  if (try_cluster(bar, parity)) return;
  const unsigned long long t0 = globaltimer_ns();
  while (!try_cluster(bar, parity)) {
    if (aborted()) return;
    if (globaltimer_ns() - t0 > kWaitLimitNs) { raise_timeout(); return; }
  }
}
__device__ __forceinline__ void wait_local(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return;
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try(bar, parity)) {
    if (aborted()) return;
    if (globaltimer_ns() - t0 > kWaitLimitNs) { raise_timeout(); return; }
  }
}
__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_dsmem(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void fence_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 96;" ::: "memory"); }

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// `sbo` bytes apart (the leading offset is unused for this layout).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused): 16 B
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;                         // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
      :: "r"(tmem_d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               :: "r"(bar) : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Packed fp32 pair helpers (fma.rn.f32x2).
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void fma2(uint64_t &acc, uint64_t a, uint64_t x) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(x));
}

// Byte offset of 16-byte chunk `j` of row `r` inside a 1024-byte, 8-row atom
// written by TMA (or by hand) with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t j) { return r * 128u + ((j ^ (r & 7u)) << 4); }

// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1) phase1_tc_kernel(const __grid_constant__ Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const uint32_t base = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t cta = cluster_rank();
  const int n = p.n, S = p.S, CL = p.CL;
  const uint32_t vbytes = p.vbytes;                    // one stage: n * kKB atoms of 1 KB

  // barriers
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + p.off_bar);
  const uint32_t b0 = base + p.off_bar;
  auto FULL = [&](int b) { return b0 + 8u * (0 + b); };
  auto VFREE = [&](int b) { return b0 + 8u * (2 + b); };
  auto MMADONE = [&](int b) { return b0 + 8u * (4 + b); };
  auto TFREE = [&](int b) { return b0 + 8u * (6 + b); };
  const uint32_t PREADY = b0 + 8u * 8;
  auto AREADY = [&](int b) { return b0 + 8u * (9 + b); };
  auto OUTDONE = [&](int b) { return b0 + 8u * (11 + b); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 13);

  float *ps = reinterpret_cast<float *>(sm + p.off_ps);    // inbox [CL][8/CL][n][kPs]
  float *al = reinterpret_cast<float *>(sm + p.off_al);    // [2][8][S][kAl] alpha

  if (threadIdx.x == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(FULL(b), 1);
      mbar_init(VFREE(b), 8 + 3);
      mbar_init(MMADONE(b), 1);
      mbar_init(TFREE(b), 3);
      mbar_init(AREADY(b), CL);
      mbar_init(OUTDONE(b), 8);
    }
    mbar_init(PREADY, CL);
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }

  // Folded query slice, bf16 hi / lo, as the B operand: row q holds the hi
  // part of query q, row kMaxS + q its lo part, unused rows are zero; K-atom
  // kb of all kNQ rows is contiguous (8-row groups 1 KB apart).
  {
    const int gq = kNQ / 8;
    const int chunks = kNQ * (kDc / 8);
    for (int c = threadIdx.x; c < chunks; c += kThreads) {
      const int row = c / (kDc / 8), ch = c % (kDc / 8);
      const int q = row < kMaxS ? row : row - kMaxS;
      float v[8];
      if (q < S) {
        const int d = (int)cta * kDc + ch * 8;
        const float4 w0 = ld_f4(p.q + (size_t)q * p.D + d), w1 = ld_f4(p.q + (size_t)q * p.D + d + 4);
        float4 g0 = make_float4(1.f, 1.f, 1.f, 1.f), g1 = g0;
        if (p.g) { g0 = ld_f4(p.g + (size_t)q * p.D + d); g1 = ld_f4(p.g + (size_t)q * p.D + d + 4); }
        const float qe[8] = {w0.x * g0.x, w0.y * g0.y, w0.z * g0.z, w0.w * g0.w,
                             w1.x * g1.x, w1.y * g1.y, w1.z * g1.z, w1.w * g1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float hi = __bfloat162float(__float2bfloat16_rn(qe[e]));
          v[e] = row < kMaxS ? hi : qe[e] - hi;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
      }
      const int kb = ch >> 3, j = ch & 7;
      const uint32_t off = p.off_q + (uint32_t)(kb * gq + (row >> 3)) * 1024u + swz(row & 7, j);
      *reinterpret_cast<uint4 *>(sm + off) = Elt<__nv_bfloat16>::pack(v);
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> tensor core
  cluster_sync_all();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem_base = *tmem_slot;

  const int64_t tiles = (p.rows + kTile - 1) / kTile;
  const int64_t cid = cluster_id(), ncl = cluster_count();
  const int64_t my_tiles = tiles > cid ? (tiles - cid + ncl - 1) / ncl : 0;
  const uint32_t idesc = idesc_bf16(128, kNQ);

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      for (int64_t j = 0; j < my_tiles; ++j) {
        const int b = (int)(j & 1);
        const int64_t tile = cid + j * ncl;
        if (j >= 2) wait_local(VFREE(b), (uint32_t)(((j - 2) >> 1) & 1));
        mbar_expect_tx(FULL(b), vbytes);
        const uint32_t vb = base + (b ? p.off_v1 : 0u);
        for (int kb = 0; kb < kKB; ++kb)
          for (int i = 0; i < n; ++i)
            tma_load_2d(vb + (uint32_t)(kb * n + i) * 1024u, &p.tmap[i], (int)cta * kDc + kb * 64,
                        (int)(tile * kTile), FULL(b));
      }
      // drain: the last stages this CTA filled have landed before it may exit
      for (int64_t j = my_tiles - 2 < 0 ? 0 : my_tiles - 2; j < my_tiles; ++j)
        wait_local(FULL((int)(j & 1)), (uint32_t)((j >> 1) & 1));
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      for (int64_t j = 0; j < my_tiles; ++j) {
        const int b = (int)(j & 1);
        wait_local(FULL(b), (uint32_t)((j >> 1) & 1));
        if (j >= 2) wait_local(TFREE(b), (uint32_t)(((j - 2) >> 1) & 1));
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t vb = base + (b ? p.off_v1 : 0u);
        const uint32_t qb = base + p.off_q;
        const uint32_t gq = (uint32_t)(kNQ / 8);
        for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = sw128_desc(vb + (uint32_t)(kb * n) * 1024u + kk * 32u, 1024u);
            const uint64_t bq = sw128_desc(qb + (uint32_t)kb * gq * 1024u + kk * 32u, 1024u);
            mma_bf16(tmem_base + (uint32_t)b * 64u, a, bq, idesc, (kb | kk) != 0);
          }
        }
        mma_commit(MMADONE(b));
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 3) {
    // ---------------- epilogue: scores, sums of squares, cluster reduce ----------------
    const int e = threadIdx.x - kEpiWarp0 * 32;          // 0..95 = TMEM lane = MMA row
    const int r = e, src = r >> 3, tok = r & 7;
    const bool live = r < 8 * n;
    for (int64_t j = 0; j < my_tiles; ++j) {
      const int b = (int)(j & 1);
      const uint32_t ph = (uint32_t)((j >> 1) & 1);
      const int64_t tile = cid + j * ncl;
      wait_local(FULL(b), ph);
      wait_local(MMADONE(b), ph);
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      float acc[48];
      const uint32_t taddr = tmem_base + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)b * 64u;
      tmem_ld16(taddr, acc);
      tmem_ld16(taddr + 16, acc + 16);
      tmem_ld16(taddr + 32, acc + 32);
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(TFREE(b));
      // partial sum of squares of row (src, tok) over this CTA's slice
      float sq = 0.f;
      if (live) {
        const unsigned char *vrow = sm + (b ? p.off_v1 : 0u) + src * 1024;
        for (int kb = 0; kb < kKB; ++kb) {
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            float x[8];
            Elt<__nv_bfloat16>::unpack(
                *reinterpret_cast<const uint4 *>(vrow + kb * n * 1024 + swz(tok, jj)), x);
#pragma unroll
            for (int q = 0; q < 8; ++q) sq = fmaf(x[q], x[q], sq);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(VFREE(b));
      // every CTA has finished reading this CTA's previous partials, and every
      // CTA's output warps are done with the alpha slot about to be refilled
      if (j >= 1) wait_cluster(AREADY((int)((j - 1) & 1)), (uint32_t)(((j - 1) >> 1) & 1));
      if (j >= 2) wait_local(OUTDONE(b), (uint32_t)(((j - 2) >> 1) & 1));
      // Push this row's partial scores and sum of squares into the inbox of
      // the CTA that reduces token `tok` (tok % CL): slot [this CTA][tok / CL][src].
      if (live) {
        const int owner = tok % CL, u = tok / CL;
        const uint32_t dst = map_rank(base + p.off_ps +
                                      (uint32_t)((((int)cta * (kTile / CL) + u) * n + src) * kPs) * 4u,
                                      (uint32_t)owner);
#pragma unroll
        for (int q = 0; q < kMaxS; ++q)
          if (q < S) st_dsmem(dst + 4u * q, acc[q] + acc[kMaxS + q]);
        st_dsmem(dst + 4u * kMaxS, sq);
      }
      fence_cluster();
      epi_bar();
      if (e == 0)
        for (int k = 0; k < CL; ++k) arrive_remote(map_rank(PREADY, (uint32_t)k));
      wait_cluster(PREADY, (uint32_t)(j & 1));
      // reduce the tokens t == cta (mod CL) from the local inbox: scores,
      // softmax, alpha, m, lse
      const int per = kTile / CL;
      for (int pr = e; pr < per * S; pr += 96) {
        const int u = pr / S, q = pr % S;
        const int t = (int)cta + CL * u;
        float sc[kMaxN];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kMaxN; ++i) {
          sc[i] = -INFINITY;
          if (i < n) {
            float dot = 0.f, sq2 = 0.f;
            for (int k = 0; k < CL; ++k) {
              const float *slot = ps + ((k * per + u) * n + i) * kPs;
              dot += slot[q];
              sq2 += slot[kMaxS];
            }
            sc[i] = dot * rsqrtf(fmaf(sq2, p.inv_D, p.eps));
            m = fmaxf(m, sc[i]);
          }
        }
        float den = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxN; ++i) {
          sc[i] = i < n ? expf(sc[i] - m) : 0.f;
          den += sc[i];
        }
        const float inv = 1.f / den;
        const uint32_t aoff = p.off_al + (uint32_t)(((b * kTile + t) * S + q) * kAl) * 4u;
        for (int k = 0; k < CL; ++k) {
          const uint32_t ra = map_rank(base + aoff, (uint32_t)k);
#pragma unroll
          for (int i = 0; i < kMaxN; ++i)
            if (i < n) st_dsmem(ra + 4u * i, sc[i] * inv);
        }
        const int64_t row = tile * kTile + t;
        if (row < p.rows) {
          p.out_lse[(size_t)q * p.rows + row] = m + logf(den);
          if (p.out_max) p.out_max[(size_t)q * p.rows + row] = m;
        }
      }
      fence_cluster();
      epi_bar();
      if (e == 0)
        for (int k = 0; k < CL; ++k) arrive_remote(map_rank(AREADY(b), (uint32_t)k));
    }
  } else {
    // ---------------- output warps: o_q = sum_i alpha_qi v_i for one token ----------------
    const int ow = warp < kEpiWarp0 ? warp - 2 : warp - (kEpiWarp0 + 3) + 2;   // 0..7
    const int t = ow;
    for (int64_t j = 0; j < my_tiles; ++j) {
      const int b = (int)(j & 1);
      const uint32_t ph = (uint32_t)((j >> 1) & 1);
      const int64_t tile = cid + j * ncl;
      const int64_t row = tile * kTile + t;
      wait_local(FULL(b), ph);
      wait_cluster(AREADY(b), ph);
      if (row < p.rows) {
        const unsigned char *vb = sm + (b ? p.off_v1 : 0u);
        const float *arow = al + (size_t)((b * kTile + t) * S) * kAl;
#pragma unroll 1
        for (int it = 0; it < 2; ++it) {
          const int ch = lane + 32 * it;                 // 16-byte chunk of the slice
          const int kb = ch >> 3, jj = ch & 7;
          uint64_t x[kMaxN][4];
#pragma unroll
          for (int i = 0; i < kMaxN; ++i) {
            if (i < n) {
              const uint4 v = *reinterpret_cast<const uint4 *>(vb + (kb * n + i) * 1024 + swz(t, jj));
              float f[8];
              Elt<__nv_bfloat16>::unpack(v, f);
#pragma unroll
              for (int m2 = 0; m2 < 4; ++m2) x[i][m2] = pk(f[2 * m2], f[2 * m2 + 1]);
            }
          }
          char *dst = static_cast<char *>(p.out) +
                      ((size_t)row * p.D + (size_t)cta * kDc + (size_t)ch * 8) * 2;
          const size_t qstride = (size_t)p.rows * p.D * 2;
#pragma unroll 2
          for (int q = 0; q < S; ++q) {
            const float4 a0 = *reinterpret_cast<const float4 *>(arow + q * kAl);
            const float4 a1 = *reinterpret_cast<const float4 *>(arow + q * kAl + 4);
            const float a2 = arow[q * kAl + 8];
            const float av[kMaxN] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w, a2};
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int i = 0; i < kMaxN; ++i) {
              if (i < n) {
                const uint64_t ai = pk(av[i], av[i]);
#pragma unroll
                for (int m2 = 0; m2 < 4; ++m2) fma2(acc[m2], ai, x[i][m2]);
              }
            }
            float h[8];
#pragma unroll
            for (int m2 = 0; m2 < 4; ++m2) upk(acc[m2], h[2 * m2], h[2 * m2 + 1]);
            st_stream(dst + (size_t)q * qstride, Elt<__nv_bfloat16>::pack(h));
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(VFREE(b));
        mbar_arrive(OUTDONE(b));
      }
    }
  }

  __syncwarp();
  cluster_sync_all();   // no CTA leaves while a peer may still touch its shared memory
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem_base), "r"(kTmemCols));
  }
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

struct Layout {
  uint32_t off_v1, off_q, off_ps, off_al, off_bar, vbytes, total;
};

Layout layout(int n, int S) {
  Layout L;
  const int NQ = kNQ;
  L.vbytes = (uint32_t)(n * kKB * 1024);
  L.off_v1 = L.vbytes;
  L.off_q = 2 * L.vbytes;
  L.off_ps = L.off_q + (uint32_t)(kKB * NQ * 128);
  L.off_al = L.off_ps + (uint32_t)(kTile * kMaxN * kPs * 4);   // inbox: 8 tokens x n rows
  L.off_bar = L.off_al + (uint32_t)(2 * kTile * S * kAl * 4);
  L.off_bar = (L.off_bar + 15) & ~15u;
  // The MMA's A operand spans 128 rows (16 KB per K-atom); rows beyond the
  // n * 8 staged ones read whatever follows (their results are unused), so
  // keep at least 16 KB past the start of the last K-atom of stage 1.
  uint32_t need = L.off_bar + 14 * 8 + 16;
  const uint32_t a_reach = L.off_v1 + (uint32_t)((kKB - 1) * n * 1024) + 16 * 1024;
  if (need < a_reach) need = a_reach;
  L.total = need + 1024;   // alignment slack
  return L;
}

}  // namespace tc

bool phase1_tc_supported(int n, int D, int dtype, int S) {
  if (dtype != ATTNRES_BF16 || n < 1 || n > tc::kMaxN || S < 1 || S > tc::kMaxS) return false;
  if (D % tc::kDc != 0) return false;
  const int CL = D / tc::kDc;
  if (CL != 1 && CL != 2 && CL != 4 && CL != 8) return false;
  if (tc::layout(n, S).total > 227 * 1024) return false;
  return tc::encode_fn() != nullptr;
}

cudaError_t launch_phase1_tc(const Phase1Args &a) {
  using namespace tc;
  auto encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  Params p;
  memset(&p, 0, sizeof(p));
  for (int i = 0; i < a.n; ++i) {
    cuuint64_t dims[2] = {(cuuint64_t)a.D, (cuuint64_t)a.rows};
    cuuint64_t strides[1] = {(cuuint64_t)a.D * 2};
    cuuint32_t box[2] = {64, kTile};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(&p.tmap[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(a.blocks[i]),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  const Layout L = layout(a.n, a.S);
  p.q = a.queries;
  p.g = a.gains;
  p.out = a.out;
  p.out_max = a.out_max;
  p.out_lse = a.out_lse;
  p.rows = a.rows;
  p.n = a.n;
  p.S = a.S;
  p.D = a.D;
  p.CL = a.D / kDc;
  p.eps = a.eps;
  p.inv_D = 1.f / (float)a.D;
  p.off_v1 = L.off_v1;
  p.off_q = L.off_q;
  p.off_ps = L.off_ps;
  p.off_al = L.off_al;
  p.off_bar = L.off_bar;
  p.vbytes = L.vbytes;

  cudaError_t e = cudaFuncSetAttribute(phase1_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)L.total);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = a.stream;
  cfg.gridDim = dim3((unsigned)p.CL, 1, 1);
  int max_clusters = 0;
  e = cudaOccupancyMaxActiveClusters(&max_clusters, phase1_tc_kernel, &cfg);
  if (e != cudaSuccess) return e;
  if (max_clusters < 1) return cudaErrorInvalidConfiguration;
  const int64_t tiles = (a.rows + kTile - 1) / kTile;
  const int64_t ncl = tiles < max_clusters ? tiles : max_clusters;
  cfg.gridDim = dim3((unsigned)(ncl * p.CL), 1, 1);
  e = cudaLaunchKernelEx(&cfg, phase1_tc_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace attnres
