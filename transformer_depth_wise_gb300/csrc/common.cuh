// common.cuh -- device helpers shared by the AttnRes kernels (sm_103a).
//
// Rows move as 16-byte vectors (8 bf16 or 4 fp32 elements).  Arithmetic is
// fp32 throughout; a bf16 element widens to fp32 exactly by placing its 16
// bits in the high half of an fp32 word.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attnres.h"

namespace attnres {

constexpr int kMaxSources = ATTNRES_MAX_SOURCES;
constexpr int kMaxQueries = ATTNRES_MAX_QUERIES;

// Element traits: EPV = elements per 16-byte vector.
template <typename T> struct Elt;
template <> struct Elt<float> {
  static constexpr int EPV = 4;
  static __device__ __forceinline__ void unpack(const uint4 &v, float *x) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  static __device__ __forceinline__ uint4 pack(const float *x) {
    return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                      __float_as_uint(x[3]));
  }
  static __device__ __forceinline__ void unpack_again(const uint4 &v, float *x) { unpack(v, x); }
};
template <> struct Elt<__nv_bfloat16> {
  static constexpr int EPV = 8;
  static __device__ __forceinline__ void unpack_word(uint32_t w, float &lo, float &hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
  }
  static __device__ __forceinline__ void unpack(const uint4 &v, float *x) {
    unpack_word(v.x, x[0], x[1]); unpack_word(v.y, x[2], x[3]);
    unpack_word(v.z, x[4], x[5]); unpack_word(v.w, x[6], x[7]);
  }
  // Same, but re-derived at the point of use (the compiler may not keep an
  // earlier unpacked copy alive across a reduction: saves registers).
  static __device__ __forceinline__ void unpack_again(const uint4 &v, float *x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      asm volatile("shl.b32 %0, %2, 16;\n\tand.b32 %1, %2, 0xffff0000;" : "=r"(lo), "=r"(hi) : "r"(w[i]));
      x[2 * i] = __uint_as_float(lo);
      x[2 * i + 1] = __uint_as_float(hi);
    }
  }
  static __device__ __forceinline__ uint32_t pack_word(float lo, float hi) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest even
    return *reinterpret_cast<uint32_t *>(&b);
  }
  static __device__ __forceinline__ uint4 pack(const float *x) {
    return make_uint4(pack_word(x[0], x[1]), pack_word(x[2], x[3]), pack_word(x[4], x[5]),
                      pack_word(x[6], x[7]));
  }
};

// Streaming 16-byte load: read-only path, no L1 allocation (each source
// byte is consumed once by the CTA that loads it).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The same at a constant byte offset from `p`, folded into the instruction.
template <int OFF>
__device__ __forceinline__ uint4 ld_stream_at(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "n"(OFF));
  return v;
}

// L2 eviction policies (createpolicy, sm_80+) for loads and stores with an
// explicit cache hint: data read again soon is kept (evict_last), data used
// for the last time goes first (evict_first).
__device__ __forceinline__ uint64_t l2_policy_keep() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_drop() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte read-only load, no L1 allocation, with an L2 policy.
__device__ __forceinline__ uint4 ld_hint(const void *p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint4 ld_hint_at(const void *p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4+%5], %6;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "n"(OFF), "l"(policy));
  return v;
}
// 16-byte store with an L2 policy.
__device__ __forceinline__ void st_hint(void *p, const uint4 &v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy) : "memory");
}
// Vector k (0..3) of a thread's slice with an L2 policy (as ld_stream_vec).
template <int TPR>
__device__ __forceinline__ uint4 ld_hint_vec(const char *base, int k, int tpr, uint64_t policy) {
  if (TPR > 0) {
    switch (k) {
      case 0: return ld_hint_at<0>(base, policy);
      case 1: return ld_hint_at<TPR * 16>(base, policy);
      case 2: return ld_hint_at<TPR * 32>(base, policy);
      default: return ld_hint_at<TPR * 48>(base, policy);
    }
  }
  return ld_hint(base + (size_t)k * tpr * 16, policy);
}

// Vector k (0..3) of a thread's slice of a row: `base` points at the thread's
// first vector and the slice's vectors lie tpr * 16 bytes apart.  With the
// thread count TPR built in, the offset is folded into the load; in unrolled
// loops k is a constant and the switch disappears.
template <int TPR>
__device__ __forceinline__ uint4 ld_stream_vec(const char *base, int k, int tpr) {
  if (TPR > 0) {
    switch (k) {
      case 0: return ld_stream_at<0>(base);
      case 1: return ld_stream_at<TPR * 16>(base);
      case 2: return ld_stream_at<TPR * 32>(base);
      default: return ld_stream_at<TPR * 48>(base);
    }
  }
  return ld_stream(base + (size_t)k * tpr * 16);
}

// Plain 16-byte load through L1 (small, reused operands: queries, gains, u).
__device__ __forceinline__ float4 ld_f4(const float *p) {
  return __ldg(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ void st_vec(void *p, const uint4 &v) {
  *reinterpret_cast<uint4 *>(p) = v;
}

// Streaming store (evict-first): outputs are not re-read by this kernel.
__device__ __forceinline__ void st_stream(void *p, const uint4 &v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
               :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Sum over the TEAM lanes of an aligned power-of-two lane group of a warp.
template <int TEAM>
__device__ __forceinline__ float team_sum_shfl(float v) {
#pragma unroll
  for (int o = TEAM / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum of K values over a whole CTA.  Each warp reduces with shuffles, lane 0
// publishes to red[parity][warp][K], one barrier, then every thread sums the
// warps' values.  Alternating `parity` between consecutive calls makes a
// second barrier unnecessary (a slot is rewritten only after every thread
// has passed the barrier of the call in between).
template <int K>
__device__ __forceinline__ void cta_sum(float (&v)[K], float *red /*[2][32][K]*/, int parity) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = team_sum_shfl<32>(v[k]);
  float *slot = red + parity * 32 * K;
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) slot[warp * K + k] = v[k];
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < K; ++k) v[k] = 0.f;
  for (int w = 0; w < nwarps; ++w) {
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] += slot[w * K + k];
  }
}

// The synthetic sublayer's nonlinearity, 0.5 tanh(z), from the identity
// tanh z = 1 - 2 / (e^{2z} + 1):  0.5 tanh z = 0.5 - 1 / (e^{2z} + 1).
// One fast exponential and one fast reciprocal instead of a full-precision
// tanh: the absolute error stays near 1e-7 for every z (e^{2z} overflowing
// to infinity gives 0.5, underflowing to 0 gives -0.5), far below one bf16
// or the fp32 tolerance step of the stored partial it is added to.
__device__ __forceinline__ float half_tanh(float z) {
  return 0.5f - __fdividef(1.f, __expf(2.f * z) + 1.f);
}

// Ask L2 to fetch `bytes` (a multiple of 16) from a 16-byte aligned global
// address, without staging anything on the SM: one instruction per row.
__device__ __forceinline__ void prefetch_l2_bulk(const void *gmem, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gmem), "r"(bytes) : "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  A kernel launched with launch_dependent()
// is set up by the hardware while the kernel before it on the stream drains,
// and its first instruction, grid_dependency_wait(), returns once that grid
// has completed and its writes are visible; every kernel launched this way
// starts with it, so no access to another kernel's data comes earlier (the
// caller may have just written the query or gain on the same stream).  No
// kernel triggers its dependents early: CTAs launched into the few SMs an
// earlier grid has left idle crowded onto them, and measured on a GB300 the
// early trigger was slower everywhere (Full stack 26.9 -> 28.4 ms, its
// two-phase schedule 9.04 -> 9.96 ms, decode graph 188 -> 196 us).  For a
// kernel launched without the attribute the wait is a no-op.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kern` with programmatic stream serialization: its launch overlaps
// the end of the previous kernel on the stream (it must call
// grid_dependency_wait() before touching any data).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (one 64-bit register, fma.rn.f32x2 = two FMAs per
// instruction) and the element pairs of a 16-byte vector.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pair(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpair(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ float pair_sum(uint64_t v) {
  float lo, hi;
  unpair(v, lo, hi);
  return lo + hi;
}
__device__ __forceinline__ void fma_pair(uint64_t &acc, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
__device__ __forceinline__ void scale_pair(uint64_t &acc, uint64_t s) {
  asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc) : "l"(s), "l"(0ull));
}

template <typename T> struct Pairs;
template <> struct Pairs<float> {
  static constexpr int NP = 2;  // pairs per 16-byte vector
  static __device__ __forceinline__ void split(const uint4 &v, uint64_t *x) {
    x[0] = ((uint64_t)v.y << 32) | v.x;
    x[1] = ((uint64_t)v.w << 32) | v.z;
  }
};
template <> struct Pairs<__nv_bfloat16> {
  static constexpr int NP = 4;
  static __device__ __forceinline__ void split(const uint4 &v, uint64_t *x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = ((uint64_t)(w[i] & 0xffff0000u) << 32) | (uint64_t)(w[i] << 16);
  }
};

// Sum of K (a power of two, <= 32) values over a whole CTA, every thread
// getting all K totals.  Each warp reduce-scatters (butterflies down to K
// lanes' worth, then halving steps: lane l ends with the warp's total of
// value l % K, 31 shuffles for K = 32 and fewer for smaller K instead of
// 5 K), lanes < K publish to red[parity][warp][K], one barrier, each lane
// adds the warps' totals of its value, and K shuffles hand every total to
// every lane.  Alternating `parity` between calls saves a second barrier.
// MAXW: the most warps a CTA of the caller has ([2][MAXW][K] scratch).
template <int K, int MAXW = 32>
__device__ __forceinline__ void cta_sum_rs(float (&v)[K], float *red /*[2][MAXW][K]*/, int parity) {
  static_assert(K >= 1 && K <= 32 && (K & (K - 1)) == 0, "K: power of two <= 32");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  float b[K];
#pragma unroll
  for (int i = 0; i < K; ++i) b[i] = v[i];
#pragma unroll
  for (int o = 16; o >= K; o >>= 1) {  // plain butterflies over the lane bits no value is kept by
#pragma unroll
    for (int i = 0; i < K; ++i) b[i] += __shfl_xor_sync(0xffffffffu, b[i], o);
  }
#pragma unroll
  for (int o = K / 2; o > 0; o >>= 1) {  // halving: keep the upper or lower half
    const bool up = lane & o;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = up ? b[i] : b[i + o];
      const float keep = up ? b[i + o] : b[i];
      b[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  float *slot = red + parity * MAXW * K;
  if (lane < K) slot[warp * K + lane] = b[0];
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < nwarps; ++w) t += slot[w * K + (lane & (K - 1))];
#pragma unroll
  for (int i = 0; i < K; ++i) v[i] = __shfl_sync(0xffffffffu, t, i);
}

}  // namespace attnres

// ---------------------------------------------------------------------------
// mbarrier / bulk-copy helpers (sm_90+ PTX, used on sm_103a)
// ---------------------------------------------------------------------------
namespace attnres {

// Upper bound on any single wait inside a kernel, in SM clock cycles (about
// 2 s at 2 GHz).  A wait that runs out sets the translation unit's error flag
// and gives up instead of spinning forever.  The waits of a kernel's normal
// work take their limit from the launch (attnres_set_wait_limit can shorten
// it); the drain at a kernel's end, which waits for the CTA's own copies and
// tensor-core operations still in flight, always uses this one.
constexpr long long kDrainLimitCycles = 4000000000ll;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait for the phase of `parity` to complete, for at most `limit` SM clock
// cycles; false if the limit ran out (the caller then stops issuing work and
// drains what it has in flight).  try_wait itself parks the thread for a
// while, so the clock is read only between tries.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, long long limit) {
  if (mbar_try(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// 1-D bulk copy global -> shared (this CTA), completion counted on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

}  // namespace attnres

// Per translation unit: a device flag that records a wait that ran out, and
// a host function (declared in launch.h) that reads and clears it.
#define ATTNRES_DEFINE_ERROR_FLAG(host_fn)                                            \
  namespace attnres {                                                               \
  static __device__ unsigned int g_error_flag = 0;                                  \
  __device__ __forceinline__ void raise_timeout() { atomicOr(&g_error_flag, 1u); }  \
  unsigned int host_fn() {                                                          \
    unsigned int v = 0, zero = 0;                                                   \
    if (cudaMemcpyFromSymbol(&v, g_error_flag, sizeof(v)) != cudaSuccess) return 2; \
    if (v) cudaMemcpyToSymbol(g_error_flag, &zero, sizeof(zero));                   \
    return v;                                                                       \
  }                                                                                 \
  }
