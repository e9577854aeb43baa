// fnorm_device.cuh -- device-side building blocks shared by the libfnorm
// kernels: the Chan/Welford statistics triple and its merges, thread-block
// cluster and distributed-shared-memory primitives, 128-bit vector access for
// fp32/bf16, TMA bulk copies with mbarriers, and bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fnorm_internal.h"

namespace fnorm {

constexpr unsigned kFullMask = 0xffffffffu;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// ---------------------------------------------------------------------------
// Statistics triple and the pairwise (Chan et al.) combination.
//
// Page Kimi-K2.6__l2_p79, block 1, merges per-thread Welford states in a
// shared-memory tree with: n = na + nb, d = mean_b - mean_a,
// mean = mean_a + d*nb/n, M2 = M2a + M2b + d^2*na*nb/n, and notes that an
// empty partner (count 0) leaves the other unchanged. Page Kimi-K2.6__l1_p34,
// block 2, applies the same combination across warp shuffles. The counts are
// carried as floats (exact up to 2^24 per merged group).
// ---------------------------------------------------------------------------
struct Stat {
  float n;
  float mean;
  float m2;
};

__device__ __forceinline__ Stat stat_empty() { return Stat{0.f, 0.f, 0.f}; }

__device__ __forceinline__ Stat chan_merge(const Stat& a, const Stat& b) {
  if (b.n == 0.f) return a;
  if (a.n == 0.f) return b;
  const float n = a.n + b.n;
  const float fb = b.n / n;       // weight of b in the merged mean
  const float d = b.mean - a.mean;
  Stat r;
  r.n = n;
  r.mean = fmaf(d, fb, a.mean);
  r.m2 = a.m2 + b.m2 + d * d * (a.n * fb);   // d^2 * na*nb/n
  return r;
}

// Tree reduction over `width` consecutive lanes (a power of two <= 32). The
// result is valid in the first lane of each segment; the other lanes hold
// partial values. The tree shape is fixed, so results are reproducible.
template <int WIDTH>
__device__ __forceinline__ Stat warp_merge(Stat s) {
#pragma unroll
  for (int off = WIDTH / 2; off > 0; off >>= 1) {
    Stat o;
    o.n = __shfl_down_sync(kFullMask, s.n, off, WIDTH);
    o.mean = __shfl_down_sync(kFullMask, s.mean, off, WIDTH);
    o.m2 = __shfl_down_sync(kFullMask, s.m2, off, WIDTH);
    s = chan_merge(s, o);
  }
  return s;
}

// warp_merge for partials of equal count in every lane of the segment (slices
// that fill their threads' slots exactly): each step merges two partials of
// the same count, so the weight b.n/n is exactly 1/2 and the count need not
// travel. The arithmetic is chan_merge's with that weight (the same bits),
// without its division and zero checks.
template <int WIDTH>
__device__ __forceinline__ Stat warp_merge_eq(Stat s) {
#pragma unroll
  for (int off = WIDTH / 2; off > 0; off >>= 1) {
    const float om = __shfl_down_sync(kFullMask, s.mean, off, WIDTH);
    const float o2 = __shfl_down_sync(kFullMask, s.m2, off, WIDTH);
    const float d = om - s.mean;
    s.mean = fmaf(d, 0.5f, s.mean);
    s.m2 = s.m2 + o2 + d * d * (s.n * 0.5f);
    s.n = s.n + s.n;
  }
  return s;
}

// ---------------------------------------------------------------------------
// Element storage: a "slot" is one 16-byte vector of W = 16/sizeof(T)
// elements, kept in registers as a uint4 in the input type's encoding.
// ---------------------------------------------------------------------------
template <class T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int W = 4;
  __device__ static __forceinline__ float get(const uint4& v, int j) {
    const unsigned w = j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  __device__ static __forceinline__ float get_opaque(const uint4& v, int j) { return get(v, j); }
  __device__ static __forceinline__ void set(uint4& v, int j, float f) {
    const unsigned w = __float_as_uint(f);
    if (j == 0) v.x = w; else if (j == 1) v.y = w; else if (j == 2) v.z = w; else v.w = w;
  }
  __device__ static __forceinline__ float load1(const float* p) { return __ldg(p); }
  __device__ static __forceinline__ void store1(float* p, float f) { *p = f; }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int W = 8;
  __device__ static __forceinline__ float get(const uint4& v, int j) {
    const unsigned w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((j & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  // The same widening as an opaque one-instruction asm that the compiler
  // re-does at every use instead of keeping 8 widened values per slot live
  // across the passes (which doubles a slot's registers and spills in the
  // kernels that hold 8 slots per thread).
  __device__ static __forceinline__ float get_opaque(const uint4& v, int j) {
    const unsigned w = (j >> 1) == 0 ? v.x : (j >> 1) == 1 ? v.y : (j >> 1) == 2 ? v.z : v.w;
    unsigned r;
    if (j & 1)
      asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(r) : "r"(w));
    else
      asm volatile("shl.b32 %0, %1, 16;" : "=r"(r) : "r"(w));
    return __uint_as_float(r);
  }
  // (low / high value of the word w) - c in one instruction: the
  // mixed-precision subtraction (sub.rn.f32.bf16, PTX ISA) takes the bf16
  // operand from its half of the word; widening bf16 to fp32 is exact, so the
  // result is the fp32 subtraction's, rounded once (the same bits as
  // widening and subtracting). Used by the packed-pair forms, where it
  // replaces a widening and a paired addition.
  __device__ static __forceinline__ float diff_lo(unsigned w, float c) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tsub.rn.f32.bf16 %0, lo, %2;\n\t}"
        : "=f"(r) : "r"(w), "f"(c));
    return r;
  }
  __device__ static __forceinline__ float diff_hi(unsigned w, float c) {
    float r;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tsub.rn.f32.bf16 %0, hi, %2;\n\t}"
        : "=f"(r) : "r"(w), "f"(c));
    return r;
  }
  __device__ static __forceinline__ void set(uint4& v, int j, float f) {
    // f is a bf16 value widened to fp32 (exact), so its low 16 bits are zero
    const unsigned b = __float_as_uint(f) >> 16;
    unsigned* w = (j >> 1) == 0 ? &v.x : (j >> 1) == 1 ? &v.y : (j >> 1) == 2 ? &v.z : &v.w;
    *w = (j & 1) ? ((*w & 0x0000ffffu) | (b << 16)) : ((*w & 0xffff0000u) | b);
  }
  __device__ static __forceinline__ float load1(const __nv_bfloat16* p) {
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p));
    return __uint_as_float(static_cast<unsigned>(u) << 16);
  }
  __device__ static __forceinline__ void store1(__nv_bfloat16* p, float f) {
    *p = __float2bfloat16_rn(f);
  }
};

__device__ __forceinline__ uint4 ld_v4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
  *reinterpret_cast<uint4*>(p) = v;
}

// Store W fp32 results as Tout at p (16-byte aligned for the vector forms).
template <class Tout, int W>
struct VecStore;

template <>
struct VecStore<float, 4> {   // 16 bytes
  __device__ static __forceinline__ void run(float* p, const float (&o)[4]) {
    st_v4(p, make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                        __float_as_uint(o[3])));
  }
};
template <>
struct VecStore<float, 8> {   // 32 bytes: two 16-byte stores
  __device__ static __forceinline__ void run(float* p, const float (&o)[8]) {
    st_v4(p, make_uint4(__float_as_uint(o[0]), __float_as_uint(o[1]), __float_as_uint(o[2]),
                        __float_as_uint(o[3])));
    st_v4(p + 4, make_uint4(__float_as_uint(o[4]), __float_as_uint(o[5]), __float_as_uint(o[6]),
                            __float_as_uint(o[7])));
  }
};
__device__ __forceinline__ unsigned pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half)
  return *reinterpret_cast<const unsigned*>(&h);
}
template <>
struct VecStore<__nv_bfloat16, 8> {   // 16 bytes
  __device__ static __forceinline__ void run(__nv_bfloat16* p, const float (&o)[8]) {
    st_v4(p, make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                        pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7])));
  }
};
template <>
struct VecStore<__nv_bfloat16, 4> {   // 8 bytes
  __device__ static __forceinline__ void run(__nv_bfloat16* p, const float (&o)[4]) {
    *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]));
  }
};

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory (PTX ISA: special
// registers %cluster_ctarank etc., barrier.cluster, mapa, ld.shared::cluster).
// A kernel launched without a cluster dimension runs as 1-CTA clusters.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned cluster_ctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_nctarank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned cluster_id_x() {
  unsigned r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ unsigned ncluster_x() {
  unsigned r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
// All threads of all CTAs of the cluster; release/acquire orders the shared
// memory writes before the barrier with the remote reads after it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t local_addr, unsigned rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel is launched so that it may start
// while the previous kernel in the stream is finishing; before its first
// access to global memory a kernel waits until all prerequisite grids have
// completed and their writes are visible (griddepcontrol.wait), and near its
// end it lets the next launch begin (griddepcontrol.launch_dependents). Both
// are no-ops for a kernel launched without the attribute.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// mbarrier + TMA bulk copy (cp.async.bulk, non-tensor form: 16-byte aligned
// addresses, size a multiple of 16), all waits bounded by %globaltimer.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  unsigned done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// Waits for the phase with the given parity to complete, for at most
// kWaitLimitNs. On expiry records kErrTimeout in *err and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity, unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, kErrTimeout);
      return false;
    }
  }
}
// 16-byte store into the shared memory of CTA `rank` of the cluster, whose
// mbarrier (same offset as `local_bar` here) receives the completed bytes.
__device__ __forceinline__ void st_async_v4(const void* local_dst, const uint64_t* local_bar,
                                            unsigned rank, const float4& v) {
  const uint32_t dst = dsmem_map(smem_u32(local_dst), rank);
  const uint32_t bar = dsmem_map(smem_u32(local_bar), rank);
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::
          "r"(dst),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
      : "memory");
}

// Global -> this CTA's shared memory, completion signalled on `bar`.
__device__ __forceinline__ void tma_bulk_g2s(void* smem_dst, const void* gmem_src, unsigned bytes,
                                             uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace fnorm
