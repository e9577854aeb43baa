// in_kernels.cuh -- InstanceNorm forward kernels (with optional per-channel
// affine parameters).
//
// What is computed (page Kimi-K2.6__l1_p34, blocks 1-2; the same statistics
// as the InstanceNorm3d step of page Kimi-K2.6__l2_p79, block 1): for every
// (n,c) slice of S contiguous elements, the mean and the biased variance, then
// y = (x - mean) * rsqrt(var + eps), or with affine parameters
// y = (x - mean) * (rsqrt(var + eps) * gamma_c) + beta_c.
//
// How (GB300 design, not the pages' H100 plan of one 512-thread block per slice
// reading the slice twice):
//  * The slice is held ON CHIP while its statistics are formed, so it is read
//    from HBM once and written once. Each thread owns 16-byte slots (4 fp32 or
//    8 bf16 values) in registers, loaded with 128-bit coalesced loads, and in
//    the split form also slots in shared memory filled by a TMA bulk copy
//    that is issued for the next slice while the current one is processed.
//  * Per thread, an exact two-pass mean/M2 over its own values (shifted by its
//    first value so a constant slice gives M2 = 0 and the exact mean). bf16
//    slices spread over clusters of more than 8 CTAs, which are issue-bound,
//    instead take one pass of sums shifted by the thread's first value (at
//    most 128 values, so the cancellation stays bounded) and normalise, both
//    as packed fp32 pairs. Then
//    the Chan pairwise merge: warp shuffles -> shared memory across warps ->
//    the CTAs of a thread-block cluster when one slice spans several CTAs (up
//    to 16, i.e. 2 MiB of input per slice; partials pushed with st.async).
//    Every merge runs in a fixed tree, so results are reproducible, and every
//    CTA of a cluster computes bit-identical statistics.
//  * Kernel shapes:
//      group    -- G lanes of a warp per slice (S up to 256 slots);
//      split    -- one CTA or one cluster per slice, registers (+ staged
//                  shared memory): the default for 16-byte-aligned slices;
//      resident -- one CTA or one cluster per slice, registers only, with
//                  element-wise access (unaligned inputs, S % vector != 0);
//      stream   -- slices beyond cluster capacity: one cluster per slice,
//                  statistics pass then a normalisation pass that walks the
//                  slice backwards so its most recently read part is still in
//                  L2.
//  * Grids are persistent: as many CTAs/clusters as fit on the SMs at once,
//    each looping over slices.
#pragma once

#include "fnorm_device.cuh"
#include "fnorm_internal.h"

namespace fnorm {

// Exact two-pass statistics of the first `nvalid` values of a thread's slots
// (values in (k, j) order: slot k, element j). Invalid values are ignored.
// Widened value j of a 16-byte slot; OPAQUE re-does the widening at every use
// (see Elem<__nv_bfloat16>::get_opaque).
template <class E, bool OPAQUE>
__device__ __forceinline__ float widen(const uint4& v, int j) {
  return OPAQUE ? E::get_opaque(v, j) : E::get(v, j);
}

template <class Tin, int NV, bool OPAQUE = false>
__device__ __forceinline__ Stat tile_stat_full(const uint4 (&r)[NV]) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  const float x0 = widen<E, OPAQUE>(r[0], 0);
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int j = 0; j < W; ++j) s[j & 3] += widen<E, OPAQUE>(r[k], j) - x0;
  constexpr float n = static_cast<float>(NV * W);
  const float mean = x0 + ((s[0] + s[1]) + (s[2] + s[3])) * (1.0f / n);
  float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float d = widen<E, OPAQUE>(r[k], j) - mean;
      q[j & 3] = fmaf(d, d, q[j & 3]);
    }
  return Stat{n, mean, (q[0] + q[1]) + (q[2] + q[3])};
}

template <class Tin, int NV, bool FAST = true, bool OPAQUE = false>
__device__ __forceinline__ Stat tile_stat(const uint4 (&r)[NV], int nvalid) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  if (FAST && nvalid == NV * W) return tile_stat_full<Tin, NV, OPAQUE>(r);   // no per-value predicates
  if (nvalid <= 0) return stat_empty();
  const float x0 = widen<E, OPAQUE>(r[0], 0);
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float d = widen<E, OPAQUE>(r[k], j) - x0;
      s[j & 3] += (k * W + j < nvalid) ? d : 0.f;
    }
  const float n = static_cast<float>(nvalid);
  const float mean = x0 + ((s[0] + s[1]) + (s[2] + s[3])) / n;
  float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float d = widen<E, OPAQUE>(r[k], j) - mean;
      q[j & 3] += (k * W + j < nvalid) ? d * d : 0.f;
    }
  return Stat{n, mean, (q[0] + q[1]) + (q[2] + q[3])};
}

// Packed pair arithmetic for bf16 inputs: the two values of one 32-bit word of
// a slot (elements 2i, 2i+1) less a constant, as an fp32 pair, processed by
// one f32x2 instruction (__fadd2_rn / __ffma2_rn), which halves the
// floating-point instructions of slices that are issue-bound (a byte of bf16
// holds twice the values of fp32). The pair comes from two mixed-precision
// subtractions (Elem<bf16>::diff_lo / diff_hi): the same bits as widening the
// pair and adding (-c, -c), one instruction fewer per pair (bf16 S = 2^20:
// 5698 -> 5838 GB/s). The scalar loops keep the widening: there the mixed
// form measured 2-4 % slower (S = 256, 4096, 16384, 65536).
__device__ __forceinline__ float2 bf16_pair_diff(unsigned w, float c) {
  using E = Elem<__nv_bfloat16>;
  return make_float2(E::diff_lo(w, c), E::diff_hi(w, c));
}

// Shifted sums of a thread's bf16 values in one pass: d = x - K (K the
// thread's first value), s += d, q += d^2, as pairs (words 0, 2 into 01;
// 1, 3 into 23). mean = K + S/n and M2 = Q - S^2/n follow; K is one of the
// values, so (K - mean)^2 <= M2 and the cancellation is bounded by the
// thread's count (at most 128 values in the kernels that use it).
__device__ __forceinline__ void bf16_acc_onepass(const uint4& v, float K, float2& s01, float2& s23,
                                                 float2& q01, float2& q23) {
  float2 d = bf16_pair_diff(v.x, K);
  s01 = __fadd2_rn(s01, d);
  q01 = __ffma2_rn(d, d, q01);
  d = bf16_pair_diff(v.y, K);
  s23 = __fadd2_rn(s23, d);
  q23 = __ffma2_rn(d, d, q23);
  d = bf16_pair_diff(v.z, K);
  s01 = __fadd2_rn(s01, d);
  q01 = __ffma2_rn(d, d, q01);
  d = bf16_pair_diff(v.w, K);
  s23 = __fadd2_rn(s23, d);
  q23 = __ffma2_rn(d, d, q23);
}

// o = (v - mean) * a + b
__device__ __forceinline__ void bf16_norm(const uint4& v, float mean, float2 a2, float2 b2, float (&o)[8]) {
  const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 r = __ffma2_rn(bf16_pair_diff(w[i], mean), a2, b2);
    o[2 * i] = r.x;
    o[2 * i + 1] = r.y;
  }
}

__device__ __forceinline__ int clamp_int(int64_t v, int lo, int hi) {
  return v < lo ? lo : (v > hi ? hi : static_cast<int>(v));
}

// Warp partials -> one CTA partial (valid in thread 0 of warp 0). `uniform`
// (the same for every thread of the CTA): every thread holds a partial of the
// same count, so the merges take the equal-count form (warp_merge_eq: the
// same tree and the same bits, no division).
template <int THREADS>
__device__ __forceinline__ Stat cta_merge(Stat st, Stat* warp_part, bool uniform = false) {
  constexpr int NWARP = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  st = uniform ? warp_merge_eq<32>(st) : warp_merge<32>(st);
  if (NWARP == 1) return st;
  if (lane == 0) warp_part[warp] = st;
  __syncthreads();
  Stat s2 = stat_empty();
  if (warp == 0) {
    if (lane < NWARP) s2 = warp_part[lane];
    s2 = uniform ? warp_merge_eq<(NWARP > 1 ? NWARP : 2)>(s2) : warp_merge<32>(s2);
  }
  return s2;
}

// CTA partial (valid in thread 0) -> slice statistics shared by the whole
// cluster; returns (mean, rstd) to every thread of the CTA. `cta_part` is a
// 2-entry shared array indexed by iteration parity, so one cluster barrier per
// slice suffices: a CTA rewrites entry (it & 1) only after every CTA of the
// cluster has passed the barrier of iteration it+1, i.e. after their reads.
template <int THREADS>
__device__ __forceinline__ float2 cluster_finalize(const Stat& cta, Stat* cta_part, float2* fin,
                                                   unsigned csize, int it, float eps) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (csize == 1) {
    if (threadIdx.x == 0) *fin = make_float2(cta.mean, rsqrtf(cta.m2 / cta.n + eps));
  } else {
    if (threadIdx.x == 0) cta_part[it & 1] = cta;
    cluster_sync();
    if (warp == 0) {
      Stat s = stat_empty();
      if (lane < static_cast<int>(csize)) {
        const uint32_t a = dsmem_map(smem_u32(&cta_part[it & 1]), lane);
        s.n = ld_dsmem_f32(a);
        s.mean = ld_dsmem_f32(a + 4);
        s.m2 = ld_dsmem_f32(a + 8);
      }
      s = warp_merge<16>(s);
      if (lane == 0) *fin = make_float2(s.mean, rsqrtf(s.m2 / s.n + eps));
    }
  }
  __syncthreads();
  return *fin;
}

// Output coefficients of slice q: y = (x - mean) * a + b, with a = rstd * gamma_c
// and b = beta_c for the affine form and a = rstd, b = 0 without it.
__device__ __forceinline__ float2 in_affine(const InParams& p, int64_t q, float rstd) {
  float a = rstd, b = 0.f;
  if (p.gamma != nullptr || p.beta != nullptr) {
    const int64_t c = q % p.C;
    if (p.gamma != nullptr) a = rstd * __ldg(p.gamma + c);
    if (p.beta != nullptr) b = __ldg(p.beta + c);
  }
  return make_float2(a, b);
}

// ---------------------------------------------------------------------------
// Resident: one CTA (cluster size 1) or one cluster per slice.
// Slot (k, t) of CTA rank r is vector r*THREADS*NV + k*THREADS + t of the
// slice (vector mode) or, element-wise, elements
// r*THREADS*NV*W + (k*W + j)*THREADS + t for j < W.
// ---------------------------------------------------------------------------
// Register budget: 64 per thread for 8 slots (32 data registers), 48 for 4.
constexpr int resident_min_blocks(int threads, int nv) {
  return ((nv >= 8 ? 1024 : 1280) / threads) > 0 ? (nv >= 8 ? 1024 : 1280) / threads : 1;
}

template <class Tin, class Tout, int THREADS, int NV, bool VEC>
__global__ void __launch_bounds__(THREADS, resident_min_blocks(THREADS, NV))
    in_resident_kernel(const InParams p) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ Stat cta_part[2];
  __shared__ float2 fin;

  const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
  const unsigned cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x;
  const Tin* __restrict__ x = static_cast<const Tin*>(p.x);
  Tout* __restrict__ y = static_cast<Tout*>(p.y);
  const int64_t S = p.S;

  // The valid prefix of this thread's values is the same for every slice.
  int nvalid;
  int64_t first;   // vector index (VEC) or element index of slot (0, 0)
  if (VEC) {
    first = static_cast<int64_t>(crank) * THREADS * NV + tid;
    const int64_t nvec = S / W;
    const int kvalid = first < nvec ? clamp_int((nvec - first + THREADS - 1) / THREADS, 0, NV) : 0;
    nvalid = kvalid * W;
  } else {
    first = static_cast<int64_t>(crank) * THREADS * NV * W + tid;
    nvalid = first < S ? clamp_int((S - first + THREADS - 1) / THREADS, 0, NV * W) : 0;
  }

  pdl_wait();
  int it = 0;
  for (int64_t q = cid; q < p.NC; q += ncl, ++it) {
    const Tin* xs = x + q * S;
    Tout* ys = y + q * S;
    uint4 r[NV];
    if (VEC) {
      const uint4* xv = reinterpret_cast<const uint4*>(xs) + first;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        r[k] = (k * W < nvalid) ? ld_v4(xv + k * THREADS) : make_uint4(0, 0, 0, 0);
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        r[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (k * W + j < nvalid)
            E::set(r[k], j, E::load1(xs + first + static_cast<int64_t>(k * W + j) * THREADS));
      }
    }

    // (no full-tile fast path here: a second unrolled copy of the two-pass would
    // push the 64-register budget of 8 bf16 slots per thread into spills)
    const Stat cta = cta_merge<THREADS>(tile_stat<Tin, NV, false, true>(r, nvalid), warp_part);
    const float2 mr = cluster_finalize<THREADS>(cta, cta_part, &fin, csize, it, p.eps);
    if (crank == 0 && tid == 0) {
      if (p.mean_out) p.mean_out[q] = mr.x;
      if (p.rstd_out) p.rstd_out[q] = mr.y;
    }
    const float2 ab = in_affine(p, q, mr.y);

    if (VEC) {
      Tout* yv = ys + first * W;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (k * W < nvalid) {
          float o[W];
#pragma unroll
          for (int j = 0; j < W; ++j) o[j] = fmaf(E::get_opaque(r[k], j) - mr.x, ab.x, ab.y);
          VecStore<Tout, W>::run(yv + static_cast<int64_t>(k) * THREADS * W, o);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (k * W + j < nvalid)
            Elem<Tout>::store1(ys + first + static_cast<int64_t>(k * W + j) * THREADS,
                               fmaf(E::get_opaque(r[k], j) - mr.x, ab.x, ab.y));
    }
  }
  pdl_trigger();
  // No CTA may leave while another can still read its shared memory.
  if (csize > 1) cluster_sync();
}

// ---------------------------------------------------------------------------
// Group: G consecutive lanes per slice, 256-thread CTAs, 32/G slices per warp
// per step. Slot (k, l) of lane l of the group is vector k*G + l of the slice
// (vector mode) or elements (k*W + j)*G + l.
// ---------------------------------------------------------------------------
// Up to 4 slots per lane: 64 registers, four 256-thread CTAs per SM.
template <class Tin, class Tout, int G, int NV, bool VEC>
__global__ void __launch_bounds__(256, NV >= 8 ? 2 : 4) in_group_kernel(const InParams p) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  constexpr int GPW = 32 / G;
  const int lane = threadIdx.x & 31;
  const int gl = lane % G, gw = lane / G;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x) >> 5;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * 8;
  const Tin* __restrict__ x = static_cast<const Tin*>(p.x);
  Tout* __restrict__ y = static_cast<Tout*>(p.y);
  const int64_t S = p.S;

  int nvalid_lane;
  if (VEC) {
    const int64_t nvec = S / W;
    nvalid_lane = gl < nvec ? clamp_int((nvec - gl + G - 1) / G, 0, NV) * W : 0;
  } else {
    nvalid_lane = gl < S ? clamp_int((S - gl + G - 1) / G, 0, NV * W) : 0;
  }

  pdl_wait();
  // The loop bound is uniform across the warp, so every lane reaches every
  // shuffle; groups past the end of the tensor carry empty statistics.
  for (int64_t base = warp_id * GPW; base < p.NC; base += nwarps * GPW) {
    const int64_t q = base + gw;
    const bool active = q < p.NC;
    const int nvalid = active ? nvalid_lane : 0;
    const Tin* xs = x + q * S;
    uint4 r[NV];
    if (VEC) {
      const uint4* xv = reinterpret_cast<const uint4*>(xs) + gl;
#pragma unroll
      for (int k = 0; k < NV; ++k)
        r[k] = (k * W < nvalid) ? ld_v4(xv + k * G) : make_uint4(0, 0, 0, 0);
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        r[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (k * W + j < nvalid) E::set(r[k], j, E::load1(xs + (k * W + j) * G + gl));
      }
    }
    Stat st = warp_merge<G>(tile_stat<Tin, NV>(r, nvalid));
    // broadcast the group's statistics from its first lane
    const float n = __shfl_sync(kFullMask, st.n, 0, G);
    const float mean = __shfl_sync(kFullMask, st.mean, 0, G);
    const float m2 = __shfl_sync(kFullMask, st.m2, 0, G);
    if (!active) continue;
    const float rstd = rsqrtf(m2 / n + p.eps);
    if (gl == 0) {
      if (p.mean_out) p.mean_out[q] = mean;
      if (p.rstd_out) p.rstd_out[q] = rstd;
    }
    const float2 ab = in_affine(p, q, rstd);
    Tout* ys = y + q * S;
    if (VEC) {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (k * W < nvalid) {
          float o[W];
#pragma unroll
          for (int j = 0; j < W; ++j) o[j] = fmaf(E::get(r[k], j) - mean, ab.x, ab.y);
          VecStore<Tout, W>::run(ys + static_cast<int64_t>(k * G + gl) * W, o);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (k * W + j < nvalid)
            Elem<Tout>::store1(ys + (k * W + j) * G + gl, fmaf(E::get(r[k], j) - mean, ab.x, ab.y));
    }
  }
  pdl_trigger();
}

// ---------------------------------------------------------------------------
// Stream (fallback for long slices): one cluster per slice, tiles of
// THREADS*U slots, statistics pass then normalisation pass in reverse tile
// order. Tiles are split between the CTAs of the cluster in contiguous runs.
// ---------------------------------------------------------------------------
template <class Tin, class Tout, int THREADS, int U, bool VEC>
__device__ __forceinline__ void stream_load_tile(const Tin* xs, int64_t S, int64_t tile,
                                                 uint4 (&r)[U], int& nvalid) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  const int tid = threadIdx.x;
  if (VEC) {
    const int64_t nvec = S / W;
    const int64_t v0 = tile * THREADS * U + tid;
    nvalid = v0 < nvec ? clamp_int((nvec - v0 + THREADS - 1) / THREADS, 0, U) * W : 0;
    const uint4* xv = reinterpret_cast<const uint4*>(xs) + v0;
#pragma unroll
    for (int k = 0; k < U; ++k) r[k] = (k * W < nvalid) ? ld_v4(xv + k * THREADS) : make_uint4(0, 0, 0, 0);
  } else {
    const int64_t e0 = tile * THREADS * U * W + tid;
    nvalid = e0 < S ? clamp_int((S - e0 + THREADS - 1) / THREADS, 0, U * W) : 0;
#pragma unroll
    for (int k = 0; k < U; ++k) {
      r[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < W; ++j)
        if (k * W + j < nvalid)
          E::set(r[k], j, E::load1(xs + e0 + static_cast<int64_t>(k * W + j) * THREADS));
    }
  }
}

template <class Tin, class Tout, int THREADS, int U, bool VEC>
__global__ void __launch_bounds__(THREADS) in_stream_kernel(const InParams p) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ Stat cta_part[2];
  __shared__ float2 fin;
  const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
  const unsigned cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x;
  const Tin* __restrict__ x = static_cast<const Tin*>(p.x);
  Tout* __restrict__ y = static_cast<Tout*>(p.y);
  const int64_t S = p.S;
  const int64_t tile_elems = static_cast<int64_t>(THREADS) * U * W;
  const int64_t ntiles = (S + tile_elems - 1) / tile_elems;
  const int64_t t0 = ntiles * crank / csize, t1 = ntiles * (crank + 1) / csize;

  pdl_wait();
  int it = 0;
  for (int64_t q = cid; q < p.NC; q += ncl, ++it) {
    const Tin* xs = x + q * S;
    Tout* ys = y + q * S;
    Stat acc = stat_empty();
    for (int64_t t = t0; t < t1; ++t) {
      uint4 r[U];
      int nvalid;
      stream_load_tile<Tin, Tout, THREADS, U, VEC>(xs, S, t, r, nvalid);
      acc = chan_merge(acc, tile_stat<Tin, U>(r, nvalid));
    }
    const Stat cta = cta_merge<THREADS>(acc, warp_part);
    const float2 mr = cluster_finalize<THREADS>(cta, cta_part, &fin, csize, it, p.eps);
    if (crank == 0 && tid == 0) {
      if (p.mean_out) p.mean_out[q] = mr.x;
      if (p.rstd_out) p.rstd_out[q] = mr.y;
    }
    const float2 ab = in_affine(p, q, mr.y);
    for (int64_t t = t1 - 1; t >= t0; --t) {
      uint4 r[U];
      int nvalid;
      stream_load_tile<Tin, Tout, THREADS, U, VEC>(xs, S, t, r, nvalid);
      if (VEC) {
        Tout* yv = ys + (t * THREADS * U + tid) * W;
#pragma unroll
        for (int k = 0; k < U; ++k) {
          if (k * W < nvalid) {
            float o[W];
#pragma unroll
            for (int j = 0; j < W; ++j) o[j] = fmaf(E::get(r[k], j) - mr.x, ab.x, ab.y);
            VecStore<Tout, W>::run(yv + static_cast<int64_t>(k) * THREADS * W, o);
          }
        }
      } else {
        const int64_t e0 = t * tile_elems + tid;
#pragma unroll
        for (int k = 0; k < U; ++k)
#pragma unroll
          for (int j = 0; j < W; ++j)
            if (k * W + j < nvalid)
              Elem<Tout>::store1(ys + e0 + static_cast<int64_t>(k * W + j) * THREADS,
                                 fmaf(E::get(r[k], j) - mr.x, ab.x, ab.y));
      }
    }
  }
  pdl_trigger();
  if (csize > 1) cluster_sync();
}

// ---------------------------------------------------------------------------
// Split-resident (vector access only): one CTA or one cluster per slice. A
// CTA's chunk of the slice is THREADS*(NS + NR) 16-byte slots: the first
// THREADS*NS slots are staged in shared memory by one TMA bulk copy
// (cp.async.bulk + mbarrier), the remaining THREADS*NR are held in registers
// (128-bit loads). Splitting the chunk between the two on-chip stores lets a
// 512-thread CTA hold 128 KiB while two CTAs share an SM, so one SM keeps two
// slices' traffic in flight. Per slice:
//   wait for the staged part -> exact per-thread two-pass over both parts ->
//   warp/CTA Chan merge -> cluster exchange -> normalise and store the staged
//   part -> barrier -> bulk-copy the NEXT slice's staged part (prefetch) ->
//   normalise and store the register part -> load the next register part.
// Cluster exchange: instead of a cluster-wide barrier per slice, each CTA
// pushes its partial (n, mean, M2) into slot [rank] of every CTA of the
// cluster with st.async, which completes bytes on the receiver's mbarrier;
// each CTA waits only for its own barrier and merges the csize slots in rank
// order, so all CTAs obtain bit-identical statistics. Two slot sets and two
// barriers alternate by slice parity; a CTA can reuse a set only after every
// CTA has consumed it (it needs their next partials first).
// Dynamic shared memory: THREADS*NS*16 bytes.
// ---------------------------------------------------------------------------
constexpr int split_min_blocks(int threads, int nr) {
  return ((nr >= 8 ? 1024 : 1280) / threads) > 0 ? (nr >= 8 ? 1024 : 1280) / threads : 1;
}

template <int THREADS>
__device__ __forceinline__ float2 cluster_exchange(const Stat& cta, float4 (*slots)[kMaxCluster],
                                                   uint64_t* xbar, float2* fin, unsigned csize,
                                                   unsigned crank, int it, float eps,
                                                   unsigned* err, bool& xfailed) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (csize == 1) {
    if (threadIdx.x == 0) *fin = make_float2(cta.mean, rsqrtf(cta.m2 / cta.n + eps));
  } else {
    const int b = it & 1;
    const unsigned phase = (static_cast<unsigned>(it) >> 1) & 1u;
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&xbar[b], csize * 16u);
      const float4 v = make_float4(cta.n, cta.mean, cta.m2, 0.f);
      for (unsigned r = 0; r < csize; ++r) st_async_v4(&slots[b][crank], &xbar[b], r, v);
    }
    if (warp == 0) {
      if (!xfailed && !mbar_wait_bounded(&xbar[b], phase, err)) xfailed = true;
      Stat s = stat_empty();
      if (lane < static_cast<int>(csize)) {
        const float4 v = slots[b][lane];
        s = Stat{v.x, v.y, v.z};
      }
      s = warp_merge<16>(s);
      if (lane == 0) *fin = make_float2(s.mean, rsqrtf(s.m2 / s.n + eps));
    }
  }
  __syncthreads();
  return *fin;
}

template <class Tin, class Tout, int THREADS, int NR, int NS, bool PACK>
__global__ void __launch_bounds__(THREADS, split_min_blocks(THREADS, NR))
    in_split_kernel(const InParams p) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  // bf16 input, PACK: one pass of shifted sums for the statistics and the
  // normalisation, both as packed pairs (bf16_acc_onepass, bf16_norm). The
  // plan sets PACK for slices spread over clusters of more than 8 CTAs, where
  // a slice's arithmetic sits between the arrival of its data and the cluster
  // exchange (bf16 S = 2^20, 16-CTA clusters: 5002 -> 5720 GB/s, 6235 with the
  // mixed-precision pairs and equal-count merges), and for slices held by one
  // 64-thread CTA (bf16 S = 4096: 5967-5995 -> 6130-6143 GB/s); with 8, 4 or
  // 1 larger CTAs per slice it measured 2-7 % slower (S = 16384 ... 2^18), and
  // those keep the exact two-pass scalar loops.
  constexpr bool kPackedBf16 = PACK && W == 8;
  extern __shared__ __align__(128) uint4 stage[];   // [NS][THREADS] slots
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ __align__(16) float4 slots[2][kMaxCluster];
  __shared__ float2 fin;
  __shared__ __align__(8) uint64_t tma_bar;
  __shared__ __align__(8) uint64_t xbar[2];
  __shared__ __align__(8) uint64_t dbg_bar;

  const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
  const unsigned cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x;
  const Tin* __restrict__ x = static_cast<const Tin*>(p.x);
  Tout* __restrict__ y = static_cast<Tout*>(p.y);
  const int64_t S = p.S;
  const int64_t nvec = S / W;
  constexpr int64_t kChunk = static_cast<int64_t>(THREADS) * (NR + NS);
  const int64_t base = static_cast<int64_t>(crank) * kChunk;          // first vector of the chunk
  const int64_t cvec = base < nvec ? (nvec - base < kChunk ? nvec - base : kChunk) : 0;
  const int64_t svec = cvec < int64_t(THREADS) * NS ? cvec : int64_t(THREADS) * NS;
  const int64_t rvec = cvec - svec;
  const unsigned sbytes = static_cast<unsigned>(svec * 16);
  const int ns_valid = (NS > 0 && tid < svec) ? clamp_int((svec - tid + THREADS - 1) / THREADS, 0, NS) : 0;
  const int nr_valid = (NR > 0 && tid < rvec) ? clamp_int((rvec - tid + THREADS - 1) / THREADS, 0, NR) : 0;
  const int64_t rbase = base + int64_t(THREADS) * NS + tid;   // vector of register slot 0
  const int nvalid = (ns_valid + nr_valid) * W;

  if (tid == 0) {
    mbar_init(&tma_bar, 1);
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  if (csize > 1) cluster_sync();   // peers' barriers exist before anyone signals them
  else __syncthreads();

  pdl_wait();
  bool failed = false, xfailed = false;
  unsigned tparity = 0;
  if (tid == 0 && sbytes > 0 && cid < p.NC) {
    mbar_arrive_expect_tx(&tma_bar, sbytes);
    tma_bulk_g2s(stage, reinterpret_cast<const uint4*>(x + cid * S) + base, sbytes, &tma_bar);
  }
  uint4 r[NR > 0 ? NR : 1];
  if (cid < p.NC) {
    const uint4* xv = reinterpret_cast<const uint4*>(x + cid * S) + rbase;
#pragma unroll
    for (int k = 0; k < NR; ++k) r[k] = (k < nr_valid) ? ld_v4(xv + k * THREADS) : make_uint4(0, 0, 0, 0);
  }

  int it = 0;
  for (int64_t q = cid; q < p.NC; q += ncl, ++it) {
    if (sbytes > 0 && !failed) {
      const bool ok = mbar_wait_bounded(&tma_bar, tparity, p.err);
      failed = __syncthreads_or(!ok) != 0;
      if (!failed) tparity ^= 1u;
    }
    // exact two-pass over this thread's values, shifted by its first value
    Stat st = stat_empty();
    if (kPackedBf16 && nvalid > 0) {
      // one pass of shifted sums as pairs (bf16_acc_onepass)
      const float K = E::get_opaque(ns_valid > 0 ? stage[tid] : r[0], 0);
      float2 s01 = make_float2(0.f, 0.f), s23 = s01, q01 = s01, q23 = s01;
#pragma unroll
      for (int k = 0; k < NS; ++k)
        if (k < ns_valid) bf16_acc_onepass(stage[k * THREADS + tid], K, s01, s23, q01, q23);
#pragma unroll
      for (int k = 0; k < NR; ++k)
        if (k < nr_valid) bf16_acc_onepass(r[k], K, s01, s23, q01, q23);
      const float n = static_cast<float>(nvalid);
      const float sd = (s01.x + s01.y) + (s23.x + s23.y), qd = (q01.x + q01.y) + (q23.x + q23.y);
      st = Stat{n, K + sd / n, fmaxf(qd - sd * (sd / n), 0.f)};
    } else if (nvalid > 0) {
      const float x0 = E::get_opaque(ns_valid > 0 ? stage[tid] : r[0], 0);
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        if (k < ns_valid) {
          const uint4 v = stage[k * THREADS + tid];
#pragma unroll
          for (int j = 0; j < W; ++j) s4[j & 3] += E::get_opaque(v, j) - x0;
        }
      }
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        if (k < nr_valid) {
#pragma unroll
          for (int j = 0; j < W; ++j) s4[j & 3] += E::get_opaque(r[k], j) - x0;
        }
      }
      const float n = static_cast<float>(nvalid);
      const float mean = x0 + ((s4[0] + s4[1]) + (s4[2] + s4[3])) / n;
      float q4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < NS; ++k) {
        if (k < ns_valid) {
          const uint4 v = stage[k * THREADS + tid];
#pragma unroll
          for (int j = 0; j < W; ++j) {
            const float d = E::get_opaque(v, j) - mean;
            q4[j & 3] = fmaf(d, d, q4[j & 3]);
          }
        }
      }
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        if (k < nr_valid) {
#pragma unroll
          for (int j = 0; j < W; ++j) {
            const float d = E::get_opaque(r[k], j) - mean;
            q4[j & 3] = fmaf(d, d, q4[j & 3]);
          }
        }
      }
      st = Stat{n, mean, (q4[0] + q4[1]) + (q4[2] + q4[3])};
    }
    // equal-count merges where every thread of the CTA holds its full share,
    // in the packed form only: there the merge lies between the data's
    // arrival and the cluster exchange (bf16 S = 2^20: 5838 -> 6240 GB/s);
    // in the scalar kernels it measured 3-7 % slower (fewer instructions,
    // but the loads' latency more exposed: long-scoreboard stalls 3.6 -> 5.4
    // per issue at S = 16384)
    const Stat cta = cta_merge<THREADS>(st, warp_part, kPackedBf16 && cvec == kChunk);
    const float2 mr = cluster_exchange<THREADS>(cta, slots, xbar, &fin, csize, crank, it, p.eps,
                                                p.err, xfailed);
    if (crank == 0 && tid == 0) {
      if (p.mean_out) p.mean_out[q] = mr.x;
      if (p.rstd_out) p.rstd_out[q] = mr.y;
    }
    const float2 ab = in_affine(p, q, mr.y);
    Tout* yq = y + q * S;
    // staged part
#pragma unroll
    for (int k = 0; k < NS; ++k) {
      if (k < ns_valid) {
        const uint4 v = stage[k * THREADS + tid];
        float o[W];
        if constexpr (kPackedBf16) {
          bf16_norm(v, mr.x, make_float2(ab.x, ab.x), make_float2(ab.y, ab.y), o);
        } else {
#pragma unroll
          for (int j = 0; j < W; ++j) o[j] = fmaf(E::get_opaque(v, j) - mr.x, ab.x, ab.y);
        }
        VecStore<Tout, W>::run(yq + (base + int64_t(k) * THREADS + tid) * W, o);
      }
    }
    const int64_t qn = q + ncl;
    if (NS > 0) {
      __syncthreads();   // the stage has been read; refill it with the next slice
      if (tid == 0 && sbytes > 0 && qn < p.NC && !failed) {
        mbar_arrive_expect_tx(&tma_bar, sbytes);
        tma_bulk_g2s(stage, reinterpret_cast<const uint4*>(x + qn * S) + base, sbytes, &tma_bar);
      }
    }
    // register part
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      if (k < nr_valid) {
        float o[W];
        if constexpr (kPackedBf16) {
          bf16_norm(r[k], mr.x, make_float2(ab.x, ab.x), make_float2(ab.y, ab.y), o);
        } else {
#pragma unroll
          for (int j = 0; j < W; ++j) o[j] = fmaf(E::get_opaque(r[k], j) - mr.x, ab.x, ab.y);
        }
        VecStore<Tout, W>::run(yq + (rbase + int64_t(k) * THREADS) * W, o);
      }
    }
    if (qn < p.NC) {
      const uint4* xv = reinterpret_cast<const uint4*>(x + qn * S) + rbase;
#pragma unroll
      for (int k = 0; k < NR; ++k) r[k] = (k < nr_valid) ? ld_v4(xv + k * THREADS) : make_uint4(0, 0, 0, 0);
    }
  }
  pdl_trigger();
  if (csize > 1) cluster_sync();   // no CTA leaves while a peer may still signal it
  if (failed && sbytes > 0) mbar_wait_bounded(&tma_bar, tparity, p.err);
  // Test hook, after the last cluster barrier so no peer waits on this CTA: a
  // wait on a barrier nothing completes must expire, record the timeout in the
  // error word and return.
  if (p.debug_timeout && cid == 0 && crank == 0 && tid == 0) mbar_wait_bounded(&dbg_bar, 0, p.err);
}

// ---------------------------------------------------------------------------
// Host side: kernel selection, persistent grid sizing, cluster launch.
// ---------------------------------------------------------------------------
template <class K>
static cudaError_t launch_clustered(K kernel, int grid, int threads, int cluster, size_t smem,
                                    cudaStream_t stream, const InParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[nattr].val.programmaticStreamSerializationAllowed = 1;
  ++nattr;
  if (cluster > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = cluster;
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <class K>
static int max_active_clusters(K kernel, int threads, int cluster, size_t smem) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cluster > 8) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  if (cluster <= 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return per_sm * device_info().sm_count;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <class Tin, class Tout, bool VEC>
static void* pick_kernel(const InPlan& plan) {
  switch (plan.path) {
    case InPath::kResident:
#define FNORM_RES(T, V)                                 \
  if (plan.threads == T && plan.nv == V)                \
    return reinterpret_cast<void*>(&in_resident_kernel<Tin, Tout, T, V, VEC>);
      FNORM_RES(128, 4) FNORM_RES(256, 4) FNORM_RES(256, 8) FNORM_RES(512, 8) FNORM_RES(1024, 8)
#undef FNORM_RES
      return nullptr;
    case InPath::kGroup:
#define FNORM_GRP(G, V)                                 \
  if (plan.group == G && plan.nv == V)                  \
    return reinterpret_cast<void*>(&in_group_kernel<Tin, Tout, G, V, VEC>);
      FNORM_GRP(8, 1) FNORM_GRP(8, 4) FNORM_GRP(32, 2) FNORM_GRP(32, 4) FNORM_GRP(32, 8)
#undef FNORM_GRP
      return nullptr;
    case InPath::kStream:
      if (plan.threads == kStreamThreads && plan.nv == kStreamUnroll)
        return reinterpret_cast<void*>(
            &in_stream_kernel<Tin, Tout, kStreamThreads, kStreamUnroll, VEC>);
      if (plan.threads == kStreamThreads && plan.nv == kStreamUnrollFew)
        return reinterpret_cast<void*>(
            &in_stream_kernel<Tin, Tout, kStreamThreads, kStreamUnrollFew, VEC>);
      return nullptr;
    case InPath::kSplit:
      if (!VEC) return nullptr;
      if (plan.packed) {
        if constexpr (Elem<Tin>::W == 8) {
#define FNORM_SPLIT_P(T, R, SM)                                      \
  if (plan.threads == T && plan.nv == R && plan.ns == SM)            \
    return reinterpret_cast<void*>(&in_split_kernel<Tin, Tout, T, R, SM, true>);
          FNORM_SPLIT_P(256, 8, 8) FNORM_SPLIT_P(512, 8, 8) FNORM_SPLIT_P(1024, 8, 8)
          FNORM_SPLIT_P(64, 8, 0)
#undef FNORM_SPLIT_P
        }
        return nullptr;
      }
#define FNORM_SPLIT(T, R, SM)                                        \
  if (plan.threads == T && plan.nv == R && plan.ns == SM)            \
    return reinterpret_cast<void*>(&in_split_kernel<Tin, Tout, T, R, SM, false>);
      FNORM_SPLIT(128, 8, 8) FNORM_SPLIT(256, 8, 8) FNORM_SPLIT(512, 8, 8) FNORM_SPLIT(1024, 8, 8)
      FNORM_SPLIT(64, 8, 0) FNORM_SPLIT(128, 8, 0) FNORM_SPLIT(256, 8, 0) FNORM_SPLIT(512, 8, 0)
      FNORM_SPLIT(1024, 8, 0)
#undef FNORM_SPLIT
      return nullptr;
  }
  return nullptr;
}

// Dynamic shared memory of a plan (the pipelined path's stage buffer).
inline size_t in_plan_smem(const InPlan& plan) {
  return plan.path == InPath::kSplit ? static_cast<size_t>(plan.threads) * plan.ns * 16 : 0;
}

template <class Tin, class Tout>
static void* pick(const InPlan& plan) {
  return plan.vec ? pick_kernel<Tin, Tout, true>(plan) : pick_kernel<Tin, Tout, false>(plan);
}

using InKernelFn = void (*)(InParams);

template <class Tin, class Tout>
int in_max_active_clusters_t(const InPlan& plan) {
  void* k = pick<Tin, Tout>(plan);
  if (!k) return 0;
  const int threads = plan.path == InPath::kGroup ? 256 : plan.threads;
  const int cl = plan.path == InPath::kGroup ? 1 : plan.cluster;
  return max_active_clusters(reinterpret_cast<InKernelFn>(k), threads, cl, in_plan_smem(plan));
}

template <class Tin, class Tout>
cudaError_t in_launch_t(const InParams& p, const InPlan& plan, cudaStream_t stream) {
  void* k = pick<Tin, Tout>(plan);
  if (!k) return cudaErrorInvalidConfiguration;
  const InKernelFn fn = reinterpret_cast<InKernelFn>(k);
  const int threads = plan.path == InPath::kGroup ? 256 : plan.threads;
  const int cl = plan.path == InPath::kGroup ? 1 : plan.cluster;
  if (cl > 8) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  const size_t smem = in_plan_smem(plan);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_clustered(fn, plan.grid, threads, cl, smem, stream, p);
}

}  // namespace fnorm
