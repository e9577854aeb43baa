// in_kernels.cuh -- InstanceNorm forward kernels (affine = False).
//
// What is computed (page Kimi-K2.6__l1_p34, blocks 1-2; the same statistics
// as the InstanceNorm3d step of page Kimi-K2.6__l2_p79, block 1): for every
// (n,c) slice of S contiguous elements, the mean and the biased variance, then
// y = (x - mean) * rsqrt(var + eps).
//
// How (GB300 design, not the pages' H100 plan of one 512-thread block per slice
// reading the slice twice):
//  * The slice is held in REGISTERS while its statistics are formed, so it is
//    read from HBM once and written once. Each thread owns NV 16-byte slots
//    (4 fp32 or 8 bf16 values) loaded with 128-bit coalesced loads.
//  * Per thread, an exact two-pass mean/M2 over its own registers (shifted by
//    its first value so a constant slice gives M2 = 0 and the exact mean), then
//    the Chan pairwise merge: warp shuffles -> shared memory across warps ->
//    distributed shared memory across the CTAs of a thread-block cluster when
//    one slice spans several CTAs (up to 16, i.e. 2 MiB of input per slice).
//    Every merge runs in a fixed tree, so results are reproducible, and every
//    CTA of a cluster computes bit-identical statistics.
//  * Three shapes of the same idea:
//      group    -- G lanes of a warp per slice (S up to 256 slots);
//      resident -- one CTA or one cluster per slice;
//      stream   -- fallback for slices beyond cluster capacity: one cluster per
//                  slice, statistics pass then a normalisation pass that walks
//                  the slice backwards so its most recently read part is still
//                  in L2.
//  * Grids are persistent: as many CTAs/clusters as fit on the 152 SMs at
//    once, each looping over slices.
#pragma once

#include "fnorm_device.cuh"
#include "fnorm_internal.h"

namespace fnorm {

// Exact two-pass statistics of the first `nvalid` values of a thread's slots
// (values in (k, j) order: slot k, element j). Invalid values are ignored.
template <class Tin, int NV>
__device__ __forceinline__ Stat tile_stat(const uint4 (&r)[NV], int nvalid) {
  using E = Elem<Tin>;
  constexpr int W = E::W;
  if (nvalid <= 0) return stat_empty();
  const float x0 = E::get(r[0], 0);
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float d = E::get(r[k], j) - x0;
      s[j & 3] += (k * W + j < nvalid) ? d : 0.f;
    }
  const float n = static_cast<float>(nvalid);
  const float mean = x0 + ((s[0] + s[1]) + (s[2] + s[3])) / n;
  float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float d = E::get(r[k], j) - mean;
      q[j & 3] += (k * W + j < nvalid) ? d * d : 0.f;
    }
  return Stat{n, mean, (q[0] + q[1]) + (q[2] + q[3])};
}

__device__ __forceinline__ int clamp_int(int64_t v, int lo, int hi) {
  return v < lo ? lo : (v > hi ? hi : static_cast<int>(v));
}

// Warp partials -> one CTA partial (valid in thread 0 of warp 0).
template <int THREADS>
__device__ __forceinline__ Stat cta_merge(Stat st, Stat* warp_part) {
  constexpr int NWARP = THREADS / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  st = warp_merge<32>(st);
  if (NWARP == 1) return st;
  if (lane == 0) warp_part[warp] = st;
  __syncthreads();
  Stat s2 = stat_empty();
  if (warp == 0) {
    if (lane < NWARP) s2 = warp_part[lane];
    s2 = warp_merge<32>(s2);
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

    const Stat cta = cta_merge<THREADS>(tile_stat<Tin, NV>(r, nvalid), warp_part);
    const float2 mr = cluster_finalize<THREADS>(cta, cta_part, &fin, csize, it, p.eps);
    if (crank == 0 && tid == 0) {
      if (p.mean_out) p.mean_out[q] = mr.x;
      if (p.rstd_out) p.rstd_out[q] = mr.y;
    }

    if (VEC) {
      Tout* yv = ys + first * W;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (k * W < nvalid) {
          float o[W];
#pragma unroll
          for (int j = 0; j < W; ++j) o[j] = (E::get(r[k], j) - mr.x) * mr.y;
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
                               (E::get(r[k], j) - mr.x) * mr.y);
    }
  }
  // No CTA may leave while another can still read its shared memory.
  if (csize > 1) cluster_sync();
}

// ---------------------------------------------------------------------------
// Group: G consecutive lanes per slice, 256-thread CTAs, 32/G slices per warp
// per step. Slot (k, l) of lane l of the group is vector k*G + l of the slice
// (vector mode) or elements (k*W + j)*G + l.
// ---------------------------------------------------------------------------
template <class Tin, class Tout, int G, int NV, bool VEC>
__global__ void __launch_bounds__(256) in_group_kernel(const InParams p) {
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
    Tout* ys = y + q * S;
    if (VEC) {
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        if (k * W < nvalid) {
          float o[W];
#pragma unroll
          for (int j = 0; j < W; ++j) o[j] = (E::get(r[k], j) - mean) * rstd;
          VecStore<Tout, W>::run(ys + static_cast<int64_t>(k * G + gl) * W, o);
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int j = 0; j < W; ++j)
          if (k * W + j < nvalid)
            Elem<Tout>::store1(ys + (k * W + j) * G + gl, (E::get(r[k], j) - mean) * rstd);
    }
  }
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
            for (int j = 0; j < W; ++j) o[j] = (E::get(r[k], j) - mr.x) * mr.y;
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
                                 (E::get(r[k], j) - mr.x) * mr.y);
      }
    }
  }
  if (csize > 1) cluster_sync();
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
  cudaLaunchAttribute attr[1];
  int nattr = 0;
  if (cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    nattr = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <class K>
static int max_active_clusters(K kernel, int threads, int cluster) {
  if (cluster > 8) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
  }
  if (cluster <= 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    return per_sm * device_info().sm_count;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
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
      if (plan.threads == kStreamThreads)
        return reinterpret_cast<void*>(
            &in_stream_kernel<Tin, Tout, kStreamThreads, kStreamUnroll, VEC>);
      return nullptr;
  }
  return nullptr;
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
  return max_active_clusters(reinterpret_cast<InKernelFn>(k), threads, cl);
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
  return launch_clustered(fn, plan.grid, threads, cl, 0, stream, p);
}

}  // namespace fnorm
