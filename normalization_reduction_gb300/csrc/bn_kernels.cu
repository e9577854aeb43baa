// bn_kernels.cu -- training-mode BatchNorm forward with a trailing scale
// (page Kimi-K2.6__l2_p73, blocks 1-2: BatchNorm2d in training mode, batch
// statistics per channel over (N, H, W), affine gamma/beta, then
// x * scaling_factor; the running statistics are updated with momentum, the
// running variance from the unbiased estimate as page Kimi-K2.6__l2_p79,
// block 1, states).
//
// A channel's values are N runs of S contiguous elements, C*S apart. A channel
// of the page's tensor (128 x 126 x 126 fp32 = 8.1 MB) is far larger than any
// on-chip store, so x is read twice, in two launches over "units" (one run,
// or a chunk of <= 16384 values of a longer run), in memory order:
//   1. statistics -- one CTA per unit; in vector mode the whole unit is in
//                    flight at once (bn_stats_split_kernel: 128-bit register
//                    loads plus one TMA bulk copy into shared memory), exact
//                    two-pass per thread, Chan merges -> one partial
//                    (n, mean, M2) per unit in the caller's workspace;
//   2. apply      -- one CTA per unit, in the reverse of memory order so the
//                    last ~100 MB the statistics pass read are still in L2
//                    (bn_apply_staged_kernel: the unit's TMA copy is issued
//                    before the channel's partials are merged in a fixed tree,
//                    so every CTA of a channel obtains bit-identical
//                    statistics); y = (x - mean)*A + B with A = scale*gamma*rstd,
//                    B = scale*beta; evict-first stores keep the reusable
//                    input in L2. The CTA of (n = 0, chunk 0) writes the saved
//                    statistics and updates the running statistics.
// Eval mode (running statistics) is one elementwise pass (bn_eval_*_kernel).
// Element-wise (unaligned or S % 4 != 0) inputs take register-only kernels
// with the same unit order and results.
#include <atomic>

#include "fnorm_device.cuh"
#include "fnorm_internal.h"
#include "in_kernels.cuh"

namespace fnorm {

// Thread-level statistics of elements [lo, hi) of run xr in tiles of
// THREADS*U*4 elements (vector mode: lo and the run length are multiples of 4).
template <int THREADS, int U, bool VEC>
__device__ __forceinline__ Stat bn_range_stat(const float* xr, int64_t lo, int64_t hi) {
  Stat acc = stat_empty();
  const int tid = threadIdx.x;
  constexpr int64_t TILE = static_cast<int64_t>(THREADS) * U * 4;
  for (int64_t t = lo; t < hi; t += TILE) {
    uint4 r[U];
    int nvalid;
    if (VEC) {
      const int64_t v0 = t / 4 + tid, vend = hi / 4;
      nvalid = v0 < vend ? clamp_int((vend - v0 + THREADS - 1) / THREADS, 0, U) * 4 : 0;
      const uint4* xv = reinterpret_cast<const uint4*>(xr) + v0;
#pragma unroll
      for (int k = 0; k < U; ++k) r[k] = (k * 4 < nvalid) ? ld_v4(xv + k * THREADS) : make_uint4(0, 0, 0, 0);
    } else {
      const int64_t e0 = t + tid;
      nvalid = e0 < hi ? clamp_int((hi - e0 + THREADS - 1) / THREADS, 0, U * 4) : 0;
#pragma unroll
      for (int k = 0; k < U; ++k) {
        r[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (k * 4 + j < nvalid)
            Elem<float>::set(r[k], j, __ldg(xr + e0 + static_cast<int64_t>(k * 4 + j) * THREADS));
      }
    }
    acc = chan_merge(acc, tile_stat<float, U>(r, nvalid));
  }
  return acc;
}

// Units (run, chunk) in memory order: unit m covers chunk m % chunks of run
// m / chunks = n*C + c. Its partial goes to partials[c][n*chunks + k].
struct BnUnit {
  int64_t run, n, c, k, lo, hi;
};
__device__ __forceinline__ BnUnit bn_unit(const BnParams& p, int64_t m) {
  BnUnit u;
  u.run = m / p.chunks;
  u.k = m - u.run * p.chunks;
  u.n = u.run / p.C;
  u.c = u.run - u.n * p.C;
  u.lo = u.k * p.chunk;
  u.hi = (u.lo + p.chunk < p.S) ? u.lo + p.chunk : p.S;
  return u;
}
__device__ __forceinline__ float4* bn_partial(const BnParams& p, const BnUnit& u) {
  if (p.part_cstride)   // strided placement (InstanceNorm, output buffer as scratch)
    return p.partials + u.c * p.part_cstride + (u.n * p.chunks + u.k) * p.part_kstride;
  return p.partials + u.c * (p.N * p.chunks) + u.n * p.chunks + u.k;
}

template <int THREADS, int U, bool VEC>
__global__ void __launch_bounds__(THREADS, 4) bn_stats_kernel(const BnParams p) {
  __shared__ Stat warp_part[THREADS / 32];
  const BnUnit u = bn_unit(p, static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x);
  const float* xr = p.x + u.run * p.S;
  pdl_wait();
  const Stat cta = cta_merge<THREADS>(bn_range_stat<THREADS, U, VEC>(xr, u.lo, u.hi), warp_part);
  if (threadIdx.x == 0) *bn_partial(p, u) = make_float4(cta.n, cta.mean, cta.m2, 0.f);
  pdl_trigger();
}

// Statistics pass in vector mode for units of up to kBnChunk values: the
// whole unit is in flight at once -- the first THREADS*NR vectors by 128-bit
// register loads, the rest by one TMA bulk copy into shared memory issued
// first -- so that four CTAs per SM keep ~256 KB of reads outstanding. Each
// thread takes the exact two-pass statistics of its register values, then of
// its staged values, and merges the two.
template <int THREADS, int NR, int NS>
__global__ void __launch_bounds__(THREADS, 4) bn_stats_split_kernel(const BnParams p) {
  extern __shared__ __align__(128) uint4 stage[];   // (THREADS * NS) vectors
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ uint64_t bar;
  __shared__ uint64_t dbg_bar;
  const int tid = threadIdx.x;
  const BnUnit u = bn_unit(p, static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x);
  const uint4* xv = reinterpret_cast<const uint4*>(p.x + u.run * p.S + u.lo);
  constexpr int RV = THREADS * NR;
  const int nvec = static_cast<int>((u.hi - u.lo) / 4);
  const int svec = nvec > RV ? nvec - RV : 0;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  // The apply launch may be scheduled as soon as every CTA of this grid has
  // started (its CTAs then wait in griddepcontrol.wait for this grid to
  // complete), which hides its launch behind the last wave of this one.
  pdl_trigger();
  if (tid == 0 && svec > 0) {
    mbar_arrive_expect_tx(&bar, static_cast<unsigned>(svec) * 16u);
    tma_bulk_g2s(stage, xv + RV, static_cast<unsigned>(svec) * 16u, &bar);
  }
  const int rvec = nvec < RV ? nvec : RV;
  const int kr = tid < rvec ? clamp_int((rvec - tid + THREADS - 1) / THREADS, 0, NR) : 0;
  uint4 r[NR];
#pragma unroll
  for (int k = 0; k < NR; ++k) r[k] = k < kr ? ld_v4(xv + k * THREADS + tid) : make_uint4(0, 0, 0, 0);
  Stat st = tile_stat<float, NR>(r, kr * 4);
  if (svec > 0) {
    // a wait that gives up has flagged the error; it is retried once (bounded)
    // so that the copy is not in flight when the CTA leaves
    if (!mbar_wait_bounded(&bar, 0, p.err)) mbar_wait_bounded(&bar, 0, p.err);
    const int ks = tid < svec ? clamp_int((svec - tid + THREADS - 1) / THREADS, 0, NS) : 0;
#pragma unroll
    for (int k = 0; k < NS; ++k) r[k] = k < ks ? stage[k * THREADS + tid] : make_uint4(0, 0, 0, 0);
    st = chan_merge(st, tile_stat<float, NS>(r, ks * 4));
  }
  const Stat cta = cta_merge<THREADS>(st, warp_part);
  if (tid == 0) *bn_partial(p, u) = make_float4(cta.n, cta.mean, cta.m2, 0.f);
  // Test hook: one CTA waits on a barrier nothing completes; the wait must
  // expire, record the timeout in the error word and return.
  if (p.debug_timeout && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
    mbar_wait_bounded(&dbg_bar, 0, p.err);
}

// The channel's statistics, merged in a fixed order from `count` partials
// part[i * istride] (read through L2 when LOADCG: partials written by other
// SMs of the same launch), as the apply coefficients (mean, A, B) for every
// thread of the CTA; with `first` the CTA also writes the saved statistics
// and updates the running statistics (count = all values of the channel, all
// ranks; unbiased variance for the running estimate).
template <int THREADS, bool LOADCG>
__device__ __forceinline__ float4 bn_channel_coef(const BnParams& p, int64_t c, const float4* part,
                                                  int64_t count, int64_t istride, bool first,
                                                  Stat* warp_part, float4* coef) {
  Stat acc = stat_empty();
  for (int64_t i = threadIdx.x; i < count; i += THREADS) {
    const float4 v = LOADCG ? __ldcg(part + i * istride) : part[i * istride];
    acc = chan_merge(acc, Stat{v.x, v.y, v.z});
  }
  const Stat s = cta_merge<THREADS>(acc, warp_part);
  if (threadIdx.x == 0) {
    const float var = s.m2 / s.n;
    const float rstd = rsqrtf(var + p.eps);
    const int64_t gc = p.affine_period ? c % p.affine_period : c;
    const float g = p.gamma ? p.gamma[gc] : 1.f;
    const float bt = p.beta ? p.beta[gc] : 0.f;
    *coef = make_float4(s.mean, p.scale * g * rstd, p.scale * bt, 0.f);
    if (first) {
      if (p.save_mean) p.save_mean[c] = s.mean;
      if (p.save_rstd) p.save_rstd[c] = rstd;
      if (p.running_mean && p.running_var) {
        const double cnt = static_cast<double>(s.n);
        const double mom = p.momentum;
        const double unbiased = static_cast<double>(s.m2) / (cnt - 1.0);
        p.running_mean[c] = static_cast<float>((1.0 - mom) * p.running_mean[c] +
                                               mom * static_cast<double>(s.mean));
        p.running_var[c] = static_cast<float>((1.0 - mom) * p.running_var[c] + mom * unbiased);
      }
    }
  }
  __syncthreads();
  return *coef;
}

template <int THREADS, int U, bool VEC>
__global__ void __launch_bounds__(THREADS, 4) bn_apply_kernel(const BnParams p) {
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ float4 coef;
  // units in the reverse of memory order: the statistics pass read the last
  // units most recently, so they are still in L2
  const int64_t nb = static_cast<int64_t>(gridDim.x);
  const int64_t lin = static_cast<int64_t>(gridDim.y) * nb - 1 -
                      (static_cast<int64_t>(blockIdx.y) * nb + blockIdx.x);
  int64_t c, b, lo, hi, off;
  if (p.N == 0) {
    // an empty shard still merges the statistics and updates the running
    // statistics (one CTA per channel) but has nothing to normalise
    c = lin;
    b = 0;
    lo = hi = off = 0;
  } else {
    const BnUnit u = bn_unit(p, lin);
    c = u.c;
    b = u.n * p.chunks + u.k;
    lo = u.lo;
    hi = u.hi;
    off = u.run * p.S;
  }
  const float* xr = p.x + off;
  float* yr = p.y + off;
  pdl_wait();

  // channel statistics: the channel's partials (or the ranks' statistics)
  // merged in a fixed order
  const float4 cf = bn_channel_coef<THREADS, false>(p, c, p.stats + c * p.stats_cstride +
                                                             b * p.stats_kstride,
                                                    p.stats_count, p.stats_istride, b == 0,
                                                    warp_part, &coef);

  const int tid = threadIdx.x;
  constexpr int64_t TILE = static_cast<int64_t>(THREADS) * U * 4;
  const int64_t ntiles = (hi - lo + TILE - 1) / TILE;
  for (int64_t ti = ntiles - 1; ti >= 0; --ti) {
    const int64_t t = lo + ti * TILE;
    if (VEC) {
      const int64_t v0 = t / 4 + tid, vend = hi / 4;
      const uint4* xv = reinterpret_cast<const uint4*>(xr) + v0;
      float4* yv = reinterpret_cast<float4*>(yr) + v0;
      uint4 r[U];
#pragma unroll
      for (int k2 = 0; k2 < U; ++k2)
        if (v0 + k2 * THREADS < vend) r[k2] = ld_v4(xv + k2 * THREADS);
#pragma unroll
      for (int k2 = 0; k2 < U; ++k2) {
        if (v0 + k2 * THREADS < vend) {
          float o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = fmaf(Elem<float>::get(r[k2], j) - cf.x, cf.y, cf.z);
          __stcs(yv + k2 * THREADS, make_float4(o[0], o[1], o[2], o[3]));
        }
      }
    } else {
      for (int64_t e = t + tid; e < t + TILE && e < hi; e += THREADS)
        __stcs(yr + e, fmaf(__ldg(xr + e) - cf.x, cf.y, cf.z));
    }
  }
}

// Apply pass in vector mode: the CTA's unit (<= kBnChunk values) is fetched
// by one TMA bulk copy into shared memory, issued before the channel's
// statistics are merged so that the merge overlaps the copy; then every
// thread normalises staged vectors and streams them out. Same unit order,
// statistics merge and side outputs as bn_apply_kernel.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 3) bn_apply_staged_kernel(const BnParams p) {
  extern __shared__ __align__(128) uint4 stage[];   // kBnChunk / 4 vectors
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ float4 coef;
  __shared__ uint64_t bar;
  __shared__ uint64_t dbg_bar;
  const int tid = threadIdx.x;
  const int64_t nb = static_cast<int64_t>(gridDim.x);
  const int64_t lin = static_cast<int64_t>(gridDim.y) * nb - 1 -
                      (static_cast<int64_t>(blockIdx.y) * nb + blockIdx.x);
  const BnUnit u = bn_unit(p, lin);
  const int64_t off = u.run * p.S + u.lo;
  const int nvec = static_cast<int>((u.hi - u.lo) / 4);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (tid == 0 && nvec > 0) {
    mbar_arrive_expect_tx(&bar, static_cast<unsigned>(nvec) * 16u);
    tma_bulk_g2s(stage, p.x + off, static_cast<unsigned>(nvec) * 16u, &bar);
  }
  // (with the output buffer as scratch, the unit's own copy of the
  // statistics lies at the start of its output range: read here, before the
  // barrier in bn_channel_coef, and overwritten by this CTA's stores below)
  const float4 cf = bn_channel_coef<THREADS, false>(
      p, u.c, p.stats + u.c * p.stats_cstride + (u.n * p.chunks + u.k) * p.stats_kstride,
      p.stats_count, p.stats_istride, u.n == 0 && u.k == 0, warp_part, &coef);
  if (nvec > 0) {
    // a wait that gives up has flagged the error; it is retried once (bounded)
    // so that the copy is not in flight when the CTA leaves
    if (!mbar_wait_bounded(&bar, 0, p.err)) mbar_wait_bounded(&bar, 0, p.err);
    float4* yv = reinterpret_cast<float4*>(p.y + off);
#pragma unroll 4
    for (int j = tid; j < nvec; j += THREADS) {
      const uint4 r = stage[j];
      float o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = fmaf(Elem<float>::get(r, q) - cf.x, cf.y, cf.z);
      __stcs(yv + j, make_float4(o[0], o[1], o[2], o[3]));
    }
  }
  // Test hook: one CTA waits on a barrier nothing completes; the wait must
  // expire, record the timeout in the error word and return.
  if (p.debug_timeout && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
    mbar_wait_bounded(&dbg_bar, 0, p.err);
}

// ---------------------------------------------------------------------------
// Resident form (one cooperative launch): a persistent grid of THREADS-thread
// CTAs walks the units in memory order (unit b + i*G for CTA b), computing the
// statistics as bn_stats_split_kernel does; the staged part (up to THREADS*NS
// vectors) of each CTA's last unit stays in shared memory across a grid-wide
// barrier; then every CTA normalises its units in reverse order -- the
// resident one first, the others re-read (the most recent ones from L2).
// The grid barrier is an arrival counter in the workspace (zeroed by the
// host before the launch) that thread 0 of each CTA polls for at most the
// wait limit; an expired wait sets the error word and the kernel finishes
// (results then invalid). Partials written by other SMs are read through L2.
// ---------------------------------------------------------------------------
template <int THREADS, int NR, int NS>
__global__ void __launch_bounds__(THREADS, 4) bn_resident_kernel(const BnParams p) {
  extern __shared__ __align__(128) uint4 stage[];   // THREADS * NS vectors
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ float4 coef;
  __shared__ uint64_t bar;
  __shared__ uint64_t dbg_bar;
  constexpr int RV = THREADS * NR;
  const int tid = threadIdx.x;
  const int64_t G = gridDim.x;
  const int64_t units = p.N * p.C * p.chunks;
  const int64_t mine = blockIdx.x < units ? (units - blockIdx.x + G - 1) / G : 0;
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  unsigned tph = 0;       // parity of the TMA barrier's next completion
  bool failed = false;    // a bounded wait expired (error word set)

  // ---- phase 1: statistics of every unit of this CTA
  for (int64_t i = 0; i < mine; ++i) {
    const BnUnit u = bn_unit(p, blockIdx.x + i * G);
    const uint4* xv = reinterpret_cast<const uint4*>(p.x + u.run * p.S + u.lo);
    const int nvec = static_cast<int>((u.hi - u.lo) / 4);
    const int svec = nvec > RV ? nvec - RV : 0;
    if (tid == 0 && svec > 0 && !failed) {
      mbar_arrive_expect_tx(&bar, static_cast<unsigned>(svec) * 16u);
      tma_bulk_g2s(stage, xv + RV, static_cast<unsigned>(svec) * 16u, &bar);
    }
    const int rvec = nvec < RV ? nvec : RV;
    const int kr = tid < rvec ? clamp_int((rvec - tid + THREADS - 1) / THREADS, 0, NR) : 0;
    uint4 r[NR];
#pragma unroll
    for (int k = 0; k < NR; ++k) r[k] = k < kr ? ld_v4(xv + k * THREADS + tid) : make_uint4(0, 0, 0, 0);
    Stat st = tile_stat<float, NR>(r, kr * 4);
    if (svec > 0) {
      // an expired wait is retried once (bounded) so that the copy is not in
      // flight when the CTA leaves; no further copies are issued
      if (!failed && !mbar_wait_bounded(&bar, tph, p.err)) {
        mbar_wait_bounded(&bar, tph, p.err);
        failed = true;
      }
      tph ^= 1u;
      const int ks = tid < svec ? clamp_int((svec - tid + THREADS - 1) / THREADS, 0, NS) : 0;
#pragma unroll
      for (int k = 0; k < NS; ++k) r[k] = k < ks ? stage[k * THREADS + tid] : make_uint4(0, 0, 0, 0);
      st = chan_merge(st, tile_stat<float, NS>(r, ks * 4));
    }
    // (cta_merge's barrier also orders this unit's reads of the stage before
    // the next unit's copy into it)
    const Stat cta = cta_merge<THREADS>(st, warp_part);
    if (tid == 0) *bn_partial(p, u) = make_float4(cta.n, cta.mean, cta.m2, 0.f);
    failed = __syncthreads_or(failed);
  }

  // ---- grid-wide barrier: every partial is written before any is merged
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(p.grid_counter, 1u);
    const unsigned target = static_cast<unsigned>(G);
    if (atomicAdd(p.grid_counter, 0u) < target) {
      const unsigned long long t0 = globaltimer_ns();
      while (atomicAdd(p.grid_counter, 0u) < target) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicOr(p.err, kErrTimeout);
          break;
        }
      }
    }
    __threadfence();
  }
  __syncthreads();

  // ---- phase 2: normalise the units in reverse order, the resident one first
  for (int64_t i = mine - 1; i >= 0; --i) {
    const BnUnit u = bn_unit(p, blockIdx.x + i * G);
    const int64_t off = u.run * p.S + u.lo;
    const uint4* xv = reinterpret_cast<const uint4*>(p.x + off);
    const int nvec = static_cast<int>((u.hi - u.lo) / 4);
    const int svec = nvec > RV ? nvec - RV : 0;
    const bool resident = i == mine - 1;
    if (!resident && tid == 0 && svec > 0 && !failed) {
      mbar_arrive_expect_tx(&bar, static_cast<unsigned>(svec) * 16u);
      tma_bulk_g2s(stage, xv + RV, static_cast<unsigned>(svec) * 16u, &bar);
    }
    // the channel's statistics: its partials merged in a fixed order
    const float4 cf = bn_channel_coef<THREADS, true>(p, u.c, p.partials + u.c * (p.N * p.chunks),
                                                     p.N * p.chunks, 1, u.n == 0 && u.k == 0,
                                                     warp_part, &coef);
    const int rvec = nvec < RV ? nvec : RV;
    const int kr = tid < rvec ? clamp_int((rvec - tid + THREADS - 1) / THREADS, 0, NR) : 0;
    uint4 r[NR];
#pragma unroll
    for (int k = 0; k < NR; ++k) r[k] = k < kr ? ld_v4(xv + k * THREADS + tid) : make_uint4(0, 0, 0, 0);
    float4* yv = reinterpret_cast<float4*>(p.y + off);
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      if (k < kr) {
        float o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = fmaf(Elem<float>::get(r[k], q) - cf.x, cf.y, cf.z);
        __stcs(yv + k * THREADS + tid, make_float4(o[0], o[1], o[2], o[3]));
      }
    }
    if (svec > 0) {
      if (!resident) {
        if (!failed && !mbar_wait_bounded(&bar, tph, p.err)) {
          mbar_wait_bounded(&bar, tph, p.err);
          failed = true;
        }
        tph ^= 1u;
      }
      for (int j = tid; j < svec; j += THREADS) {
        const uint4 v = stage[j];
        float o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = fmaf(Elem<float>::get(v, q) - cf.x, cf.y, cf.z);
        __stcs(yv + RV + j, make_float4(o[0], o[1], o[2], o[3]));
      }
    }
    failed = __syncthreads_or(failed);   // the stage is read before the next copy
  }
  // Test hook: one CTA waits on a barrier nothing completes; the wait must
  // expire, record the timeout in the error word and return.
  if (p.debug_timeout && blockIdx.x == 0 && tid == 0) mbar_wait_bounded(&dbg_bar, 0, p.err);
}

// ---------------------------------------------------------------------------
// Column form for short runs (S <= kBnColMaxS, e.g. BatchNorm over [N, C]):
// x is read as N rows of W = C*S values. Units of one run would be a handful
// of values each, so instead
//   1. bn_col_stats_kernel -- a CTA covers THREADS columns x kBnColRows rows;
//      each thread takes the exact two-pass statistics of its column's rows
//      -> partial[j][row block] (channel c owns columns [c*S, (c+1)*S), so its
//      partials are contiguous);
//   2. bn_col_merge_kernel -- one CTA per channel merges them in a fixed
//      order into (mean, A, B), the saved and the running statistics;
//   3. bn_col_apply_kernel -- elementwise, each thread walks one column down
//      the rows with its channel's coefficients.
// ---------------------------------------------------------------------------
template <int THREADS, int R>
__global__ void __launch_bounds__(THREADS) bn_col_stats_kernel(const BnParams p) {
  const int64_t W = p.C * p.S;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x;
  const int64_t nrb = (p.N + R - 1) / R;
  pdl_wait();
  for (int64_t rb = blockIdx.y; rb < nrb; rb += gridDim.y) {
    if (j < W) {
      const int64_t r0 = rb * R;
      const int rows = static_cast<int>(p.N - r0 < R ? p.N - r0 : R);
      float v[R];
#pragma unroll
      for (int k = 0; k < R; ++k) v[k] = k < rows ? __ldg(p.x + (r0 + k) * W + j) : 0.f;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < R; ++k) sum += k < rows ? v[k] - v[0] : 0.f;
      const float n = static_cast<float>(rows);
      const float mean = v[0] + sum / n;
      float m2 = 0.f;
#pragma unroll
      for (int k = 0; k < R; ++k) {
        const float d = v[k] - mean;
        m2 += k < rows ? d * d : 0.f;
      }
      p.partials[j * nrb + rb] = make_float4(n, mean, m2, 0.f);
    }
  }
  pdl_trigger();
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) bn_col_merge_kernel(const BnParams p) {
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ float4 coef;
  const int64_t c = blockIdx.x;
  const int64_t count = p.S * ((p.N + kBnColRows - 1) / kBnColRows);
  pdl_wait();
  const float4 cf = bn_channel_coef<THREADS, false>(p, c, p.partials + c * count, count, 1, true,
                                                    warp_part, &coef);
  if (threadIdx.x == 0) p.local_out[c] = cf;   // the channel's (mean, A, B)
  pdl_trigger();
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) bn_col_apply_kernel(const BnParams p) {
  const int64_t W = p.C * p.S;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x;
  pdl_wait();
  if (j < W) {
    const float4 cf = p.local_out[j / p.S];
    for (int64_t r = blockIdx.y; r < p.N; r += gridDim.y)
      p.y[r * W + j] = fmaf(__ldg(p.x + r * W + j) - cf.x, cf.y, cf.z);
  }
  pdl_trigger();
}

// Multi-rank apply for short runs (column form): each thread folds the R
// ranks' statistics of its column's channel in rank order (the same fold on
// every rank, so every rank obtains the same bits), then walks its column;
// the thread of the channel's first column in the first row group writes the
// saved statistics and updates the running statistics.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) bn_col_apply_stats_kernel(const BnParams p) {
  const int64_t W = p.C * p.S;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x;
  pdl_wait();
  if (j < W) {
    const int64_t c = j / p.S;
    Stat s = stat_empty();
    for (int64_t r = 0; r < p.stats_count; ++r) {
      const float4 v = p.stats[c * p.stats_cstride + r * p.stats_istride];
      s = chan_merge(s, Stat{v.x, v.y, v.z});
    }
    const float rstd = rsqrtf(s.m2 / s.n + p.eps);
    const float g = p.gamma ? p.gamma[c] : 1.f;
    const float bt = p.beta ? p.beta[c] : 0.f;
    const float4 cf = make_float4(s.mean, p.scale * g * rstd, p.scale * bt, 0.f);
    if (blockIdx.y == 0 && j == c * p.S) {
      if (p.save_mean) p.save_mean[c] = s.mean;
      if (p.save_rstd) p.save_rstd[c] = rstd;
      if (p.running_mean && p.running_var) {
        const double cnt = static_cast<double>(s.n);
        const double mom = p.momentum;
        const double unbiased = static_cast<double>(s.m2) / (cnt - 1.0);
        p.running_mean[c] = static_cast<float>((1.0 - mom) * p.running_mean[c] +
                                               mom * static_cast<double>(s.mean));
        p.running_var[c] = static_cast<float>((1.0 - mom) * p.running_var[c] + mom * unbiased);
      }
    }
    for (int64_t r = blockIdx.y; r < p.N; r += gridDim.y)
      p.y[r * W + j] = fmaf(__ldg(p.x + r * W + j) - cf.x, cf.y, cf.z);
  }
  pdl_trigger();
}

// Local statistics of a rank's shard: one CTA per channel merges the
// channel's partials in a fixed order into local_out[c] = (n, mean, M2, 0).
template <int THREADS>
__global__ void __launch_bounds__(THREADS) bn_merge_kernel(const BnParams p) {
  __shared__ Stat warp_part[THREADS / 32];
  const int64_t c = blockIdx.x;
  pdl_wait();
  const float4* part = p.stats + c * p.stats_cstride;
  Stat acc = stat_empty();
  // four loads in flight per thread before they are merged, in the same order
  // as one at a time (the partials may lie 64 KiB apart, each its own sector):
  // x[1,1,8192,8192] through the output-scratch route 3704-3780 -> 3961-3964
  // GB/s, through the workspace 3999-4014 -> 4073-4103 (eight: no better)
  constexpr int B = 4;
  int64_t i = threadIdx.x;
  for (; i + (B - 1) * THREADS < p.stats_count; i += B * THREADS) {
    float4 v[B];
#pragma unroll
    for (int b = 0; b < B; ++b) v[b] = part[(i + b * THREADS) * p.stats_istride];
#pragma unroll
    for (int b = 0; b < B; ++b) acc = chan_merge(acc, Stat{v[b].x, v[b].y, v[b].z});
  }
  for (; i < p.stats_count; i += THREADS) {
    const float4 v = part[i * p.stats_istride];
    acc = chan_merge(acc, Stat{v.x, v.y, v.z});
  }
  const Stat s = cta_merge<THREADS>(acc, warp_part);
  if (p.local_copies > 1) {
    // one copy per unit of the channel (output buffer as scratch): every
    // thread has read its partials before cta_merge's barrier, and the copies
    // overwrite them only after this one
    __shared__ float4 merged;
    if (threadIdx.x == 0) merged = make_float4(s.n, s.mean, s.m2, 0.f);
    __syncthreads();
    for (int64_t i = threadIdx.x; i < p.local_copies; i += THREADS)
      p.local_out[c * p.local_cstride + i * p.local_kstride] = merged;
  } else if (threadIdx.x == 0) {
    p.local_out[c] = make_float4(s.n, s.mean, s.m2, 0.f);
  }
  pdl_trigger();
}

// ---------------------------------------------------------------------------
// Eval mode (running statistics; page Kimi-K2.6__l2_p73, blocks 1-2): one
// elementwise pass, y = (x - running_mean_c) * A_c + B_c with
// A_c = scale * gamma_c * rsqrt(running_var_c + eps) and B_c = scale * beta_c.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 bn_eval_coef(const BnParams& p, int64_t c) {
  const float rstd = rsqrtf(__ldg(p.running_var + c) + p.eps);
  const float g = p.gamma ? __ldg(p.gamma + c) : 1.f;
  const float bt = p.beta ? __ldg(p.beta + c) : 0.f;
  return make_float4(__ldg(p.running_mean + c), p.scale * g * rstd, p.scale * bt, 0.f);
}

// Long runs: one CTA per (run, chunk), U vectors per thread in flight.
template <int THREADS, int U, bool VEC>
__global__ void __launch_bounds__(THREADS) bn_eval_kernel(const BnParams p) {
  const int64_t c = blockIdx.y, b = blockIdx.x;
  const int64_t n = b / p.chunks, k = b - n * p.chunks;
  const int64_t off = (n * p.C + c) * p.S;
  const float* xr = p.x + off;
  float* yr = p.y + off;
  const int64_t lo = k * p.chunk, hi = (lo + p.chunk < p.S) ? lo + p.chunk : p.S;
  const int tid = threadIdx.x;
  pdl_wait();
  const float4 cf = bn_eval_coef(p, c);
  constexpr int64_t TILE = static_cast<int64_t>(THREADS) * U * 4;
  for (int64_t t = lo; t < hi; t += TILE) {
    if (VEC) {
      const int64_t v0 = t / 4 + tid, vend = hi / 4;
      const uint4* xv = reinterpret_cast<const uint4*>(xr) + v0;
      float4* yv = reinterpret_cast<float4*>(yr) + v0;
      uint4 r[U];
#pragma unroll
      for (int k2 = 0; k2 < U; ++k2)
        if (v0 + k2 * THREADS < vend) r[k2] = ld_v4(xv + k2 * THREADS);
#pragma unroll
      for (int k2 = 0; k2 < U; ++k2) {
        if (v0 + k2 * THREADS < vend) {
          float o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) o[j] = fmaf(Elem<float>::get(r[k2], j) - cf.x, cf.y, cf.z);
          yv[k2 * THREADS] = make_float4(o[0], o[1], o[2], o[3]);
        }
      }
    } else {
      for (int64_t e = t + tid; e < t + TILE && e < hi; e += THREADS)
        yr[e] = fmaf(__ldg(xr + e) - cf.x, cf.y, cf.z);
    }
  }
  pdl_trigger();
}

// Long runs in vector mode: one CTA per unit (<= kBnChunk values) fetched by
// one TMA bulk copy into shared memory, so that the whole unit is in flight
// while the channel's coefficients are formed.
template <int THREADS>
__global__ void __launch_bounds__(THREADS, 3) bn_eval_staged_kernel(const BnParams p) {
  extern __shared__ __align__(128) uint4 stage[];   // kBnChunk / 4 vectors
  __shared__ uint64_t bar;
  __shared__ uint64_t dbg_bar;
  const int tid = threadIdx.x;
  const BnUnit u = bn_unit(p, static_cast<int64_t>(blockIdx.y) * gridDim.x + blockIdx.x);
  const int64_t off = u.run * p.S + u.lo;
  const int nvec = static_cast<int>((u.hi - u.lo) / 4);
  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  if (tid == 0 && nvec > 0) {
    mbar_arrive_expect_tx(&bar, static_cast<unsigned>(nvec) * 16u);
    tma_bulk_g2s(stage, p.x + off, static_cast<unsigned>(nvec) * 16u, &bar);
  }
  const float4 cf = bn_eval_coef(p, u.c);
  if (nvec > 0) {
    // a wait that gives up has flagged the error; it is retried once (bounded)
    // so that the copy is not in flight when the CTA leaves
    if (!mbar_wait_bounded(&bar, 0, p.err)) mbar_wait_bounded(&bar, 0, p.err);
    float4* yv = reinterpret_cast<float4*>(p.y + off);
#pragma unroll 4
    for (int j = tid; j < nvec; j += THREADS) {
      const uint4 r = stage[j];
      float o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = fmaf(Elem<float>::get(r, q) - cf.x, cf.y, cf.z);
      yv[j] = make_float4(o[0], o[1], o[2], o[3]);
    }
  }
  pdl_trigger();
  // Test hook: one CTA waits on a barrier nothing completes; the wait must
  // expire, record the timeout in the error word and return.
  if (p.debug_timeout && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0)
    mbar_wait_bounded(&dbg_bar, 0, p.err);
}

// Very short runs (S <= kBnColMaxS, e.g. [N, C]): x as N rows of C*S values;
// each thread walks one column down the rows with its channel's coefficients.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) bn_eval_col_kernel(const BnParams p) {
  const int64_t W = p.C * p.S;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x;
  pdl_wait();
  if (j < W) {
    const float4 cf = bn_eval_coef(p, j / p.S);
    for (int64_t r = blockIdx.y; r < p.N; r += gridDim.y)
      p.y[r * W + j] = fmaf(__ldg(p.x + r * W + j) - cf.x, cf.y, cf.z);
  }
  pdl_trigger();
}

// Short runs (S < kBnEvalFlatBelow): a grid-stride loop over vectors (or
// elements), each finding its channel from its index.
template <int THREADS, bool VEC>
__global__ void __launch_bounds__(THREADS) bn_eval_flat_kernel(const BnParams p) {
  const int64_t per_run = VEC ? p.S / 4 : p.S;
  const int64_t units = p.N * p.C * per_run;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * THREADS;
  pdl_wait();
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * THREADS + threadIdx.x; u < units;
       u += stride) {
    const float4 cf = bn_eval_coef(p, (u / per_run) % p.C);
    if (VEC) {
      const uint4 r = ld_v4(reinterpret_cast<const uint4*>(p.x) + u);
      float o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) o[j] = fmaf(Elem<float>::get(r, j) - cf.x, cf.y, cf.z);
      reinterpret_cast<float4*>(p.y)[u] = make_float4(o[0], o[1], o[2], o[3]);
    } else {
      p.y[u] = fmaf(__ldg(p.x + u) - cf.x, cf.y, cf.z);
    }
  }
  pdl_trigger();
}

// Stream-ordered launch with programmatic dependent launch allowed; `smem`
// bytes of dynamic shared memory.
static cudaError_t bn_launch_one(void (*kernel)(BnParams), dim3 grid, cudaStream_t stream,
                                 const BnParams& p, size_t smem = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kBnThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Allows `bytes` of dynamic shared memory for a staged kernel, once per device.
// (Setting the attribute is idempotent, so racing host threads are harmless.)
static cudaError_t allow_smem(void (*kernel)(BnParams), size_t bytes,
                              std::atomic<bool> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(bytes));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}

// One staged unit of kBnChunk fp32 values per CTA.
constexpr size_t kBnStageBytes = static_cast<size_t>(kBnChunk) * 4;

// The statistics pass: the split kernel in vector mode (unless
// FNORM_BN_SPLIT=0 asks for the register-only kernel), the register-only
// kernel otherwise.
static cudaError_t bn_launch_stats(const BnParams& p, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.N * p.chunks), static_cast<unsigned>(p.C), 1);
  if (p.vec && p.split)
    return bn_launch_one(&bn_stats_split_kernel<kBnThreads, kBnSplitRegs, kBnSplitStaged>, grid,
                         stream, p, static_cast<size_t>(kBnThreads) * kBnSplitStaged * 16);
  return p.vec ? bn_launch_one(&bn_stats_kernel<kBnThreads, kBnStatsUnroll, true>, grid, stream, p)
               : bn_launch_one(&bn_stats_kernel<kBnThreads, kBnStatsUnroll, false>, grid, stream, p);
}

// The apply pass over N*chunks x C units (at least one CTA per channel).
static cudaError_t bn_launch_apply_pass(const BnParams& p, cudaStream_t stream) {
  const int64_t nb = p.N * p.chunks > 0 ? p.N * p.chunks : 1;
  const dim3 grid(static_cast<unsigned>(nb), static_cast<unsigned>(p.C), 1);
  if (p.vec && p.split && p.N > 0) {
    static std::atomic<bool> done[64];
    const cudaError_t e = allow_smem(&bn_apply_staged_kernel<kBnThreads>, kBnStageBytes, done);
    if (e != cudaSuccess) return e;
    return bn_launch_one(&bn_apply_staged_kernel<kBnThreads>, grid, stream, p, kBnStageBytes);
  }
  return p.vec ? bn_launch_one(&bn_apply_kernel<kBnThreads, kBnUnroll, true>, grid, stream, p)
               : bn_launch_one(&bn_apply_kernel<kBnThreads, kBnUnroll, false>, grid, stream, p);
}

cudaError_t bn_launch(const BnParams& p, cudaStream_t stream) {
  cudaError_t e = bn_launch_stats(p, stream);
  if (e != cudaSuccess) return e;
  return bn_launch_apply_pass(p, stream);
}

cudaError_t bn_launch_resident(const BnParams& p, cudaStream_t stream) {
  auto kernel = &bn_resident_kernel<kBnThreads, kBnSplitRegs, kBnSplitStaged>;
  const size_t smem = static_cast<size_t>(kBnThreads) * kBnSplitStaged * 16;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBnThreads, smem);
  if (e != cudaSuccess) return e;
  const int64_t units = p.N * p.C * p.chunks;
  const int64_t cap = static_cast<int64_t>(per_sm) * device_info().sm_count;
  if (cap <= 0) return cudaErrorCooperativeLaunchTooLarge;
  e = cudaMemsetAsync(p.grid_counter, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units < cap ? units : cap), 1, 1);
  cfg.blockDim = dim3(kBnThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t bn_launch_columns(const BnParams& p, cudaStream_t stream) {
  const int64_t W = p.C * p.S;
  const int64_t nrb = (p.N + kBnColRows - 1) / kBnColRows;
  const unsigned gx = static_cast<unsigned>((W + kBnThreads - 1) / kBnThreads);
  const unsigned gy_stats = static_cast<unsigned>(nrb < 65535 ? nrb : 65535);
  cudaError_t e = bn_launch_one(&bn_col_stats_kernel<kBnThreads, kBnColRows>,
                                dim3(gx, gy_stats, 1), stream, p);
  if (e != cudaSuccess) return e;
  e = bn_launch_one(&bn_col_merge_kernel<kBnThreads>, dim3(static_cast<unsigned>(p.C), 1, 1),
                    stream, p);
  if (e != cudaSuccess) return e;
  // enough row groups per column tile to fill the GPU
  const int64_t want = (static_cast<int64_t>(device_info().sm_count) * 8 + gx - 1) / gx;
  const int64_t gy = want < p.N ? (want < 65535 ? want : 65535) : p.N;
  return bn_launch_one(&bn_col_apply_kernel<kBnThreads>,
                       dim3(gx, static_cast<unsigned>(gy > 0 ? gy : 1), 1), stream, p);
}

// Column grid for short runs: THREADS columns per CTA, enough row groups to
// fill the GPU.
static dim3 bn_col_grid(const BnParams& p) {
  const int64_t W = p.C * p.S;
  const unsigned gx = static_cast<unsigned>((W + kBnThreads - 1) / kBnThreads);
  const int64_t want = (static_cast<int64_t>(device_info().sm_count) * 8 + gx - 1) / gx;
  const int64_t gy = want < p.N ? (want < 65535 ? want : 65535) : p.N;
  return dim3(gx > 0 ? gx : 1, static_cast<unsigned>(gy > 0 ? gy : 1), 1);
}

cudaError_t bn_launch_columns_local_stats(const BnParams& p, cudaStream_t stream) {
  const int64_t W = p.C * p.S;
  const int64_t nrb = (p.N + kBnColRows - 1) / kBnColRows;
  const unsigned gx = static_cast<unsigned>((W + kBnThreads - 1) / kBnThreads);
  cudaError_t e = bn_launch_one(&bn_col_stats_kernel<kBnThreads, kBnColRows>,
                                dim3(gx, static_cast<unsigned>(nrb < 65535 ? nrb : 65535), 1),
                                stream, p);
  if (e != cudaSuccess) return e;
  BnParams q = p;   // the channel's partials are contiguous: [c][S * row blocks]
  q.stats = p.partials;
  q.stats_cstride = p.S * nrb;
  q.stats_istride = 1;
  q.stats_count = p.S * nrb;
  return bn_launch_one(&bn_merge_kernel<kBnThreads>, dim3(static_cast<unsigned>(p.C), 1, 1),
                       stream, q);
}

cudaError_t bn_launch_columns_apply_stats(const BnParams& p, cudaStream_t stream) {
  return bn_launch_one(&bn_col_apply_stats_kernel<kBnThreads>, bn_col_grid(p), stream, p);
}

cudaError_t bn_launch_local_stats(const BnParams& p, cudaStream_t stream) {
  cudaError_t e = bn_launch_stats(p, stream);
  if (e != cudaSuccess) return e;
  return bn_launch_one(&bn_merge_kernel<kBnThreads>, dim3(static_cast<unsigned>(p.C), 1, 1),
                       stream, p);
}

cudaError_t bn_launch_eval(const BnParams& p, cudaStream_t stream) {
  if (p.S >= kBnEvalFlatBelow) {
    const dim3 grid(static_cast<unsigned>(p.N * p.chunks), static_cast<unsigned>(p.C), 1);
    if (p.vec && p.split) {
      static std::atomic<bool> done[64];
      const cudaError_t e = allow_smem(&bn_eval_staged_kernel<kBnThreads>, kBnStageBytes, done);
      if (e != cudaSuccess) return e;
      return bn_launch_one(&bn_eval_staged_kernel<kBnThreads>, grid, stream, p, kBnStageBytes);
    }
    return p.vec ? bn_launch_one(&bn_eval_kernel<kBnThreads, kBnUnroll, true>, grid, stream, p)
                 : bn_launch_one(&bn_eval_kernel<kBnThreads, kBnUnroll, false>, grid, stream, p);
  }
  if (p.S <= kBnColMaxS) {
    const int64_t W = p.C * p.S;
    const unsigned gx = static_cast<unsigned>((W + kBnThreads - 1) / kBnThreads);
    const int64_t want = (static_cast<int64_t>(device_info().sm_count) * 8 + gx - 1) / gx;
    const int64_t gy = want < p.N ? (want < 65535 ? want : 65535) : p.N;
    return bn_launch_one(&bn_eval_col_kernel<kBnThreads>,
                         dim3(gx, static_cast<unsigned>(gy > 0 ? gy : 1), 1), stream, p);
  }
  const int64_t units = p.N * p.C * (p.vec ? p.S / 4 : p.S);
  const int64_t cap = static_cast<int64_t>(device_info().sm_count) * (2048 / kBnThreads);
  int64_t blocks = (units + kBnThreads - 1) / kBnThreads;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid(static_cast<unsigned>(blocks), 1, 1);
  return p.vec ? bn_launch_one(&bn_eval_flat_kernel<kBnThreads, true>, grid, stream, p)
               : bn_launch_one(&bn_eval_flat_kernel<kBnThreads, false>, grid, stream, p);
}

cudaError_t bn_launch_apply(const BnParams& p, cudaStream_t stream) {
  return bn_launch_apply_pass(p, stream);
}

}  // namespace fnorm
