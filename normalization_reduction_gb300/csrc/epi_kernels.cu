// epi_kernels.cu -- the fused post-convolution epilogue
//   y[n,s] = max_c  m_c * clamp(InstanceNorm(x[n,c,:] * m_c)[s], lo, hi)
// (page Kimi-K2.6__l2_p79, block 1: multiply by the per-channel multiplier,
// InstanceNorm3d over D*H*W, clamp to [-1, 1], multiply again, max over the
// channel dimension; output [N, D, H, W]).
//
// The page plans two kernels (per-(n,c) statistics, then one thread per output
// position looping over channels), which reads the convolution output twice
// from HBM. Here one launch does both: a thread-block cluster owns a sample n,
// and CTA r of the cluster owns a contiguous range of output positions FOR
// ALL C CHANNELS. The statistics are formed on x and the multiplier is folded
// in exactly by the affine identity
//   IN(m x) = (x - mean_x) * m / sqrt(m^2 var_x + eps),
// so z_c = m_c * clamp((x - mean_x) * a_c, lo, hi) with a_c = m_c*rsqrt(m_c^2 var_x + eps).
// Kernels (the plan picks the first that applies):
//  * epi_range_l2_kernel (default; 16-byte aligned, S % 4 == 0): each warp
//    reduces some channels over the CTA's range from HBM (per-lane sums
//    shifted by the lane's first value for ranges of at most
//    kEpiOnePassMaxPer vectors, exact two-pass register tiles beyond; Chan
//    merges), keeping the first KS vectors of each channel's range in shared
//    memory; the C partials are pushed with st.async into every CTA of the
//    cluster (completing on the receiver's mbarrier, all CTAs merge in rank
//    order: bit-identical results); the output pass takes the kept vectors
//    from shared memory and re-reads the rest of the range, which the
//    statistics pass has just brought into L2 (the whole input of the page's
//    shape, 103 MB, fits in L2), and writes max_c z_c (+ argmax; without the
//    index the clamp is a saturating FMA and channels go in pairs through a
//    three-input max).
//  * epi_stream_kernel (inputs that are not 16-byte aligned or too wide):
//    one cluster per sample, CTAs owning whole channels, each slice read twice
//    with element-wise loads.
#include "fnorm_device.cuh"
#include "fnorm_internal.h"
#include "in_kernels.cuh"

namespace fnorm {

// Instrumented builds only (build.py --phases defines FNORM_PHASE_TRACE; the
// product library has none of this): thread 0 of each of the first
// kEpiPhaseCtas CTAs of the L2-form kernel records the %globaltimer value at
// each phase boundary of its first sample -- start, statistics done, partials
// exchanged, coefficients formed, kept part written, sample done -- into
// g_epi_phase[cta][phase], read by fnorm_phase_trace_read (each launch
// overwrites the previous one's stamps).
#ifdef FNORM_PHASE_TRACE
constexpr int kEpiPhases = 6;
constexpr int kEpiPhaseCtas = 2048;
__device__ unsigned long long g_epi_phase[kEpiPhaseCtas * kEpiPhases];
#define FNORM_EPI_STAMP(k)                                                      \
  if (tid == 0 && it == 0 && blockIdx.x < kEpiPhaseCtas)                      \
    g_epi_phase[blockIdx.x * kEpiPhases + (k)] = globaltimer_ns();
#else
#define FNORM_EPI_STAMP(k)
#endif

size_t epi_range_l2_smem(int64_t C, int cluster, int keep) {
  return static_cast<size_t>(C) * 16 + 2 * static_cast<size_t>(C) * cluster * 16 +
         static_cast<size_t>(C) * keep * 16 + ((static_cast<size_t>(C) * 4 + 15) & ~size_t(15));
}

size_t epi_stream_smem(int64_t C, int cluster) {
  return static_cast<size_t>(C) * 16 + static_cast<size_t>((C + cluster - 1) / cluster) * 16;
}

__device__ __forceinline__ float epi_z(float v, const float4& cf, float lo, float hi) {
  return cf.z * fminf(fmaxf((v - cf.x) * cf.y, lo), hi);
}

// Channel coefficients (mean_x, a_c, m_c) from a channel's statistic.
__device__ __forceinline__ float4 epi_coef(const Stat& s, float mc, float eps) {
  const float var = s.m2 / s.n;
  return make_float4(s.mean, mc * rsqrtf(mc * mc * var + eps), mc, 0.f);
}

__device__ __forceinline__ void epi_update(float z, int c, float& best, int& arg) {
  if (z > best) {
    best = z;
    arg = c;
  }
}

// Per-channel output coefficients: z_c = clamp(x*A + B, lo_c, hi_c) with
// A = m_c*a_c, B = -mean_x*A, and (lo_c, hi_c) = m_c*(lo, hi) ordered for the
// sign of m_c -- the same value as m_c*clamp((x - mean_x)*a_c, lo, hi) since
// multiplying by m_c is monotone (order-reversing for m_c < 0).
__device__ __forceinline__ float4 epi_out_coef(const Stat& s, float mc, float eps, float lo,
                                               float hi) {
  const float var = s.m2 / s.n;
  const float A = mc * (mc * rsqrtf(mc * mc * var + eps));
  const float l = mc * lo, h = mc * hi;
  return make_float4(A, -s.mean * A, fminf(l, h), fmaxf(l, h));
}

__device__ __forceinline__ float epi_zc(float v, const float4& k) {
  return fminf(fmaxf(fmaf(v, k.x, k.y), k.z), k.w);
}

// Range kernel, L2 form: a cluster per sample, CTA r owning a range of
// positions of all channels, st.async exchange of the per-channel partials.
// The statistics pass streams x from
// HBM with 128-bit loads, 8 per lane in flight, leaving it in L2; the output
// pass reads the CTA's range again from L2 (4 channels' loads in flight per
// thread). For the page's shape a sample is 806 KB and the whole input
// 103 MB, below the 126 MB L2; with 256-thread CTAs in 4-CTA clusters every
// sample's cluster is resident at once, so HBM still sees one read of x.
// 16-byte load cached in L2 only (ld.global.cg): the statistics pass's reads
// of x. Measured on the page's shape with 160 vectors kept per channel (60 KB
// of L1): 28.7 against 29.0 us per call with the read-only path (__ldg); with
// the current 118 (124 KB of L1) the two measure the same. The output pass
// keeps its streaming loads (.cg there was slower: 31.6 us), and loads that
// skip the L1 allocation were slower in either pass (34.4 us).
__device__ __forceinline__ uint4 ld_v4_l2(const void* p) {
  uint4 v;
  asm("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

template <bool WANT_ARG>
__device__ __forceinline__ void epi_take(const uint4& u, const float4& k, int c, float (&best)[4],
                                         int (&arg)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float z = epi_zc(Elem<float>::get(u, j), k);
    if (WANT_ARG) {
      if (z > best[j]) {
        best[j] = z;
        arg[j] = c;
      }
    } else {
      best[j] = fmaxf(best[j], z);
    }
  }
}

// Shifted sums of one lane's fp32 values: with K the lane's first value,
// d = x - K, S = sum d, Q = sum d^2, the lane's statistics are mean = K + S/n,
// M2 = Q - S^2/n. K is one of the values, so (K - mean)^2 <= M2 and
// Q <= (n + 1) M2: the cancellation grows with n, which the plan bounds
// (kEpiOnePassMaxPer vectors per CTA range, at most 160 values per lane; longer
// ranges take exact two-pass tiles). Three floating-point operations per value
// instead of the four of an exact two-pass tile plus a merge per tile, issued
// as pairs (__fadd2_rn / __ffma2_rn, two fp32 lanes per instruction);
// x - K is x + (-K), which is exact.
struct LaneSums {
  float2 s01, s23, q01, q23;
  float2 nk;   // (-K, -K)
  int cnt;     // vectors accumulated
};

__device__ __forceinline__ LaneSums lane_sums_begin(float K) {
  LaneSums a;
  a.s01 = a.s23 = a.q01 = a.q23 = make_float2(0.f, 0.f);
  a.nk = make_float2(-K, -K);
  a.cnt = 0;
  return a;
}

// Adds r's values (cnt is counted by the caller).
__device__ __forceinline__ void lane_sums_acc(LaneSums& a, const uint4& r) {
  const float2 d01 = __fadd2_rn(make_float2(__uint_as_float(r.x), __uint_as_float(r.y)), a.nk);
  const float2 d23 = __fadd2_rn(make_float2(__uint_as_float(r.z), __uint_as_float(r.w)), a.nk);
  a.s01 = __fadd2_rn(a.s01, d01);
  a.s23 = __fadd2_rn(a.s23, d23);
  a.q01 = __ffma2_rn(d01, d01, a.q01);
  a.q23 = __ffma2_rn(d23, d23, a.q23);
}

__device__ __forceinline__ Stat lane_sums_stat(const LaneSums& a) {
  if (a.cnt == 0) return stat_empty();
  const float n = 4.f * static_cast<float>(a.cnt);
  const float S = (a.s01.x + a.s01.y) + (a.s23.x + a.s23.y);
  const float Q = (a.q01.x + a.q01.y) + (a.q23.x + a.q23.y);
  return Stat{n, S / n - a.nk.x, fmaxf(Q - S * (S / n), 0.f)};
}

// max(a, b, c) in one instruction (three-input max); like fmaxf it ignores a
// NaN operand, so it equals fmaxf(fmaxf(a, b), c).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Saturating form of the clamp, for the output without the index: with
// w = h - l, min(max(v A + B, l), h) = l + w sat(v A/w + (B - l)/w), where sat
// clamps to [0, 1] in the fused multiply-add (and maps NaN to 0, as the
// min/max form maps it to l); w = 0 gives l. Two instructions per value
// instead of three; the value may differ from the min/max form in the last
// bits (the rounding of A/w and (B - l)/w, and of the second FMA).
__device__ __forceinline__ float4 epi_sat_coef(const float4& k) {
  const float w = k.w - k.z;
  if (!(w > 0.f)) return make_float4(0.f, 0.f, k.z, 0.f);
  return make_float4(k.x / w, (k.y - k.z) / w, k.z, w);
}

__device__ __forceinline__ float epi_zsat(float v, const float4& k) {
  float t;
  asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(t) : "f"(v), "f"(k.x), "f"(k.y));
  return fmaf(t, k.w, k.z);
}

// best = max(best, z_a, z_b) for two channels (saturating coefficients).
__device__ __forceinline__ void epi_take_pair_sat(const uint4& ua, const float4& ka, const uint4& ub,
                                                  const float4& kb, float (&best)[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j)
    best[j] = fmax3(best[j], epi_zsat(Elem<float>::get(ua, j), ka), epi_zsat(Elem<float>::get(ub, j), kb));
}

// z of one channel: the min/max clamp with the index, the saturating one without.
template <bool WANT_ARG>
__device__ __forceinline__ float epi_z(float v, const float4& k) {
  return WANT_ARG ? epi_zc(v, k) : epi_zsat(v, k);
}

template <bool WANT_ARG>
__device__ __forceinline__ void epi_take_any(const uint4& u, const float4& k, int c, float (&best)[4],
                                             int (&arg)[4]) {
  if (WANT_ARG) {
    epi_take<true>(u, k, c, best, arg);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) best[j] = fmaxf(best[j], epi_zsat(Elem<float>::get(u, j), k));
  }
}

// KEEP >= 0 fixes the kept vectors per channel at compile time (the common
// full-size case); KEEP < 0 takes p.keep. ONEPASS selects the shifted lane
// sums for the statistics (ranges of at most kEpiOnePassMaxPer vectors), else
// exact two-pass tiles.
template <int THREADS, bool WANT_ARG, int KEEP, bool ONEPASS>
__global__ void __launch_bounds__(THREADS, 4) epi_range_l2_kernel(const EpiParams p) {
  extern __shared__ __align__(16) float4 dyn[];
  __shared__ __align__(8) uint64_t xbar[2];
  __shared__ __align__(8) uint64_t dbg_bar;
  constexpr int NWARP = THREADS / 32;
  constexpr int U = 8;    // 16-byte loads per lane per statistics tile
  constexpr int G = 4;    // channels loaded together in the output pass
  const int64_t S = p.S;
  const int C = static_cast<int>(p.C);
  const int64_t per = p.per;
  const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
  const unsigned cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float4* coef = dyn;          // [C]
  float4* slots = dyn + C;     // [2][C][csize]
  // [C][KS]: the first KS position vectors of each channel of the range, kept
  // from the statistics pass for the output pass (fewer L2 re-reads)
  uint4* keep = reinterpret_cast<uint4*>(slots + 2 * C * csize);
  const int KS = KEEP >= 0 ? KEEP : p.keep;
  float* mloc = reinterpret_cast<float*>(keep + static_cast<size_t>(C) * KS);   // [C]
  const int64_t nv4 = S / 4;
  const int64_t v0 = per * crank;
  const int vr = static_cast<int>(v0 < nv4 ? (nv4 - v0 < per ? nv4 - v0 : per) : 0);

  if (tid == 0) {
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  if (csize > 1) cluster_sync();
  else __syncthreads();
  pdl_wait();
  // The next launch may be scheduled once every CTA of this grid has started
  // (the grid never exceeds the co-resident capacity); its CTAs take free
  // slots and wait in griddepcontrol.wait, which hides its launch.
  pdl_trigger();
  for (int c = tid; c < C; c += THREADS) mloc[c] = __ldg(p.m + c);   // read after the barriers below

  bool xfailed = false;
  int it = 0;
  for (int64_t n = cid; n < p.N; n += ncl, ++it) {
    const int b = it & 1;
    float4* sl = slots + size_t(b) * C * csize;
    if (tid == 0) mbar_arrive_expect_tx(&xbar[b], static_cast<unsigned>(C) * csize * 16u);
    FNORM_EPI_STAMP(0)
    const uint4* xn = reinterpret_cast<const uint4*>(p.x + n * C * S) + v0;
    for (int c = warp; c < C; c += NWARP) {
      const uint4* xc = xn + int64_t(c) * nv4 + lane;
      Stat acc = stat_empty();
      LaneSums ls = lane_sums_begin(
          ONEPASS && lane < vr ? __ldg(reinterpret_cast<const float*>(xc)) : 0.f);
      int t = 0;
      for (; t + 32 * U <= vr; t += 32 * U) {   // full tiles
        uint4 r[U];
#pragma unroll
        for (int u = 0; u < U; ++u) r[u] = ld_v4_l2(xc + t + u * 32);
        if (t == 0) {
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (u * 32 + lane < KS) keep[c * KS + u * 32 + lane] = r[u];
        }
        if (ONEPASS) {
#pragma unroll
          for (int u = 0; u < U; ++u) lane_sums_acc(ls, r[u]);
          ls.cnt += U;
        } else {
          acc = chan_merge(acc, tile_stat_full<float, U>(r));
        }
      }
      if (vr - t > 4 * 32) {                     // long ragged tail: one predicated tile
        uint4 r[U];
        int nvalid = 0;
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const bool v = t + u * 32 + lane < vr;
          r[u] = v ? ld_v4_l2(xc + t + u * 32) : make_uint4(0, 0, 0, 0);
          nvalid += v ? 4 : 0;
          if (t == 0 && v && u * 32 + lane < KS) keep[c * KS + u * 32 + lane] = r[u];
        }
        if (ONEPASS) {
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (t + u * 32 + lane < vr) {
              lane_sums_acc(ls, r[u]);
              ++ls.cnt;
            }
        } else {
          acc = chan_merge(acc, tile_stat<float, U>(r, nvalid));
        }
        t = vr;
      }
      for (; t < vr; t += 32) {                  // short tail: one vector per lane
        const bool v = t + lane < vr;
        uint4 r1[1];
        r1[0] = v ? ld_v4_l2(xc + t) : make_uint4(0, 0, 0, 0);
        if (v && t + lane < KS) keep[c * KS + t + lane] = r1[0];
        if (ONEPASS) {
          if (v) {
            lane_sums_acc(ls, r1[0]);
            ++ls.cnt;
          }
        } else {
          acc = chan_merge(acc, tile_stat<float, 1>(r1, v ? 4 : 0));
        }
      }
      if (ONEPASS) acc = lane_sums_stat(ls);
      acc = warp_merge<32>(acc);
      const float4 v = make_float4(__shfl_sync(kFullMask, acc.n, 0), __shfl_sync(kFullMask, acc.mean, 0),
                                   __shfl_sync(kFullMask, acc.m2, 0), 0.f);
      for (unsigned rr = lane; rr < csize; rr += 32)
        st_async_v4(&sl[size_t(c) * csize + crank], &xbar[b], rr, v);
    }
    // Warps park at the CTA barrier while one warp waits for the partials.
    __syncthreads();
    FNORM_EPI_STAMP(1)
    bool ok = true;
    if (warp == 0 && !xfailed)
      ok = mbar_wait_bounded(&xbar[b], (static_cast<unsigned>(it) >> 1) & 1u, p.err);
    if (__syncthreads_or(!ok)) xfailed = true;
    FNORM_EPI_STAMP(2)
    // Channel coefficients: segments of W lanes (W = csize rounded up to a
    // power of two) each merge one channel's csize partials in a fixed tree
    // (the same bits in every CTA), so a warp does 32/W channels at once.
    {
      const int W = csize <= 2 ? 2 : csize <= 4 ? 4 : csize <= 8 ? 8 : 16;
      const int per_warp = 32 / W, seg = lane / W, r = lane - seg * W;
      for (int c0 = warp * per_warp; c0 < C; c0 += NWARP * per_warp) {
        const int c = c0 + seg;
        Stat s = stat_empty();
        if (c < C && r < static_cast<int>(csize)) {
          const float4 v = sl[size_t(c) * csize + r];
          s = Stat{v.x, v.y, v.z};
        }
        s = W == 2 ? warp_merge<2>(s) : W == 4 ? warp_merge<4>(s) : W == 8 ? warp_merge<8>(s)
                                                                        : warp_merge<16>(s);
        if (r == 0 && c < C) {
          const float4 k = epi_out_coef(s, mloc[c], p.eps, p.lo, p.hi);
          coef[c] = WANT_ARG ? k : epi_sat_coef(k);
        }
      }
    }
    __syncthreads();
    FNORM_EPI_STAMP(3)
    const int vk = vr < KS ? vr : KS;
    for (int v = tid; v < vk; v += THREADS) {   // positions kept on chip
      float best[4];
      int arg[4] = {0, 0, 0, 0};
      {
        const uint4 u = keep[v];
        const float4 k = coef[0];
#pragma unroll
        for (int j = 0; j < 4; ++j) best[j] = epi_z<WANT_ARG>(Elem<float>::get(u, j), k);
      }
      int c = 1;
      if (!WANT_ARG)
        for (; c + 2 <= C; c += 2)
          epi_take_pair_sat(keep[c * KS + v], coef[c], keep[(c + 1) * KS + v], coef[c + 1], best);
      for (; c < C; ++c) epi_take_any<WANT_ARG>(keep[c * KS + v], coef[c], c, best, arg);
      const int64_t pos = (v0 + v) * 4;
      __stcs(reinterpret_cast<float4*>(p.y + n * S + pos), make_float4(best[0], best[1], best[2], best[3]));
      if (WANT_ARG) {
        longlong2* ao = reinterpret_cast<longlong2*>(p.argmax + n * S + pos);
        __stcs(ao, make_longlong2(arg[0], arg[1]));
        __stcs(ao + 1, make_longlong2(arg[2], arg[3]));
      }
    }
    FNORM_EPI_STAMP(4)
    for (int v = vk + tid; v < vr; v += THREADS) {
      const uint4* xv = xn + v;
      float best[4];
      int arg[4] = {0, 0, 0, 0};
      {
        const uint4 u = __ldcs(xv);
        const float4 k = coef[0];
#pragma unroll
        for (int j = 0; j < 4; ++j) best[j] = epi_z<WANT_ARG>(Elem<float>::get(u, j), k);
      }
      int c = 1;
      for (; c + G <= C; c += G) {
        uint4 u[G];
#pragma unroll
        for (int g = 0; g < G; ++g) u[g] = __ldcs(xv + int64_t(c + g) * nv4);
        if (WANT_ARG) {
#pragma unroll
          for (int g = 0; g < G; ++g) epi_take<WANT_ARG>(u[g], coef[c + g], c + g, best, arg);
        } else {
#pragma unroll
          for (int g = 0; g < G; g += 2) epi_take_pair_sat(u[g], coef[c + g], u[g + 1], coef[c + g + 1], best);
        }
      }
      for (; c < C; ++c) epi_take_any<WANT_ARG>(__ldcs(xv + int64_t(c) * nv4), coef[c], c, best, arg);
      const int64_t pos = (v0 + v) * 4;
      __stcs(reinterpret_cast<float4*>(p.y + n * S + pos), make_float4(best[0], best[1], best[2], best[3]));
      if (WANT_ARG) {
        longlong2* ao = reinterpret_cast<longlong2*>(p.argmax + n * S + pos);
        __stcs(ao, make_longlong2(arg[0], arg[1]));
        __stcs(ao + 1, make_longlong2(arg[2], arg[3]));
      }
    }
    __syncthreads();   // coefficients consumed before the next sample rewrites them
    FNORM_EPI_STAMP(5)
  }
  pdl_trigger();
  if (csize > 1) cluster_sync();
  // Test hook, after the last cluster barrier so no peer waits on this CTA:
  // a wait on a barrier nothing completes must expire, record the timeout in
  // the error word and return.
  if (p.debug_timeout && cid == 0 && crank == 0) mbar_wait_bounded(&dbg_bar, 0, p.err);
}

// Fallback: cluster per sample, CTA rank r owns channels r, r+csize, ...;
// statistics by streaming each owned slice from global memory, then output
// positions split across the cluster, reading every channel again.
template <int THREADS>
__global__ void __launch_bounds__(THREADS) epi_stream_kernel(const EpiParams p) {
  extern __shared__ __align__(16) float4 dyn4[];
  __shared__ Stat warp_part[THREADS / 32];
  const int64_t S = p.S;
  const int C = static_cast<int>(p.C);
  const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
  const unsigned cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x;
  float4* coef = dyn4;       // [C]
  float4* loc = dyn4 + C;    // [ceil(C / csize)]
  constexpr int TILE = THREADS * 16;   // elements per tile: 16 per thread

  pdl_wait();
  for (int64_t n = cid; n < p.N; n += ncl) {
    for (int c = static_cast<int>(crank), jl = 0; c < C; c += csize, ++jl) {
      const float* xs = p.x + (n * C + c) * S;
      Stat acc = stat_empty();
      for (int64_t t0 = 0; t0 < S; t0 += TILE) {
        uint4 r[4];
        const int64_t e0 = t0 + tid;
        const int nvalid = e0 < S ? clamp_int((S - e0 + THREADS - 1) / THREADS, 0, 16) : 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          r[k] = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (k * 4 + j < nvalid)
              Elem<float>::set(r[k], j, __ldg(xs + e0 + static_cast<int64_t>(k * 4 + j) * THREADS));
        }
        acc = chan_merge(acc, tile_stat<float, 4>(r, nvalid));
      }
      const Stat cta = cta_merge<THREADS>(acc, warp_part);
      if (tid == 0) loc[jl] = epi_coef(cta, __ldg(p.m + c), p.eps);
      __syncthreads();
    }
    cluster_sync();
    for (int c = tid; c < C; c += THREADS) {
      const unsigned owner = c % csize;
      const int jl = c / csize;
      coef[c] = ld_dsmem_f4(dsmem_map(smem_u32(loc + jl), owner));
    }
    __syncthreads();
    const int64_t per = (S + csize - 1) / csize;
    const int64_t s0 = per * crank, s1 = (s0 + per < S) ? s0 + per : S;
    for (int64_t s = s0 + tid; s < s1; s += THREADS) {
      const float* xp = p.x + n * C * S + s;
      float best = epi_z(__ldg(xp), coef[0], p.lo, p.hi);
      int arg = 0;
      for (int c = 1; c < C; ++c) {
        const float z = epi_z(__ldg(xp + static_cast<int64_t>(c) * S), coef[c], p.lo, p.hi);
        if (z > best) { best = z; arg = c; }
      }
      p.y[n * S + s] = best;
      if (p.argmax) p.argmax[n * S + s] = arg;
    }
    cluster_sync();
  }
  pdl_trigger();
}

using EpiKernelFn = void (*)(EpiParams);

static EpiKernelFn epi_kernel(const EpiPlan& plan) {
  if (plan.threads != kEpiThreads) return nullptr;
  switch (plan.path) {
    case EpiPath::kRangeL2:
      if (plan.keep == kEpiKeepMax) {
        if (plan.onepass)
          return plan.want_arg ? &epi_range_l2_kernel<kEpiThreads, true, kEpiKeepMax, true>
                               : &epi_range_l2_kernel<kEpiThreads, false, kEpiKeepMax, true>;
        return plan.want_arg ? &epi_range_l2_kernel<kEpiThreads, true, kEpiKeepMax, false>
                             : &epi_range_l2_kernel<kEpiThreads, false, kEpiKeepMax, false>;
      }
      if (plan.onepass)
        return plan.want_arg ? &epi_range_l2_kernel<kEpiThreads, true, -1, true>
                             : &epi_range_l2_kernel<kEpiThreads, false, -1, true>;
      return plan.want_arg ? &epi_range_l2_kernel<kEpiThreads, true, -1, false>
                           : &epi_range_l2_kernel<kEpiThreads, false, -1, false>;
    case EpiPath::kStream: return &epi_stream_kernel<kEpiThreads>;
  }
  return nullptr;
}

static cudaError_t epi_prepare(EpiKernelFn fn, const EpiPlan& plan) {
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(plan.smem));
  if (e == cudaSuccess && plan.cluster > 8)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e;
}

int epi_max_active_clusters(const EpiPlan& plan) {
  EpiKernelFn fn = epi_kernel(plan);
  if (!fn || epi_prepare(fn, plan) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.cluster, 1, 1);
  cfg.blockDim = dim3(plan.threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t epi_launch(const EpiParams& p, const EpiPlan& plan, cudaStream_t stream) {
  EpiKernelFn fn = epi_kernel(plan);
  if (!fn) return cudaErrorInvalidConfiguration;
  cudaError_t e = epi_prepare(fn, plan);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid, 1, 1);
  cfg.blockDim = dim3(plan.threads, 1, 1);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace fnorm

#ifdef FNORM_PHASE_TRACE
// Instrumented builds only: copies the first n phase stamps (see
// g_epi_phase) to host memory; returns the CUDA error code.
extern "C" __attribute__((visibility("default"))) int fnorm_phase_trace_read(
    unsigned long long* out, int n) {
  if (n > fnorm::kEpiPhaseCtas * fnorm::kEpiPhases) n = fnorm::kEpiPhaseCtas * fnorm::kEpiPhases;
  return static_cast<int>(
      cudaMemcpyFromSymbol(out, fnorm::g_epi_phase, sizeof(unsigned long long) * n));
}
#endif
