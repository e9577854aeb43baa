// epi_kernels.cu -- the fused post-convolution epilogue
//   y[n,s] = max_c  m_c * clamp(InstanceNorm(x[n,c,:] * m_c)[s], lo, hi)
// (page Kimi-K2.6__l2_p79, block 1: multiply by the per-channel multiplier,
// InstanceNorm3d over D*H*W, clamp to [-1, 1], multiply again, max over the
// channel dimension; output [N, D, H, W]).
//
// The page plans two kernels (per-(n,c) statistics, then one thread per output
// position looping over channels), which reads the convolution output twice.
// Here one thread-block cluster owns one sample n:
//  * each CTA pulls the full slices of its cpc channels into shared memory with
//    TMA bulk copies (cp.async.bulk + mbarrier, bounded waits);
//  * it forms their statistics from shared memory (exact per-thread two-pass
//    over 16-value register tiles, Chan merges across tiles, warps and CTAs);
//  * after a cluster barrier every CTA reads the channel coefficients of all
//    CTAs and, for its share of the output positions, the C channel values at
//    each position through distributed shared memory, and writes the maximum
//    (and optionally its channel index) with 128-bit stores.
// HBM sees one read of x and one write of y. The statistics are formed on x,
// and the multiplier is folded in exactly by the affine identity
//   IN(m x) = (x - mean_x) * m / sqrt(m^2 var_x + eps),
// so z_c = m_c * clamp((x - mean_x) * a_c, lo, hi) with a_c = m_c*rsqrt(m_c^2 var_x + eps).
//
// A second kernel covers inputs that do not fit (or are not 16-byte aligned):
// the same cluster-per-sample structure, reading each slice twice from global
// memory with element-wise loads.
#include "fnorm_device.cuh"
#include "fnorm_internal.h"
#include "in_kernels.cuh"

namespace fnorm {

static __host__ __device__ __forceinline__ size_t align16(size_t v) { return (v + 15) & ~size_t(15); }

size_t epi_resident_smem(int64_t C, int64_t S, int cpc) {
  return align16(static_cast<size_t>(cpc) * S * sizeof(float)) + static_cast<size_t>(C) * 16 +
         static_cast<size_t>(cpc) * 16;
}

size_t epi_stream_smem(int64_t C, int cluster) {
  return static_cast<size_t>(C) * 16 + static_cast<size_t>((C + cluster - 1) / cluster) * 16;
}

__device__ __forceinline__ float epi_z(float v, const float4& cf, float lo, float hi) {
  return cf.z * fminf(fmaxf((v - cf.x) * cf.y, lo), hi);
}

// Channel coefficients (mean_x, a_c, m_c) from a CTA-level statistic.
__device__ __forceinline__ float4 epi_coef(const Stat& s, float mc, float eps) {
  const float var = s.m2 / s.n;
  return make_float4(s.mean, mc * rsqrtf(mc * mc * var + eps), mc, 0.f);
}

template <int THREADS>
__global__ void __launch_bounds__(THREADS) epi_resident_kernel(const EpiParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ Stat warp_part[THREADS / 32];
  __shared__ __align__(8) uint64_t bar;
  __shared__ __align__(8) uint64_t dbg_bar;

  const int64_t S = p.S;
  const int C = static_cast<int>(p.C);
  const int cpc = p.cpc;
  float* xs = reinterpret_cast<float*>(smem_raw);                                   // [cpc][S]
  float4* coef = reinterpret_cast<float4*>(smem_raw + align16(size_t(cpc) * S * 4));  // [C]
  float4* loc = coef + C;                                                            // [cpc]

  const unsigned crank = cluster_ctarank(), csize = cluster_nctarank();
  const unsigned cid = cluster_id_x(), ncl = ncluster_x();
  const int tid = threadIdx.x;
  const int c0 = static_cast<int>(crank) * cpc;
  const int nch = C - c0 < 0 ? 0 : (C - c0 < cpc ? C - c0 : cpc);
  const int64_t nv4 = S / 4;

  if (tid == 0) {
    mbar_init(&bar, 1);
    mbar_init(&dbg_bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Test hook: a wait on a barrier nothing completes must expire, record the
  // timeout and let the kernel carry on.
  if (p.debug_timeout && cid == 0 && crank == 0) mbar_wait_bounded(&dbg_bar, 0, p.err);

  bool failed = false;
  unsigned parity = 0;
  for (int64_t n = cid; n < p.N; n += ncl) {
    const float* xn = p.x + n * C * S;
    if (nch > 0 && !failed) {
      if (tid == 0) {
        mbar_arrive_expect_tx(&bar, static_cast<unsigned>(nch * S * 4));
        for (int j = 0; j < nch; ++j)
          tma_bulk_g2s(xs + j * S, xn + (c0 + j) * S, static_cast<unsigned>(S * 4), &bar);
      }
      const bool ok = mbar_wait_bounded(&bar, parity, p.err);
      failed = __syncthreads_or(!ok) != 0;
      if (!failed) parity ^= 1u;
    }

    // Statistics of this CTA's channels.
    for (int j = 0; j < nch; ++j) {
      const uint4* v4 = reinterpret_cast<const uint4*>(xs + j * S);
      Stat acc = stat_empty();
      for (int64_t i = tid; i < nv4; i += THREADS * 4) {
        uint4 r[4];
        int nvalid = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const bool v = i + u * THREADS < nv4;
          r[u] = v ? v4[i + u * THREADS] : make_uint4(0, 0, 0, 0);
          nvalid += v ? 4 : 0;
        }
        acc = chan_merge(acc, tile_stat<float, 4>(r, nvalid));
      }
      const Stat cta = cta_merge<THREADS>(acc, warp_part);
      if (tid == 0) loc[j] = epi_coef(cta, __ldg(p.m + c0 + j), p.eps);
      __syncthreads();
    }
    cluster_sync();

    // Every channel's coefficients, from the CTA that owns it.
    for (int c = tid; c < C; c += THREADS) {
      const int owner = c / cpc, j = c - owner * cpc;
      coef[c] = ld_dsmem_f4(dsmem_map(smem_u32(loc + j), owner));
    }
    __syncthreads();

    // Output positions [p0, p1) in units of 4.
    const int64_t per = (nv4 + csize - 1) / csize;
    const int64_t p0 = per * crank, p1 = (p0 + per < nv4) ? p0 + per : nv4;
    const uint32_t xs_base = smem_u32(xs);
    for (int64_t pv = p0 + tid; pv < p1; pv += THREADS) {
      float best[4];
      int arg[4];
      {
        const float4 v = ld_dsmem_f4(dsmem_map(xs_base + static_cast<uint32_t>(pv * 16), 0));
        const float4 cf = coef[0];
        best[0] = epi_z(v.x, cf, p.lo, p.hi);
        best[1] = epi_z(v.y, cf, p.lo, p.hi);
        best[2] = epi_z(v.z, cf, p.lo, p.hi);
        best[3] = epi_z(v.w, cf, p.lo, p.hi);
        arg[0] = arg[1] = arg[2] = arg[3] = 0;
      }
      int c = 1;
      // groups of four channels: issue the four remote loads, then compute
      for (; c + 4 <= C; c += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int cc = c + u, owner = cc / cpc, j = cc - owner * cpc;
          v[u] = ld_dsmem_f4(
              dsmem_map(xs_base + static_cast<uint32_t>((j * S + pv * 4) * 4), owner));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 cf = coef[c + u];
          const float z0 = epi_z(v[u].x, cf, p.lo, p.hi), z1 = epi_z(v[u].y, cf, p.lo, p.hi);
          const float z2 = epi_z(v[u].z, cf, p.lo, p.hi), z3 = epi_z(v[u].w, cf, p.lo, p.hi);
          if (z0 > best[0]) { best[0] = z0; arg[0] = c + u; }
          if (z1 > best[1]) { best[1] = z1; arg[1] = c + u; }
          if (z2 > best[2]) { best[2] = z2; arg[2] = c + u; }
          if (z3 > best[3]) { best[3] = z3; arg[3] = c + u; }
        }
      }
      for (; c < C; ++c) {
        const int owner = c / cpc, j = c - owner * cpc;
        const float4 v =
            ld_dsmem_f4(dsmem_map(xs_base + static_cast<uint32_t>((j * S + pv * 4) * 4), owner));
        const float4 cf = coef[c];
        const float z0 = epi_z(v.x, cf, p.lo, p.hi), z1 = epi_z(v.y, cf, p.lo, p.hi);
        const float z2 = epi_z(v.z, cf, p.lo, p.hi), z3 = epi_z(v.w, cf, p.lo, p.hi);
        if (z0 > best[0]) { best[0] = z0; arg[0] = c; }
        if (z1 > best[1]) { best[1] = z1; arg[1] = c; }
        if (z2 > best[2]) { best[2] = z2; arg[2] = c; }
        if (z3 > best[3]) { best[3] = z3; arg[3] = c; }
      }
      float* yo = p.y + n * S + pv * 4;
      *reinterpret_cast<float4*>(yo) = make_float4(best[0], best[1], best[2], best[3]);
      if (p.argmax) {
        longlong2* ao = reinterpret_cast<longlong2*>(p.argmax + n * S + pv * 4);
        ao[0] = make_longlong2(arg[0], arg[1]);
        ao[1] = make_longlong2(arg[2], arg[3]);
      }
    }
    // No CTA may overwrite (or release) shared memory another CTA still reads.
    cluster_sync();
  }
  if (failed && nch > 0) mbar_wait_bounded(&bar, parity, p.err);   // let copies in flight land
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
}

using EpiKernelFn = void (*)(EpiParams);

static EpiKernelFn epi_kernel(const EpiPlan& plan) {
  if (plan.threads != kEpiThreads) return nullptr;
  return plan.path == EpiPath::kResident ? &epi_resident_kernel<kEpiThreads>
                                         : &epi_stream_kernel<kEpiThreads>;
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, p);
}

}  // namespace fnorm
