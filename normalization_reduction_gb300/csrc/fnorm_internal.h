// fnorm_internal.h -- host-side contract between the C ABI (fnorm_api.cu)
// and the kernel translation units: parameter blocks, launch plans and the
// launcher entry points each kernel file defines.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fnorm.h"

namespace fnorm {

// Device error word codes (kernels OR them into the word the host passes in).
constexpr unsigned kErrTimeout = 1u;

// ---------------------------------------------------------------- InstanceNorm
struct InParams {
  const void* x;
  void* y;
  int64_t NC;
  int64_t S;
  float eps;
  float* mean_out;
  float* rstd_out;
  unsigned* err;
  const float* gamma;   // [C] per-channel scale (nullptr: 1)
  const float* beta;    // [C] per-channel shift (nullptr: 0)
  int64_t C;            // channels: slice q belongs to channel q % C
  int debug_timeout;    // test hook (split kernel): wait on an mbarrier nobody completes
};

enum class InPath : int {
  kGroup = 0,     // G lanes per slice, slice held in registers (short slices)
  kResident = 1,  // one CTA or one cluster of CTAs per slice, slice held in registers
  kStream = 2,    // one cluster per slice, two reads (statistics, then normalise)
  kSplit = 3,     // one CTA or cluster per slice, chunk split between shared memory (TMA,
                  // prefetched) and registers; st.async cluster exchange
};

struct InPlan {
  InPath path;
  bool vec;      // 16-byte vector access (else element-wise)
  int threads;   // CTA size
  int nv;        // 16-byte slots per thread (group / resident), register slots (split)
  int ns;        // staged (shared-memory) slots per thread (split)
  int group;     // lanes per slice (group path)
  int cluster;   // CTAs per slice (resident / stream); 1 = no cluster
  int grid;      // CTAs to launch (0: the launcher sizes the persistent grid)
  bool packed;   // split path, bf16 input, cluster > 8: packed pair arithmetic
};

// Launch plans the kernel files provide, listed so the dispatcher can choose
// among them: resident (threads, nv) and group (group, nv) shapes.
constexpr int kResidentShapes[][2] = {{128, 4}, {256, 4}, {256, 8}, {512, 8}, {1024, 8}};
// Split shapes: (threads, register slots, staged slots) per thread.
constexpr int kSplitShapes[][3] = {{128, 8, 8}, {256, 8, 8}, {512, 8, 8}, {1024, 8, 8},
                                   {64, 8, 0},  {128, 8, 0}, {256, 8, 0}, {512, 8, 0},
                                   {1024, 8, 0}};
constexpr int kGroupShapes[][2] = {{8, 1}, {8, 4}, {32, 2}, {32, 4}, {32, 8}};
constexpr int kStreamThreads = 512;
constexpr int kStreamUnroll = 4;       // 16-byte loads per thread per tile (many slices)
constexpr int kStreamUnrollFew = 8;    // ... when few slices keep few CTAs busy
constexpr int kMaxCluster = 16;

// Defined in in_kernels.cuh and instantiated per (Tin, Tout) in in_*.cu.
// in_launch_t returns the launch's error code; in_max_active_clusters_t the
// largest number of co-resident clusters (CTAs for cluster size 1) of the plan
// on the current device, 0 if the plan cannot run.
template <class Tin, class Tout>
cudaError_t in_launch_t(const InParams& p, const InPlan& plan, cudaStream_t stream);
template <class Tin, class Tout>
int in_max_active_clusters_t(const InPlan& plan);

// ---------------------------------------------------------------- Epilogue
struct EpiParams {
  const float* x;
  const float* m;
  float* y;
  int64_t* argmax;
  int64_t N;
  int64_t C;
  int64_t S;
  float eps;
  float lo;
  float hi;
  int64_t per;         // position vectors (of 4) per CTA (range path)
  int debug_timeout;   // test hook: wait on an mbarrier nobody completes
  int keep;            // position vectors per channel kept in shared memory between passes (L2 path)
  unsigned* err;
};

enum class EpiPath : int { kStream = 1, kRangeL2 = 2 };

struct EpiPlan {
  EpiPath path;
  int threads;
  int cluster;
  int64_t per;
  bool want_arg;
  size_t smem;   // dynamic shared memory bytes
  int grid;      // CTAs (multiple of cluster)
  int keep;      // L2 path: position vectors per channel kept on chip
  bool onepass;  // L2 path: shifted lane sums for the statistics (per <= kEpiOnePassMaxPer)
};

constexpr int kEpiThreads = 256;
constexpr int kEpiStreamCluster = 8;
constexpr int kEpiMaxChannels = 8192;

cudaError_t epi_launch(const EpiParams& p, const EpiPlan& plan, cudaStream_t stream);
int epi_max_active_clusters(const EpiPlan& plan);
size_t epi_range_l2_smem(int64_t C, int cluster, int keep);
// L2 path: the leading position vectors of each channel of a CTA's range that
// stay in shared memory from the statistics pass to the output pass: as many
// as fit kEpiSmemBudget (118 for 16 channels in 4-CTA clusters), at most
// kEpiKeepMax (compiled in for that case).
constexpr int kEpiKeepMax = 118;
// L2 path: CTA ranges of at most this many position vectors (at most 40 per
// lane, 160 values) take the shifted one-pass lane sums for the statistics.
constexpr int64_t kEpiOnePassMaxPer = 1280;
// L2 path: dynamic shared memory per CTA, kept part included, such that four
// CTAs per SM (with their static shared memory and the 1 KB per CTA the
// system reserves) fit the 132 KB shared-memory carveout; the rest of the
// SM's 256 KB stays L1, which this kernel's loads need in flight (page's
// shape: 28.7 us per call keeping 160 vectors per channel with a 196 KB
// carveout, 28.1 us keeping 118; 96 or 64 kept, same carveout: 28.8 us).
constexpr int kEpiSmemBudget = 33 * 1024 - 1024 - 64;
size_t epi_stream_smem(int64_t C, int cluster);

// ---------------------------------------------------------------- BatchNorm
struct BnParams {
  const float* x;
  float* y;
  const float* gamma;
  const float* beta;
  float scale;
  float* running_mean;
  float* running_var;
  float momentum;
  float eps;
  float* save_mean;
  float* save_rstd;
  int64_t N;
  int64_t C;
  int64_t S;
  int64_t chunk;        // elements of one (n,c) run one CTA reduces
  int64_t chunks;       // chunks per run
  float4* partials;     // [C][N*chunks] (count, mean, M2, -)
  // Statistics the apply pass merges for channel c: stats[c*stats_cstride +
  // i*stats_istride] for i < stats_count. Local: the partials (cstride =
  // N*chunks, istride = 1). Multi-rank: gathered [R][C] (cstride 1, istride C).
  const float4* stats;
  int64_t stats_cstride;
  int64_t stats_istride;
  int64_t stats_count;
  float4* local_out;    // [C] merged local statistics (local-stats call), else null
  // Strided placement, for InstanceNorm on few long slices with the output
  // buffer as scratch (zero: the workspace layouts above). The partial of unit
  // (c, n, k) goes to partials[c * part_cstride + (n * chunks + k) * part_kstride];
  // the merge writes local_copies copies of channel c's statistics to
  // local_out[c * local_cstride + i * local_kstride]; the apply pass reads
  // unit (c, n, k)'s statistics from stats + c * stats_cstride + (n * chunks +
  // k) * stats_kstride.
  int64_t part_cstride;
  int64_t part_kstride;
  int64_t local_cstride;
  int64_t local_kstride;
  int64_t local_copies;
  int64_t stats_kstride;
  // gamma/beta index of BatchNorm channel c: c % affine_period (InstanceNorm
  // as a BatchNorm over [1, N*C, S]: slice q takes gamma[q % C]); 0: c
  int64_t affine_period;
  unsigned* grid_counter;  // resident kernel: grid-barrier arrivals (zeroed before the launch)
  bool vec;
  bool split;           // statistics pass by the register + TMA-staged kernel (vector mode)
  int debug_timeout;    // test hook (staged kernels): wait on an mbarrier nobody completes
  unsigned* err;
};

constexpr int kBnThreads = 256;
constexpr int kBnUnroll = 4;        // apply pass: 16-byte loads per thread per tile
constexpr int kBnStatsUnroll = 8;   // statistics pass
constexpr int64_t kBnChunk = 16384;   // elements per CTA in the two streaming passes
constexpr int kBnSplitRegs = 8;     // split statistics kernel: vectors per thread in registers
constexpr int kBnSplitStaged = 8;   // ... and in TMA-staged shared memory (a whole kBnChunk unit)
static_assert(kBnThreads * (kBnSplitRegs + kBnSplitStaged) * 4 >= kBnChunk,
              "a unit must fit the split statistics kernel");

cudaError_t bn_launch(const BnParams& p, cudaStream_t stream);          // stats + apply
cudaError_t bn_launch_local_stats(const BnParams& p, cudaStream_t stream);  // stats + merge
cudaError_t bn_launch_apply(const BnParams& p, cudaStream_t stream);         // apply only
cudaError_t bn_launch_eval(const BnParams& p, cudaStream_t stream);          // eval mode, one pass
// Short runs (S <= kBnColMaxS): column statistics, channel merge, apply. Uses
// p.partials ([C*S][row blocks]) and p.local_out ([C] coefficients).
cudaError_t bn_launch_columns(const BnParams& p, cudaStream_t stream);
cudaError_t bn_launch_columns_local_stats(const BnParams& p, cudaStream_t stream);
cudaError_t bn_launch_columns_apply_stats(const BnParams& p, cudaStream_t stream);
constexpr int64_t kBnColMaxS = 16;   // runs this short take the column form (training)
constexpr int kBnColRows = 32;       // rows per column-statistics partial
// Single cooperative launch (statistics, grid barrier, apply) keeping part of x
// on chip; returns cudaErrorCooperativeLaunchTooLarge when the grid cannot be
// co-resident (the caller then uses bn_launch).
cudaError_t bn_launch_resident(const BnParams& p, cudaStream_t stream);

// fnorm_batchnorm_train's argument checks other than the workspace's (see
// fnorm_api.cu); *total receives N*C*S.
fnorm_status bn_train_check(const float* x, const float* y, const float* gamma,
                            const float* beta, float scale, const float* running_mean,
                            const float* running_var, float momentum, float eps,
                            const float* save_mean, const float* save_rstd, int64_t N, int64_t C,
                            int64_t S, int64_t* total);
constexpr int64_t kBnEvalFlatBelow = 1024;   // runs shorter than this take the flat eval kernel

// ---------------------------------------------------------------- helpers
struct DeviceInfo {
  int sm_count;
  int max_smem_optin;
  int cluster_launch;
};
const DeviceInfo& device_info();   // current device, cached

}  // namespace fnorm
