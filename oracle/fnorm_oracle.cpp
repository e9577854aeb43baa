// fnorm_oracle.cpp -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
//
// A plain, slow, single-threaded float64 CPU statement of what libfnorm
// computes. Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg may load it. It shares no code, header, table or constant
// with the CUDA library, and it never reads anything the CUDA library wrote.
//
// Sources: three web pages, each an agent transcript about replacing a
// PyTorch forward with a CUDA kernel (titles as on the pages):
//   [p79] Kimi-K2.6__l2_p79 -- Conv3d -> x*m_c -> InstanceNorm3d ->
//         clamp[-1,1] -> x*m_c -> max over channels.
//   [p73] Kimi-K2.6__l2_p73 -- Conv2d -> BatchNorm2d -> x*2.0.
//   [p34] Kimi-K2.6__l1_p34 -- InstanceNorm2d(64).
// Each page is a sequence of reasoning blocks; "block k" counts them from 1.
//
// Functions: InstanceNorm (float64, fp32 and bf16 storage), InstanceNorm with
// per-channel affine parameters, the fused epilogue of [p79], BatchNorm in
// training mode with running statistics and in eval mode (both followed by
// the scale of [p73]), and bf16 rounding helpers. Each is pinned by the test
// suite's pins (no function is "parity unpinned").
//
// Every result is the plain definition evaluated in float64 with the inputs
// taken exactly (fp32 and bf16 values are exact in float64) and rounded once
// to the output type at the end. Mean and variance use the textbook two-pass
// form: mean first, then the mean of squared deviations.
//
// Compile with -ffp-contract=off so that x86 and Arm hosts round alike.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------
// Storage conversions. bf16 is the upper half of an IEEE binary32.
// ---------------------------------------------------------------------------
double bf16_to_double(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Round a float64 value to the nearest bf16 value, ties to even, in a single
// rounding step (no detour through binary32). bf16 keeps 8 significant bits;
// its smallest normal is 2^-126 and its subnormal spacing is 2^-133.
uint16_t double_to_bf16(double v) {
  if (std::isnan(v)) return 0x7FC0;
  const uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  const double a = std::fabs(v);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return static_cast<uint16_t>(sign | 0x7F80);
  int e = 0;
  std::frexp(a, &e);                      // a = f * 2^e with f in [0.5, 1)
  const int ulp_exp = (e - 1 >= -126) ? (e - 8) : -133;
  const double q = std::ldexp(a, -ulp_exp);   // exact: scaling by 2^k
  const double r = std::nearbyint(q);         // default mode: ties to even
  const double res = std::ldexp(r, ulp_exp);  // exact
  if (res >= std::ldexp(1.0, 128)) return static_cast<uint16_t>(sign | 0x7F80);
  const float f = static_cast<float>(res);    // exact: res has <= 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return static_cast<uint16_t>(sign | (u >> 16));
}

// ---------------------------------------------------------------------------
// Biased mean and variance of n values, two passes.
// [p79 block 1] the per-(n,c) mean over the spatial extent and the variance
// as the mean of squared deviations (divide by the element count, not n-1);
// [p34 block 2] the same statistics per (n,c) slice of InstanceNorm2d.
// ---------------------------------------------------------------------------
void moments(const double* v, int64_t n, double* mean, double* var) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s += v[i];
  const double mu = s / static_cast<double>(n);
  double q = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    const double d = v[i] - mu;
    q += d * d;
  }
  *mean = mu;
  *var = q / static_cast<double>(n);
}

// (v - mean) / sqrt(var + eps) -- the normalisation step of [p79 block 1]
// and [p34 block 2].
double normalize(double v, double mean, double var, double eps) {
  return (v - mean) / std::sqrt(var + eps);
}

// clamp(t, lo, hi) = min(max(t, lo), hi), the reading of torch.clamp given in
// [p79 block 1].
double clamp(double t, double lo, double hi) {
  return std::fmin(std::fmax(t, lo), hi);
}

template <class Load, class Store>
int instancenorm_impl(Load load, Store store, int64_t NC, int64_t S, double eps,
                      double* mean_out, double* var_out) {
  if (NC < 0 || S < 0 || !(eps >= 0.0)) return 1;
  std::vector<double> v(static_cast<size_t>(S));
  for (int64_t q = 0; q < NC; ++q) {
    for (int64_t i = 0; i < S; ++i) v[i] = load(q * S + i);
    double mean = 0.0, var = 0.0;
    if (S > 0) moments(v.data(), S, &mean, &var);
    for (int64_t i = 0; i < S; ++i) store(q * S + i, normalize(v[i], mean, var, eps));
    if (mean_out) mean_out[q] = mean;
    if (var_out) var_out[q] = var;
  }
  return 0;
}

}  // namespace

extern "C" {

// Nearest-even rounding of float64 values to bf16 bit patterns, and back.
void fnorm_oracle_round_bf16(const double* v, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16(v[i]);
}
void fnorm_oracle_bf16_to_f64(const uint16_t* b, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_to_double(b[i]);
}

// InstanceNorm forward, affine=False, per (n,c) slice of S contiguous values.
// x and y are [NC][S]; mean_out/var_out (optional, [NC]) receive the biased
// statistics in float64. Returns 0, or 1 on a bad argument.
// [p34 block 1] InstanceNorm2d(64) on x[112,64,512,512]; [p79 block 1] the
// InstanceNorm3d step. eps = 1e-5 is the module default both pages use.
int fnorm_oracle_instancenorm_f64(const double* x, double* y, int64_t NC, int64_t S, double eps,
                                  double* mean_out, double* var_out) {
  return instancenorm_impl([&](int64_t i) { return x[i]; },
                           [&](int64_t i, double r) { y[i] = r; }, NC, S, eps, mean_out, var_out);
}

int fnorm_oracle_instancenorm_f32(const float* x, float* y, int64_t NC, int64_t S, double eps,
                                  double* mean_out, double* var_out) {
  return instancenorm_impl([&](int64_t i) { return static_cast<double>(x[i]); },
                           [&](int64_t i, double r) { y[i] = static_cast<float>(r); }, NC, S, eps,
                           mean_out, var_out);
}

int fnorm_oracle_instancenorm_bf16(const uint16_t* x, uint16_t* y, int64_t NC, int64_t S,
                                   double eps, double* mean_out, double* var_out) {
  return instancenorm_impl([&](int64_t i) { return bf16_to_double(x[i]); },
                           [&](int64_t i, double r) { y[i] = double_to_bf16(r); }, NC, S, eps,
                           mean_out, var_out);
}

// The post-convolution epilogue of [p79 block 1], for x [N][C][S] and a
// per-channel multiplier m [C]:
//   v      = x * m_c                        (the first multiply)
//   t      = InstanceNorm(v) over S          (per (n,c), biased, eps)
//   z_c    = m_c * clamp(t, lo, hi)          (clamp, then the second multiply)
//   y[n,s] = max over c of z_c[n,s]          (output [N][S])
// Each z_c is rounded to binary32 before the max, so the argmax is decided in
// the pages' fp32 precision; ties go to the lowest channel index.
// argmax (optional, [N][S]) gets that index; second (optional, [N][S]) gets the
// runner-up value (-inf when C == 1), which lets a caller see near-ties.
int fnorm_oracle_epilogue_f32(const float* x, const float* m, float* y, int64_t* argmax,
                              float* second, int64_t N, int64_t C, int64_t S, double eps,
                              double lo, double hi) {
  if (N < 0 || C < 1 || S < 0 || !(eps >= 0.0) || !(lo <= hi)) return 1;
  std::vector<double> v(static_cast<size_t>(S));
  std::vector<float> z(static_cast<size_t>(C * S));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t c = 0; c < C; ++c) {
      const double mc = static_cast<double>(m[c]);
      const float* xs = x + (n * C + c) * S;
      for (int64_t s = 0; s < S; ++s) v[s] = static_cast<double>(xs[s]) * mc;  // exact
      double mean = 0.0, var = 0.0;
      if (S > 0) moments(v.data(), S, &mean, &var);
      for (int64_t s = 0; s < S; ++s)
        z[c * S + s] = static_cast<float>(mc * clamp(normalize(v[s], mean, var, eps), lo, hi));
    }
    for (int64_t s = 0; s < S; ++s) {
      float best = z[s];
      float runner = -INFINITY;
      int64_t arg = 0;
      for (int64_t c = 1; c < C; ++c) {
        const float zc = z[c * S + s];
        if (zc > best) {
          runner = best;
          best = zc;
          arg = c;
        } else if (zc > runner) {
          runner = zc;
        }
      }
      y[n * S + s] = best;
      if (argmax) argmax[n * S + s] = arg;
      if (second) second[n * S + s] = runner;
    }
  }
  return 0;
}

// Training-mode BatchNorm forward followed by a scale factor, [p73 blocks 1-2]
// (Conv2d -> BatchNorm2d -> x*2.0), for x [N][C][S]:
//   per channel c over all (n, s): batch mean and biased variance;
//   y = scale * (gamma_c * (x - mean_c) / sqrt(var_c + eps) + beta_c);
//   running_mean <- (1 - momentum) * running_mean + momentum * mean_c;
//   running_var  <- (1 - momentum) * running_var  + momentum * var_c * n/(n-1),
// the running variance taking the unbiased (Bessel-corrected) estimate as
// [p79 block 1] states for running statistics. gamma/beta may be null (1 / 0);
// running_mean/running_var may be null (no update). save_mean/save_var
// (optional, [C]) receive the batch statistics. Needs N*S >= 2.
int fnorm_oracle_batchnorm_train_f32(const float* x, float* y, const float* gamma,
                                     const float* beta, double scale, double* running_mean,
                                     double* running_var, double momentum, double eps, int64_t N,
                                     int64_t C, int64_t S, double* save_mean, double* save_var) {
  if (N < 0 || C < 0 || S < 0 || !(eps >= 0.0)) return 1;
  const int64_t cnt = N * S;
  if (C > 0 && cnt < 2) return 1;
  std::vector<double> v(static_cast<size_t>(cnt));
  for (int64_t c = 0; c < C; ++c) {
    for (int64_t n = 0; n < N; ++n)
      for (int64_t s = 0; s < S; ++s) v[n * S + s] = static_cast<double>(x[(n * C + c) * S + s]);
    double mean = 0.0, var = 0.0;
    moments(v.data(), cnt, &mean, &var);
    const double g = gamma ? static_cast<double>(gamma[c]) : 1.0;
    const double b = beta ? static_cast<double>(beta[c]) : 0.0;
    for (int64_t n = 0; n < N; ++n)
      for (int64_t s = 0; s < S; ++s)
        y[(n * C + c) * S + s] =
            static_cast<float>(scale * (g * normalize(v[n * S + s], mean, var, eps) + b));
    if (running_mean) running_mean[c] = (1.0 - momentum) * running_mean[c] + momentum * mean;
    if (running_var) {
      const double unbiased = var * static_cast<double>(cnt) / static_cast<double>(cnt - 1);
      running_var[c] = (1.0 - momentum) * running_var[c] + momentum * unbiased;
    }
    if (save_mean) save_mean[c] = mean;
    if (save_var) save_var[c] = var;
  }
  return 0;
}

// InstanceNorm with per-channel affine parameters (the module's affine=True
// option; [p34 block 2] notes the module default is affine=False): for slice
// q = n*C + c,
//   y = gamma_c * (x - mean) / sqrt(var + eps) + beta_c,
// the affine step being the one [p73 block 1] writes for BatchNorm
// (normalise, multiply by gamma, add beta). gamma/beta (optional, [C]) default
// to 1 / 0. x and y are [N*C][S] float64; mean_out/var_out as above.
int fnorm_oracle_instancenorm_affine_f64(const double* x, double* y, const double* gamma,
                                         const double* beta, int64_t N, int64_t C, int64_t S,
                                         double eps, double* mean_out, double* var_out) {
  if (N < 0 || C < 0 || S < 0 || !(eps >= 0.0)) return 1;
  std::vector<double> v(static_cast<size_t>(S));
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t c = 0; c < C; ++c) {
      const int64_t q = n * C + c;
      for (int64_t i = 0; i < S; ++i) v[i] = x[q * S + i];
      double mean = 0.0, var = 0.0;
      if (S > 0) moments(v.data(), S, &mean, &var);
      const double g = gamma ? gamma[c] : 1.0;
      const double b = beta ? beta[c] : 0.0;
      for (int64_t i = 0; i < S; ++i) y[q * S + i] = g * normalize(v[i], mean, var, eps) + b;
      if (mean_out) mean_out[q] = mean;
      if (var_out) var_out[q] = var;
    }
  }
  return 0;
}

// Eval-mode BatchNorm followed by a scale factor, [p73 block 1] (in eval mode
// the module normalises with its running statistics, not the batch's) and
// [p73 block 2] (the per-channel factor gamma*scale/sqrt(running_var + eps)
// and shift the pages fold into the convolution): for x [N][C][S],
//   y = scale * (gamma_c * (x - running_mean_c) / sqrt(running_var_c + eps) + beta_c).
// Nothing is updated. gamma/beta (optional, [C]) default to 1 / 0.
int fnorm_oracle_batchnorm_eval_f64(const double* x, double* y, const double* gamma,
                                    const double* beta, double scale, const double* running_mean,
                                    const double* running_var, double eps, int64_t N, int64_t C,
                                    int64_t S) {
  if (N < 0 || C < 0 || S < 0 || !(eps >= 0.0) || !running_mean || !running_var) return 1;
  for (int64_t n = 0; n < N; ++n) {
    for (int64_t c = 0; c < C; ++c) {
      const double g = gamma ? gamma[c] : 1.0;
      const double b = beta ? beta[c] : 0.0;
      const int64_t base = (n * C + c) * S;
      for (int64_t s = 0; s < S; ++s)
        y[base + s] =
            scale * (g * normalize(x[base + s], running_mean[c], running_var[c], eps) + b);
    }
  }
  return 0;
}

}  // extern "C"
