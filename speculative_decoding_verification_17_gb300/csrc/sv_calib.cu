// sv_calib.cu — calibration of the logit-gap gate and the scores of the conformal gate.
//
//  gate_risk_coverage  "Speculative Pre-Positioning", section 2.4, Eq. (13)-(14): coverage and
//                      false-accept risk of the gate over a threshold grid, with the Wilson
//                      intervals of section 4, and the smallest threshold that meets a risk
//                      budget. One or two launches. In the first, every CTA bins its decision
//                      points (four per thread and step, 16-byte loads) by the number of
//                      thresholds below their gap (a bucket table over the grid, then the
//                      gap's own bucket searched) into a shared histogram, folds it into a
//                      global one, and the last CTA turns the histogram into per-threshold
//                      counts with one suffix scan. The second (grids of more than 256
//                      thresholds; the last CTA does it for smaller ones) forms every
//                      threshold's rates and Wilson intervals in double, one thread each over
//                      many SMs.
//  conformal_residual  the "speculative-decoding-plan.md" conformal gate's calibration score:
//                      the sup-norm distance of a draft row from the true row. A streaming
//                      max over two rows (16-byte loads, four pairs in flight per thread),
//                      folded into the output with an atomic maximum on the float's bits.
//  conformal_quantile  the split-conformal quantile of those scores: a radix select over the
//                      scores' order-preserving keys in three passes (11, 11, 10 bits); up to
//                      8192 scores in one CTA with the keys in shared memory, beyond that one
//                      cooperative launch whose passes each end in a grid-wide rendezvous:
//                      the CTA whose arrival completes the pass picks the digit from the
//                      pass's global histogram and publishes it to the others.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "specverify_calib.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

int device_sm_count();  // sv_common.cu

namespace {

constexpr int kCalThreads = 256;

// Wilson score interval of k successes in n trials at the normal quantile z, clamped to
// [0, 1]; NaN for n = 0. Each operation is rounded on its own (the half-width's product is
// kept out of a fused multiply-add), so the result matches the formula evaluated step by step.
__device__ void wilson(double k, double n, double z, double& lo, double& hi) {
  if (!(n > 0.0)) {
    lo = hi = __longlong_as_double(0x7ff8000000000000LL);
    return;
  }
  const double p = k / n;
  const double z2 = z * z;
  const double denom = 1.0 + z2 / n;
  const double centre = (p + z2 / (2.0 * n)) / denom;
  const double half = __dmul_rn(z / denom, sqrt(p * (1.0 - p) / n + z2 / (4.0 * n * n)));
  const double a = centre - half, b = centre + half;
  lo = a < 0.0 ? 0.0 : a;
  hi = b > 1.0 ? 1.0 : b;
}

// In place: a[i] <- a[i] + a[i+1] + ... + a[n-1] (inclusive suffix sums), all threads.
__device__ void block_suffix_sums(unsigned int* a, int n, unsigned int* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int per = (n + kCalThreads - 1) / kCalThreads;
  const int b0 = threadIdx.x * per;
  const int b1 = min(b0 + per, n);
  unsigned int tot = 0;
  for (int i = b0; i < b1; ++i) tot += a[i];
  unsigned int incl = tot;  // this thread and the later lanes of its warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int v = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += v;
  }
  if (lane == 0) warp_tot[w] = incl;
  __syncthreads();
  unsigned int run = incl - tot;
  for (int v = w + 1; v < kCalThreads / 32; ++v) run += warp_tot[v];
  for (int i = b1 - 1; i >= b0; --i) {
    run += a[i];
    a[i] = run;
  }
  __syncthreads();
}

// In place: a[i] <- a[0] + ... + a[i-1] (exclusive prefix sums), all threads.
__device__ void block_prefix_sums(unsigned int* a, int n, unsigned int* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int per = (n + kCalThreads - 1) / kCalThreads;
  const int b0 = threadIdx.x * per;
  const int b1 = min(b0 + per, n);
  unsigned int tot = 0;
  for (int i = b0; i < b1; ++i) tot += a[i];
  unsigned int incl = tot;  // this thread and the earlier lanes of its warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  unsigned int run = incl - tot;
  for (int v = 0; v < w; ++v) run += warp_tot[v];
  for (int i = b0; i < b1; ++i) {
    const unsigned int x = a[i];
    a[i] = run;
    run += x;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ risk-coverage sweep
struct SweepArgs {
  const float* gap;
  const int32_t* token;
  const int32_t* full;
  int N;
  const int32_t* answer;
  int n_answer;
  const float* taus;
  int T;
  double z, r_max;
  sv_calib_point* out;
  int32_t* out_idx;
  unsigned int* acc;  // [T + 1]: accepted points by bin b = #{t : taus[t] < gap}
  unsigned int* bad;  // [T + 1]: the wrong ones among them
  unsigned int* cnt;  // CTA arrivals
  int* state;         // [3]: broken grid flag, T - (smallest qualifying t) or 0, arrivals of
                      // sweep_points_kernel
  bool vec;           // gap, token and full_token all start on a 16-byte boundary
};

// The bin of a gap g, b = #{t : tau[t] < g}, comes from a bucket table when the grid's ends
// are finite: bucket(x) = floor((x - tau[0]) * NB / (tau[T-1] - tau[0])), clamped to
// [0, NB), is non-decreasing in x, so every threshold of an earlier bucket lies below g and
// every one of a later bucket above it. b is then first[bucket(g)] (the thresholds of the
// earlier buckets) plus the count of g's own bucket's thresholds below g: a search over that
// bucket only, no step at all for a uniform grid. Membership in the answer set is one bit of a
// shared-memory bitmap over [answer[0], answer[n-1]] when that span has at most kAnswerBits
// tokens (every vocabulary up to 262144 tokens); a wider set is searched, in shared memory when
// it has at most kSmemAnswer entries.
constexpr int kSmemAnswer = 4096;
constexpr int kAnswerBits = 1 << 18;
__host__ __device__ inline int sweep_buckets(int T) {
  int nb = 64;
  while (nb < 2 * T && nb < 8192) nb <<= 1;
  return nb;
}
// the answer region holds the bitmap or, for a wider set, its copy
inline size_t sweep_answer_bytes(int n_answer) {
  if (n_answer <= 0) return 0;
  return std::max((size_t)kAnswerBits / 8,
                  (size_t)(n_answer <= kSmemAnswer ? n_answer : 0) * sizeof(int32_t));
}
inline size_t sweep_smem(int T, int n_answer) {
  return (size_t)T * sizeof(float) + 2 * (size_t)(T + 1) * sizeof(unsigned int) +
         (size_t)(sweep_buckets(T) + 1) * sizeof(unsigned int) + sweep_answer_bytes(n_answer);
}

__device__ __forceinline__ int sweep_bucket(float x, float lo, float scale, int nb) {
  const float v = (x - lo) * scale;
  return (int)fminf(fmaxf(v, 0.0f), (float)(nb - 1));  // NaN (0 * inf) goes to bucket 0
}

// Threshold t's point from its counts: coverage, risk and their Wilson intervals, in double
// as section 4's formulas are written; t joins the qualifying set (atomicMax on T - t in
// *rev) when its risk is within r_max.
__device__ void threshold_point(const SweepArgs& A, int t, unsigned int acc, unsigned int bad,
                                int* rev) {
  const double nan = __longlong_as_double(0x7ff8000000000000LL);
  const double n = (double)A.N;
  sv_calib_point p;
  p.accepted = acc;
  p.wrong = bad;
  p.coverage = A.N > 0 ? (double)acc / n : nan;
  wilson((double)acc, n, A.z, p.cov_lo, p.cov_hi);
  if (acc > 0) {
    p.risk = (double)bad / (double)acc;
    wilson((double)bad, (double)acc, A.z, p.risk_lo, p.risk_hi);
    if (p.risk <= A.r_max) atomicMax(rev, A.T - t);
  } else {
    p.risk = p.risk_lo = p.risk_hi = nan;
  }
  A.out[t] = p;
}

// Grids up to this size get their points from sweep_kernel's last CTA; larger ones from
// sweep_points_kernel, over many SMs (the double-precision intervals of a large grid on one
// SM take longer than a second launch).
constexpr int kPointsInLastCta = 256;

__global__ void __launch_bounds__(kCalThreads) sweep_kernel(const SweepArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int T = A.T;
  const int NB = sweep_buckets(T);
  float* tau = reinterpret_cast<float*>(smem);
  unsigned int* hacc = reinterpret_cast<unsigned int*>(tau + T);
  unsigned int* hbad = hacc + T + 1;
  unsigned int* first = hbad + T + 1;  // [NB + 1]
  int32_t* ans_s = reinterpret_cast<int32_t*>(first + NB + 1);
  unsigned int* bits = reinterpret_cast<unsigned int*>(ans_s);  // the same region
  // the bitmap's span; the set is sorted, so a span of 0 or less (an unsorted set) or one
  // wider than the bitmap is searched instead
  const unsigned amin = A.n_answer > 0 ? (unsigned)__ldg(A.answer) : 0u;
  const int64_t span =
      A.n_answer > 0 ? (int64_t)__ldg(A.answer + A.n_answer - 1) - (int32_t)amin + 1 : 0;
  const bool bitmap = span > 0 && span <= kAnswerBits;
  const unsigned range = bitmap ? (unsigned)span : 0u;
  const bool ans_in_smem = !bitmap && A.n_answer <= kSmemAnswer;
  const int32_t* ans = ans_in_smem ? ans_s : A.answer;
  __shared__ unsigned int warp_tot[kCalThreads / 32];
  __shared__ int last;
  for (int t = threadIdx.x; t < T; t += kCalThreads) tau[t] = __ldg(A.taus + t);
  for (int b = threadIdx.x; b <= T; b += kCalThreads) hacc[b] = hbad[b] = 0;
  if (bitmap) {
    for (unsigned w = threadIdx.x; w < (range + 31) / 32; w += kCalThreads) bits[w] = 0u;
    __syncthreads();
    for (int i = threadIdx.x; i < A.n_answer; i += kCalThreads) {
      const unsigned u = (unsigned)__ldg(A.answer + i) - amin;
      if (u < range) atomicOr(&bits[u >> 5], 1u << (u & 31));
    }
  } else if (ans_in_smem) {
    for (int i = threadIdx.x; i < A.n_answer; i += kCalThreads) ans_s[i] = __ldg(A.answer + i);
  }
  __syncthreads();

  const float t0 = tau[0];
  const float tlo = tau[0], thi = tau[T - 1];
  const bool table = isfinite(tlo) && isfinite(thi);
  const float scale = table && thi > tlo ? (float)NB / (thi - tlo) : 0.0f;
  if (table) {
    // first[j] = #{t : bucket(tau[t]) < j}: a lower bound over the non-decreasing buckets
    for (int j = threadIdx.x; j <= NB; j += kCalThreads) {
      int lo = 0;
      for (int n = T; n > 0;) {
        const int half = n >> 1;
        if (sweep_bucket(tau[lo + half], tlo, scale, NB) < j) {
          lo += half + 1;
          n -= half + 1;
        } else {
          n = half;
        }
      }
      first[j] = (unsigned)lo;
    }
  }
  __syncthreads();
  // Four decision points at a time: each point's membership in A (a bit of the bitmap, or a
  // branch-free lower bound of a fixed number of steps) and its bin b = #{t : tau[t] < g}
  // (accepted at every t < b), so the four lookups overlap and the lanes stay converged.
  auto bin4 = [&](const float (&g)[4], const int (&tok)[4], const int (&full)[4]) {
    bool ok[4];
    int ib[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      ok[p] = g[p] > t0 && A.n_answer > 0;  // below every threshold (or NaN): accepted nowhere
      ib[p] = 0;
    }
    if (bitmap) {
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const unsigned u = (unsigned)tok[p] - amin;
        ok[p] = ok[p] && u < range && ((bits[u >> 5] >> (u & 31)) & 1u);
      }
    } else {
      int ia[4] = {0, 0, 0, 0};
      for (int n = A.n_answer; n > 1;) {
        const int half = n >> 1;
#pragma unroll
        for (int p = 0; p < 4; ++p)
          if (ans[ia[p] + half] < tok[p]) ia[p] += half;
        n -= half;
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int la = ia[p] + (ans[ia[p]] < tok[p]);  // first entry >= tok
        ok[p] = ok[p] && la < A.n_answer && ans[la] == tok[p];
      }
    }
    int b[4];
    if (table) {
      // the thresholds of earlier buckets, then those of g's bucket that lie below g
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int j = ok[p] ? sweep_bucket(g[p], tlo, scale, NB) : 0;
        int lo = (int)first[j];
        const int hi = (int)first[j + 1];
        for (int n = hi - lo; n > 0;) {
          const int half = n >> 1;
          if (tau[lo + half] < g[p]) {
            lo += half + 1;
            n -= half + 1;
          } else {
            n = half;
          }
        }
        b[p] = lo;
      }
    } else {
      for (int n = T; n > 1;) {
        const int half = n >> 1;
#pragma unroll
        for (int p = 0; p < 4; ++p)
          if (tau[ib[p] + half] < g[p]) ib[p] += half;
        n -= half;
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) b[p] = ib[p] + (tau[ib[p]] < g[p]);
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      if (!ok[p]) continue;
      const int bb = b[p] < 1 ? 1 : (b[p] > T ? T : b[p]);  // >= 1 since tau[0] < g
      atomicAdd(&hacc[bb], 1u);
      if (tok[p] != full[p]) atomicAdd(&hbad[bb], 1u);
    }
  };
  const int64_t stride = (int64_t)gridDim.x * kCalThreads;
  const int64_t tid = (int64_t)blockIdx.x * kCalThreads + threadIdx.x;
  // four points per thread and step, two steps' six 16-byte loads issued together
  const int64_t n4 = A.vec ? A.N / 4 : 0;
  const float4* gap4 = reinterpret_cast<const float4*>(A.gap);
  const int4* tok4 = reinterpret_cast<const int4*>(A.token);
  const int4* full4 = reinterpret_cast<const int4*>(A.full);
  for (int64_t q = tid; q < n4; q += 2 * stride) {
    const bool two = q + stride < n4;
    const float4 g = __ldcs(gap4 + q);
    const int4 t = __ldcs(tok4 + q);
    const int4 f = __ldcs(full4 + q);
    float4 g2 = make_float4(0.f, 0.f, 0.f, 0.f);
    int4 t2 = make_int4(0, 0, 0, 0), f2 = make_int4(0, 0, 0, 0);
    if (two) {
      g2 = __ldcs(gap4 + q + stride);
      t2 = __ldcs(tok4 + q + stride);
      f2 = __ldcs(full4 + q + stride);
    }
    {
      const float gg[4] = {g.x, g.y, g.z, g.w};
      const int tt[4] = {t.x, t.y, t.z, t.w}, ff[4] = {f.x, f.y, f.z, f.w};
      bin4(gg, tt, ff);
    }
    if (two) {
      const float gg[4] = {g2.x, g2.y, g2.z, g2.w};
      const int tt[4] = {t2.x, t2.y, t2.z, t2.w}, ff[4] = {f2.x, f2.y, f2.z, f2.w};
      bin4(gg, tt, ff);
    }
  }
  // the rest (or everything, for inputs off the 16-byte grid), four points per step
  for (int64_t i0 = 4 * n4 + 4 * tid; i0 < A.N; i0 += 4 * stride) {
    float gg[4];
    int tt[4], ff[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const bool in = i0 + p < A.N;
      gg[p] = in ? __ldcs(A.gap + i0 + p) : __int_as_float(0x7fc00000);  // NaN: not accepted
      tt[p] = in ? __ldcs(A.token + i0 + p) : 0;
      ff[p] = in ? __ldcs(A.full + i0 + p) : 0;
    }
    bin4(gg, tt, ff);
  }
  __syncthreads();
  // a grid of one CTA keeps its histogram in shared memory: no global fold, no arrival
  const bool solo = gridDim.x == 1;
  if (!solo) {
    for (int b = 1 + threadIdx.x; b <= T; b += kCalThreads) {
      if (hacc[b]) atomicAdd(A.acc + b, hacc[b]);
      if (hbad[b]) atomicAdd(A.bad + b, hbad[b]);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      last = arrive_last(A.cnt, gridDim.x);
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
  }

  // the grid must be non-decreasing without NaN
  int broken = 0;
  for (int t = threadIdx.x; t < T; t += kCalThreads)
    broken |= (tau[t] != tau[t]) || (t > 0 && tau[t] < tau[t - 1]);
  broken = __syncthreads_or(broken);
  const double nan = __longlong_as_double(0x7ff8000000000000LL);
  if (broken) {
    for (int t = threadIdx.x; t < T; t += kCalThreads)
      A.out[t] = sv_calib_point{-1, -1, nan, nan, nan, nan, nan, nan};
    if (threadIdx.x == 0) {
      *A.out_idx = -2;
      *A.state = 1;
    }
    return;
  }
  // accepted(t) = sum of bins b > t, written back over the histograms for
  // sweep_points_kernel, which forms each threshold's rates and intervals
  if (!solo) {
    for (int b = threadIdx.x; b <= T; b += kCalThreads) {
      hacc[b] = b ? __ldcg(A.acc + b) : 0u;
      hbad[b] = b ? __ldcg(A.bad + b) : 0u;
    }
    __syncthreads();
  }
  block_suffix_sums(hacc, T + 1, warp_tot);
  block_suffix_sums(hbad, T + 1, warp_tot);
  if (T <= kPointsInLastCta) {  // a small grid: the points here, no second launch
    __shared__ int rev;
    if (threadIdx.x == 0) rev = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < T; t += kCalThreads)
      threshold_point(A, t, hacc[t + 1], hbad[t + 1], &rev);
    __syncthreads();
    if (threadIdx.x == 0) *A.out_idx = rev == 0 ? -1 : T - rev;
    return;
  }
  for (int t = threadIdx.x; t < T; t += kCalThreads) {
    A.acc[t + 1] = hacc[t + 1];
    A.bad[t + 1] = hbad[t + 1];
  }
}

// The coverage, risk and Wilson intervals of every threshold (one thread each, in double, as
// the formulas of section 4 are written), spread over many SMs, and the smallest t whose risk
// is within r_max. Launched after sweep_kernel on the same stream.
constexpr int kPointThreads = 32;  // one warp per CTA: the FP64 chains spread over more SMs
__global__ void __launch_bounds__(kPointThreads) sweep_points_kernel(const SweepArgs A) {
  __shared__ int last;
  if (__ldcg(A.state) != 0) return;  // a broken grid: sweep_kernel wrote the outcome
  const int t = blockIdx.x * kPointThreads + threadIdx.x;
  if (t < A.T) threshold_point(A, t, __ldcg(A.acc + t + 1), __ldcg(A.bad + t + 1), A.state + 1);
  __syncthreads();
  if (threadIdx.x == 0) last = arrive_last(reinterpret_cast<unsigned int*>(A.state + 2), gridDim.x);
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  const int rev = __ldcg(A.state + 1);
  *A.out_idx = rev == 0 ? -1 : A.T - rev;
}

struct SweepLayout {
  size_t acc, bad, cnt, state, total;
};
SweepLayout sweep_layout(int T) {
  SweepLayout L{};
  size_t o = 0;
  L.acc = o; o = round_up(o + (size_t)(T + 1) * sizeof(unsigned int), 256);
  L.bad = o; o = round_up(o + (size_t)(T + 1) * sizeof(unsigned int), 256);
  L.cnt = o; o = round_up(o + sizeof(unsigned int), 256);
  L.state = o; o = round_up(o + 3 * sizeof(int), 256);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ conformal residual
// One CTA per (row pair, piece of kResidPieceVec vectors); 16-byte loads of both rows.
constexpr int kResidPieceVec = 4096;  // 64 KiB of each row
constexpr int kResidUnroll = 4;

struct ResidArgs {
  const void* a;
  const void* b;
  int N, V;
  int pieces;    // pieces per row
  float* out;
};

template <typename E>
__device__ __forceinline__ void resid_fold(float x, float y, float& m, bool& nan) {
  const float d = x == y ? 0.0f : fabsf(x - y);
  nan |= d != d;
  m = fmaxf(m, d);
}

template <typename E, bool kVec>
__global__ void __launch_bounds__(kCalThreads) resid_kernel(const ResidArgs A) {
  const int64_t u = blockIdx.x;
  const int row = (int)(u / A.pieces);
  const int piece = (int)(u - (int64_t)row * A.pieces);
  float m = 0.0f;
  bool nan = false;
  if (kVec) {
    const int64_t nvec = (int64_t)A.V / E::kPerVec;  // rows hold whole vectors here
    const uint4* ra = reinterpret_cast<const uint4*>(A.a) + (int64_t)row * nvec;
    const uint4* rb = reinterpret_cast<const uint4*>(A.b) + (int64_t)row * nvec;
    const int64_t v0 = (int64_t)piece * kResidPieceVec;
    const int64_t v1 = min(v0 + kResidPieceVec, nvec);
    for (int64_t v = v0 + threadIdx.x; v < v1; v += kResidUnroll * kCalThreads) {
      uint4 xa[kResidUnroll], xb[kResidUnroll];
#pragma unroll
      for (int q = 0; q < kResidUnroll; ++q) {
        const int64_t vq = v + (int64_t)q * kCalThreads;
        if (vq < v1) {
          xa[q] = __ldcs(ra + vq);
          xb[q] = __ldcs(rb + vq);
        } else {
          xa[q] = xb[q] = make_uint4(0u, 0u, 0u, 0u);  // equal: contributes 0
        }
      }
#pragma unroll
      for (int q = 0; q < kResidUnroll; ++q)
#pragma unroll
        for (int l = 0; l < E::kPerVec; ++l)
          resid_fold<E>(E::get(xa[q], l), E::get(xb[q], l), m, nan);
    }
  } else {
    // rows off the 16-byte grid: logit by logit (coalesced)
    const int64_t pe = (int64_t)kResidPieceVec * E::kPerVec;
    const int64_t j0 = (int64_t)piece * pe;
    const int64_t j1 = min(j0 + pe, (int64_t)A.V);
    const int64_t base = (int64_t)row * A.V;
    for (int64_t j = j0 + threadIdx.x; j < j1; j += kCalThreads)
      resid_fold<E>(E::load1(A.a, base + j), E::load1(A.b, base + j), m, nan);
  }
  // CTA maximum, then one atomic maximum on the non-negative float's bits (NaN above +inf)
  __shared__ float wm[kCalThreads / 32];
  __shared__ int wn[kCalThreads / 32];
  m = warp_max_f(m);
  nan = __any_sync(0xffffffffu, nan);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    wm[w] = m;
    wn[w] = nan;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int v = 1; v < kCalThreads / 32; ++v) {
      m = fmaxf(m, wm[v]);
      nan |= wn[v] != 0;
    }
    const unsigned int bits = nan ? 0x7fc00000u : __float_as_uint(m);
    atomicMax(reinterpret_cast<unsigned int*>(A.out) + row, bits);
  }
}

// ------------------------------------------------------------------ conformal quantile
constexpr int kSelBins = 2048;
constexpr int kSelectPasses = 3;
constexpr int kSelUnroll = 4;
constexpr uint64_t kSelWaitNs = 2000000000ull;  // 2 s: far past any legitimate barrier wait
constexpr unsigned int kSelTimedOut = 0x7fc00001u;  // quiet NaN, payload 1

struct SelectState {
  unsigned int cnt[4];     // CTA arrivals at each pass's grid barrier
  unsigned int pick[kSelectPasses][4];  // per pass: the digit, the keys below it, published
  unsigned int hist[kSelectPasses][kSelBins];
};

// Order-preserving key of a float (NaN canonicalised, above +inf; -0 below +0).
__device__ __forceinline__ unsigned int float_key(float x) {
  unsigned int u = __float_as_uint(x);
  if (x != x) u = 0x7fc00000u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(unsigned int k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The whole radix select in one cooperative launch. Each pass: every CTA counts the keys that
// share the prefix chosen so far into a shared histogram of the next digit (sixteen scores per
// thread and step, four 16-byte loads in flight) and adds it to the pass's global histogram;
// the CTA whose arrival completes the pass reads that histogram and picks the digit d, the
// one with (keys below it) < want <= (keys below it) + count(d), and publishes it; the other
// CTAs wait for it (one reader of the histogram: all of them reading its 8 KB at once made
// the pick take ~6 us a pass). The first two passes load the scores with an L2 evict-last
// policy, so the next pass finds them in L2. A pass completes at gridDim.x + extra arrivals
// (extra = 0; 1 only in the barrier self-test, where no pass can complete); every wait is
// bounded by limit_ns.
__global__ void __launch_bounds__(kCalThreads) select_kernel(const float* r, int n, int64_t rank,
                                                             SelectState* st, float* out,
                                                             unsigned int extra,
                                                             uint64_t limit_ns) {
  __shared__ unsigned int h[kSelBins];
  __shared__ unsigned int warp_tot[kCalThreads / 32];
  __shared__ unsigned int s_digit, s_before;
  __shared__ int s_last, s_ok;
  const int64_t stride = (int64_t)gridDim.x * kCalThreads;
  const int64_t tid = (int64_t)blockIdx.x * kCalThreads + threadIdx.x;
  const int64_t n4 = (reinterpret_cast<uintptr_t>(r) % 16 == 0) ? n / 4 : 0;
  const float4* r4 = reinterpret_cast<const float4*>(r);
  unsigned int prefix = 0u;
  unsigned int want = (unsigned int)rank;
  for (int pass = 0; pass < kSelectPasses; ++pass) {
    const int width = pass == 2 ? 10 : 11;
    const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    const unsigned int mask = (1u << width) - 1u;
    for (int b = threadIdx.x; b < kSelBins; b += kCalThreads) h[b] = 0;
    if (threadIdx.x == 0) s_digit = s_before = 0u;
    __syncthreads();
    auto count = [&](float x) {
      const unsigned int key = float_key(x);
      if (pass == 0 || (key >> (shift + width)) == prefix) atomicAdd(&h[(key >> shift) & mask], 1u);
    };
    const uint64_t pol = l2_policy(pass + 1 < kSelectPasses);
    int64_t q = tid;
    for (; q + (kSelUnroll - 1) * stride < n4; q += kSelUnroll * stride) {
      float4 x[kSelUnroll];
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u)
        asm("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
            : "=f"(x[u].x), "=f"(x[u].y), "=f"(x[u].z), "=f"(x[u].w)
            : "l"(r4 + q + u * stride), "l"(pol));
#pragma unroll
      for (int u = 0; u < kSelUnroll; ++u) {
        count(x[u].x);
        count(x[u].y);
        count(x[u].z);
        count(x[u].w);
      }
    }
    for (; q < n4; q += stride) {
      const float4 x = __ldg(r4 + q);
      count(x.x);
      count(x.y);
      count(x.z);
      count(x.w);
    }
    for (int64_t i = 4 * n4 + tid; i < n; i += stride) count(__ldg(r + i));
    __syncthreads();
    for (int b = threadIdx.x; b <= (int)mask; b += kCalThreads)
      if (h[b]) atomicAdd(&st->hist[pass][b], h[b]);
    // arrival: release this CTA's histogram adds; the last arrival acquires every CTA's
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      unsigned int seen;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                   : "=r"(seen)
                   : "l"(&st->cnt[pass])
                   : "memory");
      s_last = seen + 1 == gridDim.x + extra;
    }
    __syncthreads();
    if (s_last) {
      // the pass is complete: this CTA picks the digit for every CTA
      for (int b = threadIdx.x; b < kSelBins; b += kCalThreads)
        h[b] = b <= (int)mask ? __ldcg(&st->hist[pass][b]) : 0u;
      __syncthreads();
      // counts before the prefix sums, kept per thread for the check below
      constexpr int per = kSelBins / kCalThreads;
      unsigned int own[per];
#pragma unroll
      for (int i = 0; i < per; ++i) own[i] = h[threadIdx.x * per + i];
      __syncthreads();
      block_prefix_sums(h, kSelBins, warp_tot);
#pragma unroll
      for (int i = 0; i < per; ++i) {
        const int b = threadIdx.x * per + i;
        const unsigned int before = h[b];
        if (b <= (int)mask && own[i] > 0 && before < want && want <= before + own[i]) {
          s_digit = (unsigned int)b;
          s_before = before;
        }
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        st->pick[pass][0] = s_digit;
        st->pick[pass][1] = s_before;
        asm volatile("st.release.gpu.global.u32 [%0], 1;" ::"l"(&st->pick[pass][2]) : "memory");
      }
    } else if (threadIdx.x == 0) {
      // wait (bounded) for the last arrival to publish the digit
      unsigned int done = 0;
      const uint64_t t0 = globaltimer_ns();
      while (true) {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                     : "=r"(done)
                     : "l"(&st->pick[pass][2])
                     : "memory");
        if (done || globaltimer_ns() - t0 > limit_ns) break;
        __nanosleep(128);
      }
      s_ok = done != 0;
      if (done) {
        s_digit = __ldcg(&st->pick[pass][0]);
        s_before = __ldcg(&st->pick[pass][1]);
      }
    }
    __syncthreads();
    if (!s_last && !s_ok) {  // the wait ran out: the timeout sentinel
      if (blockIdx.x == 0 && threadIdx.x == 0) *out = __uint_as_float(kSelTimedOut);
      return;
    }
    prefix = (prefix << width) | s_digit;
    want -= s_before;
    __syncthreads();
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) *out = key_float(prefix);
}


// The whole select in one CTA for small score sets: the keys stay in shared memory.
constexpr int kSmallSelect = 8192;

__global__ void __launch_bounds__(kCalThreads) select_small_kernel(const float* r, int n,
                                                                   int rank, float* out) {
  __shared__ unsigned int keys[kSmallSelect];
  __shared__ unsigned int h[kSelBins];
  __shared__ unsigned int warp_tot[kCalThreads / 32];
  __shared__ unsigned int s_prefix, s_want;
  for (int i = threadIdx.x; i < n; i += kCalThreads) keys[i] = float_key(__ldg(r + i));
  if (threadIdx.x == 0) {
    s_prefix = 0u;
    s_want = (unsigned int)rank;
  }
  constexpr int per = kSelBins / kCalThreads;
  for (int pass = 0; pass < kSelectPasses; ++pass) {
    const int width = pass == 2 ? 10 : 11;
    const int shift = pass == 0 ? 21 : pass == 1 ? 10 : 0;
    const unsigned int mask = (1u << width) - 1u;
    for (int b = threadIdx.x; b < kSelBins; b += kCalThreads) h[b] = 0;
    __syncthreads();
    const unsigned int prefix = s_prefix, want = s_want;
    for (int i = threadIdx.x; i < n; i += kCalThreads) {
      const unsigned int key = keys[i];
      if (pass == 0 || (key >> (shift + width)) == prefix) atomicAdd(&h[(key >> shift) & mask], 1u);
    }
    __syncthreads();
    unsigned int own[per];
#pragma unroll
    for (int i = 0; i < per; ++i) own[i] = h[threadIdx.x * per + i];
    __syncthreads();
    block_prefix_sums(h, kSelBins, warp_tot);
#pragma unroll
    for (int i = 0; i < per; ++i) {
      const int b = threadIdx.x * per + i;
      const unsigned int before = h[b];
      if (b <= (int)mask && own[i] > 0 && before < want && want <= before + own[i]) {
        s_prefix = (prefix << width) | (unsigned int)b;
        s_want = want - before;
      }
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) *out = key_float(s_prefix);
}

__global__ void store_inf(float* out) { *out = __uint_as_float(0x7f800000u); }

}  // namespace
}  // namespace sv

// ============================================================================================
// C ABI
// ============================================================================================
using namespace sv;

extern "C" size_t gate_risk_coverage_workspace(int N, int T) {
  if (N < 0 || T < 1 || T > SV_MAX_TAUS) return 0;
  return sweep_layout(T).total;
}

extern "C" sv_status gate_risk_coverage(const float* gap, const int32_t* token,
                                        const int32_t* full_token, int N,
                                        const int32_t* answer_set, int n_answer,
                                        const float* taus, int T, double z, double r_max,
                                        sv_calib_point* out_points, int32_t* out_tau_index,
                                        void* workspace, size_t workspace_bytes,
                                        sv_stream_t stream) {
  if (N < 0 || n_answer < 0 || T < 1) return SV_ERR_INVALID_ARG;
  if (T > SV_MAX_TAUS) return SV_ERR_UNSUPPORTED;
  if (!std::isfinite(z) || z < 0.0) return SV_ERR_INVALID_ARG;
  if (!taus || !out_points || !out_tau_index || (n_answer > 0 && !answer_set))
    return SV_ERR_INVALID_ARG;
  if (N > 0 && (!gap || !token || !full_token)) return SV_ERR_INVALID_ARG;
  if (!aligned_to(taus, 4) || !aligned_to(out_points, 8) || !aligned_to(out_tau_index, 4) ||
      (gap && !aligned_to(gap, 4)) || (token && !aligned_to(token, 4)) ||
      (full_token && !aligned_to(full_token, 4)) || (answer_set && !aligned_to(answer_set, 4)))
    return SV_ERR_INVALID_ARG;
  const SweepLayout L = sweep_layout(T);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  SweepArgs A;
  A.gap = gap;
  A.token = token;
  A.full = full_token;
  A.N = N;
  A.answer = answer_set;
  A.n_answer = n_answer;
  A.taus = taus;
  A.T = T;
  A.z = z;
  A.r_max = r_max;
  A.out = out_points;
  A.out_idx = out_tau_index;
  char* ws = static_cast<char*>(workspace);
  A.acc = reinterpret_cast<unsigned int*>(ws + L.acc);
  A.bad = reinterpret_cast<unsigned int*>(ws + L.bad);
  A.cnt = reinterpret_cast<unsigned int*>(ws + L.cnt);
  A.state = reinterpret_cast<int*>(ws + L.state);
  A.vec = aligned_to(gap, 16) && aligned_to(token, 16) && aligned_to(full_token, 16);
  const size_t smem = sweep_smem(T, n_answer);
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(sweep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // every resident CTA slot of the GPU, but no more than one CTA per 2048 points; the
  // occupancy answer is kept per device for the last shared-memory size asked (a host query
  // that would otherwise delay every launch)
  static std::atomic<unsigned long long> occ_cache[64];  // (smem << 16) | per_sm
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  int per_sm = 0;
  const unsigned long long cached = dev >= 0 && dev < 64 ? occ_cache[dev].load() : 0ull;
  if (cached && (cached >> 16) == (unsigned long long)smem) {
    per_sm = (int)(cached & 0xffffu);
  } else {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sweep_kernel, kCalThreads, smem);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < 64 && per_sm > 0)
      occ_cache[dev].store(((unsigned long long)smem << 16) | (unsigned)(per_sm & 0xffff));
  }
  const int64_t want = ((int64_t)N + 8 * kCalThreads - 1) / (8 * kCalThreads);
  const int64_t slots = (int64_t)std::max(per_sm, 1) * device_sm_count();
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, slots));
  // the workspace's histograms and counters start at zero; a grid of one CTA with the points
  // in that CTA (T <= kPointsInLastCta) uses none of them
  if (grid > 1 || T > kPointsInLastCta) {
    e = cudaMemsetAsync(workspace, 0, L.total, st);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  sweep_kernel<<<grid, kCalThreads, smem, st>>>(A);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e);
  if (T <= kPointsInLastCta) return SV_OK;
  sweep_points_kernel<<<(T + kPointThreads - 1) / kPointThreads, kPointThreads, 0, st>>>(A);
  return launch_status();
}

extern "C" sv_status conformal_residual(const void* draft_logits, const void* true_logits,
                                        sv_dtype dtype, int N, int V, float* out_resid,
                                        sv_stream_t stream) {
  if (N < 0 || V < 1) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (N == 0) return SV_OK;
  if (!draft_logits || !true_logits || !out_resid) return SV_ERR_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned_to(draft_logits, eb) || !aligned_to(true_logits, eb) ||
      !aligned_to(out_resid, 4))
    return SV_ERR_INVALID_ARG;
  const bool vec = aligned_to(draft_logits, 16) && aligned_to(true_logits, 16) &&
                   ((int64_t)V * eb) % 16 == 0;
  const int per_vec = 16 / eb;
  const int64_t piece_elems = (int64_t)kResidPieceVec * per_vec;
  const int pieces = (int)(((int64_t)V + piece_elems - 1) / piece_elems);
  const int64_t units = (int64_t)N * pieces;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(out_resid, 0, (size_t)N * sizeof(float), st);
  if (e != cudaSuccess) return cuda_fail(e);
  ResidArgs A{draft_logits, true_logits, N, V, pieces, out_resid};
  const unsigned grid = (unsigned)units;
  if (dtype == SV_F32) {
    if (vec) resid_kernel<F32, true><<<grid, kCalThreads, 0, st>>>(A);
    else resid_kernel<F32, false><<<grid, kCalThreads, 0, st>>>(A);
  } else {
    if (vec) resid_kernel<BF16, true><<<grid, kCalThreads, 0, st>>>(A);
    else resid_kernel<BF16, false><<<grid, kCalThreads, 0, st>>>(A);
  }
  return launch_status();
}

namespace sv {

// The cooperative radix-select launch of conformal_quantile (more than kSmallSelect scores):
// clear the state, size the grid, launch. extra and limit_ns go to the grid barriers.
sv_status launch_select(const float* resid, int n, int64_t rank, float* out_q, void* workspace,
                        unsigned int extra, uint64_t limit_ns, cudaStream_t st) {
  const size_t need = round_up(sizeof(SelectState), 256);
  cudaError_t e = cudaMemsetAsync(workspace, 0, need, st);
  if (e != cudaSuccess) return cuda_fail(e);
  SelectState* S = static_cast<SelectState*>(workspace);
  // A cooperative launch: every CTA must be resident at once for the grid barriers. Up to
  // four CTAs per SM (as many as fit), no more than one CTA per 4096 scores; the occupancy
  // answer is kept per device (a host query that would otherwise delay every launch).
  static std::atomic<int> occ_cache[64];
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  int per_sm = dev >= 0 && dev < 64 ? occ_cache[dev].load() : 0;
  if (per_sm <= 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, select_kernel, kCalThreads, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    if (per_sm <= 0) return SV_ERR_UNSUPPORTED;
    if (dev >= 0 && dev < 64) occ_cache[dev].store(per_sm);
  }
  const int64_t want = ((int64_t)n + 16 * kCalThreads - 1) / (16 * kCalThreads);
  const int64_t slots = (int64_t)std::min(per_sm, 4) * device_sm_count();
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, slots));
  const float* r = resid;
  int nn = n;
  int64_t rk64 = rank;
  float* o = out_q;
  unsigned int ex = extra;
  uint64_t lim = limit_ns;
  void* args[] = {&r, &nn, &rk64, &S, &o, &ex, &lim};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(select_kernel), dim3(grid),
                                  dim3(kCalThreads), args, 0, st);
  if (e != cudaSuccess) return cuda_fail(e);
  return SV_OK;
}

}  // namespace sv

extern "C" size_t conformal_quantile_workspace(int n) {
  if (n < 1) return 0;
  return round_up(sizeof(SelectState), 256);
}

extern "C" sv_status conformal_quantile(const float* resid, int n, double q, float* out_q,
                                        void* workspace, size_t workspace_bytes,
                                        sv_stream_t stream) {
  if (n < 1 || !(q > 0.0) || !(q <= 1.0)) return SV_ERR_INVALID_ARG;
  if (!resid || !out_q || !aligned_to(resid, 4) || !aligned_to(out_q, 4))
    return SV_ERR_INVALID_ARG;
  const size_t need = round_up(sizeof(SelectState), 256);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < need)
    return SV_ERR_WORKSPACE;
  const double rk = std::ceil((double)(n + 1) * q);  // 1 <= rk <= n + 1
  const int64_t rank = (int64_t)rk;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (rank > (int64_t)n) {
    store_inf<<<1, 1, 0, st>>>(out_q);  // the rank is past the largest score
    return launch_status();
  }
  if (n <= kSmallSelect) {
    select_small_kernel<<<1, kCalThreads, 0, st>>>(resid, n, (int)rank, out_q);
    return launch_status();
  }
  return launch_select(resid, n, rank, out_q, workspace, 0u, kSelWaitNs, st);
}

extern "C" sv_status conformal_quantile_barrier_selftest(const float* resid, int n,
                                                         float* out_q, void* workspace,
                                                         size_t workspace_bytes,
                                                         unsigned int wait_us,
                                                         sv_stream_t stream) {
  if (n <= kSmallSelect || wait_us < 1 || wait_us > 100000) return SV_ERR_INVALID_ARG;
  if (!resid || !out_q || !aligned_to(resid, 4) || !aligned_to(out_q, 4))
    return SV_ERR_INVALID_ARG;
  const size_t need = round_up(sizeof(SelectState), 256);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < need)
    return SV_ERR_WORKSPACE;
  // one arrival more than the grid at every barrier: none completes, every wait runs out
  return launch_select(resid, n, (int64_t)(n / 2 + 1), out_q, workspace, 1u,
                       (uint64_t)wait_us * 1000ull, reinterpret_cast<cudaStream_t>(stream));
}

