// sv_gate.cu — the top-1/top-2 logit-gap confidence gate.
//
// "Speculative Pre-Positioning", section 2.4: gamma = l(1) - l(2), the gap between the two
// largest logits of the cached distribution (Eq. (11)); the gate fires iff gamma > tau and
// the argmax lies in the fast-answer set A (Eq. (12)); section 3.4, Algorithm 2 serves the
// argmax when it fires and falls through otherwise. The page notes that this single scan of
// the vocabulary is the whole critical path of the fast answer (section 2.2, Eq. (3)), so
// the scan is the kernel: every logit is read once from HBM by the bulk copies of
// sv_stream.cuh, each lane keeps a running (l1, argmax, l2) triple over its share of a row
// segment, each warp reduces its lanes once per segment, and the triples of a row are merged
// by the CTA that completes the row.
//
// The conformal gate of the "speculative-decoding-plan.md" note ("Axis 1 reuses the gate we
// already have: 2*tau <= gamma") is the same scan with another threshold rule: row n*K + k
// holds step n's early-exit logits at layer k, the row admits iff 2 Q[k] <= gamma, and the
// step takes its earliest admitting layer (an atomic maximum of (K - k, a_hat) per step,
// read by the row that completes the step).
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "specverify_calib.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"
#include "sv_top2.cuh"

namespace sv {

struct GateArgs {
  const void* logits;
  int N, V, nch, nseg;
  double tau;
  const int32_t* answer;
  int n_answer;
  bool aligned;
  int32_t* out_token;
  float* out_gap;
  uint8_t* out_fire;
  WarpTop2* part;  // [N][nseg][kWarps]
  unsigned int* row_cnt;
  // conformal gate only
  const float* Q;                // [K]
  int K;                         // layers per step (rows n*K .. n*K + K - 1)
  int32_t* out_layer;            // [N / K]
  unsigned long long* best;      // [N / K]: max of (K - k) << 32 | a_hat over admitting rows
  unsigned int* step_cnt;        // [N / K]
};

template <typename ET, bool kConformal = false>
struct GateOp : Top2Scan<ET> {
  using Args = GateArgs;
  using Base = Top2Scan<ET>;
  using typename Base::E;
  using typename Base::Smem;

  __device__ static bool unit(const Args& A, int64_t u, Seg& g) {
    const int r = (int)(u / A.nseg);
    const int seg = (int)(u - (int64_t)r * A.nseg);
    g.row = static_cast<const char*>(A.logits) + (int64_t)r * A.V * (16 / E::kPerVec);
    g.rid = r;
    g.r = r;
    g.slot = 0;
    g.seg = seg;
    g.keep = false;
    g.c0 = seg * kSegChunks;
    g.c1 = min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring&) {
    const int row = g.r;
    const int lane = threadIdx.x & 31;
    if (!Base::row_complete(A, g, sm)) return;
    if (threadIdx.x < 32) {
      bool poison;
      const Top2 b = Base::row_top2(A, g, sm, poison);
      if (kConformal) {
        if (lane == 0) conformal_finish(A, row, b, !(b.i1 == kNoIndex || poison));
      } else if (lane == 0) {
        if (b.i1 == kNoIndex || poison) {
          A.out_token[row] = -1;
          A.out_gap[row] = __int_as_float(0x7fc00000);
          A.out_fire[row] = 0;
        } else {
          const double gap = (double)b.m1 - (double)b.m2;
          const bool fire =
              gap > A.tau && A.n_answer > 0 && in_sorted(A.answer, A.n_answer, b.i1);
          A.out_token[row] = b.i1;
          A.out_gap[row] = (float)gap;
          A.out_fire[row] = fire ? 1 : 0;
        }
      }
    }
  }

  // One row of the conformal gate (lane 0 of the CTA that completed it).
  __device__ static void conformal_finish(const Args& A, int row, const Top2& b, bool ok) {
    const int K = A.K;
    const int n = row / K, k = row - n * K;
    const double gap = ok ? (double)b.m1 - (double)b.m2 : 0.0;
    if (A.out_gap) A.out_gap[row] = ok ? (float)gap : __int_as_float(0x7fc00000);
    const bool admit = ok && 2.0 * (double)__ldg(A.Q + k) <= gap;
    if (K == 1) {
      A.out_layer[n] = admit ? 0 : 1;
      A.out_token[n] = admit ? b.i1 : -1;
      return;
    }
    if (admit)
      atomicMax(A.best + n, ((unsigned long long)(K - k) << 32) | (unsigned int)b.i1);
    __threadfence();
    if (!arrive_last(A.step_cnt + n, (unsigned)K)) return;
    __threadfence();
    const unsigned long long v = atomicOr(A.best + n, 0ull);  // an atomic read
    const int hi = (int)(v >> 32);
    A.out_layer[n] = hi ? K - hi : K;
    A.out_token[n] = hi ? (int)(unsigned int)(v & 0xffffffffull) : -1;
  }
};

}  // namespace sv

using namespace sv;

extern "C" size_t logit_gap_gate_workspace(int N, int V, sv_dtype dtype) {
  if (N < 0 || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return gate_layout(N, V, dtype).total;
}

extern "C" sv_status logit_gap_gate(const void* logits, sv_dtype dtype, int N, int V, float tau,
                                    const int32_t* answer_set, int n_answer, int32_t* out_token,
                                    float* out_gap, uint8_t* out_fire, void* workspace,
                                    size_t workspace_bytes, sv_stream_t stream) {
  if (N < 0 || V < 2 || n_answer < 0) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (N == 0) return SV_OK;
  if (!logits || !out_token || !out_gap || !out_fire || (n_answer > 0 && !answer_set))
    return SV_ERR_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned_to(logits, eb) || !aligned_to(out_token, 4) || !aligned_to(out_gap, 4) ||
      (answer_set && !aligned_to(answer_set, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = (int64_t)N * nseg;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const GateLayout L = gate_layout(N, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  GateArgs A{};
  A.logits = logits;
  A.N = N;
  A.V = V;
  A.nch = (int)nch;
  A.nseg = nseg;
  A.tau = (double)tau;
  A.answer = answer_set;
  A.n_answer = n_answer;
  A.aligned = aligned_to(logits, 16) && ((int64_t)V * eb) % 16 == 0;
  A.out_token = out_token;
  A.out_gap = out_gap;
  A.out_fire = out_fire;
  char* ws = static_cast<char*>(workspace);
  A.part = reinterpret_cast<WarpTop2*>(ws + L.part);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const sv_status cleared = launch_clear(ws + L.ctl, L.total - L.ctl, st);
  if (cleared != SV_OK) return cleared;
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_segments<GateOp<F32>>(A, units, ctl, st);
  return launch_segments<GateOp<BF16>>(A, units, ctl, st);
}

namespace {
struct ConfGateLayout {
  size_t part, ctl, row_cnt, best, step_cnt, total;
};
ConfGateLayout conf_gate_layout(int N, int K, int V, sv_dtype d) {
  const size_t rows = (size_t)N * (size_t)K;
  const size_t nseg = static_cast<size_t>(num_segments(num_chunks(V, d)));
  ConfGateLayout L{};
  size_t o = 0;
  L.part = o;     o = round_up(o + rows * nseg * kWarpsPerChunk * sizeof(WarpTop2), 256);
  L.ctl = o;      o = round_up(o + sizeof(CallCtl), 256);
  L.row_cnt = o;  o = round_up(o + rows * sizeof(unsigned int), 256);
  L.best = o;     o = round_up(o + (size_t)N * sizeof(unsigned long long), 256);
  L.step_cnt = o; o = round_up(o + (size_t)N * sizeof(unsigned int), 256);
  L.total = o;
  return L;
}
}  // namespace

extern "C" size_t conformal_admit_workspace(int N, int K, int V, sv_dtype dtype) {
  if (N < 0 || K < 1 || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  if ((int64_t)N * K > 0x7fffffffLL) return 0;
  return conf_gate_layout(N, K, V, dtype).total;
}

extern "C" sv_status conformal_admit(const void* logits, sv_dtype dtype, int N, int K, int V,
                                     const float* Q, int32_t* out_layer, int32_t* out_token,
                                     float* out_gap, void* workspace, size_t workspace_bytes,
                                     sv_stream_t stream) {
  if (N < 0 || K < 1 || V < 2) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (N == 0) return SV_OK;
  if (!logits || !Q || !out_layer || !out_token) return SV_ERR_INVALID_ARG;
  const int eb = elem_bytes(dtype);
  if (!aligned_to(logits, eb) || !aligned_to(Q, 4) || !aligned_to(out_layer, 4) ||
      !aligned_to(out_token, 4) || (out_gap && !aligned_to(out_gap, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)N * K;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = rows * nseg;
  if (rows > 0x7fffffffLL || units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const ConfGateLayout L = conf_gate_layout(N, K, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  GateArgs A{};
  A.logits = logits;
  A.N = (int)rows;
  A.V = V;
  A.nch = (int)nch;
  A.nseg = nseg;
  A.tau = 0.0;
  A.answer = nullptr;
  A.n_answer = 0;
  A.aligned = aligned_to(logits, 16) && ((int64_t)V * eb) % 16 == 0;
  A.out_token = out_token;
  A.out_gap = out_gap;
  A.out_fire = nullptr;
  char* ws = static_cast<char*>(workspace);
  A.part = reinterpret_cast<WarpTop2*>(ws + L.part);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.Q = Q;
  A.K = K;
  A.out_layer = out_layer;
  A.best = reinterpret_cast<unsigned long long*>(ws + L.best);
  A.step_cnt = reinterpret_cast<unsigned int*>(ws + L.step_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const sv_status cleared = launch_clear(ws + L.ctl, L.total - L.ctl, st);
  if (cleared != SV_OK) return cleared;
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_segments<GateOp<F32, true>>(A, units, ctl, st);
  return launch_segments<GateOp<BF16, true>>(A, units, ctl, st);
}
