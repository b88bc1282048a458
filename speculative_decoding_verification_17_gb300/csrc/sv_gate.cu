// sv_gate.cu — the top-1/top-2 logit-gap confidence gate.
//
// "Speculative Pre-Positioning", section 2.4: gamma = l(1) - l(2), the gap between the two
// largest logits of the cached distribution (Eq. (11)); the gate fires iff gamma > tau and
// the argmax lies in the fast-answer set A (Eq. (12)); section 3.4, Algorithm 2 serves the
// argmax when it fires and falls through otherwise. The page notes that this single scan of
// the vocabulary is the whole critical path of the fast answer (section 2.2, Eq. (3)), so
// the scan is the kernel: every (row, 32 KiB chunk) unit is read once from HBM by one bulk
// copy (sv_stream.cuh), reduced to an (l1, argmax, l2) triple, and the triples of a row are
// merged by the CTA that finishes the row's last chunk.
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"

namespace sv {

constexpr int kPoisonedTop2 = -2;  // marks a chunk whose copy never landed

struct GateArgs {
  const void* logits;
  int N, V, nch;
  double tau;
  const int32_t* answer;
  int n_answer;
  bool aligned;
  int32_t* out_token;
  float* out_gap;
  uint8_t* out_fire;
  ChunkTop2* chunk;
  unsigned int* row_cnt;
};

// Top-2 state of a multiset with the lowest index of its maximum; i1 == kNoIndex = empty.
struct Top2 {
  float m1, m2;
  int i1;
};

__device__ __forceinline__ Top2 top2_merge(const Top2& A, const Top2& B) {
  if (B.i1 == kNoIndex) return A;
  if (A.i1 == kNoIndex) return B;
  if (A.m1 > B.m1 || (A.m1 == B.m1 && A.i1 < B.i1)) return {A.m1, fmaxf(A.m2, B.m1), A.i1};
  return {B.m1, fmaxf(B.m2, A.m1), B.i1};
}

__device__ __forceinline__ Top2 warp_top2(Top2 t) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Top2 u;
    u.m1 = __shfl_xor_sync(0xffffffffu, t.m1, o);
    u.m2 = __shfl_xor_sync(0xffffffffu, t.m2, o);
    u.i1 = __shfl_xor_sync(0xffffffffu, t.i1, o);
    t = top2_merge(t, u);
  }
  return t;
}

__device__ __forceinline__ bool in_sorted(const int32_t* a, int n, int v) {
  int lo = 0, hi = n;  // first index with a[i] >= v
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) < v) lo = mid + 1;
    else hi = mid;
  }
  return lo < n && __ldg(a + lo) == v;
}

template <typename ET>
struct GateOp {
  using Args = GateArgs;
  using E = ET;
  static constexpr uint32_t kPad = E::kNaNBits;  // NaN padding is skipped
  struct Smem {
    float m1[kWarps], m2[kWarps];
    int i1[kWarps];
    int row_last;
  };

  __device__ static bool unit_row(const Args& A, int64_t u, const void*& row, int64_t& j0,
                                  int64_t& j1) {
    const int r = (int)(u / A.nch);
    const int c = (int)(u - (int64_t)r * A.nch);
    row = static_cast<const char*>(A.logits) + (int64_t)r * A.V * (16 / E::kPerVec);
    j0 = (int64_t)c * E::kChunk;
    j1 = j0 + E::kChunk < A.V ? j0 + E::kChunk : (int64_t)A.V;
    return true;
  }

  __device__ static void process(const Args& A, int64_t u, const void* rowp, int64_t j0,
                                 int64_t j1, const unsigned char* chunk, bool poisoned,
                                 Smem& sm) {
    const int row = (int)(u / A.nch);
    const int c = (int)(u - (int64_t)row * A.nch);
    Top2 t{-INFINITY, -INFINITY, kNoIndex};
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const uint4 v = chunk_vec<E>(chunk, it, j0, j1, kPad);
      const int jb = (int)(j0 + (int64_t)(it * kThreads + threadIdx.x) * E::kPerVec);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) {
        const float z = E::get(v, l);
        if (z != z) continue;
        if (t.i1 == kNoIndex) {
          t.m1 = z;
          t.i1 = jb + l;
        } else if (z > t.m1) {
          t.m2 = t.m1;
          t.m1 = z;
          t.i1 = jb + l;
        } else {
          t.m2 = fmaxf(t.m2, z);
        }
      }
    }
    t = warp_top2(t);
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
      sm.m1[w] = t.m1;
      sm.m2[w] = t.m2;
      sm.i1[w] = t.i1;
    }
    cbar();
    if (threadIdx.x == 0) {
      Top2 b{sm.m1[0], sm.m2[0], sm.i1[0]};
      for (int q = 1; q < kWarps; ++q) b = top2_merge(b, Top2{sm.m1[q], sm.m2[q], sm.i1[q]});
      ChunkTop2* p = A.chunk + (int64_t)row * A.nch + c;
      p->m1 = b.m1;
      p->i1 = poisoned ? kPoisonedTop2 : b.i1;
      p->m2 = b.m2;
      sm.row_last = arrive_last(A.row_cnt + row, (unsigned)A.nch);
    }
    cbar();
    if (!sm.row_last) return;
    __threadfence();

    if (threadIdx.x < 32) {
      Top2 b{-INFINITY, -INFINITY, kNoIndex};
      bool poison = false;
      for (int cc = lane; cc < A.nch; cc += 32) {
        const ChunkTop2* p = A.chunk + (int64_t)row * A.nch + cc;
        const int pi = __ldcg(&p->i1);
        poison |= pi == kPoisonedTop2;
        if (pi != kPoisonedTop2) b = top2_merge(b, Top2{__ldcg(&p->m1), __ldcg(&p->m2), pi});
      }
      b = warp_top2(b);
      poison = __any_sync(0xffffffffu, poison);
      if (lane == 0) {
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
  const int64_t units = (int64_t)N * nch;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const GateLayout L = gate_layout(N, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  GateArgs A;
  A.logits = logits;
  A.N = N;
  A.V = V;
  A.nch = (int)nch;
  A.tau = (double)tau;
  A.answer = answer_set;
  A.n_answer = n_answer;
  A.aligned = aligned_to(logits, 16) && ((int64_t)V * eb) % 16 == 0;
  A.out_token = out_token;
  A.out_gap = out_gap;
  A.out_fire = out_fire;
  char* ws = static_cast<char*>(workspace);
  A.chunk = reinterpret_cast<ChunkTop2*>(ws + L.chunk);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws + L.ctl, 0, L.total - L.ctl, st);
  if (e != cudaSuccess) return cuda_fail(e);
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_units<GateOp<F32>>(A, units, ctl, st);
  return launch_units<GateOp<BF16>>(A, units, ctl, st);
}
