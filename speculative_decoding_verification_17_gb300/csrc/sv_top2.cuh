// sv_top2.cuh — the top-1/top-2 scan of a logit row on the segment driver, shared by the
// logit-gap gate (sv_gate.cu) and the ready-distribution cache's record step (sv_cache.cu).
//
// Each lane keeps a running (l1, argmax, l2) triple over its share of a row segment: per ring
// stage the stage's top two by a tournament, folded into the triple; each warp reduces its
// lanes once per segment; the CTA that completes the row merges the warp partials.
#pragma once

#include <cmath>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"

namespace sv {

constexpr int kPoisonedTop2 = -2;  // marks a share of which a copy never landed

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

// ---- the top two of a lane's ring stage, as a tournament of (largest, second) pairs ----
// Two sets with tops (H1, L1) and (H2, L2) have top two H = max(H1, H2) and
// L = max(min(H1, H2), max(L1, L2)) (a tie keeps both copies: the multiset's second largest).
// The maxima propagate NaN, so a stage holding a NaN gives Ms = NaN and is rescanned.
__device__ __forceinline__ uint32_t bmaxn2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float fmaxn(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// bf16: packed pairs, each 16-bit half keeping the top two of its own half of the stage.
template <int N>
__device__ __forceinline__ void stage_top2(const uint4 (&v)[N], float& Ms, float& ms) {
  uint32_t H[2 * N], L[2 * N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    H[2 * i] = bmaxn2(v[i].x, v[i].y);
    L[2 * i] = bmin2(v[i].x, v[i].y);
    H[2 * i + 1] = bmaxn2(v[i].z, v[i].w);
    L[2 * i + 1] = bmin2(v[i].z, v[i].w);
  }
#pragma unroll
  for (int q = N; q >= 1; q >>= 1)
#pragma unroll
    for (int i = 0; i < q; ++i) {
      const uint32_t h = bmaxn2(H[i], H[i + q]);
      L[i] = bmaxn2(bmin2(H[i], H[i + q]), bmaxn2(L[i], L[i + q]));
      H[i] = h;
    }
  const float ha = __uint_as_float(H[0] << 16), hb = __uint_as_float(H[0] & 0xffff0000u);
  const float la = __uint_as_float(L[0] << 16), lb = __uint_as_float(L[0] & 0xffff0000u);
  Ms = fmaxn(ha, hb);
  ms = fmaxn(fminf(ha, hb), fmaxn(la, lb));
}

// fp32: the same tournament on the stage's 4N logits.
template <int N>
__device__ __forceinline__ void stage_top2_f32(const uint4 (&v)[N], float& Ms, float& ms) {
  float H[2 * N], L[2 * N];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float a = __uint_as_float(v[i].x), b = __uint_as_float(v[i].y);
    const float c = __uint_as_float(v[i].z), d = __uint_as_float(v[i].w);
    H[2 * i] = fmaxn(a, b);
    L[2 * i] = fminf(a, b);
    H[2 * i + 1] = fmaxn(c, d);
    L[2 * i + 1] = fminf(c, d);
  }
#pragma unroll
  for (int q = N; q >= 1; q >>= 1)
#pragma unroll
    for (int i = 0; i < q; ++i) {
      const float h = fmaxn(H[i], H[i + q]);
      L[i] = fmaxn(fminf(H[i], H[i + q]), fmaxn(L[i], L[i + q]));
      H[i] = h;
    }
  Ms = H[0];
  ms = L[0];
}

// The scan part of an op over whole rows: its tile, padding, accumulator, per-stage fold and
// per-segment warp reduction. Args must provide `part` (WarpTop2 [rows][nseg][kWarps]) and
// `nseg`; Smem must provide `wpart` (float4 [kWarps]) and `row_last`.
template <typename ET>
struct Top2Scan {
  using E = ET;
  using T = SV_TILE(4, 2, 4);  // a light scan: half-chunk stages, 4 CTAs per SM
  static constexpr uint32_t kPad = E::kNaNBits;  // NaN padding is skipped
  struct Smem {
    float4 wpart[kWarps];  // the warp partials of this segment
    int row_last;
  };

  // One lane's running top-2 over the segment, in increasing logit index.
  struct Acc {
    Top2 t;
    bool poison;
  };

  __device__ static __forceinline__ void seg_begin(Acc& a) {
    a.t = Top2{-INFINITY, -INFINITY, kNoIndex};
    a.poison = false;
  }

  template <class Args>
  __device__ static __forceinline__ void warp_slice(const Args&, const Seg&, int64_t j0,
                                                    const uint4 (&v)[T::kStageVec],
                                                    bool poison, Acc& acc) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    acc.poison |= poison;
    Top2& t = acc.t;
    // The stage's top two by a tournament (a NaN anywhere makes Ms NaN); folded into the
    // lane's state, with the stage scanned for the index only when its maximum takes over.
    float Ms, ms;
    if constexpr (E::kPerVec == 8) stage_top2(v, Ms, ms);
    else stage_top2_f32(v, Ms, ms);
    if (Ms == Ms) {
      const bool take = Ms > t.m1 || t.i1 == kNoIndex;
      t.m2 = fmaxf(fminf(t.m1, Ms), fmaxf(t.m2, ms));
      if (take) {
        t.m1 = Ms;
        t.i1 = first_index(v, j0, w, lane, Ms);
      }
      return;
    }
    // a stage with NaN entries (or the row's NaN-padded end): logit by logit, NaN skipped
#pragma unroll
    for (int it = 0; it < T::kStageVec; ++it) {
      const int jb = (int)(j0 + (int64_t)warp_vec_slot<T::kStageVec>(w, it, lane) * E::kPerVec);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) {
        const float z = E::get(v[it], l);
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
  }

  // Lowest index of the lane's stage logits equal to M (one of them is).
  __device__ static __forceinline__ int first_index(const uint4 (&v)[T::kStageVec], int64_t j0,
                                                    int w, int lane, float M) {
#pragma unroll
    for (int it = 0; it < T::kStageVec; ++it) {
      const int jb = (int)(j0 + (int64_t)warp_vec_slot<T::kStageVec>(w, it, lane) * E::kPerVec);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l)
        if (E::get(v[it], l) == M) return jb + l;
    }
    return kNoIndex;
  }

  template <class Args, class S>
  __device__ static __forceinline__ void prologue(const Args&, const Seg&, S&) {}

  template <class Args, class S>
  __device__ static __forceinline__ void seg_end(const Args& A, const Seg& g, Acc& acc, S& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool poison = __any_sync(0xffffffffu, acc.poison);
    const Top2 t = warp_top2(acc.t);
    if (lane == 0) {
      const float4 out =
          make_float4(t.m1, __int_as_float(poison ? kPoisonedTop2 : t.i1), t.m2, 0.0f);
      sm.wpart[w] = out;
      if (g.nseg > 1)
        *reinterpret_cast<float4*>(A.part + ((g.rid * A.nseg + g.seg) * kWarps + w)) = out;
    }
  }


  // Whether this CTA completes the row (all threads; thread 0 arrives on the row counter). A
  // row of one segment is complete here: no counter, and its partials are this CTA's.
  template <class Args, class S>
  __device__ static bool row_complete(const Args& A, const Seg& g, S& sm) {
    if (threadIdx.x == 0)
      sm.row_last = g.nseg == 1 || arrive_last(A.row_cnt + g.rid, (unsigned)g.nseg);
    __syncthreads();
    if (!sm.row_last) return false;
    if (g.nseg > 1) __threadfence();
    return true;
  }

  // The row's top two from its warp partials (warp 0; every lane gets the result).
  template <class Args, class S>
  __device__ static Top2 row_top2(const Args& A, const Seg& g, const S& sm, bool& poison) {
    const int lane = threadIdx.x & 31;
    const int np = A.nseg * kWarps;
    const WarpTop2* wp = A.part + (int64_t)g.rid * np;
    Top2 b{-INFINITY, -INFINITY, kNoIndex};
    bool bad = false;
    for (int q = lane; q < np; q += 32) {
      const float4 pv =
          g.nseg > 1 ? __ldcg(reinterpret_cast<const float4*>(wp + q)) : sm.wpart[q];
      const int pi = __float_as_int(pv.y);
      bad |= pi == kPoisonedTop2;
      if (pi != kPoisonedTop2) b = top2_merge(b, Top2{pv.x, pv.z, pi});
    }
    b = warp_top2(b);
    poison = __any_sync(0xffffffffu, bad);
    return b;
  }
};

}  // namespace sv
