// sv_verify.cu — sampled (modified rejection) and greedy speculative-decoding verify.
//
// Sampled verify, as "Speculative Decoding: The Physics of Stolen Time in Autoregressive
// Inference" states it in section 2 (accept with min(1, p/q), resample a rejection from
// norm(max(0, p - q))) and section 1, stage 3 (keep the longest accepted prefix; a bonus
// token from p when all k are accepted), and as the "speculative-decoding-plan.md" design
// note restates it under "The acceptance math (standard speculative sampling)".
//
// Greedy verify, as "The Inference Wall, Part 7" states it under "How speculative decoding
// works" (accept while the draft token is the target's own pick, then emit the target's
// pick).
//
// One kernel launch per call (after a small memset of the call's counters). Unit = (request
// r, row slot, segment of up to four 32 KiB chunks), one CTA each (sv_stream.cuh); a request
// has 2k+1 row slots in the sampled verify (target rows 0..k, then draft rows 0..k-1) and k+1
// in the greedy verify. Units of rows a request does not need (past its n_r) exit at once.
//
//  pass 1 (every warp slice of 4 KiB)  the slice maximum m, the integer-valued reference
//                           K = ceil(m*s) with s = log2(e)/T in fp32, and the sum of
//                           2^(z*s - K) in fp32 (compensated across the warp); in the greedy
//                           verify the slice argmax.
//  row finish (the CTA that completes the row)  K_row = max K; S = sum of slice sums times
//                           2^(K - K_row), exact powers of two, in double; p(x) =
//                           2^(z_x*s - K_row) / S in double.
//  request finish (the CTA that completes the request)  ratios p_i(x_i)/q_i(x_i) in double
//                           against the uniforms, the accepted prefix a, then one draw: the
//                           residual max(0, p_a - q_a) (one extra pass over the rejected row
//                           pair, which L2 still holds, for per-chunk residual masses, then one
//                           chunk scanned in vocabulary order), or the bonus from p_n (chunk
//                           masses from the pass-1 partials, one chunk scanned).
#include <cmath>
#include <cstdint>
#include <mutex>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"

#ifndef SV_RESID_RING
#define SV_RESID_RING 1  // residual pass through the TMA ring (0: register loads)
#endif

namespace sv {

constexpr int kPoisoned = -2;  // an index that marks a slice whose copy never landed

template <typename E>
__device__ __forceinline__ const void* row_ptr(const void* base, int64_t row, int V) {
  return static_cast<const char*>(base) + row * (int64_t)V * (16 / E::kPerVec);
}

template <typename E>
__device__ __forceinline__ int64_t chunk_end(int64_t j0, int V) {
  return j0 + E::kChunk < V ? j0 + E::kChunk : (int64_t)V;
}

// ============================================================================================
// In-order draw inside one chunk
// ============================================================================================
struct ScanSmem {
  double seg_tot[kWarps];
  int seg_last[kWarps];
  double owner_excl;
  int owner;
  int result;
};

// Inverse-CDF draw inside the chunk that starts at j0: the first logit j, in vocabulary
// order, whose running weight exceeds `target` (chunk units); when rounding leaves the
// target at or past the chunk's total, the last logit with positive weight. Warp w owns the
// contiguous segment [j0 + w*kSeg, j0 + (w+1)*kSeg) and reads it in rounds of 32*kPerVec
// logits (one coalesced 16-byte vector per lane per round, two rounds loaded at once).
// Lane sums are sequential fp32, round totals come from an inclusive warp scan in double,
// segment totals are sequential sums of round totals. The owning warp replays exactly the
// same loads and arithmetic, so the crossing is found there.
// VW provides: using Raw; Raw load(int64_t j) const; void weights(const Raw&, float (&)[]),
// with zero weight past the end of the row. Every consumer thread must call this.
template <typename E, typename VW>
__device__ int scan_chunk(int64_t j0, double target, bool take_last, const VW& vw,
                          ScanSmem& sm) {
  constexpr int kSeg = E::kChunk / kWarps;
  constexpr int kRound = 32 * E::kPerVec;
  constexpr int kRounds = kSeg / kRound;
  constexpr int kBatch = 2;  // rounds loaded at once
  static_assert(kRounds * kRound == kSeg && kRounds % kBatch == 0, "whole rounds and batches");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t seg0 = j0 + (int64_t)warp * kSeg;

  double seg = 0.0;
  int lastpos = -1;
#pragma unroll 1
  for (int b = 0; b < kRounds; b += kBatch) {
    typename VW::Raw raw[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q)
      raw[q] = vw.load(seg0 + (b + q) * kRound + lane * E::kPerVec);
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      float w[E::kPerVec];
      vw.weights(raw[q], w);
      float ls = 0.0f;
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) {
        ls += w[l];
        if (w[l] > 0.0f) lastpos = (int)(seg0 + (b + q) * kRound + lane * E::kPerVec + l);
      }
      const double incl = warp_scan_d((double)ls);
      seg += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  lastpos = __reduce_max_sync(0xffffffffu, lastpos);
  if (lane == 0) {
    sm.seg_tot[warp] = seg;
    sm.seg_last[warp] = lastpos;
  }
  cbar();
  if (threadIdx.x == 0) {
    double run = 0.0;
    int owner = -1, last = -1;
    for (int w = 0; w < kWarps; ++w) {
      if (owner < 0 && !take_last && sm.seg_tot[w] > 0.0 && run + sm.seg_tot[w] > target) {
        owner = w;
        sm.owner_excl = run;
      }
      if (owner < 0) run += sm.seg_tot[w];
      last = max(last, sm.seg_last[w]);
    }
    sm.owner = owner;
    sm.result = owner < 0 ? last : sm.seg_last[owner];
  }
  cbar();
  if (warp == sm.owner) {
    // replay: the same loads (identical bits) and the same arithmetic, round by round
    double run = sm.owner_excl;
#pragma unroll 1
    for (int ro = 0; ro < kRounds; ++ro) {
      const typename VW::Raw raw = vw.load(seg0 + ro * kRound + lane * E::kPerVec);
      float w[E::kPerVec];
      vw.weights(raw, w);
      float ls = 0.0f;
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) ls += w[l];
      const double incl = warp_scan_d((double)ls);
      const double tot = __shfl_sync(0xffffffffu, incl, 31);
      if (run + tot > target) {
        const unsigned bal = __ballot_sync(0xffffffffu, ls > 0.0f && run + incl > target);
        const int L = bal ? __ffs(bal) - 1 : 31;
        const double excl = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == L) {
          double r2 = run + (lane ? excl : 0.0);
          int t = -1, lp = -1;
#pragma unroll
          for (int l = 0; l < E::kPerVec; ++l) {
            if (w[l] > 0.0f) lp = (int)(seg0 + ro * kRound + lane * E::kPerVec + l);
            r2 += (double)w[l];
            if (t < 0 && r2 > target && w[l] > 0.0f) t = lp;
          }
          if (t >= 0 || lp >= 0) sm.result = t >= 0 ? t : lp;
        }
        break;  // warp-uniform
      }
      run += tot;
    }
  }
  cbar();
  return sm.result;
}

// Chunk choice for an inverse-CDF draw over per-chunk masses mass(c), c in [0, nch): the
// first chunk whose running total exceeds target. Run by one full warp. Returns the chunk
// (or, when rounding leaves none, the last chunk with positive mass and take_last = true)
// and the running total before it.
template <typename MF>
__device__ int pick_chunk(int nch, double target, MF mass, double& before, bool& take_last) {
  const int lane = threadIdx.x & 31;
  double run = 0.0;
  int last_pos = -1;
  double last_before = 0.0;
  for (int c0 = 0; c0 < nch; c0 += 32) {
    const int c = c0 + lane;
    const double m = c < nch ? mass(c) : 0.0;
    const double incl = warp_scan_d(m);
    const bool cross = c < nch && m > 0.0 && run + incl > target;
    const unsigned bal = __ballot_sync(0xffffffffu, cross);
    if (bal) {
      const int fl = __ffs(bal) - 1;
      before = run + __shfl_sync(0xffffffffu, incl - m, fl);
      take_last = false;
      return c0 + fl;
    }
    const unsigned pos = __ballot_sync(0xffffffffu, c < nch && m > 0.0);
    if (pos) {
      const int ll = 31 - __clz(pos);
      last_pos = c0 + ll;
      last_before = run + __shfl_sync(0xffffffffu, incl - m, ll);
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
  }
  before = last_before;
  take_last = true;
  return last_pos;
}

// ============================================================================================
// Sampled verify
// ============================================================================================
struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* num_draft;
  const float* uniforms;
  int B, k, V, nch, nseg;
  float s;       // log2(e) / T, rounded to fp32
  bool aligned;  // every row starts on a 16-byte boundary
  int32_t* out_tokens;
  int32_t* out_accept_len;
  float* out_p;
  float* out_q;
  float* out_resid;
  WarpSoftmax* part;  // [B * (2k+1)][nch][kWarps]
  RowSoftmax* row;
  double* resid;      // [B][nch][kWarps] residual partial masses
  unsigned int* row_cnt;
  unsigned int* req_cnt;
};

// 2^d for an integer d <= 0, exactly (0 below the double range).
__device__ __forceinline__ double pow2i(int d) {
  return d < -1022 ? 0.0 : __longlong_as_double((long long)(1023 + d) << 52);
}

// Residual weight max(0, p_j - q_j) with both normalisers folded in (row units).
struct ResidW {
  float s, cp, cq, ip, iq;
  __device__ __forceinline__ float operator()(float zp, float zq) const {
    const float ep = ex2(fmaf(zp, s, cp));
    const float eq = ex2(fmaf(zq, s, cq));
    return fmaxf(0.0f, fmaf(ep, ip, -(eq * iq)));
  }
};

template <typename E>
struct ResidScan {
  const void* rp;
  const void* rq;
  int64_t j1;
  bool aligned;
  ResidW wf;
  struct Raw {
    uint4 p, q;
  };
  __device__ __forceinline__ Raw load(int64_t j) const {
    return {load_vec<E>(rp, j, j1, aligned, E::kNegInfBits),
            load_vec<E>(rq, j, j1, aligned, E::kNegInfBits)};
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) w[l] = wf(E::get(r.p, l), E::get(r.q, l));
  }
};

template <typename E>
struct BonusScan {
  const void* row;
  int64_t j1;
  bool aligned;
  float s, c;  // weight 2^(z*s + c), c = -K of the row
  using Raw = uint4;
  __device__ __forceinline__ Raw load(int64_t j) const {
    return load_vec<E>(row, j, j1, aligned, E::kNegInfBits);
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) w[l] = ex2(fmaf(E::get(r, l), s, c));
  }
};

// The same weights read from a chunk staged in shared memory (vector i of the chunk at
// p + 16*i, likewise q), for the in-chunk scan after a bulk copy of the chosen chunk.
template <typename E>
struct ResidScanSmem {
  const unsigned char* p;
  const unsigned char* q;
  int64_t j0, j1;
  ResidW wf;
  struct Raw {
    uint4 p, q;
  };
  __device__ __forceinline__ Raw load(int64_t j) const {
    if (j >= j1) return {E::pad_vec(E::kNegInfBits), E::pad_vec(E::kNegInfBits)};
    const int i = (int)((j - j0) / E::kPerVec);
    return {lds16(p + i * 16), lds16(q + i * 16)};
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) w[l] = wf(E::get(r.p, l), E::get(r.q, l));
  }
};

template <typename E>
struct BonusScanSmem {
  const unsigned char* p;
  int64_t j0, j1;
  float s, c;
  using Raw = uint4;
  __device__ __forceinline__ Raw load(int64_t j) const {
    if (j >= j1) return E::pad_vec(E::kNegInfBits);
    return lds16(p + (int)((j - j0) / E::kPerVec) * 16);
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) w[l] = ex2(fmaf(E::get(r, l), s, c));
  }
};

// Stage chunk [j0, j1) of a row into ring stage `st` with one bulk copy (thread 0), then wait
// for it (every thread). False if the copy never landed.
template <typename E>
__device__ bool stage_chunk(Ring& ring, int st, const void* row, int64_t j0, int64_t j1) {
  if (threadIdx.x == 0) {
    const uint32_t bytes = (uint32_t)((j1 - j0) * (16 / E::kPerVec));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive_expect_tx(&ring.full[st], bytes);
    bulk_g2s(ring.buf + st * kChunkBytes, static_cast<const char*>(row) + j0 * (16 / E::kPerVec),
             bytes, &ring.full[st]);
  }
  return ring_wait(ring, st);
}

__device__ __forceinline__ WarpSoftmax ld_part(const WarpSoftmax* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  return {v.x, v.y, v.z, v.w};
}

__device__ __forceinline__ RowSoftmax ld_row(const RowSoftmax* p) {
  RowSoftmax r;
  r.S = __ldcg(&p->S);
  r.px = __ldcg(&p->px);
  r.K = __ldcg(&p->K);
  r.status = __ldcg(&p->status);
  return r;
}

// Mass of a warp slice in units of 2^K (K the row reference): exact power-of-two scaling.
__device__ __forceinline__ double part_mass(const WarpSoftmax& w, float K) {
  if (!(w.K > -INFINITY)) return w.K == -INFINITY ? 0.0 : w.hi;  // empty, or NaN (poisoned)
  return ((double)w.hi + (double)w.lo) * pow2i((int)(w.K - K));
}

template <typename ET>
struct SampleOp {
  using Args = SampleArgs;
  using E = ET;
  static constexpr uint32_t kPad = E::kNegInfBits;
  struct Smem {
    float red[2 * kWarps];
    int row_last, req_last;
    int a, err, chunk, take_last;
    double W, before;
    ScanSmem scan;
  };

  __device__ static __forceinline__ int n_of(const Args& A, int r, bool& ok) {
    const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
    ok = nraw >= 0 && nraw <= A.k;
    return ok ? nraw : A.k;
  }

  __device__ static bool unit(const Args& A, int64_t u, Seg& g) {
    const int R = 2 * A.k + 1;
    const int r = (int)(u / ((int64_t)R * A.nseg));
    const int rem = (int)(u - (int64_t)r * R * A.nseg);
    const int slot = rem / A.nseg;
    const int seg = rem - slot * A.nseg;
    bool ok;
    const int n = n_of(A, r, ok);
    const bool is_target = slot <= A.k;
    const int i = is_target ? slot : slot - A.k - 1;
    if (is_target ? i > n : i >= n) return false;
    g.row = is_target ? row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + i, A.V)
                      : row_ptr<E>(A.draft, (int64_t)r * A.k + i, A.V);
    g.rid = (int64_t)r * R + slot;
    g.r = r;
    g.slot = slot;
    g.c0 = seg * kSegChunks;
    g.c1 = min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  // Pass 1 for one warp slice: its maximum m, the integer reference K = ceil(m*s) and the
  // sum of 2^(z*s - K) (pairwise in fp32 per lane, compensated across the warp).
  __device__ static void warp_chunk(const Args& A, const Seg& g, int c,
                                    const uint4 (&v)[kVecPerThread], bool poison) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float tmax = -INFINITY;
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) tmax = fmaxf(tmax, E::max_vec(v[it]));
    const float m = warp_max_f(tmax);
    WarpSoftmax out;
    if (poison || !(m > -INFINITY && m < INFINITY)) {
      // no finite logit: a masked slice carries no mass; NaN or +inf poison the row
      bool nan = false;
#pragma unroll
      for (int it = 0; it < kVecPerThread; ++it)
#pragma unroll
        for (int l = 0; l < E::kPerVec; ++l) nan |= E::get(v[it], l) != E::get(v[it], l);
      nan = __any_sync(0xffffffffu, nan);
      const float bad = __int_as_float(0x7fc00000);
      out = (poison || nan || m == INFINITY) ? WarpSoftmax{bad, bad, 0.0f, 0.0f}
                                             : WarpSoftmax{-INFINITY, 0.0f, 0.0f, 0.0f};
    } else {
      const float s = A.s;
      const float K = ceilf(m * s);
      // logits two at a time: packed fp32x2 FMA and adds, two SFU exp2 per pair
      const float2 s2 = make_float2(s, s), c2 = make_float2(-K, -K);
      float2 part[kVecPerThread];
#pragma unroll
      for (int it = 0; it < kVecPerThread; ++it) {
        float2 e[E::kPerVec / 2];
#pragma unroll
        for (int p = 0; p < E::kPerVec / 2; ++p) {
          const float2 x = __ffma2_rn(E::get2(v[it], p), s2, c2);
          e[p] = make_float2(ex2(x.x), ex2(x.y));
        }
#pragma unroll
        for (int q = E::kPerVec / 4; q >= 1; q >>= 1)
#pragma unroll
          for (int p = 0; p < q; ++p) e[p] = __fadd2_rn(e[p], e[p + q]);
        part[it] = e[0];
      }
#pragma unroll
      for (int q = kVecPerThread / 2; q >= 1; q >>= 1)
#pragma unroll
        for (int l = 0; l < q; ++l) part[l] = __fadd2_rn(part[l], part[l + q]);
      float hi = part[0].x + part[0].y, lo = 0.0f;
      warp_sum_compensated(hi, lo);
      out = WarpSoftmax{K, hi, lo, 0.0f};
    }
    if (lane == 0) {
      float4* p = reinterpret_cast<float4*>(A.part + ((g.rid * A.nch + c) * kWarps + w));
      *p = make_float4(out.K, out.hi, out.lo, 0.0f);
    }
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring& ring);
  __device__ static void finish_request(const Args& A, int r, int n, bool n_ok, Smem& sm,
                                        Ring& ring);
  __device__ static void residual_masses(const Args& A, const ResidScan<E>& rs, double* part,
                                         Smem& sm, Ring& ring);
};

template <typename ET>
__device__ void SampleOp<ET>::finish(const Args& A, const Seg& g, Smem& sm, Ring& ring) {
  const int r = g.r;
  bool n_ok;
  const int n = n_of(A, r, n_ok);
  const int i = g.slot <= A.k ? g.slot : g.slot - A.k - 1;
  const float s = A.s;
  if (threadIdx.x == 0) sm.row_last = arrive_last(A.row_cnt + g.rid, (unsigned)g.nseg);
  __syncthreads();
  if (!sm.row_last) return;
  __threadfence();

  // ---- row finish: merge the warp partials of the row (warp 0) ----
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int np = A.nch * kWarps;
    const WarpSoftmax* wp = A.part + g.rid * np;
    float K = -INFINITY;
    bool poison = false;
    for (int q = lane; q < np; q += 32) {
      const WarpSoftmax w = ld_part(wp + q);
      poison |= (w.K != w.K) || (w.hi != w.hi);
      if (w.K > K) K = w.K;
    }
    poison = __any_sync(0xffffffffu, poison);
    K = warp_max_f(K);
    double S = 0.0;
    if (K > -INFINITY)
      for (int q = lane; q < np; q += 32) S += part_mass(ld_part(wp + q), K);
    S = warp_sum_d(S);
    if (lane == 0) {
      int status = (!poison && K > -INFINITY && isfinite(S) && S > 0.0) ? 0 : 1;
      double px = 0.0;
      if (i < n) {
        const int32_t xi = __ldg(A.tokens + (int64_t)r * A.k + i);
        if (xi < 0 || xi >= A.V) {
          status = status ? status : 2;
        } else if (status == 0) {
          const float zx = E::load1(g.row, xi);
          px = exp2((double)zx * (double)s - (double)K) / S;
        }
      }
      RowSoftmax* rs = A.row + g.rid;
      rs->S = S;
      rs->px = px;
      rs->K = K;
      rs->status = status;
      sm.req_last = arrive_last(A.req_cnt + r, (unsigned)(2 * n + 1));
    }
  }
  __syncthreads();
  if (!sm.req_last) return;
  __threadfence();
  finish_request(A, r, n, n_ok, sm, ring);
}

// Per-warp residual masses of every chunk of the rejected pair (rs), into part[c][warp].
// With the TMA ring (aligned rows) the pair streams through the two stages half a chunk at a
// time: a stage holds 16 KiB of the target row and the same 16 KiB of the draft row, two bulk
// copies completing on the stage barrier, and the last warp out of a stage starts the copy
// of the half two ahead. Without it, every thread loads its vectors from global memory.
template <typename ET>
__device__ void SampleOp<ET>::residual_masses(const Args& A, const ResidScan<E>& rs,
                                              double* part, Smem& sm, Ring& ring) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (!ring.usable || !SV_RESID_RING) {
    for (int c = 0; c < A.nch; ++c) {
      const int64_t j0 = (int64_t)c * E::kChunk;
      ResidScan<E> q = rs;
      q.j1 = chunk_end<E>(j0, A.V);
      float acc = 0.0f;
#pragma unroll
      for (int h = 0; h < kVecPerThread; h += 2) {
        typename ResidScan<E>::Raw raw[2];
#pragma unroll
        for (int t = 0; t < 2; ++t)
          raw[t] = q.load(j0 + (int64_t)((h + t) * kThreads + tid) * E::kPerVec);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float w[E::kPerVec];
          q.weights(raw[t], w);
#pragma unroll
          for (int l = 0; l < E::kPerVec; ++l) acc += w[l];
        }
      }
      float hi = acc, lo = 0.0f;
      warp_sum_compensated(hi, lo);
      if (lane == 0) part[(int64_t)c * kWarps + warp] = (double)hi + (double)lo;
    }
    return;
  }
  constexpr int kHalf = E::kChunk / 2;           // logits per half chunk
  constexpr int kHalfBytes = kChunkBytes / 2;    // 16 KiB
  constexpr int kHalfVecPerLane = kVecPerThread / 2;
  const int nh = 2 * A.nch;
  auto issue = [&](int h) {
    const int st = h % kStages;
    const int64_t b = (int64_t)(h >> 1) * E::kChunk + (int64_t)(h & 1) * kHalf;
    const int64_t e = b + kHalf < A.V ? b + kHalf : (int64_t)A.V;
    const uint32_t bytes = e > b ? (uint32_t)((e - b) * (16 / E::kPerVec)) : 0u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (bytes == 0) {
      mbar_arrive(&ring.full[st]);
      return;
    }
    mbar_arrive_expect_tx(&ring.full[st], 2 * bytes);
    bulk_g2s(ring.buf + st * kChunkBytes, static_cast<const char*>(rs.rp) + b * (16 / E::kPerVec),
             bytes, &ring.full[st]);
    bulk_g2s(ring.buf + st * kChunkBytes + kHalfBytes,
             static_cast<const char*>(rs.rq) + b * (16 / E::kPerVec), bytes, &ring.full[st]);
  };
  if (tid == 0)
    for (int h = 0; h < kStages && h < nh; ++h) issue(h);
  // every thread follows the same barrier phases
  float acc = 0.0f;
  bool timed_out = false;
  for (int h = 0; h < nh; ++h) {
    const int st = h % kStages;
    if (!ring_wait(ring, st)) timed_out = true;
    const int64_t b = (int64_t)(h >> 1) * E::kChunk + (int64_t)(h & 1) * kHalf;
    const int64_t e = b + kHalf < A.V ? b + kHalf : (int64_t)A.V;
    const unsigned char* buf = ring.buf + st * kChunkBytes;
    uint4 vp[kHalfVecPerLane], vq[kHalfVecPerLane];
#pragma unroll
    for (int it = 0; it < kHalfVecPerLane; ++it) {
      const int slot = warp * (kHalfVecPerLane * 32) + it * 32 + lane;
      const bool in = b + (int64_t)slot * E::kPerVec < e;
      vp[it] = in ? lds16(buf + slot * 16) : E::pad_vec(E::kNegInfBits);
      vq[it] = in ? lds16(buf + kHalfBytes + slot * 16) : E::pad_vec(E::kNegInfBits);
    }
    __syncwarp();
    if (lane == 0 && atomic_add_acq_rel_cta(&ring.released[st], 1) == kWarps - 1) {
      ring.released[st] = 0;
      if (h + kStages < nh) issue(h + kStages);
    }
#pragma unroll
    for (int it = 0; it < kHalfVecPerLane; ++it) {
      float w[E::kPerVec];
      rs.weights(typename ResidScan<E>::Raw{vp[it], vq[it]}, w);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) acc += w[l];
    }
    if (h & 1) {  // both halves of chunk h/2 are in
      float hi = acc, lo = 0.0f;
      warp_sum_compensated(hi, lo);
      if (lane == 0) part[(int64_t)(h >> 1) * kWarps + warp] = (double)hi + (double)lo;
      acc = 0.0f;
    }
  }
  if (__any_sync(0xffffffffu, timed_out) && lane == 0) {
    atomicOr(&ring.ctl->error, 1u);
    for (int c = 0; c < A.nch; ++c) part[(int64_t)c * kWarps + warp] = __longlong_as_double(0x7ff8000000000000ll);
  }
}

template <typename ET>
__device__ void SampleOp<ET>::finish_request(const Args& A, int r, int n, bool n_ok, Smem& sm,
                                             Ring& ring) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = 2 * A.k + 1;
  const int32_t* x = A.tokens + (int64_t)r * A.k;
  const float* u = A.uniforms + (int64_t)r * (A.k + 1);

  // ---- accept tests (warp 0; lane i is draft position i) ----
  if (tid < 32) {
    bool bad = !n_ok;
    bool reject = false;
    double pt = 0.0, pq = 0.0;
    if (n_ok && lane < n) {
      const RowSoftmax t = ld_row(A.row + (int64_t)r * R + lane);
      const RowSoftmax q = ld_row(A.row + (int64_t)r * R + A.k + 1 + lane);
      const float ui = __ldg(u + lane);
      bad = t.status != 0 || q.status != 0 || !(ui >= 0.0f && ui < 1.0f);
      pt = t.px;
      pq = q.px;
      reject = !((double)ui < pt / pq);
    }
    if (n_ok && lane == 0) {
      const RowSoftmax t = ld_row(A.row + (int64_t)r * R + n);
      const float uk = __ldg(u + A.k);
      bad = bad || t.status != 0 || !(uk >= 0.0f && uk < 1.0f);
    }
    const bool err = __any_sync(0xffffffffu, bad);
    const unsigned rej = __ballot_sync(0xffffffffu, reject);
    const int a = rej ? __ffs(rej) - 1 : n;
    if (lane < A.k) {
      const float nan = __int_as_float(0x7fc00000);
      if (A.out_p) A.out_p[(int64_t)r * A.k + lane] = err ? nan : (lane < n ? (float)pt : 0.0f);
      if (A.out_q) A.out_q[(int64_t)r * A.k + lane] = err ? nan : (lane < n ? (float)pq : 0.0f);
    }
    if (lane == 0) {
      sm.a = a;
      sm.err = err;
    }
  }
  __syncthreads();
  const int a = sm.a;
  if (sm.err) {
    if (tid <= A.k) A.out_tokens[(int64_t)r * (A.k + 1) + tid] = -1;
    if (tid == 0) {
      A.out_accept_len[r] = -1;
      if (A.out_resid) A.out_resid[r] = __int_as_float(0x7fc00000);
    }
    return;
  }

  const float s = A.s;
  int t = -1;
  double W = 0.0;
  bool drew = false;
  if (a < n) {
    // ---- residual norm(max(0, p_a - q_a)): per-chunk masses, then one chunk ----
    ResidScan<E> rs;
    rs.rp = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + a, A.V);
    rs.rq = row_ptr<E>(A.draft, (int64_t)r * A.k + a, A.V);
    rs.aligned = A.aligned;
    const RowSoftmax tp = ld_row(A.row + (int64_t)r * R + a);
    const RowSoftmax dq = ld_row(A.row + (int64_t)r * R + A.k + 1 + a);
    rs.wf.s = s;
    rs.wf.cp = -tp.K;
    rs.wf.cq = -dq.K;
    rs.wf.ip = (float)(1.0 / tp.S);
    rs.wf.iq = (float)(1.0 / dq.S);
    double* part = A.resid + (int64_t)r * A.nch * kWarps;  // [nch][kWarps]
    residual_masses(A, rs, part, sm, ring);
    __syncthreads();
    // chunk masses R_c = sum over warps (fixed order) and W = sum_c R_c (warp 0)
    if (tid < 32) {
      double wsum = 0.0;
      for (int c = lane; c < A.nch; c += 32) {
        double rc = 0.0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) rc += part[(int64_t)c * kWarps + w];
        part[(int64_t)c * kWarps] = rc;
        wsum += rc;
      }
      wsum = warp_sum_d(wsum);
      if (lane == 0) sm.W = wsum;
    }
    __syncthreads();
    W = sm.W;
    if (W > 0.0) {
      const double target = (double)__ldg(u + A.k) * W;
      if (tid < 32) {
        double before;
        bool tl;
        const int c = pick_chunk(
            A.nch, target, [&](int cc) { return part[(int64_t)cc * kWarps]; }, before, tl);
        if (lane == 0) {
          sm.chunk = c < 0 ? 0 : (c >= A.nch ? A.nch - 1 : c);
          sm.before = before;
          sm.take_last = tl;
        }
      }
      __syncthreads();
      const int64_t j0 = (int64_t)sm.chunk * E::kChunk;
      rs.j1 = chunk_end<E>(j0, A.V);
      if (ring.usable) {
        // the chosen chunk of both rows into the two stages, then the scan from shared memory
        __syncthreads();  // nobody still reads the ring
        const bool ok0 = stage_chunk<E>(ring, 0, rs.rp, j0, rs.j1);
        const bool ok1 = stage_chunk<E>(ring, 1, rs.rq, j0, rs.j1);
        ResidScanSmem<E> ss{ring.buf, ring.buf + kChunkBytes, j0, rs.j1, rs.wf};
        t = scan_chunk<E>(j0, target - sm.before, sm.take_last != 0, ss, sm.scan);
        if (!__syncthreads_and(ok0 && ok1)) t = -1;
      } else {
        t = scan_chunk<E>(j0, target - sm.before, sm.take_last != 0, rs, sm.scan);
      }
      drew = true;
    }
  }
  if (!drew) {
    // ---- bonus draw from p_row (row n after full acceptance; row a if the residual
    //      vanished through rounding); everything in units of 2^K of that row ----
    const int brow = a;
    const int64_t rid = (int64_t)r * R + brow;
    const RowSoftmax rsw = ld_row(A.row + rid);
    const WarpSoftmax* wp = A.part + rid * A.nch * kWarps;
    const double target = (double)__ldg(u + A.k) * rsw.S;
    if (tid < 32) {
      double before;
      bool tl;
      const int c = pick_chunk(
          A.nch, target,
          [&](int cc) {
            double mass = 0.0;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) mass += part_mass(ld_part(wp + cc * kWarps + w), rsw.K);
            return mass;
          },
          before, tl);
      if (lane == 0) {
        sm.chunk = c < 0 ? 0 : (c >= A.nch ? A.nch - 1 : c);
        sm.before = before;
        sm.take_last = tl;
      }
    }
    __syncthreads();
    BonusScan<E> bs;
    bs.row = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + brow, A.V);
    bs.aligned = A.aligned;
    bs.s = s;
    bs.c = -rsw.K;
    const int64_t j0 = (int64_t)sm.chunk * E::kChunk;
    bs.j1 = chunk_end<E>(j0, A.V);
    if (ring.usable) {
      __syncthreads();  // nobody still reads the ring
      const bool ok = stage_chunk<E>(ring, 0, bs.row, j0, bs.j1);
      BonusScanSmem<E> ss{ring.buf, j0, bs.j1, s, bs.c};
      t = scan_chunk<E>(j0, target - sm.before, sm.take_last != 0, ss, sm.scan);
      if (!__syncthreads_and(ok)) t = -1;
    } else {
      t = scan_chunk<E>(j0, target - sm.before, sm.take_last != 0, bs, sm.scan);
    }
  }

  // ---- emit ----
  if (tid <= A.k) {
    int32_t val = -1;
    if (tid < a) val = __ldg(x + tid);
    else if (tid == a) val = t;
    A.out_tokens[(int64_t)r * (A.k + 1) + tid] = val;
  }
  if (tid == 0) {
    A.out_accept_len[r] = a;
    if (A.out_resid) A.out_resid[r] = a < n ? (float)W : 0.0f;
  }
}

// ============================================================================================
// Greedy verify
// ============================================================================================
struct GreedyArgs {
  const void* target;
  const int32_t* tokens;
  const int32_t* num_draft;
  int B, k, V, nch, nseg;
  bool aligned;
  int32_t* out_tokens;
  int32_t* out_accept_len;
  WarpArgmax* part;  // [B * (k+1)][nch][kWarps]
  int* row;
  unsigned int* row_cnt;
  unsigned int* req_cnt;
};

// (value, index) with the larger value first, then the lower index; kNoIndex = empty.
__device__ __forceinline__ void argmax_merge(float& v, int& idx, float v2, int idx2) {
  if (idx2 == kNoIndex) return;
  if (idx == kNoIndex || v2 > v || (v2 == v && idx2 < idx)) {
    v = v2;
    idx = idx2;
  }
}

__device__ __forceinline__ void warp_argmax(float& v, int& idx) {
  // NaN never enters: v is -inf for an empty lane, and idx breaks the tie with real -inf.
  const int key = f2key(v);
  const int kmax = __reduce_max_sync(0xffffffffu, key);
  const unsigned cand = (key == kmax) ? (unsigned)idx : 0xffffffffu;
  const unsigned best = __reduce_min_sync(0xffffffffu, cand);
  v = key2f(kmax);
  idx = (int)best;
}

template <typename ET>
struct GreedyOp {
  using Args = GreedyArgs;
  using E = ET;
  static constexpr uint32_t kPad = E::kNaNBits;  // NaN padding is never chosen
  struct Smem {
    int row_last, req_last;
    int g[SV_MAX_K + 1];
  };

  __device__ static __forceinline__ int n_of(const Args& A, int r, bool& ok) {
    const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
    ok = nraw >= 0 && nraw <= A.k;
    return ok ? nraw : A.k;
  }

  __device__ static bool unit(const Args& A, int64_t u, Seg& g) {
    const int R = A.k + 1;
    const int r = (int)(u / ((int64_t)R * A.nseg));
    const int rem = (int)(u - (int64_t)r * R * A.nseg);
    const int i = rem / A.nseg;
    const int seg = rem - i * A.nseg;
    bool ok;
    if (i > n_of(A, r, ok)) return false;
    g.row = row_ptr<E>(A.target, (int64_t)r * R + i, A.V);
    g.rid = (int64_t)r * R + i;
    g.r = r;
    g.slot = i;
    g.c0 = seg * kSegChunks;
    g.c1 = min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  __device__ static void warp_chunk(const Args& A, const Seg& g, int c,
                                    const uint4 (&v)[kVecPerThread], bool poison) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t j0 = (int64_t)c * E::kChunk;
    float best = -INFINITY;
    int bidx = kNoIndex;
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const int jb = (int)(j0 + (int64_t)warp_vec_slot(w, it, lane) * E::kPerVec);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) {
        const float z = E::get(v[it], l);
        // in increasing j: the first comparable logit, then only strictly larger ones
        if (z > best || (bidx == kNoIndex && z == z)) {
          best = z;
          bidx = jb + l;
        }
      }
    }
    warp_argmax(best, bidx);
    if (lane == 0) {
      WarpArgmax* p = A.part + ((g.rid * A.nch + c) * kWarps + w);
      *reinterpret_cast<float2*>(p) = make_float2(best, __int_as_float(poison ? kPoisoned : bidx));
    }
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring&) {
    const int r = g.r;
    bool n_ok;
    const int n = n_of(A, r, n_ok);
    const int R = A.k + 1;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) sm.row_last = arrive_last(A.row_cnt + g.rid, (unsigned)g.nseg);
    __syncthreads();
    if (!sm.row_last) return;
    __threadfence();

    if (threadIdx.x < 32) {
      const int np = A.nch * kWarps;
      const WarpArgmax* wp = A.part + g.rid * np;
      float bv = -INFINITY;
      int bi = kNoIndex;
      bool poison = false;
      for (int q = lane; q < np; q += 32) {
        const float2 pv = __ldcg(reinterpret_cast<const float2*>(wp + q));
        const int pi = __float_as_int(pv.y);
        poison |= pi == kPoisoned;
        argmax_merge(bv, bi, pv.x, pi == kPoisoned ? kNoIndex : pi);
      }
      warp_argmax(bv, bi);
      poison = __any_sync(0xffffffffu, poison);
      if (lane == 0) {
        A.row[g.rid] = (bi == kNoIndex || poison) ? -1 : bi;
        sm.req_last = arrive_last(A.req_cnt + r, (unsigned)(n + 1));
      }
    }
    __syncthreads();
    if (!sm.req_last) return;
    __threadfence();

    // ---- request finish (warp 0; lane i is position i) ----
    if (threadIdx.x < 32) {
      bool bad = !n_ok;
      bool mism = false;
      if (n_ok && lane <= n) {
        const int gi = __ldcg(A.row + (int64_t)r * R + lane);
        bad = gi < 0;
        if (lane < n) {
          const int32_t xi = __ldg(A.tokens + (int64_t)r * A.k + lane);
          bad = bad || xi < 0 || xi >= A.V;
          mism = xi != gi;
        }
        sm.g[lane] = gi;
      }
      const bool err = __any_sync(0xffffffffu, bad);
      const unsigned mm = __ballot_sync(0xffffffffu, mism);
      const int a = mm ? __ffs(mm) - 1 : n;
      __syncwarp();
      if (lane <= A.k) {
        int32_t out = -1;
        if (!err) {
          if (lane < a) out = __ldg(A.tokens + (int64_t)r * A.k + lane);
          else if (lane == a) out = sm.g[a];
        }
        A.out_tokens[(int64_t)r * R + lane] = out;
      }
      if (lane == 0) A.out_accept_len[r] = err ? -1 : a;
    }
  }
};

}  // namespace sv

// ============================================================================================
// C ABI
// ============================================================================================
using namespace sv;

namespace {

bool rows_aligned(const void* base, int V, sv_dtype d) {
  return aligned_to(base, 16) && ((int64_t)V * elem_bytes(d)) % 16 == 0;
}

}  // namespace

extern "C" size_t spec_verify_sample_workspace(int B, int k, int V, sv_dtype dtype) {
  if (B < 0 || k < 1 || k > SV_MAX_K || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return sample_layout(B, k, V, dtype).total;
}

extern "C" sv_status spec_verify_sample(const void* target_logits, const void* draft_logits,
                                        sv_dtype dtype, const int32_t* draft_tokens,
                                        const int32_t* num_draft, const float* uniforms, int B,
                                        int k, int V, float temperature, int32_t* out_tokens,
                                        int32_t* out_accept_len, float* out_p_draft,
                                        float* out_q_draft, float* out_resid_mass,
                                        void* workspace, size_t workspace_bytes,
                                        sv_stream_t stream) {
  if (B < 0 || k < 1 || V < 2) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (!(temperature >= 1e-4f && temperature <= 1e4f)) return SV_ERR_INVALID_ARG;
  if (k > SV_MAX_K) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  const int eb = elem_bytes(dtype);
  if (!target_logits || !draft_logits || !draft_tokens || !uniforms || !out_tokens ||
      !out_accept_len)
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, eb) || !aligned_to(draft_logits, eb) ||
      !aligned_to(draft_tokens, 4) || !aligned_to(uniforms, 4) || !aligned_to(out_tokens, 4) ||
      !aligned_to(out_accept_len, 4) || (num_draft && !aligned_to(num_draft, 4)) ||
      (out_p_draft && !aligned_to(out_p_draft, 4)) ||
      (out_q_draft && !aligned_to(out_q_draft, 4)) ||
      (out_resid_mass && !aligned_to(out_resid_mass, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = (int64_t)B * (2 * k + 1) * nseg;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const SampleLayout L = sample_layout(B, k, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;

  SampleArgs A;
  A.target = target_logits;
  A.draft = draft_logits;
  A.tokens = draft_tokens;
  A.num_draft = num_draft;
  A.uniforms = uniforms;
  A.B = B;
  A.k = k;
  A.V = V;
  A.nch = (int)nch;
  A.nseg = nseg;
  A.s = (float)(1.4426950408889634074 / (double)temperature);
  A.aligned = rows_aligned(target_logits, V, dtype) && rows_aligned(draft_logits, V, dtype);
  A.out_tokens = out_tokens;
  A.out_accept_len = out_accept_len;
  A.out_p = out_p_draft;
  A.out_q = out_q_draft;
  A.out_resid = out_resid_mass;
  char* ws = static_cast<char*>(workspace);
  A.part = reinterpret_cast<WarpSoftmax*>(ws + L.part);
  A.row = reinterpret_cast<RowSoftmax*>(ws + L.row);
  A.resid = reinterpret_cast<double*>(ws + L.resid);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.req_cnt = reinterpret_cast<unsigned int*>(ws + L.req_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the control word and the counters (the last regions) start every call at zero
  cudaError_t e = cudaMemsetAsync(ws + L.ctl, 0, L.total - L.ctl, st);
  if (e != cudaSuccess) return cuda_fail(e);
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_segments<SampleOp<F32>>(A, units, ctl, st);
  return launch_segments<SampleOp<BF16>>(A, units, ctl, st);
}

extern "C" size_t spec_verify_greedy_workspace(int B, int k, int V, sv_dtype dtype) {
  if (B < 0 || k < 1 || k > SV_MAX_K || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return greedy_layout(B, k, V, dtype).total;
}

extern "C" sv_status spec_verify_greedy(const void* target_logits, sv_dtype dtype,
                                        const int32_t* draft_tokens, const int32_t* num_draft,
                                        int B, int k, int V, int32_t* out_tokens,
                                        int32_t* out_accept_len, void* workspace,
                                        size_t workspace_bytes, sv_stream_t stream) {
  if (B < 0 || k < 1 || V < 2) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (k > SV_MAX_K) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  const int eb = elem_bytes(dtype);
  if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len)
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, eb) || !aligned_to(draft_tokens, 4) ||
      !aligned_to(out_tokens, 4) || !aligned_to(out_accept_len, 4) ||
      (num_draft && !aligned_to(num_draft, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = (int64_t)B * (k + 1) * nseg;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const GreedyLayout L = greedy_layout(B, k, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;

  GreedyArgs A;
  A.target = target_logits;
  A.tokens = draft_tokens;
  A.num_draft = num_draft;
  A.B = B;
  A.k = k;
  A.V = V;
  A.nch = (int)nch;
  A.nseg = nseg;
  A.aligned = rows_aligned(target_logits, V, dtype);
  A.out_tokens = out_tokens;
  A.out_accept_len = out_accept_len;
  char* ws = static_cast<char*>(workspace);
  A.part = reinterpret_cast<WarpArgmax*>(ws + L.part);
  A.row = reinterpret_cast<int*>(ws + L.row);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.req_cnt = reinterpret_cast<unsigned int*>(ws + L.req_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws + L.ctl, 0, L.total - L.ctl, st);
  if (e != cudaSuccess) return cuda_fail(e);
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_segments<GreedyOp<F32>>(A, units, ctl, st);
  return launch_segments<GreedyOp<BF16>>(A, units, ctl, st);
}

// ============================================================================================
// Greedy verify without caller-provided scratch
// ============================================================================================
// Some callers cannot allocate device memory at all: an engine that has handed every byte of
// the device to its own pool, or code on a path where cudaMalloc's implicit synchronisation
// is not allowed. For them the greedy verify can use a scratch buffer that lives in this
// library's own device image: a fixed array every GPU that loads the library holds until the
// process exits. Its device address is looked up once per device, on the first call made with
// that device current.
namespace {

constexpr size_t kGreedyScratchBytes = size_t(8) << 20;  // 8 MiB
constexpr int kMaxScratchDevices = 64;

static __device__ __align__(256) unsigned char g_greedy_scratch[kGreedyScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxScratchDevices] = {};

// Device address of g_greedy_scratch on the current device (looked up on first use).
sv_status greedy_scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxScratchDevices) return SV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_greedy_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SV_OK;
}

}  // namespace

extern "C" sv_status spec_verify_greedy_noalloc(const void* target_logits, sv_dtype dtype,
                                                const int32_t* draft_tokens,
                                                const int32_t* num_draft, int B, int k, int V,
                                                int32_t* out_tokens, int32_t* out_accept_len,
                                                sv_stream_t stream) {
  if (B < 0 || k < 1 || V < 2) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (k > SV_MAX_K) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  if (greedy_layout(B, k, V, dtype).total > kGreedyScratchBytes) return SV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const sv_status st = greedy_scratch_address(&scratch);
  if (st != SV_OK) return st;
  return spec_verify_greedy(target_logits, dtype, draft_tokens, num_draft, B, k, V, out_tokens,
                            out_accept_len, scratch, kGreedyScratchBytes, stream);
}
