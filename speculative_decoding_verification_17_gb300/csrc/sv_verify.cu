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
// One kernel launch per call (after a small memset of the call's counters). Unit =
// (request r, row slot, chunk c); a request has 2k+1 row slots in the sampled verify
// (target rows 0..k, then draft rows 0..k-1) and k+1 in the greedy verify. Units of rows a
// request does not need (past its n_r) are skipped.
//
//  pass 1 (every unit)      chunk max m_c (exact, raw logits) and, in the sampled verify,
//                           S_c = sum_j 2^(z_j*s + c_c) with s = log2(e)/T in fp32 and
//                           c_c = fp32(-m_c*s); in the greedy verify the chunk argmax.
//  row finish (last chunk)  m = max m_c; S = sum_c S_c * 2^(-c_c - m*s) in double (the
//                           exponent is exact, so every chunk is rescaled to the same
//                           reference); p(x) = 2^(z_x*s - m*s) / S in double.
//  request finish (last row)  ratios p_i(x_i)/q_i(x_i) in double against the uniforms, the
//                           accepted prefix a, then one draw: the residual max(0, p_a - q_a)
//                           (one extra pass over the rejected row pair, which L2 still
//                           holds, for per-chunk residual masses, then one chunk scanned in
//                           vocabulary order), or the bonus from p_n (chunk masses are the
//                           pass-1 partials, one chunk scanned).
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"

namespace sv {

constexpr int kPoisoned = -2;  // a chunk index that marks a chunk whose copy never landed

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
  int B, k, V, nch;
  float s;       // log2(e) / T, rounded to fp32
  bool aligned;  // every row starts on a 16-byte boundary
  int32_t* out_tokens;
  int32_t* out_accept_len;
  float* out_p;
  float* out_q;
  float* out_resid;
  ChunkSoftmax* chunk;
  RowSoftmax* row;
  double* resid;  // [B][nch][kWarps] residual partial masses
  unsigned int* row_cnt;
  unsigned int* req_cnt;
};

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
  float s, cc;
  using Raw = uint4;
  __device__ __forceinline__ Raw load(int64_t j) const {
    return load_vec<E>(row, j, j1, aligned, E::kNegInfBits);
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) w[l] = ex2(fmaf(E::get(r, l), s, cc));
  }
};

__device__ __forceinline__ ChunkSoftmax ld_chunk(const ChunkSoftmax* p) {
  ChunkSoftmax c;
  c.S = __ldcg(&p->S);
  c.m = __ldcg(&p->m);
  return c;
}

__device__ __forceinline__ RowSoftmax ld_row(const RowSoftmax* p) {
  RowSoftmax r;
  r.S = __ldcg(&p->S);
  r.px = __ldcg(&p->px);
  r.m = __ldcg(&p->m);
  r.status = __ldcg(&p->status);
  return r;
}

// Exponent that rescales a chunk's partial sum onto its row's reference m*s (exact).
__device__ __forceinline__ double chunk_to_row(float mc, float s, double ms) {
  const float cc = __fmul_rn(-mc, s);
  return -(double)cc - ms;
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

  __device__ static __forceinline__ void decode(const Args& A, int64_t u, int& r, int& slot,
                                                int& c) {
    const int R = 2 * A.k + 1;
    r = (int)(u / ((int64_t)R * A.nch));
    const int rem = (int)(u - (int64_t)r * R * A.nch);
    slot = rem / A.nch;
    c = rem - slot * A.nch;
  }
  __device__ static __forceinline__ int n_of(const Args& A, int r, bool& ok) {
    const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
    ok = nraw >= 0 && nraw <= A.k;
    return ok ? nraw : A.k;
  }

  __device__ static bool unit_row(const Args& A, int64_t u, const void*& row, int64_t& j0,
                                  int64_t& j1) {
    int r, slot, c;
    decode(A, u, r, slot, c);
    bool ok;
    const int n = n_of(A, r, ok);
    const bool is_target = slot <= A.k;
    const int i = is_target ? slot : slot - A.k - 1;
    if (is_target ? i > n : i >= n) return false;
    row = is_target ? row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + i, A.V)
                    : row_ptr<E>(A.draft, (int64_t)r * A.k + i, A.V);
    j0 = (int64_t)c * E::kChunk;
    j1 = chunk_end<E>(j0, A.V);
    return true;
  }

  __device__ static void process(const Args& A, int64_t u, const void* rowp, int64_t j0,
                                 int64_t j1, const unsigned char* chunk, bool poisoned,
                                 Smem& sm);
  __device__ static void finish_request(const Args& A, int r, int n, bool n_ok, Smem& sm);
};

template <typename ET>
__device__ void SampleOp<ET>::process(const Args& A, int64_t u, const void* rowp, int64_t j0,
                                      int64_t j1, const unsigned char* chunk, bool poisoned,
                                      Smem& sm) {
  int r, slot, c;
  decode(A, u, r, slot, c);
  bool n_ok;
  const int n = n_of(A, r, n_ok);
  const int i = slot <= A.k ? slot : slot - A.k - 1;
  const float s = A.s;
  const int R = 2 * A.k + 1;

  // ---- pass 1: chunk maximum and chunk sum ----
  float tmax = -INFINITY;
#pragma unroll
  for (int it = 0; it < kVecPerThread; ++it)
    tmax = fmaxf(tmax, E::max_vec(chunk_vec<E>(chunk, it, j0, j1, kPad)));
  const float m = block_max_f(tmax, sm.red);
  double S;
  if (poisoned || m == -INFINITY || m == INFINITY) {
    // no finite logit here: a masked chunk carries no mass; NaN or +inf poison the row
    int nan = 0;
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const uint4 v = chunk_vec<E>(chunk, it, j0, j1, kPad);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) nan |= E::get(v, l) != E::get(v, l);
    }
    const bool bad = cbar_or(nan) || m == INFINITY || poisoned;
    S = bad ? __longlong_as_double(0x7ff8000000000000ll) : 0.0;
  } else {
    const float cc = __fmul_rn(-m, s);
    float part[kVecPerThread];
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const uint4 v = chunk_vec<E>(chunk, it, j0, j1, kPad);
      float e[E::kPerVec];
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) e[l] = ex2(fmaf(E::get(v, l), s, cc));
#pragma unroll
      for (int w = E::kPerVec / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int l = 0; l < w; ++l) e[l] = e[l] + e[l + w];
      part[it] = e[0];
    }
#pragma unroll
    for (int w = kVecPerThread / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int l = 0; l < w; ++l) part[l] = part[l] + part[l + w];
    S = block_sum_fd_t0(part[0], sm.red);  // valid in thread 0, the only reader
  }

  const int64_t rid = (int64_t)r * R + slot;
  if (threadIdx.x == 0) {
    ChunkSoftmax* p = A.chunk + rid * A.nch + c;
    p->S = S;
    p->m = m;
    sm.row_last = arrive_last(A.row_cnt + rid, (unsigned)A.nch);
  }
  cbar();
  if (!sm.row_last) return;
  __threadfence();

  // ---- row finish: merge the chunk partials (warp 0) ----
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const ChunkSoftmax* cs = A.chunk + rid * A.nch;
    float mrow = -INFINITY;
    for (int cc = lane; cc < A.nch; cc += 32) mrow = fmaxf(mrow, __ldcg(&cs[cc].m));
    mrow = warp_max_f(mrow);
    const double ms = (double)mrow * (double)s;
    double Srow = 0.0;
    for (int cc = lane; cc < A.nch; cc += 32) {
      const ChunkSoftmax q = ld_chunk(cs + cc);
      if (q.m == -INFINITY) Srow += q.S;  // 0, or NaN for a poisoned chunk
      else Srow += q.S * exp2(chunk_to_row(q.m, s, ms));
    }
    Srow = warp_sum_d(Srow);
    if (lane == 0) {
      int status = (isfinite(mrow) && isfinite(Srow) && Srow > 0.0) ? 0 : 1;
      double px = 0.0;
      if (i < n) {
        const int32_t xi = __ldg(A.tokens + (int64_t)r * A.k + i);
        if (xi < 0 || xi >= A.V) {
          status = status ? status : 2;
        } else if (status == 0) {
          const float zx = E::load1(rowp, xi);
          px = exp2((double)zx * (double)s - ms) / Srow;
        }
      }
      RowSoftmax* rs = A.row + rid;
      rs->S = Srow;
      rs->px = px;
      rs->m = mrow;
      rs->status = status;
      sm.req_last = arrive_last(A.req_cnt + r, (unsigned)(2 * n + 1));
    }
  }
  cbar();
  if (!sm.req_last) return;
  __threadfence();
  finish_request(A, r, n, n_ok, sm);
}

template <typename ET>
__device__ void SampleOp<ET>::finish_request(const Args& A, int r, int n, bool n_ok, Smem& sm) {
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
  cbar();
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
    rs.wf.cp = __fmul_rn(-tp.m, s);
    rs.wf.cq = __fmul_rn(-dq.m, s);
    rs.wf.ip = (float)(1.0 / (tp.S * exp2((double)rs.wf.cp + (double)tp.m * (double)s)));
    rs.wf.iq = (float)(1.0 / (dq.S * exp2((double)rs.wf.cq + (double)dq.m * (double)s)));
    double* part = A.resid + (int64_t)r * A.nch * kWarps;  // [nch][kWarps]
    // every warp walks all chunks on its own (no barrier per chunk): four vectors in flight
    // per thread at a time, one compensated warp sum per chunk
    for (int c = 0; c < A.nch; ++c) {
      const int64_t j0 = (int64_t)c * E::kChunk;
      rs.j1 = chunk_end<E>(j0, A.V);
      float acc = 0.0f;
#pragma unroll
      for (int h = 0; h < kVecPerThread; h += 2) {
        typename ResidScan<E>::Raw raw[2];
#pragma unroll
        for (int q = 0; q < 2; ++q)
          raw[q] = rs.load(j0 + (int64_t)((h + q) * kThreads + tid) * E::kPerVec);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float w[E::kPerVec];
          rs.weights(raw[q], w);
#pragma unroll
          for (int l = 0; l < E::kPerVec; ++l) acc += w[l];
        }
      }
      float hi = acc, lo = 0.0f;
      warp_sum_compensated(hi, lo);
      if (lane == 0) part[(int64_t)c * kWarps + warp] = (double)hi + (double)lo;
    }
    cbar();
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
    cbar();
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
      cbar();
      const int64_t j0 = (int64_t)sm.chunk * E::kChunk;
      rs.j1 = chunk_end<E>(j0, A.V);
      t = scan_chunk<E>(j0, target - sm.before, sm.take_last != 0, rs, sm.scan);
      drew = true;
    }
  }
  if (!drew) {
    // ---- bonus draw from p_row (row n after full acceptance; row a if the residual
    //      vanished through rounding) ----
    const int brow = a;
    const int64_t rid = (int64_t)r * R + brow;
    const RowSoftmax rsw = ld_row(A.row + rid);
    const double ms = (double)rsw.m * (double)s;
    const ChunkSoftmax* cs = A.chunk + rid * A.nch;
    const double target = (double)__ldg(u + A.k) * rsw.S;
    if (tid < 32) {
      double before;
      bool tl;
      const int c = pick_chunk(
          A.nch, target,
          [&](int cc) {
            const ChunkSoftmax q = ld_chunk(cs + cc);
            return q.m == -INFINITY ? 0.0 : q.S * exp2(chunk_to_row(q.m, s, ms));
          },
          before, tl);
      if (lane == 0) {
        sm.chunk = c < 0 ? 0 : (c >= A.nch ? A.nch - 1 : c);
        sm.before = before;
        sm.take_last = tl;
      }
    }
    cbar();
    const int c = sm.chunk;
    const ChunkSoftmax q = ld_chunk(cs + c);
    const double scale = exp2(chunk_to_row(q.m, s, ms));
    BonusScan<E> bs;
    bs.row = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + brow, A.V);
    bs.aligned = A.aligned;
    bs.s = s;
    bs.cc = __fmul_rn(-q.m, s);
    const int64_t j0 = (int64_t)c * E::kChunk;
    bs.j1 = chunk_end<E>(j0, A.V);
    t = scan_chunk<E>(j0, (target - sm.before) / scale, sm.take_last != 0, bs, sm.scan);
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
  int B, k, V, nch;
  bool aligned;
  int32_t* out_tokens;
  int32_t* out_accept_len;
  ChunkArgmax* chunk;
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
    float v[kWarps];
    int idx[kWarps];
    int row_last, req_last;
    int g[SV_MAX_K + 1];
  };

  __device__ static __forceinline__ void decode(const Args& A, int64_t u, int& r, int& i,
                                                int& c) {
    const int R = A.k + 1;
    r = (int)(u / ((int64_t)R * A.nch));
    const int rem = (int)(u - (int64_t)r * R * A.nch);
    i = rem / A.nch;
    c = rem - i * A.nch;
  }
  __device__ static __forceinline__ int n_of(const Args& A, int r, bool& ok) {
    const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
    ok = nraw >= 0 && nraw <= A.k;
    return ok ? nraw : A.k;
  }

  __device__ static bool unit_row(const Args& A, int64_t u, const void*& row, int64_t& j0,
                                  int64_t& j1) {
    int r, i, c;
    decode(A, u, r, i, c);
    bool ok;
    if (i > n_of(A, r, ok)) return false;
    row = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + i, A.V);
    j0 = (int64_t)c * E::kChunk;
    j1 = chunk_end<E>(j0, A.V);
    return true;
  }

  __device__ static void process(const Args& A, int64_t u, const void* rowp, int64_t j0,
                                 int64_t j1, const unsigned char* chunk, bool poisoned,
                                 Smem& sm) {
    int r, i, c;
    decode(A, u, r, i, c);
    bool n_ok;
    const int n = n_of(A, r, n_ok);
    const int R = A.k + 1;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;

    float best = -INFINITY;
    int bidx = kNoIndex;
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const uint4 v = chunk_vec<E>(chunk, it, j0, j1, kPad);
      const int jb = (int)(j0 + (int64_t)(it * kThreads + threadIdx.x) * E::kPerVec);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) {
        const float z = E::get(v, l);
        // in increasing j: the first comparable logit, then only strictly larger ones
        if (z > best || (bidx == kNoIndex && z == z)) {
          best = z;
          bidx = jb + l;
        }
      }
    }
    warp_argmax(best, bidx);
    if (lane == 0) {
      sm.v[w] = best;
      sm.idx[w] = bidx;
    }
    cbar();
    const int64_t rid = (int64_t)r * R + i;
    if (threadIdx.x == 0) {
      float bv = sm.v[0];
      int bi = sm.idx[0];
      for (int q = 1; q < kWarps; ++q) argmax_merge(bv, bi, sm.v[q], sm.idx[q]);
      ChunkArgmax* p = A.chunk + rid * A.nch + c;
      p->v = bv;
      p->idx = poisoned ? kPoisoned : bi;
      sm.row_last = arrive_last(A.row_cnt + rid, (unsigned)A.nch);
    }
    cbar();
    if (!sm.row_last) return;
    __threadfence();

    if (threadIdx.x < 32) {
      float bv = -INFINITY;
      int bi = kNoIndex;
      bool poison = false;
      for (int cc = lane; cc < A.nch; cc += 32) {
        const ChunkArgmax* p = A.chunk + rid * A.nch + cc;
        const int pi = __ldcg(&p->idx);
        poison |= pi == kPoisoned;
        argmax_merge(bv, bi, __ldcg(&p->v), pi == kPoisoned ? kNoIndex : pi);
      }
      warp_argmax(bv, bi);
      poison = __any_sync(0xffffffffu, poison);
      if (lane == 0) {
        A.row[rid] = (bi == kNoIndex || poison) ? -1 : bi;
        sm.req_last = arrive_last(A.req_cnt + r, (unsigned)(n + 1));
      }
    }
    cbar();
    if (!sm.req_last) return;
    __threadfence();

    // ---- request finish (warp 0; lane i is position i) ----
    if (threadIdx.x < 32) {
      bool bad = !n_ok;
      bool mism = false;
      if (n_ok && lane <= n) {
        const int g = __ldcg(A.row + (int64_t)r * R + lane);
        bad = g < 0;
        if (lane < n) {
          const int32_t xi = __ldg(A.tokens + (int64_t)r * A.k + lane);
          bad = bad || xi < 0 || xi >= A.V;
          mism = xi != g;
        }
        sm.g[lane] = g;
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
  const int64_t units = (int64_t)B * (2 * k + 1) * nch;
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
  A.s = (float)(1.4426950408889634074 / (double)temperature);
  A.aligned = rows_aligned(target_logits, V, dtype) && rows_aligned(draft_logits, V, dtype);
  A.out_tokens = out_tokens;
  A.out_accept_len = out_accept_len;
  A.out_p = out_p_draft;
  A.out_q = out_q_draft;
  A.out_resid = out_resid_mass;
  char* ws = static_cast<char*>(workspace);
  A.chunk = reinterpret_cast<ChunkSoftmax*>(ws + L.chunk);
  A.row = reinterpret_cast<RowSoftmax*>(ws + L.row);
  A.resid = reinterpret_cast<double*>(ws + L.resid);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.req_cnt = reinterpret_cast<unsigned int*>(ws + L.req_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the control word and the counters (the last regions) start every call at zero
  cudaError_t e = cudaMemsetAsync(ws + L.ctl, 0, L.total - L.ctl, st);
  if (e != cudaSuccess) return cuda_fail(e);
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_units<SampleOp<F32>>(A, units, ctl, st);
  return launch_units<SampleOp<BF16>>(A, units, ctl, st);
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
  const int64_t units = (int64_t)B * (k + 1) * nch;
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
  A.aligned = rows_aligned(target_logits, V, dtype);
  A.out_tokens = out_tokens;
  A.out_accept_len = out_accept_len;
  char* ws = static_cast<char*>(workspace);
  A.chunk = reinterpret_cast<ChunkArgmax*>(ws + L.chunk);
  A.row = reinterpret_cast<int*>(ws + L.row);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.req_cnt = reinterpret_cast<unsigned int*>(ws + L.req_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(ws + L.ctl, 0, L.total - L.ctl, st);
  if (e != cudaSuccess) return cuda_fail(e);
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_units<GreedyOp<F32>>(A, units, ctl, st);
  return launch_units<GreedyOp<BF16>>(A, units, ctl, st);
}
