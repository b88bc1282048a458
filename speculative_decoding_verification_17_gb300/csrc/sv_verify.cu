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
// One kernel launch per call. Unit = (request r, row slot, chunk c); a request has
// 2k+1 row slots in the sampled verify (target rows 0..k, then draft rows 0..k-1) and k+1
// in the greedy verify. Units of rows a request does not need (past its n_r) exit at once.
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

namespace sv {

struct SampleArgs {
  const void* target;
  const void* draft;
  const int32_t* tokens;
  const int32_t* num_draft;
  const float* uniforms;
  int B, k, V, nch;
  float s;  // log2(e) / T, rounded to fp32
  bool aligned;  // every row starts on a 16-byte boundary
  int32_t* out_tokens;
  int32_t* out_accept_len;
  float* out_p;
  float* out_q;
  float* out_resid;
  ChunkSoftmax* chunk;
  RowSoftmax* row;
  double* resid;
  unsigned int* row_cnt;
  unsigned int* req_cnt;
};

template <typename E>
__device__ __forceinline__ const void* row_ptr(const void* base, int64_t row, int V) {
  return static_cast<const char*>(base) + row * (int64_t)V * (16 / E::kPerVec);
}

// Sum of 2^(z*s + c) over one 16-byte vector of logits, pairwise.
template <typename E>
__device__ __forceinline__ float vec_exp_sum(const uint4& v, float s, float c) {
  float e[E::kPerVec];
#pragma unroll
  for (int l = 0; l < E::kPerVec; ++l) e[l] = ex2(fmaf(E::get(v, l), s, c));
#pragma unroll
  for (int w = E::kPerVec / 2; w >= 1; w >>= 1)
#pragma unroll
    for (int l = 0; l < w; ++l) e[l] = e[l] + e[l + w];
  return e[0];
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

struct ScanSmem {
  double tot[kWarps];
  int first[kWarps];
  int result;
  int lastpos;
};

// Inverse-CDF draw inside one chunk: the first logit j in [j0, j1), in vocabulary order,
// whose running weight exceeds `target` (chunk units). When rounding leaves the target at
// or past the chunk's total, the last logit with positive weight. Each thread owns a
// contiguous run of the chunk; the thread whose run holds the crossing re-walks it with
// exactly the same double additions, so the crossing is always found there.
// weight(j) returns the weight of logit j. Every thread of the block must call this.
template <typename E, typename WF>
__device__ int scan_chunk(int64_t j0, int64_t j1, double target, bool take_last, WF weight,
                          ScanSmem& sm) {
  constexpr int kRun = E::kChunk / kThreads;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t b = j0 + (int64_t)tid * kRun;
  const int64_t e = b + kRun < j1 ? b + kRun : j1;
  double sum = 0.0;
  int lastpos = -1;
  for (int64_t j = b; j < e; ++j) {
    const float wj = weight(j);
    sum += (double)wj;
    if (wj > 0.0f) lastpos = (int)j;
  }
  // block exclusive scan of the per-thread sums
  double incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.tot[w] = incl;
  if (tid == 0) {
    sm.result = -1;
    sm.lastpos = -1;
  }
  __syncthreads();
  double excl = incl - sum;
  for (int i = 0; i < w; ++i) excl += sm.tot[i];
  const bool cross = !take_last && sum > 0.0 && excl + sum > target;
  const unsigned bal = __ballot_sync(0xffffffffu, cross);
  if (lane == 0) sm.first[w] = bal ? w * 32 + __ffs(bal) - 1 : kThreads;
  if (lastpos >= 0) atomicMax(&sm.lastpos, lastpos);
  __syncthreads();
  int owner = kThreads;
  for (int i = 0; i < kWarps; ++i) owner = min(owner, sm.first[i]);
  if (owner == tid) {
    double run = excl;
    int t = lastpos;
    for (int64_t j = b; j < e; ++j) {
      run += (double)weight(j);
      if (run > target) {
        t = (int)j;
        break;
      }
    }
    sm.result = t;
  }
  __syncthreads();
  const int t = owner < kThreads ? sm.result : sm.lastpos;
  __syncthreads();
  return t;
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
    double incl = m;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
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

// Rescale exponent of a chunk's partial sum onto its row's reference m*s.
__device__ __forceinline__ double chunk_to_row(float mc, float s, double ms) {
  const float cc = __fmul_rn(-mc, s);
  return -(double)cc - ms;
}

struct FinishSmem {
  int a;
  int err;
  double W;
  ScanSmem scan;
  int chunk;
  int take_last;
  double before;
};

template <typename E>
__device__ void finish_sample_request(const SampleArgs& A, int r, int n, bool n_ok,
                                      float* red, FinishSmem& fs) {
  const int tid = threadIdx.x, lane = tid & 31;
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
      fs.a = a;
      fs.err = err;
    }
  }
  __syncthreads();
  const int a = fs.a;
  if (fs.err) {
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
    const void* rp = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + a, A.V);
    const void* rq = row_ptr<E>(A.draft, (int64_t)r * A.k + a, A.V);
    const RowSoftmax tp = ld_row(A.row + (int64_t)r * R + a);
    const RowSoftmax dq = ld_row(A.row + (int64_t)r * R + A.k + 1 + a);
    ResidW wf;
    wf.s = s;
    wf.cp = __fmul_rn(-tp.m, s);
    wf.cq = __fmul_rn(-dq.m, s);
    wf.ip = (float)(1.0 / (tp.S * exp2((double)wf.cp + (double)tp.m * (double)s)));
    wf.iq = (float)(1.0 / (dq.S * exp2((double)wf.cq + (double)dq.m * (double)s)));
    double* rm = A.resid + (int64_t)r * A.nch;
    double Wt0 = 0.0;  // accumulated by thread 0
    for (int c = 0; c < A.nch; ++c) {
      const int64_t j0 = (int64_t)c * E::kChunk;
      const int64_t j1 = j0 + E::kChunk < A.V ? j0 + E::kChunk : A.V;
      float acc = 0.0f;
#pragma unroll 2
      for (int it = 0; it < kVecPerThread; ++it) {
        uint4 vp[1], vq[1];
        const int64_t j = j0 + (int64_t)(it * kThreads + tid) * E::kPerVec;
        if (A.aligned && j + E::kPerVec <= j1) {
          vp[0] = ld_stream16(static_cast<const char*>(rp) + j * (16 / E::kPerVec));
          vq[0] = ld_stream16(static_cast<const char*>(rq) + j * (16 / E::kPerVec));
#pragma unroll
          for (int l = 0; l < E::kPerVec; ++l) acc += wf(E::get(vp[0], l), E::get(vq[0], l));
        } else {
          for (int l = 0; l < E::kPerVec; ++l)
            if (j + l < j1) acc += wf(E::load1(rp, j + l), E::load1(rq, j + l));
        }
      }
      const double Rc = block_sum_fd_t0(acc, red);
      if (tid == 0) {
        rm[c] = Rc;
        Wt0 += Rc;
      }
      __syncthreads();  // red[] is rewritten by the next chunk
    }
    if (tid == 0) fs.W = Wt0;
    __syncthreads();  // rm[] and W visible to the whole block
    W = fs.W;
    if (W > 0.0) {
      const double target = (double)__ldg(u + A.k) * W;
      if (tid < 32) {
        double before;
        bool tl;
        const int c = pick_chunk(A.nch, target, [&](int cc) { return rm[cc]; }, before, tl);
        if (lane == 0) {
          fs.chunk = c < 0 ? 0 : (c >= A.nch ? A.nch - 1 : c);
          fs.before = before;
          fs.take_last = tl;
        }
      }
      __syncthreads();
      const int c = fs.chunk;
      const int64_t j0 = (int64_t)c * E::kChunk;
      const int64_t j1 = j0 + E::kChunk < A.V ? j0 + E::kChunk : A.V;
      t = scan_chunk<E>(j0, j1, target - fs.before, fs.take_last != 0,
                        [&](int64_t j) { return wf(E::load1(rp, j), E::load1(rq, j)); },
                        fs.scan);
      drew = true;
    }
  }
  if (!drew) {
    // ---- bonus draw from p_row (row n after full acceptance; row a if the residual
    //      vanished through rounding) ----
    const int brow = a;
    const int64_t rid = (int64_t)r * R + brow;
    const RowSoftmax rs = ld_row(A.row + rid);
    const double ms = (double)rs.m * (double)s;
    const ChunkSoftmax* cs = A.chunk + rid * A.nch;
    const double target = (double)__ldg(u + A.k) * rs.S;
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
        fs.chunk = c < 0 ? 0 : (c >= A.nch ? A.nch - 1 : c);
        fs.before = before;
        fs.take_last = tl;
      }
    }
    __syncthreads();
    const int c = fs.chunk;
    const ChunkSoftmax q = ld_chunk(cs + c);
    const float cc = __fmul_rn(-q.m, s);
    const double scale = exp2(chunk_to_row(q.m, s, ms));
    const int64_t j0 = (int64_t)c * E::kChunk;
    const int64_t j1 = j0 + E::kChunk < A.V ? j0 + E::kChunk : A.V;
    const void* rp = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + brow, A.V);
    t = scan_chunk<E>(j0, j1, (target - fs.before) / scale, fs.take_last != 0,
                      [&](int64_t j) { return ex2(fmaf(E::load1(rp, j), s, cc)); }, fs.scan);
  }

  // ---- emit ----
  if (tid <= A.k) {
    int32_t v = -1;
    if (tid < a) v = __ldg(x + tid);
    else if (tid == a) v = t;
    A.out_tokens[(int64_t)r * (A.k + 1) + tid] = v;
  }
  if (tid == 0) {
    A.out_accept_len[r] = a;
    if (A.out_resid) A.out_resid[r] = a < n ? (float)W : 0.0f;
  }
}

template <typename E>
__global__ void __launch_bounds__(kThreads, 4) sample_kernel(const SampleArgs A) {
  __shared__ float red[2 * kWarps];
  __shared__ int s_row_last, s_req_last;
  __shared__ FinishSmem fs;

  const int R = 2 * A.k + 1;
  const int64_t unit = blockIdx.x;
  const int r = (int)(unit / ((int64_t)R * A.nch));
  const int rem = (int)(unit - (int64_t)r * R * A.nch);
  const int slot = rem / A.nch;
  const int c = rem - slot * A.nch;
  const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
  const bool n_ok = nraw >= 0 && nraw <= A.k;
  const int n = n_ok ? nraw : A.k;
  const bool is_target = slot <= A.k;
  const int i = is_target ? slot : slot - A.k - 1;
  if (is_target ? i > n : i >= n) return;

  const void* rowp = is_target ? row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + i, A.V)
                               : row_ptr<E>(A.draft, (int64_t)r * A.k + i, A.V);
  const int64_t j0 = (int64_t)c * E::kChunk;
  const int64_t j1 = j0 + E::kChunk < A.V ? j0 + E::kChunk : A.V;
  const float s = A.s;

  // ---- pass 1: chunk maximum and chunk sum ----
  uint4 v[kVecPerThread];
  load_chunk<E>(rowp, j0, j1, A.aligned, E::kNegInfBits, v);
  const float m = block_max_f(E::max_all(v), red);
  double S;
  if (m == -INFINITY || m == INFINITY) {
    // no finite logit here: a masked chunk carries no mass; NaN or +inf poison the row
    int nan = 0;
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it)
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) nan |= E::get(v[it], l) != E::get(v[it], l);
    const bool bad = __syncthreads_or(nan) || m == INFINITY;
    S = bad ? __longlong_as_double(0x7ff8000000000000ll) : 0.0;
  } else {
    const float cc = __fmul_rn(-m, s);
    float part[kVecPerThread];
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) part[it] = vec_exp_sum<E>(v[it], s, cc);
#pragma unroll
    for (int w = kVecPerThread / 2; w >= 1; w >>= 1)
#pragma unroll
      for (int l = 0; l < w; ++l) part[l] = part[l] + part[l + w];
    S = block_sum_fd_t0(part[0], red);  // valid in thread 0, the only reader
  }

  const int64_t rid = (int64_t)r * R + slot;
  if (threadIdx.x == 0) {
    ChunkSoftmax* p = A.chunk + rid * A.nch + c;
    p->S = S;
    p->m = m;
    s_row_last = arrive_last(A.row_cnt + rid, (unsigned)A.nch);
  }
  __syncthreads();
  if (!s_row_last) return;
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
      s_req_last = arrive_last(A.req_cnt + r, (unsigned)(2 * n + 1));
    }
  }
  __syncthreads();
  if (!s_req_last) return;
  __threadfence();
  finish_sample_request<E>(A, r, n, n_ok, red, fs);
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

template <typename E>
__global__ void __launch_bounds__(kThreads, 4) greedy_kernel(const GreedyArgs A) {
  __shared__ float sv[kWarps];
  __shared__ int si[kWarps];
  __shared__ int s_row_last, s_req_last;
  __shared__ int s_g[SV_MAX_K + 1];

  const int R = A.k + 1;
  const int64_t unit = blockIdx.x;
  const int r = (int)(unit / ((int64_t)R * A.nch));
  const int rem = (int)(unit - (int64_t)r * R * A.nch);
  const int i = rem / A.nch;
  const int c = rem - i * A.nch;
  const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
  const bool n_ok = nraw >= 0 && nraw <= A.k;
  const int n = n_ok ? nraw : A.k;
  if (i > n) return;

  const void* rowp = row_ptr<E>(A.target, (int64_t)r * R + i, A.V);
  const int64_t j0 = (int64_t)c * E::kChunk;
  const int64_t j1 = j0 + E::kChunk < A.V ? j0 + E::kChunk : A.V;
  uint4 v[kVecPerThread];
  load_chunk<E>(rowp, j0, j1, A.aligned, E::kNaNBits, v);  // NaN padding is never chosen
  float best = -INFINITY;
  int bidx = kNoIndex;
#pragma unroll
  for (int it = 0; it < kVecPerThread; ++it) {
    const int jb = (int)(j0 + (int64_t)(it * kThreads + threadIdx.x) * E::kPerVec);
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
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    sv[w] = best;
    si[w] = bidx;
  }
  __syncthreads();
  const int64_t rid = (int64_t)r * R + i;
  if (threadIdx.x == 0) {
    float bv = sv[0];
    int bi = si[0];
    for (int q = 1; q < kWarps; ++q) argmax_merge(bv, bi, sv[q], si[q]);
    ChunkArgmax* p = A.chunk + rid * A.nch + c;
    p->v = bv;
    p->idx = bi;
    s_row_last = arrive_last(A.row_cnt + rid, (unsigned)A.nch);
  }
  __syncthreads();
  if (!s_row_last) return;
  __threadfence();

  if (threadIdx.x < 32) {
    float bv = -INFINITY;
    int bi = kNoIndex;
    for (int cc = lane; cc < A.nch; cc += 32) {
      const ChunkArgmax* p = A.chunk + rid * A.nch + cc;
      argmax_merge(bv, bi, __ldcg(&p->v), __ldcg(&p->idx));
    }
    warp_argmax(bv, bi);
    if (lane == 0) {
      A.row[rid] = bi == kNoIndex ? -1 : bi;
      s_req_last = arrive_last(A.req_cnt + r, (unsigned)(n + 1));
    }
  }
  __syncthreads();
  if (!s_req_last) return;
  __threadfence();

  // ---- request finish (warp 0; lane i is position i) ----
  if (threadIdx.x < 32) {
    bool bad = !n_ok;
    bool mism = false;
    int g = -1;
    if (n_ok && lane <= n) {
      g = __ldcg(A.row + (int64_t)r * R + lane);
      bad = g < 0;
      if (lane < n) {
        const int32_t xi = __ldg(A.tokens + (int64_t)r * A.k + lane);
        bad = bad || xi < 0 || xi >= A.V;
        mism = xi != g;
      }
      s_g[lane] = g;
    }
    const bool err = __any_sync(0xffffffffu, bad);
    const unsigned mm = __ballot_sync(0xffffffffu, mism);
    const int a = mm ? __ffs(mm) - 1 : n;
    __syncwarp();
    if (lane <= A.k) {
      int32_t out = -1;
      if (!err) {
        if (lane < a) out = __ldg(A.tokens + (int64_t)r * A.k + lane);
        else if (lane == a) out = s_g[a];
      }
      A.out_tokens[(int64_t)r * R + lane] = out;
    }
    if (lane == 0) {
      A.out_accept_len[r] = err ? -1 : a;
    }
  }
}

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
  // counters (the last two regions) start every call at zero
  cudaError_t e = cudaMemsetAsync(ws + L.row_cnt, 0, L.total - L.row_cnt, st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dtype == SV_F32)
    sample_kernel<F32><<<(unsigned)units, kThreads, 0, st>>>(A);
  else
    sample_kernel<BF16><<<(unsigned)units, kThreads, 0, st>>>(A);
  return launch_status();
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
  cudaError_t e = cudaMemsetAsync(ws + L.row_cnt, 0, L.total - L.row_cnt, st);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dtype == SV_F32)
    greedy_kernel<F32><<<(unsigned)units, kThreads, 0, st>>>(A);
  else
    greedy_kernel<BF16><<<(unsigned)units, kThreads, 0, st>>>(A);
  return launch_status();
}
