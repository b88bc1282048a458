// sv_confidence.cu — the draft-side confidence stop (variable-length drafting).
//
// The "speculative-decoding-plan.md" design note, the variable-length drafting paragraph
// after "The acceptance math (standard speculative sampling)": the draft keeps proposing
// while its own confidence stays above a floor, by top probability or an inverse-entropy
// gate, and stops early when it gets unsure. Here the draft logits of k positions exist and
// one call finds, per request, the first position whose confidence is below the floor.
//
// One unit per (request, draft row below n_in, segment), on the segment driver
// (sv_stream.cuh):
//  pass 1 (each lane)  per ring stage the lane maximum and the integer reference
//                      K = ceil(m*s); S = sum of 2^x and, for the entropy, the moment
//                      B = sum of 2^x * x, with x = z*s - K (packed fp32x2 FMAs, SFU exp2),
//                      folded into the lane's running compensated pairs after exact
//                      power-of-two rescaling (B' = 2^d (B + d S) for a reference moved by
//                      d <= 0); the lane's largest logit m.
//  row finish          the row's K, m, S and B merged in float-float sums, published.
//  request finish      one lane per position, in double: c = 2^(m*s - K) / S, or c = 1/H with
//                      H = ln S - ln2 * B / S (in nats); the stop by ballot.
// A request that reads no row (n_in = 0, or a bad count) has one empty unit that writes its
// outputs.
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"

namespace sv {

struct ConfArgs {
  const void* draft;
  const int32_t* num_draft;
  int B, k, V, nch, nseg;
  float s;       // log2(e) / T, rounded to fp32
  double floor;  // the confidence floor
  bool aligned;  // every row starts on a 16-byte boundary
  int32_t* out_num_draft;
  float* out_conf;
  ConfPartial* part;  // [B * k][nseg][kWarps]
  ConfRow* row;       // [B * k]
  unsigned int* row_cnt;
  unsigned int* req_cnt;
};

template <typename E>
__device__ __forceinline__ const void* conf_row_ptr(const void* base, int64_t row, int V) {
  return static_cast<const char*>(base) + row * (int64_t)V * (16 / E::kPerVec);
}

__device__ __forceinline__ ConfRow ld_conf_row(const ConfRow* p) {
  ConfRow r;
  r.S = __ldcg(&p->S);
  r.Bm = __ldcg(&p->Bm);
  r.K = __ldcg(&p->K);
  r.m = __ldcg(&p->m);
  r.status = __ldcg(&p->status);
  return r;
}

template <typename ET, bool kEntropy>
struct ConfOp {
  using Args = ConfArgs;
  using E = ET;
  using T = SV_TILE(8, 2, 3);  // exp-heavy, like the sampled verify
  static constexpr uint32_t kPad = E::kNegInfBits;
  struct Smem {
    ConfPartial wpart[kWarps];  // the warp partials of this segment
    int row_last, req_last;
  };
  // One lane's running state over the segment: S = hi + lo and B = bh + bl in units of 2^K,
  // the largest logit m, and whether it saw a NaN, +inf or a copy that never landed.
  struct Acc {
    float K, hi, lo, bh, bl, m;
    bool bad;
  };

  __device__ static __forceinline__ int n_of(const Args& A, int r, bool& ok) {
    const int nraw = A.num_draft ? __ldg(A.num_draft + r) : A.k;
    ok = nraw >= 0 && nraw <= A.k;
    return ok ? nraw : 0;
  }

  __device__ static bool unit(const Args& A, int64_t u, Seg& g) {
    const int r = (int)(u / ((int64_t)A.k * A.nseg));
    const int rem = (int)(u - (int64_t)r * A.k * A.nseg);
    const int i = rem / A.nseg;
    const int seg = rem - i * A.nseg;
    bool ok;
    const int n = n_of(A, r, ok);
    const bool empty = n == 0;  // reads no row: unit (0, 0) only writes the outputs
    if (empty ? (i != 0 || seg != 0) : i >= n) return false;
    g.row = conf_row_ptr<E>(A.draft, (int64_t)r * A.k + i, A.V);
    g.rid = (int64_t)r * A.k + i;
    g.r = r;
    g.slot = i;
    g.seg = seg;
    g.keep = false;
    g.c0 = empty ? 0 : seg * kSegChunks;
    g.c1 = empty ? 0 : min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  __device__ static __forceinline__ void seg_begin(Acc& a) {
    a.K = -INFINITY;
    a.hi = a.lo = a.bh = a.bl = 0.0f;
    a.m = -INFINITY;
    a.bad = false;
  }

  __device__ static __forceinline__ void prologue(const Args&, const Seg&, Smem&) {}

  __device__ static __forceinline__ void warp_slice(const Args& A, const Seg&, int64_t,
                                                    const uint4 (&v)[T::kStageVec],
                                                    bool poison, Acc& acc) {
    constexpr int kStageVec = T::kStageVec;
    const float m = E::max_lane(v);
    acc.bad |= poison;
    if (m > -INFINITY && m < INFINITY) {
      acc.m = fmaxf(acc.m, m);
      const float s = A.s;
      const float K = ceilf(m * s);
      const float2 s2 = make_float2(s, s), c2 = make_float2(-K, -K);
      const float2 lo2 = make_float2(-256.0f, -256.0f);  // a masked logit's x: 0 * x = 0
      float2 part[kStageVec], bpart[kStageVec];
#pragma unroll
      for (int it = 0; it < kStageVec; ++it) {
        float2 e[E::kPerVec / 2], b[E::kPerVec / 2];
#pragma unroll
        for (int p = 0; p < E::kPerVec / 2; ++p) {
          const float2 x = __ffma2_rn(E::get2(v[it], p), s2, c2);
          e[p] = make_float2(ex2(x.x), ex2(x.y));
          if (kEntropy)
            b[p] = __fmul2_rn(e[p], make_float2(fmaxf(x.x, lo2.x), fmaxf(x.y, lo2.y)));
        }
#pragma unroll
        for (int q = E::kPerVec / 4; q >= 1; q >>= 1)
#pragma unroll
          for (int p = 0; p < q; ++p) {
            e[p] = __fadd2_rn(e[p], e[p + q]);
            if (kEntropy) b[p] = __fadd2_rn(b[p], b[p + q]);
          }
        part[it] = e[0];
        if (kEntropy) bpart[it] = b[0];
      }
#pragma unroll
      for (int q = kStageVec / 2; q >= 1; q >>= 1)
#pragma unroll
        for (int l = 0; l < q; ++l) {
          part[l] = __fadd2_rn(part[l], part[l + q]);
          if (kEntropy) bpart[l] = __fadd2_rn(bpart[l], bpart[l + q]);
        }
      // fold into the running pairs at the larger of the two references
      const float Kn = fmaxf(K, acc.K);
      const float da = acc.K - Kn, db = K - Kn;  // <= 0 (da = -inf at the start)
      const float sa = pow2_nonpos(da), sb = pow2_nonpos(db);
      const float sum = part[0].x + part[0].y;
      float hi, e;
      two_sum(acc.hi * sa, sum * sb, hi, e);
      if (kEntropy) {
        const bool has = acc.K > -INFINITY;
        const float ba = has ? (acc.bh + da * acc.hi) * sa : 0.0f;
        const float bla = has ? (acc.bl + da * acc.lo) * sa : 0.0f;
        const float bs = (bpart[0].x + bpart[0].y + db * sum) * sb;
        float bhn, be;
        two_sum(ba, bs, bhn, be);
        acc.bl = bla + be;
        acc.bh = bhn;
      }
      acc.lo = fmaf(acc.lo, sa, e);
      acc.hi = hi;
      acc.K = Kn;
    } else if (m == -INFINITY) {
      // no finite logit here: masked entries carry no mass, a NaN poisons the row
      bool nan = false;
#pragma unroll
      for (int it = 0; it < kStageVec; ++it) nan |= E::has_nan(v[it]);
      acc.bad |= nan;
    } else {
      acc.bad = true;  // +inf, or nothing but NaN
    }
  }

  // End of the segment: the warp's reference K (the largest lane K), every lane rescaled to
  // it (B with its shift), compensated warp sums; lane 0 stores the partial.
  __device__ static __forceinline__ void seg_end(const Args& A, const Seg& g, Acc& acc,
                                                 Smem& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool bad = __any_sync(0xffffffffu, acc.bad);
    const float K = warp_max_f(acc.K);
    const float m = warp_max_f(acc.m);
    ConfPartial out{};
    if (bad) {
      out.K = __int_as_float(0x7fc00000);
    } else if (!(K > -INFINITY)) {
      out.K = -INFINITY;
      out.m = -INFINITY;
    } else {
      const bool has = acc.K > -INFINITY;
      const float d = has ? acc.K - K : 0.0f;
      const float sc = has ? pow2_nonpos(d) : 0.0f;
      float hi = acc.hi * sc, lo = acc.lo * sc;
      float bh = has ? (acc.bh + d * acc.hi) * sc : 0.0f;
      float bl = has ? (acc.bl + d * acc.lo) * sc : 0.0f;
      warp_sum_compensated(hi, lo);
      if (kEntropy) warp_sum_compensated(bh, bl);
      out.K = K;
      out.m = m;
      out.hi = hi;
      out.lo = lo;
      out.bhi = kEntropy ? bh : 0.0f;
      out.blo = kEntropy ? bl : 0.0f;
    }
    if (lane == 0) {
      sm.wpart[w] = out;
      if (g.nseg > 1) A.part[(g.rid * A.nseg + g.seg) * kWarps + w] = out;
    }
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring&);
  __device__ static void finish_request(const Args& A, int r, int n, Smem& sm);
};

template <typename ET, bool kEntropy>
__device__ void ConfOp<ET, kEntropy>::finish(const Args& A, const Seg& g, Smem& sm, Ring&) {
  const int r = g.r;
  bool n_ok;
  const int n = n_of(A, r, n_ok);
  if (n == 0) {  // the empty unit of a request that reads no row
    if (threadIdx.x < A.k) {
      const float v = n_ok ? 0.0f : __int_as_float(0x7fc00000);
      if (A.out_conf) A.out_conf[(int64_t)r * A.k + threadIdx.x] = v;
    }
    if (threadIdx.x == 0) A.out_num_draft[r] = n_ok ? 0 : -1;
    return;
  }
  // a row of one segment is complete here: no counter, and its partials are this CTA's
  if (threadIdx.x == 0)
    sm.row_last = g.nseg == 1 || arrive_last(A.row_cnt + g.rid, (unsigned)g.nseg);
  __syncthreads();
  if (!sm.row_last) return;
  if (g.nseg > 1) __threadfence();

  // ---- row finish: merge the warp partials (warp 0) ----
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int np = A.nseg * kWarps;
    const ConfPartial* wp = A.part + g.rid * np;
    auto part_q = [&](int q) -> ConfPartial {
      if (g.nseg > 1) {
        ConfPartial c;
        c.K = __ldcg(&wp[q].K);
        c.m = __ldcg(&wp[q].m);
        c.hi = __ldcg(&wp[q].hi);
        c.lo = __ldcg(&wp[q].lo);
        c.bhi = __ldcg(&wp[q].bhi);
        c.blo = __ldcg(&wp[q].blo);
        return c;
      }
      return sm.wpart[q];
    };
    float K = -INFINITY, m = -INFINITY;
    bool poison = false;
    for (int q = lane; q < np; q += 32) {
      const ConfPartial w = part_q(q);
      poison |= w.K != w.K;
      if (w.K > K) K = w.K;
      if (w.m > m) m = w.m;
    }
    poison = __any_sync(0xffffffffu, poison);
    K = warp_max_f(K);
    m = warp_max_f(m);
    DF S{0.0f, 0.0f}, Bm{0.0f, 0.0f};
    if (K > -INFINITY)
      for (int q = lane; q < np; q += 32) {
        const ConfPartial w = part_q(q);
        if (w.K > -INFINITY) {
          const float d = w.K - K, sc = pow2_nonpos(d);
          S = df_add(S, df_add(DF{w.hi * sc, 0.0f}, DF{w.lo * sc, 0.0f}));
          if (kEntropy)
            Bm = df_add(Bm, df_add(DF{(w.bhi + d * w.hi) * sc, 0.0f},
                                   DF{(w.blo + d * w.lo) * sc, 0.0f}));
        }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      S = df_add(S, df_shfl_xor(S, o));
      if (kEntropy) Bm = df_add(Bm, df_shfl_xor(Bm, o));
    }
    if (lane == 0) {
      const double Sd = (double)S.hi + (double)S.lo;
      ConfRow* rw = A.row + g.rid;
      rw->S = Sd;
      rw->Bm = (double)Bm.hi + (double)Bm.lo;
      rw->K = K;
      rw->m = m;
      rw->status = (!poison && K > -INFINITY && isfinite(Sd) && Sd > 0.0) ? 0 : 1;
      sm.req_last = arrive_last(A.req_cnt + r, (unsigned)n);
    }
  }
  __syncthreads();
  if (!sm.req_last) return;
  __threadfence();
  finish_request(A, r, n, sm);
}

// The request's stop (warp 0; lane i is draft position i): c_i in double, then the first
// position below the floor.
template <typename ET, bool kEntropy>
__device__ void ConfOp<ET, kEntropy>::finish_request(const Args& A, int r, int n, Smem&) {
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  bool bad = false, below = false;
  double c = 0.0;
  if (lane < n) {
    const ConfRow w = ld_conf_row(A.row + (int64_t)r * A.k + lane);
    bad = w.status != 0;
    if (!bad) {
      if (kEntropy) {
        const double H = log(w.S) - 0.69314718055994530942 * w.Bm / w.S;
        c = H > 0.0 ? 1.0 / H : (double)INFINITY;
      } else {
        // the top probability 2^(m*s - K) / S; m*s is exact in double
        c = exp2((double)w.m * (double)A.s - (double)w.K) / w.S;
      }
      below = c < A.floor;
    }
  }
  const bool err = __any_sync(0xffffffffu, bad);
  const unsigned b = __ballot_sync(0xffffffffu, lane < n && below);
  const int stop = b ? __ffs(b) - 1 : n;
  if (lane < A.k && A.out_conf)
    A.out_conf[(int64_t)r * A.k + lane] =
        err ? __int_as_float(0x7fc00000) : (lane < n ? (float)c : 0.0f);
  if (lane == 0) A.out_num_draft[r] = err ? -1 : stop;
}

}  // namespace sv

// ============================================================================================
// C ABI
// ============================================================================================
using namespace sv;

extern "C" size_t draft_confidence_workspace(int B, int k, int V, sv_dtype dtype) {
  if (B < 0 || k < 1 || k > SV_MAX_K || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return conf_layout(B, k, V, dtype).total;
}

extern "C" sv_status draft_confidence_stop(const void* draft_logits, sv_dtype dtype,
                                           const int32_t* num_draft, int B, int k, int V,
                                           float temperature, sv_conf_mode mode,
                                           float floor_val, int32_t* out_num_draft,
                                           float* out_conf, void* workspace,
                                           size_t workspace_bytes, sv_stream_t stream) {
  if (B < 0 || k < 1 || V < 2) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (!(temperature >= 1e-4f && temperature <= 1e4f)) return SV_ERR_INVALID_ARG;
  if (mode != SV_CONF_TOP_PROB && mode != SV_CONF_INV_ENTROPY) return SV_ERR_INVALID_ARG;
  if (!std::isfinite(floor_val)) return SV_ERR_INVALID_ARG;
  if (k > SV_MAX_K) return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  const int eb = elem_bytes(dtype);
  if (!draft_logits || !out_num_draft) return SV_ERR_INVALID_ARG;
  if (!aligned_to(draft_logits, eb) || !aligned_to(out_num_draft, 4) ||
      (num_draft && !aligned_to(num_draft, 4)) || (out_conf && !aligned_to(out_conf, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = (int64_t)B * k * nseg;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const ConfLayout L = conf_layout(B, k, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;

  ConfArgs A;
  A.draft = draft_logits;
  A.num_draft = num_draft;
  A.B = B;
  A.k = k;
  A.V = V;
  A.nch = (int)nch;
  A.nseg = nseg;
  A.s = (float)(1.4426950408889634074 / (double)temperature);
  A.floor = (double)floor_val;
  A.aligned = aligned_to(draft_logits, 16) && ((int64_t)V * eb) % 16 == 0;
  A.out_num_draft = out_num_draft;
  A.out_conf = out_conf;
  char* ws = static_cast<char*>(workspace);
  A.part = reinterpret_cast<ConfPartial*>(ws + L.part);
  A.row = reinterpret_cast<ConfRow*>(ws + L.row);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.req_cnt = reinterpret_cast<unsigned int*>(ws + L.req_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const sv_status cleared = launch_clear(ws + L.ctl, L.total - L.ctl, st);
  if (cleared != SV_OK) return cleared;
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  const bool ent = mode == SV_CONF_INV_ENTROPY;
  if (dtype == SV_F32)
    return ent ? launch_segments<ConfOp<F32, true>>(A, units, ctl, st)
               : launch_segments<ConfOp<F32, false>>(A, units, ctl, st);
  return ent ? launch_segments<ConfOp<BF16, true>>(A, units, ctl, st)
             : launch_segments<ConfOp<BF16, false>>(A, units, ctl, st);
}
