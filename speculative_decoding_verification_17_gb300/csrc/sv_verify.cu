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
// One kernel launch per call (after a small kernel that clears the call's counters), plus, for
// rows of at least 8 chunks, a second one (draw_kernel) for the draws of the batch's last
// requests, split over their chunks. Unit = (request r, row slot, segment of up to
// kSegChunks 32 KiB chunks), one CTA each (sv_stream.cuh); a request has 2k+1 row slots in
// the sampled verify (target rows 0..k, then draft rows 0..k-1) and k+1 in the greedy
// verify. Units of rows a request does not need (past its n_r) exit at once.
//
//  pass 1 (each lane, over its share of the segment)  per ring stage the lane maximum m, the
//                           integer-valued reference K = ceil(m*s) with s = log2(e)/T in
//                           fp32 and the sum of 2^(z*s - K) in fp32, folded into a running
//                           compensated pair; per segment one warp reduction to a partial
//                           (K, hi, lo); for fp32 rows, row n also keeps each stage's warp
//                           sums (its bonus draw's sub-range masses); in the greedy verify the
//                           running argmax.
//  row finish (the CTA that completes the row)  K_row = max K; S = sum of partial sums times
//                           2^(K - K_row), exact powers of two, in float-float; the row
//                           publishes S, K_row and its draft token's logit z_x.
//  request finish (the CTA that completes the request)  the accept tests u_i < p_i/q_i with
//                           p = 2^y/S, y = z_x*s - K (an fp32 ratio, re-tested exactly in
//                           double near the decision boundary), the accepted prefix a, then
//                           one draw: the residual max(0, p_a - q_a) or the bonus p_n, as the
//                           masses of every 4 KiB-or-smaller sub-range (one pass over the
//                           pair or row; for an fp32 bonus, pass 1's), the sub-range where u*W
//                           falls (one warp), and that sub-range scanned in vocabulary order
//                           (float-float sums throughout).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"

#ifndef SV_KEEP_BONUS_MASSES
#define SV_KEEP_BONUS_MASSES 1  // pass 1 keeps row n's sub-range masses for the bonus draw
#endif
#ifndef SV_RESID_RING
#define SV_RESID_RING 1  // residual pass through the TMA ring (0: register loads)
#endif

namespace sv {

int device_sm_count();  // sv_common.cu

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
// In-order draw inside one sub-range of a chunk
// ============================================================================================
struct ScanSmem {
  DF wtot[kWarps];  // each warp's total weight
  int first;        // the first vector whose running weight passes the target
  int lastpos;      // the sub-range's last token of positive weight
  int result;
};

// Inverse-CDF draw inside the sub-range that starts at s0 (kRounds * 32 16-byte vectors; the
// weights are zero past its end): the first logit j, in vocabulary order, whose running
// weight exceeds `target` (in the sub-range's units); when rounding leaves the target at or
// past the sub-range's total, or take_last is set, the last logit with positive weight.
// Thread t < kRounds * 32 takes vector t and sums its weights in order in fp32; a float-float
// scan of those sums over the block places the crossing vector, and its thread walks it. The
// scan adds in another order than the masses that chose the sub-range; where that moves the
// answer, the target lies within rounding of a boundary, and the walk falls back to the last
// positive weight. Every consumer thread calls this.
// VW provides: using Raw; Raw load(int64_t j) const; void weights(const Raw&, float (&)[]).
template <typename E, int kRounds, typename VW>
__device__ int scan_sub(int64_t s0, DF target, bool take_last, const VW& vw, ScanSmem& sm) {
  constexpr int kVec = kRounds * 32;
  static_assert(kVec <= kThreads, "one vector per thread");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    sm.first = kThreads;
    sm.lastpos = -1;
  }
  const int64_t base = s0 + (int64_t)tid * E::kPerVec;
  float wt[E::kPerVec];
  float acc = 0.0f;
  int lp = -1;
  if (tid < kVec) {
    const typename VW::Raw raw = vw.load(base);
    vw.weights(raw, wt);
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) {
      acc += wt[l];
      if (wt[l] > 0.0f) lp = (int)(base + l);
    }
  } else {
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) wt[l] = 0.0f;
  }
  const DF incl = df_warp_scan(DF{acc, 0.0f});
  DF ex = df_shfl_up(incl, 1);
  if (lane == 0) ex = DF{0.0f, 0.0f};
  if (lane == 31) sm.wtot[warp] = incl;
  cbar();
  DF start{0.0f, 0.0f};
  for (int w = 0; w < warp; ++w) start = df_add(start, sm.wtot[w]);
  start = df_add(start, ex);
  const DF through = df_add(start, DF{acc, 0.0f});
  const unsigned bl =
      __ballot_sync(0xffffffffu, !take_last && acc > 0.0f && df_gt(through, target));
  if (bl && lane == __ffs(bl) - 1) atomicMin(&sm.first, tid);
  const int lpw = __reduce_max_sync(0xffffffffu, lp);
  if (lane == 0 && lpw >= 0) atomicMax(&sm.lastpos, lpw);
  cbar();
  const int first = sm.first;
  if (tid == first) {
    int tk = -1;
    DF rr = start;
#pragma unroll
    for (int l = 0; l < E::kPerVec; ++l) {
      rr = df_add(rr, DF{wt[l], 0.0f});
      if (wt[l] > 0.0f && tk < 0 && df_gt(rr, target)) tk = (int)(base + l);
    }
    sm.result = tk < 0 ? lp : tk;  // rounding inside the vector: its last positive weight
  }
  if (tid == 0 && first == kThreads) sm.result = sm.lastpos;
  cbar();
  return sm.result;
}

// u * a for a float u, as a float-float number (about 48 bits).
__device__ __forceinline__ DF df_mul_f(DF a, float u) {
  const float p = a.hi * u;
  float e = fmaf(a.hi, u, -p);
  e = fmaf(a.lo, u, e);
  const float h = __fadd_rn(p, e);
  return {h, __fsub_rn(e, __fsub_rn(h, p))};
}

// The inverse-CDF choice of a sub-range, by one full warp: over the n masses part[f],
// f in [0, n), in vocabulary order, the first f whose running total exceeds u * W, W the
// total. Lane l sums the block [l*m, (l+1)*m), m = ceil(n/32), in float-float; a warp scan
// of the block sums gives each block's running total and W; the lane whose block first
// passes the target walks it. When rounding leaves no such f, the last f of positive mass,
// with take_last. Returns f (-1 when nothing has positive mass) and, in every lane, W and the
// target's offset into f (target minus the running total before f).
__device__ int pick_flat(int n, float u, const DF* part, DF& W, DF& offset, bool& take_last) {
  auto mass = [&](int f) { return part[f]; };
  const int lane = threadIdx.x & 31;
  const int m = (n + 31) / 32;
  const int f0 = lane * m, f1 = min(f0 + m, n);
  DF bs{0.0f, 0.0f};
  int lastf = -1;
  for (int f = f0; f < f1; ++f) {
    const DF x = mass(f);
    bs = df_add(bs, x);
    if (x.hi > 0.0f) lastf = f;
  }
  const DF incl = df_warp_scan(bs);
  W = DF{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
  const DF tgt = df_mul_f(W, u);
  DF ex = df_shfl_up(incl, 1);
  if (lane == 0) ex = DF{0.0f, 0.0f};
  const unsigned bal = __ballot_sync(0xffffffffu, lastf >= 0 && df_gt(incl, tgt));
  int pick = -1;
  DF before{0.0f, 0.0f};
  bool tl = true;
  int L;
  if (bal) {
    L = __ffs(bal) - 1;
    if (lane == L) {
      DF run = ex;
      for (int f = f0; f < f1; ++f) {
        const DF x = mass(f);
        const DF nr = df_add(run, x);
        if (x.hi > 0.0f && df_gt(nr, tgt)) {
          pick = f;
          before = run;
          tl = false;
          break;
        }
        run = nr;
      }
      if (pick < 0) pick = lastf;  // rounding inside the block: its last positive mass
    }
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, lastf >= 0);
    L = pos ? 31 - __clz(pos) : 0;
    if (lane == L) pick = lastf;
  }
  pick = __shfl_sync(0xffffffffu, pick, L);
  tl = __shfl_sync(0xffffffffu, tl ? 1 : 0, L) != 0;
  before = DF{__shfl_sync(0xffffffffu, before.hi, L), __shfl_sync(0xffffffffu, before.lo, L)};
  offset = df_add(tgt, DF{-before.hi, -before.lo});
  take_last = tl;
  return pick;
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
  WarpSoftmax* part;  // [B * (2k+1)][nseg][kWarps]
  RowSoftmax* row;
  DF* resid;          // [B][nch * 2 * kWarps] the sub-range masses of a request's draw
  WarpSoftmax* bmass;  // [B][nch * kWarps] pass 1's masses of every 4 KiB sub-range of each
                       // request's target row n, (K, hi, lo): its bonus draw's masses
  unsigned int* row_cnt;
  unsigned int* req_cnt;
  int keep_pos;             // rows of draft positions < keep_pos are copied with evict_last
  int defer;                // the last `defer` requests draw in draw_kernel
  int* draw_a;              // [B] their accepted prefix, or -1 for a data error
  int dcpc;                 // chunks per draw_kernel CTA
  unsigned int* draw_cnt;   // [B] their arrival counters in draw_kernel
};

// Residual weight max(0, p_j - q_j) with both normalisers folded in (row units).
struct ResidW {
  float s, cp, cq, ip, iq;
  __device__ __forceinline__ float operator()(float zp, float zq) const {
    const float ep = ex2(fmaf(zp, s, cp));
    const float eq = ex2(fmaf(zq, s, cq));
    return fmaxf(0.0f, fmaf(ep, ip, -(eq * iq)));
  }
  // The same for two logit pairs at once, with packed fp32x2 arithmetic (each lane of a
  // packed FMA or multiply rounds exactly like the scalar one, so the weights are identical).
  __device__ __forceinline__ float2 pair(float2 zp, float2 zq) const {
    const float2 xp = __ffma2_rn(zp, make_float2(s, s), make_float2(cp, cp));
    const float2 xq = __ffma2_rn(zq, make_float2(s, s), make_float2(cq, cq));
    const float2 ep = make_float2(ex2(xp.x), ex2(xp.y));
    const float2 eq = make_float2(ex2(xq.x), ex2(xq.y));
    const float2 nq = __fmul2_rn(eq, make_float2(-iq, -iq));
    const float2 d = __ffma2_rn(ep, make_float2(ip, ip), nq);
    return make_float2(fmaxf(0.0f, d.x), fmaxf(0.0f, d.y));
  }
};

// The weights of a draw: over a row pair, the residual (kRows = 2), or over one row, the
// bonus 2^(z*s + c) with c = -K of the row (kRows = 1). Each gives its rows, the load of one
// 16-byte vector of every row from global memory (load, zero weight past j1) or from shared
// memory holding the rows `stride` bytes apart (lds), the padding, and the weights of a
// loaded vector.
template <typename E>
struct ResidScan {
  static constexpr int kRows = 2;
  const void* rp;
  const void* rq;
  int64_t j1;
  bool aligned;
  ResidW wf;
  struct Raw {
    uint4 p, q;
  };
  __device__ __forceinline__ const void* row(int i) const { return i == 0 ? rp : rq; }
  __device__ __forceinline__ Raw load(int64_t j) const {
    return {load_vec<E>(rp, j, j1, aligned, E::kNegInfBits),
            load_vec<E>(rq, j, j1, aligned, E::kNegInfBits)};
  }
  __device__ __forceinline__ Raw lds(const unsigned char* base, int stride, int vec) const {
    return {lds16(base + vec * 16), lds16(base + stride + vec * 16)};
  }
  __device__ __forceinline__ Raw pad() const {
    return {E::pad_vec(E::kNegInfBits), E::pad_vec(E::kNegInfBits)};
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int p = 0; p < E::kPerVec / 2; ++p) {
      const float2 v = wf.pair(E::get2(r.p, p), E::get2(r.q, p));
      w[2 * p] = v.x;
      w[2 * p + 1] = v.y;
    }
  }
};

template <typename E>
struct BonusScan {
  static constexpr int kRows = 1;
  const void* rp;
  int64_t j1;
  bool aligned;
  float s, c;
  using Raw = uint4;
  __device__ __forceinline__ const void* row(int) const { return rp; }
  __device__ __forceinline__ Raw load(int64_t j) const {
    return load_vec<E>(rp, j, j1, aligned, E::kNegInfBits);
  }
  __device__ __forceinline__ Raw lds(const unsigned char* base, int, int vec) const {
    return lds16(base + vec * 16);
  }
  __device__ __forceinline__ Raw pad() const { return E::pad_vec(E::kNegInfBits); }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
#pragma unroll
    for (int p = 0; p < E::kPerVec / 2; ++p) {
      const float2 x = __ffma2_rn(E::get2(r, p), make_float2(s, s), make_float2(c, c));
      w[2 * p] = ex2(x.x);
      w[2 * p + 1] = ex2(x.y);
    }
  }
};

// Logits [j0, j1) of the rows of VW in shared memory (staged for the scan, or a piece the mass
// pass left in the ring), read back for the in-sub-range scan with the same weights.
template <typename E, class VW>
struct StagedScan {
  const VW* vw;
  const unsigned char* buf;  // logit j0 of row 0; row i starts `stride` bytes after row i-1
  int stride;
  int64_t j0, j1;
  using Raw = typename VW::Raw;
  __device__ __forceinline__ Raw load(int64_t j) const {
    if (j >= j1) return vw->pad();
    return vw->lds(buf, stride, (int)((j - j0) / E::kPerVec));
  }
  __device__ __forceinline__ void weights(const Raw& r, float (&w)[E::kPerVec]) const {
    vw->weights(r, w);
  }
};

constexpr int pow2_floor(int x) { return x >= 2 ? 2 * pow2_floor(x / 2) : 1; }

// The finishing passes see the ring (RingBytes) as two stages (its halves, on stage barriers
// 0 and 1). A draw over VW streams pieces of kPieceBytes of every row per stage, and it scans
// the chosen chunk from the ring when a whole chunk of every row fits (else from global
// memory).
template <class VW, int RingBytes>
struct DrawRing {
  static constexpr int kRingBytes = RingBytes;
  static constexpr int kHalf = kRingBytes / 2;
  static constexpr int kPieceBytes =
      pow2_floor(kHalf / VW::kRows < kChunkBytes ? kHalf / VW::kRows : kChunkBytes);
  static constexpr int kPiecesPerChunk = kChunkBytes / kPieceBytes;
  static constexpr int kVecPerLane = kPieceBytes / 16 / kThreads;
  static constexpr bool kStagedScan = VW::kRows * kChunkBytes <= kRingBytes;
  static_assert(kVecPerLane >= 1, "a piece gives every thread at least one vector");
};

// Masses of every sub-range of the rows of VW, into part[h * kWarps + warp]: piece h of the
// rows (DrawRing's pieces, kPiecesPerChunk per chunk) splits into kWarps contiguous
// sub-ranges of kVecPerLane*32 vectors, and warp w sums the w-th; false if a copy never
// landed (the masses are then NaN). With the TMA ring (aligned rows) the rows stream through
// the two halves of the ring a piece at a time: a half holds the same piece of every row, one
// bulk copy each, completing on its barrier, and the last warp out of a half starts the copy
// of the piece two ahead. Without it, every thread loads its vectors from global memory.
// Every thread calls this.
template <typename E, int RingBytes, class VW>
__device__ bool chunk_masses(int c0, int c1, int V, const VW& vw, DF* part, Ring& ring) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  using DR = DrawRing<VW, RingBytes>;
  constexpr int kPieceElems = DR::kPieceBytes / 16 * E::kPerVec;
  constexpr int kPer = DR::kPiecesPerChunk;
  constexpr int kVec = DR::kVecPerLane;
  const int h0 = c0 * kPer, np = c1 * kPer;  // the pieces [h0, np) of chunks [c0, c1)
  auto piece = [&](int h, int64_t& b, int64_t& e) {
    b = (int64_t)(h / kPer) * E::kChunk + (int64_t)(h % kPer) * kPieceElems;
    e = b + kPieceElems < V ? b + kPieceElems : (int64_t)V;
  };
  // each vector's weights in a pairwise tree of packed fp32x2 adds, then into the lane's
  // running pair; a piece's warp sum is the mass of its sub-range
  auto fold = [&](const typename VW::Raw (&raw)[kVec], float2& acc2) {
#pragma unroll
    for (int it = 0; it < kVec; ++it) {
      float w[E::kPerVec];
      vw.weights(raw[it], w);
      float2 t[E::kPerVec / 2];
#pragma unroll
      for (int p = 0; p < E::kPerVec / 2; ++p) t[p] = make_float2(w[2 * p], w[2 * p + 1]);
#pragma unroll
      for (int q = E::kPerVec / 4; q >= 1; q >>= 1)
#pragma unroll
        for (int p = 0; p < q; ++p) t[p] = __fadd2_rn(t[p], t[p + q]);
      acc2 = __fadd2_rn(acc2, t[0]);
    }
  };
  auto store = [&](int h, float2 acc2) {
    float hi = acc2.x + acc2.y, lo = 0.0f;
    warp_sum_compensated(hi, lo);
    if (lane == 0) part[(int64_t)h * kWarps + warp] = df_add(DF{hi, 0.0f}, DF{lo, 0.0f});
  };
  if (!ring.usable || !SV_RESID_RING) {
    for (int h = h0; h < np; ++h) {
      int64_t b, e;
      piece(h, b, e);
      VW q = vw;
      q.j1 = e;
      typename VW::Raw raw[kVec];
#pragma unroll
      for (int it = 0; it < kVec; ++it)
        raw[it] = q.load(b + (int64_t)(warp * (kVec * 32) + it * 32 + lane) * E::kPerVec);
      float2 acc2 = make_float2(0.0f, 0.0f);
      fold(raw, acc2);
      store(h, acc2);
    }
    return true;
  }
  auto issue = [&](int h) {
    const int st = (h - h0) & 1;
    int64_t b, e;
    piece(h, b, e);
    const uint32_t bytes = e > b ? (uint32_t)((e - b) * (16 / E::kPerVec)) : 0u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (bytes == 0) {
      mbar_arrive(&ring.full[st]);
      return;
    }
    mbar_arrive_expect_tx(&ring.full[st], VW::kRows * bytes);
#pragma unroll
    for (int i = 0; i < VW::kRows; ++i) {
      void* dst = ring.buf + st * DR::kHalf + i * DR::kPieceBytes;
      const void* src = static_cast<const char*>(vw.row(i)) + b * (16 / E::kPerVec);
      if (SV_L2_KEEP_POS > 0)
        bulk_g2s(dst, src, bytes, &ring.full[st], l2_policy(false));  // the rows' last read
      else
        bulk_g2s(dst, src, bytes, &ring.full[st]);
    }
  };
  if (tid == 0)
    for (int h = h0; h < h0 + 2 && h < np; ++h) issue(h);
  // every thread follows the same barrier phases
  bool timed_out = false;
  for (int h = h0; h < np; ++h) {
    const int st = (h - h0) & 1;
    if (!ring_wait(ring, st)) timed_out = true;
    int64_t b, e;
    piece(h, b, e);
    const unsigned char* buf = ring.buf + st * DR::kHalf;
    typename VW::Raw raw[kVec];
#pragma unroll
    for (int it = 0; it < kVec; ++it) {
      const int slot = warp * (kVec * 32) + it * 32 + lane;
      if (b + (int64_t)slot * E::kPerVec < e)
        raw[it] = vw.lds(buf, DR::kPieceBytes, slot);
      else
        raw[it] = vw.pad();
    }
    __syncwarp();
    if (lane == 0 && atomic_add_acq_rel_cta(&ring.released[st], 1) == kWarps - 1) {
      ring.released[st] = 0;
      if (h + 2 < np) issue(h + 2);
    }
    float2 acc2 = make_float2(0.0f, 0.0f);
    fold(raw, acc2);
    store(h, acc2);
  }
  if (__any_sync(0xffffffffu, timed_out)) {
    if (lane == 0) {
      atomicOr(&ring.ctl->error, 1u);
      for (int h = h0; h < np; ++h)
        part[(int64_t)h * kWarps + warp] = DF{__int_as_float(0x7fc00000), 0.0f};
    }
    return false;
  }
  return true;
}

__device__ __forceinline__ WarpSoftmax ld_part(const WarpSoftmax* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  return {v.x, v.y, v.z, v.w};
}

__device__ __forceinline__ RowSoftmax ld_row(const RowSoftmax* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  RowSoftmax r;
  r.S_hi = v.x;
  r.S_lo = v.y;
  r.zx = v.z;
  r.K = v.w;
  r.status = __ldcg(&p->status);
  return r;
}

// The accept test of one drafted position, u < p(x)/q(x), with p(x) = 2^(yp)/Sp and
// q(x) = 2^(yq)/Sq, y = zx*s - K. The ratio is formed in fp32: the exponent difference
// d = yp - yq as a float-float (each product zx*s split exactly by an FMA), 2^round(d) times
// ex2 of the remainder, times Sq/Sp. Its relative error is a few 1e-7; where u lies within
// 4e-6 * max(1, ratio) of it (or d is out of the fast path's range), the test is redone in
// double with the exponent exact, as u*Sp < 2^(yp - yq)*Sq (q(x) = 0 accepts, p(x) = q(x) =
// 0 rejects). So the decision equals the exact one wherever the exact margin is above ~1e-6.
__device__ __forceinline__ bool accept_test(float u, const RowSoftmax& t, const RowSoftmax& q,
                                            float s) {
  const float ph = t.zx * s, pl = fmaf(t.zx, s, -ph);
  const float qh = q.zx * s, ql = fmaf(q.zx, s, -qh);
  float dh, de, d2, de2;
  two_sum(ph, -qh, dh, de);
  two_sum(dh, q.K - t.K, d2, de2);
  const float dl = de + de2 + (pl - ql);
  if (fabsf(d2) <= 64.0f && fabsf(t.K) < 8.0e6f && fabsf(q.K) < 8.0e6f) {
    const float n = rintf(d2);
    const float e = ex2((d2 - n) + dl);
    const float rho = scalbnf(e * (q.S_hi / t.S_hi), (int)n);
    if (fabsf(u - rho) > 4.0e-6f * fmaxf(1.0f, rho)) return u < rho;
  }
  const double sd = (double)s;
  const double yp = (double)t.zx * sd - (double)t.K;
  const double yq = (double)q.zx * sd - (double)q.K;
  return (double)u * ((double)t.S_hi + (double)t.S_lo) <
         exp2(yp - yq) * ((double)q.S_hi + (double)q.S_lo);
}

enum DrawStatus { kDrawOk = 0, kDrawNoMass = 1, kDrawFailed = 2 };

template <typename ET>
struct SampleOp {
  using Args = SampleArgs;
  using E = ET;
  using T = SV_TILE(8, 2, 3);  // exp-heavy: whole-chunk stages, 3 CTAs of 80 registers
  static constexpr uint32_t kPad = E::kNegInfBits;
  static constexpr int kSmemChunks = 32;  // rows of up to this many chunks keep the
                                          // draw's chunk masses in shared memory
  // For fp32 rows pass 1 keeps the masses of row n's sub-ranges for the bonus draw: a ring
  // stage is one chunk, and warp w's eighth of it one sub-range of that draw. bf16 rows
  // re-read row n instead: their pass 1 issues twice the logits per byte, and there the
  // per-stage reduction cost more than the passes it saves. A ring of smaller stages, in a
  // build that forces one, keeps none.
  static constexpr bool kStageSums = SV_KEEP_BONUS_MASSES && std::is_same<ET, F32>::value &&
                                     T::kStageBytes == kChunkBytes;
  struct Smem {
    float4 wpart[kWarps];  // the warp partials of this segment
    float zx;              // the logit of the row's draft token, when prefetched
    int row_last, req_last;
    int a, err, chunk, take_last;
    DF W;
    DF before;
    RowSoftmax ra, qa, rn;  // the statistics of target row a, draft row a and target row n
    ScanSmem scan;
    DF cm[kSmemChunks * 2 * kWarps];  // the draw's sub-range masses
  };
  // One lane's running softmax sum over the segment: hi + lo (an unevaluated pair) in units
  // of 2^K, K an integer with K >= s * (the largest logit seen), and whether it saw a NaN,
  // +inf or a copy that never landed.
  struct Acc {
    float K, hi, lo;
    bool bad;
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
    g.seg = seg;
    g.keep = i < A.keep_pos;  // the early positions hold most rejections
    g.sums = kStageSums && is_target && i == n;  // row n: keep its sub-range masses
    g.c0 = seg * kSegChunks;
    g.c1 = min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  __device__ static __forceinline__ void seg_begin(Acc& a) {
    a.K = -INFINITY;
    a.hi = 0.0f;
    a.lo = 0.0f;
    a.bad = false;
  }

  // Slot of a row in its request: draft position i (target rows 0..k, draft rows k+1..2k).
  __device__ static __forceinline__ int position(const Args& A, const Seg& g) {
    return g.slot <= A.k ? g.slot : g.slot - A.k - 1;
  }

  // A row of one segment is merged by this CTA: fetch its draft token's logit while the
  // first stages are in flight.
  __device__ static __forceinline__ void prologue(const Args& A, const Seg& g, Smem& sm) {
    // a dependent draw_kernel (launched with programmatic serialization) may start its CTAs
    // as this grid's slots free up; they wait for this grid's completion before any read
    if (A.defer > 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x != 0 || g.nseg != 1) return;
    bool ok;
    const int n = n_of(A, g.r, ok);
    const int i = position(A, g);
    if (i >= n) return;
    const int32_t xi = __ldg(A.tokens + (int64_t)g.r * A.k + i);
    if (xi >= 0 && xi < A.V) sm.zx = E::load1(g.row, xi);
  }

  // Pass 1, one ring stage: the lane's maximum m over its vectors, the integer reference
  // K = ceil(m*s), the sum of 2^(z*s - K) (logits two at a time: packed fp32x2 FMA and adds,
  // two SFU exp2 per pair, a pairwise tree), then folded into the lane's running pair after
  // rescaling the side with the smaller reference by an exact power of two.
  __device__ static __forceinline__ void warp_slice(const Args& A, const Seg& g, int64_t j0,
                                                    const uint4 (&v)[T::kStageVec],
                                                    bool poison, Acc& acc) {
    constexpr int kStageVec = T::kStageVec;
    const float m = E::max_lane(v);
    acc.bad |= poison;
    float Ks = -INFINITY, ssum = 0.0f;  // the lane's stage sum, in units of 2^Ks
    if (m > -INFINITY && m < INFINITY) {
      const float s = A.s;
      const float K = ceilf(m * s);
      const float2 s2 = make_float2(s, s), c2 = make_float2(-K, -K);
      float2 part[kStageVec];
#pragma unroll
      for (int it = 0; it < kStageVec; ++it) {
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
      for (int q = kStageVec / 2; q >= 1; q >>= 1)
#pragma unroll
        for (int l = 0; l < q; ++l) part[l] = __fadd2_rn(part[l], part[l + q]);
      const float Kn = fmaxf(K, acc.K);
      const float sa = pow2_nonpos(acc.K - Kn);
      Ks = K;
      ssum = part[0].x + part[0].y;
      const float sum = ssum * pow2_nonpos(K - Kn);
      float hi, e;
      two_sum(acc.hi * sa, sum, hi, e);
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
    if (kStageSums && g.sums) stage_mass(A, g, j0, Ks, ssum);
  }

  // Row n's stage (one chunk): the warp's sub-range mass, every lane's stage sum scaled to
  // the warp's largest reference (exact), with a compensated warp sum; lane 0 stores it. A
  // row with NaN or +inf logits never draws, so what its lanes give is never used.
  __device__ static __forceinline__ void stage_mass(const Args& A, const Seg& g, int64_t j0,
                                                    float Ks, float ssum) {
    const float Kw = warp_max_f(Ks);
    float hi = Ks > -INFINITY ? ssum * pow2_nonpos(Ks - Kw) : 0.0f, lo = 0.0f;
    warp_sum_compensated(hi, lo);
    if ((threadIdx.x & 31) == 0) {
      const int64_t c = j0 / E::kChunk;
      *reinterpret_cast<float4*>(A.bmass + ((int64_t)g.r * A.nch + c) * kWarps +
                                 (threadIdx.x >> 5)) = make_float4(Kw, hi, lo, 0.0f);
    }
  }

  // End of the segment: the warp's reference K = the largest lane reference, every lane's
  // pair scaled to it (exact), and the compensated warp sum; lane 0 stores the partial.
  __device__ static __forceinline__ void seg_end(const Args& A, const Seg& g, Acc& acc,
                                                 Smem& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool bad = __any_sync(0xffffffffu, acc.bad);
    const float K = warp_max_f(acc.K);
    float4 out;
    if (bad) {
      const float nan = __int_as_float(0x7fc00000);
      out = make_float4(nan, nan, 0.0f, 0.0f);
    } else if (!(K > -INFINITY)) {
      out = make_float4(-INFINITY, 0.0f, 0.0f, 0.0f);
    } else {
      const float sc = pow2_nonpos(acc.K - K);
      float hi = acc.hi * sc, lo = acc.lo * sc;
      warp_sum_compensated(hi, lo);
      out = make_float4(K, hi, lo, 0.0f);
    }
    if (lane == 0) {
      sm.wpart[w] = out;
      if (g.nseg > 1)
        *reinterpret_cast<float4*>(A.part + ((g.rid * A.nseg + g.seg) * kWarps + w)) = out;
    }
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring& ring);
  __device__ static void finish_request(const Args& A, int r, int n, bool n_ok, Smem& sm,
                                        Ring& ring);
  template <class VW>
  __device__ static int draw(const Args& A, const VW& vw, DF* part, float u, Smem& sm,
                             Ring& ring, int& t, DF& W, bool kept = false);
  template <class VW>
  __device__ static int draw_select(const Args& A, const VW& vw, DF* part, bool landed, float u,
                                    Smem& sm, Ring& ring, int& t, DF& W, int res_lo = 0,
                                    int res_hi = 0);
  __device__ static void emit(const Args& A, int r, int a, int n, int t, DF W, int st);
  // Row n's sub-range masses as pass 1 kept them, chunks [c0, c1), into part[c * kWarps + w]
  // in units of 2^K (K: row n's reference; exact power-of-two scaling). Every thread calls
  // this.
  __device__ static void kept_masses(const Args& A, int r, float K, int c0, int c1, DF* part) {
    const float4* src = reinterpret_cast<const float4*>(A.bmass + (int64_t)r * A.nch * kWarps);
    for (int i = c0 * kWarps + threadIdx.x; i < c1 * kWarps; i += kThreads) {
      const float4 m = __ldcg(src + i);
      const float sc = m.x > -INFINITY ? pow2_nonpos(m.x - K) : 0.0f;
      part[i] = DF{m.y * sc, m.z * sc};
    }
  }
  template <class F>
  __device__ static void with_draw_weights(const Args& A, int r, int a, int n, bool bonus,
                                           F&& f, const RowSoftmax* tp_pre = nullptr,
                                           const RowSoftmax* dq_pre = nullptr);
};

template <typename ET>
__device__ void SampleOp<ET>::finish(const Args& A, const Seg& g, Smem& sm, Ring& ring) {
  const int r = g.r;
  bool n_ok;
  const int n = n_of(A, r, n_ok);
  const int i = position(A, g);
  // a row of one segment is complete here: no counter, and its partials are this CTA's
  if (threadIdx.x == 0)
    sm.row_last = g.nseg == 1 || arrive_last(A.row_cnt + g.rid, (unsigned)g.nseg);
  __syncthreads();
  if (!sm.row_last) return;
  if (g.nseg > 1) __threadfence();

  // ---- row finish: merge the warp partials of the row (warp 0; from shared memory when
  //      the row is this one segment) ----
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int np = A.nseg * kWarps;
    const WarpSoftmax* wp = A.part + g.rid * np;
    auto part_q = [&](int q) {
      if (g.nseg > 1) return ld_part(wp + q);
      const float4 v = sm.wpart[q];
      return WarpSoftmax{v.x, v.y, v.z, v.w};
    };
    float K = -INFINITY;
    bool poison = false;
    for (int q = lane; q < np; q += 32) {
      const WarpSoftmax w = part_q(q);
      poison |= (w.K != w.K) || (w.hi != w.hi);
      if (w.K > K) K = w.K;
    }
    poison = __any_sync(0xffffffffu, poison);
    K = warp_max_f(K);
    // S = sum of the partials in units of 2^K (exact power-of-two scaling), in float-float
    DF Sd{0.0f, 0.0f};
    if (K > -INFINITY)
      for (int q = lane; q < np; q += 32) {
        const WarpSoftmax w = part_q(q);
        if (w.K > -INFINITY) {
          const float sc = pow2_nonpos(w.K - K);
          Sd = df_add(Sd, df_add(DF{w.hi * sc, 0.0f}, DF{w.lo * sc, 0.0f}));
        }
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Sd = df_add(Sd, df_shfl_xor(Sd, o));
    if (lane == 0) {
      int status = (!poison && K > -INFINITY && isfinite(Sd.hi) && Sd.hi > 0.0f) ? 0 : 1;
      float zx = 0.0f;
      if (i < n) {
        const int32_t xi = __ldg(A.tokens + (int64_t)r * A.k + i);
        if (xi < 0 || xi >= A.V) status = status ? status : 2;
        else if (status == 0) zx = g.nseg == 1 ? sm.zx : E::load1(g.row, xi);
      }
      RowSoftmax* rs = A.row + g.rid;
      rs->S_hi = Sd.hi;
      rs->S_lo = Sd.lo;
      rs->zx = zx;
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

// One inverse-CDF draw with the weights vw: the masses of every sub-range (one pass over the
// rows through the ring, or already in part when kept), then draw_select: their total W, the
// sub-range in which u*W falls, and that sub-range scanned in vocabulary order. Every thread
// calls this. Returns a DrawStatus; t is the drawn token.
template <typename ET>
template <class VW>
__device__ int SampleOp<ET>::draw(const Args& A, const VW& vw, DF* part, float u, Smem& sm,
                                  Ring& ring, int& t, DF& W, bool kept) {
  using DR = DrawRing<VW, T::kRingBytes>;
  // the masses' layouts (Smem::cm, the workspace's resid region, draw_kernel's copy) hold
  // 2 * kWarps sub-ranges per chunk: a ring whose pieces are smaller than that would overflow
  // them, so such a shape does not build
  static_assert(DR::kPiecesPerChunk * kWarps <= 2 * kWarps,
                "the draw's pieces give more sub-ranges per chunk than the masses' layout holds");
  const bool landed = kept || chunk_masses<E, T::kRingBytes>(0, A.nch, A.V, vw, part, ring);
  __syncthreads();
  // the mass pass through the ring leaves its last two pieces there
  const int np = A.nch * DR::kPiecesPerChunk;
  const bool in_ring = !kept && landed && ring.usable && SV_RESID_RING;
  return draw_select(A, vw, part, landed, u, sm, ring, t, W, in_ring ? max(0, np - 2) : 0,
                     in_ring ? np : 0);
}

// The rest of a draw, from the sub-range masses in part (every chunk's, in vocabulary
// order): their total W and the sub-range in which u*W falls (one warp, pick_flat), then that
// sub-range scanned in vocabulary order by the whole CTA. Every thread calls this.
template <typename ET>
template <class VW>
__device__ int SampleOp<ET>::draw_select(const Args& A, const VW& vw, DF* part, bool landed,
                                         float u, Smem& sm, Ring& ring, int& t, DF& W,
                                         int res_lo, int res_hi) {
  const int tid = threadIdx.x, lane = tid & 31;
  using DR = DrawRing<VW, T::kRingBytes>;
  constexpr int kSubs = DR::kPiecesPerChunk * kWarps;  // sub-ranges of a chunk
  constexpr int kSubElems = DR::kVecPerLane * 32 * E::kPerVec;
  constexpr int kPieceElems = DR::kPieceBytes / 16 * E::kPerVec;
  // one warp: W and the sub-range in which u*W falls (the flat pick over every chunk's
  // sub-range masses, in vocabulary order)
  if (tid < 32) {
    DF Wd, off;
    bool tl;
    const int f = pick_flat(A.nch * kSubs, u, part, Wd, off, tl);
    if (lane == 0) {
      sm.W = Wd;
      sm.chunk = f < 0 ? 0 : f;
      sm.before = off;
      sm.take_last = tl;
    }
  }
  __syncthreads();
  W = sm.W;
  if (!landed || W.hi != W.hi) return kDrawFailed;
  if (!(W.hi > 0.0f)) return kDrawNoMass;
  const int c = sm.chunk / kSubs, q = sm.chunk - (sm.chunk / kSubs) * kSubs;
  const int64_t s0 = (int64_t)c * E::kChunk + (int64_t)(q / kWarps) * kPieceElems +
                     (int64_t)(q % kWarps) * kSubElems;
  VW sq = vw;
  sq.j1 = s0 + kSubElems < A.V ? s0 + kSubElems : (int64_t)A.V;
  if (!ring.usable) {
    t = scan_sub<E, DR::kVecPerLane>(s0, sm.before, sm.take_last != 0, sq, sm.scan);
    return kDrawOk;
  }
  // the mass pass left its last pieces [res_lo, res_hi) in the ring (piece h in half h & 1,
  // row i at i * kPieceBytes): a sub-range inside one of them is scanned from there
  const int h = c * DR::kPiecesPerChunk + q / kWarps;
  if (h >= res_lo && h < res_hi) {
    const StagedScan<E, VW> rs{&sq, ring.buf + (h & 1) * DR::kHalf, DR::kPieceBytes,
                               (int64_t)c * E::kChunk + (int64_t)(q / kWarps) * kPieceElems,
                               sq.j1};
    t = scan_sub<E, DR::kVecPerLane>(s0, sm.before, sm.take_last != 0, rs, sm.scan);
    return kDrawOk;
  }
  // nobody reads the ring any more (the barrier above): stage the sub-range of every row
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)((sq.j1 - s0) * (16 / E::kPerVec));
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
    for (int i = 0; i < VW::kRows; ++i) {
      mbar_arrive_expect_tx(&ring.full[i], bytes);
      bulk_g2s(ring.buf + i * kChunkBytes,
               static_cast<const char*>(vw.row(i)) + s0 * (16 / E::kPerVec), bytes,
               &ring.full[i]);
    }
  }
  bool ok = true;
#pragma unroll
  for (int i = 0; i < VW::kRows; ++i) ok &= ring_wait(ring, i);
  const StagedScan<E, VW> ss{&sq, ring.buf, kChunkBytes, s0, sq.j1};
  t = scan_sub<E, DR::kVecPerLane>(s0, sm.before, sm.take_last != 0, ss, sm.scan);
  if (!__syncthreads_and(ok)) {
    if (tid == 0) atomicOr(&ring.ctl->error, 1u);
    return kDrawFailed;
  }
  return kDrawOk;
}

// The weights of request r's draw, handed to f: the residual max(0, p_a - q_a) (a < n, not
// bonus), or the bonus draw from p of target row a (a = n after full acceptance, or a row
// whose residual vanished through rounding), in units of 2^K of that row. The rows'
// statistics come from tp_pre (target row a) and dq_pre (draft row a) when the caller holds
// them, else from the workspace.
template <typename ET>
template <class F>
__device__ void SampleOp<ET>::with_draw_weights(const Args& A, int r, int a, int n, bool bonus,
                                                F&& f, const RowSoftmax* tp_pre,
                                                const RowSoftmax* dq_pre) {
  const int R = 2 * A.k + 1;
  if (a < n && !bonus) {
    const RowSoftmax tp = tp_pre ? *tp_pre : ld_row(A.row + (int64_t)r * R + a);
    const RowSoftmax dq = dq_pre ? *dq_pre : ld_row(A.row + (int64_t)r * R + A.k + 1 + a);
    ResidScan<E> rs;
    rs.rp = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + a, A.V);
    rs.rq = row_ptr<E>(A.draft, (int64_t)r * A.k + a, A.V);
    rs.j1 = A.V;
    rs.aligned = A.aligned;
    rs.wf.s = A.s;
    rs.wf.cp = -tp.K;
    rs.wf.cq = -dq.K;
    rs.wf.ip = 1.0f / tp.S_hi;  // S_lo is below half an ulp of S_hi
    rs.wf.iq = 1.0f / dq.S_hi;
    f(rs);
  } else {
    const RowSoftmax rw = tp_pre ? *tp_pre : ld_row(A.row + (int64_t)r * R + a);
    BonusScan<E> bs;
    bs.rp = row_ptr<E>(A.target, (int64_t)r * (A.k + 1) + a, A.V);
    bs.j1 = A.V;
    bs.aligned = A.aligned;
    bs.s = A.s;
    bs.c = -rw.K;
    f(bs);
  }
}

// Write request r's outputs: the accepted drafts, the drawn token t and -1 padding, the
// accept length and the residual mass; or, when the draw did not succeed (st), the error
// sentinel. Every thread calls this.
template <typename ET>
__device__ void SampleOp<ET>::emit(const Args& A, int r, int a, int n, int t, DF W, int st) {
  const int tid = threadIdx.x;
  if (st != kDrawOk) {  // a data error, or a copy that never landed: the error sentinel
    if (tid <= A.k) A.out_tokens[(int64_t)r * (A.k + 1) + tid] = -1;
    if (tid == 0) {
      A.out_accept_len[r] = -1;
      if (A.out_resid) A.out_resid[r] = __int_as_float(0x7fc00000);
    }
    return;
  }
  if (tid <= A.k) {
    int32_t val = -1;
    if (tid < a) val = __ldg(A.tokens + (int64_t)r * A.k + tid);
    else if (tid == a) val = t;
    A.out_tokens[(int64_t)r * (A.k + 1) + tid] = val;
  }
  if (tid == 0) {
    A.out_accept_len[r] = a;
    if (A.out_resid) A.out_resid[r] = a < n ? W.hi : 0.0f;
  }
}

template <typename ET>
__device__ void SampleOp<ET>::finish_request(const Args& A, int r, int n, bool n_ok, Smem& sm,
                                             Ring& ring) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int R = 2 * A.k + 1;
  const float* u = A.uniforms + (int64_t)r * (A.k + 1);

  // ---- accept tests (warp 0; lane i is draft position i); the statistics of the rows the
  //      draw uses stay in shared memory ----
  if (tid < 32) {
    bool bad = !n_ok;
    bool reject = false;
    float pt = 0.0f, pq = 0.0f;
    // every load first (one round trip), then the tests
    RowSoftmax t{}, q{}, tn{};
    float ui = 0.0f, uk = 0.0f;
    const bool pos = n_ok && lane < n;
    if (pos) {
      t = ld_row(A.row + (int64_t)r * R + lane);
      q = ld_row(A.row + (int64_t)r * R + A.k + 1 + lane);
      ui = __ldg(u + lane);
    }
    if (n_ok && lane == 0) {
      tn = ld_row(A.row + (int64_t)r * R + n);
      uk = __ldg(u + A.k);
    }
    if (pos) {
      bad = t.status != 0 || q.status != 0 || !(ui >= 0.0f && ui < 1.0f);
      reject = !accept_test(ui, t, q, A.s);
      // the optional p and q outputs, in fp32
      pt = ex2(fmaf(t.zx, A.s, -t.K)) / t.S_hi;
      pq = ex2(fmaf(q.zx, A.s, -q.K)) / q.S_hi;
    }
    if (n_ok && lane == 0) {
      bad = bad || tn.status != 0 || !(uk >= 0.0f && uk < 1.0f);
      sm.rn = tn;
    }
    const bool err = __any_sync(0xffffffffu, bad);
    const unsigned rej = __ballot_sync(0xffffffffu, reject);
    const int a = rej ? __ffs(rej) - 1 : n;
    if (lane == a && a < n) {
      sm.ra = t;
      sm.qa = q;
    }
    if (lane < A.k) {
      const float nan = __int_as_float(0x7fc00000);
      if (A.out_p) A.out_p[(int64_t)r * A.k + lane] = err ? nan : (lane < n ? pt : 0.0f);
      if (A.out_q) A.out_q[(int64_t)r * A.k + lane] = err ? nan : (lane < n ? pq : 0.0f);
    }
    if (lane == 0) {
      sm.a = a;
      sm.err = err;
    }
  }
  __syncthreads();
  const int a = sm.a;
  // a deferred request (one of the launch's last): its draw follows in draw_kernel, the
  // launch after this one, split over its chunks
  if (A.defer > 0 && r >= A.B - A.defer) {
    if (tid == 0) A.draw_a[r] = sm.err ? -1 : a;
    if (sm.err) emit(A, r, a, n, -1, DF{0.0f, 0.0f}, kDrawFailed);
    return;
  }
  int t = -1;
  DF W{0.0f, 0.0f};
  int st = kDrawFailed;
  if (!sm.err) {
    const float uk = __ldg(u + A.k);
    DF* part = A.nch <= kSmemChunks  // [nch][up to 2 * kWarps]
                       ? sm.cm
                       : A.resid + (int64_t)r * A.nch * (2 * kWarps);
    st = kDrawNoMass;
    if (a < n)  // the residual norm(max(0, p_a - q_a))
      with_draw_weights(
          A, r, a, n, false,
          [&](const auto& vw) { st = draw(A, vw, part, uk, sm, ring, t, W); }, &sm.ra, &sm.qa);
    if (st == kDrawNoMass) {
      // the bonus draw from p (row n after full acceptance, from the masses pass 1 kept; row
      // a if the residual vanished through rounding, with a pass of its own)
      DF Wb;
      const bool kept = kStageSums && a == n;
      if (kept) kept_masses(A, r, sm.rn.K, 0, A.nch, part);
      with_draw_weights(
          A, r, a, n, true,
          [&](const auto& vw) { st = draw(A, vw, part, uk, sm, ring, t, Wb, kept); },
          a == n ? &sm.rn : &sm.ra);
      if (st == kDrawNoMass) st = kDrawFailed;
    }
  }
  emit(A, r, a, n, t, W, st);
}

// The draws of the deferred requests (the last `defer` of the batch), one CTA per (request,
// run of A.dcpc chunks): each computes the sub-range masses of its chunks of the request's
// draw rows, as the request's own finisher would, and the CTA that completes the request
// takes the rest of the draw (the same code on the same masses, so the same token) and
// writes its outputs. Launched right after segment_kernel<SampleOp> on the same stream,
// which wrote each deferred request's accepted prefix (or -1 for a data error) and every
// row's statistics.
template <typename E>
__global__ void __launch_bounds__(kThreads, SampleOp<E>::T::kCtasPerSm)
    draw_kernel(const SampleArgs A, CallCtl* ctl) {
  using Op = SampleOp<E>;
  constexpr int kSubsMax = 2 * kWarps;
  extern __shared__ __align__(128) unsigned char ring_buf[];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ int released[2];
  __shared__ typename Op::Smem sm;
  // the verify launch before this one must be complete, its writes visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nct = (A.nch + A.dcpc - 1) / A.dcpc;  // CTAs per request
  const int r = A.B - A.defer + (int)(blockIdx.x / (unsigned)nct);
  const int c0 = (int)(blockIdx.x % (unsigned)nct) * A.dcpc;
  const int c1 = min(c0 + A.dcpc, A.nch);
  const int a = __ldcg(A.draw_a + r);
  if (a < 0) return;  // a data error: the verify wrote the sentinel
  bool n_ok;
  const int n = Op::n_of(A, r, n_ok);
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    released[0] = released[1] = 0;
    fence_barrier_init();
  }
  __syncthreads();
  Ring ring{ring_buf, full, released, 0u, ctl, A.aligned};
  DF* gpart = A.resid + (int64_t)r * A.nch * (2 * kWarps);
  bool landed = true;
  if (Op::kStageSums && a == n) {  // the bonus draw: row n's masses are pass 1's
    Op::kept_masses(A, r, ld_row(A.row + (int64_t)r * (2 * A.k + 1) + n).K, c0, c1, gpart);
  } else {
    Op::with_draw_weights(A, r, a, n, false, [&](const auto& vw) {
      landed = chunk_masses<E, Op::T::kRingBytes>(c0, c1, A.V, vw, gpart, ring);
    });
  }
  __syncthreads();  // every warp's masses are stored
  if (tid == 0) sm.req_last = arrive_last(A.draw_cnt + r, (unsigned)nct);
  __syncthreads();
  if (!sm.req_last) return;
  __threadfence();
  // the masses of every chunk, into shared memory (written by the request's other CTAs)
  for (int i = tid; i < A.nch * kSubsMax; i += kThreads)
    sm.cm[i] = DF{__ldcg(&gpart[i].hi), __ldcg(&gpart[i].lo)};
  __syncthreads();
  const float uk = __ldg(A.uniforms + (int64_t)r * (A.k + 1) + A.k);
  int t = -1, st = kDrawFailed;
  DF W{0.0f, 0.0f};
  Op::with_draw_weights(A, r, a, n, false, [&](const auto& vw) {
    st = Op::draw_select(A, vw, sm.cm, landed, uk, sm, ring, t, W);
  });
  if (st == kDrawNoMass && a < n) {  // the residual vanished through rounding: p_a
    DF Wb;
    Op::with_draw_weights(A, r, a, n, true, [&](const auto& vw) {
      st = Op::draw(A, vw, sm.cm, uk, sm, ring, t, Wb);
    });
  }
  if (st == kDrawNoMass) st = kDrawFailed;
  Op::emit(A, r, a, n, t, W, st);
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
  WarpArgmax* part;  // [B * (k+1)][nseg][kWarps]
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

// TileT: half-chunk stages, two deep, 4 CTAs per SM for grids of many waves (a light scan);
// four deep, 3 CTAs per SM for grids of up to two waves, where each CTA's first bytes in
// flight set the time (a 64 KiB row is then requested at once).
template <typename ET, class TileT = SV_TILE(4, 2, 4)>
struct GreedyOp {
  using Args = GreedyArgs;
  using E = ET;
  using T = TileT;
  static constexpr uint32_t kPad = E::kNaNBits;  // NaN padding is never chosen
  struct Smem {
    float2 wpart[kWarps];  // the warp partials of this segment
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
    g.seg = seg;
    g.keep = false;
    g.c0 = seg * kSegChunks;
    g.c1 = min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  // One lane's running argmax over the segment, in increasing logit index.
  struct Acc {
    float best;
    int bidx;
    bool poison;
  };

  __device__ static __forceinline__ void seg_begin(Acc& a) {
    a.best = -INFINITY;
    a.bidx = kNoIndex;
    a.poison = false;
  }

  __device__ static __forceinline__ void warp_slice(const Args&, const Seg&, int64_t j0,
                                                    const uint4 (&v)[T::kStageVec],
                                                    bool poison, Acc& acc) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    acc.poison |= poison;
#pragma unroll
    for (int it = 0; it < T::kStageVec; ++it) {
      const int jb = (int)(j0 + (int64_t)warp_vec_slot<T::kStageVec>(w, it, lane) * E::kPerVec);
#pragma unroll
      for (int l = 0; l < E::kPerVec; ++l) {
        const float z = E::get(v[it], l);
        // in increasing j: the first comparable logit, then only strictly larger ones
        if (z > acc.best || (acc.bidx == kNoIndex && z == z)) {
          acc.best = z;
          acc.bidx = jb + l;
        }
      }
    }
  }

  __device__ static __forceinline__ void prologue(const Args&, const Seg&, Smem&) {}

  __device__ static __forceinline__ void seg_end(const Args& A, const Seg& g, Acc& acc,
                                                 Smem& sm) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const bool poison = __any_sync(0xffffffffu, acc.poison);
    warp_argmax(acc.best, acc.bidx);
    if (lane == 0) {
      const float2 out = make_float2(acc.best, __int_as_float(poison ? kPoisoned : acc.bidx));
      sm.wpart[w] = out;
      if (g.nseg > 1)
        *reinterpret_cast<float2*>(A.part + ((g.rid * A.nseg + g.seg) * kWarps + w)) = out;
    }
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring&) {
    const int r = g.r;
    bool n_ok;
    const int n = n_of(A, r, n_ok);
    const int R = A.k + 1;
    const int lane = threadIdx.x & 31;
    // a row of one segment is complete here: no counter, and its partials are this CTA's
    if (threadIdx.x == 0)
      sm.row_last = g.nseg == 1 || arrive_last(A.row_cnt + g.rid, (unsigned)g.nseg);
    __syncthreads();
    if (!sm.row_last) return;
    if (g.nseg > 1) __threadfence();

    if (threadIdx.x < 32) {
      const int np = A.nseg * kWarps;
      const WarpArgmax* wp = A.part + g.rid * np;
      float bv = -INFINITY;
      int bi = kNoIndex;
      bool poison = false;
      for (int q = lane; q < np; q += 32) {
        const float2 pv =
            g.nseg > 1 ? __ldcg(reinterpret_cast<const float2*>(wp + q)) : sm.wpart[q];
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

// How many of the batch's last requests leave their draw to draw_kernel. A request's draw
// runs in one CTA after its last row, one chunk after another, and re-reads 2 of the
// request's 2k+1 rows; the last requests' draws run on while little else does. The requests
// deferred are the last M, M = kDeferScale * slots * 2 / ((2k+1) * CTAs per request): the
// share of the launch whose draw re-reads would outlast its streaming (kDeferScale = 16,
// measured on B=512, k=8, V=128256 bf16 and B=256, k=4, V=151936 fp32). Rows of fewer than
// kDeferMinChunks chunks gain less than the second launch costs; rows of more than
// kSmemChunks chunks do not hold their masses in shared memory.
#ifndef SV_DEFER_SCALE
#define SV_DEFER_SCALE 16
#endif
#ifndef SV_DEFER_MIN_CHUNKS
#define SV_DEFER_MIN_CHUNKS 8
#endif
#ifndef SV_DRAW_PDL
#define SV_DRAW_PDL 1
#endif
constexpr int64_t kDeferMinChunks = SV_DEFER_MIN_CHUNKS;
int deferred_requests(int B, int k, int nseg, int64_t nch) {
  constexpr int kSmemChunks = SampleOp<F32>::kSmemChunks;
  if (SV_DEFER_SCALE <= 0 || nch < kDeferMinChunks || nch > kSmemChunks) return 0;
  const int64_t slots = (int64_t)device_sm_count() * SampleOp<F32>::T::kCtasPerSm;
  const int64_t rows = 2 * k + 1;
  const int64_t per_request = rows * nseg;
  const int64_t m = (SV_DEFER_SCALE * slots * 2 + rows * per_request - 1) / (rows * per_request);
  return (int)std::min<int64_t>(m, B);
}

// How many draft positions' rows (target and draft) pass 1 copies with evict_last. Most
// rejections fall on the first positions, and the draw then finds that pair in L2 if it was
// kept; keeping more than L2 can hold pushes the kept rows out of each other's way. The rows
// kept while a wave of CTAs is resident stay within kKeepBytes: positions
// kKeepBytes / (requests resident * 2 rows * row bytes), at least 1 (measured: 2 for B=512,
// k=8, V=128256 bf16 and 1 for B=256, k=4, V=151936 fp32 were each the best setting).
constexpr int64_t kKeepBytes = 32ll << 20;
int keep_positions(int k, int nseg, int V, sv_dtype d) {
  if (SV_L2_KEEP_POS <= 0) return 0;
  const int64_t slots = (int64_t)device_sm_count() * SampleOp<F32>::T::kCtasPerSm;
  const int64_t per_request = (int64_t)(2 * k + 1) * nseg;
  const int64_t resident = std::max<int64_t>(1, slots / per_request);
  const int64_t per_position = resident * 2 * (int64_t)V * elem_bytes(d);
  const int64_t p = kKeepBytes / per_position;
  return (int)std::max<int64_t>(1, std::min<int64_t>(p, k));
}

// Chunks per draw_kernel CTA: one, unless the deferred requests' chunks outnumber the CTA
// slots of one wave; then as many as make them fit one (each CTA streams its chunks through
// its ring, which keeps two pieces in flight across them): the kernel is latency-bound, and a
// second or third wave waits for the first.
#ifndef SV_DRAW_ONE_WAVE
#define SV_DRAW_ONE_WAVE 1
#endif
int draw_chunks_per_cta(int defer, int64_t nch) {
  if (defer <= 0 || !SV_DRAW_ONE_WAVE) return 1;
  const int64_t slots = (int64_t)device_sm_count() * SampleOp<F32>::T::kCtasPerSm;
  const int64_t units = (int64_t)defer * nch;
  return (int)std::max<int64_t>(1, std::min<int64_t>(nch, (units + slots - 1) / slots));
}

// Launch draw_kernel for the deferred requests (CTAs of draw_chunks_per_cta chunks of one
// request).
template <typename E>
sv_status launch_draws(const SampleArgs& A, CallCtl* ctl, cudaStream_t st) {
  constexpr int kRingBytes = SampleOp<E>::T::kRingBytes;
  static std::atomic<unsigned long long> ready{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (!(ready.load() & bit)) {
    e = cudaFuncSetAttribute(draw_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRingBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(draw_kernel<E>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return cuda_fail(e);
    if (bit) ready.fetch_or(bit);
  }
  // programmatic serialization: the CTAs may become resident while the verify launch
  // finishes, and wait in griddepcontrol.wait for its completion
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((int64_t)A.defer * ((A.nch + A.dcpc - 1) / A.dcpc)), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kRingBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = SV_DRAW_PDL;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, draw_kernel<E>, A, ctl);
  return e == cudaSuccess ? SV_OK : cuda_fail(e);
}

}  // namespace

extern "C" size_t spec_verify_sample_workspace(int B, int k, int V, sv_dtype dtype) {
  if (B < 0 || k < 1 || k > SV_MAX_K || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return sample_layout(B, k, V, dtype).total;
}

extern "C" int spec_verify_sample_launches(int B, int k, int V, sv_dtype dtype) {
  if (B <= 0 || k < 1 || k > SV_MAX_K || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  const int64_t nch = num_chunks(V, dtype);
  return deferred_requests(B, k, num_segments(nch), nch) > 0 ? 3 : 2;  // with the clear
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
  A.resid = reinterpret_cast<DF*>(ws + L.resid);
  A.bmass = reinterpret_cast<WarpSoftmax*>(ws + L.bmass);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  A.req_cnt = reinterpret_cast<unsigned int*>(ws + L.req_cnt);
  A.draw_a = reinterpret_cast<int*>(ws + L.draw_a);
  A.draw_cnt = reinterpret_cast<unsigned int*>(ws + L.draw_cnt);
  A.defer = deferred_requests(B, k, nseg, nch);
  A.dcpc = draw_chunks_per_cta(A.defer, nch);
  A.keep_pos = keep_positions(k, nseg, V, dtype);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // the control word and the counters (the last regions) start every call at zero
  const sv_status cleared = launch_clear(ws + L.ctl, L.total - L.ctl, st);
  if (cleared != SV_OK) return cleared;
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  sv_status s = dtype == SV_F32 ? launch_segments<SampleOp<F32>>(A, units, ctl, st)
                                : launch_segments<SampleOp<BF16>>(A, units, ctl, st);
  if (s != SV_OK || A.defer == 0) return s;
  return dtype == SV_F32 ? launch_draws<F32>(A, ctl, st) : launch_draws<BF16>(A, ctl, st);
}

extern "C" size_t spec_verify_greedy_workspace(int B, int k, int V, sv_dtype dtype) {
  if (B < 0 || k < 1 || k > SV_MAX_K || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return greedy_layout(B, k, V, dtype).total;
}

namespace {

// The host checks of a greedy-verify call, in the order both greedy entry points apply them:
// sizes and dtype, then the pointers and their alignment, then the grid size. SV_OK for a
// call that has work to launch; `empty` is set for B = 0 (a no-op).
sv_status greedy_check(const void* target_logits, sv_dtype dtype, const int32_t* draft_tokens,
                       const int32_t* num_draft, int B, int k, int V, const int32_t* out_tokens,
                       const int32_t* out_accept_len, bool& empty) {
  empty = false;
  if (B < 0 || k < 1 || V < 2) return SV_ERR_INVALID_ARG;
  if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
  if (k > SV_MAX_K) return SV_ERR_UNSUPPORTED;
  if (B == 0) {
    empty = true;
    return SV_OK;
  }
  const int eb = elem_bytes(dtype);
  if (!target_logits || !draft_tokens || !out_tokens || !out_accept_len)
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(target_logits, eb) || !aligned_to(draft_tokens, 4) ||
      !aligned_to(out_tokens, 4) || !aligned_to(out_accept_len, 4) ||
      (num_draft && !aligned_to(num_draft, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t units = (int64_t)B * (k + 1) * num_segments(num_chunks(V, dtype));
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  return SV_OK;
}

}  // namespace

extern "C" sv_status spec_verify_greedy(const void* target_logits, sv_dtype dtype,
                                        const int32_t* draft_tokens, const int32_t* num_draft,
                                        int B, int k, int V, int32_t* out_tokens,
                                        int32_t* out_accept_len, void* workspace,
                                        size_t workspace_bytes, sv_stream_t stream) {
  bool empty = false;
  const sv_status chk = greedy_check(target_logits, dtype, draft_tokens, num_draft, B, k, V,
                                     out_tokens, out_accept_len, empty);
  if (chk != SV_OK || empty) return chk;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = (int64_t)B * (k + 1) * nseg;
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
  const sv_status cleared = launch_clear(ws + L.ctl, L.total - L.ctl, st);
  if (cleared != SV_OK) return cleared;
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  using Deep = SV_TILE(4, 4, 3);
  if (units <= 2 * (int64_t)device_sm_count() * Deep::kCtasPerSm) {  // up to two waves
    if (dtype == SV_F32) return launch_segments<GreedyOp<F32, Deep>>(A, units, ctl, st);
    return launch_segments<GreedyOp<BF16, Deep>>(A, units, ctl, st);
  }
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
// that device current, and kept for the life of the process: a cudaDeviceReset (or any other
// teardown of the device's primary context) after that first call is not supported, since
// the kept address would then name memory the new context does not hold.
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
  // the same checks, in the same order, as spec_verify_greedy; then the scratch limit
  bool empty = false;
  const sv_status chk = greedy_check(target_logits, dtype, draft_tokens, num_draft, B, k, V,
                                     out_tokens, out_accept_len, empty);
  if (chk != SV_OK || empty) return chk;
  if (greedy_layout(B, k, V, dtype).total > kGreedyScratchBytes) return SV_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const sv_status st = greedy_scratch_address(&scratch);
  if (st != SV_OK) return st;
  return spec_verify_greedy(target_logits, dtype, draft_tokens, num_draft, B, k, V, out_tokens,
                            out_accept_len, scratch, kGreedyScratchBytes, stream);
}
