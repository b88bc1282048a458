// sv_cache.cu — the ready-distribution cache of "Speculative Pre-Positioning".
//
//  record      Algorithm 1 (section 3.2) for a batch of updated sessions: the ready logits of
//              each session are scanned once by the gate's top-1/top-2 scan (sv_top2.cuh) on
//              the segment driver; the CTA that completes a row writes the session's slot
//              (decision point, argmax, gamma in double, entry tokens, flags) and, when asked,
//              every warp also stores the row it read into the session's distribution row.
//              A session whose entry would over-commit its cell budget gets one empty unit
//              that reads nothing and only clears the slot.
//  serve       Algorithm 2 (section 3.4) for a batch of requests, one warp each: validity,
//              the exact-entry eligibility test (lanes compare the entry tokens), then the
//              gate of Eq. (12) on the slot's cached (argmax, gamma): no vocabulary scan on the
//              request's path, since the scan ran when the distribution was recorded.
//  invalidate  section 3.6 and Figure 3: an atomic exchange clears a slot's flags.
// The counters of Eq. (8) (consumed and wasted pre-positions) and of each outcome are kept in
// the table's statistics with 64-bit atomics.
#include <cmath>
#include <cstdint>

#include "specverify.h"
#include "specverify_cache.h"
#include "sv_device.cuh"
#include "sv_host.h"
#include "sv_stream.cuh"
#include "sv_top2.cuh"

namespace sv {

struct RecordArgs {
  const void* logits;
  int M, V, nch, nseg;
  bool aligned;
  const int32_t* session;
  const int64_t* end_pos;
  const int32_t* entry_tokens;  // [M, max_entry]
  const int32_t* entry_len;
  const int64_t* headroom;
  sv_cache_slot* slots;
  int32_t* entry_store;  // [S, max_entry]
  int S, max_entry;
  sv_cache_stats* stats;
  void* dist_store;      // [S, V] or null
  int32_t* out_status;   // [M] or null
  WarpTop2* part;        // [M][nseg][kWarps]
  unsigned int* row_cnt;
};

__device__ __forceinline__ void count(uint64_t* c) {
  atomicAdd(reinterpret_cast<unsigned long long*>(c), 1ull);
}

// A slot leaves the valid state (record, skip): an unconsumed pre-position was wasted.
__device__ __forceinline__ void retire(sv_cache_slot* s, sv_cache_stats* st) {
  const unsigned int old = atomicExch(&s->flags, 0u);
  if ((old & SV_CACHE_VALID) && !(old & SV_CACHE_CONSUMED)) count(&st->wasted);
  atomicAdd(&s->epoch, 1u);
}

// Logit l of a 16-byte vector, stored at index j of a row (its raw bits: exact).
template <typename E>
__device__ __forceinline__ void store_logit(char* row, int64_t j, const uint4& v, int l) {
  if constexpr (E::kPerVec == 4) {
    const uint32_t w = l == 0 ? v.x : l == 1 ? v.y : l == 2 ? v.z : v.w;
    reinterpret_cast<uint32_t*>(row)[j] = w;
  } else {
    const uint32_t w = (l >> 1) == 0 ? v.x : (l >> 1) == 1 ? v.y : (l >> 1) == 2 ? v.z : v.w;
    reinterpret_cast<uint16_t*>(row)[j] = (uint16_t)((l & 1) ? (w >> 16) : (w & 0xffffu));
  }
}

template <typename ET>
struct RecordOp : Top2Scan<ET> {
  using Args = RecordArgs;
  using Base = Top2Scan<ET>;
  using typename Base::E;
  using typename Base::Smem;
  using T = typename Base::T;
  using Acc = typename Base::Acc;

  // 0: record; 1: skipped on the cell budget; -1: an argument out of range
  __device__ static __forceinline__ int row_kind(const Args& A, int m) {
    const int sid = __ldg(A.session + m);
    const int L = __ldg(A.entry_len + m);
    const int64_t n_s = __ldg(A.end_pos + m);
    if (sid < 0 || sid >= A.S || L < 0 || L > A.max_entry || n_s < 0) return -1;
    return (int64_t)L > __ldg(A.headroom + m) ? 1 : 0;
  }

  __device__ static bool unit(const Args& A, int64_t u, Seg& g) {
    const int m = (int)(u / A.nseg);
    const int seg = (int)(u - (int64_t)m * A.nseg);
    const bool empty = row_kind(A, m) != 0;  // reads nothing: unit (m, 0) writes the outcome
    if (empty && seg != 0) return false;
    g.row = static_cast<const char*>(A.logits) + (int64_t)m * A.V * (16 / E::kPerVec);
    g.rid = m;
    g.r = m;
    g.slot = empty ? -1 : __ldg(A.session + m);
    g.seg = seg;
    g.keep = false;
    g.c0 = empty ? 0 : seg * kSegChunks;
    g.c1 = empty ? 0 : min(g.c0 + kSegChunks, A.nch);
    g.nseg = A.nseg;
    return true;
  }

  // The scan's fold, and the row's copy into the session's distribution row when one is kept.
  __device__ static __forceinline__ void warp_slice(const Args& A, const Seg& g, int64_t j0,
                                                    const uint4 (&v)[T::kStageVec],
                                                    bool poison, Acc& acc) {
    Base::warp_slice(A, g, j0, v, poison, acc);
    if (!A.dist_store) return;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    char* dst = static_cast<char*>(A.dist_store) + (int64_t)g.slot * A.V * (16 / E::kPerVec);
#pragma unroll
    for (int it = 0; it < T::kStageVec; ++it) {
      const int64_t jb = j0 + (int64_t)warp_vec_slot<T::kStageVec>(w, it, lane) * E::kPerVec;
      if (A.aligned && jb + E::kPerVec <= A.V) {
        __stcs(reinterpret_cast<uint4*>(dst) + jb / E::kPerVec, v[it]);
      } else {
        // the row's end, or rows off the 16-byte grid: logit by logit, inside the row
#pragma unroll
        for (int l = 0; l < E::kPerVec; ++l)
          if (jb + l < A.V) store_logit<E>(dst, jb + l, v[it], l);
      }
    }
  }

  __device__ static void finish(const Args& A, const Seg& g, Smem& sm, Ring&) {
    const int m = g.r;
    if (g.c1 == 0) {  // the empty unit of a skipped or bad row
      if (threadIdx.x == 0) {
        const int kind = row_kind(A, m);
        if (kind < 0) {
          count(&A.stats->bad);
        } else {
          retire(A.slots + __ldg(A.session + m), A.stats);
          count(&A.stats->skipped);
        }
        if (A.out_status) A.out_status[m] = kind < 0 ? SV_CACHE_BAD : SV_SKIPPED;
      }
      return;
    }
    if (!Base::row_complete(A, g, sm)) return;
    if (threadIdx.x >= 32) return;
    bool poison;
    const Top2 b = Base::row_top2(A, g, sm, poison);
    const int lane = threadIdx.x;
    const int sid = g.slot;
    const int L = __ldg(A.entry_len + m);
    sv_cache_slot* s = A.slots + sid;
    if (poison) {  // a copy never landed: nothing trustworthy to record
      if (lane == 0) {
        retire(s, A.stats);
        count(&A.stats->bad);
        if (A.out_status) A.out_status[m] = SV_CACHE_BAD;
      }
      return;
    }
    for (int i = lane; i < L; i += 32)
      A.entry_store[(int64_t)sid * A.max_entry + i] =
          __ldg(A.entry_tokens + (int64_t)m * A.max_entry + i);
    __syncwarp();
    if (lane == 0) {
      retire(s, A.stats);
      const bool some = b.i1 != kNoIndex;
      s->position = __ldg(A.end_pos + m) + L;
      s->gap = some ? (double)b.m1 - (double)b.m2 : __longlong_as_double(0x7ff8000000000000LL);
      s->token = some ? b.i1 : -1;
      s->entry_len = L;
      __threadfence_block();
      atomicExch(&s->flags, SV_CACHE_VALID | SV_CACHE_DECODED);
      count(&A.stats->pre_positions);
      if (A.out_status) A.out_status[m] = SV_RECORDED;
    }
  }
};

// ------------------------------------------------------------------------------ serve
struct ServeArgs {
  sv_cache_slot* slots;
  const int32_t* entry_store;
  int S, max_entry;
  sv_cache_stats* stats;
  const int32_t* session;
  const int64_t* start;
  const int32_t* req_tokens;
  const int32_t* req_len;
  int R;
  double tau;
  const int32_t* answer;
  int n_answer;
  bool exact;
  int32_t* out_token;
  int32_t* out_reason;
};

constexpr int kServeThreads = 256;

__global__ void __launch_bounds__(kServeThreads) serve_kernel(const ServeArgs A) {
  const int lane = threadIdx.x & 31;
  const int64_t r = ((int64_t)blockIdx.x * kServeThreads + threadIdx.x) >> 5;
  if (r >= A.R) return;
  const int sid = __ldg(A.session + r);
  const int L = __ldg(A.req_len + r);
  int reason, token = -1;
  if (sid < 0 || sid >= A.S || L < 0 || L > A.max_entry) {
    reason = SV_CACHE_BAD;
  } else {
    sv_cache_slot* s = A.slots + sid;
    const unsigned int flags = *reinterpret_cast<volatile unsigned int*>(&s->flags);
    if (!(flags & SV_CACHE_VALID)) {
      reason = SV_FALL_INVALID;
    } else {
      bool eligible = true;  // warp-uniform throughout
      if (A.exact) {
        const int Ls = s->entry_len;
        eligible = L == Ls && __ldg(A.start + r) == s->position - Ls;
        for (int i0 = 0; eligible && i0 < L; i0 += 32) {
          const int i = i0 + lane;
          const bool same = i >= L || __ldg(A.req_tokens + r * A.max_entry + i) ==
                                          A.entry_store[(int64_t)sid * A.max_entry + i];
          eligible = __all_sync(0xffffffffu, same);
        }
      }
      if (!eligible) {
        reason = SV_FALL_INELIGIBLE;
      } else {
        if (lane == 0) {
          const unsigned int old = atomicOr(&s->flags, SV_CACHE_CONSUMED);
          if (!(old & SV_CACHE_CONSUMED)) count(&A.stats->consumed);
        }
        const int tok = s->token;
        bool inA = false;
        if (A.n_answer > 0 && tok >= 0) {
          int lo = 0, hi = A.n_answer;  // first entry >= tok
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(A.answer + mid) < tok) lo = mid + 1;
            else hi = mid;
          }
          inA = lo < A.n_answer && __ldg(A.answer + lo) == tok;
        }
        if (s->gap > A.tau && inA) {
          reason = SV_SERVE_FAST;
          token = tok;
        } else {
          reason = SV_FALL_GATE;
        }
      }
    }
  }
  if (lane == 0) {
    A.out_token[r] = token;
    A.out_reason[r] = reason;
    uint64_t* c = reason == SV_SERVE_FAST ? &A.stats->fast
                  : reason == SV_FALL_INVALID ? &A.stats->fall_invalid
                  : reason == SV_FALL_INELIGIBLE ? &A.stats->fall_ineligible
                  : reason == SV_FALL_GATE ? &A.stats->fall_gate
                  : &A.stats->bad;
    count(c);
  }
}

__global__ void __launch_bounds__(kServeThreads) invalidate_kernel(sv_cache_slot* slots, int S,
                                                                   sv_cache_stats* stats,
                                                                   const int32_t* session,
                                                                   int n) {
  const int64_t i = (int64_t)blockIdx.x * kServeThreads + threadIdx.x;
  if (i >= n) return;
  const int sid = __ldg(session + i);
  if (sid < 0 || sid >= S) {
    count(&stats->bad);
    return;
  }
  retire(slots + sid, stats);
}

struct RecordLayout {
  size_t part, ctl, row_cnt, total;
};
inline RecordLayout record_layout(int M, int V, sv_dtype d) {
  const size_t nseg = static_cast<size_t>(num_segments(num_chunks(V, d)));
  RecordLayout L{};
  size_t o = 0;
  L.part = o;    o = round_up(o + static_cast<size_t>(M) * nseg * kWarpsPerChunk * sizeof(WarpTop2), 256);
  L.ctl = o;     o = round_up(o + sizeof(CallCtl), 256);
  L.row_cnt = o; o = round_up(o + static_cast<size_t>(M) * sizeof(unsigned int), 256);
  L.total = o;
  return L;
}

}  // namespace sv

// ============================================================================================
// C ABI
// ============================================================================================
using namespace sv;

static_assert(sizeof(sv_cache_slot) == 32, "sv_cache_slot is 32 bytes");
static_assert(sizeof(sv_cache_stats) == 72, "sv_cache_stats is 9 counters");

extern "C" size_t ready_cache_record_workspace(int M, int V, sv_dtype dtype) {
  if (M < 0 || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return 0;
  return record_layout(M, V, dtype).total;
}

static bool table_ok(const sv_cache_slot* slots, const void* entry_store, int S, int max_entry,
                     const sv_cache_stats* stats) {
  return slots && entry_store && stats && S >= 1 && max_entry >= 1 && max_entry <= 4096 &&
         aligned_to(slots, 32) && aligned_to(entry_store, 4) && aligned_to(stats, 8);
}

extern "C" sv_status ready_cache_record(sv_cache_slot* slots, int32_t* entry_store, int S,
                                        int max_entry, sv_cache_stats* stats,
                                        const int32_t* session, const int64_t* end_pos,
                                        const int32_t* entry_tokens, const int32_t* entry_len,
                                        const int64_t* headroom, int M, const void* ready_logits,
                                        sv_dtype dtype, int V, void* dist_store,
                                        int32_t* out_status, void* workspace,
                                        size_t workspace_bytes, sv_stream_t stream) {
  if (M < 0 || V < 2 || (dtype != SV_F32 && dtype != SV_BF16)) return SV_ERR_INVALID_ARG;
  if (!table_ok(slots, entry_store, S, max_entry, stats)) return SV_ERR_INVALID_ARG;
  if (M == 0) return SV_OK;
  const int eb = elem_bytes(dtype);
  if (!session || !end_pos || !entry_tokens || !entry_len || !headroom || !ready_logits)
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(session, 4) || !aligned_to(end_pos, 8) || !aligned_to(entry_tokens, 4) ||
      !aligned_to(entry_len, 4) || !aligned_to(headroom, 8) || !aligned_to(ready_logits, eb) ||
      (dist_store && !aligned_to(dist_store, eb)) || (out_status && !aligned_to(out_status, 4)))
    return SV_ERR_INVALID_ARG;
  const int64_t nch = num_chunks(V, dtype);
  const int nseg = num_segments(nch);
  const int64_t units = (int64_t)M * nseg;
  if (units > 0x7fffffffLL) return SV_ERR_UNSUPPORTED;
  const RecordLayout L = record_layout(M, V, dtype);
  if (!workspace || !aligned_to(workspace, 256) || workspace_bytes < L.total)
    return SV_ERR_WORKSPACE;
  RecordArgs A;
  A.logits = ready_logits;
  A.M = M;
  A.V = V;
  A.nch = (int)nch;
  A.nseg = nseg;
  // the copy into the distribution rows takes 16-byte stores only when those rows sit on the
  // same grid as the ready rows
  A.aligned = aligned_to(ready_logits, 16) && ((int64_t)V * eb) % 16 == 0 &&
              (!dist_store || aligned_to(dist_store, 16));
  A.session = session;
  A.end_pos = end_pos;
  A.entry_tokens = entry_tokens;
  A.entry_len = entry_len;
  A.headroom = headroom;
  A.slots = slots;
  A.entry_store = entry_store;
  A.S = S;
  A.max_entry = max_entry;
  A.stats = stats;
  A.dist_store = dist_store;
  A.out_status = out_status;
  char* ws = static_cast<char*>(workspace);
  A.part = reinterpret_cast<WarpTop2*>(ws + L.part);
  A.row_cnt = reinterpret_cast<unsigned int*>(ws + L.row_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const sv_status cleared = launch_clear(ws + L.ctl, L.total - L.ctl, st);
  if (cleared != SV_OK) return cleared;
  CallCtl* ctl = reinterpret_cast<CallCtl*>(ws + L.ctl);
  if (dtype == SV_F32) return launch_segments<RecordOp<F32>>(A, units, ctl, st);
  return launch_segments<RecordOp<BF16>>(A, units, ctl, st);
}

extern "C" sv_status ready_cache_serve(sv_cache_slot* slots, const int32_t* entry_store, int S,
                                       int max_entry, sv_cache_stats* stats,
                                       const int32_t* session, const int64_t* start,
                                       const int32_t* req_tokens, const int32_t* req_len, int R,
                                       float tau, const int32_t* answer_set, int n_answer,
                                       int exact, int32_t* out_token, int32_t* out_reason,
                                       sv_stream_t stream) {
  if (R < 0 || n_answer < 0) return SV_ERR_INVALID_ARG;
  if (!table_ok(slots, entry_store, S, max_entry, stats)) return SV_ERR_INVALID_ARG;
  if (R == 0) return SV_OK;
  if (!session || !start || !req_tokens || !req_len || !out_token || !out_reason ||
      (n_answer > 0 && !answer_set))
    return SV_ERR_INVALID_ARG;
  if (!aligned_to(session, 4) || !aligned_to(start, 8) || !aligned_to(req_tokens, 4) ||
      !aligned_to(req_len, 4) || !aligned_to(out_token, 4) || !aligned_to(out_reason, 4) ||
      (answer_set && !aligned_to(answer_set, 4)))
    return SV_ERR_INVALID_ARG;
  ServeArgs A{slots, entry_store, S, max_entry, stats, session, start, req_tokens, req_len, R,
              (double)tau, answer_set, n_answer, exact != 0, out_token, out_reason};
  const int64_t threads = (int64_t)R * 32;
  const unsigned grid = (unsigned)((threads + kServeThreads - 1) / kServeThreads);
  serve_kernel<<<grid, kServeThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(A);
  return launch_status();
}

extern "C" sv_status ready_cache_invalidate(sv_cache_slot* slots, int S, sv_cache_stats* stats,
                                            const int32_t* session, int n, sv_stream_t stream) {
  if (n < 0 || S < 1 || !slots || !stats || !aligned_to(slots, 32) || !aligned_to(stats, 8))
    return SV_ERR_INVALID_ARG;
  if (n == 0) return SV_OK;
  if (!session || !aligned_to(session, 4)) return SV_ERR_INVALID_ARG;
  const unsigned grid = (unsigned)(((int64_t)n + kServeThreads - 1) / kServeThreads);
  invalidate_kernel<<<grid, kServeThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      slots, S, stats, session, n);
  return launch_status();
}
