// sv_host.h — host-side helpers of the C ABI: status bookkeeping, argument checks and the
// workspace layouts shared by each *_workspace() query and its launcher.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

// Record a CUDA error for sv_last_cuda_error() and turn it into SV_ERR_CUDA.
sv_status cuda_fail(cudaError_t e);

// Zero `bytes` (a multiple of 16) at the 16-byte aligned device address p, on stream st,
// with a small kernel after which a segment kernel launched with programmatic serialization
// may start at once (sv_common.cu).
sv_status launch_clear(void* p, size_t bytes, cudaStream_t st);
#ifndef SV_CLEAR_KERNEL
#define SV_CLEAR_KERNEL 1
#endif

// Status of the launch just issued on this thread.
inline sv_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SV_OK : cuda_fail(e);
}

inline bool aligned_to(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline int elem_bytes(sv_dtype d) { return d == SV_F32 ? 4 : 2; }

// Logits per chunk (the unit of work of one CTA): 32 KiB of logits.
inline int64_t chunk_elems(sv_dtype d) { return d == SV_F32 ? 8192 : 16384; }

inline int64_t num_chunks(int V, sv_dtype d) {
  const int64_t c = chunk_elems(d);
  return (static_cast<int64_t>(V) + c - 1) / c;
}

// Per-call control word, cleared with the counters: bit 0 is set when a bounded wait for a
// chunk copy ran out (the affected rows are then reported as data errors).
struct CallCtl {
  unsigned int error;
  unsigned int pad[3];
};

// A CTA handles a row segment of up to kSegChunks consecutive chunks (a build may override
// the count to try other values).
#ifndef SV_SEG_CHUNKS
#define SV_SEG_CHUNKS 8
#endif
constexpr int kSegChunks = SV_SEG_CHUNKS;

inline int num_segments(int64_t nch) { return (int)((nch + kSegChunks - 1) / kSegChunks); }

// Partial results are kept per (row, segment, warp): warp w of a CTA reduces the w-th 4 KiB
// slice of every chunk of its segment on its own.
constexpr int kWarpsPerChunk = 8;

// Softmax partial of one warp's share of a segment: sum of 2^(z*s - K) over it, carried as
// an unevaluated float pair (hi + lo), with an integer-valued reference K >= m*s for its
// maximum m. K = -inf marks a share without a finite logit (no mass), K = NaN a poisoned
// share (NaN or +inf logits, or a copy that never landed).
struct WarpSoftmax {
  float K;
  float hi;
  float lo;
  float pad;
};

// Merged softmax statistics of one row: S = S_hi + S_lo (a float-float pair) = sum of
// 2^(z*s - K) over the row, K = the largest reference of its partials (an integer), and
// zx = the logit of the row's draft token; its probability is 2^(zx*s - K) / S.
struct RowSoftmax {
  float S_hi, S_lo;
  float zx;
  float K;
  int status;  // 0 ok, 1 not a distribution, 2 draft token out of range
  int pad[3];
};

// Confidence partial of one warp's share of a draft-row segment: S = hi + lo = sum of
// 2^(z*s - K) and B = bhi + blo = sum of 2^(z*s - K) * (z*s - K) (the entropy's moment; 0
// in the top-probability variant), with the integer reference K, and the largest logit m.
// K = -inf: no finite logit; K = NaN: poisoned.
struct ConfPartial {
  float K, m;
  float hi, lo;
  float bhi, blo;
  float pad[2];
};

// Merged statistics of one draft row for the confidence stop (in units of 2^K).
struct ConfRow {
  double S;
  double Bm;   // the entropy's moment
  float K, m;  // the row's reference and largest logit
  int status;  // 0 ok, 1 not a distribution
  int pad;
};

struct WarpArgmax {
  float v;  // largest logit of the warp's share
  int idx;  // its lowest index; kNoIndex when the share holds no comparable logit, -2 poisoned
};

struct WarpTop2 {
  float m1;  // largest logit
  int i1;    // lowest index holding it (kNoIndex if none, -2 poisoned)
  float m2;  // largest logit of the share with one copy of m1 removed
  int pad;
};

// Workspace regions. Everything from `ctl` to `total` is cleared at the start of a call.
struct SampleLayout {
  size_t part, row, resid, bmass, draw_a, ctl, row_cnt, req_cnt, draw_cnt, total;
};
inline SampleLayout sample_layout(int B, int k, int V, sv_dtype d) {
  const size_t R = 2 * static_cast<size_t>(k) + 1;
  const size_t nch = static_cast<size_t>(num_chunks(V, d));
  const size_t nseg = static_cast<size_t>(num_segments(num_chunks(V, d)));
  SampleLayout L{};
  size_t o = 0;
  L.part = o;    o = round_up(o + B * R * nseg * kWarpsPerChunk * sizeof(WarpSoftmax), 256);
  L.row = o;     o = round_up(o + B * R * sizeof(RowSoftmax), 256);
  L.resid = o;   o = round_up(o + B * nch * 2 * kWarpsPerChunk * sizeof(double), 256);
  L.bmass = o;   o = round_up(o + B * nch * kWarpsPerChunk * sizeof(WarpSoftmax), 256);
  L.draw_a = o;  o = round_up(o + B * sizeof(int), 256);
  L.ctl = o;     o = round_up(o + sizeof(CallCtl), 256);
  L.row_cnt = o; o = round_up(o + B * R * sizeof(unsigned int), 256);
  L.req_cnt = o; o = round_up(o + B * sizeof(unsigned int), 256);
  L.draw_cnt = o; o = round_up(o + B * sizeof(unsigned int), 256);
  L.total = o;
  return L;
}

struct GreedyLayout {
  size_t part, row, ctl, row_cnt, req_cnt, total;
};
inline GreedyLayout greedy_layout(int B, int k, int V, sv_dtype d) {
  const size_t R = static_cast<size_t>(k) + 1;
  const size_t nseg = static_cast<size_t>(num_segments(num_chunks(V, d)));
  GreedyLayout L{};
  size_t o = 0;
  L.part = o;    o = round_up(o + B * R * nseg * kWarpsPerChunk * sizeof(WarpArgmax), 256);
  L.row = o;     o = round_up(o + B * R * sizeof(int), 256);
  L.ctl = o;     o = round_up(o + sizeof(CallCtl), 256);
  L.row_cnt = o; o = round_up(o + B * R * sizeof(unsigned int), 256);
  L.req_cnt = o; o = round_up(o + B * sizeof(unsigned int), 256);
  L.total = o;
  return L;
}

struct ConfLayout {
  size_t part, row, ctl, row_cnt, req_cnt, total;
};
inline ConfLayout conf_layout(int B, int k, int V, sv_dtype d) {
  const size_t R = static_cast<size_t>(k);
  const size_t nseg = static_cast<size_t>(num_segments(num_chunks(V, d)));
  ConfLayout L{};
  size_t o = 0;
  L.part = o;    o = round_up(o + B * R * nseg * kWarpsPerChunk * sizeof(ConfPartial), 256);
  L.row = o;     o = round_up(o + B * R * sizeof(ConfRow), 256);
  L.ctl = o;     o = round_up(o + sizeof(CallCtl), 256);
  L.row_cnt = o; o = round_up(o + B * R * sizeof(unsigned int), 256);
  L.req_cnt = o; o = round_up(o + B * sizeof(unsigned int), 256);
  L.total = o;
  return L;
}

struct GateLayout {
  size_t part, ctl, row_cnt, total;
};
inline GateLayout gate_layout(int N, int V, sv_dtype d) {
  const size_t nseg = static_cast<size_t>(num_segments(num_chunks(V, d)));
  GateLayout L{};
  size_t o = 0;
  L.part = o;
  o = round_up(o + static_cast<size_t>(N) * nseg * kWarpsPerChunk * sizeof(WarpTop2), 256);
  L.ctl = o;     o = round_up(o + sizeof(CallCtl), 256);
  L.row_cnt = o; o = round_up(o + static_cast<size_t>(N) * sizeof(unsigned int), 256);
  L.total = o;
  return L;
}

}  // namespace sv
