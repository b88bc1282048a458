// sv_stream.cuh — the driver that feeds logit chunks to a row operation.
//
// A row of V logits is cut into chunks of kChunkBytes (32 KiB). The unit of work of one
// CTA (kThreads threads; the operation's Tile sets the CTAs per SM) is a row segment of up
// to kSegChunks consecutive chunks. Warp w always owns the contiguous eighth w of a ring
// stage. Each lane folds its share of every stage of the segment into a running accumulator
// of its own, and the warp reduces the lanes once, at the end of the segment, into one
// partial per (row, segment, warp); pass 1 has no CTA-wide barrier at all.
//
// For a row that starts on a 16-byte boundary the segment streams through a kStages-deep
// shared-memory ring: thread 0 starts one cp.async.bulk (TMA) per stage, each completing on
// that stage's mbarrier; the last warp to finish reading a stage (a shared counter) starts
// the copy kStages stages ahead into it, so the next stages land while the current one is
// reduced. For rows that are not 16-byte aligned the CTA stages each piece into the ring with
// plain loads, logit by logit. Every mbarrier wait is bounded: a copy that never lands
// poisons its row (the request gets the error sentinel) and sets a bit in the call's control
// word.
//
// After the segment, thread 0 publishes it (one acquire-release atomic on the row's counter,
// after a CTA barrier; a row of one segment needs none); the CTA that completes a row merges
// its partials, and the one that completes a request finishes the request. No CTA ever
// waits for another one.
//
// An operation Op provides:
//   using E; static constexpr uint32_t kPad; struct Smem; struct Args (with bool aligned);
//   struct Acc (one lane's running state over the segment);
//   static bool unit(const Args&, int64_t u, Seg& g);       false: unit not needed
//   static void seg_begin(Acc&);
//   static void prologue(const Args&, const Seg&, Smem&);  all threads, while the first
//       stages are in flight (a place to start loads the finish will need)
//   using T = Tile<...> (the ring's shape);
//   static void warp_slice(const Args&, const Seg&, int64_t j0,
//                          const uint4 (&v)[T::kStageVec], bool poison, Acc&);
//       one warp, the ring stage that starts at logit j0 of the row, the warp's vectors v
//       (lane l holds vector warp_vec_slot<T::kStageVec>(w, it, l) of the stage in v[it],
//       logits past the row's end set to kPad); folds them into the lane's accumulator
//   static void seg_end(const Args&, const Seg&, Acc&, Smem&);  one warp: reduce and store
//       its partial (in shared memory as well, where a row of one segment merges it)
//   static void finish(const Args&, const Seg&, Smem&, Ring&);  all threads, after the segment
#pragma once

#include <atomic>

#include <cuda_runtime.h>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

// The shape of an operation's ring: 16-byte vectors per thread in one stage (a stage holds
// kThreads * Vec * 16 bytes: 32 KiB at 8, a whole chunk), ring depth, and CTAs resident per
// SM (shared memory: Ctas * kRingBytes <= 227 KiB; registers: 65536 / (Ctas * kThreads) per
// thread). Each operation picks its own: exp-heavy passes want long stages, light scans more
// warps per SM. A build may force one shape on every operation (SV_STAGE_VEC, SV_STAGES and
// SV_CTAS_PER_SM together) to compare shapes. The chunks per segment, kSegChunks, are set in
// sv_host.h, since the workspace layouts depend on them.
template <int Vec, int Stages, int Ctas>
struct Tile {
  static constexpr int kStageVec = Vec;
  static constexpr int kStages = Stages;
  static constexpr int kCtasPerSm = Ctas;
  static constexpr int kStageBytes = kThreads * Vec * 16;
  static constexpr int kRingBytes = Stages * kStageBytes;
  static_assert(kChunkBytes % kStageBytes == 0, "a chunk is a whole number of stages");
  static_assert(Stages >= 2 && Stages <= 8, "ring depth");
  static_assert(kRingBytes >= kChunkBytes, "the finishing passes need a chunk of ring");
  static_assert(Ctas * (kRingBytes + 2048) <= 232448, "shared memory of Ctas CTAs");
};
#if defined(SV_STAGE_VEC) && defined(SV_STAGES) && defined(SV_CTAS_PER_SM)
#define SV_TILE(vec, stages, ctas) Tile<SV_STAGE_VEC, SV_STAGES, SV_CTAS_PER_SM>
#else
#define SV_TILE(vec, stages, ctas) Tile<vec, stages, ctas>
#endif

// L2 priority of the pass-1 copies: with SV_L2_KEEP_POS > 0 the rows an operation marks as
// likely to be read again (Seg::keep) are copied with evict_last and all others with
// evict_first; with 0 every copy keeps its default priority. (The sampled verify marks the
// rows of its first draft positions, how many chosen per call from a budget of L2 bytes.)
#ifndef SV_L2_KEEP_POS
#define SV_L2_KEEP_POS 1
#endif
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far past any legitimate wait

// A row segment: the row (its first logit), its slot, and its chunks [c0, c1).
struct Seg {
  const void* row;
  int64_t rid;  // row id in the workspace tables
  int r;        // request (or gate row)
  int slot;     // row slot inside the request
  int c0, c1;
  int seg;      // index of this segment in the row
  int nseg;     // segments of this row
  bool keep;    // likely to be read again soon (a hint for the L2)
  bool sums = false;  // the operation keeps per-stage sums of this row (its own use)
};

// The CTA's shared-memory ring as the finishing code may reuse it once pass 1 is done:
// its buffer, the stage barriers and release counters, how many phases each stage's barrier
// has completed, and the call's control word. `usable` is false for rows read without TMA.
struct Ring {
  unsigned char* buf;
  uint64_t* full;
  int* released;
  uint32_t phase;  // bit s: parity of the next wait on stage s
  CallCtl* ctl;
  bool usable;
};

// Wait (bounded) for the next phase of stage s; every thread of the CTA calls this for every
// use of the stage, in the same order, so all keep the same phase bits.
__device__ __forceinline__ bool ring_wait(Ring& R, int s) {
  const bool ok = mbar_wait(&R.full[s], (R.phase >> s) & 1u, kWaitLimitNs);
  R.phase ^= 1u << s;
  return ok;
}

// Index, within a ring stage of Vec vectors per thread, of the 16-byte vector lane `lane`
// of warp `w` holds in slot `it`: warp w reads the w-th contiguous eighth of the stage.
template <int Vec>
__device__ __forceinline__ int warp_vec_slot(int w, int it, int lane) {
  return w * (Vec * 32) + it * 32 + lane;
}

// Copy logits [j0, j1) of a row into a ring stage, completing on its barrier.
template <typename E>
__device__ __forceinline__ void issue_stage(const Seg& g, int64_t j0, int64_t j1,
                                            unsigned char* dst, uint64_t* bar) {
  const uint32_t bytes = (uint32_t)((j1 - j0) * (16 / E::kPerVec));
  // the warps' shared-memory reads of this stage come before the async copy that overwrites it
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive_expect_tx(bar, bytes);
  const void* src = static_cast<const char*>(g.row) + j0 * (16 / E::kPerVec);
  if (SV_L2_KEEP_POS > 0)
    bulk_g2s(dst, src, bytes, bar, l2_policy(g.keep));
  else
    bulk_g2s(dst, src, bytes, bar);
}

template <class Op>
__global__ void __launch_bounds__(kThreads, Op::T::kCtasPerSm)
    segment_kernel(const typename Op::Args A, CallCtl* ctl) {
  using E = typename Op::E;
  constexpr int kStageVec = Op::T::kStageVec;
  constexpr int kStages = Op::T::kStages;
  constexpr int kStageBytes = Op::T::kStageBytes;
  constexpr int64_t kStageElems = (int64_t)kStageBytes / 16 * E::kPerVec;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ int released[kStages];
  __shared__ typename Op::Smem sm;

  Seg g;
  if (!Op::unit(A, (int64_t)blockIdx.x, g)) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t jb = (int64_t)g.c0 * E::kChunk;
  const int64_t je = (int64_t)g.c1 * E::kChunk < A.V ? (int64_t)g.c1 * E::kChunk : (int64_t)A.V;
  const int ns = (int)((je - jb + kStageElems - 1) / kStageElems);  // stages of the segment

  typename Op::Acc acc;
  Op::seg_begin(acc);
  if (A.aligned) {
    if (threadIdx.x == 0) {
      for (int s = 0; s < kStages; ++s) {
        mbar_init(&full[s], 1);
        released[s] = 0;
      }
      fence_barrier_init();
      for (int q = 0; q < kStages && q < ns; ++q) {
        const int64_t j0 = jb + q * kStageElems;
        issue_stage<E>(g, j0, j0 + kStageElems < je ? j0 + kStageElems : je,
                       ring + q * kStageBytes, &full[q]);
      }
    }
    __syncthreads();
    Op::prologue(A, g, sm);
    for (int si = 0; si < ns; ++si) {
      const int s = si % kStages;
      const bool ok = mbar_wait(&full[s], (uint32_t)((si / kStages) & 1), kWaitLimitNs);
      const bool poison = __any_sync(0xffffffffu, !ok);
      if (poison && lane == 0) atomicOr(&ctl->error, 1u);
      const int64_t j0 = jb + si * kStageElems;
      const int64_t j1 = j0 + kStageElems < je ? j0 + kStageElems : je;
      const unsigned char* buf = ring + s * kStageBytes;
      uint4 v[kStageVec];
      if (j1 - j0 == kStageElems) {  // a whole stage (CTA-uniform): no per-vector bound
#pragma unroll
        for (int it = 0; it < kStageVec; ++it)
          v[it] = lds16(buf + warp_vec_slot<kStageVec>(warp, it, lane) * 16);
      } else {
#pragma unroll
        for (int it = 0; it < kStageVec; ++it) {
          const int slot = warp_vec_slot<kStageVec>(warp, it, lane);
          v[it] = (j0 + (int64_t)slot * E::kPerVec < j1) ? lds16(buf + slot * 16)
                                                          : E::pad_vec(Op::kPad);
        }
      }
      __syncwarp();
      if (lane == 0) {  // the last warp out of a stage refills it kStages stages ahead
        if (atomic_add_acq_rel_cta(&released[s], 1) == kWarps - 1) {
          released[s] = 0;
          if (si + kStages < ns) {
            const int64_t n0 = j0 + kStages * kStageElems;
            issue_stage<E>(g, n0, n0 + kStageElems < je ? n0 + kStageElems : je,
                           ring + s * kStageBytes, &full[s]);
          }
        }
      }
      Op::warp_slice(A, g, j0, v, poison, acc);
    }
  } else {
    // rows off the 16-byte grid: the CTA stages each piece into the ring with plain loads
    // (logit by logit, coalesced), then every warp reads its vectors as above
    Op::prologue(A, g, sm);
    for (int si = 0; si < ns; ++si) {
      const int64_t j0 = jb + si * kStageElems;
      const int64_t j1 = j0 + kStageElems < je ? j0 + kStageElems : je;
      __syncthreads();  // the previous piece has been read
#pragma unroll 1
      for (int i = threadIdx.x; i < kStageBytes / 16; i += kThreads) {
        const uint4 w = load_vec<E>(g.row, j0 + (int64_t)i * E::kPerVec, j1, false, Op::kPad);
        *reinterpret_cast<uint4*>(ring + i * 16) = w;
      }
      __syncthreads();
      uint4 v[kStageVec];
#pragma unroll
      for (int it = 0; it < kStageVec; ++it)
        v[it] = lds16(ring + warp_vec_slot<kStageVec>(warp, it, lane) * 16);
      Op::warp_slice(A, g, j0, v, false, acc);
    }
  }
  Op::seg_end(A, g, acc, sm);
  __syncthreads();  // every warp partial of the segment is stored
  Ring ring_state;
  ring_state.buf = ring;
  ring_state.full = full;
  ring_state.released = released;
  ring_state.phase = 0;
  if (A.aligned)
    for (int q = 0; q < kStages; ++q)
      ring_state.phase |= (uint32_t)(((ns - q + kStages - 1) / kStages) & 1) << q;
  ring_state.ctl = ctl;
  ring_state.usable = A.aligned;
  // the counters this finish uses were cleared by the launch before this one on the stream:
  // wait for it (nothing before this point touches them)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  Op::finish(A, g, sm, ring_state);
}

// Launch the segments of a row operation. `ctl` lies in the region the caller just cleared.
template <class Op>
sv_status launch_segments(const typename Op::Args& A, long long units, CallCtl* ctl,
                          cudaStream_t st) {
  if (units <= 0) return SV_OK;
  constexpr int kRingBytes = Op::T::kRingBytes;
  // Host-side function attributes (no stream work): the ring's dynamic shared memory and the
  // carveout that fits the op's CTAs. They are set once per device (bit d of `ready`); if a
  // launch is refused anyway (the context was reset since), they are set again and the
  // launch is retried once.
  static std::atomic<unsigned long long> ready{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  auto set_attributes = [&]() -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(
        segment_kernel<Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(segment_kernel<Op>,
                               cudaFuncAttributePreferredSharedMemoryCarveout,
                               cudaSharedmemCarveoutMaxShared);
    if (r == cudaSuccess && bit) ready.fetch_or(bit);
    return r;
  };
  if (!(ready.load() & bit)) {
    e = set_attributes();
    if (e != cudaSuccess) return cuda_fail(e);
  }
  // programmatic serialization: the CTAs may start while the clear of the call's counters
  // (the launch before this one) runs; they wait for it before the finishing phase
  auto launch = [&]() -> cudaError_t {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)units, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kRingBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = SV_CLEAR_KERNEL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, segment_kernel<Op>, A, ctl);
  };
  e = launch();
  if (e != cudaSuccess && bit) {  // attributes lost with a reset context: set them, retry
    (void)cudaGetLastError();
    ready.fetch_and(~bit);
    if (set_attributes() == cudaSuccess) e = launch();
  }
  return e == cudaSuccess ? SV_OK : cuda_fail(e);
}

}  // namespace sv
