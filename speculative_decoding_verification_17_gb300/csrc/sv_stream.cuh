// sv_stream.cuh — the two drivers that feed (row, chunk) units to a row operation.
//
// stream_kernel (rows 16-byte aligned): a persistent kernel, two CTAs per SM. Each CTA has
// one producer warp and kWarps consumer warps. The producer claims the next unit from a
// global counter (units are claimed in index order, so a request's units run close together
// in time), skips units the operation does not need, and copies the unit's 32 KiB chunk
// with one cp.async.bulk (TMA) into a kStages-deep shared-memory ring, completing on the
// stage's "full" mbarrier. The consumers wait on that barrier, move their vectors into
// registers, release the stage on its "empty" mbarrier and run the operation. So up to
// kStages chunks per CTA are in flight while the consumers compute or finish a row or a
// request, and a CTA that is busy finishing simply claims fewer units. Every wait is
// bounded by kWaitLimitNs; a wait that runs out sets a bit in the call's control word and
// the CTA stops.
//
// direct_kernel (any alignment): one CTA of kThreads threads per unit, loading straight into
// registers (logit by logit when a row is not 16-byte aligned).
//
// An operation Op provides:
//   using E;                        element type (F32 / BF16)
//   static constexpr uint32_t kPad; bit pattern read for logits past the end of a row
//   struct Smem;                    its shared-memory state
//   struct Args;                    kernel arguments (with a bool `aligned`)
//   static bool unit_row(const Args&, int64_t u, const void*& row, int64_t& j0, int64_t& j1);
//       false when unit u is not needed; else the row and the chunk [j0, j1)
//   static void process(const Args&, int64_t u, const void* row, int64_t j0, int64_t j1,
//                       const uint4 (&v)[kVecPerThread], Smem&);
//       run by the kThreads consumers with the chunk in registers
#pragma once

#include <atomic>
#include <cuda_runtime.h>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kStages = 3;
constexpr int kStreamThreads = kThreads + 32;          // consumers + one producer warp
constexpr int kRingBytes = kStages * kChunkBytes;      // 96 KiB of dynamic shared memory
constexpr uint64_t kWaitLimitNs = 2000000000ull;       // 2 s: far past any legitimate wait

template <class Op>
__global__ void __launch_bounds__(kStreamThreads, 2)
    stream_kernel(const typename Op::Args A, long long units, StreamCtl* ctl) {
  using E = typename Op::E;
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kStages];
  __shared__ __align__(8) uint64_t empty[kStages];
  __shared__ long long unit_of[kStages];
  __shared__ typename Op::Smem sm;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kWarps) {  // ---- producer ----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (;;) {
        long long u;
        const void* src = nullptr;
        uint32_t bytes = 0;
        for (;;) {
          u = (long long)atomicAdd(&ctl->next_unit, 1ull);
          if (u >= units) {
            u = -1;
            break;
          }
          const void* row;
          int64_t j0, j1;
          if (Op::unit_row(A, u, row, j0, j1)) {
            src = static_cast<const char*>(row) + j0 * (16 / E::kPerVec);
            bytes = (uint32_t)((j1 - j0) * (16 / E::kPerVec));
            break;
          }
        }
        if (!mbar_wait(&empty[stage], phase ^ 1u, kWaitLimitNs)) {
          atomicOr(&ctl->error, 1u);
          break;
        }
        unit_of[stage] = u;
        if (u < 0) {
          mbar_arrive(&full[stage]);  // no more work: consumers stop at this stage
          break;
        }
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_g2s(ring + stage * kChunkBytes, src, bytes, &full[stage]);
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    return;
  }

  // ---- consumers ----
  int stage = 0;
  uint32_t phase = 0;
  for (;;) {
    if (!mbar_wait(&full[stage], phase, kWaitLimitNs)) {
      if (lane == 0) atomicOr(&ctl->error, 2u);
      break;
    }
    const long long u = unit_of[stage];
    if (u < 0) break;
    const void* row;
    int64_t j0, j1;
    Op::unit_row(A, u, row, j0, j1);
    const unsigned char* buf = ring + stage * kChunkBytes;
    uint4 v[kVecPerThread];
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const int slot = it * kThreads + threadIdx.x;
      v[it] = (j0 + (int64_t)slot * E::kPerVec < j1) ? lds16(buf + slot * 16)
                                                      : E::pad_vec(Op::kPad);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    Op::process(A, u, row, j0, j1, v, sm);
    if (++stage == kStages) {
      stage = 0;
      phase ^= 1u;
    }
  }
}

template <class Op>
__global__ void __launch_bounds__(kThreads, 2) direct_kernel(const typename Op::Args A) {
  using E = typename Op::E;
  __shared__ typename Op::Smem sm;
  const long long u = blockIdx.x;
  const void* row;
  int64_t j0, j1;
  if (!Op::unit_row(A, u, row, j0, j1)) return;
  uint4 v[kVecPerThread];
  load_chunk<E>(row, j0, j1, A.aligned, Op::kPad, v);
  Op::process(A, u, row, j0, j1, v, sm);
}

// Launch the units of a row operation: the persistent TMA kernel for aligned rows, the
// direct kernel otherwise. `ctl` lies in the counter region the caller has just cleared.
template <class Op>
sv_status launch_units(const typename Op::Args& A, long long units, StreamCtl* ctl,
                       cudaStream_t st) {
  if (units <= 0) return SV_OK;
  if (!A.aligned) {
    direct_kernel<Op><<<(unsigned)units, kThreads, 0, st>>>(A);
    return launch_status();
  }
  static std::atomic<int> cached_grid[64];  // per device: CTAs resident at once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  // a host-side function attribute (no stream work); set on every call so it also holds
  // in a context created after the first call
  e = cudaFuncSetAttribute(stream_kernel<Op>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kRingBytes);
  if (e != cudaSuccess) return cuda_fail(e);
  int grid = (dev >= 0 && dev < 64) ? cached_grid[dev].load(std::memory_order_relaxed) : 0;
  if (grid == 0) {
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel<Op>,
                                                      kStreamThreads, kRingBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    grid = sms * (per_sm > 0 ? per_sm : 1);
    if (dev >= 0 && dev < 64) cached_grid[dev].store(grid, std::memory_order_relaxed);
  }
  const long long g = units < grid ? units : grid;
  stream_kernel<Op><<<(unsigned)g, kStreamThreads, kRingBytes, st>>>(A, units, ctl);
  return launch_status();
}

}  // namespace sv
