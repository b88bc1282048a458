// sv_stream.cuh — the driver that feeds (row, chunk) units to a row operation.
//
// unit_kernel: one CTA of kThreads threads per unit, up to kCtasPerSm CTAs resident per SM.
// For a row that starts on a 16-byte boundary, thread 0 fetches the unit's chunk (32 KiB)
// with a single cp.async.bulk (TMA) into shared memory, completing on an mbarrier; a row
// that does not is staged logit by logit by all threads. The operation then reads the
// chunk from shared memory. Many small CTAs per SM keep several chunks in flight per SM
// and hide each other's fixed costs (the barrier waits, the fence and atomic that publish a
// partial), and the register budget of kCtasPerSm CTAs is what every code path of an
// operation is written for. The wait on the bulk copy is bounded; a copy that never lands
// poisons its row (the request gets the error sentinel) and sets a bit in the call's
// control word.
//
// An operation Op provides:
//   using E;                        element type (F32 / BF16)
//   static constexpr uint32_t kPad; bit pattern read for logits past the end of a row
//   struct Smem;                    its shared-memory state
//   struct Args;                    kernel arguments (with a bool `aligned`)
//   static bool unit_row(const Args&, int64_t u, const void*& row, int64_t& j0, int64_t& j1);
//       false when unit u is not needed; else the row and the chunk [j0, j1)
//   static void process(const Args&, int64_t u, const void* row, int64_t j0, int64_t j1,
//                       const unsigned char* chunk, bool poisoned, Smem&);
//       run by all kThreads threads; 16-byte vector s of the chunk is at chunk + 16*s
#pragma once

#include <cuda_runtime.h>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

// CTAs resident per SM: shared memory allows 6 (32 KiB chunk each); 5 leaves the sampled
// verify's request-finishing code 48 registers per thread without spilling. A build may set
// SV_CTAS_PER_SM to try another value.
#ifndef SV_CTAS_PER_SM
#define SV_CTAS_PER_SM 5
#endif
constexpr int kCtasPerSm = SV_CTAS_PER_SM;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far past any legitimate wait

// Vector `it` of this thread from a chunk staged in shared memory (pad past the end).
template <typename E>
__device__ __forceinline__ uint4 chunk_vec(const unsigned char* chunk, int it, int64_t j0,
                                           int64_t j1, uint32_t pad) {
  const int slot = it * kThreads + threadIdx.x;
  return (j0 + (int64_t)slot * E::kPerVec < j1) ? lds16(chunk + slot * 16) : E::pad_vec(pad);
}

template <class Op>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
    unit_kernel(const typename Op::Args A, CallCtl* ctl) {
  using E = typename Op::E;
  extern __shared__ __align__(128) unsigned char chunk[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ typename Op::Smem sm;

  const long long u = blockIdx.x;
  const void* row;
  int64_t j0, j1;
  if (!Op::unit_row(A, u, row, j0, j1)) return;
  bool poisoned = false;
  if (A.aligned) {
    if (threadIdx.x == 0) {
      mbar_init(&bar, 1);
      fence_barrier_init();
      const uint32_t bytes = (uint32_t)((j1 - j0) * (16 / E::kPerVec));
      mbar_arrive_expect_tx(&bar, bytes);
      bulk_g2s(chunk, static_cast<const char*>(row) + j0 * (16 / E::kPerVec), bytes, &bar);
    }
    __syncthreads();
    if (!mbar_wait(&bar, 0, kWaitLimitNs)) {
      poisoned = true;
      if (threadIdx.x == 0) atomicOr(&ctl->error, 1u);
    }
    poisoned = __syncthreads_or(poisoned);
  } else {
#pragma unroll
    for (int it = 0; it < kVecPerThread; ++it) {
      const int slot = it * kThreads + threadIdx.x;
      const int64_t j = j0 + (int64_t)slot * E::kPerVec;
      if (j < j1) {
        const uint4 v = load_vec<E>(row, j, j1, false, Op::kPad);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(chunk + slot * 16)),
                     "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
    }
    __syncthreads();
  }
  Op::process(A, u, row, j0, j1, chunk, poisoned, sm);
}

// Launch the units of a row operation. `ctl` lies in the region the caller has just cleared.
template <class Op>
sv_status launch_units(const typename Op::Args& A, long long units, CallCtl* ctl,
                       cudaStream_t st) {
  if (units <= 0) return SV_OK;
  // ask for the largest shared-memory carveout so kCtasPerSm CTAs fit on an SM (a host-side
  // function attribute, no stream work; set on every call so it holds in any context)
  cudaError_t e = cudaFuncSetAttribute(unit_kernel<Op>,
                                       cudaFuncAttributePreferredSharedMemoryCarveout,
                                       cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return cuda_fail(e);
  unit_kernel<Op><<<(unsigned)units, kThreads, kChunkBytes, st>>>(A, ctl);
  return launch_status();
}

}  // namespace sv
