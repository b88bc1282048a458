// sv_device.cuh — device building blocks shared by the verify, gate and proposer kernels.
//
// A logit row of V entries is cut into chunks of kChunkBytes (32 KiB: 8192 fp32 or 16384
// bf16 logits); see sv_stream.cuh for how chunks reach the kThreads threads of a CTA.
// Block-level synchronisation uses named barrier 1 over kThreads threads (cbar).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kThreads = 256;  // consumer threads
constexpr int kWarps = kThreads / 32;
constexpr int kVecPerThread = 8;
constexpr int kChunkBytes = kThreads * kVecPerThread * 16;  // 32 KiB
constexpr int kNoIndex = 0x7fffffff;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- consumer-group barriers ---------------------------------------------------------------
__device__ __forceinline__ void cbar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
}

// Barrier that also returns whether any consumer thread passed pred != 0.
__device__ __forceinline__ bool cbar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q;\n"
      "  setp.ne.u32 p, %1, 0;\n"
      "  bar.red.or.pred q, 1, %2, p;\n"
      "  selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kThreads)
      : "memory");
  return r != 0;
}

// ---- element types -------------------------------------------------------------------------
struct F32 {
  static constexpr int kPerVec = 4;               // logits per 16-byte vector
  static constexpr int kChunk = kChunkBytes / 4;  // logits per chunk
  static constexpr uint32_t kNegInfBits = 0xff800000u;
  static constexpr uint32_t kNaNBits = 0x7fc00000u;
  __device__ static __forceinline__ float get(const uint4& v, int l) {
    const uint32_t w = l == 0 ? v.x : l == 1 ? v.y : l == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  __device__ static __forceinline__ float load1(const void* row, int64_t j) {
    return __ldg(static_cast<const float*>(row) + j);
  }
  __device__ static __forceinline__ uint32_t bits1(const void* row, int64_t j) {
    return __float_as_uint(load1(row, j));
  }
  __device__ static __forceinline__ uint4 pad_vec(uint32_t pad) {
    return make_uint4(pad, pad, pad, pad);
  }
  // Logits 2p and 2p+1 of a vector.
  __device__ static __forceinline__ float2 get2(const uint4& v, int p) {
    return p == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  // Largest logit of a vector (NaN ignored, as fmaxf does).
  __device__ static __forceinline__ float max_vec(const uint4& v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  // Largest logit of N vectors (NaN ignored), as a balanced tree.
  template <int N>
  __device__ static __forceinline__ float max_lane(const uint4 (&v)[N]) {
    float m[N];
#pragma unroll
    for (int i = 0; i < N; ++i) m[i] = max_vec(v[i]);
#pragma unroll
    for (int q = N / 2; q >= 1; q >>= 1)
#pragma unroll
      for (int i = 0; i < q; ++i) m[i] = fmaxf(m[i], m[i + q]);
    return m[0];
  }
  __device__ static __forceinline__ bool has_nan(const uint4& v) {
    return ((v.x & 0x7fffffffu) > 0x7f800000u) | ((v.y & 0x7fffffffu) > 0x7f800000u) |
           ((v.z & 0x7fffffffu) > 0x7f800000u) | ((v.w & 0x7fffffffu) > 0x7f800000u);
  }
};

struct BF16 {
  static constexpr int kPerVec = 8;
  static constexpr int kChunk = kChunkBytes / 2;
  static constexpr uint32_t kNegInfBits = 0xff80u;
  static constexpr uint32_t kNaNBits = 0x7fc0u;
  // bf16 is the upper half of a binary32: widening is a shift, exact.
  __device__ static __forceinline__ float get(const uint4& v, int l) {
    const uint32_t w = (l >> 1) == 0 ? v.x : (l >> 1) == 1 ? v.y : (l >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((l & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ static __forceinline__ float load1(const void* row, int64_t j) {
    const uint16_t b = __ldg(static_cast<const unsigned short*>(row) + j);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  __device__ static __forceinline__ uint32_t bits1(const void* row, int64_t j) {
    return static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(row) + j));
  }
  __device__ static __forceinline__ uint4 pad_vec(uint32_t pad) {
    const uint32_t w = pad | (pad << 16);
    return make_uint4(w, w, w, w);
  }
  // Logits 2p and 2p+1 of a vector (one packed bf16 pair, widened exactly).
  __device__ static __forceinline__ float2 get2(const uint4& v, int p) {
    const uint32_t w = p == 0 ? v.x : p == 1 ? v.y : p == 2 ? v.z : v.w;
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static __forceinline__ uint32_t max2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
  }
  // Largest logit of a vector, reduced on packed bf16 pairs (max.bf16x2 returns the other
  // operand when one is NaN, as fmaxf does); exact, widened only at the end.
  __device__ static __forceinline__ float max_vec(const uint4& v) {
    const uint32_t m = max2(max2(v.x, v.y), max2(v.z, v.w));
    return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u));
  }
  // Largest logit of N vectors: a balanced tree of packed pair maxima, widened once.
  template <int N>
  __device__ static __forceinline__ float max_lane(const uint4 (&v)[N]) {
    uint32_t m[N];
#pragma unroll
    for (int i = 0; i < N; ++i) m[i] = max2(max2(v[i].x, v[i].y), max2(v[i].z, v[i].w));
#pragma unroll
    for (int q = N / 2; q >= 1; q >>= 1)
#pragma unroll
      for (int i = 0; i < q; ++i) m[i] = max2(m[i], m[i + q]);
    return fmaxf(__uint_as_float(m[0] << 16), __uint_as_float(m[0] & 0xffff0000u));
  }
  __device__ static __forceinline__ bool nan2(uint32_t w) {
    return ((w & 0x7fffu) > 0x7f80u) | (((w >> 16) & 0x7fffu) > 0x7f80u);
  }
  __device__ static __forceinline__ bool has_nan(const uint4& v) {
    return nan2(v.x) | nan2(v.y) | nan2(v.z) | nan2(v.w);
  }
};

// ---- loads ---------------------------------------------------------------------------------
// Streaming 16-byte load: read-only path, no L1 allocation, 256-byte L2 fetch granularity.
// L2 keeps its normal eviction priority so a rejected row pair is still there when the
// request's finishing consumers re-read it.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// One 16-byte vector of logits j .. j+kPerVec-1 of a row (entries at or past j1 read as
// `pad`); fetched whole when the row is 16-byte aligned, else one logit at a time.
template <typename E>
__device__ __forceinline__ uint4 load_vec(const void* row, int64_t j, int64_t j1, bool aligned,
                                          uint32_t pad) {
  if (aligned && j + E::kPerVec <= j1)
    return ld_stream16(static_cast<const char*>(row) + j * (16 / E::kPerVec));
  uint32_t w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (E::kPerVec == 4) {
      w[q] = (j + q < j1) ? E::bits1(row, j + q) : pad;
    } else {
      const uint32_t lo = (j + 2 * q < j1) ? E::bits1(row, j + 2 * q) : pad;
      const uint32_t hi = (j + 2 * q + 1 < j1) ? E::bits1(row, j + 2 * q + 1) : pad;
      w[q] = lo | (hi << 16);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---- arithmetic ----------------------------------------------------------------------------
// 2^x on the SFU (the hardware ex2 instruction, flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^d for an integer-valued d <= 0, built from its exponent bits (exact; 0 for d < -126,
// including d = -inf).
__device__ __forceinline__ float pow2_nonpos(float d) {
  return __uint_as_float((uint32_t)((int)fmaxf(d, -127.0f) + 127) << 23);
}

// Order-preserving map of a non-NaN float onto int32 (for integer max reductions).
__device__ __forceinline__ int f2key(float f) {
  const int i = __float_as_int(f);
  return i ^ ((i >> 31) & 0x7fffffff);
}
__device__ __forceinline__ float key2f(int k) {
  return __int_as_float(k ^ ((k >> 31) & 0x7fffffff));
}

// Error-free sum of two floats (Knuth's TwoSum): a + b = s + e exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// A float-float number: an unevaluated sum hi + lo with |lo| <= ulp(hi)/2, about 48 bits.
// Its arithmetic runs on the FP32 pipes; this GPU's FP64 pipe is far slower, and the draw's
// scans are latency chains of such additions.
struct DF {
  float hi, lo;
};

// a + b, renormalised. Commutative to the bit (TwoSum's error term is exact), so a butterfly
// of these leaves the same sum in every lane.
__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float h = __fadd_rn(s, e);
  return {h, __fsub_rn(e, __fsub_rn(h, s))};
}

__device__ __forceinline__ bool df_gt(DF a, DF b) {
  return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo);
}

__device__ __forceinline__ DF df_from_double(double d) {
  const float h = __double2float_rn(d);
  return {h, __double2float_rn(d - (double)h)};
}

__device__ __forceinline__ DF df_shfl_xor(DF a, int o) {
  return {__shfl_xor_sync(0xffffffffu, a.hi, o), __shfl_xor_sync(0xffffffffu, a.lo, o)};
}

__device__ __forceinline__ DF df_shfl_up(DF a, int o) {
  return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}

// Inclusive warp scan of float-float values (Hillis-Steele).
__device__ __forceinline__ DF df_warp_scan(DF x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const DF y = df_shfl_up(x, o);
    if (lane >= o) x = df_add(y, x);
  }
  return x;
}

// Warp sum of floats carried as an unevaluated (hi, lo) pair: every level adds exactly.
__device__ __forceinline__ void warp_sum_compensated(float& hi, float& lo) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
    float s, e;
    two_sum(hi, h2, s, e);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, l2), e);
  }
}

__device__ __forceinline__ double warp_sum_d(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Inclusive warp scan (Hillis-Steele) in double.
__device__ __forceinline__ double warp_scan_d(double x) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

__device__ __forceinline__ float warp_max_f(float x) {  // x must not be NaN
  return key2f(__reduce_max_sync(0xffffffffu, f2key(x)));
}

// Consumer-group maximum of a non-NaN float; every consumer gets it. `red`: kWarps floats.
__device__ __forceinline__ float block_max_f(float x, float* red) {
  x = warp_max_f(x);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = x;
  cbar();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) m = fmaxf(m, red[i]);
  cbar();
  return m;
}

// Consumer-group sum of per-thread floats: compensated (exact) within each warp, the kWarps
// warp results merged in double by thread 0 only (GB300's FP64 rate is a small fraction of
// its FP32 rate, so no other thread touches double here). Valid in thread 0. `red` holds
// 2*kWarps floats and must not be rewritten before the next consumer barrier.
__device__ __forceinline__ double block_sum_fd_t0(float x, float* red) {
  float hi = x, lo = 0.0f;
  warp_sum_compensated(hi, lo);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    red[2 * w] = hi;
    red[2 * w + 1] = lo;
  }
  cbar();
  double s = 0.0;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 0; i < kWarps; ++i) s += (double)red[2 * i] + (double)red[2 * i + 1];
  }
  return s;
}

// ---- completion counters -------------------------------------------------------------------
// Count this CTA in on a completion counter; true for the CTA that arrives last. Called by
// one thread after a CTA barrier that follows the stores the CTA publishes: the add is a
// release at GPU scope (cumulative over what the barrier ordered before it) and an acquire
// for the arriving thread. The counters are cleared before every launch, by the call's clear
// kernel on the same stream (the segment kernel waits for it before its finishing phase).
__device__ __forceinline__ bool arrive_last(unsigned int* counter, unsigned int expected) {
  unsigned int prev;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
               : "=r"(prev)
               : "l"(counter)
               : "memory");
  return prev == expected - 1;
}

// Shared-memory atomic add with acquire-release ordering at CTA scope: the caller's earlier
// accesses (and, after __syncwarp, its warp's) are ordered before the add, and the thread
// that sees the final count is ordered after every earlier add.
__device__ __forceinline__ int atomic_add_acq_rel_cta(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_u32(p)), "r"(v)
               : "memory");
  return old;
}

// ---- mbarrier and bulk-copy (TMA) primitives ----------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Wait for the given phase parity of an mbarrier for at most limit_ns; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}
// Bulk copy (TMA, non-tensor) of `bytes` (a multiple of 16) from 16-byte aligned global
// memory into this CTA's shared memory, completing on `bar`, with the copy's default L2
// eviction priority, or with the priority of an L2 cache policy made by l2_policy().
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                        uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// An L2 cache policy for every line a copy touches: evicted last (keep) or first.
__device__ __forceinline__ uint64_t l2_policy(bool keep) {
  uint64_t p;
  if (keep)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint4 lds16(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

}  // namespace sv
