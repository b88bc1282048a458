// sv_ngram.cu — prompt-lookup n-gram draft proposer.
//
// "The Inference Wall, Part 7", section "What S is in this experiment, and what 'ngram'
// actually means": take the last few tokens of the text the request holds, find the same
// phrase earlier in that text, trying prompt_lookup_max tokens first and shortening to
// prompt_lookup_min, and copy the (up to) k tokens that followed it; with nothing earlier
// there is no proposal.
//
// The kernel evaluates every candidate end position at once instead of trying one phrase
// length after another: for each e <= L-2 it counts l_e, how many tokens ending at e match
// the tokens ending at L-1 (capped at n_max). The longest phrase with an earlier
// occurrence has length max_e l_e, and its earliest occurrence is the smallest e reaching
// that maximum, which is the result of the page's longest-first search. One CTA per
// request; a single packed (l_e, -e) maximum picks the winner.
//
// The history streams through shared memory in tiles of kTile end positions, each with the
// n_max - 1 tokens before it: every thread issues its asynchronous copies of a tile at once
// (cp.async, no register round trip), so a tile costs one memory latency, and the match
// counts then read shared memory only. The first tile always starts at token 0, so its
// copies (16 bytes each where the row allows) are issued before the history length is
// known, and the two loads overlap; the suffix is read from that tile when it holds it.
#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kNgramThreads = 256;
constexpr int kMaxPhrase = 64;
constexpr int kTile = 8192;  // end positions per shared-memory tile (32 KiB of tokens)

__device__ __forceinline__ void cp_async4(int32_t* dst, const int32_t* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async16(int32_t* dst, const int32_t* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(
    const int32_t* __restrict__ history, const int32_t* __restrict__ hist_len, int L_max,
    int n_max, int n_min, int k, int32_t* __restrict__ out_draft,
    int32_t* __restrict__ out_num) {
  __shared__ int32_t suffix[kMaxPhrase];
  __shared__ __align__(16) int32_t tile[kTile + kMaxPhrase];
  __shared__ unsigned int s_best[kNgramThreads / 32];
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int32_t* h = history + (int64_t)r * L_max;
  // the first tile, tokens [0, n0), requested before the length arrives
  const int n0 = L_max < kTile + kMaxPhrase ? L_max : kTile + kMaxPhrase;
  if ((reinterpret_cast<uintptr_t>(h) & 15) == 0) {
    const int n16 = n0 / 4;
    for (int i = tid; i < n16; i += kNgramThreads) cp_async16(tile + 4 * i, h + 4 * i);
    for (int i = 4 * n16 + tid; i < n0; i += kNgramThreads) cp_async4(tile + i, h + i);
  } else {
    for (int i = tid; i < n0; i += kNgramThreads) cp_async4(tile + i, h + i);
  }
  const int L = __ldg(hist_len + r);
  int32_t* d = out_draft + (int64_t)r * k;
  if (L < 0 || L > L_max) {
    cp_async_wait_all();  // no copy outlives the CTA
    for (int i = tid; i < k; i += kNgramThreads) d[i] = -1;
    if (tid == 0) out_num[r] = -1;
    return;
  }
  const int ns = n_max < L ? n_max : L;
  // suffix[t] = h[L-1-t]: from the first tile when it holds the last token
  const bool suffix_in_tile = L <= n0;
  if (!suffix_in_tile && tid < ns) cp_async4(suffix + tid, h + L - 1 - tid);
  cp_async_wait_all();
  __syncthreads();
  if (suffix_in_tile && tid < ns) suffix[tid] = tile[L - 1 - tid];

  // key = (l_e << 24) | (2^24 - 1 - e): the larger match first, then the smaller e
  unsigned int best = 0;
  int lo = 0, t1 = 0;  // the tile in shared memory holds tokens [lo, t1)
  for (int t0 = n_min - 1; t0 <= L - 2; t0 += kTile) {
    // end positions [t0, t1) read tokens [lo, t1): lo <= e - (n_max - 1) for every e >= t0
    t1 = t0 + kTile < L - 1 ? t0 + kTile : L - 1;
    lo = t0 - (n_max - 1) > 0 ? t0 - (n_max - 1) : 0;
    __syncthreads();  // the previous tile has been read; the suffix is in place
    if (lo > 0) {  // later tiles (the first one, from token 0, is in place)
      for (int i = tid; i < t1 - lo; i += kNgramThreads) cp_async4(tile + i, h + lo + i);
      cp_async_wait_all();
      __syncthreads();
    }
    for (int e = t0 + tid; e < t1; e += kNgramThreads) {
      int m = 0;
      const int cap = n_max < e + 1 ? n_max : e + 1;
      while (m < cap && tile[e - m - lo] == suffix[m]) ++m;
      if (m >= n_min) {
        const unsigned int key = ((unsigned)m << 24) | (0xffffffu - (unsigned)e);
        best = key > best ? key : best;
      }
    }
  }
  cp_async_wait_all();  // the suffix's copies, when no tile was loaded
  best = __reduce_max_sync(0xffffffffu, best);
  if (lane == 0) s_best[w] = best;
  __syncthreads();
  unsigned int b = s_best[0];
#pragma unroll
  for (int q = 1; q < kNgramThreads / 32; ++q) b = s_best[q] > b ? s_best[q] : b;
  int cnt = 0, start = 0;
  if (b != 0) {
    const int e = (int)(0xffffffu - (b & 0xffffffu));
    start = e + 1;
    cnt = L - start < k ? L - start : k;
  }
  // the proposal, from the last tile or the suffix where they hold it
  for (int i = tid; i < k; i += kNgramThreads) {
    int32_t v = -1;
    if (i < cnt) {
      const int j = start + i;
      v = (j >= lo && j < t1) ? tile[j - lo] : (j >= L - ns ? suffix[L - 1 - j] : __ldg(h + j));
    }
    d[i] = v;
  }
  if (tid == 0) out_num[r] = cnt;
}

}  // namespace sv

using namespace sv;

extern "C" sv_status ngram_propose(const int32_t* history, const int32_t* hist_len, int B,
                                   int L_max, int n_max, int n_min, int k, int32_t* out_draft,
                                   int32_t* out_num_draft, sv_stream_t stream) {
  if (B < 0 || L_max < 1 || L_max >= (1 << 24)) return SV_ERR_INVALID_ARG;
  if (n_min < 1 || n_max < n_min || n_max > kMaxPhrase || k < 1 || k > 64)
    return SV_ERR_INVALID_ARG;
  if (B == 0) return SV_OK;
  if (!history || !hist_len || !out_draft || !out_num_draft) return SV_ERR_INVALID_ARG;
  if (!aligned_to(history, 4) || !aligned_to(hist_len, 4) || !aligned_to(out_draft, 4) ||
      !aligned_to(out_num_draft, 4))
    return SV_ERR_INVALID_ARG;
  ngram_kernel<<<(unsigned)B, kNgramThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      history, hist_len, L_max, n_max, n_min, k, out_draft, out_num_draft);
  return launch_status();
}
