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
#include <cstdint>

#include "specverify.h"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kNgramThreads = 256;
constexpr int kMaxPhrase = 64;

__global__ void __launch_bounds__(kNgramThreads) ngram_kernel(
    const int32_t* __restrict__ history, const int32_t* __restrict__ hist_len, int L_max,
    int n_max, int n_min, int k, int32_t* __restrict__ out_draft,
    int32_t* __restrict__ out_num) {
  __shared__ int32_t suffix[kMaxPhrase];
  __shared__ unsigned int s_best[kNgramThreads / 32];
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int L = __ldg(hist_len + r);
  int32_t* d = out_draft + (int64_t)r * k;
  if (L < 0 || L > L_max) {
    for (int i = tid; i < k; i += kNgramThreads) d[i] = -1;
    if (tid == 0) out_num[r] = -1;
    return;
  }
  const int32_t* h = history + (int64_t)r * L_max;
  const int ns = n_max < L ? n_max : L;
  if (tid < ns) suffix[tid] = __ldg(h + L - 1 - tid);  // suffix[t] = h[L-1-t]
  __syncthreads();

  // key = (l_e << 24) | (2^24 - 1 - e): the larger match first, then the smaller e
  unsigned int best = 0;
  for (int e = n_min - 1 + tid; e <= L - 2; e += kNgramThreads) {
    int m = 0;
    const int cap = n_max < e + 1 ? n_max : e + 1;
    while (m < cap && __ldg(h + e - m) == suffix[m]) ++m;
    if (m >= n_min) {
      const unsigned int key = ((unsigned)m << 24) | (0xffffffu - (unsigned)e);
      best = key > best ? key : best;
    }
  }
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
  for (int i = tid; i < k; i += kNgramThreads) d[i] = i < cnt ? __ldg(h + start + i) : -1;
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
