// Causal multi-query / grouped-query attention, SIMT form: one warp per
// (query row, head), online softmax over the cached keys 0..pos (only those
// after pos - window with a sliding window).  Query head h reads K/V head
// h / (n_head / n_kv) (yelogs.com nanochat story, "technical details and
// official Q&A": multi-query attention; apidog.com/th "train your own
// ChatGPT", "how nanochat works" item 1: grouped-query attention and sliding
// windows; item 5: causal attention, SDPA scale 1/sqrt(head_dim)).  Used for
// the fp32 model.
#pragma once

#include "nc_common.cuh"

namespace nc {

// Q [M, n_head*hd] with rows m = b*T + t at position pos0[b] + t (each row
// of the batch continues its own cache); caches [B_max][n_kv][cache_S][hd];
// O [M, n_head*hd]; window 0 = unrestricted.
template <typename TA, typename TC>
__global__ void attn_simt_kernel(const TA* __restrict__ Q, const TC* __restrict__ Kc,
                                 const TC* __restrict__ Vc, TA* __restrict__ O, int M, int n_head,
                                 int n_kv, int hd, int T, const int* __restrict__ pos0, int cache_S,
                                 int window) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M * n_head) return;
  const int m = warp / n_head, h = warp % n_head;
  const int b = m / T, pos = pos0[b] + (m % T);
  const int per = hd / 32;
  const float scale = rsqrtf((float)hd);
  float q[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
  const TA* qr = Q + (size_t)m * n_head * hd + h * hd;
  for (int i = 0; i < per; ++i) q[i] = to_f(qr[lane + 32 * i]) * scale;
  float run_max = -INFINITY, run_sum = 0.f;
  const int g = h / (n_head / n_kv);
  const TC* kb = Kc + ((size_t)b * n_kv + g) * cache_S * hd;
  const TC* vb = Vc + ((size_t)b * n_kv + g) * cache_S * hd;
  const int s0 = window > 0 ? max(0, pos - window + 1) : 0;
  for (int s = s0; s <= pos; ++s) {
    float dot = 0.f;
    for (int i = 0; i < per; ++i) dot = fmaf(q[i], to_f(kb[(size_t)s * hd + lane + 32 * i]), dot);
    dot = warp_sum(dot);
    const float new_max = fmaxf(run_max, dot);
    const float corr = __expf(run_max - new_max);
    const float p = __expf(dot - new_max);
    run_sum = run_sum * corr + p;
    for (int i = 0; i < per; ++i)
      acc[i] = acc[i] * corr + p * to_f(vb[(size_t)s * hd + lane + 32 * i]);
    run_max = new_max;
  }
  TA* orow = O + (size_t)m * n_head * hd + h * hd;
  const float inv = 1.f / run_sum;
  for (int i = 0; i < per; ++i) orow[lane + 32 * i] = from_f<TA>(acc[i] * inv);
}

}  // namespace nc
