// Causal multi-query attention, SIMT form: one warp per (query row, head),
// online softmax over the cached keys 0..pos.  Every query head reads the
// single shared K/V head (yelogs.com nanochat story, "technical details and
// official Q&A": multi-query attention; apidog.com/th "train your own
// ChatGPT", "how nanochat works" item 5: causal attention, SDPA scale
// 1/sqrt(head_dim)).  Used for the fp32 model and as the simple path.
#pragma once

#include "nc_common.cuh"

namespace nc {

// Q [M, n_head*hd] with rows m = b*T + t at position pos0 + t; caches
// [B_max][cache_S][hd]; O [M, n_head*hd].
template <typename TA, typename TC>
__global__ void attn_simt_kernel(const TA* __restrict__ Q, const TC* __restrict__ Kc,
                                 const TC* __restrict__ Vc, TA* __restrict__ O, int M, int n_head,
                                 int hd, int T, int pos0, int cache_S) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= M * n_head) return;
  const int m = warp / n_head, h = warp % n_head;
  const int b = m / T, pos = pos0 + (m % T);
  const int per = hd / 32;
  const float scale = rsqrtf((float)hd);
  float q[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
  const TA* qr = Q + (size_t)m * n_head * hd + h * hd;
  for (int i = 0; i < per; ++i) q[i] = to_f(qr[lane + 32 * i]) * scale;
  float run_max = -INFINITY, run_sum = 0.f;
  const TC* kb = Kc + (size_t)b * cache_S * hd;
  const TC* vb = Vc + (size_t)b * cache_S * hd;
  for (int s = 0; s <= pos; ++s) {
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
