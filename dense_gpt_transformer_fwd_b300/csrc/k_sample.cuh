// Next-token sampling from fp32 logits on the device, and the KV-cache row
// clone of batch generation: the engine steps on either side of the forward
// pass (apidog.com/th "train your own ChatGPT", "how nanochat works" item 6:
// KV cache, prefill and decode, batch generation that clones the cache for
// parallel sampling; szyisi.cn "$100 ... ChatGPT clone", inference engine
// paragraph).
//
// Sampling rule (the pages name sampling but give no rule; the plainest
// reading):
//   temperature 0: the argmax, the lowest index among equal maxima;
//   otherwise: candidates ordered by (logit descending, index ascending), the
//   first top_k kept (top_k 0 keeps all), weights w_i = exp((l_i - l_0) / T)
//   in fp64, cumulative sums C_j = w_0 + ... + w_j in that order, and the
//   first candidate with C_j > u * C_last is taken, u in [0, 1) a given draw.
//
// One CTA of 1024 threads per row.  The kept candidates (at most
// SAMPLE_MAX_KEEP) are found by a radix select on order-preserving 32-bit
// keys of the logits (four 8-bit passes with shared-memory histograms), ties
// at the threshold taken in index order by a block scan, sorted by a bitonic
// sort of 64-bit (value, index) keys, weighted in parallel, and summed in
// candidate order by one thread, so the cumulative sums are the sequential
// ones of the rule.
#pragma once

#include "nc_common.cuh"

namespace nc {

constexpr int SAMPLE_THREADS = 1024;
constexpr int SAMPLE_MAX_KEEP = 1024;

// order-preserving key of a float (larger float -> larger key); -0 maps to +0
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// exclusive scan of one int per thread over the block (thread order);
// returns the thread's offset and writes the block total to *total
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[32 + lane] = w;                       // inclusive warp prefix
  }
  __syncthreads();
  const int before = warp > 0 ? s_warp[32 + warp - 1] : 0;
  *total = s_warp[32 + (blockDim.x >> 5) - 1];
  __syncthreads();
  return before + x - v;
}

// logits [B][ld] fp32 (row b at logits + b * ld, V valid columns), u [B] draws
__global__ void __launch_bounds__(SAMPLE_THREADS) sample_kernel(const float* __restrict__ logits, int ld, int V,
                                                                 double temperature, int top_k,
                                                                 const double* __restrict__ u,
                                                                 int32_t* __restrict__ out) {
  __shared__ unsigned int hist[256];
  __shared__ int s_scan[64];
  __shared__ unsigned long long cand[SAMPLE_MAX_KEEP];
  __shared__ double wsum[SAMPLE_MAX_KEEP];
  __shared__ int s_misc[4];
  const int b = blockIdx.x, tid = threadIdx.x;
  const float* row = logits + (size_t)b * ld;
  // each thread owns the contiguous index range [lo, hi) (index order = thread order)
  const int per = (V + SAMPLE_THREADS - 1) / SAMPLE_THREADS;
  const int lo = min(V, tid * per), hi = min(V, lo + per);

  if (temperature <= 0.0) {
    // greedy: max of (key, ~index) = the largest logit, lowest index on ties
    unsigned long long best = 0;
    for (int i = lo; i < hi; ++i) {
      const unsigned long long k = ((unsigned long long)float_key(row[i]) << 32) | (0xFFFFFFFFu - (unsigned)i);
      best = k > best ? k : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
      best = y > best ? y : best;
    }
    if ((tid & 31) == 0) cand[tid >> 5] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long m = 0;
      for (int w = 0; w < SAMPLE_THREADS / 32; ++w) m = cand[w] > m ? cand[w] : m;
      out[b] = (int32_t)(0xFFFFFFFFu - (unsigned)(m & 0xFFFFFFFFu));
    }
    return;
  }

  const int K = (top_k <= 0 || top_k > V) ? V : top_k;   // candidates kept (<= SAMPLE_MAX_KEEP)
  // ---- radix select: the K-th largest key (prefix), and how many ties at it are kept
  uint32_t prefix = 0, pmask = 0;
  int need = K;                                          // ranks still to place at or below `prefix`
  if (K < V) {
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int i = tid; i < 256; i += SAMPLE_THREADS) hist[i] = 0;
      __syncthreads();
      for (int i = lo; i < hi; ++i) {
        const uint32_t k = float_key(row[i]);
        if ((k & pmask) == prefix) atomicAdd(&hist[(k >> shift) & 0xFF], 1u);
      }
      __syncthreads();
      if (tid == 0) {
        int acc = 0, bin = 0;
        for (bin = 255; bin > 0; --bin) {
          if (acc + (int)hist[bin] >= need) break;
          acc += (int)hist[bin];
        }
        s_misc[0] = bin;
        s_misc[1] = need - acc;
      }
      __syncthreads();
      prefix |= (uint32_t)s_misc[0] << shift;
      pmask |= 0xFFu << shift;
      need = s_misc[1];
      __syncthreads();
    }
  }
  // ---- compaction: every key above the threshold, then `need` ties in index order
  int n_gt = 0, n_eq = 0;
  for (int i = lo; i < hi; ++i) {
    const uint32_t k = float_key(row[i]);
    if (K == V || k > prefix) ++n_gt;
    else if (k == prefix) ++n_eq;
  }
  int tot_gt = 0, tot_eq = 0;
  const int off_gt = block_exclusive_scan(n_gt, s_scan, &tot_gt);
  const int off_eq = block_exclusive_scan(n_eq, s_scan, &tot_eq);
  {
    int g = off_gt, e = off_eq;
    for (int i = lo; i < hi; ++i) {
      const uint32_t k = float_key(row[i]);
      const unsigned long long key = ((unsigned long long)k << 32) | (0xFFFFFFFFu - (unsigned)i);
      if (K == V || k > prefix) {
        cand[g++] = key;
      } else if (k == prefix) {
        if (e < need) cand[tot_gt + e] = key;
        ++e;
      }
    }
  }
  // pad to the sort width with the smallest key
  int width = 1;
  while (width < K) width <<= 1;
  for (int i = K + tid; i < width; i += SAMPLE_THREADS) cand[i] = 0ull;
  __syncthreads();
  // ---- bitonic sort, descending
  for (int size = 2; size <= width; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < width; i += SAMPLE_THREADS) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long a = cand[i], c = cand[j];
          if (desc ? (a < c) : (a > c)) {
            cand[i] = c;
            cand[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  // ---- weights in fp64, then the sequential cumulative sums
  const double l0 = (double)key_float((uint32_t)(cand[0] >> 32));
  for (int i = tid; i < K; i += SAMPLE_THREADS)
    wsum[i] = exp(((double)key_float((uint32_t)(cand[i] >> 32)) - l0) / temperature);
  __syncthreads();
  if (tid == 0) {
    double c = 0.0;
    for (int i = 0; i < K; ++i) {
      c += wsum[i];
      wsum[i] = c;
    }
  }
  __syncthreads();
  const double target = u[b] * wsum[K - 1];
  // the first candidate whose cumulative weight exceeds the target
  if (tid == 0) s_misc[2] = K - 1;
  __syncthreads();
  for (int i = tid; i < K; i += SAMPLE_THREADS)
    if (wsum[i] > target && (i == 0 || !(wsum[i - 1] > target))) atomicMin(&s_misc[2], i);
  __syncthreads();
  if (tid == 0) out[b] = (int32_t)(0xFFFFFFFFu - (unsigned)(cand[s_misc[2]] & 0xFFFFFFFFu));
}

// Batch generation: rows [0, n) of every layer's K and V cache become copies
// of row `src` (each of its n_kv K/V heads: the first copy_bytes bytes of a
// head's sequence of seq_bytes), and every row's device length becomes len
// (and, when given, its last token prev_tok[b] becomes src's).
// grid = (n, n_layer, 2 * n_kv: K or V, then the head).
__global__ void kv_clone_kernel(char* __restrict__ k_base, char* __restrict__ v_base, size_t layer_bytes,
                                size_t seq_bytes, int n_kv, int src, size_t copy_bytes, int* __restrict__ d_len,
                                int len, int32_t* __restrict__ prev_tok) {
  const int b = blockIdx.x, l = blockIdx.y;
  const int is_v = (int)blockIdx.z / n_kv, g = (int)blockIdx.z % n_kv;
  if (l == 0 && blockIdx.z == 0 && threadIdx.x == 0) {
    d_len[b] = len;
    if (prev_tok && b != src) prev_tok[b] = prev_tok[src];   // the smear's previous token
  }
  if (b == src) return;
  char* base = (is_v ? v_base : k_base) + (size_t)l * layer_bytes;
  const uint4* from = reinterpret_cast<const uint4*>(base + ((size_t)src * n_kv + g) * seq_bytes);
  uint4* to = reinterpret_cast<uint4*>(base + ((size_t)b * n_kv + g) * seq_bytes);
  const size_t n16 = copy_bytes / 16;
  for (size_t i = threadIdx.x; i < n16; i += blockDim.x) to[i] = from[i];
}

}  // namespace nc
