// Row-wise kernels of the forward pass: token embedding + RMSNorm, the
// parameter-free RMSNorm before each projection, the RoPE/QK-norm/KV-cache
// write that follows an unfused QKV projection, and an fp32 SIMT GEMM used by
// the fp32 model.
//
// Sources: yelogs.com nanochat story, "technical details and official Q&A"
// (RMSNorm without learnable parameters after the token embedding and before
// the MLP, QK norm, RoPE without absolute positions, untied embedding);
// geoz.com.cn NanoChat article, "development tricks" (precomputed rotary
// embeddings, KV cache).
#pragma once

#include "nc_common.cuh"

namespace nc {

// One warp per row: x[m] = rms(E[tok[m]]) in fp32, h[m] = TA(rms(x[m])).
// With ss_out (decode, norm folded into the next projection) h[m] = TA(x[m])
// instead, and ss_out[t * ss_ld + m] = sum of x[m][j]^2 over the 128-column
// block t (d a multiple of 128).
// An out-of-range token raises NC_DEVFLAG_TOKEN and reads row 0 instead.
template <typename TW, typename TA>
__global__ void embed_rmsnorm_kernel(const int32_t* __restrict__ tok, const TW* __restrict__ E,
                                     float* __restrict__ x, TA* __restrict__ h, int M, int d,
                                     int vocab, float eps, int* err, float* __restrict__ ss_out, int ss_ld) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (warp >= M) return;
  int t = tok[warp];
  if (t < 0 || t >= vocab) {
    if (lane == 0) atomicOr(err, NC_DEVFLAG_TOKEN);
    t = 0;
  }
  const TW* e = E + (size_t)t * d;
  float ss = 0.f;
  for (int j = lane; j < d; j += 32) {
    const float v = to_f(e[j]);
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  const float r0 = rsqrtf(ss / d + eps);
  if (ss_out) {
    for (int t = 0; t < d / 128; ++t) {
      float st = 0.f;
      for (int j = 128 * t + lane; j < 128 * (t + 1); j += 32) {
        const float v = to_f(e[j]) * r0;
        x[(size_t)warp * d + j] = v;
        h[(size_t)warp * d + j] = from_f<TA>(v);
        st = fmaf(v, v, st);
      }
      st = warp_sum(st);
      if (lane == 0) ss_out[(size_t)t * ss_ld + warp] = st;
    }
    return;
  }
  // second norm of the (already normalised) row: its mean square is ss*r0^2/d
  float ss1 = 0.f;
  for (int j = lane; j < d; j += 32) {
    const float v = to_f(e[j]) * r0;
    x[(size_t)warp * d + j] = v;
    ss1 = fmaf(v, v, ss1);
  }
  ss1 = warp_sum(ss1);
  const float r1 = rsqrtf(ss1 / d + eps);
  for (int j = lane; j < d; j += 32) h[(size_t)warp * d + j] = from_f<TA>(x[(size_t)warp * d + j] * r1);
}

// One warp per output row: h[i] = TA(rms(x[src_row(i)])), src_row(i) =
// i*stride + (last ? last[i] : 0): stride 1 and no `last` for all rows;
// stride T and last[i] = the index of row i's last token for the last
// position of each row.
template <typename TA>
__global__ void rmsnorm_kernel(const float* __restrict__ x, TA* __restrict__ h, int rows, int d,
                               int stride, const int* __restrict__ last, float eps, int* len_inc) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  // the final norm of a decode step on the generic path (fp32 models, or a
  // batch wider than the decode GEMMs) advances every row's device-side
  // cache length; every kernel of the step that reads them has finished
  // (stream order)
  if (len_inc && blockIdx.x == 0)
    for (int i = threadIdx.x; i < rows; i += blockDim.x) len_inc[i] += 1;
  if (warp >= rows) return;
  const float* xr = x + ((size_t)warp * stride + (last ? last[warp] : 0)) * d;
  float ss = 0.f;
  if ((d & 127) == 0) {
    for (int j = lane * 4; j < d; j += 128) {
      const float4 v = *reinterpret_cast<const float4*>(xr + j);
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  } else {
    for (int j = lane; j < d; j += 32) ss = fmaf(xr[j], xr[j], ss);
  }
  ss = warp_sum(ss);
  const float r = rsqrtf(ss / d + eps);
  TA* hr = h + (size_t)warp * d;
  for (int j = lane; j < d; j += 32) hr[j] = from_f<TA>(xr[j] * r);
}

// Last position of each row with the RMSNorm folded into the unembedding:
// h_out[i] = h[src(i)] and ss_out[t * ss_ld_out + i] = ss[t * ss_ld + src(i)]
// for the n_ss column blocks t, src(i) = i * stride + last[i].  A copy of what
// the last residual epilogue wrote, so the last-position logits are the same
// bits as the all-position ones.  One warp per row, 16-byte copies (d a
// multiple of 8).
template <typename TA>
__global__ void gather_last_kernel(const TA* __restrict__ h, const float* __restrict__ ss, int ss_ld, int n_ss,
                                   TA* __restrict__ h_out, float* __restrict__ ss_out, int ss_ld_out, int rows,
                                   int d, int stride, const int* __restrict__ last) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  pdl_wait();
  if (warp >= rows) return;
  const int src = warp * stride + last[warp];
  const uint4* hs = reinterpret_cast<const uint4*>(h + (size_t)src * d);
  uint4* hd = reinterpret_cast<uint4*>(h_out + (size_t)warp * d);
  for (int j = lane; j < d * (int)sizeof(TA) / 16; j += 32) hd[j] = hs[j];
  for (int t = lane; t < n_ss; t += 32) ss_out[(size_t)t * ss_ld_out + warp] = ss[(size_t)t * ss_ld + src];
}

// fp32 SIMT GEMM, C = A W^T with an elementwise epilogue.  64x64 tile per
// 256-thread block, 4x4 outputs per thread.
enum SimtEpi : int { SEPI_STORE = 0, SEPI_RESID = 1, SEPI_RELU2 = 2, SEPI_LOGITS = 3 };

template <int EPI>
__global__ void __launch_bounds__(256) gemm_simt_f32_kernel(const float* __restrict__ A,
                                                             const float* __restrict__ W,
                                                             float* __restrict__ out, int M, int N,
                                                             int K, int ldo, float cap) {
  constexpr int BMS = 64, BNS = 64, BKS = 16;
  __shared__ float As[BKS][BMS + 4];
  __shared__ float Ws[BKS][BNS + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int m0 = blockIdx.y * BMS, n0 = blockIdx.x * BNS;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BKS) {
    for (int i = threadIdx.x; i < BMS * BKS; i += 256) {
      const int r = i / BKS, kk = i % BKS;
      const int m = m0 + r, k = k0 + kk, n = n0 + r;
      As[kk][r] = (m < M && k < K) ? A[(size_t)m * K + k] : 0.f;
      Ws[kk][r] = (n < N && k < K) ? W[(size_t)n * K + k] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BKS; ++kk) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float* o = out + (size_t)m * ldo + n;
      const float v = acc[i][j];
      if constexpr (EPI == SEPI_STORE) *o = v;
      if constexpr (EPI == SEPI_RESID) *o += v;
      if constexpr (EPI == SEPI_RELU2) { const float r = fmaxf(v, 0.f); *o = r * r; }
      if constexpr (EPI == SEPI_LOGITS) *o = cap * tanhf(v / cap);
    }
  }
}

// One warp per (row m, head slot): slots [0, n_head) are query heads, then
// n_kv key heads, then n_kv value heads.  q and k: RoPE at the row's
// position pos0[b] + t, then RMSNorm over head_dim; v: copied.  q goes to
// Q [M, n_head*hd], k and v of K/V head g to the cache row (b, g, pos).  Each lane holds
// elements lane + 32 i, so both members of a rotation pair (j, j + hd/2) sit
// in the same lane.
template <typename TA, typename TC>
__global__ void qkv_post_kernel(const float* __restrict__ qkv, TA* __restrict__ q_out,
                                TC* __restrict__ k_cache, TC* __restrict__ v_cache,
                                const float* __restrict__ rope_cos, const float* __restrict__ rope_sin,
                                int M, int n_head, int n_kv, int hd, int T, const int* __restrict__ pos0,
                                int cache_S, float eps) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int slots = n_head + 2 * n_kv;
  if (warp >= M * slots) return;
  const int m = warp / slots, head = warp % slots;
  const int b = m / T, pos = pos0[b] + (m % T);
  const int per = hd / 32, half = hd / 2;     // hd in {64, 128}
  const float* src = qkv + (size_t)m * (slots * hd) + head * hd;
  float v[4];
  for (int i = 0; i < per; ++i) v[i] = src[lane + 32 * i];
  if (head < n_head + n_kv) {                   // query or key: RoPE + QK-norm
    float ss = 0.f;
    for (int i = 0; i < per; ++i) ss = fmaf(v[i], v[i], ss);
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / hd + eps);
    for (int i = 0; i < per / 2; ++i) {
      const int j = lane + 32 * i;             // first member of the pair, j < hd/2
      const float c = rope_cos[(size_t)pos * half + j], s = rope_sin[(size_t)pos * half + j];
      const float x0 = v[i] * r, x1 = v[i + per / 2] * r;
      v[i] = x0 * c - x1 * s;
      v[i + per / 2] = x0 * s + x1 * c;
    }
  }
  if (head < n_head) {
    TA* dst = q_out + (size_t)m * (n_head * hd) + head * hd;
    for (int i = 0; i < per; ++i) dst[lane + 32 * i] = from_f<TA>(v[i]);
  } else {
    const bool is_v = head >= n_head + n_kv;
    const int g = is_v ? head - n_head - n_kv : head - n_head;
    TC* dst = (is_v ? v_cache : k_cache) + (((size_t)b * n_kv + g) * cache_S + pos) * hd;
    for (int i = 0; i < per; ++i) dst[lane + 32 * i] = from_f<TC>(v[i]);
  }
}

// Per-row cache bookkeeping of one call, written on the device in stream
// order for rows base .. base + n - 1: pos0[b] = the row's cache length
// before the call (the position of its first new token), len[b] = its length
// after the call, last[b] = the index of its last token in the call's
// [B][T] token array.  The values travel in the kernel's parameters, so the
// host may reuse its buffers at once.
constexpr int ROWSET_MAX = 256;
struct RowSet {
  int n, base;
  int32_t pos0[ROWSET_MAX], len[ROWSET_MAX], last[ROWSET_MAX];
};
__global__ void set_rows_kernel(const RowSet rs, int* __restrict__ pos0, int* __restrict__ len,
                                int* __restrict__ last) {
  pdl_trigger();
  pdl_wait();
  for (int i = threadIdx.x; i < rs.n; i += blockDim.x) {
    pos0[rs.base + i] = rs.pos0[i];
    len[rs.base + i] = rs.len[i];
    last[rs.base + i] = rs.last[i];
  }
}

// max |src[i]| over n values, as the bit pattern of a non-negative float
// (those order like unsigned integers): atomicMax into *amax (zeroed before)
__global__ void absmax_kernel(const float* __restrict__ src, size_t n, unsigned int* amax) {
  float m = 0.f;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    m = fmaxf(m, fabsf(src[i]));
  m = warp_max(m);
  if ((threadIdx.x & 31) == 0) atomicMax(amax, __float_as_uint(m));
}

// FP8 weights (FP8 E4M3 values times one power-of-two scale per matrix):
// q[i] = e4m3(src[i] / scale) (round to nearest even, saturating at 448), and
// deq[i] = bf16(e4m3 value * scale), the exact 16-bit image the prefill GEMMs
// use (an E4M3 value has 3 mantissa bits; times a power of two it is a bf16
// value).  inv_scale = 1 / scale, both powers of two: the products are exact.
__global__ void quantize_e4m3_kernel(const float* __restrict__ src, size_t n, float inv_scale, float scale,
                                     uint8_t* __restrict__ q, __nv_bfloat16* __restrict__ deq) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const __nv_fp8_storage_t c = __nv_cvt_float_to_fp8(src[i] * inv_scale, __NV_SATFINITE, __NV_E4M3);
    q[i] = c;
    const __half h(__nv_cvt_fp8_to_halfraw(c, __NV_E4M3));
    deq[i] = __float2bfloat16_rn(__half2float(h) * scale);
  }
}

// ------------------------------------------------ later-architecture extras
// (apidog.com/th "how nanochat works" item 1: value embeddings, per-layer
// residual lambdas, smear, backout; parity-only features of a later version)

__device__ __forceinline__ float sigmoidf_(float z) { return 1.f / (1.f + __expf(-z)); }

// Smear, one warp per row m = b*T + t of a call whose row b starts at
// position pos0[b]: x[m] += lambda * sigmoid(x[m][:SC] . w) * x_prev, x_prev
// the previous token's normed embedding rms(E[prev]) (the previous token of
// the call, or prev_tok[b] from the row's earlier calls; none at position 0).
// x[m] holds rms(E[tok[m]]) on entry (written by the embedding kernel).
template <typename TW>
__global__ void smear_kernel(const int32_t* __restrict__ tok, const TW* __restrict__ E, float* __restrict__ x,
                             int M, int T, int d, int vocab, const int* __restrict__ pos0,
                             const int32_t* __restrict__ prev_tok, const float* __restrict__ w,
                             const float* __restrict__ lambda, int SC, float eps) {
  const int m = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (m >= M) return;
  const int b = m / T, t = m - b * T;
  int prev = t > 0 ? tok[m - 1] : (pos0[b] > 0 ? prev_tok[b] : -1);
  if (prev < 0) return;
  if (prev >= vocab) prev = 0;                     // flagged by the embedding kernel
  float* xr = x + (size_t)m * d;
  float g = 0.f;
  for (int c = lane; c < SC; c += 32) g = fmaf(xr[c], w[c], g);
  g = warp_sum(g);
  const TW* e = E + (size_t)prev * d;
  float ss = 0.f;
  for (int j = lane; j < d; j += 32) {
    const float v = to_f(e[j]);
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  const float f = *lambda * sigmoidf_(g) * rsqrtf(ss / d + eps);
  __syncwarp();
  for (int j = lane; j < d; j += 32) xr[j] = fmaf(f, to_f(e[j]), xr[j]);
}

// x = a x + c x0 elementwise, a = *pa, c = *pc (the residual and x0 lambdas of a layer)
__global__ void lambda_mix_kernel(float* __restrict__ x, const float* __restrict__ x0, size_t n,
                                  const float* __restrict__ pa, const float* __restrict__ pc) {
  const float a = *pa, c = *pc;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    x[i] = fmaf(a, x[i], c * x0[i]);
}

// x -= lambda * x_mid elementwise (backout)
__global__ void backout_kernel(float* __restrict__ x, const float* __restrict__ x_mid, size_t n,
                               const float* __restrict__ lambda) {
  const float l = *lambda;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    x[i] = fmaf(-l, x_mid[i], x[i]);
}

// Value embedding of a layer, one warp per (row m, K/V head g): gate =
// 3 sigmoid(h[m][:C] . G[g]) and the cached value row (b, g, pos) becomes
// v + gate * VE[tok[m]][g]; the same in the transposed copy V^T when given.
// h is the block's normed input (the operand of the QKV projection).
template <typename TA, typename TC>
__global__ void value_embed_kernel(const TA* __restrict__ h, int d, const int32_t* __restrict__ tok, int vocab,
                                   const float* __restrict__ ve, const float* __restrict__ gate_w, int C,
                                   TC* __restrict__ v_cache, TC* __restrict__ vt, int vt_S, int M, int T,
                                   int n_kv, int hd, int cache_S, const int* __restrict__ pos0) {
  const int wi = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wi >= M * n_kv) return;
  const int m = wi / n_kv, g = wi - m * n_kv;
  const int b = m / T, pos = pos0[b] + (m - b * T);
  int tk = tok[m];
  if (tk < 0 || tk >= vocab) tk = 0;               // flagged by the embedding kernel
  float z = 0.f;
  for (int c = lane; c < C; c += 32) z = fmaf(to_f(h[(size_t)m * d + c]), gate_w[(size_t)g * C + c], z);
  z = warp_sum(z);
  const float gate = 3.f * sigmoidf_(z);
  const float* e = ve + ((size_t)tk * n_kv + g) * hd;
  TC* vr = v_cache + (((size_t)b * n_kv + g) * cache_S + pos) * hd;
  for (int j = lane; j < hd; j += 32) {
    const TC nv = from_f<TC>(fmaf(gate, e[j], to_f(vr[j])));
    vr[j] = nv;
    if (vt) vt[((size_t)(b * n_kv + g) * hd + j) * vt_S + pos] = nv;
  }
}

// prev_tok[b] = the last token of row b in this call (index last[b], or T - 1)
__global__ void set_prev_tok_kernel(const int32_t* __restrict__ tok, int B, int T, const int* __restrict__ last,
                                    int32_t* __restrict__ prev_tok) {
  for (int b = threadIdx.x; b < B; b += blockDim.x) prev_tok[b] = tok[(size_t)b * T + (last ? last[b] : T - 1)];
}

// fp32 -> bf16 (round to nearest even) weight conversion
__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                   size_t n) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
       i += (size_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

}  // namespace nc
