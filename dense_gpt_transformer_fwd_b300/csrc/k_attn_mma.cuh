// Causal multi-query attention for the decode step on the tensor cores (bf16
// in, fp32 accumulate, mma.sync): scores, softmax and P.V stay on chip.
//
// Multi-query attention: every query head reads the single K/V head
// (yelogs.com nanochat story, "technical details and official Q&A"); scale
// 1/sqrt(head_dim) as in SDPA (apidog.com/th "train your own ChatGPT", "how
// nanochat works" item 5).
//
// Decode kernel (split over the context): one CTA = one batch row and a
// chunk of 128 cached keys; the row's n_head query vectors form the 16-row
// A operand (heads padded to 16), each warp handles 32 keys; partial (max,
// sum, output) go to a workspace, and the last CTA of the row to finish
// (a per-row counter) merges the chunks into the bf16 output.
#pragma once

#include "nc_common.cuh"

namespace nc {

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  const int n = pred ? 16 : 0;   // zero-fill when pred is false
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// A [rows][128] bf16 tile in shared memory, rows of 256 B split in 16 chunks
// of 16 B; chunk c of row r is stored at chunk c ^ (r & 7) to keep ldmatrix
// conflict-free.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + row * 256 + ((chunk ^ (row & 7)) << 4);
}

constexpr int ATT_HD = 128;

// ---------------------------------------------------------------- decode --
// Q: [B][n_head*128] (one new position per row, at pos = ctx-1); keys 0..ctx-1.
// Partial results per (row b, chunk c): m, l [B][nchunk][16][2], o [B][nchunk][16][128].
constexpr int DEC_CHUNK = 128;             // keys per CTA
constexpr int DEC_KPW = DEC_CHUNK / 4;     // keys per warp

__global__ void __launch_bounds__(128) attn_decode_mma_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Kc,
    const __nv_bfloat16* __restrict__ Vc, float* __restrict__ part_o, float* __restrict__ part_ml,
    __nv_bfloat16* __restrict__ O, int* __restrict__ counters, int n_head, int cache_S, int ctx,
    const int* __restrict__ pos_dev, float scale_log2) {
  pdl_trigger();
  // with pos_dev the context is read on the device (the step is graph-replayable);
  // the length only changes at the end of a step, so it may be read before
  // waiting for the previous kernel.  Chunks beyond the context exit.
  if (pos_dev) ctx = *pos_dev + 1;
  const int nchunk = (ctx + DEC_CHUNK - 1) / DEC_CHUNK;
  if ((int)blockIdx.x >= nchunk) return;
  extern __shared__ __align__(128) uint8_t att_smem[];
  const uint32_t sQ = smem_u32(att_smem);                     // 16 rows
  const uint32_t sK = sQ + 16 * 256;                           // DEC_CHUNK keys
  const uint32_t sV = sK + DEC_CHUNK * 256;
  float* red = reinterpret_cast<float*>(att_smem + (16 + 2 * DEC_CHUNK) * 256);  // [4][16][2]
  float* ored = reinterpret_cast<float*>(att_smem + 16 * 256);  // [4][16][128], aliases K/V
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk_id = blockIdx.x, b = blockIdx.y;
  const int k0 = chunk_id * DEC_CHUNK;
  const int ldq = n_head * ATT_HD;
  const __nv_bfloat16* kb = Kc + (size_t)b * cache_S * ATT_HD;
  const __nv_bfloat16* vb = Vc + (size_t)b * cache_S * ATT_HD;
  // keys before the newest were written by earlier calls: stream them now
  for (int i = tid; i < DEC_CHUNK * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    const int key = k0 + r;
    if (key >= ctx - 1) continue;
    const size_t off = (size_t)key * ATT_HD + c * 8;
    cp_async16(swz(sK, r, c), kb + off, true);
    cp_async16(swz(sV, r, c), vb + off, true);
  }
  cp_async_commit();
  pdl_wait();                                                  // q and the newest K/V row
  for (int i = tid; i < 16 * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    const bool ok = r < n_head;
    cp_async16(swz(sQ, r, c), Q + (size_t)b * ldq + (ok ? r : 0) * ATT_HD + c * 8, ok);
  }
  for (int i = tid; i < DEC_CHUNK * 16; i += 128) {
    const int r = i >> 4, c = i & 15;
    const int key = k0 + r;
    if (key < ctx - 1) continue;
    const bool ok = key < ctx;
    const size_t off = (size_t)(ok ? key : 0) * ATT_HD + c * 8;
    cp_async16(swz(sK, r, c), kb + off, ok);
    cp_async16(swz(sV, r, c), vb + off, ok);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  uint32_t qf[8][4];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
    ldsm_x4(swz(sQ, row, kk * 2 + (lane >> 4)), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
  }
  constexpr int NT = DEC_KPW / 8;                              // 8-key tiles per warp
  const int wk = warp * DEC_KPW;
  float s[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
    for (int jp = 0; jp < NT / 2; ++jp) {
      const int key = wk + jp * 16 + (lane & 7) + (lane >> 4) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(swz(sK, key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
      mma_bf16(s[2 * jp], qf[kk], b0, b1);
      mma_bf16(s[2 * jp + 1], qf[kk], b2, b3);
    }
  }
  float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int key = k0 + wk + j * 8 + (lane & 3) * 2 + e;
      const bool ok = key < ctx;
      s[j][e] = ok ? s[j][e] * scale_log2 : -INFINITY;
      s[j][2 + e] = ok ? s[j][2 + e] * scale_log2 : -INFINITY;
      mx_lo = fmaxf(mx_lo, s[j][e]);
      mx_hi = fmaxf(mx_hi, s[j][2 + e]);
    }
  mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
  mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
  mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
  mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
  // a warp whose keys all lie beyond ctx has max -inf: subtract 0 so exp2 gives 0, not NaN
  const float ml = mx_lo == -INFINITY ? 0.f : mx_lo, mh = mx_hi == -INFINITY ? 0.f : mx_hi;
  float sum_lo = 0.f, sum_hi = 0.f;
  uint32_t pf[NT / 2][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const float p0 = exp2f(s[j][0] - ml), p1 = exp2f(s[j][1] - ml);
    const float p2 = exp2f(s[j][2] - mh), p3 = exp2f(s[j][3] - mh);
    sum_lo += p0 + p1;
    sum_hi += p2 + p3;
    pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16(p0, p1);
    pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16(p2, p3);
  }
  sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 1);
  sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 2);
  sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 1);
  sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 2);
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < NT / 2; ++kk) {
#pragma unroll
    for (int jp = 0; jp < 8; ++jp) {
      const int key = wk + kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(swz(sV, key, jp * 2 + (lane >> 4)), b0, b1, b2, b3);
      mma_bf16(o[2 * jp], pf[kk], b0, b1);
      mma_bf16(o[2 * jp + 1], pf[kk], b2, b3);
    }
  }
  // ---- merge the 4 warps: per head row, rescale to the CTA max
  const int rlo = lane >> 2, rhi = rlo + 8;
  if ((lane & 3) == 0) {
    red[(warp * 16 + rlo) * 2 + 0] = mx_lo;
    red[(warp * 16 + rlo) * 2 + 1] = sum_lo;
    red[(warp * 16 + rhi) * 2 + 0] = mx_hi;
    red[(warp * 16 + rhi) * 2 + 1] = sum_hi;
  }
  __syncthreads();                                             // all warps done with K/V
  float cm_lo = -INFINITY, cm_hi = -INFINITY;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    cm_lo = fmaxf(cm_lo, red[(w * 16 + rlo) * 2]);
    cm_hi = fmaxf(cm_hi, red[(w * 16 + rhi) * 2]);
  }
  const float f_lo = mx_lo == -INFINITY ? 0.f : exp2f(mx_lo - cm_lo);
  const float f_hi = mx_hi == -INFINITY ? 0.f : exp2f(mx_hi - cm_hi);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = j * 8 + (lane & 3) * 2;
    ored[(warp * 16 + rlo) * 128 + col] = o[j][0] * f_lo;
    ored[(warp * 16 + rlo) * 128 + col + 1] = o[j][1] * f_lo;
    ored[(warp * 16 + rhi) * 128 + col] = o[j][2] * f_hi;
    ored[(warp * 16 + rhi) * 128 + col + 1] = o[j][3] * f_hi;
  }
  __syncthreads();
  // thread = output column; loop over head rows
  const size_t pbase = ((size_t)b * nchunk + chunk_id) * 16;
  for (int r = 0; r < n_head; ++r) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) acc += ored[(w * 16 + r) * 128 + tid];
    part_o[(pbase + r) * 128 + tid] = acc;
  }
  if (tid < n_head) {
    float cm = -INFINITY, cl = 0.f;
    for (int w = 0; w < 4; ++w) cm = fmaxf(cm, red[(w * 16 + tid) * 2]);
    for (int w = 0; w < 4; ++w) {
      const float mw = red[(w * 16 + tid) * 2];
      if (mw != -INFINITY) cl += red[(w * 16 + tid) * 2 + 1] * exp2f(mw - cm);
    }
    part_ml[(pbase + tid) * 2 + 0] = cm;
    part_ml[(pbase + tid) * 2 + 1] = cl;
  }

  // ---- the last chunk CTA of row b to finish merges every chunk (chunk
  // order fixed, so the result does not depend on which CTA is last)
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&counters[b], 1) == nchunk - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (tid == 0) counters[b] = 0;                               // ready for the next call
  float* wts = ored;                                           // [nchunk][16] merge weights
  float* inv_l = red;                                          // [16]
  __syncthreads();                                             // ored / red no longer read
  const size_t rb = (size_t)b * nchunk * 16;
  if (tid < n_head) {
    float gm = -INFINITY;
    for (int c = 0; c < nchunk; ++c) gm = fmaxf(gm, __ldcg(part_ml + (rb + c * 16 + tid) * 2));
    float l = 0.f;
    for (int c = 0; c < nchunk; ++c) {
      const float mc = __ldcg(part_ml + (rb + c * 16 + tid) * 2);
      const float f = mc == -INFINITY ? 0.f : exp2f(mc - gm);
      wts[c * 16 + tid] = f;
      l += __ldcg(part_ml + (rb + c * 16 + tid) * 2 + 1) * f;
    }
    inv_l[tid] = 1.f / l;
  }
  __syncthreads();
  // thread = output column; all chunks of two heads requested at once
  for (int h0 = 0; h0 < n_head; h0 += 2) {
    float acc[2] = {0.f, 0.f};
    for (int c0 = 0; c0 < nchunk; c0 += 8) {
      float o8[2][8];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int c = c0 + i, h = h0 + hh;
          o8[hh][i] = (c < nchunk && h < n_head) ? __ldcg(part_o + (rb + c * 16 + h) * 128 + tid) : 0.f;
        }
#pragma unroll
      for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c0 + i < nchunk && h0 + hh < n_head) acc[hh] += o8[hh][i] * wts[(c0 + i) * 16 + h0 + hh];
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
      if (h0 + hh < n_head)
        O[((size_t)b * n_head + h0 + hh) * ATT_HD + tid] = f2bf(acc[hh] * inv_l[h0 + hh]);
  }
}

constexpr size_t ATT_DECODE_SMEM = (16 + 2 * DEC_CHUNK) * 256 + 4 * 16 * 2 * 4;

}  // namespace nc
