// Causal multi-query attention for the decode step on the tensor cores (bf16
// in, fp32 accumulate, mma.sync): scores, softmax and P.V stay on chip.
//
// Multi-query attention: every query head reads the single K/V head
// (yelogs.com nanochat story, "technical details and official Q&A"); scale
// 1/sqrt(head_dim) as in SDPA (apidog.com/th "train your own ChatGPT", "how
// nanochat works" item 5).
//
// Decode kernel (split over the context): one CTA = one batch row and a
// group of consecutive 128-key sub-chunks streamed through a cp.async ring;
// the row's n_head query vectors form the 16-row A operand (heads padded to
// 16), each of 8 warps handles 16 keys of every sub-chunk with a running
// softmax.  A row covered by one group writes its output directly; otherwise
// the groups of the row form a thread-block cluster, and they merge their
// partial (max, sum, output) through distributed shared memory into the bf16
// output.
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

// A [rows][128] bf16 tile in shared memory, rows of 256 B split in 16 chunks
// of 16 B; chunk c of row r is stored at chunk c ^ (r & 7) to keep ldmatrix
// conflict-free.
__device__ __forceinline__ uint32_t swz(uint32_t base, int row, int chunk) {
  return base + row * 256 + ((chunk ^ (row & 7)) << 4);
}

constexpr int ATT_HD = 128;

// ---------------------------------------------------------------- decode --
// Q: [B][n_head*128] (one new position per row, at pos = ctx-1); keys 0..ctx-1.
// With pos_dev, row b's context is pos_dev[b] + 1 (per-row cache lengths).
// Grouped-query attention (apidog.com/th item 1): grid.y runs over the K/V
// sequences s = b * n_kv + g, and the CTA serves the n_head / n_kv query heads
// of K/V head g; a sliding window (window > 0) limits the keys to the last
// `window` positions (the sub-chunks before it are skipped).
// CTA (group g, row b) streams `group` consecutive sub-chunks of DEC_SUB keys
// (keys [g*group*DEC_SUB, ...)) through a DEC_STAGES-deep cp.async ring and
// keeps a running (max, sum, output) per warp across them; each of the
// DEC_WARPS warps owns DEC_KPW keys of every sub-chunk.  One CTA fills most of
// an SM's shared memory: its ring keeps two 64 KB sub-chunks in flight and
// its 8 warps hide each other's MMA/softmax latency.  Partial results per
// (row b, group g) stay in the CTA's shared memory: the groups of a row are
// the CTAs of one thread-block cluster (grid.x = cluster size <=
// DEC_MAX_GROUPS), which merge through distributed shared memory.
constexpr int DEC_CHUNK = 128;             // a group covers at least this many keys
constexpr int DEC_MAX_GROUPS = 8;          // portable cluster size
constexpr int DEC_SUB = 128;               // keys per pipeline stage
constexpr int DEC_STAGES = 3;
constexpr int DEC_WARPS = 8;
constexpr int DEC_THREADS = DEC_WARPS * 32;
constexpr int DEC_KPW = DEC_SUB / DEC_WARPS;   // keys per warp per sub-chunk (two 8-key MMA tiles)
constexpr uint32_t DEC_STAGE_BYTES = 2 * DEC_SUB * 256;   // K and V rows of a sub-chunk
static_assert(DEC_KPW == 16, "the score tile loop assumes 16 keys per warp");
static_assert(DEC_CHUNK % DEC_SUB == 0 || DEC_SUB % DEC_CHUNK == 0, "partial buffers sized by DEC_CHUNK");

// TO: the output type (bf16, or f16 when the next projection's activations are f16)
template <typename TO>
__global__ void __launch_bounds__(DEC_THREADS) attn_decode_mma_kernel(
    const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ Kc,
    const __nv_bfloat16* __restrict__ Vc, TO* __restrict__ O, int n_head, int cache_S, int ctx_arg,
    const int* __restrict__ pos_dev, float scale_log2, int group, int n_kv, int window) {
  pdl_trigger();
  const int grp = blockIdx.x, bs = blockIdx.y;                 // K/V sequence bs = b * n_kv + g
  const int b = bs / n_kv, g = bs % n_kv;
  const int nq = n_head / n_kv, h0 = g * nq;                   // query heads h0 .. h0 + nq - 1
  int c_begin = grp * group;                                   // first sub-chunk of this CTA
  // With pos_dev the context is read on the device (the step is
  // graph-replayable).  The previous step advances the length in its last
  // kernel, which may still be running when this kernel starts (dependent
  // launches chain), so a length read before the wait is the current one or
  // one less.  The keys below that early length minus one were written two
  // or more steps ago either way: they are streamed before the wait.  The
  // exact context is read after it and the remaining keys are loaded then.
  // Groups beyond the context have no keys (they still take part in the
  // cluster's barriers).  A windowed layer loads nothing early (its first
  // sub-chunk depends on the exact context).
  const int early_keys = window > 0 ? 0 : (pos_dev ? pos_dev[b] - 1 : ctx_arg - 1);   // keys [0, early_keys)
  const int n_early = max(0, min(group, (early_keys + DEC_SUB - 1) / DEC_SUB - c_begin));
  extern __shared__ __align__(128) uint8_t att_smem[];
  const uint32_t sQ = smem_u32(att_smem);                     // 16 rows
  const uint32_t sS = sQ + 16 * 256;                           // DEC_STAGES x (K, V) sub-chunks
  float* red = reinterpret_cast<float*>(att_smem + 16 * 256 + DEC_STAGES * DEC_STAGE_BYTES);  // [DEC_WARPS][16][2]
  float* ored = reinterpret_cast<float*>(att_smem + 16 * 256);  // [DEC_WARPS][16][128], aliases the stages
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, ocol = tid & 127;
  const int ldq = n_head * ATT_HD;
  const __nv_bfloat16* kb = Kc + (size_t)bs * cache_S * ATT_HD;
  const __nv_bfloat16* vb = Vc + (size_t)bs * cache_S * ATT_HD;
  // rows of sub-chunk i: keys (c_begin + i) * DEC_SUB + r.  `early`: only
  // the keys below key_lim (written by earlier calls); otherwise the keys the
  // early pass did not load (below early_lim nothing is reloaded), with keys
  // >= ctx zero-filled
  int ctx = ctx_arg;
  auto load_sub = [&](int i, bool early, int key_lim, int early_lim) {
    const uint32_t sk = sS + (i % DEC_STAGES) * DEC_STAGE_BYTES, sv = sk + DEC_SUB * 256;
    const int k0 = (c_begin + i) * DEC_SUB;
    for (int e = tid; e < DEC_SUB * 16; e += DEC_THREADS) {
      const int r = e >> 4, c = e & 15;
      const int key = k0 + r;
      if (early ? key >= key_lim : key < early_lim) continue;
      const bool ok = early || key < ctx;                      // early keys all exist
      const size_t off = (size_t)(ok ? key : 0) * ATT_HD + c * 8;
      cp_async16(swz(sk, r, c), kb + off, ok);
      cp_async16(swz(sv, r, c), vb + off, ok);
    }
  };
  const int pre_early = n_early < DEC_STAGES - 1 ? n_early : DEC_STAGES - 1;
  for (int i = 0; i < pre_early; ++i) {
    load_sub(i, true, early_keys, 0);
    cp_async_commit();
  }
  pdl_wait();                                                  // q and the newest K/V row
  if (pos_dev) ctx = pos_dev[b] + 1;
  const int klo = window > 0 ? max(0, ctx - window) : 0;     // the first key inside the window
  const int s_first = klo / DEC_SUB;
  c_begin = s_first + grp * group;
  const int nsub = (ctx + DEC_SUB - 1) / DEC_SUB;
  const int ngroups = (nsub - s_first + group - 1) / group;
  const int n = max(0, min(group, nsub - c_begin));
  const int pre = n < DEC_STAGES - 1 ? n : DEC_STAGES - 1;
  for (int e = tid; e < 16 * 16; e += DEC_THREADS) {
    const int r = e >> 4, c = e & 15;
    const bool ok = r < nq;
    cp_async16(swz(sQ, r, c), Q + (size_t)b * ldq + (h0 + (ok ? r : 0)) * ATT_HD + c * 8, ok);
  }
  // the keys of the first `pre` sub-chunks not loaded early (sub-chunks the
  // early pass did not start are loaded whole)
  for (int i = 0; i < pre; ++i) load_sub(i, false, 0, i < pre_early ? early_keys : 0);
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
  float m_lo = -INFINITY, m_hi = -INFINITY;                    // running max (quad-uniform)
  float sum_lo = 0.f, sum_hi = 0.f;                            // this lane's share of the sums
  float o[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  for (int i = 0; i < n; ++i) {
    if (i + DEC_STAGES - 1 < n) load_sub(i + DEC_STAGES - 1, false, 0, 0);
    cp_async_commit();
    cp_async_wait<DEC_STAGES - 1>();
    __syncthreads();
    const uint32_t sK = sS + (i % DEC_STAGES) * DEC_STAGE_BYTES, sV = sK + DEC_SUB * 256;
    const int k0 = (c_begin + i) * DEC_SUB;
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
    float mx_lo = m_lo, mx_hi = m_hi;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = k0 + wk + j * 8 + (lane & 3) * 2 + e;
        const bool ok = key < ctx && key >= klo;
        s[j][e] = ok ? s[j][e] * scale_log2 : -INFINITY;
        s[j][2 + e] = ok ? s[j][2 + e] * scale_log2 : -INFINITY;
        mx_lo = fmaxf(mx_lo, s[j][e]);
        mx_hi = fmaxf(mx_hi, s[j][2 + e]);
      }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    // rows with no valid key so far keep max -inf: subtract 0 so exp2 gives 0, not NaN
    const float ml = mx_lo == -INFINITY ? 0.f : mx_lo, mh = mx_hi == -INFINITY ? 0.f : mx_hi;
    const float c_lo = m_lo == -INFINITY ? 0.f : exp2f(m_lo - ml);
    const float c_hi = m_hi == -INFINITY ? 0.f : exp2f(m_hi - mh);
    m_lo = mx_lo;
    m_hi = mx_hi;
    sum_lo *= c_lo;
    sum_hi *= c_hi;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= c_lo;
      o[j][1] *= c_lo;
      o[j][2] *= c_hi;
      o[j][3] *= c_hi;
    }
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
    __syncthreads();                                           // the stage may be refilled
  }
  sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 1);
  sum_lo += __shfl_xor_sync(0xffffffffu, sum_lo, 2);
  sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 1);
  sum_hi += __shfl_xor_sync(0xffffffffu, sum_hi, 2);
  // ---- merge the 4 warps: per head row, rescale to the CTA max
  const int rlo = lane >> 2, rhi = rlo + 8;
  if ((lane & 3) == 0) {
    red[(warp * 16 + rlo) * 2 + 0] = m_lo;
    red[(warp * 16 + rlo) * 2 + 1] = sum_lo;
    red[(warp * 16 + rhi) * 2 + 0] = m_hi;
    red[(warp * 16 + rhi) * 2 + 1] = sum_hi;
  }
  __syncthreads();                                             // all warps done with K/V
  float cm_lo = -INFINITY, cm_hi = -INFINITY;
#pragma unroll
  for (int w = 0; w < DEC_WARPS; ++w) {
    cm_lo = fmaxf(cm_lo, red[(w * 16 + rlo) * 2]);
    cm_hi = fmaxf(cm_hi, red[(w * 16 + rhi) * 2]);
  }
  const float f_lo = m_lo == -INFINITY ? 0.f : exp2f(m_lo - cm_lo);
  const float f_hi = m_hi == -INFINITY ? 0.f : exp2f(m_hi - cm_hi);
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int col = j * 8 + (lane & 3) * 2;
    ored[(warp * 16 + rlo) * 128 + col] = o[j][0] * f_lo;
    ored[(warp * 16 + rlo) * 128 + col + 1] = o[j][1] * f_lo;
    ored[(warp * 16 + rhi) * 128 + col] = o[j][2] * f_hi;
    ored[(warp * 16 + rhi) * 128 + col + 1] = o[j][3] * f_hi;
  }
  __syncthreads();
  // per head row: the CTA's max and sum over its warps
  float cm = -INFINITY, cl = 0.f;
  if (tid < nq) {
    for (int w = 0; w < DEC_WARPS; ++w) cm = fmaxf(cm, red[(w * 16 + tid) * 2]);
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float mw = red[(w * 16 + tid) * 2];
      if (mw != -INFINITY) cl += red[(w * 16 + tid) * 2 + 1] * exp2f(mw - cm);
    }
  }
  if (ngroups == 1) {
    // group 0 covered the whole context: normalise and write the output (no
    // CTA of the cluster waits on a cluster barrier in this case)
    if (grp != 0) return;
    float* inv_l1 = reinterpret_cast<float*>(att_smem);         // the Q tile is in registers
    if (tid < nq) inv_l1[tid] = 1.f / cl;
    __syncthreads();
    // thread = output column of every other head row
    for (int r = tid >> 7; r < nq; r += DEC_THREADS / 128) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < DEC_WARPS; ++w) acc += ored[(w * 16 + r) * 128 + ocol];
      O[((size_t)b * n_head + h0 + r) * ATT_HD + ocol] = from_f<TO>(acc * inv_l1[r]);
    }
    return;
  }
  // ---- merge the groups of row b (the CTAs of this cluster, rank = grp):
  // each parks its partial (o summed over its warps, m, l) in its own shared
  // memory; after a cluster barrier CTA q merges head rows q, q + G, ... from
  // every rank in rank order (the result does not depend on timing)
  float* po = reinterpret_cast<float*>(att_smem + 16 * 256 + DEC_WARPS * 16 * 128 * 4);  // [16][128]
  float* pml = po + 16 * 128;                                                            // [16][2]
  for (int r = tid >> 7; r < nq; r += DEC_THREADS / 128) {
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) acc += ored[(w * 16 + r) * 128 + ocol];
    po[r * 128 + ocol] = acc;
  }
  if (tid < nq) {
    pml[tid * 2 + 0] = cm;
    pml[tid * 2 + 1] = cl;
  }
  cluster_sync_all();
  const int G = (int)gridDim.x;
  const uint32_t po_s = smem_u32(po), pml_s = smem_u32(pml);
  for (int r = grp + G * (tid >> 7); r < nq; r += G * (DEC_THREADS / 128)) {
    float mg[DEC_MAX_GROUPS], lg[DEC_MAX_GROUPS], og[DEC_MAX_GROUPS];
#pragma unroll
    for (int g = 0; g < DEC_MAX_GROUPS; ++g) {
      const bool in = g < G;
      mg[g] = in ? ld_cluster_f32(pml_s + r * 8, (uint32_t)g) : -INFINITY;
      lg[g] = in ? ld_cluster_f32(pml_s + r * 8 + 4, (uint32_t)g) : 0.f;
      og[g] = in ? ld_cluster_f32(po_s + (r * 128 + ocol) * 4, (uint32_t)g) : 0.f;
    }
    float gm = -INFINITY;
#pragma unroll
    for (int g = 0; g < DEC_MAX_GROUPS; ++g) gm = fmaxf(gm, mg[g]);
    float l = 0.f, acc = 0.f;
#pragma unroll
    for (int g = 0; g < DEC_MAX_GROUPS; ++g) {
      if (g >= G) break;
      const float f = mg[g] == -INFINITY ? 0.f : exp2f(mg[g] - gm);
      l += lg[g] * f;
      acc += og[g] * f;
    }
    O[((size_t)b * n_head + h0 + r) * ATT_HD + ocol] = from_f<TO>(acc * (1.f / l));
  }
  cluster_sync_all();                                          // remote reads done before any CTA exits
}

constexpr size_t ATT_DECODE_SMEM = 16 * 256 + DEC_STAGES * (size_t)DEC_STAGE_BYTES + DEC_WARPS * 16 * 2 * 4;

}  // namespace nc
