// Decode-step projections: C[b, n] = sum_k A[b, k] W[n, k] for a handful of
// rows b (the batch, B <= 128) on the 5th-generation tensor cores.
//
// With one new token per row the weight matrix is read once per step and
// each weight is used B times, so these products are bound by HBM bandwidth,
// not by the tensor core.  The operands are swapped relative to the prefill
// GEMM: the MMA's 128-row operand is a tile of 128 weight rows, its N operand
// is the batch (padded to a multiple of 16), so the accumulator in TMEM is
// D[n][b] (lane = weight row).  To keep every SM streaming weights, K is
// split across CTAs: grid = (N / 128) x splits, each CTA owns one weight tile
// and K / splits of its columns, with its loads in flight at once.  The
// splits of one tile form a thread-block cluster: each CTA parks its fp32
// partial D in its own shared memory, and after a cluster barrier CTA r sums
// the partials of every CTA (distributed shared memory, in rank order, so
// the result is deterministic) for the batch rows b = r (mod splits) and
// applies the fused epilogue:
//   EPI_QKV    (the tile is one head) QK-norm + RoPE at the row's position;
//              q -> Q, k and v -> the KV cache row (b, pos)
//   EPI_RESID  x[b, n] += sum                      (fp32 residual stream)
//   EPI_RELU2  u[b, n] = bf16(relu(sum)^2)         (MLP hidden)
//   EPI_LOGITS logits[b, n] = cap * tanh(sum/cap)  (fp32; used with 1 split)
//
// Bias-free projections, QK norm, RoPE, ReLU^2 and the logit softcap follow
// the nanochat pages (yelogs.com story, "technical details and official Q&A";
// geoz.com.cn "development tricks").
//
// 128 threads: warp 0 lane 0 issues the TMA loads, warp 1 lane 0 the MMAs,
// then all four warps (warp w reads TMEM lanes 32w..32w+31) run the
// epilogue.  Every mbarrier wait is bounded.  Launched as a programmatic
// dependent of the previous kernel, the CTA streams its first weight blocks
// into shared memory before it waits for that kernel's results.
//
// FP8 weights (FP8 = true; the FP8 training path of apidog.com/th "how
// nanochat works" item 3, here for inference): each weight matrix is stored
// as FP8 E4M3 values times one power-of-two scale, so a step streams one
// byte per weight instead of two.  The TMA brings 128 x 64 E4M3 tiles (64-byte
// swizzle); four more warps (256 threads) widen each tile exactly to f16 in a
// 128-byte-swizzled tile, which the tensor core reads as the A operand of a
// kind::f16 MMA with f16 activations; the scale multiplies the accumulated
// sums in the epilogue, whose activation outputs are then f16.
#pragma once

#include <cuda.h>
#include <type_traits>
#include "k_gemm_tc.cuh"
#include "nc_common.cuh"

namespace nc {

struct SkinnyArgs {
  int B, N, K;                    // rows, weight rows, reduction length
  int splits, kb_per;             // K split into `splits` ranges of kb_per 64-wide blocks
                                  // (the cluster size along grid y)
  // epilogue outputs
  float* x;                       // EPI_RESID: [B][N] fp32, += ; EPI_LOGITS: [B][N] fp32 out
  __nv_bfloat16* out_bf;          // EPI_QKV: Q [B][n_head*128]
  void* out_act;                  // EPI_RELU2: [B][N] activations (bf16, or f16 with FP8 weights)
  float w_scale;                  // the weight matrix's scale (1 for bf16 weights)
  __nv_bfloat16* k_cache;         // EPI_QKV: this layer's K [B_max][n_kv][S][128]
  __nv_bfloat16* v_cache;
  const float* rope_cos;          // [S][64]
  const float* rope_sin;
  const int* pos_dev;             // EPI_QKV: [B] position of each row's new token (device)
  int n_head, n_kv, cache_S;
  float eps, softcap;
  int* err;
  unsigned long long wait_limit_ns;
  // RMSNorm folded into the epilogues (decode): a residual epilogue also
  // writes h_out = bf16(x) and, per row b, the sum of squares of its 128
  // columns to ss_out[tile * ss_ld + b]; a consumer of h (QKV, MLP up, logits)
  // scales row b of its result by r_b = 1 / sqrt(sum_t ss_in[t * ss_ld + b] / K
  // + eps), summed over the n_ss column blocks in order.  Null: no folding.
  void* h_out;                    // activations (bf16, or f16 with FP8 weights)
  float* ss_out;
  const float* ss_in;
  int n_ss, ss_ld;
  int* len_inc;                   // EPI_LOGITS: the step's final kernel advances every row's cache length
};

// column blocks of 128 in a folded RMSNorm (d_model <= 2048)
constexpr int SK_MAX_SS = 16;

template <int NB, bool FP8 = false>
struct SkCfg {
  static constexpr int THREADS = FP8 ? 256 : 128;         // FP8: four converter warps more
  static constexpr uint32_t W_BYTES = 128 * 64 * 2;      // 16 KB: the MMA's 16-bit weight tile
  static constexpr uint32_t W8_BYTES = FP8 ? 128 * 64 : 0;   // 8 KB: the E4M3 tile the TMA brings
  static constexpr uint32_t A_BYTES = NB * 64 * 2;
  static constexpr uint32_t STAGE_BYTES = W_BYTES + A_BYTES + W8_BYTES;
  static constexpr uint32_t TMA_BYTES = (FP8 ? W8_BYTES : W_BYTES) + A_BYTES;   // per stage
  static constexpr int STAGES = (int)(98304 / STAGE_BYTES) < 2 ? 2 : (int)(98304 / STAGE_BYTES);
  static constexpr uint32_t TMEM_COLS = NB < 32 ? 32 : NB;
  // + barriers and flags (256 B), row scales [NB], slack
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + NB * 4 + 512 + 16;
  static_assert((size_t)STAGES * STAGE_BYTES >= (size_t)NB * 128 * 4, "partial tile must fit the ring");
};

__device__ __forceinline__ float4 ld_dsmem_v4(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  float4 v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(remote) : "memory");
  return v;
}

// Sum of the S partial tiles P_q[b][n] (q = 0..S-1, in rank order) for the
// batch rows b = rank (mod S) of this CTA, then the fused epilogue.  Warp w
// takes every 4th of those rows, lane l the columns 4l..4l+3 of the tile, so
// every distributed-shared-memory read is 16 bytes and a warp reads 512
// contiguous bytes.  RPB rows per warp are in flight at once (RPB x S reads,
// plus the residual for EPI_RESID), which makes the reduction one or two
// round trips instead of one per row.
template <int S, int EPI, typename TA>
__device__ __forceinline__ void sk_reduce_epilogue(const SkinnyArgs& args, uint32_t psm, const float* r_s,
                                                   int rank, int warp, int lane, int tile, float inv_cap) {
  constexpr int RPB = 16 / S > 8 ? 8 : 16 / S;
  const int c = 4 * lane;
  const int n0 = tile * 128;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  // EPI_QKV: the tile is one head: a query head, one of the n_kv key heads,
  // or one of the n_kv value heads (K/V head g)
  const bool is_v = EPI == EPI_QKV && tile >= args.n_head + args.n_kv;
  const int g = tile < args.n_head ? 0 : (is_v ? tile - args.n_head - args.n_kv : tile - args.n_head);
  for (int b0 = rank + S * warp; b0 < args.B; b0 += 4 * S * RPB) {
    float4 part[RPB][S], xo[RPB];
#pragma unroll
    for (int i = 0; i < RPB; ++i) {
      const int b = b0 + 4 * S * i;
      const bool in = b < args.B;
#pragma unroll
      for (int q = 0; q < S; ++q) part[i][q] = in ? ld_dsmem_v4(psm + (b * 128 + c) * 4, (uint32_t)q) : zero;
      if constexpr (EPI == EPI_RESID)
        xo[i] = in ? *reinterpret_cast<const float4*>(args.x + (size_t)b * args.N + n0 + c) : zero;
    }
#pragma unroll
    for (int i = 0; i < RPB; ++i) {
      const int b = b0 + 4 * S * i;
      if (b >= args.B) break;
      float v[4] = {part[i][0].x, part[i][0].y, part[i][0].z, part[i][0].w};
#pragma unroll
      for (int q = 1; q < S; ++q) {
        v[0] += part[i][q].x;
        v[1] += part[i][q].y;
        v[2] += part[i][q].z;
        v[3] += part[i][q].w;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] *= args.w_scale;    // 1 for bf16 weights (exact)
      if constexpr (EPI != EPI_RESID) {
        const float rb = r_s[b];                     // folded RMSNorm of the input row
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] *= rb;
      }
      if constexpr (EPI == EPI_QKV) {
        // the row's new token sits at its own position (per-row cache lengths)
        const int pos = args.pos_dev[b];
        if (!is_v) {
          const float4 cs = __ldg(reinterpret_cast<const float4*>(args.rope_cos + (size_t)pos * 64 + 4 * (lane & 15)));
          const float4 sn = __ldg(reinterpret_cast<const float4*>(args.rope_sin + (size_t)pos * 64 + 4 * (lane & 15)));
          // QK norm over the head's 128 dims, then RoPE on pairs (j, j + 64):
          // lanes 0..15 hold j = 4l..4l+3, lanes 16..31 their partners
          float ss = v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3];
          ss = warp_sum(ss);
          const float r = rsqrtf(ss * (1.f / 128.f) + args.eps);
          const float c4[4] = {cs.x, cs.y, cs.z, cs.w}, s4[4] = {sn.x, sn.y, sn.z, sn.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float own = v[k] * r;
            const float other = __shfl_xor_sync(0xffffffffu, own, 16);
            v[k] = lane < 16 ? own * c4[k] - other * s4[k] : other * s4[k] + own * c4[k];
          }
        }
        __nv_bfloat16* dst;
        if (tile < args.n_head)
          dst = args.out_bf + (size_t)b * args.n_head * 128 + tile * 128;
        else
          dst = (is_v ? args.v_cache : args.k_cache) + (((size_t)b * args.n_kv + g) * args.cache_S + pos) * 128;
        uint2 pk;
        pk.x = pack_bf16(v[0], v[1]);
        pk.y = pack_bf16(v[2], v[3]);
        *reinterpret_cast<uint2*>(dst + c) = pk;
      } else {
        const size_t o = (size_t)b * args.N + n0 + c;
        if constexpr (EPI == EPI_RESID) {
          const float4 xn = make_float4(xo[i].x + v[0], xo[i].y + v[1], xo[i].z + v[2], xo[i].w + v[3]);
          *reinterpret_cast<float4*>(args.x + o) = xn;
          if (args.h_out) {
            uint2 pk;
            pk.x = pack2<TA>(xn.x, xn.y);
            pk.y = pack2<TA>(xn.z, xn.w);
            *reinterpret_cast<uint2*>(static_cast<TA*>(args.h_out) + o) = pk;
            const float ss = warp_sum(xn.x * xn.x + xn.y * xn.y + xn.z * xn.z + xn.w * xn.w);
            if (lane == 0) args.ss_out[(size_t)tile * args.ss_ld + b] = ss;
          }
        } else if constexpr (EPI == EPI_RELU2) {
          float r[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float t = fmaxf(v[k], 0.f);
            r[k] = t * t;
          }
          uint2 pk;
          pk.x = pack2<TA>(r[0], r[1]);
          pk.y = pack2<TA>(r[2], r[3]);
          *reinterpret_cast<uint2*>(static_cast<TA*>(args.out_act) + o) = pk;
        } else {
          *reinterpret_cast<float4*>(args.x + o) =
              make_float4(softcap_f(v[0], inv_cap, args.softcap), softcap_f(v[1], inv_cap, args.softcap),
                          softcap_f(v[2], inv_cap, args.softcap), softcap_f(v[3], inv_cap, args.softcap));
        }
      }
    }
  }
}

// 16 E4M3 values (one 16-byte chunk) -> 16 f16 values, exactly (every E4M3
// value is an f16 value)
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 v, uint32_t (&h)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    h[2 * i] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
    h[2 * i + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
  }
}
__device__ __forceinline__ uint4 ld_shared_v4u(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}

template <int NB, int EPI, bool FP8>
__global__ void __launch_bounds__(SkCfg<NB, FP8>::THREADS)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                       const SkinnyArgs args) {
  using C = SkCfg<NB, FP8>;
  using TA = typename std::conditional<FP8, __half, __nv_bfloat16>::type;   // activation type
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t sk_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sk_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sW = smem;                                // MMA weight tiles (16-bit)
  uint8_t* sA = smem + STAGES * C::W_BYTES;          // activation tiles
  uint8_t* sW8 = sA + STAGES * C::A_BYTES;           // FP8: E4M3 tiles from the TMA
  uint64_t* bars = reinterpret_cast<uint64_t*>(sW8 + STAGES * C::W8_BYTES);
  // bars: full[STAGES], empty[STAGES], converted[STAGES], done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 1);
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);   // [0] abort
  float* r_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);   // [NB] row scales
  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, CONV = 2 * STAGES, DONE = 3 * STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int n0 = tile * 128;
  const int kb0 = split * args.kb_per;
  const int nkb = args.kb_per;
  const uint64_t limit = args.wait_limit_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);
      mbar_init(bar(EMPTY + s), 1);
      mbar_init(bar(CONV + s), 4);                   // one arrival per converter warp
    }
    mbar_init(bar(DONE), 1);
    flags[0] = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  auto fail = [&]() {
    atomicOr(args.err, NC_DEVFLAG_TIMEOUT);
    flags[0] = 1;
  };
  // the weight tile of a stage as the TMA writes it
  auto w_dst = [&](int s) { return smem_u32(FP8 ? sW8 + s * C::W8_BYTES : sW + s * C::W_BYTES); };

  pdl_trigger();
  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ producer
    // weights do not depend on the previous kernel: the first `pre` weight
    // blocks are requested before waiting for it, their activation blocks after
    int issued[STAGES];
    for (int s = 0; s < STAGES; ++s) issued[s] = -1;
    const int pre = nkb < STAGES ? nkb : STAGES;
    for (int kb = 0; kb < pre; ++kb) {
      mbar_arrive_expect_tx(bar(FULL + kb), C::TMA_BYTES);
      tma_load_2d(w_dst(kb), &tmW, bar(FULL + kb), (kb0 + kb) * 64, n0);
      issued[kb] = 0;
    }
    pdl_wait();
    for (int kb = 0; kb < pre; ++kb)
      tma_load_2d(smem_u32(sA + kb * C::A_BYTES), &tmA, bar(FULL + kb), (kb0 + kb) * 64, 0);
    uint32_t stage = pre == STAGES ? 0 : pre, phase = pre == STAGES ? 1 : 0;
    bool ok = true;
    for (int kb = pre; kb < nkb; ++kb) {
      if (flags[0] || !mbar_wait(bar(EMPTY + stage), phase ^ 1, limit)) {
        if (!flags[0]) fail();
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(bar(FULL + stage), C::TMA_BYTES);
      tma_load_2d(w_dst(stage), &tmW, bar(FULL + stage), (kb0 + kb) * 64, n0);
      tma_load_2d(smem_u32(sA + stage * C::A_BYTES), &tmA, bar(FULL + stage), (kb0 + kb) * 64, 0);
      issued[stage] = (int)phase;
      if (++stage == STAGES) { stage = 0; phase ^= 1; }
    }
    if (!ok)
      for (int s = 0; s < STAGES; ++s)
        if (issued[s] >= 0) mbar_wait(bar(FULL + s), (uint32_t)issued[s], limit);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = FP8 ? idesc_f16_f32(128, NB) : idesc_bf16_f32(128, NB);
    uint32_t stage = 0, phase = 0;
    bool any = false;
    for (int kb = 0; kb < nkb; ++kb) {
      // FP8: the converter warps have widened the stage's weights (they
      // waited for its copies first)
      if (flags[0] || !mbar_wait(bar(FULL + stage), phase, limit) ||
          (FP8 && !mbar_wait(bar(CONV + stage), phase, limit))) {
        if (!flags[0]) fail();
        break;
      }
      tc_fence_after();
      const uint64_t dw = smem_desc_sw128(smem_u32(sW + stage * C::W_BYTES));
      const uint64_t da = smem_desc_sw128(smem_u32(sA + stage * C::A_BYTES));
#pragma unroll
      for (int k = 0; k < 4; ++k)
        tc_mma_f16(tmem_base, desc_add(dw, k * 32), desc_add(da, k * 32), idesc, (kb | k) != 0);
      any = true;
      tc_commit(bar(EMPTY + stage));
      if (++stage == STAGES) { stage = 0; phase ^= 1; }
    }
    // completion of every issued MMA (also the drain on the abort path)
    if (any) tc_commit(bar(DONE));
    else mbar_arrive(bar(DONE));
  } else if (FP8 && warp >= 4) {
    // ------------------------------------------------------- FP8 converters
    // thread = weight row r: its 64 E4M3 bytes (64-byte swizzle: chunk c at
    // c ^ ((r >> 1) & 3)) become 64 f16 (128-byte swizzle: chunk c at c ^ (r & 7))
    const int r = 32 * (warp - 4) + lane;
    uint32_t stage = 0, phase = 0;
    for (int kb = 0; kb < nkb; ++kb) {
      const bool ok = !flags[0] && mbar_wait(bar(FULL + stage), phase, limit);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!flags[0]) fail();
        break;
      }
      const uint32_t w8 = smem_u32(sW8 + stage * C::W8_BYTES) + r * 64;
      const uint32_t w16 = smem_u32(sW + stage * C::W_BYTES) + r * 128;
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t h[8];
        e4m3x16_to_f16(ld_shared_v4u(w8 + ((c8 ^ ((r >> 1) & 3)) << 4)), h);
        st_shared_v4u(w16 + (((2 * c8) ^ (r & 7)) << 4), h[0], h[1], h[2], h[3]);
        st_shared_v4u(w16 + (((2 * c8 + 1) ^ (r & 7)) << 4), h[4], h[5], h[6], h[7]);
      }
      fence_async_smem();                            // the tensor core reads what was written
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(CONV + stage));
      if (++stage == STAGES) { stage = 0; phase ^= 1; }
    }
  }
  __syncwarp();

  // ------------------------------------------------------------- epilogue
  pdl_wait();                                        // x / positions of the previous kernels
  // row scales (all n_ss loads in flight, summed in block order), while the
  // MMAs run
  if (threadIdx.x < NB) {
    float r = 1.f;
    if (args.ss_in && threadIdx.x < args.B) {
      float p[SK_MAX_SS];
#pragma unroll
      for (int i = 0; i < SK_MAX_SS; ++i)
        p[i] = i < args.n_ss ? args.ss_in[(size_t)i * args.ss_ld + threadIdx.x] : 0.f;
      float t = 0.f;
#pragma unroll
      for (int i = 0; i < SK_MAX_SS; ++i) t += p[i];
      r = rsqrtf(t / (float)args.K + args.eps);
    }
    r_s[threadIdx.x] = r;
  }
  if (EPI == EPI_LOGITS && args.len_inc && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x < args.B)
    args.len_inc[threadIdx.x] += 1;                  // every reader of the lengths has finished
  const bool done_ok = mbar_wait(bar(DONE), 0, limit);
  if (!done_ok) fail();
  tc_fence_after();
  const int row = 32 * (warp & 3) + lane;            // weight row n0 + row (warps 0..3)
  const uint32_t taddr = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16);
  // the same decision in every thread: the TMEM loads below are warp-collective;
  // only warps 0..3 (one per TMEM lane quarter) run the epilogue
  const bool run = __syncthreads_and(done_ok) && !flags[0];
  const bool epi = run && warp < 4;
  const float inv_cap = 1.f / args.softcap;

  if (args.splits == 1 && EPI == EPI_LOGITS) {
    if (epi) {
#pragma unroll 1
      for (int c = 0; c < NB; c += 32) {
        float v[32];
        tmem_ld32(taddr + c, v);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c + j < args.B)
            args.x[(size_t)(c + j) * args.N + n0 + row] =
                softcap_f(v[j] * args.w_scale * r_s[c + j], inv_cap, args.softcap);
      }
    }
  } else {
    // this CTA's partial D[n][b] -> own shared memory as P[b][n] (the ring is
    // free: every load has landed and every MMA has read it)
    const uint32_t psm = smem_u32(smem);
    if (epi) {
#pragma unroll 1
      for (int c = 0; c < NB; c += 32) {
        float v[32];
        tmem_ld32(taddr + c, v);
#pragma unroll
        for (int j = 0; j < 32; ++j)
          asm volatile("st.shared.f32 [%0], %1;" ::"r"(psm + ((c + j) * 128 + row) * 4), "f"(v[j]) : "memory");
      }
    }
    cluster_sync_all();                              // every CTA of the tile reaches it once
    if (epi) {
      const int rank = (int)cluster_ctarank();
      switch (args.splits) {
        case 1: sk_reduce_epilogue<1, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        case 2: sk_reduce_epilogue<2, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        case 3: sk_reduce_epilogue<3, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        case 4: sk_reduce_epilogue<4, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        case 5: sk_reduce_epilogue<5, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        case 6: sk_reduce_epilogue<6, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        case 7: sk_reduce_epilogue<7, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
        default: sk_reduce_epilogue<8, EPI, TA>(args, psm, r_s, rank, warp, lane, tile, inv_cap); break;
      }
    }
    cluster_sync_all();                              // remote reads done before any CTA exits
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::TMEM_COLS);
}

}  // namespace nc
