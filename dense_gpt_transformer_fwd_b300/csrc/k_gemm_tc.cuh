// Persistent bf16 GEMM on the 5th-generation tensor cores (sm_103a):
//   acc[m, n] = sum_k A[m, k] * W[n, k]          (A [M, K], W [N, K], both K-major)
// with the consumer of each projection fused into the epilogue.
//
// The projections are the bias-free Linear layers of the nanochat-style GPT
// (yelogs.com nanochat story, "technical details and official Q&A": no bias,
// QK norm, ReLU^2, logit softcap; apidog.com/th "train your own ChatGPT",
// "how nanochat works" item 3: F.linear with the weight in the compute dtype).
//
// Roles inside one CTA (320 threads, one CTA per SM):
//   warp 0        TMA producer: A and W tiles (128 B swizzle) into a ring of
//                 STAGES shared-memory slots, completion on mbarriers
//   warp 1        TMEM owner + MMA issuer: tcgen05.mma kind::f16, M = 128,
//                 N = BN, K = 16 per instruction; two TMEM accumulators so the
//                 epilogue of tile i overlaps the main loop of tile i + 1
//   warps 2..9    epilogue, two warps per TMEM lane quarter (a warp may only
//                 read the 32 TMEM lanes of its quarter, warp % 4), each
//                 owning half of the tile's columns: tcgen05.ld, fused math,
//                 then 32-row x 128-byte chunks staged in a swizzled shared
//                 buffer and written by TMA bulk tensor stores.  With the
//                 RMSNorm folded into the projections, the residual epilogue
//                 reads x (coalesced, through the staging buffer), stores
//                 x + acc, bf16(x + acc) and the rows' sums of squares, and
//                 the next projection scales its rows by 1/rms(x); without
//                 it, x += acc is a TMA reduce-add in L2.
// Tiles are visited m-fastest, so that CTAs resident at the same time share
// the W tile, or n-fastest when the A operand is the larger one (it is then
// read from DRAM once while the W tiles stay in L2).
#pragma once

#include <cuda.h>
#include "nc_common.cuh"

namespace nc {

enum GemmEpi : int {
  EPI_QKV = 0,     // RoPE + QK-norm on q and k heads; q -> Q, k/v -> KV cache
  EPI_RESID = 1,   // x[m, n] += acc                     (fp32 residual stream)
  EPI_RELU2 = 2,   // out = bf16(relu(acc)^2)            (MLP hidden)
  EPI_LOGITS = 3,  // out = cap * tanh(acc / cap)        (fp32 logits)
  EPI_STORE = 4,   // out = acc                          (fp32, tests)
};

struct GemmArgs {
  int M, N, K;
  // EPI_QKV
  __nv_bfloat16* k_cache;         // this layer's K: [B_max][n_kv][S][128]
  __nv_bfloat16* v_cache;         // this layer's V: [B_max][n_kv][S][128]
  const float* rope_cos;          // [S][64]
  const float* rope_sin;          // [S][64]
  const float2* rope_cs_t;        // the same factors dim-major as (cos, sin) pairs: [64][S]
  // K and V caches of all layers as [rows][128] bf16 tensor maps in device
  // memory ([0] K, [1] V; 32 x 64 boxes); this layer's cache row (b, g, pos)
  // of K/V head g is kv_row0 + (b * n_kv + g) * cache_S + pos
  const CUtensorMap* tm_kv;
  long long kv_row0;
  int n_head, n_kv, T, cache_S;
  const int* pos0;                // [B] each row's first position (its cache length before the call)
  __nv_bfloat16* vt;              // optional V^T [B_max * n_kv][128][vt_S] for the prefill attention
  int vt_S;
  float eps;
  // EPI_LOGITS
  float softcap;
  // RMSNorm folded into the projections (the identity (r x) W^T = r (x W^T)):
  // with row_ss, the A operand holds bf16(x) unnormalised and the consumer
  // epilogues (EPI_QKV, EPI_RELU2, EPI_LOGITS) scale accumulator row m by
  // r_m = rsqrt(sum_t row_ss[t * ss_ld + m] * inv_d + eps), the sums of
  // squares of x's column blocks t < ss_blocks.  With h_out, EPI_RESID reads
  // x (x_in, [M][N] fp32), stores x + acc by TMA, and writes bf16(x + acc) to
  // h_out ([M][N]) and each row's sum of squares over every block of BN / 2
  // columns to ss_out[block * ss_ld + m].
  const float* row_ss;
  int ss_blocks, ss_ld;
  float inv_d;
  const float* x_in;
  __nv_bfloat16* h_out;
  float* ss_out;
  // tile order: 0 = m fastest (CTAs running together share a W tile),
  // 1 = n fastest (they share an A panel, each read from DRAM once)
  int n_fast;
  // error reporting
  int* err;
  unsigned long long wait_limit_ns;
};

// CL = 0: one CTA per 128 x BN tile; 2: CTA pairs computing a 256 x BN tile
// with tcgen05.mma.cta_group::2 (each CTA holds its 128 rows of A and half of
// the W tile)
template <int BN, int EPI, int CL = 0>
struct TcCfg {
  // K per pipeline stage: 128 (two 64-column boxes per operand) for CTA pairs,
  // which halves the per-stage barrier and commit work per FLOP
  static constexpr int BM = 128, BK = CL == 2 ? 128 : 64;
  static constexpr int KBOX = BK / 64;                 // 64-column TMA boxes per operand
  static constexpr int EPI_WARPS = 8;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  // the QKV epilogue stages both halves of a head (RoPE pairs dims j, j+64)
  static constexpr int EP_BUFS = EPI == EPI_QKV ? 2 : 1;
  static constexpr uint32_t EP_BUF = 4096;             // 32 rows x 128 B
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = (CL == 2 ? BN / 2 : BN) * BK * 2;   // W rows held by this CTA
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr size_t EP_TOTAL = (size_t)EPI_WARPS * EP_BUFS * EP_BUF;
  static constexpr size_t SMEM_CAP = 232448 - 1024 - 256;
  static constexpr int STAGES_FIT = (int)((SMEM_CAP - EP_TOTAL) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
  // two accumulators of BN columns, allocated as a power of two (>= 32)
  static constexpr uint32_t TMEM_COLS = 2 * BN <= 32 ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  static_assert(BN % 32 == 0 && 2 * BN <= 512, "two accumulators must fit tensor memory");
  static_assert(EPI != EPI_QKV || BN % 256 == 0, "the QKV epilogue takes whole heads per warp");
  static_assert(EPI != EPI_RELU2 || BN % 128 == 0, "the ReLU^2 epilogue works in 64-column chunks");
  static constexpr size_t SMEM = 1024 + STAGES * (size_t)STAGE_BYTES + EP_TOTAL + 256;
  static_assert(STAGES >= 2, "shared memory too small for the pipeline");
  static_assert(SMEM <= 232448, "shared memory over the sm_103a per-block limit");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// softcap = cap * tanh(z / cap) with the single-instruction hardware tanh
// (PTX tanh.approx.f32, one MUFU op; relative error about 2^-11, i.e. at
// most ~7e-3 absolute at the cap of 15).  Saturates to +-cap for large |z|.
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float softcap_f(float z, float inv_cap, float cap) {
  return cap * tanh_approx(z * inv_cap);
}

// Address of 16-byte chunk `cc` (0..7) of row `r` in a 32 x 128 B staging
// buffer with the 128-byte TMA swizzle (chunk index XOR row % 8).
__device__ __forceinline__ uint32_t ep_addr(uint32_t buf, int r, int cc) {
  return buf + r * 128 + ((cc ^ (r & 7)) << 4);
}

// shared -> global tensor reduce-add (x += staged tile, performed in L2)
__device__ __forceinline__ void tma_reduce_add_2d(const void* tmap, uint32_t src, int c0, int c1) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

// ------------------------------------------------- CTA-pair (cta_group::2)
// Tensor memory is allocated and freed collectively by one warp of each CTA
// of the pair; the address is written to each CTA's shared memory.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// TMA load into this CTA's shared memory whose completed bytes are counted on
// an mbarrier of either CTA of the pair (bar is a shared::cluster address)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void* tmap, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// D[256 x N] (+)= A[256 x 16] B[N x 16]^T across the pair: rows 0..127 of A and
// D live in the issuing CTA, rows 128..255 in its peer (same addresses); B's
// first N/2 rows in the issuing CTA, the rest in the peer
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          bar),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local_smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_smem), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

__device__ __forceinline__ void cluster_barrier_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// tmB's box is BN/2 rows x 64 columns.
// CL = 2: launched as clusters of two CTAs along M.  The even CTA (the
// leader) issues tcgen05.mma.cta_group::2 for the 256-row tile of the pair;
// each CTA loads its own 128 rows of A and BN/2 rows of W, and both CTAs'
// loads count on the leader's full barrier.  The
// leader's MMA commits arrive on both CTAs' empty and tfull barriers; both
// CTAs' epilogue warps release an accumulator on the leader's tempty barrier.
// Each CTA now needs 32 KB of shared memory per 64-wide K block instead of
// 48 KB, so the ring holds 6 stages and covers the load latency.
template <int BN, int EPI, int CL = 0>
__global__ void __launch_bounds__(TcCfg<BN, EPI, CL>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const GemmArgs args) {
  static_assert(CL == 0 || CL == 2, "one CTA per tile, or CTA pairs on cta_group::2");
  constexpr bool PAIR = CL == 2;                   // tiles come in vertical pairs
  using C = TcCfg<BN, EPI, CL>;
  constexpr int BM = C::BM, BK = C::BK, STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint8_t* sE = sB + STAGES * C::B_BYTES;                       // epilogue staging buffers
  uint64_t* bars = reinterpret_cast<uint64_t*>(sE + C::EP_TOTAL);
  // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_m = (args.M + BM - 1) / BM;
  const int num_n = args.N / BN;
  // work units: tiles, or (PAIR) pairs of vertically adjacent tiles, m fastest
  const int num_m2 = (num_m + 1) / 2;
  const int rank = PAIR ? (int)(blockIdx.x & 1) : 0;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustride = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int num_units = PAIR ? num_m2 * num_n : num_m * num_n;
  const int num_mu = PAIR ? num_m2 : num_m;          // m positions of a unit
  auto unit_m = [&](int u) { return args.n_fast ? u / num_n : u % num_mu; };
  auto unit_n = [&](int u) { return args.n_fast ? u % num_n : u / num_mu; };
  auto unit_m0 = [&](int u) { return PAIR ? (unit_m(u) * 2 + rank) * BM : unit_m(u) * BM; };
  auto unit_n0 = [&](int u) { return unit_n(u) * BN; };
  const int KB = (args.K + BK - 1) / BK;
  const uint64_t limit = args.wait_limit_ns;

  auto bar = [&](int i) { return smem_u32(bars + i); };
  const int FULL = 0, EMPTY = STAGES, TFULL = 2 * STAGES, TEMPTY = 2 * STAGES + 2,
            DRAIN = 2 * STAGES + 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar(FULL + s), 1);
      mbar_init(bar(EMPTY + s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar(TFULL + a), 1);
      mbar_init(bar(TEMPTY + a), PAIR ? 2 * C::EPI_WARPS : 32 * C::EPI_WARPS);
    }
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
  }
  // Launched as a programmatic dependent of the previous kernel: every
  // thread waits for that kernel's results here, after the set-up above and
  // before taking tensor memory, so that a CTA waiting here never holds TMEM
  // a CTA of the previous kernel on the same SM may still need.
  pdl_trigger();
  pdl_wait();
  if constexpr (PAIR) {
    // the peer's barriers are initialised before any remote arrive or copy
    __syncthreads();
    cluster_barrier_all();
  }
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
    else
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    atomicOr(args.err, NC_DEVFLAG_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued[STAGES];
      for (int s = 0; s < STAGES; ++s) issued[s] = -1;   // parity of an outstanding load
      bool ok = true;
      for (int u = unit0; ok && u < num_units; u += ustride) {
        const int m0 = unit_m0(u), n0 = unit_n0(u);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_test_wait(bar(EMPTY + stage), phase ^ 1) && (*abort_flag || !mbar_wait(bar(EMPTY + stage), phase ^ 1, limit))) {
            if (!*abort_flag) fail();
            ok = false;
            break;
          }
          if constexpr (PAIR) {
            // this CTA's A rows and its half of the W tile; the bytes of both
            // CTAs count on the leader's full barrier, whose one arrival (with
            // the pair's total bytes) is the leader's.  A plain CTA-scope
            // arrive: a cluster-scope release here would wait for this
            // thread's earlier copies and serialise the ring.
            const uint32_t fb = cluster_addr(bar(FULL + stage), 0);
            if (rank == 0) mbar_arrive_expect_tx(bar(FULL + stage), 2 * C::STAGE_BYTES);
#pragma unroll
            for (int h = 0; h < C::KBOX; ++h) {
              tma_load_2d_pair(smem_u32(sA + stage * C::A_BYTES + h * (C::A_BYTES / C::KBOX)), &tmA, fb,
                               kb * BK + 64 * h, m0);
              tma_load_2d_pair(smem_u32(sB + stage * C::B_BYTES + h * (C::B_BYTES / C::KBOX)), &tmB, fb,
                               kb * BK + 64 * h, n0 + rank * (BN / 2));
            }
            issued[stage] = (int)phase;
            if (++stage == STAGES) { stage = 0; phase ^= 1; }
            continue;
          }
          mbar_arrive_expect_tx(bar(FULL + stage), C::STAGE_BYTES);
          tma_load_2d(smem_u32(sA + stage * C::A_BYTES), &tmA, bar(FULL + stage), kb * BK, m0);
          // W boxes are BN/2 rows; the two halves sit back to back in the stage
          tma_load_2d(smem_u32(sB + stage * C::B_BYTES), &tmB, bar(FULL + stage), kb * BK, n0);
          tma_load_2d(smem_u32(sB + stage * C::B_BYTES + C::B_BYTES / 2), &tmB, bar(FULL + stage), kb * BK,
                      n0 + BN / 2);
          issued[stage] = (int)phase;
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      if (!ok && (!PAIR || rank == 0)) {
        // let every copy still in flight land before the CTA exits (in a pair
        // the leader's full barriers also count the peer's copies, and the
        // peer waits for the leader at the final cluster barrier)
        for (int s = 0; s < STAGES; ++s)
          if (issued[s] >= 0) mbar_wait(bar(FULL + s), (uint32_t)issued[s], limit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {
      constexpr uint32_t idesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true, any = false;
      for (int u = unit0; ok && u < num_units; u += ustride, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_test_wait(bar(TEMPTY + acc), acc_phase ^ 1) && (*abort_flag || !mbar_wait(bar(TEMPTY + acc), acc_phase ^ 1, limit))) {
          if (!*abort_flag) fail();
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_test_wait(bar(FULL + stage), phase) && (*abort_flag || !mbar_wait(bar(FULL + stage), phase, limit))) {
            if (!*abort_flag) fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sA + stage * C::A_BYTES);
          const uint32_t b0 = smem_u32(sB + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // 16-column step k: box k / 4 of the stage, 32 bytes per step inside it
            const uint32_t ao = (k >> 2) * (C::A_BYTES / C::KBOX) + (k & 3) * 32;
            const uint32_t bo = (k >> 2) * (C::B_BYTES / C::KBOX) + (k & 3) * 32;
            if constexpr (PAIR)
              tc_mma_f16_pair(d_tmem, smem_desc_sw128(a0 + ao), smem_desc_sw128(b0 + bo), idesc, (kb | k) != 0);
            else
              tc_mma_f16(d_tmem, smem_desc_sw128(a0 + k * 32), smem_desc_sw128(b0 + k * 32), idesc,
                         (kb | k) != 0);
          }
          any = true;
          if constexpr (PAIR)
            tc_commit_pair(bar(EMPTY + stage), (uint16_t)0x3);
          else
            tc_commit(bar(EMPTY + stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (ok) {
          if constexpr (PAIR)
            tc_commit_pair(bar(TFULL + acc), (uint16_t)0x3);
          else
            tc_commit(bar(TFULL + acc));
        }
      }
      if (!ok && any) {
        // every issued MMA must finish before TMEM is released
        if constexpr (PAIR)
          tc_commit_pair(bar(DRAIN), (uint16_t)0x1);
        else
          tc_commit(bar(DRAIN));
        mbar_wait(bar(DRAIN), 0, limit);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = warp - 2;                         // 0..7
    const int q = warp & 3;                         // TMEM lane quarter of this warp
    constexpr int HALF = BN / 2;                    // columns owned by this warp
    const int ch0 = (e >> 2) * HALF;                // first owned column in the tile
    const uint32_t buf0 = smem_u32(sE + e * C::EP_BUFS * C::EP_BUF);
    const float inv_cap = 1.0f / args.softcap;
    // folded RMSNorm: 1 / rms(x) of row r, its block sums added in block order
    auto row_rscale = [&](int r) {
      const float* ssr = args.row_ss + (r < args.M ? r : args.M - 1);
      float t = 0.f;
      for (int bi = 0; bi < args.ss_blocks; ++bi) t += __ldcg(ssr + (size_t)bi * args.ss_ld);
      return rsqrtf(t * args.inv_d + args.eps);
    };
    // The ReLU^2 and logits epilogues request the next unit's block sums at
    // the start of a unit and add them at its end, so that their latency
    // overlaps this unit's work (these epilogues are short next to their
    // loads when K is small).
    constexpr bool SS_AHEAD = EPI == EPI_RELU2 || EPI == EPI_LOGITS;
    constexpr int SS_MAXB = 16;
    const bool ss_ahead = SS_AHEAD && args.row_ss != nullptr && args.ss_blocks <= SS_MAXB;
    float ss_next[SS_AHEAD ? SS_MAXB : 1];
    float rscale_next = 1.f;
    if (ss_ahead && unit0 < num_units) rscale_next = row_rscale(unit_m0(unit0) + 32 * q + lane);
    int local = 0;
    for (int u = unit0; u < num_units; u += ustride, ++local) {
      const int acc = local & 1;
      // the epilogue reads TMEM with warp-collective loads: every lane of the
      // warp leaves or stays together
      const bool full = !*abort_flag && mbar_wait(bar(TFULL + acc), (local >> 1) & 1, limit);
      if (!__all_sync(0xffffffffu, full)) {
        if (!*abort_flag) fail();
        break;
      }
      tc_fence_after();
      const int m0 = unit_m0(u), n0 = unit_n0(u);
      const int row0 = m0 + 32 * q;                 // first row of this warp
      const int my_row = row0 + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * q) << 16) + acc * BN + ch0;
      // folded RMSNorm: this row's 1 / rms(x)
      float rscale = 1.f;
      if constexpr (SS_AHEAD) {
        if (ss_ahead) {
          rscale = rscale_next;
          const int un = u + ustride;
          if (un < num_units) {
            const int rn = unit_m0(un) + 32 * q + lane;
            const float* ssr = args.row_ss + (rn < args.M ? rn : args.M - 1);
#pragma unroll
            for (int bi = 0; bi < SS_MAXB; ++bi)
              ss_next[bi] = bi < args.ss_blocks ? __ldcg(ssr + (size_t)bi * args.ss_ld) : 0.f;
          }
        } else if (args.row_ss != nullptr) {
          rscale = row_rscale(my_row);
        }
      } else if (args.row_ss != nullptr) {
        rscale = row_rscale(my_row);
      }

      if constexpr (EPI == EPI_RESID) {
        if (args.h_out != nullptr) {
          // x = x + acc, read here and stored by TMA; bf16(x) and the row's
          // sum of squares over this warp's 128 columns for the next norm.
          // 32 columns per chunk.  x is read coalesced (8 lanes per 128-byte
          // row, 4 rows per load) one chunk ahead, staged in the swizzled
          // buffer, and read back one row per lane, where the sum is formed
          // in place; bf16(x) is read from there in the coalesced layout
          // again and stored, and the TMA stores the fp32 x.
          // this warp's columns are one norm block of HALF columns
          const bool row_ok = my_row < args.M;
          const int lr = lane >> 3, lp = lane & 7;      // coalesced role: row 4i + lr, 16-byte piece lp
          const float* xw = args.x_in + (size_t)n0 + ch0 + 4 * lp;
          auto load_x = [&](int c, float4 (&xv)[8]) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = row0 + 4 * i + lr;
              xv[i] = r < args.M ? *reinterpret_cast<const float4*>(xw + (size_t)r * args.N + c)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          };
          __nv_bfloat16* hw = args.h_out + (size_t)n0 + ch0 + 4 * lp;
          float4 xc[8], xn[8];
          load_x(0, xc);
          float ss = 0.f;
#pragma unroll
          for (int c = 0; c < HALF; c += 32) {
            if (c + 32 < HALF) load_x(c + 32, xn);
            float v[32];
            tmem_ld32(taddr + c, v);
            if (lane == 0) bulk_wait_read<0>();     // the previous store has read the buffer
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) st_shared_v4(ep_addr(buf0, 4 * i + lr, lp), xc[i].x, xc[i].y, xc[i].z, xc[i].w);
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              const float4 t = ld_shared_v4(ep_addr(buf0, lane, cc));
              v[4 * cc] += t.x;
              v[4 * cc + 1] += t.y;
              v[4 * cc + 2] += t.z;
              v[4 * cc + 3] += t.w;
              st_shared_v4(ep_addr(buf0, lane, cc), v[4 * cc], v[4 * cc + 1], v[4 * cc + 2], v[4 * cc + 3]);
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = row0 + 4 * i + lr;
              const float4 t = ld_shared_v4(ep_addr(buf0, 4 * i + lr, lp));
              if (r < args.M)
                *reinterpret_cast<uint2*>(hw + (size_t)r * args.N + c) =
                    make_uint2(pack_bf16x2(t.x, t.y), pack_bf16x2(t.z, t.w));
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, buf0, n0 + ch0 + c, row0);
              bulk_commit();
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) ss = fmaf(v[j], v[j], ss);
            if (c + 32 < HALF) {
#pragma unroll
              for (int i = 0; i < 8; ++i) xc[i] = xn[i];
            }
          }
          if (row_ok) args.ss_out[(size_t)((n0 + ch0) / HALF) * args.ss_ld + my_row] = ss;
        } else {
          // x += acc as a TMA reduce-add in L2 (x is not read into the SM)
#pragma unroll 1
          for (int c = 0; c < HALF; c += 32) {
            float v[32];
            tmem_ld32(taddr + c, v);
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              st_shared_v4(ep_addr(buf0, lane, cc), v[4 * cc], v[4 * cc + 1], v[4 * cc + 2], v[4 * cc + 3]);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tmC, buf0, n0 + ch0 + c, row0);
              bulk_commit();
            }
          }
        }
      } else if constexpr (EPI == EPI_LOGITS || EPI == EPI_STORE) {
        // 32 fp32 columns per chunk
        const float sc = inv_cap * rscale;
#pragma unroll 1
        for (int c = 0; c < HALF; c += 32) {
          float v[32];
          tmem_ld32(taddr + c, v);
          if constexpr (EPI == EPI_LOGITS) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = args.softcap * tanh_approx(v[j] * sc);
          }
          if (lane == 0) bulk_wait_read<0>();       // the previous store has read the buffer
          __syncwarp();
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            st_shared_v4(ep_addr(buf0, lane, cc), v[4 * cc], v[4 * cc + 1], v[4 * cc + 2], v[4 * cc + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, buf0, n0 + ch0 + c, row0);
            bulk_commit();
          }
        }
      } else if constexpr (EPI == EPI_RELU2) {
        // 64 bf16 columns per chunk
#pragma unroll 1
        for (int c = 0; c < HALF; c += 64) {
          float v0[32], v1[32];
          tmem_ld32(taddr + c, v0);
          tmem_ld32(taddr + c + 32, v1);
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // relu(r z)^2 with the row's norm scale r > 0
            const float a0 = fmaxf(v0[2 * j] * rscale, 0.f), a1 = fmaxf(v0[2 * j + 1] * rscale, 0.f);
            const float b0 = fmaxf(v1[2 * j] * rscale, 0.f), b1 = fmaxf(v1[2 * j + 1] * rscale, 0.f);
            w[j] = pack_bf16x2(a0 * a0, a1 * a1);
            w[16 + j] = pack_bf16x2(b0 * b0, b1 * b1);
          }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            st_shared_v4u(ep_addr(buf0, lane, cc), w[4 * cc], w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, buf0, n0 + ch0 + c, row0);
            bulk_commit();
          }
        }
      } else if constexpr (EPI == EPI_QKV) {
        // BN covers BN/128 whole heads (head_dim 128); each warp owns HALF/128
        // heads.  Columns [0, n_head*128) are query heads, then the n_kv key
        // heads, then the n_kv value heads.  The two halves of a head (dims
        // 0..63, 64..127) go to the warp's two staging buffers.
        const int b_last = (args.M - 1) / args.T;
        const int b = min(my_row / args.T, b_last);     // rows >= M use the last row's start
        const int pos = args.pos0[b] + (my_row - b * args.T);
        const int pos_c = pos < args.cache_S ? pos : args.cache_S - 1;   // rows >= M only
        const uint32_t bufA = buf0, bufB = buf0 + C::EP_BUF;
        // the warp's 32 rows are consecutive positions of one sequence (then
        // the K/V cache rows are consecutive too): TMA stores to the cache
        const int b0w = row0 / args.T;
        const bool kv_tma = args.tm_kv != nullptr && row0 + 32 <= args.M && (row0 + 31) / args.T == b0w;
#pragma unroll 1
        for (int hh = 0; hh < HALF / 128; ++hh) {
          const int head = ((n0 + ch0) >> 7) + hh;
          const bool is_v = head >= args.n_head + args.n_kv;
          // K/V head of a key or value column block
          const int g = head < args.n_head ? 0 : (is_v ? head - args.n_head - args.n_kv : head - args.n_head);
          const uint32_t hbase = taddr + hh * 128;
          // RoPE factors of dims c..c+31 at this row's position from the
          // dim-major tables: for each dim the warp reads 32 consecutive
          // positions (128 contiguous bytes).  Chunk 0's are requested before
          // the QK-norm pass so that their latency overlaps it.
          float rc[32], rs[32];
          auto load_rope = [&](int c) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const float2 t = __ldg(args.rope_cs_t + (size_t)(c + j) * args.cache_S + pos_c);
              rc[j] = t.x;
              rs[j] = t.y;
            }
          };
          // the row's norm scale r, then for q and k heads the QK-norm of
          // r * acc: r * rsqrt(r^2 mean(acc^2) + eps)
          float scale = rscale;
          if (!is_v) {
            load_rope(0);
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
              float v[32];
              tmem_ld32(hbase + c, v);
#pragma unroll
              for (int j = 0; j < 32; ++j) s4[j & 3] = fmaf(v[j], v[j], s4[j & 3]);
            }
            const float ms = ((s4[0] + s4[1]) + (s4[2] + s4[3])) * (1.f / 128.f);
            scale = rscale * rsqrtf(rscale * rscale * ms + args.eps);
          }
          if (lane == 0) bulk_wait_read<0>();       // both buffers free
          __syncwarp();
#pragma unroll 1
          for (int c = 0; c < 64; c += 32) {
            float a[32], bb[32];
            if (!is_v && c > 0) load_rope(c);
            tmem_ld32(hbase + c, a);
            tmem_ld32(hbase + 64 + c, bb);
            if (!is_v) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float x0 = a[j] * scale, x1 = bb[j] * scale;
                a[j] = x0 * rc[j] - x1 * rs[j];
                bb[j] = x0 * rs[j] + x1 * rc[j];
              }
            } else if (args.row_ss != nullptr) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                a[j] *= scale;
                bb[j] *= scale;
              }
            }
            if (is_v && args.vt != nullptr && my_row < args.M) {
              // transposed copy V^T[b][dim][pos]: lanes (consecutive positions)
              // write consecutive addresses for each dim
              __nv_bfloat16* vt = args.vt + (size_t)(b * args.n_kv + g) * 128 * args.vt_S + pos;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                vt[(size_t)(c + j) * args.vt_S] = f2bf(a[j]);
                vt[(size_t)(64 + c + j) * args.vt_S] = f2bf(bb[j]);
              }
            }
            // columns c..c+31 of each half = 16-byte chunks c/8 .. c/8+3
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int cc = (c >> 3) + k;
              st_shared_v4u(ep_addr(bufA, lane, cc), pack_bf16x2(a[8 * k], a[8 * k + 1]),
                            pack_bf16x2(a[8 * k + 2], a[8 * k + 3]), pack_bf16x2(a[8 * k + 4], a[8 * k + 5]),
                            pack_bf16x2(a[8 * k + 6], a[8 * k + 7]));
              st_shared_v4u(ep_addr(bufB, lane, cc), pack_bf16x2(bb[8 * k], bb[8 * k + 1]),
                            pack_bf16x2(bb[8 * k + 2], bb[8 * k + 3]), pack_bf16x2(bb[8 * k + 4], bb[8 * k + 5]),
                            pack_bf16x2(bb[8 * k + 6], bb[8 * k + 7]));
            }
          }
          if (head < args.n_head) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, bufA, head * 128, row0);
              tma_store_2d(&tmC, bufB, head * 128 + 64, row0);
              bulk_commit();
            }
          } else if (kv_tma) {
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              const CUtensorMap* tkv = args.tm_kv + (is_v ? 1 : 0);
              const int crow = (int)(args.kv_row0 + ((long long)b0w * args.n_kv + g) * args.cache_S +
                                     args.pos0[b0w] + (row0 - b0w * args.T));
              tma_store_2d(tkv, bufA, 0, crow);
              tma_store_2d(tkv, bufB, 64, crow);
              bulk_commit();
            }
          } else {
            // key / value rows go to the cache row (b, pos): 256 B per row,
            // lane l writes 32-bit words l and l + 32
            __syncwarp();
#pragma unroll 4
            for (int r = 0; r < 32; ++r) {
              const int m = row0 + r;
              if (m < args.M) {
                const int rb = m / args.T;
                const int rp = args.pos0[rb] + (m - rb * args.T);
                uint32_t* dst = reinterpret_cast<uint32_t*>(
                    (is_v ? args.v_cache : args.k_cache) + (((size_t)rb * args.n_kv + g) * args.cache_S + rp) * 128);
                const uint32_t off = ((lane >> 2) ^ (r & 7)) * 16 + (lane & 3) * 4;
                dst[lane] = ld_shared_u32(bufA + r * 128 + off);
                dst[lane + 32] = ld_shared_u32(bufB + r * 128 + off);
              }
            }
            __syncwarp();
          }
        }
      }
      tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(cluster_addr(bar(TEMPTY + acc), 0));
      } else {
        mbar_arrive(bar(TEMPTY + acc));
      }
      if constexpr (SS_AHEAD) {
        if (ss_ahead && u + ustride < num_units) {
          // the same block order as row_rscale: the same value
          float t = 0.f;
#pragma unroll
          for (int bi = 0; bi < SS_MAXB; ++bi)
            if (bi < args.ss_blocks) t += ss_next[bi];
          rscale_next = rsqrtf(t * args.inv_d + args.eps);
        }
      }
    }
    if (lane == 0) bulk_wait_all();                 // stores done before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // (pair) no CTA leaves while its peer may still signal its barriers or
  // write its tensor memory
  if constexpr (PAIR) cluster_barrier_all();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace nc
