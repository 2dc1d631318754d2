// Causal multi-query attention for the prefill on the 5th-generation tensor
// cores (sm_103a): flash-style, scores S and output O accumulate in TMEM,
// operands are fed by TMA, the online softmax runs one thread per row.
//
// Multi-query attention: every query head reads the single K/V head
// (yelogs.com nanochat story, "technical details and official Q&A"); scale
// 1/sqrt(head_dim) as in SDPA (apidog.com/th "train your own ChatGPT", "how
// nanochat works" item 5); query t attends to keys 0..t.
//
// Grouped-query attention with sliding windows (apidog.com/th item 1): query
// head h reads K/V head h / G, G = n_head / n_kv (G = n_head is multi-query
// attention), and a layer with a window sees only the last `window` keys.
//
// One work item = one batch row, one tile of 128 query positions and TWO
// query heads of one K/V group (tiles "A" and "B"), which share every K and V
// tile it loads (with G odd, the last pair of a group repeats its one head in
// tile B and does not store it).  The kernel is persistent: one CTA per SM
// runs its items one after another with the same barriers, tensor memory and
// K/V ring, and loads the next item's queries while the current item's last
// products run.  The
// queries of row b of a prefill chunk sit at positions p0 .. p0 + T - 1,
// p0 = pos0[b], and read the keys 0 .. p0 + T - 1 of the cache (p0 = 0 for a
// whole prompt; a later chunk continues each row's cache).  Per 128-key
// block j:
//   S_t   = Q_t K_j^T          tcgen05.mma M=128 N=128 K=128   (TMEM, fp32)
//   P_t   = exp2(S_t * c - m)  softmax threads, bf16, back into TMEM over S_t
//   O_t  += P_t V_j            tcgen05.mma M=128 N=128 K=128, A (= P_t) from
//                              TMEM, B (= V_j^T) from shared memory
// TMEM columns: S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512); P_t
// takes the first 64 columns of S_t (two bf16 per column, row r in lane r)
// once the softmax has read S_t.  Keeping P out of shared memory leaves the
// P V product one shared-memory operand instead of two.  The tensor core
// runs the MMAs one thread issues in issue order, so S_t(j+1), issued after
// P_t(j) V_j, overwrites P_t(j) only after that product has read it.
// The running max m is only raised when a block's max exceeds it by more
// than 2^8 (in the exp2 domain); O and the running sum are then rescaled by
// the same thread (it owns that TMEM lane).  The final O / l is exact either
// way, since numerator and denominator share the reference m.
//
// Operands (all K-major bf16 tiles with the 128-byte swizzle, boxes of 64
// columns x 128 rows): Q from the query buffer viewed as [B][T][n_head*128];
// K from this layer's cache [B_max * n_kv][S][128]; V from a transposed copy
// V^T [B_max * n_kv][128][S_vt] that the QKV epilogue writes during the prefill, so
// that P V is again an A * B^T product with B = V^T.  O is staged in the P
// buffer and written by a TMA store into the attention output
// [B][T][n_head*128]; the tensor maps clip rows t >= T.
//
// Warp roles (320 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 2..5 softmax of tile A, warps 6..9 softmax of tile B (warp w
// reads TMEM lanes 32*(w%4) .. +31, i.e. rows of its quarter).  The shared
// memory buffer of each tile stages its output for the TMA store.
// Every mbarrier wait is bounded; on expiry the kernel records
// NC_DEVFLAG_TIMEOUT, lets its copies and MMAs drain, frees TMEM and returns.
#pragma once

#include <cuda.h>
#include "nc_common.cuh"

namespace nc {

struct AttnTcArgs {
  int B, T, n_head, n_qt;          // n_qt = ceil(T / 128)
  int n_kv;                        // K/V heads; query head h reads K/V head h / (n_head / n_kv)
  int window;                      // sliding window (keys p - window + 1 .. p); 0 = unrestricted
  const int* pos0;                 // [B] position of each row's first query (its cache length before the chunk)
  float scale_log2;                // log2(e) / sqrt(head_dim)
  int* err;
  unsigned long long wait_limit_ns;
};

constexpr int ATC_THREADS = 320;
constexpr uint32_t ATC_HALF = 16384;                 // 128 rows x 128 B
constexpr uint32_t ATC_TILE = 2 * ATC_HALF;          // 128 rows x 128 bf16
constexpr uint32_t ATC_OFF_Q = 0;                    // 2 tiles
constexpr uint32_t ATC_OFF_KV = 2 * ATC_TILE;        // ring of 3 slots: K_0 V_0 K_1 V_1 ...
constexpr uint32_t ATC_OFF_P = 5 * ATC_TILE;         // 2 tiles: the output staging of each head
constexpr uint32_t ATC_OFF_BAR = 7 * ATC_TILE;
constexpr size_t ATC_SMEM = 1024 + 7 * (size_t)ATC_TILE + 256;

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 32 lanes x 32 consecutive fp32 columns, registers -> TMEM
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16_2(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}
// D (TMEM) (+)= A B^T with A read from tensor memory (M = 128 lanes, K = 16:
// 8 columns of bf16 pairs) and B from shared memory
__device__ __forceinline__ void tc_mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns, registers -> TMEM
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// byte address of bf16 element (row r, column c) of a 128 x 128 tile stored
// as two K-major 128-byte-swizzled halves (columns 0..63, 64..127)
__device__ __forceinline__ uint32_t atc_addr(uint32_t tile, int r, int c) {
  return tile + (c >> 6) * ATC_HALF + r * 128 + ((((c & 63) >> 3) ^ (r & 7)) << 4) + (c & 7) * 2;
}

// bar.red.or over the `n` threads of named barrier `id`: every thread gets
// the OR of the predicates (a barrier like bar.sync)
__device__ __forceinline__ bool named_bar_or(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

// One work item: a batch row, a tile of 128 query positions and a pair of
// query heads of one K/V group.
struct AtcItem {
  int b, h0, h1, bkv, q0, qpos0, jfirst, nb;
};

__global__ void __launch_bounds__(ATC_THREADS, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ,   // q   [B][T][NQ]
                           const __grid_constant__ CUtensorMap tmK,   // K   [B_max][S][128]
                           const __grid_constant__ CUtensorMap tmVt,  // V^T [B_max][128][S_vt]
                           const __grid_constant__ CUtensorMap tmO,   // att [B][T][NQ]
                           const AttnTcArgs args) {
  extern __shared__ uint8_t atc_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(atc_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s0 = smem_u32(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ATC_OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 18);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(bars + i); };
  // barrier indices
  const int QFULL = 0, KVFULL = 1, KVFREE = 4, SFULL = 7, SFREE = 9, PFULL = 11, PVDONE = 13,
            DRAIN = 15, QFREE = 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.n_head / args.n_kv;             // query heads per K/V head
  const int pg_n = (G + 1) >> 1;                     // head pairs per group
  const int pairs = args.n_kv * pg_n;
  const int per_qt = args.B * pairs;
  const int n_items = args.n_qt * per_qt;
  const uint64_t limit = args.wait_limit_ns;
  // Persistent: CTA c takes the items of rounds k = 0, 1, ...: item
  // k * grid + c, or k * grid + grid - 1 - c in odd rounds (heavy query tiles
  // come first, so the snake order evens out the key blocks per CTA)
  auto item_index = [&](int k) {
    const int G2 = (int)gridDim.x, c = (int)blockIdx.x;
    return k * G2 + ((k & 1) ? G2 - 1 - c : c);
  };
  auto item_of = [&](int w) {
    AtcItem it;
    const int qt = args.n_qt - 1 - w / per_qt;
    const int rest = w % per_qt;
    it.b = rest / pairs;
    const int hp = rest % pairs;
    const int g = hp / pg_n;
    it.h0 = g * G + 2 * (hp % pg_n);                 // tile A's head
    it.h1 = min(it.h0 + 1, g * G + G - 1);           // tile B's head (== h0: not stored)
    it.bkv = it.b * args.n_kv + g;                   // K/V cache sequence
    it.q0 = qt * 128;
    // query row r sits at position qpos0 + r and sees keys max(0, qpos0 + r -
    // window + 1) .. qpos0 + r; the keys of the cache end at pos0 + T - 1
    const int p0 = args.pos0[it.b];
    it.qpos0 = p0 + it.q0;
    const int last_key = min(it.qpos0 + 127, p0 + args.T - 1);
    it.jfirst = args.window > 0 ? max(0, it.qpos0 - args.window + 1) / 128 : 0;
    it.nb = last_key / 128 + 1 - it.jfirst;          // key blocks jfirst .. jfirst + nb - 1
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar(QFULL), 1);
    mbar_init(bar(QFREE), 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(bar(KVFULL + i), 1);
      mbar_init(bar(KVFREE + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(SFULL + i), 1);
      mbar_init(bar(SFREE + i), 128);
      mbar_init(bar(PFULL + i), 128);
      mbar_init(bar(PVDONE + i), 1);
    }
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmVt);
    tma_prefetch_desc(&tmO);
  }
  // programmatic dependent of the QKV projection: wait for its results before
  // taking tensor memory (see the GEMM kernel)
  pdl_trigger();
  pdl_wait();
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto fail = [&]() {
    atomicOr(args.err, NC_DEVFLAG_TIMEOUT);
    *abort_flag = 1;
  };
  auto wait = [&](int i, uint32_t parity) -> bool {
    if (*abort_flag) return false;
    if (mbar_wait(bar(i), parity, limit)) return true;
    fail();
    return false;
  };
  // the softmax warps read TMEM with warp-collective loads: a wait they take
  // ends the same way for every lane of the warp
  auto wait_warp = [&](int i, uint32_t parity) -> bool {
    const bool r = wait(i, parity);
    return __all_sync(0xffffffffu, r);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // per item: Q (once the previous item's S products have read the Q
    // tiles), then K_0, V_0, K_1, V_1, ... round a ring of three slots: ring
    // tile i (counted over all items) uses slot i % 3, so V_{j+1} reuses the
    // slot of K_j (free once both heads' S_j are done) and is in flight long
    // before P V_{j+1} needs it
    if (lane == 0) {
      bool ok = true;
      int inflight[3] = {-1, -1, -1};                // parity of loads in flight
      int q_inflight = -1;
      int kv_i = 0;
      for (int k = 0; ok; ++k) {
        const int w = item_index(k);
        if (w >= n_items) break;
        const AtcItem it = item_of(w);
        if (k > 0 && !wait(QFREE, (k - 1) & 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(QFULL), 2 * ATC_TILE);
        for (int t = 0; t < 2; ++t)
          for (int h = 0; h < 2; ++h)
            tma_load_3d(s0 + ATC_OFF_Q + t * ATC_TILE + h * ATC_HALF, &tmQ, bar(QFULL),
                        (t == 0 ? it.h0 : it.h1) * 128 + 64 * h, it.q0, it.b);
        q_inflight = k & 1;
        for (int i = 0; i < 2 * it.nb; ++i, ++kv_i) {
          const int slot = kv_i % 3, round = kv_i / 3, j = it.jfirst + (i >> 1);
          if (!wait(KVFREE + slot, (round & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(KVFULL + slot), ATC_TILE);
          const uint32_t dst = s0 + ATC_OFF_KV + slot * ATC_TILE;
          for (int h = 0; h < 2; ++h) {
            if ((i & 1) == 0)
              tma_load_3d(dst + h * ATC_HALF, &tmK, bar(KVFULL + slot), 64 * h, j * 128, it.bkv);
            else
              tma_load_3d(dst + h * ATC_HALF, &tmVt, bar(KVFULL + slot), j * 128 + 64 * h, 0, it.bkv);
          }
          inflight[slot] = round & 1;
        }
      }
      if (!ok) {
        // let every copy still in flight land before the CTA exits
        if (q_inflight >= 0) mbar_wait(bar(QFULL), (uint32_t)q_inflight, limit);
        for (int sl = 0; sl < 3; ++sl)
          if (inflight[sl] >= 0) mbar_wait(bar(KVFULL + sl), (uint32_t)inflight[sl], limit);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // per item: S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...  so
    // that the softmax of one head overlaps the tensor-core work of the other
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
      auto issue_s = [&](int t, int ks) {
        const uint64_t dq = smem_desc_sw128(s0 + ATC_OFF_Q + t * ATC_TILE);
        const uint64_t dk = smem_desc_sw128(s0 + ATC_OFF_KV + ks * ATC_TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * ATC_HALF + (kk & 3) * 32;
          tc_mma_f16(tmem_base + t * 128, desc_add(dq, off), desc_add(dk, off), idesc, kk != 0);
        }
        tc_commit(bar(SFULL + t));
      };
      auto issue_pv = [&](int t, int vs, bool first) {
        // P_t in TMEM columns t*128 + 8kk .. +7 for keys 16kk .. 16kk+15
        const uint64_t dv = smem_desc_sw128(s0 + ATC_OFF_KV + vs * ATC_TILE);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * ATC_HALF + (kk & 3) * 32;
          tc_mma_f16_tmem_a(tmem_base + 256 + t * 128, tmem_base + t * 128 + 8 * kk, desc_add(dv, off), idesc,
                            (!first || kk != 0) ? 1u : 0u);
        }
        tc_commit(bar(PVDONE + t));
      };
      // counted over all items: S products issued and P tiles consumed per
      // tile; ring tile kv_base is this item's K_0 (slot i % 3, phase (i / 3) & 1)
      int sn[2] = {0, 0}, pn[2] = {0, 0};
      int kv_base = 0;
      bool ok = true, any = false;
      for (int k = 0; ok; ++k) {
        const int w = item_index(k);
        if (w >= n_items) break;
        const int nb = item_of(w).nb;
        if (!wait(QFULL, k & 1) || !wait(KVFULL + kv_base % 3, (kv_base / 3) & 1)) { ok = false; break; }
        for (int t = 0; ok && t < 2; ++t) {
          // S_t (and P_t over it) free: the softmax has read the previous S_t
          if (sn[t] > 0 && !wait(SFREE + t, (sn[t] - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_s(t, kv_base % 3);
          ++sn[t];
          any = true;
        }
        if (!ok) break;
        tc_commit(bar(KVFREE + kv_base % 3));
        if (nb == 1) tc_commit(bar(QFREE));           // the item's last S products were issued
        for (int j = 0; ok && j < nb; ++j) {
          const bool more = j + 1 < nb;
          const int iv = kv_base + 2 * j + 1, ik = kv_base + 2 * j + 2;
          if (!wait(KVFULL + iv % 3, (iv / 3) & 1)) { ok = false; break; }
          for (int t = 0; ok && t < 2; ++t) {
            if (!wait(PFULL + t, pn[t] & 1)) { ok = false; break; }
            tc_fence_after();
            issue_pv(t, iv % 3, j == 0);
            ++pn[t];
            if (t == 1) tc_commit(bar(KVFREE + iv % 3));
            if (more) {
              if (t == 0 && !wait(KVFULL + ik % 3, (ik / 3) & 1)) { ok = false; break; }
              if (!wait(SFREE + t, (sn[t] - 1) & 1)) { ok = false; break; }
              tc_fence_after();
              issue_s(t, ik % 3);
              ++sn[t];
              if (t == 1) {
                tc_commit(bar(KVFREE + ik % 3));
                if (j + 2 == nb) tc_commit(bar(QFREE));
              }
            }
          }
        }
        kv_base += 2 * nb;
      }
      if (!ok && any) {
        // every issued MMA must finish before TMEM is released
        tc_commit(bar(DRAIN));
        mbar_wait(bar(DRAIN), 0, limit);
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int t = (warp - 2) >> 2;                  // tile: 0 = head h0, 1 = head h1
    const int qd = warp & 3;                        // TMEM lane quarter
    const int r = 32 * qd + lane;                   // row of the tile = query q0 + r
    const uint32_t lane_off = (uint32_t)(32 * qd) << 16;
    const uint32_t tS = tmem_base + lane_off + t * 128;
    const uint32_t tO = tmem_base + lane_off + 256 + t * 128;
    const uint32_t pbuf = s0 + ATC_OFF_P + t * ATC_TILE;  // this head's output staging tile
    const float sl2 = args.scale_log2;
    int sc = 0;                                     // S_t tiles consumed over all items
    bool ok = true;
    for (int k = 0;; ++k) {
      const int w = item_index(k);
      if (w >= n_items) break;
      const AtcItem it = item_of(w);
      float m = -INFINITY;                          // reference max (raw score units)
      float l = 0.f;                                // running sum of exp2((s - m) * sl2)
      for (int j = 0; ok && j < it.nb; ++j, ++sc) {
        if (!wait_warp(SFULL + t, sc & 1)) { ok = false; break; }
        tc_fence_after();
        float v[128];
        tmem_ld128(tS, v);                          // the whole row of S_t
        tc_fence_before();
        mbar_arrive(bar(SFREE + t));                // S_t may be overwritten
        const int jb = it.jfirst + j;               // the key block
        const int lim = it.qpos0 + r - jb * 128;    // last key of the block this row may see
        if (lim < 127) {                            // a diagonal block: later keys are in the future
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) v[c] = -INFINITY;
        }
        if (args.window > 0) {
          const int lo = lim - args.window + 1;     // first key of the block inside the window
          if (lo > 0) {
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c < lo) v[c] = -INFINITY;
          }
        }
        // row max as a tree (8 independent chains of three-input maxima)
        float mk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mk[i] = fmaxf(v[i], v[8 + i]);
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mk[i] = fmax3(mk[i], v[c + i], v[c + 8 + i]);
        const float mx = fmaxf(fmaxf(fmaxf(mk[0], mk[1]), fmaxf(mk[2], mk[3])),
                               fmaxf(fmaxf(mk[4], mk[5]), fmaxf(mk[6], mk[7])));
        bool rescale = false;
        float factor = 1.f;
        if (mx > m && (m == -INFINITY || (mx - m) * sl2 > 8.f)) {
          factor = ex2_approx((m - mx) * sl2);      // 0 when m = -inf
          l *= factor;
          m = mx;
          rescale = j > 0;
        }
        // no key seen yet (a window can mask a whole block of a row): P = 0
        const float mb = m == -INFINITY ? 0.f : m * sl2;
        // the previous P_t V product has finished: P_t and O_t may be written
        if (sc > 0 && !wait_warp(PVDONE + t, (sc - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        // P = exp2(s * sl2 - m * sl2) in bf16, 32 columns at a time into the
        // first half of the row's S_t columns (S_t has been read); row sum in
        // 8 partial sums, kept as 4 pairs (column c goes to partial c % 8)
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nmbx2 = f2_pack(-mb, -mb);
        uint64_t lk2[4] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 128; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 a = f2_unpack(f2_fma(f2_pack(v[c + 2 * i], v[c + 2 * i + 1]), sl2x2, nmbx2));
            const float p0 = ex2_approx(a.x), p1 = ex2_approx(a.y);
            lk2[i & 3] = f2_add(lk2[i & 3], f2_pack(p0, p1));
            pk[i] = pack_bf16_2(p0, p1);
          }
          tmem_st16u(tS + (c >> 1), pk);
        }
        float lk[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 t = f2_unpack(lk2[i]);
          lk[2 * i] = t.x;
          lk[2 * i + 1] = t.y;
        }
        l += ((lk[0] + lk[1]) + (lk[2] + lk[3])) + ((lk[4] + lk[5]) + (lk[6] + lk[7]));
        // tcgen05.ld / tcgen05.st are warp-collective: the whole warp takes the
        // rescale path when any of its rows needs it, each row with its own
        // factor (1 for rows that keep their reference max)
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? factor : 1.f;
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            float o[32];
            tmem_ld32(tO + c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= f;
            tmem_st32(tO + c, o);
          }
        }
        tmem_wait_st();                             // P (and a rescaled O) written
        tc_fence_before();
        mbar_arrive(bar(PFULL + t));
      }
      // ---- the item's output: O / l -> bf16 -> staging tile -> TMA store
      if (ok && !wait_warp(PVDONE + t, (sc - 1) & 1)) ok = false;
      // every thread of the tile meets both barriers once per item; the
      // second one also decides, for all of them alike, whether to go on
      named_bar_sync(1 + t, 128);                   // the previous item's store has read the tile
      if (ok) {
        tc_fence_after();
        const float inv = 1.f / l;
        float v[128];
        tmem_ld128(tO, v);
#pragma unroll
        for (int kq = 0; kq < 16; ++kq)
          st_shared_v4u(atc_addr(pbuf, r, 8 * kq), pack_bf16_2(v[8 * kq] * inv, v[8 * kq + 1] * inv),
                        pack_bf16_2(v[8 * kq + 2] * inv, v[8 * kq + 3] * inv),
                        pack_bf16_2(v[8 * kq + 4] * inv, v[8 * kq + 5] * inv),
                        pack_bf16_2(v[8 * kq + 6] * inv, v[8 * kq + 7] * inv));
        fence_async_smem();
      }
      const bool stop = named_bar_or(1 + t, 128, !ok || *abort_flag);
      if (threadIdx.x == 64 + 128 * t) {
        if (!stop && (t == 0 || it.h1 != it.h0)) {
          const int head = t == 0 ? it.h0 : it.h1;
          tma_store_3d(&tmO, pbuf, head * 128, it.q0, it.b);
          tma_store_3d(&tmO, pbuf + ATC_HALF, head * 128 + 64, it.q0, it.b);
          bulk_commit();
        }
        bulk_wait_read<0>();
      }
      if (stop) break;
    }
    if (threadIdx.x == 64 + 128 * t) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 512);
}

// V^T[s][dim][p] = V[s][p][dim] for the K/V sequences s = b * n_kv + g
// (s < gridDim.y) and p in [0, P_b), P_b = pos0[b]: the transposed value
// operand of the prefill attention for the positions written before the
// current chunk (by an earlier chunk or by decode steps).  One CTA per (64
// positions, sequence): 64 cache rows of 256 B through shared memory, read
// and written with coalesced accesses.  Positions >= P_b are not touched.
__global__ void __launch_bounds__(256) vt_fill_kernel(const __nv_bfloat16* __restrict__ V,
                                                      __nv_bfloat16* __restrict__ vt, int cache_S, int vt_S,
                                                      const int* __restrict__ pos0, int n_kv) {
  __shared__ __align__(16) __nv_bfloat16 tile[64][128 + 8];
  const int b = blockIdx.y, p0 = blockIdx.x * 64;   // b: the K/V sequence
  const int P = pos0[b / n_kv];
  if (p0 >= P) return;
  for (int e = threadIdx.x; e < 64 * 16; e += 256) {
    const int r = e >> 4, c = e & 15;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (p0 + r < P) v = *reinterpret_cast<const uint4*>(V + ((size_t)b * cache_S + p0 + r) * 128 + c * 8);
    *reinterpret_cast<uint4*>(&tile[r][c * 8]) = v;
  }
  __syncthreads();
  __nv_bfloat16* dst = vt + (size_t)b * 128 * vt_S + p0;
  for (int e = threadIdx.x; e < 128 * 32; e += 256) {
    const int d = e >> 5, j = (e & 31) * 2;
    if (p0 + j + 1 < P) {
      __nv_bfloat162 pr;
      pr.x = tile[j][d];
      pr.y = tile[j + 1][d];
      *reinterpret_cast<__nv_bfloat162*>(dst + (size_t)d * vt_S + j) = pr;
    } else if (p0 + j < P) {
      dst[(size_t)d * vt_S + j] = tile[j][d];
    }
  }
}

}  // namespace nc
