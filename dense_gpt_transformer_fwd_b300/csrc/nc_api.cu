// Runtime behind the nc C ABI: model object, weight upload and bf16
// conversion, RoPE table, KV cache, activation workspace, TMA descriptors,
// and the per-call kernel sequence of the forward pass (prefill and decode).
//
// Forward pass, per the nanochat pages (yelogs.com story "technical details and
// official Q&A"; geoz.com.cn "development tricks"; apidog.com/th "how nanochat
// works" items 1, 3, 5, 6):
//   x = rms(E[tok]);  h = rms(x)
//   per layer: [q;k;v] = h Wqkv^T;  q, k <- rms(rope(.)) ;  cache <- k, v
//              x += attn(q, cache) Wo^T;  h = rms(x)
//              x += relu(h Wfc^T)^2 Wproj^T;  h = rms(x)
//   logits = cap * tanh(h Wu^T / cap)
// The 16-bit path folds every h = rms(x) into the projection that consumes
// h: it multiplies its fp32 result by 1/rms(x), and its operand is bf16(x)
// (written, with per-block sums of squares, by the kernel that produced x).
#include "nc.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <type_traits>
#include <utility>
#include <vector>

#include "k_attn_mma.cuh"
#include "k_attn_simt.cuh"
#include "k_attn_tc.cuh"
#include "k_gemm_skinny.cuh"
#include "k_gemm_tc.cuh"
#include "k_rowops.cuh"
#include "k_sample.cuh"
#include "nc_common.cuh"

using namespace nc;

namespace {

constexpr int64_t kGuardElems = 2048;       // sentinel guard before and after each cache
// form of the prefill GEMMs: CTA pairs on tcgen05.mma.cta_group::2 (see launch_gemm_tc)
constexpr int kPrefillCluster = 2;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
// log2(e) / sqrt(128): attention scale folded into the exp2 of the softmax
constexpr float kAttnScaleLog2 = 1.4426950408889634f * 0.08838834764831845f;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool load_encode() {
  if (g_encode) return true;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// 2-D tensor map over a row-major [rows][cols] matrix of bf16 or fp32, box =
// box_cols x box_rows with box_cols * elem = 128 bytes (one swizzle row),
// 128-byte swizzle, zero fill out of bounds.
bool make_tmap(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
               bool f32 = false) {
  if (!load_encode()) return false;
  const uint64_t eb = f32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || (cols * eb) % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * eb};
  cuuint32_t box[2] = {(cuuint32_t)(128 / eb), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(tm, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over a row-major [rows][cols] byte matrix (FP8 E4M3 weights): box
// 64 bytes x box_rows, 64-byte swizzle (chunk c of row r at c ^ ((r >> 1) & 3)).
bool make_tmap8(CUtensorMap* tm, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  if (!load_encode()) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || cols % 16) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D bf16 tensor map, dims/box innermost first, 128-byte swizzle (box[0] =
// 64 elements = one swizzle row), zero fill out of bounds.
bool make_tmap3(CUtensorMap* tm, const void* ptr, const uint64_t dims[3], const uint64_t strides_b[2],
                const uint32_t box[3]) {
  if (!load_encode()) return false;
  if ((reinterpret_cast<uintptr_t>(ptr) & 15) || strides_b[0] % 16 || strides_b[1] % 16) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides_b[0], strides_b[1]};
  cuuint32_t bx[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), d, st, bx, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Where a buffer lives: PTR_HOST (pageable or pinned host memory),
// PTR_DEVICE (memory of device `dev`, or managed memory) or PTR_OTHER_DEVICE
// (device memory of another GPU, which no call accepts).
enum PtrKind { PTR_HOST = 0, PTR_DEVICE = 1, PTR_OTHER_DEVICE = 2 };
PtrKind ptr_kind(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return PTR_HOST;
  }
  if (a.type == cudaMemoryTypeManaged) return PTR_DEVICE;
  if (a.type == cudaMemoryTypeDevice) return a.device == dev ? PTR_DEVICE : PTR_OTHER_DEVICE;
  return PTR_HOST;
}

// last CUDA error this thread turned into NC_ERR_CUDA / NC_ERR_OOM
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

// A failed allocation (or launch configuration) also stays in the runtime's
// per-thread last-error slot, where the next cudaGetLastError() check of a
// later call would find it: clear it here.  Sticky errors (a faulted
// context) cannot be cleared this way and are reported again by later calls.
nc_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return NC_OK;
  g_last_cuda_error = e;
  cudaGetLastError();
  return e == cudaErrorMemoryAllocation ? NC_ERR_OOM : NC_ERR_CUDA;
}

#define NC_TRY(expr)                                  \
  do {                                                \
    cudaError_t e_ = (expr);                          \
    if (e_ != cudaSuccess) return from_cuda(e_);      \
  } while (0)

inline unsigned blocks_for_warps(int64_t warps, int threads = 256) {
  return (unsigned)((warps * 32 + threads - 1) / threads);
}

// The intermediates of one decode step on the decode GEMMs: the fp32
// residual x [rows][d], h = bf16(x) [rows][d], per-128-column sums of squares
// of x ss [d/128][ss_ld], the query q and attention output att [rows][n_head*128],
// the MLP hidden u [rows][d_mlp], and the tensor maps the decode GEMMs read
// h, att and u through (boxes of NB rows x 64 columns).
struct DecodeBufs {
  float* x = nullptr;
  void* h = nullptr;
  void* q = nullptr;
  void* att = nullptr;
  void* u = nullptr;
  float* ss = nullptr;
  int ss_ld = 0;
  CUtensorMap tm_h_nb{}, tm_att_nb{}, tm_u_nb{};
};

// ------------------------------------------------ no-allocation decode scratch
// nc_decode_step_noalloc keeps the decode step's intermediates (a DecodeBufs
// set) in this file-scope device array instead of model memory, so that a
// decode step can run for callers that may not allocate.  Limits: at most
// kNaRows rows, d_model <= kNaD, n_head * 128 <= kNaNQ, d_mlp <= kNaF; the
// array is 4.5 MiB and every GPU that loads the library holds it until the
// process exits.
constexpr int kNaRows = 128, kNaD = 2048, kNaNQ = 2048, kNaF = 8192;
constexpr size_t na_round(size_t b) { return (b + 255) / 256 * 256; }
constexpr size_t kNaOffX = 0;
constexpr size_t kNaOffH = kNaOffX + na_round((size_t)kNaRows * kNaD * 4);
constexpr size_t kNaOffQ = kNaOffH + na_round((size_t)kNaRows * kNaD * 2);
constexpr size_t kNaOffAtt = kNaOffQ + na_round((size_t)kNaRows * kNaNQ * 2);
constexpr size_t kNaOffU = kNaOffAtt + na_round((size_t)kNaRows * kNaNQ * 2);
constexpr size_t kNaOffSS = kNaOffU + na_round((size_t)kNaRows * kNaF * 2);
constexpr size_t kNaBytes = kNaOffSS + na_round((size_t)(kNaD / 128) * kNaRows * 4);
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaBytes];

// Device address of the scratch on device `dev`, which must be current.  In
// host code the array's name is a host-side stand-in, not a device address:
// the address is looked up with cudaGetSymbolAddress once per device (at the
// creation of the first model on it) and cached.
constexpr int kNaMaxDevices = 64;
std::mutex g_na_mutex;
void* g_na_addr[kNaMaxDevices] = {};

cudaError_t noalloc_scratch(int dev, void** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_na_mutex);
  if (!g_na_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_na_addr[dev] = p;
  }
  *out = g_na_addr[dev];
  return cudaSuccess;
}

}  // namespace

struct nc_model {
  nc_config cfg{};
  int device = 0, num_sms = 148;
  bool bf16 = true;
  size_t wbytes = 2;                   // bytes per weight / activation / cache element
  void* weights = nullptr;             // compute dtype, canonical order
  const void* E = nullptr;
  const void* Wu = nullptr;
  std::vector<const void*> wqkv, wo, wfc, wproj;
  float* rope_cos = nullptr;           // [max_seq][hd/2]
  float* rope_sin = nullptr;
  float2* rope_cs_t = nullptr;         // [hd/2][max_seq] (cos, sin): the dim-major copy for the prefill QKV epilogue
  CUtensorMap* d_tm_kv = nullptr;      // device: K and V caches of all layers as [rows][128] bf16
  void* k_alloc = nullptr;             // [guard][L][B_max][S][hd][guard]
  void* v_alloc = nullptr;
  int64_t kv_elems = 0, layer_elems = 0;
  int32_t length = 0, batch = 0;
  int64_t max_rows = 0;
  float* x = nullptr;                  // fp32 residual [max_rows][d]
  void* h = nullptr;                   // GEMM input [max_rows][d]: bf16(x), or rms(x) where no fold applies
  void* q = nullptr;                   // [max_rows][n_head*hd]
  void* att = nullptr;                 // [max_rows][n_head*hd]
  void* u = nullptr;                   // [max_rows][d_mlp]
  float* c32 = nullptr;                // fp32 path: raw QKV [max_rows][(n_head+2)*hd]
  void* h_last = nullptr;              // [max_batch][d]
  float* ss_part = nullptr;            // decode: [d / 128][max_batch] per-block sums of squares of x
  float* ss_rows = nullptr;            // prefill (16-bit models): [d / 96 at most][max_rows] the same per
                                       // row, over blocks of 128 or 96 columns
  int32_t* tok_stage = nullptr;
  float* logit_stage = nullptr;
  size_t logit_stage_bytes = 0;
  int* err = nullptr;
  int64_t launches = 0;
  uint64_t wait_limit_ns = kDefaultWaitNs;
  // per-kernel-class event timing (nc_profile_begin / nc_profile_end)
  struct ProfRec {
    int cls;
    cudaEvent_t a, b;
    int64_t launches;
  };
  bool profiling = false;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<ProfRec> recs;
  // per-row cache lengths: host mirror, and device arrays [max_batch] that the
  // kernels read: the length (decode), the start position of the current
  // call's tokens (prefill) and the index of each row's last token
  std::vector<int32_t> lens;
  int* d_len = nullptr;
  int* d_pos0 = nullptr;
  int* d_last = nullptr;
  // decode-step skinny GEMMs (bf16, B <= sk_nb)
  int sk_nb = 0;                       // padded batch of the MMA N operand: 32, 64 or 128 (0 = off)
  int sk_splits[4] = {1, 1, 1, 1};     // K splits of QKV, O-proj, FC, PROJ
  std::vector<CUtensorMap> tm_w128;    // per layer Wqkv, Wo, Wfc, Wproj, box 64 x 128 rows
  std::vector<CUtensorMap> tm_w96;     // per layer Wo, Wproj, box 64 x 96 rows (192-wide residual tiles;
                                       // empty unless d_model % 192 == 0)
  CUtensorMap tm_wu128{};
  // FP8 models: the projection weights as E4M3 bytes (per layer Wqkv, Wo, Wfc,
  // Wproj, then Wu), one power-of-two scale per matrix, and their tensor maps
  // (box 64 bytes x 128 rows, 64-byte swizzle) for the decode GEMMs; the bf16
  // buffer above holds their exact dequantized image for the prefill
  bool fp8 = false;
  void* w8 = nullptr;
  // later-architecture extras (NC_EXTRA_* bits): their fp32 parameters
  // (the packed tail after Wu) and the buffers they need
  int extras = 0;
  float* ex_params = nullptr;          // device copy of the tail (bf16 models; fp32 models point into weights)
  std::vector<const float*> ve_table, ve_gate;   // per layer (null where no value embedding)
  const float* resid_l = nullptr;      // [L]
  const float* x0_l = nullptr;         // [L]
  const float* smear_w = nullptr;      // [smear_channels]
  const float* smear_lambda = nullptr;
  const float* backout_lambda = nullptr;
  float* x0 = nullptr;                 // [max_rows][d] the residual entering block 0
  float* x_mid = nullptr;              // [max_rows][d] the residual after block L/2 - 1
  int32_t* prev_tok = nullptr;         // [max_batch] each row's last token (smear)
  std::vector<float> w8_scale;
  std::vector<CUtensorMap> tm_w8;
  DecodeBufs dbuf;                     // the decode step's intermediates in the workspace above
  DecodeBufs dbuf_na;                  // the same in the no-allocation scratch (nc_decode_step_noalloc)
  bool noalloc_ok = false;             // the model's shape fits the no-allocation scratch
  // captured decode step
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t g_exec = nullptr;
  int g_B = 0;
  const void* g_tok = nullptr;
  const void* g_logits = nullptr;
  int64_t g_launches = 0;
  void* vt = nullptr;                  // prefill V^T [max_batch][128][vt_S] (bf16)
  int vt_S = 0;
  CUtensorMap tm_vt{};                 // 3-D map over vt, box 64 keys x 128 dims
  std::vector<CUtensorMap> tm_kc;      // per layer 3-D map over the K cache, box 64 x 128 keys
  // A-operand maps (box 64 x 128), epilogue maps (box 128 B x 32); weight maps below
  CUtensorMap tm_h{}, tm_att{}, tm_u{}, tm_hlast{};
  CUtensorMap tm_q_st{}, tm_x_st{}, tm_u_st{};

  void* kc(int l) const { return static_cast<char*>(k_alloc) + (kGuardElems + l * layer_elems) * wbytes; }
  void* vc(int l) const { return static_cast<char*>(v_alloc) + (kGuardElems + l * layer_elems) * wbytes; }
};

namespace {

void free_model(nc_model* m) {
  if (!m) return;
  for (cudaEvent_t e : m->ev_pool) cudaEventDestroy(e);
  if (m->g_exec) cudaGraphExecDestroy(m->g_exec);
  if (m->cap_stream) cudaStreamDestroy(m->cap_stream);
  void* ptrs[] = {m->weights, m->rope_cos, m->rope_sin, m->rope_cs_t, m->d_tm_kv,
                  m->k_alloc, m->v_alloc, m->x,
                  m->h,       m->q,        m->att,      m->u,       m->c32,     m->h_last,
                  m->tok_stage, m->logit_stage, m->err, m->vt, m->d_len, m->d_pos0, m->d_last, m->ss_part, m->ss_rows,
                  m->w8, m->ex_params, m->x0, m->x_mid, m->prev_tok};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  delete m;
}

// FP8 models: every projection matrix (per layer Wqkv, Wo, Wfc, Wproj, then
// Wu) of the fp32 weights `src` (device, canonical order) becomes E4M3 bytes
// in m->w8 with one power-of-two scale per matrix, 2**ceil(log2(amax / 448)),
// and its exact dequantized image replaces the matrix in the bf16 buffer.
cudaError_t quantize_fp8_weights(nc_model* m, const float* src) {
  const nc_config& c = m->cfg;
  const int64_t d = c.d_model, nh = c.n_head, nkv = c.n_kv_head, F = c.d_mlp, V = c.vocab;
  const int64_t NQKV = (nh + 2 * nkv) * 128, NQ = nh * 128;
  std::vector<std::pair<int64_t, int64_t>> mats;         // (element offset, count)
  int64_t off = V * d;                                    // after E
  for (int l = 0; l < c.n_layer; ++l)
    for (int64_t n : {NQKV * d, d * NQ, F * d, d * F}) {
      mats.push_back({off, n});
      off += n;
    }
  mats.push_back({off, V * d});                           // Wu
  int64_t total = 0;
  for (auto& mt : mats) total += mt.second;
  cudaError_t e = cudaMalloc(&m->w8, total);
  if (e != cudaSuccess) return e;
  unsigned int* d_amax = nullptr;
  e = cudaMalloc(&d_amax, mats.size() * sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  std::vector<unsigned int> amax(mats.size());
  e = cudaMemset(d_amax, 0, mats.size() * sizeof(unsigned int));
  for (size_t i = 0; e == cudaSuccess && i < mats.size(); ++i) {
    absmax_kernel<<<2 * m->num_sms, 256>>>(src + mats[i].first, (size_t)mats[i].second, d_amax + i);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpy(amax.data(), d_amax, mats.size() * sizeof(unsigned int), cudaMemcpyDeviceToHost);
  cudaFree(d_amax);
  if (e != cudaSuccess) return e;
  uint8_t* q = static_cast<uint8_t*>(m->w8);
  __nv_bfloat16* img = static_cast<__nv_bfloat16*>(m->weights);
  m->w8_scale.clear();
  for (size_t i = 0; i < mats.size(); ++i) {
    float a;
    std::memcpy(&a, &amax[i], sizeof(a));
    double scale = 1.0;
    if (a > 0.f) {
      int ex = 0;
      const double mant = std::frexp((double)a / 448.0, &ex);   // a / 448 = mant * 2^ex, mant in [0.5, 1)
      scale = std::ldexp(1.0, mant == 0.5 ? ex - 1 : ex);
    }
    m->w8_scale.push_back((float)scale);
    quantize_e4m3_kernel<<<4 * m->num_sms, 256>>>(src + mats[i].first, (size_t)mats[i].second,
                                                  (float)(1.0 / scale), (float)scale, q, img + mats[i].first);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    q += mats[i].second;
  }
  return cudaSuccess;
}

cudaEvent_t next_event(nc_model* m) {
  if (m->ev_used == m->ev_pool.size()) {
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    m->ev_pool.push_back(e);
  }
  return m->ev_pool[m->ev_used++];
}

// Brackets the kernels launched in its lifetime with two events when the
// model is profiling; attributes them to one kernel class.
struct KScope {
  nc_model* m;
  cudaStream_t s;
  size_t rec = SIZE_MAX;
  int64_t l0 = 0;
  KScope(nc_model* m_, int cls, cudaStream_t s_) : m(m_), s(s_) {
    if (!m->profiling) return;
    cudaEvent_t a = next_event(m), b = next_event(m);
    if (!a || !b) return;
    cudaEventRecord(a, s);
    l0 = m->launches;
    rec = m->recs.size();
    m->recs.push_back({cls, a, b, 0});
  }
  ~KScope() {
    if (rec == SIZE_MAX) return;
    cudaEventRecord(m->recs[rec].b, s);
    m->recs[rec].launches = m->launches - l0;
  }
};

nc_status validate(const nc_config* c) {
  if (!c) return NC_ERR_INVALID_ARG;
  if (c->n_layer < 1 || c->d_model < 32 || c->n_head < 1 || c->head_dim < 32 || c->d_mlp < 1 ||
      c->vocab < 1 || c->max_batch < 1 || c->max_seq < 1 || !(c->rope_base > 0.f) ||
      !(c->softcap > 0.f) || !(c->rms_eps >= 0.f) ||
      (c->dtype != NC_F32 && c->dtype != NC_BF16 && c->dtype != NC_FP8))
    return NC_ERR_INVALID_ARG;
  if (c->n_kv_head < 1 || c->n_head % c->n_kv_head || c->window < 0) return NC_ERR_INVALID_ARG;
  if (c->window > 0 && c->n_layer > 64) return NC_ERR_UNSUPPORTED;   // one bit per layer
  if (c->extras & ~NC_EXTRA_ALL) return NC_ERR_INVALID_ARG;
  if ((c->extras & NC_EXTRA_VALUE_EMBED) && (c->ve_gate_channels < 1 || c->ve_gate_channels > c->d_model))
    return NC_ERR_INVALID_ARG;
  if ((c->extras & NC_EXTRA_SMEAR) && (c->smear_channels < 1 || c->smear_channels > c->d_model))
    return NC_ERR_INVALID_ARG;
  if (c->dtype == NC_BF16 || c->dtype == NC_FP8) {
    if (c->head_dim != 128 || c->d_model % 256 || c->d_mlp % 256 || c->vocab % 256 ||
        ((c->n_head + 2 * c->n_kv_head) * 128) % 256 || c->n_head > 16 || c->n_head % 2)
      return NC_ERR_UNSUPPORTED;
  } else {
    if ((c->head_dim != 64 && c->head_dim != 128) || c->d_model % 32) return NC_ERR_UNSUPPORTED;
  }
  return NC_OK;
}

// Launch with programmatic stream serialization when `pdl` is set: the
// kernel may start while the previous kernel in the stream is running and
// waits for it with griddepcontrol.wait (every kernel of the library does).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// Decode attention: the grid.x groups of a row form one thread-block cluster
// (they merge through distributed shared memory); `pdl` as for launch_k.  TO
// is the output (activation) type.
template <typename TO = __nv_bfloat16, typename... Args>
cudaError_t launch_attn_decode(bool pdl, dim3 grid, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(DEC_THREADS, 1, 1);
  cfg.dynamicSmemBytes = ATT_DECODE_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = grid.x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, attn_decode_mma_kernel<TO>, std::forward<Args>(args)...);
}

// Prefill GEMM; tb is a weight map with a box of BN/2 rows.  cl selects the
// form (with at least two M tiles): 0 one CTA per tile, 2 CTA pairs computing
// 256-row tiles with tcgen05.mma.cta_group::2.
template <int BN, int EPI, int CL>
cudaError_t set_gemm_smem() {
  return cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI, CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)TcCfg<BN, EPI, CL>::SMEM);
}

template <int BN, int EPI, int CL>
cudaError_t launch_gemm_cl(nc_model* m, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                           const GemmArgs& a, cudaStream_t s) {
  using C = TcCfg<BN, EPI, CL>;
  const int num_m = (a.M + 127) / 128, num_n = a.N / BN;
  const int units = ((num_m + 1) / 2) * num_n;
  const int pairs = units < m->num_sms / 2 ? units : m->num_sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, EPI, CL>, ta, tb, tc, a);
  m->launches++;
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BN, int EPI>
cudaError_t launch_gemm_tc(nc_model* m, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const GemmArgs& a, cudaStream_t s, int cl = 0) {
  const int num_m = (a.M + 127) / 128, num_n = a.N / BN;
  if (num_m * num_n == 0) return cudaSuccess;
  if (cl == 2 && num_m >= 2) return launch_gemm_cl<BN, EPI, 2>(m, ta, tb, tc, a, s);
  using C = TcCfg<BN, EPI, 0>;
  const int tiles = num_m * num_n;
  const int grid = tiles < m->num_sms ? tiles : m->num_sms;
  const cudaError_t e = launch_k(true, gemm_tc_kernel<BN, EPI, 0>, dim3(grid), dim3(C::THREADS), C::SMEM, s, ta, tb,
                                 tc, a);
  m->launches++;
  return e != cudaSuccess ? e : cudaGetLastError();
}

// K split for a decode-step GEMM with `tiles` weight tiles and `kb` 64-wide
// K blocks: the divisor of kb, at most the portable cluster size 8, that puts
// the CTA count closest to one per SM.
int choose_splits(int tiles, int kb, int sms) {
  int best = 1, best_gap = 1 << 30;
  for (int sp = 1; sp <= kb && sp <= 8; ++sp) {
    if (kb % sp) continue;
    const int gap = std::abs(tiles * sp - sms);
    if (gap < best_gap) {
      best = sp;
      best_gap = gap;
    }
  }
  return best;
}

// Decode attention launch shape: sub-chunks of DEC_SUB keys per CTA (a
// group covers at least DEC_CHUNK keys) chosen for one wave of one CTA per SM
// over the batch (a CTA holds most of an SM's shared memory), at most
// DEC_MAX_GROUPS groups (one cluster) per row; grid.x covers max_seq.  A batch
// of num_sms / 2 rows or more gets one CTA per row, which writes its output
// without a merge.
void decode_attn_shape(const nc_model* m, int B, int window, int* group, int* grid_x) {
  int max_sub = (m->cfg.max_seq + DEC_SUB - 1) / DEC_SUB;
  // a window of W keys spans at most ceil(W / DEC_SUB) + 1 sub-chunks
  if (window > 0) max_sub = std::min(max_sub, (window + DEC_SUB - 1) / DEC_SUB + 1);
  int target = m->num_sms / (B * m->cfg.n_kv_head);    // one CTA per SM over the K/V sequences
  if (target < 1) target = 1;
  if (target > DEC_MAX_GROUPS) target = DEC_MAX_GROUPS;
  int g = (max_sub + target - 1) / target;
  const int min_g = (DEC_CHUNK + DEC_SUB - 1) / DEC_SUB;
  if (g < min_g) g = min_g;
  *group = g;
  *grid_x = (max_sub + g - 1) / g;
}

// Sliding window of layer l: the config's window where bit l of
// window_layers is set, else 0 (the whole causal context).
int layer_window(const nc_model* m, int l) {
  const nc_config& c = m->cfg;
  return (c.window > 0 && l < 64 && ((c.window_layers >> l) & 1ull)) ? c.window : 0;
}

// Tile width of a residual projection (N = d_model columns) on CTA pairs:
// 192 where weight maps for it exist and it finishes in fewer column-time
// units, i.e. ceil(units / pairs) * BN is smaller (the last wave of 256-wide
// tiles can leave most pairs idle: d_model 1536 at 16384 rows is 384 units
// of 256 on 74 pairs, 5.2 waves, against 512 units of 192, 6.9 waves).
int resid_bn(const nc_model* m, int M, int N) {
  const int num_m = (M + 127) / 128;
  if (m->tm_w96.empty() || N % 192 || num_m < 2) return 256;
  const int pairs = m->num_sms / 2, m2 = (num_m + 1) / 2;
  auto cost = [&](int bn) { return (int64_t)((m2 * (N / bn) + pairs - 1) / pairs) * bn; };
  return cost(192) < cost(256) ? 192 : 256;
}

GemmArgs base_args(nc_model* m, int M, int N, int K) {
  GemmArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = M;
  a.N = N;
  a.K = K;
  a.err = m->err;
  a.wait_limit_ns = m->wait_limit_ns;
  a.eps = m->cfg.rms_eps;
  a.softcap = m->cfg.softcap;
  a.n_fast = (int64_t)M * K >= (int64_t)N * K;   // the A operand is at least as large as W
  return a;
}

template <int EPI>
cudaError_t launch_simt_gemm(nc_model* m, const float* A, const float* W, float* out, int M, int N,
                             int K, int ldo, cudaStream_t s) {
  dim3 grid((N + 63) / 64, (M + 63) / 64);
  gemm_simt_f32_kernel<EPI><<<grid, 256, 0, s>>>(A, W, out, M, N, K, ldo, m->cfg.softcap);
  m->launches++;
  return cudaGetLastError();
}

// The whole forward pass over M = B*T rows; row b's tokens sit at positions
// p0_b .. p0_b + T - 1.  A prefill (p0_b = 0 for new sequences, or a later
// chunk continuing each row's cache) reads p0_b from d_pos0 and, for
// last_only, each row's last token index from d_last (both written by
// set_rows before the call); `max_p0` is the largest p0_b.  With `decode`, one
// generic decode step (T = 1, p0_b = the row's length, read from d_len).
nc_status forward(nc_model* m, const int32_t* tok, int B, int T, int max_p0, float* logits,
                  bool last_only, cudaStream_t s, bool decode = false) {
  const nc_config& c = m->cfg;
  const int M = B * T, d = c.d_model, hd = c.head_dim, nh = c.n_head, F = c.d_mlp, V = c.vocab;
  const int nkv = c.n_kv_head;
  const int NQKV = (nh + 2 * nkv) * hd, NQ = nh * hd;
  const float eps = c.rms_eps;
  const int out_rows = last_only ? B : M;
  const bool bf = m->bf16;
  const int* pos0 = decode ? m->d_len : m->d_pos0;    // [B] first position of each row's tokens
  using bf16 = __nv_bfloat16;
  // 16-bit models without the extras fold the RMSNorms into the projections:
  // the embedding kernel and every residual epilogue write h = bf16(x) and
  // the per-128-column sums of squares of x (ss_rows, [d/128][M]), and the
  // next projection scales its rows by 1/rms(x), the unembedding included
  // (last_only: each row's last position of h and its sums are gathered
  // first).  A decode step on this path keeps its final norm kernel, which
  // also advances the rows' lengths.
  const bool fold = bf && !m->extras;
  const bool fold_final = fold && !decode;
  int ss_w = 128;                     // columns per sum-of-squares block of the last writer of h
  auto fold_in = [&](GemmArgs& a) {
    a.row_ss = m->ss_rows;
    a.ss_blocks = d / ss_w;
    a.ss_ld = M;
    a.inv_d = 1.f / (float)d;
  };
  auto fold_out = [&](GemmArgs& a) {
    a.x_in = m->x;
    a.h_out = static_cast<bf16*>(m->h);
    a.ss_out = m->ss_rows;
    a.ss_ld = M;
  };

  CUtensorMap tm_qa[2];  // q and att viewed as [B][T][n_head*128], box 64 x 128 rows
  if (bf && T > 1) {
    const uint64_t dims[3] = {(uint64_t)NQ, (uint64_t)T, (uint64_t)B};
    const uint64_t strides[2] = {(uint64_t)NQ * 2, (uint64_t)T * NQ * 2};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_tmap3(&tm_qa[0], m->q, dims, strides, box) || !make_tmap3(&tm_qa[1], m->att, dims, strides, box))
      return NC_ERR_CUDA;
  }
  {  // x = rms(E[tok]); h = bf16(x) and its sums of squares (folded), or h = rms(x)
    KScope ks(m, NC_K_EMBED, s);
    if (bf)
      embed_rmsnorm_kernel<bf16, bf16><<<blocks_for_warps(M), 256, 0, s>>>(
          tok, static_cast<const bf16*>(m->E), m->x, static_cast<bf16*>(m->h), M, d, V, eps, m->err,
          fold ? m->ss_rows : (float*)nullptr, M);
    else
      embed_rmsnorm_kernel<float, float><<<blocks_for_warps(M), 256, 0, s>>>(
          tok, static_cast<const float*>(m->E), m->x, static_cast<float*>(m->h), M, d, V, eps, m->err,
          (float*)nullptr, 0);
    m->launches++;
    NC_TRY(cudaGetLastError());
  }
  // later-architecture extras (the parameters are fp32 on the device)
  const size_t xn = (size_t)M * d;
  const unsigned ew_blocks = (unsigned)std::min<size_t>((xn + 255) / 256, (size_t)8 * m->num_sms);
  auto renorm = [&]() -> cudaError_t {              // h = rms(x) after x changed
    if (bf)
      rmsnorm_kernel<bf16><<<blocks_for_warps(M), 256, 0, s>>>(m->x, static_cast<bf16*>(m->h), M, d, 1, nullptr,
                                                               eps, nullptr);
    else
      rmsnorm_kernel<float><<<blocks_for_warps(M), 256, 0, s>>>(m->x, static_cast<float*>(m->h), M, d, 1, nullptr,
                                                                eps, nullptr);
    m->launches++;
    return cudaGetLastError();
  };
  if (m->extras) {
    KScope ks(m, NC_K_EMBED, s);
    if (m->extras & NC_EXTRA_SMEAR) {
      // x_t += lambda sigmoid(x_t[:SC] . w) rms(E[previous token]); then the
      // rows' last tokens are kept for the next call
      if (bf)
        smear_kernel<bf16><<<blocks_for_warps(M), 256, 0, s>>>(tok, static_cast<const bf16*>(m->E), m->x, M, T, d,
                                                               V, pos0, m->prev_tok, m->smear_w, m->smear_lambda,
                                                               c.smear_channels, eps);
      else
        smear_kernel<float><<<blocks_for_warps(M), 256, 0, s>>>(tok, static_cast<const float*>(m->E), m->x, M, T,
                                                                d, V, pos0, m->prev_tok, m->smear_w,
                                                                m->smear_lambda, c.smear_channels, eps);
      m->launches++;
      NC_TRY(cudaGetLastError());
      set_prev_tok_kernel<<<1, 256, 0, s>>>(tok, B, T, decode ? nullptr : m->d_last, m->prev_tok);
      m->launches++;
      NC_TRY(cudaGetLastError());
      if (!(m->extras & NC_EXTRA_RESID_LAMBDAS)) NC_TRY(renorm());
    }
    if (m->extras & NC_EXTRA_RESID_LAMBDAS)
      NC_TRY(cudaMemcpyAsync(m->x0, m->x, xn * 4, cudaMemcpyDeviceToDevice, s));
  }
  for (int l = 0; l < c.n_layer; ++l) {
    if (m->extras & NC_EXTRA_RESID_LAMBDAS) {
      // x = resid_l x + x0_l x0 before the block, then its normed input
      KScope ks(m, NC_K_NORM, s);
      lambda_mix_kernel<<<ew_blocks, 256, 0, s>>>(m->x, m->x0, xn, m->resid_l + l, m->x0_l + l);
      m->launches++;
      NC_TRY(cudaGetLastError());
      NC_TRY(renorm());
    }
    if (bf && T > 1 && max_p0 > 0) {
      // a later prefill chunk: the attention's V^T operand of the positions
      // cached before it (the QKV epilogue below writes the chunk's own)
      KScope ks(m, NC_K_ATTN, s);
      vt_fill_kernel<<<dim3((max_p0 + 63) / 64, B * nkv), 256, 0, s>>>(
          static_cast<const bf16*>(m->vc(l)), static_cast<bf16*>(m->vt), c.max_seq, m->vt_S, m->d_pos0, nkv);
      m->launches++;
      NC_TRY(cudaGetLastError());
    }
    {  // [q;k;v] = h Wqkv^T; RoPE + QK-norm; q -> Q, k/v -> cache
      KScope ks(m, NC_K_QKV, s);
      if (bf) {
        GemmArgs a = base_args(m, M, NQKV, d);
        a.k_cache = static_cast<bf16*>(m->kc(l));
        a.v_cache = static_cast<bf16*>(m->vc(l));
        a.rope_cos = m->rope_cos;
        a.rope_sin = m->rope_sin;
        a.rope_cs_t = m->rope_cs_t;
        a.tm_kv = m->d_tm_kv;
        a.kv_row0 = kGuardElems / 128 + (long long)l * c.max_batch * nkv * c.max_seq;
        a.n_head = nh;
        a.n_kv = nkv;
        a.T = T;
        a.pos0 = pos0;
        a.cache_S = c.max_seq;
        if (T > 1) {
          a.vt = static_cast<bf16*>(m->vt);
          a.vt_S = m->vt_S;
        }
        if (fold) fold_in(a);
        NC_TRY((launch_gemm_tc<256, EPI_QKV>(m, m->tm_h, m->tm_w128[4 * l + 0], m->tm_q_st, a, s, kPrefillCluster)));
      } else {
        NC_TRY(launch_simt_gemm<SEPI_STORE>(m, static_cast<const float*>(m->h),
                                            static_cast<const float*>(m->wqkv[l]), m->c32, M, NQKV,
                                            d, NQKV, s));
        qkv_post_kernel<float, float><<<blocks_for_warps((int64_t)M * (nh + 2 * nkv)), 256, 0, s>>>(
            m->c32, static_cast<float*>(m->q), static_cast<float*>(m->kc(l)),
            static_cast<float*>(m->vc(l)), m->rope_cos, m->rope_sin, M, nh, nkv, hd, T, pos0, c.max_seq,
            eps);
        m->launches++;
        NC_TRY(cudaGetLastError());
      }
      if (m->ve_table.size() && m->ve_table[l]) {
        // value embedding: v += 3 sigmoid(h[:C] G^T) VE[tok] in the cache (and V^T)
        const int warps = M * nkv;
        if (bf)
          value_embed_kernel<bf16, bf16><<<blocks_for_warps(warps), 256, 0, s>>>(
              static_cast<const bf16*>(m->h), d, tok, V, m->ve_table[l], m->ve_gate[l], c.ve_gate_channels,
              static_cast<bf16*>(m->vc(l)), T > 1 ? static_cast<bf16*>(m->vt) : nullptr, m->vt_S, M, T, nkv, hd,
              c.max_seq, pos0);
        else
          value_embed_kernel<float, float><<<blocks_for_warps(warps), 256, 0, s>>>(
              static_cast<const float*>(m->h), d, tok, V, m->ve_table[l], m->ve_gate[l], c.ve_gate_channels,
              static_cast<float*>(m->vc(l)), nullptr, 0, M, T, nkv, hd, c.max_seq, pos0);
        m->launches++;
        NC_TRY(cudaGetLastError());
      }
    }
    {  // causal MQA attention over the cache
      KScope ks(m, NC_K_ATTN, s);
      if (bf && T > 1) {
        AttnTcArgs aa;
        aa.B = B;
        aa.T = T;
        aa.pos0 = pos0;
        aa.n_head = nh;
        aa.n_kv = nkv;
        aa.window = layer_window(m, l);
        aa.n_qt = (T + 127) / 128;
        aa.scale_log2 = kAttnScaleLog2;
        aa.err = m->err;
        aa.wait_limit_ns = m->wait_limit_ns;
        // CTAs: query tiles x rows x K/V heads x head pairs of a group
        // persistent: one CTA per SM over the items (query tiles x rows x K/V
        // heads x head pairs of a group)
        const int items = aa.n_qt * B * nkv * ((nh / nkv + 1) / 2);
        NC_TRY(launch_k(true, attn_prefill_tc_kernel, dim3(std::min(items, m->num_sms)), dim3(ATC_THREADS), ATC_SMEM,
                        s, tm_qa[0], m->tm_kc[l], m->tm_vt, tm_qa[1], aa));
        m->launches++;
        NC_TRY(cudaGetLastError());
      } else if (bf) {
        // one position per row (T == 1): row b's context is pos0[b] + 1
        int group = 2, gx = 1;
        const int win = layer_window(m, l);
        decode_attn_shape(m, B, win, &group, &gx);
        NC_TRY(launch_attn_decode(false, dim3(gx, B * nkv), s, static_cast<const bf16*>(m->q),
                                  static_cast<const bf16*>(m->kc(l)), static_cast<const bf16*>(m->vc(l)),
                                  static_cast<bf16*>(m->att), nh, (int)c.max_seq, 0, pos0, kAttnScaleLog2,
                                  group, nkv, win));
        m->launches++;
      } else {
        attn_simt_kernel<float, float><<<blocks_for_warps((int64_t)M * nh), 256, 0, s>>>(
            static_cast<const float*>(m->q), static_cast<const float*>(m->kc(l)),
            static_cast<const float*>(m->vc(l)), static_cast<float*>(m->att), M, nh, nkv, hd, T, pos0,
            c.max_seq, layer_window(m, l));
        m->launches++;
        NC_TRY(cudaGetLastError());
      }
    }
    {  // x += att Wo^T
      KScope ks(m, NC_K_OPROJ, s);
      if (bf) {
        GemmArgs a = base_args(m, M, d, NQ);
        if (fold) fold_out(a);
        if (resid_bn(m, M, d) == 192) {
          NC_TRY((launch_gemm_tc<192, EPI_RESID>(m, m->tm_att, m->tm_w96[2 * l + 0], m->tm_x_st, a, s, kPrefillCluster)));
          ss_w = 96;
        } else {
          NC_TRY((launch_gemm_tc<256, EPI_RESID>(m, m->tm_att, m->tm_w128[4 * l + 1], m->tm_x_st, a, s, kPrefillCluster)));
          ss_w = 128;
        }
      } else {
        NC_TRY(launch_simt_gemm<SEPI_RESID>(m, static_cast<const float*>(m->att),
                                            static_cast<const float*>(m->wo[l]), m->x, M, d, NQ, d, s));
      }
    }
    if (!fold) {  // h = rms(x)
      KScope ks(m, NC_K_NORM, s);
      if (bf)
        rmsnorm_kernel<bf16><<<blocks_for_warps(M), 256, 0, s>>>(m->x, static_cast<bf16*>(m->h), M, d, 1,
                                                                 nullptr, eps, nullptr);
      else
        rmsnorm_kernel<float><<<blocks_for_warps(M), 256, 0, s>>>(m->x, static_cast<float*>(m->h), M, d, 1,
                                                                  nullptr, eps, nullptr);
      m->launches++;
      NC_TRY(cudaGetLastError());
    }
    {  // u = relu(h Wfc^T)^2
      KScope ks(m, NC_K_FC, s);
      if (bf) {
        GemmArgs a = base_args(m, M, F, d);
        if (fold) fold_in(a);
        NC_TRY((launch_gemm_tc<256, EPI_RELU2>(m, m->tm_h, m->tm_w128[4 * l + 2], m->tm_u_st, a, s, kPrefillCluster)));
      } else {
        NC_TRY(launch_simt_gemm<SEPI_RELU2>(m, static_cast<const float*>(m->h),
                                            static_cast<const float*>(m->wfc[l]),
                                            static_cast<float*>(m->u), M, F, d, F, s));
      }
    }
    {  // x += u Wproj^T
      KScope ks(m, NC_K_PROJ, s);
      if (bf) {
        GemmArgs a = base_args(m, M, d, F);
        if (fold) fold_out(a);
        if (resid_bn(m, M, d) == 192) {
          NC_TRY((launch_gemm_tc<192, EPI_RESID>(m, m->tm_u, m->tm_w96[2 * l + 1], m->tm_x_st, a, s, kPrefillCluster)));
          ss_w = 96;
        } else {
          NC_TRY((launch_gemm_tc<256, EPI_RESID>(m, m->tm_u, m->tm_w128[4 * l + 3], m->tm_x_st, a, s, kPrefillCluster)));
          ss_w = 128;
        }
      } else {
        NC_TRY(launch_simt_gemm<SEPI_RESID>(m, static_cast<const float*>(m->u),
                                            static_cast<const float*>(m->wproj[l]), m->x, M, d, F, d, s));
      }
    }
    if (m->extras & NC_EXTRA_BACKOUT) {
      // keep the residual after the first half; subtract it after the last block
      const int mid = c.n_layer / 2 - 1;
      if (l == mid) NC_TRY(cudaMemcpyAsync(m->x_mid, m->x, xn * 4, cudaMemcpyDeviceToDevice, s));
      if (l == c.n_layer - 1 && mid >= 0) {
        KScope ks(m, NC_K_NORM, s);
        backout_kernel<<<ew_blocks, 256, 0, s>>>(m->x, m->x_mid, xn, m->backout_lambda);
        m->launches++;
        NC_TRY(cudaGetLastError());
      }
    }
    if (fold_final && last_only && l == c.n_layer - 1) {
      // the last position of each row: bf16(x) and its sums of squares
      KScope ks(m, NC_K_NORM, s);
      gather_last_kernel<bf16><<<blocks_for_warps(B), 256, 0, s>>>(
          static_cast<const bf16*>(m->h), m->ss_rows, M, d / ss_w, static_cast<bf16*>(m->h_last), m->ss_part, B, B,
          d, T, m->d_last);
      m->launches++;
      NC_TRY(cudaGetLastError());
    }
    if (!fold || (l == c.n_layer - 1 && !fold_final)) {
      // h = rms(x): next block's pre-attention norm, or the final norm
      KScope ks(m, NC_K_NORM, s);
      const bool final_last = last_only && l == c.n_layer - 1;
      const int rows = final_last ? B : M;
      void* dst = final_last ? m->h_last : m->h;
      // a decode step on this generic path advances the device-side length in
      // its final norm
      int* len_inc = (decode && l == c.n_layer - 1) ? m->d_len : nullptr;
      const int* last = final_last ? m->d_last : nullptr;
      if (bf)
        rmsnorm_kernel<bf16><<<blocks_for_warps(rows), 256, 0, s>>>(
            m->x, static_cast<bf16*>(dst), rows, d, final_last ? T : 1, last, eps, len_inc);
      else
        rmsnorm_kernel<float><<<blocks_for_warps(rows), 256, 0, s>>>(
            m->x, static_cast<float*>(dst), rows, d, final_last ? T : 1, last, eps, len_inc);
      m->launches++;
      NC_TRY(cudaGetLastError());
    }
  }
  {  // logits = cap * tanh(h Wu^T / cap)
    KScope ks(m, NC_K_LMHEAD, s);
    if (bf) {
      GemmArgs a = base_args(m, out_rows, V, d);
      if (fold_final) {
        fold_in(a);
        if (last_only) {
          a.row_ss = m->ss_part;
          a.ss_ld = B;
        }
      }
      CUtensorMap tm_out;
      if (!make_tmap(&tm_out, logits, out_rows, V, 32, true)) return NC_ERR_INVALID_ARG;
      NC_TRY((launch_gemm_tc<256, EPI_LOGITS>(m, last_only ? m->tm_hlast : m->tm_h, m->tm_wu128, tm_out, a, s, kPrefillCluster)));
    } else {
      NC_TRY(launch_simt_gemm<SEPI_LOGITS>(
          m, static_cast<const float*>(last_only ? m->h_last : m->h),
          static_cast<const float*>(m->Wu), logits, out_rows, V, d, V, s));
    }
  }
  return NC_OK;
}

template <int NB, int EPI, bool FP8>
cudaError_t launch_skinny(nc_model* m, const CUtensorMap& tw, const CUtensorMap& ta, SkinnyArgs a, int tiles,
                          cudaStream_t s) {
  using C = SkCfg<NB, FP8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, a.splits, 1);
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = a.splits;   // the K splits of one tile form a cluster
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, gemm_skinny_kernel<NB, EPI, FP8>, tw, ta, a);
  m->launches++;
  return e != cudaSuccess ? e : cudaGetLastError();
}

SkinnyArgs skinny_args(nc_model* m, int B, int N, int K, int splits) {
  SkinnyArgs a;
  std::memset(&a, 0, sizeof(a));
  a.B = B;
  a.N = N;
  a.K = K;
  a.splits = splits;
  a.kb_per = K / 64 / splits;
  a.eps = m->cfg.rms_eps;
  a.softcap = m->cfg.softcap;
  a.err = m->err;
  a.wait_limit_ns = m->wait_limit_ns;
  a.w_scale = 1.f;
  return a;
}

// One decode step of the bf16 model for B <= NB rows on the skinny GEMMs.
// Every kernel takes the position from the device-side length, so the
// sequence is the same at every step and can be replayed as a CUDA graph.
template <int NB, bool FP8>
nc_status forward_decode_nb(nc_model* m, const DecodeBufs& db, const int32_t* tok, int B, float* logits,
                            cudaStream_t s) {
  const nc_config& c = m->cfg;
  const int d = c.d_model, nh = c.n_head, F = c.d_mlp, V = c.vocab;
  const int nkv = c.n_kv_head;
  const int NQKV = (nh + 2 * nkv) * 128, NQ = nh * 128;
  const float eps = c.rms_eps;
  using bf16 = __nv_bfloat16;
  // the decode GEMMs' activations: bf16, or f16 with FP8 weights (the tensor
  // core takes the same type for both operands)
  using TA = typename std::conditional<FP8, __half, bf16>::type;
  // weight map and scale of matrix g (0 Wqkv, 1 Wo, 2 Wfc, 3 Wproj) of layer l
  auto wmap = [&](int l, int g) -> const CUtensorMap& { return FP8 ? m->tm_w8[4 * l + g] : m->tm_w128[4 * l + g]; };
  auto wscale = [&](int l, int g) { return FP8 ? m->w8_scale[4 * l + g] : 1.f; };
  // RMSNorm folded into the projections: every residual update writes
  // h = TA(x) and per-block sums of squares; QKV, MLP up and lm_head scale
  // their rows by 1/rms(x) (r (x W^T) = (r x) W^T)
  const int ss_ld = db.ss_ld, n_ss = d / 128;
  auto fold_in = [&](SkinnyArgs& a) {
    a.ss_in = db.ss;
    a.n_ss = n_ss;
    a.ss_ld = ss_ld;
  };
  auto fold_out = [&](SkinnyArgs& a) {
    a.h_out = db.h;
    a.ss_out = db.ss;
    a.ss_ld = ss_ld;
  };
  {
    KScope ks(m, NC_K_EMBED, s);
    embed_rmsnorm_kernel<bf16, TA><<<blocks_for_warps(B), 256, 0, s>>>(
        tok, static_cast<const bf16*>(m->E), db.x, static_cast<TA*>(db.h), B, d, V, eps, m->err, db.ss, ss_ld);
    m->launches++;
    NC_TRY(cudaGetLastError());
  }
  for (int l = 0; l < c.n_layer; ++l) {
    {
      KScope ks(m, NC_K_QKV, s);
      SkinnyArgs a = skinny_args(m, B, NQKV, d, m->sk_splits[0]);
      a.out_bf = static_cast<bf16*>(db.q);
      a.k_cache = static_cast<bf16*>(m->kc(l));
      a.v_cache = static_cast<bf16*>(m->vc(l));
      a.rope_cos = m->rope_cos;
      a.rope_sin = m->rope_sin;
      a.pos_dev = m->d_len;
      a.n_head = nh;
      a.n_kv = nkv;
      a.cache_S = c.max_seq;
      a.w_scale = wscale(l, 0);
      fold_in(a);
      NC_TRY((launch_skinny<NB, EPI_QKV, FP8>(m, wmap(l, 0), db.tm_h_nb, a, NQKV / 128, s)));
    }
    {
      KScope ks(m, NC_K_ATTN, s);
      int group = 2, gx = 1;
      const int win = layer_window(m, l);
      decode_attn_shape(m, B, win, &group, &gx);
      NC_TRY(launch_attn_decode<TA>(true, dim3(gx, B * nkv), s, static_cast<const bf16*>(db.q),
                                    static_cast<const bf16*>(m->kc(l)), static_cast<const bf16*>(m->vc(l)),
                                    static_cast<TA*>(db.att), nh, (int)c.max_seq, 0,
                                    static_cast<const int*>(m->d_len), kAttnScaleLog2, group, nkv, win));
      m->launches++;
    }
    {
      KScope ks(m, NC_K_OPROJ, s);
      SkinnyArgs a = skinny_args(m, B, d, NQ, m->sk_splits[1]);
      a.x = db.x;
      a.w_scale = wscale(l, 1);
      fold_out(a);
      NC_TRY((launch_skinny<NB, EPI_RESID, FP8>(m, wmap(l, 1), db.tm_att_nb, a, d / 128, s)));
    }
    {
      KScope ks(m, NC_K_FC, s);
      SkinnyArgs a = skinny_args(m, B, F, d, m->sk_splits[2]);
      a.out_act = db.u;
      a.w_scale = wscale(l, 2);
      fold_in(a);
      NC_TRY((launch_skinny<NB, EPI_RELU2, FP8>(m, wmap(l, 2), db.tm_h_nb, a, F / 128, s)));
    }
    {
      KScope ks(m, NC_K_PROJ, s);
      SkinnyArgs a = skinny_args(m, B, d, F, m->sk_splits[3]);
      a.x = db.x;
      a.w_scale = wscale(l, 3);
      fold_out(a);
      NC_TRY((launch_skinny<NB, EPI_RESID, FP8>(m, wmap(l, 3), db.tm_u_nb, a, d / 128, s)));
    }
  }
  {
    KScope ks(m, NC_K_LMHEAD, s);
    SkinnyArgs a = skinny_args(m, B, V, d, 1);
    a.x = logits;
    fold_in(a);
    a.len_inc = m->d_len;                            // the step's last kernel
    a.w_scale = FP8 ? m->w8_scale[4 * c.n_layer] : 1.f;
    NC_TRY((launch_skinny<NB, EPI_LOGITS, FP8>(m, FP8 ? m->tm_w8[4 * c.n_layer] : m->tm_wu128, db.tm_h_nb, a,
                                               V / 128, s)));
  }
  return NC_OK;
}

// Every kernel a model can launch is loaded and given its dynamic shared
// memory limit here, on the model's device, when the model is created.  The
// CUDA runtime loads kernels lazily and function attributes are per device,
// so no later call loads a module or sets an attribute (a first launch could
// otherwise allocate device memory inside a call).
template <int EPI>
cudaError_t configure_gemm_tc() {
  cudaError_t e = set_gemm_smem<256, EPI, 0>();
  if (e == cudaSuccess) e = set_gemm_smem<256, EPI, 2>();
  if (e == cudaSuccess && EPI == EPI_RESID) e = set_gemm_smem<192, EPI_RESID, 0>();
  if (e == cudaSuccess && EPI == EPI_RESID) e = set_gemm_smem<192, EPI_RESID, 2>();
  return e;
}
template <int NB, bool FP8>
cudaError_t configure_skinny() {
  const int sm = (int)SkCfg<NB, FP8>::SMEM;
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<NB, EPI_QKV, FP8>, a, sm);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_skinny_kernel<NB, EPI_RESID, FP8>, a, sm);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_skinny_kernel<NB, EPI_RELU2, FP8>, a, sm);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(gemm_skinny_kernel<NB, EPI_LOGITS, FP8>, a, sm);
  return e;
}
template <typename K>
cudaError_t load_kernel(K* k) {
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, k);
}

cudaError_t configure_kernels(const nc_model* m) {
  using bf16 = __nv_bfloat16;
  cudaError_t e = cudaSuccess;
  auto step = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
  };
  if (m->bf16) {
    step(configure_gemm_tc<EPI_QKV>());
    step(configure_gemm_tc<EPI_RESID>());
    step(configure_gemm_tc<EPI_RELU2>());
    step(configure_gemm_tc<EPI_LOGITS>());
    step(configure_gemm_tc<EPI_STORE>());
    if (m->fp8) {
      step(configure_skinny<32, true>());
      step(configure_skinny<64, true>());
      step(configure_skinny<128, true>());
      step(cudaFuncSetAttribute(attn_decode_mma_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)ATT_DECODE_SMEM));
      step(load_kernel(embed_rmsnorm_kernel<bf16, __half>));
      step(load_kernel(absmax_kernel));
      step(load_kernel(quantize_e4m3_kernel));
    }
    step(configure_skinny<32, false>());
    step(configure_skinny<64, false>());
    step(configure_skinny<128, false>());
    step(cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)ATC_SMEM));
    step(cudaFuncSetAttribute(attn_decode_mma_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)ATT_DECODE_SMEM));
    step(load_kernel(embed_rmsnorm_kernel<bf16, bf16>));
    step(load_kernel(rmsnorm_kernel<bf16>));
    step(load_kernel(vt_fill_kernel));
    step(load_kernel(set_rows_kernel));
  } else {
    step(load_kernel(gemm_simt_f32_kernel<SEPI_STORE>));
    step(load_kernel(gemm_simt_f32_kernel<SEPI_RESID>));
    step(load_kernel(gemm_simt_f32_kernel<SEPI_RELU2>));
    step(load_kernel(gemm_simt_f32_kernel<SEPI_LOGITS>));
    step(load_kernel(qkv_post_kernel<float, float>));
    step(load_kernel(attn_simt_kernel<float, float>));
    step(load_kernel(embed_rmsnorm_kernel<float, float>));
    step(load_kernel(rmsnorm_kernel<float>));
    step(load_kernel(set_rows_kernel));
  }
  step(load_kernel(sample_kernel));
  step(load_kernel(kv_clone_kernel));
  if (m->extras) {
    step(load_kernel(smear_kernel<__nv_bfloat16>));
    step(load_kernel(smear_kernel<float>));
    step(load_kernel(lambda_mix_kernel));
    step(load_kernel(backout_kernel));
    step(load_kernel(value_embed_kernel<__nv_bfloat16, __nv_bfloat16>));
    step(load_kernel(value_embed_kernel<float, float>));
    step(load_kernel(set_prev_tok_kernel));
  }
  return e;
}

// the decode GEMMs fold the RMSNorms into their epilogues; models with the
// later-architecture extras decode on the generic one-position pass
bool decode_on_skinny(const nc_model* m, int B) {
  return m->bf16 && m->sk_nb > 0 && B <= m->sk_nb && m->extras == 0;
}

nc_status forward_decode(nc_model* m, const int32_t* tok, int B, float* logits, cudaStream_t s,
                         const DecodeBufs* db = nullptr) {
  if (!decode_on_skinny(m, B)) return forward(m, tok, B, 1, 0, logits, false, s, true);
  const DecodeBufs& b = db ? *db : m->dbuf;
  if (m->fp8) {
    switch (m->sk_nb) {
      case 32: return forward_decode_nb<32, true>(m, b, tok, B, logits, s);
      case 64: return forward_decode_nb<64, true>(m, b, tok, B, logits, s);
      default: return forward_decode_nb<128, true>(m, b, tok, B, logits, s);
    }
  }
  switch (m->sk_nb) {
    case 32: return forward_decode_nb<32, false>(m, b, tok, B, logits, s);
    case 64: return forward_decode_nb<64, false>(m, b, tok, B, logits, s);
    default: return forward_decode_nb<128, false>(m, b, tok, B, logits, s);
  }
}

// Decode step through a CUDA graph of the whole step.  The first step with a
// given (B, logit buffer) runs eagerly; the second captures the
// step on a model-owned stream; every step is then one graph launch on the
// caller's stream.  Profiling runs the step eagerly.
nc_status decode_graph(nc_model* m, const int32_t* tok, int B, float* logits, cudaStream_t s) {
  if (!decode_on_skinny(m, B) || m->profiling) return forward_decode(m, tok, B, logits, s);
  // the graph reads the tokens from the model's staging buffer
  if (tok != m->tok_stage) {
    NC_TRY(cudaMemcpyAsync(m->tok_stage, tok, (size_t)B * 4, cudaMemcpyDeviceToDevice, s));
    tok = m->tok_stage;
  }
  const bool same = m->g_B == B && m->g_tok == tok && m->g_logits == logits;
  if (!same) {
    if (m->g_exec) {
      cudaGraphExecDestroy(m->g_exec);
      m->g_exec = nullptr;
    }
    m->g_B = B;
    m->g_tok = tok;
    m->g_logits = logits;
    return forward_decode(m, tok, B, logits, s);
  }
  if (!m->g_exec) {
    if (!m->cap_stream) NC_TRY(cudaStreamCreateWithFlags(&m->cap_stream, cudaStreamNonBlocking));
    const int64_t l0 = m->launches;
    NC_TRY(cudaStreamBeginCapture(m->cap_stream, cudaStreamCaptureModeThreadLocal));
    nc_status st = forward_decode(m, tok, B, logits, m->cap_stream);
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(m->cap_stream, &g);
    m->g_launches = m->launches - l0;
    m->launches = l0;
    if (st != NC_OK) {
      if (g) cudaGraphDestroy(g);
      return st;
    }
    if (e != cudaSuccess) return from_cuda(e);
    e = cudaGraphInstantiate(&m->g_exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
      m->g_exec = nullptr;
      return from_cuda(e);
    }
  }
  NC_TRY(cudaGraphLaunch(m->g_exec, s));
  m->launches += m->g_launches;
  return NC_OK;
}

// Resolve the token and logit buffers to device memory, staging host buffers.
nc_status run_call(nc_model* m, const int32_t* tokens, int B, int T, int max_p0, float* logits,
                   bool last_only, cudaStream_t s, bool decode) {
  const int M = B * T;
  const PtrKind tk = ptr_kind(tokens, m->device), lk = ptr_kind(logits, m->device);
  if (tk == PTR_OTHER_DEVICE || lk == PTR_OTHER_DEVICE) return NC_ERR_INVALID_ARG;
  const int32_t* tok_dev = tokens;
  if (tk == PTR_HOST) {
    NC_TRY(cudaMemcpyAsync(m->tok_stage, tokens, (size_t)M * 4, cudaMemcpyHostToDevice, s));
    tok_dev = m->tok_stage;
  }
  const size_t out_bytes = (size_t)(last_only ? B : M) * m->cfg.vocab * 4;
  float* out_dev = logits;
  const bool host_out = lk == PTR_HOST;
  if (host_out) {
    if (m->logit_stage_bytes < out_bytes) {
      NC_TRY(cudaStreamSynchronize(s));
      if (m->logit_stage) cudaFree(m->logit_stage);
      m->logit_stage = nullptr;
      m->logit_stage_bytes = 0;
      NC_TRY(cudaMalloc(&m->logit_stage, out_bytes));
      m->logit_stage_bytes = out_bytes;
    }
    out_dev = m->logit_stage;
  }
  nc_status st = decode ? decode_graph(m, tok_dev, B, out_dev, s)
                        : forward(m, tok_dev, B, T, max_p0, out_dev, last_only, s);
  if (st != NC_OK) return st;
  if (host_out) NC_TRY(cudaMemcpyAsync(logits, out_dev, out_bytes, cudaMemcpyDeviceToHost, s));
  return NC_OK;
}

__global__ void wait_nothing_kernel(int* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(smem_u32(&bar), 0, limit_ns)) atomicOr(err, NC_DEVFLAG_TIMEOUT);
}

}  // namespace

extern "C" {

const char* nc_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no error" : cudaGetErrorString(g_last_cuda_error);
}

const char* nc_status_string(nc_status s) {
  switch (s) {
    case NC_OK: return "ok";
    case NC_ERR_INVALID_ARG: return "invalid argument";
    case NC_ERR_UNSUPPORTED: return "unsupported configuration";
    case NC_ERR_OOM: return "out of device memory";
    case NC_ERR_STATE: return "invalid state for this call";
    case NC_ERR_CAPACITY: return "KV cache full";
    case NC_ERR_TOKEN: return "token id out of range";
    case NC_ERR_TIMEOUT: return "device wait timed out";
    case NC_ERR_CUDA: return "CUDA error";
    case NC_ERR_SCRATCH_LIMIT: return "beyond the no-allocation decode scratch (rows, widths or model type)";
  }
  return "unknown status";
}

nc_status nc_model_create(const nc_config* cfg, const float* weights, nc_model** out) {
  if (!out) return NC_ERR_INVALID_ARG;
  *out = nullptr;
  nc_status st = validate(cfg);
  if (st != NC_OK) return st;
  if (!weights) return NC_ERR_INVALID_ARG;
  nc_model* m = new (std::nothrow) nc_model();
  if (!m) return NC_ERR_OOM;
  m->cfg = *cfg;
  m->bf16 = cfg->dtype == NC_BF16 || cfg->dtype == NC_FP8;   // FP8: bf16 compute, FP8 decode weights
  m->fp8 = cfg->dtype == NC_FP8;
  m->wbytes = m->bf16 ? 2 : 4;
  const nc_config& c = m->cfg;
  const int64_t d = c.d_model, hd = c.head_dim, nh = c.n_head, F = c.d_mlp, V = c.vocab;
  const int64_t nkv = c.n_kv_head;
  const int64_t NQKV = (nh + 2 * nkv) * hd, NQ = nh * hd;
  const int64_t layer_params = NQKV * d + d * NQ + F * d + d * F;
  const int64_t n_params = 2 * V * d + c.n_layer * layer_params;   // E, the blocks, Wu
  // the extras' parameters follow Wu: value-embedding tables of the even
  // layers [V][n_kv * hd], their gates [n_kv][C]; residual and x0 lambdas [L]
  // each; smear gate [SC] and lambda; backout lambda
  const int n_ve = (cfg->extras & NC_EXTRA_VALUE_EMBED) ? (c.n_layer + 1) / 2 : 0;
  const int64_t n_extra = n_ve * (V * nkv * hd + nkv * (int64_t)c.ve_gate_channels) +
                          ((cfg->extras & NC_EXTRA_RESID_LAMBDAS) ? 2 * c.n_layer : 0) +
                          ((cfg->extras & NC_EXTRA_SMEAR) ? c.smear_channels + 1 : 0) +
                          ((cfg->extras & NC_EXTRA_BACKOUT) ? 1 : 0);
  m->extras = cfg->extras;

#define CREATE_TRY(expr)                       \
  do {                                         \
    cudaError_t e_ = (expr);                   \
    if (e_ != cudaSuccess) {                   \
      free_model(m);                           \
      return from_cuda(e_);                    \
    }                                          \
  } while (0)

  CREATE_TRY(cudaGetDevice(&m->device));
  CREATE_TRY(cudaDeviceGetAttribute(&m->num_sms, cudaDevAttrMultiProcessorCount, m->device));

  // weights: upload fp32, convert to the compute dtype
  CREATE_TRY(cudaMalloc(&m->weights, n_params * m->wbytes));
  if (m->bf16) {
    float* tmp = nullptr;
    const PtrKind wk = ptr_kind(weights, m->device);
    if (wk == PTR_OTHER_DEVICE) {
      free_model(m);
      return NC_ERR_INVALID_ARG;
    }
    const bool dev_src = wk == PTR_DEVICE;
    if (!dev_src) {
      CREATE_TRY(cudaMalloc(&tmp, (n_params + n_extra) * 4));
      cudaError_t e = cudaMemcpy(tmp, weights, (n_params + n_extra) * 4, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        cudaFree(tmp);
        free_model(m);
        return from_cuda(e);
      }
    }
    f32_to_bf16_kernel<<<4 * m->num_sms, 256>>>(dev_src ? weights : tmp,
                                                 static_cast<__nv_bfloat16*>(m->weights), n_params);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && m->fp8) e = quantize_fp8_weights(m, dev_src ? weights : tmp);
    if (e == cudaSuccess && n_extra > 0) {
      // the extras stay fp32
      e = cudaMalloc(&m->ex_params, n_extra * 4);
      if (e == cudaSuccess)
        e = cudaMemcpy(m->ex_params, (dev_src ? weights : tmp) + n_params, n_extra * 4, cudaMemcpyDeviceToDevice);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (tmp) cudaFree(tmp);
    CREATE_TRY(e);
  } else {
    CREATE_TRY(cudaMalloc(&m->ex_params, (n_extra > 0 ? n_extra : 1) * 4));
    CREATE_TRY(cudaMemcpy(m->weights, weights, n_params * 4, cudaMemcpyDefault));
    if (n_extra > 0) CREATE_TRY(cudaMemcpy(m->ex_params, weights + n_params, n_extra * 4, cudaMemcpyDefault));
  }
  if (n_extra > 0) {
    const float* p = m->ex_params;
    m->ve_table.assign(c.n_layer, nullptr);
    m->ve_gate.assign(c.n_layer, nullptr);
    for (int l = 0; l < c.n_layer && n_ve; l += 2) {
      m->ve_table[l] = p;
      p += V * nkv * hd;
    }
    for (int l = 0; l < c.n_layer && n_ve; l += 2) {
      m->ve_gate[l] = p;
      p += nkv * c.ve_gate_channels;
    }
    if (m->extras & NC_EXTRA_RESID_LAMBDAS) {
      m->resid_l = p;
      m->x0_l = p + c.n_layer;
      p += 2 * c.n_layer;
    }
    if (m->extras & NC_EXTRA_SMEAR) {
      m->smear_w = p;
      m->smear_lambda = p + c.smear_channels;
      p += c.smear_channels + 1;
    }
    if (m->extras & NC_EXTRA_BACKOUT) m->backout_lambda = p;
    if (!n_ve) m->ve_table.clear();
  }
  {
    const char* p = static_cast<const char*>(m->weights);
    const size_t wb = m->wbytes;
    m->E = p;
    p += V * d * wb;
    for (int l = 0; l < c.n_layer; ++l) {
      m->wqkv.push_back(p);
      p += NQKV * d * wb;
      m->wo.push_back(p);
      p += d * NQ * wb;
      m->wfc.push_back(p);
      p += F * d * wb;
      m->wproj.push_back(p);
      p += d * F * wb;
    }
    m->Wu = p;
  }

  // RoPE table, computed in double on the host: theta = p * base^(-2j/hd)
  {
    const int64_t half = hd / 2;
    std::vector<float> cs(c.max_seq * half), sn(c.max_seq * half);
    for (int64_t p = 0; p < c.max_seq; ++p)
      for (int64_t j = 0; j < half; ++j) {
        const double inv = std::pow((double)c.rope_base, -2.0 * (double)j / (double)hd);
        const double th = (double)p * inv;
        cs[p * half + j] = (float)std::cos(th);
        sn[p * half + j] = (float)std::sin(th);
      }
    CREATE_TRY(cudaMalloc(&m->rope_cos, cs.size() * 4));
    CREATE_TRY(cudaMalloc(&m->rope_sin, sn.size() * 4));
    CREATE_TRY(cudaMemcpy(m->rope_cos, cs.data(), cs.size() * 4, cudaMemcpyHostToDevice));
    CREATE_TRY(cudaMemcpy(m->rope_sin, sn.data(), sn.size() * 4, cudaMemcpyHostToDevice));
    std::vector<float2> cst(cs.size());
    for (int64_t p = 0; p < c.max_seq; ++p)
      for (int64_t j = 0; j < half; ++j) cst[j * c.max_seq + p] = make_float2(cs[p * half + j], sn[p * half + j]);
    CREATE_TRY(cudaMalloc(&m->rope_cs_t, cst.size() * sizeof(float2)));
    CREATE_TRY(cudaMemcpy(m->rope_cs_t, cst.data(), cst.size() * sizeof(float2), cudaMemcpyHostToDevice));
  }

  // KV cache with sentinel guards
  m->layer_elems = (int64_t)c.max_batch * nkv * c.max_seq * hd;
  m->kv_elems = 2 * kGuardElems + c.n_layer * m->layer_elems;
  CREATE_TRY(cudaMalloc(&m->k_alloc, m->kv_elems * m->wbytes));
  CREATE_TRY(cudaMalloc(&m->v_alloc, m->kv_elems * m->wbytes));
  CREATE_TRY(cudaMemset(m->k_alloc, 0xFF, m->kv_elems * m->wbytes));
  CREATE_TRY(cudaMemset(m->v_alloc, 0xFF, m->kv_elems * m->wbytes));

  // workspace
  m->max_rows = (int64_t)c.max_batch * c.max_seq;
  const int64_t R = m->max_rows;
  CREATE_TRY(cudaMalloc(&m->x, R * d * 4));
  CREATE_TRY(cudaMalloc(&m->h, R * d * m->wbytes));
  CREATE_TRY(cudaMalloc(&m->q, R * NQ * m->wbytes));
  CREATE_TRY(cudaMalloc(&m->att, R * NQ * m->wbytes));
  CREATE_TRY(cudaMalloc(&m->u, R * F * m->wbytes));
  CREATE_TRY(cudaMalloc(&m->h_last, (int64_t)c.max_batch * d * m->wbytes));
  // (decode: [d/128 + 1][max_batch]; a last-position prefill gathers up to d/96 blocks)
  CREATE_TRY(cudaMalloc(&m->ss_part, (int64_t)(d / 64 + 1) * c.max_batch * 4));
  if (m->bf16) CREATE_TRY(cudaMalloc(&m->ss_rows, (d / 64) * R * 4));
  if (!m->bf16) CREATE_TRY(cudaMalloc(&m->c32, R * NQKV * 4));
  CREATE_TRY(cudaMalloc(&m->tok_stage, R * 4));
  if (m->extras & NC_EXTRA_RESID_LAMBDAS) CREATE_TRY(cudaMalloc(&m->x0, R * d * 4));
  if (m->extras & NC_EXTRA_BACKOUT) CREATE_TRY(cudaMalloc(&m->x_mid, R * d * 4));
  if (m->extras & NC_EXTRA_SMEAR) {
    CREATE_TRY(cudaMalloc(&m->prev_tok, (size_t)c.max_batch * 4));
    CREATE_TRY(cudaMemset(m->prev_tok, 0, (size_t)c.max_batch * 4));
  }
  if (m->bf16) {
    m->vt_S = (c.max_seq + 127) / 128 * 128;
    CREATE_TRY(cudaMalloc(&m->vt, (int64_t)c.max_batch * nkv * 128 * m->vt_S * 2));
    CREATE_TRY(cudaMemset(m->vt, 0, (int64_t)c.max_batch * nkv * 128 * m->vt_S * 2));
  }
  CREATE_TRY(configure_kernels(m));
  CREATE_TRY(cudaMalloc(&m->err, sizeof(int)));
  CREATE_TRY(cudaMalloc(&m->d_len, (size_t)c.max_batch * sizeof(int)));
  CREATE_TRY(cudaMalloc(&m->d_pos0, (size_t)c.max_batch * sizeof(int)));
  CREATE_TRY(cudaMalloc(&m->d_last, (size_t)c.max_batch * sizeof(int)));
  CREATE_TRY(cudaMemset(m->d_len, 0, (size_t)c.max_batch * sizeof(int)));
  CREATE_TRY(cudaMemset(m->d_pos0, 0, (size_t)c.max_batch * sizeof(int)));
  CREATE_TRY(cudaMemset(m->d_last, 0, (size_t)c.max_batch * sizeof(int)));
  m->lens.assign(c.max_batch, 0);
  if (m->bf16 && d <= SK_MAX_SS * 128) {
    // decode-step skinny GEMMs: batch padded to 32, 64 or 128 columns
    m->sk_nb = c.max_batch <= 32 ? 32 : (c.max_batch <= 64 ? 64 : 128);
    const int64_t Ns[4] = {NQKV, d, F, d}, Ks[4] = {d, NQ, d, F};
    for (int g = 0; g < 4; ++g)
      m->sk_splits[g] = choose_splits((int)(Ns[g] / 128), (int)(Ks[g] / 64), m->num_sms);
  }
  CREATE_TRY(cudaMemset(m->h, 0, R * d * m->wbytes));
  CREATE_TRY(cudaMemset(m->att, 0, R * NQ * m->wbytes));
  CREATE_TRY(cudaMemset(m->u, 0, R * F * m->wbytes));
  CREATE_TRY(cudaMemset(m->h_last, 0, (int64_t)c.max_batch * d * m->wbytes));
  CREATE_TRY(cudaMemset(m->err, 0, sizeof(int)));

  if (m->bf16) {
    bool ok = make_tmap(&m->tm_h, m->h, R, d, 128) && make_tmap(&m->tm_att, m->att, R, NQ, 128) &&
              make_tmap(&m->tm_u, m->u, R, F, 128) &&
              make_tmap(&m->tm_hlast, m->h_last, c.max_batch, d, 128) &&
              make_tmap(&m->tm_q_st, m->q, R, NQ, 32) && make_tmap(&m->tm_u_st, m->u, R, F, 32) &&
              make_tmap(&m->tm_x_st, m->x, R, d, 32, true);
    {
      const uint64_t dims[3] = {(uint64_t)m->vt_S, 128, (uint64_t)(c.max_batch * nkv)};
      const uint64_t strides[2] = {(uint64_t)m->vt_S * 2, (uint64_t)m->vt_S * 256};
      const uint32_t box[3] = {64, 128, 1};
      ok = ok && make_tmap3(&m->tm_vt, m->vt, dims, strides, box);
    }
    ok = ok && make_tmap(&m->tm_wu128, m->Wu, V, d, 128);
    // the decode step's intermediates in the workspace
    DecodeBufs& db = m->dbuf;
    db.x = m->x;
    db.h = m->h;
    db.q = m->q;
    db.att = m->att;
    db.u = m->u;
    db.ss = m->ss_part;
    db.ss_ld = c.max_batch;
    if (m->sk_nb > 0)
      ok = ok && make_tmap(&db.tm_h_nb, db.h, R, d, m->sk_nb) && make_tmap(&db.tm_att_nb, db.att, R, NQ, m->sk_nb) &&
           make_tmap(&db.tm_u_nb, db.u, R, F, m->sk_nb);
    // ... and in the no-allocation scratch, when the shape fits it
    if (ok && m->sk_nb > 0 && d <= kNaD && NQ <= kNaNQ && F <= kNaF) {
      void* base = nullptr;
      CREATE_TRY(noalloc_scratch(m->device, &base));
      char* b0 = static_cast<char*>(base);
      DecodeBufs& na = m->dbuf_na;
      na.x = reinterpret_cast<float*>(b0 + kNaOffX);
      na.h = b0 + kNaOffH;
      na.q = b0 + kNaOffQ;
      na.att = b0 + kNaOffAtt;
      na.u = b0 + kNaOffU;
      na.ss = reinterpret_cast<float*>(b0 + kNaOffSS);
      na.ss_ld = kNaRows;
      ok = make_tmap(&na.tm_h_nb, na.h, kNaRows, d, m->sk_nb) && make_tmap(&na.tm_att_nb, na.att, kNaRows, NQ, m->sk_nb) &&
           make_tmap(&na.tm_u_nb, na.u, kNaRows, F, m->sk_nb);
      m->noalloc_ok = ok;
    }
    m->tm_w128.resize(4 * c.n_layer);
    for (int l = 0; ok && l < c.n_layer; ++l)
      ok = make_tmap(&m->tm_w128[4 * l + 0], m->wqkv[l], NQKV, d, 128) &&
           make_tmap(&m->tm_w128[4 * l + 1], m->wo[l], d, NQ, 128) &&
           make_tmap(&m->tm_w128[4 * l + 2], m->wfc[l], F, d, 128) &&
           make_tmap(&m->tm_w128[4 * l + 3], m->wproj[l], d, F, 128);
    if (ok && d % 192 == 0) {
      m->tm_w96.resize(2 * c.n_layer);
      for (int l = 0; ok && l < c.n_layer; ++l)
        ok = make_tmap(&m->tm_w96[2 * l + 0], m->wo[l], d, NQ, 96) &&
             make_tmap(&m->tm_w96[2 * l + 1], m->wproj[l], d, F, 96);
    }
    if (ok && m->fp8) {
      // E4M3 matrices in the order quantize_fp8_weights wrote them
      m->tm_w8.resize(4 * c.n_layer + 1);
      const uint8_t* q = static_cast<const uint8_t*>(m->w8);
      const int64_t rows[4] = {NQKV, d, F, d}, cols[4] = {d, NQ, d, F};
      for (int l = 0; ok && l < c.n_layer; ++l)
        for (int g = 0; ok && g < 4; ++g) {
          ok = make_tmap8(&m->tm_w8[4 * l + g], q, rows[g], cols[g], 128);
          q += rows[g] * cols[g];
        }
      ok = ok && make_tmap8(&m->tm_w8[4 * c.n_layer], q, V, d, 128);
    }
    m->tm_kc.resize(c.n_layer);
    for (int l = 0; ok && l < c.n_layer; ++l) {
      const uint64_t dims[3] = {128, (uint64_t)c.max_seq, (uint64_t)(c.max_batch * nkv)};
      const uint64_t strides[2] = {256, (uint64_t)c.max_seq * 256};
      const uint32_t box[3] = {64, 128, 1};
      ok = make_tmap3(&m->tm_kc[l], m->kc(l), dims, strides, box);
    }
    // K and V caches of all layers (guards included) as [rows][128] for the
    // prefill QKV epilogue's TMA stores
    CUtensorMap kv[2];
    ok = ok && make_tmap(&kv[0], m->k_alloc, (uint64_t)(m->kv_elems / 128), 128, 32) &&
         make_tmap(&kv[1], m->v_alloc, (uint64_t)(m->kv_elems / 128), 128, 32);
    if (ok) {
      CREATE_TRY(cudaMalloc(&m->d_tm_kv, sizeof(kv)));
      CREATE_TRY(cudaMemcpy(m->d_tm_kv, kv, sizeof(kv), cudaMemcpyHostToDevice));
    }
    if (!ok) {
      free_model(m);
      return NC_ERR_CUDA;
    }
  }
  CREATE_TRY(cudaDeviceSynchronize());
  *out = m;
  return NC_OK;
#undef CREATE_TRY
}

void nc_model_destroy(nc_model* m) {
  if (!m) return;
  cudaDeviceSynchronize();
  free_model(m);
}

nc_status nc_kv_reset(nc_model* m, nc_stream_t) {
  if (!m) return NC_ERR_INVALID_ARG;
  m->length = 0;
  m->batch = 0;
  std::fill(m->lens.begin(), m->lens.end(), 0);
  return NC_OK;
}

nc_status nc_prefill_rows(nc_model* m, const int32_t* tokens, int32_t B, int32_t T, const int32_t* row_len,
                          float* logits, int32_t last_only, nc_stream_t stream) {
  if (!m || !tokens || !logits) return NC_ERR_INVALID_ARG;
  if (B < 1 || B > m->cfg.max_batch || T < 1 || T > m->cfg.max_seq) return NC_ERR_INVALID_ARG;
  const bool fresh = m->length == 0;
  // a later chunk of the same rows continues the cache
  if (!fresh && B != m->batch) return NC_ERR_INVALID_ARG;
  std::vector<int32_t> p0(B), len(B), last(B);
  int max_p0 = 0;
  for (int b = 0; b < B; ++b) {
    const int n = row_len ? row_len[b] : T;
    if (n < 1 || n > T) return NC_ERR_INVALID_ARG;
    p0[b] = fresh ? 0 : m->lens[b];
    // the padded tokens of a shorter row are computed too: every row needs
    // room for T positions
    if (T > m->cfg.max_seq - p0[b]) return NC_ERR_CAPACITY;
    len[b] = p0[b] + n;
    last[b] = n - 1;
    max_p0 = std::max(max_p0, (int)p0[b]);
  }
  for (int base = 0; base < B; base += ROWSET_MAX) {
    RowSet rs;
    rs.base = base;
    rs.n = std::min(ROWSET_MAX, B - base);
    for (int i = 0; i < rs.n; ++i) {
      rs.pos0[i] = p0[base + i];
      rs.len[i] = len[base + i];
      rs.last[i] = last[base + i];
    }
    set_rows_kernel<<<1, 256, 0, stream>>>(rs, m->d_pos0, m->d_len, m->d_last);
    m->launches++;
    NC_TRY(cudaGetLastError());
  }
  nc_status st = run_call(m, tokens, B, T, max_p0, logits, last_only != 0, stream, false);
  if (st != NC_OK) return st;
  for (int b = 0; b < B; ++b) m->lens[b] = len[b];
  m->length = *std::max_element(len.begin(), len.end());
  m->batch = B;
  return NC_OK;
}

nc_status nc_prefill(nc_model* m, const int32_t* tokens, int32_t B, int32_t T, float* logits,
                     int32_t last_only, nc_stream_t stream) {
  return nc_prefill_rows(m, tokens, B, T, nullptr, logits, last_only, stream);
}

nc_status nc_decode_step(nc_model* m, const int32_t* tokens, int32_t B, float* logits,
                         nc_stream_t stream) {
  if (!m || !tokens || !logits) return NC_ERR_INVALID_ARG;
  if (m->length == 0) return NC_ERR_STATE;
  if (B != m->batch) return NC_ERR_INVALID_ARG;
  if (m->length >= m->cfg.max_seq) return NC_ERR_CAPACITY;   // the longest row is full
  nc_status st = run_call(m, tokens, B, 1, 0, logits, false, stream, true);
  if (st != NC_OK) return st;
  for (int b = 0; b < B; ++b) m->lens[b] += 1;
  m->length += 1;
  return NC_OK;
}

nc_status nc_decode_step_noalloc(nc_model* m, const int32_t* tokens, int32_t B, float* logits,
                                 nc_stream_t stream) {
  if (!m || !tokens || !logits) return NC_ERR_INVALID_ARG;
  if (!m->bf16) return NC_ERR_UNSUPPORTED;
  if (m->length == 0) return NC_ERR_STATE;
  if (B != m->batch) return NC_ERR_INVALID_ARG;
  if (m->length >= m->cfg.max_seq) return NC_ERR_CAPACITY;
  if (!m->noalloc_ok || B > kNaRows || !decode_on_skinny(m, B)) return NC_ERR_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != m->device) return NC_ERR_INVALID_ARG;
  if (ptr_kind(tokens, m->device) != PTR_DEVICE || ptr_kind(logits, m->device) != PTR_DEVICE)
    return NC_ERR_INVALID_ARG;
  // the step's intermediates live in the file-scope scratch (its device
  // address was looked up when the model was created); the kernels were
  // loaded and configured then too, and the step is launched kernel by
  // kernel: nothing here allocates.  Per-kernel profiling events are not
  // recorded for this call.
  const bool prof = m->profiling;
  m->profiling = false;
  const nc_status st = forward_decode(m, tokens, B, logits, stream, &m->dbuf_na);
  m->profiling = prof;
  if (st != NC_OK) return st;
  for (int b = 0; b < B; ++b) m->lens[b] += 1;
  m->length += 1;
  return NC_OK;
}

nc_status nc_kv_clone(nc_model* m, int32_t src, int32_t n, nc_stream_t stream) {
  if (!m) return NC_ERR_INVALID_ARG;
  if (m->length == 0) return NC_ERR_STATE;
  if (src < 0 || src >= m->batch || n < 1 || n > m->cfg.max_batch) return NC_ERR_INVALID_ARG;
  const size_t wb = m->wbytes, hd = (size_t)m->cfg.head_dim;
  char* k0 = static_cast<char*>(m->k_alloc) + kGuardElems * wb;
  char* v0 = static_cast<char*>(m->v_alloc) + kGuardElems * wb;
  const int len = m->lens[src];
  const int nkv = m->cfg.n_kv_head;
  kv_clone_kernel<<<dim3(n, m->cfg.n_layer, 2 * nkv), 256, 0, stream>>>(
      k0, v0, (size_t)m->layer_elems * wb, (size_t)m->cfg.max_seq * hd * wb, nkv, src, (size_t)len * hd * wb,
      m->d_len, len, m->prev_tok);
  m->launches++;
  NC_TRY(cudaGetLastError());
  for (int b = 0; b < n; ++b) m->lens[b] = len;
  m->length = len;
  m->batch = n;
  return NC_OK;
}

nc_status nc_sample(nc_model* m, const float* logits, int32_t B, double temperature, int32_t top_k,
                    const double* u, int32_t* tokens, nc_stream_t stream) {
  if (!m || !logits || !tokens || B < 1 || B > m->cfg.max_batch) return NC_ERR_INVALID_ARG;
  if (!(temperature >= 0.0) || !std::isfinite(temperature)) return NC_ERR_INVALID_ARG;
  if (temperature > 0.0 && !u) return NC_ERR_INVALID_ARG;
  const int V = m->cfg.vocab;
  const int kept = (top_k <= 0 || top_k > V) ? V : top_k;
  if (temperature > 0.0 && kept > SAMPLE_MAX_KEEP) return NC_ERR_UNSUPPORTED;
  if (ptr_kind(logits, m->device) != PTR_DEVICE || ptr_kind(tokens, m->device) != PTR_DEVICE ||
      (temperature > 0.0 && ptr_kind(u, m->device) != PTR_DEVICE))
    return NC_ERR_INVALID_ARG;
  sample_kernel<<<B, SAMPLE_THREADS, 0, stream>>>(logits, V, V, temperature, top_k, u, tokens);
  m->launches++;
  NC_TRY(cudaGetLastError());
  return NC_OK;
}

nc_status nc_sync_status(nc_model* m, nc_stream_t stream) {
  if (!m) return NC_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return NC_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return NC_ERR_CUDA;
  int flags = 0;
  if (cudaMemcpy(&flags, m->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return NC_ERR_CUDA;
  if (flags) cudaMemset(m->err, 0, sizeof(int));
  if (flags & NC_DEVFLAG_TIMEOUT) return NC_ERR_TIMEOUT;
  if (flags & NC_DEVFLAG_TOKEN) return NC_ERR_TOKEN;
  if (flags) return NC_ERR_CUDA;
  return NC_OK;
}

nc_status nc_kv_length(const nc_model* m, int32_t* length, int32_t* batch) {
  if (!m) return NC_ERR_INVALID_ARG;
  if (length) *length = m->length;
  if (batch) *batch = m->batch;
  return NC_OK;
}

nc_status nc_kv_row_lengths(const nc_model* m, int32_t* lengths) {
  if (!m || !lengths) return NC_ERR_INVALID_ARG;
  for (int b = 0; b < m->batch; ++b) lengths[b] = m->lens[b];
  return NC_OK;
}

nc_status nc_kv_layout(const nc_model* m, int64_t* total_bytes, int64_t* guard_elems,
                       int32_t* elem_bytes) {
  if (!m) return NC_ERR_INVALID_ARG;
  if (total_bytes) *total_bytes = m->kv_elems * (int64_t)m->wbytes;
  if (guard_elems) *guard_elems = kGuardElems;
  if (elem_bytes) *elem_bytes = (int32_t)m->wbytes;
  return NC_OK;
}

nc_status nc_kv_read(nc_model* m, void* k_dst, void* v_dst, nc_stream_t stream) {
  if (!m || !k_dst || !v_dst) return NC_ERR_INVALID_ARG;
  const size_t bytes = m->kv_elems * m->wbytes;
  NC_TRY(cudaMemcpyAsync(k_dst, m->k_alloc, bytes, cudaMemcpyDefault, stream));
  NC_TRY(cudaMemcpyAsync(v_dst, m->v_alloc, bytes, cudaMemcpyDefault, stream));
  return NC_OK;
}

int64_t nc_launch_count(const nc_model* m) { return m ? m->launches : -1; }

nc_status nc_gemm_bf16(nc_model* m, const void* A, const void* W, float* C, int32_t M, int32_t N,
                       int32_t K, nc_stream_t stream) {
  if (!m || !A || !W || !C || M < 1 || N < 256 || K < 8 || N % 256 || K % 8) return NC_ERR_INVALID_ARG;
  if (ptr_kind(A, m->device) != PTR_DEVICE || ptr_kind(W, m->device) != PTR_DEVICE ||
      ptr_kind(C, m->device) != PTR_DEVICE)
    return NC_ERR_INVALID_ARG;
  // M > 128 runs the CTA-pair form the prefill uses
  const int cl = M > 128 ? kPrefillCluster : 0;
  CUtensorMap ta, tb;
  if (!make_tmap(&ta, A, M, K, 128) || !make_tmap(&tb, W, N, K, 128)) return NC_ERR_INVALID_ARG;
  CUtensorMap tc;
  if (!make_tmap(&tc, C, M, N, 32, true)) return NC_ERR_INVALID_ARG;
  GemmArgs a = base_args(m, M, N, K);
  NC_TRY((launch_gemm_tc<256, EPI_STORE>(m, ta, tb, tc, a, stream, cl)));
  return NC_OK;
}

nc_status nc_debug_wait_timeout(nc_model* m, int64_t limit_ns, nc_stream_t stream) {
  if (!m || limit_ns < 0 || limit_ns > 10000000000ll) return NC_ERR_INVALID_ARG;
  wait_nothing_kernel<<<1, 32, 0, stream>>>(m->err, (unsigned long long)limit_ns);
  m->launches++;
  NC_TRY(cudaGetLastError());
  return NC_OK;
}

nc_status nc_profile_begin(nc_model* m) {
  if (!m) return NC_ERR_INVALID_ARG;
  m->recs.clear();
  m->ev_used = 0;
  m->profiling = true;
  return NC_OK;
}

nc_status nc_profile_end(nc_model* m, nc_stream_t stream, double* ms, int64_t* launches) {
  if (!m || !ms || !launches) return NC_ERR_INVALID_ARG;
  m->profiling = false;
  for (int i = 0; i < NC_KCLASS_COUNT; ++i) {
    ms[i] = 0.0;
    launches[i] = 0;
  }
  NC_TRY(cudaStreamSynchronize(stream));
  for (const auto& r : m->recs) {
    float t = 0.f;
    NC_TRY(cudaEventElapsedTime(&t, r.a, r.b));
    ms[r.cls] += t;
    launches[r.cls] += r.launches;
  }
  m->recs.clear();
  m->ev_used = 0;
  return NC_OK;
}

nc_status nc_set_wait_limit(nc_model* m, int64_t limit_ns) {
  if (!m || limit_ns < 1000 || limit_ns > 60000000000ll) return NC_ERR_INVALID_ARG;
  m->wait_limit_ns = (uint64_t)limit_ns;
  return NC_OK;
}

}  // extern "C"
