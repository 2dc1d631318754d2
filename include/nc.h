/*
 * nc.h -- C ABI of the B300-native forward pass of a nanochat-style GPT.
 *
 * The model (yelogs.com nanochat story, "technical details and official Q&A";
 * apidog.com/th "train your own ChatGPT", "how nanochat works" item 1) is a
 * dense decoder-only transformer: untied token embedding E and unembedding
 * Wu, parameter-free RMSNorm after the embedding, before attention, before
 * the MLP and before the unembedding; bias-free QKV projection; RoPE from a
 * precomputed table (geoz.com.cn NanoChat article, "development tricks");
 * parameter-free QK-norm; causal multi-query attention (one K/V head shared by
 * every query head) with scale 1/sqrt(head_dim); output projection and
 * residual; ReLU^2 MLP and residual; logits = softcap * tanh(z / softcap).
 * The inference engine runs it as a full-sequence prefill that fills a KV
 * cache, then one-token decode steps over that cache (szyisi.cn "$100 ...
 * ChatGPT clone", inference engine paragraph; apidog.com/th item 6).
 *
 * Conventions
 *  - Every pointer argument may be a device pointer or a host pointer (pinned
 *    or pageable); the library checks with cudaPointerGetAttributes and stages
 *    host buffers through model-owned device memory on the given stream.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream)
 *    unless a host buffer forces a synchronous copy.  A model is not
 *    thread-safe: one host thread drives it.
 *  - Argument and state errors are returned immediately, with nothing
 *    enqueued.  Conditions found on the device (a token id outside [0, vocab),
 *    an expired bounded wait inside a kernel) are recorded in a device error
 *    word and returned by nc_sync_status().
 *  - No C++ exception crosses this interface.
 */
#ifndef NC_H_
#define NC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define NC_API __attribute__((visibility("default")))
#else
#define NC_API
#endif

typedef struct CUstream_st* nc_stream_t; /* the same type as cudaStream_t */

typedef enum {
  NC_OK = 0,
  NC_ERR_INVALID_ARG = 1, /* a null pointer, a size out of range, a bad config field */
  NC_ERR_UNSUPPORTED = 2, /* a config this build has no kernels for */
  NC_ERR_OOM = 3,         /* device allocation failed */
  NC_ERR_STATE = 4,       /* prefill on a non-empty cache, decode before prefill */
  NC_ERR_CAPACITY = 5,    /* the KV cache is full (length == max_seq) */
  NC_ERR_TOKEN = 6,       /* (device) a token id outside [0, vocab) was seen */
  NC_ERR_TIMEOUT = 7,     /* (device) a bounded pipeline wait expired */
  NC_ERR_CUDA = 8,        /* a CUDA runtime error */
  NC_ERR_SCRATCH_LIMIT = 9 /* nc_decode_step_noalloc: the batch or the model is beyond its fixed scratch */
} nc_status;

typedef enum { NC_F32 = 0, NC_BF16 = 1, NC_FP8 = 2 } nc_dtype;

/*
 * Model shape and capacity.  Shapes of the pages' models: d20 has d_model
 * 1280, 10 heads of dim 128 (szyisi.cn, "pre-training"); d12/d24 follow the
 * same depth rule (d_model = 64 * depth, heads of 128, MLP = 4 * d_model);
 * vocab 65536 = 2**16 (szyisi.cn, tokenizer section).
 *   n_kv_head: K/V heads, dividing n_head; query head h reads K/V head
 *            h / (n_head / n_kv_head).  1 is multi-query attention (yelogs.com
 *            architecture answer); more is grouped-query attention
 *            (apidog.com/th "how nanochat works" item 1).
 *   window / window_layers: sliding-window attention (apidog.com/th item 1,
 *            a pattern such as "SSSL" of short and long windows): a layer
 *            whose bit is set lets a query at position p see only the keys
 *            p - window + 1 .. p.
 *   NC_BF16: weights, activations and the KV cache in bf16 with fp32
 *            accumulation and an fp32 residual stream; needs head_dim == 128,
 *            d_model, d_mlp and n_head*head_dim multiples of 256, vocab a
 *            multiple of 256.
 *   NC_FP8:  as NC_BF16, with FP8 projection weights (the FP8 path of
 *            apidog.com/th "how nanochat works" item 3): each of Wqkv, Wo, Wfc,
 *            Wproj and Wu is rounded at creation to E4M3 values (nearest
 *            even, saturating) times one power-of-two scale per matrix,
 *            2^ceil(log2(amax / 448)).  Decode steps stream the E4M3 bytes
 *            (half the weight traffic) and widen them exactly to f16, with f16
 *            activations; prefill runs the bf16 path on the exact bf16 image
 *            of the same rounded weights.  E stays bf16.
 *   NC_F32:  everything fp32 (SIMT kernels); head_dim 64 or 128.
 *   rms_eps sits inside the square root: x / sqrt(mean(x^2) + eps).
 *   max_batch / max_seq size the KV cache [n_layer][max_batch][n_kv_head][max_seq][head_dim]
 *   (K and V each) and the activation workspace (max_batch * max_seq rows).
 */
/*
 * Later-architecture extras (apidog.com/th "how nanochat works" item 1 and
 * its list of automated improvements; parity-only features of a later
 * version of the model).  Bits of nc_config.extras:
 *   NC_EXTRA_VALUE_EMBED   layers 0, 2, 4, ... add 3 sigmoid(h[:C] G_l^T) VE_l[tok]
 *                          to v per K/V head (h the block's normed input,
 *                          C = ve_gate_channels)
 *   NC_EXTRA_RESID_LAMBDAS before block l: x = resid_l x + x0_l x0, x0 the
 *                          residual that enters block 0
 *   NC_EXTRA_SMEAR         after the embedding norm: x_t += lambda
 *                          sigmoid(x_t[:smear_channels] . w) x_{t-1}, x_{t-1}
 *                          the previous token's normed embedding (none before
 *                          a sequence's first token)
 *   NC_EXTRA_BACKOUT       after the last block: x -= lambda x_mid, x_mid the
 *                          residual after block n_layer / 2 - 1
 * Their fp32 parameters follow Wu in the packed weights, in this order: the
 * tables VE_l [vocab][n_kv_head * head_dim] of the even layers, then their
 * gates G_l [n_kv_head][ve_gate_channels]; resid lambdas [n_layer], x0
 * lambdas [n_layer]; the smear gate [smear_channels] and lambda [1]; the
 * backout lambda [1] (each group present only when its bit is set).  Decode
 * steps of such a model run the generic one-position pass.
 */
enum {
  NC_EXTRA_VALUE_EMBED = 1,
  NC_EXTRA_RESID_LAMBDAS = 2,
  NC_EXTRA_SMEAR = 4,
  NC_EXTRA_BACKOUT = 8,
  NC_EXTRA_ALL = 15
};

typedef struct {
  int32_t n_layer, d_model, n_head, n_kv_head, head_dim, d_mlp, vocab;
  float rope_base, softcap, rms_eps;
  int32_t dtype; /* nc_dtype */
  int32_t max_batch, max_seq;
  int32_t window;          /* sliding window in positions; 0 = every layer sees its whole causal context */
  int32_t reserved;        /* 0 */
  uint64_t window_layers;  /* bit l set: layer l uses the sliding window (n_layer <= 64 when window > 0) */
  int32_t extras;          /* NC_EXTRA_* bits; 0 = the base model */
  int32_t ve_gate_channels, smear_channels;
  int32_t reserved2;       /* 0 */
} nc_config;

typedef struct nc_model nc_model;

/*
 * Create a model on the current CUDA device.
 *   weights: packed fp32 values, canonical order (PyTorch Linear [out, in]
 *            row-major, as F.linear takes them: apidog.com/th item 3):
 *            E[vocab][d]; for each layer Wqkv[(n_head+2)*hd][d] (query heads,
 *            then the key head, then the value head), Wo[d][n_head*hd],
 *            Wfc[d_mlp][d], Wproj[d][d_mlp]; then Wu[vocab][d].
 *            Host or device memory; copied (and rounded to bf16, nearest-even,
 *            for NC_BF16), so the caller may free it when the call returns.
 *   out:     receives the model; *out is NULL on failure.
 * Synchronous.  The model owns its weights, KV cache, RoPE table and workspace.
 */
NC_API nc_status nc_model_create(const nc_config* cfg, const float* weights, nc_model** out);

/* Free everything the model owns.  NULL is ignored.  Synchronizes the device. */
NC_API void nc_model_destroy(nc_model* m);

/*
 * Empty the KV cache (length := 0, no prefill batch), so that the next call
 * must be a prefill.  The inference engine's KV cache is filled by the prefill
 * and extended by each decode step (szyisi.cn "$100 ... ChatGPT clone",
 * inference engine paragraph; apidog.com/th "how nanochat works" item 6);
 * this call starts a new sequence.  Host-side bookkeeping only: `stream` is
 * not used, nothing is enqueued, and the cache contents and the device copy
 * of the length are left as they are (the next prefill's embedding kernel
 * rewrites the device length before any kernel reads it).
 */
NC_API nc_status nc_kv_reset(nc_model* m, nc_stream_t stream);

/*
 * Prefill (szyisi.cn inference engine paragraph: the prompt is processed in
 * one pass that fills the KV cache; apidog.com/th "how nanochat works" item 6;
 * yelogs.com architecture answer for the forward pass itself): the full
 * forward pass over tokens[B][T] at positions p0 .. p0 + T - 1, where p0 is
 * the cache length before the call.
 *  - On an empty cache (p0 = 0) it starts B new sequences.
 *  - On a non-empty cache it is the next chunk of the same B rows (chunked
 *    prefill): each chunk attends to every cached position and to its own
 *    earlier positions, so prefilling a prompt in chunks gives the logits of
 *    prefilling it at once.  Decode steps may come between chunks.
 * K/V of the T positions are written to rows [0, B) of the cache and the
 * cache length becomes p0 + T.
 *   tokens:    int32 [B][T], ids in [0, vocab).
 *   logits:    fp32 [B][T][vocab], or [B][vocab] (position p0 + T - 1) if last_only.
 * Errors: NC_ERR_INVALID_ARG if B is outside [1, max_batch], T outside
 * [1, max_seq], or (non-empty cache) B differs from the cached batch;
 * NC_ERR_CAPACITY if p0 + T > max_seq.
 */
NC_API nc_status nc_prefill(nc_model* m, const int32_t* tokens, int32_t B, int32_t T, float* logits,
                     int32_t last_only, nc_stream_t stream);

/*
 * Prefill with a length per row: as nc_prefill, but row b holds row_len[b]
 * tokens (1 <= row_len[b] <= T) at the start of its T-token slot, the rest of
 * the slot being padding.  Each row has its own cache length: row b's tokens
 * sit at positions p_b .. p_b + row_len[b] - 1, p_b being its length before
 * the call, and its length becomes p_b + row_len[b].  A batch of prompts of
 * different lengths is prefilled in one call this way, and decode steps then
 * append each row's token at its own position.  (The engine serves a batch of
 * sequences from one KV cache: apidog.com/th "how nanochat works" item 6.)
 *   row_len: int32 [B] in host memory; NULL means T for every row.
 *   logits:  fp32 [B][T][vocab] (the padding positions hold unspecified
 *            values), or [B][vocab] at each row's last token if last_only.
 * The padding tokens are computed and their K/V written past the row's
 * length (a later call overwrites them), so every row needs room for T
 * positions: NC_ERR_CAPACITY if p_b + T > max_seq for some row.  Other errors
 * as nc_prefill; NC_ERR_INVALID_ARG for a row_len outside [1, T].
 */
NC_API nc_status nc_prefill_rows(nc_model* m, const int32_t* tokens, int32_t B, int32_t T,
                                 const int32_t* row_len, float* logits, int32_t last_only, nc_stream_t stream);

/*
 * Decode step (szyisi.cn inference engine paragraph and geoz.com.cn
 * "development tricks": each new token attends to the cached keys and values
 * instead of recomputing the prefix): one new token per row at position
 * p = the row's current length, attending to its cached positions 0..p;
 * appends K/V at p; the row's length := p + 1.
 *   tokens: int32 [B]; logits: fp32 [B][vocab].
 * Errors: NC_ERR_STATE before any prefill; NC_ERR_INVALID_ARG if B differs from
 * the prefill's B; NC_ERR_CAPACITY if the longest row's length == max_seq.
 */
NC_API nc_status nc_decode_step(nc_model* m, const int32_t* tokens, int32_t B, float* logits,
                         nc_stream_t stream);

/*
 * Decode step that allocates nothing.  The pages have no counterpart to this
 * call.  It is for callers that cannot allocate device memory while they
 * decode: a serving loop that has handed every free byte to other models'
 * KV caches, a host framework that owns the device allocator and forbids
 * allocations outside it, or code running where an allocation would
 * synchronise the device.  nc_decode_step may allocate: it grows a staging
 * buffer the first time it is given host logits, and it instantiates a CUDA
 * graph of the step.  This call never calls cudaMalloc, cudaFree or any other
 * allocating routine.
 *
 * Same arguments, state rules and results as nc_decode_step, except:
 *  - tokens and logits must be device pointers on the model's device (host
 *    buffers would need staging memory), and the current device must be the
 *    model's device: otherwise NC_ERR_INVALID_ARG;
 *  - the step's intermediates (residual, activations, queries, attention
 *    output, MLP hidden, norm partial sums) live in one fixed scratch array in
 *    device memory, a static part of the library of 4.5 MiB that every GPU
 *    loading the library holds until the process exits.  It serves at most
 *    128 rows of a bf16 model with d_model <= 2048, n_head * 128 <= 2048 and
 *    d_mlp <= 8192; anything larger (or an fp32 model) returns
 *    NC_ERR_SCRATCH_LIMIT with nothing enqueued;
 *  - the scratch's device address is looked up when the first model is
 *    created on a device, and every kernel the step uses is loaded and
 *    configured at model creation, so the call itself does no set-up;
 *  - the step is launched kernel by kernel, not through a CUDA graph.
 * Every call of every model on a device shares the one scratch array, which
 * keeps the last call's contents.  No value in it has to start at zero: each
 * value a step reads was written earlier in the same step, and rows past the
 * batch only feed results that are discarded.  Calls that can overlap on the
 * GPU (on different streams, or on different models) race on the scratch:
 * order them, for example by issuing them on one stream.
 */
NC_API nc_status nc_decode_step_noalloc(nc_model* m, const int32_t* tokens, int32_t B,
                                        float* logits, nc_stream_t stream);

/*
 * Batch generation (apidog.com/th "how nanochat works" item 6: the engine
 * clones the KV cache to sample several continuations of one prompt in
 * parallel): rows [0, n) of the cache become copies of row `src` for every
 * position it holds, every row's length becomes src's, and the batch
 * becomes n.  Typical use: prefill a prompt
 * with B = 1, clone it to n rows, then decode the n rows with different
 * sampled tokens.  Asynchronous on `stream`.
 * Errors: NC_ERR_STATE on an empty cache; NC_ERR_INVALID_ARG if src is not a
 * cached row or n is outside [1, max_batch].
 */
NC_API nc_status nc_kv_clone(nc_model* m, int32_t src, int32_t n, nc_stream_t stream);

/*
 * Next tokens from logits on the device (apidog.com/th item 6 and szyisi.cn
 * inference engine paragraph name sampling but give no rule; this is the
 * plainest reading):
 *  - temperature == 0: the argmax of each row, the lowest index among equal
 *    maxima (u and top_k are not used; u may be NULL);
 *  - temperature > 0: the candidates in the order (logit descending, index
 *    ascending), the first top_k of them (top_k <= 0 keeps all), weights
 *    w_i = exp((l_i - l_0) / temperature) in fp64, cumulative sums
 *    C_j = w_0 + ... + w_j in that order, and the first candidate with
 *    C_j > u[b] * C_last.
 *   logits: fp32 [B][vocab] (device); u: fp64 [B] draws in [0, 1) (device);
 *   tokens: int32 [B] (device), written on `stream`; they may be passed
 *           straight to the next nc_decode_step.
 * At most 1024 candidates are kept with temperature > 0 (top_k <= 1024, or
 * vocab <= 1024): otherwise NC_ERR_UNSUPPORTED.  NC_ERR_INVALID_ARG for null
 * or host pointers, B outside [1, max_batch], a negative or non-finite
 * temperature.
 */
NC_API nc_status nc_sample(nc_model* m, const float* logits, int32_t B, double temperature, int32_t top_k,
                           const double* u, int32_t* tokens, nc_stream_t stream);

/*
 * Synchronize `stream`, then report (and clear) the device error word:
 * NC_ERR_TOKEN, NC_ERR_TIMEOUT, or a pending CUDA error as NC_ERR_CUDA.
 */
NC_API nc_status nc_sync_status(nc_model* m, nc_stream_t stream);

/*
 * The cache length (the longest row's, when rows differ) and the batch
 * (0 before the first prefill).
 */
NC_API nc_status nc_kv_length(const nc_model* m, int32_t* length, int32_t* batch);

/* Each cached row's length: lengths[b] for b < batch (host memory). */
NC_API nc_status nc_kv_row_lengths(const nc_model* m, int32_t* lengths);

/*
 * Test hook: copy the whole K and V caches, guard regions included, into
 * k_dst / v_dst (device or host), each `nc_kv_bytes` bytes.  Layout of each:
 * [guard][n_layer][max_batch][n_kv_head][max_seq][head_dim][guard], elements of
 * `elem_bytes` (2 for NC_BF16, 4 for NC_F32); guards are `guard_elems`
 * elements.  At creation the whole buffer holds the sentinel byte 0xFF; a
 * position is written only when prefill or decode computes it.
 */
NC_API nc_status nc_kv_layout(const nc_model* m, int64_t* total_bytes, int64_t* guard_elems,
                       int32_t* elem_bytes);
NC_API nc_status nc_kv_read(nc_model* m, void* k_dst, void* v_dst, nc_stream_t stream);

/*
 * Number of kernels this model has launched since creation (every kernel of
 * every call, including graph replays).  Used to report launches per step.
 */
NC_API int64_t nc_launch_count(const nc_model* m);

/*
 * Building block, test hook: C[M][N] = A[M][K] * W[N][K]^T with bf16 A and W
 * (device pointers, row-major, K a multiple of 8, N a multiple of 256) and
 * fp32 C (device), on the tcgen05 tensor-core GEMM of the prefill path.
 * Uses the model's error word for timeouts.
 */
NC_API nc_status nc_gemm_bf16(nc_model* m, const void* A, const void* W, float* C, int32_t M, int32_t N,
                       int32_t K, nc_stream_t stream);

/*
 * Failure-detection hook: launch one CTA that waits, with the library's
 * bounded wait, on an mbarrier that nothing arrives at, for at most
 * limit_ns nanoseconds.  nc_sync_status() then returns NC_ERR_TIMEOUT and the
 * CUDA context stays usable.
 */
NC_API nc_status nc_debug_wait_timeout(nc_model* m, int64_t limit_ns, nc_stream_t stream);

/* Upper bound (ns) on every pipeline wait inside the kernels; default 2e9. */
NC_API nc_status nc_set_wait_limit(nc_model* m, int64_t limit_ns);

/*
 * Per-kernel timing with CUDA events on the calling stream.  Between
 * nc_profile_begin and nc_profile_end every kernel the model launches is
 * bracketed by two events; nc_profile_end synchronizes the stream and returns,
 * per kernel class, the summed device time (ms) and the number of launches.
 * Classes (index into the arrays, NC_KCLASS_COUNT entries each):
 */
enum {
  NC_K_EMBED = 0,   /* token embedding + RMSNorm                   */
  NC_K_QKV = 1,     /* QKV projection + RoPE + QK-norm + cache write */
  NC_K_ATTN = 2,    /* causal MQA attention (all its kernels)       */
  NC_K_OPROJ = 3,   /* output projection + residual                 */
  NC_K_NORM = 4,    /* RMSNorm kernels where no projection folds the norm
                       (fp32 model, the extras, the last-position gather,
                       the final norm of a generic decode step)        */
  NC_K_FC = 5,      /* MLP up-projection + ReLU^2                    */
  NC_K_PROJ = 6,    /* MLP down-projection + residual               */
  NC_K_LMHEAD = 7,  /* unembedding + softcap                        */
  NC_KCLASS_COUNT = 8
};
NC_API nc_status nc_profile_begin(nc_model* m);
NC_API nc_status nc_profile_end(nc_model* m, nc_stream_t stream, double* ms, int64_t* launches);

/* Static description of a status code. */
NC_API const char* nc_status_string(nc_status s);

/*
 * Description of the CUDA runtime error behind the last NC_ERR_CUDA or
 * NC_ERR_OOM returned on the calling thread ("no error" if none).  The
 * string is static; the state is per host thread.
 */
NC_API const char* nc_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* NC_H_ */
