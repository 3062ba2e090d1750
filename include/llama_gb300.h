/*
 * llama_gb300.h -- C ABI of the GB300 (sm_103a) Llama2 decoder forward.
 *
 * The library computes the decoder-only forward pass of a Llama2-style model
 * in its two phases ("Llama2架构与推理全解析" §2.1, Prefill and Decode):
 *
 *   h = embed(token_ids)
 *   for each layer:  h = h + attn(rmsnorm(h), kv_cache)
 *                    h = h + ffn(rmsnorm(h))
 *   logits = lm_head(rmsnorm(h))
 *
 * (the main-computation pseudocode of §2.3), with RMSNorm (§1.2), SwiGLU
 * (§1.3), RoPE (§1.4), grouped-query attention (§1.5) and a KV cache that the
 * caller owns (§2.4). Prefill returns the first prediction and decode appends
 * one token per sequence to the cache (§3.4 generation loop).
 *
 * Conventions shared by every entry point
 *  - All device buffers are allocated by the caller (e.g. with PyTorch) and
 *    passed as plain pointers; the library never allocates device memory. It
 *    keeps a small host-side context whose device state lives in the caller's
 *    workspace (llama_workspace_bytes).
 *  - Row-major storage everywhere. Projection weights are [out, in]
 *    (y = x W^T), which is the pages' x W with W stored [in, out].
 *  - dtype LLAMA_BF16: weights, gains, embedding, LM head, KV cache are bf16
 *    (options: an FP8 E4M3 KV cache, llama_kv.kv_dtype, and E4M3 projection
 *    weights with per-row scales, llama_config.weight_dtype);
 *    dtype LLAMA_F32: all of them are fp32. In both cases the residual
 *    stream (hidden) and the logits are fp32 and every reduction (GEMM,
 *    softmax, norm statistics) accumulates in fp32.
 *  - Token ids, positions and page-table entries are int32.
 *  - Calls enqueue work on the context's stream and return without
 *    synchronising, except llama_sync_status and llama_decode_step_host.
 *  - Every entry point returns an llama_status code. Errors found on the
 *    host (bad pointer, size, layout) are returned at once and nothing is
 *    enqueued. Errors found by kernels (a token id >= vocab, a position past
 *    the cache, a page id outside the pool, a device wait that ran out of
 *    time) set a device status word; the offending access is skipped and the
 *    next llama_sync_status returns LLAMA_ERR_DEVICE_CHECK. Nothing traps.
 *  - One context per stream; a context is not thread-safe.
 */
#ifndef LLAMA_GB300_H
#define LLAMA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum llama_status {
  LLAMA_OK = 0,
  LLAMA_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad layout */
  LLAMA_ERR_UNSUPPORTED = 2,   /* shape the kernels do not implement */
  LLAMA_ERR_OUT_OF_RANGE = 3,  /* size above what the context was built for */
  LLAMA_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  LLAMA_ERR_DEVICE_CHECK = 5,  /* a kernel flagged bad data or a wait timeout */
  LLAMA_ERR_WORKSPACE = 6      /* workspace null, misaligned or too small */
} llama_status;

typedef enum llama_dtype { LLAMA_F32 = 0, LLAMA_BF16 = 1 } llama_dtype;

/* Device status word bits (llama_last_device_flags). */
#define LLAMA_FLAG_TOKEN_RANGE 0x1u   /* token id outside [0, vocab) */
#define LLAMA_FLAG_POS_RANGE 0x2u     /* position outside the cache */
#define LLAMA_FLAG_PAGE_RANGE 0x4u    /* page id outside [0, n_pages) */
#define LLAMA_FLAG_WAIT_TIMEOUT 0x8u  /* a bounded device wait expired */
#define LLAMA_FLAG_INDEX 0x10u        /* bounds-check builds only: a kernel's shared-memory
                                         layout or an index invariant failed its check */

/* Model and sizing. Values of the size table ("Llama2架构与推理全解析" §1.6):
 * 7B = {32, 4096, 32, 32, 128, 11008, 32000}, 70B = {80, 8192, 64, 8, 128,
 * 28672, 32000}; rms_eps 1e-5 (§1.2 gives 1e-5 .. 1e-6), rope_theta 10000. */
typedef struct llama_config {
  int32_t n_layers;
  int32_t hidden;        /* H */
  int32_t n_q_heads;     /* query heads */
  int32_t n_kv_heads;    /* K/V heads; n_q_heads % n_kv_heads == 0 (GQA, §1.5) */
  int32_t head_dim;      /* d, even */
  int32_t intermediate;  /* SwiGLU width I */
  int32_t vocab;         /* V (ignored when has_embed_head == 0) */
  float rms_eps;
  float rope_theta;
  int32_t dtype;         /* llama_dtype */
  int32_t max_batch;     /* most sequences in one call */
  int32_t max_tokens;    /* most prompt rows (B*T) in one prefill call */
  int32_t max_seq;       /* positions 0 .. max_seq-1 may be used (RoPE table size) */
  int32_t has_embed_head;/* 1: token ids in, logits out; 0: hidden in/out only */
  int32_t weight_dtype;  /* projection weights (wqkv, wo, w_gate, w_up, w_down):
                            LLAMA_W_MODEL in the config's dtype, or LLAMA_W_E4M3 */
} llama_config;


/* Projection weights as FP8 E4M3 (bf16 models only; FP8 as the latency option
 * of "Llama2架构全景解析" §3.2): each matrix is [rows, cols] bytes plus an fp32
 * scale per row, row m standing for e4m3(byte) * scale[m]
 * (llama_quantize_rows_e4m3 makes both from bf16). Activations, norms, the
 * embedding and the LM head keep the config's dtype. The GEMMs stream one
 * byte per weight and apply the row scale to their accumulators. */
#define LLAMA_W_MODEL 0
#define LLAMA_W_E4M3 1

/* One layer's weights (device pointers, dtype of the config).
 *   attn_norm, ffn_norm : [H]                       RMSNorm gains
 *   wqkv                : [(n_q + 2 n_kv) d, H]     Q rows, then K rows, then V rows
 *   wo                  : [H, n_q d]
 *   w_gate, w_up        : [I, H]
 *   w_down              : [H, I]
 *   *_scale             : fp32 [rows of that matrix], weight_dtype LLAMA_W_E4M3
 *                         only (the matrices are then E4M3 bytes); else ignored
 * The pointers must stay valid for the life of the context. */
typedef struct llama_layer_weights {
  const void* attn_norm;
  const void* wqkv;
  const void* wo;
  const void* ffn_norm;
  const void* w_gate;
  const void* w_up;
  const void* w_down;
  const float* wqkv_scale;
  const float* wo_scale;
  const float* w_gate_scale;
  const float* w_up_scale;
  const float* w_down_scale;
} llama_layer_weights;

/* Whole-model weights. embed and lm_head are separate [V, H] matrices (the
 * pages: no weight tying); final_norm is [H]. All three may be NULL when
 * has_embed_head == 0. layers is a HOST array of n_layers entries, read
 * during llama_init only. */
typedef struct llama_weights {
  const void* embed;
  const void* final_norm;
  const void* lm_head;
  const llama_layer_weights* layers;
} llama_weights;

/* KV cache, owned by the caller (device memory, dtype of the config).
 * Contiguous (page_size == 0):
 *   k, v : [n_layers][batch_capacity][n_kv][capacity][d]
 *   sequence b of a call uses slot b; positions must be < capacity.
 * Paged (page_size > 0, a multiple of 16; PagedAttention):
 *   k, v       : [n_layers][n_pages][n_kv][page_size][d]
 *   page_table : DEVICE int32 [batch][max_pages_per_seq]; token m of sequence
 *                b lives in page page_table[b][m / page_size], slot
 *                m % page_size.
 * The cache stores the RoPE-rotated K and the plain V.
 * Element type (kv_dtype): LLAMA_KV_MODEL (0) — the config's dtype; or
 * LLAMA_KV_E4M3 (1) — one FP8 E4M3 byte per value (bf16 models only, head_dim
 * 128): a stored byte q means e4m3(q) * k_scale for K, * v_scale for V; values
 * are written as e4m3(x / scale), nearest with ties to even, saturating at
 * +-448 (the FP8 option of "Llama2架构全景解析" §3.2; half the bytes the decode
 * attention streams). An E4M3 cache serves prefill and decode; llama_extend and
 * llama_attention_decode_noalloc answer UNSUPPORTED for it. */
#define LLAMA_KV_MODEL 0
#define LLAMA_KV_E4M3 1
typedef struct llama_kv {
  void* k;
  void* v;
  int32_t page_size;
  int32_t capacity;
  int32_t batch_capacity;
  int32_t n_pages;
  const int32_t* page_table;
  int32_t max_pages_per_seq;
  int32_t kv_dtype;  /* LLAMA_KV_MODEL or LLAMA_KV_E4M3 */
  float k_scale;     /* E4M3 only, > 0 */
  float v_scale;     /* E4M3 only, > 0 */
} llama_kv;

typedef struct llama_ctx llama_ctx;

/* Bytes of device workspace llama_init needs for cfg (256-byte aligned). */
int llama_workspace_bytes(const llama_config* cfg, size_t* bytes);

/* Build a context. workspace: device buffer of at least
 * llama_workspace_bytes bytes, 256-byte aligned, owned by the caller and
 * untouched by anyone else while the context lives. stream: a cudaStream_t
 * (NULL = legacy default stream). Enqueues the RoPE table fill on stream.
 * On success *out receives the context (free with llama_free). */
int llama_init(const llama_config* cfg, const llama_weights* w, void* workspace,
               size_t workspace_bytes, void* stream, llama_ctx** out);

/* Change the stream later calls enqueue on. */
int llama_set_stream(llama_ctx* ctx, void* stream);

/* Prefill a fresh prompt ("Llama2架构与推理全解析" §2.1): tokens is DEVICE
 * int32 [B, T]; token t of each sequence sits at position t. Writes the
 * rotated K and the V of positions 0..T-1 of every layer into kv, then
 * the logits of each sequence's last row into logits (DEVICE fp32 [B, V]).
 * next_ids (DEVICE int32 [B], may be NULL) receives the greedy choice
 * (argmax, lowest index on ties; §2.5). */
int llama_prefill(llama_ctx* ctx, const int32_t* tokens, int32_t B, int32_t T,
                  const llama_kv* kv, float* logits, int32_t* next_ids);

/* One decode step ("Llama2架构与推理全解析" §2.4, §3.4 decode_one): tokens and
 * positions are DEVICE int32 [B]; sequence b's token is at position
 * positions[b], its K/V are appended there, and it attends to keys
 * 0..positions[b]. Writes logits (DEVICE fp32 [B, V]) and, if next_ids is not
 * NULL, the greedy choice per sequence. */
int llama_decode_step(llama_ctx* ctx, const int32_t* tokens, const int32_t* positions,
                      int32_t B, const llama_kv* kv, float* logits, int32_t* next_ids);

/* llama_decode_step with HOST buffers: copies tokens/positions (HOST int32
 * [B]) to the device, runs the step, copies logits (HOST fp32 [B, V], may be
 * NULL) and next_ids (HOST int32 [B], may be NULL) back, and synchronises the
 * stream. Returns the status of the step including device flags. Host buffers
 * should be pinned for asynchronous copies. */
int llama_decode_step_host(llama_ctx* ctx, const int32_t* tokens_host,
                           const int32_t* positions_host, int32_t B, const llama_kv* kv,
                           float* logits_host, int32_t* next_ids_host);

/* The layer stack alone on a hidden state (no embedding, final norm or LM
 * head), for single-layer workloads. hidden is DEVICE fp32, updated in place.
 *   llama_prefill_hidden: hidden [B*T, H], rows of sequence b at b*T .. b*T+T-1,
 *                         fresh prompt at positions 0..T-1.
 *   llama_decode_hidden : hidden [B, H], positions DEVICE int32 [B]. */
int llama_prefill_hidden(llama_ctx* ctx, float* hidden, int32_t B, int32_t T,
                         const llama_kv* kv);
int llama_decode_hidden(llama_ctx* ctx, float* hidden, const int32_t* positions, int32_t B,
                        const llama_kv* kv);

/* Extend step of continuous batching ("Llama2架构全景解析" §3.1 and
 * "基于LLAMA2与PyTorch的高效推理框架实践指南" §三.2 name continuous batching;
 * prefill, §2.1 of "Llama2架构与推理全解析", and decode, §2.4, are its two
 * special cases): one call feeds new tokens of B sequences, each any number of
 * rows at any position — whole prompts of different lengths, a piece of a
 * prompt whose earlier pieces are already cached, or single decode tokens,
 * mixed in one batch. Rows are packed: sequence b owns rows cu_rows[b] ..
 * cu_rows[b+1] - 1 (cu_rows[0] = 0, cu_rows[B] = n_rows, non-decreasing), the
 * first at position start_pos[b] and the rest at consecutive positions; the
 * cache slots of sequence b are those of batch index (or page-table row) b.
 * Every row's rotated K and its V are appended first; row i of sequence b
 * then attends over keys 0 .. start_pos[b] + i of b (its cached keys, the
 * earlier rows of its piece and itself).
 *   tokens   : DEVICE int32 [n_rows]
 *   cu_rows  : DEVICE int32 [B + 1];  start_pos: DEVICE int32 [B]
 *   max_rows : host int, the largest cu_rows[b+1] - cu_rows[b] (sizes the grid)
 *   logits   : DEVICE fp32 [B, V] for the last row of each sequence; next_ids
 *              [B] the greedy ids (or NULL)
 * n_rows <= max(max_batch, max_tokens), B <= max_batch; bf16 models only
 * (UNSUPPORTED otherwise). Positions past the cache, page ids outside the pool
 * and a last row outside [0, n_rows) set device flags (llama_sync_status);
 * malformed cu_rows are the caller's error. Asynchronous. */
int llama_extend(llama_ctx* ctx, const int32_t* tokens, int32_t n_rows, const int32_t* cu_rows,
                 const int32_t* start_pos, int32_t B, int32_t max_rows, const llama_kv* kv,
                 float* logits, int32_t* next_ids);
/* The layer stack of llama_extend on a hidden state: hidden [n_rows, H] fp32,
 * updated in place (for models without embedding and LM head). */
int llama_extend_hidden(llama_ctx* ctx, float* hidden, int32_t n_rows, const int32_t* cu_rows,
                        const int32_t* start_pos, int32_t B, int32_t max_rows,
                        const llama_kv* kv);

/* Capture one decode step into a CUDA graph owned by the context (the launch
 * overhead of a step's ~9 kernels per layer goes away on replay). The device
 * buffers are fixed at capture: tokens [B], positions [B], kv, logits [B, V],
 * next_ids [B] (may be NULL). With advance = 1 the graph ends by adding 1 to
 * every position, so passing next_ids as tokens makes each replay one step
 * of the greedy generation loop ("Llama2架构与推理全解析" §3.4). The context's
 * stream must not be the legacy default stream. A new capture replaces the
 * previous graph. Device-side flags are reported by llama_sync_status as for
 * direct calls. */
int llama_graph_capture_decode(llama_ctx* ctx, const int32_t* tokens, int32_t* positions,
                               int32_t B, const llama_kv* kv, float* logits, int32_t* next_ids,
                               int32_t advance);
/* Replay the captured step on the context's stream. */
int llama_graph_launch(llama_ctx* ctx);

/* E4M3 weights with one scale per row, on the device: for each row m of the
 * bf16 matrix w [rows, cols], scales[m] = max_k |w[m,k]| / 448 (1 for an
 * all-zero row) and codes[m,k] = e4m3(w[m,k] / scales[m]), nearest with ties
 * to even, saturating at +-448 (fp32 arithmetic). w, codes: 16-byte aligned,
 * cols a multiple of 16; codes [rows, cols] bytes, scales [rows] fp32.
 * stream is a cudaStream_t (NULL: the legacy default stream). Asynchronous;
 * INVALID_ARG for null or misaligned pointers or bad sizes. */
int llama_quantize_rows_e4m3(const void* w, int32_t rows, int32_t cols, void* codes,
                             float* scales, void* stream);

/* Synchronise the stream, then read and clear the device status word.
 * Returns LLAMA_OK, LLAMA_ERR_CUDA or LLAMA_ERR_DEVICE_CHECK. */
int llama_sync_status(llama_ctx* ctx);

/* Flags (LLAMA_FLAG_*) seen by the last llama_sync_status. */
uint32_t llama_last_device_flags(const llama_ctx* ctx);

/* Test of the timeout path: enqueue one kernel whose bounded wait, the one
 * every pipelined kernel uses, waits on a shared-memory barrier that nothing
 * completes. After limit_us microseconds (1 .. 1000000) it sets
 * LLAMA_FLAG_WAIT_TIMEOUT and returns; the next llama_sync_status reports
 * LLAMA_ERR_DEVICE_CHECK and the context stays usable. INVALID_ARG for a
 * limit outside that range. Asynchronous. */
int llama_check_wait_timeout(llama_ctx* ctx, int32_t limit_us);

/* 1 when the library was compiled with LLAMA_BOUNDS_CHECK (kernels check
 * their shared-memory layout against the launch's dynamic shared memory and
 * their index invariants, set LLAMA_FLAG_INDEX and skip the work on a
 * failure), else 0. */
int32_t llama_bounds_checked(void);

/* Static description of a status code. */
const char* llama_strerror(int status);

/* Release the host context (the workspace stays the caller's). */
int llama_free(llama_ctx* ctx);

/* ---- Per-kernel timing. kind: one of LLAMA_KERNEL_* below. When enabled,
 * every launch of that kernel class is bracketed by CUDA events on the
 * context's stream; llama_profile_read returns the summed device time (ms)
 * and the launch count since the last reset, synchronising the stream. */
#define LLAMA_KERNEL_RMSNORM 0
#define LLAMA_KERNEL_GEMM 1
#define LLAMA_KERNEL_ROPE_APPEND 2
#define LLAMA_KERNEL_ATTN_DECODE 3
#define LLAMA_KERNEL_ATTN_PREFILL 4
#define LLAMA_KERNEL_EMBED 5
#define LLAMA_KERNEL_ARGMAX 6
#define LLAMA_KERNEL_SAMPLE 7
#define LLAMA_KERNEL_COUNT 8
int llama_profile_enable(llama_ctx* ctx, uint32_t kind_mask);
int llama_profile_read(llama_ctx* ctx, int32_t kind, double* total_ms, int64_t* launches);
/* Launches of this library's kernels enqueued since context creation. */
int64_t llama_launch_count(const llama_ctx* ctx);

/* ---- Single operations, each one kernel (or one kernel plus its split
 * combine) of the forward pass on caller buffers, enqueued on the context's
 * stream. "T" below is the config dtype (bf16 or fp32). ---- */

/* RMSNorm ("Llama2架构与推理全解析" §1.2): out[r] = x[r] / sqrt(mean(x[r]^2) + eps)
 * * gamma over H columns. x fp32 [rows, H] (row r read at x + r*in_stride*H),
 * gamma T [H], out T [rows, H]. in_stride >= 1 selects every in_stride-th row
 * starting at row in_offset. */
int llama_op_rmsnorm(llama_ctx* ctx, const float* x, int32_t rows, int32_t in_stride,
                     int32_t in_offset, const void* gamma, void* out);

/* Linear layer y = x W^T (§1.3 notation x W) with a fused epilogue.
 *   x T [n_rows, K] (or the pair layout, LLAMA_EPI_SPLIT_X); w T [M, K];
 *   w_up T [M, K] (SWIGLU only).
 *   epilogue LLAMA_EPI_STORE_F32 : out fp32 [n_rows, M] = x W^T
 *            LLAMA_EPI_RESID_F32 : out fp32 [n_rows, M] += x W^T (residual add)
 *            LLAMA_EPI_STORE_T   : out T [n_rows, M] = x W^T
 *            LLAMA_EPI_SWIGLU    : out T [n_rows, M] = silu(x W^T) * (x W_up^T)
 * bf16 runs on the tcgen05 tensor cores, fp32 on the CUDA cores. */
#define LLAMA_EPI_STORE_F32 0
#define LLAMA_EPI_RESID_F32 1
#define LLAMA_EPI_STORE_T 2
#define LLAMA_EPI_SWIGLU 3
/* OR-ed into epilogue (bf16, n_rows <= 128): x carries each row as a pair,
 * rows [0, n_rows) = bf16(v) and rows [L, L + n_rows) = bf16(v - bf16(v)),
 * L = n_rows rounded up to a multiple of 16, and the product uses both (about
 * 16 significant bits of v). STORE_T and SWIGLU outputs are written the same
 * way: rows [0, n_rows) and [L, L + n_rows) of out. The library's decode path
 * carries every GEMM operand this way. */
#define LLAMA_EPI_SPLIT_X 16
int llama_op_linear(llama_ctx* ctx, const void* x, int32_t n_rows, const void* w,
                    const void* w_up, int32_t M, int32_t K, int32_t epilogue, void* out);

/* RoPE + KV append (§1.4, §2.4): qkv fp32 [rows, (n_q + 2 n_kv) d] as the Q/K/V
 * projection wrote it; row r is sequence r / rows_per_seq at position
 * positions[r] (DEVICE int32 [rows]). Writes the rotated Q to q_out T
 * [rows, n_q d], the rotated K and the V into layer `layer` of kv, and, if
 * k_out/v_out are not NULL, also to k_out/v_out T [rows, n_kv d]. */
int llama_op_rope_append(llama_ctx* ctx, const float* qkv, int32_t rows, int32_t rows_per_seq,
                         const int32_t* positions, int32_t layer, const llama_kv* kv,
                         void* q_out, void* k_out, void* v_out);

/* Decode attention over the cache (§2.3, §2.4, §1.5): q T [B, n_q, d] (rotated),
 * sequence b attends keys 0..positions[b] of layer `layer`; out T [B, n_q d].
 * positions[b] must lie in [0, min(cache slots, max_seq)): a position outside
 * sets LLAMA_FLAG_POS_RANGE and its output rows are undefined (a negative
 * position gives zeros). */
int llama_op_attention_decode(llama_ctx* ctx, const void* q, const int32_t* positions,
                              int32_t B, int32_t layer, const llama_kv* kv, void* out);

/* Decode attention that allocates nothing. The pages have no counterpart to
 * this entry point: it exists for callers that cannot allocate device memory
 * at the moment they need attention, such as a framework that owns all device
 * memory through its own pool (and forbids other allocators), a plugin loaded
 * into such a framework, or code running while a stream is captured into a
 * CUDA graph (an allocation would break the capture).
 * Same computation and argument meaning as llama_op_attention_decode, but it
 * takes the model config instead of a context, plus a cudaStream_t (NULL =
 * legacy default stream); q, positions, out and kv are the caller's. The
 * key-split partial sums live in an 8 MiB array inside the library's device
 * image: one per GPU that loads the library, held until the process exits.
 * The first call on a device (with that device current) looks up the array's
 * address and sets kernel attributes; make that first call before any stream
 * capture. Calls share the array: calls that overlap on the GPU race and must
 * be serialised by the caller. Shapes whose partial sums would exceed 8 MiB
 * return LLAMA_ERR_OUT_OF_RANGE and enqueue nothing (the partial sums are
 * sized for every slot of the cache: positions may go up to the cache's
 * capacity - 1, whatever cfg->max_seq says). bf16 and head_dim 128 only.
 * Range problems in positions or the page table are still skipped on the
 * device but are not reported (there is no status word): a negative position
 * gives zero output rows, a page id outside the pool reads zeros. */
int llama_attention_decode_noalloc(const llama_config* cfg, const void* q,
                                   const int32_t* positions, int32_t B, int32_t layer,
                                   const llama_kv* kv, void* out, void* stream);

/* Causal prefill attention (§2.1, §2.3) of fresh prompts: q T [B*T, n_q, d],
 * k, v T [B*T, n_kv, d] (k rotated); row t attends keys 0..t of its own
 * sequence; out T [B*T, n_q d]. */
int llama_op_attention_prefill(llama_ctx* ctx, const void* q, const void* k, const void* v,
                               int32_t B, int32_t T, void* out);

/* Embedding row lookup (§2.3): out fp32 [n, H] = table[tokens[i]]. */
int llama_op_embed(llama_ctx* ctx, const int32_t* tokens, int32_t n, void* out);

/* Greedy choice (§2.5): ids[b] = argmax_v logits[b, v], lowest index on ties. */
int llama_op_argmax(llama_ctx* ctx, const float* logits, int32_t B, int32_t V, int32_t* ids);

/* ---- Sampling of the next token ("Llama2架构与推理全解析" §2.5 from logits to
 * sampling, §3.3 sampling parameters; "Llama2架构全景解析" §2.2 step 3:
 * probs = softmax(logits / T), then a draw). Per row b of logits, in order:
 *   1. repetition penalty r: every distinct id among history[b][0 .. history_len[b])
 *      has its logit divided by r if positive, multiplied by r otherwise;
 *   2. temperature T: s = logit / T; T == 0 gives the greedy choice (argmax,
 *      lowest index on ties) and ignores the rest;
 *   3. top-k: keep the k largest s (ties to the lower index);
 *   4. softmax over the kept ids;
 *   5. top-p: keep the smallest prefix of that order whose probability
 *      reaches p;
 *   6. renormalise and draw with uniforms[b] in [0, 1): the first kept id, in
 *      ascending id order, whose cumulative probability exceeds the uniform
 *      (the last kept id if rounding leaves none).
 * The draw is deterministic given the inputs. Random numbers are the caller's:
 * uniforms[b] is drawn by the caller (any generator). */
typedef struct {
  float temperature;        /* >= 0; 0: greedy */
  int32_t top_k;            /* <= 0 or >= V: off */
  float top_p;              /* (0, 1]; 1: off */
  float repetition_penalty; /* > 0; 1: off */
} llama_sampling;

/* logits: [B, V] fp32 device rows (contiguous), V <= 32768;
 * history: [B, history_stride] int32 device ids or NULL (then no penalty),
 * history_len: [B] int32 device counts (may be NULL when history is NULL);
 * uniforms: [B] fp32 device; next_ids: [B] int32 device output. All pointers
 * stay the caller's. Returns INVALID_ARG for NULL buffers or parameters out of
 * range, UNSUPPORTED for V above 32768. History ids outside [0, V)
 * are skipped and set LLAMA_FLAG_TOKEN_RANGE. Asynchronous on the context's
 * stream; one kernel launch. */
int llama_sample(llama_ctx* ctx, const float* logits, int32_t B, int32_t V,
                 const llama_sampling* params,
                 const int32_t* history, const int32_t* history_len, int32_t history_stride,
                 const float* uniforms, int32_t* next_ids);

#ifdef __cplusplus
}
#endif
#endif /* LLAMA_GB300_H */
