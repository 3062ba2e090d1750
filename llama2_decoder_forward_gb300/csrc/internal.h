// Host-side declarations shared by the library's translation units: kernel
// argument blocks and launcher entry points (all enqueue on a caller stream).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/llama_gb300.h"

namespace llgb {

// ------------------------------------------------------------------ launching
// Every kernel is launched with programmatic stream serialization: it may
// start while the previous kernel on the stream drains, runs its prologue
// (barriers, descriptors, weight prefetch) and then waits in-kernel
// (griddepcontrol.wait) before touching activations. set_pdl(false) turns
// this off (plain stream order).
void set_pdl(bool on);
bool pdl_enabled();

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, int cluster_z, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (pdl_enabled()) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_z > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = 1;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = cluster_z;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------ RoPE + append
struct RopeAppendArgs {
  const float* qkv;          // [rows, (n_q + 2 n_kv) d] fp32
  const int32_t* positions;  // [rows] or null (position = r % rows_per_seq)
  // extend steps (separate RoPE kernel only): row r belongs to the sequence b
  // with cu_rows[b] <= r < cu_rows[b + 1] and sits at start_pos[b] + r - cu_rows[b]
  const int32_t* cu_rows;    // [n_seq + 1] or null
  const int32_t* start_pos;  // [n_seq]
  int n_seq;
  // FP8 E4M3 cache: byte = e4m3(x / scale); the K/V side buffers then hold the
  // unscaled e4m3 values (exact in bf16)
  int kv_fp8;
  float k_scale, v_scale;
  const float2* rope;        // [max_seq, d/2] (cos, sin)
  void* q_out;               // [rows, n_q d]
  size_t q_lo;               // >0: also store bf16(q - bf16(q)) q_lo elements further
  void* k_out;               // [rows, n_kv d] or null
  void* v_out;               // [rows, n_kv d] or null
  void* k_cache;
  void* v_cache;
  const int32_t* page_table;
  uint32_t* status;
  int rows_per_seq, n_q, n_kv, head_dim, max_seq, layer;
  int page_size, capacity, batch_cap, n_pages, max_pages;
};

cudaError_t launch_embed(int dtype, const int32_t* tokens, const void* table, int V, int H, int n,
                         float* out, uint32_t* status, cudaStream_t st);
// row_end: optional [rows] — output row r normalises input row row_end[r] - 1
// (the last row of sequence r in a packed batch; in_stride/in_offset unused),
// rows outside [0, n_in) flag LLAMA_FLAG_TOKEN_RANGE and give zeros.
cudaError_t launch_rmsnorm(int dtype, const float* x, int rows, int in_stride, int in_offset,
                           const void* gamma, int H, float eps, void* out, int lo_rows,
                           cudaStream_t st, const int32_t* row_end = nullptr, int n_in = 0,
                           uint32_t* status = nullptr);
cudaError_t launch_rope_table(float2* tab, int max_seq, int head_dim, double theta,
                              cudaStream_t st);
cudaError_t launch_rope_append(int dtype, const RopeAppendArgs& a, int rows, cudaStream_t st);
cudaError_t launch_argmax(const float* logits, int B, int V, int32_t* ids, cudaStream_t st);
cudaError_t launch_advance_positions(int32_t* positions, int B, cudaStream_t st);
// E4M3 rows of a bf16 [rows, cols] matrix with per-row scales (cols % 16 == 0).
cudaError_t launch_quantize_rows_e4m3(const void* w, int rows, int cols, void* codes,
                                      float* scales, cudaStream_t st);
// One bounded wait that nothing completes: sets LLAMA_FLAG_WAIT_TIMEOUT after limit_ns.
cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, cudaStream_t st);

// ------------------------------------------------------------------ GEMM
// y[n, m] (epilogue) sum_k x[n, k] * w[m, k]; x has N rows, w has M rows.
// Internal epilogue of the Q/K/V projection: RoPE on Q and K, Q to its pair
// buffer, K and V into the cache (the work of the RoPE/append kernel).
constexpr int kEpiRope = 4;

struct GemmCall {
  int dtype;
  int epi;                    // LLAMA_EPI_*
  int M, N, K;
  const void* x;              // [N, K]   (fp32 path)
  const void* w;              // [M, K]
  const void* w_up;           // [M, K]   (SWIGLU)
  const CUtensorMap* map_w;   // bf16 path: weights, box {64, 128}, SWIZZLE_128B
  const CUtensorMap* map_up;  // bf16 path, SWIGLU
  const CUtensorMap* map_x;   // bf16 path: activations, box {64, n_tile}
  int n_tile;                 // bf16 path: MMA N (multiple of 16, <= 256)
  int split;                  // bf16 path: x rows [0,N) hold bf16(v), rows [L, L+N) hold
                              // bf16(v - bf16(v)), L = round16(N); both are multiplied
  size_t out_lo;              // bf16 outputs: also store the remainder out_lo elements on
  const RopeAppendArgs* rope; // kEpiRope: where the rotated Q and the K/V rows go
  // Fused RMSNorm (bf16). Producer (RESID_F32): also store the bf16 pair of
  // x_new * norm_gamma[m] in norm_out ([N][M] hi, norm_lo elements further
  // lo) and the sum of x_new^2 over each 128-feature tile in
  // ssq_out[tile][ssq_ld]. Consumer: scale row n's outputs by
  // 1 / sqrt(sum over ssq_tiles of ssq_in[t][n] / norm_h + norm_eps).
  const void* norm_gamma = nullptr;
  void* norm_out = nullptr;
  size_t norm_lo = 0;
  float* ssq_out = nullptr;
  const float* ssq_in = nullptr;
  int ssq_tiles = 0, ssq_ld = 0, norm_h = 0;
  float norm_eps = 0.f;
  // E4M3 weights (bf16 path): map_w / map_up are byte tensors, box {64, 128},
  // no swizzle; row m stands for code * w_scale[m] (u_scale[m] for W_up).
  // Null: bf16 weights.
  const float* w_scale = nullptr;
  const float* u_scale = nullptr;
  void* out;
  int ldo;
  uint32_t* status;
  int sm_count;
};
// Activation rows one bf16 GEMM tile reads (MMA N) for N logical rows; the
// activation descriptor's box holds gemm_box_rows of them.
int gemm_n_tile(int N, int split);
inline int gemm_box_rows(int N, int split) {
  return split ? gemm_n_tile(N, split) / 2 : gemm_n_tile(N, split);
}
cudaError_t launch_gemm(const GemmCall& g, cudaStream_t st);
cudaError_t gemm_prepare();  // sets kernel attributes once per process
// Prefill-sized bf16 pair-operand projections (at least 0.9 tiles of 128
// rows x 256 features per SM): the persistent kernel with the activation rows
// on the MMA's M side. launch_gemm takes this path whenever it applies.
bool gemm_tm_shape(int epi, int M, int N, int split, int sm_count);  // by shape alone
bool gemm_tm_applies(const GemmCall& g);
cudaError_t launch_gemm_tm(const GemmCall& g, cudaStream_t st);
cudaError_t gemm_tm_prepare();

// ------------------------------------------------------------------ attention
struct AttnDecodeArgs {
  const void* q;             // [B, n_q, d]
  size_t q_lo;               // >0: q + q_lo holds the bf16 remainders of q (pair operand)
  const int32_t* positions;  // [B]
  const CUtensorMap* map_k;  // bf16: 3D {d, rows per layer, layers}, box {64, box_rows, 1}, SW128
  const CUtensorMap* map_v;
  const CUtensorMap* map_k16;  // the same views with box {64, 16, 1} (partial tiles, 16-key pages)
  const CUtensorMap* map_v16;
  int box_rows;              // 64 (one box per half of a full 64-key tile) or 16 (one per 16 keys)
  const void* k_cache;       // fp32 path
  const void* v_cache;
  const int32_t* page_table;
  void* out;                 // [B, n_q d]
  size_t out_lo;             // >0: also store bf16 remainders out_lo elements further
  float* partial;            // split partials (workspace)
  size_t partial_bytes;
  uint32_t* status;
  int B, n_q, n_kv, head_dim, layer;
  int page_size, capacity, batch_cap, n_pages, max_pages;
  int max_keys;              // upper bound of positions[b] + 1 (sizes the split count)
  // extend steps: only sequences with one new row (cu_rows[b+1] - cu_rows[b]
  // == 1) are handled, their q / output row being cu_rows[b]; null: row b
  const int32_t* cu_rows = nullptr;
  // FP8 E4M3 cache (key-major groups only): maps over bytes, box {128, rows, 1}
  int kv_fp8 = 0;
  float k_scale = 1.f, v_scale = 1.f;
  int sm_count;
};
size_t attn_decode_partial_bytes(int B, int n_q, int head_dim, int max_keys, int sm_count,
                                 int n_kv);
cudaError_t launch_attn_decode(int dtype, const AttnDecodeArgs& a, cudaStream_t st);
// Rows of the K/V cache boxes: 64 when every 64-key tile is contiguous in
// the cache (no paging, or pages of a multiple of 64 keys), else 16.
inline int attn_decode_box_rows(int page_size) { return page_size % 64 == 0 ? 64 : 16; }
// Kernel launches one decode-attention call makes (1, or 2 with a split merge).
int attn_decode_launches(int B, int n_kv, int max_keys, int sm_count, int dtype);

struct AttnPrefillArgs {
  const void* q;             // [B*T, n_q, d]
  int q_lo_rows;             // >0: row q_lo_rows + r holds the bf16 remainder of q row r
  const void* k;             // [B*T, n_kv, d]
  const void* v;
  const CUtensorMap* map_q;  // bf16: 3D {d, heads, rows}, box {64, 1, 64}, SW128
  const CUtensorMap* map_k;
  const CUtensorMap* map_v;
  void* out;                 // [B*T, n_q d]
  size_t out_lo;             // >0: also store bf16 remainders out_lo elements further
  uint32_t* status;
  int B, T, n_q, n_kv, head_dim;
  // Extend (bf16 only): packed sequences and K/V read from the cache.
  // cu_rows [B+1] / start_pos [B] on the device; T is then the longest
  // sequence's row count and n_rows the packed total. The maps are the
  // cache's 3D views {d, rows per layer, layers} with box {64, box_rows, 1}
  // (map_k, map_v) and box {64, 16, 1} (map_k16, map_v16).
  const int32_t* cu_rows = nullptr;
  const int32_t* start_pos = nullptr;
  int n_rows = 0;
  int from_cache = 0, box_rows = 16, layer = 0;
  int page_size = 0, capacity = 0, batch_cap = 0, n_pages = 0, max_pages = 0;
  const int32_t* page_table = nullptr;
  const CUtensorMap* map_k16 = nullptr;
  const CUtensorMap* map_v16 = nullptr;
  // K/V read as stored values times these (the FP8 cache's unscaled values)
  float k_scale = 1.f, v_scale = 1.f;
};
cudaError_t launch_attn_prefill(int dtype, const AttnPrefillArgs& a, cudaStream_t st);
cudaError_t attn_prepare();
// bf16 prefill attention on tcgen05 (k_prefill_tc.cu)
cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t st);
cudaError_t attn_prefill_tc_prepare();

// ---- token sampling (k_sample.cu)
struct SampleCall {
  const float* logits;  // [B, ldl] fp32, V used per row
  int B, V, ldl;
  float temperature;    // 0: greedy
  int top_k;            // <= 0 or >= V: off
  float top_p;          // >= 1: off
  float penalty;        // 1: off
  const int32_t* history;      // [B, history_stride] ids (penalty only)
  const int32_t* history_len;  // [B]
  int history_stride;
  const float* uniforms;       // [B] in [0, 1)
  int32_t* next_ids;           // [B]
  uint32_t* status;
};
constexpr int kSampleMaxVocab = 32768;  // 64 entries per thread of one 512-thread CTA
int sample_chunk(int V);
size_t sample_smem_bytes(int V);
cudaError_t sample_prepare();
cudaError_t launch_sample(const SampleCall& c, cudaStream_t st);

}  // namespace llgb
