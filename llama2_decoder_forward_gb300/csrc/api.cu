// C ABI of the library: configuration checks, the workspace layout, TMA
// descriptors, and the host orchestration of prefill and decode
// ("Llama2架构与推理全解析" §2.3 main computation, §2.1 two phases, §3.4
// generation loop). Every step of the forward pass runs in this library's
// kernels; the host only validates arguments and enqueues launches.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <tuple>
#include <vector>

#include "internal.h"

using namespace llgb;

namespace {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
// bf16 GEMM and attention operands are carried as a pair hi = bf16(v),
// lo = bf16(v - hi): rows [0, n) and [L, L + n) of the buffer, L = n rounded
// up to 16. Products use both, keeping about 16 significant bits of v; only
// the KV cache holds single bf16 values. (The extra MMA work is free while
// decode is bound by weight bytes; it doubles the prefill's tensor work.)
inline int round16(int v) { return (v + 15) / 16 * 16; }
// Remainder-row offset of the pair layout for `rows` activation rows (0 for fp32).
inline int pair_rows(const llama_config& cf, int rows) {
  return cf.dtype == LLAMA_BF16 ? round16(rows) : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_once;
cudaError_t g_prep_err = cudaSuccess;

bool load_encode() {
  std::call_once(g_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    g_prep_err = gemm_prepare();
    if (g_prep_err == cudaSuccess) g_prep_err = attn_prepare();
    if (g_prep_err == cudaSuccess) g_prep_err = sample_prepare();
  });
  return g_encode != nullptr && g_prep_err == cudaSuccess;
}

int elem_size(int dtype) { return dtype == LLAMA_BF16 ? 2 : 4; }

int sm_count_or_default() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
    return n;
  cudaGetLastError();
  return 152;
}

// Workspace layout (byte offsets from the workspace base).
struct Layout {
  size_t status, rope, x, u, qkv, q, kside, vside, o, a, u_last, logits, ids, tok, pos, apart,
      ssq, total;
  size_t apart_bytes;
  int R;
};

int check_config(const llama_config* c) {
  if (!c) return LLAMA_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->hidden < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 ||
      c->head_dim < 2 || c->intermediate < 1 || c->max_batch < 1 || c->max_tokens < 0 ||
      c->max_seq < 1)
    return LLAMA_ERR_INVALID_ARG;
  if (c->has_embed_head != 0 && c->has_embed_head != 1) return LLAMA_ERR_INVALID_ARG;
  if (c->has_embed_head && c->vocab < 1) return LLAMA_ERR_INVALID_ARG;
  if (c->dtype != LLAMA_F32 && c->dtype != LLAMA_BF16) return LLAMA_ERR_INVALID_ARG;
  if (c->weight_dtype != LLAMA_W_MODEL && c->weight_dtype != LLAMA_W_E4M3)
    return LLAMA_ERR_INVALID_ARG;
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return LLAMA_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0) return LLAMA_ERR_INVALID_ARG;
  if (c->head_dim % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  // 16-byte row pitches for TMA and vector loads
  if (c->hidden % 8 != 0 || c->intermediate % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  if (c->weight_dtype == LLAMA_W_E4M3) {  // byte rows: 16-byte pitches for TMA
    if (c->dtype != LLAMA_BF16 || c->hidden % 16 != 0 || c->intermediate % 16 != 0)
      return LLAMA_ERR_UNSUPPORTED;
  }
  if (c->dtype == LLAMA_BF16) {
    if (c->head_dim != 128) return LLAMA_ERR_UNSUPPORTED;
    if (c->n_q_heads / c->n_kv_heads > 16) return LLAMA_ERR_UNSUPPORTED;
  } else {
    if (c->head_dim > 256) return LLAMA_ERR_UNSUPPORTED;
    if ((size_t)(c->max_seq + c->head_dim + 32) * 4 > 200 * 1024) return LLAMA_ERR_UNSUPPORTED;
  }
  return LLAMA_OK;
}

Layout make_layout(const llama_config* c, int sm_count) {
  Layout L{};
  const size_t es = elem_size(c->dtype);
  const int R = std::max(c->max_batch, c->max_tokens);
  L.R = R;
  const size_t H = c->hidden, d = c->head_dim, nq = c->n_q_heads, nkv = c->n_kv_heads,
               I = c->intermediate, V = c->has_embed_head ? c->vocab : 0;
  const size_t qkv_rows = (nq + 2 * nkv) * d;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes);
    return o;
  };
  L.status = take(16);
  L.rope = take((size_t)c->max_seq * (d / 2) * sizeof(float) * 2);
  L.x = take((size_t)R * H * 4);
  // GEMM operands in the hi/lo pair layout: rows [0, R) and [round16(R), ..+R)
  const size_t RA = 2 * (size_t)round16(std::max(R, 1));
  L.u = take(RA * H * es);
  // fp32 Q/K/V rows between the projection and RoPE (bf16 decode applies RoPE in the GEMM epilogue)
  L.qkv = take((size_t)R * qkv_rows * 4);
  L.q = take(RA * nq * d * es);
  L.kside = take((size_t)std::max(c->max_tokens, 1) * nkv * d * es);
  L.vside = take((size_t)std::max(c->max_tokens, 1) * nkv * d * es);
  L.o = take(RA * nq * d * es);
  L.a = take(RA * I * es);
  L.u_last = take(2 * (size_t)round16(c->max_batch) * H * es);
  L.logits = take((size_t)c->max_batch * std::max<size_t>(V, 1) * 4);
  L.ids = take((size_t)c->max_batch * 4);
  L.tok = take((size_t)c->max_batch * 4);
  L.pos = take((size_t)c->max_batch * 4);
  L.apart_bytes = attn_decode_partial_bytes(c->max_batch, (int)nq, (int)d, c->max_seq, sm_count,
                                            (int)nkv);
  L.apart = take(std::max<size_t>(L.apart_bytes, 16));
  // fused RMSNorm: per-(128-feature tile, row) sums of squares of the residual stream
  L.ssq = take((H + 127) / 128 * (size_t)R * 4);
  L.total = off;
  return L;
}

struct Key2 {
  const void* p;
  uint64_t a, b, c, d, e, f;
  bool operator<(const Key2& o) const {
    return std::tie(p, a, b, c, d, e, f) < std::tie(o.p, o.a, o.b, o.c, o.d, o.e, o.f);
  }
};

}  // namespace

struct llama_ctx {
  llama_config cfg;
  cudaStream_t stream = nullptr;
  int device = 0, sm_count = 152, es = 2;
  const void *embed = nullptr, *final_norm = nullptr, *lm_head = nullptr;
  std::vector<llama_layer_weights> layers;
  char* ws = nullptr;
  Layout L;
  uint32_t* status = nullptr;
  float2* rope = nullptr;
  std::map<Key2, CUtensorMap> maps;
  // E4M3 projection weights: weight pointer -> its per-row scales
  std::map<const void*, const float*> wscale;
  uint32_t prof_mask = 0;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> ev[LLAMA_KERNEL_COUNT];
  size_t ev_used[LLAMA_KERNEL_COUNT] = {};
  int64_t launches = 0;
  uint32_t last_flags = 0;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  int64_t graph_launches = 0;  // kernels in one replay of the captured step

  template <typename T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(ws + off);
  }
};

namespace {

// 2D row-major [rows, cols] bf16 tensor, box {64, box_rows}, 128-byte swizzle.
const CUtensorMap* map2d(llama_ctx* c, const void* ptr, uint64_t rows, uint64_t cols,
                         uint32_t box_rows) {
  Key2 k{ptr, 2, rows, cols, box_rows, 0, 0};
  auto it = c->maps.find(k);
  if (it != c->maps.end()) return &it->second;
  CUtensorMap m;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nullptr;
  return &c->maps.emplace(k, m).first->second;
}

// 2D row-major [rows, cols] byte tensor (E4M3 weights), box {64, 128}, no
// swizzle (the GEMM converts the tile to bf16 itself).
const CUtensorMap* map2d_u8(llama_ctx* c, const void* ptr, uint64_t rows, uint64_t cols) {
  Key2 k{ptr, 5, rows, cols, 128, 0, 0};
  auto it = c->maps.find(k);
  if (it != c->maps.end()) return &it->second;
  CUtensorMap m;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nullptr;
  return &c->maps.emplace(k, m).first->second;
}

// 3D [d2][d1][d0] bf16 tensor (d0 innermost), box {64, b1, b2}, 128-byte swizzle.
// 3D [d2][d1][d0] byte tensor (the FP8 cache, d0 = 128), box {128, b1, b2},
// 128-byte swizzle.
const CUtensorMap* map3d_u8(llama_ctx* c, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                            uint32_t b1, uint32_t b2) {
  Key2 k{ptr, 4, d0, d1, d2, b1, b2};
  auto it = c->maps.find(k);
  if (it != c->maps.end()) return &it->second;
  CUtensorMap m;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0, d0 * d1};
  cuuint32_t box[3] = {128, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nullptr;
  return &c->maps.emplace(k, m).first->second;
}

const CUtensorMap* map3d(llama_ctx* c, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint32_t b1, uint32_t b2) {
  Key2 k{ptr, 3, d0, d1, d2, b1, b2};
  auto it = c->maps.find(k);
  if (it != c->maps.end()) return &it->second;
  CUtensorMap m;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return nullptr;
  return &c->maps.emplace(k, m).first->second;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Keep the descriptor cache bounded (callers that keep passing new buffers);
// the weight descriptors are rebuilt on demand after a trim.
void trim_maps(llama_ctx* c) {
  if (c->maps.size() > 4096) c->maps.clear();
}

// Bracket one kernel class with events when profiling is on.
struct Prof {
  llama_ctx* c;
  int kind;
  bool on;
  cudaEvent_t e1 = nullptr;
  Prof(llama_ctx* c_, int k) : c(c_), kind(k), on((c_->prof_mask >> k) & 1u) {
    if (!on) return;
    auto& v = c->ev[kind];
    if (c->ev_used[kind] == v.size()) {
      cudaEvent_t a, b;
      if (cudaEventCreate(&a) != cudaSuccess) { on = false; return; }
      if (cudaEventCreate(&b) != cudaSuccess) { cudaEventDestroy(a); on = false; return; }
      v.push_back({a, b});
    }
    auto& pr = v[c->ev_used[kind]++];
    cudaEventRecord(pr.first, c->stream);
    e1 = pr.second;
  }
  ~Prof() {
    if (on) cudaEventRecord(e1, c->stream);
  }
};

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? LLAMA_OK : LLAMA_ERR_CUDA; }

int check_kv(const llama_ctx* c, const llama_kv* kv, int B) {
  if (!kv || !kv->k || !kv->v) return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(kv->k) || !aligned16(kv->v)) return LLAMA_ERR_INVALID_ARG;
  if (kv->kv_dtype != LLAMA_KV_MODEL && kv->kv_dtype != LLAMA_KV_E4M3) return LLAMA_ERR_INVALID_ARG;
  if (kv->kv_dtype == LLAMA_KV_E4M3) {
    if (c->cfg.dtype != LLAMA_BF16 || c->cfg.head_dim != 128 ||
        c->cfg.n_q_heads / c->cfg.n_kv_heads > 8)
      return LLAMA_ERR_UNSUPPORTED;
    if (!(kv->k_scale > 0.f) || !(kv->v_scale > 0.f) || !std::isfinite(kv->k_scale) ||
        !std::isfinite(kv->v_scale))
      return LLAMA_ERR_INVALID_ARG;
  }
  const uint64_t nkv = c->cfg.n_kv_heads;
  uint64_t rows;
  if (kv->page_size == 0) {
    if (kv->capacity < 1 || kv->batch_capacity < B) return LLAMA_ERR_INVALID_ARG;
    rows = (uint64_t)kv->batch_capacity * nkv * kv->capacity;
  } else {
    if (kv->page_size < 0 || !kv->page_table || kv->n_pages < 1 || kv->max_pages_per_seq < 1)
      return LLAMA_ERR_INVALID_ARG;
    if (c->cfg.dtype == LLAMA_BF16 && kv->page_size % 16 != 0) return LLAMA_ERR_UNSUPPORTED;
    rows = (uint64_t)kv->n_pages * nkv * kv->page_size;
  }
  if (rows + 64 >= (1ull << 31)) return LLAMA_ERR_UNSUPPORTED;  // int32 TMA row coordinates
  return LLAMA_OK;
}

// ---------------------------------------------------------------- single steps
int do_rmsnorm(llama_ctx* c, const float* x, int rows, int stride, int offset, const void* gamma,
               void* out, int lo_rows = 0, const int32_t* row_end = nullptr, int n_in = 0) {
  Prof pf(c, LLAMA_KERNEL_RMSNORM);
  c->launches++;
  return cuda_rc(launch_rmsnorm(c->cfg.dtype, x, rows, stride, offset, gamma, c->cfg.hidden,
                                c->cfg.rms_eps, out, lo_rows, c->stream, row_end, n_in,
                                c->status));
}

// split: x holds the hi/lo pair layout of its N rows; out_lo: bf16 outputs also
// store their remainder out_lo elements further on.
// RMSNorm folded into the projections (bf16): the residual GEMM that updates
// x also writes the next projection's input pair x * gamma and the tile sums
// of x^2 (producer); the next projection scales each row by 1/rms from those
// sums (consumer).
struct NormFuse {
  const void* gamma = nullptr;  // producer
  void* out = nullptr;
  size_t lo = 0;
  bool consume = false;         // consumer
};

// rope: the Q/K/V projection's RoPE + cache-append epilogue (bf16 only).
int do_gemm(llama_ctx* c, int epi, const void* x, int N, int K, const void* w, const void* wu,
            int M, void* out, int ldo, int split = 0, size_t out_lo = 0,
            const RopeAppendArgs* rope = nullptr, const NormFuse* nf = nullptr) {
  GemmCall g{};
  g.rope = rope;
  if (nf) {
    float* ssq = c->at<float>(c->L.ssq);
    g.norm_gamma = nf->gamma;
    g.norm_out = nf->out;
    g.norm_lo = nf->lo;
    g.ssq_out = nf->gamma ? ssq : nullptr;
    g.ssq_in = nf->consume ? ssq : nullptr;
    g.ssq_tiles = (c->cfg.hidden + 127) / 128;
    g.ssq_ld = c->L.R;
    g.norm_h = c->cfg.hidden;
    g.norm_eps = c->cfg.rms_eps;
  }
  g.split = split;
  g.out_lo = out_lo;
  g.dtype = c->cfg.dtype;
  g.epi = epi;
  g.M = M;
  g.N = N;
  g.K = K;
  g.x = x;
  g.w = w;
  g.w_up = wu;
  g.out = out;
  g.ldo = ldo;
  g.status = c->status;
  g.sm_count = c->sm_count;
  if (c->cfg.dtype == LLAMA_BF16) {
    if (!aligned16(x) || !aligned16(w) || (wu && !aligned16(wu))) return LLAMA_ERR_INVALID_ARG;
    trim_maps(c);
    g.n_tile = gemm_n_tile(N, split);
    if (!c->wscale.empty()) {  // E4M3 projection weights
      auto iw = c->wscale.find(w);
      if (iw != c->wscale.end()) g.w_scale = iw->second;
      if (wu) {
        auto iu = c->wscale.find(wu);
        if (iu != c->wscale.end()) g.u_scale = iu->second;
      }
      if ((wu != nullptr) && ((g.w_scale != nullptr) != (g.u_scale != nullptr)))
        return LLAMA_ERR_INVALID_ARG;
    }
    if (g.w_scale) {
      g.map_w = map2d_u8(c, w, M, K);
      g.map_up = wu ? map2d_u8(c, wu, M, K) : nullptr;
    } else {
      g.map_w = map2d(c, w, M, K, 128);
      g.map_up = wu ? map2d(c, wu, M, K, 128) : nullptr;
    }
    g.map_x = map2d(c, x, split ? (uint64_t)round16(N) + N : (uint64_t)N, K,
                    gemm_box_rows(N, split));
    if (!g.map_w || !g.map_x || (wu && !g.map_up)) return LLAMA_ERR_CUDA;
  }
  Prof pf(c, LLAMA_KERNEL_GEMM);
  c->launches++;
  return cuda_rc(launch_gemm(g, c->stream));
}

RopeAppendArgs rope_args(const llama_ctx* c, const float* qkv, int rows_per_seq,
                         const int32_t* positions, int layer, const llama_kv* kv, void* q_out,
                         void* k_out, void* v_out, size_t q_lo) {
  RopeAppendArgs a{};
  a.q_lo = q_lo;
  a.qkv = qkv;
  a.positions = positions;
  a.rope = c->rope;
  a.q_out = q_out;
  a.k_out = k_out;
  a.v_out = v_out;
  a.k_cache = kv->k;
  a.v_cache = kv->v;
  a.page_table = kv->page_table;
  a.status = c->status;
  a.rows_per_seq = rows_per_seq;
  a.n_q = c->cfg.n_q_heads;
  a.n_kv = c->cfg.n_kv_heads;
  a.head_dim = c->cfg.head_dim;
  a.max_seq = c->cfg.max_seq;
  a.layer = layer;
  a.page_size = kv->page_size;
  a.capacity = kv->capacity;
  a.batch_cap = kv->batch_capacity;
  a.n_pages = kv->n_pages;
  a.max_pages = kv->max_pages_per_seq;
  a.kv_fp8 = kv->kv_dtype == LLAMA_KV_E4M3;
  a.k_scale = kv->k_scale;
  a.v_scale = kv->v_scale;
  return a;
}

// Packed sequences of an extend step: sequence b owns rows cu_rows[b] ..
// cu_rows[b+1]-1, the first at position start_pos[b]; max_rows bounds the
// rows of one sequence.
struct RowMap {
  const int32_t* cu_rows;
  const int32_t* start_pos;
  int B, max_rows;
};

int do_rope_append(llama_ctx* c, const float* qkv, int rows, int rows_per_seq,
                   const int32_t* positions, int layer, const llama_kv* kv, void* q_out,
                   void* k_out, void* v_out, size_t q_lo = 0, const RowMap* rm = nullptr) {
  RopeAppendArgs a =
      rope_args(c, qkv, rows_per_seq, positions, layer, kv, q_out, k_out, v_out, q_lo);
  if (rm) {
    a.cu_rows = rm->cu_rows;
    a.start_pos = rm->start_pos;
    a.n_seq = rm->B;
  }
  Prof pf(c, LLAMA_KERNEL_ROPE_APPEND);
  c->launches++;
  return cuda_rc(launch_rope_append(c->cfg.dtype, a, rows, c->stream));
}

int do_attn_decode(llama_ctx* c, const void* q, const int32_t* positions, int B, int layer,
                   const llama_kv* kv, void* out, size_t out_lo = 0, size_t q_lo = 0,
                   const int32_t* cu_rows = nullptr) {
  AttnDecodeArgs a{};
  a.cu_rows = cu_rows;
  a.out_lo = out_lo;
  a.q_lo = q_lo;
  a.q = q;
  a.positions = positions;
  a.k_cache = kv->k;
  a.v_cache = kv->v;
  a.page_table = kv->page_table;
  a.out = out;
  a.partial = c->at<float>(c->L.apart);
  a.partial_bytes = c->L.apart_bytes;
  a.status = c->status;
  a.B = B;
  a.n_q = c->cfg.n_q_heads;
  a.n_kv = c->cfg.n_kv_heads;
  a.head_dim = c->cfg.head_dim;
  a.layer = layer;
  a.page_size = kv->page_size;
  a.capacity = kv->capacity;
  a.batch_cap = kv->batch_capacity;
  a.n_pages = kv->n_pages;
  a.max_pages = kv->max_pages_per_seq;
  const int cap_keys = kv->page_size ? kv->max_pages_per_seq * kv->page_size : kv->capacity;
  a.max_keys = std::max(1, std::min(cap_keys, c->cfg.max_seq));
  a.sm_count = c->sm_count;
  a.kv_fp8 = kv->kv_dtype == LLAMA_KV_E4M3;
  a.k_scale = kv->k_scale;
  a.v_scale = kv->v_scale;
  if (a.kv_fp8) {  // byte views of the cache
    trim_maps(c);
    const uint64_t d = c->cfg.head_dim, nkv = c->cfg.n_kv_heads;
    const uint64_t rows = kv->page_size ? (uint64_t)kv->n_pages * nkv * kv->page_size
                                        : (uint64_t)kv->batch_capacity * nkv * kv->capacity;
    a.box_rows = attn_decode_box_rows(kv->page_size);
    a.map_k = map3d_u8(c, kv->k, d, rows, c->cfg.n_layers, a.box_rows, 1);
    a.map_v = map3d_u8(c, kv->v, d, rows, c->cfg.n_layers, a.box_rows, 1);
    a.map_k16 = map3d_u8(c, kv->k, d, rows, c->cfg.n_layers, 16, 1);
    a.map_v16 = map3d_u8(c, kv->v, d, rows, c->cfg.n_layers, 16, 1);
    if (!a.map_k || !a.map_v || !a.map_k16 || !a.map_v16) return LLAMA_ERR_CUDA;
  } else if (c->cfg.dtype == LLAMA_BF16) {
    trim_maps(c);
    const uint64_t d = c->cfg.head_dim, nkv = c->cfg.n_kv_heads;
    const uint64_t rows = kv->page_size ? (uint64_t)kv->n_pages * nkv * kv->page_size
                                        : (uint64_t)kv->batch_capacity * nkv * kv->capacity;
    a.box_rows = attn_decode_box_rows(kv->page_size);
    a.map_k = map3d(c, kv->k, d, rows, c->cfg.n_layers, a.box_rows, 1);
    a.map_v = map3d(c, kv->v, d, rows, c->cfg.n_layers, a.box_rows, 1);
    a.map_k16 = map3d(c, kv->k, d, rows, c->cfg.n_layers, 16, 1);
    a.map_v16 = map3d(c, kv->v, d, rows, c->cfg.n_layers, 16, 1);
    if (!a.map_k || !a.map_v || !a.map_k16 || !a.map_v16) return LLAMA_ERR_CUDA;
  }
  Prof pf(c, LLAMA_KERNEL_ATTN_DECODE);
  c->launches += attn_decode_launches(B, a.n_kv, a.max_keys, c->sm_count, c->cfg.dtype);
  return cuda_rc(launch_attn_decode(c->cfg.dtype, a, c->stream));
}

int do_attn_prefill(llama_ctx* c, const void* q, const void* k, const void* v, int B, int T,
                    void* out, size_t out_lo = 0, int q_lo_rows = 0, float k_scale = 1.f,
                    float v_scale = 1.f) {
  AttnPrefillArgs a{};
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.out_lo = out_lo;
  a.q_lo_rows = q_lo_rows;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.status = c->status;
  a.B = B;
  a.T = T;
  a.n_q = c->cfg.n_q_heads;
  a.n_kv = c->cfg.n_kv_heads;
  a.head_dim = c->cfg.head_dim;
  if (c->cfg.dtype == LLAMA_BF16) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return LLAMA_ERR_INVALID_ARG;
    trim_maps(c);
    const uint64_t d = c->cfg.head_dim, rows = (uint64_t)B * T;
    a.map_q = map3d(c, q, d, c->cfg.n_q_heads, rows + (uint64_t)q_lo_rows, 1, 64);
    a.map_k = map3d(c, k, d, c->cfg.n_kv_heads, rows, 1, 64);
    a.map_v = map3d(c, v, d, c->cfg.n_kv_heads, rows, 1, 64);
    if (!a.map_q || !a.map_k || !a.map_v) return LLAMA_ERR_CUDA;
  }
  Prof pf(c, LLAMA_KERNEL_ATTN_PREFILL);
  c->launches++;
  return cuda_rc(launch_attn_prefill(c->cfg.dtype, a, c->stream));
}

// Attention of an extend step: every packed row over keys 0 .. its position
// of its sequence, read from the cache (the rows' own K/V already appended).
int do_attn_extend(llama_ctx* c, const void* q, int n_rows, const RowMap& rm, int layer,
                   const llama_kv* kv, void* out, size_t out_lo, int q_lo_rows) {
  if (c->cfg.dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (!aligned16(q)) return LLAMA_ERR_INVALID_ARG;
  AttnPrefillArgs a{};
  a.out_lo = out_lo;
  a.q_lo_rows = q_lo_rows;
  a.q = q;
  a.out = out;
  a.status = c->status;
  a.B = rm.B;
  a.T = rm.max_rows;
  a.n_q = c->cfg.n_q_heads;
  a.n_kv = c->cfg.n_kv_heads;
  a.head_dim = c->cfg.head_dim;
  a.cu_rows = rm.cu_rows;
  a.start_pos = rm.start_pos;
  a.n_rows = n_rows;
  a.from_cache = 1;
  a.box_rows = attn_decode_box_rows(kv->page_size);
  a.layer = layer;
  a.page_size = kv->page_size;
  a.capacity = kv->capacity;
  a.batch_cap = kv->batch_capacity;
  a.n_pages = kv->n_pages;
  a.max_pages = kv->max_pages_per_seq;
  a.page_table = kv->page_table;
  trim_maps(c);
  const uint64_t d = c->cfg.head_dim, nkv = c->cfg.n_kv_heads;
  const uint64_t crow = kv->page_size ? (uint64_t)kv->n_pages * nkv * kv->page_size
                                      : (uint64_t)kv->batch_capacity * nkv * kv->capacity;
  a.map_q = map3d(c, q, d, c->cfg.n_q_heads, (uint64_t)n_rows + (uint64_t)q_lo_rows, 1, 64);
  a.map_k = map3d(c, kv->k, d, crow, c->cfg.n_layers, a.box_rows, 1);
  a.map_v = map3d(c, kv->v, d, crow, c->cfg.n_layers, a.box_rows, 1);
  a.map_k16 = map3d(c, kv->k, d, crow, c->cfg.n_layers, 16, 1);
  a.map_v16 = map3d(c, kv->v, d, crow, c->cfg.n_layers, 16, 1);
  if (!a.map_q || !a.map_k || !a.map_v || !a.map_k16 || !a.map_v16) return LLAMA_ERR_CUDA;
  Prof pf(c, LLAMA_KERNEL_ATTN_PREFILL);
  c->launches++;
  return cuda_rc(launch_attn_prefill(c->cfg.dtype, a, c->stream));
}

#define TRY(expr)                   \
  do {                              \
    const int _rc = (expr);         \
    if (_rc != LLAMA_OK) return _rc; \
  } while (0)

// One decoder layer on rows x[0..rows): h = h + attn(rmsnorm(h)); h = h + ffn(rmsnorm(h)).
// rm: an extend step (packed rows of several sequences at any positions);
// B, T, positions and prefill are then unused.
int run_layer(llama_ctx* c, int l, float* x, int rows, int B, int T, const int32_t* positions,
              const llama_kv* kv, bool prefill, const RowMap* rm = nullptr) {
  const llama_config& cf = c->cfg;
  const llama_layer_weights& lw = c->layers[l];
  const int H = cf.hidden, d = cf.head_dim, nq = cf.n_q_heads, nkv = cf.n_kv_heads,
            I = cf.intermediate;
  const int qkv_rows = (nq + 2 * nkv) * d;
  void* u = c->at<void>(c->L.u);
  float* qkv = c->at<float>(c->L.qkv);
  void* q = c->at<void>(c->L.q);
  void* o = c->at<void>(c->L.o);
  void* a = c->at<void>(c->L.a);
  const int lo = pair_rows(cf, rows);
  const int sp = lo ? 1 : 0;
  // bf16: the RMSNorms after the first ride on the residual GEMMs (the layers
  // run in order, so layer l > 0 finds its normalised input pair and the row
  // sums left by layer l - 1's down projection)
  const bool fuse = cf.dtype == LLAMA_BF16;
  NormFuse consume;
  consume.consume = true;
  const NormFuse* qkv_nf = fuse && l > 0 ? &consume : nullptr;
  if (!qkv_nf) TRY(do_rmsnorm(c, x, rows, 1, 0, lw.attn_norm, u, lo));
  void* ks = prefill ? c->at<void>(c->L.kside) : nullptr;
  void* vs = prefill ? c->at<void>(c->L.vside) : nullptr;
  const int rps = prefill ? T : 1;
  const int32_t* pos = prefill ? nullptr : positions;
  const size_t q_lo = (size_t)lo * nq * d;
  // prefill Q/K/V on the token-major GEMM (bf16 weights, prefill-sized rows)
  const bool tm_qkv = prefill && cf.dtype == LLAMA_BF16 && d % 16 == 0 &&
                      (c->wscale.empty() || c->wscale.find(lw.wqkv) == c->wscale.end()) &&
                      gemm_tm_shape(kEpiRope, qkv_rows, rows, sp, c->sm_count);
  if (rm) {  // extend: RoPE/append, then attention over the cache
    TRY(do_gemm(c, LLAMA_EPI_STORE_F32, u, rows, H, lw.wqkv, nullptr, qkv_rows, qkv, qkv_rows, sp,
                0, nullptr, qkv_nf));
    TRY(do_rope_append(c, qkv, rows, 1, nullptr, l, kv, q, nullptr, nullptr, q_lo, rm));
    TRY(do_attn_extend(c, q, rows, *rm, l, kv, o, q_lo, lo));  // pieces of 2+ rows
    TRY(do_attn_decode(c, q, rm->start_pos, rm->B, l, kv, o, q_lo, q_lo, rm->cu_rows));  // 1 row
  } else if (cf.dtype == LLAMA_BF16 && (!prefill || tm_qkv)) {
    // Q/K/V projection with RoPE and the cache append in its epilogue. A
    // prefill takes it only on the persistent token-major GEMM, whose
    // epilogue overlaps the next tile's MMAs; with one tile per CTA the
    // per-element work stalled the tensor pipe for longer than the separate
    // pass over the fp32 rows takes.
    const RopeAppendArgs ra = rope_args(c, nullptr, rps, pos, l, kv, q, ks, vs, q_lo);
    TRY(do_gemm(c, kEpiRope, u, rows, H, lw.wqkv, nullptr, qkv_rows, nullptr, qkv_rows, sp, 0,
                &ra, qkv_nf));
    if (prefill) {
      const bool f8 = kv->kv_dtype == LLAMA_KV_E4M3;
      TRY(do_attn_prefill(c, q, ks, vs, B, T, o, q_lo, lo, f8 ? kv->k_scale : 1.f,
                          f8 ? kv->v_scale : 1.f));
    } else {
      TRY(do_attn_decode(c, q, positions, B, l, kv, o, q_lo, q_lo));
    }
  } else {
    TRY(do_gemm(c, LLAMA_EPI_STORE_F32, u, rows, H, lw.wqkv, nullptr, qkv_rows, qkv, qkv_rows, sp,
                0, nullptr, qkv_nf));
    TRY(do_rope_append(c, qkv, rows, rps, pos, l, kv, q, ks, vs, q_lo));
    const bool f8 = kv->kv_dtype == LLAMA_KV_E4M3;  // side buffers hold unscaled E4M3 values
    if (prefill)
      TRY(do_attn_prefill(c, q, ks, vs, B, T, o, q_lo, lo, f8 ? kv->k_scale : 1.f,
                          f8 ? kv->v_scale : 1.f));
    else
      TRY(do_attn_decode(c, q, positions, B, l, kv, o, q_lo, q_lo));
  }
  if (fuse) {
    NormFuse ffn;  // O projection + residual, then the pre-FFN norm's input pair
    ffn.gamma = lw.ffn_norm;
    ffn.out = u;
    ffn.lo = (size_t)lo * H;
    TRY(do_gemm(c, LLAMA_EPI_RESID_F32, o, rows, nq * d, lw.wo, nullptr, H, x, H, sp, 0, nullptr,
                &ffn));
    TRY(do_gemm(c, LLAMA_EPI_SWIGLU, u, rows, H, lw.w_gate, lw.w_up, I, a, I, sp, (size_t)lo * I,
                nullptr, &consume));
    NormFuse next;  // down projection + residual, then the next layer's pre-attention pair
    next.gamma = l + 1 < cf.n_layers ? c->layers[l + 1].attn_norm : nullptr;
    next.out = u;
    next.lo = (size_t)lo * H;
    TRY(do_gemm(c, LLAMA_EPI_RESID_F32, a, rows, I, lw.w_down, nullptr, H, x, H, sp, 0, nullptr,
                next.gamma ? &next : nullptr));
  } else {
    TRY(do_gemm(c, LLAMA_EPI_RESID_F32, o, rows, nq * d, lw.wo, nullptr, H, x, H, sp));
    TRY(do_rmsnorm(c, x, rows, 1, 0, lw.ffn_norm, u, lo));
    TRY(do_gemm(c, LLAMA_EPI_SWIGLU, u, rows, H, lw.w_gate, lw.w_up, I, a, I, sp, (size_t)lo * I));
    TRY(do_gemm(c, LLAMA_EPI_RESID_F32, a, rows, I, lw.w_down, nullptr, H, x, H, sp));
  }
  return LLAMA_OK;
}

// Final RMSNorm + LM head (+ greedy choice) on rows stride*b + offset of x.
// row_end (extend): sequence b's last row is row_end[b] - 1 of the n_in rows.
int run_head(llama_ctx* c, const float* x, int B, int stride, int offset, float* logits,
             int32_t* next_ids, const int32_t* row_end = nullptr, int n_in = 0) {
  const llama_config& cf = c->cfg;
  void* ul = c->at<void>(c->L.u_last);
  const int lo = pair_rows(cf, B);
  TRY(do_rmsnorm(c, x, B, stride, offset, c->final_norm, ul, lo, row_end, n_in));
  TRY(do_gemm(c, LLAMA_EPI_STORE_F32, ul, B, cf.hidden, c->lm_head, nullptr, cf.vocab, logits,
              cf.vocab, lo ? 1 : 0));
  if (next_ids) {
    Prof pf(c, LLAMA_KERNEL_ARGMAX);
    c->launches++;
    TRY(cuda_rc(launch_argmax(logits, B, cf.vocab, next_ids, c->stream)));
  }
  return LLAMA_OK;
}

int check_ctx(const llama_ctx* c) { return c ? LLAMA_OK : LLAMA_ERR_INVALID_ARG; }

}  // namespace

// ======================================================================== C ABI
extern "C" {

const char* llama_strerror(int s) {
  switch (s) {
    case LLAMA_OK: return "ok";
    case LLAMA_ERR_INVALID_ARG: return "invalid argument";
    case LLAMA_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case LLAMA_ERR_OUT_OF_RANGE: return "size above the context's limits";
    case LLAMA_ERR_CUDA: return "CUDA call failed";
    case LLAMA_ERR_DEVICE_CHECK: return "a kernel flagged bad input or a wait timeout";
    case LLAMA_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    default: return "unknown status";
  }
}

int llama_workspace_bytes(const llama_config* cfg, size_t* bytes) {
  if (!bytes) return LLAMA_ERR_INVALID_ARG;
  TRY(check_config(cfg));
  *bytes = make_layout(cfg, sm_count_or_default()).total;
  return LLAMA_OK;
}

int llama_init(const llama_config* cfg, const llama_weights* w, void* workspace,
               size_t workspace_bytes, void* stream, llama_ctx** out) {
  if (!out || !w) return LLAMA_ERR_INVALID_ARG;
  *out = nullptr;
  TRY(check_config(cfg));
  if (!w->layers) return LLAMA_ERR_INVALID_ARG;
  if (cfg->has_embed_head && (!w->embed || !w->final_norm || !w->lm_head))
    return LLAMA_ERR_INVALID_ARG;
  const bool w8 = cfg->weight_dtype == LLAMA_W_E4M3;
  for (int l = 0; l < cfg->n_layers; ++l) {
    const llama_layer_weights& lw = w->layers[l];
    const void* ps[7] = {lw.attn_norm, lw.wqkv, lw.wo, lw.ffn_norm, lw.w_gate, lw.w_up, lw.w_down};
    for (const void* p : ps)
      if (!p || !aligned16(p)) return LLAMA_ERR_INVALID_ARG;
    if (w8) {
      const float* sc[5] = {lw.wqkv_scale, lw.wo_scale, lw.w_gate_scale, lw.w_up_scale,
                            lw.w_down_scale};
      for (const float* p : sc)
        if (!p || (reinterpret_cast<uintptr_t>(p) % 4) != 0) return LLAMA_ERR_INVALID_ARG;
    }
  }
  if (cfg->has_embed_head && (!aligned16(w->embed) || !aligned16(w->lm_head)))
    return LLAMA_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0)
    return LLAMA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return LLAMA_ERR_CUDA;
  }
  if (!load_encode()) return LLAMA_ERR_CUDA;
  // LLAMA_GB300_PDL=0: launch in plain stream order (no programmatic overlap)
  const char* pdl = getenv("LLAMA_GB300_PDL");
  set_pdl(!(pdl && pdl[0] == '0'));
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  Layout L = make_layout(cfg, sms);
  if (workspace_bytes < L.total) return LLAMA_ERR_WORKSPACE;
  llama_ctx* c = new (std::nothrow) llama_ctx();
  if (!c) return LLAMA_ERR_INVALID_ARG;
  c->cfg = *cfg;
  c->stream = reinterpret_cast<cudaStream_t>(stream);
  c->device = dev;
  c->sm_count = sms;
  c->es = elem_size(cfg->dtype);
  c->embed = w->embed;
  c->final_norm = w->final_norm;
  c->lm_head = w->lm_head;
  c->layers.assign(w->layers, w->layers + cfg->n_layers);
  c->ws = reinterpret_cast<char*>(workspace);
  c->L = L;
  c->status = c->at<uint32_t>(L.status);
  c->rope = c->at<float2>(L.rope);
  int rc = LLAMA_OK;
  if (cudaMemsetAsync(c->ws, 0, L.rope, c->stream) != cudaSuccess) rc = LLAMA_ERR_CUDA;
  if (rc == LLAMA_OK &&
      launch_rope_table(c->rope, cfg->max_seq, cfg->head_dim, (double)cfg->rope_theta,
                        c->stream) != cudaSuccess)
    rc = LLAMA_ERR_CUDA;
  c->launches = 1;
  if (rc == LLAMA_OK && cfg->dtype == LLAMA_BF16) {  // weight descriptors
    const uint64_t H = cfg->hidden, d = cfg->head_dim, nq = cfg->n_q_heads,
                   nkv = cfg->n_kv_heads, I = cfg->intermediate;
    for (const auto& lw : c->layers) {
      if (w8) {
        c->wscale[lw.wqkv] = lw.wqkv_scale;
        c->wscale[lw.wo] = lw.wo_scale;
        c->wscale[lw.w_gate] = lw.w_gate_scale;
        c->wscale[lw.w_up] = lw.w_up_scale;
        c->wscale[lw.w_down] = lw.w_down_scale;
        if (!map2d_u8(c, lw.wqkv, (nq + 2 * nkv) * d, H) || !map2d_u8(c, lw.wo, H, nq * d) ||
            !map2d_u8(c, lw.w_gate, I, H) || !map2d_u8(c, lw.w_up, I, H) ||
            !map2d_u8(c, lw.w_down, H, I))
          rc = LLAMA_ERR_CUDA;
      } else if (!map2d(c, lw.wqkv, (nq + 2 * nkv) * d, H, 128) ||
                 !map2d(c, lw.wo, H, nq * d, 128) || !map2d(c, lw.w_gate, I, H, 128) ||
                 !map2d(c, lw.w_up, I, H, 128) || !map2d(c, lw.w_down, H, I, 128)) {
        rc = LLAMA_ERR_CUDA;
      }
    }
    if (cfg->has_embed_head && !map2d(c, c->lm_head, cfg->vocab, H, 128)) rc = LLAMA_ERR_CUDA;
  }
  if (rc != LLAMA_OK) {
    delete c;
    return rc;
  }
  *out = c;
  return LLAMA_OK;
}

int llama_set_stream(llama_ctx* c, void* stream) {
  TRY(check_ctx(c));
  c->stream = reinterpret_cast<cudaStream_t>(stream);
  return LLAMA_OK;
}

int llama_free(llama_ctx* c) {
  if (!c) return LLAMA_ERR_INVALID_ARG;
  if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
  if (c->graph) cudaGraphDestroy(c->graph);
  for (auto& v : c->ev)
    for (auto& pr : v) {
      cudaEventDestroy(pr.first);
      cudaEventDestroy(pr.second);
    }
  delete c;
  return LLAMA_OK;
}

int llama_prefill(llama_ctx* c, const int32_t* tokens, int32_t B, int32_t T, const llama_kv* kv,
                  float* logits, int32_t* next_ids) {
  TRY(check_ctx(c));
  const llama_config& cf = c->cfg;
  if (!cf.has_embed_head) return LLAMA_ERR_UNSUPPORTED;
  if (!tokens || !logits || B < 1 || T < 1) return LLAMA_ERR_INVALID_ARG;
  if (B > cf.max_batch || (int64_t)B * T > cf.max_tokens || T > cf.max_seq)
    return LLAMA_ERR_OUT_OF_RANGE;
  TRY(check_kv(c, kv, B));
  const int cap = kv->page_size ? kv->max_pages_per_seq * kv->page_size : kv->capacity;
  if (T > cap) return LLAMA_ERR_OUT_OF_RANGE;
  const int rows = B * T;
  float* x = c->at<float>(c->L.x);
  {
    Prof pf(c, LLAMA_KERNEL_EMBED);
    c->launches++;
    TRY(cuda_rc(launch_embed(cf.dtype, tokens, c->embed, cf.vocab, cf.hidden, rows, x, c->status,
                             c->stream)));
  }
  for (int l = 0; l < cf.n_layers; ++l) TRY(run_layer(c, l, x, rows, B, T, nullptr, kv, true));
  return run_head(c, x, B, T, T - 1, logits, next_ids);
}

namespace {
int check_extend(const llama_ctx* c, int32_t n_rows, const int32_t* cu_rows,
                 const int32_t* start_pos, int32_t B, int32_t max_rows, const llama_kv* kv) {
  const llama_config& cf = c->cfg;
  if (!cu_rows || !start_pos || B < 1 || n_rows < 1 || max_rows < 1 || max_rows > n_rows)
    return LLAMA_ERR_INVALID_ARG;
  if (cf.dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (B > cf.max_batch || n_rows > std::max(cf.max_batch, cf.max_tokens))
    return LLAMA_ERR_OUT_OF_RANGE;
  TRY(check_kv(c, kv, B));
  return kv->kv_dtype == LLAMA_KV_MODEL ? LLAMA_OK : LLAMA_ERR_UNSUPPORTED;
}
}  // namespace

int llama_extend(llama_ctx* c, const int32_t* tokens, int32_t n_rows, const int32_t* cu_rows,
                 const int32_t* start_pos, int32_t B, int32_t max_rows, const llama_kv* kv,
                 float* logits, int32_t* next_ids) {
  TRY(check_ctx(c));
  const llama_config& cf = c->cfg;
  if (!cf.has_embed_head) return LLAMA_ERR_UNSUPPORTED;
  if (!tokens || !logits) return LLAMA_ERR_INVALID_ARG;
  TRY(check_extend(c, n_rows, cu_rows, start_pos, B, max_rows, kv));
  float* x = c->at<float>(c->L.x);
  {
    Prof pf(c, LLAMA_KERNEL_EMBED);
    c->launches++;
    TRY(cuda_rc(launch_embed(cf.dtype, tokens, c->embed, cf.vocab, cf.hidden, n_rows, x, c->status,
                             c->stream)));
  }
  const RowMap rm{cu_rows, start_pos, B, max_rows};
  for (int l = 0; l < cf.n_layers; ++l)
    TRY(run_layer(c, l, x, n_rows, B, 0, nullptr, kv, false, &rm));
  return run_head(c, x, B, 0, 0, logits, next_ids, cu_rows + 1, n_rows);
}

int llama_extend_hidden(llama_ctx* c, float* hidden, int32_t n_rows, const int32_t* cu_rows,
                        const int32_t* start_pos, int32_t B, int32_t max_rows,
                        const llama_kv* kv) {
  TRY(check_ctx(c));
  if (!hidden) return LLAMA_ERR_INVALID_ARG;
  TRY(check_extend(c, n_rows, cu_rows, start_pos, B, max_rows, kv));
  const RowMap rm{cu_rows, start_pos, B, max_rows};
  for (int l = 0; l < c->cfg.n_layers; ++l)
    TRY(run_layer(c, l, hidden, n_rows, B, 0, nullptr, kv, false, &rm));
  return LLAMA_OK;
}

int llama_decode_step(llama_ctx* c, const int32_t* tokens, const int32_t* positions, int32_t B,
                      const llama_kv* kv, float* logits, int32_t* next_ids) {
  TRY(check_ctx(c));
  const llama_config& cf = c->cfg;
  if (!cf.has_embed_head) return LLAMA_ERR_UNSUPPORTED;
  if (!tokens || !positions || !logits || B < 1) return LLAMA_ERR_INVALID_ARG;
  if (B > cf.max_batch) return LLAMA_ERR_OUT_OF_RANGE;
  TRY(check_kv(c, kv, B));
  float* x = c->at<float>(c->L.x);
  {
    Prof pf(c, LLAMA_KERNEL_EMBED);
    c->launches++;
    TRY(cuda_rc(launch_embed(cf.dtype, tokens, c->embed, cf.vocab, cf.hidden, B, x, c->status,
                             c->stream)));
  }
  for (int l = 0; l < cf.n_layers; ++l) TRY(run_layer(c, l, x, B, B, 1, positions, kv, false));
  return run_head(c, x, B, 1, 0, logits, next_ids);
}

int llama_decode_step_host(llama_ctx* c, const int32_t* tokens_host,
                           const int32_t* positions_host, int32_t B, const llama_kv* kv,
                           float* logits_host, int32_t* next_ids_host) {
  TRY(check_ctx(c));
  if (!tokens_host || !positions_host || B < 1) return LLAMA_ERR_INVALID_ARG;
  if (B > c->cfg.max_batch) return LLAMA_ERR_OUT_OF_RANGE;
  int32_t* tok = c->at<int32_t>(c->L.tok);
  int32_t* pos = c->at<int32_t>(c->L.pos);
  float* lg = c->at<float>(c->L.logits);
  int32_t* ids = c->at<int32_t>(c->L.ids);
  const size_t nb = (size_t)B * sizeof(int32_t);
  if (cudaMemcpyAsync(tok, tokens_host, nb, cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
      cudaMemcpyAsync(pos, positions_host, nb, cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  TRY(llama_decode_step(c, tok, pos, B, kv, lg, ids));
  if (logits_host &&
      cudaMemcpyAsync(logits_host, lg, (size_t)B * c->cfg.vocab * sizeof(float),
                      cudaMemcpyDeviceToHost, c->stream) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  if (next_ids_host &&
      cudaMemcpyAsync(next_ids_host, ids, nb, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  return llama_sync_status(c);
}

int llama_prefill_hidden(llama_ctx* c, float* hidden, int32_t B, int32_t T, const llama_kv* kv) {
  TRY(check_ctx(c));
  const llama_config& cf = c->cfg;
  if (!hidden || B < 1 || T < 1) return LLAMA_ERR_INVALID_ARG;
  if (B > cf.max_batch || (int64_t)B * T > cf.max_tokens || T > cf.max_seq)
    return LLAMA_ERR_OUT_OF_RANGE;
  TRY(check_kv(c, kv, B));
  const int cap = kv->page_size ? kv->max_pages_per_seq * kv->page_size : kv->capacity;
  if (T > cap) return LLAMA_ERR_OUT_OF_RANGE;
  for (int l = 0; l < cf.n_layers; ++l)
    TRY(run_layer(c, l, hidden, B * T, B, T, nullptr, kv, true));
  return LLAMA_OK;
}

int llama_decode_hidden(llama_ctx* c, float* hidden, const int32_t* positions, int32_t B,
                        const llama_kv* kv) {
  TRY(check_ctx(c));
  if (!hidden || !positions || B < 1) return LLAMA_ERR_INVALID_ARG;
  if (B > c->cfg.max_batch) return LLAMA_ERR_OUT_OF_RANGE;
  TRY(check_kv(c, kv, B));
  for (int l = 0; l < c->cfg.n_layers; ++l)
    TRY(run_layer(c, l, hidden, B, B, 1, positions, kv, false));
  return LLAMA_OK;
}

int llama_graph_capture_decode(llama_ctx* c, const int32_t* tokens, int32_t* positions, int32_t B,
                               const llama_kv* kv, float* logits, int32_t* next_ids,
                               int32_t advance) {
  TRY(check_ctx(c));
  if (!c->stream) return LLAMA_ERR_UNSUPPORTED;  // the legacy stream cannot be captured
  if (!tokens || !positions || !logits || B < 1) return LLAMA_ERR_INVALID_ARG;
  if (advance != 0 && advance != 1) return LLAMA_ERR_INVALID_ARG;
  if (c->graph_exec) {
    cudaGraphExecDestroy(c->graph_exec);
    c->graph_exec = nullptr;
  }
  if (c->graph) {
    cudaGraphDestroy(c->graph);
    c->graph = nullptr;
  }
  const uint32_t prof = c->prof_mask;
  c->prof_mask = 0;  // no timing events inside the graph
  if (cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    c->prof_mask = prof;
    return LLAMA_ERR_CUDA;
  }
  const int64_t n0 = c->launches;
  int rc = llama_decode_step(c, tokens, positions, B, kv, logits, next_ids);
  if (rc == LLAMA_OK && advance) {
    rc = cuda_rc(launch_advance_positions(positions, B, c->stream));
    c->launches++;
  }
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(c->stream, &g);
  c->prof_mask = prof;
  c->graph_launches = c->launches - n0;
  c->launches = n0;
  if (rc != LLAMA_OK || ec != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    cudaGetLastError();
    return rc != LLAMA_OK ? rc : LLAMA_ERR_CUDA;
  }
  if (cudaGraphInstantiate(&c->graph_exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return LLAMA_ERR_CUDA;
  }
  c->graph = g;
  return LLAMA_OK;
}

int llama_graph_launch(llama_ctx* c) {
  TRY(check_ctx(c));
  if (!c->graph_exec) return LLAMA_ERR_INVALID_ARG;
  if (cudaGraphLaunch(c->graph_exec, c->stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  c->launches += c->graph_launches;
  return LLAMA_OK;
}

int llama_sync_status(llama_ctx* c) {
  TRY(check_ctx(c));
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  uint32_t flags = 0;
  if (cudaMemcpy(&flags, c->status, sizeof(flags), cudaMemcpyDeviceToHost) != cudaSuccess)
    return LLAMA_ERR_CUDA;
  c->last_flags = flags;
  if (flags) {
    if (cudaMemset(c->status, 0, sizeof(uint32_t)) != cudaSuccess) return LLAMA_ERR_CUDA;
    return LLAMA_ERR_DEVICE_CHECK;
  }
  return LLAMA_OK;
}

uint32_t llama_last_device_flags(const llama_ctx* c) { return c ? c->last_flags : 0u; }

int32_t llama_bounds_checked(void) {
#if defined(LLAMA_BOUNDS_CHECK) && LLAMA_BOUNDS_CHECK
  return 1;
#else
  return 0;
#endif
}

int llama_quantize_rows_e4m3(const void* w, int32_t rows, int32_t cols, void* codes,
                             float* scales, void* stream) {
  if (!w || !codes || !scales || rows < 1 || cols < 16 || cols % 16 != 0)
    return LLAMA_ERR_INVALID_ARG;
  if (!aligned16(w) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) % 4) != 0)
    return LLAMA_ERR_INVALID_ARG;
  return cuda_rc(launch_quantize_rows_e4m3(w, rows, cols, codes, scales,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int llama_check_wait_timeout(llama_ctx* c, int32_t limit_us) {
  TRY(check_ctx(c));
  if (limit_us < 1 || limit_us > 1000000) return LLAMA_ERR_INVALID_ARG;
  c->launches++;
  return cuda_rc(launch_wait_check(c->status, (uint64_t)limit_us * 1000u, c->stream));
}

int llama_profile_enable(llama_ctx* c, uint32_t mask) {
  TRY(check_ctx(c));
  c->prof_mask = mask;
  for (size_t& u : c->ev_used) u = 0;
  return LLAMA_OK;
}

int llama_profile_read(llama_ctx* c, int32_t kind, double* total_ms, int64_t* launches) {
  TRY(check_ctx(c));
  if (kind < 0 || kind >= LLAMA_KERNEL_COUNT || !total_ms || !launches)
    return LLAMA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(c->stream) != cudaSuccess) return LLAMA_ERR_CUDA;
  double tot = 0.0;
  for (size_t i = 0; i < c->ev_used[kind]; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, c->ev[kind][i].first, c->ev[kind][i].second) != cudaSuccess)
      return LLAMA_ERR_CUDA;
    tot += ms;
  }
  *total_ms = tot;
  *launches = (int64_t)c->ev_used[kind];
  c->ev_used[kind] = 0;
  return LLAMA_OK;
}

int64_t llama_launch_count(const llama_ctx* c) { return c ? c->launches : 0; }

// ---------------------------------------------------------------- single operations
int llama_op_rmsnorm(llama_ctx* c, const float* x, int32_t rows, int32_t in_stride,
                     int32_t in_offset, const void* gamma, void* out) {
  TRY(check_ctx(c));
  if (!x || !gamma || !out || rows < 1 || in_stride < 1 || in_offset < 0)
    return LLAMA_ERR_INVALID_ARG;
  return do_rmsnorm(c, x, rows, in_stride, in_offset, gamma, out);
}

int llama_op_linear(llama_ctx* c, const void* x, int32_t n_rows, const void* w, const void* w_up,
                    int32_t M, int32_t K, int32_t epilogue, void* out) {
  TRY(check_ctx(c));
  if (!x || !w || !out || n_rows < 1 || M < 1 || K < 1) return LLAMA_ERR_INVALID_ARG;
  const int split = (epilogue & LLAMA_EPI_SPLIT_X) ? 1 : 0;
  epilogue &= ~LLAMA_EPI_SPLIT_X;
  if (epilogue < LLAMA_EPI_STORE_F32 || epilogue > LLAMA_EPI_SWIGLU) return LLAMA_ERR_INVALID_ARG;
  if (epilogue == LLAMA_EPI_SWIGLU && !w_up) return LLAMA_ERR_INVALID_ARG;
  if (c->cfg.dtype == LLAMA_BF16 && K % 8 != 0) return LLAMA_ERR_UNSUPPORTED;
  if (split && c->cfg.dtype != LLAMA_BF16) return LLAMA_ERR_UNSUPPORTED;
  if (n_rows > std::max(c->cfg.max_batch, c->cfg.max_tokens)) return LLAMA_ERR_OUT_OF_RANGE;
  const bool t_out = epilogue == LLAMA_EPI_SWIGLU || epilogue == LLAMA_EPI_STORE_T;
  return do_gemm(c, epilogue, x, n_rows, K, w, epilogue == LLAMA_EPI_SWIGLU ? w_up : nullptr, M,
                 out, M, split, (split && t_out) ? (size_t)round16(n_rows) * M : 0);
}

int llama_op_rope_append(llama_ctx* c, const float* qkv, int32_t rows, int32_t rows_per_seq,
                         const int32_t* positions, int32_t layer, const llama_kv* kv, void* q_out,
                         void* k_out, void* v_out) {
  TRY(check_ctx(c));
  if (!qkv || !q_out || rows < 1 || rows_per_seq < 1 || layer < 0 || layer >= c->cfg.n_layers)
    return LLAMA_ERR_INVALID_ARG;
  TRY(check_kv(c, kv, (rows + rows_per_seq - 1) / rows_per_seq));
  return do_rope_append(c, qkv, rows, rows_per_seq, positions, layer, kv, q_out, k_out, v_out);
}

int llama_op_attention_decode(llama_ctx* c, const void* q, const int32_t* positions, int32_t B,
                              int32_t layer, const llama_kv* kv, void* out) {
  TRY(check_ctx(c));
  if (!q || !positions || !out || B < 1 || layer < 0 || layer >= c->cfg.n_layers)
    return LLAMA_ERR_INVALID_ARG;
  if (B > c->cfg.max_batch) return LLAMA_ERR_OUT_OF_RANGE;
  TRY(check_kv(c, kv, B));
  return do_attn_decode(c, q, positions, B, layer, kv, out);
}

int llama_op_attention_prefill(llama_ctx* c, const void* q, const void* k, const void* v,
                               int32_t B, int32_t T, void* out) {
  TRY(check_ctx(c));
  if (!q || !k || !v || !out || B < 1 || T < 1) return LLAMA_ERR_INVALID_ARG;
  if (c->cfg.dtype == LLAMA_F32 && (size_t)(T + c->cfg.head_dim + 32) * 4 > 200 * 1024)
    return LLAMA_ERR_OUT_OF_RANGE;
  return do_attn_prefill(c, q, k, v, B, T, out);
}

int llama_op_embed(llama_ctx* c, const int32_t* tokens, int32_t n, void* out) {
  TRY(check_ctx(c));
  if (!c->cfg.has_embed_head) return LLAMA_ERR_UNSUPPORTED;
  if (!tokens || !out || n < 1) return LLAMA_ERR_INVALID_ARG;
  Prof pf(c, LLAMA_KERNEL_EMBED);
  c->launches++;
  return cuda_rc(launch_embed(c->cfg.dtype, tokens, c->embed, c->cfg.vocab, c->cfg.hidden, n,
                              reinterpret_cast<float*>(out), c->status, c->stream));
}

int llama_sample(llama_ctx* c, const float* logits, int32_t B, int32_t V, const llama_sampling* sp,
                 const int32_t* history, const int32_t* history_len, int32_t history_stride,
                 const float* uniforms, int32_t* next_ids) {
  TRY(check_ctx(c));
  if (!logits || !sp || !uniforms || !next_ids || B < 1) return LLAMA_ERR_INVALID_ARG;
  if (!(sp->temperature >= 0.f) || !(sp->top_p > 0.f && sp->top_p <= 1.f) ||
      !(sp->repetition_penalty > 0.f) || !std::isfinite(sp->temperature) ||
      !std::isfinite(sp->repetition_penalty))
    return LLAMA_ERR_INVALID_ARG;
  if (history && (!history_len || history_stride < 0)) return LLAMA_ERR_INVALID_ARG;
  if (V < 1) return LLAMA_ERR_INVALID_ARG;
  if (V > kSampleMaxVocab) return LLAMA_ERR_UNSUPPORTED;
  SampleCall sc{};
  sc.logits = logits;
  sc.B = B;
  sc.V = V;
  sc.ldl = V;
  sc.temperature = sp->temperature;
  sc.top_k = sp->top_k;
  sc.top_p = sp->top_p;
  sc.penalty = sp->repetition_penalty;
  sc.history = history;
  sc.history_len = history_len;
  sc.history_stride = history_stride;
  sc.uniforms = uniforms;
  sc.next_ids = next_ids;
  sc.status = c->status;
  Prof pf(c, LLAMA_KERNEL_SAMPLE);
  c->launches++;
  return cuda_rc(launch_sample(sc, c->stream));
}

int llama_op_argmax(llama_ctx* c, const float* logits, int32_t B, int32_t V, int32_t* ids) {
  TRY(check_ctx(c));
  if (!logits || !ids || B < 1 || V < 1) return LLAMA_ERR_INVALID_ARG;
  Prof pf(c, LLAMA_KERNEL_ARGMAX);
  c->launches++;
  return cuda_rc(launch_argmax(logits, B, V, ids, c->stream));
}

}  // extern "C"
