// Decode attention for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// moment they need this kernel: a host framework that owns every byte of
// device memory through its own pool and forbids other allocators, a plugin
// loaded into such a framework, or code that runs while a stream is being
// captured into a CUDA graph, where an allocation would break the capture.
// The regular path needs a caller workspace for the key-split partial sums;
// this entry point keeps them in a fixed array that lives in the library's
// own device image instead, so nothing is allocated at call time.
//
// The array is kNoAllocScratchBytes (8 MiB) and exists once per GPU that
// loads the library, until the process exits. Calls share it: two calls that
// overlap on the GPU (different streams, or graphs replayed concurrently)
// race on it and must be serialised by the caller. Nothing in it has to start
// at zero: every key split writes its own slice before the merge reads it.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;

// Key-split partial sums of the decode attention (see the header comment).
static __device__ __align__(256) float g_attn_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};
bool g_prepared[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Once per device, with that device current: the scratch array's device
// address (the host-side symbol is only a stand-in and must never be handed
// to a kernel) and the kernels' shared-memory attributes.
int setup_device(int dev, void** scratch) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return LLAMA_ERR_UNSUPPORTED;
  if (!g_encode_fn) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return LLAMA_ERR_CUDA;
    g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (!g_prepared[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return LLAMA_ERR_CUDA;
    }
    if (llgb::attn_prepare() != cudaSuccess) return LLAMA_ERR_CUDA;
    g_scratch_addr[dev] = p;
    g_prepared[dev] = true;
  }
  *scratch = g_scratch_addr[dev];
  return LLAMA_OK;
}

bool encode_cache_map(CUtensorMap* m, void* base, uint64_t d, uint64_t rows, uint64_t layers,
                      uint32_t box_rows) {
  cuuint64_t dims[3] = {d, rows, layers};
  cuuint64_t strides[2] = {d * 2, d * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode_fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" int llama_attention_decode_noalloc(const llama_config* cfg, const void* q,
                                              const int32_t* positions, int32_t B, int32_t layer,
                                              const llama_kv* kv, void* out, void* stream) {
  if (!cfg || !q || !positions || !out || !kv || !kv->k || !kv->v || B < 1)
    return LLAMA_ERR_INVALID_ARG;
  if (cfg->dtype != LLAMA_BF16 || cfg->head_dim != 128 || kv->kv_dtype != LLAMA_KV_MODEL)
    return LLAMA_ERR_UNSUPPORTED;
  if (cfg->n_layers < 1 || cfg->n_q_heads < 1 || cfg->n_kv_heads < 1 || cfg->max_seq < 1 ||
      cfg->n_q_heads % cfg->n_kv_heads != 0 || layer < 0 || layer >= cfg->n_layers)
    return LLAMA_ERR_INVALID_ARG;
  if (cfg->n_q_heads / cfg->n_kv_heads > 16) return LLAMA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(out) || !aligned16(kv->k) || !aligned16(kv->v))
    return LLAMA_ERR_INVALID_ARG;
  const uint64_t nkv = cfg->n_kv_heads, d = cfg->head_dim;
  uint64_t rows;
  int cap_keys;
  if (kv->page_size == 0) {
    if (kv->capacity < 1 || kv->batch_capacity < B) return LLAMA_ERR_INVALID_ARG;
    rows = (uint64_t)kv->batch_capacity * nkv * kv->capacity;
    cap_keys = kv->capacity;
  } else {
    if (kv->page_size < 0 || kv->page_size % 16 != 0) return LLAMA_ERR_UNSUPPORTED;
    if (!kv->page_table || kv->n_pages < 1 || kv->max_pages_per_seq < 1)
      return LLAMA_ERR_INVALID_ARG;
    rows = (uint64_t)kv->n_pages * nkv * kv->page_size;
    cap_keys = kv->max_pages_per_seq * kv->page_size;
  }
  if (rows + 64 >= (1ull << 31)) return LLAMA_ERR_UNSUPPORTED;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return LLAMA_ERR_CUDA;
  }
  void* scratch = nullptr;
  const int rc = setup_device(dev, &scratch);
  if (rc != LLAMA_OK) return rc;

  // The split plan covers every slot of the cache (not only max_seq of them):
  // there is no status word here to report a position the plan would miss.
  const int max_keys = cap_keys;
  const size_t need = llgb::attn_decode_partial_bytes(B, cfg->n_q_heads, (int)d,
                                                      max_keys < 1 ? 1 : max_keys, sms, (int)nkv);
  if (need > kNoAllocScratchBytes) return LLAMA_ERR_OUT_OF_RANGE;

  CUtensorMap mk, mv, mk16, mv16;
  const int box_rows = llgb::attn_decode_box_rows(kv->page_size);
  if (!encode_cache_map(&mk, kv->k, d, rows, cfg->n_layers, box_rows) ||
      !encode_cache_map(&mv, kv->v, d, rows, cfg->n_layers, box_rows) ||
      !encode_cache_map(&mk16, kv->k, d, rows, cfg->n_layers, 16) ||
      !encode_cache_map(&mv16, kv->v, d, rows, cfg->n_layers, 16))
    return LLAMA_ERR_CUDA;
  llgb::AttnDecodeArgs a{};
  a.q = q;
  a.positions = positions;
  a.map_k = &mk;
  a.map_v = &mv;
  a.map_k16 = &mk16;
  a.map_v16 = &mv16;
  a.box_rows = box_rows;
  a.k_cache = kv->k;
  a.v_cache = kv->v;
  a.page_table = kv->page_table;
  a.out = out;
  a.out_lo = 0;
  a.partial = static_cast<float*>(scratch);
  a.partial_bytes = kNoAllocScratchBytes;
  a.status = nullptr;
  a.B = B;
  a.n_q = cfg->n_q_heads;
  a.n_kv = cfg->n_kv_heads;
  a.head_dim = (int)d;
  a.layer = layer;
  a.page_size = kv->page_size;
  a.capacity = kv->capacity;
  a.batch_cap = kv->batch_capacity;
  a.n_pages = kv->n_pages;
  a.max_pages = kv->max_pages_per_seq;
  a.max_keys = max_keys < 1 ? 1 : max_keys;
  a.sm_count = sms;
  return llgb::launch_attn_decode(LLAMA_BF16, a, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? LLAMA_OK
             : LLAMA_ERR_CUDA;
}
