// Token sampling from the LM head's logits ("Llama2架构与推理全解析" §2.5 from
// logits to sampling, §3.3 sampling parameters; "Llama2架构全景解析"
// §2.2 step 3, probs = softmax(logits / T) and a draw).
//
// One CTA of 512 threads per sequence. Thread t owns the CH consecutive
// vocabulary entries [t*CH, t*CH + CH): their scaled logits s live in its
// registers and their unnormalised probabilities e in shared memory, stored
// transposed (entry j of thread t at j*512 + t) so that the per-thread walks
// are conflict-free. Steps, in the order of the definition:
//   1. repetition penalty: the sequence's history marks a bitmap; marked
//      logits are divided by r when positive, multiplied by r otherwise;
//   2. temperature: s = z / T (T == 0: argmax, lowest index on ties);
//   3. top-k: the k-th largest s found by a bitwise search over the
//      order-preserving 32-bit key of s (count of keys >= candidate), ties
//      at the threshold kept in ascending index order;
//   4. e = exp(s - max s) over the kept entries;
//   5. top-p: the same search over the kept mass (sum of e over keys >=
//      candidate) finds the smallest prefix of the descending order whose
//      mass reaches p * sum(e); ties at the threshold are kept in index order
//      while the mass is still short of it;
//   6. draw: u * sum(e) is located in the running sum of e in ascending
//      vocabulary order (the last kept entry if rounding leaves none).
// Every reduction and scan runs in a fixed order, so a draw is reproducible.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace llgb {

constexpr int SAMPLE_THREADS = 512;
constexpr int kSampleWarps = SAMPLE_THREADS / 32;

// Order-preserving map of a float to an unsigned key (larger float, larger key).
__device__ __forceinline__ uint32_t float_key(float s) {
  const uint32_t b = __float_as_uint(s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <typename T, typename Op>
__device__ __forceinline__ T warp_reduce(T v, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide reduction: warp butterflies, then every thread folds the 16 warp
// results in warp order. `red` holds one value per warp; it is free again on
// return.
template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, T* red, Op op) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_reduce(v, op);
  if (lane == 0) red[warp] = v;
  __syncthreads();
  T r = red[0];
#pragma unroll 4
  for (int w = 1; w < kSampleWarps; ++w) r = op(r, red[w]);
  __syncthreads();
  return r;
}

// Exclusive prefix of v over threads in thread order.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x = x + y;
  }
  const T ex = __shfl_up_sync(0xffffffffu, x, 1);
  if (lane == 31) red[warp] = x;
  __syncthreads();
  T off = T(0);
  for (int w = 0; w < warp; ++w) off = off + red[w];
  __syncthreads();
  return off + (lane == 0 ? T(0) : ex);
}

struct SampleArgs {
  const float* logits;
  int ldl, V;
  float temperature, top_p, penalty;
  int top_k;
  const int32_t* history;
  const int32_t* history_len;
  int history_stride;
  const float* uniforms;
  int32_t* next_ids;
  uint32_t* status;
};

template <int CH>
__global__ void __launch_bounds__(SAMPLE_THREADS, 1) sample_kernel(SampleArgs a) {
  grid_dep_wait();  // the logits come from the LM head
  grid_dep_launch();
  extern __shared__ float e_sm[];  // [CH][512] unnormalised probabilities, then the bitmap
  uint32_t* seen = reinterpret_cast<uint32_t*>(e_sm + CH * SAMPLE_THREADS);
  // bounds-check builds: the probabilities and the bitmap fit the launch, and
  // the row fits the chunks
  if (!bc_smem(e_sm, (uint32_t)(CH * SAMPLE_THREADS * 4 + ((a.V + 31) >> 5) * 4), 4,
               threadIdx.x == 0 ? a.status : nullptr) ||
      !bc_ok(a.V <= CH * SAMPLE_THREADS, threadIdx.x == 0 ? a.status : nullptr))
    return;
  __shared__ int red_i[kSampleWarps];
  __shared__ float red_f[kSampleWarps];
  __shared__ uint32_t red_u[kSampleWarps];
  const int b = blockIdx.x, t = threadIdx.x;
  const int V = a.V, v0 = t * CH;
  const float* row = a.logits + (size_t)b * a.ldl;
  auto add_i = [](int x, int y) { return x + y; };
  auto add_f = [](float x, float y) { return x + y; };

  // 1. repetition penalty: mark the history's distinct ids
  const bool pen = a.penalty != 1.f && a.history != nullptr;
  if (pen) {
    const int nw = (V + 31) >> 5;
    for (int i = t; i < nw; i += SAMPLE_THREADS) seen[i] = 0u;
    __syncthreads();
    const int len = a.history_len ? a.history_len[b] : 0;
    const int32_t* hist = a.history + (size_t)b * a.history_stride;
    for (int i = t; i < len; i += SAMPLE_THREADS) {
      const int id = hist[i];
      if (id >= 0 && id < V)
        atomicOr(&seen[id >> 5], 1u << (id & 31));
      else
        flag(a.status, LLAMA_FLAG_TOKEN_RANGE);
    }
    __syncthreads();
  }
  // the scaled logits are kept as their order-preserving keys (one register each)
  uint32_t key[CH];
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    const int v = v0 + j;
    float z = v < V ? row[v] : -INFINITY;
    if (pen && v < V && ((seen[v >> 5] >> (v & 31)) & 1u)) z = z > 0.f ? z / a.penalty : z * a.penalty;
    key[j] = float_key(a.temperature == 0.f ? z : z / a.temperature);
  }

  // 2. greedy limit: the largest key, lowest index on ties
  if (a.temperature == 0.f) {
    uint32_t best = 0;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if (v0 + j < V && (key[j] > best || bi == INT_MAX)) {
        best = key[j];
        bi = v0 + j;
      }
    const uint32_t m = block_reduce(best, red_u, [](uint32_t x, uint32_t y) { return max(x, y); });
    const int w = block_reduce(best == m ? bi : INT_MAX, red_i,
                               [](int x, int y) { return min(x, y); });
    if (t == 0) a.next_ids[b] = w;
    return;
  }

  // 3. top-k
  uint64_t kept = 0;
#pragma unroll
  for (int j = 0; j < CH; ++j)
    if (v0 + j < V) kept |= 1ull << j;
  if (a.top_k > 0 && a.top_k < V) {
    uint32_t kap = 0;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = kap | (1u << bit);
      int c = 0;
#pragma unroll
      for (int j = 0; j < CH; ++j) c += ((kept >> j) & 1ull) && key[j] >= cand;
      if (block_reduce(c, red_i, add_i) >= a.top_k) kap = cand;
    }
    int gt = 0, ties = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if ((kept >> j) & 1ull) {
        gt += key[j] > kap;
        ties += key[j] == kap;
      }
    const int need = a.top_k - block_reduce(gt, red_i, add_i);
    int rank = block_exclusive_scan(ties, red_i);
    uint64_t keep = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if ((kept >> j) & 1ull) {
        if (key[j] > kap) keep |= 1ull << j;
        if (key[j] == kap) {
          if (rank < need) keep |= 1ull << j;
          ++rank;
        }
      }
    kept = keep;
  }

  // 4. unnormalised probabilities of the kept entries
  uint32_t kmax = 0;
#pragma unroll
  for (int j = 0; j < CH; ++j)
    if ((kept >> j) & 1ull) kmax = max(kmax, key[j]);
  const float mx =
      key_float(block_reduce(kmax, red_u, [](uint32_t x, uint32_t y) { return max(x, y); }));
  float tot = 0.f;
#pragma unroll
  for (int j = 0; j < CH; ++j) {
    const float e = ((kept >> j) & 1ull) ? expf(key_float(key[j]) - mx) : 0.f;
    e_sm[j * SAMPLE_THREADS + t] = e;
    tot += e;
  }
  const float Z1 = block_reduce(tot, red_f, add_f);

  // 5. top-p
  if (a.top_p < 1.f) {
    const float target = a.top_p * Z1;
    uint32_t kap = 0;
    for (int bit = 31; bit >= 0; --bit) {
      const uint32_t cand = kap | (1u << bit);
      float m = 0.f;
#pragma unroll
      for (int j = 0; j < CH; ++j)
        if (((kept >> j) & 1ull) && key[j] >= cand) m += e_sm[j * SAMPLE_THREADS + t];
      if (block_reduce(m, red_f, add_f) >= target) kap = cand;
    }
    float gt = 0.f, tie_mass = 0.f;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if ((kept >> j) & 1ull) {
        if (key[j] > kap) gt += e_sm[j * SAMPLE_THREADS + t];
        if (key[j] == kap) tie_mass += e_sm[j * SAMPLE_THREADS + t];
      }
    const float m_gt = block_reduce(gt, red_f, add_f);
    float before = block_exclusive_scan(tie_mass, red_f);
    uint64_t keep = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if ((kept >> j) & 1ull) {
        if (key[j] > kap) keep |= 1ull << j;
        if (key[j] == kap) {
          if (m_gt + before < target) keep |= 1ull << j;
          before += e_sm[j * SAMPLE_THREADS + t];
        }
      }
    kept = keep;
  }

  // 6. draw in ascending vocabulary order
  float mine = 0.f;
  int last = -1;
#pragma unroll
  for (int j = 0; j < CH; ++j)
    if ((kept >> j) & 1ull) {
      mine += e_sm[j * SAMPLE_THREADS + t];
      last = v0 + j;
    }
  const float Z2 = block_reduce(mine, red_f, add_f);
  const float goal = a.uniforms[b] * Z2;
  float c = block_exclusive_scan(mine, red_f);
  int pick = INT_MAX;
#pragma unroll
  for (int j = 0; j < CH; ++j)
    if ((kept >> j) & 1ull) {
      c += e_sm[j * SAMPLE_THREADS + t];
      if (c > goal && pick == INT_MAX) pick = v0 + j;
    }
  pick = block_reduce(pick, red_i, [](int x, int y) { return min(x, y); });
  if (pick == INT_MAX) pick = block_reduce(last, red_i, [](int x, int y) { return max(x, y); });
  if (t == 0) a.next_ids[b] = pick;
}

int sample_chunk(int V) {
  int ch = 1;
  while (ch * SAMPLE_THREADS < V) ch <<= 1;
  return ch;
}

size_t sample_smem_bytes(int V) {
  const int ch = sample_chunk(V);
  return (size_t)ch * SAMPLE_THREADS * sizeof(float) + (size_t)((V + 31) / 32) * 4;
}

template <int CH>
static cudaError_t set_sample_attr() {
  return cudaFuncSetAttribute(sample_kernel<CH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)sample_smem_bytes(CH * SAMPLE_THREADS));
}

cudaError_t sample_prepare() {
  cudaError_t e;
  if ((e = set_sample_attr<1>()) != cudaSuccess) return e;
  if ((e = set_sample_attr<2>()) != cudaSuccess) return e;
  if ((e = set_sample_attr<4>()) != cudaSuccess) return e;
  if ((e = set_sample_attr<8>()) != cudaSuccess) return e;
  if ((e = set_sample_attr<16>()) != cudaSuccess) return e;
  if ((e = set_sample_attr<32>()) != cudaSuccess) return e;
  return set_sample_attr<64>();
}

cudaError_t launch_sample(const SampleCall& c, cudaStream_t st) {
  SampleArgs a;
  a.logits = c.logits;
  a.ldl = c.ldl;
  a.V = c.V;
  a.temperature = c.temperature;
  a.top_p = c.top_p;
  a.penalty = c.penalty;
  a.top_k = c.top_k;
  a.history = c.history;
  a.history_len = c.history_len;
  a.history_stride = c.history_stride;
  a.uniforms = c.uniforms;
  a.next_ids = c.next_ids;
  a.status = c.status;
  const size_t sm = sample_smem_bytes(c.V);
  const dim3 grid(c.B), block(SAMPLE_THREADS);
  switch (sample_chunk(c.V)) {
    case 1: return launch_k(sample_kernel<1>, grid, block, sm, st, 0, a);
    case 2: return launch_k(sample_kernel<2>, grid, block, sm, st, 0, a);
    case 4: return launch_k(sample_kernel<4>, grid, block, sm, st, 0, a);
    case 8: return launch_k(sample_kernel<8>, grid, block, sm, st, 0, a);
    case 16: return launch_k(sample_kernel<16>, grid, block, sm, st, 0, a);
    case 32: return launch_k(sample_kernel<32>, grid, block, sm, st, 0, a);
    case 64: return launch_k(sample_kernel<64>, grid, block, sm, st, 0, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace llgb
