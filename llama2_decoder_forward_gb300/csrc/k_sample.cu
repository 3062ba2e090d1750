// Token sampling from the LM head's logits ("Llama2架构与推理全解析" §2.5 from
// logits to sampling, §3.3 sampling parameters; "Llama2架构全景解析"
// §2.2 step 3, probs = softmax(logits / T) and a draw).
//
// One CTA of 512 threads per sequence. Thread t owns the CH consecutive
// vocabulary entries [t*CH, t*CH + CH): the row is read along its length
// (coalesced) into shared memory and each thread takes its entries from there
// (the slot index XORed with the lane, so neither side has bank conflicts);
// their scaled logits live in its registers as order-preserving 32-bit keys,
// a 64-bit mask marks the entries still kept, and their unnormalised
// probabilities are stored in shared memory transposed (entry j of thread t
// at j*512 + t). Steps, in the order of the definition:
//   1. repetition penalty: the sequence's history marks a bitmap; marked
//      logits are divided by r when positive, multiplied by r otherwise;
//   2. temperature: s = z / T (T == 0: argmax, lowest index on ties); the
//      divisions are products with 1/r and 1/T;
//   3. top-k: the k-th largest key by a radix select, 4 bits per pass from
//      the top: each pass counts the keys that still match the threshold's
//      prefix in 16 buckets of their next 4 bits and keeps the bucket where
//      the count from the top reaches k (once the tied keys fit, they move to
//      a short list that the remaining passes read instead); the candidates
//      start as the keys >= the smallest of the first k threads' maxima, a
//      bound the k-th largest key cannot be below; ties at the threshold are
//      kept in ascending index order;
//   4. e = exp(s - max s) over the kept entries;
//   5. top-p: the same radix select over the kept mass (sum of e per bucket)
//      finds the smallest prefix of the descending order whose mass reaches
//      p * sum(e); ties at the threshold are kept in index order while the
//      mass is still short of it;
//   6. draw: u * sum(e) is located in the running sum of e in ascending
//      vocabulary order (the last kept entry if rounding leaves none).
// Bucket totals are per-thread parts in shared memory added in a fixed
// order, and so is every other reduction and scan, so a draw is
// reproducible.
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

// Exclusive prefix of v over threads in thread order (and, through `total`,
// the sum over all threads).
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* red, T* total = nullptr) {
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
  if (total) {
    T all = off;
    for (int w = warp; w < kSampleWarps; ++w) all = all + red[w];
    *total = all;
  }
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

constexpr int kBins = 16;        // radix of the threshold searches (4 bits per pass)
constexpr int kListMax = 4096;   // entries a search moves to its shared-memory list
static_assert(kSampleWarps == kBins, "one warp adds up each bucket");

// Staging slot of entry j of thread t (see the header).
template <int CH>
__device__ __forceinline__ int stage_pos(int t, int j) {
  return t * CH + (CH >= 32 ? (j ^ (t & 31)) : j);
}

// Bucket totals of one radix pass: hist[d * 512 + t] is thread t's part of
// bucket d; warp d adds bucket d over the threads in a fixed order (lane l
// takes threads l, l + 32, ..., l + 480; then a butterfly) and its lane 0
// writes tot[d].
template <typename T>
__device__ __forceinline__ void bucket_totals(const T* hist, T* tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T* h = hist + warp * SAMPLE_THREADS + lane;
  T c[4];  // four chains of four threads each, then their pairwise sum
#pragma unroll
  for (int q = 0; q < 4; ++q)
    c[q] = ((h[32 * (4 * q)] + h[32 * (4 * q + 1)]) + h[32 * (4 * q + 2)]) + h[32 * (4 * q + 3)];
  const T r = warp_reduce((c[0] + c[1]) + (c[2] + c[3]), [](T x, T y) { return x + y; });
  if (lane == 0) tot[warp] = r;
}

// The bucket of a pass: from the top, the first bucket d at which the amount
// above the current prefix (`above`) plus buckets d..15 reaches `target`;
// bucket 0 when none does (for masses only rounding can cause that). Returns
// d and adds the buckets above d to `above`. Every thread reads the 16 totals
// and takes the same decision.
template <typename T>
__device__ __forceinline__ uint32_t pick_bucket(const T* tot, T target, T& above) {
  T c = above;
  uint32_t sel = 0;
  bool found = false;
#pragma unroll
  for (int d = kBins - 1; d >= 1; --d) {
    const T v = tot[d];
    if (!found && c + v >= target) {
      sel = (uint32_t)d;
      found = true;
    }
    if (!found) c = c + v;
  }
  above = c;
  return sel;
}

// Is key k still tied with the threshold, whose bits above `shift + 4` are
// those of kap?
__device__ __forceinline__ bool on_prefix(uint32_t k, uint32_t kap, int shift) {
  return shift >= 28 || (k >> (shift + 4)) == (kap >> (shift + 4));
}

// Radix select among this thread's candidate entries `cand` (keys in key[],
// weights w(j): 1 to count, e to weigh): the largest key kap such that the
// weight of the candidates >= kap reaches `target` (4 bits per pass from the
// top). While more than kListMax candidates are tied with the prefix, a pass
// reads every candidate from the registers; then the tied ones move to the
// shared-memory list (key, weight) and the remaining passes read the list.
// n_tied: the number of candidates when known (counting), else -1. Returns
// kap; `above` gets the weight of the candidates > kap and `tie` this
// thread's candidates equal to kap.
template <int CH, typename T, typename W>
__device__ __forceinline__ uint32_t radix_select(const uint32_t (&key)[CH], uint64_t cand,
                                                 int n_tied, T target, W w, T* hist, T* tot,
                                                 uint32_t* lkey, T* lw, int* red_i, T& above,
                                                 uint64_t& tie) {
  const int t = threadIdx.x;
  uint32_t kap = 0;
  above = T(0);
  bool listed = false;
  int n = 0;
#pragma unroll 1
  for (int shift = 32 - 4; shift >= 0; shift -= 4) {
    if (!listed && n_tied <= kListMax) {  // move the tied candidates to the list if they fit
      uint64_t act = 0;
#pragma unroll
      for (int j = 0; j < CH; ++j)
        act |= (uint64_t)(((cand >> j) & 1ull) && on_prefix(key[j], kap, shift)) << j;
      int total;
      int off = block_exclusive_scan(__popcll((long long)act), red_i, &total);
      if (total <= kListMax) {
#pragma unroll
        for (int j = 0; j < CH; ++j)
          if ((act >> j) & 1ull) {
            lkey[off] = key[j];
            lw[off] = w(j);
            ++off;
          }
        listed = true;
        n = total;
        __syncthreads();
      }
    }
#pragma unroll
    for (int d = 0; d < kBins; ++d) hist[d * SAMPLE_THREADS + t] = T(0);
    if (listed) {
      for (int i = t; i < n; i += SAMPLE_THREADS) {
        const uint32_t k = lkey[i];
        if (on_prefix(k, kap, shift)) hist[((k >> shift) & 15u) * SAMPLE_THREADS + t] += lw[i];
      }
    } else if (cand) {  // every candidate, branch-free (weight 0 when off the prefix)
#pragma unroll
      for (int j = 0; j < CH; ++j) {
        const bool on = ((cand >> j) & 1ull) && on_prefix(key[j], kap, shift);
        hist[((key[j] >> shift) & 15u) * SAMPLE_THREADS + t] += on ? w(j) : T(0);
      }
    }
    __syncthreads();
    bucket_totals(hist, tot);
    __syncthreads();
    const uint32_t sel = pick_bucket(tot, target, above);
    kap |= sel << shift;
    n_tied = n_tied < 0 ? -1 : (int)tot[sel];  // counting: the candidates now tied
  }
  tie = 0;
#pragma unroll
  for (int j = 0; j < CH; ++j) tie |= (uint64_t)(((cand >> j) & 1ull) && key[j] == kap) << j;
  return kap;
}

template <int CH>
__global__ void __launch_bounds__(SAMPLE_THREADS, 1) sample_kernel(SampleArgs a) {
  grid_dep_wait();  // the logits come from the LM head
  grid_dep_launch();
  // [CH][512]: first the staged row, then the unnormalised probabilities
  extern __shared__ float e_sm[];
  float* hist = e_sm + CH * SAMPLE_THREADS;  // [16][512] per-thread bucket parts
  int* hist_i = reinterpret_cast<int*>(hist);
  uint32_t* lkey = reinterpret_cast<uint32_t*>(hist + kBins * SAMPLE_THREADS);  // search list
  float* lw = reinterpret_cast<float*>(lkey + kListMax);
  int* lw_i = reinterpret_cast<int*>(lw);
  uint32_t* seen = reinterpret_cast<uint32_t*>(lw + kListMax);  // history bitmap
  // bounds-check builds: the buffers and the bitmap fit the launch, and the
  // row fits the chunks
  if (!bc_smem(e_sm,
               (uint32_t)(((CH + kBins) * SAMPLE_THREADS + 2 * kListMax + ((a.V + 31) >> 5)) * 4),
               4, threadIdx.x == 0 ? a.status : nullptr) ||
      !bc_ok(a.V <= CH * SAMPLE_THREADS, threadIdx.x == 0 ? a.status : nullptr))
    return;
  __shared__ int red_i[kSampleWarps];
  __shared__ float red_f[kSampleWarps];
  __shared__ uint32_t red_u[kSampleWarps];
  __shared__ int tot_i[kBins];
  __shared__ float tot_f[kBins];
  const int b = blockIdx.x, t = threadIdx.x;
  const int V = a.V, v0 = t * CH;
  const float* row = a.logits + (size_t)b * a.ldl;
  auto add_f = [](float x, float y) { return x + y; };

  // the row, read along its length, into the staging slots
  {
    float z[CH];
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int v = t + SAMPLE_THREADS * k;
      z[k] = v < V ? row[v] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < CH; ++k) {
      const int v = t + SAMPLE_THREADS * k;
      e_sm[stage_pos<CH>(v / CH, v % CH)] = z[k];
    }
  }
  // 1. repetition penalty: mark the history's distinct ids
  const bool pen = a.penalty != 1.f && a.history != nullptr;
  if (pen) {
    const int nw = (V + 31) >> 5;
    for (int i = t; i < nw; i += SAMPLE_THREADS) seen[i] = 0u;
    __syncthreads();
    const int len = a.history_len ? a.history_len[b] : 0;
    const int32_t* hist_ids = a.history + (size_t)b * a.history_stride;
    for (int i = t; i < len; i += SAMPLE_THREADS) {
      const int id = hist_ids[i];
      if (id >= 0 && id < V)
        atomicOr(&seen[id >> 5], 1u << (id & 31));
      else
        flag(a.status, LLAMA_FLAG_TOKEN_RANGE);
    }
  }
  __syncthreads();
  // 2. the scaled logits as keys, one register each
  uint32_t key[CH];
  uint64_t kept = 0;
  {
    const float inv_t = a.temperature == 0.f ? 1.f : 1.f / a.temperature;
    const float inv_r = 1.f / a.penalty;
#pragma unroll
    for (int j = 0; j < CH; ++j) {
      const int v = v0 + j;
      float z = e_sm[stage_pos<CH>(t, j)];
      if (pen && v < V && ((seen[v >> 5] >> (v & 31)) & 1u)) z = z > 0.f ? z * inv_r : z * a.penalty;
      key[j] = float_key(z * inv_t);
      if (v < V) kept |= 1ull << j;
    }
  }

  // greedy limit: the largest key, lowest index on ties
  if (a.temperature == 0.f) {
    uint32_t best = 0;
    int bi = INT_MAX;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if (((kept >> j) & 1ull) && (key[j] > best || bi == INT_MAX)) {
        best = key[j];
        bi = v0 + j;
      }
    const uint32_t m = block_reduce(best, red_u, [](uint32_t x, uint32_t y) { return max(x, y); });
    const int w = block_reduce(best == m ? bi : INT_MAX, red_i,
                               [](int x, int y) { return min(x, y); });
    if (t == 0) a.next_ids[b] = w;
    return;
  }

  // 3. top-k: radix select of the k-th largest key among the kept entries
  if (a.top_k > 0 && a.top_k < V) {
    // Candidates: when k threads own entries, the keys >= L, the smallest of
    // the largest keys of threads 0..k-1. Those k keys are >= L, so the k-th
    // largest is too, and usually few keys pass (the search can then start on
    // the list).
    uint64_t cand = kept;
    int n_cand = V;
    if (a.top_k <= (V + CH - 1) / CH) {
      uint32_t tmax = 0;
#pragma unroll
      for (int j = 0; j < CH; ++j)
        if ((kept >> j) & 1ull) tmax = max(tmax, key[j]);
      const uint32_t L = block_reduce(t < a.top_k ? tmax : 0xffffffffu, red_u,
                                      [](uint32_t x, uint32_t y) { return min(x, y); });
      cand = 0;
#pragma unroll
      for (int j = 0; j < CH; ++j) cand |= (uint64_t)(((kept >> j) & 1ull) && key[j] >= L) << j;
      n_cand = -1;
    }
    int above;
    uint64_t act;
    const uint32_t kap = radix_select<CH>(key, cand, n_cand, a.top_k, [](int) { return 1; },
                                          hist_i, tot_i, lkey, lw_i, red_i, above, act);
    // kap is the k-th largest key: `above` entries exceed it, `act` equal it
    const int need = a.top_k - above;
    int rank = block_exclusive_scan(__popcll((long long)act), red_i);
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

  // 5. top-p: radix select over the kept mass
  if (a.top_p < 1.f) {
    const float target = a.top_p * Z1;
    float above;
    uint64_t act;
    const uint32_t kap =
        radix_select<CH>(key, kept, -1, target, [&](int j) { return e_sm[j * SAMPLE_THREADS + t]; },
                         hist, tot_f, lkey, lw, red_i, above, act);
    // kap: the smallest key of the prefix; `above` is the kept mass beyond it
    float tie_mass = 0.f;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if ((act >> j) & 1ull) tie_mass += e_sm[j * SAMPLE_THREADS + t];
    float before = block_exclusive_scan(tie_mass, red_f);
    uint64_t keep = 0;
#pragma unroll
    for (int j = 0; j < CH; ++j)
      if ((kept >> j) & 1ull) {
        if (key[j] > kap) keep |= 1ull << j;
        if (key[j] == kap) {
          if (above + before < target) keep |= 1ull << j;
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
  return ((size_t)(ch + kBins) * SAMPLE_THREADS + 2 * kListMax + (size_t)((V + 31) / 32)) * 4;
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
