// Row-wise kernels of the decoder forward: embedding gather, RMSNorm, the
// RoPE table, RoPE + KV-cache append, and the greedy argmax.
//
// "Llama2架构与推理全解析": §2.3 (embedding lookup, residual stream),
// §1.2 (RMSNorm), §1.4 (RoPE), §2.4 (KV cache append), §2.5 (greedy choice).
#include "common.cuh"
#include "internal.h"

namespace llgb {

// ------------------------------------------------------------------ embedding
// out[r, :] = (fp32) table[tokens[r], :]. A token id outside [0, V) sets
// LLAMA_FLAG_TOKEN_RANGE and yields a zero row.
template <typename T>
__global__ void embed_kernel(const int32_t* __restrict__ tokens, const T* __restrict__ table,
                             int V, int H, float* __restrict__ out, uint32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = blockIdx.x;
  const int tok = tokens[r];
  const bool ok = tok >= 0 && tok < V;
  if (!ok && threadIdx.x == 0) flag(status, LLAMA_FLAG_TOKEN_RANGE);
  const T* src = table + (size_t)(ok ? tok : 0) * H;
  float* dst = out + (size_t)r * H;
  for (int i = threadIdx.x; i < H; i += blockDim.x) dst[i] = ok ? to_f32(src[i]) : 0.f;
}

// ------------------------------------------------------------------ RMSNorm
// One CTA per row: y = x / sqrt(mean(x^2) + eps) * gamma; statistics in fp32.
// Input row r is x + (r * in_stride + in_offset) * H. With lo_rows > 0 the bf16
// remainder y - bf16(y) is also written to row r + lo_rows (hi/lo operand pair).
template <typename T>
__device__ __forceinline__ void store_y(T* yr, size_t lo, int i, float v) {
  const T hi = from_f32<T>(v);
  yr[i] = hi;
  if (lo) yr[lo + i] = from_f32<T>(v - to_f32(hi));
}

template <typename T>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x, int in_stride,
                                                      int in_offset, const T* __restrict__ gamma,
                                                      int H, float eps, T* __restrict__ out,
                                                      int lo_rows, const int32_t* row_end,
                                                      int n_in, uint32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  const size_t lo = (size_t)lo_rows * H;
  __shared__ float red[8];
  const int r = blockIdx.x;
  const float* xr = x + ((size_t)r * in_stride + in_offset) * H;
  T* yr = out + (size_t)r * H;
  if (row_end) {  // the last row of packed sequence r
    const int src = row_end[r] - 1;
    if (src < 0 || src >= n_in) {
      if (threadIdx.x == 0) flag(status, LLAMA_FLAG_TOKEN_RANGE);
      for (int i = threadIdx.x; i < H; i += blockDim.x) store_y(yr, lo, i, 0.f);
      return;
    }
    xr = x + (size_t)src * H;
  }
  float ss = 0.f;
  const bool vec = (H % 4) == 0;
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
      float4 v = x4[i];
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  } else {
    for (int i = threadIdx.x; i < H; i += blockDim.x) ss += xr[i] * xr[i];
  }
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float inv = 1.0f / sqrtf(red[0] / (float)H + eps);
  if (vec) {
    const float4* x4 = reinterpret_cast<const float4*>(xr);
    for (int i = threadIdx.x; i < H / 4; i += blockDim.x) {
      float4 v = x4[i];
      const int c = i * 4;
      float g0 = to_f32(gamma[c]), g1 = to_f32(gamma[c + 1]), g2 = to_f32(gamma[c + 2]),
            g3 = to_f32(gamma[c + 3]);
      store_y(yr, lo, c, v.x * inv * g0);
      store_y(yr, lo, c + 1, v.y * inv * g1);
      store_y(yr, lo, c + 2, v.z * inv * g2);
      store_y(yr, lo, c + 3, v.w * inv * g3);
    }
  } else {
    for (int i = threadIdx.x; i < H; i += blockDim.x)
      store_y(yr, lo, i, xr[i] * inv * to_f32(gamma[i]));
  }
}

// ------------------------------------------------------------------ RoPE table
// tab[m * (d/2) + j] = (cos(m * theta_j), sin(m * theta_j)), theta_j =
// base^(-2j/d), evaluated in fp64 and rounded once to fp32.
__global__ void rope_table_kernel(float2* __restrict__ tab, int max_seq, int half, double base) {
  grid_dep_wait();
  grid_dep_launch();
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)max_seq * half) return;
  const int m = (int)(i / half), j = (int)(i % half);
  const double inv = pow(base, -2.0 * (double)j / (double)(2 * half));
  double s, c;
  sincos((double)m * inv, &s, &c);
  tab[i] = make_float2((float)c, (float)s);
}

// ------------------------------------------------------------------ RoPE + KV append
// Row r of qkv (fp32, Q heads | K heads | V heads) belongs to sequence
// r / rows_per_seq at position positions[r] (or r % rows_per_seq when
// positions is null). Each thread takes 8 consecutive values (two 128-bit
// loads), rotates adjacent pairs of Q and K by their position's angles, and
// writes Q to q_out and K, V into the cache slot (and to k_out / v_out when
// given). Positions outside the cache, or page ids outside the pool, set a
// status flag and skip the cache write.
// Eight consecutive values to dst: 16-byte stores when dst is 16-byte aligned
// (always, for the layouts this library sets up), else element by element.
__device__ __forceinline__ void store8(bf16* dst, const bf16 (&o)[8]) {
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = (uint32_t)__bfloat16_as_ushort(o[2 * k]) |
             ((uint32_t)__bfloat16_as_ushort(o[2 * k + 1]) << 16);
    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[k] = o[k];
  }
}
__device__ __forceinline__ void store8(float* dst, const float (&o)[8]) {
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(o[4], o[5], o[6], o[7]);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) dst[k] = o[k];
  }
}

template <typename T>
__global__ void __launch_bounds__(256) rope_append_kernel(RopeAppendArgs a) {
  grid_dep_wait();
  grid_dep_launch();
  const int r = blockIdx.y;
  int b, pos;
  if (a.cu_rows) {  // packed rows of several sequences: find r's sequence
    int lo = 0, hi = a.n_seq - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.cu_rows[mid] <= r) lo = mid; else hi = mid - 1;
    }
    b = lo;
    pos = a.start_pos[b] + r - a.cu_rows[b];
  } else {
    b = r / a.rows_per_seq;
    pos = a.positions ? a.positions[r] : (r % a.rows_per_seq);
  }
  const int d = a.head_dim;
  const int qw = a.n_q * d, kw = a.n_kv * d;
  const int width = qw + 2 * kw;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const int c = i * 8;
  if (c >= width) return;
  const float* src = a.qkv + (size_t)r * width + c;
  float v[8];
  {
    float4 lo = *reinterpret_cast<const float4*>(src);
    float4 hi = *reinterpret_cast<const float4*>(src + 4);
    v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
    v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
  }
  const bool is_v = c >= qw + kw;
  const bool pos_ok = pos >= 0 && pos < a.max_seq;
  if (!pos_ok && c == 0) flag(a.status, LLAMA_FLAG_POS_RANGE);
  if (!is_v) {
    const int dd = (c < qw ? c : c - qw) % d;
    const float2* tab = a.rope + (size_t)(pos_ok ? pos : 0) * (d / 2) + dd / 2;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 cs = tab[p];
      const float x0 = v[2 * p], x1 = v[2 * p + 1];
      v[2 * p] = x0 * cs.x - x1 * cs.y;
      v[2 * p + 1] = x0 * cs.y + x1 * cs.x;
    }
  }
  T o[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) o[k] = from_f32<T>(v[k]);
  if (c < qw) {
    T* dst = reinterpret_cast<T*>(a.q_out) + (size_t)r * qw + c;
    store8(dst, o);
    if (a.q_lo) {
      T ol[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ol[k] = from_f32<T>(v[k] - to_f32(o[k]));
      store8(dst + a.q_lo, ol);
    }
    return;
  }
  const int ck = is_v ? c - qw - kw : c - qw;  // column within the K (or V) block
  const int g = ck / d, dd = ck % d;
  uint8_t q8[8];
  if (a.kv_fp8) {  // the cache holds e4m3(x / scale); the side buffers its e4m3 value
    const float sc = is_v ? a.v_scale : a.k_scale;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      q8[k] = f32_to_e4m3(v[k] / sc);
      o[k] = from_f32<T>(e4m3_to_f32(q8[k]));
    }
  }
  T* side = reinterpret_cast<T*>(is_v ? a.v_out : a.k_out);
  if (side) store8(side + (size_t)r * kw + ck, o);
  // cache slot
  size_t slot;
  if (a.page_size == 0) {
    if (!pos_ok || pos >= a.capacity) {
      if (dd == 0) flag(a.status, LLAMA_FLAG_POS_RANGE);
      return;
    }
    slot = (((size_t)a.layer * a.batch_cap + b) * a.n_kv + g) * a.capacity + pos;
  } else {
    const int pi = pos_ok ? pos / a.page_size : -1;
    if (pi < 0 || pi >= a.max_pages) {
      if (dd == 0) flag(a.status, LLAMA_FLAG_POS_RANGE);
      return;
    }
    const int page = a.page_table[(size_t)b * a.max_pages + pi];
    if (page < 0 || page >= a.n_pages) {
      if (dd == 0) flag(a.status, LLAMA_FLAG_PAGE_RANGE);
      return;
    }
    slot = (((size_t)a.layer * a.n_pages + page) * a.n_kv + g) * a.page_size + pos % a.page_size;
  }
  if (a.kv_fp8) {
    uint8_t* cache8 = reinterpret_cast<uint8_t*>(is_v ? a.v_cache : a.k_cache) + slot * d + dd;
    uint2 w;
    w.x = q8[0] | (q8[1] << 8) | (q8[2] << 16) | ((uint32_t)q8[3] << 24);
    w.y = q8[4] | (q8[5] << 8) | (q8[6] << 16) | ((uint32_t)q8[7] << 24);
    *reinterpret_cast<uint2*>(cache8) = w;
    return;
  }
  store8(reinterpret_cast<T*>(is_v ? a.v_cache : a.k_cache) + slot * d + dd, o);
}

// ------------------------------------------------------------------ greedy argmax
// ids[b] = index of the largest logit of row b; ties go to the lowest index.
__global__ void __launch_bounds__(1024) argmax_kernel(const float* __restrict__ logits, int V,
                                                      int32_t* __restrict__ ids) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float sv[32];
  __shared__ int si[32];
  const float* row = logits + (size_t)blockIdx.x * V;
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int i = threadIdx.x; i < V; i += blockDim.x) {
    const float x = row[i];
    if (x > best || (x == best && i < bi)) { best = x; bi = i; }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
  }
  if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = best; si[threadIdx.x >> 5] = bi; }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int nw = blockDim.x >> 5;
    best = threadIdx.x < nw ? sv[threadIdx.x] : -INFINITY;
    bi = threadIdx.x < nw ? si[threadIdx.x] : 0x7fffffff;
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if (threadIdx.x == 0) ids[blockIdx.x] = bi == 0x7fffffff ? 0 : bi;
  }
}

// ------------------------------------------------------------------ positions += 1
// Advances every sequence by one position (used at the end of a captured
// decode step so that graph replays walk through the sequence).
__global__ void advance_positions_kernel(int32_t* __restrict__ positions, int B) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) positions[b] += 1;
}

// ------------------------------------------------------------------ launchers
static bool g_pdl = true;
void set_pdl(bool on) { g_pdl = on; }
bool pdl_enabled() { return g_pdl; }

cudaError_t launch_embed(int dtype, const int32_t* tokens, const void* table, int V, int H, int n,
                         float* out, uint32_t* status, cudaStream_t st) {
  if (dtype == LLAMA_BF16)
    return launch_k(embed_kernel<bf16>, dim3(n), dim3(256), 0, st, 0, tokens, (const bf16*)table, V,
                    H, out, status);
  return launch_k(embed_kernel<float>, dim3(n), dim3(256), 0, st, 0, tokens, (const float*)table,
                  V, H, out, status);
}

cudaError_t launch_rmsnorm(int dtype, const float* x, int rows, int in_stride, int in_offset,
                           const void* gamma, int H, float eps, void* out, int lo_rows,
                           cudaStream_t st, const int32_t* row_end, int n_in, uint32_t* status) {
  if (dtype == LLAMA_BF16)
    return launch_k(rmsnorm_kernel<bf16>, dim3(rows), dim3(256), 0, st, 0, x, in_stride, in_offset,
                    (const bf16*)gamma, H, eps, (bf16*)out, lo_rows, row_end, n_in, status);
  return launch_k(rmsnorm_kernel<float>, dim3(rows), dim3(256), 0, st, 0, x, in_stride, in_offset,
                  (const float*)gamma, H, eps, (float*)out, 0, row_end, n_in, status);
}

cudaError_t launch_rope_table(float2* tab, int max_seq, int head_dim, double theta,
                              cudaStream_t st) {
  const long long n = (long long)max_seq * (head_dim / 2);
  return launch_k(rope_table_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, 0, tab,
                  max_seq, head_dim / 2, theta);
}

cudaError_t launch_rope_append(int dtype, const RopeAppendArgs& a, int rows, cudaStream_t st) {
  const int width = (a.n_q + 2 * a.n_kv) * a.head_dim;
  dim3 grid((width / 8 + 255) / 256, rows);
  if (dtype == LLAMA_BF16) return launch_k(rope_append_kernel<bf16>, grid, dim3(256), 0, st, 0, a);
  return launch_k(rope_append_kernel<float>, grid, dim3(256), 0, st, 0, a);
}

cudaError_t launch_argmax(const float* logits, int B, int V, int32_t* ids, cudaStream_t st) {
  return launch_k(argmax_kernel, dim3(B), dim3(1024), 0, st, 0, logits, V, ids);
}

}  // namespace llgb

namespace llgb {
// Check of the bounded device wait: one thread waits, with the helper every
// pipeline uses, on a shared-memory mbarrier whose phase nothing completes.
// The wait runs out after limit_ns, sets LLAMA_FLAG_WAIT_TIMEOUT in the
// status word and the kernel returns normally.
__global__ void wait_check_kernel(uint32_t* status, uint64_t limit_ns) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, status, limit_ns);
  }
}

// E4M3 weights, one CTA per row: the row's largest magnitude (exact in fp32),
// scale = amax / 448 (1 for an all-zero row), then every value divided by the
// scale (IEEE fp32 division) and rounded to E4M3, nearest even, saturating.
__global__ void __launch_bounds__(256) quantize_rows_e4m3_kernel(const bf16* __restrict__ w,
                                                                  int cols,
                                                                  uint8_t* __restrict__ codes,
                                                                  float* __restrict__ scales) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float red[8];
  const size_t row = blockIdx.x;
  const bf16* src = w + row * cols;
  float amax = 0.f;
  for (int k = threadIdx.x * 8; k < cols; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + k);
    const bf16* e = reinterpret_cast<const bf16*>(&v);
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(__bfloat162float(e[j])));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const float s = amax > 0.f ? amax / 448.0f : 1.0f;
  if (threadIdx.x == 0) scales[row] = s;
  uint8_t* dst = codes + row * cols;
  for (int k = threadIdx.x * 8; k < cols; k += 256 * 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src + k);
    const bf16* e = reinterpret_cast<const bf16*>(&v);
    uint32_t b[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      b[j >> 2] |= (uint32_t)f32_to_e4m3(__bfloat162float(e[j]) / s) << (8 * (j & 3));
    *reinterpret_cast<uint2*>(dst + k) = make_uint2(b[0], b[1]);
  }
}

cudaError_t launch_quantize_rows_e4m3(const void* w, int rows, int cols, void* codes,
                                      float* scales, cudaStream_t st) {
  // a plain launch: the stream may be the legacy default stream
  quantize_rows_e4m3_kernel<<<rows, 256, 0, st>>>(reinterpret_cast<const bf16*>(w), cols,
                                                  reinterpret_cast<uint8_t*>(codes), scales);
  return cudaGetLastError();
}

cudaError_t launch_wait_check(uint32_t* status, uint64_t limit_ns, cudaStream_t st) {
  return launch_k(wait_check_kernel, dim3(1), dim3(32), 0, st, 0, status, limit_ns);
}

cudaError_t launch_advance_positions(int32_t* positions, int B, cudaStream_t st) {
  return launch_k(advance_positions_kernel, dim3((B + 127) / 128), dim3(128), 0, st, 0, positions, B);
}
}  // namespace llgb
