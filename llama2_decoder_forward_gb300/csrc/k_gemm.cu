// Linear layers y = x W^T of the decoder forward with fused epilogues.
//
// Every projection of the layer ("Llama2架构与推理全解析" §2.3: Q/K/V, output
// projection; §1.3: SwiGLU gate/up and down; the LM head) is one GEMM whose
// A operand is the weight matrix W [M, K] and whose B operand is the
// activation block x [N, K] (both K-major). The accumulator tile is 128
// weight rows x n_tile activation rows in tensor memory, so a decode step with
// 8..64 sequences still fills the 128-row MMA, and the epilogue thread that
// owns weight row m writes output column m for every activation row: stores
// are coalesced along m.
//
// bf16 path (tcgen05, sm_103a): one CTA per (n tile, m tile, k split);
// warp 0 issues TMA loads (128-byte swizzle) into a ring of shared-memory
// stages, warp 1 owns the tensor memory and issues tcgen05.mma (M=128,
// N=n_tile, K=16) per stage, warps 2..5 read the accumulator with tcgen05.ld
// and apply the epilogue. SwiGLU runs two MMAs per K step (gate rows and up
// rows of the same 128 features) into two accumulators, so silu(g)*u is
// formed in registers. When the grid would leave SMs idle (decode), K is
// split over up to 8 CTAs that form one thread-block cluster: each stages its
// fp32 sums in shared memory and the cluster adds them through distributed
// shared memory in split order (deterministic), each CTA finishing a slice of
// the tile's columns.
//
// E4M3 weights (W8 instantiations): the weight tiles arrive as bytes, the
// epilogue warps convert each to a bf16 tile in shared memory before the MMA
// (E4M3 is exact in bf16), and the per-row scale multiplies the accumulator.
//
// fp32 path: plain CUDA-core FMAs in fp32 (no TF32), one thread per output.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "rope_epi.cuh"

namespace llgb {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int GEMM_THREADS = 192;
constexpr int kMaxDynSmem = 232448;  // 227 KB per CTA
constexpr int kRasterGroup = 16;     // activation tiles a group of consecutive CTAs shares

struct TcParams {
  RopeAppendArgs rope;  // kEpiRope only
  // fused RMSNorm (see GemmCall)
  const bf16* norm_gamma;
  bf16* norm_out;
  size_t norm_lo;
  float* ssq_out;
  const float* ssq_in;
  int ssq_tiles, ssq_ld;
  float norm_inv_h, norm_eps;
  int M, N, K;
  int n_tile, num_kb, splits, n_tiles;
  int stages;
  int nconv;  // W8: converted-tile buffers (1 or 2)
  uint32_t tmem_cols;
  int lo;      // >0 (hi/lo mode): TMEM column offset of the remainder product (= ncol)
  int lo_rows; // hi/lo mode: activation row r's remainder is row lo_rows + r
  int ncol;    // output columns one tile produces (n_tile, or n_tile / 2 in the hi/lo mode)
  size_t out_lo;  // >0: bf16 outputs also write their remainder out_lo elements further
  // E4M3 weights (W8 kernels): row m of W (and of W_up) stands for
  // code * w_scale[m] (u_scale[m]); the scale multiplies the accumulator
  const float* w_scale;
  const float* u_scale;
  void* out;
  int ldo;
  uint32_t* status;
};

// Store one output element. For bf16 outputs with out_lo > 0 the value is
// kept as a pair: hi = bf16(v) at idx and lo = bf16(v - hi) at idx + out_lo.
template <int EPI, typename T>
__device__ __forceinline__ void epi_apply(void* out, size_t idx, float g, float u,
                                          size_t out_lo = 0) {
  if (EPI == LLAMA_EPI_STORE_F32) {
    reinterpret_cast<float*>(out)[idx] = g;
  } else if (EPI == LLAMA_EPI_RESID_F32) {
    reinterpret_cast<float*>(out)[idx] += g;
  } else {
    const float v = EPI == LLAMA_EPI_STORE_T ? g : silu_mul(g, u);  // STORE_T: g
    const T hi = from_f32<T>(v);
    reinterpret_cast<T*>(out)[idx] = hi;
    if (out_lo) reinterpret_cast<T*>(out)[idx + out_lo] = from_f32<T>(v - to_f32(hi));
  }
}

// Q/K/V projection epilogue. A RopeFeat describes output feature m (Q heads,
// then K heads, then V heads; features 2j and 2j+1 of a head form a RoPE
// pair); rope_emit stores that feature of token row r given its own sum and
// its pair partner's. Q and K are rotated by the token's angle; Q goes to its
// bf16 pair buffer, K and V to the cache slot (and to the prefill side
// buffers when given). Positions outside the RoPE table or the cache and page
// ids outside the pool are flagged and their cache writes skipped.
struct RopeFeat {
  int kind;   // 0 = Q, 1 = K, 2 = V
  int col;    // column within the Q, K or V block
  int g, dd;  // head and dimension within it
  bool odd;
};

__device__ __forceinline__ RopeFeat rope_feat(const RopeAppendArgs& a, int m) {
  const int d = a.head_dim, qw = a.n_q * d, kw = a.n_kv * d;
  RopeFeat f;
  f.kind = m < qw ? 0 : (m < qw + kw ? 1 : 2);
  f.col = f.kind == 0 ? m : (f.kind == 1 ? m - qw : m - qw - kw);
  f.g = f.col / d;
  f.dd = f.col - f.g * d;
  f.odd = f.dd & 1;
  return f;
}

// (cos, sin) of feature f's pair at position pos (identity for V and for
// positions outside the table); rope_cs2 also returns the next pair's (f.dd
// a multiple of 4: one 16-byte load).
__device__ __forceinline__ float2 rope_cs(const RopeAppendArgs& a, const RopeFeat& f, int pos) {
  if (f.kind == 2 || pos < 0) return make_float2(1.f, 0.f);
  return __ldg(a.rope + (size_t)pos * (a.head_dim / 2) + (f.dd >> 1));
}
__device__ __forceinline__ float4 rope_cs2(const RopeAppendArgs& a, const RopeFeat& f, int pos) {
  if (f.kind == 2 || pos < 0) return make_float4(1.f, 0.f, 1.f, 0.f);
  return __ldg(reinterpret_cast<const float4*>(a.rope + (size_t)pos * (a.head_dim / 2) +
                                               (f.dd >> 1)));
}

// Stores feature f of token row r: own is its sum, partner the other member
// of its RoPE pair, cs the pair's angle.
__device__ __forceinline__ void rope_emit(const RopeAppendArgs& a, const RopeFeat& f, int r,
                                          const TokInfo& t, float2 cs, float own, float partner) {
  const int d = a.head_dim;
  const float v = f.kind == 2 ? own
                  : f.odd     ? own * cs.x + partner * cs.y
                              : own * cs.x - partner * cs.y;
  const bf16 hi = __float2bfloat16_rn(v);
  if (f.kind == 0) {
    bf16* q = reinterpret_cast<bf16*>(a.q_out) + (size_t)r * a.n_q * d + f.col;
    q[0] = hi;
    if (a.q_lo) q[a.q_lo] = __float2bfloat16_rn(v - __bfloat162float(hi));
    return;
  }
  const bool is_v = f.kind == 2;
  const uint8_t q8 = a.kv_fp8 ? f32_to_e4m3(v / (is_v ? a.v_scale : a.k_scale)) : 0;
  bf16* side = reinterpret_cast<bf16*>(is_v ? a.v_out : a.k_out);
  if (side) side[(size_t)r * a.n_kv * d + f.col] = a.kv_fp8 ? __float2bfloat16_rn(e4m3_to_f32(q8)) : hi;
  if (t.kv >= 0) {
    const long long slot = t.kv + (long long)f.g * (a.page_size ? a.page_size : a.capacity);
    if (a.kv_fp8)
      reinterpret_cast<uint8_t*>(is_v ? a.v_cache : a.k_cache)[slot * d + f.dd] = q8;
    else
      reinterpret_cast<bf16*>(is_v ? a.v_cache : a.k_cache)[slot * d + f.dd] = hi;
  }
}

// Four consecutive features f0 .. f0+3 of token row r (two whole RoPE pairs,
// one kind, one head: f0.dd a multiple of 4) from their sums g, with the
// pairs' angles cs (x, y: first pair; z, w: second): the same values as four
// rope_emit calls, stored 8 bytes at a time where the destination allows.
__device__ __forceinline__ void st4_bf16(bf16* dst, const float (&v)[4], bool lo_part) {
  bf16 h[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const bf16 hi = __float2bfloat16_rn(v[e]);
    h[e] = lo_part ? __float2bfloat16_rn(v[e] - __bfloat162float(hi)) : hi;
  }
  if ((reinterpret_cast<uintptr_t>(dst) & 7u) == 0) {
    const uint32_t w0 = (uint32_t)__bfloat16_as_ushort(h[0]) | ((uint32_t)__bfloat16_as_ushort(h[1]) << 16);
    const uint32_t w1 = (uint32_t)__bfloat16_as_ushort(h[2]) | ((uint32_t)__bfloat16_as_ushort(h[3]) << 16);
    *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) dst[e] = h[e];
  }
}
__device__ __forceinline__ void rope_emit4(const RopeAppendArgs& a, const RopeFeat& f0, int r,
                                           const TokInfo& t, float4 cs, const float (&g)[4],
                                           int valid) {
  if (valid < 4) {  // a partial item at the end of the rows: element by element
    for (int e = 0; e < valid; ++e) {
      RopeFeat f = f0;
      f.col += e;
      f.dd += e;
      f.odd = e & 1;
      rope_emit(a, f, r, t, e < 2 ? make_float2(cs.x, cs.y) : make_float2(cs.z, cs.w), g[e],
                g[e ^ 1]);
    }
    return;
  }
  const int d = a.head_dim;
  float v[4];
  if (f0.kind == 2) {
#pragma unroll
    for (int e = 0; e < 4; ++e) v[e] = g[e];
  } else {
    v[0] = g[0] * cs.x - g[1] * cs.y;
    v[1] = g[1] * cs.x + g[0] * cs.y;
    v[2] = g[2] * cs.z - g[3] * cs.w;
    v[3] = g[3] * cs.z + g[2] * cs.w;
  }
  if (f0.kind == 0) {
    bf16* q = reinterpret_cast<bf16*>(a.q_out) + (size_t)r * a.n_q * d + f0.col;
    st4_bf16(q, v, false);
    if (a.q_lo) st4_bf16(q + a.q_lo, v, true);
    return;
  }
  const bool is_v = f0.kind == 2;
  if (a.kv_fp8) {  // the cache holds e4m3(x / scale); the side buffers its e4m3 value
    const float sc = is_v ? a.v_scale : a.k_scale;
    uint8_t q8[4];
    float dq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      q8[e] = f32_to_e4m3(v[e] / sc);
      dq[e] = e4m3_to_f32(q8[e]);
    }
    bf16* side = reinterpret_cast<bf16*>(is_v ? a.v_out : a.k_out);
    if (side) st4_bf16(side + (size_t)r * a.n_kv * d + f0.col, dq, false);
    if (t.kv >= 0) {
      const long long slot = t.kv + (long long)f0.g * (a.page_size ? a.page_size : a.capacity);
      uint8_t* c8 = reinterpret_cast<uint8_t*>(is_v ? a.v_cache : a.k_cache) + slot * d + f0.dd;
      if ((reinterpret_cast<uintptr_t>(c8) & 3u) == 0)
        *reinterpret_cast<uint32_t*>(c8) = (uint32_t)q8[0] | ((uint32_t)q8[1] << 8) |
                                           ((uint32_t)q8[2] << 16) | ((uint32_t)q8[3] << 24);
      else
        for (int e = 0; e < 4; ++e) c8[e] = q8[e];
    }
    return;
  }
  bf16* side = reinterpret_cast<bf16*>(is_v ? a.v_out : a.k_out);
  if (side) st4_bf16(side + (size_t)r * a.n_kv * d + f0.col, v, false);
  if (t.kv >= 0) {
    const long long slot = t.kv + (long long)f0.g * (a.page_size ? a.page_size : a.capacity);
    st4_bf16(reinterpret_cast<bf16*>(is_v ? a.v_cache : a.k_cache) + slot * d + f0.dd, v, false);
  }
}

// 16 accumulator columns starting at col for this thread's TMEM lane; in the
// hi/lo operand mode the column col + lo holds the product with the
// remainders and is added.
__device__ __forceinline__ void load_acc16(uint32_t tq, int col, int lo, float (&v)[16]) {
  uint32_t a[16], b[16];
  tmem_ld16(tq + col, a);
  if (lo) tmem_ld16(tq + col + lo, b);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 16; ++j)
    v[j] = lo ? __uint_as_float(a[j]) + __uint_as_float(b[j]) : __uint_as_float(a[j]);
}

// Split-K cluster reduction: CTA k of the cluster finishes columns
// [c_beg, c_end) of the tile; a work item is 4 consecutive rows of one column.
// Sums of 16 values over the 32 lanes of a warp (v[j] summed over lanes, for
// every j) in 16 shuffles: each halving step keeps half of the indices and
// adds the partner lane's copies of them. On return lane l holds the sum for
// index 8*b4 + 4*b3 + 2*b2 + b1 (b_i: bit i of l); lanes l and l ^ 1 agree.
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane, int& index) {
  float a8[8], a4[4], a2[2];
  const bool h4 = lane & 16, h3 = lane & 8, h2 = lane & 4, h1 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float send = h4 ? v[i] : v[i + 8];
    a8[i] = (h4 ? v[i + 8] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = h3 ? a8[i] : a8[i + 4];
    a4[i] = (h3 ? a8[i + 4] : a8[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = h2 ? a4[i] : a4[i + 2];
    a2[i] = (h2 ? a4[i + 2] : a4[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  const float send = h1 ? a2[0] : a2[1];
  float a1 = (h1 ? a2[1] : a2[0]) + __shfl_xor_sync(0xffffffffu, send, 2);
  a1 += __shfl_xor_sync(0xffffffffu, a1, 1);
  index = (h4 ? 8 : 0) + (h3 ? 4 : 0) + (h2 ? 2 : 0) + (h1 ? 1 : 0);
  return a1;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct RedSlice {
  int c_beg, items;
};
__device__ __forceinline__ RedSlice red_slice(const TcParams& p, int k) {
  RedSlice r;
  r.c_beg = (k * p.ncol) / p.splits;
  const int c_end = min(((k + 1) * p.ncol) / p.splits, min(p.ncol, p.N));
  r.items = max(0, c_end - r.c_beg) * (BM / 4);
  return r;
}

// E4M3 weight tile -> bf16 tile for the MMA. The source is the TMA box of
// 128 rows x 64 bytes without swizzle (row r at r * 64); the destination is
// the 128-row x 64-element bf16 tile in the 128-byte-swizzle layout the bf16
// path loads by TMA (16-byte chunk j of row r at r * 128 + ((j ^ (r & 7)) << 4)).
// Thread t of the 128 takes 16 bytes (quarter q = t % 4) of rows t / 4 + 32i:
// a warp reads 512 contiguous bytes, and each group of 8 threads writes the
// even chunks of one row and the odd chunks of the next, so neither side has
// bank conflicts. E4M3 values are exact in f16 and in bf16.
__device__ __forceinline__ void e4m3_tile_to_bf16(uint32_t src, uint32_t dst, int t) {
  const int q = t & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 32 + (t >> 2);
    uint32_t w[4];
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                 : "r"(src + r * 64 + q * 16));
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t lo, hi;  // f16 pairs of bytes (0, 1) and (2, 3)
      e4m3x4_to_f16x2x2(w[j], lo, hi);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
      const __nv_bfloat162 ab = __floats2bfloat162_rn(a.x, a.y);
      const __nv_bfloat162 bb = __floats2bfloat162_rn(b.x, b.y);
      o[2 * j] = *reinterpret_cast<const uint32_t*>(&ab);
      o[2 * j + 1] = *reinterpret_cast<const uint32_t*>(&bb);
    }
    const uint32_t row = dst + r * 128;
    const uint32_t c0 = (uint32_t)((2 * q) ^ (r & 7)) << 4, c1 = (uint32_t)((2 * q + 1) ^ (r & 7)) << 4;
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + c0), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3])
                 : "memory");
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(row + c1), "r"(o[4]), "r"(o[5]),
                 "r"(o[6]), "r"(o[7])
                 : "memory");
  }
}

template <int EPI, bool W8>
__global__ void __launch_bounds__(GEMM_THREADS, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmU,
                   const __grid_constant__ CUtensorMap tmX, TcParams p) {
  constexpr bool DUAL = EPI == LLAMA_EPI_SWIGLU;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // weight tiles as loaded: bf16, or E4M3 bytes (W8)
  const uint32_t a_bytes = BM * BK * (W8 ? 1 : 2);
  const uint32_t b_bytes = (uint32_t)p.n_tile * BK * 2;
  const uint32_t stage_bytes = a_bytes * (DUAL ? 2 : 1) + b_bytes;
  const int S = p.stages;
  // W8: p.nconv buffers of converted bf16 weight tiles (gate then up) after the stages
  const uint32_t conv_bytes = W8 ? BM * BK * 2 * (DUAL ? 2 : 1) : 0;
  const int NC = W8 ? p.nconv : 0;
  uint8_t* conv = smem + (size_t)S * stage_bytes;
  uint8_t* bar_block = conv + (size_t)NC * conv_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(bar_block);
  uint64_t* empty = full + S;
  uint64_t* accf = empty + S;
  // ctl[0]: TMEM base address, ctl[1]: abort, ctl[2]: this CTA reduces the tile
  volatile uint32_t* ctl = reinterpret_cast<volatile uint32_t*>(accf + 1);
  // W8: converted buffer c is full (128 converter arrivals) / free (MMA commit)
  uint64_t* cfull = accf + 3;
  uint64_t* cempty = cfull + 2;
  // kEpiRope: the tile's tokens (ncol entries after the 256-byte barrier block)
  TokInfo* tok = reinterpret_cast<TokInfo*>(bar_block + 256);
  // RMSNorm scales of the tile's rows (consumers), after the token table
  float* scl = reinterpret_cast<float*>(bar_block + 256 + (EPI == kEpiRope ? 16 * p.ncol : 0));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.z;
  // Tile order (no K split): CTAs run in launch order, so consecutive ones
  // take kRasterGroup activation tiles of one weight tile, then the same
  // activation tiles of the next weight tile. The activations and weights the
  // running CTAs read then stay in L2 instead of every wave streaming all the
  // activation tiles from HBM again.
  int tile_n = blockIdx.x, tile_m = blockIdx.y;
  if (p.splits == 1 && gridDim.x > 1) {
    const int id = blockIdx.y * gridDim.x + blockIdx.x;
    const int per_group = kRasterGroup * (int)gridDim.y;
    const int g0 = (id / per_group) * kRasterGroup;
    const int gn = min(kRasterGroup, (int)gridDim.x - g0);
    const int r = id - (id / per_group) * per_group;
    tile_n = g0 + r % gn;
    tile_m = r / gn;
  }

  const int kb0 = (int)(((long long)split * p.num_kb) / p.splits);
  const int kb1 = (int)(((long long)(split + 1) * p.num_kb) / p.splits);

  {  // bounds-check builds: the layout fits the launch, the split sums fit the
     // stages they reuse, output rows fit their stride (same for every CTA)
    const uint32_t tables = 256 + (EPI == kEpiRope ? 16 * p.ncol : 0) + (p.ssq_in ? 4 * p.ncol : 0);
    const uint32_t staged = p.splits > 1 ? (uint32_t)p.ncol * BM * 4 * (DUAL ? 2 : 1)
                                         : (EPI == LLAMA_EPI_RESID_F32 ? 16u * p.ncol : 0u);
    uint32_t* st = threadIdx.x == 0 ? p.status : nullptr;
    const uint32_t body = (uint32_t)S * stage_bytes + (uint32_t)NC * conv_bytes;
    const bool fits = bc_smem(smem, body + tables, 1024, st) &&
                      bc_ok(16u * S + 56u <= 256u, st) &&  // barrier block
                      bc_ok(!W8 || NC == 1 || NC == 2, st);
    const bool red_fits = bc_ok(staged <= body, st);
    const bool rows_fit = bc_ok(EPI == kEpiRope || p.M <= p.ldo, st);
    if (!fits || !red_fits || !rows_fit) {
      grid_dep_wait();
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    ctl[1] = 0;
    ctl[2] = 0;
    if (W8) {
      for (int c = 0; c < NC; ++c) {
        mbar_init(&cfull[c], 128);
        mbar_init(&cempty[c], 1);
      }
    }
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    if (DUAL) tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(const_cast<uint32_t*>(ctl), p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl[0];

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      const uint64_t pol_w = l2_policy_evict_first();  // weights are streamed once
      const uint32_t b_off = a_bytes * (DUAL ? 2 : 1);
      // The weights do not depend on the previous kernel: fill the first
      // stages with them before waiting, then add the activation tiles.
      const int npre = min(S, kb1 - kb0);
      for (int i = 0; i < npre; ++i) {
        uint8_t* st = smem + (size_t)i * stage_bytes;
        mbar_arrive_expect_tx(&full[i], stage_bytes);
        tma_load_2d_hint(st, &tmW, &full[i], (kb0 + i) * BK, tile_m * BM, pol_w);
        if (DUAL) tma_load_2d_hint(st + a_bytes, &tmU, &full[i], (kb0 + i) * BK, tile_m * BM, pol_w);
      }
      // activation tile: one box of n_tile rows, or in the hi/lo mode the hi
      // rows and the remainder rows of the same ncol activations back to back
      // activations are read by every weight tile's CTA: kept in L2 ahead of
      // the streamed weights
      const uint64_t pol_x = l2_policy_evict_last();
      auto load_x = [&](uint8_t* dst, uint64_t* bar, int kb) {
        if (p.lo) {
          tma_load_2d_hint(dst, &tmX, bar, kb * BK, tile_n * p.ncol, pol_x);
          tma_load_2d_hint(dst + (uint32_t)p.ncol * BK * 2, &tmX, bar, kb * BK,
                           p.lo_rows + tile_n * p.ncol, pol_x);
        } else {
          tma_load_2d_hint(dst, &tmX, bar, kb * BK, tile_n * p.n_tile, pol_x);
        }
      };
      grid_dep_wait();
      grid_dep_launch();
      for (int i = 0; i < npre; ++i)
        load_x(smem + (size_t)i * stage_bytes + b_off, &full[i], kb0 + i);
      int s = npre % S, issued = npre;
      uint32_t ph = npre == S ? 1u : 0u;
      bool ok = true;
      for (int kb = kb0 + npre; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[s], ph ^ 1, p.status)) {
          ok = false;
          ctl[1] = 1;
          break;
        }
        uint8_t* st = smem + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_2d_hint(st, &tmW, &full[s], kb * BK, tile_m * BM, pol_w);
        if (DUAL) tma_load_2d_hint(st + a_bytes, &tmU, &full[s], kb * BK, tile_m * BM, pol_w);
        load_x(st + b_off, &full[s], kb);
        ++issued;
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) {  // let the copies already in flight land before the CTA exits
        for (int i = 0; i < issued && i < S; ++i) {
          if (--s < 0) {
            s = S - 1;
            ph ^= 1;
          }
          mbar_wait(&full[s], ph, p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(BM, p.n_tile);
      int s = 0, c = 0;
      uint32_t ph = 0, cph = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (ctl[1] || !mbar_wait(&full[s], ph, p.status) ||
            (W8 && !mbar_wait(&cfull[c], cph, p.status))) {
          ctl[1] = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(smem + (size_t)s * stage_bytes);
        // weights: the stage's bf16 tiles, or (W8) the converted buffer
        const uint32_t w0 = W8 ? smem_u32(conv + (size_t)c * conv_bytes) : a0;
        const uint32_t up_off = W8 ? BM * BK * 2 : a_bytes;
        const uint64_t da = smem_desc_sw128(w0);
        const uint64_t du = smem_desc_sw128(w0 + up_off);
        const uint64_t db = smem_desc_sw128(a0 + a_bytes * (DUAL ? 2 : 1));
#pragma unroll
        for (int k = 0; k < BK / 16; ++k) {  // advance 32 bytes (16 bf16) along K
          const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
          tc_mma_f16(tmem, da + 2 * k, db + 2 * k, idesc, acc);
          if (DUAL) tc_mma_f16(tmem + p.n_tile, du + 2 * k, db + 2 * k, idesc, acc);
        }
        tc_commit(&empty[s]);
        if (W8) {
          tc_commit(&cempty[c]);
          if (++c == NC) {
            c = 0;
            cph ^= 1;
          }
        }
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
      tc_commit(accf);
      mbar_wait(accf, 0, p.status);  // every MMA retired before teardown
    }
  } else {  // ---------------- epilogue warps 2..5
    if (W8) {
      // first the weight converters: every stage's E4M3 tiles to bf16, in
      // k-block order, into the conversion buffers (weights only: no
      // dependency on the previous kernel)
      const int t = threadIdx.x - 64;
      int s = 0, c = 0;
      uint32_t ph = 0, cph = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (ctl[1] || !mbar_wait(&full[s], ph, p.status) ||
            !mbar_wait(&cempty[c], cph ^ 1, p.status)) {
          ctl[1] = 1;
          break;
        }
        const uint32_t src = smem_u32(smem + (size_t)s * stage_bytes);
        const uint32_t dst = smem_u32(conv + (size_t)c * conv_bytes);
        e4m3_tile_to_bf16(src, dst, t);
        if (DUAL) e4m3_tile_to_bf16(src + a_bytes, dst + BM * BK * 2, t);
        fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
        mbar_arrive(&cfull[c]);
        if (++c == NC) {
          c = 0;
          cph ^= 1;
        }
        if (++s == S) {
          s = 0;
          ph ^= 1;
        }
      }
    }
    grid_dep_wait();  // the residual and the outputs belong to the previous kernels' order
    grid_dep_launch();
    if (EPI == kEpiRope) {  // token table, filled while the MMAs run
      for (int i = threadIdx.x - 64; i < p.ncol; i += 128) {
        const int r = tile_n * p.ncol + i;
        tok[i] = r < p.N ? rope_token(p.rope, r) : TokInfo{-1, -1, 0};
      }
    }
    if (p.ssq_in) {  // RMSNorm scale of each row: its tile sums, added in tile order
      for (int i = threadIdx.x - 64; i < p.ncol; i += 128) {
        const int r = tile_n * p.ncol + i;
        float ss = 0.f;
        if (r < p.N)
          for (int tt = 0; tt < p.ssq_tiles; ++tt) ss += p.ssq_in[(size_t)tt * p.ssq_ld + r];
        scl[i] = 1.0f / sqrtf(ss * p.norm_inv_h + p.norm_eps);
      }
    }
    if (EPI == kEpiRope || p.ssq_in) epi_bar();
    const bool ok = mbar_wait(accf, 0, p.status);
    tc_fence_after();
    if (ok && !ctl[1]) {
      const int q = warp & 3;  // TMEM lane quadrant this warp may read
      const int r = q * 32 + lane;
      const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
      const int up = p.n_tile;  // first TMEM column of the up-projection accumulator
      if (p.splits == 1) {
        const int gm = tile_m * BM + r;
        const int n0 = tile_n * p.ncol;
        const int nvalid = min(p.ncol, p.N - n0);
        const RopeFeat rf = EPI == kEpiRope ? rope_feat(p.rope, min(gm, p.M - 1)) : RopeFeat{};
        const float wsc = W8 ? p.w_scale[min(gm, p.M - 1)] : 1.f;
        const float usc = W8 && DUAL ? p.u_scale[min(gm, p.M - 1)] : 1.f;
        for (int c0 = 0; c0 < nvalid; c0 += 16) {
          float g[16], u[16];
          load_acc16(tq, c0, p.lo, g);
          if (DUAL) load_acc16(tq, up + c0, p.lo, u);
          if (W8) {  // E4M3 weights: the row scale (before any use of the sums)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              g[j] *= wsc;
              if (DUAL) u[j] *= usc;
            }
          }
          if (p.ssq_in) {  // the input rows were normalised up to this scale
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              g[j] *= scl[c0 + j];
              if (DUAL) u[j] *= scl[c0 + j];
            }
          }
          if (EPI == LLAMA_EPI_RESID_F32 && p.norm_gamma) {
            // x_new, its normalised-input pair for the next projection, and
            // the per-row sums of squares of this tile's 128 features
            float* o = reinterpret_cast<float*>(p.out);
            const bool row_ok = gm < p.M;
            const float gam = row_ok ? __bfloat162float(p.norm_gamma[gm]) : 0.f;
            float res[16], ss[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              res[j] = (row_ok && c0 + j < nvalid) ? o[(size_t)(n0 + c0 + j) * p.ldo + gm] : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float xn = res[j] + g[j];
              ss[j] = 0.f;
              if (row_ok && c0 + j < nvalid) {
                const size_t idx = (size_t)(n0 + c0 + j) * p.ldo + gm;
                o[idx] = xn;
                const float y = xn * gam;
                const bf16 hi = __float2bfloat16_rn(y);
                p.norm_out[idx] = hi;
                if (p.norm_lo)
                  p.norm_out[idx + p.norm_lo] = __float2bfloat16_rn(y - __bfloat162float(hi));
                ss[j] = xn * xn;
              }
            }
            int jx;
            const float tot = warp_sum16(ss, lane, jx);
            if ((lane & 1) == 0)  // [4 quadrants][ncol] column sums of this warp's 32 rows
              reinterpret_cast<float*>(smem)[q * p.ncol + c0 + jx] = tot;
            continue;
          }
          if (EPI == kEpiRope) {
            float partner[16];  // the RoPE partner feature sits in the neighbouring lane
#pragma unroll
            for (int j = 0; j < 16; ++j) partner[j] = __shfl_xor_sync(0xffffffffu, g[j], 1);
            // the chunk's angles: all loads issued before any store
            float2 cs[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) cs[j] = rope_cs(p.rope, rf, tok[c0 + j].pos);
            if (gm < p.M) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < nvalid)
                  rope_emit(p.rope, rf, n0 + c0 + j, tok[c0 + j], cs[j], g[j], partner[j]);
            }
          } else if (gm < p.M) {
            if (EPI == LLAMA_EPI_RESID_F32) {
              // read the 16 residual values before writing any (one round trip)
              float* o = reinterpret_cast<float*>(p.out);
              float res[16];
#pragma unroll
              for (int j = 0; j < 16; ++j)
                res[j] = c0 + j < nvalid ? o[(size_t)(n0 + c0 + j) * p.ldo + gm] : 0.f;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < nvalid) o[(size_t)(n0 + c0 + j) * p.ldo + gm] = res[j] + g[j];
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < nvalid)
                  epi_apply<EPI, bf16>(p.out, (size_t)(n0 + c0 + j) * p.ldo + gm, g[j],
                                       DUAL ? u[j] : 0.f, p.out_lo);
            }
          }
        }
      } else {
        // this split's sums -> shared memory, column-major [col][128 rows]
        // (the direct path's norm sums are finished below)
        float* red = reinterpret_cast<float*>(smem);
        for (int c0 = 0; c0 < p.ncol; c0 += 16) {
          float g[16];
          load_acc16(tq, c0, p.lo, g);
#pragma unroll
          for (int j = 0; j < 16; ++j) red[(c0 + j) * BM + r] = g[j];
          if (DUAL) {
            load_acc16(tq, up + c0, p.lo, g);
#pragma unroll
            for (int j = 0; j < 16; ++j) red[(p.ncol + c0 + j) * BM + r] = g[j];
          }
        }
      }
    }
    if (EPI == LLAMA_EPI_RESID_F32 && p.norm_gamma && p.splits == 1) {
      epi_bar();  // every quadrant's column sums are in shared memory
      const int n0 = tile_n * p.ncol;
      const float* wsum = reinterpret_cast<const float*>(smem);
      for (int i = threadIdx.x - 64; i < p.ncol; i += 128)
        if (ok && !ctl[1] && n0 + i < p.N)
          p.ssq_out[(size_t)tile_m * p.ssq_ld + n0 + i] =
              wsum[i] + wsum[p.ncol + i] + wsum[2 * p.ncol + i] + wsum[3 * p.ncol + i];
    }
  }
  if (p.splits > 1) {
    // The splits of this tile form one cluster: after every CTA has staged its
    // sums, CTA k adds column slice k of all splits in split order (the same
    // order on every run) and applies the epilogue. One work item is 4
    // consecutive rows of one column (a 16-byte remote load per split).
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2 && !ctl[1]) {
      const int t = threadIdx.x - 64;
      const int S = p.splits;
      const RedSlice sl = red_slice(p, (int)cluster_ctarank());
      const uint32_t red0 = smem_u32(smem);
      for (int it = t; it < sl.items; it += 128) {
        const int c = sl.c_beg + it / (BM / 4), rq = (it % (BM / 4)) * 4;
        const uint32_t og = red0 + (uint32_t)(c * BM + rq) * 4u;
        const uint32_t ou = red0 + (uint32_t)((p.ncol + c) * BM + rq) * 4u;
        float4 gv[8], uv[8];
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2)
          if (s2 < S) {
            gv[s2] = dsmem_ld4(dsmem_addr(og, s2));
            if (DUAL) uv[s2] = dsmem_ld4(dsmem_addr(ou, s2));
          }
        float g[4] = {0.f, 0.f, 0.f, 0.f}, u[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int s2 = 0; s2 < 8; ++s2)
          if (s2 < S) {
            g[0] += gv[s2].x; g[1] += gv[s2].y; g[2] += gv[s2].z; g[3] += gv[s2].w;
            if (DUAL) { u[0] += uv[s2].x; u[1] += uv[s2].y; u[2] += uv[s2].z; u[3] += uv[s2].w; }
          }
        const int gm0 = tile_m * BM + rq;
        if (W8) {  // E4M3 weights: the row scales of the split-ordered sums
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int m = min(gm0 + e, p.M - 1);
            g[e] *= p.w_scale[m];
            if (DUAL) u[e] *= p.u_scale[m];
          }
        }
        if (p.ssq_in) {
          const float sc = scl[c];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            g[e] *= sc;
            u[e] *= sc;
          }
        }
        if (EPI == kEpiRope) {  // rows gm0..gm0+3: two complete RoPE pairs
          const TokInfo ti = tok[c];
          const RopeFeat f0 = rope_feat(p.rope, gm0);
          const float4 cs = rope_cs2(p.rope, f0, ti.pos);
          rope_emit4(p.rope, f0, c, ti, cs, g, min(4, p.M - gm0));
        } else if (EPI == LLAMA_EPI_RESID_F32) {
          float* o = reinterpret_cast<float*>(p.out) + (size_t)c * p.ldo + gm0;
          // a whole item with 16-byte aligned rows: vector loads and stores
          const bool vec = gm0 + 4 <= p.M && (reinterpret_cast<uintptr_t>(o) & 15u) == 0;
          float res[4];
          if (vec) {
            const float4 r4 = *reinterpret_cast<const float4*>(o);
            res[0] = r4.x; res[1] = r4.y; res[2] = r4.z; res[3] = r4.w;
            *reinterpret_cast<float4*>(o) =
                make_float4(res[0] + g[0], res[1] + g[1], res[2] + g[2], res[3] + g[3]);
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) res[e] = gm0 + e < p.M ? o[e] : 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (gm0 + e < p.M) o[e] = res[e] + g[e];
          }
          if (p.norm_gamma) {  // normalised-input pair and this tile's sum of squares
            float ss = 0.f;
            if (vec) {
              float y[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float xn = res[e] + g[e];
                y[e] = xn * __bfloat162float(p.norm_gamma[gm0 + e]);
                ss += xn * xn;
              }
              bf16* dst = p.norm_out + (size_t)c * p.ldo + gm0;
              st4_bf16(dst, y, false);
              if (p.norm_lo) st4_bf16(dst + p.norm_lo, y, true);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (gm0 + e < p.M) {
                  const float xn = res[e] + g[e];
                  const float y = xn * __bfloat162float(p.norm_gamma[gm0 + e]);
                  const bf16 hi = __float2bfloat16_rn(y);
                  const size_t idx = (size_t)c * p.ldo + gm0 + e;
                  p.norm_out[idx] = hi;
                  if (p.norm_lo)
                    p.norm_out[idx + p.norm_lo] = __float2bfloat16_rn(y - __bfloat162float(hi));
                  ss += xn * xn;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
            if ((threadIdx.x & 31) == 0) p.ssq_out[(size_t)tile_m * p.ssq_ld + c] = ss;
          }
        } else if (EPI == LLAMA_EPI_SWIGLU && gm0 + 4 <= p.M) {  // a whole item
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = silu_mul(g[e], u[e]);
          bf16* dst = reinterpret_cast<bf16*>(p.out) + (size_t)c * p.ldo + gm0;
          st4_bf16(dst, v, false);
          if (p.out_lo) st4_bf16(dst + p.out_lo, v, true);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (gm0 + e < p.M)
              epi_apply<EPI, bf16>(p.out, (size_t)c * p.ldo + gm0 + e, g[e], u[e], p.out_lo);
        }
      }
    }
    __syncwarp();
    cluster_sync_all();  // no CTA leaves while another still reads its shared memory
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

// ------------------------------------------------------------------ fp32 CUDA-core path
template <int EPI>
__global__ void gemm_f32_kernel(const float* __restrict__ x, const float* __restrict__ w,
                                const float* __restrict__ wu, int M, int N, int K, void* out,
                                int ldo) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = blockIdx.y;
  if (m >= M || n >= N) return;
  const float* xr = x + (size_t)n * K;
  const float* wr = w + (size_t)m * K;
  float acc = 0.f, accu = 0.f;
  if (EPI == LLAMA_EPI_SWIGLU) {
    const float* ur = wu + (size_t)m * K;
    for (int k = 0; k < K; ++k) {
      acc = fmaf(xr[k], wr[k], acc);
      accu = fmaf(xr[k], ur[k], accu);
    }
  } else {
    for (int k = 0; k < K; ++k) acc = fmaf(xr[k], wr[k], acc);
  }
  epi_apply<EPI, float>(out, (size_t)n * ldo + m, acc, accu);
}

// ------------------------------------------------------------------ planning
struct Plan {
  int n_tile, ncol, lo, lo_rows, stages, nconv, splits, m_tiles, n_tiles, num_kb, ctas_per_sm;
  size_t smem;
  uint32_t tmem_cols;
};

static int round16(int v) { return (v + 15) / 16 * 16; }

int gemm_n_tile(int N, int split) {
  if (split) return 2 * std::min(128, round16(N));
  return N >= 256 ? 256 : std::max(16, round16(N));
}

// rope: the Q/K/V epilogue's token table (16 bytes per tile column) follows
// the barrier block.
static Plan make_plan(int M, int N, int K, bool dual, int split, int sm_count, bool rope,
                      bool scale, bool w8) {
  Plan pl{};
  pl.n_tile = gemm_n_tile(N, split);
  pl.lo = split ? pl.n_tile / 2 : 0;
  pl.ncol = split ? pl.lo : pl.n_tile;
  pl.lo_rows = split ? round16(N) : 0;
  const int width = pl.n_tile * (dual ? 2 : 1);  // accumulator columns
  pl.tmem_cols = 32;
  while ((int)pl.tmem_cols < width) pl.tmem_cols <<= 1;
  const int stage_bytes = BM * BK * (w8 ? 1 : 2) * (dual ? 2 : 1) + pl.n_tile * BK * 2;
  // two CTAs per SM while both fit in tensor memory: narrow (decode) tiles,
  // and the single-accumulator prefill tiles, whose epilogues then overlap
  // the other CTA's K loop (two stages each)
  const bool two = (pl.n_tile <= 128 && pl.tmem_cols <= 256) || (!dual && pl.n_tile == 256 && N > 512);
  const int budget = two ? 112 * 1024 : 224 * 1024;
  const int extra = (rope ? 16 * pl.ncol : 0) + (scale ? 4 * pl.ncol : 0);
  // E4M3 weights: buffers of converted bf16 tiles besides the (smaller)
  // stages; two while three stages still fit, else one (converting a k-block
  // takes far less time than streaming its bytes)
  const int conv1 = w8 ? BM * BK * 2 * (dual ? 2 : 1) : 0;
  pl.nconv = w8 ? 2 : 0;
  if (w8 && (budget - 2048 - extra - 2 * conv1) / stage_bytes < 3) pl.nconv = 1;
  const int conv = pl.nconv * conv1;
  pl.stages = std::max(2, std::min(w8 ? 12 : 8, (budget - 2048 - extra - conv) / stage_bytes));
  pl.smem = (size_t)pl.stages * stage_bytes + conv + 1024 + 256 + extra;
  pl.ctas_per_sm = std::max(1, std::min(two ? 2 : 1, (int)(233472 / (pl.smem + 1024))));
  pl.m_tiles = (M + BM - 1) / BM;
  pl.n_tiles = (N + pl.ncol - 1) / pl.ncol;
  pl.num_kb = (K + BK - 1) / BK;
  const int tiles = pl.m_tiles * pl.n_tiles;
  const int slots = std::max(1, sm_count) * pl.ctas_per_sm;
  // Split K only for a single activation tile (decode) whose split sums fit
  // in the stage buffers; choose the count minimising waves x (k-blocks per
  // CTA + a fixed cost of about kFixedKb k-blocks for launch, first-load
  // latency and the cluster reduction).
  constexpr int kFixedKb = 4;
  const size_t red_bytes = (size_t)pl.ncol * (dual ? 2 : 1) * BM * sizeof(float);
  const bool can_split = pl.n_tiles == 1 && red_bytes <= (size_t)pl.stages * stage_bytes + conv;
  const int max_split = can_split ? std::min(8, pl.num_kb) : 1;
  long best = -1;
  pl.splits = 1;
  for (int s = 1; s <= max_split; ++s) {
    const long ctas = (long)tiles * s;
    const long waves = (ctas + slots - 1) / slots;
    const long cost = waves * ((pl.num_kb + s - 1) / s + kFixedKb);
    if (best < 0 || cost < best) {
      best = cost;
      pl.splits = s;
    }
  }
  return pl;
}

template <int EPI>
static cudaError_t set_attr() {
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<EPI, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemm_tc_kernel<EPI, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

cudaError_t gemm_prepare() {
  cudaError_t e;
  if ((e = set_attr<LLAMA_EPI_STORE_F32>()) != cudaSuccess) return e;
  if ((e = set_attr<LLAMA_EPI_RESID_F32>()) != cudaSuccess) return e;
  if ((e = set_attr<LLAMA_EPI_STORE_T>()) != cudaSuccess) return e;
  if ((e = set_attr<kEpiRope>()) != cudaSuccess) return e;
  if ((e = set_attr<LLAMA_EPI_SWIGLU>()) != cudaSuccess) return e;
  return gemm_tm_prepare();
}

template <int EPI, bool W8>
static cudaError_t launch_tc(const GemmCall& g, const Plan& pl, cudaStream_t st) {
  TcParams p;
  if (g.rope) p.rope = *g.rope;
  p.norm_gamma = reinterpret_cast<const bf16*>(g.norm_gamma);
  p.norm_out = reinterpret_cast<bf16*>(g.norm_out);
  p.norm_lo = g.norm_lo;
  p.ssq_out = g.ssq_out;
  p.ssq_in = g.ssq_in;
  p.ssq_tiles = g.ssq_tiles;
  p.ssq_ld = g.ssq_ld;
  p.norm_inv_h = g.norm_h > 0 ? 1.0f / (float)g.norm_h : 0.f;
  p.norm_eps = g.norm_eps;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.n_tile = pl.n_tile;
  p.num_kb = pl.num_kb;
  p.splits = pl.splits;
  p.n_tiles = pl.n_tiles;
  p.stages = pl.stages;
  p.nconv = pl.nconv;
  p.tmem_cols = pl.tmem_cols;
  p.lo = pl.lo;
  p.lo_rows = pl.lo_rows;
  p.ncol = pl.ncol;
  p.out_lo = g.out_lo;
  p.w_scale = g.w_scale;
  p.u_scale = g.u_scale;
  p.out = g.out;
  p.ldo = g.ldo;
  p.status = g.status;
  const CUtensorMap* up = g.map_up ? g.map_up : g.map_w;
  return launch_k(gemm_tc_kernel<EPI, W8>, dim3(pl.n_tiles, pl.m_tiles, pl.splits),
                  dim3(GEMM_THREADS), pl.smem, st, pl.splits, *g.map_w, *up, *g.map_x, p);
}

template <int EPI>
static cudaError_t launch_tc(const GemmCall& g, const Plan& pl, cudaStream_t st) {
  return g.w_scale ? launch_tc<EPI, true>(g, pl, st) : launch_tc<EPI, false>(g, pl, st);
}

template <int EPI>
static cudaError_t launch_f32(const GemmCall& g, cudaStream_t st) {
  dim3 grid((g.M + 127) / 128, g.N);
  return launch_k(gemm_f32_kernel<EPI>, grid, dim3(128), 0, st, 0, (const float*)g.x,
                  (const float*)g.w, (const float*)g.w_up, g.M, g.N, g.K, g.out, g.ldo);
}

cudaError_t launch_gemm(const GemmCall& g, cudaStream_t st) {
  if (g.dtype == LLAMA_F32) {
    switch (g.epi) {
      case LLAMA_EPI_STORE_F32: return launch_f32<LLAMA_EPI_STORE_F32>(g, st);
      case LLAMA_EPI_RESID_F32: return launch_f32<LLAMA_EPI_RESID_F32>(g, st);
      case LLAMA_EPI_STORE_T: return launch_f32<LLAMA_EPI_STORE_T>(g, st);
      default: return launch_f32<LLAMA_EPI_SWIGLU>(g, st);
    }
  }
  if (gemm_tm_applies(g)) return launch_gemm_tm(g, st);
  const bool dual = g.epi == LLAMA_EPI_SWIGLU;
  if (g.w_scale && dual != (g.u_scale != nullptr)) return cudaErrorInvalidValue;
  const Plan pl = make_plan(g.M, g.N, g.K, dual, g.split, g.sm_count, g.epi == kEpiRope,
                            g.ssq_in != nullptr, g.w_scale != nullptr);
  if (pl.n_tile != g.n_tile) return cudaErrorInvalidValue;
  switch (g.epi) {
    case LLAMA_EPI_STORE_F32: return launch_tc<LLAMA_EPI_STORE_F32>(g, pl, st);
    case LLAMA_EPI_RESID_F32: return launch_tc<LLAMA_EPI_RESID_F32>(g, pl, st);
    case LLAMA_EPI_STORE_T: return launch_tc<LLAMA_EPI_STORE_T>(g, pl, st);
    case kEpiRope: return g.rope ? launch_tc<kEpiRope>(g, pl, st) : cudaErrorInvalidValue;
    default: return launch_tc<LLAMA_EPI_SWIGLU>(g, pl, st);
  }
}

}  // namespace llgb
