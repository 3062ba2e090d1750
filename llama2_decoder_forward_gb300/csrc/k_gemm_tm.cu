// Prefill projections with the activation rows on the MMA's M side.
//
// The same products as gemm_tc_kernel ("Llama2架构与推理全解析" §2.3: Q/K/V
// and output projections; §1.3: SwiGLU gate/up and down): y[n, m] = sum_k
// x[n, k] w[m, k], the activations carried as the bf16 pair hi + lo. Here
// the A operand is a tile of 128 activation rows (tokens) and B is 256
// weight rows, so the two halves of the pair are two A tiles that accumulate
// into one tensor-memory accumulator (hi W + lo W). With the weights on M
// (gemm_tc_kernel) the pair doubles the N side instead, and a 64-wide
// k-block brings 48 KB for 512 cycles of MMA work (94 bytes per cycle); here
// it brings 64 KB (16 KB hi, 16 KB lo, 32 KB of weights) for 1024 cycles
// (64 bytes per cycle), below what the L2 delivers into one SM.
//
// Persistent: one CTA per SM walks the tiles t = blockIdx.x, + gridDim.x, ...
// Two accumulators of 256 columns each fill the 512 tensor-memory columns,
// so the epilogue of one tile runs while the MMAs of the next fill the other
// accumulator. Warp 0 issues the TMA loads into a ring of 3 stages of 64 KB,
// warp 1 the MMAs (M = 128, N = 256, K = 16), warps 2..5 read the
// accumulator (thread = token row, tcgen05.ld 32x32b) and apply the
// epilogue: store fp32, add into the fp32 residual (and, for the fused
// RMSNorm, store the next projection's input pair x * gamma and the per-row
// sums of x^2 per 128 features), silu(gate) * up as a bf16 pair, or, for the
// Q/K/V projection, RoPE and the KV-cache append (each thread holds whole
// RoPE pairs of its token: features 2j and 2j + 1 are neighbouring
// accumulator columns). SwiGLU loads 128 gate rows and the same 128 up rows as the two halves of B, so
// columns 0..127 of the accumulator hold the gate sums and 128..255 the up
// sums of the same features.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "rope_epi.cuh"

namespace llgb {

namespace {

constexpr int TM_BM = 128;  // activation rows per tile (MMA M)
constexpr int TM_BN = 256;  // weight rows per tile (MMA N)
constexpr int TM_BK = 64;   // K per stage: one 128-byte swizzle row of bf16
constexpr int TM_STAGES = 3;
constexpr int TM_THREADS = 192;
constexpr uint32_t TM_A_BYTES = TM_BM * TM_BK * 2;                // one half of the pair
constexpr uint32_t TM_B_BYTES = TM_BN * TM_BK * 2;                // two 128-row weight boxes
constexpr uint32_t TM_STAGE_BYTES = 2 * TM_A_BYTES + TM_B_BYTES;  // 64 KB
constexpr uint32_t TM_TMEM_COLS = 2 * TM_BN;                      // two accumulators
constexpr int TM_GROUP = 16;  // activation tiles consecutive tiles share
constexpr size_t TM_SMEM = (size_t)TM_STAGES * TM_STAGE_BYTES + 1024 + 256;

struct TmParams {
  RopeAppendArgs rope;  // kEpiRope only
  int M, N, K, num_kb;
  int lo_rows;  // activation row n's remainder is row lo_rows + n of the map
  int n_tok, n_feat, tiles;
  int fw;  // output features per tile: 256, or 128 for SwiGLU
  void* out;
  int ldo;
  size_t out_lo;  // >0: bf16 outputs also store their remainder out_lo elements further
  // fused RMSNorm: producer (RESID_F32 with norm_gamma) and consumer (ssq_in)
  const bf16* norm_gamma;
  bf16* norm_out;
  size_t norm_lo;
  float* ssq_out;
  const float* ssq_in;
  int ssq_tiles, ssq_ld;
  float norm_inv_h, norm_eps;
  uint32_t* status;
};

// Tile t -> (activation tile, weight tile). Consecutive tiles take
// TM_GROUP activation tiles of one weight tile, then the same activation
// tiles of the next weight tile: the CTAs running at once share a few
// weight tiles and one group's activations, which stay in L2.
__device__ __forceinline__ void tm_tile(const TmParams& p, int t, int& tok, int& feat) {
  const int per_group = TM_GROUP * p.n_feat;
  const int g = t / per_group;
  const int r = t - g * per_group;
  const int tok0 = g * TM_GROUP;
  const int gn = min(TM_GROUP, p.n_tok - tok0);
  tok = tok0 + r % gn;
  feat = r / gn;
}

// 16 consecutive values at src / dst, valid of them inside the matrix
// (16-byte accesses when all 16 are valid and the address allows).
__device__ __forceinline__ void ld16_f32(const float* src, float (&v)[16], int valid) {
  if (valid >= 16 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 q = reinterpret_cast<const float4*>(src)[i];
      v[4 * i] = q.x;
      v[4 * i + 1] = q.y;
      v[4 * i + 2] = q.z;
      v[4 * i + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = j < valid ? src[j] : 0.f;
  }
}
__device__ __forceinline__ void st16_f32(float* dst, const float (&v)[16], int valid) {
  if (valid >= 16 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      reinterpret_cast<float4*>(dst)[i] =
          make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < valid) dst[j] = v[j];
  }
}
__device__ __forceinline__ void ld16_bf16(const bf16* src, float (&v)[16], int valid) {
  if (valid >= 16 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(src) + i);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        v[8 * i + 2 * e] = f.x;
        v[8 * i + 2 * e + 1] = f.y;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = j < valid ? __bfloat162float(src[j]) : 0.f;
  }
}
// The bf16 pair of 16 values: hi = bf16(v) at dst, and, when lo > 0,
// bf16(v - hi) lo elements further.
__device__ __forceinline__ void st16_pair(bf16* dst, size_t lo, const float (&v)[16], int valid) {
  uint32_t h[8], r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) split_pack(v[2 * i], v[2 * i + 1], h[i], r[i]);
  const bool vec = valid >= 16 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 &&
                   (lo == 0 || (reinterpret_cast<uintptr_t>(dst + lo) & 15u) == 0);
  if (vec) {
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(h[0], h[1], h[2], h[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(h[4], h[5], h[6], h[7]);
    if (lo) {
      reinterpret_cast<uint4*>(dst + lo)[0] = make_uint4(r[0], r[1], r[2], r[3]);
      reinterpret_cast<uint4*>(dst + lo)[1] = make_uint4(r[4], r[5], r[6], r[7]);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < valid) {
        const uint32_t hw = h[j >> 1], rw = r[j >> 1];
        dst[j] = __ushort_as_bfloat16((uint16_t)((j & 1) ? hw >> 16 : hw & 0xFFFFu));
        if (lo) dst[lo + j] = __ushort_as_bfloat16((uint16_t)((j & 1) ? rw >> 16 : rw & 0xFFFFu));
      }
  }
}

// The Q/K/V epilogue for 16 consecutive features m.. of token row n (one
// head of one kind: m and the head size are multiples of 16) from their sums
// g: RoPE on Q and K by the token's angle (feature pairs 2j, 2j + 1 rotated
// together), Q to its bf16 pair buffer, K and V to the cache slot (bf16, or
// E4M3 of x / scale) and to the side buffers when given. The same values as
// the separate RoPE/append kernel and gemm_tc_kernel's epilogue.
__device__ __forceinline__ void tm_rope16(const RopeAppendArgs& a, int n, int m, const TokInfo& ti,
                                          const float (&g)[16]) {
  const int d = a.head_dim, qw = a.n_q * d, kw = a.n_kv * d;
  const int kind = m < qw ? 0 : (m < qw + kw ? 1 : 2);
  const int col = m - (kind == 0 ? 0 : (kind == 1 ? qw : qw + kw));
  const int gh = col / d, dd = col - gh * d;
  float v[16];
  if (kind == 2 || ti.pos < 0) {  // V, or a position outside the table (angle 0)
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = g[j];
  } else {
    const float4* cs = reinterpret_cast<const float4*>(a.rope + (size_t)ti.pos * (d / 2) + (dd >> 1));
    // the separate RoPE kernel's expressions term for term, so that both
    // round (and contract into FMAs) alike and write bit-identical values
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // pairs (4i, 4i+1) and (4i+2, 4i+3)
      const float4 c = __ldg(cs + i);
      const float x0 = g[4 * i], x1 = g[4 * i + 1], x2 = g[4 * i + 2], x3 = g[4 * i + 3];
      v[4 * i] = x0 * c.x - x1 * c.y;
      v[4 * i + 1] = x0 * c.y + x1 * c.x;
      v[4 * i + 2] = x2 * c.z - x3 * c.w;
      v[4 * i + 3] = x2 * c.w + x3 * c.z;
    }
  }
  if (kind == 0) {
    st16_pair(reinterpret_cast<bf16*>(a.q_out) + (size_t)n * qw + col, a.q_lo, v, 16);
    return;
  }
  const bool is_v = kind == 2;
  bf16* side = reinterpret_cast<bf16*>(is_v ? a.v_out : a.k_out);
  const long long slot =
      ti.kv < 0 ? -1 : ti.kv + (long long)gh * (a.page_size ? a.page_size : a.capacity);
  if (a.kv_fp8) {  // the cache holds e4m3(x / scale); the side buffers its e4m3 value
    const float sc = is_v ? a.v_scale : a.k_scale;
    uint32_t w[4];
    float dq[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[i] = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint8_t q8 = f32_to_e4m3(v[4 * i + e] / sc);
        dq[4 * i + e] = e4m3_to_f32(q8);
        w[i] |= (uint32_t)q8 << (8 * e);
      }
    }
    if (side) st16_pair(side + (size_t)n * kw + col, 0, dq, 16);
    if (slot >= 0) {
      uint8_t* c8 = reinterpret_cast<uint8_t*>(is_v ? a.v_cache : a.k_cache) + slot * d + dd;
      if ((reinterpret_cast<uintptr_t>(c8) & 15u) == 0) {
        *reinterpret_cast<uint4*>(c8) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) c8[j] = (uint8_t)(w[j >> 2] >> (8 * (j & 3)));
      }
    }
    return;
  }
  if (side) st16_pair(side + (size_t)n * kw + col, 0, v, 16);
  if (slot >= 0)
    st16_pair(reinterpret_cast<bf16*>(is_v ? a.v_cache : a.k_cache) + slot * d + dd, 0, v, 16);
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(TM_THREADS, 1)
    gemm_tm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmU,
                   const __grid_constant__ CUtensorMap tmX, TmParams p) {
  constexpr bool DUAL = EPI == LLAMA_EPI_SWIGLU;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)TM_STAGES * TM_STAGE_BYTES);
  uint64_t* empty = full + TM_STAGES;
  uint64_t* tfull = empty + TM_STAGES;  // accumulator b holds a finished tile
  uint64_t* tempty = tfull + 2;         // accumulator b was read (128 epilogue threads)
  uint64_t* mdone = tempty + 2;         // every MMA retired (teardown)
  // ctl[0]: tensor-memory base address, ctl[1]: abort
  volatile uint32_t* ctl = reinterpret_cast<volatile uint32_t*>(mdone + 1);
  static_assert((2 * TM_STAGES + 5) * 8 + 8 <= 256, "barrier block");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (!bc_smem(smem, TM_STAGES * TM_STAGE_BYTES + 256, 1024,
               threadIdx.x == 0 ? p.status : nullptr)) {
    grid_dep_wait();
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < TM_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(mdone, 1);
    ctl[1] = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmW);
    if (DUAL) tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) tmem_alloc(const_cast<uint32_t*>(ctl), TM_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl[0];

  if (warp == 0) {
    if (lane == 0) {  // ---------------- TMA producer
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();  // read by every weight tile's CTA
      // The two 128-row halves of a stage's weight tile: rows wrow.. and
      // wrow + 128.. of W, or (SwiGLU) the same rows of W_gate and W_up.
      auto load_w = [&](uint8_t* st, uint64_t* bar, int kb, int feat) {
        uint8_t* b = st + 2 * TM_A_BYTES;
        const int wrow = feat * (DUAL ? 128 : TM_BN);
        tma_load_2d_hint(b, &tmW, bar, kb * TM_BK, wrow, pol_w);
        if (DUAL)
          tma_load_2d_hint(b + TM_B_BYTES / 2, &tmU, bar, kb * TM_BK, wrow, pol_w);
        else
          tma_load_2d_hint(b + TM_B_BYTES / 2, &tmW, bar, kb * TM_BK, wrow + 128, pol_w);
      };
      auto load_x = [&](uint8_t* st, uint64_t* bar, int kb, int tok) {
        tma_load_2d_hint(st, &tmX, bar, kb * TM_BK, tok * TM_BM, pol_x);
        tma_load_2d_hint(st + TM_A_BYTES, &tmX, bar, kb * TM_BK, p.lo_rows + tok * TM_BM, pol_x);
      };
      // The weights do not depend on the previous kernel: the first tile's
      // first stages get them before the dependency wait.
      int t = blockIdx.x, tok = 0, feat = 0, npre = 0;
      if (t < p.tiles) {
        tm_tile(p, t, tok, feat);
        npre = min(TM_STAGES, p.num_kb);
        for (int i = 0; i < npre; ++i) {
          uint8_t* st = smem + (size_t)i * TM_STAGE_BYTES;
          mbar_arrive_expect_tx(&full[i], TM_STAGE_BYTES);
          load_w(st, &full[i], i, feat);
        }
      }
      grid_dep_wait();
      grid_dep_launch();
      for (int i = 0; i < npre; ++i) load_x(smem + (size_t)i * TM_STAGE_BYTES, &full[i], i, tok);
      int s = npre % TM_STAGES, issued = npre, kb_first = npre;
      uint32_t ph = npre == TM_STAGES ? 1u : 0u;
      bool ok = true;
      for (; t < p.tiles && ok; t += gridDim.x) {
        tm_tile(p, t, tok, feat);
        for (int kb = kb_first; kb < p.num_kb; ++kb) {
          if (ctl[1] || !mbar_wait(&empty[s], ph ^ 1, p.status)) {
            ok = false;
            ctl[1] = 1;
            break;
          }
          uint8_t* st = smem + (size_t)s * TM_STAGE_BYTES;
          mbar_arrive_expect_tx(&full[s], TM_STAGE_BYTES);
          load_w(st, &full[s], kb, feat);
          load_x(st, &full[s], kb, tok);
          ++issued;
          if (++s == TM_STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        kb_first = 0;
      }
      if (!ok) {  // let the copies already in flight land before the CTA exits
        for (int i = 0; i < issued && i < TM_STAGES; ++i) {
          if (--s < 0) {
            s = TM_STAGES - 1;
            ph ^= 1;
          }
          mbar_wait(&full[s], ph, p.status);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {  // ---------------- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(TM_BM, TM_BN);
      int s = 0, lt = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++lt) {
        const int b = lt & 1;
        // accumulator b's previous tile has been read by the epilogue
        if (ctl[1] || !mbar_wait(&tempty[b], ((uint32_t)(lt >> 1) & 1u) ^ 1u, p.status)) {
          ok = false;
          ctl[1] = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * TM_BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (ctl[1] || !mbar_wait(&full[s], ph, p.status)) {
            ok = false;
            ctl[1] = 1;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(smem + (size_t)s * TM_STAGE_BYTES);
          const uint64_t dh = smem_desc_sw128(a0);
          const uint64_t dl = smem_desc_sw128(a0 + TM_A_BYTES);
          const uint64_t dw = smem_desc_sw128(a0 + 2 * TM_A_BYTES);
#pragma unroll
          for (int k = 0; k < TM_BK / 16; ++k) {  // advance 32 bytes (16 bf16) along K
            tc_mma_f16(d, dh + 2 * k, dw + 2 * k, idesc, (kb > 0 || k > 0) ? 1u : 0u);
            tc_mma_f16(d, dl + 2 * k, dw + 2 * k, idesc, 1u);
          }
          tc_commit(&empty[s]);
          if (++s == TM_STAGES) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) tc_commit(&tfull[b]);
      }
      tc_commit(mdone);
      mbar_wait(mdone, 0, p.status);  // every MMA retired before teardown
    }
  } else {  // ---------------- epilogue warps 2..5: thread = token row
    grid_dep_wait();  // the residual and the norm sums belong to the previous kernels
    grid_dep_launch();
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    const int r = q * 32 + lane;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16);
    int lt = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++lt) {
      const int b = lt & 1;
      // the warp stays converged for the tcgen05.ld below: it goes on only
      // when every lane saw the accumulator finished
      const bool ok = !ctl[1] && mbar_wait(&tfull[b], (uint32_t)(lt >> 1) & 1u, p.status);
      if (!__all_sync(0xffffffffu, ok)) {
        ctl[1] = 1;
        break;
      }
      tc_fence_after();
      int tok, feat;
      tm_tile(p, t, tok, feat);
      const int n = tok * TM_BM + r;
      const bool row_ok = n < p.N;
      float scl = 1.f;
      if (p.ssq_in && row_ok) {  // RMSNorm scale of the row: its tile sums in tile order
        float ss = 0.f;
        for (int tt = 0; tt < p.ssq_tiles; ++tt) ss += p.ssq_in[(size_t)tt * p.ssq_ld + n];
        scl = 1.0f / sqrtf(ss * p.norm_inv_h + p.norm_eps);
      }
      const TokInfo ti =
          EPI == kEpiRope && row_ok ? rope_token(p.rope, n) : TokInfo{-1, -1, 0};
      const uint32_t tb = tq + (uint32_t)(b * TM_BN);
      const int m0 = feat * p.fw;
      const size_t row = (size_t)(row_ok ? n : 0) * p.ldo;
      const int nchunks = p.fw / 16;
      float ssq0 = 0.f, ssq1 = 0.f;  // sums of x^2 over features m0.. and m0 + 128..
      for (int c = 0; c < nchunks; ++c) {
        const int c0 = c * 16;
        float g[16], u[16];
        {
          uint32_t a[16], a2[16];
          tmem_ld16(tb + c0, a);
          if (DUAL) tmem_ld16(tb + 128 + c0, a2);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            g[j] = __uint_as_float(a[j]) * scl;
            u[j] = DUAL ? __uint_as_float(a2[j]) * scl : 0.f;
          }
        }
        if (c == nchunks - 1) {  // the accumulator is free for the tile after next
          tc_fence_before();
          mbar_arrive(&tempty[b]);
        }
        const int m = m0 + c0;
        const int valid = row_ok ? min(16, p.M - m) : 0;
        if (valid <= 0) continue;
        if (EPI == kEpiRope) {
          tm_rope16(p.rope, n, m, ti, g);
        } else if (EPI == LLAMA_EPI_STORE_F32) {
          st16_f32(reinterpret_cast<float*>(p.out) + row + m, g, valid);
        } else if (EPI == LLAMA_EPI_RESID_F32) {
          float* o = reinterpret_cast<float*>(p.out) + row + m;
          float xn[16];
          ld16_f32(o, xn, valid);
#pragma unroll
          for (int j = 0; j < 16; ++j) xn[j] += g[j];
          st16_f32(o, xn, valid);
          if (p.norm_gamma) {  // the next projection's input pair and the sums of x^2
            float gam[16];
            ld16_bf16(p.norm_gamma + m, gam, valid);
            float y[16];
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              y[j] = xn[j] * gam[j];
              if (j < valid) s += xn[j] * xn[j];
            }
            if (c0 < 128)
              ssq0 += s;
            else
              ssq1 += s;
            st16_pair(p.norm_out + row + m, p.norm_lo, y, valid);
          }
        } else {  // STORE_T (g) or SWIGLU (silu(g) * u): a bf16 pair
          float v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = DUAL ? silu_mul(g[j], u[j]) : g[j];
          st16_pair(reinterpret_cast<bf16*>(p.out) + row + m, p.out_lo, v, valid);
        }
      }
      if (EPI == LLAMA_EPI_RESID_F32 && p.norm_gamma && row_ok) {
        // one sum per 128-feature tile of the output, as gemm_tc_kernel stores them
        p.ssq_out[(size_t)(m0 / 128) * p.ssq_ld + n] = ssq0;
        if (p.fw > 128 && m0 + 128 < p.M) p.ssq_out[(size_t)(m0 / 128 + 1) * p.ssq_ld + n] = ssq1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TM_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side
bool gemm_tm_shape(int epi, int M, int N, int split, int sm_count) {
  if (!split) return false;
  if (epi != LLAMA_EPI_STORE_F32 && epi != LLAMA_EPI_RESID_F32 && epi != LLAMA_EPI_STORE_T &&
      epi != LLAMA_EPI_SWIGLU && epi != kEpiRope)
    return false;
  if (gemm_box_rows(N, split) != TM_BM) return false;  // 128-row activation boxes
  const int fw = epi == LLAMA_EPI_SWIGLU ? 128 : TM_BN;
  const long tiles = (long)((N + TM_BM - 1) / TM_BM) * ((M + fw - 1) / fw);
  // about one tile for every SM or more: at 144 tiles on 152 SMs (the O and
  // down projections of a 1052-row extend step) this kernel measured 2.7 %
  // faster for the whole step than the weights-on-M tiles
  return tiles * 10 >= 9L * std::max(1, sm_count);
}

bool gemm_tm_applies(const GemmCall& g) {
  if (g.dtype != LLAMA_BF16 || g.w_scale) return false;
  if (g.epi == kEpiRope) {
    if (!g.rope || g.rope->head_dim % 16 != 0) return false;
  } else if (g.rope || g.M > g.ldo) {
    return false;
  }
  return gemm_tm_shape(g.epi, g.M, g.N, g.split, g.sm_count);
}

template <int EPI>
static cudaError_t launch_tm(const GemmCall& g, cudaStream_t st) {
  TmParams p{};
  if (g.rope) p.rope = *g.rope;
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.num_kb = (g.K + TM_BK - 1) / TM_BK;
  p.lo_rows = (g.N + 15) / 16 * 16;
  p.fw = EPI == LLAMA_EPI_SWIGLU ? 128 : TM_BN;
  p.n_tok = (g.N + TM_BM - 1) / TM_BM;
  p.n_feat = (g.M + p.fw - 1) / p.fw;
  p.tiles = p.n_tok * p.n_feat;
  p.out = g.out;
  p.ldo = g.ldo;
  p.out_lo = g.out_lo;
  p.norm_gamma = reinterpret_cast<const bf16*>(g.norm_gamma);
  p.norm_out = reinterpret_cast<bf16*>(g.norm_out);
  p.norm_lo = g.norm_lo;
  p.ssq_out = g.ssq_out;
  p.ssq_in = g.ssq_in;
  p.ssq_tiles = g.ssq_tiles;
  p.ssq_ld = g.ssq_ld;
  p.norm_inv_h = g.norm_h > 0 ? 1.0f / (float)g.norm_h : 0.f;
  p.norm_eps = g.norm_eps;
  p.status = g.status;
  const int grid = std::min(p.tiles, std::max(1, g.sm_count));
  const CUtensorMap* up = g.map_up ? g.map_up : g.map_w;
  return launch_k(gemm_tm_kernel<EPI>, dim3(grid), dim3(TM_THREADS), TM_SMEM, st, 0, *g.map_w,
                  *up, *g.map_x, p);
}

cudaError_t launch_gemm_tm(const GemmCall& g, cudaStream_t st) {
  if (!gemm_tm_applies(g) || !g.map_w || !g.map_x || (g.epi == LLAMA_EPI_SWIGLU && !g.map_up))
    return cudaErrorInvalidValue;
  switch (g.epi) {
    case LLAMA_EPI_STORE_F32: return launch_tm<LLAMA_EPI_STORE_F32>(g, st);
    case LLAMA_EPI_RESID_F32: return launch_tm<LLAMA_EPI_RESID_F32>(g, st);
    case LLAMA_EPI_STORE_T: return launch_tm<LLAMA_EPI_STORE_T>(g, st);
    case kEpiRope: return launch_tm<kEpiRope>(g, st);
    default: return launch_tm<LLAMA_EPI_SWIGLU>(g, st);
  }
}

cudaError_t gemm_tm_prepare() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e;
  if ((e = cudaFuncSetAttribute(gemm_tm_kernel<LLAMA_EPI_STORE_F32>, a, (int)TM_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(gemm_tm_kernel<LLAMA_EPI_RESID_F32>, a, (int)TM_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(gemm_tm_kernel<LLAMA_EPI_STORE_T>, a, (int)TM_SMEM)) != cudaSuccess)
    return e;
  if ((e = cudaFuncSetAttribute(gemm_tm_kernel<kEpiRope>, a, (int)TM_SMEM)) != cudaSuccess)
    return e;
  return cudaFuncSetAttribute(gemm_tm_kernel<LLAMA_EPI_SWIGLU>, a, (int)TM_SMEM);
}

}  // namespace llgb
