// Grouped-query scaled dot-product attention ("Llama2架构与推理全解析" §2.3:
// scores q.k / sqrt(d), causal mask, softmax, weighted sum of V; §1.5 GQA:
// query head h reads K/V head h / G; §2.4: decode reads the whole cache).
//
// Decode (bf16, head_dim 128): one CTA per (sequence, K/V head, key split).
// A producer warp copies K and V of 16-key sub-tiles (one page of a paged
// cache, or 16 consecutive slots of a contiguous one) from HBM into shared
// memory with TMA (128-byte swizzle) into a 3-stage mbarrier ring; every
// query head of the group shares the tile. Four consumer warps each take one
// sub-tile per stage and run S = Q K^T and O += P V on mma.sync (the G query
// heads are the 16-row M side, zero-padded), with an online softmax in fp32
// (base-2 exponent, the running maximum subtracted before exp). The four
// warps' (max, sum, O) are merged through shared memory; with several key
// splits a small kernel merges the splits the same way.
//
// Prefill (bf16) runs on the tcgen05 tensor cores (k_prefill_tc.cu).
//
// fp32 configs use plain CUDA-core kernels (exact fp32, exp on the CUDA
// math library) for both phases.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace llgb {

constexpr int AD = 128;  // head_dim of the tensor-core kernels
constexpr float kLog2e = 1.4426950408889634f;

// ======================================================================== decode
constexpr int SUBK = 16;                               // keys per TMA box / page granule
constexpr int DTILE = 64;                              // keys per stage
constexpr int DSTAGES = 3;
constexpr int DEC_THREADS = 160;                       // 4 consumer warps + producer warp
constexpr uint32_t HALF_BYTES = SUBK * 128;            // 16 rows x 64 dims x bf16
constexpr uint32_t SUB_BYTES = 2 * HALF_BYTES;         // 16 rows x 128 dims
constexpr uint32_t TILE_HALF = DTILE * 128;            // 64 keys x 64 dims x bf16: 8 KB
constexpr uint32_t DSTAGE_BYTES = 4 * TILE_HALF;       // K and V, two dim halves each: 32 KB
// Stage layout: K dims 0-63 [64 keys][128 B], K dims 64-127, V dims 0-63,
// V dims 64-127; 16-key sub-tile j of a half starts at j * HALF_BYTES.
constexpr size_t DEC_SMEM = DSTAGES * DSTAGE_BYTES + 1024 + 256;
// FP8 E4M3 cache: one byte per value, so a 64-key tile of K (or V) is one
// 128-byte-swizzled box of 64 rows x 128 bytes; three CTAs per SM.
constexpr int F8_STAGES = 3;
constexpr uint32_t F8_TILE = DTILE * 128;  // K (or V) of 64 keys: 8 KB
constexpr uint32_t F8_SUB = SUBK * 128;    // 16 keys: 2 KB
constexpr uint32_t F8_STAGE = 2 * F8_TILE;
constexpr size_t DEC_SMEM_F8 = F8_STAGES * F8_STAGE + 1024 + 256;

struct DecParams {
  const bf16* q;
  size_t q_lo;
  const int32_t* positions;
  const int32_t* page_table;
  bf16* out;
  size_t out_lo;
  float* part;
  uint32_t* status;
  int n_q, n_kv, G, layer;
  int page_size, capacity, batch_cap, n_pages, max_pages;
  int splits, keys_per_split;
  int box_rows;  // 64: one TMA box per K/V half of a tile; 16: one per sub-tile
  float scale_log2;
  // extend steps: sequence b is handled only when it has exactly one new row,
  // which is row cu_rows[b] of q and of the output (null: row b)
  const int32_t* cu_rows;
  float v_scale;  // FP8 cache: V bytes are e4m3 * v_scale (1 otherwise; K's scale is in scale_log2)
  // keys the launch covers: min(cache slots, splits * keys_per_split)
  int key_limit;
};

// Number of keys sequence b attends (positions[b] + 1). A position below 0
// or one whose keys the launch does not cover (past the cache, or past the
// key range the split plan was sized for) is flagged; the sequence then
// attends no keys (negative position) or the covered keys only.
__device__ __forceinline__ int decode_keys(int pos, int key_limit, uint32_t* status, bool report) {
  if (pos < 0 || pos + 1 > key_limit) {
    if (report) flag(status, LLAMA_FLAG_POS_RANGE);
    return pos < 0 ? 0 : key_limit;
  }
  return pos + 1;
}

// Row index (within one layer's [rows, d] view of the cache) of the 16-key
// sub-tile starting at key k0 of sequence b, K/V head g. A page id outside the
// pool is flagged and mapped to a row range that TMA fills with zeros.
__device__ __forceinline__ int kv_row(const DecParams& p, int b, int g, int k0) {
  if (p.page_size == 0) return (b * p.n_kv + g) * p.capacity + k0;
  const int pi = k0 / p.page_size;
  const int page = pi < p.max_pages ? p.page_table[(size_t)b * p.max_pages + pi] : -1;
  if (page < 0 || page >= p.n_pages) {
    flag(p.status, LLAMA_FLAG_PAGE_RANGE);
    return -4 * SUBK;
  }
  return (page * p.n_kv + g) * p.page_size + (k0 % p.page_size);
}

__device__ __forceinline__ void cons_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// Consumer warps, tensor-core variant: the G query heads of the group are the
// M rows of mma.sync (zero-padded to 16); Q and P are carried as bf16 pairs.
// Leaves this warp's running max, sum and O in shared memory for the merge.
__device__ __forceinline__ void decode_consume_mma(const DecParams& p, uint8_t* smem,
                                                   uint64_t* full, uint64_t* empty,
                                                   volatile uint32_t* abort_flag, int b, int g,
                                                   int kbeg, int kend, int n_sub, int n_tiles,
                                                   int warp, int lane) {
  const int G = p.G;
  const int r0 = lane >> 2;
  // Q fragments (the G heads of the group as rows 0..G-1 of a 16-row tile);
  // with a pair operand the remainder fragments ride along (two MMAs each)
  uint32_t qa[8][4], ql[8][4];
  {
    const bf16* qb = p.q + ((size_t)b * p.n_q + (size_t)g * G) * AD;
    const bf16* qr = qb + p.q_lo;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int col = kk * 16 + 2 * (lane & 3);
      const int offs[4] = {r0 * AD + col, (r0 + 8) * AD + col, r0 * AD + col + 8,
                           (r0 + 8) * AD + col + 8};
      const bool ok[4] = {r0 < G, r0 + 8 < G, r0 < G, r0 + 8 < G};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qa[kk][i] = ok[i] ? *reinterpret_cast<const uint32_t*>(qb + offs[i]) : 0u;
        ql[kk][i] = (ok[i] && p.q_lo) ? *reinterpret_cast<const uint32_t*>(qr + offs[i]) : 0u;
      }
    }
  }
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  float oacc[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const int mi = lane >> 3, rr = lane & 7;

  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % DSTAGES;
    const uint32_t ph = (t / DSTAGES) & 1;
    if (*abort_flag) break;
    if (!mbar_wait(&full[s], ph, p.status)) {
      *abort_flag = 1;
      break;
    }
    const int sub = 4 * t + warp;
    if (sub < n_sub) {
      uint8_t* st = smem + s * DSTAGE_BYTES;
      const int k0 = kbeg + sub * SUBK;
      const int nvalid = min(SUBK, kend - k0);
      const uint32_t kbase = smem_u32(st + warp * HALF_BYTES);
      uint8_t* vptr = st + 2 * TILE_HALF + warp * HALF_BYTES;
      if (nvalid < SUBK) {  // rows past the last key may hold anything: zero them
        const int nz = (SUBK - nvalid) * 16;
        for (int i = lane; i < nz; i += 32) {
          const int row = nvalid + (i >> 4), half = (i >> 3) & 1, chunk = i & 7;
          *reinterpret_cast<uint4*>(vptr + half * TILE_HALF + row * 128 + chunk * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const uint32_t vbase = smem_u32(vptr);
      // S = Q K^T over 16 keys
      float sc[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sc[0][i] = sc[1][i] = 0.f;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int half = kk >> 2;
        const int chunk = (kk & 3) * 2 + (mi & 1);
        const int row = ((mi >> 1) << 3) + rr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kbase + half * TILE_HALF + swz128(row, chunk), b0, b1, b2, b3);
        mma_bf16_16816(sc[0], qa[kk], b0, b1);
        mma_bf16_16816(sc[1], qa[kk], b2, b3);
        if (p.q_lo) {
          mma_bf16_16816(sc[0], ql[kk], b0, b1);
          mma_bf16_16816(sc[1], ql[kk], b2, b3);
        }
      }
      // online softmax in base 2
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int key = nb * 8 + 2 * (lane & 3) + (i & 1);
          const float v = key < nvalid ? sc[nb][i] * p.scale_log2 : -INFINITY;
          sc[nb][i] = v;
          mx[i >> 1] = fmaxf(mx[i >> 1], v);
        }
      float corr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mnew = fmaxf(mrow[h], mx[h]);
        corr[h] = mnew == -INFINITY ? 1.f : ex2(mrow[h] - mnew);
        mrow[h] = mnew;
      }
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int nb = 0; nb < 2; ++nb)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int h = i >> 1;
          const float pv = mrow[h] == -INFINITY ? 0.f : ex2(sc[nb][i] - mrow[h]);
          sc[nb][i] = pv;
          ps[h] += pv;
        }
      lrow[0] = lrow[0] * corr[0] + ps[0];
      lrow[1] = lrow[1] * corr[1] + ps[1];
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        oacc[dn][0] *= corr[0];
        oacc[dn][1] *= corr[0];
        oacc[dn][2] *= corr[1];
        oacc[dn][3] *= corr[1];
      }
      // P as a bf16 pair: hi = bf16(p), lo = bf16(p - hi); O += P_hi V + P_lo V
      uint32_t pa[4], pl[4];
      split_pack(sc[0][0], sc[0][1], pa[0], pl[0]);
      split_pack(sc[0][2], sc[0][3], pa[1], pl[1]);
      split_pack(sc[1][0], sc[1][1], pa[2], pl[2]);
      split_pack(sc[1][2], sc[1][3], pa[3], pl[3]);
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int c16 = dp * 2 + (mi >> 1);
        const int row = ((mi & 1) << 3) + rr;
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vbase + (c16 >> 3) * TILE_HALF + swz128(row, c16 & 7), b0, b1, b2, b3);
        mma_bf16_16816(oacc[2 * dp], pa, b0, b1);
        mma_bf16_16816(oacc[2 * dp + 1], pa, b2, b3);
        mma_bf16_16816(oacc[2 * dp], pl, b0, b1);
        mma_bf16_16816(oacc[2 * dp + 1], pl, b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

  // ---- this warp's (max, sum, O) to shared memory for the 4-warp merge
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
  }
  float* so = reinterpret_cast<float*>(smem);  // [4][16][128]
  float* sm = so + 4 * 16 * AD;                // [4][16]
  float* sl = sm + 64;                         // [4][16]
  cons_bar();  // every consumer is done with the stage buffers
#pragma unroll
  for (int dn = 0; dn < 16; ++dn)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = r0 + (i >= 2 ? 8 : 0);
      const int col = dn * 8 + 2 * (lane & 3) + (i & 1);
      so[(warp * 16 + row) * AD + col] = oacc[dn][i];
    }
  if ((lane & 3) == 0) {
    sm[warp * 16 + r0] = mrow[0];
    sm[warp * 16 + r0 + 8] = mrow[1];
    sl[warp * 16 + r0] = lrow[0];
    sl[warp * 16 + r0 + 8] = lrow[1];
  }
}

// Consumer warps, key-major tensor-core variant for groups of at most 8 query
// heads: S^T = K Q^T puts the 16 keys of a sub-tile on the M rows and the
// group's heads on N = 8, and O^T = V^T P^T puts 16 head dims on M, so MHA
// wastes no MMA rows. Q and P are bf16 pairs (two MMAs each); P^T reaches
// operand layout through movmatrix transposes. Lane l tracks heads 2(l%4) and
// 2(l%4)+1. Same shared-memory output as the other variant.
constexpr int kKeyMajorMaxG = 8;
__device__ __forceinline__ void decode_consume_keymajor(const DecParams& p, uint8_t* smem,
                                                        uint64_t* full, uint64_t* empty,
                                                        volatile uint32_t* abort_flag, int b,
                                                        int g, int kbeg, int kend, int n_sub,
                                                        int n_tiles, int warp, int lane) {
  const int G = p.G;
  const int hq = lane >> 2;             // head of this lane's Q^T columns (B operand)
  const int hc = 2 * (lane & 3);        // first of the two heads this lane accumulates
  // Q^T fragments: b0/b1 = Q[head lane/4][16 kk + 2(l%4) + {0,1} (+8)]
  uint32_t qh[8][2], ql[8][2];
  {
    const bf16* qb = p.q + ((size_t)b * p.n_q + (size_t)g * G + hq) * AD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int col = kk * 16 + 2 * (lane & 3);
      const bool ok = hq < G;
      qh[kk][0] = ok ? *reinterpret_cast<const uint32_t*>(qb + col) : 0u;
      qh[kk][1] = ok ? *reinterpret_cast<const uint32_t*>(qb + col + 8) : 0u;
      ql[kk][0] = (ok && p.q_lo) ? *reinterpret_cast<const uint32_t*>(qb + p.q_lo + col) : 0u;
      ql[kk][1] = (ok && p.q_lo) ? *reinterpret_cast<const uint32_t*>(qb + p.q_lo + col + 8) : 0u;
    }
  }
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float oacc[8][4];  // O^T tile dt: rows d = 16 dt + l/4 (+8), columns heads hc, hc+1
#pragma unroll
  for (int i = 0; i < 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const int mi = lane >> 3, rr = lane & 7;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % DSTAGES;
    const uint32_t ph = (t / DSTAGES) & 1;
    if (*abort_flag) break;
    if (!mbar_wait(&full[s], ph, p.status)) {
      *abort_flag = 1;
      break;
    }
    const int sub = 4 * t + warp;
    if (sub < n_sub) {
      uint8_t* st = smem + s * DSTAGE_BYTES;
      const int k0 = kbeg + sub * SUBK;
      const int nvalid = min(SUBK, kend - k0);
      const uint32_t kbase = smem_u32(st + warp * HALF_BYTES);
      uint8_t* vptr = st + 2 * TILE_HALF + warp * HALF_BYTES;
      if (nvalid < SUBK) {  // rows past the last key may hold anything: zero them
        const int nz = (SUBK - nvalid) * 16;
        for (int i = lane; i < nz; i += 32) {
          const int row = nvalid + (i >> 4), half = (i >> 3) & 1, chunk = i & 7;
          *reinterpret_cast<uint4*>(vptr + half * TILE_HALF + row * 128 + chunk * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const uint32_t vbase = smem_u32(vptr);
      // S^T (16 keys x 8 heads): hi and lo parts of Q in separate chains
      float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        // A = K[16 keys][16 dims]: matrices (keys 0-7, c), (keys 8-15, c), (0-7, c+1), (8-15, c+1)
        const int row = ((mi & 1) << 3) + rr;
        const int chunk = (kk & 3) * 2 + (mi >> 1);
        uint32_t a[4];
        ldsm_x4(kbase + (kk >> 2) * TILE_HALF + swz128(row, chunk), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(sh, a, qh[kk][0], qh[kk][1]);
        if (p.q_lo) mma_bf16_16816(sl, a, ql[kk][0], ql[kk][1]);
      }
      // lane holds S^T[key l/4 (+8)][heads hc, hc+1]; online softmax per head
      float sv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = (lane >> 2) + (i >= 2 ? 8 : 0);
        sv[i] = key < nvalid ? (sh[i] + sl[i]) * p.scale_log2 : -INFINITY;
      }
      float corr[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float mx = fmaxf(sv[j], sv[j + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m_run[j], mx);
        corr[j] = mnew == m_run[j] ? 1.f : ex2(m_run[j] - mnew);  // unchanged max: exactly 1
        m_run[j] = mnew;
      }
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = i & 1;
        pv[i] = m_run[j] == -INFINITY ? 0.f : ex2(sv[i] - m_run[j]);
      }
      l_run[0] = l_run[0] * corr[0] + pv[0] + pv[2];
      l_run[1] = l_run[1] * corr[1] + pv[1] + pv[3];
      // once the running maxima settle most sub-tiles leave them unchanged
      if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
        for (int dt = 0; dt < 8; ++dt) {
          oacc[dt][0] *= corr[0];
          oacc[dt][1] *= corr[1];
          oacc[dt][2] *= corr[0];
          oacc[dt][3] *= corr[1];
        }
      }
      // P^T as the B operand (16 keys x 8 heads): transpose the two 8x8 halves
      uint32_t p0h, p0l, p1h, p1l;
      split_pack(pv[0], pv[1], p0h, p0l);  // keys 0-7
      split_pack(pv[2], pv[3], p1h, p1l);  // keys 8-15
      const uint32_t bh0 = movmatrix_t(p0h), bh1 = movmatrix_t(p1h);
      const uint32_t bl0 = movmatrix_t(p0l), bl1 = movmatrix_t(p1l);
      // O^T += V^T P^T: A = V^T[16 dims][16 keys] from V[key][dim] by transposed loads
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) {
        const int c16 = dt * 2 + (mi & 1);
        const int row = ((mi >> 1) << 3) + rr;
        uint32_t a[4];
        ldsm_x4_t(vbase + (c16 >> 3) * TILE_HALF + swz128(row, c16 & 7), a[0], a[1], a[2], a[3]);
        mma_bf16_16816(oacc[dt], a, bh0, bh1);
        mma_bf16_16816(oacc[dt], a, bl0, bl1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // ---- this warp's (max, sum, O) to shared memory for the 4-warp merge
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
  }
  float* so = reinterpret_cast<float*>(smem);  // [4][16][128]
  float* smx = so + 4 * 16 * AD;               // [4][16]
  float* ssum = smx + 64;                      // [4][16]
  cons_bar();  // every consumer is done with the stage buffers
#pragma unroll
  for (int dt = 0; dt < 8; ++dt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int head = hc + (i & 1);
      const int d = dt * 16 + (lane >> 2) + (i >= 2 ? 8 : 0);
      if (head < G) so[(warp * 16 + head) * AD + d] = oacc[dt][i];
    }
  if (lane < 4) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (hc + j < G) {
        smx[warp * 16 + hc + j] = m_run[j];
        ssum[warp * 16 + hc + j] = l_run[j];
      }
  }
}

// Consumer warps for an FP8 E4M3 cache (groups of at most 8 query heads),
// key-major like decode_consume_keymajor but on f16 tensor-core MMAs: E4M3
// values are exact in f16, so K and V enter the MMA unrounded; Q and P are
// single f16 values (11 significant bits, against the 4 of every cached value:
// a second, remainder MMA would buy nothing here). The stage holds K
// [64 keys][128 bytes] then V the same.
//  * S^T = K Q^T: ldmatrix on the byte rows gives each lane 4 consecutive
//    dims of a key; their two f16 pairs serve as the fragment's k-columns
//    (2t, 2t+1) and (2t+8, 2t+9). The head dims are thus taken in a permuted
//    order, and Q's fragments use the same order, so the dot products are
//    unchanged.
//  * O^T += V^T P^T: the A fragment needs one dim of two keys per register,
//    so each lane loads 4-byte words (4 dims) of its 4 keys and pairs bytes
//    of two keys with a byte permute. The output dims come out permuted:
//    row r of m-tile mt is dim 64*(mt/4) + 4*r + mt%4, undone when O is
//    written. K's scale is in scale_log2, V's is applied at the output.
__device__ __forceinline__ void decode_consume_fp8(const DecParams& p, uint8_t* smem,
                                                   uint64_t* full, uint64_t* empty,
                                                   volatile uint32_t* abort_flag, int b, int g,
                                                   int kbeg, int kend, int n_sub, int n_tiles,
                                                   int warp, int lane) {
  const int G = p.G;
  const int hq = lane >> 2;   // head of this lane's Q^T column (B operand), also its row group
  const int t4 = lane & 3;
  const int hc = 2 * t4;      // first of the two heads this lane accumulates
  // Q^T fragments (f16), dims in the permuted order: chunk kk of 16 dims;
  // register 0 holds dims 4t, 4t+1 and register 1 dims 4t+2, 4t+3
  uint32_t qh[8][2];
  {
    const bf16* qb = p.q + ((size_t)b * p.n_q + (size_t)g * G + hq) * AD;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = kk * 16 + 4 * t4 + 2 * j;
        float v0 = 0.f, v1 = 0.f;
        if (hq < G) {
          v0 = __bfloat162float(qb[col]) + (p.q_lo ? __bfloat162float(qb[p.q_lo + col]) : 0.f);
          v1 = __bfloat162float(qb[col + 1]) +
               (p.q_lo ? __bfloat162float(qb[p.q_lo + col + 1]) : 0.f);
        }
        const __half2 h2 = __floats2half2_rn(v0, v1);
        qh[kk][j] = *reinterpret_cast<const uint32_t*>(&h2);
      }
  }
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float oacc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const int mi = lane >> 3, rr = lane & 7;
  for (int t = 0; t < n_tiles; ++t) {
    const int s = t % F8_STAGES;
    const uint32_t ph = (t / F8_STAGES) & 1;
    if (*abort_flag) break;
    if (!mbar_wait(&full[s], ph, p.status)) {
      *abort_flag = 1;
      break;
    }
    const int sub = 4 * t + warp;
    if (sub < n_sub) {
      uint8_t* st = smem + s * F8_STAGE;
      const int k0 = kbeg + sub * SUBK;
      const int nvalid = min(SUBK, kend - k0);
      const uint32_t kbase = smem_u32(st + warp * F8_SUB);
      const uint8_t* vsub = st + F8_TILE + warp * F8_SUB;
      const uint32_t vbase = smem_u32(vsub);
      if (nvalid < SUBK) {  // V rows past the last key may hold anything: zero them
        const int nz = (SUBK - nvalid) * 8;
        for (int i = lane; i < nz; i += 32)
          *reinterpret_cast<uint4*>(const_cast<uint8_t*>(vsub) + (nvalid + (i >> 3)) * 128 +
                                    (i & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
        __syncwarp();
      }
      // V words (loaded first, used after the softmax): keys 2t, 2t+1, 2t+8, 2t+9; dims 64h + 32e + 4(l/4) .. +3
      uint32_t w[4][2][2];
#pragma unroll
      for (int kq = 0; kq < 4; ++kq) {
        const int key = (kq & 1) + 2 * t4 + (kq >> 1) * 8;
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int off = 64 * h + 32 * e + 4 * hq;
            w[kq][h][e] = lds32(vbase + key * 128 + (((off >> 4) ^ (key & 7)) << 4) + (off & 15));
          }
      }
      // S^T (16 keys x 8 heads), even and odd k-steps in separate chains
      float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {  // dims 32kp .. 32kp + 31: two k-steps
        const int row = ((mi & 1) << 3) + rr;
        const int chunk = kp * 2 + (mi >> 1);
        uint32_t r[4];
        ldsm_x4(kbase + swz128(row, chunk), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a[4];  // key rows g (r[2h]) and g + 8 (r[2h+1]); dims 4t, 4t+1 then 4t+2, 4t+3
          e4m3x4_to_f16x2x2(r[2 * h], a[0], a[2]);
          e4m3x4_to_f16x2x2(r[2 * h + 1], a[1], a[3]);
          const int kk = 2 * kp + h;
          mma_f16_16816(h ? sl : sh, a, qh[kk][0], qh[kk][1]);
        }
      }
      // lane holds S^T[key l/4 (+8)][heads hc, hc+1]; online softmax per head
      float sv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int key = (lane >> 2) + (i >= 2 ? 8 : 0);
        sv[i] = key < nvalid ? (sh[i] + sl[i]) * p.scale_log2 : -INFINITY;
      }
      float corr[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float mx = fmaxf(sv[j], sv[j + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m_run[j], mx);
        corr[j] = mnew == m_run[j] ? 1.f : ex2(m_run[j] - mnew);  // unchanged max: exactly 1
        m_run[j] = mnew;
      }
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = i & 1;
        pv[i] = m_run[j] == -INFINITY ? 0.f : ex2(sv[i] - m_run[j]);
      }
      l_run[0] = l_run[0] * corr[0] + pv[0] + pv[2];
      l_run[1] = l_run[1] * corr[1] + pv[1] + pv[3];
      // once the running maxima settle most sub-tiles leave them unchanged
      if (__any_sync(0xffffffffu, corr[0] != 1.f || corr[1] != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          oacc[mt][0] *= corr[0];
          oacc[mt][1] *= corr[1];
          oacc[mt][2] *= corr[0];
          oacc[mt][3] *= corr[1];
        }
      }
      // P^T as the B operand (16 keys x 8 heads), f16
      const __half2 p0 = __floats2half2_rn(pv[0], pv[1]);  // keys 0-7
      const __half2 p1 = __floats2half2_rn(pv[2], pv[3]);  // keys 8-15
      const uint32_t bh0 = movmatrix_t(*reinterpret_cast<const uint32_t*>(&p0));
      const uint32_t bh1 = movmatrix_t(*reinterpret_cast<const uint32_t*>(&p1));
      // O^T += V^T P^T over 8 m-tiles of permuted dims; one byte permute
      // gathers the key pairs of two m-tiles (bytes j and j + 1 of both keys)
#pragma unroll
      for (int mp = 0; mp < 4; ++mp) {  // m-tiles 2mp and 2mp + 1
        const int h = mp >> 1, j = (mp & 1) * 2;
        const uint32_t sel = (uint32_t)j | ((uint32_t)(4 + j) << 4) | ((uint32_t)(j + 1) << 8) |
                             ((uint32_t)(5 + j) << 12);
        uint32_t a0[4], a1[4];
        e4m3x4_to_f16x2x2(__byte_perm(w[0][h][0], w[1][h][0], sel), a0[0], a1[0]);
        e4m3x4_to_f16x2x2(__byte_perm(w[0][h][1], w[1][h][1], sel), a0[1], a1[1]);
        e4m3x4_to_f16x2x2(__byte_perm(w[2][h][0], w[3][h][0], sel), a0[2], a1[2]);
        e4m3x4_to_f16x2x2(__byte_perm(w[2][h][1], w[3][h][1], sel), a0[3], a1[3]);
        mma_f16_16816(oacc[2 * mp], a0, bh0, bh1);
        mma_f16_16816(oacc[2 * mp + 1], a1, bh0, bh1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  // ---- this warp's (max, sum, O) to shared memory for the 4-warp merge
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
    l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
  }
  float* so = reinterpret_cast<float*>(smem);  // [4][16][128]
  float* smx = so + 4 * 16 * AD;               // [4][16]
  float* ssum = smx + 64;                      // [4][16]
  cons_bar();  // every consumer is done with the stage buffers
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int head = hc + (i & 1);
      const int d = 64 * (mt >> 2) + 4 * ((lane >> 2) + (i >= 2 ? 8 : 0)) + (mt & 3);
      if (head < G) so[(warp * 16 + head) * AD + d] = oacc[mt][i];
    }
  if (lane < 4) {
#pragma unroll
    for (int j = 0; j < 2; ++j)
      if (hc + j < G) {
        smx[warp * 16 + hc + j] = m_run[j];
        ssum[warp * 16 + hc + j] = l_run[j];
      }
  }
}

template <bool KEYMAJOR, bool FP8>
__global__ void __launch_bounds__(DEC_THREADS, FP8 ? 4 : 2)
    attn_decode_kernel(const __grid_constant__ CUtensorMap mapK,
                       const __grid_constant__ CUtensorMap mapV,
                       const __grid_constant__ CUtensorMap mapK16,
                       const __grid_constant__ CUtensorMap mapV16, DecParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int NS = FP8 ? F8_STAGES : DSTAGES;
  constexpr uint32_t SB = FP8 ? F8_STAGE : DSTAGE_BYTES;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + NS * SB);
  uint64_t* empty = full + NS;
  volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(empty + NS);

  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  static_assert((4 * 16 * AD + 128) * sizeof(float) <= (size_t)NS * SB,
                "the 4-warp merge area (O, max, sum) aliases the stage ring");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int qrow = b;  // row of q and of the output
  if (p.cu_rows) {
    qrow = p.cu_rows[b];
    if (p.cu_rows[b + 1] - qrow != 1) {  // longer pieces go to the prefill-style kernel
      grid_dep_wait();
      return;
    }
  }
  // positions and the page table are caller inputs, complete before the step
  const int n_keys = decode_keys(p.positions[b], p.key_limit, p.status,
                                 split == 0 && threadIdx.x == 0);
  const int kbeg = split * p.keys_per_split;
  const int kend = min(n_keys, kbeg + p.keys_per_split);
  if (kbeg >= kend) {  // this split has no keys (the merge skips it)
    grid_dep_wait();
    if (p.splits == 1 && threadIdx.x < AD) {
      // a sequence without keys: zero output rows, as the split merge writes
      for (int r = 0; r < p.G; ++r) {
        const size_t oh = (size_t)qrow * p.n_q + (size_t)g * p.G + r;
        p.out[oh * AD + threadIdx.x] = __float2bfloat16_rn(0.f);
        if (p.out_lo) p.out[oh * AD + threadIdx.x + p.out_lo] = __float2bfloat16_rn(0.f);
      }
    }
    return;
  }
  const int n_sub = (kend - kbeg + SUBK - 1) / SUBK;
  const int n_tiles = (n_sub + 3) / 4;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 4) {  // ------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      tma_prefetch_desc(&mapK16);
      tma_prefetch_desc(&mapV16);
      const uint64_t pol_kv = l2_policy_evict_first();  // the cache is streamed once
      int issued = 0;
      bool ok = true, waited = false;
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % NS;
        const uint32_t ph = (t / NS) & 1;
        // Keys below the new token were cached by earlier steps and can be
        // fetched while the previous kernel finishes; the tile holding the
        // new token's K/V (written by the RoPE/append kernel) waits for it.
        if (!waited && kbeg + (t + 1) * DTILE >= n_keys) {
          grid_dep_wait();
          grid_dep_launch();
          waited = true;
        }
        if (!mbar_wait(&empty[s], ph ^ 1, p.status)) {
          ok = false;
          *abort_flag = 1;
          break;
        }
        const int nsub = min(4, n_sub - 4 * t);
        uint8_t* st = smem + s * SB;
        if (FP8) {  // K tile at st, V tile at st + F8_TILE, [keys][128 bytes] each
          if (p.box_rows == DTILE && nsub == 4) {
            const int row = kv_row(p, b, g, kbeg + t * DTILE);
            mbar_arrive_expect_tx(&full[s], F8_STAGE);
            tma_load_3d_hint(st, &mapK, &full[s], 0, row, p.layer, pol_kv);
            tma_load_3d_hint(st + F8_TILE, &mapV, &full[s], 0, row, p.layer, pol_kv);
          } else {
            mbar_arrive_expect_tx(&full[s], nsub * 2 * F8_SUB);
            for (int j = 0; j < nsub; ++j) {
              const int row = kv_row(p, b, g, kbeg + (4 * t + j) * SUBK);
              tma_load_3d_hint(st + j * F8_SUB, &mapK16, &full[s], 0, row, p.layer, pol_kv);
              tma_load_3d_hint(st + F8_TILE + j * F8_SUB, &mapV16, &full[s], 0, row, p.layer,
                               pol_kv);
            }
          }
        } else if (p.box_rows == DTILE && nsub == 4) {  // 64 contiguous keys: one box per half
          const int row = kv_row(p, b, g, kbeg + t * DTILE);
          mbar_arrive_expect_tx(&full[s], DSTAGE_BYTES);
          tma_load_3d_hint(st, &mapK, &full[s], 0, row, p.layer, pol_kv);
          tma_load_3d_hint(st + TILE_HALF, &mapK, &full[s], 64, row, p.layer, pol_kv);
          tma_load_3d_hint(st + 2 * TILE_HALF, &mapV, &full[s], 0, row, p.layer, pol_kv);
          tma_load_3d_hint(st + 3 * TILE_HALF, &mapV, &full[s], 64, row, p.layer, pol_kv);
        } else {
          mbar_arrive_expect_tx(&full[s], nsub * SUB_BYTES * 2);
          for (int j = 0; j < nsub; ++j) {
            const int row = kv_row(p, b, g, kbeg + (4 * t + j) * SUBK);
            uint8_t* kd = st + j * HALF_BYTES;
            uint8_t* vd = st + 2 * TILE_HALF + j * HALF_BYTES;
            tma_load_3d_hint(kd, &mapK16, &full[s], 0, row, p.layer, pol_kv);
            tma_load_3d_hint(kd + TILE_HALF, &mapK16, &full[s], 64, row, p.layer, pol_kv);
            tma_load_3d_hint(vd, &mapV16, &full[s], 0, row, p.layer, pol_kv);
            tma_load_3d_hint(vd + TILE_HALF, &mapV16, &full[s], 64, row, p.layer, pol_kv);
          }
        }
        ++issued;
      }
      if (!ok) {
        for (int t = issued - 1; t >= 0 && t >= issued - NS; --t)
          mbar_wait(&full[t % NS], (t / NS) & 1, p.status);
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  grid_dep_wait();  // q comes from the RoPE/append kernel
  grid_dep_launch();
  if (FP8)
    decode_consume_fp8(p, smem, full, empty, abort_flag, qrow, g, kbeg, kend, n_sub, n_tiles, warp,
                       lane);
  else if (KEYMAJOR)
    decode_consume_keymajor(p, smem, full, empty, abort_flag, qrow, g, kbeg, kend, n_sub, n_tiles,
                            warp, lane);
  else
    decode_consume_mma(p, smem, full, empty, abort_flag, qrow, g, kbeg, kend, n_sub, n_tiles, warp,
                       lane);
  const int G = p.G;
  float* so = reinterpret_cast<float*>(smem);  // [4][16][128]
  float* sm = so + 4 * 16 * AD;                // [4][16]
  float* sl = sm + 64;                         // [4][16]
  cons_bar();
  if (*abort_flag) return;
  const int t = threadIdx.x;  // output dim
  for (int r = 0; r < G; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, sm[w * 16 + r]);
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float mw = sm[w * 16 + r];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L += sl[w * 16 + r] * f;
        O += so[(w * 16 + r) * AD + t] * f;
      }
    }
    const size_t bh = (size_t)b * p.n_q + (size_t)g * G + r;
    if (p.splits == 1) {
      const size_t oh = (size_t)qrow * p.n_q + (size_t)g * G + r;
      const float v = L > 0.f ? O / L * p.v_scale : 0.f;
      const bf16 hi = __float2bfloat16_rn(v);
      p.out[oh * AD + t] = hi;
      if (p.out_lo) p.out[oh * AD + t + p.out_lo] = __float2bfloat16_rn(v - __bfloat162float(hi));
    } else {
      float* pp = p.part + (bh * p.splits + split) * (AD + 2);
      pp[t] = O;
      if (t == 0) {
        pp[AD] = M;
        pp[AD + 1] = L;
      }
    }
  }
}

// Merge the key splits of (sequence, head) bh: rescale each split's sum and
// output by 2^(m_s - max m) and normalise.
__global__ void attn_combine_kernel(const float* __restrict__ part,
                                    const int32_t* __restrict__ positions, int n_q, int splits,
                                    int keys_per_split, int key_limit, int d, void* out,
                                    size_t out_lo, const int32_t* cu_rows, float v_scale) {
  grid_dep_wait();
  grid_dep_launch();
  const int bh = blockIdx.x;
  const int b = bh / n_q;
  size_t oh = bh;  // output row-head
  if (cu_rows) {
    if (cu_rows[b + 1] - cu_rows[b] != 1) return;
    oh = (size_t)cu_rows[b] * n_q + (bh - (size_t)b * n_q);
  }
  const int n_keys = decode_keys(positions[b], key_limit, nullptr, false);
  const int used = min(splits, (n_keys + keys_per_split - 1) / keys_per_split);
  const float* pp = part + (size_t)bh * splits * (d + 2);
  float M = -INFINITY;
  for (int s = 0; s < used; ++s) M = fmaxf(M, pp[(size_t)s * (d + 2) + d]);
  for (int t = threadIdx.x; t < d; t += blockDim.x) {
    float L = 0.f, O = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < used; ++s) {
        const float* ps = pp + (size_t)s * (d + 2);
        const float f = ps[d] == -INFINITY ? 0.f : exp2f(ps[d] - M);
        L += ps[d + 1] * f;
        O += ps[t] * f;
      }
    }
    const float v = L > 0.f ? O / L * v_scale : 0.f;
    const bf16 hi = __float2bfloat16_rn(v);
    reinterpret_cast<bf16*>(out)[oh * d + t] = hi;
    if (out_lo)
      reinterpret_cast<bf16*>(out)[oh * d + t + out_lo] =
          __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

// ======================================================================== fp32 CUDA-core kernels
// Decode: one CTA per (query head, sequence); scores in shared memory.
__global__ void attn_decode_f32_kernel(const float* __restrict__ q, const int32_t* positions,
                                       const float* __restrict__ kc, const float* __restrict__ vc,
                                       const int32_t* page_table, float* __restrict__ out,
                                       int n_q, int n_kv, int d, int layer, int page_size,
                                       int capacity, int batch_cap, int n_pages, int max_pages,
                                       uint32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ float sh[];
  const int h = blockIdx.x, b = blockIdx.y;
  const int g = h / (n_q / n_kv);
  const int cap_keys = page_size ? max_pages * page_size : capacity;
  const int n = decode_keys(positions[b], cap_keys, nullptr, false);
  float* qs = sh;
  float* sc = sh + d;
  float* red = sc + cap_keys;
  for (int i = threadIdx.x; i < d; i += blockDim.x) qs[i] = q[((size_t)b * n_q + h) * d + i];
  __syncthreads();
  auto slot = [&](int m) -> long long {
    if (page_size == 0) return (((long long)layer * batch_cap + b) * n_kv + g) * capacity + m;
    const int page = page_table[(size_t)b * max_pages + m / page_size];
    if (page < 0 || page >= n_pages) return -1;
    return (((long long)layer * n_pages + page) * n_kv + g) * page_size + m % page_size;
  };
  const float scale = 1.0f / sqrtf((float)d);
  for (int m = threadIdx.x; m < n; m += blockDim.x) {
    const long long sl = slot(m);
    float s = 0.f;
    if (sl >= 0) {
      const float* kr = kc + sl * d;
      for (int i = 0; i < d; ++i) s = fmaf(qs[i], kr[i], s);
    } else {
      flag(status, LLAMA_FLAG_PAGE_RANGE);
    }
    sc[m] = s * scale;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int m = threadIdx.x; m < n; m += blockDim.x) mx = fmaxf(mx, sc[m]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = -INFINITY;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
  __syncthreads();
  for (int m = threadIdx.x; m < n; m += blockDim.x) sc[m] = expf(sc[m] - mx);
  __syncthreads();
  float sum = 0.f;
  for (int m = 0; m < n; ++m) sum += sc[m];
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float o = 0.f;
    for (int m = 0; m < n; ++m) {
      const long long sl = slot(m);
      if (sl >= 0) o = fmaf(sc[m], vc[sl * d + i], o);
    }
    out[((size_t)b * n_q + h) * d + i] = n > 0 ? o / sum : 0.f;
  }
}

// Prefill: one CTA per (row, head, sequence), keys 0..row of its sequence.
__global__ void attn_prefill_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                                        const float* __restrict__ v, float* __restrict__ out,
                                        int T, int n_q, int n_kv, int d) {
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ float sh[];
  const int t = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int g = h / (n_q / n_kv);
  const int n = t + 1;
  float* qs = sh;
  float* sc = sh + d;
  float* red = sc + T;
  const size_t r = (size_t)b * T + t;
  for (int i = threadIdx.x; i < d; i += blockDim.x) qs[i] = q[(r * n_q + h) * d + i];
  __syncthreads();
  const float scale = 1.0f / sqrtf((float)d);
  for (int m = threadIdx.x; m < n; m += blockDim.x) {
    const float* kr = k + (((size_t)b * T + m) * n_kv + g) * d;
    float s = 0.f;
    for (int i = 0; i < d; ++i) s = fmaf(qs[i], kr[i], s);
    sc[m] = s * scale;
  }
  __syncthreads();
  float mx = -INFINITY;
  for (int m = threadIdx.x; m < n; m += blockDim.x) mx = fmaxf(mx, sc[m]);
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  mx = -INFINITY;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, red[w]);
  __syncthreads();
  for (int m = threadIdx.x; m < n; m += blockDim.x) sc[m] = expf(sc[m] - mx);
  __syncthreads();
  float sum = 0.f;
  for (int m = 0; m < n; ++m) sum += sc[m];
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    float o = 0.f;
    for (int m = 0; m < n; ++m) o = fmaf(sc[m], v[(((size_t)b * T + m) * n_kv + g) * d + i], o);
    out[(r * n_q + h) * d + i] = o / sum;
  }
}

// ======================================================================== host side
static void decode_plan(int B, int n_kv, int max_keys, int sm_count, int& splits, int& kps) {
  const int slots = std::max(1, sm_count) * 2;
  const int pairs = std::max(1, B * n_kv);
  int s = 1;
  while (pairs * s < 2 * slots && s < 16 && (max_keys + 2 * s - 1) / (2 * s) >= 256) s *= 2;
  kps = (max_keys + s - 1) / s;
  kps = std::min(kps, 2048);
  kps = std::max(DTILE, (kps + DTILE - 1) / DTILE * DTILE);
  splits = (max_keys + kps - 1) / kps;
}

size_t attn_decode_partial_bytes(int B, int n_q, int head_dim, int max_keys, int sm_count,
                                 int n_kv) {
  int splits, kps;
  decode_plan(B, n_kv, max_keys, sm_count, splits, kps);
  if (splits <= 1) return 0;
  return (size_t)B * n_q * splits * (head_dim + 2) * sizeof(float);
}

cudaError_t attn_prepare() {
  cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DEC_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_decode_kernel<true, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DEC_SMEM);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_decode_kernel<true, true>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)DEC_SMEM_F8);
  if (e != cudaSuccess) return e;
  return attn_prefill_tc_prepare();
}

cudaError_t launch_attn_decode(int dtype, const AttnDecodeArgs& a, cudaStream_t st) {
  int splits, kps;
  decode_plan(a.B, a.n_kv, a.max_keys, a.sm_count, splits, kps);
  if (dtype == LLAMA_F32) {
    const int cap_keys = a.page_size ? a.max_pages * a.page_size : a.capacity;
    const size_t sm = (size_t)(a.head_dim + cap_keys + 32) * sizeof(float);
    if (sm > 200 * 1024) return cudaErrorInvalidValue;
    if (sm > 48 * 1024)
      cudaFuncSetAttribute(attn_decode_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm);
    return launch_k(attn_decode_f32_kernel, dim3(a.n_q, a.B), dim3(128), sm, st, 0,
                    (const float*)a.q, a.positions, (const float*)a.k_cache,
                    (const float*)a.v_cache, a.page_table, (float*)a.out, a.n_q, a.n_kv,
                    a.head_dim, a.layer, a.page_size, a.capacity, a.batch_cap, a.n_pages,
                    a.max_pages, a.status);
  }
  if (a.head_dim != AD) return cudaErrorInvalidValue;
  if (splits > 1 && (size_t)a.B * a.n_q * splits * (AD + 2) * sizeof(float) > a.partial_bytes) {
    // workspace sized for fewer splits: one split per sequence
    splits = 1;
    kps = std::max(DTILE, (a.max_keys + DTILE - 1) / DTILE * DTILE);
  }
  DecParams p;
  p.q = (const bf16*)a.q;
  p.q_lo = a.q_lo;
  p.positions = a.positions;
  p.page_table = a.page_table;
  p.out = (bf16*)a.out;
  p.out_lo = a.out_lo;
  p.part = a.partial;
  p.status = a.status;
  p.n_q = a.n_q;
  p.n_kv = a.n_kv;
  p.G = a.n_q / a.n_kv;
  p.layer = a.layer;
  p.page_size = a.page_size;
  p.capacity = a.capacity;
  p.batch_cap = a.batch_cap;
  p.n_pages = a.n_pages;
  p.max_pages = a.max_pages;
  p.splits = splits;
  p.keys_per_split = kps;
  p.box_rows = a.box_rows == DTILE ? DTILE : SUBK;
  p.cu_rows = a.cu_rows;
  p.scale_log2 = kLog2e / sqrtf((float)AD) * (a.kv_fp8 ? a.k_scale : 1.f);
  p.v_scale = a.kv_fp8 ? a.v_scale : 1.f;
  const int cap_keys = a.page_size ? a.max_pages * a.page_size : a.capacity;
  p.key_limit = (int)std::min<long long>(cap_keys, (long long)splits * kps);
  const bool keymajor = p.G <= kKeyMajorMaxG;
  if (a.kv_fp8 && !keymajor) return cudaErrorInvalidValue;
  const dim3 grid(splits, a.n_kv, a.B), block(DEC_THREADS);
  cudaError_t e =
      a.kv_fp8 ? launch_k(attn_decode_kernel<true, true>, grid, block, DEC_SMEM_F8, st, 0,
                          *a.map_k, *a.map_v, *a.map_k16, *a.map_v16, p)
      : keymajor ? launch_k(attn_decode_kernel<true, false>, grid, block, DEC_SMEM, st, 0,
                            *a.map_k, *a.map_v, *a.map_k16, *a.map_v16, p)
                 : launch_k(attn_decode_kernel<false, false>, grid, block, DEC_SMEM, st, 0,
                            *a.map_k, *a.map_v, *a.map_k16, *a.map_v16, p);
  if (e != cudaSuccess || splits == 1) return e;
  return launch_k(attn_combine_kernel, dim3(a.B * a.n_q), dim3(AD), 0, st, 0,
                  (const float*)a.partial, a.positions, a.n_q, splits, kps, p.key_limit, AD, a.out,
                  a.out_lo, a.cu_rows, p.v_scale);
}

int attn_decode_launches(int B, int n_kv, int max_keys, int sm_count, int dtype) {
  if (dtype == LLAMA_F32) return 1;
  int splits, kps;
  decode_plan(B, n_kv, max_keys, sm_count, splits, kps);
  return splits > 1 ? 2 : 1;
}

cudaError_t launch_attn_prefill(int dtype, const AttnPrefillArgs& a, cudaStream_t st) {
  if (dtype == LLAMA_F32) {
    const size_t sm = (size_t)(a.head_dim + a.T + 32) * sizeof(float);
    if (sm > 200 * 1024) return cudaErrorInvalidValue;
    if (sm > 48 * 1024)
      cudaFuncSetAttribute(attn_prefill_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)sm);
    return launch_k(attn_prefill_f32_kernel, dim3(a.T, a.n_q, a.B), dim3(128), sm, st, 0,
                    (const float*)a.q, (const float*)a.k, (const float*)a.v, (float*)a.out, a.T,
                    a.n_q, a.n_kv, a.head_dim);
  }
  return launch_attn_prefill_tc(a, st);
}

}  // namespace llgb
