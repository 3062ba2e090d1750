// Causal prefill attention on the 5th-generation tensor cores (tcgen05):
// scores q.k / sqrt(d), the causal mask, a numerically stable softmax and the
// weighted sum of V ("Llama2架构与推理全解析" §2.1 prefill, §2.3 attention; §1.5
// GQA: query head h reads K/V head h / G), computed FlashAttention-style so
// the T x T score matrix never leaves the SM.
//
// One CTA per (128 query rows, query head, sequence); 384 threads:
//   warp 0     TMA producer of the Q tile (and its bf16 remainder rows) and
//              of the K tiles (128 keys each) into a 3-slot mbarrier ring; a
//              slot frees as soon as S_j = Q K_j^T is computed;
//   warp 10    TMA producer of the V tiles into a 2-slot ring; a slot frees
//              once O += P_j V_j is computed;
//   warp 1     tensor-memory owner; one thread issues the score MMAs
//              S_j = Q K_j^T into one of two S buffers in tensor memory;
//   warp 11    one thread issues O += P_j V_j into the O accumulator in
//              tensor memory (two issuing threads, because issuing and the
//              barrier waits between MMA groups, not the tensor pipe, bound
//              a single thread at these small MMA shapes);
//   warps 2-9  softmax, two groups of four warps: a thread of group k owns
//              one query row (its tensor-memory lane) and keys 64k .. 64k+63
//              of every tile. It reads its half of S_j with tcgen05.ld,
//              masks, exchanges the row's tile maximum with its partner in the
//              other group through shared memory, keeps the running max and
//              its half of the sum, writes its half of P_j (bf16, as a hi/lo
//              pair when Q is one) into tensor memory, rescales O when needed
//              and at the end normalises and stores its 64 of the row's 128
//              output dims.
// Q is the score MMAs' A operand straight from its TMA tile in shared memory,
// and P the PV MMAs' A operand in tensor memory. That leaves tensor memory for
// three S buffers and the O accumulator. S has three buffers, and P_j is written over S_j (each thread
// replaces its own scores): the MMAs of S_{j+1} and S_{j+2} run while the
// softmax works on S_j, and S_{j+3} reuses buffer j % 3 once O += P_j V_j has
// completed. With 128-key tiles the score MMAs have N = 128, where one thread
// issues them faster than the tensor pipe executes them (at N = 64 issuing
// bounded them).
// The running max is applied lazily: O and the sum are rescaled only when a
// row's max grows by more than 2^8, otherwise P keeps the older max, which
// leaves the normalised result unchanged. Key tiles past the diagonal are
// skipped; the diagonal tile and the last partial tile are masked per key.
//
// Operand layouts:
//   Q  A operand in shared memory, K-major, 128-byte swizzled as TMA writes
//      it: [128 rows][64 dims] per dim half, the remainder tile Q_TILE
//      further;
//   K  B operand in shared memory, K-major, 128-byte swizzled as TMA writes
//      it: [128 keys][64 dims] per dim half;
//   P  A operand in tensor memory, in the S buffer of its tile: keys 64k ..
//      64k+63 at columns 64k .. 64k+31 (column c holds two consecutive keys),
//      their remainders at columns 64k+32 .. 64k+63;
//   V  B operand in shared memory, MN-major: [128 keys][64 dims] per dim half
//      (the dims are the MMA's N, contiguous in memory); 8-key groups 1024
//      bytes apart, the two dim halves KV_HALF bytes apart.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace llgb {

namespace {

constexpr int TQ = 128;          // query rows per CTA: MMA M, one tensor-memory lane each
constexpr int TK = 128;          // keys per tile
constexpr int TBOX = 64;         // rows of the Q/K/V boxes of the 64-row views
constexpr int TSUB = 16;         // keys per box of a 16-row (paged) cache view
constexpr int KSTAGES = 3;       // K tiles in flight
constexpr int VSTAGES = 2;       // V tiles in flight
constexpr int TC_THREADS = 384;  // Q/K producer, S issuer, two softmax warpgroups, V producer, PV issuer
constexpr int V_WARP = 10;
constexpr int PV_WARP = 11;
constexpr uint32_t KV_HALF = TK * 128;     // 128 keys x 64 dims bf16: 16 KB
constexpr uint32_t KV_TILE = 2 * KV_HALF;  // 128 keys x 128 dims: 32 KB (one K or V slot)
constexpr uint32_t Q_HALF = TQ * 128;      // 128 rows x 64 dims: 16 KB
constexpr uint32_t Q_TILE = 2 * Q_HALF;    // 32 KB; the remainder tile follows
constexpr uint32_t OFF_K = 2 * Q_TILE;
constexpr uint32_t OFF_V = OFF_K + KSTAGES * KV_TILE;
constexpr uint32_t OFF_BAR = OFF_V + VSTAGES * KV_TILE;
// exchange area of the two softmax groups: fp32 [2][2 groups][128 rows] (the
// tile maxima, double-buffered by tile parity; after the loop the final sums
// go to the buffer the last tile did not use) and int [2][2 groups][4
// quadrants] "this warp is on track" flags
constexpr uint32_t OFF_X = OFF_BAR + 256;
constexpr uint32_t OFF_XOK = OFF_X + 2 * 2 * 128 * 4;
constexpr size_t TC_SMEM = OFF_XOK + 2 * 2 * 4 * 4;  // the dynamic base is 1024-byte aligned (checked)
static_assert(TC_SMEM <= 232448, "227 KB of shared memory per CTA");
// tensor-memory columns: three S (then P) buffers of 128 columns, the O accumulator
constexpr int NSB = 3;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t O_COL = NSB * TK;
constexpr float kRescaleLog2 = 8.f;  // rescale O when a row max grows by more than 2^8

struct TcPreParams {
  bf16* out;
  size_t out_lo;
  uint32_t* status;
  int q_lo_rows;  // > 0: Q rows have bf16 remainders at row q_lo_rows + r; P is a pair too
  int T, n_q, n_kv, G, n_qtiles;
  float scale_log2, v_scale;
  const int32_t* cu_rows;
  const int32_t* start_pos;
  int n_rows;
  int from_cache, box_rows, layer, page_size, capacity, batch_cap, n_pages, max_pages;
  const int32_t* page_table;
};

// Shared-memory descriptor of an MN-major operand written by TMA with 128-byte
// swizzling: 64 contiguous MN elements per 128-byte row, 8-row (K) groups 1024
// bytes apart (stride byte offset), consecutive 64-element MN blocks `lbo`
// bytes apart (leading byte offset).
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)(1024u >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate):
// the A operand is read from tensor memory (row m = lane m).
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread, registers -> tensor memory.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


// The two softmax warps that own the same 32 rows (one per group) meet here.
// Both always pass the same sequence of these barriers: every decision to
// leave the tile loop is taken right after one, from flags both warps read.
__device__ __forceinline__ void pair_bar(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
}

// Cache row of the keys starting at k0 (a multiple of 16) of sequence b, K/V
// head g; a page id outside the pool is flagged and mapped to rows TMA fills
// with zeros.
__device__ __forceinline__ int tc_kv_row(const TcPreParams& p, int b, int g, int k0) {
  if (p.page_size == 0) return (b * p.n_kv + g) * p.capacity + k0;
  const int pi = k0 / p.page_size;
  const int page = pi < p.max_pages ? p.page_table[(size_t)b * p.max_pages + pi] : -1;
  if (page < 0 || page >= p.n_pages) {
    flag(p.status, LLAMA_FLAG_PAGE_RANGE);
    return -4 * TSUB;
  }
  return (page * p.n_kv + g) * p.page_size + (k0 % p.page_size);
}

// K or V tile of keys k0 .. k0 + nvalid - 1 into ring slot `dst`, completing
// on barrier fb: per 64-key block one 64-row box per dim half when the view
// has them and the block is full, else 16-key boxes for the keys the sequence
// has.
__device__ __forceinline__ void load_kv_tile(const TcPreParams& p, const CUtensorMap* m64,
                                             const CUtensorMap* m16, uint8_t* dst, uint64_t* fb,
                                             int b, int g, int rowbase, int k0, int nvalid) {
  if (!p.from_cache) {
    mbar_arrive_expect_tx(fb, KV_TILE);
    for (int rb = 0; rb < TK / TBOX; ++rb) {
      tma_load_3d(dst + rb * TBOX * 128, m64, fb, 0, g, rowbase + k0 + rb * TBOX);
      tma_load_3d(dst + KV_HALF + rb * TBOX * 128, m64, fb, 64, g, rowbase + k0 + rb * TBOX);
    }
    return;
  }
  uint32_t bytes = 0;
  for (int rb = 0; rb < TK / TBOX; ++rb) {
    const int nv = min(TBOX, nvalid - rb * TBOX);
    if (nv > 0)
      bytes += (p.box_rows == TBOX && nv == TBOX) ? 2 * TBOX * 128
                                                  : 2 * ((nv + TSUB - 1) / TSUB) * TSUB * 128;
  }
  mbar_arrive_expect_tx(fb, bytes);
  for (int rb = 0; rb < TK / TBOX; ++rb) {
    const int nv = min(TBOX, nvalid - rb * TBOX);
    uint8_t* d = dst + rb * TBOX * 128;
    if (nv <= 0) break;
    if (p.box_rows == TBOX && nv == TBOX) {
      const int row = tc_kv_row(p, b, g, k0 + rb * TBOX);
      tma_load_3d(d, m64, fb, 0, row, p.layer);
      tma_load_3d(d + KV_HALF, m64, fb, 64, row, p.layer);
    } else {
      for (int jj = 0; jj < (nv + TSUB - 1) / TSUB; ++jj) {
        const int row = tc_kv_row(p, b, g, k0 + rb * TBOX + jj * TSUB);
        tma_load_3d(d + jj * TSUB * 128, m16, fb, 0, row, p.layer);
        tma_load_3d(d + KV_HALF + jj * TSUB * 128, m16, fb, 64, row, p.layer);
      }
    }
  }
}

// A producer's ring: every tile's K (or V) into slot kt % NS once the
// consumer freed it; on an abort the copies in flight are waited for.
template <int NS>
__device__ __forceinline__ void produce_ring(const TcPreParams& p, const CUtensorMap* m64,
                                             const CUtensorMap* m16, uint8_t* slots, uint64_t* full,
                                             uint64_t* empty, volatile uint32_t* ctl, int n_kt,
                                             int n_keys, int b, int g, int rowbase) {
  int issued = 0;
  for (int kt = 0; kt < n_kt; ++kt) {
    const int s = kt % NS;
    if (ctl[1] || !mbar_wait_ready(&empty[s], ((kt / NS) & 1) ^ 1, p.status)) {
      ctl[1] = 1;
      for (int t = issued - 1; t >= 0 && t >= issued - NS; --t)
        mbar_wait_ready(&full[t % NS], (t / NS) & 1, p.status);
      return;
    }
    const int k0 = kt * TK;
    load_kv_tile(p, m64, m16, slots + s * KV_TILE, &full[s], b, g, rowbase, k0,
                 min(TK, n_keys - k0));
    ++issued;
  }
}

__global__ void __launch_bounds__(TC_THREADS, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap mapQ,
                           const __grid_constant__ CUtensorMap mapK,
                           const __grid_constant__ CUtensorMap mapV,
                           const __grid_constant__ CUtensorMap mapK16,
                           const __grid_constant__ CUtensorMap mapV16, TcPreParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need 1024-byte alignment
    if (threadIdx.x == 0) flag(p.status, LLAMA_FLAG_INDEX);
    grid_dep_wait();
    return;
  }
  uint64_t* qfull = reinterpret_cast<uint64_t*>(smem + OFF_BAR);  // Q tile in shared memory
  uint64_t* kfull = qfull + 1;
  uint64_t* kempty = kfull + KSTAGES;
  uint64_t* vfull = kempty + KSTAGES;
  uint64_t* vempty = vfull + VSTAGES;
  uint64_t* sfull = vempty + VSTAGES;  // [NSB] S_j is in tensor memory buffer j % NSB
  // [NSB] P_j is in tensor memory (O rescaled if needed). One per buffer: the
  // softmax may finish later tiles before the PV thread looks at tile j, but
  // not tile j + NSB (S_{j+NSB} waits for O += P_j V_j), so a buffer's
  // barrier is at most one phase ahead of its waiter and parity identifies it
  uint64_t* pready = sfull + NSB;
  uint64_t* odone = pready + NSB;      // [NSB] O += P_j V_j has completed (buffer j % NSB free)
  uint64_t* mfin = odone + NSB;        // [2] every S / PV MMA issued has completed (teardown)
  // ctl[0]: tensor-memory base address, ctl[1]: abort
  volatile uint32_t* ctl = reinterpret_cast<volatile uint32_t*>(mfin + 2);
  static_assert((1 + 2 * KSTAGES + 2 * VSTAGES + 3 * NSB + 2) * 8 + 8 <= OFF_X - OFF_BAR,
                "barrier block");
  const bool pair = p.q_lo_rows > 0;

  grid_dep_wait();  // q, k, v come from the RoPE/append kernel
  grid_dep_launch();
  const int qt = p.n_qtiles - 1 - (int)blockIdx.x;  // longest rows first
  const int h = blockIdx.y, b = blockIdx.z;
  const int g = h / p.G;
  const int q0 = qt * TQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rowbase = p.cu_rows ? p.cu_rows[b] : b * p.T;
  const int n_b = p.cu_rows ? p.cu_rows[b + 1] - rowbase : p.T;  // this sequence's rows
  const int start = p.start_pos ? p.start_pos[b] : 0;             // position of its first row
  if (q0 >= n_b) return;
  if (p.cu_rows && p.from_cache && n_b == 1) return;  // single new rows: the decode kernel's
  if (p.from_cache) {  // the sequence's keys must fit its cache slots
    const int cap_keys = p.page_size ? p.max_pages * p.page_size : p.capacity;
    if (start < 0 || start > cap_keys - n_b) {
      if (threadIdx.x == 0) flag(p.status, LLAMA_FLAG_POS_RANGE);
      return;
    }
  }
  const int n_keys = start + n_b;  // keys 0 .. n_keys - 1 exist once the rows are appended
  const int n_kt = (start + min(q0 + TQ, n_b) - 1) / TK + 1;

  if (threadIdx.x == 0) {
    mbar_init(qfull, 1);
    for (int s = 0; s < KSTAGES; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < VSTAGES; ++s) {
      mbar_init(&vfull[s], 1);
      mbar_init(&vempty[s], 1);
    }
    for (int i = 0; i < NSB; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&odone[i], 1);
      mbar_init(&pready[i], 8);
    }
    mbar_init(&mfin[0], 1);
    mbar_init(&mfin[1], 1);
    ctl[1] = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(const_cast<uint32_t*>(ctl), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl[0];

  if (warp == 0) {  // ----------------------------------------------- Q and K producer
    if (lane == 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      if (p.from_cache) tma_prefetch_desc(&mapK16);
      mbar_arrive_expect_tx(qfull, pair ? 2 * Q_TILE : Q_TILE);
      for (int t = 0; t < (pair ? 2 : 1); ++t) {
        const int row0 = (t ? p.q_lo_rows : 0) + rowbase + q0;
        for (int half = 0; half < 2; ++half)
          for (int rb = 0; rb < 2; ++rb)
            tma_load_3d(smem + t * Q_TILE + half * Q_HALF + rb * (Q_HALF / 2), &mapQ, qfull,
                        64 * half, h, row0 + 64 * rb);
      }
      produce_ring<KSTAGES>(p, &mapK, &mapK16, smem + OFF_K, kfull, kempty, ctl, n_kt, n_keys, b,
                            g, rowbase);
      mbar_wait_ready(qfull, 0, p.status);  // no copy may still be in flight when the CTA exits
    }
  } else if (warp == V_WARP) {  // --------------------------------------- V producer
    if (lane == 0) {
      tma_prefetch_desc(&mapV);
      if (p.from_cache) tma_prefetch_desc(&mapV16);
      produce_ring<VSTAGES>(p, &mapV, &mapV16, smem + OFF_V, vfull, vempty, ctl, n_kt, n_keys, b,
                            g, rowbase);
    }
  } else if (warp == 1 || warp == PV_WARP) {  // ---------------------------- MMA issuers
    if (lane == 0) {
      const bool is_s = warp == 1;
      const uint32_t id_s = idesc_bf16_f32(TQ, TK);
      const uint32_t id_o = idesc_bf16_f32(TQ, 128) | (1u << 16);  // B (V) MN-major
      // descriptors of K slot 0 and V slot 0; a slot, a dim half or a K step
      // moves the start-address field (address / 16) by a constant, so the
      // issue loop is a few adds per MMA (issuing bounds these small MMAs)
      const uint64_t kdesc0 = smem_desc_sw128(smem_u32(smem + OFF_K));
      const uint64_t vdesc0 = smem_desc_sw128_mn(smem_u32(smem + OFF_V), KV_HALF);
      // Q: the A operand of the score MMAs, read from its TMA tile (hi, then
      // the remainder tile Q_TILE further)
      const uint64_t qdesc0 = smem_desc_sw128(smem_u32(smem));
      bool ok = !is_s || mbar_wait_ready(qfull, 0, p.status);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int sb = j % NSB;
        if (is_s) {  // S_j = Q K_j^T, into the buffer P_{j-NSB} leaves
          const int s = j % KSTAGES;
          if (ctl[1] || !mbar_wait_ready(&kfull[s], (j / KSTAGES) & 1, p.status) ||
              (j >= NSB && !mbar_wait_ready(&odone[sb], ((j - NSB) / NSB) & 1, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t kd = kdesc0 + (uint64_t)(s * (KV_TILE >> 4));
          const uint32_t d = tmem + (uint32_t)sb * TK;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // 16 dims per MMA: 32 bytes of Q and of K rows
            tc_mma_f16(d, qdesc0 + ((kk >> 2) * Q_HALF + (kk & 3) * 32) / 16,
                       kd + ((kk >> 2) * KV_HALF + (kk & 3) * 32) / 16, id_s, kk > 0 ? 1u : 0u);
          if (pair)
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc_mma_f16(d, qdesc0 + (Q_TILE + (kk >> 2) * Q_HALF + (kk & 3) * 32) / 16,
                         kd + ((kk >> 2) * KV_HALF + (kk & 3) * 32) / 16, id_s, 1u);
          tc_commit(&sfull[sb]);
          tc_commit(&kempty[s]);
        } else {  // O += P_j V_j
          const int s = j % VSTAGES;
          if (ctl[1] || !mbar_wait_ready(&pready[sb], (j / NSB) & 1, p.status) ||
              !mbar_wait_ready(&vfull[s], (j / VSTAGES) & 1, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t vd = vdesc0 + (uint64_t)(s * (KV_TILE >> 4));
          const uint32_t pc = tmem + TK * (uint32_t)sb;
          const uint32_t oc = tmem + O_COL;
          // 16 keys per MMA: 8 P columns (keys 64g + 16m .. at 64g + 8m), two 8-key V groups
#pragma unroll
          for (int kk = 0; kk < TK / 16; ++kk)
            tc_mma_f16_ts(oc, pc + 64u * (kk >> 2) + 8u * (kk & 3), vd + kk * (2048 / 16), id_o,
                          (j > 0 || kk > 0) ? 1u : 0u);
          if (pair)
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk)
              tc_mma_f16_ts(oc, pc + 64u * (kk >> 2) + 32u + 8u * (kk & 3), vd + kk * (2048 / 16),
                            id_o, 1u);
          tc_commit(&odone[sb]);
          tc_commit(&vempty[s]);
        }
      }
      if (!ok) ctl[1] = 1;
      uint64_t* fin = &mfin[is_s ? 0 : 1];
      tc_commit(fin);
      mbar_wait_ready(fin, 0, p.status);  // this thread's MMAs retired before the tensor memory is freed
    }
  } else {  // --------------------------------------------------------- softmax warps
    const int quad = warp & 3;          // tensor-memory lane quadrant this warp may access
    const int grp = (warp - 2) >> 2;    // 0: keys 0-63 of a tile, O dims 0-63; 1: the rest
    const int r = quad * 32 + lane;
    const int qrow = q0 + r;
    const int qpos = start + qrow;
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem + OFF_X);                  // [2][2][128]
    volatile int* xok = reinterpret_cast<volatile int*>(smem + OFF_XOK);  // [2][2][4]
    const float c = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;  // m_used: the row's reference max, log2 units
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const bool good =
          __all_sync(0xffffffffu, ok && !ctl[1] && mbar_wait_ready(&sfull[j % NSB], (j / NSB) & 1, p.status));
      float sv[64];
      float pm = -INFINITY;
      const uint32_t sc = (uint32_t)(j % NSB) * TK + 64u * grp;  // this thread's S (then P) columns
      if (good) {
        tc_fence_after();
        uint32_t u[4][16];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld16(tl + sc + 16u * q, u[q]);
        tmem_ld_wait();
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 16; ++i) sv[16 * q + i] = __uint_as_float(u[q][i]);
        const int k0 = j * TK + 64 * grp;  // this thread's first key of the tile
        // a tile below the CTA's first row and inside the sequence needs no mask
        const bool full = j * TK + TK - 1 <= start + q0 && j * TK + TK <= n_keys;
        if (!full) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (k0 + i > qpos || k0 + i >= n_keys) sv[i] = -INFINITY;
        }
        float mx[4] = {sv[0], sv[1], sv[2], sv[3]};  // raw scores; the scale is positive
#pragma unroll
        for (int i = 4; i < 64; ++i) mx[i & 3] = fmaxf(mx[i & 3], sv[i]);
        pm = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      }
      const int xb = (j & 1) * 2;
      xch[(xb + grp) * 128 + r] = pm;
      if (lane == 0) xok[(xb + grp) * 4 + quad] = good ? 1 : 0;
      pair_bar(quad);
      if (!xok[xb * 4 + quad] || !xok[(xb + 1) * 4 + quad]) {  // both warps leave together
        ok = false;
        break;
      }
      const float mt = fmaxf(xch[xb * 128 + r], xch[(xb + 1) * 128 + r]) * c;  // row tile max, log2
      const float m_new = fmaxf(m_used, mt);
      const bool need = m_new > m_used + kRescaleLog2;  // also the first finite max
      const float f = m_used == -INFINITY ? 0.f : ex2(m_used - m_new);
      const bool rescale = __any_sync(0xffffffffu, need && j > 0);
      if (rescale) {
        // O must not be in flight: wait for O += P_{j-1} V_{j-1}. PV_{j-1-NSB}
        // completed before S_{j-1} was computed and PV_{j-1+NSB} needs a later
        // tile's P, so the barrier is on tile j - 1 - NSB or j - 1 and parity
        // identifies it
        if (!__all_sync(0xffffffffu, mbar_wait_ready(&odone[(j - 1) % NSB],
                                                     ((j - 1) / NSB) & 1, p.status))) {
          ok = false;  // the next tile's flags take both warps out of the loop
          ctl[1] = 1;
          continue;
        }
        tc_fence_after();
        const float fo = need ? f : 1.f;  // rescale this thread's 64 O dims
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t u[16];
          const uint32_t oc = O_COL + 64u * grp + 16u * q;
          tmem_ld16(tl + oc, u);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * fo);
          tmem_st16(tl + oc, u);
        }
      }
      if (need) {
        l *= f;
        m_used = m_new;
      }
      const int nvalid = min(TK, n_keys - j * TK);
      if (nvalid < TK) {
        // V rows past the last key may hold anything (P is 0 there, but
        // 0 * NaN is not): zero them, once V_j has landed, before the MMA
        // reads the tile (V_{j+2} cannot land in this slot before O += P_j V_j)
        if (!__all_sync(0xffffffffu, mbar_wait_ready(&vfull[j % VSTAGES], (j / VSTAGES) & 1, p.status))) {
          ok = false;
          ctl[1] = 1;
          continue;
        }
        uint8_t* vt = smem + OFF_V + (j % VSTAGES) * KV_TILE;
        const int nz = (TK - nvalid) * 16;
        for (int i = threadIdx.x - 64; i < nz; i += 256) {
          const int row = nvalid + (i >> 4), half = (i >> 3) & 1, chunk = i & 7;
          *reinterpret_cast<uint4*>(vt + half * KV_HALF + row * 128 + chunk * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // the MMA reads V through the async proxy
      }
      // e = 2^(s c - m) and this thread's 64 keys of P row r over its scores
      // (keys at columns sc .. sc+31, the remainders at sc+32 .. sc+63; all
      // scores are in registers), one 32-key half at a time so the packing
      // and stores of one half overlap the exponentials of the other
      const float mu = m_used == -INFINITY ? 0.f : m_used;
      float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
        for (int i = 32 * hh; i < 32 * hh + 32; ++i) {
          const float e = ex2(fmaf(sv[i], c, -mu));  // masked keys: -inf -> 0
          sv[i] = e;
          ls[i & 3] += e;
        }
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) split_pack(sv[32 * hh + 2 * i], sv[32 * hh + 2 * i + 1], ph[i], pl[i]);
        tmem_st16(tl + sc + 16u * hh, ph);
        if (pair) tmem_st16(tl + sc + 32u + 16u * hh, pl);
      }
      l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pready[j % NSB]);
    }
    // ---- epilogue: this thread's 64 dims of O / l (l = both groups' halves)
    const int last = n_kt - 1;
    const bool done =
        ok && !ctl[1] && mbar_wait_ready(&odone[last % NSB], (last / NSB) & 1, p.status);
    const int xs = (n_kt & 1) * 2;  // the exchange buffer the last tile did not use
    xch[(xs + grp) * 128 + r] = l;
    pair_bar(quad);
    if (done && !ctl[1]) {
      tc_fence_after();
      const float lt = xch[xs * 128 + r] + xch[(xs + 1) * 128 + r];
      const float inv = lt > 0.f ? p.v_scale / lt : 0.f;
      const bool row_ok = qrow < n_b && rowbase + qrow < p.n_rows;
      bf16* dst = p.out + (size_t)(rowbase + qrow) * p.n_q * 128 + (size_t)h * 128 + 64 * grp;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t u[16];
        tmem_ld16(tl + O_COL + 64u * grp + 16u * q, u);
        tmem_ld_wait();
        uint32_t hi[8], lo[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          split_pack(__uint_as_float(u[2 * i]) * inv, __uint_as_float(u[2 * i + 1]) * inv, hi[i],
                     lo[i]);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + 16 * q);
          d4[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
          d4[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
          if (p.out_lo) {
            uint4* l4 = reinterpret_cast<uint4*>(dst + 16 * q + p.out_lo);
            l4[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            l4[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
          }
        }
      }
    } else {
      ctl[1] = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

cudaError_t attn_prefill_tc_prepare() {
  return cudaFuncSetAttribute(attn_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)TC_SMEM);
}

cudaError_t launch_attn_prefill_tc(const AttnPrefillArgs& a, cudaStream_t st) {
  if (a.head_dim != 128) return cudaErrorInvalidValue;
  if (a.from_cache && (!a.map_k16 || !a.map_v16)) return cudaErrorInvalidValue;
  TcPreParams p;
  p.out = (bf16*)a.out;
  p.out_lo = a.out_lo;
  p.status = a.status;
  p.q_lo_rows = a.q_lo_rows;
  p.T = a.T;
  p.n_q = a.n_q;
  p.n_kv = a.n_kv;
  p.G = a.n_q / a.n_kv;
  p.n_qtiles = (a.T + TQ - 1) / TQ;
  p.scale_log2 = 1.4426950408889634f / sqrtf(128.f) * a.k_scale;
  p.v_scale = a.v_scale;
  p.cu_rows = a.cu_rows;
  p.start_pos = a.start_pos;
  p.n_rows = a.cu_rows ? a.n_rows : a.B * a.T;
  p.from_cache = a.from_cache;
  p.box_rows = a.box_rows == TBOX ? TBOX : TSUB;
  p.layer = a.layer;
  p.page_size = a.page_size;
  p.capacity = a.capacity;
  p.batch_cap = a.batch_cap;
  p.n_pages = a.n_pages;
  p.max_pages = a.max_pages;
  p.page_table = a.page_table;
  const CUtensorMap* k16 = a.from_cache ? a.map_k16 : a.map_k;
  const CUtensorMap* v16 = a.from_cache ? a.map_v16 : a.map_v;
  return launch_k(attn_prefill_tc_kernel, dim3(p.n_qtiles, a.n_q, a.B), dim3(TC_THREADS), TC_SMEM,
                  st, 0, *a.map_q, *a.map_k, *a.map_v, *k16, *v16, p);
}

}  // namespace llgb
