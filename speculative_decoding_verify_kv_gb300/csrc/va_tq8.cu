// Tensor-core split-KV partial kernel for Q8_0 caches, sm_103a (tcgen05 +
// TMEM + bulk copies), in transposed form.
//
// One CTA owns (sequence, KV head, KV chunk, block of at most 96 query rows
// of that KV head) and reads every K/V byte of its chunk once for all of
// those rows (hipfire PR #695, alpineQ comments: one block reuses each Q8
// K/V fetch across several verifier rows).  Per 128-token tile:
//
//   S^T = K Q^T      tcgen05.mma, M = 128 tokens, N = query rows, K = D.
//                    A = the K tile in TMEM, B = Q^T in shared memory.
//   softmax          one thread per token: scores in log2 units against a
//                    per-row running maximum that moves only when a score
//                    passes it by more than 2^kSlack (then O^T and the row sums
//                    are rescaled); masks (context visible to every row,
//                    chain rows causal by index, tree rows by ancestor
//                    mask); P = 2^(s c - m) into shared memory as fp16 P^T;
//                    fp32 row sums per thread.
//   O^T += V^T P^T   tcgen05.mma, M = 128 values of d, N = query rows,
//                    K = 16 tokens per step; A = the V tile (MN-major),
//                    B = P^T (MN-major), both in shared memory.
//
// Tokens sit on the MMA's M axis and query rows on N, so a KV head's 96
// rows (16 draft rows x 6 query heads) fill N without padding to 128, and
// O^T's lanes are values of d, so the partial rows leave TMEM as coalesced
// stores.  At the end each row's (m, l, O) goes to its partial slot; the
// merge kernel combines the slots (hipfire PR #817 "FA2 split-KV",
// sections "Summary" and "Performance").
//
// Q8_0 arithmetic.  A K element d*q (fp16 scale d, int8 code q) has up to
// 18 significant bits, more than fp16's 11.  It enters the MMA as two fp16
// parts: hi = fp16(d*q) and lo = fma(d, q, -hi), the rounding residual,
// which fp16 holds exactly (its lowest bit is that of d*q), so hi + lo ==
// d*q exactly whenever |d*q| < 65504.  S^T takes one MMA per part and K
// step; Q (bf16) is exact in fp16 after a per-row power-of-two rescale,
// folded back into the score multiplier c.  V elements are fp16(d*q) (one
// rounding) and P is fp16, as the P.V product's precision allows.
//
// Warp roles (16 warps, four warpgroups with their own register budgets):
//   3 V producer (raw V rows into shared memory by 1-D bulk copies; L2
//     prefetch of K and V tiles ahead), 1 TMEM owner + S^T issuer, 2 P.V
//     issuer, 0 idle after the prologue;
//   4..7 softmax (warp & 3 = TMEM lane quadrant = 32 tokens, every row),
//     also the O^T rescale and the epilogue;
//   8..11 K dequantisation (one token row per thread, read from L2, into
//     TMEM);
//   12..15 V dequantisation (one token row per thread, into shared memory);
//   4..15 stage Q^T in the prologue.
// Every wait is bounded (VA_DEV_TIMEOUT); after a timeout the CTA drains
// its copies and MMAs, frees TMEM and writes NaN partials.
#include <string.h>

#include "va_common.cuh"
#include "va_sm100.cuh"

namespace va {
using namespace sm100;

namespace tq8 {

constexpr int kTT = 128;      // tokens per tile (the MMA's M)
constexpr int kNR = 96;       // query rows per CTA at most (the MMA's N)
constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kLaunchRegs = 128;  // 65536 registers / 512 threads
constexpr int kPrefetch = 4;     // L2 prefetch distance in tiles
constexpr uint64_t kWaitNs = 2000000000ull;
// A row's running maximum m (log2 units) moves only when one of its scores
// passes m + kSlack: P = 2^(s c - m) stays below 2^kSlack, well inside
// fp16 (P^T) and fp32 (row sums, O^T).
constexpr float kSlack = 14.f;

// TMEM columns (512 allocated): O^T half h (d in [128h, 128h + 128)) at
// COL_O + h*kNR; S^T buffer b at COL_S + b*kNR; K slot k at COL_K + 64k
// (hi parts in its first 32 columns, lo parts in the next 32).
constexpr int COL_O = 0;
constexpr int COL_S = 2 * kNR;
constexpr int COL_K = 4 * kNR;
constexpr int TMEM_COLS = 512;
static_assert(COL_K + 128 <= TMEM_COLS, "TMEM map");

// Warp roles.
constexpr int W_PROD = 0, W_SMMA = 1, W_PV = 2, W_PRODV = 3;
constexpr int W_SM0 = 4;    // softmax warps 4..7
constexpr int W_KDQ0 = 8;   // K dequantisation warps 8..11
constexpr int W_VDQ0 = 12;  // V dequantisation warps 12..15
constexpr int kRoleWarps = 4;  // warps per softmax / dequantisation role (one per quadrant)
// Per-thread register budgets of the four warpgroups; their sum stays within
// the registers the block is launched with (4 x kLaunchRegs), so the
// softmax warpgroup's setmaxnreg.inc is covered by the other warpgroups'
// decrements.
constexpr int REG_CTRL = 72, REG_SM = 256, REG_KDQ = 120, REG_VDQ = 56;
static_assert(REG_CTRL + REG_SM + REG_KDQ + REG_VDQ <= 4 * kLaunchRegs, "register split");

template <int D>
struct Cfg {
  static constexpr int NB = D / 32;                 // Q8 blocks per row
  static constexpr int RB = NB * 34;                // raw bytes per token row
  static constexpr int NW = RB / 4;                 // raw words per token row
  static constexpr int DV = D < 128 ? 128 : D;      // V / O^T extent along d
  static constexpr int DH = DV / 128;               // O^T halves
  static constexpr int NFILL = D / 64;              // K slot fills (64 d each) per tile
  static constexpr int NRAW = D == 256 ? 1 : 2;     // raw V row buffers
  static constexpr int NVB = D == 256 ? 1 : 2;      // fp16 V tile buffers
  static constexpr int QT_BLK = kNR * 128;          // one 64-d column block of Q^T
  static constexpr int QT_BYTES = (D / 64) * QT_BLK;
  static constexpr int PT_BLK = kTT * 128;          // one 64-row block of P^T
  static constexpr int PT_BYTES = 2 * PT_BLK;       // one P^T buffer (rows 0..127)
  static constexpr int NPB = 2;                     // P^T buffers
  static constexpr int VT_BLK = kTT * 128;          // one 64-d column block of a V tile
  static constexpr int VT_BYTES = (DV / 64) * VT_BLK;
  static constexpr int RAW_BYTES = (kTT * RB + 127) / 128 * 128;
  static constexpr int OFF_QT = 0;
  static constexpr int OFF_PT = OFF_QT + QT_BYTES;
  static constexpr int OFF_VT = OFF_PT + NPB * PT_BYTES;
  static constexpr int OFF_RV = OFF_VT + NVB * VT_BYTES;
  static constexpr int SMEM = OFF_RV + NRAW * RAW_BYTES + 1024;
};

enum {
  B_RVF = 0,    // [2] raw V rows of the buffer's tile landed
  B_RVE = 2,    // [2] raw V buffer read by the V dequantisation warps
  B_KSF = 4,    // [2] K slot written (TMEM)
  B_KSE = 6,    // [2] the S^T MMAs reading a K slot completed
  B_STF = 8,    // [2] S^T of the buffer's tile complete
  B_STE = 10,   // [2] S^T buffer read by the softmax
  B_PF = 12,    // [2] P^T buffer written
  B_PE = 14,    // [2] the P.V MMAs reading a P^T buffer completed
  B_VF = 16,    // [2] fp16 V tile written
  B_VE = 18,    // [2] V tile free again
  B_OF = 20,    // the last P.V completed
  B_DRAIN = 21, // [2] S^T issuer, P.V issuer
  B_COUNT = 23
};

// Byte offset of 16-byte chunk `chunk` (< 8) of row `row` inside a
// 128-byte-swizzled block whose rows are 128 bytes apart.
__device__ __forceinline__ uint32_t sw128(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Load a raw Q8_0 row (RB bytes) into words, with the widest loads its
// alignment allows (rows are RB bytes apart from a 16-byte-aligned base).
template <int D>
__device__ __forceinline__ void load_row(uint32_t (&w)[Cfg<D>::NW], const unsigned char* src) {
  constexpr int RB = Cfg<D>::RB;
  if (RB % 16 == 0) {
#pragma unroll
    for (int k = 0; k < RB / 16; ++k) {
      const uint4 v = reinterpret_cast<const uint4*>(src)[k];
      w[4 * k] = v.x;
      w[4 * k + 1] = v.y;
      w[4 * k + 2] = v.z;
      w[4 * k + 3] = v.w;
    }
  } else if (RB % 8 == 0) {
#pragma unroll
    for (int k = 0; k < RB / 8; ++k) {
      const uint2 v = reinterpret_cast<const uint2*>(src)[k];
      w[2 * k] = v.x;
      w[2 * k + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int k = 0; k < RB / 4; ++k) w[k] = reinterpret_cast<const uint32_t*>(src)[k];
  }
}

// Scale and the eight 4-code words of Q8_0 block b of a row held in words.
// The block starts at byte 34 b: an odd block starts two bytes into a word.
__device__ __forceinline__ void q8_block(const uint32_t* w, int b, __half2& d2, uint32_t (&code)[8]) {
  const int o = 34 * b;
  const int wo = o >> 2;
  uint32_t sbits;
  if (o & 2) {
    sbits = w[wo] >> 16;
#pragma unroll
    for (int q = 0; q < 8; ++q) code[q] = w[wo + 1 + q];
  } else {
    sbits = w[wo] & 0xFFFFu;
#pragma unroll
    for (int q = 0; q < 8; ++q) code[q] = __funnelshift_r(w[wo + q], w[wo + q + 1], 16);
  }
  d2 = __half2half2(__ushort_as_half((unsigned short)sbits));
}

// Four int8 codes -> two fp16 pairs holding the codes exactly: each byte
// b + 128 becomes the fp16 value 1024 + (b + 128) (exponent byte 0x64),
// minus 1152.
__device__ __forceinline__ void codes_to_h2(uint32_t code, __half2& a, __half2& b) {
  const uint32_t x = code ^ 0x80808080u;
  uint32_t lo = __byte_perm(x, 0x64646464u, 0x4140);
  uint32_t hi = __byte_perm(x, 0x64646464u, 0x4342);
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));
  a = __hsub2(*reinterpret_cast<__half2*>(&lo), bias);
  b = __hsub2(*reinterpret_cast<__half2*>(&hi), bias);
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Move this warpgroup's per-thread register limit from the launch count to N.
template <int N>
__device__ __forceinline__ void set_regs() {
  if constexpr (N > kLaunchRegs) setmaxnreg_inc<N>();
  else if constexpr (N < kLaunchRegs) setmaxnreg_dec<N>();
}

}  // namespace tq8

template <int D, bool PAGED>
__global__ void __launch_bounds__(tq8::kThreads, 1)
    tq8_partial_kernel(const Params p) {
  using namespace tq8;
  using C = Cfg<D>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int err_s;
  // Per-row state of the online softmax (row r of the CTA = sequence-local
  // query row rb*kNR + r).  cm_s holds (c, m_eff): the score multiplier and
  // the maximum P is taken against (+inf for a row with no visible token
  // yet, so its P is 0); m_s the running maximum itself (log2 units, -inf
  // before the first visible token); thr_s the raw score above which the
  // maximum moves; f_s the rescale factor of the current tile.  Padded rows
  // have c = 0 and m_eff = thr = +inf.
  __shared__ __align__(16) float2 cm_s[kNR];
  __shared__ __align__(16) float m_s[kNR];
  __shared__ __align__(16) float thr_s[kNR];
  __shared__ float rc_s[kNR];            // 1 / c (0 for padded rows)
  __shared__ __align__(16) float f_s[kNR];
  __shared__ long long slot_s[kNR];      // partial slot index of each row
  __shared__ int jr_s[kNR];              // local row index (in the sequence) of each row
  __shared__ unsigned anc_s[kNR];        // ancestor mask of each row
  __shared__ unsigned flag_s[2][4];      // [tile parity][softmax warp]: a row passed its trigger

  // The merge kernel may launch now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;");
  // Launched as a programmatic dependent of the previous work on the
  // stream: nothing is read or written before that work has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, s = blockIdx.z;

  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  if (err & VA_DEV_BAD_ROWS) {
    if (tid == 0) flag(p.status, err);
    return;
  }
  int rb, slot, nsub;  // row block, chunk, the sequence's chunk count
  if (!cta_work(p, n, blockIdx.x, &rb, &slot, &nsub)) return;
  const int G = p.G;
  const int R = n * G;
  if (rb * kNR >= R) return;
  const int Rb = min(kNR, R - rb * kNR);   // valid rows of this CTA
  const int NR = (Rb + 15) / 16 * 16;      // MMA N
  const int L = ctx + n;
  int lo, hi, slo, shi;
  split_range(L, p.S, 0, &lo, &hi);
  sub_range(lo, hi, nsub, p.min_sub, slot, &slo, &shi);
  const int ntiles = (shi - slo + kTT - 1) / kTT;
  if (ntiles == 0 && !err) {
    // An empty chunk (short span): its rows' slots become (-inf, 0) at once,
    // without the prologue.  The sequence's other CTAs check its parents.
    if (tid < Rb) {
      const int rs = rb * kNR + tid;
      const long long si0 = slot_index(p, slot, row0 + rs / G, kvh * G + rs % G);
      p.ws_ml[2 * si0] = -INFINITY;
      p.ws_ml[2 * si0 + 1] = 0.f;
    }
    return;
  }
  const int kind = seq_kind_of(p, s);
  // Tree sequence with a tree scratch KV: its draft positions (>= ctx) are
  // read from the scratch rows by the dequantising threads, and the cache
  // covers the context only.
  const bool scratch = uses_scratch(p, kind);
  const int cend = scratch ? min(shi, ctx) : shi;  // cache tokens of the chunk end here

  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  unsigned char* const qt = sm + C::OFF_QT;
  auto ptb = [&](int b) { return sm + C::OFF_PT + b * C::PT_BYTES; };
  auto vt = [&](int b) { return sm + C::OFF_VT + b * C::VT_BYTES; };
  auto rawv = [&](int b) { return sm + C::OFF_RV + b * C::RAW_BYTES; };

  // Raw-row copies of tile i of tensor kv (0 = K, 1 = V): the cache tokens
  // [t0, end16) in whole 16-token groups, one bulk copy (contiguous) or one
  // per 16-token page (paged).  A tile with no cache tokens completes its
  // barrier phase at once.
  auto tile_span = [&](int i, int* t0, int* nload) {
    *t0 = slo + i * kTT;
    const int end16 = min(*t0 + kTT, (cend + kPage - 1) / kPage * kPage);
    *nload = max(0, end16 - *t0);
  };
  // Block ids of a tile's pages, all loads in flight together.
  auto tile_blocks = [&](int t0, int npg, int (&blk)[kTT / kPage]) {
#pragma unroll
    for (int pg = 0; pg < kTT / kPage; ++pg)
      blk[pg] = pg < npg ? p.block_table[(long long)s * p.max_blocks + t0 / kPage + pg] : 0;
  };
  auto prefetch = [&](int i, int kv) {
    if (i >= ntiles) return;
    int t0, nload;
    tile_span(i, &t0, &nload);
    if (nload <= 0) return;
    const unsigned char* src = (const unsigned char*)(kv ? p.v : p.k);
    if (!PAGED) {
      const long long row = ((long long)s * p.KVH + kvh) * p.capacity + t0;
      bulk_prefetch_l2(src + row * C::RB, (uint32_t)(nload * C::RB));
    } else {
      int blk[kTT / kPage];
      tile_blocks(t0, nload / kPage, blk);
#pragma unroll
      for (int pg = 0; pg < kTT / kPage; ++pg)
        if (pg < nload / kPage)
          bulk_prefetch_l2(src + ((long long)blk[pg] * p.KVH + kvh) * kPage * C::RB,
                           kPage * C::RB);
    }
  };
  auto issue_v = [&](int i, uint64_t pol) {
    int t0, nload;
    tile_span(i, &t0, &nload);
    const int b = i % C::NRAW;
    unsigned char* dst = rawv(b);
    const uint32_t fb = bar(B_RVF + b);
    const unsigned char* src = (const unsigned char*)p.v;
    int blk[kTT / kPage];
    if (PAGED) tile_blocks(t0, nload / kPage, blk);
    mbar_arrive_expect_tx(fb, (uint32_t)(nload * C::RB));
    if (nload > 0) {
      if (!PAGED) {
        const long long row = ((long long)s * p.KVH + kvh) * p.capacity + t0;
        bulk_g2s(smem_u32(dst), src + row * C::RB, (uint32_t)(nload * C::RB), fb, pol);
      } else {
#pragma unroll
        for (int pg = 0; pg < kTT / kPage; ++pg)
          if (pg < nload / kPage)
            bulk_g2s(smem_u32(dst + pg * kPage * C::RB),
                     src + ((long long)blk[pg] * p.KVH + kvh) * kPage * C::RB, kPage * C::RB,
                     fb, pol);
      }
    }
  };

  // Contiguous cache without a detected error: tile 0's copies go out now
  // (every address is in range: the span was checked against the capacity).
  const bool early = !PAGED && !err && ntiles > 0;
  if (tid == 0) {
    err_s = 0;
    abort_s = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_RVF + b), 1);
      mbar_init(bar(B_RVE + b), kRoleWarps);
      mbar_init(bar(B_KSF + b), kRoleWarps);
      mbar_init(bar(B_KSE + b), 1);
      mbar_init(bar(B_STF + b), 1);
      mbar_init(bar(B_STE + b), kRoleWarps);
      mbar_init(bar(B_VF + b), kRoleWarps);
      mbar_init(bar(B_PF + b), kRoleWarps);
      mbar_init(bar(B_PE + b), 1);
      mbar_init(bar(B_VE + b), 1);
      mbar_init(bar(B_DRAIN + b), 1);
    }
    mbar_init(bar(B_OF), 1);
    fence_barrier_init();
    if (early) {
      // K rows go straight from L2 to the K dequantisation warps: bring
      // the first tiles of K into L2 and V tile 0 into shared memory.
      const uint64_t pol = policy_evict_first();
      for (int i = 0; i <= kPrefetch; ++i) prefetch(i, 0);
      issue_v(0, pol);
      for (int i = 1; i <= kPrefetch; ++i) prefetch(i, 1);
    }
  }

  // Warps 4..15: Q^T into shared memory (fp16, each row rescaled by a power
  // of two so that its largest |q| lies in [0.5, 1); the factor goes into
  // the score multiplier c), the row tables, and the initial running maxima.
  // Rows past this CTA's valid rows are zero.
  if (warp >= W_SM0) {
    constexpr int NSW = kWarps - W_SM0;  // staging warps
    const int ws = warp - W_SM0;
    constexpr int CPR = D / 8;           // 16-byte chunks per Q row
    constexpr int RPI = 32 / CPR;        // rows per warp per step
    constexpr int NIT = (kNR + NSW * RPI - 1) / (NSW * RPI);
    const int chunk = lane % CPR, sub = lane / CPR;
    uint4 v[NIT];
#pragma unroll
    for (int k = 0; k < NIT; ++k) {
      const int r = RPI * (ws + NSW * k) + sub;
      v[k] = make_uint4(0u, 0u, 0u, 0u);
      if (r < Rb) {
        const int rs = rb * kNR + r;
        const long long qi = ((long long)(row0 + rs / G) * p.H + kvh * G + rs % G) * D;
        v[k] = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(p.q) + qi)[chunk];
      }
    }
#pragma unroll
    for (int k = 0; k < NIT; ++k) {
      const int r = RPI * (ws + NSW * k) + sub;
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
      float amax = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        amax = fmaxf(amax, fabsf(__uint_as_float(w[m] << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(w[m] & 0xFFFF0000u)));
      }
#pragma unroll
      for (int off = CPR / 2; off > 0; off >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      int e = 0;
      if (amax > 0.f) frexpf(amax, &e);
      const float qscale = ldexpf(1.f, -e);
      uint32_t h[4];
#pragma unroll
      for (int m = 0; m < 4; ++m)
        h[m] = h2u(__floats2half2_rn(__uint_as_float(w[m] << 16) * qscale,
                                     __uint_as_float(w[m] & 0xFFFF0000u) * qscale));
      if (r < kNR) {
        *reinterpret_cast<uint4*>(qt + (chunk / 8) * C::QT_BLK + sw128(r, chunk % 8)) =
            make_uint4(h[0], h[1], h[2], h[3]);
        if (chunk == 0) {
          const float c = ldexpf(p.scale_log2, e);
          cm_s[r] = r < Rb ? make_float2(c, INFINITY) : make_float2(0.f, INFINITY);
          rc_s[r] = r < Rb ? 1.f / c : 0.f;
        }
      }
    }
    // Row tables (row r of the CTA = sequence-local query row rb*kNR + r).
    const int tsm = tid - W_SM0 * 32;
    if (tsm < kNR) {
      const int r = tsm;
      int j = -1;
      unsigned anc = 0u;
      if (r < Rb && !err) {
        j = (rb * kNR + r) / G;
        bool bad = false;
        anc = row_mask(kind, p.parent + row0, j, &bad);
        if (bad) atomicOr(&err_s, (int)VA_DEV_BAD_PARENT);
      }
      jr_s[r] = j;
      anc_s[r] = anc;
      m_s[r] = -INFINITY;
      thr_s[r] = r < Rb ? -INFINITY : INFINITY;
      f_s[r] = 1.f;
      long long si = 0;
      if (r < Rb) {
        const int rs = rb * kNR + r;
        si = slot_index(p, slot, row0 + rs / G, kvh * G + rs % G);
      }
      slot_s[r] = si;
    }
  }
  // D = 64: the V tiles' second 64-d block stays zero (O^T's lanes 64..127).
  if (D < 128 && warp >= W_VDQ0) {
    for (int b = 0; b < C::NVB; ++b)
      for (int k = tid - W_VDQ0 * 32; k < C::VT_BLK / 16; k += 128)
        reinterpret_cast<uint4*>(vt(b) + C::VT_BLK)[k] = make_uint4(0u, 0u, 0u, 0u);
  }
  // Paged cache: every block-table entry the chunk reads must be in range.
  if (PAGED && !err && ntiles > 0) {
    const int pg0 = slo / kPage, pg1 = (cend + kPage - 1) / kPage;
    for (int pg = pg0 + tid; pg < pg1; pg += kThreads) {
      const int blk = p.block_table[(long long)s * p.max_blocks + pg];
      if (blk < 0 || blk >= p.num_blocks) atomicOr(&err_s, (int)VA_DEV_BAD_BLOCK);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();
  err |= (unsigned)err_s;

  if (err || ntiles == 0) {
    if (early && tid == 0) {
      // Let the copies already issued land before the CTA goes away.
      int dummy = 0;
      volatile int* never = &dummy;
      mbar_wait(bar(B_RVF), 0, never, kWaitNs);
    }
    if (err && tid == 0) flag(p.status, err);
    if (tid < Rb) {
      const int rs = rb * kNR + tid;
      const long long si = slot_index(p, slot, row0 + rs / G, kvh * G + rs % G);
      p.ws_ml[2 * si] = err ? NAN : -INFINITY;
      p.ws_ml[2 * si + 1] = err ? NAN : 0.f;
    }
    return;
  }

  if (warp == W_SMMA) {
    tmem_alloc(smem_u32(&tmem_base_s), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tmem_base_s;
  volatile int* abort_p = &abort_s;
  auto fail = [&]() {
    *abort_p = 1;
    flag(p.status, VA_DEV_TIMEOUT);
  };
  int dummy_never = 0;
  volatile int* never = &dummy_never;

  // Role dispatch.  Each warpgroup first sets its register budget (every
  // warp of a warpgroup executes the same setmaxnreg).
  if (warp < W_SM0) {
   set_regs<REG_CTRL>();
   if (warp == W_PRODV) {
    // ------------------------------------------------------------ producer
    // The V tiles into the raw buffer once the V dequantisation warps have
    // read the buffer's last tile; K and V kPrefetch tiles ahead in L2 (the
    // K dequantisation warps read K rows from L2 themselves).
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = early ? 1 : 0;
      bool ok = true;
      if (!early)
        for (int i = 0; i <= kPrefetch; ++i) prefetch(i, 0);
      for (int i = issued; i < ntiles && ok; ++i) {
        const int b = i % C::NRAW;
        ok = mbar_wait(bar(B_RVE + b), ((i / C::NRAW) & 1) ^ 1, abort_p, kWaitNs);
        if (!ok) break;
        issue_v(i, pol);
        issued = i + 1;
        for (int j = (i == 0 ? 1 : i + kPrefetch); j <= i + kPrefetch; ++j) {
          if (i > 0) prefetch(j, 0);
          prefetch(j, 1);
        }
      }
      if (!ok) fail();
      if (*abort_p) {
        // Make sure no copy of ours is still landing in shared memory.
        for (int i = max(0, issued - C::NRAW); i < issued; ++i)
          mbar_wait(bar(B_RVF + i % C::NRAW), (i / C::NRAW) & 1, never, kWaitNs);
      }
    }
   } else if (warp == W_SMMA) {
    // ------------------------------------------------------------ S^T issuer
    // S^T(i) into buffer i & 1 once the softmax has read that buffer's
    // previous tile: per K slot fill (64 values of d), four K steps of 16,
    // each an MMA of the hi part and one of the lo part.
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(kTT, NR, false, false);
      const uint32_t qt_a = smem_u32(qt);
      bool ok = true, any = false;
      int g = 0;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int b = i & 1;
        ok = mbar_wait(bar(B_STE + b), ((i >> 1) & 1) ^ 1, abort_p, kWaitNs);
        for (int f = 0; f < C::NFILL && ok; ++f, ++g) {
          const int ks = g & 1;
          ok = mbar_wait(bar(B_KSF + ks), (g >> 1) & 1, abort_p, kWaitNs);
          if (!ok) break;
          tc_fence_after();
          const uint32_t dcol = tm + COL_S + b * kNR;
          const uint32_t a_hi = tm + COL_K + ks * 64, a_lo = a_hi + 32;
          const uint64_t bd0 = sdesc_sw128(qt_a + f * C::QT_BLK, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = bd0 + (uint64_t)((kk * 32) >> 4);
            mma_ts(dcol, a_hi + kk * 8, bd, idesc, (f | kk) ? 1u : 0u);
            mma_ts(dcol, a_lo + kk * 8, bd, idesc, 1u);
          }
          any = true;
          mma_commit(bar(B_KSE + ks));
        }
        if (ok) mma_commit(bar(B_STF + b));
      }
      if (!ok) fail();
      if (any) {
        mma_commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, never, kWaitNs);
      }
    }
   } else if (warp == W_PV) {
    // ------------------------------------------------------------ P.V issuer
    // O^T += V^T P^T once the softmax has written P^T(i) (and rescaled O^T
    // if its maxima moved) and the V tile is ready; per half of d, eight K
    // steps of 16 tokens.  Completion frees P^T and the V buffer.
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, NR, false, true, true);
      bool ok = true, any = false;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int vb = i % C::NVB;
        const int pb = i & 1;
        ok = mbar_wait(bar(B_PF + pb), (i >> 1) & 1, abort_p, kWaitNs) &&
             mbar_wait(bar(B_VF + vb), (i / C::NVB) & 1, abort_p, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        const uint32_t vt_a = smem_u32(vt(vb));
        const uint64_t bd0 = sdesc_sw128(smem_u32(ptb(pb)), C::PT_BLK, 1024);
#pragma unroll
        for (int h = 0; h < C::DH; ++h) {
          const uint64_t ad0 = sdesc_sw128(vt_a + 2 * h * C::VT_BLK, C::VT_BLK, 1024);
#pragma unroll
          for (int kk = 0; kk < kTT / 16; ++kk) {
            const uint64_t step = (uint64_t)((kk * 2048) >> 4);
            mma_ss(tm + COL_O + h * kNR, ad0 + step, bd0 + step, idesc,
                   (i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        any = true;
        mma_commit(bar(B_PE + pb));
        mma_commit(bar(B_VE + vb));
      }
      if (ok) mma_commit(bar(B_OF));
      if (!ok) fail();
      if (any) {
        mma_commit(bar(B_DRAIN + 1));
        mbar_wait(bar(B_DRAIN + 1), 0, never, kWaitNs);
      }
    }
   }
  } else if (warp < W_KDQ0) {
    // ------------------------------------------------------------ softmax
    // Warp w & 3 = TMEM lane quadrant: this thread's token of each tile and,
    // for O^T, 32 values of d in each half.  Every thread covers all rows;
    // S^T comes into registers once per tile.
    set_regs<REG_SM>();
    const int quad = warp & 3;
    const int t = quad * 32 + lane;          // token of the tile; row owner in the epilogue
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    constexpr int NCH = kNR / 16;
    const int nch = NR / 16;
    float l[kNR];
#pragma unroll
    for (int r = 0; r < kNR; ++r) l[r] = 0.f;
    bool ok = true;
    // A failed wait does not leave the loop: each iteration meets the same
    // named barriers as the other softmax warps, so a failing warp keeps
    // arriving there (skipping the work) until the loop ends.
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;                     // S^T buffer and P^T buffer of this tile
      unsigned char* const pt = ptb(b);
      if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_STF + b), (i >> 1) & 1, abort_p, kWaitNs)))
        ok = false;
      tc_fence_after();
      const uint32_t scol = tm + lane_base + COL_S + b * kNR;
      const int tp = slo + i * kTT + t;
      const int cls = tp >= shi ? 2 : (tp < ctx ? 0 : 1);  // context / draft / past the chunk
      uint32_t su[kNR];
      if (ok) {
        tmem_ld32_into<0>(scol, su);
        tmem_ld32_into<32>(scol + 32, su);
        tmem_ld32_into<64>(scol + 64, su);
        tmem_wait_ld();
      }
#define SV(r) __uint_as_float(su[r])
      // Draft token: rows that may not see it get -inf (padded rows keep
      // their finite score; their c = 0 and m_eff = +inf give P = 0).
      auto mask_draft = [&]() {
        const int a = tp - ctx;
#pragma unroll
        for (int r = 0; r < kNR; ++r)
          if (r < Rb && !draft_visible(kind, anc_s[r], jr_s[r], a)) su[r] = 0xFF800000u;  // -inf
      };
      if (cls == 1) mask_draft();
      if (i == 0) {
        // Seed each row's running maximum with the chunk's first token
        // (thread t = 0; it lies inside the chunk, and a draft row that may
        // not see it has its score masked to -inf): typical scores then stay
        // within 2^kSlack of the seed and the first tile needs no rescale.
        if (t == 0) {
#pragma unroll
          for (int r = 0; r < kNR; r += 4)
            *reinterpret_cast<float4*>(&f_s[r]) = make_float4(SV(r), SV(r + 1), SV(r + 2), SV(r + 3));
        }
        bar_sync(1, 128);
        if (t < Rb && ok) {
          const float x = f_s[t] * cm_s[t].x;
          const bool vis = x != -INFINITY;
          m_s[t] = vis ? x : -INFINITY;
          cm_s[t].y = vis ? x : INFINITY;
          thr_s[t] = vis ? (x + kSlack) * rc_s[t] : -INFINITY;
        }
        bar_sync(1, 128);
      }
      // Pass 1: does any visible score pass its row's trigger?
      bool hit = false;
      if (ok && cls != 2) {
#pragma unroll
        for (int r = 0; r < kNR; r += 4) {
          const float4 th = *reinterpret_cast<const float4*>(&thr_s[r]);
          hit |= (SV(r) > th.x) | (SV(r + 1) > th.y) | (SV(r + 2) > th.z) | (SV(r + 3) > th.w);
        }
      }
      const bool any = __any_sync(0xffffffffu, hit);
      if (lane == 0) flag_s[i & 1][quad] = any ? 1u : 0u;
      bar_sync(1, 128);
      const bool need = (flag_s[i & 1][0] | flag_s[i & 1][1] | flag_s[i & 1][2] | flag_s[i & 1][3]) != 0u;
      bool pe_done = false;
      if (need) {
        // Some row's maximum moves by more than 2^8 (or has not been set).
        // The previous tile's P.V must have landed (it also releases this
        // tile's P^T buffer, used as scratch here, and O^T for the rescale).
        if (i > 0) {
          if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_PE + ((i - 1) & 1)), ((i - 1) >> 1) & 1,
                                                       abort_p, kWaitNs)))
            ok = false;
          pe_done = true;
        }
        // The P^T buffer (free now) holds bf16(s*c) of every (token, row),
        // -inf where not visible; each owner thread r then takes its row's
        // maximum over the 128 tokens.
#pragma unroll
        for (int r = 0; r < kNR; r += 8) {
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 cm = *reinterpret_cast<const float4*>(&cm_s[r + 2 * q]);
            const float x0 = cls == 2 ? -INFINITY : SV(r + 2 * q) * cm.x;
            const float x1 = cls == 2 ? -INFINITY : SV(r + 2 * q + 1) * cm.z;
            const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
            pk[q] = *reinterpret_cast<const uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(pt + (r >> 6) * C::PT_BLK + sw128(t, (r & 63) >> 3)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        bar_sync(1, 128);
        if (t < Rb) {
          const int r = t;
          const unsigned char* col = pt + (r >> 6) * C::PT_BLK + ((r & 7) << 1);
          float Mk[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) Mk[k] = -INFINITY;
#pragma unroll 2
          for (int tk = 0; tk < kTT; tk += 8) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const unsigned short bits =
                  *reinterpret_cast<const unsigned short*>(col + sw128(tk + k, (r & 63) >> 3));
              Mk[k] = fmaxf(Mk[k], __uint_as_float((uint32_t)bits << 16));
            }
          }
          const float M = fmaxf(fmaxf(fmaxf(Mk[0], Mk[1]), fmaxf(Mk[2], Mk[3])),
                                fmaxf(fmaxf(Mk[4], Mk[5]), fmaxf(Mk[6], Mk[7])));
          const float m_old = m_s[r];
          const bool upd = M != -INFINITY && (m_old == -INFINITY || M > m_old + kSlack);
          const float m_new = upd ? M : m_old;
          const float f = upd ? (m_old == -INFINITY ? 0.f : ex2_approx(m_old - m_new)) : 1.f;
          m_s[r] = m_new;
          cm_s[r].y = m_new == -INFINITY ? INFINITY : m_new;
          thr_s[r] = m_new == -INFINITY ? -INFINITY : (m_new + kSlack) * rc_s[r];
          f_s[r] = f;
        }
        bar_sync(1, 128);
#pragma unroll
        for (int r = 0; r < kNR; r += 4) {
          const float4 f4 = *reinterpret_cast<const float4*>(&f_s[r]);
          l[r] *= f4.x;
          l[r + 1] *= f4.y;
          l[r + 2] *= f4.z;
          l[r + 3] *= f4.w;
        }
        if (i > 0 && ok) {
          // O^T columns of every row, this quadrant's lanes (values of d).
          tc_fence_after();
#pragma unroll 1
          for (int h = 0; h < C::DH; ++h) {
            const uint32_t oc = tm + lane_base + COL_O + h * kNR;
            uint32_t ou[kNR];
            tmem_ld32_into<0>(oc, ou);
            tmem_ld32_into<32>(oc + 32, ou);
            tmem_ld32_into<64>(oc + 64, ou);
            tmem_wait_ld();
#pragma unroll
            for (int r = 0; r < kNR; r += 4) {
              const float4 f4 = *reinterpret_cast<const float4*>(&f_s[r]);
              ou[r] = __float_as_uint(__uint_as_float(ou[r]) * f4.x);
              ou[r + 1] = __float_as_uint(__uint_as_float(ou[r + 1]) * f4.y);
              ou[r + 2] = __float_as_uint(__uint_as_float(ou[r + 2]) * f4.z);
              ou[r + 3] = __float_as_uint(__uint_as_float(ou[r + 3]) * f4.w);
            }
            tmem_st32_from<0>(oc, ou);
            tmem_st32_from<32>(oc + 32, ou);
            tmem_st32_from<64>(oc + 64, ou);
          }
          tmem_wait_st();
        }
        // The scores again (the S^T buffer is released only after pass 2),
        // so that they need not stay in registers through the rescale.
        if (ok) {
          tmem_ld32_into<0>(scol, su);
          tmem_ld32_into<32>(scol + 32, su);
          tmem_ld32_into<64>(scol + 64, su);
          tmem_wait_ld();
          if (cls == 1) mask_draft();
        } else {
#pragma unroll
          for (int r = 0; r < kNR; ++r) su[r] = 0u;
        }
      }
      // Pass 2: P = 2^(s c - m) into this tile's P^T buffer (fp16), row sums
      // in fp32, once the P.V of two tiles back has read that buffer.
      if (i > 1 && !pe_done && ok &&
          !__all_sync(0xffffffffu, mbar_wait(bar(B_PE + b), ((i >> 1) & 1) ^ 1, abort_p, kWaitNs)))
        ok = false;
      if (ok) {
        const float kill = cls == 2 ? -INFINITY : 0.f;
#pragma unroll
        for (int r = 0; r < kNR; r += 8) {
          uint32_t pk[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 cm = *reinterpret_cast<const float4*>(&cm_s[r + 2 * q]);
            const float p0 = ex2_approx(fmaf(SV(r + 2 * q), cm.x, -cm.y) + kill);
            const float p1 = ex2_approx(fmaf(SV(r + 2 * q + 1), cm.z, -cm.w) + kill);
            l[r + 2 * q] += p0;
            l[r + 2 * q + 1] += p1;
            pk[q] = h2u(__floats2half2_rn(p0, p1));
          }
          if (r < NR)
            *reinterpret_cast<uint4*>(pt + (r >> 6) * C::PT_BLK + sw128(t, (r & 63) >> 3)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_STE + b));
        mbar_arrive(bar(B_PF + b));
      }
    }
    // Epilogue: the last P.V; each row's sum over the 128 tokens in token
    // order (the per-thread sums pass through shared memory, in the V tile
    // area, idle now); (m, l, O) into the slot.
    if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_OF), 0, abort_p, kWaitNs))) ok = false;
    if (!ok && lane == 0) fail();
    tc_fence_after();
    // Shared memory is idle now: the row sums go to the Q^T / P^T area, O^T
    // to the V tile and raw-row area.
    constexpr int LP = kNR + 4;  // pitch (floats) of the [token][row] row sums
    constexpr int LBUF = kTT * LP * 4, OSTAGE = kNR * D * 4;
    constexpr bool LOW = LBUF <= C::OFF_VT;  // row sums below the V tiles, else after O
    static_assert(OSTAGE + (LOW ? 0 : LBUF) <= C::SMEM - 1024 - C::OFF_VT, "epilogue scratch");
    float* lbuf = reinterpret_cast<float*>(LOW ? sm : vt(0) + OSTAGE);
#pragma unroll
    for (int r = 0; r < kNR; r += 4)
      *reinterpret_cast<float4*>(lbuf + t * LP + r) = make_float4(l[r], l[r + 1], l[r + 2], l[r + 3]);
    bar_sync(1, 128);
    const bool bad = __any_sync(0xffffffffu, *abort_p != 0);
    if (t < Rb) {
      // Eight partial sums over tokens k, k + 8, ... then added in a fixed
      // order: the row's sum depends only on its own values.
      float ls[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls[k] = 0.f;
#pragma unroll 2
      for (int tk = 0; tk < kTT; tk += 8) {
#pragma unroll
        for (int k = 0; k < 8; ++k) ls[k] += lbuf[(tk + k) * LP + t];
      }
      const float lt = ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      const long long si = slot_s[t];
      p.ws_ml[2 * si] = bad ? NAN : m_s[t];
      p.ws_ml[2 * si + 1] = bad ? NAN : lt;
    }
    if (!bad) {
      // O^T half by half (every row's column in one TMEM round trip) into
      // [row][d] fp32 rows in shared memory (lanes = consecutive d), then
      // one bulk copy per row to its partial slot.
      float* ostage = reinterpret_cast<float*>(vt(0));
#pragma unroll 1
      for (int h = 0; h < C::DH; ++h) {
        const int d = 128 * h + 32 * quad + lane;
        const uint32_t oc = tm + lane_base + COL_O + h * kNR;
        uint32_t ou[kNR];
        tmem_ld32_into<0>(oc, ou);
        tmem_ld32_into<32>(oc + 32, ou);
        tmem_ld32_into<64>(oc + 64, ou);
        tmem_wait_ld();
        if (d < D) {
#pragma unroll
          for (int r = 0; r < kNR; ++r)
            if (r < Rb) ostage[r * D + d] = __uint_as_float(ou[r]);
        }
      }
      fence_proxy_async_smem();
      bar_sync(1, 128);
      if (t < Rb) {
        bulk_s2g(p.ws_acc + slot_s[t] * D, smem_u32(ostage + t * D), (uint32_t)(D * 4));
        bulk_commit_wait_all();
      }
    }
#undef SV
  } else if (warp < W_VDQ0) {
    // ------------------------------------------------------------ K dequant
    // Thread = token t of the tile (its TMEM lane).  Per tile: the token's
    // raw K row straight from L2 into registers (the producer keeps K tiles
    // ahead in L2), then per K slot fill (64 values of d) the hi and lo fp16
    // parts into the slot's two 32-column halves.
    set_regs<REG_KDQ>();
    const int quad = warp & 3;
    const int t = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const unsigned char* ksrc = reinterpret_cast<const unsigned char*>(p.k);
    const unsigned char* dsrc = reinterpret_cast<const unsigned char*>(p.dk);
    bool ok = true;
    int g = 0;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int tp = slo + i * kTT + t;
      const bool live = tp < shi;
      uint32_t w[C::NW + 1];
      w[C::NW] = 0u;
      if (live) {
        const unsigned char* src;
        if (scratch && tp >= ctx) {
          src = dsrc + scratch_row(p, row0, kvh, tp - ctx) * C::RB;
        } else if (!PAGED) {
          src = ksrc + (((long long)s * p.KVH + kvh) * p.capacity + tp) * C::RB;
        } else {
          const int blk = p.block_table[(long long)s * p.max_blocks + tp / kPage];
          src = ksrc + (((long long)blk * p.KVH + kvh) * kPage + tp % kPage) * C::RB;
        }
        load_row<D>(*reinterpret_cast<uint32_t(*)[C::NW]>(w), src);
      }
#pragma unroll
      for (int f = 0; f < C::NFILL; ++f) {
        const int ks = (g + f) & 1;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_KSE + ks), (((g + f) >> 1) & 1) ^ 1,
                                                     abort_p, kWaitNs)))
          ok = false;
        if (!ok) continue;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t hv[16], lv[16];
          __half2 d2;
          uint32_t code[8];
          q8_block(w, 2 * f + hb, d2, code);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            __half2 x0, x1;
            codes_to_h2(code[q], x0, x1);
            const __half2 h0 = __hmul2(x0, d2), h1 = __hmul2(x1, d2);
            hv[2 * q] = live ? h2u(h0) : 0u;
            hv[2 * q + 1] = live ? h2u(h1) : 0u;
            lv[2 * q] = live ? h2u(__hfma2(x0, d2, __hneg2(h0))) : 0u;
            lv[2 * q + 1] = live ? h2u(__hfma2(x1, d2, __hneg2(h1))) : 0u;
          }
          tmem_st16(tm + lane_base + COL_K + ks * 64 + hb * 16, hv);
          tmem_st16(tm + lane_base + COL_K + ks * 64 + 32 + hb * 16, lv);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_KSF + ks));
      }
      g += C::NFILL;
    }
    if (!ok && lane == 0) fail();
  } else {
    // ------------------------------------------------------------ V dequant
    // Thread = token t of the tile.  Per tile, once the raw rows have landed
    // and the V buffer is free: fp16(d*q) into the 128-byte-swizzled
    // MN-major tile (64-d column blocks, one 128-byte row per token), two Q8
    // blocks (17 words of the raw row) at a time; then the raw buffer is
    // released.  Tokens past the chunk are zeros.
    set_regs<REG_VDQ>();
    const int t = (warp - W_VDQ0) * 32 + lane;
    const unsigned char* dsrc = reinterpret_cast<const unsigned char*>(p.dv);
    bool ok = true;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int b = i % C::NRAW, vb = i % C::NVB;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_RVF + b), (i / C::NRAW) & 1, abort_p, kWaitNs) &&
                                       mbar_wait(bar(B_VE + vb), ((i / C::NVB) & 1) ^ 1, abort_p, kWaitNs))) {
        ok = false;
        break;
      }
      const int tp = slo + i * kTT + t;
      const bool live = tp < shi;
      const unsigned char* row = (scratch && tp >= ctx)
                                     ? dsrc + scratch_row(p, row0, kvh, tp - ctx) * C::RB
                                     : rawv(b) + t * C::RB;
      unsigned char* dst = vt(vb);
#pragma unroll 1
      for (int pr = 0; pr < C::NB / 2; ++pr) {
        uint32_t w[18];
        w[17] = 0u;
        if (live) {
#pragma unroll
          for (int k = 0; k < 17; ++k) w[k] = reinterpret_cast<const uint32_t*>(row + 68 * pr)[k];
        }
        unsigned char* col = dst + pr * C::VT_BLK;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          __half2 d2;
          uint32_t code[8];
          q8_block(w, hb, d2, code);
          // 8 values of d (one 16-byte chunk) at a time.
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 out = make_uint4(0u, 0u, 0u, 0u);
            if (live) {
              __half2 x0, x1, x2, x3;
              codes_to_h2(code[2 * c], x0, x1);
              codes_to_h2(code[2 * c + 1], x2, x3);
              out = make_uint4(h2u(__hmul2(x0, d2)), h2u(__hmul2(x1, d2)), h2u(__hmul2(x2, d2)),
                               h2u(__hmul2(x3, d2)));
            }
            *reinterpret_cast<uint4*>(col + sw128(t, hb * 4 + c)) = out;
          }
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_VF + vb));
        mbar_arrive(bar(B_RVE + b));
      }
    }
    if (!ok && lane == 0) fail();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_SMMA) tmem_dealloc(tm, TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Host side.

template <int D, bool PAGED>
static cudaError_t launch_tq8_t(const Params& p, dim3 grid, cudaStream_t st) {
  using C = tq8::Cfg<D>;
  static int checked = 0;  // 1 ok, -1 refused
  if (checked == 0) {
    cudaError_t e = cudaFuncSetAttribute(tq8_partial_kernel<D, PAGED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    // The warpgroups' register budgets add up to exactly the registers the
    // block is launched with; a kernel built with another count could make
    // a budget increase wait forever, so it is never launched.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, tq8_partial_kernel<D, PAGED>);
    if (e != cudaSuccess) return e;
    checked = (fa.numRegs == tq8::kLaunchRegs) ? 1 : -1;
  }
  if (checked < 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(tq8::kThreads);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, tq8_partial_kernel<D, PAGED>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int tq8_rows_per_block() { return tq8::kNR; }
int tq8_threads() { return tq8::kThreads; }

int tq8_smem_bytes(int D) {
  switch (D) {
    case 64: return tq8::Cfg<64>::SMEM;
    case 128: return tq8::Cfg<128>::SMEM;
    case 256: return tq8::Cfg<256>::SMEM;
  }
  return 0;
}

cudaError_t launch_tq8_partial(const Params& p, dim3 grid, cudaStream_t st) {
  const bool paged = p.page_size != 0;
  switch (p.D) {
    case 64: return paged ? launch_tq8_t<64, true>(p, grid, st) : launch_tq8_t<64, false>(p, grid, st);
    case 128: return paged ? launch_tq8_t<128, true>(p, grid, st) : launch_tq8_t<128, false>(p, grid, st);
    case 256: return paged ? launch_tq8_t<256, true>(p, grid, st) : launch_tq8_t<256, false>(p, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace va
