// Tensor-core split-KV partial kernel (tcgen05 + TMEM + TMA), sm_103a.
//
// One CTA owns (sequence, KV head, KV chunk) and ALL query rows of that KV
// head (n rows x G heads <= 128 per row block), so every K/V byte of its
// token range is read from HBM exactly once for every row it serves
// (hipfire PR #695, alpineQ comments: one block reuses each Q8 K/V fetch
// across several verifier rows; here across all of them).  Per 64-token
// tile:
//
//   S = Q K^T      tcgen05.mma, A = Q (TMEM), B = K tile (smem, K-major);
//                  bf16: N = 64 tokens into one of two S buffers; Q8: N =
//                  128 over [K hi rows; K lo rows] of the tile, one MMA per
//                  K step, into one S buffer (columns 0..63 Q.K_hi, 64..127
//                  Q.K_lo)
//   softmax        8 warps, one TMEM lane (= query row) per thread and one
//                  half of the tile's columns per warp; masks (chain rows
//                  causal by index, tree rows by ancestor mask); online
//                  (m, l) in log2 units; P written back over S (bf16) or
//                  into a shared-memory P tile (Q8, after the softmax has
//                  released the S buffer)
//   O += P V       tcgen05.mma, A = P (TMEM for bf16, the shared P tile for
//                  Q8), B = V tile (smem, MN-major)
//
// O (fp32, 128 lanes x D columns) lives in TMEM for the CTA's whole range.
// At the end each row's (m, l, O) goes to its partial slot; the merge
// kernel combines slots (hipfire PR #817 "FA2 split-KV", sections "Summary"
// and "Performance").
//
// Caches:
//   Q8_0, contiguous: a tile's raw 34-byte blocks arrive by one 1-D bulk
//     copy per tensor into a tile buffer; four warps per tensor dequantise
//     them in place to fp16 in the 128-byte-swizzled MMA layout,
//     zero-filling tokens past the range.  A K element d*q (up to 18
//     significant bits) becomes hi = fp16(d*q) and the residual lo =
//     fma(d, q, -hi), exact in fp16, written 64 rows below it in the same
//     column block, so the S MMA over [hi; lo] sees d*q exactly; V
//     elements are fp16(d*q) (one rounding).  Paged (a separate
//     instantiation): the same warps load the raw rows themselves through
//     the block table (a tree sequence's drafts from the tree scratch KV
//     when one is given).  Q is converted to fp16 after a per-row
//     power-of-two rescale (exact), and the scale folds into the score
//     multiplier.  P is fp16.
//   bf16: tiled TMA loads place K/V tiles directly in the MMA layout; one
//     warp zeroes V rows past the range of a ragged tile.  P is split into
//     bf16 hi + lo halves (two MMAs) so P keeps 16 significant bits.
//   Both: Q rows are staged in shared memory by warps 2.. with coalesced
//     loads during the prologue and moved into TMEM by the softmax warps.
//
// Warp roles: 0 = copy producer, 1 = TMEM owner + S MMA issuer, 2..9 =
// softmax/epilogue (two warps per TMEM lane quadrant), 13 (Q8) or 11
// (bf16) = P.V MMA issuer, Q8: 10, 11, 12, 17 dequantise K and 14, 15,
// 16, 19 V (each group spread over the four sub-partitions); bf16: 10
// fixes up V tails.
// Every wait is bounded (VA_DEV_TIMEOUT); on a timeout the CTA drains its
// own copies and MMAs, frees TMEM and writes NaN partials.
#include <limits.h>
#include <string.h>

#include "va_common.cuh"
#include "va_sm100.cuh"

namespace va {
using namespace sm100;

constexpr int kNT = 64;      // tokens per tile
constexpr int kPrefetch = 4; // L2 prefetch distance in tiles (Q8 raw stream)
constexpr int kM = 128;      // MMA rows (query rows per CTA)
constexpr uint64_t kWaitNs = 2000000000ull;

template <int D, int KVT>
struct UCfg {
  static constexpr bool kQ8 = (KVT == VA_Q8_0);
  static constexpr int RB = kQ8 ? D / 32 * 34 : D * 2;  // global bytes per token row
  static constexpr int NB = D / 32;                      // Q8 blocks per row
  static constexpr int DBLK = D / 64;                    // 64-element column blocks
  static constexpr int TILE = kNT * D * 2;               // one 16-bit tile in smem
  static constexpr int NB16 = 2;                         // Q8 tile buffers per tensor
  static constexpr int PTILE = kM * kNT * 2;             // Q8: one fp16 P tile (rows x tokens)
  static constexpr int NST = (D == 256) ? 3 : (D == 128 ? 6 : 8);  // bf16 K+V stages
  static constexpr int COL_O = 0;
  static constexpr int COL_S0 = D;
  static constexpr int COL_Q = D + 2 * kNT;
  static constexpr int TMEM_COLS = (COL_Q + D / 2 <= 256) ? 256 : 512;
  static constexpr int DQ_WARPS = kQ8 ? 8 : 1;
  // Q8: warp 13 issues the P.V MMAs and eight of warps 10..19 dequantise
  // (dq_slot).  bf16: warp 10 fixes up V tails, warp 11 issues the P.V
  // MMAs.
  static constexpr int PV_WARP = kQ8 ? 13 : 11;
  static constexpr int THREADS = (kQ8 ? 20 : 12) * 32;
  static constexpr int MAXREG = (65536 / THREADS) / 8 * 8 > 255 ? 255 : (65536 / THREADS) / 8 * 8;
  // Q8: per buffer a K tile of hi and lo parts (2 TILE) and a V tile, then
  // the P tile.
  static constexpr int SMEM_Q8 = 3 * NB16 * TILE + PTILE;
  static constexpr int SMEM_BF16 = NST * 2 * TILE;
  static constexpr int SMEM_EPI = kM * (D * 4 + 16);  // O staging at the end
  static constexpr int SMEM_MAIN = kQ8 ? SMEM_Q8 : SMEM_BF16;
  static constexpr int SMEM = (SMEM_MAIN > SMEM_EPI ? SMEM_MAIN : SMEM_EPI) + 1024 + 64;
};

// Barrier slots in static shared memory.
enum {
  B_SFULL = 0,    // [2] S of the buffer's tile is in TMEM
  B_PFULL = 2,    // [2] P of the buffer's tile is in TMEM
  B_SFREE = 4,    // [2] P.V of the buffer's tile has completed
  B_QREADY = 6,
  B_DRAIN = 7,    // [2] S issuer, P.V issuer
  B_OFINAL = 9,   // the last P.V has completed
  // Q8 tile buffers, [tensor 0 = K / 1 = V][3 slots, NB16 used]: raw bytes
  // landed, fp16 ready (K: hi and lo parts), buffer free again.
  B_QFULL = 10,   // [2][3]
  B_QREADY8 = 16, // [2][3]
  B_QEMPTY = 22,  // [2][3]
  // Q8 only (these slots are the bf16 stage barriers' in the other
  // instantiation): the P.V that read the P tile completed; the softmax has
  // read the S buffer.
  B_PFREE = 28,
  B_SCONS = 30,
  // bf16 stages [NST]: K landed, V landed, V fixed up, stage free.
  B_RFULL = 28,
  B_VFULL = 36,
  B_VREADY = 44,
  B_REMPTY = 52,
  B_COUNT = 60
};

// Byte offset of element (row, col) inside one 128-byte-swizzled column
// block whose rows are 128 bytes apart (col in 16-bit elements, < 64).
__device__ __forceinline__ uint32_t sw128_off(int row, int chunk16) {
  return (uint32_t)(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// Q8 dequantisation slot of a warp (-1: none): slots 0..3 dequantise K,
// 4..7 V.  Each group holds one warp of every sub-partition (warp index
// mod 4) except that V doubles up on sub-partition 3, whose softmax warps
// serve query rows 96..127 (idle when a KV head has at most 96 rows).
__device__ __forceinline__ int dq_slot(int warp) {
  switch (warp) {
    case 10: return 0;
    case 11: return 1;
    case 12: return 2;
    case 17: return 3;
    case 14: return 4;
    case 15: return 5;
    case 16: return 6;
    case 19: return 7;
    default: return -1;
  }
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// One Q8_0 block (fp16 scale d, 32 int8 codes q) held in words w from
// word wo (odd: the block starts two bytes into w[wo]; live false: zeros)
// -> fp16 hi = fp16(d*q) into the 16-byte chunks c0 .. c0 + 3 of token row
// t of the swizzled column block hi.  With lo (K tiles), also the residuals
// fma(d, q, -hi) into the same place of lo: a residual of d*q (at most 18
// significant bits) below hi's last bit fits fp16 exactly, so hi + lo ==
// d*q and the S MMAs over both parts see the exact K element.  A chunk is
// stored as soon as it is converted, to keep few values in registers.
__device__ __forceinline__ void dq_block_store(const uint32_t* w, int wo, bool odd, bool live,
                                               unsigned char* hi, unsigned char* lo, int t, int c0) {
  uint32_t sbits = 0u, code[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) code[q] = 0u;
  if (live) {
    if (odd) {
      sbits = w[wo] >> 16;
#pragma unroll
      for (int q = 0; q < 8; ++q) code[q] = w[wo + 1 + q];
    } else {
      sbits = w[wo] & 0xFFFFu;
#pragma unroll
      for (int q = 0; q < 8; ++q) code[q] = __funnelshift_r(w[wo + q], w[wo + q + 1], 16);
    }
  }
  const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)sbits));
  const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t hv[4], lv[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint32_t x = code[2 * c + k] ^ 0x80808080u;  // bytes q + 128
      uint32_t b0 = __byte_perm(x, 0x64646464u, 0x4140);
      uint32_t b1 = __byte_perm(x, 0x64646464u, 0x4342);
      const __half2 q0 = __hsub2(*reinterpret_cast<__half2*>(&b0), bias);  // exact codes
      const __half2 q1 = __hsub2(*reinterpret_cast<__half2*>(&b1), bias);
      __half2 a = __hmul2(q0, d2);
      __half2 e = __hmul2(q1, d2);
      hv[2 * k] = *reinterpret_cast<uint32_t*>(&a);
      hv[2 * k + 1] = *reinterpret_cast<uint32_t*>(&e);
      if (lo) {
        __half2 la = __hfma2(q0, d2, __hneg2(a));
        __half2 le = __hfma2(q1, d2, __hneg2(e));
        lv[2 * k] = *reinterpret_cast<uint32_t*>(&la);
        lv[2 * k + 1] = *reinterpret_cast<uint32_t*>(&le);
      }
    }
    const uint32_t off = sw128_off(t, c0 + c);
    *reinterpret_cast<uint4*>(hi + off) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    if (lo) *reinterpret_cast<uint4*>(lo + off) = make_uint4(lv[0], lv[1], lv[2], lv[3]);
  }
}

// Convert and store the NBH blocks of a half-row held in words w (the first
// block starting sh = 0 or 2 bytes into w[0]).  K (with lo parts): 64-d
// column blocks of hi rows then lo rows.  With sh = 0 and an even NBH the
// blocks go two at a time (68 bytes = 17 words: blocks at words 0 and 8 + 2
// bytes), the next pair's words moving down by 17 after each step, so the
// conversion is one two-block step in the code rather than NBH unrolled
// copies (which would crowd the instruction cache).
template <int NBH, int NW>
__device__ __forceinline__ void dq_half_row(uint32_t (&w)[NW], int sh, int hf, bool live,
                                            unsigned char* buf, unsigned char* lobuf, int t) {
  if (NBH % 2 == 0 && sh == 0) {
#pragma unroll 1
    for (int jp = 0; jp < NBH / 2; ++jp) {
      const int b0 = hf * NBH + 2 * jp;  // even block index in the row: chunks 0-3, then 4-7
      const int boff = (b0 >> 1) * (lobuf ? 2 : 1) * (kNT * 128);
      unsigned char* lo = lobuf ? lobuf + boff : nullptr;
      dq_block_store(w, 0, false, live, buf + boff, lo, t, 0);
      dq_block_store(w, 8, true, live, buf + boff, lo, t, 4);
#pragma unroll
      for (int q = 0; q + 17 < NW; ++q) w[q] = w[q + 17];
    }
  } else {
#pragma unroll
    for (int jb = 0; jb < NBH; ++jb) {
      const int b = hf * NBH + jb;  // block index in the row
      const int boff = (b >> 1) * (lobuf ? 2 : 1) * (kNT * 128);
      const int o = sh + 34 * jb;   // block offset in the words
      dq_block_store(w, o >> 2, o & 2, live, buf + boff, lobuf ? lobuf + boff : nullptr, t,
                     (b & 1) * 4);
    }
  }
}

// Q8_0 dequantisation by direct loads (paged caches).  A thread owns one
// half-row (token t = gtid % 64 of the tile, half hf = gtid / 64 of its
// D/32 blocks).  It loads the raw bytes of its half-row from global memory
// into registers (DqRaw, issued before the tile buffer is free, so the
// latency hides behind the wait), then converts them and writes fp16 into
// the 128-byte-swizzled K-major tile layout (eight consecutive threads take
// eight consecutive tokens of one block, so their 16-byte stores hit
// distinct bank groups).  Tokens >= valid become zeros.
template <int D>
struct DqRaw {
  static constexpr int NB = D / 32;               // blocks per row
  static constexpr int RB = NB * 34;              // bytes per row
  static constexpr int HB = RB / 2;               // bytes per half-row
  // Does the second half-row start 2 bytes into a word (D = 64 only)?  Else
  // both halves' blocks sit at the same word offsets, so one conversion
  // serves both (a second copy of the unrolled conversion would crowd the
  // instruction cache).
  static constexpr bool kOdd = (HB % 4) != 0;
  static constexpr int NW = (HB + (kOdd ? 2 : 0) + 3) / 4;
  uint32_t w[NW];
};

// `row` is in global memory (read-only for the kernel's lifetime).
template <int D>
__device__ __forceinline__ void dq_load(DqRaw<D>& r, const unsigned char* row, int hf, bool live) {
  using R = DqRaw<D>;
  if (!live) return;
  if (D == 256) {
    // 136 bytes from an 8-byte boundary: eight 16-byte loads and one 8-byte
    // load at the end (first half) or at the start (second half).
    static_assert(D != 256 || R::NW == 34, "D = 256 half-row words");
    const uint4* q = reinterpret_cast<const uint4*>(row + (hf ? R::HB + 8 : 0));
    const uint2 e = __ldg(reinterpret_cast<const uint2*>(row + (hf ? R::HB : 128)));
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldg(q + k);
    if (hf) {
      r.w[0] = e.x;
      r.w[1] = e.y;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        r.w[2 + 4 * k] = v[k].x;
        r.w[3 + 4 * k] = v[k].y;
        r.w[4 + 4 * k] = v[k].z;
        r.w[5 + 4 * k] = v[k].w;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        r.w[4 * k] = v[k].x;
        r.w[1 + 4 * k] = v[k].y;
        r.w[2 + 4 * k] = v[k].z;
        r.w[3 + 4 * k] = v[k].w;
      }
      r.w[32] = e.x;
      r.w[33] = e.y;
    }
  } else {
    const int start = hf * R::HB;
    const uint32_t* q = reinterpret_cast<const uint32_t*>(row + (start & ~3));
#pragma unroll
    for (int k = 0; k < R::NW; ++k) r.w[k] = __ldg(q + k);
  }
}

// Convert and store a loaded half-row (its words are consumed).
template <int D>
__device__ __forceinline__ void dq_convert(DqRaw<D>& r, unsigned char* buf, unsigned char* lobuf,
                                           int t, int hf, bool live) {
  // The half-row starts 0 bytes into the loaded words, or 2 (second half at
  // D = 64).
  dq_half_row<D / 64>(r.w, DqRaw<D>::kOdd && hf ? 2 : 0, hf, live, buf, lobuf, t);
}

// Dequantise, in place, the raw Q8_0 rows (RB bytes apart) at the start of
// a tile buffer into the fp16 MMA layout of the same buffer; tokens >= valid
// become zeros.  128 threads (named barrier `barid`): thread -> (token
// t = tid % 64, half-row hf = tid / 64).  Phase A reads every raw byte the
// thread needs into registers, the barrier waits for all readers, phase B
// writes the fp16 rows (eight consecutive threads take eight consecutive
// tokens of one block, so their 16-byte stores hit distinct bank groups).
template <int D>
__device__ __forceinline__ void dequant_inplace(unsigned char* buf, unsigned char* lobuf, int valid,
                                                int tid, int barid, bool work) {
  constexpr int NB = D / 32;      // blocks per row
  constexpr int RB = NB * 34;     // bytes per row
  constexpr int HB = RB / 2;      // bytes per half-row
  constexpr int NBH = NB / 2;     // blocks per half-row
  constexpr int NW = (HB + 2 + 3) / 4 + 1;
  const int t = tid & 63, hf = tid >> 6;
  const int start = t * RB + hf * HB;
  // 0 or 2; 0 unless HB is not a multiple of 4 (D = 64), which leaves one
  // unrolled conversion in the code instead of two.
  const int sh = HB % 4 ? (start & 3) : 0;
  uint32_t w[NW];
  const bool live = work && t < valid;
  if (live) {
    if (D == 256 && hf == 0) {
      // 16-byte aligned: 9 x 16-byte loads (the last 8 bytes belong to hf 1).
      const uint4* q = reinterpret_cast<const uint4*>(buf + start);
#pragma unroll
      for (int k = 0; k < 9; ++k) {
        const uint4 v = q[k];
        w[4 * k] = v.x;
        w[4 * k + 1] = v.y;
        w[4 * k + 2] = v.z;
        w[4 * k + 3] = v.w;
      }
    } else if (D == 256) {
      // 8-byte aligned half-row.
      const uint2* q = reinterpret_cast<const uint2*>(buf + start);
#pragma unroll
      for (int k = 0; k < 17; ++k) {
        const uint2 v = q[k];
        w[2 * k] = v.x;
        w[2 * k + 1] = v.y;
      }
    } else {
      const uint32_t* q = reinterpret_cast<const uint32_t*>(buf + (start - sh));
#pragma unroll
      for (int k = 0; k < NW; ++k) w[k] = q[k];
    }
  }
  named_barrier_sync(barid, 128);
  if (work) dq_half_row<NBH, NW>(w, sh, hf, live, buf, lobuf, t);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two probabilities for the P.V MMA: fp16 pair (Q8 path), or bf16
// hi pair + bf16 lo pair (bf16 path) so that hi + lo carries 16 bits.
template <bool Q8>
__device__ __forceinline__ void pack_p(float a, float b, uint32_t& hi, uint32_t& lo) {
  if (Q8) {
    __half2 h = __floats2half2_rn(a, b);
    hi = *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
    hi = *reinterpret_cast<uint32_t*>(&h);
    lo = *reinterpret_cast<uint32_t*>(&l);
  }
}

// PAGED: the cache is paged (Q8: the dequantising warps load the raw rows
// themselves; bf16: one tensor load per 16-token page); a separate
// instantiation, so the contiguous kernel carries none of that code.
template <int D, int KVT, bool PAGED>
__global__ void __launch_bounds__(UCfg<D, KVT>::THREADS, 1) __maxnreg__((UCfg<D, KVT>::MAXREG))
    umma_partial_kernel(const Params p, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV) {
  using C = UCfg<D, KVT>;
  constexpr bool Q8 = C::kQ8;
  extern __shared__ unsigned char smem_raw[];
  __shared__ __align__(8) uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ int err_s;
  __shared__ float red_max[2][2][kM];
  __shared__ float red_q[2][kM];
  __shared__ float red_l[kM];

  // The merge kernel may launch now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;");
  // Launched as a programmatic dependent of whatever precedes it on the
  // stream: the CTAs may become resident early, but nothing is read or
  // written before that work has completed and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kvh = blockIdx.y, s = blockIdx.z;

  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  if (err & VA_DEV_BAD_ROWS) {
    if (tid == 0) flag(p.status, err);
    return;
  }
  // Row block and chunk (one level of chunks: split 0, slot = chunk).
  int rb, sub, nsub;
  if (!cta_work(p, n, blockIdx.x, &rb, &sub, &nsub)) return;
  const int split = 0, slot = sub;
  const int G = p.G;
  const int R = n * G;
  if (rb * kM >= R) return;
  const int L = ctx + n;
  int lo, hi, slo, shi;
  split_range(L, p.S, split, &lo, &hi);
  sub_range(lo, hi, nsub, p.min_sub, sub, &slo, &shi);
  const int ntiles = (shi - slo + kNT - 1) / kNT;
  if (ntiles == 0 && !err) {
    // An empty chunk (short span): its rows' slots become (-inf, 0) at once,
    // without the prologue.  The sequence's other CTAs check its parents.
    if (tid < kM) {
      const int rs = rb * kM + tid;
      if (rs < R) {
        const long long si0 = slot_index(p, slot, row0 + rs / G, kvh * G + rs % G);
        p.ws_ml[2 * si0] = -INFINITY;
        p.ws_ml[2 * si0 + 1] = 0.f;
      }
    }
    return;
  }

  // Softmax-thread row identity.
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int rseq = rb * kM + r;
  const bool is_sm = (warp >= 2 && warp < 10);
  const bool rvalid = is_sm && rseq < R;
  const int j = rvalid ? rseq / G : 0;
  const int g = rvalid ? rseq % G : 0;
  const int kind = seq_kind_of(p, s);
  // Tree sequence with a tree scratch KV: draft positions (>= ctx) are read
  // from the scratch rows, and the cache (block table) covers the context
  // only.  (Paged Q8 instantiation; the host routes other caches with a
  // scratch KV to the CUDA-core kernel.)
  const bool scratch = PAGED && uses_scratch(p, kind);

  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  // Shared-memory regions.
  //   Q8: buffers (K_j, V_j), j < NB16, then the P tile.  Raw Q8 rows
  //       land at the start of a K or V tile and are dequantised in place.
  //       A K tile holds, per 64-d column block, the 64 token rows of hi
  //       parts and then the 64 rows of lo parts, so that [hi; lo] is one
  //       128-row B operand; a V tile is the fp16 values.  The P tile
  //       holds the fp16 probabilities of a tile, 128 rows of 64 tokens
  //       (K-major, 128-byte swizzle), the A operand of the P.V MMA.
  //   bf16: stages of (K tile, V tile).
  auto q8buf = [&](int kv, int j) { return sm + (3 * j + 2 * kv) * C::TILE; };
  auto q8lo = [&](int j) { return q8buf(0, j) + kNT * 128; };
  auto q8p = [&]() { return sm + 3 * C::NB16 * C::TILE; };
  auto kst = [&](int st) { return sm + st * 2 * C::TILE; };            // bf16 K stage
  auto vst = [&](int st) { return sm + st * 2 * C::TILE + C::TILE; };  // bf16 V stage
  // Contiguous Q8 cache: L2 prefetch of the raw rows of tensor kv (0 = K,
  // 1 = V), tile i.
  auto prefetch_q8 = [&](int i, int kv) {
    const unsigned char* src = (const unsigned char*)(kv ? p.v : p.k);
    const int tp = slo + i * kNT;
    const int np = min(tp + kNT, (shi + kPage - 1) / kPage * kPage) - tp;
    const long long rowp = ((long long)s * p.KVH + kvh) * p.capacity + tp;
    bulk_prefetch_l2(src + rowp * C::RB, (uint32_t)(np * C::RB));
  };
  // Contiguous Q8 cache: copy the raw rows of tensor kv, tile i, into
  // buffer i % NB16 (whose previous tile must be consumed), and pull tile
  // i + kPrefetch into L2.
  auto issue_q8 = [&](int i, int kv) {
    const int jb = i % C::NB16;
    const uint64_t pol = policy_evict_first();
    const int t0 = slo + i * kNT;
    const int nload = min(t0 + kNT, (shi + kPage - 1) / kPage * kPage) - t0;  // multiple of 16
    const unsigned char* src = (const unsigned char*)(kv ? p.v : p.k);
    unsigned char* dst = q8buf(kv, jb);
    const uint32_t fb = bar(B_QFULL + 3 * kv + jb);
    if (i + kPrefetch < ntiles) prefetch_q8(i + kPrefetch, kv);
    mbar_arrive_expect_tx(fb, (uint32_t)(nload * C::RB));
    const long long rowi = ((long long)s * p.KVH + kvh) * p.capacity + t0;
    bulk_g2s(smem_u32(dst), src + rowi * C::RB, (uint32_t)(nload * C::RB), fb, pol);
  };

  // bf16, contiguous cache: tile i's K and V by tiled TMA loads (one per
  // 64-d column block) into stage i % NST.
  auto issue_bf16 = [&](int i) {
    const int st = i % C::NST;
    const uint64_t pol = policy_evict_first();
    const int t0 = slo + i * kNT;
    mbar_arrive_expect_tx(bar(B_RFULL + st), (uint32_t)C::TILE);
    mbar_arrive_expect_tx(bar(B_VFULL + st), (uint32_t)C::TILE);
    const int plane = s * p.KVH + kvh;
    for (int db = 0; db < C::DBLK; ++db) {
      tma_load_3d(smem_u32(kst(st) + db * kNT * 128), &tmK, db * 64, t0, plane, bar(B_RFULL + st),
                  pol);
      tma_load_3d(smem_u32(vst(st) + db * kNT * 128), &tmV, db * 64, t0, plane, bar(B_VFULL + st),
                  pol);
    }
  };

  // Q8, contiguous cache: the raw rows of a tile arrive by one bulk copy per
  // tensor into the tile buffer and are dequantised in place.  Paged cache:
  // a tile would take one small copy per 16-token page, so the dequantising
  // warps load the raw rows themselves (`direct`).  Tile 0 goes to buffers
  // K0/V0, which the Q staging does not use; every address is known to be in
  // range (the span was checked against the capacity), so these copies go
  // out before the rest of the prologue.
  constexpr bool direct = Q8 && PAGED;
  // bf16, contiguous cache: likewise tile 0's tensor loads (stage 0).
  auto issue_first = [&]() {
    if (Q8) {
      issue_q8(0, 0);
      issue_q8(0, 1);
    } else {
      issue_bf16(0);
    }
  };
  const bool early = !PAGED && !err && ntiles > 0;
  constexpr int kQRow = D * 2 + 16;
  // Q staging: buffer 1 (K1 V1, 3 tiles, room for 128 rows at every D), so
  // tile 1's copies and conversions wait until Q is in TMEM.
  // bf16: from stage 1 on (stages 1 and 2 at most), so tile 1's loads
  // wait likewise.
  static_assert(!Q8 || kM * kQRow <= 3 * C::TILE, "Q staging");
  static_assert(Q8 || kM * kQRow <= (C::NST - 1) * 2 * C::TILE, "Q staging");
  unsigned char* const qstage = Q8 ? q8buf(0, 1) : kst(1);
  const int qfirst = 1;  // first tile whose buffers hold the staging

  if (tid == 0) {
    err_s = 0;
    abort_s = 0;
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_PFULL + 1), 8);
    mbar_init(bar(B_SFREE), 1);
    mbar_init(bar(B_SFREE + 1), 1);
    mbar_init(bar(B_QREADY), 8);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    mbar_init(bar(B_OFINAL), 1);
    if (Q8) {
      for (int i = 0; i < 6; ++i) {
        mbar_init(bar(B_QFULL + i), 1);
        mbar_init(bar(B_QREADY8 + i), C::DQ_WARPS / 2);
        mbar_init(bar(B_QEMPTY + i), 1);
      }
      mbar_init(bar(B_PFREE), 1);
      mbar_init(bar(B_SCONS), 8);
    } else {
      for (int i = 0; i < C::NST; ++i) {
        mbar_init(bar(B_RFULL + i), 1);
        mbar_init(bar(B_VFULL + i), 1);
        mbar_init(bar(B_VREADY + i), 1);
        mbar_init(bar(B_REMPTY + i), 1);
      }
    }
    fence_barrier_init();
    if (early) issue_first();
  }
  // Warps 2.. stage this CTA's Q rows in shared memory (rows padded to
  // kQRow bytes so that the lanes of a warp read distinct bank groups) with
  // every load in flight and consecutive lanes on consecutive 16 bytes of a
  // row, overlapping the rest of the prologue; the softmax warps move them
  // into TMEM (Q8: converted to fp16).  The staging takes buffer 1 / stage
  // 1 on (see qstage).
  if (warp >= 2) {
    constexpr int CPR = D / 8;  // 16-byte chunks per row
    constexpr int NTHR = C::THREADS - 64;
    constexpr int ITER = (kM * CPR + NTHR - 1) / NTHR;
    const int rows_blk = min(kM, R - rb * kM);
    const int total = rows_blk * CPR;
    const int t = tid - 64;
    uint4 v[ITER];
#pragma unroll
    for (int k = 0; k < ITER; ++k) {
      const int c = t + k * NTHR;
      if (c < total) {
        const int rs = rb * kM + c / CPR;
        const long long qi = ((long long)(row0 + rs / G) * p.H + kvh * G + rs % G) * D;
        v[k] = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(p.q) + qi)[c % CPR];
      }
    }
#pragma unroll
    for (int k = 0; k < ITER; ++k) {
      const int c = t + k * NTHR;
      if (c < total)
        *reinterpret_cast<uint4*>(qstage + (c / CPR) * kQRow + (c % CPR) * 16) = v[k];
    }
    named_barrier_sync(2, NTHR);
  }
  __syncthreads();
  unsigned anc = 0;
  if (rvalid && !err) {
    bool bad = false;
    anc = row_mask(kind, p.parent + row0, j, &bad);
    if (bad) atomicOr(&err_s, (int)VA_DEV_BAD_PARENT);
  }
  if (PAGED && !err && ntiles > 0) {
    const int cend = scratch ? min(shi, ctx) : shi;  // cache tokens of the range
    const int pg0 = slo / kPage, pg1 = (cend + kPage - 1) / kPage;
    for (int pg = pg0 + tid; pg < pg1; pg += blockDim.x) {
      int blk = p.block_table[(long long)s * p.max_blocks + pg];
      if (blk < 0 || blk >= p.num_blocks) atomicOr(&err_s, (int)VA_DEV_BAD_BLOCK);
    }
  }
  __syncthreads();
  err |= (unsigned)err_s;

  // Slot of this thread's row.
  const int grow = row0 + j, h = kvh * G + g;
  const long long si = slot_index(p, slot, grow, h);

  if (err || ntiles == 0) {
    if (early && tid == 0) {
      // Let the copies already issued land before the CTA goes away.
      int dummy = 0;
      volatile int* never = &dummy;
      mbar_wait(bar(Q8 ? B_QFULL : B_RFULL), 0, never, kWaitNs);
      mbar_wait(bar(Q8 ? B_QFULL + 3 : B_VFULL), 0, never, kWaitNs);
    }
    if (err && tid == 0) flag(p.status, err);
    if (rvalid) {
      p.ws_ml[2 * si] = err ? NAN : -INFINITY;
      p.ws_ml[2 * si + 1] = err ? NAN : 0.f;
    }
    return;
  }

  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_s), C::TMEM_COLS);
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


  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = Q8 ? 1 : 0;
      if (direct) {
        issued = 0;  // nothing to copy: the dequantising warps load the rows
      } else if (Q8) {
        // L2 prefetches of tiles 1.. once tile 0 (whose HBM reads they would
        // otherwise compete with) has landed.
        if (ntiles > 1 && mbar_wait(bar(B_QFULL), 0, abort_p, kWaitNs)) {
          for (int i = 1; i < min(kPrefetch, ntiles); ++i) {
            prefetch_q8(i, 0);
            prefetch_q8(i, 1);
          }
        }
        for (int i = 1; i < ntiles && !*abort_p; ++i) {
          // The buffers of tiles qfirst.. hold the Q staging until the
          // softmax warps have put Q into TMEM.
          if (i == qfirst && !mbar_wait(bar(B_QREADY), 0, abort_p, kWaitNs)) {
            fail();
            break;
          }
          const int jb = i % C::NB16;
          const uint32_t par = ((i / C::NB16) & 1) ^ 1;
          bool ok = mbar_wait(bar(B_QEMPTY + jb), par, abort_p, kWaitNs);
          if (ok) issue_q8(i, 0);
          ok = ok && mbar_wait(bar(B_QEMPTY + 3 + jb), par, abort_p, kWaitNs);
          if (ok) issue_q8(i, 1);
          if (!ok) {
            fail();
            break;
          }
          issued = i + 1;
        }
      } else {
        issued = early ? 1 : 0;
        for (int i = issued; i < ntiles; ++i) {
          const int st = i % C::NST;
          // The stages of tiles qfirst.. hold the Q staging until the
          // softmax warps have put Q into TMEM.
          if ((i == qfirst && !mbar_wait(bar(B_QREADY), 0, abort_p, kWaitNs)) ||
              !mbar_wait(bar(B_REMPTY + st), ((i / C::NST) & 1) ^ 1, abort_p, kWaitNs)) {
            fail();
            break;
          }
          const int t0 = slo + i * kNT;
          const int end16 = min(t0 + kNT, (shi + kPage - 1) / kPage * kPage);
          const int nload = end16 - t0;
          if (!PAGED) {
            issue_bf16(i);
          } else {
            const uint32_t bytes = (uint32_t)(nload * D * 2);
            mbar_arrive_expect_tx(bar(B_RFULL + st), bytes);
            mbar_arrive_expect_tx(bar(B_VFULL + st), bytes);
            for (int pg = 0; pg < nload / kPage; ++pg) {
              const int blk = p.block_table[(long long)s * p.max_blocks + t0 / kPage + pg];
              for (int db = 0; db < C::DBLK; ++db) {
                const uint32_t off = db * kNT * 128 + pg * kPage * 128;
                tma_load_4d(smem_u32(kst(st) + off), &tmK, db * 64, 0, kvh, blk,
                            bar(B_RFULL + st), pol);
                tma_load_4d(smem_u32(vst(st) + off), &tmV, db * 64, 0, kvh, blk,
                            bar(B_VFULL + st), pol);
              }
            }
          }
          issued = i + 1;
        }
      }
      // Drain: make sure no copy of ours is still landing in shared memory.
      if (!direct && *abort_p) {
        int dummy = 0;
        volatile int* never = &dummy;
        const int nslot = Q8 ? C::NB16 : C::NST;
        for (int i = max(0, issued - nslot); i < issued; ++i) {
          const int st = i % nslot;
          const uint32_t par = (i / nslot) & 1;
          mbar_wait(bar((Q8 ? B_QFULL : B_RFULL) + st), par, never, kWaitNs);
          mbar_wait(bar((Q8 ? B_QFULL + 3 : B_VFULL) + st), par, never, kWaitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ S issuer
    // bf16: S(i) = Q K_i^T into S buffer i & 1, once K_i is ready and the
    // P.V that last read that buffer (tile i - 2, whose P it held) has
    // completed.  Q8: one 128-column S buffer; per K step one MMA over the
    // 128 B rows [K_i hi; K_i lo], so columns 0..63 get Q.K_hi and 64..127
    // Q.K_lo (the softmax adds them: hi + lo = d*q exactly), once K_i is
    // ready and the softmax has read S(i - 1).
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_f16(kM, Q8 ? 2 * kNT : kNT, !Q8, false);
      bool ok = mbar_wait(bar(B_QREADY), 0, abort_p, kWaitNs);
      bool any = false;
      for (int i = 0; i < ntiles && ok; ++i) {
        const int b = i & 1;
        uint32_t kaddr;
        if (Q8) {
          const int jb = i % C::NB16;
          ok = mbar_wait(bar(B_QREADY8 + jb), (i / C::NB16) & 1, abort_p, kWaitNs);
          kaddr = smem_u32(q8buf(0, jb));
          if (ok && i >= 1) ok = mbar_wait(bar(B_SCONS), (i - 1) & 1, abort_p, kWaitNs);
        } else {
          const int st = i % C::NST;
          ok = mbar_wait(bar(B_RFULL + st), (i / C::NST) & 1, abort_p, kWaitNs);
          kaddr = smem_u32(kst(st));
          if (ok && i >= 2)
            ok = mbar_wait(bar(B_SFREE + b), ((i - 2) >> 1) & 1, abort_p, kWaitNs);
        }
        if (!ok) break;
        tc_fence_after();
        const uint64_t kd0 = sdesc_sw128(kaddr, 16, 1024);
        // Column blocks of 64 d: bf16 K tiles kNT rows apart, Q8 K tiles
        // 2 kNT rows (hi then lo).
        constexpr int CB = (Q8 ? 2 : 1) * kNT * 128;
        const uint32_t scol = tm + C::COL_S0 + (Q8 ? 0 : b * kNT);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t step = (uint64_t)(((kk >> 2) * CB + (kk & 3) * 32) >> 4);
          mma_ts(scol, tm + C::COL_Q + kk * 8, kd0 + step, ID_QK, kk > 0 ? 1u : 0u);
        }
        any = true;
        mma_commit(bar(B_SFULL + (Q8 ? 0 : b)));
        if (Q8) mma_commit(bar(B_QEMPTY + i % C::NB16));
      }
      if (!ok) fail();
      if (any) {
        // Wait (bounded, regardless of abort) until these MMAs have finished.
        int dummy = 0;
        volatile int* never = &dummy;
        mma_commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, never, kWaitNs);
      }
    }
  } else if (warp == C::PV_WARP) {
    // ------------------------------------------------------------ P.V issuer
    // O += P_t V_t once the softmax has written P_t (bf16: into S buffer
    // t & 1 in TMEM; Q8: into the P tile in shared memory) and V_t is
    // ready; its completion frees that S buffer / the P tile and V_t's
    // buffer.
    if (lane == 0) {
      constexpr uint32_t ID_PV = idesc_f16(kM, D, !Q8, true);
      bool ok = true, any = false;
      for (int t = 0; t < ntiles && ok; ++t) {
        const int bt = t & 1;
        ok = mbar_wait(bar(B_PFULL + bt), (t >> 1) & 1, abort_p, kWaitNs);
        uint32_t vaddr = 0;
        if (ok && Q8) {
          const int jb = t % C::NB16;
          ok = mbar_wait(bar(B_QREADY8 + 3 + jb), (t / C::NB16) & 1, abort_p, kWaitNs);
          vaddr = smem_u32(q8buf(1, jb));
        } else if (ok) {
          const int st = t % C::NST;
          ok = mbar_wait(bar(B_VREADY + st), (t / C::NST) & 1, abort_p, kWaitNs);
          vaddr = smem_u32(vst(st));
        }
        if (!ok) break;
        tc_fence_after();
        const uint32_t scol = tm + C::COL_S0 + bt * kNT;
        // Descriptor of the tile start; each 16-token K step adds 2048 bytes
        // to its start-address field (no carry: shared addresses < 256 KB).
        const uint64_t vd0 = sdesc_sw128(vaddr, kNT * 128, 1024);
        // Q8: P tile (K-major, one 128-byte row of 64 tokens per query
        // row); a 16-token K step is 32 bytes along the row.
        const uint64_t pd0 = sdesc_sw128(smem_u32(q8p()), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kNT / 16; ++kk) {
          const uint64_t vd = vd0 + (uint64_t)((kk * 2048) >> 4);
          if (Q8) {
            mma_ss(tm + C::COL_O, pd0 + (uint64_t)((kk * 32) >> 4), vd, ID_PV,
                   (t > 0 || kk > 0) ? 1u : 0u);
          } else {
            mma_ts(tm + C::COL_O, scol + kk * 8, vd, ID_PV, (t > 0 || kk > 0) ? 1u : 0u);
            mma_ts(tm + C::COL_O, scol + kNT / 2 + kk * 8, vd, ID_PV, 1u);
          }
        }
        any = true;
        mma_commit(bar(Q8 ? B_PFREE : B_SFREE + bt));
        if (Q8) mma_commit(bar(B_QEMPTY + 3 + t % C::NB16));
        else mma_commit(bar(B_REMPTY + t % C::NST));
      }
      if (ok) mma_commit(bar(B_OFINAL));
      if (!ok) fail();
      if (any) {
        int dummy = 0;
        volatile int* never = &dummy;
        mma_commit(bar(B_DRAIN + 1));
        mbar_wait(bar(B_DRAIN + 1), 0, never, kWaitNs);
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ softmax
    // Warps 2..9: quad = warp & 3 selects the TMEM lane quadrant (32 rows),
    // half = (warp - 2) >> 2 selects which 32 of the tile's 64 columns this
    // thread scores; the two halves of a row exchange their maxima through
    // shared memory once per tile (named barrier 5 + quad: just the two
    // warps of the quadrant).
    const int half = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const bool warp_live = __any_sync(0xffffffffu, rvalid);
    float c_r = p.scale_log2;
    {
      // Q row -> TMEM (16-bit pairs); this half loads elements
      // [half*D/2, (half+1)*D/2) with all loads in flight and writes TMEM
      // columns [half*D/4, (half+1)*D/4).  Q8 path: fp16 after a 2^-e
      // rescale of the whole row (exact), the 2^e folded into the score
      // multiplier; the two halves exchange their |q| maxima.
      constexpr int NQ = D / 16;  // uint4 per half row
      // From the shared staging copy (rows padded so the lanes of a warp
      // hit distinct bank groups).
      const uint4* qsrc = reinterpret_cast<const uint4*>(qstage + r * kQRow + half * D);
      float qscale = 1.f;
      if (Q8) {
        float amax = 0.f;
        if (rvalid) {
#pragma unroll 4
          for (int k = 0; k < NQ; ++k) {
            const uint4 q4 = qsrc[k];
            const uint32_t w[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              amax = fmaxf(amax, fabsf(__uint_as_float(w[m] << 16)));
              amax = fmaxf(amax, fabsf(__uint_as_float(w[m] & 0xFFFF0000u)));
            }
          }
        }
        red_q[half][r] = amax;
        named_barrier_sync(5 + quad, 64);  // the row's two halves
        amax = fmaxf(amax, red_q[half ^ 1][r]);
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        qscale = ldexpf(1.f, -e);
        c_r = ldexpf(p.scale_log2, e);
      }
#pragma unroll 1
      for (int c = 0; c < NQ / 4; ++c) {
        uint4 q4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) q4[k] = rvalid ? qsrc[4 * c + k] : make_uint4(0u, 0u, 0u, 0u);
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t w[4] = {q4[k].x, q4[k].y, q4[k].z, q4[k].w};
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if (Q8) {
              float a = __uint_as_float(w[m] << 16) * qscale;
              float b2 = __uint_as_float(w[m] & 0xFFFF0000u) * qscale;
              __half2 hv = __floats2half2_rn(a, b2);
              pk[4 * k + m] = *reinterpret_cast<uint32_t*>(&hv);
            } else {
              pk[4 * k + m] = w[m];
            }
          }
        }
        tmem_st16(tm + lane_base + C::COL_Q + half * (D / 4) + 16 * c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_QREADY));
    }

    float m_use = -INFINITY, l_run = 0.f;
    bool ok = true;
    // A failed wait does not leave the loop: every iteration has exactly one
    // named barrier shared with the partner warp, so a failing warp keeps
    // arriving there (skipping the work) until the loop ends.
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL + (Q8 ? 0 : b)),
                                                   Q8 ? (i & 1) : ((i >> 1) & 1), abort_p, kWaitNs)))
        ok = false;
      tc_fence_after();
      const uint32_t scol = tm + lane_base + C::COL_S0 + (Q8 ? 0 : b * kNT);
      const int t0 = slo + i * kNT + 32 * half;  // first token of this half
      const bool plain = (slo + i * kNT + kNT <= ctx) && (slo + i * kNT + kNT <= shi);
      float sv[32];
      float mx = -INFINITY;
      if (ok && warp_live) {
        uint32_t sr[32];
        tmem_ld32(scol + 32 * half, sr);
        if (Q8) {
          // S = Q.K_hi + Q.K_lo: the lo columns sit kNT further on.
          uint32_t sl[32];
          tmem_ld32(scol + kNT + 32 * half, sl);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            sr[c] = __float_as_uint(__uint_as_float(sr[c]) + __uint_as_float(sl[c]));
        } else {
          tmem_wait_ld();
        }
        if (plain && rvalid) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = __uint_as_float(sr[c]);
            mx = fmaxf(mx, sv[c]);
          }
        } else {
          const unsigned vis = rvalid ? visible_bits(kind, anc, j, ctx, shi, t0) : 0u;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = (vis >> c) & 1u ? __uint_as_float(sr[c]) : -INFINITY;
            mx = fmaxf(mx, sv[c]);
          }
        }
      }
      if (Q8) {
        // S(i) is in registers: the S issuer may overwrite the buffer.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SCONS));
      }
      // Row maximum over both halves (raw scores; c_r > 0).
      red_max[b][half][r] = mx;
      named_barrier_sync(5 + quad, 64);  // the row's two halves
      mx = fmaxf(mx, red_max[b][half ^ 1][r]);
      const float mt = mx * c_r;
      const bool need = rvalid && (m_use != -INFINITY) && (mt > m_use + 8.f);
      const float m_new = (m_use == -INFINITY || need) ? mt : m_use;
      if (ok && __any_sync(0xffffffffu, need) &&
          !__all_sync(0xffffffffu,
                      Q8 ? mbar_wait(bar(B_PFREE), (i - 1) & 1, abort_p, kWaitNs)
                         : mbar_wait(bar(B_SFREE + ((i - 1) & 1)), ((i - 1) >> 1) & 1, abort_p,
                                     kWaitNs)))
        ok = false;
      if (ok && __any_sync(0xffffffffu, need)) {
        // Rescale this half of the warp's O rows once the previous P.V landed.
        tc_fence_after();
        const float f = need ? exp2f(m_use - m_new) : 1.f;
#pragma unroll 1
        for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 16) {
          uint32_t o[16];
          tmem_ld16(tm + lane_base + C::COL_O + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * f);
          tmem_st16(tm + lane_base + C::COL_O + c0, o);
        }
        tmem_wait_st();
        l_run *= f;
      }
      m_use = m_new;
      if (ok && warp_live) {
        uint32_t ph[16], pl[16];
        float lsum = 0.f;
        // A masked score (-inf) gives 2^-inf = 0.  m_use is finite once any
        // score of the row was visible; while none was, every score here is
        // masked and the 0 offset keeps -inf * c_r + offset at -inf.
        const float mneg = m_use == -INFINITY ? 0.f : -m_use;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float a = ex2_approx(fmaf(sv[2 * c], c_r, mneg));
          const float bb = ex2_approx(fmaf(sv[2 * c + 1], c_r, mneg));
          lsum += a + bb;
          pack_p<Q8>(a, bb, ph[c], pl[c]);
        }
        if (rvalid) l_run += lsum;
        if (Q8) {
          // P(i) into the P tile once the P.V of tile i - 1 has read it:
          // this row's 32 tokens are chunks 4 half .. 4 half + 3 of its
          // 128-byte row.
          if (i >= 1 && !__all_sync(0xffffffffu, mbar_wait(bar(B_PFREE), (i - 1) & 1, abort_p,
                                                           kWaitNs)))
            ok = false;
          if (ok) {
            unsigned char* prow = q8p();
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<uint4*>(prow + sw128_off(r, 4 * half + c)) =
                  make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
          }
        } else {
          tmem_st16(scol + 16 * half, ph);
          tmem_st16(scol + kNT / 2 + 16 * half, pl);
          tmem_wait_st();
        }
      }
      if (Q8) fence_proxy_async_smem();  // P tile writes -> the MMA's reads
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL + b));
    }
    // Epilogue: the last P.V, then (m, l, O) into the slot; l adds the two
    // halves in fixed order.
    if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_OFINAL), 0, abort_p, kWaitNs))) ok = false;
    if (!ok && lane == 0) fail();
    tc_fence_after();
    if (half == 1) red_l[r] = l_run;
    named_barrier_sync(5 + quad, 64);  // the row's two halves
    const bool bad = __any_sync(0xffffffffu, *abort_p != 0);
    if (rvalid && half == 0) {
      p.ws_ml[2 * si] = bad ? NAN : m_use;
      p.ws_ml[2 * si + 1] = bad ? NAN : l_run + red_l[r];
    }
    // O rows go through shared memory (the tile buffers are idle now; rows
    // padded by 16 bytes so a warp's stores hit distinct bank groups) and
    // leave row by row with coalesced warp-wide stores.
    constexpr int kORow = D * 4 + 16;
    if (!bad && warp_live) {
#pragma unroll 1
      for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 32) {
        uint32_t o[32];
        tmem_ld32(tm + lane_base + C::COL_O + c0, o);
        tmem_wait_ld();
        if (rvalid) {
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<uint4*>(sm + r * kORow + (c0 + c) * 4) =
                make_uint4(o[c], o[c + 1], o[c + 2], o[c + 3]);
        }
      }
    }
    named_barrier_sync(1, 256);
    if (!bad) {
      // Warp w copies rows w - 2, w + 6, ... (eight warps share the rows),
      // each row with whole-warp 16-byte stores (coalesced 512-byte runs).
      const int nrows_blk = min(kM, R - rb * kM);
      for (int rr = warp - 2; rr < nrows_blk; rr += 8) {
        const int rs2 = rb * kM + rr;
        const long long si2 = slot_index(p, slot, row0 + rs2 / G, kvh * G + rs2 % G);
        const uint4* srow = reinterpret_cast<const uint4*>(sm + rr * kORow);
        uint4* grow4 = reinterpret_cast<uint4*>(p.ws_acc + si2 * D);
#pragma unroll
        for (int c = lane; c < D / 4; c += 32) grow4[c] = srow[c];
      }
    }
  } else {
    // ------------------------------------------------------------ dequant / fix-up
    if (direct && dq_slot(warp) >= 0) {
      // Paged Q8: the K and V dequantisation groups (dq_slot) each convert
      // their tensor's tiles at their own pace (warp 18 is idle, 13 issues
      // the P.V MMAs).  Per tile: load the raw half-row from global memory, wait
      // until the tile buffer is free (the MMA that read its previous tile
      // has completed; tiles from qfirst on also wait for Q to have left
      // the staging area), convert, store, release.
      const int dq = dq_slot(warp);
      const int grp = dq >> 2;  // 0 = K, 1 = V
      const int gtid = (dq & 3) * 32 + lane;
      const int t = gtid & 63, hf = gtid >> 6;
      const unsigned char* src = reinterpret_cast<const unsigned char*>(grp ? p.v : p.k);
      const unsigned char* dsrc = reinterpret_cast<const unsigned char*>(grp ? p.dv : p.dk);
      // Block-table lookups are issued a tile ahead of their use, so that
      // neither a row's address nor an L2 prefetch waits on one.
      auto row_blk = [&](int i) {
        const int tok = slo + i * kNT + t;
        return tok < shi && !(scratch && tok >= ctx)
                   ? p.block_table[(long long)s * p.max_blocks + tok / kPage]
                   : 0;
      };
      // L2 prefetch of page pg of tile k (pages holding cache tokens only;
      // their blocks were checked in the prologue): the block, then the copy.
      const int cend = scratch ? min(shi, ctx) : shi;
      auto pf_blk = [&](int k, int pg) {
        const int tp = slo + k * kNT + pg * kPage;
        return k < ntiles && tp < cend ? p.block_table[(long long)s * p.max_blocks + tp / kPage] : -1;
      };
      auto pf_issue = [&](int blk) {
        if (blk >= 0) bulk_prefetch_l2(src + ((long long)blk * p.KVH + kvh) * kPage * C::RB, kPage * C::RB);
      };
      // Lanes of the group's first warp keep its tensor kPrefetch tiles
      // ahead in L2, one page each: tiles 1..kPrefetch (16 lanes) before the
      // first conversion, then tile i + kPrefetch (4 lanes) after converting
      // tile i.
      const bool pf_warp = (dq & 3) == 0;
      static_assert(kNT == 4 * kPage && 4 * kPrefetch <= 32, "prefetch lanes");
      if (pf_warp && lane < 4 * kPrefetch) pf_issue(pf_blk(1 + lane / 4, lane % 4));
      int blk_next = row_blk(0);
      // A failed wait does not leave the loop (no named barrier here, but
      // the stores must stay out of buffers an MMA may still read).
      bool ok = true;
      for (int i = 0; i < ntiles; ++i) {
        const int jb = i % C::NB16;
        const int t0 = slo + i * kNT;
        const int tok = t0 + t;
        const bool live = ok && tok < shi;
        const bool draft = scratch && tok >= ctx;  // from the tree scratch KV
        const int blk = blk_next;
        const unsigned char* row =
            draft ? dsrc + scratch_row(p, row0, kvh, tok - ctx) * C::RB
                  : src + (((long long)blk * p.KVH + kvh) * kPage + tok % kPage) * C::RB;
        DqRaw<D> raw;
        dq_load<D>(raw, row, hf, live);
        if (i + 1 < ntiles) blk_next = row_blk(i + 1);
        const int pfb = pf_warp && lane < 4 && i >= 1 ? pf_blk(i + kPrefetch, lane) : -1;
        if (ok && !__all_sync(0xffffffffu,
                              mbar_wait(bar(B_QEMPTY + 3 * grp + jb), ((i / C::NB16) & 1) ^ 1,
                                        abort_p, kWaitNs) &&
                                  (i < qfirst || mbar_wait(bar(B_QREADY), 0, abort_p, kWaitNs)))) {
          ok = false;
          if (lane == 0) fail();
        }
        if (!ok) continue;
        dq_convert<D>(raw, q8buf(grp, jb), grp == 0 ? q8lo(jb) : nullptr, t, hf, live);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_QREADY8 + 3 * grp + jb));
        pf_issue(pfb);
      }
    } else if (Q8 && dq_slot(warp) >= 0) {
      // The K and V dequantisation groups (dq_slot) each convert their
      // tensor's tiles at their own pace, in place in the tile buffers (warp
      // 18 is idle, 13 issues the P.V MMAs).
      const int dq = dq_slot(warp);
      const int grp = dq >> 2;  // 0 = K, 1 = V
      const int gtid = (dq & 3) * 32 + lane;
      // A failed wait does not leave the loop: each iteration has one named
      // barrier shared by the group's four warps, so a failing warp keeps
      // arriving there (skipping the work) until the loop ends.
      bool ok = true;
      for (int i = 0; i < ntiles; ++i) {
        const int jb = i % C::NB16;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_QFULL + 3 * grp + jb),
                                                     (i / C::NB16) & 1, abort_p, kWaitNs))) {
          ok = false;
          if (lane == 0) fail();
        }
        dequant_inplace<D>(q8buf(grp, jb), grp == 0 ? q8lo(jb) : nullptr, shi - (slo + i * kNT),
                           gtid, 3 + grp, ok);
        if (ok) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_QREADY8 + 3 * grp + jb));
        }
      }
    } else if (!Q8 && warp == 10) {
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % C::NST;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_VFULL + st), (i / C::NST) & 1, abort_p, kWaitNs))) {
          if (lane == 0) fail();
          break;
        }
        const int valid = shi - (slo + i * kNT);
        if (valid < kNT) {
          const int rows = kNT - valid;
          const int chunks = C::DBLK * rows * 8;  // 16-byte chunks to clear
          for (int u = lane; u < chunks; u += 32) {
            const int db = u / (rows * 8);
            const int rr = valid + (u / 8) % rows;
            *reinterpret_cast<uint4*>(vst(st) + db * kNT * 128 + rr * 128 + (u & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_VREADY + st));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tm, C::TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps for the bf16 cache and the launch.

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)ptr;
  }
  return fn;
}

// Tiled map over a bf16 cache: contiguous [plane][capacity][D] with boxes
// {64, 64, 1}, or paged [block][KVH][16][D] with boxes {64, 16, 1, 1}.
static bool make_map(CUtensorMap* map, const Params& p, const void* base) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t D = (cuuint64_t)p.D;
  CUresult r;
  if (p.page_size == 0) {
    cuuint64_t dims[3] = {D, (cuuint64_t)p.capacity, (cuuint64_t)p.num_seqs * p.KVH};
    cuuint64_t strides[2] = {D * 2, (cuuint64_t)p.capacity * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kNT, 1};
    cuuint32_t es[3] = {1, 1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[4] = {D, (cuuint64_t)kPage, (cuuint64_t)p.KVH, (cuuint64_t)p.num_blocks};
    cuuint64_t strides[3] = {D * 2, (cuuint64_t)kPage * D * 2, (cuuint64_t)p.KVH * kPage * D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)kPage, 1, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
           es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

template <int D, int KVT, bool PAGED>
static cudaError_t launch_umma_t(const Params& p, dim3 grid, cudaStream_t st) {
  using C = UCfg<D, KVT>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(umma_partial_kernel<D, KVT, PAGED>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (!C::kQ8) {
    if (!make_map(&mk, p, p.k) || !make_map(&mv, p, p.v)) return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, umma_partial_kernel<D, KVT, PAGED>, p, mk, mv);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int umma_threads(int D, int kv_dtype) {
  (void)D;
  return kv_dtype == VA_Q8_0 ? UCfg<256, VA_Q8_0>::THREADS : UCfg<256, VA_BF16>::THREADS;
}

int umma_smem_bytes(int D, int kv_dtype) {
#define VA_U_SMEM(DD, KT) \
  if (D == DD && kv_dtype == KT) return UCfg<DD, KT>::SMEM;
  VA_U_SMEM(64, VA_BF16) VA_U_SMEM(64, VA_Q8_0) VA_U_SMEM(128, VA_BF16)
  VA_U_SMEM(128, VA_Q8_0) VA_U_SMEM(256, VA_BF16) VA_U_SMEM(256, VA_Q8_0)
#undef VA_U_SMEM
  return 0;
}

cudaError_t launch_umma_partial(const Params& p, dim3 grid, cudaStream_t st) {
#define VA_U_BF16(DD)                                                                     \
  if (p.D == DD && p.kv_dtype == VA_BF16)                                                 \
    return p.page_size != 0 ? launch_umma_t<DD, VA_BF16, true>(p, grid, st)              \
                            : launch_umma_t<DD, VA_BF16, false>(p, grid, st);
#define VA_U_Q8(DD)                                                                       \
  if (p.D == DD && p.kv_dtype == VA_Q8_0)                                                 \
    return p.page_size != 0 ? launch_umma_t<DD, VA_Q8_0, true>(p, grid, st)              \
                            : launch_umma_t<DD, VA_Q8_0, false>(p, grid, st);
  VA_U_BF16(64) VA_U_Q8(64) VA_U_BF16(128) VA_U_Q8(128) VA_U_BF16(256) VA_U_Q8(256)
#undef VA_U_BF16
#undef VA_U_Q8
  return cudaErrorInvalidValue;
}

}  // namespace va
