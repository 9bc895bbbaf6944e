// Tensor-core split-KV partial kernel (tcgen05 + TMEM + TMA), sm_103a.
//
// One CTA owns (sequence, KV head, split, sub-chunk) and ALL query rows of
// that KV head (n rows x G heads <= 128), so every K/V byte of its token
// range is read from HBM exactly once for every row it serves (hipfire PR
// #695, alpineQ comments: one block reuses each Q8 K/V fetch across several
// verifier rows; here across all of them).  Per 64-token tile:
//
//   S = Q K^T      tcgen05.mma, A = Q (TMEM), B = K tile (smem, K-major)
//   softmax        4 warps, one TMEM lane (= query row) per thread; masks;
//                  online (m, l) in log2 units; P written back over S
//   O += P V       tcgen05.mma, A = P (TMEM), B = V tile (smem, MN-major)
//
// O (fp32, 128 lanes x D columns) lives in TMEM for the CTA's whole range.
// At the end each row's (m, l, O) goes to its partial slot; the merge
// kernel combines slots (hipfire PR #817 "FA2 split-KV", sections "Summary"
// and "Performance").
//
// Caches:
//   Q8_0: raw 34-byte blocks arrive by 1-D bulk TMA into a staging ring;
//     8 warps dequantise them to fp16 (one rounding of d*q) straight into
//     the 128-byte-swizzled MMA layout, zero-filling tokens past the range.
//     Q is converted to fp16 after a per-row power-of-two rescale (exact),
//     and the scale folds into the score multiplier.  P is fp16.
//   bf16: tiled TMA loads place K/V tiles directly in the MMA layout; one
//     warp zeroes V rows past the range of a ragged tile.  P is split into
//     bf16 hi + lo halves (two MMAs) so P keeps 16 significant bits.
//
// Warp roles: 0 = TMA producer, 1 = TMEM owner + MMA issuer, 2..9 =
// softmax/epilogue (two warps per TMEM lane quadrant, one per half of the
// tile's columns), 10.. = Q8 dequant (4 warps for K, 4 for V) or bf16 V
// fix-up (1 warp).
// Every wait is bounded (VA_DEV_TIMEOUT); on a timeout the CTA drains its
// own copies and MMAs, frees TMEM and writes NaN partials.
#include <string.h>

#include "va_common.cuh"
#include "va_sm100.cuh"

namespace va {
using namespace sm100;

constexpr int kNT = 64;      // tokens per tile
constexpr int kM = 128;      // MMA rows (query rows per CTA)
constexpr uint64_t kWaitNs = 2000000000ull;

template <int D, int KVT>
struct UCfg {
  static constexpr bool kQ8 = (KVT == VA_Q8_0);
  static constexpr int RB = kQ8 ? D / 32 * 34 : D * 2;  // global bytes per token row
  static constexpr int NB = D / 32;                      // Q8 blocks per row
  static constexpr int DBLK = D / 64;                    // 64-element column blocks
  static constexpr int TILE = kNT * D * 2;               // one 16-bit tile in smem
  static constexpr int RAW_HALF = kNT * RB;              // raw K (or V) bytes of a tile
  static constexpr int NRH = (D == 256) ? 4 : (D == 128 ? 8 : 16);  // Q8 raw half-slots
  static constexpr int NST = (D == 256) ? 3 : (D == 128 ? 6 : 8);  // bf16 K+V stages
  static constexpr int COL_O = 0;
  static constexpr int COL_S0 = D;
  static constexpr int COL_Q = D + 2 * kNT;
  static constexpr int TMEM_COLS = (COL_Q + D / 2 <= 256) ? 256 : 512;
  static constexpr int DQ_WARPS = kQ8 ? 8 : 1;
  static constexpr int THREADS = (10 + DQ_WARPS) * 32;
  static constexpr int MAXREG = (65536 / THREADS) / 8 * 8 > 255 ? 255 : (65536 / THREADS) / 8 * 8;
  static constexpr int SMEM_Q8 = 4 * TILE + NRH * RAW_HALF;
  static constexpr int SMEM_BF16 = NST * 2 * TILE;
  static constexpr int SMEM = (kQ8 ? SMEM_Q8 : SMEM_BF16) + 1024 + 64;
};

// Barrier slots in static shared memory.
enum {
  B_SFULL = 0,    // [2]
  B_PFULL = 2,    // [2]
  B_PVDONE = 4,
  B_QREADY = 5,
  B_DRAIN = 6,
  B_OFINAL = 7,   // the last P.V has completed
  B_KREADY = 8,   // Q8: [2]
  B_KEMPTY = 10,  // Q8: [2]
  B_VREADY = 12,  // Q8: [2]; bf16: [NST]
  B_VEMPTY = 20,  // Q8: [2]
  B_RFULL = 22,   // Q8 raw half-slots: [NRH]; bf16 K full: [NST]
  B_REMPTY = 38,  // Q8 raw half-slots: [NRH]; bf16 stage empty: [NST]
  B_VFULL = 54,   // bf16 V full: [NST]
  B_COUNT = 62
};

// Byte offset of element (row, col) inside one 128-byte-swizzled column
// block whose rows are 128 bytes apart (col in 16-bit elements, < 64).
__device__ __forceinline__ uint32_t sw128_off(int row, int chunk16) {
  return (uint32_t)(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// Dequantise a tile of Q8_0 rows (raw, rows RB bytes apart) into the fp16
// MMA layout at dst; tokens >= valid become zeros.  128 threads; each takes
// its 34-byte blocks two at a time with both blocks' shared-memory loads in
// flight.  Eight consecutive threads take eight consecutive tokens of one
// block, so their 16-byte stores land in distinct bank groups.
template <int D>
__device__ __forceinline__ void dequant_tile(const unsigned char* raw, unsigned char* dst,
                                             int valid, int tid) {
  constexpr int NB = D / 32;
  constexpr int RB = NB * 34;
  constexpr int ITEMS = kNT * NB;
  constexpr int NTHR = 128;
#pragma unroll 1
  for (int u0 = tid; u0 < ITEMS; u0 += 2 * NTHR) {
    uint32_t wd[2][9];
    int tt[2], bq[2];
    bool live[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int u = u0 + k * NTHR;
      tt[k] = (u & 7) + 8 * (u / (8 * NB));
      bq[k] = (u >> 3) % NB;
      live[k] = u < ITEMS;
      if (live[k] && tt[k] < valid) {
        const int off = tt[k] * RB + bq[k] * 34;
        const uint32_t* w = reinterpret_cast<const uint32_t*>(raw + (off & ~3));
#pragma unroll
        for (int q = 0; q < 9; ++q) wd[k][q] = w[q];
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      if (!live[k]) continue;
      const int t = tt[k], b = bq[k];
      unsigned char* drow = dst + (b >> 1) * (kNT * 128);
      const int c0 = (b & 1) * 4;
      uint4 out[4];
      if (t < valid) {
        uint32_t sbits, code[8];
        if (b & 1) {  // block starts 2 bytes past a word boundary
          sbits = wd[k][0] >> 16;
#pragma unroll
          for (int q = 0; q < 8; ++q) code[q] = wd[k][q + 1];
        } else {
          sbits = wd[k][0] & 0xFFFFu;
#pragma unroll
          for (int q = 0; q < 8; ++q) code[q] = __funnelshift_r(wd[k][q], wd[k][q + 1], 16);
        }
        const __half2 d2 = __half2half2(__ushort_as_half((unsigned short)sbits));
        const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));  // 1152
        uint32_t hv[16];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t x = code[q] ^ 0x80808080u;  // bytes q + 128
          uint32_t lo = __byte_perm(x, 0x64646464u, 0x4140);
          uint32_t hi = __byte_perm(x, 0x64646464u, 0x4342);
          __half2 a = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&lo), bias), d2);
          __half2 c = __hmul2(__hsub2(*reinterpret_cast<__half2*>(&hi), bias), d2);
          hv[2 * q] = *reinterpret_cast<uint32_t*>(&a);
          hv[2 * q + 1] = *reinterpret_cast<uint32_t*>(&c);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c)
          out[c] = make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) out[c] = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(drow + sw128_off(t, c0 + c)) = out[c];
    }
  }
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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

template <int D, int KVT>
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
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rb = blockIdx.x % p.row_blocks;
  const int sp = blockIdx.x / p.row_blocks;
  const int split = sp / p.P, sub = sp % p.P, slot = sp;
  const int kvh = blockIdx.y, s = blockIdx.z;

  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  if (err & VA_DEV_BAD_ROWS) {
    if (tid == 0) flag(p.status, err);
    return;
  }
  const int G = p.G;
  const int R = n * G;
  if (rb * kM >= R) return;
  const int L = ctx + n;
  int lo, hi, slo, shi;
  split_range(L, p.S, split, &lo, &hi);
  sub_range(lo, hi, p.P, p.min_sub, sub, &slo, &shi);
  const int ntiles = (shi - slo + kNT - 1) / kNT;

  // Softmax-thread row identity.
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int rseq = rb * kM + r;
  const bool is_sm = (warp >= 2 && warp < 10);
  const bool rvalid = is_sm && rseq < R;
  const int j = rvalid ? rseq / G : 0;
  const int g = rvalid ? rseq % G : 0;
  const int kind = seq_kind_of(p, s);

  if (tid == 0) {
    err_s = 0;
    abort_s = 0;
  }
  __syncthreads();
  unsigned anc = 0;
  if (rvalid && !err) {
    bool bad = false;
    anc = row_mask(kind, p.parent + row0, j, &bad);
    if (bad) atomicOr(&err_s, (int)VA_DEV_BAD_PARENT);
  }
  if (!err && p.page_size != 0 && ntiles > 0) {
    const int pg0 = slo / kPage, pg1 = (shi + kPage - 1) / kPage;
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
    if (err && tid == 0) flag(p.status, err);
    if (rvalid) {
      p.ws_ml[2 * si] = err ? NAN : -INFINITY;
      p.ws_ml[2 * si + 1] = err ? NAN : 0.f;
    }
    return;
  }

  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (tid == 0) {
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_PFULL), 8);
    mbar_init(bar(B_PFULL + 1), 8);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_QREADY), 8);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_OFINAL), 1);
    if (Q8) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(bar(B_KREADY + i), C::DQ_WARPS / 2);
        mbar_init(bar(B_KEMPTY + i), 1);
        mbar_init(bar(B_VREADY + i), C::DQ_WARPS / 2);
        mbar_init(bar(B_VEMPTY + i), 1);
      }
      for (int i = 0; i < C::NRH; ++i) {
        mbar_init(bar(B_RFULL + i), 1);
        mbar_init(bar(B_REMPTY + i), C::DQ_WARPS / 2);
      }
    } else {
      for (int i = 0; i < C::NST; ++i) {
        mbar_init(bar(B_RFULL + i), 1);
        mbar_init(bar(B_VFULL + i), 1);
        mbar_init(bar(B_VREADY + i), 1);
        mbar_init(bar(B_REMPTY + i), 1);
      }
    }
    fence_barrier_init();
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

  // Q8: warps 2.. stage this CTA's Q rows in shared memory (the fp16 tile
  // buffers, unused until the first dequant) with every load in flight;
  // the softmax warps convert them into TMEM, then release the area.
  constexpr int kQRow = D * 2 + 16;
  if (Q8 && warp >= 2) {
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
      if (c < total) *reinterpret_cast<uint4*>(sm + (c / CPR) * kQRow + (c % CPR) * 16) = v[k];
    }
    named_barrier_sync(2, NTHR);
    if (warp >= 10) named_barrier_sync(2, NTHR);  // dequant warps wait for the release
  }

  // Shared-memory regions.
  unsigned char* k16 = sm;                      // Q8: 2 dequantised K tiles
  unsigned char* v16 = sm + 2 * C::TILE;        // Q8: 2 dequantised V tiles
  unsigned char* raw = sm + 4 * C::TILE;        // Q8: raw stages
  auto kst = [&](int st) { return sm + st * 2 * C::TILE; };            // bf16 K stage
  auto vst = [&](int st) { return sm + st * 2 * C::TILE + C::TILE; };  // bf16 V stage

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int issued = 0;
      if (Q8) {
        // Raw K_i and V_i go to their own half-slots (K, V, K, V, ...), each
        // freed as soon as its own dequantisation is done.
        for (int hh = 0; hh < 2 * ntiles; ++hh) {
          const int i = hh >> 1, slot = hh % C::NRH;
          if (!mbar_wait(bar(B_REMPTY + slot), ((hh / C::NRH) & 1) ^ 1, abort_p, kWaitNs)) {
            fail();
            break;
          }
          const int t0 = slo + i * kNT;
          const int end16 = min(t0 + kNT, (shi + kPage - 1) / kPage * kPage);
          const int nload = end16 - t0;  // multiple of 16
          const unsigned char* src = (const unsigned char*)((hh & 1) ? p.v : p.k);
          unsigned char* dst = raw + slot * C::RAW_HALF;
          mbar_arrive_expect_tx(bar(B_RFULL + slot), (uint32_t)(nload * C::RB));
          if (p.page_size == 0) {
            const long long rowi = ((long long)s * p.KVH + kvh) * p.capacity + t0;
            bulk_g2s(smem_u32(dst), src + rowi * C::RB, (uint32_t)(nload * C::RB),
                     bar(B_RFULL + slot), pol);
          } else {
            for (int pg = 0; pg < nload / kPage; ++pg) {
              const int blk = p.block_table[(long long)s * p.max_blocks + t0 / kPage + pg];
              const long long rowi = ((long long)blk * p.KVH + kvh) * kPage;
              bulk_g2s(smem_u32(dst + pg * kPage * C::RB), src + rowi * C::RB, kPage * C::RB,
                       bar(B_RFULL + slot), pol);
            }
          }
          issued = hh + 1;
        }
      } else {
        for (int i = 0; i < ntiles; ++i) {
          const int st = i % C::NST;
          if (!mbar_wait(bar(B_REMPTY + st), ((i / C::NST) & 1) ^ 1, abort_p, kWaitNs)) {
            fail();
            break;
          }
          const int t0 = slo + i * kNT;
          const int end16 = min(t0 + kNT, (shi + kPage - 1) / kPage * kPage);
          const int nload = end16 - t0;
          if (p.page_size == 0) {
            mbar_arrive_expect_tx(bar(B_RFULL + st), (uint32_t)C::TILE);
            mbar_arrive_expect_tx(bar(B_VFULL + st), (uint32_t)C::TILE);
            const int plane = s * p.KVH + kvh;
            for (int db = 0; db < C::DBLK; ++db) {
              tma_load_3d(smem_u32(kst(st) + db * kNT * 128), &tmK, db * 64, t0, plane,
                          bar(B_RFULL + st), pol);
              tma_load_3d(smem_u32(vst(st) + db * kNT * 128), &tmV, db * 64, t0, plane,
                          bar(B_VFULL + st), pol);
            }
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
      if (*abort_p) {
        int dummy = 0;
        volatile int* never = &dummy;
        const int nslot = Q8 ? C::NRH : C::NST;
        for (int i = max(0, issued - nslot); i < issued; ++i) {
          const int st = i % nslot;
          mbar_wait(bar(B_RFULL + st), (i / nslot) & 1, never, kWaitNs);
          if (!Q8) mbar_wait(bar(B_VFULL + st), (i / nslot) & 1, never, kWaitNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t ID_QK = idesc_f16(kM, kNT, !Q8, false);
      constexpr uint32_t ID_PV = idesc_f16(kM, D, !Q8, true);
      bool ok = mbar_wait(bar(B_QREADY), 0, abort_p, kWaitNs);
      bool any = false;
      auto issue_pv = [&](int t) -> bool {
        const int bt = t & 1;
        if (!mbar_wait(bar(B_PFULL + bt), (t >> 1) & 1, abort_p, kWaitNs)) return false;
        uint32_t vaddr;
        if (Q8) {
          if (!mbar_wait(bar(B_VREADY + bt), (t >> 1) & 1, abort_p, kWaitNs)) return false;
          vaddr = smem_u32(v16 + bt * C::TILE);
        } else {
          const int st = t % C::NST;
          if (!mbar_wait(bar(B_VREADY + st), (t / C::NST) & 1, abort_p, kWaitNs)) return false;
          vaddr = smem_u32(vst(st));
        }
        tc_fence_after();
        const uint32_t scol = tm + C::COL_S0 + bt * kNT;
        // Descriptor of the tile start; each 16-token K step adds 2048 bytes
        // to its start-address field (no carry: shared addresses < 256 KB).
        const uint64_t vd0 = sdesc_sw128(vaddr, kNT * 128, 1024);
#pragma unroll
        for (int kk = 0; kk < kNT / 16; ++kk) {
          const uint64_t vd = vd0 + (uint64_t)((kk * 2048) >> 4);
          mma_ts(tm + C::COL_O, scol + kk * 8, vd, ID_PV, (t > 0 || kk > 0) ? 1u : 0u);
          if (!Q8) mma_ts(tm + C::COL_O, scol + kNT / 2 + kk * 8, vd, ID_PV, 1u);
        }
        any = true;
        mma_commit(bar(B_PVDONE));
        if (Q8) mma_commit(bar(B_VEMPTY + bt));
        else mma_commit(bar(B_REMPTY + t % C::NST));
        return true;
      };
      if (ok) {
        tc_fence_after();
        for (int i = 0; i < ntiles && ok; ++i) {
          const int b = i & 1;
          uint32_t kaddr;
          if (Q8) {
            ok = mbar_wait(bar(B_KREADY + b), (i >> 1) & 1, abort_p, kWaitNs);
            kaddr = smem_u32(k16 + b * C::TILE);
          } else {
            const int st = i % C::NST;
            ok = mbar_wait(bar(B_RFULL + st), (i / C::NST) & 1, abort_p, kWaitNs);
            kaddr = smem_u32(kst(st));
          }
          if (!ok) break;
          tc_fence_after();
          const uint64_t kd0 = sdesc_sw128(kaddr, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t kd = kd0 + (uint64_t)(((kk >> 2) * (kNT * 128) + (kk & 3) * 32) >> 4);
            mma_ts(tm + C::COL_S0 + b * kNT, tm + C::COL_Q + kk * 8, kd, ID_QK,
                   kk > 0 ? 1u : 0u);
          }
          any = true;
          mma_commit(bar(B_SFULL + b));
          if (Q8) mma_commit(bar(B_KEMPTY + b));
          if (i >= 1) ok = issue_pv(i - 1);
        }
        if (ok) ok = issue_pv(ntiles - 1);
        if (ok) mma_commit(bar(B_OFINAL));
      }
      if (!ok) fail();
      if (any) {
        // Wait (bounded, regardless of abort) until our MMAs have finished.
        int dummy = 0;
        volatile int* never = &dummy;
        mma_commit(bar(B_DRAIN));
        mbar_wait(bar(B_DRAIN), 0, never, kWaitNs);
      }
    }
  } else if (warp < 10) {
    // ------------------------------------------------------------ softmax
    // Warps 2..9: quad = warp & 3 selects the TMEM lane quadrant (32 rows),
    // half = (warp - 2) >> 2 selects which 32 of the tile's 64 columns this
    // thread scores; the two halves of a row exchange their maxima through
    // shared memory once per tile.
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
      // Q8: from the shared staging copy (rows padded so the lanes of a warp
      // hit distinct bank groups); bf16: straight from global memory.
      const uint4* qsrc =
          Q8 ? reinterpret_cast<const uint4*>(sm + r * kQRow + half * D)
             : reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned short*>(p.q) +
                                              ((long long)grow * p.H + h) * D + half * (D / 2));
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
        named_barrier_sync(1, 256);
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
      if (Q8) named_barrier_sync(2, C::THREADS - 64);  // staging area free again
    }

    float m_use = -INFINITY, l_run = 0.f;
    bool ok = true;
    // A failed wait does not leave the loop: every iteration has exactly one
    // named barrier shared with the partner warp, so a failing warp keeps
    // arriving there (skipping the work) until the loop ends.
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      if (ok && !__all_sync(0xffffffffu, mbar_wait(bar(B_SFULL + b), (i >> 1) & 1, abort_p, kWaitNs)))
        ok = false;
      tc_fence_after();
      const uint32_t scol = tm + lane_base + C::COL_S0 + b * kNT;
      const int t0 = slo + i * kNT + 32 * half;  // first token of this half
      const bool plain = (slo + i * kNT + kNT <= ctx) && (slo + i * kNT + kNT <= shi);
      float sv[32];
      float mx = -INFINITY;
      if (ok && warp_live) {
        uint32_t sr[32];
        tmem_ld32(scol + 32 * half, sr);
        tmem_wait_ld();
        if (plain && rvalid) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = __uint_as_float(sr[c]);
            mx = fmaxf(mx, sv[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int t = t0 + c;
            const bool vis = rvalid && t < shi && (t < ctx || ((anc >> (t - ctx)) & 1u));
            sv[c] = vis ? __uint_as_float(sr[c]) : -INFINITY;
            mx = fmaxf(mx, sv[c]);
          }
        }
      }
      // Row maximum over both halves (raw scores; c_r > 0).
      red_max[b][half][r] = mx;
      named_barrier_sync(1, 256);
      mx = fmaxf(mx, red_max[b][half ^ 1][r]);
      const float mt = mx * c_r;
      const bool need = rvalid && (m_use != -INFINITY) && (mt > m_use + 8.f);
      const float m_new = (m_use == -INFINITY || need) ? mt : m_use;
      if (ok && __any_sync(0xffffffffu, need) &&
          !__all_sync(0xffffffffu, mbar_wait(bar(B_PVDONE), (i - 1) & 1, abort_p, kWaitNs)))
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
        const float mneg = -m_use;
        if (plain) {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float a = ex2_approx(fmaf(sv[2 * c], c_r, mneg));
            const float bb = ex2_approx(fmaf(sv[2 * c + 1], c_r, mneg));
            lsum += a + bb;
            pack_p<Q8>(a, bb, ph[c], pl[c]);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float a = sv[2 * c] == -INFINITY ? 0.f : ex2_approx(fmaf(sv[2 * c], c_r, mneg));
            const float bb =
                sv[2 * c + 1] == -INFINITY ? 0.f : ex2_approx(fmaf(sv[2 * c + 1], c_r, mneg));
            lsum += a + bb;
            pack_p<Q8>(a, bb, ph[c], pl[c]);
          }
        }
        if (rvalid) l_run += lsum;
        tmem_st16(scol + 16 * half, ph);
        if (!Q8) tmem_st16(scol + kNT / 2 + 16 * half, pl);
        tmem_wait_st();
      }
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
    named_barrier_sync(1, 256);
    const bool bad = __any_sync(0xffffffffu, *abort_p != 0);
    if (rvalid && half == 0) {
      p.ws_ml[2 * si] = bad ? NAN : m_use;
      p.ws_ml[2 * si + 1] = bad ? NAN : l_run + red_l[r];
    }
    if (!bad && warp_live) {
      float* dst = p.ws_acc + si * D;
#pragma unroll 1
      for (int c0 = half * (D / 2); c0 < (half + 1) * (D / 2); c0 += 16) {
        uint32_t o[16];
        tmem_ld16(tm + lane_base + C::COL_O + c0, o);
        tmem_wait_ld();
        if (rvalid) {
#pragma unroll
          for (int c = 0; c < 16; c += 4)
            *reinterpret_cast<float4*>(dst + c0 + c) =
                make_float4(__uint_as_float(o[c]), __uint_as_float(o[c + 1]),
                            __uint_as_float(o[c + 2]), __uint_as_float(o[c + 3]));
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dequant / fix-up
    if (Q8) {
      // Warps 10..13 dequantise K tiles, 14..17 V tiles, each group at its
      // own pace.
      const int grp = (warp - 10) >> 2;  // 0 = K, 1 = V
      const int gtid = ((warp - 10) & 3) * 32 + lane;
      unsigned char* out16 = grp ? v16 : k16;
      const int b_ready = grp ? B_VREADY : B_KREADY;
      const int b_empty = grp ? B_VEMPTY : B_KEMPTY;
      for (int i = 0; i < ntiles; ++i) {
        const int hh = 2 * i + grp, slot = hh % C::NRH, buf = i & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_RFULL + slot), (hh / C::NRH) & 1, abort_p, kWaitNs))) {
          if (lane == 0) fail();
          break;
        }
        if (!__all_sync(0xffffffffu, mbar_wait(bar(b_empty + buf), ((i >> 1) & 1) ^ 1, abort_p, kWaitNs))) {
          if (lane == 0) fail();
          break;
        }
        const int valid = shi - (slo + i * kNT);
        dequant_tile<D>(raw + slot * C::RAW_HALF, out16 + buf * C::TILE, valid, gtid);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(b_ready + buf));
          mbar_arrive(bar(B_REMPTY + slot));
        }
      }
    } else if (warp == 10) {
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

template <int D, int KVT>
static cudaError_t launch_umma_t(const Params& p, dim3 grid, cudaStream_t st) {
  using C = UCfg<D, KVT>;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(umma_partial_kernel<D, KVT>,
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
  umma_partial_kernel<D, KVT><<<grid, C::THREADS, C::SMEM, st>>>(p, mk, mv);
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
#define VA_U_CASE(DD, KT) \
  if (p.D == DD && p.kv_dtype == KT) return launch_umma_t<DD, KT>(p, grid, st);
  VA_U_CASE(64, VA_BF16) VA_U_CASE(64, VA_Q8_0) VA_U_CASE(128, VA_BF16)
  VA_U_CASE(128, VA_Q8_0) VA_U_CASE(256, VA_BF16) VA_U_CASE(256, VA_Q8_0)
#undef VA_U_CASE
  return cudaErrorInvalidValue;
}

}  // namespace va
