// Shared device-side definitions of the verify-attention kernels: launch
// parameters, the split rule, row masks, the KV gather and storage decoding.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "verify_attn.h"

namespace va {

constexpr int kPage = 16;
constexpr int kChunkAlign = 64;  // KV chunks are whole 64-token tiles
constexpr int kQ8Block = 32;
constexpr int kQ8BlockBytes = 34;
constexpr float kLn2 = 0.6931471805599453f;

// Everything a partial / merge / debug kernel needs, passed by value.
struct Params {
  int num_seqs, H, KVH, G, D;
  int total_rows, max_rows;
  int S, P, slots;        // logical splits, sub-chunks per split, S*P
  int min_sub;            // smallest sub-chunk (tokens) before a split is cut further
  int min_splits;         // the caller's split count: a sequence keeps at least this many chunks
  int mode;               // va_mode
  int kv_dtype, q_dtype;  // va_dtype
  float scale_log2;       // softmax scale * log2(e)
  const void* q;
  const int* cu_rows;
  const int* ctx_len;
  const int* parent;
  const unsigned char* seq_kind;
  const void* k;
  const void* v;
  const void* dk;         // tree scratch KV [total_rows][KVH][row], or null
  const void* dv;
  int page_size;
  long long capacity;
  const int* block_table;
  int max_blocks;
  int num_blocks;
  int row_bytes;          // bytes of one (token, KV head) row
  float* ws_acc;          // [slots][total_rows][H][D]
  float* ws_ml;           // [slots][total_rows][H][2]  (m in log2 units, l)
  float* o;               // [total_rows][H][D]
  float* lse;             // [total_rows][H]
  unsigned* status;
  int rows_per_block;     // query rows (j, g pairs) one partial CTA owns
  int row_blocks;         // ceil(max_rows * G / rows_per_block)
};

__device__ __forceinline__ void flag(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

// Split rule: chunk = ceil(L/S) rounded up to 16 tokens; split s covers
// [s*chunk, min((s+1)*chunk, L)).  Sub-chunk p of P covers a 16-aligned
// slice of that range; the number of live sub-chunks depends only on the
// chunk's own length.  Nothing here looks at other sequences.
__device__ __forceinline__ void split_range(int L, int S, int s, int* lo, int* hi) {
  int per = (L + S - 1) / S;
  int chunk = (per + kPage - 1) / kPage * kPage;
  long long a = (long long)s * chunk, b = (long long)(s + 1) * chunk;
  *lo = (int)(a < L ? a : L);
  *hi = (int)(b < L ? b : L);
}

// Chunk p of [lo, hi) cut into at most P chunks of a whole number of
// 64-token tiles, each at least min_sub tokens: the chunk length is
// ceil((hi - lo) / P) (or min_sub if larger) rounded up to 64; chunks past
// the end are empty.
__device__ __forceinline__ int sub_len(int len, int P, int min_sub) {
  int per = (len + P - 1) / P;
  if (per < min_sub) per = min_sub;
  return (per + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
}

__device__ __forceinline__ void sub_range(int lo, int hi, int P, int min_sub, int p, int* slo,
                                          int* shi) {
  const int sub = sub_len(hi - lo, P, min_sub);
  long long a = lo + (long long)p * sub, b = lo + (long long)(p + 1) * sub;
  *slo = (int)(a < hi ? a : hi);
  *shi = (int)(b < hi ? b : hi);
}

// Chunk count of a sequence with n query rows: the launch's count P shared
// out among the sequence's row blocks (each row block streams the span
// again, so a many-row sequence takes fewer, longer chunks), but at least
// the caller's split count.  It depends on the sequence alone.
__device__ __forceinline__ int seq_subs(const Params& p, int n) {
  const int rb = (n * p.G + p.rows_per_block - 1) / p.rows_per_block;
  const int c = p.P / (rb > 1 ? rb : 1);
  return c > p.min_splits ? c : p.min_splits;
}

// Work of partial CTA x (blockIdx.x) for a sequence with n query rows: its
// b row blocks times its seq_subs chunks, laid out chunk-major (x = chunk *
// b + row block).  The grid holds max(T, S * most row blocks) such CTAs per
// (KV head, sequence), which covers every sequence; false for x past this
// sequence's work.  *ts = seq_subs(p, n).
__device__ __forceinline__ bool cta_work(const Params& p, int n, int x, int* rb, int* chunk,
                                         int* ts) {
  const int rows = n * p.G;
  if (rows <= p.rows_per_block) {
    *ts = p.P > p.min_splits ? p.P : p.min_splits;
    *rb = 0;
    *chunk = x;
    return x < *ts;
  }
  const int b = (rows + p.rows_per_block - 1) / p.rows_per_block;
  *ts = seq_subs(p, n);
  *rb = x % b;
  *chunk = x / b;
  return *chunk < *ts;
}

// Number of non-empty chunks of [lo, hi) under sub_range (they come first).
__device__ __forceinline__ int live_subs(int lo, int hi, int P, int min_sub) {
  const int len = hi - lo;
  if (len <= 0) return 0;
  const int sub = sub_len(len, P, min_sub);
  const int n = (len + sub - 1) / sub;
  return n < P ? n : P;
}

// Kind of sequence s: 0 chain / direct, 1 tree.
__device__ __forceinline__ int seq_kind_of(const Params& p, int s) {
  if (p.mode == VA_MODE_CHAIN) return 0;
  if (p.mode == VA_MODE_TREE) return 1;
  return p.seq_kind[s] ? 1 : 0;
}

// Rows per sequence: chain sequences (prefill segments, draft chains and
// one-row direct rows) up to kMaxRows, tree suffixes up to kMaxTreeRows
// (their visibility is a 32-bit ancestor mask).
constexpr int kMaxRows = VA_MAX_ROWS_PER_SEQ;
constexpr int kMaxTreeRows = VA_MAX_TREE_ROWS;

// Ancestor mask of local row j: bit a set iff draft position a is visible
// to row j (a == j or a is an ancestor).  A chain row j >= 31 gets every
// bit (draft_visible decides chain visibility from j itself).  The walk strictly decreases, so it
// ends within j steps; a parent outside [-1, current) flags an error.
__device__ __forceinline__ unsigned row_mask(int kind, const int* parent_seq, int j,
                                             bool* bad) {
  if (kind == 0) return j >= 31 ? 0xFFFFFFFFu : ((1u << (j + 1)) - 1u);
  unsigned m = 1u << j;
  int cur = j;
  int par = parent_seq[j];
  while (par != -1) {
    if (par < -1 || par >= cur) {
      *bad = true;
      return m;
    }
    m |= 1u << par;
    cur = par;
    par = parent_seq[cur];
  }
  return m;
}

// Is draft position a (0 <= a < n) visible to local row j?  Chain: a <= j
// (causal).  Tree: bit a of the row's ancestor mask (n <= kMaxTreeRows).
__device__ __forceinline__ bool draft_visible(int kind, unsigned anc, int j, int a) {
  return kind == 0 ? a <= j : ((anc >> a) & 1u) != 0u;
}

// Bits c of [lo, hi) intersected with [0, 32).
__device__ __forceinline__ unsigned bit_range(int lo, int hi) {
  lo = max(lo, 0);
  hi = min(hi, 32);
  if (lo >= hi) return 0u;
  const unsigned up = hi == 32 ? 0xFFFFFFFFu : (1u << hi) - 1u;
  return up & ~((1u << lo) - 1u);
}

// Visibility of the 32 tokens t0 .. t0 + 31 of a span [., shi) to local row
// j of a sequence with ctx context tokens, as bits: context tokens, and
// draft tokens ctx + a for which draft_visible(kind, anc, j, a) holds.  The
// same decision as draft_visible token by token, in a few word operations.
__device__ __forceinline__ unsigned visible_bits(int kind, unsigned anc, int j, int ctx, int shi,
                                                 int t0) {
  unsigned m = bit_range(0, min(ctx, shi) - t0);
  if (shi > ctx) {
    unsigned dm = bit_range(ctx - t0, shi - t0);
    if (kind == 0) {
      dm &= bit_range(ctx - t0, ctx + j + 1 - t0);  // a <= j
    } else {
      const int sh = t0 - ctx;  // bit c of the window is draft position c + sh
      dm &= sh >= 0 ? (sh < 32 ? anc >> sh : 0u) : (-sh < 32 ? anc << -sh : 0u);
    }
    m |= dm;
  }
  return m;
}

// Row of token t of (sequence s, KV head kvh), counted in rows of the k/v
// array; -1 when the block table entry is out of range.
__device__ __forceinline__ long long kv_row(const Params& p, int s, int kvh, int t) {
  if (p.page_size == 0) return ((long long)s * p.KVH + kvh) * p.capacity + t;
  int blk = p.block_table[(long long)s * p.max_blocks + t / kPage];
  if (blk < 0 || blk >= p.num_blocks) return -1;
  return ((long long)blk * p.KVH + kvh) * kPage + (t % kPage);
}

// Does sequence s (of the given kind) read its draft K/V from the tree
// scratch KV (row cu_rows[s] + a for draft position a)?
__device__ __forceinline__ bool uses_scratch(const Params& p, int kind) {
  return p.dk != nullptr && kind == 1;
}

// Scratch row (counted in rows of dk / dv) of draft position a.
__device__ __forceinline__ long long scratch_row(const Params& p, int row0, int kvh, int a) {
  return (long long)(row0 + a) * p.KVH + kvh;
}

// Validate sequence s: row count and the span against capacity / the block
// table (the context only when its drafts sit in the scratch KV).  Returns
// the error bits (0 if fine).
__device__ __forceinline__ unsigned check_sequence(const Params& p, int s, int* row0, int* n,
                                                   int* ctx) {
  int r0 = p.cu_rows[s], r1 = p.cu_rows[s + 1];
  int c = p.ctx_len[s];
  *row0 = r0;
  *n = r1 - r0;
  *ctx = c;
  unsigned err = 0;
  if (r1 < r0 || r1 - r0 > p.max_rows || r0 < 0 || r1 > p.total_rows) err |= VA_DEV_BAD_ROWS;
  else if (r1 - r0 > kMaxTreeRows && seq_kind_of(p, s) == 1) err |= VA_DEV_BAD_ROWS;
  if (c < 0) err |= VA_DEV_CTX_OVERFLOW;
  if (!err) {
    long long L = (long long)c + (uses_scratch(p, seq_kind_of(p, s)) ? 0 : r1 - r0);
    if (p.page_size == 0) {
      if (L > p.capacity) err |= VA_DEV_CTX_OVERFLOW;
    } else {
      if ((L + kPage - 1) / kPage > p.max_blocks) err |= VA_DEV_CTX_OVERFLOW;
    }
  }
  return err;
}

// Storage decoding (exact for bf16 and fp16 scales; Q8 element = d*q in fp32).
__device__ __forceinline__ float bf16_bits_to_float(unsigned short b) {
  return __uint_as_float(((unsigned)b) << 16);
}

__device__ __forceinline__ float load_q(const Params& p, long long idx) {
  if (p.q_dtype == VA_F32) return reinterpret_cast<const float*>(p.q)[idx];
  return bf16_bits_to_float(reinterpret_cast<const unsigned short*>(p.q)[idx]);
}

template <int KVT>
__device__ __forceinline__ float load_kv(const void* base, long long row, int row_bytes, int d) {
  const unsigned char* r = reinterpret_cast<const unsigned char*>(base) + row * row_bytes;
  if (KVT == VA_F32) return reinterpret_cast<const float*>(r)[d];
  if (KVT == VA_BF16) return bf16_bits_to_float(reinterpret_cast<const unsigned short*>(r)[d]);
  const unsigned char* blk = r + (d / kQ8Block) * kQ8BlockBytes;
  unsigned short sb = (unsigned short)(blk[0] | (blk[1] << 8));
  float sc = __half2float(__ushort_as_half(sb));
  signed char code = (signed char)blk[2 + (d % kQ8Block)];
  return sc * (float)code;
}

// Index of the partial slot for (slot, global row, head).
__device__ __forceinline__ long long slot_index(const Params& p, int slot, int grow, int h) {
  return ((long long)slot * p.total_rows + grow) * p.H + h;
}

}  // namespace va
