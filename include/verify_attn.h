/*
 * verify_attn.h — C ABI of the GB300 speculative-decoding verify-attention
 * library (libverify_attn.so, sm_103a).
 *
 * The operation: a window of draft-token query rows per sequence attends over
 * that sequence's KV cache.  Rows are causal along a chain, or follow a
 * parent array for a fixed-width tree suffix; query heads are grouped over
 * fewer KV heads; the cache is contiguous or paged in 16-token blocks and
 * holds fp32, bf16 or Q8_0 rows.  The result per (row, head) is the softmax-
 * weighted sum of the visible V rows (O) and the natural-log sum of the
 * exponentiated scaled scores (LSE).
 *
 * Sources (the pages this library restates):
 *   - hipfire PR #695 "perf(gfx11): optimize Qwen DFlash speculative verify":
 *     section "Summary" (B=16 verify through batched flash attention), the
 *     alpineQ comments (Q8 KV, one block reusing each KV fetch across several
 *     verifier rows, the batched-partials layout and its reducer).
 *   - hipfire PR #817 "speed up long-context DFlash verify 13.4% with FA2
 *     split-KV": sections "Summary", "Default and admission policy" and
 *     "Performance" (S8 split-KV partial + merge, caller-owned partial
 *     workspace, fail-closed admission, S1 equal to the unsplit result).
 *   - lucebox PR #686 "perf(qwen35): retain speculation during paged
 *     prefill": sections "Mechanism", "State and commit invariants" and
 *     "Correctness failure found during qualification" (direct rows and a
 *     fixed-width tree suffix in one step over paged KV; tree ancestry
 *     metadata; partitioning must not depend on what shares the launch).
 *
 * Conventions for every entry point:
 *   - Pointers named "device" are CUDA device memory owned by the caller;
 *     the library never allocates, frees or keeps them past the call.
 *   - Calls are asynchronous on the given CUDA stream (a cudaStream_t passed
 *     as void*; NULL = legacy default stream).  Lengths and metadata are read
 *     on the device, so the host never synchronises.
 *   - The stream must belong to the current device (the plan uses that
 *     device's SM count); outside stream capture, a stream of another
 *     device returns VA_ERR_INVALID_ARG and launches nothing (a capturing
 *     stream's device cannot be queried without ending the capture, so
 *     there the caller's word stands).
 *   - Host-checkable errors return a status and launch nothing.
 *   - Data errors found on the device (bad parent, block id, row counts,
 *     context beyond capacity) OR a VA_DEV_* bit into *status (device word,
 *     may be NULL) and the affected rows get NaN outputs (for inconsistent
 *     row offsets, VA_DEV_BAD_ROWS, every row of that sequence).
 */
#ifndef VERIFY_ATTN_H
#define VERIFY_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum va_status {
  VA_OK = 0,
  VA_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad enum */
  VA_ERR_UNSUPPORTED = 2,         /* shape/dtype outside the supported set */
  VA_ERR_ALIGNMENT = 3,           /* a pointer is not 16-byte aligned */
  VA_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes < va_workspace_size() */
  VA_ERR_CUDA = 5                 /* a CUDA runtime call or launch failed */
} va_status;

typedef enum va_dtype {
  VA_F32 = 0,  /* IEEE fp32 */
  VA_BF16 = 1, /* bfloat16 */
  VA_Q8_0 = 2  /* 34-byte blocks: fp16 scale d (little endian), 32 int8 codes q; value d*q */
} va_dtype;

typedef enum va_mode {
  VA_MODE_CHAIN = 0, /* every sequence is a chain: row j sees context + rows 0..j */
  VA_MODE_TREE = 1,  /* every sequence is a tree over its rows (parent array) */
  VA_MODE_MIXED = 2  /* per-sequence kind from seq_kind[] */
} va_mode;

/* Device status bits (OR-ed into *status). */
#define VA_DEV_BAD_PARENT 0x1u   /* parent[j] not in [-1, j) */
#define VA_DEV_BAD_BLOCK 0x2u    /* block_table entry outside [0, num_blocks) */
#define VA_DEV_CTX_OVERFLOW 0x4u /* ctx + n exceeds capacity / the block table */
#define VA_DEV_BAD_ROWS 0x8u     /* cu_rows not ascending, n > max_rows_per_seq, total mismatch,
                                    or a tree sequence with more than VA_MAX_TREE_ROWS rows */
#define VA_DEV_TIMEOUT 0x10u     /* a bounded pipeline wait gave up */

/* Problem flags. */
#define VA_FLAG_CUDA_CORES 0x1u /* run the CUDA-core (SIMT) partial kernel for any dtype */

/*
 * The KV cache.
 *   contiguous (page_size == 0): k, v are [num_seqs][num_kv_heads][capacity][row];
 *     capacity is a multiple of 16 tokens.
 *   paged (page_size == 16): k, v are pools [num_blocks][num_kv_heads][16][row]
 *     and token t of sequence s lives in block block_table[s*max_blocks_per_seq + t/16],
 *     slot t%16 (lucebox PR #686, "Correctness failure found during
 *     qualification": 16-token blocks).
 *   row = head_dim fp32 / bf16 elements, or head_dim/32 Q8_0 blocks of 34 bytes.
 *   The draft rows' own K/V sit at positions ctx .. ctx+n-1 of the same cache,
 *   except for tree sequences when a tree scratch KV is given (draft_k,
 *   draft_v: device [total_rows][num_kv_heads][row], row r of the launch in
 *   the cache's row format, 16-byte aligned).  Then a tree sequence's draft
 *   position a reads scratch row cu_rows[s] + a, and its cache needs room
 *   for the context only (capacity, or block-table entries, for ctx_len[s]
 *   tokens).  Chain and direct sequences always read the cache: prefill and
 *   direct rows write durable KV, tree rows write scratch KV (lucebox PR
 *   #686, "State and commit invariants").  With a scratch KV, Q8_0 caches
 *   (contiguous or paged) run on the transposed tensor-core kernel and other
 *   caches on the CUDA-core kernel.
 */
typedef struct va_kv {
  va_dtype dtype;
  int32_t num_kv_heads;
  int32_t head_dim;            /* 64, 128 or 256 */
  const void *k;               /* device, 16-byte aligned */
  const void *v;               /* device, 16-byte aligned */
  int32_t page_size;           /* 0 or 16 */
  int64_t capacity;            /* contiguous only: tokens per (sequence, KV head) */
  const int32_t *block_table;  /* paged only: device [num_seqs][max_blocks_per_seq] */
  int32_t max_blocks_per_seq;  /* paged only */
  int32_t num_blocks;          /* paged only: blocks in the pool */
  const void *draft_k;         /* optional tree scratch KV (see above), or NULL */
  const void *draft_v;         /* set together with draft_k */
} va_kv;

/*
 * The query side.
 *   q: device [total_rows][num_heads][head_dim], fp32 or bf16 (bf16 for the
 *      bf16 and Q8_0 caches; fp32 or bf16 for the fp32 cache).
 *   Rows of sequence s are cu_rows[s] .. cu_rows[s+1]-1 (device array); row
 *   j of a sequence sits at KV position ctx_len[s] + j.
 *   parent: device [total_rows], the local index of each row's parent in its
 *      own sequence, -1 for a node attached to the context; must satisfy
 *      parent[j] < j.  Ignored for chain sequences (may be NULL in chain mode).
 *   seq_kind: device [num_seqs], 0 = chain (a 1-row chain is a direct/AR
 *      row), 1 = tree; read in VA_MODE_MIXED only.
 *   Query head h reads KV head h / (num_heads / num_kv_heads).
 *   scale: softmax scale; 0 selects 1/sqrt(head_dim).
 *   num_splits: S >= 1.  Sequence s's span L = ctx + n is cut into chunks
 *      of max(ceil(L/Ts), 128) tokens rounded up to a whole number of
 *      64-token tiles (at most Ts chunks).  T (>= S, <= 16 S) is fixed by S,
 *      num_kv_heads and the GPU's SM count only (one wave of CTAs per
 *      sequence and KV head); a sequence whose n * G query rows span b > 1
 *      row blocks of the partial kernel (128 rows on the tensor-core
 *      kernels, 16 on the CUDA-core kernel), each of which reads the span
 *      again, uses Ts = max(S, floor(T / b)) chunks (T otherwise); each
 *      chunk writes an fp32 online-softmax
 *      partial and a merge pass combines them in ascending order (hipfire
 *      PR #817, "Summary" and "Performance").  No choice depends on the
 *      other sequences of the launch, so a row's result depends only on
 *      its own sequence (lucebox PR #686, "Correctness failure found during
 *      qualification").
 */
/* Rows per sequence: a chain sequence (a prefill segment, a draft chain or
 * a one-row direct row; causal among its own rows) may hold up to
 * VA_MAX_ROWS_PER_SEQ rows, a tree suffix up to VA_MAX_TREE_ROWS (its
 * visibility is a 32-bit ancestor mask).  Rows beyond 128 / G per KV head
 * run as further row blocks, each reading that sequence's K/V again. */
#define VA_MAX_ROWS_PER_SEQ 1024
#define VA_MAX_TREE_ROWS 32

typedef struct va_problem {
  int32_t num_seqs;
  int32_t num_heads;
  va_dtype q_dtype;
  const void *q;
  const int32_t *cu_rows;
  const int32_t *ctx_len;
  const int32_t *parent;
  const uint8_t *seq_kind;
  int32_t total_rows;          /* host copy of cu_rows[num_seqs] */
  int32_t max_rows_per_seq;    /* host bound on rows per sequence, 1..VA_MAX_ROWS_PER_SEQ
                                  (VA_MODE_TREE: 1..VA_MAX_TREE_ROWS) */
  float scale;
  int32_t num_splits;
  uint32_t flags;              /* VA_FLAG_* */
} va_problem;

/* Library version (major*10000 + minor*100 + patch). */
int32_t va_version(void);

/*
 * Tree commit of the KV cache (the KV part of lucebox PR #686's tree commit
 * transaction, "State and commit invariants": tree rows write scratch KV;
 * the commit promotes only the accepted prefix and checks every domain
 * before it mutates any).  For each sequence s, the accepted path of m_s =
 * accepted_len[s] tree nodes, accepted_nodes[cu_rows[s] + i] for i < m_s
 * (root first), goes from the tree scratch KV (kv->draft_k / draft_v, row
 * cu_rows[s] + node) to positions ctx_len[s] + i of the cache, K and V of
 * every KV head, byte for byte.  accepted_len: device [num_seqs];
 * accepted_nodes: device [total_rows] (entries past m_s ignored).
 * Device preflight before any write, for every sequence: the row checks of
 * a verify call (VA_DEV_BAD_ROWS, VA_DEV_CTX_OVERFLOW on the context);
 * 0 <= m <= n and m = 0 unless the sequence is a tree (VA_DEV_BAD_ROWS);
 * nodes in [0, n) (VA_DEV_BAD_ROWS) forming a root path: parent[first] =
 * -1, parent[next] = previous (VA_DEV_BAD_PARENT); positions up to
 * ctx + m within capacity or the block table (VA_DEV_CTX_OVERFLOW) on
 * valid blocks (VA_DEV_BAD_BLOCK).  If the status word holds any bit after
 * the preflight, nothing is written: *status must be 0 on entry.  Host
 * checks as for the verify calls; kv->draft_k, accepted_len and status are
 * required (VA_ERR_INVALID_ARG).  The scratch must not overlap the cache.
 */
va_status verify_attn_promote(const va_problem *p, const va_kv *kv, int32_t mode,
                              const int32_t *accepted_len, const int32_t *accepted_nodes,
                              uint32_t *status, void *stream);

/* Human-readable name of a status code; never NULL. */
const char *va_status_string(va_status s);

/* Text of the CUDA error behind this thread's last VA_ERR_CUDA; never NULL. */
const char *va_last_cuda_error(void);

/*
 * Bytes of device workspace a verify call needs for this problem: the fp32
 * split partials (m, l and the unnormalised accumulator per split, row and
 * head; hipfire PR #817 "Default and admission policy": the caller-owned
 * partial workspace).  Returns 0 for an invalid problem.
 */
size_t va_workspace_size(const va_problem *p, const va_kv *kv);

/*
 * Host-only validation, no launch and no device access: the checks every
 * verify call makes before launching (fail-closed admission as in hipfire
 * PR #817 "Default and admission policy"; undersized workspace rejected).
 */
va_status va_validate(const va_problem *p, const va_kv *kv, int32_t mode, size_t ws_bytes);

/*
 * Verify attention.  o: device fp32 [total_rows][num_heads][head_dim];
 * lse: device fp32 [total_rows][num_heads] (natural log).  ws: device
 * workspace of at least va_workspace_size() bytes, 256-byte aligned;
 * its contents need no initialisation and are overwritten.
 *   verify_attn_chain: every sequence is a chain (also 1-row direct rows).
 *   verify_attn_tree:  every sequence is a tree over its rows (parent required).
 *   verify_attn_mixed: per-sequence chain or tree from seq_kind (lucebox PR
 *                      #686 "Mechanism": direct rows and tree rows in one step).
 */
va_status verify_attn_chain(const va_problem *p, const va_kv *kv, void *ws, size_t ws_bytes,
                            float *o, float *lse, uint32_t *status, void *stream);
va_status verify_attn_tree(const va_problem *p, const va_kv *kv, void *ws, size_t ws_bytes,
                           float *o, float *lse, uint32_t *status, void *stream);
va_status verify_attn_mixed(const va_problem *p, const va_kv *kv, void *ws, size_t ws_bytes,
                            float *o, float *lse, uint32_t *status, void *stream);

/*
 * Debug export of the row map and masks the kernels use: row_seq[r] is the
 * sequence of global row r; anc_mask[r] has bit a set iff draft position a
 * of that sequence is visible to row r (itself or an ancestor).  Device
 * outputs of total_rows entries each.  The mask has 32 bits: a chain row
 * j >= 31 gets every bit (the kernels decide chain visibility from j).  (lucebox PR #686 "Correctness failure
 * found during qualification": the compact row map and W8 topology checks.)
 */
va_status va_debug_row_map(const va_problem *p, int32_t mode, int32_t *row_seq,
                           uint32_t *anc_mask, uint32_t *status, void *stream);

/*
 * Debug export of the KV gather the kernels use: phys_row[s*max_len + t] is
 * the row of token t of sequence s, KV head kv_head, counted in rows of the
 * k/v array (contiguous: (s*KVH+kvh)*capacity + t; paged:
 * (block*KVH+kvh)*16 + t%16), or -1 for t >= ctx+n.  Device output of
 * num_seqs*max_len int64.
 */
va_status va_debug_gather_index(const va_problem *p, const va_kv *kv, int32_t kv_head,
                                int64_t max_len, int64_t *phys_row, uint32_t *status,
                                void *stream);

/*
 * Debug export of the KV chunks the partial kernels run (the split plan of
 * hipfire PR #817 "Summary": each sequence's span cut into chunks whose
 * partials a merge combines; lucebox PR #686 "Correctness failure found
 * during qualification": the cut must not depend on what else shares the
 * launch).  For sequence s and slot j < T (T = va_plan's slots),
 * ranges[2*(s*T + j)] and ranges[2*(s*T + j) + 1] are the first and
 * one-past-last KV position of chunk j, computed by the device functions
 * the partial kernels call: with L = ctx_len[s] + rows of s and Ts the
 * sequence's chunk count (see num_splits), a chunk has c = max(ceil(L / Ts),
 * 128) rounded up to a multiple of 64 tokens and chunk j is [min(j c, L),
 * min((j + 1) c, L)) (empty past L; slots Ts .. T - 1 are empty).  A sequence
 * whose row offsets are inconsistent gets -1, -1 and sets
 * VA_DEV_BAD_ROWS.  ranges: device int32[num_seqs * T * 2].
 */
va_status va_debug_split_ranges(const va_problem *p, const va_kv *kv, int32_t mode,
                                int32_t *ranges, uint32_t *status, void *stream);

/* Plan details for a problem (which kernel runs, splits and sub-splits). */
/* Partial kernels (va_plan_info.kernel). */
#define VA_KERNEL_CUDA_CORES 0 /* fp32 FMA, one thread block per 16 query rows */
#define VA_KERNEL_TENSOR 1     /* tcgen05, query rows on the MMA's M axis (bf16 caches) */
#define VA_KERNEL_TENSOR_Q8 2  /* tcgen05, tokens on M and query rows on N (Q8_0 caches) */

typedef struct va_plan_info {
  int32_t kernel;          /* VA_KERNEL_* */
  int32_t sub_splits;      /* T: KV chunks per sequence of one row block (equal to slots) */
  int32_t slots;           /* T partial slots per (row, head) */
  int32_t grid_x, grid_y, grid_z; /* x: max(T, S * row blocks of the longest sequence);
                                     y: KV heads; z: sequences */
  int32_t threads;
  int32_t smem_bytes;
} va_plan_info;

va_status va_plan(const va_problem *p, const va_kv *kv, int32_t mode, va_plan_info *out);

/*
 * Optional per-kernel timing for benchmarks.  While enabled (on != 0),
 * every verify call records CUDA events on its stream before the partial
 * kernel, between the partial and merge kernels, and after the merge;
 * enabling restarts at slot 0 (at most 4096 calls are kept).  Inside a
 * stream capture the records become event nodes of the graph, so a replay
 * refreshes them.  va_timing_read waits for the recorded events and writes
 * each recorded call's partial and merge durations in milliseconds
 * (host arrays of max_calls floats, either may be NULL).  Not thread-safe.
 */
va_status va_timing_enable(int32_t on);
va_status va_timing_read(int32_t max_calls, float *partial_ms, float *merge_ms,
                         int32_t *num_calls);

/*
 * Verify attention without a caller workspace and without any allocation
 * on the call path.  The pages have no counterpart to this entry point;
 * verify_attn_chain/tree/mixed, which take a caller workspace, are the
 * pages' route.
 *
 * For callers that cannot hand the library device memory per call: code
 * that owns no allocator (a plain C host program, a runtime whose device
 * memory budget is fixed up front), or a serving loop that must not call
 * into an allocator between steps.  The split partials go to scratch that
 * belongs to the library: a fixed array of VA_STATIC_WORKSPACE_BYTES in the
 * library's device image, reserved by the CUDA runtime when the library's
 * module is loaded on a device (one array per device).
 *
 * mode: VA_MODE_CHAIN, VA_MODE_TREE or VA_MODE_MIXED (same meaning as the
 * three entry points above).  p, kv, o, lse, status, stream: as for
 * verify_attn_chain.  Nothing needs initialising: the scratch holds no
 * state between calls and need not start at zero.
 *
 * Limits and errors:
 *   - Problems whose va_workspace_size() exceeds VA_STATIC_WORKSPACE_BYTES
 *     (16 MiB: e.g. 38 slots x 16 rows x 24 heads at D=256 fit,
 *     38 slots x 50 rows x 24 heads do not) return
 *     VA_ERR_WORKSPACE_TOO_SMALL before any launch; use the entry points
 *     with a caller workspace for those.
 *   - The scratch used is the current device's, and the stream must belong
 *     to that device (VA_ERR_INVALID_ARG otherwise, nothing launched).
 *   - The first call on each device looks the scratch address up with
 *     cudaGetSymbolAddress (VA_ERR_CUDA if that fails); make that first
 *     call, on every device it will be used on, outside any stream capture.
 *   - The scratch is shared by every call on a device: calls on one stream
 *     are ordered and safe, calls that can overlap in time (different
 *     streams without ordering between them, several host threads) race on
 *     it and must not be issued.
 */
#define VA_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)

va_status verify_attn_noalloc(const va_problem *p, const va_kv *kv, int32_t mode, float *o,
                              float *lse, uint32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* VERIFY_ATTN_H */
