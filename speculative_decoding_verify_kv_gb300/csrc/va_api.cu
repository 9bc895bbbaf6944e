// Host side of the C ABI: validation (fail-closed, before any launch),
// planning (kernel, splits, sub-chunks, grid), workspace sizing and the
// launches on the caller's stream.
//
// Admission follows the fail-closed rule of hipfire PR #817 "Default and
// admission policy": anything outside the supported set is rejected with a
// status, never silently routed elsewhere; an undersized workspace is
// rejected before launch.
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <vector>

#include "va_common.cuh"

namespace va {
cudaError_t launch_simt_partial(const Params& p, dim3 grid, cudaStream_t st);
int simt_smem_bytes(int D);
cudaError_t launch_umma_partial(const Params& p, dim3 grid, cudaStream_t st);
int umma_smem_bytes(int D, int kv_dtype);
int umma_threads(int D, int kv_dtype);
cudaError_t launch_tq8_partial(const Params& p, dim3 grid, cudaStream_t st);
int tq8_rows_per_block();
int tq8_threads();
int tq8_smem_bytes(int D);

static thread_local cudaError_t g_last_cuda = cudaSuccess;
static va_status note_cuda(cudaError_t e) {
  g_last_cuda = e;
  return VA_ERR_CUDA;
}
cudaError_t launch_merge(const Params& p, cudaStream_t st);
cudaError_t launch_debug_row_map(const Params& p, int* row_seq, unsigned* anc, cudaStream_t st);
cudaError_t launch_debug_split(const Params& p, int* ranges, cudaStream_t st);
cudaError_t launch_promote(const Params& p, const int* acc_len, const int* nodes,
                           cudaStream_t st);
cudaError_t launch_debug_gather(const Params& p, int kvh, long long max_len, long long* out,
                                cudaStream_t st);

constexpr int kSimtRowsPerBlock = 16;
constexpr int kSimtThreadsPerBlock = 128;
constexpr int kUmmaRowsPerBlock = 128;
constexpr int kMinSubTokens = 128;
constexpr int kMaxSubSplits = 16;

static int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

static bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

// The plan (the SM count) and the library-held scratch are the current
// device's, so a stream must belong to the current device; the default
// streams always do.  Checked outside stream capture only: querying a
// capturing stream's device is not a capturable operation and would
// invalidate the capture.
static va_status check_stream_device(cudaStream_t s) {
  if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread) return VA_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return note_cuda(e);
  if (cap != cudaStreamCaptureStatusNone) return VA_OK;
  int dev = 0, sdev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return note_cuda(e);
  e = cudaStreamGetDevice(s, &sdev);
  if (e != cudaSuccess) return note_cuda(e);
  return sdev == dev ? VA_OK : VA_ERR_INVALID_ARG;
}

static int row_bytes_of(int dtype, int D) {
  switch (dtype) {
    case VA_F32: return 4 * D;
    case VA_BF16: return 2 * D;
    case VA_Q8_0: return D / kQ8Block * kQ8BlockBytes;
  }
  return 0;
}

// Checks that need no device access.  ws_bytes < 0 skips the workspace check.
static va_status check(const va_problem* p, const va_kv* kv, int mode) {
  if (!p || !kv) return VA_ERR_INVALID_ARG;
  if (mode < VA_MODE_CHAIN || mode > VA_MODE_MIXED) return VA_ERR_INVALID_ARG;
  if (p->num_seqs < 1 || p->num_heads < 1 || kv->num_kv_heads < 1) return VA_ERR_INVALID_ARG;
  if (p->total_rows < 0 || p->num_splits < 1) return VA_ERR_INVALID_ARG;
  if (p->max_rows_per_seq < 1) return VA_ERR_INVALID_ARG;
  if (p->q_dtype < VA_F32 || p->q_dtype > VA_Q8_0) return VA_ERR_INVALID_ARG;
  if (kv->dtype < VA_F32 || kv->dtype > VA_Q8_0) return VA_ERR_INVALID_ARG;
  if (p->num_heads % kv->num_kv_heads) return VA_ERR_UNSUPPORTED;
  int G = p->num_heads / kv->num_kv_heads;
  if (G > 8) return VA_ERR_UNSUPPORTED;
  if (kv->head_dim != 64 && kv->head_dim != 128 && kv->head_dim != 256) return VA_ERR_UNSUPPORTED;
  if (p->max_rows_per_seq > kMaxRows) return VA_ERR_UNSUPPORTED;
  if (mode == VA_MODE_TREE && p->max_rows_per_seq > kMaxTreeRows) return VA_ERR_UNSUPPORTED;
  if (p->num_splits > 256) return VA_ERR_UNSUPPORTED;
  if (p->q_dtype == VA_Q8_0) return VA_ERR_UNSUPPORTED;
  if (kv->dtype != VA_F32 && p->q_dtype != VA_BF16) return VA_ERR_UNSUPPORTED;
  if (!(p->scale >= 0.f) || isinf(p->scale)) return VA_ERR_INVALID_ARG;
  if (p->flags & ~(uint32_t)VA_FLAG_CUDA_CORES) return VA_ERR_INVALID_ARG;
  if (!p->cu_rows || !p->ctx_len) return VA_ERR_INVALID_ARG;
  if (p->total_rows > 0 && !p->q) return VA_ERR_INVALID_ARG;
  if (mode != VA_MODE_CHAIN && !p->parent) return VA_ERR_INVALID_ARG;
  if (mode == VA_MODE_MIXED && !p->seq_kind) return VA_ERR_INVALID_ARG;
  if (!kv->k || !kv->v) return VA_ERR_INVALID_ARG;
  if (!kv->draft_k != !kv->draft_v) return VA_ERR_INVALID_ARG;
  if (kv->draft_k && (!aligned16(kv->draft_k) || !aligned16(kv->draft_v))) return VA_ERR_ALIGNMENT;
  if (kv->page_size == 0) {
    if (kv->capacity < 1) return VA_ERR_INVALID_ARG;
    if (kv->capacity % kPage) return VA_ERR_UNSUPPORTED;
  } else if (kv->page_size == kPage) {
    if (!kv->block_table || kv->max_blocks_per_seq < 1 || kv->num_blocks < 1)
      return VA_ERR_INVALID_ARG;
  } else {
    return VA_ERR_UNSUPPORTED;
  }
  if (!aligned16(kv->k) || !aligned16(kv->v)) return VA_ERR_ALIGNMENT;
  if (p->q && !aligned16(p->q)) return VA_ERR_ALIGNMENT;
  return VA_OK;
}

struct Plan {
  int kernel;  // VA_KERNEL_*
  int P, slots, rows_per_block, row_blocks, threads, smem;
  dim3 grid;
};

static Plan make_plan(const va_problem* p, const va_kv* kv) {
  Plan pl;
  const int G = p->num_heads / kv->num_kv_heads;
  // Kernel choice from the cache dtype, the layout, the caller's flag and
  // whether a tree scratch KV is given, never from the problem's sizes:
  // the row-major tensor-core kernel for bf16 caches without a scratch KV
  // and for Q8_0 caches except contiguous ones with a scratch KV, which the
  // transposed tensor-core kernel takes; everything else on the CUDA-core
  // kernel.
  const bool tensor_ok = kv->dtype != VA_F32 && !(p->flags & VA_FLAG_CUDA_CORES);
  const bool scratch = kv->draft_k != nullptr;
  if (tensor_ok && kv->dtype == VA_Q8_0 && kv->page_size == 0 && scratch) {
    pl.kernel = VA_KERNEL_TENSOR_Q8;
    pl.rows_per_block = tq8_rows_per_block();
    pl.threads = tq8_threads();
    pl.smem = tq8_smem_bytes(kv->head_dim);
  } else if (tensor_ok && (!scratch || kv->dtype == VA_Q8_0)) {
    pl.kernel = VA_KERNEL_TENSOR;
    pl.rows_per_block = kUmmaRowsPerBlock;
    pl.threads = umma_threads(kv->head_dim, kv->dtype);
    pl.smem = umma_smem_bytes(kv->head_dim, kv->dtype);
  } else {
    pl.kernel = VA_KERNEL_CUDA_CORES;
    pl.rows_per_block = kSimtRowsPerBlock;
    pl.threads = kSimtThreadsPerBlock;
    pl.smem = simt_smem_bytes(kv->head_dim);
  }
  const bool tensor = pl.kernel != VA_KERNEL_CUDA_CORES;
  // Each sequence's KV span is cut into at most `slots` chunks of whole
  // 64-token tiles, at least 128 tokens each (fewer when the span is
  // short), the count fixed by S, the KV head count and the SM count only:
  // never by the other sequences of the launch.  One sequence's chunks of one KV head fill one wave of CTAs
  // (the tensor-core kernel holds one CTA per SM, the CUDA-core kernel
  // about two); the count is at least S and at most S * kMaxSubSplits.
  const int target = (tensor ? 1 : 2) * sm_count();
  int slots = target / kv->num_kv_heads;
  if (slots < p->num_splits) slots = p->num_splits;
  if (slots > p->num_splits * kMaxSubSplits) slots = p->num_splits * kMaxSubSplits;
  pl.P = slots;
  pl.slots = slots;
  const int rows = p->max_rows_per_seq * G;
  pl.row_blocks = (rows + pl.rows_per_block - 1) / pl.rows_per_block;
  // Per (KV head, sequence) the CTAs of a sequence's row blocks times its
  // chunks (cta_work): T chunks for a sequence of one row block, max(S,
  // T / b) for one of b blocks, so max(T, S * row_blocks) CTAs cover all.
  const int per = pl.slots > p->num_splits * pl.row_blocks ? pl.slots
                                                           : p->num_splits * pl.row_blocks;
  pl.grid = dim3((unsigned)per, (unsigned)kv->num_kv_heads, (unsigned)p->num_seqs);
  return pl;
}

static size_t ws_bytes_for(const va_problem* p, const va_kv* kv, const Plan& pl) {
  size_t items = (size_t)pl.slots * (size_t)p->total_rows * (size_t)p->num_heads;
  size_t acc = items * (size_t)kv->head_dim * 4;
  size_t ml = items * 2 * 4;
  acc = (acc + 255) / 256 * 256;
  ml = (ml + 255) / 256 * 256;
  return acc + ml;
}

static Params make_params(const va_problem* p, const va_kv* kv, int mode, const Plan& pl,
                          void* ws, float* o, float* lse, uint32_t* status) {
  Params q;
  memset(&q, 0, sizeof(q));
  q.num_seqs = p->num_seqs;
  q.H = p->num_heads;
  q.KVH = kv->num_kv_heads;
  q.G = p->num_heads / kv->num_kv_heads;
  q.D = kv->head_dim;
  q.total_rows = p->total_rows;
  q.max_rows = p->max_rows_per_seq;
  q.S = 1;  // one level of chunks: [0, L) in pl.slots pieces
  q.P = pl.P;
  q.slots = pl.slots;
  q.min_sub = kMinSubTokens;
  q.min_splits = p->num_splits;
  q.mode = mode;
  q.kv_dtype = kv->dtype;
  q.q_dtype = p->q_dtype;
  float sc = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)kv->head_dim);
  q.scale_log2 = (float)((double)sc * 1.4426950408889634);
  q.q = p->q;
  q.cu_rows = p->cu_rows;
  q.ctx_len = p->ctx_len;
  q.parent = p->parent;
  q.seq_kind = p->seq_kind;
  q.k = kv->k;
  q.v = kv->v;
  q.dk = kv->draft_k;
  q.dv = kv->draft_v;
  q.page_size = kv->page_size;
  q.capacity = kv->capacity;
  q.block_table = kv->block_table;
  q.max_blocks = kv->max_blocks_per_seq;
  q.num_blocks = kv->num_blocks;
  q.row_bytes = row_bytes_of(kv->dtype, kv->head_dim);
  if (ws) {
    size_t items = (size_t)pl.slots * (size_t)p->total_rows * (size_t)p->num_heads;
    size_t acc = (items * (size_t)kv->head_dim * 4 + 255) / 256 * 256;
    q.ws_acc = (float*)ws;
    q.ws_ml = (float*)((char*)ws + acc);
  }
  q.o = o;
  q.lse = lse;
  q.status = (unsigned*)status;
  q.rows_per_block = pl.rows_per_block;
  q.row_blocks = pl.row_blocks;
  return q;
}

// Optional per-kernel timing: while enabled, each verify call records CUDA
// events around its partial and merge launches on the call's stream
// (slots are reused from 0 each time timing is switched on; events made
// during stream capture become event-record nodes of the graph).
struct TimingSlot {
  cudaEvent_t e[3];
};
static std::vector<TimingSlot> g_timing_slots;
static bool g_timing_on = false;
static int g_timing_next = 0;
constexpr int kMaxTimingSlots = 4096;

// Record a timing event; under stream capture as an external event node.
// Timing is best-effort: a failed record clears its error so it never
// reaches the launch checks.
static void timing_record(cudaEvent_t e, cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t r = cudaStreamIsCapturing(s, &cap);
  if (r == cudaSuccess && cap == cudaStreamCaptureStatusActive)
    r = cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
  else
    r = cudaEventRecord(e, s);
  if (r != cudaSuccess) cudaGetLastError();
}

static TimingSlot* timing_slot() {
  if (!g_timing_on || g_timing_next >= kMaxTimingSlots) return nullptr;
  if (g_timing_next >= (int)g_timing_slots.size()) {
    TimingSlot t;
    for (int i = 0; i < 3; ++i)
      if (cudaEventCreate(&t.e[i]) != cudaSuccess) return nullptr;
    g_timing_slots.push_back(t);
  }
  return &g_timing_slots[g_timing_next++];
}

static cudaError_t launch_partial(const Plan& pl, const Params& q, cudaStream_t cs) {
  switch (pl.kernel) {
    case VA_KERNEL_TENSOR_Q8: return launch_tq8_partial(q, pl.grid, cs);
    case VA_KERNEL_TENSOR: return launch_umma_partial(q, pl.grid, cs);
    default: return launch_simt_partial(q, pl.grid, cs);
  }
}

static va_status run(const va_problem* p, const va_kv* kv, int mode, void* ws, size_t ws_bytes,
                     float* o, float* lse, uint32_t* status, void* stream) {
  va_status st = check(p, kv, mode);
  if (st != VA_OK) return st;
  if (p->total_rows == 0) return VA_OK;
  if (!o || !lse) return VA_ERR_INVALID_ARG;
  if (!aligned16(o)) return VA_ERR_ALIGNMENT;
  Plan pl = make_plan(p, kv);
  size_t need = ws_bytes_for(p, kv, pl);
  if (!ws || ws_bytes < need) return VA_ERR_WORKSPACE_TOO_SMALL;
  if (((uintptr_t)ws & 255u) != 0) return VA_ERR_ALIGNMENT;
  cudaStream_t cs = (cudaStream_t)stream;
  st = check_stream_device(cs);
  if (st != VA_OK) return st;
  Params q = make_params(p, kv, mode, pl, ws, o, lse, status);
  TimingSlot* ts = timing_slot();
  // External records so that, under stream capture, they become event
  // nodes of the graph (plain records only order work inside a capture).
  if (ts) timing_record(ts->e[0], cs);
  cudaError_t e = launch_partial(pl, q, cs);
  if (e != cudaSuccess) return note_cuda(e);
  if (ts) timing_record(ts->e[1], cs);
  e = launch_merge(q, cs);
  if (e != cudaSuccess) return note_cuda(e);
  if (ts) timing_record(ts->e[2], cs);
  return VA_OK;
}

}  // namespace va

using namespace va;

extern "C" {

int32_t va_version(void) { return 100; }

const char* va_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda); }

const char* va_status_string(va_status s) {
  switch (s) {
    case VA_OK: return "ok";
    case VA_ERR_INVALID_ARG: return "invalid argument";
    case VA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case VA_ERR_ALIGNMENT: return "pointer not aligned";
    case VA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case VA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

size_t va_workspace_size(const va_problem* p, const va_kv* kv) {
  if (check(p, kv, VA_MODE_CHAIN) != VA_OK && check(p, kv, VA_MODE_MIXED) != VA_OK) return 0;
  Plan pl = make_plan(p, kv);
  return ws_bytes_for(p, kv, pl);
}

va_status va_validate(const va_problem* p, const va_kv* kv, int32_t mode, size_t ws_bytes) {
  va_status st = check(p, kv, mode);
  if (st != VA_OK) return st;
  if (p->total_rows == 0) return VA_OK;
  Plan pl = make_plan(p, kv);
  if (ws_bytes < ws_bytes_for(p, kv, pl)) return VA_ERR_WORKSPACE_TOO_SMALL;
  return VA_OK;
}

va_status va_plan(const va_problem* p, const va_kv* kv, int32_t mode, va_plan_info* out) {
  va_status st = check(p, kv, mode);
  if (st != VA_OK) return st;
  if (!out) return VA_ERR_INVALID_ARG;
  Plan pl = make_plan(p, kv);
  out->kernel = pl.kernel;
  out->sub_splits = pl.P;
  out->slots = pl.slots;
  out->grid_x = (int32_t)pl.grid.x;
  out->grid_y = (int32_t)pl.grid.y;
  out->grid_z = (int32_t)pl.grid.z;
  out->threads = pl.threads;
  out->smem_bytes = pl.smem;
  return VA_OK;
}

va_status va_timing_enable(int32_t on) {
  g_timing_on = on != 0;
  if (g_timing_on) g_timing_next = 0;
  return VA_OK;
}

va_status va_timing_read(int32_t max_calls, float* partial_ms, float* merge_ms,
                         int32_t* num_calls) {
  if (!num_calls) return VA_ERR_INVALID_ARG;
  int n = g_timing_next < max_calls ? g_timing_next : max_calls;
  for (int i = 0; i < n; ++i) {
    TimingSlot& t = g_timing_slots[i];
    cudaError_t e = cudaEventSynchronize(t.e[2]);
    if (e != cudaSuccess) return note_cuda(e);
    float a = 0.f, b = 0.f;
    if ((e = cudaEventElapsedTime(&a, t.e[0], t.e[1])) != cudaSuccess) return note_cuda(e);
    if ((e = cudaEventElapsedTime(&b, t.e[1], t.e[2])) != cudaSuccess) return note_cuda(e);
    if (partial_ms) partial_ms[i] = a;
    if (merge_ms) merge_ms[i] = b;
  }
  *num_calls = n;
  return VA_OK;
}

va_status verify_attn_chain(const va_problem* p, const va_kv* kv, void* ws, size_t ws_bytes,
                            float* o, float* lse, uint32_t* status, void* stream) {
  return run(p, kv, VA_MODE_CHAIN, ws, ws_bytes, o, lse, status, stream);
}

va_status verify_attn_tree(const va_problem* p, const va_kv* kv, void* ws, size_t ws_bytes,
                           float* o, float* lse, uint32_t* status, void* stream) {
  return run(p, kv, VA_MODE_TREE, ws, ws_bytes, o, lse, status, stream);
}

va_status verify_attn_mixed(const va_problem* p, const va_kv* kv, void* ws, size_t ws_bytes,
                            float* o, float* lse, uint32_t* status, void* stream) {
  return run(p, kv, VA_MODE_MIXED, ws, ws_bytes, o, lse, status, stream);
}

va_status va_debug_row_map(const va_problem* p, int32_t mode, int32_t* row_seq,
                           uint32_t* anc_mask, uint32_t* status, void* stream) {
  if (!p || !p->cu_rows || !p->ctx_len) return VA_ERR_INVALID_ARG;
  if (mode < VA_MODE_CHAIN || mode > VA_MODE_MIXED) return VA_ERR_INVALID_ARG;
  if (p->num_seqs < 1 || p->max_rows_per_seq < 1 || p->max_rows_per_seq > kMaxRows)
    return VA_ERR_INVALID_ARG;
  if (mode == VA_MODE_TREE && p->max_rows_per_seq > kMaxTreeRows) return VA_ERR_INVALID_ARG;
  if (mode != VA_MODE_CHAIN && !p->parent) return VA_ERR_INVALID_ARG;
  if (mode == VA_MODE_MIXED && !p->seq_kind) return VA_ERR_INVALID_ARG;
  if (p->total_rows == 0) return VA_OK;
  if (!row_seq || !anc_mask) return VA_ERR_INVALID_ARG;
  Params q;
  memset(&q, 0, sizeof(q));
  q.num_seqs = p->num_seqs;
  q.total_rows = p->total_rows;
  q.max_rows = p->max_rows_per_seq;
  q.mode = mode;
  q.cu_rows = p->cu_rows;
  q.ctx_len = p->ctx_len;
  q.parent = p->parent;
  q.seq_kind = p->seq_kind;
  q.status = (unsigned*)status;
  q.capacity = 1LL << 40;  // spans are not checked here
  cudaError_t e = launch_debug_row_map(q, row_seq, (unsigned*)anc_mask, (cudaStream_t)stream);
  return e == cudaSuccess ? VA_OK : note_cuda(e);
}

va_status va_debug_gather_index(const va_problem* p, const va_kv* kv, int32_t kv_head,
                                int64_t max_len, int64_t* phys_row, uint32_t* status,
                                void* stream) {
  va_status st = check(p, kv, VA_MODE_CHAIN);
  if (st != VA_OK) return st;
  if (kv_head < 0 || kv_head >= kv->num_kv_heads || max_len < 1 || !phys_row)
    return VA_ERR_INVALID_ARG;
  Plan pl = make_plan(p, kv);
  Params q = make_params(p, kv, VA_MODE_CHAIN, pl, nullptr, nullptr, nullptr, status);
  cudaError_t e = launch_debug_gather(q, kv_head, (long long)max_len, (long long*)phys_row,
                                      (cudaStream_t)stream);
  return e == cudaSuccess ? VA_OK : note_cuda(e);
}

va_status va_debug_split_ranges(const va_problem* p, const va_kv* kv, int32_t mode,
                                int32_t* ranges, uint32_t* status, void* stream) {
  va_status st = check(p, kv, mode);
  if (st != VA_OK) return st;
  if (!ranges) return VA_ERR_INVALID_ARG;
  if (p->num_seqs == 0) return VA_OK;
  Plan pl = make_plan(p, kv);
  Params q = make_params(p, kv, mode, pl, nullptr, nullptr, nullptr, status);
  cudaError_t e = launch_debug_split(q, (int*)ranges, (cudaStream_t)stream);
  return e == cudaSuccess ? VA_OK : note_cuda(e);
}

va_status verify_attn_promote(const va_problem* p, const va_kv* kv, int32_t mode,
                              const int32_t* accepted_len, const int32_t* accepted_nodes,
                              uint32_t* status, void* stream) {
  va_status st = check(p, kv, mode);
  if (st != VA_OK) return st;
  if (!kv->draft_k || !accepted_len || !status) return VA_ERR_INVALID_ARG;
  if (p->total_rows > 0 && !accepted_nodes) return VA_ERR_INVALID_ARG;
  Plan pl = make_plan(p, kv);
  Params q = make_params(p, kv, mode, pl, nullptr, nullptr, nullptr, status);
  cudaError_t e = launch_promote(q, accepted_len, accepted_nodes, (cudaStream_t)stream);
  return e == cudaSuccess ? VA_OK : note_cuda(e);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Verify call with library-held scratch (no allocation on the call path).
//
// The split partials go to a file-scope device array that is part of this
// module's device image: the CUDA runtime reserves it when the module is
// loaded on a device, and this library never allocates or frees it.  Its
// address on the current device is looked up once per device with
// cudaGetSymbolAddress and cached.  The partial kernel writes every (m, l)
// entry of every slot it owns before the merge kernel reads it, and the
// merge skips slots with l = 0 without reading their accumulators, so no
// part of the array has to start at zero.  One array per device serves
// every call: calls on the same stream are ordered, calls that may
// overlap in time (other streams, other host threads) race on it.

namespace va {

static __device__ __align__(256) unsigned char g_static_ws[VA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxStaticDevices = 64;
static std::atomic<void*> g_static_ws_ptr[kMaxStaticDevices];

static cudaError_t static_workspace(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxStaticDevices) return cudaErrorInvalidDevice;
  void* ptr = g_static_ws_ptr[dev].load(std::memory_order_acquire);
  if (!ptr) {
    e = cudaGetSymbolAddress(&ptr, g_static_ws);
    if (e != cudaSuccess) return e;
    if (!ptr) return cudaErrorInvalidSymbol;
    g_static_ws_ptr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return cudaSuccess;
}

}  // namespace va

extern "C" {

va_status verify_attn_noalloc(const va_problem* p, const va_kv* kv, int32_t mode, float* o,
                              float* lse, uint32_t* status, void* stream) {
  va_status st = check(p, kv, mode);
  if (st != VA_OK) return st;
  if (p->total_rows == 0) return VA_OK;
  if (!o || !lse) return VA_ERR_INVALID_ARG;
  if (!aligned16(o)) return VA_ERR_ALIGNMENT;
  Plan pl = make_plan(p, kv);
  if (ws_bytes_for(p, kv, pl) > (size_t)VA_STATIC_WORKSPACE_BYTES)
    return VA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t cs = (cudaStream_t)stream;
  st = check_stream_device(cs);
  if (st != VA_OK) return st;
  void* ws = nullptr;
  cudaError_t e = static_workspace(&ws);
  if (e != cudaSuccess) return note_cuda(e);
  Params q = make_params(p, kv, mode, pl, ws, o, lse, status);
  e = launch_partial(pl, q, cs);
  if (e != cudaSuccess) return note_cuda(e);
  e = launch_merge(q, cs);
  if (e != cudaSuccess) return note_cuda(e);
  return VA_OK;
}

}  // extern "C"
