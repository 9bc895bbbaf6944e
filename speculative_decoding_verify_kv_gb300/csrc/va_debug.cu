// Debug exports of the row map, ancestor masks and KV gather: they call the
// same device functions the partial kernels use, so a bit-exact comparison
// with the oracle checks the kernels' own indexing.
#include "va_common.cuh"

namespace va {

// One block per sequence, its threads striding over the local rows.
__global__ void debug_row_map_kernel(const Params p, int* row_seq, unsigned* anc) {
  const int s = blockIdx.x;
  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  if (err & VA_DEV_BAD_ROWS) {
    if (threadIdx.x == 0) flag(p.status, err & VA_DEV_BAD_ROWS);
    return;
  }
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    bool bad = false;
    unsigned m = row_mask(seq_kind_of(p, s), p.parent + row0, j, &bad);
    if (bad) flag(p.status, VA_DEV_BAD_PARENT);
    row_seq[row0 + j] = s;
    anc[row0 + j] = m;
  }
}

// One thread per (sequence, token < max_len).
__global__ void debug_gather_kernel(const Params p, int kvh, long long max_len, long long* out) {
  const int s = blockIdx.y;
  const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= max_len) return;
  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  long long L = (long long)ctx + n;
  long long v = -1;
  if (err) {
    if (t == 0) flag(p.status, err);
  } else if (t < L) {
    v = kv_row(p, s, kvh, (int)t);
    if (v < 0) flag(p.status, VA_DEV_BAD_BLOCK);
  }
  out[(long long)s * max_len + t] = v;
}

// One block per sequence, its threads striding over the slots: each
// chunk's [lo, hi) exactly as the partial kernels compute it.
__global__ void debug_split_kernel(const Params p, int* ranges) {
  const int s = blockIdx.x;
  int row0, n, ctx;
  const unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  for (int j = threadIdx.x; j < p.slots; j += blockDim.x) {
    int slo = -1, shi = -1;
    if (!(err & VA_DEV_BAD_ROWS)) {
      int lo, hi;
      split_range(ctx + n, p.S, 0, &lo, &hi);
      sub_range(lo, hi, seq_subs(p, n), p.min_sub, j, &slo, &shi);
    }
    ranges[2 * ((long long)s * p.slots + j)] = slo;
    ranges[2 * ((long long)s * p.slots + j) + 1] = shi;
  }
  if (threadIdx.x == 0 && (err & VA_DEV_BAD_ROWS)) flag(p.status, err & VA_DEV_BAD_ROWS);
}

cudaError_t launch_debug_split(const Params& p, int* ranges, cudaStream_t st) {
  debug_split_kernel<<<p.num_seqs, 64, 0, st>>>(p, ranges);
  return cudaGetLastError();
}

cudaError_t launch_debug_row_map(const Params& p, int* row_seq, unsigned* anc, cudaStream_t st) {
  debug_row_map_kernel<<<p.num_seqs, 32, 0, st>>>(p, row_seq, anc);
  return cudaGetLastError();
}

cudaError_t launch_debug_gather(const Params& p, int kvh, long long max_len, long long* out,
                                cudaStream_t st) {
  dim3 grid((unsigned)((max_len + 255) / 256), p.num_seqs);
  debug_gather_kernel<<<grid, 256, 0, st>>>(p, kvh, max_len, out);
  return cudaGetLastError();
}

}  // namespace va
