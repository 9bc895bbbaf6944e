// Tree commit of the KV cache: copy the accepted path of each tree sequence
// from the tree scratch KV into the durable cache, as one transaction
// (lucebox PR #686, "State and commit invariants": tree rows write scratch
// KV, the commit transaction promotes only the accepted prefix, and it
// checks every domain before it mutates any).
#include "va_common.cuh"

namespace va {

// Preflight, one thread per sequence: the rows, the accepted path (a root
// path of the tree: parent[nodes[0]] == -1, parent[nodes[i]] == nodes[i-1])
// and the destination positions ctx .. ctx+m-1 (capacity, block table).
// Errors go to the status word, which the copy kernel reads before writing.
__global__ void promote_check_kernel(const Params p, const int* acc_len, const int* nodes) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= p.num_seqs) return;
  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  if (err) {
    flag(p.status, err);
    return;
  }
  const int m = acc_len[s];
  if (m < 0 || m > n || (m > 0 && seq_kind_of(p, s) != 1)) {
    flag(p.status, VA_DEV_BAD_ROWS);
    return;
  }
  int prev = -1;
  for (int i = 0; i < m; ++i) {
    const int a = nodes[row0 + i];
    if (a < 0 || a >= n) {
      flag(p.status, VA_DEV_BAD_ROWS);
      return;
    }
    if (p.parent[row0 + a] != prev) {
      flag(p.status, VA_DEV_BAD_PARENT);
      return;
    }
    prev = a;
  }
  const long long end = (long long)ctx + m;
  if (p.page_size == 0) {
    if (end > p.capacity) flag(p.status, VA_DEV_CTX_OVERFLOW);
  } else {
    const long long pages = (end + kPage - 1) / kPage;
    if (pages > p.max_blocks) {
      flag(p.status, VA_DEV_CTX_OVERFLOW);
      return;
    }
    for (long long pg = ctx / kPage; pg < pages; ++pg) {
      const int blk = p.block_table[(long long)s * p.max_blocks + pg];
      if (blk < 0 || blk >= p.num_blocks) {
        flag(p.status, VA_DEV_BAD_BLOCK);
        return;
      }
    }
  }
}

// Copy, one block per (sequence, KV head, tensor): path row i of sequence s
// (scratch row cu_rows[s] + nodes[i]) -> cache position ctx + i, in 32-bit
// words.  Nothing is written when the status word carries any bit.
__global__ void promote_copy_kernel(const Params p, const int* acc_len, const int* nodes) {
  if (*reinterpret_cast<volatile const unsigned*>(p.status) != 0u) return;
  const int s = blockIdx.x, kvh = blockIdx.y, kv = blockIdx.z;
  const int row0 = p.cu_rows[s], ctx = p.ctx_len[s], m = acc_len[s];
  const int W = p.row_bytes / 4;
  const uint32_t* src = reinterpret_cast<const uint32_t*>(kv ? p.dv : p.dk);
  uint32_t* dst = reinterpret_cast<uint32_t*>(const_cast<void*>(kv ? p.v : p.k));
  for (int w = threadIdx.x; w < m * W; w += blockDim.x) {
    const int i = w / W, c = w % W;
    const long long srow = scratch_row(p, row0, kvh, nodes[row0 + i]);
    const long long drow = kv_row(p, s, kvh, ctx + i);
    dst[drow * W + c] = src[srow * W + c];
  }
}

cudaError_t launch_promote(const Params& p, const int* acc_len, const int* nodes,
                           cudaStream_t st) {
  promote_check_kernel<<<(p.num_seqs + 127) / 128, 128, 0, st>>>(p, acc_len, nodes);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  promote_copy_kernel<<<dim3(p.num_seqs, p.KVH, 2), 256, 0, st>>>(p, acc_len, nodes);
  return cudaGetLastError();
}

}  // namespace va
