// CUDA-core split-KV partial kernel.
//
// One CTA owns (sequence, KV head, split, sub-chunk, block of 16 query rows)
// and walks its token range in tiles of 32 tokens: decode K/V into shared
// memory as fp32, score every (row, token) pair, mask, update the online
// softmax (m in log2 units, l) and accumulate P.V in registers.  It writes
// one fp32 partial (m, l, acc[D]) per (row, head) into its slot of the
// workspace; the merge kernel combines the slots.
//
// This is the kernel for the fp32 cache and for row blocks too small to
// fill a tensor-core tile; it serves every dtype, so tests can also run it
// as a second implementation next to the tensor-core kernel.
//
// Restated from: hipfire PR #817 "FA2 split-KV" sections "Summary" and
// "Performance" (split partials + merge), hipfire PR #695 alpineQ comments
// (one block serves several verifier rows from one KV fetch), lucebox PR
// #686 "State and commit invariants" (tree ancestry masks).
#include <string.h>

#include "va_common.cuh"

namespace va {

constexpr int kSimtRows = 16;    // query rows per CTA
constexpr int kSimtTile = 32;    // tokens per tile
constexpr int kSimtThreads = 128;

template <int D>
constexpr int simt_smem_floats() {
  return kSimtRows * D + kSimtTile * (D + 1) + kSimtTile * D + kSimtRows * kSimtTile;
}

template <int D, int KVT>
__global__ void __launch_bounds__(kSimtThreads) simt_partial_kernel(const Params p) {
  constexpr int NK = D / 32;  // accumulator columns per lane
  extern __shared__ float sm[];
  float* Qs = sm;                              // [16][D]
  float* Ks = Qs + kSimtRows * D;              // [32][D+1]
  float* Vs = Ks + kSimtTile * (D + 1);        // [32][D]
  float* Ps = Vs + kSimtTile * D;              // [16][32]
  __shared__ float alpha_s[kSimtRows];
  __shared__ unsigned mask_s[kSimtRows];
  __shared__ int bad_s;

  // The merge kernel may launch now; it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;");
  // Programmatic dependent of the preceding work on the stream: nothing is
  // read or written before that work has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kvh = blockIdx.y, s = blockIdx.z;

  int row0, n, ctx;
  unsigned err = check_sequence(p, s, &row0, &n, &ctx);
  if (err & VA_DEV_BAD_ROWS) {
    if (tid == 0) flag(p.status, err);
    return;  // the rows of this sequence are unknown
  }
  // Row block and chunk (one level of chunks: split 0, slot = chunk).
  int rb, sub, nsub;
  if (!cta_work(p, n, blockIdx.x, &rb, &sub, &nsub)) return;
  const int split = 0, slot = sub;
  const int R = n * p.G;
  const int rbase = rb * kSimtRows;
  if (rbase >= R) return;
  const int nrows = min(kSimtRows, R - rbase);
  const int L = ctx + n;
  const int kind = seq_kind_of(p, s);
  const bool scratch = uses_scratch(p, kind);  // drafts from the tree scratch KV

  if (tid == 0) bad_s = 0;
  __syncthreads();
  if (tid < nrows) {
    int j = (rbase + tid) / p.G;
    bool bad = false;
    mask_s[tid] = row_mask(kind, p.parent + row0, j, &bad);
    if (bad) atomicOr(&bad_s, 1);
  }
  __syncthreads();
  if (bad_s) err |= VA_DEV_BAD_PARENT;

  int lo, hi, slo, shi;
  split_range(L, p.S, split, &lo, &hi);
  sub_range(lo, hi, nsub, p.min_sub, sub, &slo, &shi);

  // Q rows of this block -> shared (fp32).
  for (int i = tid; i < nrows * D; i += kSimtThreads) {
    int rl = i / D, d = i % D;
    int r = rbase + rl, j = r / p.G, g = r % p.G;
    long long qi = ((long long)(row0 + j) * p.H + (kvh * p.G + g)) * D + d;
    Qs[rl * D + d] = load_q(p, qi);
  }

  float m_run[4], l_run[4];
  float acc[4][NK];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int k = 0; k < NK; ++k) acc[i][k] = 0.f;
  }

  if (!err) {
    for (int t0 = slo; t0 < shi; t0 += kSimtTile) {
      __syncthreads();
      // Decode the K/V tile; tokens past the range become zeros.
      for (int i = tid; i < kSimtTile * D; i += kSimtThreads) {
        int t = i / D, d = i % D;
        int tok = t0 + t;
        float kx = 0.f, vx = 0.f;
        if (tok < shi && tok >= ctx && scratch) {
          const long long row = scratch_row(p, row0, kvh, tok - ctx);
          kx = load_kv<KVT>(p.dk, row, p.row_bytes, d);
          vx = load_kv<KVT>(p.dv, row, p.row_bytes, d);
        } else if (tok < shi) {
          long long row = kv_row(p, s, kvh, tok);
          if (row < 0) {
            atomicOr(&bad_s, 2);
          } else {
            kx = load_kv<KVT>(p.k, row, p.row_bytes, d);
            vx = load_kv<KVT>(p.v, row, p.row_bytes, d);
          }
        }
        Ks[t * (D + 1) + d] = kx;
        Vs[t * D + d] = vx;
      }
      __syncthreads();
      if (bad_s & 2) {
        err |= VA_DEV_BAD_BLOCK;
        break;
      }
      // Scores: lane = token, rows warp + 4i.
      const int tok = t0 + lane;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = warp + 4 * i;
        if (rl >= nrows) continue;
        float dot = 0.f;
#pragma unroll 8
        for (int d = 0; d < D; ++d) dot = fmaf(Qs[rl * D + d], Ks[lane * (D + 1) + d], dot);
        bool vis = tok < shi &&
                   (tok < ctx || draft_visible(kind, mask_s[rl], (rbase + rl) / p.G, tok - ctx));
        float s2 = vis ? dot * p.scale_log2 : -INFINITY;
        float mt = s2;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        float m_new = fmaxf(m_run[i], mt);
        float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run[i] - m_new);
        float pr = vis ? exp2f(s2 - m_new) : 0.f;
        float ps = pr;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l_run[i] = l_run[i] * alpha + ps;
        m_run[i] = m_new;
        Ps[rl * kSimtTile + lane] = pr;
        if (lane == 0) alpha_s[rl] = alpha;
      }
      __syncthreads();
      // acc[row][d] = alpha * acc + sum_t P[row][t] V[t][d]; lane owns d = lane + 32k.
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = warp + 4 * i;
        if (rl >= nrows) continue;
        const float a = alpha_s[rl];
#pragma unroll
        for (int k = 0; k < NK; ++k) acc[i][k] *= a;
        for (int t = 0; t < kSimtTile; ++t) {
          const float pv = Ps[rl * kSimtTile + t];
#pragma unroll
          for (int k = 0; k < NK; ++k) acc[i][k] = fmaf(pv, Vs[t * D + lane + 32 * k], acc[i][k]);
        }
      }
    }
  }
  if (err) {
    if (tid == 0) flag(p.status, err);
  }
  // Write this CTA's slot for its rows (an empty range writes l = 0).
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = warp + 4 * i;
    if (rl >= nrows) continue;
    const int r = rbase + rl, j = r / p.G, g = r % p.G;
    const int grow = row0 + j, h = kvh * p.G + g;
    const long long si = slot_index(p, slot, grow, h);
    if (lane == 0) {
      p.ws_ml[2 * si] = err ? NAN : m_run[i];
      p.ws_ml[2 * si + 1] = err ? NAN : l_run[i];
    }
    float* dst = p.ws_acc + si * D;
#pragma unroll
    for (int k = 0; k < NK; ++k) dst[lane + 32 * k] = acc[i][k];
  }
}

template <int D, int KVT>
static cudaError_t launch_simt_t(const Params& p, dim3 grid, cudaStream_t st) {
  constexpr int smem = simt_smem_floats<D>() * 4;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(simt_partial_kernel<D, KVT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kSimtThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, simt_partial_kernel<D, KVT>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int simt_smem_bytes(int D) {
  switch (D) {
    case 64: return simt_smem_floats<64>() * 4;
    case 128: return simt_smem_floats<128>() * 4;
    default: return simt_smem_floats<256>() * 4;
  }
}

cudaError_t launch_simt_partial(const Params& p, dim3 grid, cudaStream_t st) {
#define VA_SIMT_CASE(DD, KT) \
  if (p.D == DD && p.kv_dtype == KT) return launch_simt_t<DD, KT>(p, grid, st);
  VA_SIMT_CASE(64, VA_F32) VA_SIMT_CASE(64, VA_BF16) VA_SIMT_CASE(64, VA_Q8_0)
  VA_SIMT_CASE(128, VA_F32) VA_SIMT_CASE(128, VA_BF16) VA_SIMT_CASE(128, VA_Q8_0)
  VA_SIMT_CASE(256, VA_F32) VA_SIMT_CASE(256, VA_BF16) VA_SIMT_CASE(256, VA_Q8_0)
#undef VA_SIMT_CASE
  return cudaErrorInvalidValue;
}

}  // namespace va
