// Merge of the split partials.
//
// Per (row, head): M = max over live slots of m_s, then l = sum 2^(m_s - M)
// l_s and acc = sum 2^(m_s - M) acc_s, O = acc / l and LSE = (M + log2 l)
// * ln 2.  A slot with l = 0 is an empty chunk and is skipped; a NaN slot
// (device-detected error) makes the row NaN.  The summation order is fixed
// (slot groups in ascending order, then groups in ascending order), so a
// row's output depends only on its own slots.
//
// Restated from hipfire PR #817 "FA2 split-KV" sections "Summary" and
// "Performance" (S8 partials combined by a merge pass; S1 equals the
// unsplit result) and hipfire PR #695 alpineQ comments (the reducer of the
// batched-partials layout).
#include <string.h>

#include "va_common.cuh"

namespace va {

constexpr int kMergeThreads = 256;

// One CTA per (row, head).  Warp 0 finds M over the live slots; then D/4
// column threads x (256 / (D/4)) slot groups accumulate float4 columns of
// their slots, and the groups are added in fixed group order.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const Params p) {
  constexpr int TC = D / 4;
  constexpr int NG = kMergeThreads / TC;
  __shared__ float4 red[NG][TC];
  __shared__ float lred[NG];
  __shared__ float M_s;
  __shared__ int nan_s;
  // Launched as a programmatic dependent of the partial kernel: wait here
  // until that grid has finished and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long item = blockIdx.x;
  const int grow = (int)(item / p.H), h = (int)(item % p.H);
  const int tcol = threadIdx.x % TC, grp = threadIdx.x / TC;
  if (threadIdx.x < 32) {
    float M = -INFINITY;
    int nan = 0;
    for (int sl = threadIdx.x; sl < p.slots; sl += 32) {
      const long long si = slot_index(p, sl, grow, h);
      const float m = p.ws_ml[2 * si], l = p.ws_ml[2 * si + 1];
      if (isnan(m) || isnan(l)) nan = 1;
      if (l > 0.f) M = fmaxf(M, m);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      nan |= __shfl_xor_sync(0xffffffffu, nan, o);
    }
    if (threadIdx.x == 0) {
      M_s = M;
      nan_s = nan;
    }
  }
  __syncthreads();
  const float M = M_s;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
  // Slots grp, grp+NG, ... in batches of 8 with every load of a batch in
  // flight before any is used.
  for (int s0 = grp; s0 < p.slots; s0 += 8 * NG) {
    float mm[8], ll[8];
    float4 aa[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int sl = s0 + k * NG;
      mm[k] = 0.f;
      ll[k] = 0.f;
      if (sl < p.slots) {
        const long long si = slot_index(p, sl, grow, h);
        mm[k] = p.ws_ml[2 * si];
        ll[k] = p.ws_ml[2 * si + 1];
        aa[k] = *reinterpret_cast<const float4*>(p.ws_acc + si * D + 4 * tcol);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (!(ll[k] > 0.f)) continue;
      const float w = exp2f(mm[k] - M);
      lsum = fmaf(w, ll[k], lsum);
      acc.x = fmaf(w, aa[k].x, acc.x);
      acc.y = fmaf(w, aa[k].y, acc.y);
      acc.z = fmaf(w, aa[k].z, acc.z);
      acc.w = fmaf(w, aa[k].w, acc.w);
    }
  }
  red[grp][tcol] = acc;
  if (tcol == 0) lred[grp] = lsum;
  __syncthreads();
  if (grp == 0) {
    float4 t = red[0][tcol];
    float lt = lred[0];
#pragma unroll
    for (int g = 1; g < NG; ++g) {
      const float4 b = red[g][tcol];
      t.x += b.x;
      t.y += b.y;
      t.z += b.z;
      t.w += b.w;
      lt += lred[g];
    }
    const bool nan = nan_s != 0;
    const float inv = 1.f / lt;
    float4 out = nan ? make_float4(NAN, NAN, NAN, NAN)
                     : make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
    *reinterpret_cast<float4*>(p.o + item * D + 4 * tcol) = out;
    if (tcol == 0) p.lse[item] = nan ? NAN : (M + log2f(lt)) * kLn2;
  }
}

template <int D>
static cudaError_t launch_merge_t(const Params& p, cudaStream_t st, long long items) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)items);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel<D>, p);
}

cudaError_t launch_merge(const Params& p, cudaStream_t st) {
  long long items = (long long)p.total_rows * p.H;
  if (items == 0) return cudaSuccess;
  cudaError_t e;
  switch (p.D) {
    case 64: e = launch_merge_t<64>(p, st, items); break;
    case 128: e = launch_merge_t<128>(p, st, items); break;
    case 256: e = launch_merge_t<256>(p, st, items); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace va
