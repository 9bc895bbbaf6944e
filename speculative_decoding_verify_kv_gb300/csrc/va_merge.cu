// Warp-level merge of the split partials.
//
// One warp per (row, head): M = max over live slots of m_s, then in
// ascending slot order l = sum 2^(m_s - M) l_s and acc = sum 2^(m_s - M)
// acc_s; O = acc / l and LSE = (M + log2 l) * ln 2.  A slot with l = 0 is
// an empty chunk and is skipped; a NaN slot (device-detected error) makes
// the row NaN.  The order is fixed, so a row's output depends only on its
// own slots.
//
// Restated from hipfire PR #817 "FA2 split-KV" sections "Summary" and
// "Performance" (S8 partials combined by a merge pass; S1 equals the
// unsplit result) and hipfire PR #695 alpineQ comments (the reducer of the
// batched-partials layout).
#include "va_common.cuh"

namespace va {

constexpr int kMergeWarps = 8;

template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const Params p) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const long long item = (long long)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const long long items = (long long)p.total_rows * p.H;
  if (item >= items) return;
  const int grow = (int)(item / p.H), h = (int)(item % p.H);

  float M = -INFINITY;
  bool nan = false;
  for (int sl = 0; sl < p.slots; ++sl) {
    long long si = slot_index(p, sl, grow, h);
    float m = p.ws_ml[2 * si], l = p.ws_ml[2 * si + 1];
    if (isnan(m) || isnan(l)) nan = true;
    if (l > 0.f) M = fmaxf(M, m);
  }
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  float lsum = 0.f;
  for (int sl = 0; sl < p.slots; ++sl) {
    long long si = slot_index(p, sl, grow, h);
    float m = p.ws_ml[2 * si], l = p.ws_ml[2 * si + 1];
    if (!(l > 0.f)) continue;
    float w = exp2f(m - M);
    lsum = fmaf(w, l, lsum);
    const float* a = p.ws_acc + si * D;
#pragma unroll
    for (int k = 0; k < PER; ++k) acc[k] = fmaf(w, a[lane + 32 * k], acc[k]);
  }
  const float inv = 1.f / lsum;
  float* o = p.o + item * D;
#pragma unroll
  for (int k = 0; k < PER; ++k) o[lane + 32 * k] = nan ? NAN : acc[k] * inv;
  if (lane == 0) p.lse[item] = nan ? NAN : (M + log2f(lsum)) * kLn2;
}

cudaError_t launch_merge(const Params& p, cudaStream_t st) {
  long long items = (long long)p.total_rows * p.H;
  if (items == 0) return cudaSuccess;
  dim3 grid((unsigned)((items + kMergeWarps - 1) / kMergeWarps));
  switch (p.D) {
    case 64: merge_kernel<64><<<grid, kMergeWarps * 32, 0, st>>>(p); break;
    case 128: merge_kernel<128><<<grid, kMergeWarps * 32, 0, st>>>(p); break;
    case 256: merge_kernel<256><<<grid, kMergeWarps * 32, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace va
