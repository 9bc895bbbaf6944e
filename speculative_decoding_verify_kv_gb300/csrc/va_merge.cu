// Merge of the split partials.
//
// Per (row, head): M = max over live slots of m_s, then l = sum 2^(m_s - M)
// l_s and acc = sum 2^(m_s - M) acc_s, O = acc / l and LSE = (M + log2 l)
// * ln 2.  A slot with l = 0 is an empty chunk and is skipped; a NaN slot
// (device-detected error) makes the row NaN.  The summation order is fixed
// (slots of a group in ascending order, then groups in ascending order), so
// a row's output depends only on its own slots.  Rows of a sequence whose
// row range is inconsistent (VA_DEV_BAD_ROWS) are NaN.
//
// Restated from hipfire PR #817 "FA2 split-KV" sections "Summary" and
// "Performance" (S8 partials combined by a merge pass; S1 equals the
// unsplit result) and hipfire PR #695 alpineQ comments (the reducer of the
// batched-partials layout).
#include <string.h>

#include "va_common.cuh"

namespace va {

constexpr int kMergeThreads = 256;

// One CTA per (row, head): D/4 column threads x (256 / (D/4)) slot groups.
// Group g takes slots g, g + NG, ... in ascending order and issues every
// load of its slots (m, l and a float4 of acc, up to BATCH at once) before
// using any, so the merge costs one round trip to the partials up to
// NG x BATCH slots (40 at D = 256: the 38 of a long-context call).  The
// register cap keeps three CTAs on an SM, so a call's merge CTAs (384 at
// 16 rows x 24 heads) run in one wave on 152 SMs.  Each group keeps its own
// maximum M_g; the groups are then combined in ascending group order with
// the overall maximum M:  l = sum_g 2^(M_g - M) l_g, acc likewise.
template <int D>
__global__ void __launch_bounds__(kMergeThreads, 3) merge_kernel(const Params p) {
  constexpr int TC = D / 4;
  constexpr int NG = kMergeThreads / TC;
  constexpr int BATCH = 10;  // slots per group loaded together
  __shared__ float4 red[NG][TC];
  __shared__ float lred[NG], mred[NG];
  // Launched as a programmatic dependent of the partial kernel: wait here
  // until that grid has finished and its writes are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // A programmatic dependent launched after this kernel (the next call's
  // partial kernel) may now become resident; it waits for this grid to
  // complete before it touches memory.
  asm volatile("griddepcontrol.launch_dependents;");
  const long long item = blockIdx.x;
  const int grow = (int)(item / p.H), h = (int)(item % p.H);
  const int tcol = threadIdx.x % TC, grp = threadIdx.x / TC;
  float Mg = -INFINITY, lg = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // The row's sequence: the last s with cu_rows[s] <= row.  A row that no
  // sequence covers, or whose sequence has inconsistent rows (the partial
  // kernel flags VA_DEV_BAD_ROWS and writes none of its slots), comes out
  // NaN, so that scratch left by an earlier call never reaches O.
  int s_lo = 0, s_hi = p.num_seqs - 1;
  while (s_lo < s_hi) {
    const int mid = (s_lo + s_hi + 1) >> 1;
    if (p.cu_rows[mid] <= grow) s_lo = mid;
    else s_hi = mid - 1;
  }
  int sr0, sn, sctx;
  int nan = !(p.cu_rows[s_lo] <= grow && grow < p.cu_rows[s_lo + 1]) ||
            (check_sequence(p, s_lo, &sr0, &sn, &sctx) & VA_DEV_BAD_ROWS) != 0u;
  // Slots past the sequence's last non-empty chunk hold nothing of this
  // call: with one level of chunks they are the trailing empty ones of the
  // partial kernels' sub_range cut, so only the first `live` are read (at
  // least one: a sequence with rows has a non-empty span).
  int live = p.slots;
  if (!nan && p.S == 1 && sctx >= 0) {
    int lo0, hi0;
    split_range(sctx + sn, 1, 0, &lo0, &hi0);
    live = max(1, live_subs(lo0, hi0, seq_subs(p, sn), p.min_sub));
  }
  for (int s0 = grp; s0 < live && !nan; s0 += BATCH * NG) {
    float mm[BATCH], ll[BATCH];
    float4 aa[BATCH];
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      const int sl = s0 + k * NG;
      mm[k] = -INFINITY;
      ll[k] = 0.f;
      aa[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (sl < live) {
        const long long si = slot_index(p, sl, grow, h);
        mm[k] = p.ws_ml[2 * si];
        ll[k] = p.ws_ml[2 * si + 1];
        aa[k] = *reinterpret_cast<const float4*>(p.ws_acc + si * D + 4 * tcol);
      }
    }
    // A slot with l = 0 is an empty chunk (its acc is never read as data);
    // a NaN (m, l) is a device-detected error and poisons the row.
    float bm = Mg;
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      if (isnan(mm[k]) || isnan(ll[k])) nan = 1;
      if (ll[k] > 0.f) bm = fmaxf(bm, mm[k]);
    }
    if (bm > Mg) {
      const float f = exp2f(Mg - bm);  // 0 while nothing was live
      lg *= f;
      acc.x *= f;
      acc.y *= f;
      acc.z *= f;
      acc.w *= f;
      Mg = bm;
    }
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      if (!(ll[k] > 0.f)) continue;
      const float w = exp2f(mm[k] - Mg);
      lg = fmaf(w, ll[k], lg);
      acc.x = fmaf(w, aa[k].x, acc.x);
      acc.y = fmaf(w, aa[k].y, acc.y);
      acc.z = fmaf(w, aa[k].z, acc.z);
      acc.w = fmaf(w, aa[k].w, acc.w);
    }
  }
  red[grp][tcol] = acc;
  if (tcol == 0) {
    lred[grp] = lg;
    mred[grp] = Mg;
  }
  const bool bad = __syncthreads_or(nan) != 0;
  if (grp == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < NG; ++g)
      if (lred[g] > 0.f) M = fmaxf(M, mred[g]);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    float lt = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      if (!(lred[g] > 0.f)) continue;
      const float w = exp2f(mred[g] - M);
      const float4 b = red[g][tcol];
      t.x = fmaf(w, b.x, t.x);
      t.y = fmaf(w, b.y, t.y);
      t.z = fmaf(w, b.z, t.z);
      t.w = fmaf(w, b.w, t.w);
      lt = fmaf(w, lred[g], lt);
    }
    const float inv = 1.f / lt;
    float4 out = bad ? make_float4(NAN, NAN, NAN, NAN)
                     : make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
    *reinterpret_cast<float4*>(p.o + item * D + 4 * tcol) = out;
    if (tcol == 0) p.lse[item] = bad ? NAN : (M + log2f(lt)) * kLn2;
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
