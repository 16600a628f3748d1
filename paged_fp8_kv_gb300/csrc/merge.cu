// Merge of split-KV partial results (sequences the plan cut into > 1 chunk).
//
// Source: the "mjolnir/t5_decode.py" page, `reduction` kernel: only the
// splits a sequence ran are read (the workspace is never initialised), every
// part is rescaled to the common maximum (weight 0 for an empty part),
//   O = scale_o * sum_j w_j o_j / sum_j w_j l_j      (0 when the sum is 0)
//   LSE = max_j m_j + ln(sum_j w_j l_j),
// and unsplit sequences are left untouched (decode wrote them).
//
// kWPR warps share one (packed row, kv head, sequence) and stride over its
// splits; lane l owns d = 4l..4l+3 (16-byte loads).  Each warp keeps a
// running (max, sum, O) and folds in kUnroll splits per step, whose loads
// are all issued before any is used, so a long split list costs few memory
// round trips.  The warp results are combined in a fixed order: the result
// does not depend on timing.  kWPR follows the longest split list (1 warp
// per row for a few splits, 16 for hundreds).

#include <cuda_runtime.h>

#include "mj_kernels.h"

namespace mj {
namespace {

constexpr int kCtaWarps = 4;  // warps per CTA when a row needs fewer
constexpr int kUnroll = 8;

struct Running {
  float m, l, o[4];
};

// Folds part (mj, lj, oj) into r: both rescaled to the larger maximum.
__device__ __forceinline__ void fold(Running& r, float mj, float lj, const float4& oj) {
  if (mj == -INFINITY) return;  // an empty part adds nothing
  const float mn = fmaxf(r.m, mj);
  const float a = (r.m == -INFINITY) ? 0.f : __expf(r.m - mn);
  const float w = __expf(mj - mn);
  r.l = fmaf(r.l, a, w * lj);
  r.o[0] = fmaf(r.o[0], a, w * oj.x);
  r.o[1] = fmaf(r.o[1], a, w * oj.y);
  r.o[2] = fmaf(r.o[2], a, w * oj.z);
  r.o[3] = fmaf(r.o[3], a, w * oj.w);
  r.m = mn;
}

template <int kWPR>
__global__ void __launch_bounds__((kWPR > kCtaWarps ? kWPR : kCtaWarps) * 32) merge_kernel(const DecodeDev a) {
  constexpr int kRows = kWPR >= kCtaWarps ? 1 : kCtaWarps / kWPR;  // rows per CTA
  constexpr int kMergeWarps = kWPR;
  const int lane = threadIdx.x & 31;
  const int rsub = (threadIdx.x >> 5) / kWPR;  // row within the CTA
  const int warp = (threadIdx.x >> 5) % kWPR;  // warp within the row
  const int n = blockIdx.x * kRows + rsub, g = blockIdx.y, b = blockIdx.z;
  int nsp = a.n_splits[b];
  if (nsp <= 1) return;  // uniform over the CTA
  nsp = nsp < a.max_splits ? nsp : a.max_splits;
  const bool live = n < a.n_q;

  __shared__ float s_m[kRows][kMergeWarps], s_l[kRows][kMergeWarps];
  __shared__ __align__(16) float s_o[kRows][kMergeWarps][kHeadDimDev];

  Running r{-INFINITY, 0.f, {0.f, 0.f, 0.f, 0.f}};
  const int64_t row0 = part_row(a, b, g, 0, live ? n : 0);
  const int64_t split_stride = a.n_q;  // rows between consecutive slots
  for (int j0 = warp; live && j0 < nsp; j0 += kMergeWarps * kUnroll) {
    float mj[kUnroll], lj[kUnroll];
    float4 oj[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = j0 + u * kMergeWarps;
      mj[u] = -INFINITY;
      lj[u] = 0.f;
      oj[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < nsp) {
        const int64_t pr = row0 + j * split_stride;
        mj[u] = a.m_part[pr];
        lj[u] = a.l_part[pr];
        oj[u] = *reinterpret_cast<const float4*>(&a.o_part[pr * kHeadDimDev + lane * 4]);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) fold(r, mj[u], lj[u], oj[u]);
  }
  if (lane == 0) {
    s_m[rsub][warp] = r.m;
    s_l[rsub][warp] = r.l;
  }
  *reinterpret_cast<float4*>(&s_o[rsub][warp][lane * 4]) = make_float4(r.o[0], r.o[1], r.o[2], r.o[3]);
  __syncthreads();

  // combine: 128 threads per row (kRows rows per CTA share the CTA's threads)
  const int tpr = blockDim.x / kRows;  // threads per row, >= 32
  const int cr = threadIdx.x / tpr;
  const int cn = blockIdx.x * kRows + cr;
  for (int d = threadIdx.x % tpr; cn < a.n_q && d < kHeadDimDev; d += tpr) {
    float m_all = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) m_all = fmaxf(m_all, s_m[cr][w]);
    float l_all = 0.f, o_all = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float ww = (s_m[cr][w] == -INFINITY) ? 0.f : __expf(s_m[cr][w] - m_all);
      l_all = fmaf(ww, s_l[cr][w], l_all);
      o_all = fmaf(ww, s_o[cr][w][d], o_all);
    }
    const float inv = l_all > 0.f ? a.scale_o / l_all : 0.f;
    const int64_t orow = b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + cn) * kHeadDimDev;
    a.o[orow + d] = __float2bfloat16_rn(o_all * inv);
    if (d == 0) a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + cn] = m_all + logf(l_all);
  }
}

template <int kWPR>
cudaError_t launch_merge_t(const DecodeDev& a, cudaStream_t stream) {
  constexpr int kRows = kWPR >= kCtaWarps ? 1 : kCtaWarps / kWPR;
  constexpr int kThreads = (kWPR > kCtaWarps ? kWPR : kCtaWarps) * 32;
  dim3 grid((a.n_q + kRows - 1) / kRows, a.h_k, a.num_seqs);
  merge_kernel<kWPR><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const DecodeDev& a, int max_n_splits, cudaStream_t stream) {
  // about kUnroll splits per warp in one round of loads
  if (max_n_splits <= kUnroll) return launch_merge_t<1>(a, stream);
  if (max_n_splits <= 4 * kUnroll) return launch_merge_t<4>(a, stream);
  return launch_merge_t<16>(a, stream);
}

}  // namespace mj
