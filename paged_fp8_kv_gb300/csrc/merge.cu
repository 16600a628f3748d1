// Merge of split-KV partial results (sequences the plan cut into > 1 chunk).
//
// Source: the "mjolnir/t5_decode.py" page, `reduction` kernel: only the
// splits a sequence ran are read (the workspace is never initialised), every
// part is rescaled to the common maximum (weight 0 for an empty part),
//   O = scale_o * sum_j w_j o_j / sum_j w_j l_j      (0 when the sum is 0)
//   LSE = max_j m_j + ln(sum_j w_j l_j),
// and unsplit sequences are left untouched (decode wrote them).
//
// One CTA per (packed row, kv head, sequence); 8 warps stride over the
// splits, lane l owns d = 4l..4l+3 (16-byte loads); the 8 warp results are
// combined in a fixed order, so the result does not depend on timing.

#include <cuda_runtime.h>

#include "mj_kernels.h"

namespace mj {
namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const DecodeDev a) {
  const int n = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  int nsp = a.n_splits[b];
  if (nsp <= 1) return;
  nsp = nsp < a.max_splits ? nsp : a.max_splits;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  __shared__ __align__(16) float s_o[kMergeWarps][kHeadDimDev];

  // pass 1: this warp's maximum
  float m_w = -INFINITY;
  for (int j = warp; j < nsp; j += kMergeWarps) m_w = fmaxf(m_w, a.m_part[part_row(a, b, g, j, n)]);
  // pass 2: rescaled sums
  float l_w = 0.f;
  float4 o_w = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int j = warp; j < nsp; j += kMergeWarps) {
    const int64_t pr = part_row(a, b, g, j, n);
    const float mj = a.m_part[pr];
    const float lj = a.l_part[pr];
    const float4 oj = *reinterpret_cast<const float4*>(&a.o_part[pr * kHeadDimDev + lane * 4]);
    const float wj = (mj == -INFINITY) ? 0.f : __expf(mj - m_w);
    l_w = fmaf(wj, lj, l_w);
    o_w.x = fmaf(wj, oj.x, o_w.x);
    o_w.y = fmaf(wj, oj.y, o_w.y);
    o_w.z = fmaf(wj, oj.z, o_w.z);
    o_w.w = fmaf(wj, oj.w, o_w.w);
  }
  if (lane == 0) {
    s_m[warp] = m_w;
    s_l[warp] = l_w;
  }
  *reinterpret_cast<float4*>(&s_o[warp][lane * 4]) = o_w;
  __syncthreads();

  if (threadIdx.x < kHeadDimDev) {
    const int d = threadIdx.x;
    float m_all = -INFINITY;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) m_all = fmaxf(m_all, s_m[w]);
    float l_all = 0.f, o_all = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float ww = (s_m[w] == -INFINITY) ? 0.f : __expf(s_m[w] - m_all);
      l_all = fmaf(ww, s_l[w], l_all);
      o_all = fmaf(ww, s_o[w][d], o_all);
    }
    const float inv = l_all > 0.f ? a.scale_o / l_all : 0.f;
    const int64_t orow = b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + n) * kHeadDimDev;
    a.o[orow + d] = __float2bfloat16_rn(o_all * inv);
    if (d == 0) a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + n] = m_all + logf(l_all);
  }
}

}  // namespace

cudaError_t launch_merge(const DecodeDev& a, cudaStream_t stream) {
  dim3 grid(a.n_q, a.h_k, a.num_seqs);
  merge_kernel<<<grid, kMergeWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mj
