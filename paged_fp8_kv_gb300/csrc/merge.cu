// Merge of split-KV partial results (sequences the plan cut into > 1 chunk).
//
// Source: the "mjolnir/t5_decode.py" page, `reduction` kernel: only the
// splits a sequence ran are read (the workspace is never initialised), every
// part is rescaled to the common maximum (weight 0 for an empty part),
//   O = scale_o * sum_j w_j o_j / sum_j w_j l_j      (0 when the sum is 0)
//   LSE = max_j m_j + ln(sum_j w_j l_j),
// and unsplit sequences are left untouched (decode wrote them).
//
// One (packed row, kv head, sequence) is served by kWPR warps, each taking
// up to kPer consecutive splits: lane j of a warp loads split j's (m, l),
// every lane copies the 16-byte piece d = 4 lane .. 4 lane + 3 of every one
// of its splits' o into shared memory with asynchronous copies, all issued
// before any is waited for (one memory round trip; register loads would be
// scheduled one latency each).  The
// warp's maximum comes from the (m, l) lanes, so O is one pass of FMAs in
// split order with no rescaling.  With kWPR > 1 the warps' (max, sum, O)
// are combined in warp order through shared memory.  Every sum runs in a
// fixed order: the result does not depend on timing.
//
// A sequence with more splits than the launch covers (kWPR x kPer, sized
// from the caller's max_n_splits hint) or than max_splits is not merged: its
// rows are left as they were and MJ_ERR_INVALID_ARG goes to the status word.
//
// The kernel is launched as a programmatic dependent of the decode kernel:
// its CTAs can be resident before the decode grid ends and read the split
// counts (the plan's, which the decode grid does not write) meanwhile; each
// waits for the decode grid before reading the partials or exiting.

#include <cuda_runtime.h>

#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

constexpr int kCtaWarps = 4;  // warps per CTA when a row needs fewer
constexpr int kStatusInvalidArg = 1;  // MJ_ERR_INVALID_ARG

// kWPR warps per row, each staging up to kPer splits (4, 8 or 16: the
// staging area, kPer x 512 B a warp, sets how many CTAs fit an SM)
template <int kWPR, int kPer>
__global__ void __launch_bounds__((kWPR > kCtaWarps ? kWPR : kCtaWarps) * 32) merge_kernel(const DecodeDev a) {
  constexpr int kRowsPerCta = kWPR >= kCtaWarps ? 1 : kCtaWarps / kWPR;
  const int lane = threadIdx.x & 31;
  const int wic = threadIdx.x >> 5;         // warp in the CTA
  const int w = wic % kWPR;                 // warp within the row
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + wic / kWPR;  // (b, g, n), n fastest
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.h_k * a.n_q;
  const int n = static_cast<int>(row % a.n_q);
  const int g = static_cast<int>((row / a.n_q) % a.h_k);
  const int b = static_cast<int>(row / (static_cast<int64_t>(a.n_q) * a.h_k));
  // The split count comes from the plan, which the decode grid does not
  // write and which was complete before any decode CTA passed its own wait
  // (this grid launches only after all of them have): it is read while the
  // decode grid drains.  Every CTA then waits for the decode grid's
  // completion (its partials complete and visible) before any other global
  // access or its exit, and the unpack after it may launch.
  const int nsp = row < rows ? a.n_splits[b] : 0;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  if (row >= rows) return;  // uniform over a row's warps (kWPR > 1: one row per CTA)
  if (nsp <= 1) return;  // unsplit: decode wrote O; uniform over the row's warps
  if (nsp > kWPR * kPer || nsp > a.max_splits) {
    // more splits than this launch was sized for (a max_n_splits hint below
    // the plan's largest count) or than the workspace holds: refuse the row
    // instead of merging a subset of its partials
    if (w == 0 && lane == 0 && a.status) atomicExch(a.status, kStatusInvalidArg);
    return;
  }
  const int j0 = w * kPer;
  const int cnt = nsp - j0 < kPer ? nsp - j0 : kPer;  // this warp's splits (may be <= 0)
  const int64_t pr0 = part_row(a, b, g, 0, n);
  const int64_t split_stride = a.n_q;  // rows between consecutive slots
  float m = -INFINITY, l = 0.f;
  if (lane < cnt) {
    const int64_t pr = pr0 + (j0 + lane) * split_stride;
    m = a.m_part[pr];
    l = a.l_part[pr];
  }
  // copies of this warp's splits, all in flight at once, into its kPer x
  // 512 B of the (dynamic) staging area; slots past its last split are
  // zero-filled without a read (their weight is 0)
  extern __shared__ __align__(16) float4 s_stage[];
  float4* const st = s_stage + wic * kPer * 32;
  const int jmax = nsp - 1;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int j = j0 + u < jmax ? j0 + u : jmax;
    cp_async16(st + u * 32 + lane, &a.o_part[(pr0 + j * split_stride) * kHeadDimDev + lane * 4], u < cnt);
  }
  cp_async_commit();
  // this warp's maximum, weights and weighted row sum
  float mw = m;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
  const float wt = (m == -INFINITY) ? 0.f : __expf(m - mw);
  float lw = wt * l;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
  float4 ow = make_float4(0.f, 0.f, 0.f, 0.f);
  cp_async_wait<0>();  // this lane's copies (it reads only its own)
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const float wu = __shfl_sync(0xffffffffu, wt, u);  // 0 past this warp's splits
    const float4 o = st[u * 32 + lane];
    ow.x = fmaf(wu, o.x, ow.x);
    ow.y = fmaf(wu, o.y, ow.y);
    ow.z = fmaf(wu, o.z, ow.z);
    ow.w = fmaf(wu, o.w, ow.w);
  }
  float mx = mw, lsum = lw;
  if constexpr (kWPR > 1) {
    __shared__ float s_m[kWPR], s_l[kWPR];
    __shared__ __align__(16) float s_o[kWPR][kHeadDimDev];
    if (lane == 0) {
      s_m[w] = mw;
      s_l[w] = lw;
    }
    *reinterpret_cast<float4*>(&s_o[w][lane * 4]) = ow;
    __syncthreads();
    if (w != 0) return;
    mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < kWPR; ++v) mx = fmaxf(mx, s_m[v]);
    lsum = 0.f;
    ow = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int v = 0; v < kWPR; ++v) {
      const float f = (s_m[v] == -INFINITY) ? 0.f : __expf(s_m[v] - mx);
      lsum = fmaf(f, s_l[v], lsum);
      const float4 ov = *reinterpret_cast<const float4*>(&s_o[v][lane * 4]);
      ow.x = fmaf(f, ov.x, ow.x);
      ow.y = fmaf(f, ov.y, ow.y);
      ow.z = fmaf(f, ov.z, ow.z);
      ow.w = fmaf(f, ov.w, ow.w);
    }
  }
  const float inv = lsum > 0.f ? a.scale_o / lsum : 0.f;
  const int64_t orow = b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + n) * kHeadDimDev;
  const __nv_bfloat162 lo2 = __floats2bfloat162_rn(ow.x * inv, ow.y * inv);
  const __nv_bfloat162 hi2 = __floats2bfloat162_rn(ow.z * inv, ow.w * inv);
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t*>(&lo2);
  packed.y = *reinterpret_cast<const uint32_t*>(&hi2);
  *reinterpret_cast<uint2*>(a.o + orow + lane * 4) = packed;
  if (lane == 0) a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + n] = mx + logf(lsum);
}

template <int kWPR, int kPer>
cudaError_t launch_merge_t(const DecodeDev& a, cudaStream_t stream) {
  constexpr int kRowsPerCta = kWPR >= kCtaWarps ? 1 : kCtaWarps / kWPR;
  constexpr int kThreads = (kWPR > kCtaWarps ? kWPR : kCtaWarps) * 32;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.h_k * a.n_q;
  const dim3 grid(static_cast<unsigned>((rows + kRowsPerCta - 1) / kRowsPerCta), 1, 1);
  const size_t smem = kThreads / 32 * kPer * 32 * 16;  // the staging area: kPer x 512 B a warp
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(merge_kernel<kWPR, kPer>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(merge_kernel<kWPR, kPer>, grid, dim3(kThreads, 1, 1), smem, stream, a);
}

}  // namespace

cudaError_t launch_merge(const DecodeDev& a, int max_n_splits, cudaStream_t stream) {
  if (max_n_splits <= 4) return launch_merge_t<1, 4>(a, stream);
  if (max_n_splits <= 8) return launch_merge_t<1, 8>(a, stream);
  if (max_n_splits <= 16) return launch_merge_t<1, 16>(a, stream);
  if (max_n_splits <= 64) return launch_merge_t<4, 16>(a, stream);
  return launch_merge_t<16, 16>(a, stream);
}

}  // namespace mj
