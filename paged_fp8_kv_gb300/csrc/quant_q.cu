// Fused fp8 query quantisation and pack.
//
// Source: the "mjolnir/t5_decode.py" page, `quantize_q_fp8` and `pack_q`
// (host helpers section).  For sequence b and kv head g the group is the
// q_len tokens x h_r query heads x d values of Q that share one kv head; its
// descale is max(amax, 1e-6) / 448 in fp32 (448: the largest e4m3 value),
// and every element is stored as e4m3(q / descale), rounded to nearest even
// and saturating, in the packed row (b, g, qi*h_r + hr).  The page does this
// in two host-side tensor passes and a separate pack; here one kernel reads
// the bf16 rows in vLLM's layout and writes the packed e4m3 rows and the
// descales.
//
// One CTA per (b, g), 64 to 512 threads by the group's size.  Pass 1 reads
// the group's rows as 16-byte vectors, up to eight vectors' loads in flight
// per thread, and reduces |q| to its maximum (warp shuffles, then shared
// memory).  Pass 2 quantises from the same registers when the group fits
// one sweep of the block (up to 4096 vectors, 512 rows of d = 128), else
// reads the rows again (L2 hits), and writes 16 codes per vector as one
// 16-byte store.  The division is IEEE fp32 (round to nearest), as on the page, so
// codes are a function of the inputs alone.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

constexpr int kMaxThreads = 512;
constexpr int kUnroll = 8;  // 16-element vectors per thread and sweep
constexpr float kE4m3Max = 448.f;
constexpr float kAmaxFloor = 1e-6f;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 w, float* x) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(u[i] << 16);
    x[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(kMaxThreads)
    quantize_pack_q_kernel(const uint4* __restrict__ q, uint4* __restrict__ q_packed, float* __restrict__ q_descale,
                           int q_len, int h_k, int h_r, int head_dim) {
  // a programmatic dependent: no global load or store before the grid
  // ahead of this one has completed; the next kernel may launch now
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int bg = blockIdx.x;  // b * h_k + g
  const int b = bg / h_k, g = bg % h_k;
  const int nthr = blockDim.x;
  const int rows = q_len * h_r;
  const int v16_per_row = head_dim / 16;  // 16 elements: two bf16 vectors in, one code vector out
  const int total = rows * v16_per_row;
  const int64_t row_vecs = head_dim / 8;  // bf16 vectors per row
  auto src_vec = [&](int i) -> const uint4* {
    const int row = i / v16_per_row, v = i % v16_per_row;
    const int qi = row / h_r, hr = row % h_r;
    const int64_t vllm_row = (static_cast<int64_t>(b) * q_len + qi) * (static_cast<int64_t>(h_k) * h_r) +
                             static_cast<int64_t>(g) * h_r + hr;
    return q + vllm_row * row_vecs + 2 * v;
  };

  // pass 1: the group's largest magnitude (kUnroll vectors' loads issued
  // before any is used).  A group that fits one sweep of the block keeps
  // its values in these registers for pass 2.
  const bool one_sweep = total <= nthr * kUnroll;
  uint4 w[kUnroll][2];
  float amax = 0.f;
  for (int base = threadIdx.x; base < total; base += nthr * kUnroll) {
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * nthr;
      if (i < total) {
        const uint4* s = src_vec(i);
        w[u][0] = s[0];
        w[u][1] = s[1];
      } else {
        w[u][0] = w[u][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      float x[16];
      bf16x8_to_f32(w[u][0], x);
      bf16x8_to_f32(w[u][1], x + 8);
#pragma unroll
      for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[e]));
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  __shared__ float s_amax[kMaxThreads / 32];
  if ((threadIdx.x & 31) == 0) s_amax[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_amax[0];
  for (int v = 1; v < nthr / 32; ++v) amax = fmaxf(amax, s_amax[v]);
  const float descale = __fdiv_rn(fmaxf(amax, kAmaxFloor), kE4m3Max);
  if (threadIdx.x == 0) q_descale[bg] = descale;

  // pass 2: codes, 16 per vector, in the packed row order (row-major:
  // vector i is row i / v16_per_row, columns 16 (i % v16_per_row) ..)
  uint4* const dst = q_packed + static_cast<int64_t>(bg) * rows * v16_per_row;
  for (int base = threadIdx.x; base < total; base += nthr * kUnroll) {
    if (!one_sweep) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int i = base + u * nthr;
        if (i < total) {
          const uint4* s = src_vec(i);
          w[u][0] = s[0];
          w[u][1] = s[1];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = base + u * nthr;
      if (i >= total) break;
      float x[16];
      bf16x8_to_f32(w[u][0], x);
      bf16x8_to_f32(w[u][1], x + 8);
      uint32_t c[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint16_t c01 = ptx::f32x2_to_e4m3x2(__fdiv_rn(x[4 * k], descale), __fdiv_rn(x[4 * k + 1], descale));
        const uint16_t c23 =
            ptx::f32x2_to_e4m3x2(__fdiv_rn(x[4 * k + 2], descale), __fdiv_rn(x[4 * k + 3], descale));
        c[k] = static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
      }
      dst[i] = make_uint4(c[0], c[1], c[2], c[3]);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_pack_q(const void* q_vllm, void* q_packed, float* q_descale, int num_seqs, int q_len,
                                   int h_k, int h_r, int head_dim, cudaStream_t stream) {
  const int64_t groups = static_cast<int64_t>(num_seqs) * h_k;
  if (groups == 0) return cudaSuccess;
  // threads: about one vector each (the divisions of a thread run one
  // after another), 64 .. 512; larger groups take up to kUnroll vectors a
  // thread per sweep
  const int64_t vecs = static_cast<int64_t>(q_len) * h_r * (head_dim / 16);
  int threads = 64;
  while (threads < kMaxThreads && threads < vecs) threads *= 2;
  return launch_pdl(quantize_pack_q_kernel, dim3(static_cast<unsigned>(groups), 1, 1), dim3(threads, 1, 1), 0, stream,
                    static_cast<const uint4*>(q_vllm), static_cast<uint4*>(q_packed), q_descale, q_len, h_k, h_r,
                    head_dim);
}

}  // namespace mj
