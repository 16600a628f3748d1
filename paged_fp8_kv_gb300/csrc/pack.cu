// Query / output layout permutation (source: the "mjolnir/t5_decode.py"
// page, `pack_q` and `unpack_o`): vLLM rows (b*q_len + qi, g*h_r + hr) <->
// packed rows (b, g, qi*h_r + hr).  Each row is head_dim contiguous
// elements; threads move 16-byte vectors, consecutive threads consecutive
// vectors of the destination.

#include <cuda_runtime.h>

#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

__global__ void permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                    int64_t total_vec, int vec_per_row, int q_len, int h_k, int h_r,
                                    bool to_packed) {
  // a programmatic dependent: no global load or store before the grid
  // ahead of this one has completed; the next kernel may launch now
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
  if (i >= total_vec) return;
  const int64_t row = i / vec_per_row;
  const int v = static_cast<int>(i % vec_per_row);
  const int n_q = q_len * h_r;
  // destination row index -> (b, g, qi, hr)
  int64_t b, g, qi, hr;
  if (to_packed) {  // dst row = (b*h_k + g)*n_q + qi*h_r + hr
    const int64_t n = row % n_q;
    const int64_t bg = row / n_q;
    g = bg % h_k;
    b = bg / h_k;
    qi = n / h_r;
    hr = n % h_r;
  } else {  // dst row = (b*q_len + qi)*(h_k*h_r) + g*h_r + hr
    const int64_t h = row % (h_k * h_r);
    const int64_t bq = row / (h_k * h_r);
    qi = bq % q_len;
    b = bq / q_len;
    g = h / h_r;
    hr = h % h_r;
  }
  const int64_t vllm_row = (b * q_len + qi) * (h_k * h_r) + g * h_r + hr;
  const int64_t packed_row = (b * h_k + g) * n_q + qi * h_r + hr;
  const int64_t src_row = to_packed ? vllm_row : packed_row;
  dst[row * vec_per_row + v] = src[src_row * vec_per_row + v];
}

}  // namespace

cudaError_t launch_permute_rows(const void* src, void* dst, int elem_bytes, int num_seqs, int q_len,
                                int h_k, int h_r, int head_dim, bool to_packed, cudaStream_t stream) {
  const int vec_per_row = head_dim * elem_bytes / 16;
  const int64_t rows = static_cast<int64_t>(num_seqs) * q_len * h_k * h_r;
  const int64_t total = rows * vec_per_row;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  return launch_pdl(permute_rows_kernel, dim3(static_cast<unsigned>(blocks), 1, 1), dim3(threads, 1, 1), 0, stream,
                    static_cast<const uint4*>(src), static_cast<uint4*>(dst), total, vec_per_row, q_len, h_k, h_r,
                    to_packed);
}

}  // namespace mj
