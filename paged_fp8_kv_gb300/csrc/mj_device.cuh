// Device-side helpers and the kernel argument block shared by the decode,
// merge and layout kernels of libmj (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace mj {

// Everything a decode launch needs, by value (kernel parameter space).
struct DecodeDev {
  const void* q;
  int64_t q_seq;
  const uint8_t* k;
  const uint8_t* v;
  int64_t k_page, k_row, k_head, v_page, v_row, v_head;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* work;
  const int32_t* n_splits;
  const float* qd;
  const float* kd;
  const float* vd;
  int64_t qd_seq, qd_head, kd_seq, kd_head, vd_seq, vd_head;
  float softmax_scale, scale_o;
  __nv_bfloat16* o;
  int64_t o_seq;
  float* lse;
  float* o_part;  // [b][g][slot][n][d]
  float* m_part;  // [b][g][slot][n]
  float* l_part;
  int32_t* status;
  int32_t num_seqs, h_k, n_q, q_len, h_r, page_size, max_blocks, causal, max_splits, num_work;
  int32_t num_pages;
  int32_t l2_prefetch;  // tiles the producer prefetches into L2 ahead (0 = off)
};

constexpr float kLog2e = 1.4426950408889634f;

// Exact e4m3 -> f16 of two packed codes (low byte -> low half).  Every e4m3
// value, subnormals and NaN included, is representable in f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

// Four e4m3 codes (one 32-bit word, byte 0 first) -> four floats, exactly.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* out) {
  const uint32_t lo = e4m3x2_to_f16x2(static_cast<uint16_t>(w & 0xFFFFu));
  const uint32_t hi = e4m3x2_to_f16x2(static_cast<uint16_t>(w >> 16));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&lo));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hi));
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(c));
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// 2^x with the hardware approximation (ex2.approx; flushes results below
// 2^-126 to zero, which only drops probabilities far below fp32 resolution
// of the row sum).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  const int n = valid ? 16 : 0;  // 0 source bytes: fill 16 zero bytes
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Index helpers for the partial-result workspace.
__device__ __forceinline__ int64_t part_row(const DecodeDev& a, int b, int g, int slot, int n) {
  return ((static_cast<int64_t>(b) * a.h_k + g) * a.max_splits + slot) * a.n_q + n;
}

}  // namespace mj
