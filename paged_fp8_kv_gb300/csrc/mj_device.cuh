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
  int32_t l2_prefetch;     // tiles the producer prefetches into L2 ahead (0 = off)
  int32_t kv_evict_first;  // K/V tile loads with an L2 EVICT_FIRST policy (0 = off)
  int32_t kv_format;       // mj_kv_format of the K/V pools
  const uint8_t* ks;       // nvfp4 scale planes: row r of (page, g) at page*x_page + g*x_head + 8r
  const uint8_t* vs;
  int64_t ks_page, ks_head, vs_page, vs_head;
};

// Bits per K/V code of a pool format (mj_kv_format: e4m3, e3m2, e2m3, e2m1,
// nvfp4).
__host__ __device__ constexpr int kv_bits(int kv_format) {
  return kv_format == 0 ? 8 : ((kv_format == 3 || kv_format == 4) ? 4 : 6);
}

// The kind::f8f6f4 operand format code of a pool format (nvfp4 reaches the
// MMA converted to e4m3).
__host__ __device__ constexpr uint32_t kv_mma_format(int kv_format) {
  return kv_format == 1 ? 4u : (kv_format == 2 ? 3u : (kv_format == 3 ? 5u : 0u));
}


// Bytes a TMA load of `rows` K/V rows (one head, d = 128 codes each) reads
// from global memory and credits to its mbarrier: the packed size (the
// shared-memory copy of a narrow row takes 128 bytes whatever the format).
__host__ __device__ constexpr uint32_t kv_box_bytes(int kv_format, int rows) {
  return static_cast<uint32_t>(rows) * 16u * static_cast<uint32_t>(kv_bits(kv_format));
}

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

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed fp32 pairs (one instruction for two lanes of arithmetic on sm_100
// and later): (a0, a1) * (b0, b1) + (c0, c1) and (a0, a1) + (b0, b1), round
// to nearest, each lane exactly as its scalar instruction.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  const uint64_t ua = (static_cast<uint64_t>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x);
  const uint64_t ub = (static_cast<uint64_t>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x);
  const uint64_t uc = (static_cast<uint64_t>(__float_as_uint(c.y)) << 32) | __float_as_uint(c.x);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(ua), "l"(ub), "l"(uc));
  return make_float2(__uint_as_float(static_cast<uint32_t>(r)), __uint_as_float(static_cast<uint32_t>(r >> 32)));
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  const uint64_t ua = (static_cast<uint64_t>(__float_as_uint(a.y)) << 32) | __float_as_uint(a.x);
  const uint64_t ub = (static_cast<uint64_t>(__float_as_uint(b.y)) << 32) | __float_as_uint(b.x);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ua), "l"(ub));
  return make_float2(__uint_as_float(static_cast<uint32_t>(r)), __uint_as_float(static_cast<uint32_t>(r >> 32)));
}

// Packed half-precision helpers for the exponentials and the P split.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
  uint32_t y;
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}
__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t add_f16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// N values 0 <= x <= 448 (N a multiple of 4) as e4m3 hi and lo parts, four
// codes a word: x is rounded to half precision (11 significant bits), hi =
// e4m3(x), lo = e4m3((x - hi) 2^kLoShift) (the difference is exact in half
// precision, and |x - hi| <= x 2^-4, so a shift up to 4 stays in range and
// keeps the lo part clear of e4m3's subnormal floor), so hi + lo 2^-kLoShift
// carries about 8 significant bits of x.
template <int N, int kLoShift = 0>
__device__ __forceinline__ void split_e4m3_hilo(const float* x, uint32_t* hi, uint32_t* lo) {
  static_assert(kLoShift >= 0 && kLoShift <= 4, "lo shift");
  constexpr uint32_t kScale2 = (15u + kLoShift) << 10 | (15u + kLoShift) << 26;  // (2^s, 2^s) in halves
#pragma unroll
  for (int w = 0; w < N / 4; ++w) {
    const uint32_t h01 = f32x2_to_f16x2(x[4 * w], x[4 * w + 1]);
    const uint32_t h23 = f32x2_to_f16x2(x[4 * w + 2], x[4 * w + 3]);
    const uint16_t e01 = f16x2_to_e4m3x2(h01);
    const uint16_t e23 = f16x2_to_e4m3x2(h23);
    uint32_t d01 = sub_f16x2(h01, e4m3x2_to_f16x2(e01));
    uint32_t d23 = sub_f16x2(h23, e4m3x2_to_f16x2(e23));
    if (kLoShift > 0) {
      d01 = mul_f16x2(d01, kScale2);
      d23 = mul_f16x2(d23, kScale2);
    }
    const uint16_t l01 = f16x2_to_e4m3x2(d01);
    const uint16_t l23 = f16x2_to_e4m3x2(d23);
    hi[w] = static_cast<uint32_t>(e01) | (static_cast<uint32_t>(e23) << 16);
    lo[w] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
  }
}

// Reduces R per-lane values over the 32 lanes (max or sum), scattered by
// recursive halving: each step keeps half of the live values and adds the
// partner lane's copy of them.  On return v[0] holds the warp total of
// column warp_col<R>(lane) (and, for R = 64, v[1] that of column + 32).
template <int R, bool kMax>
__device__ __forceinline__ void warp_reduce_scatter(float* v, int lane) {
  auto op = [](float x, float y) { return kMax ? fmaxf(x, y) : x + y; };
  if constexpr (R == 64) {
    warp_reduce_scatter<32, kMax>(v, lane);
    warp_reduce_scatter<32, kMax>(v + 32, lane);
    v[1] = v[32];
  } else {
    int width = R;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      if (width > 1) {
        const bool upper = (lane & off) != 0;
        const int half = width >> 1;
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
          if (i < half) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
          }
        }
        width = half;
      } else {
        v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], off));
      }
    }
  }
}

// Column held by a lane after warp_reduce_scatter<R>: the lane bits that
// chose upper halves, most significant first; lanes that agree on them hold
// the same total (only the lowest of them stores it).
template <int R>
__device__ __forceinline__ int warp_col(int lane) {
  constexpr int kShift = R >= 32 ? 0 : (R == 16 ? 1 : 2);
  return lane >> kShift;
}
template <int R>
__device__ __forceinline__ bool warp_col_writer(int lane) {
  constexpr int kMask = R >= 32 ? 0 : (R == 16 ? 1 : 3);
  return (lane & kMask) == 0;
}

// One nvfp4 group: 16 e2m1 codes (8 bytes, element 2i in the low nibble of
// byte i) and their e4m3 scale -> 16 e4m3 codes of code * scale * 2^-3,
// rounded to nearest even.  Every step before the rounding is exact in half
// precision: an e2m1 value has two significant bits and an e4m3 scale four,
// so the product has at most six, between 2^-13 and 336.
__device__ __forceinline__ uint4 nvfp4_group_to_e4m3(uint2 codes, uint32_t scale_code) {
  // the scale / 8 in both halves of a packed pair
  const uint32_t s2 = e4m3x2_to_f16x2(static_cast<uint16_t>(scale_code & 0xFFu));
  uint32_t sh;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(sh) : "r"(s2), "r"(0x30003000u));  // (0.125, 0.125)
  sh = __byte_perm(sh, 0, 0x1010);  // low half in both halves
  const uint32_t w[2] = {codes.x, codes.y};
  uint32_t out[4];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w[k]));
    uint16_t e[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t prod;
      asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(prod) : "r"(h[j]), "r"(sh));
      asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(e[j]) : "r"(prod));
    }
    out[2 * k] = static_cast<uint32_t>(e[0]) | (static_cast<uint32_t>(e[1]) << 16);
    out[2 * k + 1] = static_cast<uint32_t>(e[2]) | (static_cast<uint32_t>(e[3]) << 16);
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// Index helpers for the partial-result workspace.
__device__ __forceinline__ int64_t part_row(const DecodeDev& a, int b, int g, int slot, int n) {
  return ((static_cast<int64_t>(b) * a.h_k + g) * a.max_splits + slot) * a.n_q + n;
}

}  // namespace mj
