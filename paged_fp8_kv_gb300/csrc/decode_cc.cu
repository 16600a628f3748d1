// Split-KV paged decode attention on the CUDA cores (narrow query tiles).
//
// One CTA serves one work item (a contiguous range of 128-row KV tiles of one
// sequence), one kv head and NT packed query rows.  Sources: the
// "mjolnir/t5_decode.py" page — `decode` kernel (work-item fetch, paged
// gather, masking by select, online softmax with the descales folded into
// the exponent, the -inf guard, the epilogue's final-vs-partial split) and
// the module docstring (causal tail, packing).  This kernel keeps P in fp32:
// there is no P quantisation on the CUDA cores.
//
// Data flow per 64-key stage (KT rows):
//   cp.async 16-byte page gathers -> shared ring (STAGES deep, rows padded to
//   144 bytes so that row-parallel 16-byte reads are conflict free);
//   QK: two threads per key, each a half of d, exact e4m3 dequant in
//   registers, Q broadcast from shared memory as fp32;
//   block max over the stage (warp shuffles + one shared-memory step);
//   p = 2^((s - m) * c) with c = softmax_scale * qd * kd * log2(e);
//   PV: warp w takes keys w*16.., lane l owns d = 4l..4l+3 for all NT rows.

#include <cuda_runtime.h>

#include "mj_device.cuh"
#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

constexpr int kThreads = 128;
constexpr int kKT = 64;       // keys per stage
constexpr int kStages = 3;    // ring depth
constexpr int kRowB = 144;    // padded shared row (128 data bytes + 16)
constexpr int kWarps = kThreads / 32;

template <int NT>
struct CcSmem {
  uint8_t kv[kStages][2][kKT][kRowB];  // [stage][K|V][key][byte]
  float q[kHeadDimDev][NT];            // Q transposed: q[d][n]
  float p[kKT][NT];
  float red[kWarps][NT];
};

template <int NT, bool kQe4m3>
__global__ void __launch_bounds__(kThreads)
decode_cc_kernel(const DecodeDev a, int n_q_tiles) {
  // Launched as a programmatic dependent: no global load or store before
  // the grid ahead of this one has completed.  The merge (this grid's own
  // dependent) may launch now; its CTAs wait the same way.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  CcSmem<NT>& sm = *reinterpret_cast<CcSmem<NT>*>(smem_raw);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  // Linear grid, work item outermost (see the tensor-core kernel).
  const int g = blockIdx.x % a.h_k;
  const int rest = blockIdx.x / a.h_k;
  const int n0 = (rest % n_q_tiles) * NT;
  const int w_idx = rest / n_q_tiles;

  const int4 item = reinterpret_cast<const int4*>(a.work)[w_idx];
  const int b = item.x, t_begin = item.y, t_end = item.z, slot = item.w;
  if (t_end <= t_begin) return;  // padding item

  const int L = a.seq_lens[b];
  const int nsp = a.n_splits[b];
  const float qd = a.qd[b * a.qd_seq + g * a.qd_head];
  const float kd = a.kd[b * a.kd_seq + g * a.kd_head];
  const float vd = a.vd[b * a.vd_seq + g * a.vd_head];
  const float cta_scale = a.softmax_scale * qd * kd;  // raw score -> logit
  const float c2 = cta_scale * kLog2e;                // raw score -> log2 units

  // ---- Q tile -> shared (fp32, transposed), rows past n_q are zero
  {
    const int d = tid;  // kThreads == head_dim
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float x = 0.f;
      if (n0 + n < a.n_q) {
        const int64_t off = b * a.q_seq + (static_cast<int64_t>(g) * a.n_q + n0 + n) * kHeadDimDev + d;
        if (kQe4m3)
          x = e4m3_to_f32(static_cast<const uint8_t*>(a.q)[off]);
        else
          x = bf16_bits_to_f32(static_cast<const uint16_t*>(a.q)[off]);
      }
      sm.q[d][n] = x;
    }
  }

  // Last key each row may see (-1: none).
  int lim[NT];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int row = n0 + n;
    int l = a.causal ? L - a.q_len + row / a.h_r : L - 1;
    l = l < L - 1 ? l : L - 1;
    lim[n] = row < a.n_q ? l : -1;
  }

  // Key range of this work item, clipped to the sequence.
  const int key_begin = t_begin * kTileRowsDev;
  int key_end = t_end * kTileRowsDev;
  key_end = key_end < L ? key_end : L;
  const int n_stages = key_end > key_begin ? (key_end - key_begin + kKT - 1) / kKT : 0;

  const int64_t bt_row = static_cast<int64_t>(b) * a.max_blocks;
  const int PS = a.page_size;

  // Copy stage s (keys key_begin + s*KT ...) into ring slot s % kStages.
  auto issue = [&](int s) {
    if (s < n_stages) {
      const int kbase = key_begin + s * kKT;
      uint8_t(*dst)[kKT][kRowB] = sm.kv[s % kStages];
#pragma unroll
      for (int i = 0; i < (kKT * 8) / kThreads; ++i) {
        const int c = i * kThreads + tid;  // 16-byte chunk id
        const int r = c >> 3, col = (c & 7) * 16;
        const int j = kbase + r;
        const bool ok = j < key_end;
        int64_t koff = 0, voff = 0;
        if (ok) {
          const int64_t page = a.block_table[bt_row + j / PS];
          const int64_t rr = j % PS;
          koff = page * a.k_page + rr * a.k_row + g * a.k_head + col;
          voff = page * a.v_page + rr * a.v_row + g * a.v_head + col;
        }
        cp_async16(&dst[0][r][col], a.k + koff, ok);
        cp_async16(&dst[1][r][col], a.v + voff, ok);
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) issue(s);

  float m_run[NT], l_thr[NT];
  float o_acc[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    m_run[n] = -INFINITY;
    l_thr[n] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) o_acc[n][e] = 0.f;
  }

  const int qk_key = tid >> 1;
  const int qk_half = tid & 1;

  for (int s = 0; s < n_stages; ++s) {
    cp_async_wait<kStages - 2>();
    __syncthreads();  // stage s landed; everyone is done with stage s-1
    issue(s + kStages - 1);
    const uint8_t(*kv)[kKT][kRowB] = sm.kv[s % kStages];

    // ---- QK: scores of key qk_key for all NT rows (half of d per thread)
    float acc[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n] = 0.f;
    const uint8_t* krow = &kv[0][qk_key][qk_half * 64];
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      const uint4 raw = *reinterpret_cast<const uint4*>(krow + ch * 16);
      const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        float kf[4];
        e4m3x4_to_f32(words[wi], kf);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int d = qk_half * 64 + ch * 16 + wi * 4 + e;
#pragma unroll
          for (int n4 = 0; n4 < NT; n4 += 4) {
            const float4 qv = *reinterpret_cast<const float4*>(&sm.q[d][n4]);
            acc[n4 + 0] = fmaf(qv.x, kf[e], acc[n4 + 0]);
            acc[n4 + 1] = fmaf(qv.y, kf[e], acc[n4 + 1]);
            acc[n4 + 2] = fmaf(qv.z, kf[e], acc[n4 + 2]);
            acc[n4 + 3] = fmaf(qv.w, kf[e], acc[n4 + 3]);
          }
        }
      }
    }
    const int j = key_begin + s * kKT + qk_key;
    float sc[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      const float full = acc[n] + __shfl_xor_sync(0xffffffffu, acc[n], 1);
      sc[n] = (j <= lim[n]) ? full : -INFINITY;  // select: masked rows never leak
    }

    // ---- stage max over the 64 keys (pairs already agree)
    float mx[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float v = sc[n];
#pragma unroll
      for (int off = 2; off < 32; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
      mx[n] = v;
    }
    if (lane == 0) {
#pragma unroll
      for (int n = 0; n < NT; ++n) sm.red[warp][n] = mx[n];
    }
    __syncthreads();
    float corr[NT];
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      float t = sm.red[0][n];
#pragma unroll
      for (int w2 = 1; w2 < kWarps; ++w2) t = fmaxf(t, sm.red[w2][n]);
      const float m_new = fmaxf(m_run[n], t);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // -inf guard
      corr[n] = fast_exp2((m_run[n] - m_use) * c2);
      const float p = fast_exp2((sc[n] - m_use) * c2);
      l_thr[n] = l_thr[n] * corr[n] + (qk_half == 0 ? p : 0.f);
      if (qk_half == 0) sm.p[qk_key][n] = p;
      m_run[n] = m_new;
    }
    __syncthreads();  // p ready

    // ---- PV: O[n][4 lane .. +3] for this warp's 16 keys
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) o_acc[n][e] *= corr[n];
#pragma unroll 4
    for (int kk = warp * (kKT / kWarps); kk < (warp + 1) * (kKT / kWarps); ++kk) {
      const uint32_t vw = *reinterpret_cast<const uint32_t*>(&kv[1][kk][lane * 4]);
      float vf[4];
      e4m3x4_to_f32(vw, vf);
#pragma unroll
      for (int n4 = 0; n4 < NT; n4 += 4) {
        const float4 pv = *reinterpret_cast<const float4*>(&sm.p[kk][n4]);
        const float pp[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 4; ++e) o_acc[n4 + i][e] = fmaf(pp[i], vf[e], o_acc[n4 + i][e]);
      }
    }
  }
  cp_async_wait<0>();
  __syncthreads();  // ring is free: reuse it for the cross-warp combine

  // ---- row sums: sum over all threads
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    float v = l_thr[n];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    l_thr[n] = v;
  }
  float* obuf = reinterpret_cast<float*>(&sm.kv[0][0][0][0]);  // [warp][n][d]
  static_assert(sizeof(float) * kWarps * NT * kHeadDimDev <= sizeof(sm.kv), "combine buffer");
  if (lane == 0) {
#pragma unroll
    for (int n = 0; n < NT; ++n) sm.red[warp][n] = l_thr[n];
  }
#pragma unroll
  for (int n = 0; n < NT; ++n)
    *reinterpret_cast<float4*>(&obuf[(warp * NT + n) * kHeadDimDev + lane * 4]) =
        make_float4(o_acc[n][0], o_acc[n][1], o_acc[n][2], o_acc[n][3]);
  __syncthreads();

  const bool final_out = nsp <= 1;
  const int d = tid;
  for (int n = 0; n < NT; ++n) {
    const int row = n0 + n;
    if (row >= a.n_q) break;
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      l += sm.red[w2][n];
      o += obuf[(w2 * NT + n) * kHeadDimDev + d];
    }
    const float m_logit = m_run[n] * cta_scale;  // -inf stays -inf
    if (final_out) {
      // l >= 1 whenever a key is visible; the epsilon only turns 0/0 into 0.
      const float inv = a.scale_o * vd / (l + 1e-30f);
      const int64_t orow = b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + row) * kHeadDimDev;
      a.o[orow + d] = __float2bfloat16_rn(o * inv);
      if (d == 0) a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + row] = m_logit + logf(l);
    } else {
      const int64_t pr = part_row(a, b, g, slot, row);
      a.o_part[pr * kHeadDimDev + d] = o * vd;
      if (d == 0) {
        a.m_part[pr] = m_logit;
        a.l_part[pr] = l;
      }
    }
  }
}

template <int NT, bool kQe4m3>
cudaError_t launch_cc(const DecodeDev& a, int n_q_tiles, cudaStream_t stream) {
  const size_t smem = sizeof(CcSmem<NT>);
  auto kern = decode_cc_kernel<NT, kQe4m3>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.num_work) * n_q_tiles * a.h_k, 1, 1);
  return launch_pdl(kern, grid, dim3(kThreads, 1, 1), smem, stream, a, n_q_tiles);
}

}  // namespace

cudaError_t launch_decode_cc(const DecodeDev& a, int rows_per_cta, int n_q_tiles, bool q_e4m3,
                             cudaStream_t stream) {
  switch (rows_per_cta) {
    case 4:
      return q_e4m3 ? launch_cc<4, true>(a, n_q_tiles, stream) : launch_cc<4, false>(a, n_q_tiles, stream);
    case 8:
      return q_e4m3 ? launch_cc<8, true>(a, n_q_tiles, stream) : launch_cc<8, false>(a, n_q_tiles, stream);
    case 16:
      return q_e4m3 ? launch_cc<16, true>(a, n_q_tiles, stream) : launch_cc<16, false>(a, n_q_tiles, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

int cc_smem_bytes(int rows_per_cta) {
  switch (rows_per_cta) {
    case 4: return static_cast<int>(sizeof(CcSmem<4>));
    case 8: return static_cast<int>(sizeof(CcSmem<8>));
    case 16: return static_cast<int>(sizeof(CcSmem<16>));
    default: return 0;
  }
}

}  // namespace mj
