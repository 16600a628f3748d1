// The occupancy-pinned split-KV plan computed on the device.
//
// Source: the "mjolnir/t5_decode.py" page, `plan_split_kv` and `SplitPlan`
// (host helpers section); the schedule kernel of the paged-decode page
// builds its plan on the device for the same reason: sequence lengths that
// change from step to step inside one captured CUDA graph.  The rule is the
// host plan's, for options the caller fixes (slots per wave, max_splits,
// force_splits, min_chunk_tiles, a padded work-list length):
//
//   T_b   = max(1, ceil(L_b / 128)) tiles; T = max_b T_b
//   floor = max(min_chunk_tiles, ceil(T / max_splits))
//   chunk = max(floor, ceil(T / force_splits))   if force_splits > 0
//         = T                                    if b >= slots or max_splits == 1
//         = the least c in [floor, max(floor, T)] with sum_b ceil(T_b / c) <= slots
//   items (b, s*chunk, min(T_b, (s+1)*chunk), s), ordered by length, longest
//   first, equal lengths in (b, s) order; then (0, 0, 0, 0) up to pad_to.
//
// One CTA of 256 threads.  The tile counts sit in shared memory; the chunk
// comes from an 8-way search (each warp sums the chunk count of one probe).  Every item of length
// `chunk` precedes every shorter one, and those full-length items are
// placed in (b, s) order by a prefix sum of floor(T_b / chunk).  The rest
// (at most one item per sequence, of length T_b mod chunk) are ordered by a
// bitonic sort of (length descending, b ascending) keys, unique per
// sequence, so the order is the stable one.  Problems are reported in the
// optional status word (lengths out of range, more splits than max_splits,
// more items than pad_to); the outputs are then unspecified but every write
// stays inside the buffers.

#include <cuda_runtime.h>

#include <cstdint>

#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kTileRowsDev = 128;
constexpr int kStatusInvalid = 1;   // MJ_ERR_INVALID_ARG
constexpr int kStatusCapacity = 3;  // MJ_ERR_CAPACITY

__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

__device__ __forceinline__ int64_t warp_max(int64_t v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = max64(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ int64_t warp_sum(int64_t v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

__global__ void __launch_bounds__(kPlanThreads)
    plan_device_kernel(const int32_t* __restrict__ seq_lens, int num_seqs, int64_t max_len, int64_t slots,
                       int max_splits, int force_splits, int min_chunk, int pad_to, int sort_n,
                       int4* __restrict__ work, int32_t* __restrict__ n_splits, int32_t* __restrict__ chunk_out,
                       int32_t* __restrict__ status) {
  // a programmatic dependent: no global load or store before the grid
  // ahead of this one has completed; the next kernel may launch now
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem_raw);      // [sort_n]
  int32_t* tiles = reinterpret_cast<int32_t*>(keys + sort_n);  // [num_seqs]
  __shared__ int64_t red_a[kPlanWarps], red_b[kPlanWarps];
  __shared__ int64_t probe[kPlanWarps];
  __shared__ int ok[kPlanWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // tile counts; the longest and whether a length was out of range
  int64_t bad = 0, longest = 1;
  for (int b = tid; b < num_seqs; b += kPlanThreads) {
    int64_t L = seq_lens[b];
    if (L < 0 || L > max_len) {
      bad = 1;
      L = L < 0 ? 0 : max_len;
    }
    const int64_t t = L > 0 ? (L + kTileRowsDev - 1) / kTileRowsDev : 1;
    tiles[b] = static_cast<int32_t>(t);
    longest = max64(longest, t);
  }
  longest = warp_max(longest);
  bad = warp_max(bad);
  if (lane == 0) {
    red_a[warp] = longest;
    red_b[warp] = bad;
  }
  __syncthreads();  // also publishes tiles[]
  longest = red_a[0];
  bad = red_b[0];
  for (int v = 1; v < kPlanWarps; ++v) {
    longest = max64(longest, red_a[v]);
    bad = max64(bad, red_b[v]);
  }

  // chunk.  The least c in [lo, hi] with sum_b ceil(T_b / c) <= slots (a
  // non-increasing function of c, within bound at hi) by an 8-way search:
  // each warp evaluates one probe, the first probe within bound becomes hi
  // and the one before it, plus one, lo.
  const int64_t floor_c = max64(min_chunk, (longest + max_splits - 1) / max_splits);
  int64_t chunk;
  if (force_splits > 0) {
    chunk = max64(floor_c, (longest + force_splits - 1) / force_splits);
  } else if (num_seqs >= slots || max_splits == 1) {
    chunk = longest;
  } else {
    int64_t lo = floor_c, hi = max64(floor_c, longest);
    while (lo < hi) {  // lo, hi uniform over the block
      const int64_t p = lo + ((hi - lo) * (warp + 1)) / (kPlanWarps + 1);  // in [lo, hi)
      // tile counts and chunks fit 32 bits (at most 2^30 / 128): 32-bit divisions
      const uint32_t p32 = static_cast<uint32_t>(p);
      int64_t part = 0;
      for (int b = lane; b < num_seqs; b += 32) part += (static_cast<uint32_t>(tiles[b]) + p32 - 1) / p32;
      part = warp_sum(part);
      __syncthreads();  // the previous round's probes are read
      if (lane == 0) {
        probe[warp] = p;
        ok[warp] = part <= slots;
      }
      __syncthreads();
      int first = kPlanWarps;
      for (int v = kPlanWarps - 1; v >= 0; --v)
        if (ok[v]) first = v;
      if (first < kPlanWarps) {
        hi = probe[first];
        if (first > 0) lo = probe[first - 1] + 1;
      } else {
        lo = probe[kPlanWarps - 1] + 1;
      }
    }
    chunk = lo;
  }

  // per sequence: splits, full-length chunks and remainders (contiguous runs
  // of sequences per thread, so the prefix sums keep b order)
  const int per = (num_seqs + kPlanThreads - 1) / kPlanThreads;
  const int b0 = min(num_seqs, tid * per), b1 = min(num_seqs, b0 + per);
  const uint32_t c32 = static_cast<uint32_t>(chunk);
  int64_t my_full = 0, my_rem = 0, over = 0;
  for (int b = b0; b < b1; ++b) {
    const uint32_t t = static_cast<uint32_t>(tiles[b]);
    const uint32_t k = (t + c32 - 1) / c32;
    if (k > static_cast<uint32_t>(max_splits)) over = 1;
    n_splits[b] = static_cast<int32_t>(k);
    my_full += t / c32;
    my_rem += (t % c32) != 0;
  }
  // exclusive scans of both counts over the threads: within warps by
  // shuffles, then over the warps' totals
  int64_t inc_f = my_full, inc_r = my_rem;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t f = __shfl_up_sync(0xffffffffu, inc_f, off);
    const int64_t r = __shfl_up_sync(0xffffffffu, inc_r, off);
    if (lane >= off) {
      inc_f += f;
      inc_r += r;
    }
  }
  over = warp_max(over);
  __syncthreads();  // red_a / red_b are read
  if (lane == 31) {
    red_a[warp] = inc_f;
    red_b[warp] = inc_r;
  }
  if (lane == 0) probe[warp] = over;
  __syncthreads();
  int64_t off_full = inc_f - my_full, off_rem = inc_r - my_rem;
  int64_t full_total = 0, rem_total = 0;
  for (int v = 0; v < kPlanWarps; ++v) {
    if (v < warp) {
      off_full += red_a[v];
      off_rem += red_b[v];
    }
    full_total += red_a[v];
    rem_total += red_b[v];
    over = max64(over, probe[v]);
  }
  const int64_t n_items = full_total + rem_total;
  const bool fits = n_items <= pad_to;
  if (tid == 0) {
    if (chunk_out) *chunk_out = static_cast<int32_t>(chunk);
    if (status && (bad || over)) atomicExch(reinterpret_cast<int*>(status), kStatusInvalid);
    else if (status && !fits) atomicExch(reinterpret_cast<int*>(status), kStatusCapacity);
  }

  // full-length items in (b, s) order; remainder keys: length descending,
  // then b ascending (unique, so any correct sort keeps generation order)
  for (int b = b0; b < b1; ++b) {
    const uint32_t t = static_cast<uint32_t>(tiles[b]);
    const uint32_t f = t / c32, r = t % c32;
    if (fits)
      for (uint32_t s = 0; s < f; ++s)
        work[off_full + s] = make_int4(b, static_cast<int>(s * c32), static_cast<int>((s + 1) * c32),
                                       static_cast<int>(s));
    off_full += f;
    if (r != 0) keys[off_rem++] = ((0x7FFFFFFFull - r) << 32) | static_cast<uint64_t>(b);
  }
  for (int i = static_cast<int>(rem_total) + tid; i < sort_n; i += kPlanThreads) keys[i] = ~0ull;
  __syncthreads();
  // bitonic sort of sort_n (a power of two) keys, ascending
  for (int k = 2; k <= sort_n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < sort_n; i += kPlanThreads) {
        const int q = i ^ j;
        if (q > i) {
          const uint64_t x = keys[i], y = keys[q];
          const bool up = (i & k) == 0;
          if ((x > y) == up) {
            keys[i] = y;
            keys[q] = x;
          }
        }
      }
      __syncthreads();
    }
  }
  if (fits) {
    for (int i = tid; i < rem_total; i += kPlanThreads) {
      const int b = static_cast<int>(keys[i] & 0xFFFFFFFFull);
      const uint32_t t = static_cast<uint32_t>(tiles[b]);
      const uint32_t s = t / c32;  // the last split slot
      work[full_total + i] = make_int4(b, static_cast<int>(s * c32), static_cast<int>(t), static_cast<int>(s));
    }
    for (int64_t i = n_items + tid; i < pad_to; i += kPlanThreads) work[i] = make_int4(0, 0, 0, 0);
  }
}

}  // namespace

int plan_device_sort_n(int num_seqs) {
  int n = 1;
  while (n < num_seqs) n <<= 1;
  return n;
}

size_t plan_device_smem_bytes(int num_seqs) {
  return static_cast<size_t>(plan_device_sort_n(num_seqs)) * 8 + static_cast<size_t>(num_seqs) * 4;
}

cudaError_t launch_plan_device(const int32_t* seq_lens, int num_seqs, int64_t max_len, int64_t slots,
                               int max_splits, int force_splits, int min_chunk, int pad_to, int4* work,
                               int32_t* n_splits, int32_t* chunk_out, int32_t* status, cudaStream_t stream) {
  const int sort_n = plan_device_sort_n(num_seqs);
  const size_t smem = plan_device_smem_bytes(num_seqs);
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(plan_device_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(plan_device_kernel, dim3(1, 1, 1), dim3(kPlanThreads, 1, 1), smem, stream, seq_lens, num_seqs,
                    max_len, slots, max_splits, force_splits, min_chunk, pad_to, sort_n, work, n_splits, chunk_out,
                    status);
}

}  // namespace mj
