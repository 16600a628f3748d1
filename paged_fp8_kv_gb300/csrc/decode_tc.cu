// Split-KV paged decode attention on the 5th-generation tensor cores
// (tcgen05, kind::f8f6f4), swap-AB orientation: the 128 KV rows of a tile
// are the MMA's M, the R packed query rows of the CTA (twice, as hi and lo
// parts) are its N.
//
// Sources: the "mjolnir/t5_decode.py" page — `decode` kernel (warp roles,
// paged TMA gather with out-of-range pages read as zeros, masking by select,
// online softmax with descales folded into the exponent and the -inf guard,
// lazy O rescale, deferred column sums, final-vs-partial epilogue, P stored
// as e4m3(p * 448)); the vLLM pull request page on the swap-AB decode kernel
// (KV slots on M, live heads on N).
//
// What this kernel does differently from those designs (GB300-first):
//  * K and V are never dequantised: the e4m3 tiles the TMA lands in shared
//    memory are the MMA operands directly (K as a K-major A, V as an
//    MN-major A for O^T = V^T P).
//  * A bf16 Q is split once per CTA into two e4m3 parts, x = q * 2^s =
//    hi + lo with hi = e4m3(x), lo = e4m3(x - hi), and both parts are
//    multiplied into the same accumulator.  The power-of-two s puts the
//    tile's largest |q| in [128, 256); hi + lo carries bf16's 8 significant
//    bits exactly for every |x| >= 2^-2 (smaller values keep an error below
//    2^-10 in x units).
//  * P is split the same way, x = 448 p = hi + lo, so the PV product sees
//    about 8 significant bits of p (bf16-like) instead of e4m3's 4.
//  * The hi and lo parts are stacked along the MMA's N (Q: 2R rows of B;
//    P: 2R columns of B) so each K step is one MMA; their products land in
//    accumulator columns c and R + c, which the softmax / epilogue add.
//
// Roles (64 + 128 or 64 + 256 threads):
//   warp 0      TMA producer: K and V tiles, one box per KV page.
//   warp 1      TMEM allocator; lane 0 issues every MMA and commit.
//   warps 2..   softmax / correction / epilogue; warp w reads TMEM lanes
//               32*(w%4).. (TMEM lane = KV row for S, = head-dim row for O);
//               with 8 softmax warps two share a lane quarter, each taking
//               half of the columns.
//
// Every mbarrier wait is bounded (wall clock); a role that gives up sets a
// shared abort flag and writes MJ_ERR_TIMEOUT to the optional status word,
// the others stop at their next wait, in-flight copies and MMAs are drained
// (bounded again) and TMEM is freed before the CTA exits.

#include <cuda.h>
#include <cuda_runtime.h>

#include "mj_device.cuh"
#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
// -------------------------------------------------------- host: tensor maps

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

// (d bytes, rows in page, kv heads, pages) view of a paged e4m3 pool; one box
// is box_rows rows of box_heads heads: 128 bytes x box_rows x box_heads,
// head-major in shared memory, 128-byte swizzle.
bool make_kv_map(CUtensorMap* m, const uint8_t* base, int page_size, int h_k, int num_pages, int64_t s_row,
                 int64_t s_head, int64_t s_page, int box_rows, int box_heads, int kv_format) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {128, static_cast<cuuint64_t>(page_size), static_cast<cuuint64_t>(h_k),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(s_row), static_cast<cuuint64_t>(s_head),
                                 static_cast<cuuint64_t>(s_page)};
  const cuuint32_t box[4] = {128, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(box_heads), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType type = kv_format == 0   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : kv_format == 3 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B
                                                    : CU_TENSOR_MAP_DATA_TYPE_16U6_ALIGN16B;
  const CUresult r = enc(m, type, 4, const_cast<uint8_t*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

constexpr int kTileKV = 128;                 // KV rows per tile (MMA M)
constexpr int kKVTileBytes = kTileKV * 128;  // one K or V tile: 16 KB
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far above any legal wait
constexpr int kStatusTimeout = 5;            // MJ_ERR_TIMEOUT
// P is produced as x = 448 p 2^-kTau: a column's reference maximum m moves
// only when a score passes m + kTau (log2 units), so x stays within e4m3's
// range and most tiles need neither the column reduction nor an O
// correction; the result does not depend on m.
constexpr int kTau = 4;
constexpr float kLog2PScale = 8.807354922057604f - kTau;  // log2(448 2^-kTau)
constexpr float kPScaleInv = (1.f / 448.f) * (1 << kTau);
// P's lo part is stored as e4m3((x - hi) 2^kLoShift) and its products are
// weighted back by 2^-kLoShift when the hi and lo columns of O are added
constexpr int kLoShift = 4;
constexpr float kLoInv = 1.f / (1 << kLoShift);

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

// Shape constants of one instance: R packed query rows per CTA.
//   GEMM1 B operand (Q): kN1 rows = [hi rows | lo rows] for bf16 Q (2R), the
//     e4m3 codes for e4m3 Q (R, at least 16 as the MMA requires).
//   GEMM2 B operand (P): kN2 = 2R columns = [hi columns | lo columns].
// The hi and lo parts share one MMA per K step; their products land in
// separate accumulator columns (c and R + c) that the softmax adds.
//   kNv: the pool is nvfp4 (e2m1 codes and an e4m3 scale per 16 elements): a
//     fourth warpgroup converts each tile into the e4m3 ring from a ring of
//     packed tiles the TMA fills (codes and scales of K and V, 18 KB a tile).
template <int R, bool kQe4m3, bool kNv = false>
struct TcCfg {
  static constexpr int kN1 = kQe4m3 ? (R < 16 ? 16 : R) : 2 * R;
  static constexpr int kN2 = 2 * R;
  // 16 rows and 8 rows of bf16 Q: three stages at two CTAs per SM instead
  // of two at three; a CTA then keeps a third more of its sequence in
  // flight (GQA decode: the long sequences need no split, 109.8 -> 108.6
  // us a step; sweep N = 16: 384 -> 256 work items, 101.6 -> 98.7 us), and
  // short split chunks have most of their tiles in flight at once
  static constexpr bool kDeep16 = R == 16 || (!kQe4m3 && R == 8);
  // nvfp4: two converted stages and six packed ones (108 KB of the pool in
  // flight), one CTA per SM
  static constexpr int kStages = kNv ? 2 : (kDeep16 ? 3 : (R <= 32 ? 2 : 5));
  static constexpr int kMinBlocks = kNv ? 1 : (kDeep16 ? 2 : (R <= 16 ? 3 : (R <= 32 ? 2 : 1)));
  static constexpr int kCvtWarps = kNv ? 4 : 0;
  static constexpr int kPkStages = kNv ? 6 : 0;
  static constexpr int kPkCodes = kTileKV * 64;   // 128 rows x 64 bytes of e2m1 codes
  static constexpr int kPkScales = kTileKV * 8;   // 128 rows x 8 e4m3 scales
  static constexpr int kPkBytes = 2 * (kPkCodes + kPkScales);  // K codes, V codes, K scales, V scales
  // two P buffers let the softmax of tile i write while GEMM2(i-1) still
  // reads; R = 16 at 3 CTAs/SM has no room for the second one
  static constexpr int kPBufs = R == 16 && !kDeep16 ? 1 : 2;
  // softmax warps: four cover the 128 TMEM lanes; with R = 32 a second four
  // take the other half of the columns (two warps per lane quarter)
  static constexpr int kSmWarps = R >= 32 ? 8 : 4;
  static constexpr int kSmThreads = 32 * kSmWarps;
  static constexpr int kThreads = 64 + kSmThreads + 32 * kCvtWarps;
  static constexpr int kHalves = kSmWarps / 4;
  static constexpr int kCols = R / kHalves;  // columns per softmax thread
  static constexpr int kQBytes = kN1 * 128;    // SW128 K-major rows
  static constexpr int kPBytes = kN2 * kTileKV;  // MN-major, no swizzle
  static constexpr int kTmemCols = pow2_at_least(2 * kN1 + kN2);
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kStages * kKVTileBytes;
  static constexpr int kOffQ = 2 * kStages * kKVTileBytes;
  static constexpr int kOffP = kOffQ + kQBytes;       // [buf][kN2/16 groups][128 rows][16 B]
  static constexpr int kOffRed = kOffP + kPBufs * kPBytes;  // [4][R] floats
  static constexpr int kOffM = kOffRed + 4 * R * 4;    // [2][R] running max
  static constexpr int kOffCorr = kOffM + 2 * R * 4;   // [R] correction
  static constexpr int kOffPk = (kOffCorr + R * 4 + 1023) / 1024 * 1024;  // packed ring (nvfp4)
  static constexpr int kOffBar = kOffPk + kPkStages * kPkBytes;
  static constexpr int kNumBars = 3 * kStages + 2 + 2 + 2 + 2 + 1 + 1 + 1 + 2 * kPkStages;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static_assert(kN1 % 16 == 0 && kN1 <= 256 && kN2 % 16 == 0 && kN2 <= 256, "MMA N");
  static_assert(kMinBlocks * kTmemCols <= 512, "TMEM for kMinBlocks CTAs");
  static_assert(kMinBlocks * (kBytes + 1024) <= 233472, "shared memory for kMinBlocks CTAs");
};

struct Bars {
  uint32_t kfull, vfull, kvempty;  // + stage * 8
  uint32_t sfull, sfree;           // + buf * 8
  uint32_t pfull, pfree;  // + buf * 8
  uint32_t odone, qready, drain;
  uint32_t pkfull, pkempty;  // nvfp4 packed ring: + stage * 8
};

__device__ __forceinline__ void set_abort(volatile int* abort, int32_t* status) {
  *abort = 1;
  if (status) atomicExch(status, kStatusTimeout);
}

template <int R, bool kQe4m3, bool kNv>
__global__ void __launch_bounds__((TcCfg<R, kQe4m3, kNv>::kThreads), (TcCfg<R, kQe4m3, kNv>::kMinBlocks))
decode_tc_kernel(const DecodeDev a, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, const __grid_constant__ CUtensorMap tmap_ks,
                 const __grid_constant__ CUtensorMap tmap_vs, int n_q_tiles) {
  // Launched as a programmatic dependent: no global load or store before
  // the grid ahead of this one has completed.  The merge (this grid's own
  // dependent) may launch now; its CTAs wait the same way.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  using C = TcCfg<R, kQe4m3, kNv>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(sm);
  float* red = reinterpret_cast<float*>(sm + C::kOffRed);      // [4][R]
  float* m_s = reinterpret_cast<float*>(sm + C::kOffM);        // [2][R]
  float* corr_s = reinterpret_cast<float*>(sm + C::kOffCorr);  // [R]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffMisc + 4);
  int* q_shift = reinterpret_cast<int*>(sm + C::kOffMisc + 8);
  float* amax_red = reinterpret_cast<float*>(sm + C::kOffMisc + 16);  // [8]

  Bars bar;
  {
    uint32_t p = sbase + C::kOffBar;
    bar.kfull = p;
    p += 8 * C::kStages;
    bar.vfull = p;
    p += 8 * C::kStages;
    bar.kvempty = p;
    p += 8 * C::kStages;
    bar.sfull = p;
    p += 16;
    bar.sfree = p;
    p += 16;
    bar.pfull = p;
    p += 16;
    bar.pfree = p;
    p += 16;
    bar.odone = p;
    p += 8;
    bar.qready = p;
    p += 8;
    bar.drain = p;
    p += 8;
    bar.pkfull = p;
    p += 8 * C::kPkStages;
    bar.pkempty = p;
  }

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Linear grid, work item outermost: the plan's longest-first order holds
  // for the whole launch, and the heads / query tiles of one work item (which
  // read the same KV pages) run side by side.
  const int g = blockIdx.x % a.h_k;
  const int rest = blockIdx.x / a.h_k;
  const int qt = rest % n_q_tiles;
  const int w_idx = rest / n_q_tiles;
  const int n0 = qt * R;

  const int4 item = reinterpret_cast<const int4*>(a.work)[w_idx];
  const int b = item.x, t_begin = item.y, t_end = item.z, slot = item.w;
  if (t_end <= t_begin) return;  // padding item: uniform exit before any setup
  const int T = t_end - t_begin;
  // The producer's lane j reads page j of the first tile now, alongside the
  // sequence length (which only masks the pages past it): the first copies
  // then wait for one memory round trip after the work item, not two.
  const int PS = a.page_size;
  const int ppt = kTileKV / PS;  // pages per tile: 1, 2, 4 or 8
  const int64_t bt_row = static_cast<int64_t>(b) * a.max_blocks;
  int first_page_raw = 0;
  if (warp == 0 && lane < ppt && t_begin * ppt + lane < a.max_blocks)
    first_page_raw = a.block_table[bt_row + t_begin * ppt + lane];
  const int L = a.seq_lens[b];

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      // e4m3 stages: filled by the TMA (one arrival with its byte count), or
      // by the converter warps (one arrival each)
      ptx::mbar_init(bar.kfull + 8 * s, kNv ? C::kCvtWarps : 1);
      ptx::mbar_init(bar.vfull + 8 * s, kNv ? C::kCvtWarps : 1);
      ptx::mbar_init(bar.kvempty + 8 * s, 1);
    }
    for (int s = 0; s < C::kPkStages; ++s) {
      ptx::mbar_init(bar.pkfull + 8 * s, 1);
      ptx::mbar_init(bar.pkempty + 8 * s, C::kCvtWarps);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar.sfull + 8 * s, 1);
      ptx::mbar_init(bar.sfree + 8 * s, C::kSmWarps);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(bar.pfull + 8 * s, C::kSmWarps);
      ptx::mbar_init(bar.pfree + 8 * s, 1);
    }
    ptx::mbar_init(bar.odone, 1);
    ptx::mbar_init(bar.qready, 1);
    ptx::mbar_init(bar.drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + C::kOffMisc, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;                // S buffers: columns [0, 2 kN1)
  const uint32_t tmem_o = tmem + 2 * C::kN1;   // O: columns [2 kN1, 2 kN1 + kN2)

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Lane j handles page j of each tile: the block-table lookups of a tile
    // run in parallel, and the next tile's lookups are in flight while this
    // tile's copies are issued.
    int valid_pages = (L + PS - 1) / PS;
    valid_pages = valid_pages < a.max_blocks ? valid_pages : a.max_blocks;
    auto lookup = [&](int tile) -> int {
      const int blk = tile * ppt + lane;
      // pages past the sequence end are read out of range: zeros
      return (lane < ppt && blk < valid_pages) ? a.block_table[bt_row + blk] : a.num_pages;
    };
    if (lane == 0) {
      ptx::prefetch_tmap(&tmap_k);
      ptx::prefetch_tmap(&tmap_v);
    }
    const bool evict_first = a.kv_evict_first != 0;
    const uint64_t kv_policy = ptx::policy_evict_first();
    const uint32_t tile_tx = kv_box_bytes(a.kv_format, kTileKV);
    int next_page = (lane < ppt && t_begin * ppt + lane < valid_pages) ? first_page_raw : a.num_pages;
    int issued = 0;
    if constexpr (kNv) {
      // nvfp4: each tile's K and V codes (PS rows of 64 bytes a page) and
      // their scales (PS rows of 8 bytes a page, from the scale plane) into a
      // packed stage; the converter warps turn it into e4m3 stages
      if (lane == 0) {
        ptx::prefetch_tmap(&tmap_ks);
        ptx::prefetch_tmap(&tmap_vs);
      }
      for (int i = 0; i < T; ++i) {
        const int ps = i % C::kPkStages;
        if (i >= C::kPkStages) {
          const bool got =
              ptx::mbar_wait_bounded(bar.pkempty + 8 * ps, ((i / C::kPkStages) - 1) & 1, abort_flag, kWaitNs);
          if (__any_sync(0xffffffffu, !got)) {
            if (lane == 0) set_abort(abort_flag, a.status);
            break;
          }
        }
        const int page = next_page;
        if (i + 1 < T) next_page = lookup(t_begin + i + 1);
        const uint32_t pk = sbase + C::kOffPk + ps * C::kPkBytes;
        if (lane == 0) ptx::mbar_arrive_expect_tx(bar.pkfull + 8 * ps, C::kPkBytes);
        __syncwarp();
        if (lane < ppt) {
          const uint32_t pb = bar.pkfull + 8 * ps;
          ptx::tma_load_kv(pk + lane * PS * 64, &tmap_k, pb, 0, 0, g, page, evict_first, kv_policy);
          ptx::tma_load_kv(pk + C::kPkCodes + lane * PS * 64, &tmap_v, pb, 0, 0, g, page, evict_first, kv_policy);
          ptx::tma_load_kv(pk + 2 * C::kPkCodes + lane * PS * 8, &tmap_ks, pb, 0, 0, g, page, evict_first,
                           kv_policy);
          ptx::tma_load_kv(pk + 2 * C::kPkCodes + C::kPkScales + lane * PS * 8, &tmap_vs, pb, 0, 0, g, page,
                           evict_first, kv_policy);
        }
        issued = i + 1;
      }
      if (*abort_flag && lane == 0) {
        for (int i = (issued > C::kPkStages ? issued - C::kPkStages : 0); i < issued; ++i) {
          volatile int never = 0;
          ptx::mbar_wait_bounded(bar.pkfull + 8 * (i % C::kPkStages), (i / C::kPkStages) & 1, &never, kWaitNs / 4);
        }
      }
    } else {
    for (int i = 0; i < T; ++i) {
      const int st = i % C::kStages;
      if (i >= C::kStages) {
        const bool got =
            ptx::mbar_wait_bounded(bar.kvempty + 8 * st, ((i / C::kStages) - 1) & 1, abort_flag, kWaitNs);
        if (__any_sync(0xffffffffu, !got)) {  // leave the loop together
          if (lane == 0) set_abort(abort_flag, a.status);
          break;
        }
      }
      const int page = next_page;
      if (i + 1 < T) next_page = lookup(t_begin + i + 1);
      // L2 prefetch of a tile further ahead: its HBM latency overlaps the
      // wait for a free stage, and its TMA load later hits L2.
      const int ahead = i + a.l2_prefetch;
      if (a.l2_prefetch > 0 && ahead < T) {
        for (int pf = (i == 0 ? 1 : ahead); pf <= ahead; ++pf) {
          const int pp = lookup(t_begin + pf);
          if (lane < ppt && pp < a.num_pages) {
            ptx::tma_prefetch_l2_4d(&tmap_k, 0, 0, g, pp);
            ptx::tma_prefetch_l2_4d(&tmap_v, 0, 0, g, pp);
          }
        }
      }
      const uint32_t dk = sbase + C::kOffK + st * kKVTileBytes;
      const uint32_t dv = sbase + C::kOffV + st * kKVTileBytes;
      if (lane == 0) {  // the packed bytes the tile's boxes read (16 KB for e4m3)
        ptx::mbar_arrive_expect_tx(bar.kfull + 8 * st, tile_tx);
        ptx::mbar_arrive_expect_tx(bar.vfull + 8 * st, tile_tx);
      }
      __syncwarp();
      if (lane < ppt) {
        ptx::tma_load_kv(dk + lane * PS * 128, &tmap_k, bar.kfull + 8 * st, 0, 0, g, page, evict_first, kv_policy);
        ptx::tma_load_kv(dv + lane * PS * 128, &tmap_v, bar.vfull + 8 * st, 0, 0, g, page, evict_first, kv_policy);
      }
      issued = i + 1;
    }
    if (*abort_flag && lane == 0) {
      // drain: wait (bounded) for every tile this warp issued to land
      for (int i = (issued > C::kStages ? issued - C::kStages : 0); i < issued; ++i) {
        const int st = i % C::kStages;
        const uint32_t par = (i / C::kStages) & 1;
        volatile int never = 0;
        ptx::mbar_wait_bounded(bar.kfull + 8 * st, par, &never, kWaitNs / 4);
        ptx::mbar_wait_bounded(bar.vfull + 8 * st, par, &never, kWaitNs / 4);
      }
    }
    }  // e4m3 and the other narrow formats
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      // A = the K / V tile in the pool's format, B = e4m3 (Q and P parts)
      const uint32_t kv_fmt = kv_mma_format(a.kv_format);
      const uint32_t idesc_s = ptx::idesc_f8f6f4(kTileKV, C::kN1, false, false, kv_fmt, 0);  // S = K Q^T
      const uint32_t idesc_o = ptx::idesc_f8f6f4(kTileKV, C::kN2, true, true, kv_fmt, 0);    // O = V^T P
      const uint32_t q_base = sbase + C::kOffQ;
      bool ok = ptx::mbar_wait_bounded(bar.qready, 0, abort_flag, kWaitNs);
      // Issue GEMM1 and GEMM2 as their inputs become ready, whichever comes
      // first: GEMM2(j) must not wait behind the arrival of a later K tile,
      // or the ring's stages would be released one TMA latency late.
      int g1 = 0, g2 = 0;
      uint64_t stall_since = 0;
      while (ok && g2 < T) {
        bool progressed = false;
        if (g1 < T) {
          const int st = g1 % C::kStages;
          const int sb = g1 & 1;
          if (ptx::mbar_test_wait(bar.kfull + 8 * st, (g1 / C::kStages) & 1) &&
              (g1 < 2 || ptx::mbar_test_wait(bar.sfree + 8 * sb, ((g1 >> 1) - 1) & 1))) {
            ptx::tc_fence_after();
            const uint32_t k_base = sbase + C::kOffK + st * kKVTileBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // A = K (K-major, 128-byte swizzle, 8-row groups 1024 B apart);
              // B = Q hi|lo rows (same layout); one K step = 32 bytes of d.
              const uint64_t ad = ptx::smem_desc(k_base + kk * 32, 16, 1024, ptx::kSwizzle128B);
              const uint64_t bd = ptx::smem_desc(q_base + kk * 32, 16, 1024, ptx::kSwizzle128B);
              ptx::mma_e4m3(tmem_s + sb * C::kN1, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit(bar.sfull + 8 * sb);
            ++g1;
            progressed = true;
          }
        }
        if (g2 < g1) {
          const int st = g2 % C::kStages;
          const int pb = g2 % C::kPBufs;
          if (ptx::mbar_test_wait(bar.pfull + 8 * pb, (g2 / C::kPBufs) & 1) &&
              ptx::mbar_test_wait(bar.vfull + 8 * st, (g2 / C::kStages) & 1)) {
            ptx::tc_fence_after();
            const uint32_t v_base = sbase + C::kOffV + st * kKVTileBytes;
            const uint32_t p_base = sbase + C::kOffP + pb * C::kPBytes;
#pragma unroll
            for (int kk = 0; kk < kTileKV / 32; ++kk) {
              // A = V^T: MN-major, 128-byte swizzle, 8-row groups 1024 B
              // apart; one K step = 32 KV rows = 4 groups.  B = P hi|lo:
              // MN-major, no swizzle, 8-row core matrices 128 B apart along
              // K, 16-column groups 2048 B apart along N.
              const uint64_t ad = ptx::smem_desc(v_base + kk * 4096, 0, 1024, ptx::kSwizzle128B);
              const uint64_t bd = ptx::smem_desc(p_base + kk * 512, 128, 2048, ptx::kSwizzleNone);
              ptx::mma_e4m3(tmem_o, ad, bd, idesc_o, (g2 > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(bar.odone);
            ptx::mma_commit(bar.pfree + 8 * pb);
            ptx::mma_commit(bar.kvempty + 8 * st);
            ++g2;
            progressed = true;
          }
        }
        if (progressed) {
          stall_since = 0;
        } else {
          // Nothing ready: sleep on the event the pipeline needs next (P of
          // the oldest tile, else K of the next one) instead of spinning on
          // the issue slots the softmax warps share with this warp.
          if (g2 < g1)
            ptx::mbar_try_wait_hint(bar.pfull + 8 * (g2 % C::kPBufs), (g2 / C::kPBufs) & 1, 200);
          else if (g1 < T)
            ptx::mbar_try_wait_hint(bar.kfull + 8 * (g1 % C::kStages), (g1 / C::kStages) & 1, 200);
          const uint64_t now = ptx::globaltimer_ns();
          if (stall_since == 0) stall_since = now;
          if (*abort_flag || now - stall_since > kWaitNs) ok = false;
        }
      }
      if (!ok) set_abort(abort_flag, a.status);
      // every MMA this thread issued has completed once `drain` fires
      ptx::mma_commit(bar.drain);
      volatile int never = 0;
      ptx::mbar_wait_bounded(bar.drain, 0, &never, kWaitNs);
    }
  } else if (warp < 2 + C::kSmWarps) {
    // ------------------------------------------------- softmax warpgroup
    constexpr int kCols = C::kCols;
    constexpr int kSmT = C::kSmThreads;
    const int sw = warp - 2;          // 0 .. kSmWarps-1 within the softmax group
    const int quarter = warp & 3;     // TMEM lane quarter this warp may access
    const int col0 = (sw / 4) * kCols;  // first column of this thread's half
    const int st_tid = sw * 32 + lane;
    const int row = quarter * 32 + lane;  // TMEM lane: KV row (S) / d (O)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    constexpr int kBarSm = 1;         // named barrier id of the softmax group

    const float qd = a.qd[b * a.qd_seq + g * a.qd_head];
    const float kd = a.kd[b * a.kd_seq + g * a.kd_head];
    const float vd = a.vd[b * a.vd_seq + g * a.vd_head];

    // ---- Q tile -> shared: e4m3 rows in the 128-byte swizzled K-major
    // layout, [hi rows 0..R) [lo rows R..2R) for bf16 Q
    {
      constexpr int kChunks = (R * 8 + kSmT - 1) / kSmT;  // (row, 16-byte chunk) pairs per thread
      float amax = 0.f;
      float xv[kChunks][16];
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const int id = k * kSmT + st_tid;
        const int n = id >> 3, cc = id & 7;
        const int qrow = n0 + n;
#pragma unroll
        for (int e = 0; e < 16; ++e) xv[k][e] = 0.f;
        if (n < R && qrow < a.n_q) {
          const int64_t off = b * a.q_seq + (static_cast<int64_t>(g) * a.n_q + qrow) * kHeadDimDev + cc * 16;
          if (kQe4m3) {
            const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) + off);
            const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) e4m3x4_to_f32(w4[wi], &xv[k][wi * 4]);
          } else {
            const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + off);
            const uint4 r0 = src[0], r1 = src[1];
            const uint32_t w8[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int wi = 0; wi < 8; ++wi) {
              xv[k][2 * wi] = __uint_as_float(w8[wi] << 16);
              xv[k][2 * wi + 1] = __uint_as_float(w8[wi] & 0xFFFF0000u);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(xv[k][e]));
      }
      int shift = 0;
      if (!kQe4m3) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) amax_red[sw] = amax;
        ptx::named_bar_sync(kBarSm, kSmT);
        for (int w = 0; w < C::kSmWarps; ++w) amax = fmaxf(amax, amax_red[w]);
        if (amax > 0.f) {
          const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;  // floor(log2) for normals
          shift = 7 - e;
          shift = shift > 126 ? 126 : (shift < -126 ? -126 : shift);
        }
      }
      const float qscale = kQe4m3 ? 1.f : ldexpf(1.f, shift);
      // rows of the Q buffer no thread fills (e4m3 Q with R < 16) are zero
      if (kQe4m3 && R < C::kN1) {
        for (int id = st_tid; id < (C::kN1 - R) * 8; id += kSmT)
          *reinterpret_cast<uint4*>(sm + C::kOffQ + R * 128 + id * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const int id = k * kSmT + st_tid;
        const int n = id >> 3, cc = id & 7;
        if (n < R) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            uint16_t h01, h23, l01 = 0, l23 = 0;
            if (kQe4m3) {
              h01 = ptx::f32x2_to_e4m3x2(xv[k][4 * wi], xv[k][4 * wi + 1]);
              h23 = ptx::f32x2_to_e4m3x2(xv[k][4 * wi + 2], xv[k][4 * wi + 3]);
            } else {
              float x[4], hf[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) x[e] = xv[k][4 * wi + e] * qscale;
              h01 = ptx::f32x2_to_e4m3x2(x[0], x[1]);
              h23 = ptx::f32x2_to_e4m3x2(x[2], x[3]);
              e4m3x4_to_f32(static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16), hf);
              l01 = ptx::f32x2_to_e4m3x2(x[0] - hf[0], x[1] - hf[1]);
              l23 = ptx::f32x2_to_e4m3x2(x[2] - hf[2], x[3] - hf[3]);
            }
            hw[wi] = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
            lw[wi] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
          }
          // 128-byte swizzle: chunk cc of row n at chunk position cc ^ (n % 8)
          *reinterpret_cast<uint4*>(sm + C::kOffQ + n * 128 + ((cc ^ (n & 7)) << 4)) =
              make_uint4(hw[0], hw[1], hw[2], hw[3]);
          if (!kQe4m3) {
            const int nl = R + n;
            *reinterpret_cast<uint4*>(sm + C::kOffQ + nl * 128 + ((cc ^ (nl & 7)) << 4)) =
                make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      if (st_tid == 0) *q_shift = shift;
      if (st_tid < R) m_s[st_tid] = -INFINITY;  // running max starts at -inf
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(kBarSm, kSmT);
      if (st_tid == 0) ptx::mbar_arrive(bar.qready);
    }
    const int shift = *q_shift;
    // raw (computed) score -> logit and -> log2 units; 2^-shift undoes the Q scaling
    const float cta_scale = a.softmax_scale * qd * kd * ldexpf(1.f, -shift);
    const float c2 = cta_scale * kLog2e;
    const float head_c = kTau / c2;  // kTau in raw score units

    float l_thr[kCols];  // deferred row sums (of 448 p) for this thread's columns
#pragma unroll
    for (int c = 0; c < kCols; ++c) l_thr[c] = 0.f;
    int mb = 0;  // which half of m_s holds the running column max (raw units)

    bool ok = true;
    const int vis_all = a.causal ? L - a.q_len : L - 1;  // keys every row sees
    for (int i = 0; i < T; ++i) {
      const int sb = i & 1;
      const int j = (t_begin + i) * kTileKV + row;  // this thread's key
      if (!ptx::mbar_wait_bounded(bar.sfull + 8 * sb, (i >> 1) & 1, abort_flag, kWaitNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      float sc[kCols];
      // S row of this thread's key for its columns (hi + lo partial
      // products), masked by select: garbage or poison rows never leak
      auto load_s = [&]() {
        const uint32_t s_base = tmem_s + lane_off + sb * C::kN1;
        if constexpr (C::kHalves == 1) {
          uint32_t r[C::kN1];  // every chunk in flight, one wait
#pragma unroll
          for (int c0 = 0; c0 < C::kN1; c0 += 16) MJ_TMEM_LD16(s_base + c0, (r + c0));
          ptx::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < R; ++c) {
            sc[c] = __uint_as_float(r[c]);
            if (!kQe4m3) sc[c] += __uint_as_float(r[R + c]);
          }
        } else {
          uint32_t r[2 * kCols];
#pragma unroll
          for (int c0 = 0; c0 < kCols; c0 += 16) {
            MJ_TMEM_LD16(s_base + col0 + c0, (r + c0));
            if (!kQe4m3) MJ_TMEM_LD16(s_base + R + col0 + c0, (r + kCols + c0));
          }
          ptx::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            sc[c] = __uint_as_float(r[c]);
            if (!kQe4m3) sc[c] += __uint_as_float(r[kCols + c]);
          }
        }
        if (j > vis_all) {
#pragma unroll
          for (int c = 0; c < kCols; ++c) {
            const int n = n0 + col0 + c;
            int lim = a.causal ? L - a.q_len + n / a.h_r : L - 1;
            lim = lim < L - 1 ? lim : L - 1;
            if (j > lim) sc[c] = -INFINITY;
          }
        }
      };
      load_s();

      // Reference maxima (shared, identical for every thread): only when
      // some score passes its column's m + kTau (one barrier-reduction
      // answers that for the group) are the column maxima reduced:
      // reduce-scatter in the warp, the four warps through shared memory,
      // then thread c updates column c.  Otherwise the tile needs no
      // exchange at all.
      const float* m_now = m_s + mb * R + col0;
      bool exceed = false;
#pragma unroll
      for (int c4 = 0; c4 < kCols; c4 += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(m_now + c4);
        exceed |= (sc[c4] > m4.x + head_c) | (sc[c4 + 1] > m4.y + head_c) | (sc[c4 + 2] > m4.z + head_c) |
                  (sc[c4 + 3] > m4.w + head_c);
      }
      bool moved = false;
      if (ptx::named_bar_red_or(kBarSm, kSmT, exceed)) {
        warp_reduce_scatter<kCols, true>(sc, lane);  // in place; S is read again below
        if (warp_col_writer<kCols>(lane)) {
          const int col = col0 + warp_col<kCols>(lane);
          red[quarter * R + col] = sc[0];
          if (kCols == 64) red[quarter * R + 32 + col] = sc[1];
        }
        ptx::named_bar_sync(kBarSm, kSmT);
        bool moved_c = false;
        if (st_tid < R) {
          const int c = st_tid;
          const float t = fmaxf(fmaxf(red[c], red[R + c]), fmaxf(red[2 * R + c], red[3 * R + c]));
          const float mo = m_s[mb * R + c];
          moved_c = t > mo + head_c;
          const float mn = moved_c ? t : mo;
          // corr = 2^((m_old - m_use) c2); the -inf guard makes it 0 for a
          // column that had seen no key
          const float mu = (mn == -INFINITY) ? 0.f : mn;
          corr_s[c] = moved_c ? fast_exp2((mo - mu) * c2) : 1.f;
          m_s[(mb ^ 1) * R + c] = mn;
        }
        moved = ptx::named_bar_red_or(kBarSm, kSmT, moved_c);
        mb ^= 1;
        if (moved) {
#pragma unroll
          for (int c4 = 0; c4 < kCols; c4 += 4) {
            const float4 f = *reinterpret_cast<const float4*>(corr_s + col0 + c4);
            l_thr[c4] *= f.x;
            l_thr[c4 + 1] *= f.y;
            l_thr[c4 + 2] *= f.z;
            l_thr[c4 + 3] *= f.w;
          }
        }
        load_s();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar.sfree + 8 * sb);
      // lazy O correction (both the hi and the lo columns of a row): only
      // when some column max moved, after GEMM2(i-1)
      if (moved && i > 0) {
        if (!ptx::mbar_wait_bounded(bar.odone, (i - 1) & 1, abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // this thread's columns of O: hi [col0, col0 + kCols), lo R + those
#pragma unroll
        for (int part = 0; part < 2; ++part) {
#pragma unroll
          for (int c0 = 0; c0 < kCols; c0 += 16) {
            const int oc = (C::kHalves == 1) ? (part * 16 + c0) : (part * R + col0 + c0);
            if (C::kHalves == 1 && oc >= C::kN2) break;
            uint32_t r[16];
            MJ_TMEM_LD16(tmem_o + lane_off + oc, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              r[e] = __float_as_uint(__uint_as_float(r[e]) * corr_s[(oc + e) % R]);
            MJ_TMEM_ST16(tmem_o + lane_off + oc, r);
          }
        }
        ptx::tmem_st_wait();
      }
      // x = 448 p 2^-kTau = 2^((s - m) c2 + log2 448 - kTau), within e4m3's
      // range; the row sums keep the same factor.  The -inf guard uses 0 as
      // the reference of a column that has seen no key yet.
      {
        const float* m_new = m_s + mb * R + col0;
#pragma unroll
        for (int c4 = 0; c4 < kCols; c4 += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(m_new + c4);
          const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float m_use = (mm[e] == -INFINITY) ? 0.f : mm[e];
            const float p = fast_exp2(fmaf(sc[c4 + e], c2, fmaf(-m_use, c2, kLog2PScale)));
            l_thr[c4 + e] += p;
            sc[c4 + e] = p;
          }
        }
      }
      // P buffer i % kPBufs is free once GEMM2(i - kPBufs) finished reading it
      const int pb = i % C::kPBufs;
      if (i >= C::kPBufs &&
          !ptx::mbar_wait_bounded(bar.pfree + 8 * pb, ((i / C::kPBufs) - 1) & 1, abort_flag, kWaitNs)) {
        ok = false;
        break;
      }
      // split x = hi + lo (e4m3, through half precision); hi -> column c,
      // lo -> column R + c of the P buffer [kN2/16 groups][128 rows][16 bytes]
      {
        uint32_t hw[kCols / 4], lw[kCols / 4];
        split_e4m3_hilo<kCols, kLoShift>(sc, hw, lw);
        uint8_t* pbuf = sm + C::kOffP + pb * C::kPBytes + row * 16;
        if (R == 8) {
          *reinterpret_cast<uint4*>(pbuf) = make_uint4(hw[0], hw[1], lw[0], lw[1]);
        } else {
#pragma unroll
          for (int gq = 0; gq < kCols / 16; ++gq) {
            *reinterpret_cast<uint4*>(pbuf + (col0 / 16 + gq) * (kTileKV * 16)) =
                make_uint4(hw[4 * gq], hw[4 * gq + 1], hw[4 * gq + 2], hw[4 * gq + 3]);
            *reinterpret_cast<uint4*>(pbuf + ((R + col0) / 16 + gq) * (kTileKV * 16)) =
                make_uint4(lw[4 * gq], lw[4 * gq + 1], lw[4 * gq + 2], lw[4 * gq + 3]);
          }
        }
      }
      // rows past the sequence end: zero their V row so 0 * poison cannot
      // reach O (the TMA landed the whole last page).  Every thread of a
      // tile that reaches the end waits, so that a wait that gives up does
      // so in all warps alike.
      if ((t_begin + i + 1) * kTileKV > L) {
        const int st = i % C::kStages;
        if (!ptx::mbar_wait_bounded(bar.vfull + 8 * st, (i / C::kStages) & 1, abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        if (j >= L && col0 == 0) {
          uint4* vrow = reinterpret_cast<uint4*>(sm + C::kOffV + st * kKVTileBytes + row * 128);
#pragma unroll
          for (int e = 0; e < 8; ++e) vrow[e] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar.pfull + 8 * pb);
    }

    // ---- epilogue
    // `drain` fires once every MMA the CTA issued is done (a parity wait on
    // `odone` could not tell GEMM2(T - 1) from GEMM2(T - 3) when two P
    // buffers let two GEMM2s be in flight)
    if (ok && !ptx::mbar_wait_bounded(bar.drain, 0, abort_flag, kWaitNs)) ok = false;
    if (*abort_flag) ok = false;
    if (!ok) {
      set_abort(abort_flag, a.status);
    } else {
      ptx::tc_fence_after();
      // row sums: reduce over the 128 KV rows
      ptx::named_bar_sync(kBarSm, kSmT);  // everyone is done reading red
      warp_reduce_scatter<kCols, false>(l_thr, lane);
      if (warp_col_writer<kCols>(lane)) {
        const int col = col0 + warp_col<kCols>(lane);
        red[quarter * R + col] = l_thr[0];
        if (kCols == 64) red[quarter * R + 32 + col] = l_thr[1];
      }
      const float* m_fin = m_s + mb * R;
      ptx::named_bar_sync(kBarSm, kSmT);
      const int nsp = a.n_splits[b];
      const bool final_out = nsp <= 1;
      const float out_scale = vd * kPScaleInv;  // O and the row sums both carry 448 2^-kTau
      const int d = row;  // TMEM lane of O = head-dim index
      float o_row[kCols];  // O[d][c] = hi column c + lo column R + c
      if constexpr (C::kHalves == 1) {
#pragma unroll
        for (int c0 = 0; c0 < C::kN2; c0 += 16) {
          uint32_t r[16];
          MJ_TMEM_LD16(tmem_o + lane_off + c0, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = c0 + e;
            if (c < R)
              o_row[c] = __uint_as_float(r[e]);
            else
              o_row[c - R] += __uint_as_float(r[e]) * kLoInv;
          }
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < kCols; c0 += 16) {
          uint32_t rh[16], rl[16];
          MJ_TMEM_LD16(tmem_o + lane_off + col0 + c0, rh);
          MJ_TMEM_LD16(tmem_o + lane_off + R + col0 + c0, rl);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o_row[c0 + e] = __uint_as_float(rh[e]) + __uint_as_float(rl[e]) * kLoInv;
        }
      }
#pragma unroll
      for (int cl = 0; cl < kCols; ++cl) {
        const int c = col0 + cl;
        const int n = n0 + c;
        if (n >= a.n_q) break;
        const float l = (red[c] + red[R + c] + red[2 * R + c] + red[3 * R + c]) * kPScaleInv;
        const float o = o_row[cl] * out_scale;
        if (final_out) {
          const int64_t orow = b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + n) * kHeadDimDev;
          a.o[orow + d] = __float2bfloat16_rn(o * (a.scale_o / (l + 1e-30f)));
        } else {
          const int64_t pr = part_row(a, b, g, slot, n);
          a.o_part[pr * kHeadDimDev + d] = o;
        }
      }
      if (st_tid < R && n0 + st_tid < a.n_q) {
        const int c = st_tid, n = n0 + c;
        const float l = (red[c] + red[R + c] + red[2 * R + c] + red[3 * R + c]) * kPScaleInv;
        const float m_logit = m_fin[c] * cta_scale;
        if (final_out) {
          a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + n] = m_logit + logf(l);
        } else {
          const int64_t pr = part_row(a, b, g, slot, n);
          a.m_part[pr] = m_logit;
          a.l_part[pr] = l;
        }
      }
    }
  } else if constexpr (kNv) {
    // ---------------------------------------------- nvfp4 converter warps
    // Tile i: its packed stage (K codes, V codes, K scales, V scales, rows of
    // 64 and 8 bytes) -> e4m3 stage i % kStages in the layout the TMA gives
    // e4m3 pools (128-byte rows, 16-byte chunk cc of row r at cc ^ (r % 8)),
    // once GEMM2 of the tile that used the stage before has completed.
    // Thread j of the group converts groups j, j + 128, ... of each tile;
    // rows at or past the sequence end are written as zeros.
    const int ct = tid - (64 + C::kSmThreads);  // 0 .. 127
    bool ok = true;
    for (int i = 0; i < T; ++i) {
      const int ps = i % C::kPkStages;
      const int st = i % C::kStages;
      if (!ptx::mbar_wait_bounded(bar.pkfull + 8 * ps, (i / C::kPkStages) & 1, abort_flag, kWaitNs) ||
          (i >= C::kStages &&
           !ptx::mbar_wait_bounded(bar.kvempty + 8 * st, ((i / C::kStages) - 1) & 1, abort_flag, kWaitNs))) {
        ok = false;
        break;
      }
      const int key0 = (t_begin + i) * kTileKV;
      const uint8_t* pk = sm + C::kOffPk + ps * C::kPkBytes;
#pragma unroll
      for (int kv = 0; kv < 2; ++kv) {
        const uint8_t* codes = pk + kv * C::kPkCodes;
        const uint8_t* scales = pk + 2 * C::kPkCodes + kv * C::kPkScales;
        uint8_t* dst = sm + (kv ? C::kOffV : C::kOffK) + st * kKVTileBytes;
#pragma unroll 2
        for (int j = ct; j < kTileKV * 8; j += 128) {
          const int r = j >> 3, cc = j & 7;
          uint4 e = make_uint4(0u, 0u, 0u, 0u);
          if (key0 + r < L)
            e = nvfp4_group_to_e4m3(*reinterpret_cast<const uint2*>(codes + r * 64 + cc * 8), scales[r * 8 + cc]);
          *reinterpret_cast<uint4*>(dst + r * 128 + ((cc ^ (r & 7)) << 4)) = e;
        }
      }
      ptx::fence_proxy_async_smem();  // generic-proxy writes -> the MMA's reads
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(bar.kfull + 8 * st);
        ptx::mbar_arrive(bar.vfull + 8 * st);
        ptx::mbar_arrive(bar.pkempty + 8 * ps);
      }
    }
    if (!ok && lane == 0) set_abort(abort_flag, a.status);
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::kTmemCols);
}

// nvfp4 pools as byte tensors: the codes (64 bytes a row) and the scale
// plane (a page's rows of one head, PS x 8 bytes, seen as PS / 16 rows of
// 128 bytes); one box is one page of one head, unswizzled.
bool make_nv_map(CUtensorMap* m, const uint8_t* base, bool scales, int page_size, int h_k, int num_pages,
                 int64_t s_row, int64_t s_head, int64_t s_page) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t inner = scales ? 128 : 64;
  const cuuint64_t rows = scales ? static_cast<cuuint64_t>(page_size / 16) : static_cast<cuuint64_t>(page_size);
  const cuuint64_t dims[4] = {inner, rows, static_cast<cuuint64_t>(h_k), static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(scales ? 128 : s_row), static_cast<cuuint64_t>(s_head),
                                 static_cast<cuuint64_t>(s_page)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(inner), static_cast<cuuint32_t>(rows), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int R, bool kQe4m3, bool kNv>
cudaError_t launch_tc(const DecodeDev& a, int n_q_tiles, cudaStream_t stream) {
  CUtensorMap mk, mv, mks, mvs;
  if (kNv) {
    if (!make_nv_map(&mk, a.k, false, a.page_size, a.h_k, a.num_pages, a.k_row, a.k_head, a.k_page) ||
        !make_nv_map(&mv, a.v, false, a.page_size, a.h_k, a.num_pages, a.v_row, a.v_head, a.v_page) ||
        !make_nv_map(&mks, a.ks, true, a.page_size, a.h_k, a.num_pages, 8, a.ks_head, a.ks_page) ||
        !make_nv_map(&mvs, a.vs, true, a.page_size, a.h_k, a.num_pages, 8, a.vs_head, a.vs_page))
      return cudaErrorInvalidValue;
  } else {
    if (!make_kv_map(&mk, a.k, a.page_size, a.h_k, a.num_pages, a.k_row, a.k_head, a.k_page, a.page_size, 1,
                     a.kv_format) ||
        !make_kv_map(&mv, a.v, a.page_size, a.h_k, a.num_pages, a.v_row, a.v_head, a.v_page, a.page_size, 1,
                     a.kv_format))
      return cudaErrorInvalidValue;
    mks = mk;  // unused by these instances
    mvs = mv;
  }
  using C = TcCfg<R, kQe4m3, kNv>;
  auto kern = decode_tc_kernel<R, kQe4m3, kNv>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.num_work) * n_q_tiles * a.h_k, 1, 1);
  return launch_pdl(kern, grid, dim3(C::kThreads, 1, 1), C::kBytes, stream, a, mk, mv, mks, mvs, n_q_tiles);
}

template <int R>
cudaError_t launch_tc_q(const DecodeDev& a, int n_q_tiles, bool q_e4m3, cudaStream_t stream) {
  if (a.kv_format == 4) {  // nvfp4: e4m3 Q, up to 32 rows (validated before)
    if constexpr (R <= 32) {
      if (q_e4m3) return launch_tc<R, true, true>(a, n_q_tiles, stream);
    }
    return cudaErrorInvalidValue;
  }
  return q_e4m3 ? launch_tc<R, true, false>(a, n_q_tiles, stream) : launch_tc<R, false, false>(a, n_q_tiles, stream);
}

// ---------------------------------------------------------------- checks
// The producer's page gather and the CUDA-core kernel's dequant as
// standalone launches, so that tests can compare them byte- and bit-exact
// with the oracle: the same tensor maps (make_kv_map), the same page lookup
// (lane j fetches page j of a 128-row tile through the block table; pages
// past the sequence end are fetched out of range, as zeros), the same TMA
// boxes, and the 128-byte swizzle the MMA descriptors assume, undone here.

// grid (tiles, h_k, num_seqs), 64 threads; out rows [b][g][row][128 bytes]
__global__ void __launch_bounds__(64) gather_kv_kernel(const DecodeDev a, const __grid_constant__ CUtensorMap tmap,
                                                       uint8_t* __restrict__ out, int out_rows) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tile = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t tile_s = ptx::smem_u32(tile);
  const uint32_t bar = tile_s + kKVTileBytes;
  const int t = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int L = a.seq_lens[b];
  const int T = L > 0 ? (L + kTileKV - 1) / kTileKV : 1;
  if (t >= T) return;  // uniform over the CTA
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (tid < 32) {
    const int PS = a.page_size;
    const int ppt = kTileKV / PS;
    int valid_pages = (L + PS - 1) / PS;
    valid_pages = valid_pages < a.max_blocks ? valid_pages : a.max_blocks;
    const int blk = t * ppt + lane;
    const int page = (lane < ppt && blk < valid_pages)
                         ? a.block_table[static_cast<int64_t>(b) * a.max_blocks + blk]
                         : a.num_pages;
    if (lane == 0) ptx::mbar_arrive_expect_tx(bar, kv_box_bytes(a.kv_format, kTileKV));
    __syncwarp();
    if (lane < ppt) ptx::tma_load_4d(tile_s + lane * PS * 128, &tmap, bar, 0, 0, g, page);
  }
  volatile int never = 0;
  if (!ptx::mbar_wait_bounded(bar, 0, &never, kWaitNs)) {  // rows stay unwritten: the test fails
    ptx::mbar_wait_bounded(bar, 0, &never, kWaitNs / 4);     // (a bounded drain before leaving)
    return;
  }
  for (int i = tid; i < kTileKV * 8; i += 64) {
    const int r = i >> 3, cc = i & 7;
    const int key = t * kTileKV + r;
    if (key >= L || key >= out_rows) continue;
    const uint4 v = *reinterpret_cast<const uint4*>(tile + r * 128 + ((cc ^ (r & 7)) << 4));
    *reinterpret_cast<uint4*>(out + ((static_cast<int64_t>(b) * a.h_k + g) * out_rows + key) * 128 + cc * 16) = v;
  }
}

// 64 threads: codes 4t .. 4t + 3 through the CUDA-core kernel's conversion
__global__ void dequant_e4m3_kernel(float* __restrict__ out) {
  const uint32_t c0 = 4u * threadIdx.x;
  const uint32_t w = c0 | ((c0 + 1) << 8) | ((c0 + 2) << 16) | ((c0 + 3) << 24);
  float v[4];
  e4m3x4_to_f32(w, v);
#pragma unroll
  for (int k = 0; k < 4; ++k) out[c0 + k] = v[k];
}

// The bounded-wait primitive on its own: one warp waits on an mbarrier that
// nothing arrives on, so the wait must give up after `limit_ns`; the warp then
// reports MJ_ERR_TIMEOUT in the status word, as the decode kernels do, and the
// time it waited.  No other warp and no named barrier is involved, so the
// launch ends whatever the primitive does with its limit.
__global__ void bounded_wait_kernel(int32_t* status, int64_t* waited_ns, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbar_init();
  }
  __syncwarp();
  const uint64_t t0 = ptx::globaltimer_ns();
  const bool done = ptx::mbar_wait_bounded(b, 0, &abort_flag, limit_ns);
  const uint64_t t1 = ptx::globaltimer_ns();
  if (threadIdx.x == 0) {
    if (!done) atomicExch(status, 5);  // MJ_ERR_TIMEOUT
    if (waited_ns) *waited_ns = static_cast<int64_t>(t1 - t0);
  }
}

}  // namespace

cudaError_t launch_bounded_wait(int32_t* status, int64_t* waited_ns, uint64_t limit_ns, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(status, waited_ns, limit_ns);
  return cudaGetLastError();
}

// nvfp4 pools: rows 0 .. L - 1 converted to e4m3 by the decode kernel's
// conversion (nvfp4_group_to_e4m3), codes and scales read through the block
// table with plain loads; grid (tiles, h_k, num_seqs), 128 threads.
__global__ void __launch_bounds__(128) gather_nvfp4_kernel(const DecodeDev a, bool values, uint8_t* __restrict__ out,
                                                           int out_rows) {
  const int t = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int L = a.seq_lens[b];
  const uint8_t* pool = values ? a.v : a.k;
  const uint8_t* scales = values ? a.vs : a.ks;
  const int64_t p_page = values ? a.v_page : a.k_page, p_row = values ? a.v_row : a.k_row;
  const int64_t p_head = values ? a.v_head : a.k_head;
  const int64_t s_page = values ? a.vs_page : a.ks_page, s_head = values ? a.vs_head : a.ks_head;
  for (int j = threadIdx.x; j < kTileKV * 8; j += 128) {
    const int key = t * kTileKV + (j >> 3), cc = j & 7;
    if (key >= L || key >= out_rows) continue;
    const int page = a.block_table[static_cast<int64_t>(b) * a.max_blocks + key / a.page_size];
    const int row = key % a.page_size;
    const uint2 c = *reinterpret_cast<const uint2*>(pool + page * p_page + row * p_row + g * p_head + cc * 8);
    const uint32_t sc = scales[page * s_page + g * s_head + row * 8 + cc];
    *reinterpret_cast<uint4*>(out + ((static_cast<int64_t>(b) * a.h_k + g) * out_rows + key) * 128 + cc * 16) =
        nvfp4_group_to_e4m3(c, sc);
  }
}

cudaError_t launch_gather_kv(const DecodeDev& a, bool values, uint8_t* out, int out_rows, cudaStream_t stream) {
  if (a.kv_format == 4) {
    const int tiles = (out_rows + kTileKV - 1) / kTileKV;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(a.h_k), static_cast<unsigned>(a.num_seqs));
    gather_nvfp4_kernel<<<grid, 128, 0, stream>>>(a, values, out, out_rows);
    return cudaGetLastError();
  }
  CUtensorMap m;
  const bool ok = values ? make_kv_map(&m, a.v, a.page_size, a.h_k, a.num_pages, a.v_row, a.v_head, a.v_page,
                                       a.page_size, 1, a.kv_format)
                         : make_kv_map(&m, a.k, a.page_size, a.h_k, a.num_pages, a.k_row, a.k_head, a.k_page,
                                       a.page_size, 1, a.kv_format);
  if (!ok) return cudaErrorInvalidValue;
  const int tiles = (out_rows + kTileKV - 1) / kTileKV;
  const int smem = kKVTileBytes + 1024 + 64;  // tile, alignment slack, mbarrier
  dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(a.h_k), static_cast<unsigned>(a.num_seqs));
  gather_kv_kernel<<<grid, 64, smem, stream>>>(a, m, out, out_rows);
  return cudaGetLastError();
}

cudaError_t launch_dequant_e4m3(float* out, cudaStream_t stream) {
  dequant_e4m3_kernel<<<1, 64, 0, stream>>>(out);
  return cudaGetLastError();
}

cudaError_t launch_decode_tc(const DecodeDev& a, int rows_per_cta, int n_q_tiles, bool q_e4m3,
                             cudaStream_t stream) {
  switch (rows_per_cta) {
    case 8: return launch_tc_q<8>(a, n_q_tiles, q_e4m3, stream);
    case 16: return launch_tc_q<16>(a, n_q_tiles, q_e4m3, stream);
    case 32: return launch_tc_q<32>(a, n_q_tiles, q_e4m3, stream);
    case 64: return launch_tc_q<64>(a, n_q_tiles, q_e4m3, stream);
    default: return cudaErrorInvalidValue;
  }
}

int tc_min_blocks(int rows_per_cta, bool q_e4m3, bool nvfp4) {
  if (nvfp4) return 1;
  switch (rows_per_cta) {
    case 8: return q_e4m3 ? TcCfg<8, true>::kMinBlocks : TcCfg<8, false>::kMinBlocks;
    case 16: return q_e4m3 ? TcCfg<16, true>::kMinBlocks : TcCfg<16, false>::kMinBlocks;
    case 32: return q_e4m3 ? TcCfg<32, true>::kMinBlocks : TcCfg<32, false>::kMinBlocks;
    case 64: return q_e4m3 ? TcCfg<64, true>::kMinBlocks : TcCfg<64, false>::kMinBlocks;
    default: return 1;
  }
}

int tc_smem_bytes(int rows_per_cta, bool q_e4m3, bool nvfp4) {
  if (nvfp4) {
    switch (rows_per_cta) {
      case 8: return TcCfg<8, true, true>::kBytes;
      case 16: return TcCfg<16, true, true>::kBytes;
      case 32: return TcCfg<32, true, true>::kBytes;
      default: return 0;
    }
  }
  switch (rows_per_cta) {
    case 8: return q_e4m3 ? TcCfg<8, true>::kBytes : TcCfg<8, false>::kBytes;
    case 16: return q_e4m3 ? TcCfg<16, true>::kBytes : TcCfg<16, false>::kBytes;
    case 32: return q_e4m3 ? TcCfg<32, true>::kBytes : TcCfg<32, false>::kBytes;
    case 64: return q_e4m3 ? TcCfg<64, true>::kBytes : TcCfg<64, false>::kBytes;
    default: return 0;
  }
}

}  // namespace mj
