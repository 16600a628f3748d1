// Head-grouped split-KV paged decode attention on the tensor cores (tcgen05,
// kind::f8f6f4) for GQA caches with several kv heads: a persistent kernel,
// one CTA per SM.
//
// Sources: as for the per-head kernel in decode_tc.cu — the
// "mjolnir/t5_decode.py" page (`decode`: paged TMA gather, select masking,
// online softmax with folded descales and the -inf guard, lazy O rescale,
// final-vs-partial epilogue, 448-scaled e4m3 P) and the swap-AB decode pull
// request page (KV slots on M, live heads on N).  What a work unit computes
// is the page's; which CTA computes it is not part of the result.
//
// Why a second kernel: one CTA per kv head reads each KV row of its head as
// a separate 128-byte piece, h_k*128 bytes apart; on GB300 that pattern
// streams at about 4.9 TB/s however deep the pipeline.  Here a CTA serves G
// kv heads of a work item and fetches each page's rows of all G heads as one
// TMA box.  Under load a TMA round trip takes 2-3 us, so the SM needs about
// 150 KB outstanding: the CTA owns the SM, keeps a six-stage ring of 32 KB
// tiles, and never drains it between work units — it takes units from a
// shared counter (greedy, longest first, as the plan orders them) and its
// producer streams the next unit's tiles while the softmax finishes the
// last one.
//
// Roles (416 threads): warps 0 and 12 issue the K and the V TMA tiles;
// warp 1 (one thread)
// issues the S = K Q^T MMAs and warp 11 (one thread) the O += V^T P MMAs —
// one thread issues a tcgen05.mma only every 70-100 cycles, slower than the
// tensor pipe runs them, and a 32 KB tile takes eight; warps 2-9 are two
// softmax warpgroups taking alternate tiles, each with its own S, O and
// running max (merged per unit); warp 10 fetches the next unit, its
// descriptor and scales, and converts its Q tile to e4m3, one unit ahead.
//
// One MMA tile is 128 rows = G heads x KR = 128/G keys (head-major: row
// h*KR + k).  Its N side holds the GR = G*RH query rows of all G heads
// (column h*RH + n), twice for bf16 Q (hi | lo e4m3 parts):
//   S[row, col]  = K[row] . Q[col]       -- only the head-diagonal blocks
//                                           (head(row) == head(col)) are used
//   O[d, col]   += V[row, d] P[row, col] -- P is zero off the diagonal, so
//                                           each column sums its own head
// The MMA costs the same ~70 cycles for any N up to 128, so computing the
// off-diagonal blocks is free; the zeros of P are written once.
//
// A head's KR rows live in one warp (G = 8: half a warp; G = 4: a warp), so
// the column maxima and row sums are warp-local shuffles; one barrier per
// tile tells a warpgroup whether any head's maximum moved (then its O, whose
// TMEM lanes are the head dimension and span all heads, is corrected).

#include <cuda.h>
#include <cuda_runtime.h>

#include "mj_device.cuh"
#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

constexpr int kRows = 128;                   // MMA M: rows of one tile
constexpr int kTileBytes = kRows * 128;      // one K or V tile: 16 KB
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far above any legal wait
constexpr int kStatusTimeout = 5;            // MJ_ERR_TIMEOUT
constexpr int kWG = 2;                       // softmax warpgroups
constexpr int kThreads = 64 + 128 * kWG + 96;
constexpr int kSchedWarp = 2 + 4 * kWG;      // warp index of the scheduler
constexpr int kMma2Warp = kSchedWarp + 1;    // warp index of the GEMM2 issuer
constexpr int kVLoadWarp = kSchedWarp + 2;   // warp index of the V-tile producer
constexpr int kItemBytes = 128;              // one unit descriptor in shared memory

constexpr int pow2_at_least(int x) {
  int p = 32;
  while (p < x) p <<= 1;
  return p;
}

template <int G, int RH, bool kQe4m3>
struct GCfg {
  static constexpr int kRH = RH;
  static constexpr int KR = kRows / G;     // keys per head per tile
  static constexpr int GR = G * RH;        // query columns of the CTA
  // G = 2: a head's 64 keys span two warps (a pair), which exchange their
  // column maxima and row sums through shared memory
  static constexpr bool kPair = KR >= 64;          // a head's keys span kWph warps
  static constexpr int kWph = kPair ? KR / 32 : 1;  // warps per head (2 or 4)
  static constexpr int HPW = kPair ? 1 : 32 / KR;  // heads per warp
  static constexpr int W = HPW * RH;       // S columns a warp reads
  static constexpr int kN1 = kQe4m3 ? (GR < 16 ? 16 : GR) : 2 * GR;
  static constexpr int kN2 = 2 * GR;
  // S buffers per warpgroup: two when they fit in TMEM beside O, else one
  // (the warpgroup's next GEMM1 then waits until its softmax has read S)
  static constexpr int kSBufs = 2 * kN1 + kN2 <= 256 ? 2 : 1;
  // K and V rings: a K stage is free once its GEMM1 ran, a V stage only
  // after the tile's softmax and GEMM2, so V gets more stages
  // P is produced as x = 448 p 2^-kTau: a column's reference maximum is
  // moved only when a score passes it by kTau (log2 units); kTau = 0 is the
  // exact running maximum
  static constexpr int kTau = 4;
  static constexpr float kLog2PScale = 8.807354922057604f - kTau;  // log2(448 2^-kTau)
  static constexpr float kPScaleInv = (1.f / 448.f) * (1 << kTau);
  // P's lo part is stored as e4m3((x - hi) 2^kLoShift); its products are
  // weighted back by 2^-kLoShift when the hi and lo columns of O are added
  static constexpr int kLoShift = 4;
  static constexpr float kLoInv = 1.f / (1 << kLoShift);
  static constexpr int kStagesK = kPair ? 4 : 5;
  static constexpr int kStagesV = kPair ? (G == 1 ? 6 : 5) : 7;
  static constexpr int kQBytes = kN1 * 128;
  // P (GEMM2's B operand, MN-major, no swizzle: [16-column groups][K rows][16 B]).
  //   G >= 4: one block-diagonal buffer per warpgroup, [kN2/16][128 rows],
  //     the off-diagonal zeros written once.
  //   G = 2: per head only its own columns, [2 RH/16][KR rows] (one GEMM2
  //     MMA chain per head), and two buffers per warpgroup, so that the
  //     softmax of a tile need not wait for the previous tile's GEMM2.
  static constexpr int kPBufs = kPair ? 2 : 1;
  static constexpr int kPHeadBytes = 2 * RH * KR;  // G = 2: one head's hi | lo columns
  static constexpr int kPBufBytes = kPair ? G * kPHeadBytes : kN2 * kRows;
  static constexpr int kPBytes = kPBufs * kPBufBytes;  // per warpgroup
  static constexpr int kWgCols = pow2_at_least(kSBufs * kN1 + kN2);  // TMEM per warpgroup: S, O
  static constexpr int kTmemCols = kWG * kWgCols;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kStagesK * kTileBytes;
  static constexpr int kOffQ = (kStagesK + kStagesV) * kTileBytes;  // [2 unit slots]
  static constexpr int kOffP = kOffQ + 2 * kQBytes;          // [kWG] P buffers
  static constexpr int kOffCorr = kOffP + kWG * kPBytes;     // [kWG][2][GR]
  // per group and unit slot: [GR] max, [GR] sum.  Group 0's state needs no
  // second slot for G >= 4 (its next unit cannot end before group 1 has
  // merged this one: that unit's GEMM2s wait for both groups' O-free); the
  // G = 2 layout has room for it.
  static constexpr int kOffStat = kOffCorr + kWG * 2 * GR * 4;
  static constexpr int kStatSets = kPair ? 4 : 3;
  // pair exchange: [kWG] x ([4 warps][32] partial column values, [4][32]
  // each warp's copy of the update thresholds, [4][32] of the exponent
  // offsets, [4] each warp's lowest threshold)
  static constexpr int kOffRed = kOffStat + kStatSets * 2 * GR * 4;
  static constexpr int kRedWg = 3 * 128 + 4;  // floats per warpgroup (16-byte multiple)
  static constexpr int kRedBytes = kPair ? kWG * kRedWg * 4 : 0;
  static constexpr int kOffItem = kOffRed + kRedBytes;             // [2 slots] descriptors
  static constexpr int kOffBar = kOffItem + 2 * kItemBytes;
  static constexpr int kNumBars = 2 * (kStagesK + kStagesV) + 9 * kWG + 2 + 2 + 1 + 1 + 2 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 32 + 1024;
  static_assert(KR >= 16 && KR <= 128, "a head's rows sit within one warp, two or four");
  static_assert(kWph == 1 || kWph == 2 || kWph == 4, "warps per head");
  static_assert(kPair ? RH == 32 : (W == 8 || W == 16), "TMEM load width / one column per lane");
  static_assert(kN1 % 16 == 0 && kN2 % 16 == 0 && kN1 <= 256 && kN2 <= 256, "MMA N");
  static_assert(kTmemCols <= 512, "TMEM");
  static_assert(kBytes <= 232448, "shared memory");
  static_assert(44 + 8 * G <= kItemBytes, "unit descriptor");
  static_assert(kOffBar % 8 == 0, "mbarrier alignment");
  static_assert(16 * 128 * 4 <= kPBytes && GR % 16 == 0, "epilogue stage: 16 columns in a P buffer");
};

// Unit descriptor, written by the scheduler warp, read by every role.
template <int G>
struct Item {
  int valid, b, t_begin, TS, L, g0, n0, slot, nsp, shift;
  int u;  // unit index: its parity picks the warpgroup of the unit's first tile
  float vd[G], cs[G];  // v descale, logit scale (softmax_scale * qd * kd) per head
};

__device__ __forceinline__ void set_abort(volatile int* abort, int32_t* status) {
  *abort = 1;
  if (status) atomicExch(status, kStatusTimeout);
}

// The Q tile of a unit as e4m3 rows of `qbuf` in the 128-byte swizzled
// K-major layout: GR rows (row c = hq * RH + n: head g0 + hq, packed row
// n0 + n), for bf16 Q first the hi parts, then the lo parts (rows GR + c),
// of x = q 2^shift with the power of two shift putting the tile's largest
// |q| in [128, 256); returns shift (0 for e4m3 Q).  Run by kNT threads (ti =
// 0 .. kNT - 1); with more than one warp, `red` holds kNT / 32 floats of
// shared memory and `bar` names a barrier of exactly those threads.
template <class C, bool kQe4m3, int kNT>
__device__ __forceinline__ int convert_q_tile(const DecodeDev& a, uint8_t* qbuf, int b, int g0, int n0, int ti,
                                              float* red, int bar) {
  constexpr int GR = C::GR, RH = C::kRH;
  constexpr int kChunks = GR * 8 / kNT;  // 16-element chunks per thread
  static_assert(kChunks >= 1 && kChunks * kNT == GR * 8, "chunks");
  // one warp loads in two halves (registers); a larger group loads at once
  constexpr int kHalf = (kNT == 32 && kChunks >= 2) ? kChunks / 2 : kChunks;
  constexpr int kWords = kQe4m3 ? 1 : 2;  // 16-byte words per chunk
  const int lane = ti & 31;
  auto q_src = [&](int kc, bool& live) -> const uint4* {
    const int id = kc * kNT + ti;
    const int c = id >> 3, cc = id & 7;
    const int hq = c / RH, qrow = n0 + c % RH;
    live = qrow < a.n_q;
    const int64_t off =
        b * a.q_seq + (static_cast<int64_t>(g0 + hq) * a.n_q + (live ? qrow : 0)) * kHeadDimDev + cc * 16;
    return kQe4m3 ? reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) + off)
                  : reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + off);
  };
  int shift = 0;
  if (!kQe4m3) {
    // bf16 |q| max: integer max of the magnitude bits; the loads of a half
    // are all issued before any is used (one memory latency per half)
    uint32_t mbits = 0;
#pragma unroll
    for (int k0 = 0; k0 < kChunks; k0 += kHalf) {
      uint4 raw[kHalf][2];
#pragma unroll
      for (int u = 0; u < kHalf; ++u) {
        bool live;
        const uint4* src = q_src(k0 + u, live);
        raw[u][0] = live ? src[0] : make_uint4(0u, 0u, 0u, 0u);
        raw[u][1] = live ? src[1] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kHalf; ++u) {
        const uint32_t w8[8] = {raw[u][0].x, raw[u][0].y, raw[u][0].z, raw[u][0].w,
                                raw[u][1].x, raw[u][1].y, raw[u][1].z, raw[u][1].w};
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
          mbits = max(mbits, w8[wi] & 0x7FFFu);
          mbits = max(mbits, (w8[wi] >> 16) & 0x7FFFu);
        }
      }
    }
    float amax = __uint_as_float(mbits << 16);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if constexpr (kNT > 32) {
      if (lane == 0) red[ti >> 5] = amax;
      ptx::named_bar_sync(bar, kNT);
#pragma unroll
      for (int w = 0; w < kNT / 32; ++w) amax = fmaxf(amax, red[w]);
    }
    if (amax > 0.f) {
      const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;
      shift = 7 - e;  // max |q| 2^shift in [128, 256)
      shift = shift > 126 ? 126 : (shift < -126 ? -126 : shift);
    }
  }
  const float qscale = kQe4m3 ? 1.f : ldexpf(1.f, shift);
  if (kQe4m3 && GR < C::kN1) {
    for (int id = ti; id < (C::kN1 - GR) * 8; id += kNT)
      *reinterpret_cast<uint4*>(qbuf + GR * 128 + id * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  // the conversion pass reads the chunks again (from L1)
#pragma unroll 2
  for (int kc = 0; kc < kChunks; ++kc) {
    const int id = kc * kNT + ti;
    const int c = id >> 3, cc = id & 7;
    bool live;
    const uint4* src = q_src(kc, live);
    uint4 raw[kWords];
#pragma unroll
    for (int wd = 0; wd < kWords; ++wd) raw[wd] = live ? src[wd] : make_uint4(0u, 0u, 0u, 0u);
    float x[16];
    if (kQe4m3) {
      const uint32_t w4[4] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) e4m3x4_to_f32(w4[wi], x + wi * 4);
    } else {
      const uint32_t w8[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w,
                              raw[kWords - 1].x, raw[kWords - 1].y, raw[kWords - 1].z, raw[kWords - 1].w};
#pragma unroll
      for (int wi = 0; wi < 8; ++wi) {
        x[2 * wi] = __uint_as_float(w8[wi] << 16);
        x[2 * wi + 1] = __uint_as_float(w8[wi] & 0xFFFF0000u);
      }
    }
    uint32_t hwd[4], lwd[4];
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      uint16_t h01, h23, l01 = 0, l23 = 0;
      if (kQe4m3) {
        h01 = ptx::f32x2_to_e4m3x2(x[4 * wi], x[4 * wi + 1]);
        h23 = ptx::f32x2_to_e4m3x2(x[4 * wi + 2], x[4 * wi + 3]);
      } else {
        float xs[4], hf[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) xs[e] = x[4 * wi + e] * qscale;
        h01 = ptx::f32x2_to_e4m3x2(xs[0], xs[1]);
        h23 = ptx::f32x2_to_e4m3x2(xs[2], xs[3]);
        e4m3x4_to_f32(static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16), hf);
        l01 = ptx::f32x2_to_e4m3x2(xs[0] - hf[0], xs[1] - hf[1]);
        l23 = ptx::f32x2_to_e4m3x2(xs[2] - hf[2], xs[3] - hf[3]);
      }
      hwd[wi] = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
      lwd[wi] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
    }
    // 128-byte swizzle: chunk cc of row c at chunk position cc ^ (c % 8)
    *reinterpret_cast<uint4*>(qbuf + c * 128 + ((cc ^ (c & 7)) << 4)) = make_uint4(hwd[0], hwd[1], hwd[2], hwd[3]);
    if (!kQe4m3) {
      const int cl = GR + c;
      *reinterpret_cast<uint4*>(qbuf + cl * 128 + ((cc ^ (cl & 7)) << 4)) = make_uint4(lwd[0], lwd[1], lwd[2], lwd[3]);
    }
  }
  return shift;
}

// Named barriers: 1 + wg within a softmax warpgroup, kBarAll across both.
constexpr int kBarAll = 3;

template <int G, int RH, bool kQe4m3>
__global__ void __launch_bounds__(kThreads, 1)
decode_tcg_kernel(const DecodeDev a, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, int n_q_tiles, int num_units, int* sched) {
  // Launched as a programmatic dependent: no global load or store before
  // the grid ahead of this one has completed.  The merge (this grid's own
  // dependent) may launch now; its CTAs wait the same way.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  using C = GCfg<G, RH, kQe4m3>;
  using It = Item<G>;
  constexpr int KR = C::KR, GR = C::GR, SK = C::kStagesK, SV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(sm);
  float* corr_all = reinterpret_cast<float*>(sm + C::kOffCorr);
  float* stat_all = reinterpret_cast<float*>(sm + C::kOffStat);
  auto stat_of = [&](int w, int sl) -> float* {  // [GR] m, [GR] l of group w, unit slot sl
    return stat_all + (C::kPair ? w * 2 + sl : (w == 0 ? 0 : 1 + sl)) * 2 * GR;
  };
  float* red_all = reinterpret_cast<float*>(sm + C::kOffRed);    // pair exchange (G = 2)
  auto item = [&](int slot) -> It& { return *reinterpret_cast<It*>(sm + C::kOffItem + slot * kItemBytes); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffMisc + 4);

  // mbarriers: the K ring (full, empty), the V ring (full, empty); per
  // warpgroup S full x2, S free x2, P full, P free; unit slot full x2 /
  // empty x2; O free; MMA drain; unit descriptor full x2.
  const uint32_t bar0 = sbase + C::kOffBar;
  auto kfull = [&](int s) { return bar0 + 8u * s; };
  auto kempty = [&](int s) { return bar0 + 8u * (SK + s); };
  auto vfull = [&](int s) { return bar0 + 8u * (2 * SK + s); };
  auto vempty = [&](int s) { return bar0 + 8u * (2 * SK + SV + s); };
  constexpr int kB = 2 * (SK + SV);
  // k: 0, 1 S full; 2, 3 S free; 4, 5 P full (per P buffer); 6, 7 P free
  // (the GEMM2 that read the buffer is done); 8 O done (every GEMM2)
  auto wgbar = [&](int wg, int k) { return bar0 + 8u * (kB + 9 * wg + k); };
  auto pfull = [&](int wg, int pb) { return wgbar(wg, 4 + pb); };
  auto pfree = [&](int wg, int pb) { return wgbar(wg, 6 + pb); };
  auto ifull = [&](int slot) { return bar0 + 8u * (kB + 9 * kWG + slot); };
  auto iempty = [&](int slot) { return bar0 + 8u * (kB + 9 * kWG + 2 + slot); };
  const uint32_t ofree = bar0 + 8u * (kB + 9 * kWG + 4);
  const uint32_t drain = ofree + 8u;
  // the descriptor alone (the producer needs no Q): before the Q conversion
  auto dfull = [&](int slot) { return drain + 8u * (1 + slot); };
  // the first unit's Q tile converted (by the softmax warps)
  const uint32_t qcvt = drain + 8u * 3;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int groups = a.h_k / G;

  if (tid == 0) {
    for (int s = 0; s < SK; ++s) {
      ptx::mbar_init(kfull(s), 1);
      ptx::mbar_init(kempty(s), 1);
    }
    for (int s = 0; s < SV; ++s) {
      ptx::mbar_init(vfull(s), 1);
      ptx::mbar_init(vempty(s), 1);
    }
    for (int wg = 0; wg < kWG; ++wg) {
      ptx::mbar_init(wgbar(wg, 0), 1);
      ptx::mbar_init(wgbar(wg, 1), 1);
      ptx::mbar_init(wgbar(wg, 2), 4);
      ptx::mbar_init(wgbar(wg, 3), 4);
      ptx::mbar_init(pfull(wg, 0), 4);
      ptx::mbar_init(pfull(wg, 1), 4);
      ptx::mbar_init(pfree(wg, 0), 1);
      ptx::mbar_init(pfree(wg, 1), 1);
      ptx::mbar_init(wgbar(wg, 8), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(ifull(s), 1);
      ptx::mbar_init(dfull(s), 1);
      ptx::mbar_init(iempty(s), 2 + 4 * kWG);  // both MMA issuers, every softmax warp
    }
    ptx::mbar_init(ofree, 4 * kWG);
    ptx::mbar_init(drain, 2);
    ptx::mbar_init(qcvt, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  // P: every byte off the head diagonal stays zero for the whole kernel
  // (published to the tensor core by the fence before each P-full arrival)
  if (warp >= 2 && warp < kSchedWarp) {
    uint4* p = reinterpret_cast<uint4*>(sm + C::kOffP);
    for (int id = tid - 64; id < kWG * C::kPBytes / 16; id += 128 * kWG) p[id] = make_uint4(0u, 0u, 0u, 0u);
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + C::kOffMisc, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kSchedWarp) {
    // ----------------------------------------------------------- scheduler
    // Takes units from the shared counter (unit = work item x q tile x head
    // group, work item outermost, so the plan's longest-first order is the
    // order units are handed out), and fills a unit slot: descriptor, per-
    // head scales, and the Q tile as e4m3 (hi | lo rows for bf16 Q) in the
    // 128-byte swizzled K-major layout.
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      if (it >= 2) {
        const bool got = ptx::mbar_wait_bounded(iempty(slot), ((it >> 1) - 1) & 1, abort_flag, kWaitNs);
        if (__any_sync(0xffffffffu, !got)) {
          if (lane == 0) set_abort(abort_flag, a.status);
          break;
        }
      }
      int u = 0, b = 0, t_begin = 0, t_end = 0, wslot = 0, qt = 0, grp = 0;
      bool valid = false;
      for (bool first = it == 0;; first = false) {  // the next unit that is not padding
        // the first unit of CTA x is unit x; later ones come from the counter
        if (lane == 0) u = first ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(sched, 1);
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u >= num_units) break;
        grp = u % groups;
        const int rest = u / groups;
        qt = rest % n_q_tiles;
        const int4 wk = reinterpret_cast<const int4*>(a.work)[rest / n_q_tiles];
        b = wk.x;
        t_begin = wk.y;
        t_end = wk.z;
        wslot = wk.w;
        if (t_end > t_begin) {
          valid = true;
          break;
        }
      }
      It& I = item(slot);
      int L = 0;
      if (valid) {
        L = a.seq_lens[b];
        int key_stop = t_end * 128;
        key_stop = key_stop < L ? key_stop : L;
        const int TS = (key_stop - t_begin * 128 + KR - 1) / KR;
        if (lane == 0) {
          I.b = b;
          I.t_begin = t_begin;
          I.TS = TS < 1 ? 1 : TS;
          I.L = L;
          I.g0 = grp * G;
          I.n0 = qt * RH;
          I.slot = wslot;
          I.nsp = a.n_splits[b];
          I.u = u;
        }
      }
      if (lane == 0) I.valid = valid ? 1 : 0;
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(dfull(slot));  // the producer may start on the unit's tiles
      if (valid) {
        const int g0 = grp * G, n0 = qt * RH;
        if (lane < G) {
          const int g = g0 + lane;
          I.vd[lane] = a.vd[b * a.vd_seq + g * a.vd_head];
          I.cs[lane] = a.softmax_scale * a.qd[b * a.qd_seq + g * a.qd_head] * a.kd[b * a.kd_seq + g * a.kd_head];
        }
        if (it == 0 && C::kPair) {
          // G = 2: the first unit's Q tile (64 rows) is converted by the
          // softmax warps (idle until then, and eight times as many); the
          // 32-row instances measured slower with that code beside their
          // softmax (more register spills)
          const bool done = ptx::mbar_wait_bounded(qcvt, 0, abort_flag, kWaitNs);
          if (!done && lane == 0) set_abort(abort_flag, a.status);
        } else {
          const int shift =
              convert_q_tile<C, kQe4m3, 32>(a, sm + C::kOffQ + slot * C::kQBytes, b, g0, n0, lane, nullptr, 0);
          if (lane == 0) I.shift = shift;
        }
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ifull(slot));
      if (!valid) break;
    }
  } else if (warp == 0 || warp == kVLoadWarp) {
    // ----------------------------------------------------------- producers
    // Warp 0 loads the K tiles, warp 12 the V tiles, each as its ring's
    // stages free up (a K stage after its GEMM1, a V stage after its GEMM2):
    // two short loops, so that issuing never waits on the other tensor's
    // ring or on a busy issue slot shared with the softmax warps.
    //
    // Per tile: the rows of keys [k0, k0 + KR) of the G heads.  When a page
    // holds whole tiles (PS >= KR) that is one TMA box, all G heads of one
    // page (the per-SM rate of TMA operations, not bytes, bounds small
    // boxes); else box jb of head h on lane h * bph + jb.  Block-table
    // entries come from a register window (lane l holds block wbase + l)
    // refilled 32 blocks ahead.
    const bool is_k = warp == 0;
    const int NS = is_k ? SK : SV;
    const uint32_t ring = sbase + (is_k ? C::kOffK : C::kOffV);
    const CUtensorMap* tmap = is_k ? &tmap_k : &tmap_v;
    auto full = [&](int st) { return is_k ? kfull(st) : vfull(st); };
    auto empty = [&](int st) { return is_k ? kempty(st) : vempty(st); };
    const int PS = a.page_size;
    const int box_rows = KR < PS ? KR : PS;
    const int bph = KR / box_rows;  // boxes per head per tile
    const int h = lane / bph, jb = lane % bph;
    const bool active = lane < G * bph;
    const bool one_box = bph == 1 && box_rows == KR;
    if (lane == 0) ptx::prefetch_tmap(tmap);
    const bool evict_first = a.kv_evict_first != 0;
    const uint64_t kv_policy = ptx::policy_evict_first();
    uint32_t n = 0;  // tiles issued, over all units
    bool alive = true;
    for (int it = 0; alive; ++it) {
      const int slot = it & 1;
      const bool got = ptx::mbar_wait_bounded(dfull(slot), (it >> 1) & 1, abort_flag, kWaitNs);
      if (__any_sync(0xffffffffu, !got)) {
        if (lane == 0) set_abort(abort_flag, a.status);
        break;
      }
      const It& I = item(slot);
      if (!I.valid) break;
      const int L = I.L, TS = I.TS, g0 = I.g0;
      const int key_begin = I.t_begin * 128;
      const int64_t bt_row = static_cast<int64_t>(I.b) * a.max_blocks;
      int valid_pages = (L + PS - 1) / PS;
      valid_pages = valid_pages < a.max_blocks ? valid_pages : a.max_blocks;
      auto load_win = [&](int base) -> int {
        const int blk = base + lane;
        return blk < valid_pages ? a.block_table[bt_row + blk] : a.num_pages;
      };
      // A tile spans at most two blocks and starts on a block boundary when
      // it spans two (KR a multiple of PS); the window starts at the unit's
      // first block, so a tile never straddles two windows.
      int wbase = key_begin / PS;
      int win = load_win(wbase);
      int win_next = load_win(wbase + 32);
      for (int i = 0; i < TS; ++i, ++n) {
        const int st = n % NS;
        if (n >= static_cast<uint32_t>(NS)) {
          const bool freed = ptx::mbar_wait_bounded(empty(st), ((n / NS) - 1) & 1, abort_flag, kWaitNs);
          if (__any_sync(0xffffffffu, !freed)) {
            if (lane == 0) set_abort(abort_flag, a.status);
            alive = false;
            break;
          }
        }
        const int key0 = key_begin + i * KR;
        if (key0 / PS >= wbase + 32) {  // uniform over the warp
          wbase += 32;
          win = win_next;
          win_next = load_win(wbase + 32);
        }
        const int key = key0 + jb * box_rows;
        const int pg = __shfl_sync(0xffffffffu, win, (key / PS - wbase) & 31);
        const int page = (active && key < L) ? pg : a.num_pages;
        const int row_off = key % PS;
        const uint32_t dst = ring + st * kTileBytes;
        if (one_box) {
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(full(st), kTileBytes);
            ptx::tma_load_kv(dst, tmap, full(st), 0, row_off, g0, page, evict_first, kv_policy);
          }
        } else {
          if (lane == 0) ptx::mbar_arrive_expect_tx(full(st), kTileBytes);
          __syncwarp();
          if (active)
            ptx::tma_load_kv(dst + (h * KR + jb * box_rows) * 128, tmap, full(st), 0, row_off, g0 + h, page,
                             evict_first, kv_policy);
        }
      }
    }
    if (*abort_flag && lane == 0) {
      // drain: wait (bounded) for every tile still in flight to land
      volatile int never = 0;
      for (uint32_t i = (n > static_cast<uint32_t>(NS) ? n - NS : 0); i < n; ++i)
        ptx::mbar_wait_bounded(full(i % NS), (i / NS) & 1, &never, kWaitNs / 4);
    }
  } else if (warp == 1 || warp == kMma2Warp) {
    // ----------------------------------------------------------------- MMA
    // Tile number n counts tiles over all units (the rings' index).  Tile i
    // of unit u goes to warpgroup (i + u) & 1 — a function of the unit
    // alone, so the result does not depend on which CTA ran which units —
    // as that group's local tile t: GEMM1 (warp 1) into its S buffer
    // t % kSBufs, GEMM2 (warp 11) into its O.  Each issuer walks the
    // units in order with blocking waits; GEMM1 runs ahead as far as the S
    // buffers allow.  Shared-memory descriptors are a base plus the
    // operand's offset >> 4 (every offset stays inside the 14-bit field).
    if (lane == 0) {
      const bool gemm1 = warp == 1;
      bool ok = true;
      uint32_t n = 0;                // this issuer's tiles so far
      uint32_t tcount[2] = {0u, 0u};  // each group's tiles of the earlier units
      for (int it = 0; ok; ++it) {
        const int slot = it & 1;
        if (!ptx::mbar_wait_bounded(ifull(slot), (it >> 1) & 1, abort_flag, kWaitNs)) {
          ok = false;
          break;
        }
        const It& I = item(slot);
        if (!I.valid) break;
        const int TS = I.TS;
        const int f = I.u & 1;
        if (gemm1) {
          const uint32_t idesc_s = ptx::idesc_e4m3(kRows, C::kN1, false, false);
          const uint64_t kdesc0 = ptx::smem_desc(sbase + C::kOffK, 16, 1024, ptx::kSwizzle128B);
          const uint64_t qdesc = ptx::smem_desc(sbase + C::kOffQ + slot * C::kQBytes, 16, 1024, ptx::kSwizzle128B);
          for (int i = 0; i < TS; ++i, ++n) {
            const int st = n % SK;
            const int wg = (i + f) & 1;
            const int t = static_cast<int>(tcount[wg]) + (i >> 1), sb = t % C::kSBufs;
            if (!ptx::mbar_wait_bounded(kfull(st), (n / SK) & 1, abort_flag, kWaitNs) ||
                (t >= C::kSBufs &&
                 !ptx::mbar_wait_bounded(wgbar(wg, 2 + sb), ((t / C::kSBufs) - 1) & 1, abort_flag, kWaitNs))) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t kdesc = kdesc0 + static_cast<uint64_t>((st * kTileBytes) >> 4);
            const uint32_t d_s = tmem + wg * C::kWgCols + sb * C::kN1;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // one K step = 32 bytes of d
              ptx::mma_e4m3(d_s, kdesc + 2 * kk, qdesc + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
            ptx::mma_commit(wgbar(wg, sb));
            ptx::mma_commit(kempty(st));
          }
        } else {
          const uint32_t idesc_o = C::kPair ? ptx::idesc_e4m3(kRows, 2 * RH, true, true)
                                            : ptx::idesc_e4m3(kRows, C::kN2, true, true);
          const uint64_t vdesc0 = ptx::smem_desc(sbase + C::kOffV, 0, 1024, ptx::kSwizzle128B);
          const uint64_t pdesc0 = C::kPair ? ptx::smem_desc(sbase + C::kOffP, 128, KR * 16, ptx::kSwizzleNone)
                                           : ptx::smem_desc(sbase + C::kOffP, 128, 2048, ptx::kSwizzleNone);
          for (int i = 0; i < TS; ++i, ++n) {
            const int st = n % SV;
            const int wg = (i + f) & 1;
            const int t = static_cast<int>(tcount[wg]) + (i >> 1);
            const int pb = t % C::kPBufs;
            const bool first = i < 2;  // this group's first tile of the unit: O starts over
            if (!ptx::mbar_wait_bounded(pfull(wg, pb), (t / C::kPBufs) & 1, abort_flag, kWaitNs) ||
                !ptx::mbar_wait_bounded(vfull(st), (n / SV) & 1, abort_flag, kWaitNs) ||
                (first && it > 0 && !ptx::mbar_wait_bounded(ofree, (it - 1) & 1, abort_flag, kWaitNs))) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t vdesc = vdesc0 + static_cast<uint64_t>((st * kTileBytes) >> 4);
            const uint64_t pdesc =
                pdesc0 + static_cast<uint64_t>((wg * C::kPBytes + pb * C::kPBufBytes) >> 4);
            const uint32_t d_o = tmem + wg * C::kWgCols + C::kSBufs * C::kN1;
            if constexpr (C::kPair) {
              // per head: O[:, head h's hi | lo columns] += V_h^T P_h, K = KR keys
#pragma unroll
              for (int hh = 0; hh < G; ++hh) {
#pragma unroll
                for (int kk = 0; kk < KR / 32; ++kk)  // one K step = 32 keys (4096 B of V, 512 B of P)
                  ptx::mma_e4m3(d_o + hh * 2 * RH, vdesc + 256 * (hh * (KR / 32) + kk),
                                pdesc + ((hh * C::kPHeadBytes) >> 4) + 32 * kk, idesc_o,
                                (!first || kk > 0) ? 1u : 0u);
              }
            } else {
#pragma unroll
              for (int kk = 0; kk < kRows / 32; ++kk)  // one K step = 32 KV rows
                ptx::mma_e4m3(d_o, vdesc + 256 * kk, pdesc + 32 * kk, idesc_o, (!first || kk > 0) ? 1u : 0u);
            }
            ptx::mma_commit(pfree(wg, pb));
            if (C::kPair) ptx::mma_commit(wgbar(wg, 8));
            ptx::mma_commit(vempty(st));
          }
        }
        for (int w = 0; w < 2; ++w) tcount[w] += static_cast<uint32_t>(TS - ((w + f) & 1) + 1) >> 1;
        if (ok) ptx::mma_commit(iempty(slot));  // this unit's Q and slot are no longer read
      }
      if (!ok) set_abort(abort_flag, a.status);
      // every MMA of both issuers has completed once `drain` fires
      ptx::mma_commit(drain);
      volatile int never = 0;
      ptx::mbar_wait_bounded(drain, 0, &never, kWaitNs);
    }
  } else {
    // ------------------------------------------------ softmax warpgroups
    // A wait that gives up sets the abort flag and the work runs on (every
    // later wait returns at once), so that every warp meets the same named
    // barriers; nothing is written out after an abort.
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int st_tid = ((warp - 2) & 3) * 32 + lane;
    const int row = quarter * 32 + lane;  // TMEM lane: tile row (S) / d (O)
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int h = row / KR;               // this row's head within the group
    const int k = row % KR;               // ... and key within the tile
    const int h_first = (quarter * 32) / KR;  // first head of this warp
    const int hw = h - h_first;           // 0 .. HPW-1
    const int bar_wg = 1 + wg;
    const uint32_t tmem_s = tmem + wg * C::kWgCols;
    const uint32_t tmem_o = tmem_s + C::kSBufs * C::kN1;
    uint8_t* const pbuf_wg = sm + C::kOffP + wg * C::kPBytes;
    float* const corr_wg = corr_all + wg * 2 * GR;

    // ---- the first unit's Q tile, converted by both groups together
    if constexpr (C::kPair) {
      const int ti = tid - 64;
      const bool got = ptx::mbar_wait_bounded(dfull(0), 0, abort_flag, kWaitNs);
      const bool bad = ptx::named_bar_red_or(kBarAll, 128 * kWG, !got);
      It& I0 = item(0);
      if (!bad && I0.valid) {
        const int shift =
            convert_q_tile<C, kQe4m3, 128 * kWG>(a, sm + C::kOffQ, I0.b, I0.g0, I0.n0, ti, corr_all, kBarAll);
        if (ti == 0) I0.shift = shift;
      }
      if (bad && ti == 0) set_abort(abort_flag, a.status);
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(kBarAll, 128 * kWG);
      if (ti == 0) ptx::mbar_arrive(qcvt);
    }
    uint32_t n_base = 0;  // tiles of all earlier units
    uint32_t tb = 0;      // this group's tiles of all earlier units
    for (int it = 0;; ++it) {
      const int slot = it & 1;
      const bool got = ptx::mbar_wait_bounded(ifull(slot), (it >> 1) & 1, abort_flag, kWaitNs);
      // one decision for both groups: both take the same path through the
      // barriers below
      if (ptx::named_bar_red_or(kBarAll, 128 * kWG, !got)) {
        if (st_tid == 0) set_abort(abort_flag, a.status);
        break;
      }
      const It& I = item(slot);
      if (!I.valid) break;
      const int b = I.b, L = I.L, TS = I.TS, n0 = I.n0;
      const int key_begin = I.t_begin * 128;
      const float two_m_shift = ldexpf(1.f, -I.shift);
      const float c2 = I.cs[h] * two_m_shift * kLog2e;  // raw score -> log2 units, this row's head
      const int i0 = (wg + I.u) & 1;  // this group's first tile of the unit

      float* my_m = stat_of(wg, slot);
      float* my_l = my_m + GR;
      if constexpr (C::kPair) {
        // ---- G = 2: warps q and q ^ 1 hold one head's 64 keys.  Lane c
        // keeps column c's reference maximum m (raw units).  A tile updates
        // m only where its maximum passes m + kTau / c2 (kTau in log2 units),
        // so 448 p 2^-kTau stays within e4m3's range and most tiles need
        // neither the column reduction nor an O correction; the result does
        // not depend on m.  Each thread keeps its key's share of every row
        // sum, reduced once per unit.
        // this head's warps: lane quarters wq0 .. wq0 + kWph - 1, with their
        // own named barrier (the warpgroup's when a head fills it)
        const int wq0 = (quarter / C::kWph) * C::kWph;
        const bool head_lead = quarter == wq0;  // stores the head's stats
        const int bar_head = C::kWph == 4 ? bar_wg : 4 + 2 * wg + h;
        constexpr int kHeadThreads = 32 * C::kWph;
        float* const red = red_all + wg * C::kRedWg;    // [4 warps][32] partial values
        float* const thr = red + 128 + quarter * 32;   // this warp's copy: update thresholds (raw)
        float* const bias = red + 256 + quarter * 32;  // ... and exponent offsets (log2 units)
        float* const thr_min = red + 384 + quarter;    // ... and the lowest threshold
        const float head_c = C::kTau / c2;  // kTau in raw units of this head
        const int vis_all = a.causal ? L - a.q_len : L - 1;  // keys every column sees
        float m_lane = -INFINITY;
        float l_thr[RH];
#pragma unroll
        for (int nn = 0; nn < RH; ++nn) l_thr[nn] = 0.f;
        thr[lane] = -INFINITY;  // a fresh column: its first finite score updates it
        bias[lane] = C::kLog2PScale;
        if (lane == 0) *thr_min = -INFINITY;
        __syncwarp();
        bool ok = true;
        int t_last = -1;
        for (int i = i0; i < TS; i += 2) {
          const uint32_t n = n_base + i;
          const int t = static_cast<int>(tb) + (i >> 1);
          const int sb = t % C::kSBufs;
          const bool first = i < 2;
          const int j = key_begin + i * KR + k;  // this row's key
          t_last = t;
          if (!ptx::mbar_wait_bounded(wgbar(wg, sb), (t / C::kSBufs) & 1, abort_flag, kWaitNs)) ok = false;
          ptx::tc_fence_after();
          float sc[RH];
          {
            // this row's head's columns: hi, then lo (added)
            uint32_t r[RH];
            const uint32_t s_base = tmem_s + lane_off + sb * C::kN1 + h * RH;
            MJ_TMEM_LD16(s_base, r);
            MJ_TMEM_LD16(s_base + 16, (r + 16));
            ptx::tmem_ld_wait();
#pragma unroll
            for (int nn = 0; nn < RH; ++nn) sc[nn] = __uint_as_float(r[nn]);
            if (!kQe4m3) {
              MJ_TMEM_LD16(s_base + GR, r);
              MJ_TMEM_LD16(s_base + GR + 16, (r + 16));
              ptx::tmem_ld_wait();
#pragma unroll
              for (int nn = 0; nn < RH; ++nn) sc[nn] += __uint_as_float(r[nn]);
            }
          }
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(wgbar(wg, 2 + sb));
          if (j > vis_all) {  // select: keys past a column's limit, and garbage rows, never leak
#pragma unroll
            for (int nn = 0; nn < RH; ++nn) {
              const int qrow = n0 + nn;
              int lim = a.causal ? L - a.q_len + qrow / a.h_r : L - 1;
              lim = lim < L - 1 ? lim : L - 1;
              if (qrow >= a.n_q || j > lim) sc[nn] = -INFINITY;
            }
          }
          // may any score pass its column's threshold?  A conservative test
          // (this key's largest score against the warp's lowest threshold);
          // one barrier answers for the group, and the update below, uniform
          // over it, checks each column exactly.
          float smax = sc[0];
#pragma unroll
          for (int nn = 1; nn < RH; ++nn) smax = fmaxf(smax, sc[nn]);
          const bool any_ex = ptx::named_bar_red_or(bar_wg, 128, smax > *thr_min);
          bool any_moved = false;
          if (any_ex) {
            // column maxima over the head's 64 keys: reduce-scatter within
            // the warp (lane c ends with column c), then the partner's value
            float mx[RH];
#pragma unroll
            for (int nn = 0; nn < RH; ++nn) mx[nn] = sc[nn];
            warp_reduce_scatter<RH, true>(mx, lane);
            red[quarter * 32 + lane] = mx[0];
            ptx::named_bar_sync(bar_head, kHeadThreads);
            float tmax = mx[0];
#pragma unroll
            for (int q2 = 0; q2 < C::kWph; ++q2) tmax = fmaxf(tmax, red[(wq0 + q2) * 32 + lane]);
            const bool moved_c = tmax > thr[lane];
            const float mn = moved_c ? tmax : m_lane;
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            // the -inf guard: 0 for a column that had no finite score yet
            const float corr_c = moved_c ? fast_exp2((m_lane - mu) * c2) : 1.f;
            m_lane = mn;
            float* corr_b = corr_wg + (t & 1) * GR;
            if (head_lead) corr_b[h * RH + lane] = corr_c;
            // the partner has read red; corr_b is complete
            any_moved = ptx::named_bar_red_or(bar_wg, 128, moved_c);
            const float tn = (mn == -INFINITY) ? -INFINITY : mn + head_c;
            thr[lane] = tn;
            bias[lane] = fmaf(-mu, c2, C::kLog2PScale);
            float tlo = tn;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) tlo = fminf(tlo, __shfl_xor_sync(0xffffffffu, tlo, off));
            if (lane == 0) *thr_min = tlo;
            const float4* cb4 = reinterpret_cast<const float4*>(corr_b + h * RH);
#pragma unroll
            for (int q4 = 0; q4 < RH / 4; ++q4) {
              const float4 f = cb4[q4];
              l_thr[4 * q4] *= f.x;
              l_thr[4 * q4 + 1] *= f.y;
              l_thr[4 * q4 + 2] *= f.z;
              l_thr[4 * q4 + 3] *= f.w;
            }
            __syncwarp();
          }
          // P buffer t & 1 is free once the GEMM2 of tile t - 2 is done
          const int pb = t & 1;
          if (t >= 2 && !ptx::mbar_wait_bounded(pfree(wg, pb), ((t >> 1) - 1) & 1, abort_flag, kWaitNs)) ok = false;
          // lazy O correction (uniform over the group: TMEM access is warp-wide),
          // after the GEMM2 of tile t - 1 (t - 2's is done: the parity names it)
          if (any_moved && !first) {
            if (!ptx::mbar_wait_bounded(wgbar(wg, 8), (t - 1) & 1, abort_flag, kWaitNs)) ok = false;
            const float* corr_b = corr_wg + (t & 1) * GR;
            ptx::tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < C::kN2; c0 += 16) {
              // O columns of head c0 / (2 RH): hi | lo halves of RH each
              const int cb = (c0 / (2 * RH)) * RH + c0 % RH;
              uint32_t r[16];
              MJ_TMEM_LD16(tmem_o + lane_off + c0, r);
              ptx::tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr_b[cb + e]);
              MJ_TMEM_ST16(tmem_o + lane_off + c0, r);
            }
            ptx::tmem_st_wait();
          }
          // x = 448 p 2^-kTau, its row-sum shares, and the e4m3 split
          {
            const float4* b4 = reinterpret_cast<const float4*>(bias);
#pragma unroll
            for (int q4 = 0; q4 < RH / 4; ++q4) {
              const float4 bv = b4[q4];
              const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float x = fast_exp2(fmaf(sc[4 * q4 + e], c2, bb[e]));
                l_thr[4 * q4 + e] += x;
                sc[4 * q4 + e] = x;
              }
            }
          }
          {
            uint32_t hi[RH / 4], lo[RH / 4];
            split_e4m3_hilo<RH, C::kLoShift>(sc, hi, lo);
            // this head's P: [hi groups 0, 1 | lo groups 2, 3][KR keys][16 B]
            uint8_t* prow = pbuf_wg + pb * C::kPBufBytes + h * C::kPHeadBytes + k * 16;
            constexpr int kGS = KR * 16;  // bytes between 16-column groups
            *reinterpret_cast<uint4*>(prow) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(prow + kGS) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
            *reinterpret_cast<uint4*>(prow + 2 * kGS) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            *reinterpret_cast<uint4*>(prow + 3 * kGS) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
          }
          // rows past the sequence end: zero their V row (0 * poison must not
          // reach O; the TMA landed whole pages)
          if (key_begin + (i + 1) * KR > L) {
            const int st = n % SV;
            if (!ptx::mbar_wait_bounded(vfull(st), (n / SV) & 1, abort_flag, kWaitNs)) ok = false;
            if (j >= L) {
              uint4* vrow = reinterpret_cast<uint4*>(sm + C::kOffV + st * kTileBytes + row * 128);
#pragma unroll
              for (int e = 0; e < 8; ++e) vrow[e] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
          ptx::fence_proxy_async_smem();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(pfull(wg, pb));
          if (!ok) set_abort(abort_flag, a.status);
        }
        n_base += TS;
        tb += static_cast<uint32_t>(TS - i0 + 1) >> 1;
        // ---- end of the unit: this group's O is final once its last two
        // GEMM2s are done (each P buffer's barrier names its own)
        if (t_last >= 1 &&
            !ptx::mbar_wait_bounded(pfree(wg, (t_last - 1) & 1), ((t_last - 1) >> 1) & 1, abort_flag, kWaitNs))
          ok = false;
        if (t_last >= 0 && !ptx::mbar_wait_bounded(pfree(wg, t_last & 1), (t_last >> 1) & 1, abort_flag, kWaitNs))
          ok = false;
        if (!ok) set_abort(abort_flag, a.status);
        // row sums over the pair's 64 keys; the even warp stores the head's stats
        warp_reduce_scatter<RH, false>(l_thr, lane);
        red[quarter * 32 + lane] = l_thr[0];
        ptx::named_bar_sync(bar_head, kHeadThreads);
        if (head_lead) {
          float lsum = 0.f;  // in warp order
#pragma unroll
          for (int q2 = 0; q2 < C::kWph; ++q2) lsum += red[(wq0 + q2) * 32 + lane];
          my_m[h * RH + lane] = m_lane;
          my_l[h * RH + lane] = lsum * C::kPScaleInv;
        }
      } else {
      // deferred row sums (of 448 p 2^-kTau); reference column maxima (raw)
      // and the scores that would move them
      float l_thr[RH], m_cur[RH], thr[RH];
      const float head_c = C::kTau / c2;
      int lim[RH];                 // last visible key of column n of this row's head (-1: none)
#pragma unroll
      for (int nn = 0; nn < RH; ++nn) {
        l_thr[nn] = 0.f;
        m_cur[nn] = -INFINITY;
        thr[nn] = -INFINITY;  // a fresh column: its first finite score moves it
        const int qrow = n0 + nn;
        int l = a.causal ? L - a.q_len + qrow / a.h_r : L - 1;
        l = l < L - 1 ? l : L - 1;
        lim[nn] = qrow < a.n_q ? l : -1;
      }

      bool ok = true;
      int t_last = -1;  // this group's last local tile of the unit
      for (int i = i0; i < TS; i += 2) {
        const uint32_t n = n_base + i;
        const int t = static_cast<int>(tb) + (i >> 1);
        const int sb = t & 1;
        const bool first = i < 2;
        const int j = key_begin + i * KR + k;  // this row's key
        t_last = t;
        if (!ptx::mbar_wait_bounded(wgbar(wg, sb), (t >> 1) & 1, abort_flag, kWaitNs)) ok = false;
        ptx::tc_fence_after();
        float sc[RH];
        {
          // this warp's heads' columns (hi and lo parts), then this row's head
          uint32_t rh[C::W], rl[C::W];
          const uint32_t s_base = tmem_s + lane_off + sb * C::kN1 + h_first * RH;
          if constexpr (C::W == 8) {
            MJ_TMEM_LD8(s_base, rh);
            if (!kQe4m3) MJ_TMEM_LD8(s_base + GR, rl);
          } else {
            MJ_TMEM_LD16(s_base, rh);
            if (!kQe4m3) MJ_TMEM_LD16(s_base + GR, rl);
          }
          ptx::tmem_ld_wait();
#pragma unroll
          for (int nn = 0; nn < RH; ++nn) {
            float v = __uint_as_float(rh[nn]);
            if (!kQe4m3) v += __uint_as_float(rl[nn]);
            if (C::HPW == 2) {
              float v1 = __uint_as_float(rh[RH + nn]);
              if (!kQe4m3) v1 += __uint_as_float(rl[RH + nn]);
              v = hw ? v1 : v;
            }
            sc[nn] = (j <= lim[nn]) ? v : -INFINITY;  // select: garbage rows never leak
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(wgbar(wg, 2 + sb));

        // A column's reference maximum m moves only where a score passes
        // m + kTau / c2 (so 448 p 2^-kTau stays within e4m3's range): one
        // barrier tells the group whether any score does; only then are the
        // column maxima reduced (shuffles within the head's KR lanes).
        bool ex = false;
#pragma unroll
        for (int nn = 0; nn < RH; ++nn) ex |= sc[nn] > thr[nn];
        bool any_moved = false;
        if (ptx::named_bar_red_or(bar_wg, 128, ex)) {
          bool moved = false;
          float corr[RH];
#pragma unroll
          for (int nn = 0; nn < RH; ++nn) {
            float v = sc[nn];
#pragma unroll
            for (int off = KR / 2; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
            const bool mv = v > thr[nn];
            const float mn = mv ? v : m_cur[nn];
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            corr[nn] = mv ? fast_exp2((m_cur[nn] - mu) * c2) : 1.f;  // the -inf guard: 0 for a fresh column
            moved |= mv;
            m_cur[nn] = mn;
            thr[nn] = (mn == -INFINITY) ? -INFINITY : mn + head_c;
          }
          float* corr_b = corr_wg + sb * GR;
          if (k == 0) {
#pragma unroll
            for (int nn = 0; nn < RH; ++nn) corr_b[h * RH + nn] = corr[nn];
          }
          any_moved = ptx::named_bar_red_or(bar_wg, 128, moved);
          if (moved) {
#pragma unroll
            for (int nn = 0; nn < RH; ++nn) l_thr[nn] *= corr[nn];
          }
        }
        // This group's P buffer and O are free once the GEMM2 of its previous
        // tile finished (the one before that was waited for a tile ago, so
        // the parity names that GEMM2 alone).
        if (t > 0 && !ptx::mbar_wait_bounded(pfree(wg, 0), (t - 1) & 1, abort_flag, kWaitNs)) ok = false;
        // lazy O correction: O's TMEM lanes are head-dimension rows spanning
        // every head's columns, so any moved maximum corrects all of them
        // (the condition is uniform over the group: TMEM access is warp-wide)
        if (any_moved && !first) {
          const float* corr_b = corr_wg + sb * GR;
          ptx::tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < C::kN2; c0 += 16) {
            uint32_t r[16];
            MJ_TMEM_LD16(tmem_o + lane_off + c0, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr_b[(c0 + e) % GR]);
            MJ_TMEM_ST16(tmem_o + lane_off + c0, r);
          }
          ptx::tmem_st_wait();
        }
        // x = 448 p 2^-kTau and the row sums
#pragma unroll
        for (int nn = 0; nn < RH; ++nn) {
          const float mu = (m_cur[nn] == -INFINITY) ? 0.f : m_cur[nn];
          const float p = fast_exp2(fmaf(sc[nn], c2, fmaf(-mu, c2, C::kLog2PScale)));
          l_thr[nn] += p;
          sc[nn] = p;
        }
        {
          uint32_t hi[RH / 4], lo[RH / 4];
          split_e4m3_hilo<RH, C::kLoShift>(sc, hi, lo);
          uint8_t* prow = pbuf_wg + row * 16;
          const int ch = h * RH, cl = GR + h * RH;  // this row's hi / lo columns
          uint8_t* ph = prow + (ch / 16) * (kRows * 16) + (ch % 16);
          uint8_t* pl = prow + (cl / 16) * (kRows * 16) + (cl % 16);
          if constexpr (RH == 4) {
            *reinterpret_cast<uint32_t*>(ph) = hi[0];
            *reinterpret_cast<uint32_t*>(pl) = lo[0];
          } else {
            *reinterpret_cast<uint2*>(ph) = make_uint2(hi[0], hi[1]);
            *reinterpret_cast<uint2*>(pl) = make_uint2(lo[0], lo[1]);
          }
        }
        // rows past the sequence end: zero their V row (0 * poison must not
        // reach O; the TMA landed whole pages)
        if (key_begin + (i + 1) * KR > L) {
          const int st = n % SV;
          if (!ptx::mbar_wait_bounded(vfull(st), (n / SV) & 1, abort_flag, kWaitNs)) ok = false;
          if (j >= L) {
            uint4* vrow = reinterpret_cast<uint4*>(sm + C::kOffV + st * kTileBytes + row * 128);
#pragma unroll
            for (int e = 0; e < 8; ++e) vrow[e] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(pfull(wg, 0));
        if (!ok) set_abort(abort_flag, a.status);
      }
      n_base += TS;
      tb += static_cast<uint32_t>(TS - i0 + 1) >> 1;

      // ---- end of the unit: this group's O is final once its last GEMM2 is
      if (t_last >= 0 && !ptx::mbar_wait_bounded(pfree(wg, 0), t_last & 1, abort_flag, kWaitNs)) ok = false;
      if (!ok) set_abort(abort_flag, a.status);
      // row sums of this head: shuffles within its KR lanes
#pragma unroll
      for (int nn = 0; nn < RH; ++nn) {
        float v = l_thr[nn];
#pragma unroll
        for (int off = KR / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        l_thr[nn] = v;
      }
      if (k == 0) {
#pragma unroll
        for (int nn = 0; nn < RH; ++nn) {
          my_m[h * RH + nn] = m_cur[nn];
          my_l[h * RH + nn] = l_thr[nn] * C::kPScaleInv;
        }
      }
      }
      const bool fine = !ptx::named_bar_red_or(kBarAll, 128 * kWG, *abort_flag != 0);
      // ---- both groups: merge of their states and the output, group w
      // taking the 16-column blocks 16 w, 16 w + 32, ...  Per column: the
      // common maximum and each group's weight, folded with scale_o / l for
      // a final output (in this group's correction area).
      const bool final_out = I.nsp <= 1;
      float* w0_s = corr_wg;
      float* w1_s = corr_wg + GR;
      const int ce = st_tid;  // the column this thread merges, if its block is this group's
      const bool mine = ce < GR && ((ce >> 4) & 1) == wg;
      float mx = -INFINITY, lsum = 0.f;
      if (fine && mine) {
        const int hq = ce / RH;
        const float c2c = I.cs[hq] * two_m_shift * kLog2e;
        const float* s0 = stat_of(0, slot);
        const float* s1 = stat_of(1, slot);
        const float m0 = s0[ce], m1 = s1[ce];
        mx = fmaxf(m0, m1);
        const float f0 = (m0 == -INFINITY) ? 0.f : fast_exp2((m0 - mx) * c2c);
        const float f1 = (m1 == -INFINITY) ? 0.f : fast_exp2((m1 - mx) * c2c);
        lsum = s0[GR + ce] * f0 + s1[GR + ce] * f1;
        const float sc = final_out ? a.scale_o / (lsum + 1e-30f) : 1.f;
        w0_s[ce] = f0 * sc;
        w1_s[ce] = f1 * sc;
      }
      ptx::named_bar_sync(bar_wg, 128);
      if (fine) {
        ptx::tc_fence_after();
        const int d = row;  // TMEM lane of O = head-dimension index
        const uint32_t o0 = tmem + C::kSBufs * C::kN1;               // group 0's O
        const uint32_t o1 = tmem + C::kWgCols + C::kSBufs * C::kN1;  // group 1's O, same lanes
        // Sixteen columns at a time: O = w0 O_0 + w1 O_1 (hi + lo parts of
        // each; select, not multiply: a group with no tile left its O stale)
        // is staged column-major in this group's P buffer (idle now: its
        // last GEMM2 is done), then written out as whole rows with 16-byte
        // stores — one store per column and thread would take microseconds
        // while the KV stream saturates the memory system.
        float* stage = reinterpret_cast<float*>(pbuf_wg);
#pragma unroll 1
        for (int c0 = 16 * wg; c0 < GR; c0 += 32) {
          // TMEM columns of the hi and lo parts of output columns c0 .. c0 + 15
          const int ohi = C::kPair ? (c0 / RH) * 2 * RH + c0 % RH : c0;
          const int olo = C::kPair ? ohi + RH : GR + c0;
          float ov[16];
          {
            uint32_t rh[16], rl[16];
            MJ_TMEM_LD16(o0 + lane_off + ohi, rh);
            MJ_TMEM_LD16(o0 + lane_off + olo, rl);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float w0 = w0_s[c0 + e];
              ov[e] = w0 > 0.f ? (__uint_as_float(rh[e]) + __uint_as_float(rl[e]) * C::kLoInv) * w0 : 0.f;
            }
          }
          {
            uint32_t qh[16], ql[16];
            MJ_TMEM_LD16(o1 + lane_off + ohi, qh);
            MJ_TMEM_LD16(o1 + lane_off + olo, ql);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float w1 = w1_s[c0 + e];
              if (w1 > 0.f) ov[e] += (__uint_as_float(qh[e]) + __uint_as_float(ql[e]) * C::kLoInv) * w1;
            }
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) stage[e * kHeadDimDev + d] = ov[e];
          ptx::named_bar_sync(bar_wg, 128);
          // 16 rows x 32 four-float pieces
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int q = st_tid + 128 * r;
            const int e = q >> 5, d4 = (q & 31) * 4;
            const int c = c0 + e;
            const int hq = c / RH, qrow = n0 + c % RH;
            if (qrow < a.n_q) {
              float4 v = *reinterpret_cast<const float4*>(stage + e * kHeadDimDev + d4);
              const int g = I.g0 + hq;
              const float f = I.vd[hq] * C::kPScaleInv;
              v.x *= f;
              v.y *= f;
              v.z *= f;
              v.w *= f;
              if (final_out) {
                const __nv_bfloat162 lo2 = __floats2bfloat162_rn(v.x, v.y);
                const __nv_bfloat162 hi2 = __floats2bfloat162_rn(v.z, v.w);
                uint2 packed;
                packed.x = *reinterpret_cast<const uint32_t*>(&lo2);
                packed.y = *reinterpret_cast<const uint32_t*>(&hi2);
                const int64_t orow = b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + qrow) * kHeadDimDev;
                *reinterpret_cast<uint2*>(a.o + orow + d4) = packed;
              } else {
                const int64_t pr = part_row(a, b, g, I.slot, qrow);
                *reinterpret_cast<float4*>(a.o_part + pr * kHeadDimDev + d4) = v;
              }
            }
          }
          ptx::named_bar_sync(bar_wg, 128);  // the next block reuses the stage
        }
        // the P buffer's off-diagonal zeros again (published by the fence
        // before this group's next P-full arrival); G = 2 has none: every
        // tile rewrites its buffer whole
        if (!C::kPair)
          for (int id = st_tid; id < C::kPBytes / 16; id += 128)
            reinterpret_cast<uint4*>(pbuf_wg)[id] = make_uint4(0u, 0u, 0u, 0u);
        if (mine) {
          const int c = ce, hq = c / RH, nn = c % RH;
          const int qrow = n0 + nn, g = I.g0 + hq;
          if (qrow < a.n_q) {
            const float m_logit = mx * I.cs[hq] * two_m_shift;
            if (final_out) {
              a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + qrow] = m_logit + logf(lsum);
            } else {
              const int64_t pr = part_row(a, b, g, I.slot, qrow);
              a.m_part[pr] = m_logit;
              a.l_part[pr] = lsum;
            }
          }
        }
      }
      // both O accumulators and this slot are free again
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ptx::mbar_arrive(ofree);
        ptx::mbar_arrive(iempty(slot));
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::kTmemCols);
}

template <int G, int RH, bool kQe4m3>
cudaError_t launch_tcg(const DecodeDev& a, int n_q_tiles, int* sched, int sm_count, cudaStream_t stream) {
  using C = GCfg<G, RH, kQe4m3>;
  // the same box choice as the producer: all G heads at once when a page
  // holds whole tiles
  const int box_rows = C::KR < a.page_size ? C::KR : a.page_size;
  const int box_heads = box_rows == C::KR ? G : 1;
  CUtensorMap mk, mv;
  if (a.kv_format != 0) return cudaErrorInvalidValue;  // e4m3 pools only (validated before)
  if (!make_kv_map(&mk, a.k, a.page_size, a.h_k, a.num_pages, a.k_row, a.k_head, a.k_page, box_rows, box_heads, 0) ||
      !make_kv_map(&mv, a.v, a.page_size, a.h_k, a.num_pages, a.v_row, a.v_head, a.v_page, box_rows, box_heads, 0))
    return cudaErrorInvalidValue;
  auto kern = decode_tcg_kernel<G, RH, kQe4m3>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
  if (e != cudaSuccess) return e;
  const int num_units = a.num_work * n_q_tiles * (a.h_k / G);
  e = cudaMemsetAsync(sched, 0, sizeof(int), stream);
  if (e != cudaSuccess) return e;
  const int grid = num_units < sm_count ? num_units : sm_count;
  return launch_pdl(kern, dim3(grid, 1, 1), dim3(kThreads, 1, 1), C::kBytes, stream, a, mk, mv, n_q_tiles,
                    num_units, sched);
}

}  // namespace

bool tcg_supported(int h_k, int n_q, int* heads_per_cta, int* rows_per_head) {
  // G heads x RH rows per head: G = 8 x 4 and G = 4 x 8 (a head's keys
  // within one warp), G = 2 x 32 (a head's keys in a warp pair), G = 1 x 32
  // (one head's keys over the four warps of a group)
  int g = 0, rh = 0;
  if (n_q <= 4 && h_k % 8 == 0) {
    g = 8;
    rh = 4;
  } else if (n_q <= 8 && h_k % 4 == 0) {
    g = 4;
    rh = 8;
  } else if (n_q <= 32 && h_k % 2 == 0) {
    g = 2;
    rh = 32;
  } else if (n_q <= 32) {
    g = 1;
    rh = 32;
  }
  if (g == 0) return false;
  *heads_per_cta = g;
  *rows_per_head = rh;
  return true;
}

cudaError_t launch_decode_tcg(const DecodeDev& a, int heads_per_cta, int rows_per_head, int n_q_tiles, bool q_e4m3,
                              int* sched, int sm_count, cudaStream_t stream) {
  if (heads_per_cta == 8 && rows_per_head == 4)
    return q_e4m3 ? launch_tcg<8, 4, true>(a, n_q_tiles, sched, sm_count, stream)
                  : launch_tcg<8, 4, false>(a, n_q_tiles, sched, sm_count, stream);
  if (heads_per_cta == 4 && rows_per_head == 8)
    return q_e4m3 ? launch_tcg<4, 8, true>(a, n_q_tiles, sched, sm_count, stream)
                  : launch_tcg<4, 8, false>(a, n_q_tiles, sched, sm_count, stream);
  if (heads_per_cta == 2 && rows_per_head == 32)
    return q_e4m3 ? launch_tcg<2, 32, true>(a, n_q_tiles, sched, sm_count, stream)
                  : launch_tcg<2, 32, false>(a, n_q_tiles, sched, sm_count, stream);
  if (heads_per_cta == 1 && rows_per_head == 32)
    return q_e4m3 ? launch_tcg<1, 32, true>(a, n_q_tiles, sched, sm_count, stream)
                  : launch_tcg<1, 32, false>(a, n_q_tiles, sched, sm_count, stream);
  return cudaErrorInvalidValue;
}

int tcg_smem_bytes(int heads_per_cta, int rows_per_head, bool q_e4m3) {
  if (heads_per_cta == 8 && rows_per_head == 4) return q_e4m3 ? GCfg<8, 4, true>::kBytes : GCfg<8, 4, false>::kBytes;
  if (heads_per_cta == 4 && rows_per_head == 8) return q_e4m3 ? GCfg<4, 8, true>::kBytes : GCfg<4, 8, false>::kBytes;
  if (heads_per_cta == 2 && rows_per_head == 32)
    return q_e4m3 ? GCfg<2, 32, true>::kBytes : GCfg<2, 32, false>::kBytes;
  if (heads_per_cta == 1 && rows_per_head == 32)
    return q_e4m3 ? GCfg<1, 32, true>::kBytes : GCfg<1, 32, false>::kBytes;
  return 0;
}

}  // namespace mj
