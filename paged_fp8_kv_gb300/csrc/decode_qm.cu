// Split-KV paged decode attention on the tensor cores (tcgen05,
// kind::f8f6f4) for many packed query rows: query rows on the MMA's M.
//
// Sources: the "mjolnir/t5_decode.py" page — `decode` kernel (paged TMA
// gather with out-of-range pages read as zeros, masking by select, online
// softmax with the descales folded into the exponent and the -inf guard,
// lazy O rescale, final-vs-partial epilogue, P stored as e4m3(p * 448)).
// The swap-AB orientation of the pull request page (KV slots on M) pays off
// while the live rows are few; past 32 rows it would run one CTA per 32 rows
// and read the KV once per CTA.  Here one CTA takes 128 packed rows of one
// kv head (a q tile) and reads each KV tile once for all of them:
//   S[row, key] = Q[row] . K[key]         A = Q (K-major), B = K tile (K-major)
//   O[row, d]  += P[row, key] V[key, d]    A = P (K-major), B = V tile (MN-major)
// with 128 keys per tile.  A TMEM lane is a query row for S and for O, so
// each softmax thread owns one row: its maximum and sum are thread-local and
// its O rescale touches only its own TMEM lane.
//
// As in the swap-AB kernel, nothing is dequantised: the e4m3 K / V tiles the
// TMA lands are the operands; bf16 Q is split into hi + lo e4m3 parts
// (q 2^s = hi + lo) and P into hi + lo (448 p = hi + lo), each part an A
// operand of its own MMA into the same accumulator.
//
// Row copies (17-64 packed rows): each packed row is held 4 (2) times on
// GEMM1's M, every copy taking a quarter (half) of a tile's keys; the
// copies share the row's reference maximum and write one P row between
// them, and GEMM2 runs as O^T[d, row] += V^T[d, key] P^T[key, row] with the
// packed rows on N (A = V tile MN-major, B = P rows K-major), a quarter
// (half) of the MMA work of a 128-row O.
//
// Roles (384 threads): warps 0 and 11 issue the K and V TMA tiles into two
// rings (a K stage is freed by its GEMM1, a V stage by its GEMM2); warp 1
// (TMEM allocator) issues GEMM1 and warp 10 GEMM2 (one thread issues a
// tcgen05.mma only every 70-100 cycles); warps 2-5 and 6-9 are two softmax
// warpgroups taking alternate tiles, thread = query row, each group with its
// own S and O (128 TMEM columns each), merged per row at the end.
//
// Paired q tiles (more than 128 packed rows): one CTA takes two q tiles of
// the same kv head, warpgroup w the 128 rows of q tile w, and each KV tile
// goes to both warpgroups (a GEMM1 and a GEMM2 per group), so the KV is read
// once for 256 rows; each group writes its own rows at the end.

#include <cuda.h>
#include <cuda_runtime.h>

#include "mj_device.cuh"
#include "mj_kernels.h"
#include "sm100_ptx.cuh"

namespace mj {
namespace {

constexpr int kRows = 128;                   // query rows per CTA = MMA M; keys per tile = MMA N
constexpr int kTileBytes = kRows * 128;      // one K or V tile (128 keys x d): 16 KB
constexpr int kPartBytes = kRows * 128;      // one e4m3 operand of 128 rows x 128 bytes
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: far above any legal wait
constexpr int kStatusTimeout = 5;            // MJ_ERR_TIMEOUT
// P is produced as x = 448 p 2^-kTau: a row's reference maximum m moves only
// when the tile's maximum passes m + kTau (log2 units), so x stays within
// e4m3's range and most tiles need no O correction; the result does not
// depend on m.
constexpr int kTau = 4;
constexpr float kLog2PScale = 8.807354922057604f - kTau;  // log2(448 2^-kTau)
constexpr float kPScaleInv = (1.f / 448.f) * (1 << kTau);
constexpr int kWG = 2;                       // softmax warpgroups, alternate tiles
constexpr int kThreads = 64 + 128 * kWG + 64;
constexpr int kMma2Warp = 2 + 4 * kWG;       // 10
constexpr int kVLoadWarp = kMma2Warp + 1;    // 11
constexpr int kBarAll = 3;                   // named barrier of both warpgroups

template <bool kQe4m3, bool kPair = false, int kDup = 1>
struct QmCfg {
  // K ring: measured the bound at three stages (a stage comes back one TMA
  // round trip after its GEMM1, and the period was that over three); the
  // shared memory left beside Q and the P buffers takes one more (two with
  // e4m3 Q, which has no lo part)
  // Paired q tiles hold two Q tiles: three K and three V stages beside a
  // bf16 pair's 64 KB of Q parts (a stage then serves twice the work).
  // Row copies keep two P buffers per group; with 64 rows (two copies) those
  // fill the group's P region, so the copies' maxima and factors get a small
  // region of their own and the K ring one stage fewer (a build with one K
  // and one V stage fewer measured within 2 % on every workload).
  static constexpr int kStagesK = kPair ? (kQe4m3 ? 4 : 3) : (kQe4m3 ? 5 : 4) - (kDup == 2 ? 1 : 0);
  static constexpr int kStagesV = kPair ? (kQe4m3 ? 4 : 3) : 4;
  static constexpr int kQParts = kQe4m3 ? 1 : 2;
  static constexpr int kQTiles = kPair ? 2 : 1;
  static constexpr int kTmemCols = 512;  // per warpgroup: S (128), O (128)
  static constexpr int kWgCols = 256;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kStagesK * kTileBytes;
  static constexpr int kOffQ = (kStagesK + kStagesV) * kTileBytes;  // [q tile][hi | lo] 128 x 128 B each
  static constexpr int kOffP = kOffQ + kQTiles * kQParts * kPartBytes;  // [wg][hi | lo]
  static constexpr int kOffX = kOffP + kWG * 2 * kPartBytes;         // 64 rows: [wg] copies' maxima, factors
  static constexpr int kXBytes = kDup == 2 ? kWG * 1024 : 0;
  static constexpr int kOffStat = kOffX + kXBytes;                   // group 1: [128] max, [128] sum
  static constexpr int kOffBar = kOffStat + 2 * kRows * 4;
  static constexpr int kNumBars = 2 * (kStagesK + kStagesV) + 6 * kWG + 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kBytes = kOffMisc + 64 + 1024;
  static_assert(kBytes <= 232448, "shared memory");
};

__device__ __forceinline__ void set_abort(volatile int* abort, int32_t* status) {
  *abort = 1;
  if (status) atomicExch(status, kStatusTimeout);
}

// 128-byte-swizzled K-major row of an e4m3 operand: 16-byte chunk cc of
// row r sits at chunk position cc ^ (r % 8).
__device__ __forceinline__ uint8_t* swz(uint8_t* part, int r, int cc) {
  return part + r * 128 + ((cc ^ (r & 7)) << 4);
}

// kDup > 1: a q tile has kR = 128 / kDup packed rows, each held kDup times
// in GEMM1's M rows (row r is packed row r % kR); copy s of a row takes keys
// [s kR, (s + 1) kR) of every tile, so every softmax warp has work and each
// covers 1 / kDup of the keys.  The copies of a row share its reference
// maximum, write their key slices into one P row per packed row, and GEMM2
// runs as O^T = V^T P^T with the kR packed rows on N.
template <bool kQe4m3, int kDup, bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
decode_qm_kernel(const DecodeDev a, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v, int n_q_tiles) {
  static_assert(!kPair || kDup == 1, "paired q tiles: one copy of each row");
  constexpr int kR = kRows / kDup;   // packed rows per q tile; also keys per copy
  constexpr int kCh = kR < 64 ? kR : 64;  // S columns per TMEM round trip
  // Launched as a programmatic dependent: no global load or store before
  // the grid ahead of this one has completed.  The merge (this grid's own
  // dependent) may launch now; its CTAs wait the same way.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  using C = QmCfg<kQe4m3, kPair, kDup>;
  constexpr int SK = C::kStagesK, SV = C::kStagesV;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = ptx::smem_u32(sm);
  float* stat_m = reinterpret_cast<float*>(sm + C::kOffStat);  // group 1's row max
  float* stat_l = stat_m + kRows;                               // group 1's row sum
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::kOffMisc + 4);
  int* q_shift = reinterpret_cast<int*>(sm + C::kOffMisc + 8);        // [q tile]
  float* amax_red = reinterpret_cast<float*>(sm + C::kOffMisc + 16);  // [q tile][4]

  // mbarriers: K ring (full, empty), V ring (full, empty), per warpgroup S
  // full, S free, P full, P free; Q ready; MMA drain
  const uint32_t bar0 = sbase + C::kOffBar;
  auto kfull = [&](int s) { return bar0 + 8u * s; };
  auto kempty = [&](int s) { return bar0 + 8u * (SK + s); };
  auto vfull = [&](int s) { return bar0 + 8u * (2 * SK + s); };
  auto vempty = [&](int s) { return bar0 + 8u * (2 * SK + SV + s); };
  constexpr int kB = 2 * (SK + SV);
  // per group: 0 S full, 1 S free, 2 P full, 3 GEMM2 done (P free); with two
  // P buffers (32 rows) 2 / 3 serve even local tiles and 4 / 5 odd ones
  auto wgbar = [&](int wg, int k) { return bar0 + 8u * (kB + 6 * wg + k); };
  const uint32_t qready = bar0 + 8u * (kB + 6 * kWG);
  const uint32_t drain = qready + 8u;
  // row copies (32 / 64 packed rows): two P buffers per group (local tile t
  // writes buffer t & 1), so the softmax of tile t waits only for the GEMM2
  // of tile t - 2; each buffer has its own P-full and GEMM2-done barriers,
  // which then complete once every two tiles (never two phases ahead of a
  // waiter)
  constexpr bool kPDbl = kDup > 1;
  auto pfull_bar = [&](int wg, int t) { return wgbar(wg, (kPDbl && (t & 1)) ? 4 : 2); };
  auto g2done_bar = [&](int wg, int t) { return wgbar(wg, (kPDbl && (t & 1)) ? 5 : 3); };
  auto bar_phase = [&](int t) { return static_cast<uint32_t>(kPDbl ? (t >> 1) & 1 : t & 1); };

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  // Linear grid, work item outermost (the plan's longest-first order holds).
  const int g = blockIdx.x % a.h_k;
  const int rest = blockIdx.x / a.h_k;
  const int qt = rest % n_q_tiles;
  const int w_idx = rest / n_q_tiles;
  const int n0 = qt * kR * C::kQTiles;  // the CTA's first packed row

  const int4 item = reinterpret_cast<const int4*>(a.work)[w_idx];
  const int b = item.x, t_begin = item.y, t_end = item.z, slot = item.w;
  if (t_end <= t_begin) return;  // padding item
  const int L = a.seq_lens[b];
  const int T = t_end - t_begin;  // tiles of 128 keys
  const int key_begin = t_begin * kRows;

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
      ptx::mbar_init(wgbar(wg, 1), 4);
      ptx::mbar_init(wgbar(wg, 2), 4);
      ptx::mbar_init(wgbar(wg, 3), 1);
      ptx::mbar_init(wgbar(wg, 4), 4);
      ptx::mbar_init(wgbar(wg, 5), 1);
    }
    ptx::mbar_init(qready, C::kQTiles);  // each q tile's group
    ptx::mbar_init(drain, 2);
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

  if (warp == 0 || warp == kVLoadWarp) {
    // ----------------------------------------------------------- producers
    // Warp 0 loads K tiles, warp 11 V tiles.  A tile is keys [k0, k0 + 128)
    // of kv head g: 128 / box_rows boxes of box_rows rows (one per page when
    // pages are shorter than a tile), box jb on lane jb.  Block-table
    // entries come from a register window (lane l holds block wbase + l)
    // refilled 32 blocks ahead.
    const bool is_k = warp == 0;
    const int NS = is_k ? SK : SV;
    const uint32_t ring = sbase + (is_k ? C::kOffK : C::kOffV);
    const CUtensorMap* tmap = is_k ? &tmap_k : &tmap_v;
    auto full = [&](int st) { return is_k ? kfull(st) : vfull(st); };
    auto empty = [&](int st) { return is_k ? kempty(st) : vempty(st); };
    const int PS = a.page_size;
    const int box_rows = PS < kRows ? PS : kRows;
    const int nbox = kRows / box_rows;
    const bool active = lane < nbox;
    const int64_t bt_row = static_cast<int64_t>(b) * a.max_blocks;
    int valid_pages = (L + PS - 1) / PS;
    valid_pages = valid_pages < a.max_blocks ? valid_pages : a.max_blocks;
    auto load_win = [&](int base) -> int {
      const int blk = base + lane;
      return blk < valid_pages ? a.block_table[bt_row + blk] : a.num_pages;
    };
    if (lane == 0) ptx::prefetch_tmap(tmap);
    const bool evict_first = a.kv_evict_first != 0;
    const uint64_t kv_policy = ptx::policy_evict_first();
    const uint32_t tile_tx = kv_box_bytes(a.kv_format, kRows);
    // a tile spans nbox whole blocks (or lies in one block) and the window
    // starts at the item's first block, so a tile never straddles windows
    int wbase = key_begin / PS;
    int win = load_win(wbase);
    int win_next = load_win(wbase + 32);
    int issued = 0;
    for (int i = 0; i < T; ++i) {
      const int st = i % NS;
      if (i >= NS) {
        const bool freed = ptx::mbar_wait_bounded(empty(st), ((i / NS) - 1) & 1, abort_flag, kWaitNs);
        if (__any_sync(0xffffffffu, !freed)) {
          if (lane == 0) set_abort(abort_flag, a.status);
          break;
        }
      }
      const int key0 = key_begin + i * kRows;
      if (key0 / PS >= wbase + 32) {  // uniform over the warp
        wbase += 32;
        win = win_next;
        win_next = load_win(wbase + 32);
      }
      const int key = key0 + lane * box_rows;
      const int pg = __shfl_sync(0xffffffffu, win, (key / PS - wbase) & 31);
      const int page = (active && key < L) ? pg : a.num_pages;
      const int row_off = key % PS;
      if (lane == 0) ptx::mbar_arrive_expect_tx(full(st), tile_tx);  // packed bytes read
      __syncwarp();
      if (active)
        ptx::tma_load_kv(ring + st * kTileBytes + lane * box_rows * 128, tmap, full(st), 0, row_off, g, page,
                         evict_first, kv_policy);
      issued = i + 1;
    }
    if (*abort_flag && lane == 0) {
      volatile int never = 0;
      for (int i = (issued > NS ? issued - NS : 0); i < issued; ++i)
        ptx::mbar_wait_bounded(full(i % NS), (i / NS) & 1, &never, kWaitNs / 4);
    }
  } else if (warp == 1 || warp == kMma2Warp) {
    // ----------------------------------------------------------------- MMA
    // Unit u is (tile i, group u & 1) with the group's local tile t = u >> 1:
    // tile i = u alternates between the groups, or (paired q tiles) tile
    // i = u >> 1 goes to both, whose stage is then freed after group 1's
    // MMA.  GEMM1 (warp 1) into that group's S, GEMM2 (warp 10) into its O.
    if (lane == 0) {
      const bool gemm1 = warp == 1;
      bool ok = ptx::mbar_wait_bounded(qready, 0, abort_flag, kWaitNs);
      // A = e4m3 (Q and P parts), B = the K / V tile in the pool's format
      const uint32_t kv_fmt = kv_mma_format(a.kv_format);
      const uint32_t idesc_s = ptx::idesc_f8f6f4(kRows, kRows, false, false, 0, kv_fmt);  // S = Q K^T
      const uint32_t idesc_o = ptx::idesc_f8f6f4(kRows, kRows, false, true, 0, kv_fmt);   // O = P V, V MN-major
      // row copies: O^T = V^T P^T, M = d, N = the packed rows; A = the V tile
      // (MN-major), B = the group's P rows (K-major)
      const uint32_t idesc_ot = ptx::idesc_f8f6f4(kRows, kR, true, false, kv_fmt, 0);
      constexpr uint64_t kPtStep = (kR * 128) >> 4;  // descriptor step between the P rows' parts
      const uint64_t qdesc = ptx::smem_desc(sbase + C::kOffQ, 16, 1024, ptx::kSwizzle128B);
      const uint64_t kdesc0 = ptx::smem_desc(sbase + C::kOffK, 16, 1024, ptx::kSwizzle128B);
      const uint64_t pdesc0 = ptx::smem_desc(sbase + C::kOffP, 16, 1024, ptx::kSwizzle128B);
      const uint64_t vdesc0 = ptx::smem_desc(sbase + C::kOffV, 0, 1024, ptx::kSwizzle128B);
      constexpr uint64_t kPartStep = kPartBytes >> 4;  // descriptor step to the next operand part
      for (int u = 0; ok && u < T * C::kQTiles; ++u) {
        const int i = kPair ? u >> 1 : u;
        const int wg = u & 1, t = u >> 1;
        const bool last_use = !kPair || wg == 1;  // the tile's stage is freed after this unit
        const uint32_t tm = tmem + wg * C::kWgCols;
        if (gemm1) {
          const int st = i % SK;
          if (!ptx::mbar_wait_bounded(kfull(st), (i / SK) & 1, abort_flag, kWaitNs) ||
              (t >= 1 && !ptx::mbar_wait_bounded(wgbar(wg, 1), (t - 1) & 1, abort_flag, kWaitNs))) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t kdesc = kdesc0 + static_cast<uint64_t>((st * kTileBytes) >> 4);
          const uint64_t qd = qdesc + (kPair ? static_cast<uint64_t>(wg) * C::kQParts * kPartStep : 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // one K step = 32 bytes of d
#pragma unroll
            for (int part = 0; part < C::kQParts; ++part)
              ptx::mma_e4m3(tm, qd + part * kPartStep + 2 * kk, kdesc + 2 * kk, idesc_s,
                            (kk > 0 || part > 0) ? 1u : 0u);
          }
          ptx::mma_commit(wgbar(wg, 0));
          if (last_use) ptx::mma_commit(kempty(st));
        } else {
          const int st = i % SV;
          if (!ptx::mbar_wait_bounded(pfull_bar(wg, t), bar_phase(t), abort_flag, kWaitNs) ||
              !ptx::mbar_wait_bounded(vfull(st), (i / SV) & 1, abort_flag, kWaitNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t vdesc = vdesc0 + static_cast<uint64_t>((st * kTileBytes) >> 4);
          const uint64_t pdesc = pdesc0 + static_cast<uint64_t>(wg) * 2 * kPartStep +
                                 (kPDbl ? static_cast<uint64_t>(t & 1) * 2 * kPtStep : 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // one K step = 32 keys
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              if constexpr (kDup > 1)
                ptx::mma_e4m3(tm + kRows, vdesc + 256 * kk, pdesc + part * kPtStep + 2 * kk, idesc_ot,
                              (t > 0 || kk > 0 || part > 0) ? 1u : 0u);
              else
                ptx::mma_e4m3(tm + kRows, pdesc + part * kPartStep + 2 * kk, vdesc + 256 * kk, idesc_o,
                              (t > 0 || kk > 0 || part > 0) ? 1u : 0u);
            }
          }
          ptx::mma_commit(g2done_bar(wg, t));
          if (last_use) ptx::mma_commit(vempty(st));
        }
      }
      if (!ok) set_abort(abort_flag, a.status);
      ptx::mma_commit(drain);
      volatile int never = 0;
      ptx::mbar_wait_bounded(drain, 0, &never, kWaitNs);
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Two warpgroups take alternate tiles; in each, thread = query row r
    // (TMEM lane r of the group's S and O), warps covering the four lane
    // quarters.  A wait that gives up sets the abort flag and the loop runs
    // on (later waits return at once), so every warp takes the same path;
    // nothing is written out after an abort.
    const int wg = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int st_tid = ((warp - 2) & 3) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int bar_wg = 1 + wg;
    const uint32_t tmem_s = tmem + wg * C::kWgCols + lane_off;
    const uint32_t tmem_o = tmem_s + kRows;
    uint8_t* const pbuf = sm + C::kOffP + wg * 2 * kPartBytes;
    const int qrow = n0 + (kPair ? wg * kRows : 0) + r % kR;  // paired: group w owns q tile w
    const int cb = (r / kR) * kR;  // first key of this row's copy (uniform over a warp)
    const bool live = qrow < a.n_q;
    const float qd = a.qd[b * a.qd_seq + g * a.qd_head];
    const float kd = a.kd[b * a.kd_seq + g * a.kd_head];
    const float vd = a.vd[b * a.vd_seq + g * a.vd_head];

    // ---- Q row r -> two (bf16) or one (e4m3) K-major operand rows (group 0;
    // paired q tiles: each group its own tile, with its own scaling)
    uint8_t* const qbase = sm + C::kOffQ + (kPair ? wg * C::kQParts * kPartBytes : 0);
    int* const q_shift_g = q_shift + (kPair ? wg : 0);
    float* const amax_g = amax_red + (kPair ? 4 * wg : 0);
    if (kPair || wg == 0) {
      uint4 raw[kQe4m3 ? 8 : 16];
      const int64_t off = b * a.q_seq + (static_cast<int64_t>(g) * a.n_q + (live ? qrow : 0)) * kHeadDimDev;
      if (kQe4m3) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.q) + off);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) raw[cc] = live ? src[cc] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) *reinterpret_cast<uint4*>(swz(qbase, r, cc)) = raw[cc];
        if (st_tid == 0) *q_shift_g = 0;
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + off);
#pragma unroll
        for (int w = 0; w < 16; ++w) raw[w] = live ? src[w] : make_uint4(0u, 0u, 0u, 0u);
        uint32_t mbits = 0;  // bf16 |q| max: integer max of the magnitude bits
#pragma unroll
        for (int w = 0; w < 16; ++w) {
          const uint32_t v4[4] = {raw[w].x, raw[w].y, raw[w].z, raw[w].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) mbits = max(mbits, max(v4[e] & 0x7FFFu, (v4[e] >> 16) & 0x7FFFu));
        }
        float amax = __uint_as_float(mbits << 16);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) amax_g[(warp - 2) & 3] = amax;
        ptx::named_bar_sync(bar_wg, 128);
        amax = fmaxf(fmaxf(amax_g[0], amax_g[1]), fmaxf(amax_g[2], amax_g[3]));
        int shift = 0;
        if (amax > 0.f) {
          const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;
          shift = 7 - e;  // max |q| 2^shift in [128, 256)
          shift = shift > 126 ? 126 : (shift < -126 ? -126 : shift);
        }
        const float qscale = ldexpf(1.f, shift);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {  // 16 elements = two 16-byte words of bf16
          uint32_t hw[4], lw[4];
          const uint32_t w8[8] = {raw[2 * cc].x,     raw[2 * cc].y,     raw[2 * cc].z,     raw[2 * cc].w,
                                  raw[2 * cc + 1].x, raw[2 * cc + 1].y, raw[2 * cc + 1].z, raw[2 * cc + 1].w};
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            float x[4], hf[4];
            x[0] = __uint_as_float(w8[2 * wi] << 16) * qscale;
            x[1] = __uint_as_float(w8[2 * wi] & 0xFFFF0000u) * qscale;
            x[2] = __uint_as_float(w8[2 * wi + 1] << 16) * qscale;
            x[3] = __uint_as_float(w8[2 * wi + 1] & 0xFFFF0000u) * qscale;
            const uint16_t h01 = ptx::f32x2_to_e4m3x2(x[0], x[1]);
            const uint16_t h23 = ptx::f32x2_to_e4m3x2(x[2], x[3]);
            e4m3x4_to_f32(static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16), hf);
            const uint16_t l01 = ptx::f32x2_to_e4m3x2(x[0] - hf[0], x[1] - hf[1]);
            const uint16_t l23 = ptx::f32x2_to_e4m3x2(x[2] - hf[2], x[3] - hf[3]);
            hw[wi] = static_cast<uint32_t>(h01) | (static_cast<uint32_t>(h23) << 16);
            lw[wi] = static_cast<uint32_t>(l01) | (static_cast<uint32_t>(l23) << 16);
          }
          *reinterpret_cast<uint4*>(swz(qbase, r, cc)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(swz(qbase + kPartBytes, r, cc)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        if (st_tid == 0) *q_shift_g = shift;
      }
      ptx::fence_proxy_async_smem();
      ptx::named_bar_sync(bar_wg, 128);
      if (st_tid == 0) ptx::mbar_arrive(qready);
    }
    ptx::named_bar_sync(kBarAll, 128 * kWG);  // the Q shift is set
    const int shift = *q_shift_g;
    // raw (computed) score -> logit and -> log2 units; 2^-shift undoes the Q scaling
    const float scale_l = a.softmax_scale * qd * kd * ldexpf(1.f, -shift);
    const float c2 = scale_l * kLog2e;
    // last visible key of this row (-1: none)
    int lim = a.causal ? L - a.q_len + qrow / a.h_r : L - 1;
    lim = lim < L - 1 ? lim : L - 1;
    if (!live) lim = -1;

    float m_run = -INFINITY;  // reference row maximum (raw units)
    float l_run = 0.f;        // running row sum of x = 448 p 2^-kTau
    const float head_c = kTau / c2;  // kTau in raw score units
    bool ok = true;
    int t_last = -1;
    // A warp whose 32 rows are all past n_q computes nothing: its P rows
    // keep whatever they hold, which reaches only its own (unused) O rows.
    const bool warp_live = __any_sync(0xffffffffu, live);
    if constexpr (kDup == 1) {
      // alternate tiles, or (paired q tiles) every tile
      for (int i = kPair ? 0 : wg; i < T; i += kPair ? 1 : kWG) {
        const int t = kPair ? i : i >> 1;
        const int key0 = key_begin + i * kRows;
        t_last = t;
        if (!ptx::mbar_wait_bounded(wgbar(wg, 0), t & 1, abort_flag, kWaitNs)) ok = false;
        ptx::tc_fence_after();
        if (warp_live) {
          // pass 1: the row's masked maximum over the tile (select: garbage or
          // poison keys never leak); a tile wholly below every row's limit of
          // its warp skips the selects.  64 columns per TMEM round trip.
          // (rows past n_q produce nothing: any value will do for them)
          const bool unmasked = __all_sync(0xffffffffu, !live || key0 + kRows - 1 <= lim);
          float mt = -INFINITY;
    #pragma unroll
          for (int h0 = 0; h0 < kRows; h0 += kCh) {
            uint32_t rr[kCh];
    #pragma unroll
            for (int c0 = 0; c0 < kCh; c0 += 16) MJ_TMEM_LD16(tmem_s + h0 + c0, (rr + c0));
            ptx::tmem_ld_wait();
            if (unmasked) {
    #pragma unroll
              for (int e = 0; e < kCh; e += 2) mt = fmax3(mt, __uint_as_float(rr[e]), __uint_as_float(rr[e + 1]));
            } else {
    #pragma unroll
              for (int e = 0; e < kCh; e += 2)
                mt = fmax3(mt, (key0 + h0 + e <= lim) ? __uint_as_float(rr[e]) : -INFINITY,
                           (key0 + h0 + e + 1 <= lim) ? __uint_as_float(rr[e + 1]) : -INFINITY);
            }
          }
          if (!live) mt = -INFINITY;  // keeps the maximum of an empty row at -inf
          const bool moved = mt > m_run + head_c;
          const float m_new = moved ? mt : m_run;
          const float mu = (m_new == -INFINITY) ? 0.f : m_new;  // the -inf guard
          const float corr = moved ? fast_exp2((m_run - mu) * c2) : 1.f;  // 0 for a fresh row
          l_run *= corr;
          m_run = m_new;
          // this group's P buffer and O are free once GEMM2 of its previous tile ran
          if (t > 0 && !ptx::mbar_wait_bounded(wgbar(wg, 3), (t - 1) & 1, abort_flag, kWaitNs)) ok = false;
          // lazy O correction: each row rescales its own TMEM lane, but TMEM
          // access is warp-wide, so a warp corrects when any of its rows moved
          if (t > 0 && __any_sync(0xffffffffu, moved)) {
            ptx::tc_fence_after();
            constexpr int kOc = 64;
    #pragma unroll
            for (int h0 = 0; h0 < kRows; h0 += kOc) {
              uint32_t rr[kOc];
    #pragma unroll
              for (int c0 = 0; c0 < kOc; c0 += 16) MJ_TMEM_LD16(tmem_o + h0 + c0, (rr + c0));
              ptx::tmem_ld_wait();
    #pragma unroll
              for (int e = 0; e < kOc; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * corr);
    #pragma unroll
              for (int c0 = 0; c0 < kOc; c0 += 16) MJ_TMEM_ST16(tmem_o + h0 + c0, (rr + c0));
            }
            ptx::tmem_st_wait();
          }
          // pass 2: x = 448 p 2^-kTau = 2^((s - m) c + log2 448 - kTau) in
          // fp32 (ex2.approx.f32; x <= 448), the row sum of the unrounded x in
          // fp32, and the MMA operand split x = hi + lo through half precision
          // (x rounded to 11 significant bits, hi = e4m3(x), lo = e4m3(x - hi),
          // the difference exact in halves): about 8 significant bits of x in P.
          // (On GB300 the fp32 exponential issues at the same result rate as the
          // packed-half one, so nothing is saved by narrowing it.)
          const float bias = fmaf(-mu, c2, kLog2PScale);
          const float2 c2x2 = make_float2(c2, c2), bias2 = make_float2(bias, bias);
    #pragma unroll
          for (int h0 = 0; h0 < kRows; h0 += kCh) {
            uint32_t rr[kCh];
    #pragma unroll
            for (int c0 = 0; c0 < kCh; c0 += 16) MJ_TMEM_LD16(tmem_s + h0 + c0, (rr + c0));
            ptx::tmem_ld_wait();
            if (h0 + kCh == kRows) {
              // S is read whole: the group's next GEMM1 may overwrite it while
              // the last half is turned into P
              ptx::tc_fence_before();
              __syncwarp();
              if (lane == 0) ptx::mbar_arrive(wgbar(wg, 1));
            }
    #pragma unroll
            for (int q = 0; q < kCh / 16; ++q) {
              const int cc = h0 / 16 + q;  // 16-key chunk of the P row
              uint32_t hw[4], lw[4];
              float2 sum2 = make_float2(0.f, 0.f);
    #pragma unroll
              for (int wi = 0; wi < 4; ++wi) {
                uint16_t h8[2], l8[2];
    #pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                  const int e0 = q * 16 + wi * 4 + pr * 2;
                  float s0 = __uint_as_float(rr[e0]), s1 = __uint_as_float(rr[e0 + 1]);
                  if (!unmasked) {
                    const int c = h0 + e0;
                    s0 = (key0 + c <= lim) ? s0 : -INFINITY;
                    s1 = (key0 + c + 1 <= lim) ? s1 : -INFINITY;
                  }
                  const float2 y = fma2(make_float2(s0, s1), c2x2, bias2);
                  const float x0 = fast_exp2(y.x);
                  const float x1 = fast_exp2(y.y);
                  sum2 = add2(sum2, make_float2(x0, x1));
                  const uint32_t x2 = f32x2_to_f16x2(x0, x1);
                  const uint16_t hi8 = f16x2_to_e4m3x2(x2);
                  const uint32_t hf2 = e4m3x2_to_f16x2(hi8);
                  l8[pr] = f16x2_to_e4m3x2(sub_f16x2(x2, hf2));
                  h8[pr] = hi8;
                }
                hw[wi] = static_cast<uint32_t>(h8[0]) | (static_cast<uint32_t>(h8[1]) << 16);
                lw[wi] = static_cast<uint32_t>(l8[0]) | (static_cast<uint32_t>(l8[1]) << 16);
              }
              l_run += sum2.x + sum2.y;
              *reinterpret_cast<uint4*>(swz(pbuf, r, cc)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
              *reinterpret_cast<uint4*>(swz(pbuf + kPartBytes, r, cc)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
          }
        }
        if (!warp_live) {  // S read (a live warp released it after its last load)
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(wgbar(wg, 1));
          // and, like a live warp, it arrives on P full only after GEMM2 of the
          // group's previous tile: a group with no live row (the second q tile
          // past n_q) would otherwise complete P full a second phase before the
          // GEMM2 thread's wait on the first
          if (t > 0 && !ptx::mbar_wait_bounded(wgbar(wg, 3), (t - 1) & 1, abort_flag, kWaitNs)) ok = false;
        }
        // keys past the sequence end: zero their V rows (0 * poison must not
        // reach O; the TMA landed whole pages).  Thread r owns key row r (of
        // group 0 when both groups take the tile: its GEMM2 is issued first).
        if ((!kPair || wg == 0) && key0 + kRows > L) {
          const int st = i % SV;
          if (!ptx::mbar_wait_bounded(vfull(st), (i / SV) & 1, abort_flag, kWaitNs)) ok = false;
          if (key0 + r >= L) {
            uint4* vrow = reinterpret_cast<uint4*>(sm + C::kOffV + st * kTileBytes + r * 128);
#pragma unroll
            for (int e = 0; e < 8; ++e) vrow[e] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(wgbar(wg, 2));
        if (!ok) set_abort(abort_flag, a.status);
      }

      // ---- epilogue: this group's O is final once its last GEMM2 is done;
      // group 0 merges both groups' rows (row r's state of group 1 through
      // shared memory, its O from group 1's TMEM columns, same lanes).  With
      // paired q tiles each group writes its own rows (its state alone).
      if (t_last >= 0 && !ptx::mbar_wait_bounded(wgbar(wg, 3), t_last & 1, abort_flag, kWaitNs)) ok = false;
      if (!ok) set_abort(abort_flag, a.status);
      if (!kPair && wg == 1) {
        stat_m[r] = m_run;
        stat_l[r] = l_run;
      }
      const bool fine = !ptx::named_bar_red_or(kBarAll, 128 * kWG, *abort_flag != 0);
      if ((kPair || wg == 0) && fine) {
        ptx::tc_fence_after();
        const float m1 = kPair ? -INFINITY : stat_m[r], l1 = kPair ? 0.f : stat_l[r];
        const float mx = fmaxf(m_run, m1);
        const float f0 = (m_run == -INFINITY) ? 0.f : fast_exp2((m_run - mx) * c2);
        const float f1 = (m1 == -INFINITY) ? 0.f : fast_exp2((m1 - mx) * c2);
        const float lraw = l_run * f0 + l1 * f1;  // row sum of x, both groups
        const bool final_out = a.n_splits[b] <= 1;
        const int64_t orow = final_out ? b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + (live ? qrow : 0)) * kHeadDimDev
                                       : part_row(a, b, g, slot, live ? qrow : 0) * kHeadDimDev;
        const uint32_t o1 = tmem + C::kWgCols + kRows + lane_off;  // group 1's O, same lanes
        const float mrow = mx;
        const float l = lraw * kPScaleInv;
        const float f = vd * kPScaleInv * (final_out ? a.scale_o / (l + 1e-30f) : 1.f);
        const bool writer = live;
#pragma unroll 1
        for (int c0 = 0; c0 < kRows; c0 += 16) {
          uint32_t ra[16], rb[16];
          MJ_TMEM_LD16(tmem_o + c0, ra);
          if constexpr (kPair) {
#pragma unroll
            for (int e = 0; e < 16; ++e) rb[e] = 0u;  // no second group's state (f1 = 0)
          } else {
            MJ_TMEM_LD16(o1 + c0, rb);
          }
          ptx::tmem_ld_wait();
          float v[16];
          // select, not multiply: a group with no key left its O stale
#pragma unroll
          for (int e = 0; e < 16; ++e)
            v[e] = ((f0 > 0.f ? __uint_as_float(ra[e]) * f0 : 0.f) + (f1 > 0.f ? __uint_as_float(rb[e]) * f1 : 0.f));
          if (!writer) continue;
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] *= f;
          if (final_out) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const __nv_bfloat162 v2 = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
              pk[e] = *reinterpret_cast<const uint32_t*>(&v2);
            }
            uint4* dst = reinterpret_cast<uint4*>(a.o + orow + c0);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          } else {
            float4* dst = reinterpret_cast<float4*>(a.o_part + orow + c0);
#pragma unroll
            for (int e = 0; e < 4; ++e) dst[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          }
        }
        if (writer) {
          const float m_logit = mrow * scale_l;
          if (final_out) {
            a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + qrow] = m_logit + logf(l);
          } else {
            const int64_t pr = part_row(a, b, g, slot, qrow);
            a.m_part[pr] = m_logit;
            a.l_part[pr] = l;
          }
        }
      }
    } else {
      // ---- row copies (32 or 64 packed rows, each held 4 or 2 times): copy
      // cp of packed row qr holds keys [cp kR, (cp + 1) kR) of every tile.  The
      // copies of a row share its reference maximum (the tile maxima of their
      // key slices meet in shared memory), so their P entries are on one
      // scale and GEMM2 sums them into one row: O^T[d, row] += V^T[d, key]
      // P^T[key, row] with N = the packed rows, a quarter (half) of the MMA
      // work of a 128-row O.  The group's O^T sits in TMEM with d on the
      // lanes, so a correction scales every lane's column of each row.
      const int cp = r / kR;  // this lane's copy
      const int qr = r % kR;  // its packed row in the q tile
      constexpr int kPtPart = kR * 128;  // one e4m3 part of the group's P rows
      // [kDup][kR] tile maxima of the slices, then [2][kR] factors: after the
      // two P buffers (32 rows), or in their own region (64 rows)
      float* const mx_x = kDup == 2 ? reinterpret_cast<float*>(sm + C::kOffX + wg * 1024)
                                    : reinterpret_cast<float*>(pbuf + 4 * kPtPart);
      float* const fx = mx_x + kRows;                                      // [2][kR] per-row factors
      const int bar_red = 4 + wg;  // the group's reduction barrier
      for (int i = wg; i < T; i += kWG) {
        const int t = i >> 1;
        const int key0 = key_begin + i * kRows;
        t_last = t;
        if (!ptx::mbar_wait_bounded(wgbar(wg, 0), t & 1, abort_flag, kWaitNs)) ok = false;
        ptx::tc_fence_after();
        // the row's slice of S stays in registers, and S goes back to GEMM1
        // right after this read
        uint32_t sv[kR];
        float mt = -INFINITY;
        bool unmasked = true;
        if (warp_live) {
          unmasked = __all_sync(0xffffffffu, !live || key0 + cb + kR - 1 <= lim);
  #pragma unroll
          for (int c0 = 0; c0 < kR; c0 += 16) MJ_TMEM_LD16(tmem_s + cb + c0, (sv + c0));
          ptx::tmem_ld_wait();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(wgbar(wg, 1));
        if (warp_live) {
          if (unmasked) {
  #pragma unroll
            for (int e = 0; e < kR; e += 2) mt = fmax3(mt, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]));
          } else {
  #pragma unroll
            for (int e = 0; e < kR; e += 2)
              mt = fmax3(mt, (key0 + cb + e <= lim) ? __uint_as_float(sv[e]) : -INFINITY,
                         (key0 + cb + e + 1 <= lim) ? __uint_as_float(sv[e + 1]) : -INFINITY);
          }
          if (!live) mt = -INFINITY;  // keeps the maximum of an empty row at -inf
        }
        // the row's tile maximum over its copies; every copy then takes the
        // same decision from the same values
        mx_x[cp * kR + qr] = mt;
        ptx::named_bar_sync(bar_wg, 128);
        float mrow = -INFINITY;
  #pragma unroll
        for (int s2 = 0; s2 < kDup; ++s2) mrow = fmaxf(mrow, mx_x[s2 * kR + qr]);
        const bool moved = mrow > m_run + head_c;
        const float m_new = moved ? mrow : m_run;
        const float mu = (m_new == -INFINITY) ? 0.f : m_new;  // the -inf guard
        const float corr = moved ? fast_exp2((m_run - mu) * c2) : 1.f;  // 0 for a fresh row
        l_run *= corr;
        m_run = m_new;
        if (cp == 0) fx[qr] = corr;
        const bool any_moved = ptx::named_bar_red_or(bar_red, 128, moved);  // also: fx and mx_x reads done
        // this tile's P rows are free once the GEMM2 that last read them ran
        // (the previous tile's, or with two buffers the one before it); O^T
        // takes a correction only after the previous tile's GEMM2
        const int t_free = kPDbl ? t - 2 : t - 1;
        if (t_free >= 0 && !ptx::mbar_wait_bounded(g2done_bar(wg, t_free), bar_phase(t_free), abort_flag, kWaitNs))
          ok = false;
        if (kPDbl && t > 0 && any_moved &&
            !ptx::mbar_wait_bounded(g2done_bar(wg, t - 1), bar_phase(t - 1), abort_flag, kWaitNs))
          ok = false;
        uint8_t* const pb = pbuf + (kPDbl ? (t & 1) * 2 * kPtPart : 0);  // this tile's P rows
        if (t > 0 && any_moved) {  // lazy correction: lane d scales column qr of every row by its factor
          ptx::tc_fence_after();
  #pragma unroll
          for (int c0 = 0; c0 < kR; c0 += 16) {
            uint32_t rr[16];
            MJ_TMEM_LD16(tmem_o + c0, rr);
            ptx::tmem_ld_wait();
  #pragma unroll
            for (int e = 0; e < 16; ++e) rr[e] = __float_as_uint(__uint_as_float(rr[e]) * fx[c0 + e]);
            MJ_TMEM_ST16(tmem_o + c0, rr);
          }
          ptx::tmem_st_wait();
        }
        if (warp_live) {
          // pass 2 on the slice: x, its sum, and the hi / lo split (as for
          // 128 rows) into row qr, keys [cb, cb + kR), of the group's P rows
          const float bias = fmaf(-mu, c2, kLog2PScale);
          const float2 c2x2 = make_float2(c2, c2), bias2 = make_float2(bias, bias);
  #pragma unroll
          for (int q = 0; q < kR / 16; ++q) {
            const int cc = cb / 16 + q;  // 16-key chunk of the P row
            uint32_t hw[4], lw[4];
            float2 sum2 = make_float2(0.f, 0.f);
  #pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              uint16_t h8[2], l8[2];
  #pragma unroll
              for (int pr = 0; pr < 2; ++pr) {
                const int e0 = q * 16 + wi * 4 + pr * 2;
                float s0 = __uint_as_float(sv[e0]), s1 = __uint_as_float(sv[e0 + 1]);
                if (!unmasked) {
                  s0 = (key0 + cb + e0 <= lim) ? s0 : -INFINITY;
                  s1 = (key0 + cb + e0 + 1 <= lim) ? s1 : -INFINITY;
                }
                const float2 y = fma2(make_float2(s0, s1), c2x2, bias2);
                const float x0 = fast_exp2(y.x);
                const float x1 = fast_exp2(y.y);
                sum2 = add2(sum2, make_float2(x0, x1));
                const uint32_t x2 = f32x2_to_f16x2(x0, x1);
                const uint16_t hi8 = f16x2_to_e4m3x2(x2);
                const uint32_t hf2 = e4m3x2_to_f16x2(hi8);
                l8[pr] = f16x2_to_e4m3x2(sub_f16x2(x2, hf2));
                h8[pr] = hi8;
              }
              hw[wi] = static_cast<uint32_t>(h8[0]) | (static_cast<uint32_t>(h8[1]) << 16);
              lw[wi] = static_cast<uint32_t>(l8[0]) | (static_cast<uint32_t>(l8[1]) << 16);
            }
            l_run += sum2.x + sum2.y;
            *reinterpret_cast<uint4*>(swz(pb, qr, cc)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(swz(pb + kPtPart, qr, cc)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
        // keys past the sequence end: zero their V rows (0 * poison must not
        // reach O; the TMA landed whole pages).  Thread r owns key row r.
        if (key0 + kRows > L) {
          const int st = i % SV;
          if (!ptx::mbar_wait_bounded(vfull(st), (i / SV) & 1, abort_flag, kWaitNs)) ok = false;
          if (key0 + r >= L) {
            uint4* vrow = reinterpret_cast<uint4*>(sm + C::kOffV + st * kTileBytes + r * 128);
  #pragma unroll
            for (int e = 0; e < 8; ++e) vrow[e] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(pfull_bar(wg, t));
        if (!ok) set_abort(abort_flag, a.status);
      }

      // ---- epilogue: a row's sum over its copies (one scale), then group 0
      // merges both groups' rows (group 1's state through shared memory, its
      // O^T from its TMEM columns) and lane d writes element d of every row
      if (t_last >= 0 && !ptx::mbar_wait_bounded(g2done_bar(wg, t_last), bar_phase(t_last), abort_flag, kWaitNs))
        ok = false;
      if (!ok) set_abort(abort_flag, a.status);
      mx_x[cp * kR + qr] = l_run;  // (every read of the maxima is done: the last tile's barrier)
      ptx::named_bar_sync(bar_wg, 128);
      float lrow = 0.f;
  #pragma unroll
      for (int s2 = 0; s2 < kDup; ++s2) lrow += mx_x[s2 * kR + qr];
      if (wg == 1 && cp == 0) {
        stat_m[qr] = m_run;
        stat_l[qr] = lrow;
      }
      const bool fine = !ptx::named_bar_red_or(kBarAll, 128 * kWG, *abort_flag != 0);
      if (wg == 0 && fine) {
        ptx::tc_fence_after();
        const bool final_out = a.n_splits[b] <= 1;
        if (cp == 0) {
          const float m1 = stat_m[qr], l1 = stat_l[qr];
          const float mx = fmaxf(m_run, m1);
          const float f0 = (m_run == -INFINITY) ? 0.f : fast_exp2((m_run - mx) * c2);
          const float f1 = (m1 == -INFINITY) ? 0.f : fast_exp2((m1 - mx) * c2);
          const float l = (lrow * f0 + l1 * f1) * kPScaleInv;
          const float f = vd * kPScaleInv * (final_out ? a.scale_o / (l + 1e-30f) : 1.f);
          // 0 marks a group with no key for the row (its O^T column is stale)
          fx[qr] = f0 > 0.f ? f0 * f : 0.f;
          fx[kR + qr] = f1 > 0.f ? f1 * f : 0.f;
          if (live) {
            const float m_logit = mx * scale_l;
            if (final_out) {
              a.lse[(static_cast<int64_t>(b) * a.h_k + g) * a.n_q + qrow] = m_logit + logf(l);
            } else {
              const int64_t pr = part_row(a, b, g, slot, qrow);
              a.m_part[pr] = m_logit;
              a.l_part[pr] = l;
            }
          }
        }
        ptx::named_bar_sync(1, 128);  // group 0's barrier: the factors are written
        const int d = r;              // this lane's element of every row
        const uint32_t o1 = tmem + C::kWgCols + kRows + lane_off;  // group 1's O^T, same lanes
        const int live_rows = a.n_q - n0 < kR ? a.n_q - n0 : kR;
  #pragma unroll 1
        for (int c0 = 0; c0 < kR; c0 += 16) {
          uint32_t ra[16], rb[16];
          MJ_TMEM_LD16(tmem_o + c0, ra);
          MJ_TMEM_LD16(o1 + c0, rb);
          ptx::tmem_ld_wait();
  #pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = c0 + e;
            if (c >= live_rows) break;
            const float w0 = fx[c], w1 = fx[kR + c];
            // select, not multiply: a group with no key left its column stale
            const float v = (w0 > 0.f ? __uint_as_float(ra[e]) * w0 : 0.f) + (w1 > 0.f ? __uint_as_float(rb[e]) * w1 : 0.f);
            if (final_out) {
              a.o[b * a.o_seq + (static_cast<int64_t>(g) * a.n_q + n0 + c) * kHeadDimDev + d] = __float2bfloat16_rn(v);
            } else {
              a.o_part[part_row(a, b, g, slot, n0 + c) * kHeadDimDev + d] = v;
            }
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::kTmemCols);
}

template <bool kQe4m3, int kDup, bool kPair = false>
cudaError_t launch_qm(const DecodeDev& a, int n_q_tiles, cudaStream_t stream) {
  using C = QmCfg<kQe4m3, kPair, kDup>;
  const int box_rows = a.page_size < kRows ? a.page_size : kRows;
  CUtensorMap mk, mv;
  if (!make_kv_map(&mk, a.k, a.page_size, a.h_k, a.num_pages, a.k_row, a.k_head, a.k_page, box_rows, 1,
                   a.kv_format) ||
      !make_kv_map(&mv, a.v, a.page_size, a.h_k, a.num_pages, a.v_row, a.v_head, a.v_page, box_rows, 1,
                   a.kv_format))
    return cudaErrorInvalidValue;
  auto kern = decode_qm_kernel<kQe4m3, kDup, kPair>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(a.num_work) * n_q_tiles * a.h_k, 1, 1);
  return launch_pdl(kern, grid, dim3(kThreads, 1, 1), C::kBytes, stream, a, mk, mv, n_q_tiles);
}

}  // namespace

cudaError_t launch_decode_qm(const DecodeDev& a, int rows_per_cta, int n_q_tiles, bool q_e4m3,
                             cudaStream_t stream) {
  switch (rows_per_cta) {
    case 256:  // two q tiles of 128 rows per CTA
      return q_e4m3 ? launch_qm<true, 1, true>(a, n_q_tiles, stream) : launch_qm<false, 1, true>(a, n_q_tiles, stream);
    case 128: return q_e4m3 ? launch_qm<true, 1>(a, n_q_tiles, stream) : launch_qm<false, 1>(a, n_q_tiles, stream);
    case 64: return q_e4m3 ? launch_qm<true, 2>(a, n_q_tiles, stream) : launch_qm<false, 2>(a, n_q_tiles, stream);
    case 32: return q_e4m3 ? launch_qm<true, 4>(a, n_q_tiles, stream) : launch_qm<false, 4>(a, n_q_tiles, stream);
    default: return cudaErrorInvalidValue;
  }
}

int qm_smem_bytes(bool q_e4m3) { return q_e4m3 ? QmCfg<true>::kBytes : QmCfg<false>::kBytes; }

}  // namespace mj
