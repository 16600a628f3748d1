// C ABI entry points: argument validation, kernel choice and launches.

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdio>
#include <cstring>

#include "mj.h"
#include "mj_internal.h"
#include "mj_kernels.h"

namespace mj {

namespace {

constexpr size_t kAlign = 256;
size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WorkspaceLayout {
  size_t o_off, m_off, l_off, sched_off, total;
};

// Split partials (when the plan may split), then the persistent kernel's
// unit counter (reset by the launch itself, in the stream).
WorkspaceLayout workspace_layout(const mj_decode_params& p) {
  WorkspaceLayout w{0, 0, 0, 0, 0};
  if (p.max_splits > 1) {
    const size_t rows = static_cast<size_t>(p.num_seqs) * p.h_k * p.max_splits * p.q_len * p.h_r;
    w.o_off = 0;
    w.m_off = round_up(rows * kHeadDim * sizeof(float));
    w.l_off = w.m_off + round_up(rows * sizeof(float));
    w.total = w.l_off + round_up(rows * sizeof(float));
  }
  if (choose_kernel(p).kind == KernelKind::kTensorCoreGrouped) {
    w.sched_off = w.total;
    w.total += kAlign;
  }
  return w;
}

// SMs of the current device (the persistent kernel's grid), cached per
// device; 0 when it cannot be read.
int device_sm_count() {
  static int cache[64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// nvfp4 scale planes: present, 16-byte aligned, page and head strides
// 16-byte multiples (a page's rows of one head are 8 bytes apart).
bool scales_ok(const mj_decode_params& p, const mj_decode_args& a) {
  if (p.kv_format != MJ_KV_NVFP4) return true;
  if (!a.k_scales || !a.v_scales || !aligned16(a.k_scales) || !aligned16(a.v_scales)) return false;
  const int64_t st[4] = {a.ks_page, a.ks_head, a.vs_page, a.vs_head};
  for (int64_t s : st)
    if (s <= 0 || (s & 15) != 0 || s >= (int64_t{1} << 40)) return false;
  return true;
}

const char* kv_format_name(int f) {
  switch (f) {
    case MJ_KV_E3M2: return "e3m2";
    case MJ_KV_E2M3: return "e2m3";
    case MJ_KV_E2M1: return "e2m1";
    case MJ_KV_NVFP4: return "nvfp4";
    default: return "e4m3";
  }
}

// K/V pool pointers and byte strides: 16-byte aligned (the page gathers'
// TMA boxes), 32-byte aligned for the packed narrow formats (their TMA
// element types require it).
bool kv_layout_ok(const mj_decode_params& p, const void* k, const void* v, const int64_t (&strides)[6]) {
  // nvfp4 codes are read as bytes (16-byte rules); the MMA-read narrow
  // formats need 32
  const bool narrow = p.kv_format != MJ_KV_E4M3 && p.kv_format != MJ_KV_NVFP4;
  if (!aligned16(k) || !aligned16(v)) return false;
  if (narrow && (!aligned32(k) || !aligned32(v))) return false;
  const int64_t mask = narrow ? 31 : 15;
  for (int64_t s : strides)
    if (s <= 0 || (s & mask) != 0 || s >= (int64_t{1} << 40)) return false;
  return true;
}

constexpr int kDefaultL2Prefetch = 0;  // tiles; measured choice
constexpr int kDefaultKvEvictFirst = 1;  // measured choice (faster on every workload)
constexpr int kSmemPerSm = 233472;  // 228 KiB usable shared memory per SM
constexpr int kSmemReservedPerCta = 1024;
// Units per SM the plan cuts for the head-grouped kernel (measured, 2 to 12
// per SM): six for 8 heads x 4 rows (GQA decode), three for 2 heads x 32
// rows (spec verify: each unit boundary stalls the CTA's softmax for its
// output epilogue, a few microseconds), two for 1 head x 32 rows (sweep with
// h_k = 1: 118 us at two, 122 at three, 128 at four).
constexpr int kGroupedUnitsPerSm = 6;
constexpr int kPairUnitsPerSm = 3;
constexpr int kOneHeadUnitsPerSm = 2;
// More packed rows than this go to the query-rows kernel (measured with its
// rows held several times: 32 rows 115 us vs 121 us swap-AB on the sweep,
// 261 us vs 260 us (2-head grouped) / 278 us on the spec-verify workload,
// with no merge; at 16 rows the swap-AB kernel is as fast).
constexpr int kQRowsFrom = 16;

}  // namespace

KernelChoice choose_kernel(const mj_decode_params& p) {
  const int n_q = p.q_len * p.h_r;
  const bool e4m3 = p.q_dtype == MJ_E4M3;
  KernelChoice k{};
  k.heads_per_cta = 1;
  int smem;
  int g = 0, rh = 0;
  if (p.kernel == MJ_KERNEL_CUDA_CORE) {
    k.kind = KernelKind::kCudaCore;
    k.rows_per_cta = n_q <= 4 ? 4 : (n_q <= 8 ? 8 : 16);
    smem = cc_smem_bytes(k.rows_per_cta);
    static const char* names[2][3] = {{"cc_n4_bf16", "cc_n8_bf16", "cc_n16_bf16"},
                                      {"cc_n4_e4m3", "cc_n8_e4m3", "cc_n16_e4m3"}};
    k.name = names[e4m3][k.rows_per_cta == 4 ? 0 : (k.rows_per_cta == 8 ? 1 : 2)];
  } else if (p.kernel == MJ_KERNEL_TENSOR_CORE_QROWS ||
             (p.kernel == MJ_KERNEL_AUTO && n_q > kQRowsFrom && p.kv_format != MJ_KV_NVFP4)) {
    k.kind = KernelKind::kTensorCoreQRows;
    // up to 32 or 64 packed rows: each row held four or two times in the
    // 128 MMA rows, every copy taking that share of a tile's keys; more
    // than 128: two q tiles per CTA sharing each KV tile
    k.rows_per_cta = n_q <= 32 ? 32 : (n_q <= 64 ? 64 : (n_q <= 128 ? 128 : 256));
    smem = qm_smem_bytes(e4m3);
    static const char* names[2][4] = {{"qm_r32_bf16", "qm_r64_bf16", "qm_bf16", "qm_pair_bf16"},
                                      {"qm_r32_e4m3", "qm_r64_e4m3", "qm_e4m3", "qm_pair_e4m3"}};
    k.name = names[e4m3][k.rows_per_cta == 32 ? 0 : (k.rows_per_cta == 64 ? 1 : (k.rows_per_cta == 128 ? 2 : 3))];
  } else if (p.kernel == MJ_KERNEL_TENSOR_CORE_GROUPED && tcg_supported(p.h_k, n_q, &g, &rh)) {
    k.kind = KernelKind::kTensorCoreGrouped;
    k.rows_per_cta = rh;
    k.heads_per_cta = g;
    smem = tcg_smem_bytes(g, rh, e4m3);
    static const char* names[2][4] = {{"tcg_g8r4_bf16", "tcg_g4r8_bf16", "tcg_g2r32_bf16", "tcg_g1r32_bf16"},
                                      {"tcg_g8r4_e4m3", "tcg_g4r8_e4m3", "tcg_g2r32_e4m3", "tcg_g1r32_e4m3"}};
    k.name = names[e4m3][g == 8 ? 0 : (g == 4 ? 1 : (g == 2 ? 2 : 3))];
  } else {
    k.kind = KernelKind::kTensorCore;
    k.rows_per_cta = n_q <= 8 ? 8 : (n_q <= 16 ? 16 : (n_q <= 32 ? 32 : 64));
    smem = tc_smem_bytes(k.rows_per_cta, e4m3, p.kv_format == MJ_KV_NVFP4);
    static const char* names[2][4] = {{"tc_r8_bf16", "tc_r16_bf16", "tc_r32_bf16", "tc_r64_bf16"},
                                      {"tc_r8_e4m3", "tc_r16_e4m3", "tc_r32_e4m3", "tc_r64_e4m3"}};
    const int idx = k.rows_per_cta == 8 ? 0 : (k.rows_per_cta == 16 ? 1 : (k.rows_per_cta == 32 ? 2 : 3));
    k.name = names[e4m3][idx];
  }
  k.n_q_tiles = (n_q + k.rows_per_cta - 1) / k.rows_per_cta;
  int per_sm = kSmemPerSm / (smem + kSmemReservedPerCta);
  int cap = 16;
  if (k.kind == KernelKind::kTensorCore) cap = tc_min_blocks(k.rows_per_cta, e4m3, p.kv_format == MJ_KV_NVFP4);
  if (k.kind == KernelKind::kTensorCoreGrouped || k.kind == KernelKind::kTensorCoreQRows)
    cap = 1;  // owns the SM: all of TMEM, a deep ring
  if (per_sm > cap) per_sm = cap;
  k.ctas_per_sm = (per_sm < 1 ? 1 : per_sm) * k.heads_per_cta;
  // The persistent kernel takes units from a queue: the plan cuts about six
  // units per SM, so that the greedy queue (longest first) ends balanced.
  if (k.kind == KernelKind::kTensorCoreGrouped)
    k.ctas_per_sm *= g == 1 ? kOneHeadUnitsPerSm : (g == 2 ? kPairUnitsPerSm : kGroupedUnitsPerSm);
  return k;
}

}  // namespace mj

using namespace mj;

extern "C" const char* mj_status_string(mj_status s) {
  switch (s) {
    case MJ_OK: return "ok";
    case MJ_ERR_INVALID_ARG: return "invalid argument";
    case MJ_ERR_UNSUPPORTED: return "unsupported configuration";
    case MJ_ERR_CAPACITY: return "buffer or workspace too small";
    case MJ_ERR_CUDA: return "CUDA error";
    case MJ_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

extern "C" size_t mj_decode_workspace_bytes(const mj_decode_params* params) {
  if (check_params(params) != MJ_OK) return 0;
  return workspace_layout(*params).total;
}

extern "C" mj_status mj_kernel_name(const mj_decode_params* params, char* buf, int32_t len) {
  const mj_status st = check_params(params);
  if (st != MJ_OK) return st;
  if (!buf || len < 1) return MJ_ERR_INVALID_ARG;
  if (params->kv_format == MJ_KV_E4M3)
    std::snprintf(buf, static_cast<size_t>(len), "%s", choose_kernel(*params).name);
  else  // the KV format a narrow-pool launch reads, appended
    std::snprintf(buf, static_cast<size_t>(len), "%s_kv%s", choose_kernel(*params).name,
                  kv_format_name(params->kv_format));
  return MJ_OK;
}

extern "C" mj_status mj_decode_attn(const mj_decode_params* params, const mj_decode_args* args,
                                    mj_stream_t stream_) {
  mj_status st = check_params(params);
  if (st != MJ_OK) return st;
  if (!args) return MJ_ERR_INVALID_ARG;
  const mj_decode_params& p = *params;
  const mj_decode_args& a = *args;
  if (!a.q || !a.k || !a.v || !a.block_table || !a.seq_lens || !a.work || !a.n_splits || !a.q_descale ||
      !a.k_descale || !a.v_descale || !a.o || !a.lse)
    return MJ_ERR_INVALID_ARG;
  if (a.num_work < 1) return MJ_ERR_INVALID_ARG;
  const int64_t kv_strides[6] = {a.k_page, a.k_row, a.k_head, a.v_page, a.v_row, a.v_head};
  if (!kv_layout_ok(p, a.k, a.v, kv_strides) || !scales_ok(p, a)) return MJ_ERR_INVALID_ARG;
  const int q_bytes = p.q_dtype == MJ_E4M3 ? 1 : 2;
  if (!aligned16(a.q) || !aligned16(a.o)) return MJ_ERR_INVALID_ARG;
  if (a.q_seq_stride < 0 || ((a.q_seq_stride * q_bytes) & 15) != 0) return MJ_ERR_INVALID_ARG;
  if (a.o_seq_stride < 0 || ((a.o_seq_stride * 2) & 15) != 0) return MJ_ERR_INVALID_ARG;
  // one sequence's packed rows (h_k * n_q rows of d) must fit between two
  // sequences: a shorter O stride would make sequences overwrite each other
  const int64_t seq_elems = static_cast<int64_t>(p.h_k) * p.q_len * p.h_r * kHeadDim;
  if (p.num_seqs > 1 && (a.q_seq_stride < seq_elems || a.o_seq_stride < seq_elems)) return MJ_ERR_INVALID_ARG;
  const int64_t d_strides[6] = {a.qd_seq, a.qd_head, a.kd_seq, a.kd_head, a.vd_seq, a.vd_head};
  for (int64_t s : d_strides)
    if (s < 0) return MJ_ERR_INVALID_ARG;
  if (!(a.softmax_scale > 0.f) || !(a.scale_o == a.scale_o)) return MJ_ERR_INVALID_ARG;
  if (a.max_n_splits < 0 || a.max_n_splits > p.max_splits) return MJ_ERR_INVALID_ARG;
  const WorkspaceLayout ws = workspace_layout(p);
  if (ws.total > 0) {
    if (!a.workspace) return MJ_ERR_INVALID_ARG;
    if (a.workspace_bytes < ws.total) return MJ_ERR_CAPACITY;
    if ((reinterpret_cast<uintptr_t>(a.workspace) & (kAlign - 1)) != 0) return MJ_ERR_INVALID_ARG;
  }

  DecodeDev d{};
  d.q = a.q;
  d.q_seq = a.q_seq_stride;
  d.k = a.k;
  d.v = a.v;
  d.k_page = a.k_page;
  d.k_row = a.k_row;
  d.k_head = a.k_head;
  d.v_page = a.v_page;
  d.v_row = a.v_row;
  d.v_head = a.v_head;
  d.block_table = a.block_table;
  d.seq_lens = a.seq_lens;
  d.work = a.work;
  d.n_splits = a.n_splits;
  d.qd = a.q_descale;
  d.kd = a.k_descale;
  d.vd = a.v_descale;
  d.qd_seq = a.qd_seq;
  d.qd_head = a.qd_head;
  d.kd_seq = a.kd_seq;
  d.kd_head = a.kd_head;
  d.vd_seq = a.vd_seq;
  d.vd_head = a.vd_head;
  d.softmax_scale = a.softmax_scale;
  d.scale_o = a.scale_o;
  d.o = static_cast<__nv_bfloat16*>(a.o);
  d.o_seq = a.o_seq_stride;
  d.lse = a.lse;
  if (ws.total > 0) {
    char* base = static_cast<char*>(a.workspace);
    d.o_part = reinterpret_cast<float*>(base + ws.o_off);
    d.m_part = reinterpret_cast<float*>(base + ws.m_off);
    d.l_part = reinterpret_cast<float*>(base + ws.l_off);
  }
  d.status = a.status;
  d.num_seqs = p.num_seqs;
  d.h_k = p.h_k;
  d.n_q = p.q_len * p.h_r;
  d.q_len = p.q_len;
  d.h_r = p.h_r;
  d.page_size = p.page_size;
  d.max_blocks = p.max_blocks;
  d.causal = p.causal;
  d.max_splits = p.max_splits;
  d.num_work = a.num_work;
  d.num_pages = p.num_pages;
  d.l2_prefetch = p.l2_prefetch == 0 ? kDefaultL2Prefetch : (p.l2_prefetch < 0 ? 0 : p.l2_prefetch);
  d.kv_evict_first = p.kv_evict_first == 0 ? kDefaultKvEvictFirst : (p.kv_evict_first > 0 ? 1 : 0);
  d.kv_format = p.kv_format;
  d.ks = a.k_scales;
  d.vs = a.v_scales;
  d.ks_page = a.ks_page;
  d.ks_head = a.ks_head;
  d.vs_page = a.vs_page;
  d.vs_head = a.vs_head;

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  if (a.timing_events)
    for (int i = 0; i < 3; ++i) ev[i] = static_cast<cudaEvent_t>(a.timing_events[i]);

  const KernelChoice kc = choose_kernel(p);
  const int merge_splits = a.max_n_splits == 0 ? p.max_splits : a.max_n_splits;
  const bool merge = p.max_splits > 1 && merge_splits > 1;
  if (verbose())
    std::fprintf(stderr,
                 "mj_decode_attn: kernel=%s num_seqs=%d h_k=%d n_q=%d (q_len %d x h_r %d) page_size=%d %s "
                 "q=%s kv=%s work_items=%d merge=%s (max_n_splits %d of max_splits %d) kv_evict_first=%d\n",
                 kc.name, p.num_seqs, p.h_k, p.q_len * p.h_r, p.q_len, p.h_r, p.page_size,
                 p.causal ? "causal" : "non-causal", p.q_dtype == MJ_E4M3 ? "e4m3" : "bf16",
                 kv_format_name(p.kv_format), a.num_work, merge ? "yes" : "no", merge_splits, p.max_splits,
                 d.kv_evict_first);
  // an NVTX range around the launches, so a profiler's timeline names them
  nvtxRangePushA("mj_decode_attn");
  struct RangeEnd {
    ~RangeEnd() { nvtxRangePop(); }
  } range_end;
  cudaError_t e = cudaSuccess;
  if (ev[0] && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return MJ_ERR_CUDA;
  if (kc.kind == KernelKind::kTensorCoreQRows) {
    e = launch_decode_qm(d, kc.rows_per_cta, kc.n_q_tiles, p.q_dtype == MJ_E4M3, stream);
  } else if (kc.kind == KernelKind::kTensorCoreGrouped) {
    const int sms = device_sm_count();
    if (sms < 1) return MJ_ERR_CUDA;
    int* sched = reinterpret_cast<int*>(static_cast<char*>(a.workspace) + ws.sched_off);
    e = launch_decode_tcg(d, kc.heads_per_cta, kc.rows_per_cta, kc.n_q_tiles, p.q_dtype == MJ_E4M3, sched, sms,
                          stream);
  }
  else if (kc.kind == KernelKind::kTensorCore)
    e = launch_decode_tc(d, kc.rows_per_cta, kc.n_q_tiles, p.q_dtype == MJ_E4M3, stream);
  else
    e = launch_decode_cc(d, kc.rows_per_cta, kc.n_q_tiles, p.q_dtype == MJ_E4M3, stream);
  if (e != cudaSuccess) return MJ_ERR_CUDA;
  if (ev[1] && cudaEventRecord(ev[1], stream) != cudaSuccess) return MJ_ERR_CUDA;
  if (merge) {
    e = launch_merge(d, merge_splits, stream);
    if (e != cudaSuccess) return MJ_ERR_CUDA;
  }
  if (ev[2] && cudaEventRecord(ev[2], stream) != cudaSuccess) return MJ_ERR_CUDA;
  return MJ_OK;
}

namespace {

mj_status permute(const void* src, void* dst, int32_t elem_bytes, int32_t num_seqs, int32_t q_len,
                  int32_t h_k, int32_t h_r, int32_t head_dim, bool to_packed, mj_stream_t stream) {
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return MJ_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2) return MJ_ERR_INVALID_ARG;
  if (num_seqs < 1 || q_len < 1 || h_k < 1 || h_r < 1 || head_dim < 1) return MJ_ERR_INVALID_ARG;
  if ((head_dim * elem_bytes) % 16 != 0) return MJ_ERR_UNSUPPORTED;
  const char* s = static_cast<const char*>(src);
  const char* d = static_cast<const char*>(dst);
  const size_t bytes = static_cast<size_t>(num_seqs) * q_len * h_k * h_r * head_dim * elem_bytes;
  if (s < d + bytes && d < s + bytes) return MJ_ERR_INVALID_ARG;  // overlap
  const cudaError_t e = launch_permute_rows(src, dst, elem_bytes, num_seqs, q_len, h_k, h_r, head_dim,
                                            to_packed, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MJ_OK : MJ_ERR_CUDA;
}

}  // namespace

extern "C" mj_status mj_pack_q(const void* q_vllm, void* q_packed, int32_t elem_bytes, int32_t num_seqs,
                               int32_t q_len, int32_t h_k, int32_t h_r, int32_t head_dim,
                               mj_stream_t stream) {
  return permute(q_vllm, q_packed, elem_bytes, num_seqs, q_len, h_k, h_r, head_dim, true, stream);
}

extern "C" mj_status mj_check_gather_kv(const mj_decode_params* params, const mj_decode_args* args, int32_t values,
                                        uint8_t* out, int32_t out_rows, mj_stream_t stream) {
  const mj_status st = check_params(params);
  if (st != MJ_OK) return st;
  if (!args || !out || !aligned16(out) || out_rows < 1 || values < 0 || values > 1) return MJ_ERR_INVALID_ARG;
  const mj_decode_args& a = *args;
  if (!a.k || !a.v || !a.block_table || !a.seq_lens) return MJ_ERR_INVALID_ARG;
  const int64_t kv_strides[6] = {a.k_page, a.k_row, a.k_head, a.v_page, a.v_row, a.v_head};
  if (!kv_layout_ok(*params, a.k, a.v, kv_strides) || !scales_ok(*params, a)) return MJ_ERR_INVALID_ARG;
  DecodeDev d{};
  d.kv_format = params->kv_format;
  d.ks = a.k_scales;
  d.vs = a.v_scales;
  d.ks_page = a.ks_page;
  d.ks_head = a.ks_head;
  d.vs_page = a.vs_page;
  d.vs_head = a.vs_head;
  d.k = a.k;
  d.v = a.v;
  d.k_page = a.k_page;
  d.k_row = a.k_row;
  d.k_head = a.k_head;
  d.v_page = a.v_page;
  d.v_row = a.v_row;
  d.v_head = a.v_head;
  d.block_table = a.block_table;
  d.seq_lens = a.seq_lens;
  d.num_seqs = params->num_seqs;
  d.h_k = params->h_k;
  d.page_size = params->page_size;
  d.max_blocks = params->max_blocks;
  d.num_pages = params->num_pages;
  const cudaError_t e = launch_gather_kv(d, values != 0, out, out_rows, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MJ_OK : MJ_ERR_CUDA;
}

extern "C" mj_status mj_check_dequant_e4m3(float* out, mj_stream_t stream) {
  if (!out || (reinterpret_cast<uintptr_t>(out) & 15) != 0) return MJ_ERR_INVALID_ARG;
  return launch_dequant_e4m3(out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MJ_OK : MJ_ERR_CUDA;
}

extern "C" mj_status mj_check_bounded_wait(int32_t* status, int64_t* waited_ns, int32_t limit_us,
                                           mj_stream_t stream) {
  if (!status || (reinterpret_cast<uintptr_t>(status) & 3) != 0) return MJ_ERR_INVALID_ARG;
  if (waited_ns && (reinterpret_cast<uintptr_t>(waited_ns) & 7) != 0) return MJ_ERR_INVALID_ARG;
  if (limit_us < 1 || limit_us > 1000000) return MJ_ERR_INVALID_ARG;
  const cudaError_t e = launch_bounded_wait(status, waited_ns, static_cast<uint64_t>(limit_us) * 1000u,
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MJ_OK : MJ_ERR_CUDA;
}

namespace {

// Options as the device plan resolves them (0 -> the kernel's values, no model).
void resolve_device_opts(const mj_decode_params& p, mj_plan_opts* opts) {
  const KernelChoice kc = choose_kernel(p);
  if (opts->sm_count == 0) opts->sm_count = kDefaultSmCount;
  if (opts->ctas_per_sm == 0) opts->ctas_per_sm = kc.ctas_per_sm;
  if (opts->n_q_tiles == 0) opts->n_q_tiles = kc.n_q_tiles;
  if (opts->min_chunk_tiles == 0) opts->min_chunk_tiles = 1;
}

}  // namespace

extern "C" int32_t mj_decode_plan_max_items(const mj_decode_params* params, mj_plan_opts* opts) {
  if (check_params(params) != MJ_OK || !opts) return -1;
  if (opts->sm_count < 0 || opts->ctas_per_sm < 0 || opts->n_q_tiles < 0 || opts->force_splits < 0 ||
      opts->min_chunk_tiles < 0)
    return -1;
  resolve_device_opts(*params, opts);
  const int64_t b = params->num_seqs;
  if (opts->force_splits > 0) return static_cast<int32_t>(b * std::min(opts->force_splits, params->max_splits));
  const int64_t slots = std::max<int64_t>(
      1, static_cast<int64_t>(opts->sm_count) * opts->ctas_per_sm / (static_cast<int64_t>(params->h_k) * opts->n_q_tiles));
  // one wave's slots bound the chunks whenever the rule splits; otherwise
  // there is one item per sequence
  return static_cast<int32_t>(std::min<int64_t>(b * params->max_splits, std::max(b, slots)));
}

extern "C" mj_status mj_decode_plan_device(const mj_decode_params* params, mj_plan_opts* opts,
                                           const int32_t* seq_lens_dev, int32_t* work_dev, int32_t* n_splits_dev,
                                           int32_t* chunk_tiles_dev, int32_t* status_dev, mj_stream_t stream) {
  const mj_status st = check_params(params);
  if (st != MJ_OK) return st;
  if (!opts || !seq_lens_dev || !work_dev || !n_splits_dev) return MJ_ERR_INVALID_ARG;
  if (!aligned16(work_dev)) return MJ_ERR_INVALID_ARG;
  if (opts->sm_count < 0 || opts->ctas_per_sm < 0 || opts->n_q_tiles < 0 || opts->force_splits < 0 ||
      opts->min_chunk_tiles < 0 || opts->pad_to < 1)
    return MJ_ERR_INVALID_ARG;  // the work list has a fixed length: pad_to
  if (params->num_seqs > kMaxDevicePlanSeqs) return MJ_ERR_UNSUPPORTED;
  resolve_device_opts(*params, opts);
  const int64_t slots = std::max<int64_t>(
      1, static_cast<int64_t>(opts->sm_count) * opts->ctas_per_sm / (static_cast<int64_t>(params->h_k) * opts->n_q_tiles));
  const int64_t max_len = static_cast<int64_t>(params->max_blocks) * params->page_size;
  const cudaError_t e = launch_plan_device(seq_lens_dev, params->num_seqs, max_len, slots, params->max_splits,
                                           opts->force_splits, opts->min_chunk_tiles, opts->pad_to,
                                           reinterpret_cast<int4*>(work_dev), n_splits_dev, chunk_tiles_dev,
                                           status_dev, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MJ_OK : MJ_ERR_CUDA;
}

extern "C" mj_status mj_quantize_pack_q(const void* q_vllm, void* q_packed, float* q_descale, int32_t num_seqs,
                                        int32_t q_len, int32_t h_k, int32_t h_r, int32_t head_dim,
                                        mj_stream_t stream) {
  if (!q_vllm || !q_packed || !q_descale || !aligned16(q_vllm) || !aligned16(q_packed)) return MJ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_descale) & 3) != 0) return MJ_ERR_INVALID_ARG;
  if (num_seqs < 1 || q_len < 1 || h_k < 1 || h_r < 1 || head_dim < 1) return MJ_ERR_INVALID_ARG;
  if (head_dim % 16 != 0) return MJ_ERR_UNSUPPORTED;
  const int64_t elems = static_cast<int64_t>(num_seqs) * q_len * h_k * h_r * head_dim;
  if (static_cast<int64_t>(q_len) * h_r * head_dim > (int64_t{1} << 30) || elems > (int64_t{1} << 40))
    return MJ_ERR_UNSUPPORTED;
  const char* s = static_cast<const char*>(q_vllm);
  const char* d = static_cast<const char*>(q_packed);
  const char* f = reinterpret_cast<const char*>(q_descale);
  const size_t in_bytes = static_cast<size_t>(elems) * 2, out_bytes = static_cast<size_t>(elems);
  const size_t ds_bytes = static_cast<size_t>(num_seqs) * h_k * 4;
  if ((s < d + out_bytes && d < s + in_bytes) || (s < f + ds_bytes && f < s + in_bytes) ||
      (d < f + ds_bytes && f < d + out_bytes))
    return MJ_ERR_INVALID_ARG;  // overlap
  const cudaError_t e = launch_quantize_pack_q(q_vllm, q_packed, q_descale, num_seqs, q_len, h_k, h_r, head_dim,
                                               reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MJ_OK : MJ_ERR_CUDA;
}

extern "C" mj_status mj_unpack_o(const void* o_packed, void* o_vllm, int32_t num_seqs, int32_t q_len,
                                 int32_t h_k, int32_t h_r, int32_t head_dim, mj_stream_t stream) {
  return permute(o_packed, o_vllm, 2, num_seqs, q_len, h_k, h_r, head_dim, false, stream);
}
