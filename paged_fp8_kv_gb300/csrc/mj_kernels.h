// Launchers of the device kernels (host-callable, defined in the .cu files).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <utility>

#include "mj_device.cuh"

namespace mj {

// Launches kern as a programmatic dependent of the work before it in the
// stream: its CTAs may become resident once every CTA of the previous grid
// has called griddep_launch_dependents (or exited), hiding the launch under
// that grid's tail.  Every kernel launched this way calls griddep_wait in
// every CTA before its first global load or store and before it exits, so
// each kernel of a chain still starts its memory work after the one before
// it has completed, and so transitively after all earlier ones.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

constexpr int kHeadDimDev = 128;
constexpr int kTileRowsDev = 128;

// CUDA-core decode (rows_per_cta in {4, 8, 16}).
cudaError_t launch_decode_cc(const DecodeDev& a, int rows_per_cta, int n_q_tiles, bool q_e4m3,
                             cudaStream_t stream);
int cc_smem_bytes(int rows_per_cta);

// Tensor-core (tcgen05) decode (rows_per_cta in {8, 16, 32}).
cudaError_t launch_decode_tc(const DecodeDev& a, int rows_per_cta, int n_q_tiles, bool q_e4m3,
                             cudaStream_t stream);
// nvfp4 pools (a.kv_format 4) run instances with a converter warpgroup.
int tc_smem_bytes(int rows_per_cta, bool q_e4m3, bool nvfp4 = false);
int tc_min_blocks(int rows_per_cta, bool q_e4m3, bool nvfp4 = false);  // co-resident CTAs per SM the kernel is built for

// Head-grouped tensor-core decode: one CTA serves heads_per_cta kv heads
// (rows_per_head packed query rows each); tcg_supported picks the shape.
// Persistent: min(units, sm_count) CTAs take units from the counter at
// `sched` (device memory, zeroed by the launch in the stream).
cudaError_t launch_decode_tcg(const DecodeDev& a, int heads_per_cta, int rows_per_head, int n_q_tiles, bool q_e4m3,
                              int* sched, int sm_count, cudaStream_t stream);
int tcg_smem_bytes(int heads_per_cta, int rows_per_head, bool q_e4m3);

// Query-rows-on-M tensor-core decode: 128 packed rows of one kv head per
// CTA, one CTA per SM.
// rows_per_cta 128, 64 or 32: each packed row held 128 / rows_per_cta times,
// every copy taking that share of a tile's keys.
cudaError_t launch_decode_qm(const DecodeDev& a, int rows_per_cta, int n_q_tiles, bool q_e4m3,
                             cudaStream_t stream);
int qm_smem_bytes(bool q_e4m3);

// TMA descriptor of a paged e4m3 pool seen as (d bytes, rows in page, kv
// heads, pages); one box is box_rows rows of box_heads heads (head-major in
// shared memory), 128-byte swizzle.
// Strides are in bytes.  kv_format picks the element type: e4m3 codes are
// bytes; the narrow formats are read packed (16 codes in 8 or 12 bytes) and
// land 16 codes per 16 bytes of shared memory, the operand form of the
// kind::f8f6f4 MMA.
bool make_kv_map(CUtensorMap* m, const uint8_t* base, int page_size, int h_k, int num_pages, int64_t s_row,
                 int64_t s_head, int64_t s_page, int box_rows, int box_heads, int kv_format);

// Merge of split sequences' partials into O / LSE; max_n_splits (> 1) sizes
// the number of warps that share one row.
cudaError_t launch_merge(const DecodeDev& a, int max_n_splits, cudaStream_t stream);

// Layout permutations (vLLM <-> packed rows).
cudaError_t launch_gather_kv(const DecodeDev& a, bool values, uint8_t* out, int out_rows, cudaStream_t stream);
cudaError_t launch_dequant_e4m3(float* out, cudaStream_t stream);
cudaError_t launch_bounded_wait(int32_t* status, int64_t* waited_ns, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_plan_device(const int32_t* seq_lens, int num_seqs, int64_t max_len, int64_t slots,
                               int max_splits, int force_splits, int min_chunk, int pad_to, int4* work,
                               int32_t* n_splits, int32_t* chunk_out, int32_t* status, cudaStream_t stream);
cudaError_t launch_quantize_pack_q(const void* q_vllm, void* q_packed, float* q_descale, int num_seqs, int q_len,
                                   int h_k, int h_r, int head_dim, cudaStream_t stream);
cudaError_t launch_permute_rows(const void* src, void* dst, int elem_bytes, int num_seqs, int q_len,
                                int h_k, int h_r, int head_dim, bool to_packed, cudaStream_t stream);

}  // namespace mj
