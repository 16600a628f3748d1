/*
 * mj.h — C ABI of the paged fp8-KV split-KV decode attention library
 * (libmj.so, sm_103a / GB300).
 *
 * The operation (source: the "mjolnir/t5_decode.py" page — module docstring
 * on vLLM-shaped inputs and the causal tail; `plan_split_kv` for the plan;
 * the `decode` kernel's softmax/epilogue and the `reduction` kernel for the
 * split merge; `pack_q` / `unpack_o` for the query packing):
 *
 *   For each sequence b, kv head g and packed query row n (query token
 *   qi = n / h_r of query head h = g*h_r + n % h_r), with L = seq_lens[b]
 *   counting the q_len new tokens:
 *     visible keys   j <= L - q_len + qi (causal) or j <= L - 1 (non-causal)
 *     key/value j    K/V[block_table[b][j / page_size], j % page_size, g, :]
 *     z_j            = softmax_scale * qd[b,g] * kd[b,g] * <q_n, k_j>
 *     O[n]           = scale_o * vd[b,g] * sum_j softmax(z)_j * v_j   (bf16)
 *     LSE[n]         = log(sum_j exp(z_j))                  (natural log)
 *   A row with no visible key gets O = 0 and LSE = -inf.
 *
 * K and V are e4m3 (E4M3FN) codes; Q is bf16 or e4m3.  Scores, softmax and
 * accumulation are fp32.  The KV range of a sequence may be cut into
 * contiguous chunks (split-KV); split sequences are merged by a second
 * kernel that touches only them.
 *
 * Conventions for every entry point:
 *   - All tensors are caller-owned.  The library allocates nothing and keeps
 *     no state between calls.
 *   - "device" pointers must be valid on the current CUDA device; "host"
 *     pointers are ordinary CPU memory.
 *   - Strides are in ELEMENTS of the tensor they index, except the K/V
 *     strides, which are in bytes (equal to elements for e4m3 pools).  The
 *     head dimension is always contiguous.
 *   - Every function validates its arguments first and returns an error
 *     code without launching anything when they are bad.
 *   - Launch entry points enqueue on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and never synchronise the host, so they can be
 *     captured in a CUDA graph.
 */
#ifndef MJ_H_
#define MJ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without requiring the CUDA headers. */
typedef struct CUstream_st* mj_stream_t;

typedef enum {
  MJ_OK = 0,
  MJ_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad stride, bad shape */
  MJ_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels cover */
  MJ_ERR_CAPACITY = 3,    /* an output buffer or the workspace is too small */
  MJ_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  MJ_ERR_TIMEOUT = 5      /* written by a kernel into the status word */
} mj_status;

typedef enum { MJ_BF16 = 0, MJ_E4M3 = 1 } mj_dtype;

/* Problem shape and fixed choices.
 *   num_seqs    b >= 1
 *   q_len       query tokens per sequence (>= 1; > 1 for speculative verify)
 *   h_k, h_r    kv heads, query heads per kv head (n_q = q_len * h_r rows)
 *   head_dim    d; must be 128
 *   page_size   rows per KV page: 16, 32, 64 or 128
 *   max_blocks  row length of block_table
 *   num_pages   pages in the KV pool
 *   causal      1: causal tail; 0: every query token sees all L keys
 *   q_dtype     mj_dtype of Q (K/V are always e4m3)
 *   max_splits  partial slots per sequence, 1..256 (1 = never split)
 *   kernel      mj_kernel_pref: which decode kernel to run (0 = library's
 *               choice)
 *   l2_prefetch tensor-core kernel: KV tiles its producer pulls into L2
 *               ahead of the shared-memory loads (source: the kernel's
 *               `l2_prefetch` option on the "mjolnir/t5_decode.py" page);
 *               0 = library default, -1 = off, 1..8 = distance in tiles
 *   kv_evict_first
 *               the tensor-core kernels' K/V tile loads carry an L2
 *               EVICT_FIRST cache policy (KV is read once; source: the
 *               kernel's `kv_evict_first` option on the
 *               "mjolnir/t5_decode.py" page); 0 = library default (on),
 *               -1 = off, 1 = on; results are identical either way
 *   kv_format   mj_kv_format of the K/V pools (0 = e4m3) */
typedef struct {
  int32_t num_seqs, q_len, h_k, h_r, head_dim, page_size;
  int32_t max_blocks, num_pages, causal, q_dtype, max_splits, kernel;
  int32_t l2_prefetch, kv_evict_first, kv_format;
} mj_decode_params;

/* Element format of the K and V pools (source: the KV-format constants and
 * the narrow-format helpers of the "mjolnir/t5_decode.py" page).  Every
 * format is sign | exponent | mantissa with a bias and a subnormal binade;
 * the narrow ones have no infinities or NaN:
 *   MJ_KV_E4M3  8 bits, E4M3FN (bias 7, largest 448), one code per byte
 *   MJ_KV_E3M2  6 bits (bias 3, largest 28)
 *   MJ_KV_E2M3  6 bits (bias 1, largest 7.5)
 *   MJ_KV_E2M1  4 bits (bias 1, largest 6)
 * A row of one kv head is d codes packed little-endian into d*bits/8 bytes:
 * bit k of element i is bit (bits*i + k) % 8 of byte (bits*i + k) / 8 (fp4:
 * element 2i in the low nibble of byte i; fp6: four elements in three
 * bytes).  Every value of the narrow formats is an e4m3 value, so the
 * operation is unchanged; the tensor-core kernels feed the codes to the MMA
 * as they are (the TMA spreads each 16-element group over 16 bytes of
 * shared memory).  Narrow formats need kernel MJ_KERNEL_AUTO,
 * MJ_KERNEL_TENSOR_CORE or MJ_KERNEL_TENSOR_CORE_QROWS, K/V base pointers
 * 32-byte aligned and K/V strides multiples of 32 bytes.
 *   MJ_KV_NVFP4 e2m1 codes packed as MJ_KV_E2M1 (64 bytes a row) plus one
 *               e4m3 scale per 16 consecutive elements of a row, held in a
 *               separate scale plane (mj_decode_args.k_scales / v_scales):
 *               the 8 scales of a row are 8 consecutive bytes and the rows of
 *               one (page, head) follow each other, page_size * 8 bytes
 *               (layout (page, head, row, group)).  The value the operation
 *               uses is e4m3(code * scale * 2^-3), rounded to nearest even
 *               (the page's nvfp4 kernel value); the kernel converts each
 *               group in shared memory before the MMA.  Needs e4m3 Q,
 *               q_len*h_r <= 32 and MJ_KERNEL_AUTO or MJ_KERNEL_TENSOR_CORE;
 *               code strides are 16-byte multiples. */
typedef enum { MJ_KV_E4M3 = 0, MJ_KV_E3M2 = 1, MJ_KV_E2M3 = 2, MJ_KV_E2M1 = 3, MJ_KV_NVFP4 = 4 } mj_kv_format;

/* Decode kernel families.  Both compute the same function; the choice only
 * changes speed (and last-bit rounding).
 *   MJ_KERNEL_AUTO         the library's choice for the shape
 *   MJ_KERNEL_CUDA_CORE    fp32 CUDA-core kernel, exact e4m3 dequant in
 *                          registers, fp32 P
 *   MJ_KERNEL_TENSOR_CORE  tcgen05 swap-AB kernel: e4m3 K/V tiles straight
 *                          from TMA into the MMA, Q and P as hi+lo e4m3;
 *                          one CTA per kv head
 *   MJ_KERNEL_TENSOR_CORE_GROUPED
 *                          the same arithmetic, persistent, with one CTA per
 *                          SM taking units of 8, 4, 2 or 1 kv heads, whose
 *                          rows of each page it reads together: 8 heads for
 *                          q_len*h_r <= 4 (h_k a multiple of 8), 4 for <= 8
 *                          (h_k a multiple of 4), 2 for <= 32 (h_k even),
 *                          1 for <= 32 (any h_k); MJ_ERR_UNSUPPORTED above
 *                          32 rows
 *   MJ_KERNEL_TENSOR_CORE_QROWS
 *                          tcgen05 kernel with 128 query rows on the MMA's M
 *                          and 128 keys on N: one read of the KV per q tile
 *                          of 128 packed rows, or of 64 / 32 packed rows
 *                          each held two / four times with every copy taking
 *                          that share of the keys; above 128 rows one CTA
 *                          takes two q tiles, so the KV is read once per
 *                          256 rows; MJ_KERNEL_AUTO takes it for
 *                          q_len*h_r > 16 */
typedef enum {
  MJ_KERNEL_AUTO = 0,
  MJ_KERNEL_CUDA_CORE = 1,
  MJ_KERNEL_TENSOR_CORE = 2,
  MJ_KERNEL_TENSOR_CORE_GROUPED = 3,
  MJ_KERNEL_TENSOR_CORE_QROWS = 4
} mj_kernel_pref;

/* Plan knobs (source: `plan_split_kv`).  A field left 0 takes the
 * library's value for the kernel mj_decode_attn will launch for these
 * params, and is filled in on return, so a caller can reproduce the plan:
 *   sm_count         SMs of the target GPU (0 -> 152, a GB300)
 *   ctas_per_sm      (decode CTA, kv head) slots per SM.  0 -> the
 *                    library's choice: for the per-head kernels the
 *                    co-resident pairs (CTAs per SM), or 5/3, 8/3 or 4
 *                    times that when a model of the greedy longest-first
 *                    schedule says the finer plan ends at least 5 % sooner;
 *                    for the persistent head-grouped kernel its units per
 *                    SM times the heads one unit serves
 *   n_q_tiles        CTAs per (work item, kv head) along the packed rows
 *   force_splits     > 0: cut every sequence into this many chunks
 *   min_chunk_tiles  lower bound of the chunk size in 128-row tiles (0 -> 1)
 *   pad_to           > 0: pad the work list with empty items to this length */
typedef struct {
  int32_t sm_count, ctas_per_sm, n_q_tiles, force_splits, min_chunk_tiles, pad_to;
} mj_plan_opts;

/* Occupancy-pinned split-KV plan (host only; no CUDA call; deterministic).
 *
 * Every sequence has T_b = max(1, ceil(L_b / 128)) tiles of 128 KV rows.
 * One wave holds slots = max(1, sm_count*ctas_per_sm / (h_k*n_q_tiles))
 * work items.  The chunk size is the smallest number of tiles, at least
 * max(min_chunk_tiles, ceil(T_max / max_splits)), whose chunk count over
 * all sequences fits one wave (force_splits > 0 takes
 * max(that floor, ceil(T_max / force_splits)); a batch that already fills
 * the wave, or max_splits == 1, is not split).  Items are ordered longest
 * first, ties in (b, slot) order.
 *
 *   seq_lens_host  host int32[num_seqs]; 0 <= L_b <= max_blocks*page_size
 *   work_out       host int32[work_cap][4]: (seq, tile_begin, tile_end,
 *                  split_slot); padding items are (0, 0, 0, 0)
 *   num_work       host out: items written
 *   n_splits_out   host int32[num_seqs]: chunks per sequence
 *   chunk_tiles    host out (may be NULL)
 * Errors: MJ_ERR_INVALID_ARG (nulls, bad params, a length out of range,
 * pad_to below the item count), MJ_ERR_CAPACITY (work_cap too small). */
mj_status mj_decode_plan(const mj_decode_params* params, mj_plan_opts* opts,
                         const int32_t* seq_lens_host, int32_t* work_out, int32_t work_cap,
                         int32_t* num_work, int32_t* n_splits_out, int32_t* chunk_tiles);

/* Bytes of workspace mj_decode_attn needs: fp32 partial O, max and sum for
 * max_splits slots of every (seq, kv head, row); 0 when max_splits == 1.
 * Layout (private): o[b][g][slot][n][d], then m and l [b][g][slot][n]. */
size_t mj_decode_workspace_bytes(const mj_decode_params* params);

/* Device-side arguments of mj_decode_attn.
 *   q            device, packed (b, h_k, n_q, d) rows of q_dtype; row n of
 *                kv head g of sequence b at q + b*q_seq_stride + (g*n_q+n)*d
 *                (for q_len == 1 vLLM's (b, h_q, d) is already packed);
 *                with num_seqs > 1, q_seq_stride and o_seq_stride are at
 *                least h_k*n_q*d (MJ_ERR_INVALID_ARG otherwise)
 *   k, v         device pools of kv_format codes; the row of (page, r, g)
 *                starts at byte page*x_page + r*x_row + g*x_head, and holds
 *                d codes (d*bits/8 bytes, packed as mj_kv_format says);
 *                strides are in BYTES, each a multiple of 16 (of 32 for the
 *                narrow formats); K and V may share one buffer
 *   block_table  device int32 (b, max_blocks); entries past ceil(L/PS) are
 *                never read; entries before must be in [0, num_pages)
 *   seq_lens     device int32[b], the same values the plan saw
 *   work, n_splits, num_work   device copies of the plan's outputs
 *   *_descale    device fp32, (b, g) at b*x_seq + g*x_head (strides 0 =
 *                per tensor); finite and > 0
 *   o            device bf16, packed like q with o_seq_stride
 *   lse          device fp32 (b, h_k, n_q), contiguous
 *   workspace    device, >= mj_decode_workspace_bytes; need not be
 *                initialised; may be NULL only when that size is 0
 *                (max_splits == 1 and a kernel other than the head-grouped
 *                one, which keeps its unit counter there)
 *   status       optional device int32, caller-zeroed; kernels that give up
 *                a bounded wait write MJ_ERR_TIMEOUT there, and the merge
 *                writes MJ_ERR_INVALID_ARG for a sequence whose n_splits
 *                exceeds max_n_splits or max_splits (that sequence's O and
 *                LSE rows are then not written); NULL = off
 *   max_n_splits host hint: the plan's largest n_splits (1 = nothing was
 *                split: the merge kernel is not launched; it also sizes the
 *                merge); 0 = unknown (the merge runs, sized for max_splits).
 *                A sequence with more splits than the hint is refused by the
 *                merge (see status), never merged in part.
 *   timing_events optional: NULL, or 3 cudaEvent_t recorded on `stream`
 *                before the decode kernel, between decode and merge, and
 *                after the merge (instrumentation only)
 *   k_scales, v_scales
 *                MJ_KV_NVFP4 only (ignored otherwise): device e4m3 scale
 *                planes, 16-byte aligned; the 8 scales of row r of (page, g)
 *                at page*x_page + g*x_head + r*8 (bytes; both strides
 *                multiples of 16) */
typedef struct {
  const void* q;
  int64_t q_seq_stride;
  const uint8_t* k;
  const uint8_t* v;
  int64_t k_page, k_row, k_head, v_page, v_row, v_head;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* work;
  const int32_t* n_splits;
  int32_t num_work;
  const float* q_descale;
  const float* k_descale;
  const float* v_descale;
  int64_t qd_seq, qd_head, kd_seq, kd_head, vd_seq, vd_head;
  float softmax_scale, scale_o;
  void* o;
  int64_t o_seq_stride;
  float* lse;
  void* workspace;
  size_t workspace_bytes;
  int32_t* status;
  int32_t max_n_splits;
  void* const* timing_events;
  const uint8_t* k_scales;
  const uint8_t* v_scales;
  int64_t ks_page, ks_head, vs_page, vs_head;
} mj_decode_args;

/* Decode attention for one step: the decode kernel over every work item,
 * then, if any sequence was split (max_splits > 1), the merge kernel over
 * the split sequences.  Writes O and LSE of every (b, g, n).  Deterministic:
 * repeated calls give identical bytes.
 * Errors: MJ_ERR_INVALID_ARG, MJ_ERR_UNSUPPORTED (head_dim != 128, bad
 * page size, q_dtype), MJ_ERR_CAPACITY (workspace), MJ_ERR_CUDA. */
mj_status mj_decode_attn(const mj_decode_params* params, const mj_decode_args* args,
                         mj_stream_t stream);

/* Size of the fixed device scratch behind mj_decode_attn_static_ws. */
#define MJ_STATIC_WORKSPACE_BYTES ((size_t)32 << 20)

/* Same as mj_decode_attn, but without a caller workspace: the split partials
 * go to a fixed MJ_STATIC_WORKSPACE_BYTES device array inside the library,
 * so the call allocates nothing.  (The source pages have no counterpart;
 * this serves callers that may not allocate device memory at call time, such
 * as runtimes that give the whole device to their own arena or plugins in a
 * framework that owns the allocator.)
 *   - args->workspace / workspace_bytes are ignored; everything else is as
 *     for mj_decode_attn.
 *   - Problems whose mj_decode_workspace_bytes exceeds the array return
 *     MJ_ERR_CAPACITY before anything is launched.
 *   - The array is looked up once per device, on the first call made with
 *     that device current; make that first call before any stream capture.
 *   - Every call on a device shares the one array and nothing in it needs to
 *     start at zero (every partial is written before it is read); calls whose
 *     kernels overlap on the GPU (different streams without ordering) race on
 *     it and must be serialised by the caller.
 *   - Each GPU that loads the library keeps the array until the process
 *     exits. */
mj_status mj_decode_attn_static_ws(const mj_decode_params* params, const mj_decode_args* args,
                                   mj_stream_t stream);

/* vLLM query layout (num_seqs*q_len, h_k*h_r, d) -> packed (num_seqs, h_k,
 * q_len*h_r, d), row n = qi*h_r + hr (source: `pack_q`).  Both device,
 * contiguous, must not overlap; elem_bytes is 2 (bf16) or 1 (e4m3). */
mj_status mj_pack_q(const void* q_vllm, void* q_packed, int32_t elem_bytes, int32_t num_seqs,
                    int32_t q_len, int32_t h_k, int32_t h_r, int32_t head_dim, mj_stream_t stream);

/* The plan of mj_decode_plan computed on the device from device sequence
 * lengths, so that plan, decode and merge can be captured in one CUDA graph
 * and replayed while the lengths change (source: `plan_split_kv`; the
 * paged-decode page's schedule kernel plans on the device for the same
 * reason).  The rule and the item order are mj_decode_plan's, for the
 * options given; no model picks ctas_per_sm here (0 takes the kernel's
 * co-resident CTAs), so pass the options a host plan reported to reproduce
 * it.  The work list always has opts->pad_to rows: items, then (0,0,0,0)
 * padding; launch mj_decode_attn with num_work = pad_to and max_n_splits =
 * max_splits.
 *   opts            in/out as for mj_decode_plan; pad_to >= 1 is required
 *   seq_lens_dev    device int32[num_seqs], 0 <= L_b <= max_blocks*page_size
 *   work_dev        device int32[pad_to][4], 16-byte aligned
 *   n_splits_dev    device int32[num_seqs]
 *   chunk_tiles_dev device int32, may be NULL
 *   status_dev      device int32, may be NULL; caller-zeroed; receives
 *                   MJ_ERR_INVALID_ARG (a length out of range, more splits
 *                   than max_splits) or MJ_ERR_CAPACITY (more items than
 *                   pad_to), in which case the outputs are unspecified (every
 *                   write stays inside the buffers)
 * One single-CTA kernel on `stream`; no host sync.  Errors returned at once:
 * MJ_ERR_INVALID_ARG (params, nulls, alignment, pad_to < 1),
 * MJ_ERR_UNSUPPORTED (num_seqs > 16384), MJ_ERR_CUDA (launch). */
mj_status mj_decode_plan_device(const mj_decode_params* params, mj_plan_opts* opts, const int32_t* seq_lens_dev,
                                int32_t* work_dev, int32_t* n_splits_dev, int32_t* chunk_tiles_dev,
                                int32_t* status_dev, mj_stream_t stream);

/* The most work items the plan rule makes for these params and options,
 * whatever the sequence lengths (host only): with force_splits = 0 at most
 * max(num_seqs, slots) (the rule splits only to fill one wave of slots),
 * else num_seqs * min(force_splits, max_splits).  The tightest pad_to for
 * mj_decode_plan_device: padding items are launched as CTAs that exit at
 * once, so a loose pad_to costs launch time.  Fills opts' zero fields as
 * mj_decode_plan_device does; returns -1 for invalid params or options. */
int32_t mj_decode_plan_max_items(const mj_decode_params* params, mj_plan_opts* opts);

/* The preconditions mj_decode_attn cannot check cheaply (it reads device
 * memory it does not validate), checked on host copies for debugging: for
 * every sequence b, 0 <= L_b <= max_blocks*page_size, the block-table
 * entries of its first ceil(L_b / page_size) pages are in [0, num_pages)
 * (entries past them may hold anything), and q/k/v descales of every kv
 * head are finite and positive (the kernels take the raw-score maximum
 * before scaling).  block_table_host is [num_seqs][max_blocks]; descales
 * are indexed [b*d_seq + g*d_head] as in mj_decode_args.  Returns MJ_OK, or
 * MJ_ERR_INVALID_ARG with *bad_seq (optional) set to the first offending
 * sequence (-1 when the arguments themselves are invalid).  Host only. */
mj_status mj_check_preconditions(const mj_decode_params* params, const int32_t* block_table_host,
                                 const int32_t* seq_lens_host, const float* q_descale, const float* k_descale,
                                 const float* v_descale, int64_t qd_seq, int64_t qd_head, int64_t kd_seq,
                                 int64_t kd_head, int64_t vd_seq, int64_t vd_head, int32_t* bad_seq);

/* Verification hooks (not needed to compute anything): the decode path's
 * page gather and the CUDA-core kernel's e4m3 conversion as standalone
 * launches, for byte- and bit-exact comparison with a reference.
 *
 * mj_check_gather_kv: for every sequence b and kv head g, K (values = 0) or
 * V (values = 1) rows 0 .. L_b - 1 fetched exactly as the tensor-core
 * decode kernels fetch them (the same tensor maps over the caller's
 * strides, the same block-table lookup and TMA boxes), written densely:
 *   out[(b*h_k + g)*out_rows + row][0..127] for row < min(L_b, out_rows)
 * (device, 16-byte aligned; other rows are left as they were).  args'
 * k, v, strides, block_table and seq_lens are read; the rest is ignored.
 * mj_check_dequant_e4m3: out[c] = the fp32 value the CUDA-core kernel gives
 * e4m3 code c, c = 0..255 (device, 16-byte aligned; NaN codes give NaN).
 * Errors: MJ_ERR_INVALID_ARG, MJ_ERR_UNSUPPORTED (params), MJ_ERR_CUDA. */
mj_status mj_check_gather_kv(const mj_decode_params* params, const mj_decode_args* args, int32_t values,
                             uint8_t* out, int32_t out_rows, mj_stream_t stream);
mj_status mj_check_dequant_e4m3(float* out, mj_stream_t stream);

/* Verification hook of the kernels' bounded waits (every mbarrier wait in
 * the decode kernels gives up after a time limit, sets MJ_ERR_TIMEOUT in the
 * status word and lets the CTA drain and exit, so a lost copy or MMA cannot
 * hang the GPU).  One warp waits on an mbarrier that nothing ever completes,
 * with the same primitive and a limit of limit_us microseconds, then writes
 * MJ_ERR_TIMEOUT to *status and the nanoseconds it waited to *waited_ns.
 *   status     device int32 (caller-zeroed)
 *   waited_ns  device int64, 8-byte aligned, or NULL
 *   limit_us   1 .. 1000000
 * No counterpart on the pages (their kernel's waits have no limit).
 * Errors: MJ_ERR_INVALID_ARG, MJ_ERR_CUDA (launch). */
mj_status mj_check_bounded_wait(int32_t* status, int64_t* waited_ns, int32_t limit_us, mj_stream_t stream);

/* Fused fp8 query quantisation and pack (source: `quantize_q_fp8` and
 * `pack_q`).  For every sequence b and kv head g the group is Q's q_len
 * tokens x h_r heads x d values of that kv head;
 *   q_descale[b*h_k + g] = max(amax_group |q|, 1e-6) / 448   (fp32)
 *   q_packed[b][g][qi*h_r + hr][:] = e4m3(q / q_descale[b*h_k + g])
 * with IEEE fp32 division and e4m3 rounding to nearest even, saturating at
 * +-448.  The outputs feed mj_decode_attn with q_dtype MJ_E4M3 and
 * q_descale strides (qd_seq, qd_head) = (h_k, 1).
 *   q_vllm     device bf16 (num_seqs*q_len, h_k*h_r, head_dim), contiguous,
 *              16-byte aligned, finite values
 *   q_packed   device e4m3 (num_seqs, h_k, q_len*h_r, head_dim), 16-byte
 *              aligned
 *   q_descale  device fp32 (num_seqs, h_k)
 *   head_dim   a multiple of 16
 * The three buffers must not overlap.  One kernel launch on `stream`; no
 * host sync.  Errors: MJ_ERR_INVALID_ARG (nulls, alignment, sizes,
 * overlap), MJ_ERR_UNSUPPORTED (head_dim, a group over 2^30 values),
 * MJ_ERR_CUDA (launch). */
mj_status mj_quantize_pack_q(const void* q_vllm, void* q_packed, float* q_descale, int32_t num_seqs,
                             int32_t q_len, int32_t h_k, int32_t h_r, int32_t head_dim, mj_stream_t stream);

/* Inverse permutation for the bf16 output (source: `unpack_o`). */
mj_status mj_unpack_o(const void* o_packed, void* o_vllm, int32_t num_seqs, int32_t q_len,
                      int32_t h_k, int32_t h_r, int32_t head_dim, mj_stream_t stream);

/* Static text for a status code. */
const char* mj_status_string(mj_status status);

/* Which kernel mj_decode_attn runs for these params: writes a short name
 * (e.g. "cc_n4_bf16") into buf (NUL-terminated, truncated to len). */
mj_status mj_kernel_name(const mj_decode_params* params, char* buf, int32_t len);

#ifdef __cplusplus
}
#endif

#endif /* MJ_H_ */
