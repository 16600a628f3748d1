// Host-side internals shared by the plan, the validation and the launchers.
#pragma once

#include <cstdint>

#include "mj.h"

namespace mj {

constexpr int kTileRows = 128;  // plan unit: KV rows per tile
constexpr int kHeadDim = 128;
constexpr int kMaxSplits = 256;
constexpr int kDefaultSmCount = 152;  // GB300
constexpr int kMaxDevicePlanSeqs = 16384;  // device plan: one CTA, keys and tiles in shared memory

enum class KernelKind { kCudaCore = 0, kTensorCore = 1, kTensorCoreGrouped = 2, kTensorCoreQRows = 3 };

// The decode kernel mj_decode_attn launches for a problem, and the
// occupancy facts the plan needs about it.
struct KernelChoice {
  KernelKind kind;
  int rows_per_cta;  // packed query rows one CTA covers (per kv head)
  int heads_per_cta; // kv heads one CTA covers
  int n_q_tiles;     // CTAs along the packed rows
  int ctas_per_sm;   // co-resident (CTA, kv head) pairs per SM
  const char* name;
};

// Shape of the head-grouped tensor-core kernel for (h_k, n_q): kv heads per
// CTA and packed rows per head; false when no instance fits.
bool tcg_supported(int h_k, int n_q, int* heads_per_cta, int* rows_per_head);

// Validates the shape fields every entry point shares.
mj_status check_params(const mj_decode_params* p);

// Kernel choice for valid params.
KernelChoice choose_kernel(const mj_decode_params& p);

// MJ_VERBOSE set to a non-empty value other than "0" in the environment
// (read once per process): the entry points print what they chose to stderr.
bool verbose();

}  // namespace mj
