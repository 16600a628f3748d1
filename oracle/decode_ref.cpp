// Plain fp64 CPU oracle for paged fp8-KV decode attention.
//
// TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the benchmark's
// CPU-baseline / reference legs may load this library.  The CUDA library never
// links, includes or calls it, and it shares no code with the CUDA path.
//
// What it computes is the plain definition of softmax attention over a paged
// cache, written out without blocking, fusion or reordering (sources: the
// "mjolnir/t5_decode.py" page, module docstring on the vLLM-shaped inputs,
// `emulate_decode` for the exact fp32 attention it also returns, and the
// kernel's epilogue for the LSE convention):
//
//   for sequence b, kv head g, packed row n (query token qi = n / h_r):
//     last visible key   lim = L - q_len + qi   (causal)   or   L - 1
//     key j              K[block_table[b][j / PS], j % PS, g, :]
//     logit              z_j = softmax_scale * qd[b,g] * kd[b,g] * <q_n, k_j>
//     M = max_j z_j,  l = sum_j exp(z_j - M)
//     O[d]  = scale_o * vd[b,g] * sum_j exp(z_j - M) * v_j[d] / l
//     LSE   = M + ln l                                   (natural log)
//   A row that sees no key gets O = 0 and LSE = -inf.
//
// Input values are decoded exactly: bf16 by widening its bits, e4m3 (the
// E4M3FN variant: no infinities, S.1111.111 is NaN, largest finite 448) from
// its bit fields.  Everything after decoding is fp64.
//
// Parity pins: tests/test_oracle.py checks this file against the e4m3 values
// torch's float8_e4m3fn decodes, closed forms (one key, identical keys,
// one-hot dominance), brute-force mask enumeration, a Decimal log-sum-exp on
// tiny inputs, split-then-merge against the direct sum, and page-permutation
// invariance.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#include <atomic>

namespace {

// ---------------------------------------------------------------- decoding

// E4M3FN value of one byte, from the format definition: 1 sign bit, 4
// exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
// (m / 8) * 2^-6; exponent 15 with mantissa 7 is NaN (no infinities).
double e4m3_value(uint8_t code) {
  const int sign = code >> 7;
  const int e = (code >> 3) & 0xF;
  const int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  if (e == 0)
    mag = std::ldexp(static_cast<double>(m) / 8.0, -6);
  else
    mag = std::ldexp(1.0 + static_cast<double>(m) / 8.0, e - 7);
  return sign ? -mag : mag;
}

struct E4M3Table {
  double v[256];
  E4M3Table() {
    for (int c = 0; c < 256; ++c) v[c] = e4m3_value(static_cast<uint8_t>(c));
  }
};
const E4M3Table kE4M3;

// bf16 is the upper half of an IEEE binary32; widening is exact.
double bf16_value(uint16_t bits) {
  uint32_t w = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &w, sizeof(f));
  return static_cast<double>(f);
}

}  // namespace

extern "C" {

// Problem description.  All strides are in elements of the tensor they index.
//   q : vLLM layout (num_seqs * q_len, h_q, d); element (b, qi, h, i) at
//       b*q_seq + qi*q_tok + h*q_head + i, where packed row n of kv head g is
//       query token qi = n / h_r of query head h = g*h_r + n % h_r; bf16 bits
//       (q_is_e4m3 = 0) or e4m3 codes (q_is_e4m3 = 1)
//   k/v : e4m3 codes, element (page, r, g, i) at
//         page*x_page + r*x_row + g*x_head + i
//   descales : fp32, (b, g) at b*x_seq + g*x_head (stride 0 = broadcast)
typedef struct {
  int32_t num_seqs, q_len, h_k, h_r, head_dim, page_size, max_blocks;
  int32_t causal, q_is_e4m3;
  double softmax_scale, scale_o;
  int64_t q_seq, q_tok, q_head;
  int64_t k_page, k_row, k_head, v_page, v_row, v_head;
  int64_t qd_seq, qd_head, kd_seq, kd_head, vd_seq, vd_head;
} oracle_problem;

double oracle_e4m3_value(uint8_t code) { return kE4M3.v[code]; }
double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }

}  // extern "C"

namespace {

struct View {
  const oracle_problem* p;
  const void* q;
  const uint8_t* k;
  const uint8_t* v;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const float* qd;
  const float* kd;
  const float* vd;

  int n_q() const { return p->q_len * p->h_r; }

  double q_at(int b, int g, int n, int i) const {
    const int qi = n / p->h_r;
    const int h = g * p->h_r + n % p->h_r;
    const int64_t off = b * p->q_seq + qi * p->q_tok + static_cast<int64_t>(h) * p->q_head + i;
    if (p->q_is_e4m3) return kE4M3.v[static_cast<const uint8_t*>(q)[off]];
    return bf16_value(static_cast<const uint16_t*>(q)[off]);
  }
  // Byte offset of key/value row j of sequence b, head g.
  int64_t row_off(int b, int j, int g, int64_t x_page, int64_t x_row, int64_t x_head) const {
    const int32_t page = block_table[static_cast<int64_t>(b) * p->max_blocks + j / p->page_size];
    return page * x_page + static_cast<int64_t>(j % p->page_size) * x_row + g * x_head;
  }
  double k_at(int b, int j, int g, int i) const {
    return kE4M3.v[k[row_off(b, j, g, p->k_page, p->k_row, p->k_head) + i]];
  }
  double v_at(int b, int j, int g, int i) const {
    return kE4M3.v[v[row_off(b, j, g, p->v_page, p->v_row, p->v_head) + i]];
  }
  double qd_at(int b, int g) const { return qd[b * p->qd_seq + g * p->qd_head]; }
  double kd_at(int b, int g) const { return kd[b * p->kd_seq + g * p->kd_head]; }
  double vd_at(int b, int g) const { return vd[b * p->vd_seq + g * p->vd_head]; }

  // Index of the last key row n may see (may be negative: sees nothing).
  int64_t last_visible(int b, int n) const {
    const int64_t L = seq_lens[b];
    if (!p->causal) return L - 1;
    const int qi = n / p->h_r;
    const int64_t lim = L - p->q_len + qi;
    return lim < L - 1 ? lim : L - 1;
  }

  // Scaled logit z_j of row n against key j.
  double logit(int b, int g, int n, int j) const {
    double dot = 0.0;
    for (int i = 0; i < p->head_dim; ++i) dot += q_at(b, g, n, i) * k_at(b, j, g, i);
    return p->softmax_scale * qd_at(b, g) * kd_at(b, g) * dot;
  }

  // Softmax statistics of row n over the visible keys in [j0, j1):
  //   m = max z_j, l = sum exp(z_j - m), acc[i] = sum exp(z_j - m) v_j[i]
  // (no scale_o / v descale).  An empty range gives m = -inf, l = 0, acc = 0.
  void partial(int b, int g, int n, int64_t j0, int64_t j1, double* m_out, double* l_out,
               double* acc) const {
    const int d = p->head_dim;
    const int64_t lim = last_visible(b, n);
    const int64_t hi = (j1 - 1 < lim) ? j1 - 1 : lim;  // inclusive
    for (int i = 0; i < d; ++i) acc[i] = 0.0;
    if (hi < j0) {
      *m_out = -std::numeric_limits<double>::infinity();
      *l_out = 0.0;
      return;
    }
    std::vector<double> z(static_cast<size_t>(hi - j0 + 1));
    double m = -std::numeric_limits<double>::infinity();
    for (int64_t j = j0; j <= hi; ++j) {
      z[j - j0] = logit(b, g, n, static_cast<int>(j));
      if (z[j - j0] > m) m = z[j - j0];
    }
    double l = 0.0;
    for (int64_t j = j0; j <= hi; ++j) {
      const double w = std::exp(z[j - j0] - m);
      l += w;
      for (int i = 0; i < d; ++i) acc[i] += w * v_at(b, static_cast<int>(j), g, i);
    }
    *m_out = m;
    *l_out = l;
  }

  // Final O (d values) and LSE of one row over all its visible keys.
  void row(int b, int g, int n, double* o, double* lse) const {
    const int d = p->head_dim;
    double m, l;
    partial(b, g, n, 0, seq_lens[b], &m, &l, o);
    if (l == 0.0) {  // no visible key
      for (int i = 0; i < d; ++i) o[i] = 0.0;
      *lse = -std::numeric_limits<double>::infinity();
      return;
    }
    const double s = p->scale_o * vd_at(b, g) / l;
    for (int i = 0; i < d; ++i) o[i] *= s;
    *lse = m + std::log(l);
  }
};

}  // namespace

extern "C" {

// Full attention for a list of (b, g) units (pairs in `units`), or for every
// (b, g) in b-major order when units == NULL.  Output unit u occupies
// o[u * n_q * d ...] and lse[u * n_q ...].  `threads` <= 0 uses every
// hardware thread.  Returns 0, or -1 on a bad argument.
int oracle_attention(const oracle_problem* p, const void* q, const uint8_t* k, const uint8_t* v,
                     const int32_t* block_table, const int32_t* seq_lens, const float* qd,
                     const float* kd, const float* vd, const int32_t* units, int32_t n_units,
                     double* o, double* lse, int32_t threads) {
  if (!p || !q || !k || !v || !block_table || !seq_lens || !qd || !kd || !vd || !o || !lse)
    return -1;
  if (p->h_r <= 0 || p->q_len <= 0 || p->head_dim <= 0 || p->page_size <= 0) return -1;
  View view{p, q, k, v, block_table, seq_lens, qd, kd, vd};
  const int64_t total = units ? n_units : static_cast<int64_t>(p->num_seqs) * p->h_k;
  const int n_q = view.n_q();
  const int d = p->head_dim;
  int nt = threads > 0 ? threads : static_cast<int>(std::thread::hardware_concurrency());
  if (nt < 1) nt = 1;
  if (nt > total) nt = static_cast<int>(total > 0 ? total : 1);
  std::atomic<int64_t> next{0};
  auto worker = [&]() {
    for (;;) {
      const int64_t u = next.fetch_add(1);
      if (u >= total) return;
      int b, g;
      if (units) {
        b = units[2 * u];
        g = units[2 * u + 1];
      } else {
        b = static_cast<int>(u / p->h_k);
        g = static_cast<int>(u % p->h_k);
      }
      for (int n = 0; n < n_q; ++n)
        view.row(b, g, n, o + (u * n_q + n) * d, lse + u * n_q + n);
    }
  };
  if (nt == 1) {
    worker();
  } else {
    std::vector<std::thread> pool;
    for (int t = 0; t < nt; ++t) pool.emplace_back(worker);
    for (auto& t : pool) t.join();
  }
  return 0;
}

// Softmax statistics of one row over keys [j0, j1) (see View::partial).
int oracle_partial(const oracle_problem* p, const void* q, const uint8_t* k, const uint8_t* v,
                   const int32_t* block_table, const int32_t* seq_lens, const float* qd,
                   const float* kd, const float* vd, int32_t b, int32_t g, int32_t n, int64_t j0,
                   int64_t j1, double* m, double* l, double* acc) {
  if (!p || !m || !l || !acc) return -1;
  View view{p, q, k, v, block_table, seq_lens, qd, kd, vd};
  view.partial(b, g, n, j0, j1, m, l, acc);
  return 0;
}

// Combine n_parts partial statistics of one row (each (m_j, l_j, acc_j) from
// oracle_partial) into O and LSE: rescale every part to the common maximum,
// add, divide.  `out_scale` multiplies O (scale_o * v descale).
int oracle_merge(int32_t n_parts, int32_t d, const double* m, const double* l, const double* acc,
                 double out_scale, double* o, double* lse) {
  if (n_parts < 0 || d <= 0 || !o || !lse) return -1;
  double m_max = -std::numeric_limits<double>::infinity();
  for (int j = 0; j < n_parts; ++j)
    if (m[j] > m_max) m_max = m[j];
  double l_sum = 0.0;
  for (int i = 0; i < d; ++i) o[i] = 0.0;
  for (int j = 0; j < n_parts; ++j) {
    if (l[j] == 0.0) continue;  // an empty part contributes nothing
    const double w = std::exp(m[j] - m_max);
    l_sum += w * l[j];
    for (int i = 0; i < d; ++i) o[i] += w * acc[static_cast<int64_t>(j) * d + i];
  }
  if (l_sum == 0.0) {
    for (int i = 0; i < d; ++i) o[i] = 0.0;
    *lse = -std::numeric_limits<double>::infinity();
    return 0;
  }
  for (int i = 0; i < d; ++i) o[i] *= out_scale / l_sum;
  *lse = m_max + std::log(l_sum);
  return 0;
}

}  // extern "C"
