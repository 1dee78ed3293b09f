// Oracle for the fused attention forward pass -- TEST INFRASTRUCTURE ONLY.
//
// Only tests/, the smoke check and the benchmark's CPU-baseline leg may load
// this library.  It shares no code with the CUDA path and does not follow its
// algorithm: it materialises each row of the score matrix in float64 and runs
// a plain two-pass softmax, which is the definition the pages give.
//
// What is computed (per batch b, head h, query row i):
//   * "Attention memory" page, section "The quadratic bound": the score matrix
//     is s x s and entry (i, j) says how much token i attends to token j.
//   * same page, section "What this memory is": the scores sit between the
//     query-key product and the softmax-weighted sum of the values, so
//       s_ij = scale * <q_i, k_j>,   O_i = sum_j softmax_j(s_i.) * v_j.
//   * "PyTorch attention backends" story (masked_fill sentences): a masked
//     key is filled with minus infinity before the softmax, so it gets weight
//     exactly zero.  Key j is allowed for row i iff j < valid_b and, when
//     causal, j <= i (top-left alignment, the torch SDPA is_causal reading).
//   * "Flash attention" glossary page, first paragraph: the fused method gives
//     the same numbers as standard attention; this file is standard attention.
//   * The log-sum-exp that the fused kernel also returns is
//       LSE_i = ln sum_{allowed j} exp(s_ij)  (= m + ln l with m the row max),
//     and a row with no allowed key gives O_i = 0 and LSE_i = -inf.
//   * "Attention memory" page, sections "Formula" and "Worked example": the
//     materialised score buffer holds B * H * s^2 * e bytes.
//
// Inputs are bf16 bit patterns widened exactly to double (or, through
// attn_ref_f64_dbl, doubles).  Every product and sum is in double.
//
// Parity pins: tests/test_oracle_pins.py (worked-example bytes, row sums,
// constant V, Q = 0, causal row 0, key permutation, padding = truncation,
// one-hot peak, and torch's float64 CPU SDPA as an independent library
// routine); tests/test_oracle_mutants.py shows those pins catch planted
// mistakes in this file.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>

namespace {

double bf16_to_double(uint16_t bits) {
  const uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// Inputs either as bf16 bit patterns or as doubles (the latter lets the tests
// take finite differences of the forward pass).
struct Problem {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const double* qd;  // when non-null, q/k/v are read from qd/kd/vd instead
  const double* kd;
  const double* vd;
  int64_t B, H, S_q, S_kv, D;
  double scale;
  int causal;
  const int32_t* kv_valid_len;  // host, may be null
};

// Key j is allowed for query row i of batch b (masked_fill to -inf otherwise).
bool key_allowed(const Problem& p, int64_t b, int64_t i, int64_t j) {
  int64_t valid = p.S_kv;
  if (p.kv_valid_len != nullptr) {
    valid = std::min<int64_t>(std::max<int64_t>(p.kv_valid_len[b], 0), p.S_kv);
  }
  if (j >= valid) return false;
  if (p.causal && j > i) return false;
  return true;
}

double q_at(const Problem& p, int64_t idx) { return p.qd ? p.qd[idx] : bf16_to_double(p.q[idx]); }
double k_at(const Problem& p, int64_t idx) { return p.kd ? p.kd[idx] : bf16_to_double(p.k[idx]); }
double v_at(const Problem& p, int64_t idx) { return p.vd ? p.vd[idx] : bf16_to_double(p.v[idx]); }

// One output row: materialise the score row, then a two-pass softmax.
void one_row(const Problem& p, int64_t flat_row, double* o_row, double* lse_out,
             std::vector<double>& s_row) {
  const int64_t b = flat_row / (p.H * p.S_q);
  const int64_t h = (flat_row / p.S_q) % p.H;
  const int64_t i = flat_row % p.S_q;
  const int64_t qi = ((b * p.H + h) * p.S_q + i) * p.D;   // element offsets
  const int64_t kbh = (b * p.H + h) * p.S_kv * p.D;
  const int64_t vbh = kbh;
  const double neg_inf = -std::numeric_limits<double>::infinity();

  // Scores s_ij = scale * q_i . k_j, with masked entries set to -inf.
  s_row.assign(static_cast<size_t>(p.S_kv), neg_inf);
  for (int64_t j = 0; j < p.S_kv; ++j) {
    if (!key_allowed(p, b, i, j)) continue;
    double dot = 0.0;
    for (int64_t d = 0; d < p.D; ++d) {
      dot += q_at(p, qi + d) * k_at(p, kbh + j * p.D + d);
    }
    s_row[j] = p.scale * dot;
  }

  // Pass 1: row maximum.
  double m = neg_inf;
  for (int64_t j = 0; j < p.S_kv; ++j) m = std::max(m, s_row[j]);

  for (int64_t d = 0; d < p.D; ++d) o_row[d] = 0.0;
  if (m == neg_inf) {  // no allowed key
    *lse_out = neg_inf;
    return;
  }

  // Pass 2: exponentials, their sum, and the weighted sum of value rows.
  double l = 0.0;
  for (int64_t j = 0; j < p.S_kv; ++j) {
    if (s_row[j] == neg_inf) continue;
    const double e = std::exp(s_row[j] - m);
    l += e;
    for (int64_t d = 0; d < p.D; ++d) o_row[d] += e * v_at(p, vbh + j * p.D + d);
  }
  for (int64_t d = 0; d < p.D; ++d) o_row[d] /= l;
  *lse_out = m + std::log(l);
}

}  // namespace

extern "C" {

// Number of bytes of a materialised B x H x s x s score matrix with e bytes per
// score ("Attention memory" page, "Formula" section).
uint64_t attn_ref_score_buffer_bytes(int64_t B, int64_t H, int64_t s, int64_t e) {
  return static_cast<uint64_t>(B) * static_cast<uint64_t>(H) * static_cast<uint64_t>(s) *
         static_cast<uint64_t>(s) * static_cast<uint64_t>(e);
}

}  // extern "C"

namespace {

int run_rows(const Problem& p, const int64_t* rows, int64_t n_rows, double* o, double* lse, int threads) {
  const int64_t B = p.B, H = p.H, S_q = p.S_q, D = p.D;
  if (B < 1 || H < 1 || S_q < 0 || p.S_kv < 0 || D < 1 || n_rows < 0) return 1;
  if (n_rows > 0 && (o == nullptr || lse == nullptr)) return 1;
  if (rows == nullptr && n_rows != B * H * S_q) return 1;
  const int64_t total = B * H * S_q;
  if (rows != nullptr) {
    for (int64_t r = 0; r < n_rows; ++r)
      if (rows[r] < 0 || rows[r] >= total) return 1;
  }

  int nt = threads > 0 ? threads : static_cast<int>(std::thread::hardware_concurrency());
  nt = std::max(1, std::min<int>(nt, static_cast<int>(std::max<int64_t>(n_rows, 1))));

  auto work = [&](int tid) {
    std::vector<double> s_row;
    for (int64_t r = tid; r < n_rows; r += nt) {
      const int64_t flat = rows != nullptr ? rows[r] : r;
      one_row(p, flat, o + r * D, lse + r, s_row);
    }
  };
  if (nt == 1) {
    work(0);
  } else {
    std::vector<std::thread> pool;
    pool.reserve(static_cast<size_t>(nt));
    for (int t = 0; t < nt; ++t) pool.emplace_back(work, t);
    for (auto& th : pool) th.join();
  }
  return 0;
}

}  // namespace

extern "C" {

// Reference attention forward in float64.
//   q: bf16 bits [B][H][S_q][D]; k, v: bf16 bits [B][H][S_kv][D] (host memory)
//   kv_valid_len: host int32[B] or null (= S_kv for every batch)
//   rows: flat query-row ids (b*H + h)*S_q + i, or null for all B*H*S_q rows
//   o: n_rows x D doubles; lse: n_rows doubles (natural log)
//   threads <= 0 uses every hardware thread.
// Returns 0 on success, 1 on invalid arguments.
int attn_ref_f64(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t B, int64_t H,
                 int64_t S_q, int64_t S_kv, int64_t D, double scale, int causal,
                 const int32_t* kv_valid_len, const int64_t* rows, int64_t n_rows, double* o,
                 double* lse, int threads) {
  if (n_rows > 0 && q == nullptr) return 1;
  if (S_kv > 0 && (k == nullptr || v == nullptr)) return 1;
  const Problem p{q, k, v, nullptr, nullptr, nullptr, B, H, S_q, S_kv, D, scale, causal, kv_valid_len};
  return run_rows(p, rows, n_rows, o, lse, threads);
}

// The same computation on float64 inputs (same layouts), for finite differences.
int attn_ref_f64_dbl(const double* q, const double* k, const double* v, int64_t B, int64_t H,
                     int64_t S_q, int64_t S_kv, int64_t D, double scale, int causal,
                     const int32_t* kv_valid_len, const int64_t* rows, int64_t n_rows, double* o,
                     double* lse, int threads) {
  if (n_rows > 0 && q == nullptr) return 1;
  if (S_kv > 0 && (k == nullptr || v == nullptr)) return 1;
  const Problem p{nullptr, nullptr, nullptr, q, k, v, B, H, S_q, S_kv, D, scale, causal, kv_valid_len};
  return run_rows(p, rows, n_rows, o, lse, threads);
}

// Threads attn_ref_f64 would use for threads <= 0.
int attn_ref_hardware_threads(void) {
  return static_cast<int>(std::thread::hardware_concurrency());
}

}  // extern "C"
