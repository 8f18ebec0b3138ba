// moe_oracle.cpp -- CPU oracle of the sparse int4 MoE block.  TEST
// INFRASTRUCTURE ONLY: the test suite, the package smoke check and the
// benchmark's CPU-baseline leg call it (through oracle/cpp.py); the CUDA
// library never does, and the two share no code.
//
// What it computes follows the Swiftlet project README ("Show HN: Run an 80B
// Qwen in 4.3 GB of RAM on a Mac and a 35B on an iPhone", wpnews), section
// "How it works": each token is routed to k of E experts, a shared expert is
// always applied, and the experts are stored in MLX's affine int4 group
// quantisation (same README, its list of what was built).  Per token t:
//   1. l[e] = x_t . Wr_e (+ prior_e)
//   2. top-k of softmax(l) by the EXACT value of l (descending, ties to the
//      lowest expert id), the k probabilities renormalised to sum to one
//   3. g = sigmoid(x_t . wsg)
//   4. the pairs p = t k + j stably sorted by expert (perm, offsets)
//   5. per pair: a = Wg x, u = Wu x, h = silu(a) u, o = Wd h, W = s q + b per
//      group of G inputs (code 8c+j of a row in bits 4j..4j+3 of word c)
//   6. y_t = sum_j w_j o_j + g S(x_t), S the shared expert
// Everything is float64 (bf16 and fp32 inputs widen exactly); the selection
// uses float64 logits with a rigorous error bound and decides overlapping
// candidates with an exact integer accumulator, so it is a function of the
// inputs alone.  The stack (oracle_moe_stack) chains blocks for one token:
// n = RMSNorm(x) * norm_w (bf16), x <- bf16(x + bf16(y)) -- a reading: the
// pages show no equations between the blocks.
//
// Parallelism: OpenMP over tokens (routing) and over experts (projections);
// every sum runs in a fixed order, so results do not depend on the thread
// count.
#include <omp.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

double bf16_value(uint16_t b) {
  const uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Nearest bf16 (ties to even) of a float64 value that is far from bf16's
// overflow and underflow: keep 8 significant bits of v = m 2^e.
uint16_t bf16_round(double v) {
  if (v == 0.0) return std::signbit(v) ? 0x8000 : 0;
  int e;
  const double m = std::frexp(v, &e);                  // 1/2 <= |m| < 1
  const double r = std::ldexp(std::nearbyint(std::ldexp(m, 8)), e - 8);  // ties to even
  const float f = (float)r;                            // exact: 8 significant bits
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// Exact sum of float64 terms with at most 53 significant bits: a fixed-point
// integer in 32-bit digits, value = sum_i d[i] 2^(32 i + kLsb).  bf16 x bf16
// products (down to 2^-266) and fp32 priors (down to 2^-149) all fit; digits
// are int64 so that carries can wait until the end.
struct ExactSum {
  static constexpr int kLsb = -340;
  static constexpr int kDigits = 30;
  int64_t d[kDigits];
  ExactSum() { std::memset(d, 0, sizeof d); }
  void add(double v) {
    if (v == 0.0) return;
    int e;
    const double m = std::frexp(std::fabs(v), &e);
    const uint64_t mant = (uint64_t)std::ldexp(m, 53);  // exact integer < 2^53
    const int sh = e - 53 - kLsb;                        // bit position of mant's LSB
    unsigned __int128 w = (unsigned __int128)mant << (sh % 32);
    for (int i = sh / 32; w != 0; ++i, w >>= 32) {
      const int64_t part = (int64_t)(uint32_t)w;
      d[i] += v < 0 ? -part : part;
    }
  }
  // Propagate carries: digits 0..n-2 in [0, 2^32), the top digit signed.
  void normalise() {
    int64_t carry = 0;
    for (int i = 0; i < kDigits - 1; ++i) {
      const int64_t t = d[i] + carry;
      d[i] = t & 0xFFFFFFFFll;
      carry = (t - d[i]) / 4294967296ll;
    }
    d[kDigits - 1] += carry;
  }
};

int exact_cmp(ExactSum a, ExactSum b) {
  a.normalise();
  b.normalise();
  if (a.d[ExactSum::kDigits - 1] != b.d[ExactSum::kDigits - 1])
    return a.d[ExactSum::kDigits - 1] < b.d[ExactSum::kDigits - 1] ? -1 : 1;
  for (int i = ExactSum::kDigits - 2; i >= 0; --i)
    if (a.d[i] != b.d[i]) return a.d[i] < b.d[i] ? -1 : 1;
  return 0;
}

struct QMat {  // one int4 matrix [rows][cols]: q [rows][cols/8], s/b [rows][cols/G]
  const uint32_t* q;
  const uint16_t* s;
  const uint16_t* b;
  int rows, cols;
};

// Row r of W = s q + b, dequantised into out[cols].
void dequant_row(const QMat& m, int r, int G, double* out) {
  const uint32_t* qr = m.q + (size_t)r * (m.cols / 8);
  const uint16_t* sr = m.s + (size_t)r * (m.cols / G);
  const uint16_t* br = m.b + (size_t)r * (m.cols / G);
  for (int c = 0; c < m.cols; ++c) {
    const int code = (int)((qr[c / 8] >> (4 * (c % 8))) & 0xFu);
    out[c] = bf16_value(sr[c / G]) * code + bf16_value(br[c / G]);
  }
}

double silu(double z) { return z / (1.0 + std::exp(-z)); }

struct Block {
  int T, H, E, k, I, Is, G;
  const uint16_t* x;          // [T][H]
  const uint16_t* router_w;   // [E][H]
  const float* router_bias;   // [E] or null
  const uint16_t* gate_vec;   // [H]
  QMat sg, su, sd;            // shared expert
  const uint32_t *eq[3];      // routed experts, leading dim E: gate, up, down
  const uint16_t *es[3], *eb[3];
};

QMat expert_mat(const Block& B, int which, int e) {
  const int rows = which == 2 ? B.H : B.I, cols = which == 2 ? B.I : B.H;
  const size_t nq = (size_t)rows * (cols / 8), ns = (size_t)rows * (cols / B.G);
  return QMat{B.eq[which] + e * nq, B.es[which] + e * ns, B.eb[which] + e * ns, rows, cols};
}

// Steps 1-3 for token t: selected experts (exact order), their weights, the gate.
void route_token(const Block& B, int t, int32_t* idx, double* w, double* gate, double* logit) {
  const int H = B.H, E = B.E, k = B.k;
  const uint16_t* xt = B.x + (size_t)t * H;
  std::vector<double> xv(H), lo(E), hi(E);
  for (int h = 0; h < H; ++h) xv[h] = bf16_value(xt[h]);
  const double u = std::ldexp(1.0, -53);
  for (int e = 0; e < E; ++e) {
    const uint16_t* wr = B.router_w + (size_t)e * H;
    double s = 0.0, mag = 0.0;
    for (int h = 0; h < H; ++h) {
      const double p = xv[h] * bf16_value(wr[h]);  // exact
      s += p;
      mag += std::fabs(p);
    }
    if (B.router_bias) {
      s += (double)B.router_bias[e];
      mag += std::fabs((double)B.router_bias[e]);
    }
    // |float64 sum - exact| <= gamma_n sum|terms| (Higham, Accuracy and
    // Stability of Numerical Algorithms, Thm. 4.3); twice that, to spare
    const double bound = 2.0 * (H + 2) * u * mag;
    logit[e] = s;
    lo[e] = s - bound;
    hi[e] = s + bound;
  }
  // an expert whose upper end lies below the k-th largest lower end is beaten
  // by k experts: only the others are candidates
  std::vector<double> sorted_lo(lo);
  std::nth_element(sorted_lo.begin(), sorted_lo.begin() + (E - k), sorted_lo.end());
  const double kth = sorted_lo[E - k];
  std::vector<int> cand;
  for (int e = 0; e < E; ++e)
    if (hi[e] >= kth) cand.push_back(e);
  // candidates whose interval overlaps another candidate's get exact values
  const int C = (int)cand.size();
  std::vector<char> need(C, 0);
  for (int a = 0; a < C; ++a)
    for (int b = 0; b < C; ++b)
      if (a != b && lo[cand[a]] <= hi[cand[b]] && lo[cand[b]] <= hi[cand[a]]) need[a] = 1;
  std::vector<ExactSum> ex(C);
  for (int a = 0; a < C; ++a) {
    if (!need[a]) continue;
    const uint16_t* wr = B.router_w + (size_t)cand[a] * H;
    for (int h = 0; h < H; ++h) ex[a].add(xv[h] * bf16_value(wr[h]));
    if (B.router_bias) ex[a].add((double)B.router_bias[cand[a]]);
  }
  std::vector<int> ord(C);
  for (int a = 0; a < C; ++a) ord[a] = a;
  // exact order, ties to the lower id; two candidates of which one has no
  // exact value have disjoint intervals, and their float64 values order them
  std::sort(ord.begin(), ord.end(), [&](int a, int b) {
    int c;
    if (need[a] && need[b])
      c = exact_cmp(ex[a], ex[b]);
    else
      c = logit[cand[a]] < logit[cand[b]] ? -1 : logit[cand[a]] > logit[cand[b]] ? 1 : 0;
    if (c != 0) return c > 0;
    return cand[a] < cand[b];
  });
  // softmax over all E (max subtracted), renormalised over the selection
  double mx = logit[0];
  for (int e = 1; e < E; ++e) mx = std::max(mx, logit[e]);
  double z = 0.0;
  for (int e = 0; e < E; ++e) z += std::exp(logit[e] - mx);
  double den = 0.0;
  for (int j = 0; j < k; ++j) {
    idx[j] = cand[ord[j]];
    w[j] = std::exp(logit[idx[j]] - mx) / z;
    den += w[j];
  }
  for (int j = 0; j < k; ++j) w[j] /= den;
  double gz = 0.0;
  for (int h = 0; h < H; ++h) gz += xv[h] * bf16_value(B.gate_vec[h]);
  *gate = 1.0 / (1.0 + std::exp(-gz));
}

// o[n][H] = Wd (silu(Wg x_n) * (Wu x_n)) for the n inputs xs[n][H].
void expert_mlp(const QMat& wg, const QMat& wu, const QMat& wd, int G, const double* xs, int n,
                double* o) {
  const int I = wg.rows, H = wg.cols;
  std::vector<double> row(std::max(H, I)), a((size_t)n * I), up((size_t)n * I);
  for (int r = 0; r < I; ++r) {
    dequant_row(wg, r, G, row.data());
    for (int p = 0; p < n; ++p) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += row[h] * xs[(size_t)p * H + h];
      a[(size_t)p * I + r] = s;
    }
    dequant_row(wu, r, G, row.data());
    for (int p = 0; p < n; ++p) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += row[h] * xs[(size_t)p * H + h];
      up[(size_t)p * I + r] = s;
    }
  }
  for (size_t i = 0; i < (size_t)n * I; ++i) a[i] = silu(a[i]) * up[i];  // h
  for (int r = 0; r < H; ++r) {
    dequant_row(wd, r, G, row.data());
    for (int p = 0; p < n; ++p) {
      double s = 0.0;
      for (int i = 0; i < I; ++i) s += row[i] * a[(size_t)p * I + i];
      o[(size_t)p * H + r] = s;
    }
  }
}

// The whole block; y only for the n_rows token rows listed.
void run_block(const Block& B, const int32_t* rows, int n_rows, double* y, int32_t* topk_idx,
               double* topk_w, double* gate, double* logits, int32_t* perm, int32_t* offsets) {
  const int T = B.T, H = B.H, E = B.E, k = B.k;
#pragma omp parallel for schedule(dynamic)
  for (int t = 0; t < T; ++t)
    route_token(B, t, topk_idx + (size_t)t * k, topk_w + (size_t)t * k, gate + t,
                logits + (size_t)t * E);
  // stable counting sort of the pairs by expert
  std::vector<int> count(E, 0);
  for (int p = 0; p < T * k; ++p) ++count[topk_idx[p]];
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + count[e];
  std::vector<int> fill(offsets, offsets + E);
  for (int p = 0; p < T * k; ++p) perm[fill[topk_idx[p]]++] = p;
  // the listed rows' pairs, grouped by expert (the shared expert last, id E)
  std::vector<double> xs((size_t)n_rows * H);
  for (int r = 0; r < n_rows; ++r)
    for (int h = 0; h < H; ++h) xs[(size_t)r * H + h] = bf16_value(B.x[(size_t)rows[r] * H + h]);
  std::vector<std::vector<int>> pairs(E + 1);  // entries r * k + j (j = k: shared)
  for (int r = 0; r < n_rows; ++r) {
    for (int j = 0; j < k; ++j) pairs[topk_idx[(size_t)rows[r] * k + j]].push_back(r * (k + 1) + j);
    pairs[E].push_back(r * (k + 1) + k);
  }
  std::vector<double> o((size_t)n_rows * (k + 1) * H);
#pragma omp parallel for schedule(dynamic)
  for (int e = 0; e <= E; ++e) {
    const std::vector<int>& ps = pairs[e];
    if (ps.empty()) continue;
    std::vector<double> in(ps.size() * (size_t)H), out(ps.size() * (size_t)H);
    for (size_t n = 0; n < ps.size(); ++n)
      std::memcpy(&in[n * H], &xs[(size_t)(ps[n] / (k + 1)) * H], sizeof(double) * H);
    if (e < E)
      expert_mlp(expert_mat(B, 0, e), expert_mat(B, 1, e), expert_mat(B, 2, e), B.G, in.data(),
                 (int)ps.size(), out.data());
    else
      expert_mlp(B.sg, B.su, B.sd, B.G, in.data(), (int)ps.size(), out.data());
    for (size_t n = 0; n < ps.size(); ++n)
      std::memcpy(&o[(size_t)ps[n] * H], &out[n * H], sizeof(double) * H);
  }
  // combine in a fixed order: routed experts by rank, then the shared one
  for (int r = 0; r < n_rows; ++r) {
    const int t = rows[r];
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) acc += topk_w[(size_t)t * k + j] * o[((size_t)r * (k + 1) + j) * H + h];
      y[(size_t)r * H + h] = acc + gate[t] * o[((size_t)r * (k + 1) + k) * H + h];
    }
  }
}

Block make_block(int T, int H, int E, int k, int I, int Is, int G, const uint16_t* x,
                 const uint16_t* router_w, const float* router_bias, const uint16_t* gate_vec,
                 const uint32_t* const* sq, const uint16_t* const* ss, const uint16_t* const* sb,
                 const uint32_t* const* eq, const uint16_t* const* es, const uint16_t* const* eb) {
  Block B;
  B.T = T, B.H = H, B.E = E, B.k = k, B.I = I, B.Is = Is, B.G = G;
  B.x = x, B.router_w = router_w, B.router_bias = router_bias, B.gate_vec = gate_vec;
  B.sg = QMat{sq[0], ss[0], sb[0], Is, H};
  B.su = QMat{sq[1], ss[1], sb[1], Is, H};
  B.sd = QMat{sq[2], ss[2], sb[2], H, Is};
  for (int i = 0; i < 3; ++i) B.eq[i] = eq[i], B.es[i] = es[i], B.eb[i] = eb[i];
  return B;
}

}  // namespace

extern "C" {

// Nearest bf16 bits of each of the n float64 values.
void oracle_bf16_round(const double* v, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16_round(v[i]);
}

// The block over T tokens.  Weights: sq/ss/sb = shared {gate, up, down}
// {q, s, b}; eq/es/eb = routed {gate, up, down} {q, s, b} with leading dim E
// (slot e = expert e).  rows[n_rows]: token rows whose y is computed (y is
// [n_rows][H]); routing, perm [T k] and offsets [E+1] cover every token.
// threads: OpenMP threads (0: the default).  Returns 0.
int oracle_moe_block(int T, int H, int E, int k, int I, int Is, int G, const uint16_t* x,
                     const uint16_t* router_w, const float* router_bias, const uint16_t* gate_vec,
                     const uint32_t* const* sq, const uint16_t* const* ss,
                     const uint16_t* const* sb, const uint32_t* const* eq,
                     const uint16_t* const* es, const uint16_t* const* eb, const int32_t* rows,
                     int n_rows, int threads, double* y, int32_t* topk_idx, double* topk_w,
                     double* gate, double* logits, int32_t* perm, int32_t* offsets) {
  if (threads > 0) omp_set_num_threads(threads);
  const Block B =
      make_block(T, H, E, k, I, Is, G, x, router_w, router_bias, gate_vec, sq, ss, sb, eq, es, eb);
  run_block(B, rows, n_rows, y, topk_idx, topk_w, gate, logits, perm, offsets);
  return 0;
}

// One token through L blocks: n = bf16(x / sqrt(mean x^2 + eps) * norm_w)
// (norm_w[l] null: ones), y = block l on n (or on xn_given[l] when given),
// x <- bf16(x + bf16(y)).  Per-layer weight pointers are arrays of L.
// Outputs: xs [L+1][H] (inputs, last = result), xn [L][H], y [L][H],
// topk_idx / topk_w [L][k].
int oracle_moe_stack(int L, int H, int E, int k, int I, int Is, int G, const uint16_t* x,
                     const uint16_t* const* router_w, const float* const* router_bias,
                     const uint16_t* const* gate_vec, const uint16_t* const* norm_w, double eps,
                     const uint32_t* const* sq, const uint16_t* const* ss,
                     const uint16_t* const* sb, const uint32_t* const* eq,
                     const uint16_t* const* es, const uint16_t* const* eb,
                     const uint16_t* xn_given, int threads, uint16_t* xs, uint16_t* xn, double* y,
                     int32_t* topk_idx, double* topk_w) {
  if (threads > 0) omp_set_num_threads(threads);
  std::memcpy(xs, x, sizeof(uint16_t) * H);
  std::vector<double> gate(1), logits(E);
  std::vector<int32_t> perm(k), offsets(E + 1);
  const int32_t row0 = 0;
  for (int l = 0; l < L; ++l) {
    const uint16_t* xl = xs + (size_t)l * H;
    uint16_t* nl = xn + (size_t)l * H;
    if (xn_given) {
      std::memcpy(nl, xn_given + (size_t)l * H, sizeof(uint16_t) * H);
    } else {
      double ms = 0.0;
      for (int h = 0; h < H; ++h) ms += bf16_value(xl[h]) * bf16_value(xl[h]);
      const double r = 1.0 / std::sqrt(ms / H + eps);
      for (int h = 0; h < H; ++h)
        nl[h] = bf16_round(bf16_value(xl[h]) * r * (norm_w[l] ? bf16_value(norm_w[l][h]) : 1.0));
    }
    const Block B = make_block(1, H, E, k, I, Is, G, nl, router_w[l], router_bias[l], gate_vec[l],
                               sq + 3 * l, ss + 3 * l, sb + 3 * l, eq + 3 * l, es + 3 * l,
                               eb + 3 * l);
    double* yl = y + (size_t)l * H;
    run_block(B, &row0, 1, yl, topk_idx + (size_t)l * k, topk_w + (size_t)l * k, gate.data(),
              logits.data(), perm.data(), offsets.data());
    uint16_t* xnext = xs + (size_t)(l + 1) * H;
    for (int h = 0; h < H; ++h)
      xnext[h] = bf16_round(bf16_value(xl[h]) + bf16_value(bf16_round(yl[h])));
  }
  return 0;
}

}  // extern "C"
