/*
 * synth.c -- seeded, counter-based generator of the synthetic inputs of the
 * sparse MoE block (router weights, shared-expert gate vector, int4 expert
 * weights with their affine scales/biases, and token activations).
 *
 * This module draws random numbers and rounds them to the storage types; it
 * holds none of the MoE block's arithmetic.  Both the CPU oracle and the CUDA
 * library consume the arrays it writes.
 *
 * Generator: the SplitMix64 sequence of Steele, Lea and Flood, "Fast
 * splittable pseudorandom number generators" (OOPSLA 2014).  With state
 * `key`, output i (i = 0, 1, ...) is mix64(key + (i + 1) * 0x9E3779B97F4A7C15),
 * so any element can be drawn independently of the others (counter-based).
 * Normals use the Box-Muller transform (Box & Muller, 1958) in double.
 *
 * Distributions (the synthetic recipe of the int4 MoE workloads):
 *   packed int4 codes      q ~ U{0..15}, 8 codes per uint32 word;
 *   group scale            s = bf16(0.005 + 0.01*|N(0,1)|);   bias b = -8*s;
 *   router / shared gate   bf16 N(0, std) with std = 1/sqrt(hidden);
 *   token activations      bf16 N(0, 1).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -fPIC -shared (contraction off so
 * that x86 and aarch64 hosts round the same way).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

/* Output i of the SplitMix64 sequence whose state starts at `key`. */
uint64_t synth_draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * SYNTH_GOLDEN); }

/* Stream key for one tensor: a chain of SplitMix64 mixes over its coordinates. */
uint64_t synth_key(uint64_t seed, uint64_t workload, uint64_t layer, uint64_t tensor,
                   uint64_t index) {
  uint64_t k = mix64(seed + SYNTH_GOLDEN);
  k = mix64(k ^ (workload + SYNTH_GOLDEN));
  k = mix64(k ^ (layer + 2 * SYNTH_GOLDEN));
  k = mix64(k ^ (tensor + 3 * SYNTH_GOLDEN));
  k = mix64(k ^ (index + 4 * SYNTH_GOLDEN));
  return k;
}

/* float -> bf16 bits, round to nearest even (NaN -> canonical quiet NaN). */
static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

static inline float bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Standard normal number n of stream `key` (Box-Muller, pairs 2m and 2m+1). */
static inline double normal_at(uint64_t key, uint64_t n) {
  uint64_t m = n >> 1;
  double u1 = (double)((synth_draw(key, 2 * m) >> 11) + 1) * 0x1.0p-53; /* (0, 1] */
  double u2 = (double)(synth_draw(key, 2 * m + 1) >> 11) * 0x1.0p-53;   /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double a = 6.283185307179586476925286766559 * u2;
  return (n & 1) ? r * sin(a) : r * cos(a);
}

/* Uniform 32-bit words: word 2i is the low half of draw i, word 2i+1 the high half.
 * As packed int4 codes every nibble is U{0..15}. */
void synth_fill_u32(uint64_t key, int64_t n, uint32_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < (n + 1) / 2; ++i) {
    uint64_t d = synth_draw(key, (uint64_t)i);
    out[2 * i] = (uint32_t)d;
    if (2 * i + 1 < n) out[2 * i + 1] = (uint32_t)(d >> 32);
  }
}

/* bf16(mean + std * N(0,1)), the value rounded double -> float -> bf16. */
void synth_fill_normal_bf16(uint64_t key, int64_t n, double mean, double std, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = (float)(mean + std * normal_at(key, (uint64_t)i));
    out[i] = f32_to_bf16(v);
  }
}

/* Group scales and biases: s = bf16(0.005 + 0.01*|N(0,1)|), b = bf16(-8*s) (exact). */
void synth_fill_scale_bias(uint64_t key, int64_t n, uint16_t* s_out, uint16_t* b_out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    float v = (float)(0.005 + 0.01 * fabs(normal_at(key, (uint64_t)i)));
    uint16_t s = f32_to_bf16(v);
    s_out[i] = s;
    b_out[i] = f32_to_bf16(-8.0f * bf16_to_f32(s));
  }
}

/* Tensor ids of the stream keys. */
enum {
  T_ROUTER_W = 1,
  T_SHARED_GATE_VEC = 2,
  T_TOKENS = 3,
  T_SHARED_BASE = 10, /* + 0..5: gate_q, gate_sb, up_q, up_sb, down_q, down_sb */
  T_EXPERT_BASE = 20  /* same six, index = expert id */
};

/* One quantised matrix [rows][cols]: q words [rows][cols/8], s/b [rows][cols/group]. */
static void fill_qmatrix(uint64_t kq, uint64_t ksb, int64_t rows, int64_t cols, int64_t group,
                         uint32_t* q, uint16_t* s, uint16_t* b) {
  int64_t nw = rows * (cols / 8);
  int64_t ng = rows * (cols / group);
  for (int64_t i = 0; i < (nw + 1) / 2; ++i) {
    uint64_t d = synth_draw(kq, (uint64_t)i);
    q[2 * i] = (uint32_t)d;
    if (2 * i + 1 < nw) q[2 * i + 1] = (uint32_t)(d >> 32);
  }
  for (int64_t i = 0; i < ng; ++i) {
    float v = (float)(0.005 + 0.01 * fabs(normal_at(ksb, (uint64_t)i)));
    uint16_t sv = f32_to_bf16(v);
    s[i] = sv;
    b[i] = f32_to_bf16(-8.0f * bf16_to_f32(sv));
  }
}

/*
 * Experts e0 .. e0+n-1 of one layer, canonical (MLX affine) layout, expert-major:
 *   gate_q/up_q [n][inter][hidden/8], gate_s/gate_b/up_s/up_b [n][inter][hidden/group],
 *   down_q [n][hidden][inter/8],       down_s/down_b [n][hidden][inter/group].
 * When `shared` is nonzero the single shared expert is written instead (n must be 1).
 */
void synth_fill_experts(uint64_t seed, uint64_t workload, uint64_t layer, int shared, int64_t e0,
                        int64_t n, int64_t hidden, int64_t inter, int64_t group,
                        uint32_t* gate_q, uint16_t* gate_s, uint16_t* gate_b, uint32_t* up_q,
                        uint16_t* up_s, uint16_t* up_b, uint32_t* down_q, uint16_t* down_s,
                        uint16_t* down_b) {
  int64_t gu_w = inter * (hidden / 8), gu_g = inter * (hidden / group);
  int64_t d_w = hidden * (inter / 8), d_g = hidden * (inter / group);
  uint64_t base = shared ? T_SHARED_BASE : T_EXPERT_BASE;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t j = 0; j < 3 * n; ++j) {
    int64_t x = j / 3, m = j % 3;
    uint64_t e = shared ? 0 : (uint64_t)(e0 + x);
    uint64_t kq = synth_key(seed, workload, layer, base + 2 * m, e);
    uint64_t ks = synth_key(seed, workload, layer, base + 2 * m + 1, e);
    if (m == 0)
      fill_qmatrix(kq, ks, inter, hidden, group, gate_q + x * gu_w, gate_s + x * gu_g,
                   gate_b + x * gu_g);
    else if (m == 1)
      fill_qmatrix(kq, ks, inter, hidden, group, up_q + x * gu_w, up_s + x * gu_g,
                   up_b + x * gu_g);
    else
      fill_qmatrix(kq, ks, hidden, inter, group, down_q + x * d_w, down_s + x * d_g,
                   down_b + x * d_g);
  }
}

/* Router weight bf16 [E][hidden] and shared-expert gate vector bf16 [hidden], N(0, 1/sqrt(hidden)). */
void synth_fill_router(uint64_t seed, uint64_t workload, uint64_t layer, int64_t E,
                       int64_t hidden, uint16_t* router_w, uint16_t* shared_gate_vec) {
  double std = 1.0 / sqrt((double)hidden);
  synth_fill_normal_bf16(synth_key(seed, workload, layer, T_ROUTER_W, 0), E * hidden, 0.0, std,
                         router_w);
  synth_fill_normal_bf16(synth_key(seed, workload, layer, T_SHARED_GATE_VEC, 0), hidden, 0.0,
                         std, shared_gate_vec);
}

/* Token activations bf16 [T][hidden] ~ N(0,1) for (layer, step). */
void synth_fill_tokens(uint64_t seed, uint64_t workload, uint64_t layer, uint64_t step, int64_t T,
                       int64_t hidden, uint16_t* x) {
  synth_fill_normal_bf16(synth_key(seed, workload, layer, T_TOKENS, step), T * hidden, 0.0, 1.0,
                         x);
}
