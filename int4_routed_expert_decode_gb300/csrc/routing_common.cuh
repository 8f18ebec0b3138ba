// routing_common.cuh -- device code of the router and the exact top-k, shared
// by the standalone router kernels and the fused decode kernel.
//
// Routing follows the Swiftlet README (wpnews page, "How it works"): each
// layer sends every token to k of E experts.  The selection ranks the exact
// real logits l = x . Wr_e (+ prior_e).  A bf16 x bf16 product is exact in
// fp32; the fp32 sum below has a fixed summation structure whose depth gives
// a rigorous error bound; where two candidates are closer than twice the
// bound their exact values are compared with an integer superaccumulator
// (Kulisch accumulation), ties going to the lower expert id.
#pragma once

#include <stdint.h>

#include "device_util.cuh"

namespace moe {
namespace rt {

constexpr int kRunCache = 32;  // exact values cached per warp
constexpr int kDigits = 18;    // 32-bit digits of the superaccumulator

template <int NJ>
struct RouterShape {
  static constexpr int H = NJ * 256;
  static constexpr int HV = H / 8;  // uint4 (8 bf16) chunks per row
  static constexpr int LOG2NJ =
      (NJ >= 32) ? 5 : (NJ >= 16) ? 4 : (NJ >= 8) ? 3 : (NJ >= 4) ? 2 : (NJ >= 2) ? 1 : 0;
  // Summation depth: 8 sequential FMAs per chunk, a pairwise tree over the NJ
  // chunk sums of a lane, a 5-level butterfly across lanes, the prior.
  static constexpr int DEPTH = 8 + LOG2NJ + 6;
  // 2 * D * u (u = 2^-24): twice gamma_D (Higham, Accuracy and Stability of
  // Numerical Algorithms, Thm. 4.3, for any summation tree of depth D).
  static constexpr float kBoundScale = 2.0f * (float)DEPTH * 5.9604644775390625e-8f;
};

// 2^-120: covers products that underflow in fp32 (at most 8192 terms of 2^-150).
constexpr float kBoundFloor = 7.52316384526264e-37f;

// x . w and sum |x w| of one row: lane l holds chunks c = l + 32 j (j < NJ) of
// the row in wv and the same chunks of x in xr (8 bf16 per uint4).  Every
// lane returns the full sums.
template <int NJ>
__device__ __forceinline__ void router_row_dot_regs(const uint4 (&wv)[NJ], const uint4 (&xr)[NJ],
                                                    float& sum, float& mag) {
  float acc[NJ], mg[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const uint4 xv = xr[j];
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ww[4] = {wv[j].x, wv[j].y, wv[j].z, wv[j].w};
    float a = 0.f, m = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float x0 = bf16_lo(xw[q]), x1 = bf16_hi(xw[q]);
      const float w0 = bf16_lo(ww[q]), w1 = bf16_hi(ww[q]);
      a = fmaf(x0, w0, a);
      a = fmaf(x1, w1, a);
      m = fmaf(fabsf(x0), fabsf(w0), m);
      m = fmaf(fabsf(x1), fabsf(w1), m);
    }
    acc[j] = a;
    mg[j] = m;
  }
#pragma unroll
  for (int s = NJ / 2; s > 0; s >>= 1) {
#pragma unroll
    for (int j = 0; j < s; ++j) {
      acc[j] += acc[j + s];
      mg[j] += mg[j + s];
    }
  }
  sum = warp_sum(acc[0]);
  mag = warp_sum(mg[0]);
}

// The same with the x chunks read from shared memory (xs[lane + 32 j]).
template <int NJ>
__device__ __forceinline__ void router_row_dot(const uint4 (&wv)[NJ], const uint4* xs, int lane,
                                               float& sum, float& mag) {
  uint4 xr[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) xr[j] = xs[lane + 32 * j];
  router_row_dot_regs<NJ>(wv, xr, sum, mag);
}

// Logit with its prior and the stored bound.
template <int NJ>
__device__ __forceinline__ void router_logit_and_bound(float sum, float mag, float prior,
                                                       float& logit, float& bnd) {
  logit = sum + prior;
  bnd = RouterShape<NJ>::kBoundScale * (mag + fabsf(prior)) + kBoundFloor;
}

// ---------------------------------------------------------------- exact logits
// Value * 2^266 as a two's-complement integer in 32-bit digits held in
// int64 (headroom for carries).  A bf16 number is M * 2^(E' - 134) with
// M = 1.m (8 bits) and E' = max(e, 1); a product of two is
// Mx*Mw * 2^(Ex + Ew - 268), i.e. Mx*Mw << (Ex + Ew - 2) after scaling.  An
// fp32 prior M * 2^(E' - 150) becomes M << (E' + 116).
static __device__ __forceinline__ void add_shifted(int64_t* acc, uint64_t mant, int shift,
                                                   bool neg) {
  const int d = shift >> 5;
  const uint64_t v = mant << (shift & 31);
  const int64_t lo = (int64_t)(v & 0xFFFFFFFFull), hi = (int64_t)(v >> 32);
  if (neg) {
    acc[d] -= lo;
    acc[d + 1] -= hi;
  } else {
    acc[d] += lo;
    acc[d + 1] += hi;
  }
}

static __device__ __forceinline__ void add_bf16_product(int64_t* acc, uint32_t xb, uint32_t wb) {
  if ((xb & 0x7FFFu) == 0 || (wb & 0x7FFFu) == 0) return;
  const uint32_t ex = (xb >> 7) & 0xFFu, ew = (wb >> 7) & 0xFFu;
  const uint64_t mx = ex ? ((xb & 0x7Fu) | 0x80u) : (xb & 0x7Fu);
  const uint64_t mw = ew ? ((wb & 0x7Fu) | 0x80u) : (wb & 0x7Fu);
  const int shift = (int)(ex ? ex : 1u) + (int)(ew ? ew : 1u) - 2;
  add_shifted(acc, mx * mw, shift, ((xb ^ wb) >> 15) & 1u);
}

static __device__ __forceinline__ void add_f32(int64_t* acc, float f) {
  const uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) return;
  const uint32_t e = (u >> 23) & 0xFFu;
  const uint64_t m = e ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);
  add_shifted(acc, m, (int)(e ? e : 1u) + 116, u >> 31);
}

// Warp-cooperative exact value of x . w (+ prior); lane 0 writes the
// normalised digits to `out` (shared memory; digit 17 signed, 0..16 unsigned).
static __device__ void exact_logit_warp(const uint16_t* __restrict__ x,
                                        const uint16_t* __restrict__ w, int H,
                                        const float* prior_e, uint32_t* out) {
  const int lane = threadIdx.x & 31;
  int64_t acc[kDigits];
#pragma unroll
  for (int d = 0; d < kDigits; ++d) acc[d] = 0;
  for (int h = lane; h < H; h += 32) add_bf16_product(acc, x[h], w[h]);
  if (lane == 0 && prior_e != nullptr) add_f32(acc, *prior_e);
#pragma unroll
  for (int d = 0; d < kDigits; ++d) {
    int64_t v = acc[d];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    acc[d] = v;
  }
  if (lane == 0) {
    int64_t carry = 0;
#pragma unroll
    for (int d = 0; d < kDigits - 1; ++d) {
      const int64_t t = acc[d] + carry;
      out[d] = (uint32_t)(t & 0xFFFFFFFFll);
      carry = t >> 32;
    }
    out[kDigits - 1] = (uint32_t)(acc[kDigits - 1] + carry);
  }
  __syncwarp();
}

// -1, 0, +1 for a < b, a == b, a > b.
static __device__ __forceinline__ int exact_cmp(const uint32_t* a, const uint32_t* b) {
  const int32_t ta = (int32_t)a[kDigits - 1], tb = (int32_t)b[kDigits - 1];
  if (ta != tb) return ta < tb ? -1 : 1;
  for (int d = kDigits - 2; d >= 0; --d)
    if (a[d] != b[d]) return a[d] < b[d] ? -1 : 1;
  return 0;
}

// Order-preserving map of floats to unsigned keys (larger float, larger key).
static __device__ __forceinline__ uint32_t f32_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

static __device__ __forceinline__ float key_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Does expert a come before expert b in the exact order (larger value first,
// ties to the lower id)?  Computes both exact values (slow path for long runs).
static __device__ bool exact_before(const uint16_t* xt, const uint16_t* router_w,
                                    const float* prior, int H, int a, int b, uint32_t* scratch) {
  uint32_t* va = scratch;
  uint32_t* vb = scratch + kDigits;
  exact_logit_warp(xt, router_w + (size_t)a * H, H, prior ? prior + a : nullptr, va);
  exact_logit_warp(xt, router_w + (size_t)b * H, H, prior ? prior + b : nullptr, vb);
  const int c = exact_cmp(va, vb);
  return c > 0 || (c == 0 && a < b);
}

// Bytes of per-warp shared memory topk_select_warp needs for E experts:
// sel_idx, sel_val, the exact-value cache, scratch, and the run members'
// refined values, bounds and cache flags.
__host__ __device__ constexpr size_t topk_warp_smem(int E) {
  return (size_t)E * 8 + (size_t)(kRunCache + 2) * kDigits * 4 + (size_t)kRunCache * 12;
}

// A tight fp32 logit of one router row, by one warp.  Lane l takes the
// 8-element chunks c = l + 32 j of the row (8 sequential FMAs from zero per
// chunk, chunk sums added in order), then a 5-level butterfly, then the
// prior: depth D = 8 + H/256 + 6.  sum |x w| is computed alongside with the
// same structure; 1 + 2^-8 covers its own rounding, so
// bound = 2 D u (mag (1 + 2^-8) + |prior|) bounds the error (Higham, Accuracy
// and Stability of Numerical Algorithms, Thm. 4.3).  x is a generic pointer
// (global or shared memory); w is global.
static __device__ void tight_logit_warp(const uint16_t* __restrict__ x,
                                        const uint16_t* __restrict__ w, int H,
                                        const float* prior_e, float& logit, float& bnd) {
  const int lane = threadIdx.x & 31;
  float acc = 0.f, mag = 0.f;
  for (int j = 0; j < H / 256; ++j) {
    // x may live in shared memory (the decode kernel keeps its block input there)
    const uint4 xv = reinterpret_cast<const uint4*>(x)[lane + 32 * j];
    const uint4 wv = __ldg(reinterpret_cast<const uint4*>(w) + lane + 32 * j);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
    float sc = 0.f, mc = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float x0 = bf16_lo(xw[q]), x1 = bf16_hi(xw[q]);
      const float w0 = bf16_lo(ww[q]), w1 = bf16_hi(ww[q]);
      sc = fmaf(x0, w0, sc);
      mc = fmaf(fabsf(x0), fabsf(w0), mc);
      sc = fmaf(x1, w1, sc);
      mc = fmaf(fabsf(x1), fabsf(w1), mc);
    }
    acc += sc;
    mag += mc;
  }
  acc = warp_sum(acc);
  mag = warp_sum(mag);
  const float p = prior_e ? *prior_e : 0.f;
  logit = acc + p;
  const float depth = (float)(8 + H / 256 + 6);
  bnd = 2.0f * depth * 5.9604644775390625e-8f * (mag * 1.00390625f + fabsf(p)) + kBoundFloor;
}

// Per-lane sort of (key, id) pairs, best first: larger key, then lower id.
// Bitonic network over N (a power of two) register entries.
template <int N>
__device__ __forceinline__ void sort_lane_desc(uint32_t (&key)[N], int (&id)[N]) {
#pragma unroll
  for (int kk = 2; kk <= N; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j > 0; j >>= 1) {
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int l = i ^ j;
        if (l > i) {
          const bool l_first = key[l] > key[i] || (key[l] == key[i] && id[l] < id[i]);
          const bool i_first = key[i] > key[l] || (key[i] == key[l] && id[i] < id[l]);
          const bool swap = ((i & kk) == 0) ? l_first : i_first;
          if (swap) {
            const uint32_t tk = key[i];
            key[i] = key[l];
            key[l] = tk;
            const int ti = id[i];
            id[i] = id[l];
            id[l] = ti;
          }
        }
      }
    }
  }
}

// Swap entries p and q of the selection (and of the exact-value cache when
// `cache` is given); one warp, positions relative to `base`.
static __device__ __forceinline__ void swap_sel(int* sel_idx, float* sel_val, uint32_t* cache,
                                                int base, int p, int q) {
  const int lane = threadIdx.x & 31;
  if (cache && lane < kDigits) {
    const uint32_t tmp = cache[p * kDigits + lane];
    cache[p * kDigits + lane] = cache[q * kDigits + lane];
    cache[q * kDigits + lane] = tmp;
  }
  if (lane == 0) {
    const int ti = sel_idx[base + p];
    sel_idx[base + p] = sel_idx[base + q];
    sel_idx[base + q] = ti;
    const float tv = sel_val[base + p];
    sel_val[base + p] = sel_val[base + q];
    sel_val[base + q] = tv;
  }
  __syncwarp();
}

// Take entries best first from per-lane sorted lists (key 0 = empty), one per
// iteration, writing sel_idx/sel_val[n] (lane 0).  Stops after `limit`
// entries, when the lists run dry (*closed = 2), or -- if close_on_gap -- once
// n >= k and the next entry is more than thr below the last one taken
// (*closed = 1).  Returns n.
template <int N>
__device__ int extract_sorted(uint32_t (&key)[N], int (&id)[N], int k, int limit, float thr,
                              bool close_on_gap, int* sel_idx, float* sel_val, int* closed) {
  const int lane = threadIdx.x & 31;
  int n = 0;
  *closed = 0;
  while (n < limit) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key[0]);
    if (kmax == 0u) {
      *closed = 2;
      break;
    }
    const uint32_t win =
        __reduce_min_sync(0xffffffffu, key[0] == kmax ? (uint32_t)id[0] : 0xFFFFFFFFu);
    const float wv = key_f32(kmax);
    if (close_on_gap && n >= k) {
      const float last = sel_val[n - 1];
      if (!(last - wv <= thr)) {  // certified gap: the selection is closed
        *closed = 1;
        break;
      }
    }
    if (lane == 0) {
      sel_idx[n] = (int)win;
      sel_val[n] = wv;
    }
    if (key[0] == kmax && id[0] == (int)win) {  // pop this lane's head
#pragma unroll
      for (int i = 0; i < N - 1; ++i) {
        key[i] = key[i + 1];
        id[i] = id[i + 1];
      }
      key[N - 1] = 0u;
      id[N - 1] = 0x7FFFFFFF;
    }
    __syncwarp();
    ++n;
  }
  __syncwarp();
  return n;
}

// Reorder, by exact values, every run of neighbours of sel[0..n) closer than
// thr that reaches into the first k positions (one warp).  The run's members
// are first recomputed with tight fp32 bounds (tight_logit_warp); two
// members whose tight intervals are disjoint are ordered by them, and only
// overlapping ones are compared exactly (values cached on first use).
// cache/scratch: kRunCache*kDigits and 2*kDigits words; tl/tb/have:
// kRunCache entries each (all this warp's shared memory).
static __device__ void resolve_runs(int* sel_idx, float* sel_val, int n, int k, float thr,
                                    const uint16_t* xt, const uint16_t* router_w,
                                    const float* prior, int H, uint32_t* cache,
                                    uint32_t* scratch) {
  const int lane = threadIdx.x & 31;
  float* tl = reinterpret_cast<float*>(scratch + 2 * kDigits);
  float* tb = tl + kRunCache;
  int* have = reinterpret_cast<int*>(tb + kRunCache);
  auto ensure_exact = [&](int a0, int q) {
    if (!have[q]) {
      const int e = sel_idx[a0 + q];
      exact_logit_warp(xt, router_w + (size_t)e * H, H, prior ? prior + e : nullptr, scratch);
      if (lane < kDigits) cache[q * kDigits + lane] = scratch[lane];
      if (lane == 0) have[q] = 1;
      __syncwarp();
    }
  };
  int a = 0;
  while (a < n - 1 && a < k) {
    int b = a;
    while (b + 1 < n && sel_val[b] - sel_val[b + 1] <= thr) ++b;
    if (b > a) {
      const int m = b - a + 1;
      const int need = min(b, k - 1) - a + 1;
      if (m <= kRunCache) {
        for (int q = 0; q < m; ++q) {
          const int e = sel_idx[a + q];
          float l, bb;
          tight_logit_warp(xt, router_w + (size_t)e * H, H, prior ? prior + e : nullptr, l, bb);
          if (lane == 0) {
            tl[q] = l;
            tb[q] = bb;
            have[q] = 0;
          }
        }
        __syncwarp();
        // selection sort of the first `need` positions by (exact desc, id asc)
        for (int p = 0; p < need; ++p) {
          int best = p;
          for (int q = p + 1; q < m; ++q) {
            int c;
            if (tl[q] - tb[q] > tl[best] + tb[best]) {
              c = 1;
            } else if (tl[best] - tb[best] > tl[q] + tb[q]) {
              c = -1;
            } else {
              ensure_exact(a, q);
              ensure_exact(a, best);
              c = exact_cmp(cache + q * kDigits, cache + best * kDigits);
            }
            if (c > 0 || (c == 0 && sel_idx[a + q] < sel_idx[a + best])) best = q;
          }
          __syncwarp();
          if (best != p) {
            swap_sel(sel_idx, sel_val, cache, a, p, best);
            if (lane == 0) {
              const float t0 = tl[p], t1 = tb[p];
              const int h0 = have[p];
              tl[p] = tl[best];
              tb[p] = tb[best];
              have[p] = have[best];
              tl[best] = t0;
              tb[best] = t1;
              have[best] = h0;
            }
            __syncwarp();
          }
        }
      } else {
        for (int p = 0; p < need; ++p) {
          int best = p;
          for (int q = p + 1; q < m; ++q) {
            if (exact_before(xt, router_w, prior, H, sel_idx[a + q], sel_idx[a + best], scratch))
              best = q;
            __syncwarp();
          }
          if (best != p) swap_sel(sel_idx, sel_val, nullptr, a, p, best);
        }
      }
    }
    a = b + 1;
  }
  __syncwarp();
}

// Plain fp32 logits and bounds in global memory (read through L2).
struct PlainLogits {
  const float* l;
  const float* b;
  __device__ __forceinline__ void get(int e, float& logit, float& bnd) const {
    logit = __ldcg(l + e);
    bnd = __ldcg(b + e);
  }
  __device__ __forceinline__ int id(int e) const { return e; }
};

// The k experts of one token in exact order, by one warp.
//   src: the token's E fp32 logits and their bounds (src.get(i, logit, bound))
//        and the expert id of entry i (src.id(i); entries may be a subset of
//        the experts in any order)
//   xt: the token's bf16 x (global); router_w, prior: router weights and prior
//   smem: topk_warp_smem(E) bytes of this warp's shared memory
// On return sel_idx[0..k) / sel_val[0..k) (inside smem) hold the experts in
// descending exact logit (ties to the lower id) and their fp32 logits.
//
// Lane l holds experts l*MAXV .. l*MAXV + MAXV-1 (E <= 32*MAXV), sorted best
// first.  Extraction repeatedly takes the best head over the warp (two warp
// reductions per expert) until k are taken and the gap to the next exceeds
// 2*beta, beta = the largest bound of the token; every run of neighbours
// closer than 2*beta is then reordered by exact values.  Runs are bounded by
// gaps > 2*beta, so exact values never cross a run boundary, and experts left
// behind are beaten by k taken ones.
template <int MAXV, typename Src>
__device__ void topk_select_warp_src(const Src& src, int E, int k, const uint16_t* xt,
                                     const uint16_t* router_w, const float* prior, int H,
                                     uint8_t* smem, int** sel_idx_out, float** sel_val_out) {
  const int lane = threadIdx.x & 31;
  int* sel_idx = reinterpret_cast<int*>(smem);
  float* sel_val = reinterpret_cast<float*>(smem + (size_t)E * 4);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem + (size_t)E * 8);
  uint32_t* scratch = cache + kRunCache * kDigits;
  *sel_idx_out = sel_idx;
  *sel_val_out = sel_val;

  uint32_t key[MAXV];
  int id[MAXV];
  uint32_t bmax = 0;  // bounds are non-negative: their bits order like the values
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = lane * MAXV + i;
    float l = 0.f, bnd = 0.f;
    if (e < E) src.get(e, l, bnd);
    if (l != l) l = -INFINITY;  // a NaN logit from bad input ranks as -inf
    key[i] = (e < E) ? f32_key(l) : 0u;  // key 0: empty (below every real logit)
    id[i] = (e < E) ? src.id(e) : 0x7FFFFFFF;
    if (e < E) bmax = max(bmax, __float_as_uint(bnd));
  }
  const float thr = 2.0f * __uint_as_float(__reduce_max_sync(0xffffffffu, bmax));
  sort_lane_desc<MAXV>(key, id);
  int closed;
  const int n = extract_sorted<MAXV>(key, id, k, E, thr, true, sel_idx, sel_val, &closed);
  resolve_runs(sel_idx, sel_val, n, k, thr, xt, router_w, prior, H, cache, scratch);
}

template <int MAXV>
__device__ void topk_select_warp(const float* lrow, const float* brow, int E, int k,
                                 const uint16_t* xt, const uint16_t* router_w,
                                 const float* prior, int H, uint8_t* smem, int** sel_idx_out,
                                 float** sel_val_out) {
  topk_select_warp_src<MAXV>(PlainLogits{lrow, brow}, E, k, xt, router_w, prior, H, smem,
                             sel_idx_out, sel_val_out);
}

// The same selection by all `nw` warps of a CTA (E <= nw * 32 * V), for
// latency: warp w rank-sorts experts [32 V w, 32 V (w + 1)) across its lanes
// (best first; ties to the lower id) into `lists` (shared memory, E entries
// of (key, id)), then warp 0 merges the nw lists -- lane l < nw holds the
// head of list l -- with the closing rule and the run resolution of
// topk_select_warp_src, so the result is identical.  Every thread of the CTA
// calls; the selection is complete on return (one __syncthreads inside, none
// after: sel_idx / sel_val are written by warp 0).
//   smem: topk_warp_smem(E) bytes; lists: nw * 32 V entries of 8 bytes (whole
//   lists: the padding past E is written too); bmx: nw floats after them.
template <int V, typename Src>
__device__ void topk_select_block(const Src& src, int E, int k, const uint16_t* xt,
                                  const uint16_t* router_w, const float* prior, int H,
                                  uint8_t* smem, uint2* lists, float* bmx, int** sel_idx_out,
                                  float** sel_val_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  int* sel_idx = reinterpret_cast<int*>(smem);
  float* sel_val = reinterpret_cast<float*>(smem + (size_t)E * 4);
  uint32_t* cache = reinterpret_cast<uint32_t*>(smem + (size_t)E * 8);
  uint32_t* scratch = cache + kRunCache * kDigits;
  *sel_idx_out = sel_idx;
  *sel_val_out = sel_val;
  constexpr int L = 32 * V;  // list length
  uint32_t key[V];
  int id[V];
  uint32_t bm = 0;
#pragma unroll
  for (int v = 0; v < V; ++v) {
    const int e = warp * L + lane * V + v;
    float l = 0.f, bnd = 0.f;
    if (e < E) src.get(e, l, bnd);
    if (l != l) l = -INFINITY;
    key[v] = (e < E) ? f32_key(l) : 0u;
    id[v] = (e < E) ? src.id(e) : e;  // padding: key 0 (never taken), a distinct id
    if (e < E) bm = max(bm, __float_as_uint(bnd));
  }
  bm = __reduce_max_sync(0xffffffffu, bm);
  if (warp * L < E) {
    // rank sort of the warp's list: an entry's position is the number of
    // entries before it (larger key, or equal key and lower id), counted
    // against 64-bit keys read back from shared memory as broadcasts --
    // independent compares instead of a network of dependent shuffles
    uint64_t ck[V];
    uint64_t* cks = reinterpret_cast<uint64_t*>(lists + warp * L);
#pragma unroll
    for (int v = 0; v < V; ++v) {
      ck[v] = ((uint64_t)key[v] << 32) | (uint32_t)~(uint32_t)id[v];
      cks[lane * V + v] = ck[v];
    }
    __syncwarp();
    int rank[V];
#pragma unroll
    for (int v = 0; v < V; ++v) rank[v] = 0;
    const uint4* kp = reinterpret_cast<const uint4*>(cks);
#pragma unroll 4
    for (int u = 0; u < L / 2; ++u) {
      const uint4 w = kp[u];
      const uint64_t a0 = ((uint64_t)w.y << 32) | w.x, a1 = ((uint64_t)w.w << 32) | w.z;
#pragma unroll
      for (int v = 0; v < V; ++v) rank[v] += (int)(a0 > ck[v]) + (int)(a1 > ck[v]);
    }
    __syncwarp();
#pragma unroll
    for (int v = 0; v < V; ++v) lists[warp * L + rank[v]] = make_uint2(key[v], (uint32_t)id[v]);
  }
  if (lane == 0) bmx[warp] = __uint_as_float(bm);
  __syncthreads();
  if (warp != 0) return;
  float thr = 0.f;
  for (int w = 0; w < nw; ++w) thr = fmaxf(thr, bmx[w]);
  thr *= 2.0f;
  const int nl = (E + L - 1) / L;  // lists that hold experts
  int pos = 0;
  uint2 head = (lane < nl) ? lists[lane * L] : make_uint2(0u, 0x7FFFFFFFu);
  const int len = (lane < nl) ? min(L, E - lane * L) : 0;
  int n = 0;
  while (n < E) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, head.x);
    if (kmax == 0u) break;
    const uint32_t win = __reduce_min_sync(0xffffffffu, head.x == kmax ? head.y : 0xFFFFFFFFu);
    const float wv = key_f32(kmax);
    if (n >= k) {
      const float last = sel_val[n - 1];
      if (!(last - wv <= thr)) break;  // certified gap: the selection is closed
    }
    if (lane == 0) {
      sel_idx[n] = (int)win;
      sel_val[n] = wv;
    }
    if (head.x == kmax && head.y == win) {  // advance this list
      ++pos;
      head = pos < len ? lists[lane * L + pos] : make_uint2(0u, 0x7FFFFFFFu);
    }
    __syncwarp();
    ++n;
  }
  __syncwarp();
  resolve_runs(sel_idx, sel_val, n, k, thr, xt, router_w, prior, H, cache, scratch);
}

// Renormalised softmax weight of selected expert `lane` (lanes < k), i.e.
// exp(l_j - m) / sum_i exp(l_i - m) over the k selected logits.
static __device__ __forceinline__ float renormalised_weight(const float* sel_val, int k) {
  const int lane = threadIdx.x & 31;
  // any m that keeps exp(l - m) finite gives the same weights; the first
  // selected logit is within rounding of the largest
  const float mx = sel_val[0];
  const float ej = (lane < k) ? __expf(sel_val[lane] - mx) : 0.f;
  const float den = warp_sum(ej);
  return ej / den;
}

}  // namespace rt
}  // namespace moe
