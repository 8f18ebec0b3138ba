// router.cu -- router logits, exact top-k with renormalised softmax weights,
// and the shared-expert sigmoid gate.
//
// Routing follows the Swiftlet README (wpnews page, "How it works"): each
// layer sends every token to k of E experts.  The selection ranks the exact
// real logits l = x . Wr_e (+ prior_e): a bf16 x bf16 product is exact in
// fp32, the fp32 sum carries a rigorous error bound from its summation depth,
// and where two candidates are closer than twice the bound their exact values
// are compared with an integer superaccumulator (Kulisch accumulation), ties
// going to the lower expert id.  The weights are the softmax probabilities
// of the k selected experts renormalised to sum to one, i.e.
// w_j = exp(l_j - m) / sum_i exp(l_i - m) over the selected i.
#include <cstdio>
#include <mutex>

#include "device_util.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kRouterWarps = 8;   // one router row per warp
constexpr int kRouterTC = 8;      // tokens staged per pass
constexpr int kTopkWarps = 4;     // tokens per top-k CTA
constexpr int kRunCache = 32;     // exact values cached per warp
constexpr int kDigits = 18;       // 32-bit digits of the superaccumulator

// ---------------------------------------------------------------- logits
// Row r = blockIdx.x * 8 + warp (r == E is the shared gate vector).  Lane l
// holds the 8-element chunks c = l + 32 j, j < NJ, of the row (H = 256 NJ).
// Summation: 8 sequential FMAs per chunk, a pairwise tree over the NJ chunk
// sums, a 5-level butterfly across lanes, one addition of the prior:
// depth D = 8 + log2(NJ) + 6.  Any such sum is within gamma_D * sum|x w| of
// the exact one (Higham, Accuracy and Stability, Thm. 4.3); the bound stored
// is 2 * D * 2^-24 * (sum|x w| + |prior|) + 2^-120 (the last term covers
// products that underflow in fp32).
template <int NJ>
__global__ void __launch_bounds__(256) router_logits_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ router_w,
    const float* __restrict__ prior, const uint16_t* __restrict__ shared_gate_w, int E,
    float* __restrict__ logits, float* __restrict__ bound, float* __restrict__ gate_z) {
  constexpr int H = NJ * 256;
  constexpr int HV = H / 8;  // uint4 chunks per row
  constexpr int LOG2NJ = (NJ >= 32) ? 5 : (NJ >= 16) ? 4 : (NJ >= 8) ? 3 : (NJ >= 4) ? 2 : (NJ >= 2) ? 1 : 0;
  constexpr float kBoundScale = 2.0f * (float)(8 + LOG2NJ + 6) * 5.9604644775390625e-8f;
  extern __shared__ uint4 xs[];  // [kRouterTC][HV]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRouterWarps + warp;
  const bool active = r <= E;
  const uint16_t* wrow = (r < E) ? router_w + (size_t)r * H : shared_gate_w;
  uint4 wv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    wv[j] = active ? __ldg(reinterpret_cast<const uint4*>(wrow) + lane + 32 * j) : make_uint4(0, 0, 0, 0);
  const float pb = (r < E && prior != nullptr) ? prior[r] : 0.f;
  for (int t0 = 0; t0 < T; t0 += kRouterTC) {
    const int tc = min(kRouterTC, T - t0);
    __syncthreads();
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t0 * H);
    for (int i = threadIdx.x; i < tc * HV; i += blockDim.x) xs[i] = src[i];
    __syncthreads();
    if (!active) continue;
    for (int tt = 0; tt < tc; ++tt) {
      float acc[NJ], mag[NJ];
#pragma unroll
      for (int j = 0; j < NJ; ++j) {
        const uint4 xv = xs[tt * HV + lane + 32 * j];
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
        mag[j] = m;
      }
#pragma unroll
      for (int s = NJ / 2; s > 0; s >>= 1) {
#pragma unroll
        for (int j = 0; j < s; ++j) {
          acc[j] += acc[j + s];
          mag[j] += mag[j + s];
        }
      }
      const float sum = warp_sum(acc[0]);
      const float mg = warp_sum(mag[0]);
      if (lane == 0) {
        const int t = t0 + tt;
        if (r < E) {
          logits[(size_t)t * E + r] = sum + pb;
          bound[(size_t)t * E + r] = kBoundScale * (mg + fabsf(pb)) + 7.52316384526264e-37f;
        } else {
          gate_z[t] = sum;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- exact logits
// Value * 2^266 as a two's-complement integer in 32-bit digits held in
// int64 (headroom for carries).  A bf16 number is M * 2^(E' - 134) with
// M = 1.m (8 bits) and E' = max(e, 1); a product of two is
// Mx*Mw * 2^(Ex + Ew - 268), i.e. Mx*Mw << (Ex + Ew - 2) after scaling.  An
// fp32 prior M * 2^(E' - 150) becomes M << (E' + 116).
__device__ __forceinline__ void add_shifted(int64_t* acc, uint64_t mant, int shift, bool neg) {
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

__device__ __forceinline__ void add_bf16_product(int64_t* acc, uint32_t xb, uint32_t wb) {
  if ((xb & 0x7FFFu) == 0 || (wb & 0x7FFFu) == 0) return;
  const uint32_t ex = (xb >> 7) & 0xFFu, ew = (wb >> 7) & 0xFFu;
  const uint64_t mx = ex ? ((xb & 0x7Fu) | 0x80u) : (xb & 0x7Fu);
  const uint64_t mw = ew ? ((wb & 0x7Fu) | 0x80u) : (wb & 0x7Fu);
  const int shift = (int)(ex ? ex : 1u) + (int)(ew ? ew : 1u) - 2;
  add_shifted(acc, mx * mw, shift, ((xb ^ wb) >> 15) & 1u);
}

__device__ __forceinline__ void add_f32(int64_t* acc, float f) {
  const uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) return;
  const uint32_t e = (u >> 23) & 0xFFu;
  const uint64_t m = e ? ((u & 0x7FFFFFu) | 0x800000u) : (u & 0x7FFFFFu);
  add_shifted(acc, m, (int)(e ? e : 1u) + 116, u >> 31);
}

// Warp-cooperative exact value of x . w (+ prior); lane 0 writes the
// normalised digits to `out` (shared memory; digit 17 signed, 0..16 unsigned).
__device__ void exact_logit_warp(const uint16_t* __restrict__ x, const uint16_t* __restrict__ w,
                                 int H, const float* prior_e, uint32_t* out) {
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
__device__ __forceinline__ int exact_cmp(const uint32_t* a, const uint32_t* b) {
  const int32_t ta = (int32_t)a[kDigits - 1], tb = (int32_t)b[kDigits - 1];
  if (ta != tb) return ta < tb ? -1 : 1;
  for (int d = kDigits - 2; d >= 0; --d)
    if (a[d] != b[d]) return a[d] < b[d] ? -1 : 1;
  return 0;
}

__device__ __forceinline__ uint32_t f32_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Does expert a come before expert b in the exact order (larger value first,
// ties to the lower id)?  Computes both exact values (slow path for long runs).
__device__ bool exact_before(const uint16_t* xt, const uint16_t* router_w, const float* prior,
                             int H, int a, int b, uint32_t* scratch) {
  uint32_t* va = scratch;
  uint32_t* vb = scratch + kDigits;
  exact_logit_warp(xt, router_w + (size_t)a * H, H, prior ? prior + a : nullptr, va);
  exact_logit_warp(xt, router_w + (size_t)b * H, H, prior ? prior + b : nullptr, vb);
  const int c = exact_cmp(va, vb);
  return c > 0 || (c == 0 && a < b);
}

// ---------------------------------------------------------------- top-k
// One warp per token.  Extract experts in descending fp32 order (ties to the
// lower id) until k are taken and the gap to the next one exceeds 2*beta,
// beta = max bound of the token; then every run of neighbours closer than
// 2*beta is reordered by exact values.  Runs are bounded by gaps > 2*beta,
// so exact values never cross a run boundary.
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(
    const float* __restrict__ logits, const float* __restrict__ bound,
    const float* __restrict__ gate_z, const uint16_t* __restrict__ x,
    const uint16_t* __restrict__ router_w, const float* __restrict__ prior, int T, int E, int H,
    int k, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* __restrict__ gate) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= T) return;
  // per-warp smem: sel_idx[E], sel_val[E], cache[kRunCache][kDigits], scratch[2*kDigits]
  uint8_t* base = smem_raw + (size_t)warp * ((size_t)E * 8 + (kRunCache + 2) * kDigits * 4);
  int* sel_idx = reinterpret_cast<int*>(base);
  float* sel_val = reinterpret_cast<float*>(base + (size_t)E * 4);
  uint32_t* cache = reinterpret_cast<uint32_t*>(base + (size_t)E * 8);
  uint32_t* scratch = cache + kRunCache * kDigits;

  constexpr int MAXV = kMaxE / 32;
  float v[MAXV];
  float beta = 0.f;
  const float* lrow = logits + (size_t)t * E;
  const float* brow = bound + (size_t)t * E;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = lane + 32 * i;
    // NaN marks "not a candidate" (padding and experts already taken); a NaN
    // logit from bad input ranks as -inf.
    const float l = (e < E) ? lrow[e] : __int_as_float(0x7fc00000);
    v[i] = (e < E && l != l) ? -INFINITY : l;
    if (e < E) beta = fmaxf(beta, brow[e]);
  }
  beta = warp_max(beta);
  const float thr = 2.0f * beta;

  // extraction
  int n = 0;
  while (n < E) {
    float lb = -INFINITY;
    int li = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
      const int e = lane + 32 * i;
      if (v[i] > lb || (v[i] == lb && e < li)) {
        lb = v[i];
        li = e;
      }
    }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, li == 0x7FFFFFFF ? 0u : f32_key(lb));
    const uint32_t mine = (li != 0x7FFFFFFF && f32_key(lb) == kmax) ? (uint32_t)li : 0xFFFFFFFFu;
    const uint32_t win = __reduce_min_sync(0xffffffffu, mine);
    if (win == 0xFFFFFFFFu) break;  // no candidates left
    const float wv = __shfl_sync(0xffffffffu, lb, (int)(win & 31));
    if (n >= k) {
      const float last = sel_val[n - 1];
      if (!(last - wv <= thr)) break;  // certified gap: the selection is closed
    }
    if (lane == 0) {
      sel_idx[n] = (int)win;
      sel_val[n] = wv;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < MAXV; ++i)
      if (lane + 32 * i == (int)win) v[i] = __int_as_float(0x7fc00000);
    ++n;
  }
  __syncwarp();

  // resolve runs of neighbours closer than thr
  const uint16_t* xt = x + (size_t)t * H;
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
          exact_logit_warp(xt, router_w + (size_t)e * H, H, prior ? prior + e : nullptr,
                           scratch);
          if (lane < kDigits) cache[q * kDigits + lane] = scratch[lane];
          __syncwarp();
        }
        // selection sort of the first `need` positions by (exact desc, id asc)
        for (int p = 0; p < need; ++p) {
          int best = p;
          for (int q = p + 1; q < m; ++q) {
            const int c = exact_cmp(cache + q * kDigits, cache + best * kDigits);
            if (c > 0 || (c == 0 && sel_idx[a + q] < sel_idx[a + best])) best = q;
          }
          __syncwarp();
          if (best != p && lane < kDigits) {
            const uint32_t tmp = cache[p * kDigits + lane];
            cache[p * kDigits + lane] = cache[best * kDigits + lane];
            cache[best * kDigits + lane] = tmp;
          }
          if (best != p && lane == 0) {
            const int ti = sel_idx[a + p];
            sel_idx[a + p] = sel_idx[a + best];
            sel_idx[a + best] = ti;
            const float tv = sel_val[a + p];
            sel_val[a + p] = sel_val[a + best];
            sel_val[a + best] = tv;
          }
          __syncwarp();
        }
      } else {
        for (int p = 0; p < need; ++p) {
          int best = p;
          for (int q = p + 1; q < m; ++q) {
            if (exact_before(xt, router_w, prior, H, sel_idx[a + q], sel_idx[a + best], scratch))
              best = q;
            __syncwarp();
          }
          if (best != p && lane == 0) {
            const int ti = sel_idx[a + p];
            sel_idx[a + p] = sel_idx[a + best];
            sel_idx[a + best] = ti;
            const float tv = sel_val[a + p];
            sel_val[a + p] = sel_val[a + best];
            sel_val[a + best] = tv;
          }
          __syncwarp();
        }
      }
    }
    a = b + 1;
  }
  __syncwarp();

  // renormalised softmax weights of the k selected experts
  float mx = -INFINITY;
  for (int j = 0; j < k; ++j) mx = fmaxf(mx, sel_val[j]);
  const float ej = (lane < k) ? __expf(sel_val[lane] - mx) : 0.f;
  const float den = warp_sum(ej);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = sel_idx[lane];
    topk_w[(size_t)t * k + lane] = ej / den;
  }
  if (lane == 0) gate[t] = 1.0f / (1.0f + __expf(-gate_z[t]));
}

}  // namespace

cudaError_t launch_router(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches) {
  const int E = c.d.E, H = c.d.H;
  const int grid = (E + 1 + kRouterWarps - 1) / kRouterWarps;
  const size_t smem = (size_t)kRouterTC * H * 2;
  switch (H / 256) {
#define MOE_ROUTER_CASE(NJ)                                                                    \
  case NJ:                                                                                     \
    router_logits_kernel<NJ><<<grid, kRouterWarps * 32, smem, st>>>(                           \
        a.x, a.T, c.router_w, c.router_bias, c.shared_gate_w, E, c.ws.logits, c.ws.bound,      \
        c.ws.gate_z);                                                                          \
    break;
    MOE_ROUTER_CASE(1)
    MOE_ROUTER_CASE(2)
    MOE_ROUTER_CASE(4)
    MOE_ROUTER_CASE(8)
    MOE_ROUTER_CASE(16)
    MOE_ROUTER_CASE(32)
#undef MOE_ROUTER_CASE
    default:
      return cudaErrorInvalidValue;
  }
  ++*launches;
  return cudaGetLastError();
}

cudaError_t prepare_router(const Ctx& c) {
  const size_t smem = (size_t)kRouterTC * c.d.H * 2;
  cudaError_t e = cudaSuccess;
  switch (c.d.H / 256) {
#define MOE_ROUTER_ATTR(NJ)                                                                   \
  case NJ:                                                                                    \
    e = cudaFuncSetAttribute(router_logits_kernel<NJ>,                                        \
                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);         \
    break;
    MOE_ROUTER_ATTR(1)
    MOE_ROUTER_ATTR(2)
    MOE_ROUTER_ATTR(4)
    MOE_ROUTER_ATTR(8)
    MOE_ROUTER_ATTR(16)
    MOE_ROUTER_ATTR(32)
#undef MOE_ROUTER_ATTR
    default:
      return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  // The limit is per kernel, not per context: size it for the largest E so
  // that preparing a small context never lowers it under a larger one.
  const size_t tsmem = ((size_t)kMaxE * 8 + (kRunCache + 2) * kDigits * 4) * kTopkWarps;
  return cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)tsmem);
}

cudaError_t launch_topk(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches) {
  const int E = c.d.E;
  const size_t per_warp = (size_t)E * 8 + (kRunCache + 2) * kDigits * 4;
  const size_t smem = per_warp * kTopkWarps;
  const int grid = (a.T + kTopkWarps - 1) / kTopkWarps;
  topk_kernel<<<grid, kTopkWarps * 32, smem, st>>>(c.ws.logits, c.ws.bound, c.ws.gate_z, a.x,
                                                    c.router_w, c.router_bias, a.T, E, c.d.H,
                                                    c.d.k, a.topk_idx, a.topk_w, c.ws.gate);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free routing (moe_route_static).
//
// Some callers cannot call cudaMalloc at all: code whose device memory is
// owned by a host application's own allocator, code that must not trigger
// the implicit synchronisation an allocation can cause, code that only
// enqueues work onto streams it is handed.  For them this entry point runs
// the same router and top-k kernels as moe_forward, taking every input and
// output from the caller and keeping its intermediates (fp32 logits, their
// error bounds, the shared-gate pre-activations) in the file-scope device
// array below.  The array is loaded with the library and stays resident on
// every device that loads it until the process exits.
namespace moe {
namespace {

constexpr int kStaticMaxLogits = MOE_STATIC_ROUTE_MAX_LOGITS;  // T * E
constexpr int kStaticMaxT = MOE_STATIC_ROUTE_MAX_T;
constexpr int kStaticMaxDevices = 64;

// [0, kStaticMaxLogits): logits, [kStaticMaxLogits, 2*kStaticMaxLogits):
// bounds, then kStaticMaxT shared-gate pre-activations.  Every call writes
// each element it later reads, so nothing needs clearing between calls.
static __device__ __align__(256) float g_route_scratch[2 * kStaticMaxLogits + kStaticMaxT];

std::mutex g_static_mu;
float* g_static_ptr[kStaticMaxDevices] = {};

// Once per device, with that device current: the device address of the
// array (its host-side name is only a stand-in) and the kernels' dynamic
// shared-memory limits.
cudaError_t static_route_setup(int dev, float** out) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    float* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_route_scratch);
    if (e != cudaSuccess) return e;
    const int max_smem_router = kRouterTC * kMaxH * 2;
    const cudaError_t attrs[] = {
        cudaFuncSetAttribute(router_logits_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_router),
        cudaFuncSetAttribute(router_logits_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_router),
        cudaFuncSetAttribute(router_logits_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_router),
        cudaFuncSetAttribute(router_logits_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_router),
        cudaFuncSetAttribute(router_logits_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_router),
        cudaFuncSetAttribute(router_logits_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem_router),
        cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(((size_t)kMaxE * 8 + (kRunCache + 2) * kDigits * 4) * kTopkWarps))};
    for (cudaError_t a : attrs)
      if (a != cudaSuccess) return a;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_static(const void* x, int T, const uint16_t* router_w,
                                const float* router_bias, const uint16_t* shared_gate_w, int E,
                                int k, int hidden, int32_t* topk_idx, float* topk_w,
                                float* shared_gate, void* stream) {
  using namespace moe;
  char msg[256];
  if (T < 0 || T > kStaticMaxT) {
    snprintf(msg, sizeof msg, "moe_route_static: T=%d not in [0, %d]", T, kStaticMaxT);
    return set_global_msg(MOE_ERR_INVALID_ARG, msg);
  }
  if (E < 1 || E > kMaxE || k < 1 || k > E || k > kMaxK) {
    snprintf(msg, sizeof msg, "moe_route_static: E=%d, k=%d out of range", E, k);
    return set_global_msg(MOE_ERR_INVALID_ARG, msg);
  }
  if (hidden < 256 || hidden > kMaxH || hidden % 256 != 0) {
    snprintf(msg, sizeof msg, "moe_route_static: hidden=%d must be a multiple of 256 in [256, %d]",
             hidden, kMaxH);
    return set_global_msg(MOE_ERR_UNSUPPORTED, msg);
  }
  if ((int64_t)T * E > kStaticMaxLogits) {
    snprintf(msg, sizeof msg,
             "moe_route_static: T*E=%lld exceeds the static scratch limit of %d logits",
             (long long)T * E, kStaticMaxLogits);
    return set_global_msg(MOE_ERR_INVALID_ARG, msg);
  }
  if (T == 0) return MOE_OK;
  if (!x || !router_w || !shared_gate_w || !topk_idx || !topk_w || !shared_gate)
    return set_global_msg(MOE_ERR_INVALID_ARG, "moe_route_static: a required pointer is NULL");
  if ((((uintptr_t)x) | ((uintptr_t)router_w) | ((uintptr_t)shared_gate_w)) & 15)
    return set_global_msg(MOE_ERR_INVALID_ARG,
                          "moe_route_static: x, router_w and shared_gate_w must be 16-byte aligned");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kStaticMaxDevices)
    return set_global_msg(MOE_ERR_CUDA, "moe_route_static: no usable current device");
  float* base = nullptr;
  e = static_route_setup(dev, &base);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "moe_route_static: set-up failed: %s", cudaGetErrorString(e));
    return set_global_msg(MOE_ERR_CUDA, msg);
  }
  float* logits = base;
  float* bound = base + kStaticMaxLogits;
  float* gate_z = base + 2 * kStaticMaxLogits;
  cudaStream_t st = (cudaStream_t)stream;
  const uint16_t* xb = (const uint16_t*)x;
  const int grid = (E + 1 + kRouterWarps - 1) / kRouterWarps;
  const size_t smem = (size_t)kRouterTC * hidden * 2;
  switch (hidden / 256) {
    case 1: router_logits_kernel<1><<<grid, kRouterWarps * 32, smem, st>>>(xb, T, router_w, router_bias, shared_gate_w, E, logits, bound, gate_z); break;
    case 2: router_logits_kernel<2><<<grid, kRouterWarps * 32, smem, st>>>(xb, T, router_w, router_bias, shared_gate_w, E, logits, bound, gate_z); break;
    case 4: router_logits_kernel<4><<<grid, kRouterWarps * 32, smem, st>>>(xb, T, router_w, router_bias, shared_gate_w, E, logits, bound, gate_z); break;
    case 8: router_logits_kernel<8><<<grid, kRouterWarps * 32, smem, st>>>(xb, T, router_w, router_bias, shared_gate_w, E, logits, bound, gate_z); break;
    case 16: router_logits_kernel<16><<<grid, kRouterWarps * 32, smem, st>>>(xb, T, router_w, router_bias, shared_gate_w, E, logits, bound, gate_z); break;
    case 32: router_logits_kernel<32><<<grid, kRouterWarps * 32, smem, st>>>(xb, T, router_w, router_bias, shared_gate_w, E, logits, bound, gate_z); break;
    default:
      return set_global_msg(MOE_ERR_UNSUPPORTED, "moe_route_static: unsupported hidden size");
  }
  const size_t tsmem = ((size_t)E * 8 + (kRunCache + 2) * kDigits * 4) * kTopkWarps;
  topk_kernel<<<(T + kTopkWarps - 1) / kTopkWarps, kTopkWarps * 32, tsmem, st>>>(
      logits, bound, gate_z, xb, router_w, router_bias, T, E, hidden, k, topk_idx, topk_w,
      shared_gate);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "moe_route_static: launch failed: %s", cudaGetErrorString(e));
    return set_global_msg(MOE_ERR_CUDA, msg);
  }
  return MOE_OK;
}
