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
#include "routing_common.cuh"

namespace moe {

namespace {

using namespace rt;

constexpr int kRouterWarps = 8;   // one router row per warp
constexpr int kRouterTC = 8;      // tokens staged per pass
constexpr int kTopkWarps = 4;     // tokens per top-k CTA

// ---------------------------------------------------------------- logits
// Row r = blockIdx.x * 8 + warp (r == E is the shared gate vector).  Lane l
// holds the 8-element chunks c = l + 32 j, j < NJ, of the row (H = 256 NJ);
// router_row_dot fixes the summation structure the stored bound relies on.
template <int NJ>
__global__ void __launch_bounds__(256) router_logits_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ router_w,
    const float* __restrict__ prior, const uint16_t* __restrict__ shared_gate_w, int E,
    float* __restrict__ logits, float* __restrict__ bound, float* __restrict__ gate_z) {
  constexpr int H = RouterShape<NJ>::H;
  constexpr int HV = RouterShape<NJ>::HV;
  extern __shared__ uint4 xs[];  // [kRouterTC][HV]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRouterWarps + warp;
  const bool active = r <= E;
  const uint16_t* wrow = (r < E) ? router_w + (size_t)r * H : shared_gate_w;
  uint4 wv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    wv[j] = active ? __ldg(reinterpret_cast<const uint4*>(wrow) + lane + 32 * j)
                   : make_uint4(0, 0, 0, 0);
  const float pb = (r < E && prior != nullptr) ? prior[r] : 0.f;
  for (int t0 = 0; t0 < T; t0 += kRouterTC) {
    const int tc = min(kRouterTC, T - t0);
    __syncthreads();
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t0 * H);
    for (int i = threadIdx.x; i < tc * HV; i += blockDim.x) xs[i] = src[i];
    __syncthreads();
    if (!active) continue;
    for (int tt = 0; tt < tc; ++tt) {
      float sum, mg;
      router_row_dot<NJ>(wv, xs + tt * HV, lane, sum, mg);
      if (lane == 0) {
        const int t = t0 + tt;
        if (r < E) {
          float l, b;
          router_logit_and_bound<NJ>(sum, mg, pb, l, b);
          logits[(size_t)t * E + r] = l;
          bound[(size_t)t * E + r] = b;
        } else {
          gate_z[t] = sum;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- top-k
// One warp per token (see topk_select_warp), then the renormalised softmax
// weights of the k selected experts and the shared gate sigmoid(x . wsg).
template <int MAXV>
__global__ void __launch_bounds__(kTopkWarps * 32) topk_kernel(
    const float* __restrict__ logits, const float* __restrict__ bound,
    const float* __restrict__ gate_z, const uint16_t* __restrict__ x,
    const uint16_t* __restrict__ router_w, const float* __restrict__ prior, int T, int E, int H,
    int k, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* __restrict__ gate) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= T) return;
  int* sel_idx;
  float* sel_val;
  topk_select_warp<MAXV>(logits + (size_t)t * E, bound + (size_t)t * E, E, k, x + (size_t)t * H,
                         router_w, prior, H, smem_raw + (size_t)warp * topk_warp_smem(E),
                         &sel_idx, &sel_val);
  const float w = renormalised_weight(sel_val, k);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = sel_idx[lane];
    topk_w[(size_t)t * k + lane] = w;
  }
  if (lane == 0) gate[t] = 1.0f / (1.0f + __expf(-gate_z[t]));
}

// ---------------------------------------------------------------- many tokens
// For many tokens the logits are a GEMM [T x H] . [H x E]: register-tiled
// fp32 FMAs, each CTA a tile of kTT tokens x kTE experts over a slice of H
// (the slices split H when there are too few tiles to fill the GPU).
// Summation structure of every logit: sequential FMAs over a chunk of kTK
// terms from zero, the chunk sums of a slice added in order, the slice sums
// added in order, then the prior, so a product passes through at most
// D = kTK + H / kTK + slices + 1 roundings.  The bound uses twice
// gamma_D times an upper bound of sum |x w| + |prior| (Higham, Accuracy and
// Stability of Numerical Algorithms, Thm. 4.3); sum |x_h w_h| <= |x|_2 |w|_2
// (Cauchy-Schwarz), with the 2-norms from router_norms_kernel.
constexpr int kTT = 64, kTE = 128, kTK = 64;

// Warp per row: rows r < T are tokens (2-norm bound and x . wsg), rows
// T <= r < T + E are router rows (2-norm bound).  A warp's fp32 sum of
// squares has depth H/256 * 8 + 5 <= 261, so multiplying its square root
// by 1 + 2^-8 bounds the exact norm from above.
__global__ void __launch_bounds__(256) router_norms_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ router_w, int E,
    const uint16_t* __restrict__ wsg, int H, float* __restrict__ xnorm,
    float* __restrict__ wnorm, float* __restrict__ gate_z) {
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (row >= T + E) return;
  const bool tok = row < T;
  const uint16_t* r = tok ? x + (size_t)row * H : router_w + (size_t)(row - T) * H;
  float ss = 0.f, dz = 0.f;
  for (int c = lane; c < H / 8; c += 32) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(r) + c);
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
    uint32_t gw[4] = {0, 0, 0, 0};
    if (tok) {
      const uint4 gv = __ldg(reinterpret_cast<const uint4*>(wsg) + c);
      gw[0] = gv.x; gw[1] = gv.y; gw[2] = gv.z; gw[3] = gv.w;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a0 = bf16_lo(vw[q]), a1 = bf16_hi(vw[q]);
      ss = fmaf(a0, a0, ss);
      ss = fmaf(a1, a1, ss);
      dz = fmaf(a0, bf16_lo(gw[q]), dz);
      dz = fmaf(a1, bf16_hi(gw[q]), dz);
    }
  }
  ss = warp_sum(ss);
  dz = warp_sum(dz);
  if (lane == 0) {
    const float n = sqrtf(ss) * 1.00390625f;
    if (tok) {
      xnorm[row] = n;
      gate_z[row] = dz;
    } else {
      wnorm[row - T] = n;
    }
  }
}

// Logit bound of the structure above.
__device__ __forceinline__ void tile_logit_and_bound(float sum, float p, float xn, float wn,
                                                     int H, int slices, float& l, float& b) {
  const float scale =
      2.0f * (float)(kTK + H / kTK + slices + 1) * 5.9604644775390625e-8f * 1.00390625f;
  l = sum + p;
  b = scale * (xn * wn + fabsf(p)) + kBoundFloor;
}

// blockIdx.z = slice of H (chunks [z * cps, (z + 1) * cps)).  With one slice
// the kernel writes logits and bounds; otherwise the slice sums to
// part[z][T][E] for router_slices_kernel.
__global__ void __launch_bounds__(256, 2) router_tile_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ router_w,
    const float* __restrict__ prior, int E, int H, int cps, const float* __restrict__ xnorm,
    const float* __restrict__ wnorm, float* __restrict__ logits, float* __restrict__ bound,
    float* __restrict__ part) {
  __shared__ __align__(16) float xs[kTK][kTT];  // [h][token]
  __shared__ __align__(16) float ws[kTK][kTE];  // [h][expert]
  const int t0 = blockIdx.x * kTT, e0 = blockIdx.y * kTE;
  // thread: tokens 4 ty .. 4 ty + 3, experts 4 tx .. 4 tx + 3 and 64 + 4 tx .. 64 + 4 tx + 3
  // (consecutive lanes read consecutive 16-byte words of a shared-memory row)
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float2 tot[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) tot[i][j] = make_float2(0.f, 0.f);
  const int kbeg = blockIdx.z * cps * kTK, kend = min(H, kbeg + cps * kTK);
  // the next chunk's words of this thread, loaded while the current one is
  // multiplied (x: 2 of the 512 16-byte words, Wr: 4 of the 1024)
  static_assert(kTT * kTK / 8 == 2 * 256 && kTE * kTK / 8 == 4 * 256, "staging split");
  uint4 px[2], pw[4];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = tid + 256 * r, tt = i % kTT, hc = i / kTT;
      px[r] = t0 + tt < T
                  ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * H + k0) + hc)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = tid + 256 * r, ee = i % kTE, hc = i / kTE;
      pw[r] = e0 + ee < E ? __ldg(reinterpret_cast<const uint4*>(router_w + (size_t)(e0 + ee) * H +
                                                                  k0) + hc)
                          : make_uint4(0, 0, 0, 0);
    }
  };
  fetch(kbeg);
  for (int k0 = kbeg; k0 < kend; k0 += kTK) {
    __syncthreads();  // the previous chunk's products are done
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = tid + 256 * r, tt = i % kTT, hc = i / kTT;
      const uint32_t vw[4] = {px[r].x, px[r].y, px[r].z, px[r].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        xs[hc * 8 + 2 * q][tt] = bf16_lo(vw[q]);
        xs[hc * 8 + 2 * q + 1][tt] = bf16_hi(vw[q]);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = tid + 256 * r, ee = i % kTE, hc = i / kTE;
      const uint32_t vw[4] = {pw[r].x, pw[r].y, pw[r].z, pw[r].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        ws[hc * 8 + 2 * q][ee] = bf16_lo(vw[q]);
        ws[hc * 8 + 2 * q + 1][ee] = bf16_hi(vw[q]);
      }
    }
    __syncthreads();
    if (k0 + kTK < kend) fetch(k0 + kTK);
    float2 acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
#pragma unroll 4
    for (int h = 0; h < kTK; ++h) {
      const float4 xv = *reinterpret_cast<const float4*>(&xs[h][ty * 4]);
      const float4 wa = *reinterpret_cast<const float4*>(&ws[h][tx * 4]);
      const float4 wb = *reinterpret_cast<const float4*>(&ws[h][64 + tx * 4]);
      const float xi[4] = {xv.x, xv.y, xv.z, xv.w};
      const float2 wj[4] = {make_float2(wa.x, wa.y), make_float2(wa.z, wa.w),
                            make_float2(wb.x, wb.y), make_float2(wb.z, wb.w)};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
          acc[i][j] = __ffma2_rn(make_float2(xi[i], xi[i]), wj[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        tot[i][j] = make_float2(tot[i][j].x + acc[i][j].x, tot[i][j].y + acc[i][j].y);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int e = e0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
      if (e >= E) continue;
      const float sum = (j & 1) ? tot[i][j >> 1].y : tot[i][j >> 1].x;
      if (gridDim.z > 1) {
        part[((size_t)blockIdx.z * T + t) * E + e] = sum;
      } else {
        float l, b;
        tile_logit_and_bound(sum, prior ? prior[e] : 0.f, xnorm[t], wnorm[e], H, 1, l, b);
        logits[(size_t)t * E + e] = l;
        bound[(size_t)t * E + e] = b;
      }
    }
  }
}

// Sum of the slice sums in slice order, then the prior.
__global__ void router_slices_kernel(const float* __restrict__ part, int slices, int T, int E,
                                     int H, const float* __restrict__ prior,
                                     const float* __restrict__ xnorm,
                                     const float* __restrict__ wnorm, float* __restrict__ logits,
                                     float* __restrict__ bound) {
  const int64_t n = (int64_t)T * E;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float sum = part[i];
    for (int z = 1; z < slices; ++z) sum += part[(size_t)z * n + i];
    const int t = (int)(i / E), e = (int)(i - (int64_t)t * E);
    float l, b;
    tile_logit_and_bound(sum, prior ? prior[e] : 0.f, xnorm[t], wnorm[e], H, slices, l, b);
    logits[i] = l;
    bound[i] = b;
  }
}

// topk_kernel with the per-lane list length fitting E.
cudaError_t launch_topk_any(const float* logits, const float* bound, const float* gate_z,
                            const uint16_t* x, const uint16_t* router_w, const float* prior,
                            int T, int E, int H, int k, int32_t* topk_idx, float* topk_w,
                            float* gate, cudaStream_t st) {
  const size_t smem = topk_warp_smem(E) * kTopkWarps;
  const int grid = (T + kTopkWarps - 1) / kTopkWarps;
#define MOE_TOPK_LAUNCH(MV)                                                                    \
  topk_kernel<MV><<<grid, kTopkWarps * 32, smem, st>>>(logits, bound, gate_z, x, router_w,    \
                                                        prior, T, E, H, k, topk_idx, topk_w, gate)
  if (E <= 32) MOE_TOPK_LAUNCH(1);
  else if (E <= 64) MOE_TOPK_LAUNCH(2);
  else if (E <= 128) MOE_TOPK_LAUNCH(4);
  else if (E <= 256) MOE_TOPK_LAUNCH(8);
  else if (E <= 512) MOE_TOPK_LAUNCH(16);
  else MOE_TOPK_LAUNCH(32);
#undef MOE_TOPK_LAUNCH
  return cudaGetLastError();
}

// The dynamic shared-memory limit is per kernel, not per context: size it for
// the largest E, so that preparing a small context never lowers it under a
// larger one.
cudaError_t set_topk_smem_limits() {
  const int smem = (int)(topk_warp_smem(kMaxE) * kTopkWarps);
  const cudaError_t e[] = {
      cudaFuncSetAttribute(topk_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
      cudaFuncSetAttribute(topk_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
      cudaFuncSetAttribute(topk_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
      cudaFuncSetAttribute(topk_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
      cudaFuncSetAttribute(topk_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem),
      cudaFuncSetAttribute(topk_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)};
  for (cudaError_t x : e)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

cudaError_t set_router_smem_limit(int H) {
  const int smem = kRouterTC * H * 2;
  switch (H / 256) {
    case 1: return cudaFuncSetAttribute(router_logits_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 2: return cudaFuncSetAttribute(router_logits_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 4: return cudaFuncSetAttribute(router_logits_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 8: return cudaFuncSetAttribute(router_logits_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 16: return cudaFuncSetAttribute(router_logits_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    case 32: return cudaFuncSetAttribute(router_logits_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_router_any(const uint16_t* x, int T, const uint16_t* router_w,
                              const float* prior, const uint16_t* shared_gate_w, int E, int H,
                              float* logits, float* bound, float* gate_z, cudaStream_t st) {
  const int grid = (E + 1 + kRouterWarps - 1) / kRouterWarps;
  const size_t smem = (size_t)kRouterTC * H * 2;
#define MOE_ROUTER_LAUNCH(NJ)                                                                 \
  router_logits_kernel<NJ><<<grid, kRouterWarps * 32, smem, st>>>(x, T, router_w, prior,      \
                                                                   shared_gate_w, E, logits,  \
                                                                   bound, gate_z)
  switch (H / 256) {
    case 1: MOE_ROUTER_LAUNCH(1); break;
    case 2: MOE_ROUTER_LAUNCH(2); break;
    case 4: MOE_ROUTER_LAUNCH(4); break;
    case 8: MOE_ROUTER_LAUNCH(8); break;
    case 16: MOE_ROUTER_LAUNCH(16); break;
    case 32: MOE_ROUTER_LAUNCH(32); break;
    default: return cudaErrorInvalidValue;
  }
#undef MOE_ROUTER_LAUNCH
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches) {
  if (a.T >= kTileRouterMinT) {
    const int rows = a.T + c.d.E;
    router_norms_kernel<<<(rows + 7) / 8, 256, 0, st>>>(a.x, a.T, c.router_w, c.d.E,
                                                       c.shared_gate_w, c.d.H, c.ws.xnorm,
                                                       c.ws.wnorm, c.ws.gate_z);
    if (router_tc_supported(c.d, a.T)) {
      ++*launches;
      return launch_router_tc(c, a, st, launches);
    }
    const int tiles = ((a.T + kTT - 1) / kTT) * ((c.d.E + kTE - 1) / kTE);
    const int chunks = c.d.H / kTK;
    // slices of H so that about two CTAs per SM are busy (one slice when the tiles suffice)
    int slices = max(1, min(chunks, (2 * c.num_sms) / tiles));
    if ((int64_t)slices * a.T * c.d.E > tile_router_part_floats(c.num_sms)) slices = 1;
    const int cps = (chunks + slices - 1) / slices;
    slices = (chunks + cps - 1) / cps;
    dim3 grid((a.T + kTT - 1) / kTT, (c.d.E + kTE - 1) / kTE, slices);
    router_tile_kernel<<<grid, 256, 0, st>>>(a.x, a.T, c.router_w, c.router_bias, c.d.E, c.d.H,
                                             cps, c.ws.xnorm, c.ws.wnorm, c.ws.logits,
                                             c.ws.bound, c.ws.rpart);
    *launches += 2;
    if (slices > 1) {
      router_slices_kernel<<<2 * c.num_sms, 256, 0, st>>>(c.ws.rpart, slices, a.T, c.d.E, c.d.H,
                                                          c.router_bias, c.ws.xnorm, c.ws.wnorm,
                                                          c.ws.logits, c.ws.bound);
      ++*launches;
    }
    return cudaGetLastError();
  }
  ++*launches;
  return launch_router_any(a.x, a.T, c.router_w, c.router_bias, c.shared_gate_w, c.d.E, c.d.H,
                           c.ws.logits, c.ws.bound, c.ws.gate_z, st);
}

cudaError_t prepare_router(const Ctx& c) {
  cudaError_t e = set_router_smem_limit(c.d.H);
  if (e == cudaSuccess) e = set_topk_smem_limits();
  if (e == cudaSuccess) e = prepare_router_tc();
  return e;
}

cudaError_t launch_topk(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches) {
  if (a.T >= kTileRouterMinT && router_tc_supported(c.d, a.T))
    return launch_router_candidates(c, a, st, launches);
  ++*launches;
  return launch_topk_any(c.ws.logits, c.ws.bound, c.ws.gate_z, a.x, c.router_w, c.router_bias,
                         a.T, c.d.E, c.d.H, c.d.k, a.topk_idx, a.topk_w, c.ws.gate, st);
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
    const cudaError_t attrs[] = {set_router_smem_limit(256),  set_router_smem_limit(512),
                                 set_router_smem_limit(1024), set_router_smem_limit(2048),
                                 set_router_smem_limit(4096), set_router_smem_limit(8192),
                                 set_topk_smem_limits()};
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
  if (!hidden_supported(hidden)) {
    snprintf(msg, sizeof msg, "moe_route_static: hidden=%d not in {256, 512, 1024, 2048, 4096, 8192}",
             hidden);
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
  e = launch_router_any(xb, T, router_w, router_bias, shared_gate_w, E, hidden, logits, bound,
                        gate_z, st);
  if (e == cudaSuccess)
    e = launch_topk_any(logits, bound, gate_z, xb, router_w, router_bias, T, E, hidden, k,
                        topk_idx, topk_w, shared_gate, st);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof msg, "moe_route_static: launch failed: %s", cudaGetErrorString(e));
    return set_global_msg(MOE_ERR_CUDA, msg);
  }
  return MOE_OK;
}
