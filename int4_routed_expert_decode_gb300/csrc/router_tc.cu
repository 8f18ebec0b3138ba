// router_tc.cu -- the router for many tokens in two steps.
//
// 1. Approximate logits a[t][e] = x_t . Wr_e (+ prior_e) as a bf16 GEMM on the
//    tensor cores (tcgen05, fp32 accumulation in TMEM, operands by TMA in the
//    128-byte-swizzled K-major layout): 128 experts x 128 tokens per CTA.
// 2. Per token (one warp): every expert whose approximate logit is within 2d
//    of the k-th largest is a candidate, d = 2^-10 |x_t|_2 max_e |Wr_e|_2.
//    Candidates get certified fp32 logits with tight bounds, and the exact
//    selection of routing_common.cuh orders them (ties to the lower id); the
//    weights are the renormalised softmax of the selected logits.
//
// Why the filter is safe.  If |a_e - l_e| <= delta for every expert, the k-th
// largest approximate logit is within delta of the k-th largest exact one, so
// an expert that can be selected has a_e >= (k-th approximate) - 2 delta:
// the filter keeps it whenever delta <= d.  Error model of the tensor cores
// (kind::f16, fp32 accumulation): bf16 x bf16 products are exact; each k-step
// of 16 products is summed after aligning to the largest with at least 23
// kept bits (truncation), then added to the fp32 accumulator with rounding.
// That gives delta <= (16 2^-23 + (H/16) 2^-24) sum|x w| <= (2^-19 + H 2^-28)
// |x| |w| (Cauchy-Schwarz) -- at H = 8192 about 2^-15 |x||w|, 32 times below
// the accumulation term of d = 2^-10 |x| max_e|Wr_e| + 2^-22 max|prior| (the
// second term covers the rounding of the prior's addition).  The model is not
// taken on trust: every candidate's certified logit measures the error on
// that expert (at least |a - l| - bound), and a token whose measured error
// exceeds d/8 falls back to certifying all E experts.  The largest observed
// |a - l| and the number of fallbacks are kept for moe_router_check_stats.
#include <cuda.h>

#include "device_util.cuh"
#include "moe_internal.cuh"
#include "routing_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

using namespace rt;

constexpr int kRM = 128, kRN = 128, kRK = 64, kRStages = 4;
constexpr int kRThreads = 192;  // warp 0: TMA, warp 1: MMA, warps 2-5: epilogue
constexpr int kRTile = kRM * kRK * 2;  // 16 KiB (A and B alike)
constexpr uint64_t kRWaitNs = 1000000000ull;
constexpr int kCandWarps = 4;
constexpr int kCandCap = 64;  // candidates kept in shared memory per token
// one token's overflow scratch: the selection scratch for E entries, then E
// candidate ids, logits and bounds
__host__ __device__ constexpr size_t cand_ovf_bytes(int E) {
  return (topk_warp_smem(E) + (size_t)E * 12 + 15) & ~size_t(15);
}
// per warp: the selection scratch for kCandCap entries, then the candidate
// ids, logits and bounds
__host__ __device__ constexpr size_t cand_warp_smem() {
  return (topk_warp_smem(kCandCap) + (size_t)kCandCap * 12 + 15) & ~size_t(15);
}

struct RSmem {
  uint8_t a[kRStages][kRTile];
  uint8_t b[kRStages][kRTile];
  uint64_t full[kRStages], empty[kRStages], done;
  uint32_t tmem;
};

__device__ __forceinline__ uint64_t sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Bounded mbarrier wait (1 s): false, with MOE_ERR_TIMEOUT recorded, on expiry.
__device__ bool rwait(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && ptx::globaltimer_ns() - t0 > kRWaitNs) {
      record_error(err, MOE_ERR_TIMEOUT);
      return false;
    }
  }
}

// wmap: Wr [E][H] bf16, xmap: x [T][H] bf16; both box 64 x 128, 128-byte swizzle.
__global__ void __launch_bounds__(kRThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                     int T, int E, int H, const float* __restrict__ prior, float* __restrict__ approx,
                     int32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  RSmem& S = *reinterpret_cast<RSmem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * kRM, t0 = blockIdx.y * kRN, nk = H / kRK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRStages; ++s) {
      ptx::mbar_init(&S.full[s], 1);
      ptx::mbar_init(&S.empty[s], 1);
    }
    ptx::mbar_init(&S.done, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) ptx::tmem_alloc(&S.tmem, 128);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem;
  if (warp == 0 && lane == 0) {
    for (int c = 0; c < nk; ++c) {
      const int s = c % kRStages;
      if (c >= kRStages && !rwait(&S.empty[s], ((c / kRStages) + 1) & 1, err)) break;
      ptx::mbar_arrive_expect_tx(&S.full[s], 2 * kRTile);
      ptx::tma_load_2d(S.a[s], &wmap, c * kRK, e0, &S.full[s]);
      ptx::tma_load_2d(S.b[s], &xmap, c * kRK, t0, &S.full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // D[128 experts][128 tokens]: kind::f16, bf16 operands, fp32 accumulator
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kRN >> 3) << 17) |
                           ((uint32_t)(kRM >> 4) << 24);
    bool ok = true;
    for (int c = 0; c < nk && ok; ++c) {
      const int s = c % kRStages;
      if (!rwait(&S.full[s], (c / kRStages) & 1, err)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint64_t ad = sw128(ptx::smem_u32(S.a[s])), bd = sw128(ptx::smem_u32(S.b[s]));
#pragma unroll
      for (int kk = 0; kk < kRK / 16; ++kk)
        ptx::tc_mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (c > 0 || kk > 0) ? 1u : 0u);
      ptx::tc_commit(&S.empty[s]);
    }
    ptx::tc_commit(&S.done);  // every MMA issued has completed
  } else if (warp >= 2) {
    const int q = warp & 3;  // TMEM lane quarter: experts e0 + 32 q ..
    const bool ok = rwait(&S.done, 0, err);
    ptx::tc_fence_after();
    const int e = e0 + q * 32 + lane;
    const float p = (prior && e < E) ? prior[e] : 0.f;
    for (int n0 = 0; n0 < kRN; n0 += 16) {
      float v[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(q * 32) << 16) + n0, v);
      if (ok && e < E) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int t = t0 + n0 + i;
          if (t < T) approx[(size_t)t * E + e] = v[i] + p;
        }
      }
    }
  }
  if (warp == 1) __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 128);
  }
}

// Candidates of one token, as a top-k source: entry i is expert cid[i] with a
// certified fp32 logit and bound.
struct CandLogits {
  const int* cid;
  const float* cl;
  const float* cb;
  __device__ __forceinline__ void get(int i, float& logit, float& bnd) const {
    logit = cl[i];
    bnd = cb[i];
  }
  __device__ __forceinline__ int id(int i) const { return cid[i]; }
};

// A tight fp32 logit of router row e (e < 0: none) by a group of 8 lanes:
// lane sub = lane % 8 takes the 8-element chunks c = sub + 8 j of the row
// (8 sequential FMAs from zero per chunk, chunk sums added in order), then a
// 3-level butterfly inside the group, then the prior: depth
// D = 8 + H/64 + 3 + 1.  sum |x w| is computed alongside with the same
// structure; 1 + 2^-8 covers its own rounding, so
// bound = 2 D u (mag (1 + 2^-8) + |prior|) bounds the error (Higham, Accuracy
// and Stability of Numerical Algorithms, Thm. 4.3).
__device__ void tight_logit_group8(const uint16_t* __restrict__ x,
                                   const uint16_t* __restrict__ router_w, int H,
                                   const float* prior, int e, float& logit, float& bnd) {
  const int sub = threadIdx.x & 7;
  float acc = 0.f, mag = 0.f;
  if (e >= 0) {
    const uint4* xr = reinterpret_cast<const uint4*>(x);
    const uint4* wr = reinterpret_cast<const uint4*>(router_w + (size_t)e * H);
    // the loads of several chunks in flight at once (the sums keep their order)
#pragma unroll 8
    for (int j = 0; j < H / 64; ++j) {
      const uint4 xv = __ldg(xr + sub + 8 * j);
      const uint4 wv = __ldg(wr + sub + 8 * j);
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
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    acc += __shfl_xor_sync(0xffffffffu, acc, o);
    mag += __shfl_xor_sync(0xffffffffu, mag, o);
  }
  const float p = (prior && e >= 0) ? prior[e] : 0.f;
  logit = acc + p;
  const float depth = (float)(8 + H / 64 + 4);
  bnd = 2.0f * depth * 5.9604644775390625e-8f * (mag * 1.00390625f + fabsf(p)) + kBoundFloor;
}

// One warp per token: threshold, candidates, certified logits, exact order.
template <int MAXV>
__global__ void __launch_bounds__(kCandWarps * 32) router_candidates_kernel(
    const float* __restrict__ approx, const float* __restrict__ xnorm,
    const float* __restrict__ wnorm, const float* __restrict__ gate_z,
    const uint16_t* __restrict__ x, const uint16_t* __restrict__ router_w,
    const float* __restrict__ prior, int T, int E, int H, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, float* __restrict__ gate, uint32_t* __restrict__ rstats,
    uint8_t* __restrict__ ovf) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kCandWarps + warp;
  if (t >= T) return;
  // Candidate arrays and selection scratch: in shared memory for up to
  // kCandCap candidates (the usual case), else in this token's slice of the
  // global overflow region (E entries: many candidates, or every expert).
  uint8_t* ws = smem_raw + (size_t)warp * cand_warp_smem();
  int* cid = reinterpret_cast<int*>(ws + topk_warp_smem(kCandCap));
  float* cl = reinterpret_cast<float*>(cid + kCandCap);
  float* cb = cl + kCandCap;
  bool in_global = false;
  auto to_global = [&]() {
    ws = ovf + (size_t)t * cand_ovf_bytes(E);
    cid = reinterpret_cast<int*>(ws + topk_warp_smem(E));
    cl = reinterpret_cast<float*>(cid + E);
    cb = cl + E;
    in_global = true;
  };
  const float* arow = approx + (size_t)t * E;
  // the k-th largest approximate logit (entries in lane-major order)
  uint32_t key[MAXV];
  int id[MAXV];
  float wmax = 0.f, pmax = 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int e = lane * MAXV + i;
    float v = e < E ? __ldcg(arow + e) : 0.f;
    if (v != v) v = -INFINITY;
    key[i] = e < E ? f32_key(v) : 0u;
    id[i] = e < E ? e : 0x7FFFFFFF;
    if (e < E) {
      wmax = fmaxf(wmax, __ldg(wnorm + e));
      if (prior) pmax = fmaxf(pmax, fabsf(__ldg(prior + e)));
    }
  }
  wmax = warp_max(wmax);
  pmax = warp_max(pmax);
  uint32_t kk[MAXV];
  int ki[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    kk[i] = key[i];
    ki[i] = id[i];
  }
  sort_lane_desc<MAXV>(kk, ki);
  uint32_t kth = 0;
  for (int r = 0; r < k; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, kk[0]);
    const uint32_t win = __reduce_min_sync(0xffffffffu, kk[0] == m ? (uint32_t)ki[0] : 0xFFFFFFFFu);
    kth = m;
    if (kk[0] == m && ki[0] == (int)win) {
#pragma unroll
      for (int i = 0; i < MAXV - 1; ++i) {
        kk[i] = kk[i + 1];
        ki[i] = ki[i + 1];
      }
      kk[MAXV - 1] = 0u;
      ki[MAXV - 1] = 0x7FFFFFFF;
    }
  }
  // d bounds |a - l| for every expert: 2^-10 |x| max|Wr| the accumulation
  // (file comment), 2^-22 max|prior| the rounding of the prior's addition
  const float xn = __ldg(xnorm + t);
  const float d = 0.0009765625f * xn * wmax + 2.384185791015625e-07f * pmax;
  const float cut = key_f32(kth) - 2.0f * d;
  // candidates, in expert order (counted first to choose their storage)
  int n = 0;
#pragma unroll
  for (int i = 0; i < MAXV; ++i)
    n += __popc(__ballot_sync(0xffffffffu, key[i] != 0u && key_f32(key[i]) >= cut));
  if (n > kCandCap) to_global();
  n = 0;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    // lane-major entries: expert lane * MAXV + i; gather per i in lane order,
    // then the list is not sorted by id -- order does not matter to the selection
    const bool c = key[i] != 0u && key_f32(key[i]) >= cut;
    const unsigned bal = __ballot_sync(0xffffffffu, c);
    if (c) cid[n + __popc(bal & ((1u << lane) - 1u))] = id[i];
    n += __popc(bal);
  }
  __syncwarp();
  // certified logits of the candidates, four at a time (8 lanes each)
  auto certify = [&]() {
    for (int i = 0; i < n; i += 4) {
      const int g = lane >> 3, e = i + g < n ? cid[i + g] : -1;
      float l, b;
      tight_logit_group8(x + (size_t)t * H, router_w, H, prior, e, l, b);
      if ((lane & 7) == 0 && e >= 0) {
        cl[i + g] = l;
        cb[i + g] = b;
      }
    }
    __syncwarp();
  };
  certify();
  // Run-time check of the error model on the candidates: the tensor cores'
  // error on expert e is at least |a_e - l_e| - b_e.  If one exceeds d/8 the
  // model does not hold for this token, and every expert is certified.
  // (the statistic kept is the plain difference |a - l|, error of l included)
  float worst = 0.f, diff = 0.f;
  for (int i = lane; i < n; i += 32) {
    const float dd = fabsf(__ldcg(arow + cid[i]) - cl[i]);
    diff = fmaxf(diff, dd);
    worst = fmaxf(worst, dd - cb[i]);
  }
  worst = warp_max(worst);
  diff = warp_max(diff);
  const bool fallback = worst > 0.125f * d;
  if (lane == 0 && rstats) {
    const float denom = xn * wmax;
    if (denom > 0.f) atomicMax(rstats, __float_as_uint(diff / denom));
    if (fallback) atomicAdd(rstats + 1, 1u);
  }
  if (fallback) {
    if (!in_global) to_global();
    n = E;
    for (int e = lane; e < E; e += 32) cid[e] = e;
    __syncwarp();
    certify();
  }
  int* sel_idx;
  float* sel_val;
  // one candidate per lane when they fit (the usual case), else two or MAXV
  if (n <= 32)
    topk_select_warp_src<1>(CandLogits{cid, cl, cb}, n, k, x + (size_t)t * H, router_w, prior, H,
                            ws, &sel_idx, &sel_val);
  else if (n <= 64)
    topk_select_warp_src<2>(CandLogits{cid, cl, cb}, n, k, x + (size_t)t * H, router_w, prior, H,
                            ws, &sel_idx, &sel_val);
  else
    topk_select_warp_src<MAXV>(CandLogits{cid, cl, cb}, n, k, x + (size_t)t * H, router_w, prior,
                               H, ws, &sel_idx, &sel_val);
  const float w = renormalised_weight(sel_val, k);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = sel_idx[lane];
    topk_w[(size_t)t * k + lane] = w;
  }
  if (lane == 0) gate[t] = 1.0f / (1.0f + __expf(-gate_z[t]));
}

constexpr size_t kRSmem = sizeof(RSmem) + 1024;

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link the driver library).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encode_fn() {
  static EncodeFn fn = []() -> EncodeFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeFn>(p);
  }();
  return fn;
}

// [rows][H] bf16, box 64 x 128, 128-byte swizzle.
bool encode_rows128(CUtensorMap* m, const uint16_t* base, int rows, int H) {
  const EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dim[2] = {(cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)H * 2};
  const cuuint32_t box[2] = {kRK, 128};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dim, stride, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t cand_smem() { return (size_t)kCandWarps * cand_warp_smem(); }

}  // namespace

size_t router_tc_overflow_bytes(const Dims& d, int max_T) {
  return router_tc_supported(d, max_T) ? (size_t)max_T * cand_ovf_bytes(d.E) : 0;
}

bool router_tc_supported(const Dims& d, int T) {
  return T >= 128 && d.E >= 128 && d.E % 128 == 0 && d.E <= kMaxE && d.H % kRK == 0;
}

cudaError_t prepare_router_tc() {
  cudaError_t e = cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kRSmem);
  const int cs = (int)cand_smem();
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_candidates_kernel<4>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, cs);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_candidates_kernel<8>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, cs);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_candidates_kernel<16>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, cs);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(router_candidates_kernel<32>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, cs);
  return e;
}

// Approximate logits into c.ws.logits (after router_norms_kernel has written
// the norms and the shared gate).
cudaError_t launch_router_tc(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches) {
  const Dims& d = c.d;
  CUtensorMap wmap, xmap;
  if (!encode_rows128(&wmap, c.router_w, d.E, d.H) || !encode_rows128(&xmap, a.x, a.T, d.H))
    return cudaErrorInvalidValue;
  dim3 grid(d.E / kRM, (a.T + kRN - 1) / kRN);
  router_tc_kernel<<<grid, kRThreads, kRSmem, st>>>(wmap, xmap, a.T, d.E, d.H, c.router_bias,
                                                    c.ws.logits, c.err);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_router_candidates(const Ctx& c, const FwdArgs& a, cudaStream_t st,
                                     int* launches) {
  const Dims& d = c.d;
  const int grid = (a.T + kCandWarps - 1) / kCandWarps;
  const size_t smem = cand_smem();
#define MOE_CAND(MV)                                                                            \
  router_candidates_kernel<MV><<<grid, kCandWarps * 32, smem, st>>>(                           \
      c.ws.logits, c.ws.xnorm, c.ws.wnorm, c.ws.gate_z, a.x, c.router_w, c.router_bias, a.T,    \
      d.E, d.H, d.k, a.topk_idx, a.topk_w, c.ws.gate, c.ws.rstats, c.ws.rovf)
  if (d.E <= 128) MOE_CAND(4);
  else if (d.E <= 256) MOE_CAND(8);
  else if (d.E <= 512) MOE_CAND(16);
  else MOE_CAND(32);
#undef MOE_CAND
  ++*launches;
  return cudaGetLastError();
}

}  // namespace moe
