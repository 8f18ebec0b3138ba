// experts_general.cu -- expert-major int4 / int8 GEMV kernels for any T (the
// general path, and the only one for int8 experts), plus the deterministic
// combine.
//
// For every expert in use (and the shared expert, which takes every token)
// a CTA streams a tile of the expert's rows and applies it to all of the
// expert's tokens:
//   gate/up:  h[q, i] = silu(Wg_i . x_t) * (Wu_i . x_t)         (q = pair position)
//   down:     o[q, r] = Wd_r . h[q, :]
//   combine:  y[t, r] = sum_j w[t, j] o[inv[t*k + j], r] + g_t o[P + t, r]
// with W = s*q + b per group (MLX affine int4 or int8; Swiftlet README, its
// list of what was built).  The affine terms are folded per 32-code
// chunk: sum_c (s q_c + b) x_c = s * sum_c q_c x_c + b * sum_c x_c, the last
// sum staged once per token.
#include "device_util.cuh"
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kTC = 8;         // tokens staged per pass
constexpr int kRowsPerCta = 32;
constexpr int kWarps = 8;
constexpr int kStageBudget = 96 * 1024;  // bytes of staged vectors per CTA

struct Unit {
  const uint8_t* blob;  // null: nothing to do
  int inter;            // inner size of this expert
  int q0, n;            // pair positions [q0, q0+n) (routed) or tokens [0, n) (shared)
  int hrow0;            // first h/o row
  bool shared;
};

__device__ Unit resolve_unit(int u, const int32_t* __restrict__ used, int n_used,
                             const int32_t* __restrict__ offsets, const int32_t* table,
                             int n_slots, const uint8_t* pool, uint64_t stride,
                             const uint8_t* shared_blob, int I, int Is, int T, int P,
                             int32_t* err) {
  Unit U{nullptr, 0, 0, 0, 0, false};
  if (u == (int)gridDim.y - 1) {
    U.blob = shared_blob;
    U.inter = Is;
    U.q0 = 0;
    U.n = T;
    U.hrow0 = P;
    U.shared = true;
    return U;
  }
  if (u >= n_used) return U;
  const int e = used[u];
  const int slot = table ? table[e] : e;
  if (slot < 0 || slot >= n_slots) {
    if (threadIdx.x == 0) record_error(err, MOE_ERR_SLOT);
    return U;
  }
  U.blob = pool + (uint64_t)slot * stride;
  U.inter = I;
  U.q0 = offsets[e];
  U.n = offsets[e + 1] - offsets[e];
  U.hrow0 = U.q0;
  return U;
}

// Stage `tc` fp32 vectors of length K into xs [kTC][K] and their 32-chunk sums
// into xsum [kTC][K/32].  src(tt) gives the tt-th vector's source row.
template <typename Loader>
__device__ void stage_rows(float* xs, float* xsum, int tc, int K, Loader src) {
  for (int i = threadIdx.x; i < tc * K; i += blockDim.x) xs[i] = src(i / K, i % K);
  __syncthreads();
  const int nch = K / 32;
  for (int i = threadIdx.x; i < tc * nch; i += blockDim.x) {
    const float* p = xs + (i / nch) * K + (i % nch) * 32;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 32; ++c) s += p[c];
    xsum[i] = s;
  }
  __syncthreads();
}

// BITS: code width; a 32-code chunk is BITS/4 uint4 words.
template <int BITS>
__device__ __forceinline__ float dot_codes(const uint4* chunk, const float* xv) {
  if constexpr (BITS == 4) {
    return dot_chunk32(__ldg(chunk), xv);
  } else {
    return dot_chunk32_q8(__ldg(chunk), __ldg(chunk + 1), xv);
  }
}

template <int BITS>
__global__ void __launch_bounds__(kWarps * 32) gateup_general_kernel(
    const uint16_t* __restrict__ x, int T, int k, int H, int I, int Is, int G,
    const int32_t* __restrict__ perm, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ used, const int32_t* __restrict__ n_used, const int32_t* table,
    int n_slots, const uint8_t* __restrict__ pool, BlobLayout L, const uint8_t* shared_blob,
    BlobLayout LS, int maxI, float* __restrict__ h, int tcmax, int32_t* err) {
  extern __shared__ float smem[];
  const int P = T * k;
  const Unit U = resolve_unit(blockIdx.y, used, *n_used, offsets, table, n_slots, pool, L.stride,
                              shared_blob, I, Is, T, P, err);
  if (U.blob == nullptr || U.n == 0) return;
  const int f0 = blockIdx.x * kRowsPerCta;
  if (f0 >= U.inter) return;
  const BlobLayout& B = U.shared ? LS : L;
  const uint32_t* guq = reinterpret_cast<const uint32_t*>(U.blob + B.gu_q);
  const uint32_t* gusb = reinterpret_cast<const uint32_t*>(U.blob + B.gu_sb);
  constexpr int V = BITS / 4;  // uint4 words per 32-code chunk
  const int nch = H / 32, wrow = H * BITS / 32, grow = H / G;
  float* xs = smem;
  float* xsum = smem + tcmax * H;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q0 = 0; q0 < U.n; q0 += tcmax) {
    const int tc = min(tcmax, U.n - q0);
    __syncthreads();
    stage_rows(xs, xsum, tc, H, [&](int tt, int c) {
      const int q = q0 + tt;
      const int t = U.shared ? q : perm[U.q0 + q] / k;
      return bf16_val(x[(size_t)t * H + c]);
    });
    for (int f = f0 + warp; f < min(f0 + kRowsPerCta, U.inter); f += kWarps) {
      float pg[kTC], pu[kTC];
#pragma unroll
      for (int tt = 0; tt < kTC; ++tt) pg[tt] = pu[tt] = 0.f;
      const uint4* rg = reinterpret_cast<const uint4*>(guq + (size_t)(2 * f) * wrow);
      const uint4* ru = reinterpret_cast<const uint4*>(guq + (size_t)(2 * f + 1) * wrow);
      for (int c = lane; c < nch; c += 32) {
        const int g = (c * 32) / G;
        const uint32_t sbg = __ldg(gusb + (size_t)(2 * f) * grow + g);
        const uint32_t sbu = __ldg(gusb + (size_t)(2 * f + 1) * grow + g);
#pragma unroll
        for (int tt = 0; tt < kTC; ++tt) {
          if (tt < tc) {
            const float* xv = xs + tt * H + c * 32;
            const float xsm = xsum[tt * nch + c];
            pg[tt] += bf16_lo(sbg) * dot_codes<BITS>(rg + c * V, xv) + bf16_hi(sbg) * xsm;
            pu[tt] += bf16_lo(sbu) * dot_codes<BITS>(ru + c * V, xv) + bf16_hi(sbu) * xsm;
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTC; ++tt) {
        if (tt < tc) {
          const float a = warp_sum(pg[tt]);
          const float u = warp_sum(pu[tt]);
          if (lane == 0) h[(size_t)(U.hrow0 + q0 + tt) * maxI + f] = silu_f(a) * u;
        }
      }
    }
  }
}

template <int BITS>
__global__ void __launch_bounds__(kWarps * 32) down_general_kernel(
    int T, int k, int H, int I, int Is, int G, const int32_t* __restrict__ offsets,
    const int32_t* __restrict__ used, const int32_t* __restrict__ n_used, const int32_t* table,
    int n_slots, const uint8_t* __restrict__ pool, BlobLayout L, const uint8_t* shared_blob,
    BlobLayout LS, int maxI, const float* __restrict__ h, float* __restrict__ o, int tcmax,
    int32_t* err) {
  extern __shared__ float smem[];
  const int P = T * k;
  const Unit U = resolve_unit(blockIdx.y, used, *n_used, offsets, table, n_slots, pool, L.stride,
                              shared_blob, I, Is, T, P, err);
  if (U.blob == nullptr || U.n == 0) return;
  const int r0 = blockIdx.x * kRowsPerCta;
  if (r0 >= H) return;
  const BlobLayout& B = U.shared ? LS : L;
  const int K = U.inter;
  const uint32_t* dq = reinterpret_cast<const uint32_t*>(U.blob + B.d_q);
  const uint32_t* dsb = reinterpret_cast<const uint32_t*>(U.blob + B.d_sb);
  constexpr int V = BITS / 4;
  const int nch = K / 32, wrow = K * BITS / 32, grow = K / G;
  float* xs = smem;
  float* xsum = smem + tcmax * K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int q0 = 0; q0 < U.n; q0 += tcmax) {
    const int tc = min(tcmax, U.n - q0);
    __syncthreads();
    stage_rows(xs, xsum, tc, K, [&](int tt, int c) {
      return h[(size_t)(U.hrow0 + q0 + tt) * maxI + c];
    });
    for (int r = r0 + warp; r < min(r0 + kRowsPerCta, H); r += kWarps) {
      float pd[kTC];
#pragma unroll
      for (int tt = 0; tt < kTC; ++tt) pd[tt] = 0.f;
      const uint4* rw = reinterpret_cast<const uint4*>(dq + (size_t)r * wrow);
      for (int c = lane; c < nch; c += 32) {
        const uint32_t sb = __ldg(dsb + (size_t)r * grow + (c * 32) / G);
#pragma unroll
        for (int tt = 0; tt < kTC; ++tt) {
          if (tt < tc) {
            pd[tt] += bf16_lo(sb) * dot_codes<BITS>(rw + c * V, xs + tt * K + c * 32) +
                      bf16_hi(sb) * xsum[tt * nch + c];
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < kTC; ++tt) {
        if (tt < tc) {
          const float v = warp_sum(pd[tt]);
          if (lane == 0) o[(size_t)(U.hrow0 + q0 + tt) * H + r] = v;
        }
      }
    }
  }
}

// y[t, r] = sum_j w[t, j] o[inv[t*k+j], r] + g_t o[P + t, r], fixed j order.
__global__ void __launch_bounds__(256) combine_kernel(
    int T, int k, int H, const float* __restrict__ topk_w, const int32_t* __restrict__ inv,
    const float* __restrict__ gate, const float* __restrict__ o, uint16_t* __restrict__ y) {
  const int t = blockIdx.x;
  const int P = T * k;
  for (int r = threadIdx.x; r < H; r += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j)
      acc = fmaf(topk_w[(size_t)t * k + j], o[(size_t)inv[t * k + j] * H + r], acc);
    acc = fmaf(gate[t], o[(size_t)(P + t) * H + r], acc);
    y[(size_t)t * H + r] = f32_to_bf16_rne(acc);
  }
}

int pick_tc(int K) {
  const int budget = kStageBudget;
  int tc = budget / (K * 4 + (K / 32) * 4);
  return max(1, min(kTC, tc));
}

}  // namespace

cudaError_t prepare_general_experts(const Ctx& c) {
  // The limits are per kernel, not per context: size them for the largest
  // staging any shape can ask for (pick_tc keeps it within its budget), so
  // that preparing one context never lowers the limit under another.
  (void)c;
  const int most = kStageBudget + 1024;
  const void* fns[4] = {(const void*)gateup_general_kernel<4>, (const void*)gateup_general_kernel<8>,
                        (const void*)down_general_kernel<4>, (const void*)down_general_kernel<8>};
  for (const void* f : fns) {
    cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_general_experts(const Ctx& c, const FwdArgs& a, cudaStream_t st,
                                   int* launches) {
  const Dims& d = c.d;
  const int T = a.T, P = T * d.k;
  const int maxI = d.I > d.Is ? d.I : d.Is;
  const int units = (P < d.E ? P : d.E) + 1;  // experts in use (at most) + shared
  {
    const int tc = pick_tc(d.H);
    const size_t smem = (size_t)tc * d.H * 4 + (size_t)tc * (d.H / 32) * 4;
    dim3 grid((maxI + kRowsPerCta - 1) / kRowsPerCta, units);
    auto* gk = d.bits == 8 ? gateup_general_kernel<8> : gateup_general_kernel<4>;
    gk<<<grid, kWarps * 32, smem, st>>>(
        a.x, T, d.k, d.H, d.I, d.Is, d.G, c.ws.perm, c.ws.offsets, c.ws.used, c.ws.n_used,
        a.table, c.n_slots, c.pool, c.ex, c.shared, c.sh, maxI, c.ws.h, tc, c.err);
    ++*launches;
    record_mark(c, MOE_MARK_GATEUP, st);
  }
  {
    const int tc = pick_tc(maxI);
    const size_t smem = (size_t)tc * maxI * 4 + (size_t)tc * (maxI / 32) * 4;
    dim3 grid((d.H + kRowsPerCta - 1) / kRowsPerCta, units);
    auto* dk = d.bits == 8 ? down_general_kernel<8> : down_general_kernel<4>;
    dk<<<grid, kWarps * 32, smem, st>>>(
        T, d.k, d.H, d.I, d.Is, d.G, c.ws.offsets, c.ws.used, c.ws.n_used, a.table, c.n_slots,
        c.pool, c.ex, c.shared, c.sh, maxI, c.ws.h, c.ws.o, tc, c.err);
    ++*launches;
    record_mark(c, MOE_MARK_DOWN, st);
  }
  combine_kernel<<<T, 256, 0, st>>>(T, d.k, d.H, a.topk_w, c.ws.inv, c.ws.gate, c.ws.o, a.y);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace moe
