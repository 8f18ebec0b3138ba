// Gated DeltaNet recurrence (the linear-attention layers that make up three
// quarters of the Qwen3-Next / Qwen3.5-3.6 hybrid stack: wpnews page, Swiftlet
// README, "How it works"; creativeainews page, "How Expert Streaming Works").
//
// Per value head h, a d_v x d_k fp32 state S is carried from token to token:
//   k^ = k / sqrt(|k|^2 + eps),  q^ = q / sqrt(|q|^2 + eps) / sqrt(d_k)
//   u  = beta (v - alpha S k^)            (the delta: new value minus recall)
//   S <- alpha S + u k^T,   o = S q^ = alpha (S_old q^) + u (k^ . q^)
// The second form of o needs both dot products of the OLD state only, so one
// butterfly reduction per token serves the update and the output.
//
// Work split: row i of S (its d_k columns) is independent of every other row
// given k^ and q^, so one warp owns R consecutive rows of one (sequence, head)
// for all T tokens.  Lane l holds columns [l*C, l*C + C) of each row (C =
// d_k / 32) in registers: a row is one coalesced 4*d_k-byte read at the start
// and one write at the end, whatever T is.  Every warp normalises k and q
// itself (a warp-wide reduction of three sums), so warps never synchronise
// with one another.  The next token's q, k, v, alpha and beta are loaded
// before the current token's arithmetic to hide their latency for T > 1.
//
// For T = 1 (decode) the kernel is bound by HBM: 2 * 4 * d_k bytes of state
// per row, plus the token's inputs.
#include <cuda_runtime.h>
#include <cstdint>
#include <cstdio>
#include <cmath>

#include "moe.h"
#include "sm100_ptx.cuh"

namespace moe {
int set_global_msg(int code, const char* text);

namespace {

// Small CTAs: the register file, not a CTA count, bounds the warps per SM.
constexpr int kGdnThreads = 128;
constexpr int kGdnWarps = kGdnThreads / 32;

struct GdnArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const float* alpha;
  const float* beta;
  float* state;
  float* out;
  int B, T, Hk, Hv, dv;
  float eps;
  float inv_sqrt_dk;
};

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// C consecutive bf16 values (C in {2, 4, 8}) from a 2*C-byte aligned address.
template <int C>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float (&f)[C]) {
  if constexpr (C == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    f[0] = bf16_lo_f(w); f[1] = bf16_hi_f(w);
  } else if constexpr (C == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = bf16_lo_f(w.x); f[1] = bf16_hi_f(w.x); f[2] = bf16_lo_f(w.y); f[3] = bf16_hi_f(w.y);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    f[0] = bf16_lo_f(w.x); f[1] = bf16_hi_f(w.x); f[2] = bf16_lo_f(w.y); f[3] = bf16_hi_f(w.y);
    f[4] = bf16_lo_f(w.z); f[5] = bf16_hi_f(w.z); f[6] = bf16_lo_f(w.w); f[7] = bf16_hi_f(w.w);
  }
}

// C consecutive fp32 values from a 4*C-byte (C = 8: 16-byte) aligned address.
template <int C>
__device__ __forceinline__ void load_f32(const float* p, float (&f)[C]) {
  if constexpr (C == 2) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    f[0] = a.x; f[1] = a.y;
  } else {
#pragma unroll
    for (int i = 0; i < C; i += 4) {
      const float4 a = *reinterpret_cast<const float4*>(p + i);
      f[i] = a.x; f[i + 1] = a.y; f[i + 2] = a.z; f[i + 3] = a.w;
    }
  }
}

template <int C>
__device__ __forceinline__ void store_f32(float* p, const float (&f)[C]) {
  if constexpr (C == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(f[0], f[1]);
  } else {
#pragma unroll
    for (int i = 0; i < C; i += 4)
      *reinterpret_cast<float4*>(p + i) = make_float4(f[i], f[i + 1], f[i + 2], f[i + 3]);
  }
}

// The inputs of one token as one warp needs them.
template <int C, int R>
struct TokenIn {
  float k[C], q[C], v[R];
  float alpha, beta;
};

template <int C, int R>
__device__ __forceinline__ void load_token(const GdnArgs& a, long bt, int j, int h, int row0,
                                           int lane, TokenIn<C, R>& in) {
  const long kq_off = (bt * a.Hk + j) * (32 * C) + lane * C;
  load_bf16<C>(a.k + kq_off, in.k);
  load_bf16<C>(a.q + kq_off, in.q);
  const uint16_t* vp = a.v + (bt * a.Hv + h) * a.dv + row0;
#pragma unroll
  for (int r = 0; r < R; ++r) in.v[r] = __uint_as_float(static_cast<uint32_t>(vp[r]) << 16);
  in.alpha = a.alpha[bt * a.Hv + h];
  in.beta = a.beta[bt * a.Hv + h];
}

template <int N>
__device__ __forceinline__ void warp_sum(float (&x)[N]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] += __shfl_xor_sync(0xffffffffu, x[i], o);
}

// SEQ = false: T is 1 (a decode step), nothing is prefetched.
template <int DK, int R, bool SEQ>
__global__ void __launch_bounds__(kGdnThreads) gdn_recurrence_kernel(GdnArgs a) {
  constexpr int C = DK / 32;
  const int lane = threadIdx.x & 31;
  const long warp = static_cast<long>(blockIdx.x) * kGdnWarps + (threadIdx.x >> 5);
  const int warps_per_head = a.dv / R;
  const long n_warps = static_cast<long>(a.B) * a.Hv * warps_per_head;
  // Programmatic dependent launch: this grid may start while the previous
  // kernel in the stream finishes; every global access waits for it here.
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  if (warp >= n_warps) return;
  const long bh = warp / warps_per_head;  // sequence * Hv + value head
  const int row0 = static_cast<int>(warp - bh * warps_per_head) * R;
  const int h = static_cast<int>(bh % a.Hv);
  const long b = bh / a.Hv;
  const int j = h / (a.Hv / a.Hk);  // key head shared by a group of value heads

  float* srow = a.state + (bh * a.dv + row0) * DK + lane * C;
  float s[R][C];
#pragma unroll
  for (int r = 0; r < R; ++r) load_f32<C>(srow + static_cast<long>(r) * DK, s[r]);

  TokenIn<C, R> cur;
  load_token<C, R>(a, b * a.T, j, h, row0, lane, cur);
  const int T = SEQ ? a.T : 1;
  for (int t = 0; t < T; ++t) {
    const long bt = b * a.T + t;
    TokenIn<C, R> nxt;
    if (SEQ && t + 1 < T) load_token<C, R>(a, bt + 1, j, h, row0, lane, nxt);

    float n3[3] = {0.f, 0.f, 0.f};  // |k|^2, |q|^2, k.q
#pragma unroll
    for (int c = 0; c < C; ++c) {
      n3[0] = fmaf(cur.k[c], cur.k[c], n3[0]);
      n3[1] = fmaf(cur.q[c], cur.q[c], n3[1]);
      n3[2] = fmaf(cur.k[c], cur.q[c], n3[2]);
    }
    // Old-state recalls S k (unnormalised) and S q, per row.
    float d[2 * R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float sk = 0.f, sq = 0.f;
#pragma unroll
      for (int c = 0; c < C; ++c) {
        sk = fmaf(s[r][c], cur.k[c], sk);
        sq = fmaf(s[r][c], cur.q[c], sq);
      }
      d[2 * r] = sk;
      d[2 * r + 1] = sq;
    }
    warp_sum<3>(n3);
    warp_sum<2 * R>(d);
    const float rk = 1.0f / sqrtf(n3[0] + a.eps);
    const float rq = a.inv_sqrt_dk / sqrtf(n3[1] + a.eps);
    // Explicitly rounded steps: every row split gives bit-identical results.
    const float kq = __fmul_rn(__fmul_rn(n3[2], rk), rq);  // k^ . q^
    float kh[C];
#pragma unroll
    for (int c = 0; c < C; ++c) kh[c] = __fmul_rn(cur.k[c], rk);

    float o_mine = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float u = __fmul_rn(cur.beta, __fmaf_rn(-cur.alpha, __fmul_rn(d[2 * r], rk), cur.v[r]));
#pragma unroll
      for (int c = 0; c < C; ++c) s[r][c] = __fmaf_rn(u, kh[c], __fmul_rn(cur.alpha, s[r][c]));
      const float o = __fmaf_rn(u, kq, __fmul_rn(cur.alpha, __fmul_rn(d[2 * r + 1], rq)));
      if (lane == r) o_mine = o;
    }
    if (lane < R) a.out[(bt * a.Hv + h) * a.dv + row0 + lane] = o_mine;
    if (SEQ && t + 1 < T) cur = nxt;
  }
#pragma unroll
  for (int r = 0; r < R; ++r) store_f32<C>(srow + static_cast<long>(r) * DK, s[r]);
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// ---- T > 1 with the token inputs staged in shared memory ------------------
// One CTA = 4 warps x 4 rows = 16 consecutive rows of one (sequence, head).
// The q and k rows of kTC tokens, the CTA's 16 values of v per token and the
// gates arrive by per-thread asynchronous copies into one of two buffers
// while the previous chunk is computed; each chunk's norms (|k|^2, |q|^2,
// k.q) are computed once per CTA, a quarter of the tokens per warp.  The
// per-token loop then reads shared memory only.  Needs dv % 16 == 0 and
// 16-byte aligned q, k, v rows.
constexpr int kSeqRows = 4;                      // rows per warp
constexpr int kSeqCtaRows = kGdnWarps * kSeqRows;  // 16 rows per CTA

template <int DK>
struct SeqChunk {
  static constexpr int kTC = 4096 / DK;  // tokens per chunk: 32 for d_k = 128
  uint16_t k[kTC][DK];
  uint16_t q[kTC][DK];
  uint16_t v[kTC][kSeqCtaRows];
  float alpha[kTC], beta[kTC];
  float rk[kTC], rq[kTC], kq[kTC];
};

template <int DK>
__device__ __forceinline__ void issue_chunk(const GdnArgs& a, SeqChunk<DK>& c, long b, int h,
                                            int j, int row0, int t0, int n) {
  constexpr int kSeg = DK * 2 / 16;  // 16-byte pieces of a q or k row
  for (int i = threadIdx.x; i < n * kSeg; i += kGdnThreads) {
    const int t = i / kSeg, p = i - t * kSeg;
    const long off = ((b * a.T + t0 + t) * a.Hk + j) * DK + p * 8;
    ptx::cp_async16(&c.k[t][p * 8], a.k + off);
    ptx::cp_async16(&c.q[t][p * 8], a.q + off);
  }
  for (int i = threadIdx.x; i < 2 * n; i += kGdnThreads) {
    const int t = i >> 1, p = i & 1;
    ptx::cp_async16(&c.v[t][p * 8], a.v + ((b * a.T + t0 + t) * a.Hv + h) * a.dv + row0 + p * 8);
  }
  for (int i = threadIdx.x; i < 2 * n; i += kGdnThreads) {
    const int t = i >> 1;
    const long g = (b * a.T + t0 + t) * a.Hv + h;
    if (i & 1) ptx::cp_async4(&c.beta[t], a.beta + g);
    else ptx::cp_async4(&c.alpha[t], a.alpha + g);
  }
}

template <int DK>
__global__ void __launch_bounds__(kGdnThreads) gdn_sequence_kernel(GdnArgs a) {
  constexpr int C = DK / 32;
  constexpr int R = kSeqRows;
  constexpr int TC = SeqChunk<DK>::kTC;
  extern __shared__ __align__(16) unsigned char gdn_smem[];
  SeqChunk<DK>* buf = reinterpret_cast<SeqChunk<DK>*>(gdn_smem);

  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ctas_per_head = a.dv / kSeqCtaRows;
  const long bh = blockIdx.x / ctas_per_head;
  const int cta_row0 = static_cast<int>(blockIdx.x - bh * ctas_per_head) * kSeqCtaRows;
  const int h = static_cast<int>(bh % a.Hv);
  const long b = bh / a.Hv;
  const int j = h / (a.Hv / a.Hk);
  const int row0 = cta_row0 + warp * R;

  float* srow = a.state + (bh * a.dv + row0) * DK + lane * C;
  float s[R][C];
#pragma unroll
  for (int r = 0; r < R; ++r) load_f32<C>(srow + static_cast<long>(r) * DK, s[r]);

  const int n_chunks = (a.T + TC - 1) / TC;
  issue_chunk<DK>(a, buf[0], b, h, j, cta_row0, 0, min(TC, a.T));
  ptx::cp_async_commit();
  for (int ch = 0; ch < n_chunks; ++ch) {
    const int t0 = ch * TC, n = min(TC, a.T - t0);
    SeqChunk<DK>& c = buf[ch & 1];
    if (ch + 1 < n_chunks)
      issue_chunk<DK>(a, buf[(ch + 1) & 1], b, h, j, cta_row0, t0 + TC, min(TC, a.T - t0 - TC));
    ptx::cp_async_commit();
    ptx::cp_async_wait<1>();
    __syncthreads();
    for (int t = warp; t < n; t += kGdnWarps) {  // the chunk's norms, once per CTA
      float kf[C], qf[C];
      load_bf16<C>(&c.k[t][lane * C], kf);
      load_bf16<C>(&c.q[t][lane * C], qf);
      float n3[3] = {0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < C; ++e) {
        n3[0] = fmaf(kf[e], kf[e], n3[0]);
        n3[1] = fmaf(qf[e], qf[e], n3[1]);
        n3[2] = fmaf(kf[e], qf[e], n3[2]);
      }
      warp_sum<3>(n3);
      if (lane == 0) {
        const float rk = 1.0f / sqrtf(n3[0] + a.eps);
        const float rq = a.inv_sqrt_dk / sqrtf(n3[1] + a.eps);
        c.rk[t] = rk;
        c.rq[t] = rq;
        c.kq[t] = __fmul_rn(__fmul_rn(n3[2], rk), rq);
      }
    }
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      float kf[C], qf[C];
      load_bf16<C>(&c.k[t][lane * C], kf);
      load_bf16<C>(&c.q[t][lane * C], qf);
      float d[2 * R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int e = 0; e < C; ++e) {
          sk = fmaf(s[r][e], kf[e], sk);
          sq = fmaf(s[r][e], qf[e], sq);
        }
        d[2 * r] = sk;
        d[2 * r + 1] = sq;
      }
      warp_sum<2 * R>(d);
      const float rk = c.rk[t], rq = c.rq[t], kq = c.kq[t];
      const float alpha = c.alpha[t], beta = c.beta[t];
      float kh[C];
#pragma unroll
      for (int e = 0; e < C; ++e) kh[e] = __fmul_rn(kf[e], rk);
      float o_mine = 0.f;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v = __uint_as_float(static_cast<uint32_t>(c.v[t][warp * R + r]) << 16);
        const float u = __fmul_rn(beta, __fmaf_rn(-alpha, __fmul_rn(d[2 * r], rk), v));
#pragma unroll
        for (int e = 0; e < C; ++e) s[r][e] = __fmaf_rn(u, kh[e], __fmul_rn(alpha, s[r][e]));
        const float o = __fmaf_rn(u, kq, __fmul_rn(alpha, __fmul_rn(d[2 * r + 1], rq)));
        if (lane == r) o_mine = o;
      }
      if (lane < R) a.out[((b * a.T + t0 + t) * a.Hv + h) * a.dv + row0 + lane] = o_mine;
    }
    __syncthreads();  // every warp is done with this buffer before it is refilled
  }
#pragma unroll
  for (int r = 0; r < R; ++r) store_f32<C>(srow + static_cast<long>(r) * DK, s[r]);
}

template <int DK>
cudaError_t launch_seq(const GdnArgs& a, cudaStream_t st) {
  const size_t smem = 2 * sizeof(SeqChunk<DK>);
  static bool configured = false;  // the attribute is per function: set once
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gdn_sequence_kernel<DK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long>(a.B) * a.Hv * (a.dv / kSeqCtaRows)));
  cfg.blockDim = dim3(kGdnThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gdn_sequence_kernel<DK>, a);
}

template <int DK, int R, bool SEQ>
cudaError_t launch_r(const GdnArgs& a, cudaStream_t st) {
  const long warps = static_cast<long>(a.B) * a.Hv * a.dv / R;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((warps + kGdnWarps - 1) / kGdnWarps));
  cfg.blockDim = dim3(kGdnThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gdn_recurrence_kernel<DK, R, SEQ>, a);
}

template <int DK>
cudaError_t launch_dk(const GdnArgs& a, int R, cudaStream_t st) {
  if (a.T > 1 && a.dv % kSeqCtaRows == 0 && aligned(a.q, 16) && aligned(a.k, 16) &&
      aligned(a.v, 16))
    return launch_seq<DK>(a, st);
  if (a.T == 1) {
    switch (R) {
      case 8: return launch_r<DK, 8, false>(a, st);
      case 4: return launch_r<DK, 4, false>(a, st);
      case 2: return launch_r<DK, 2, false>(a, st);
      default: return launch_r<DK, 1, false>(a, st);
    }
  }
  switch (R) {
    case 4: return launch_r<DK, 4, true>(a, st);
    case 2: return launch_r<DK, 2, true>(a, st);
    default: return launch_r<DK, 1, true>(a, st);
  }
}

// Rows per warp: enough warps to fill every SM comes first (about 20 warps
// of 152 SMs); above that, more rows per warp put more of the state in
// flight per lane (R rows x 4*d_k bytes per warp).
int pick_rows_per_warp(long rows, int dv, int T) {
  constexpr long kFullWarps = 152L * 20;
  const int rmax = T == 1 ? 8 : 4;  // T > 1 also holds the next token's inputs
  for (int R = rmax; R > 1; R >>= 1)
    if (dv % R == 0 && rows / R >= kFullWarps) return R;
  return 1;
}

}  // namespace
}  // namespace moe

extern "C" int moe_gdn_recurrence(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const float* alpha, const float* beta, float* state, float* out,
                                  int B, int T, int Hk, int Hv, int dk, int dv, void* stream) {
  using namespace moe;
  char msg[160];
  if (B < 0 || T < 0 || Hk < 1 || Hv < 1 || dv < 1 || dv > 4096 || Hv % Hk != 0) {
    snprintf(msg, sizeof(msg), "gdn: bad sizes B=%d T=%d Hk=%d Hv=%d dv=%d", B, T, Hk, Hv, dv);
    return set_global_msg(MOE_ERR_INVALID_ARG, msg);
  }
  if (dk != 64 && dk != 128 && dk != 256) {
    snprintf(msg, sizeof(msg), "gdn: key dim %d not in {64, 128, 256}", dk);
    return set_global_msg(MOE_ERR_UNSUPPORTED, msg);
  }
  if (B == 0 || T == 0) return set_global_msg(MOE_OK, "");
  if (!q || !k || !v || !alpha || !beta || !state || !out)
    return set_global_msg(MOE_ERR_INVALID_ARG, "gdn: NULL pointer");
  const uintptr_t qk_align = static_cast<uintptr_t>(dk / 32) * 2;
  if (!aligned(state, 16) || !aligned(q, qk_align) || !aligned(k, qk_align) || !aligned(v, 2) ||
      !aligned(alpha, 4) || !aligned(beta, 4) || !aligned(out, 4))
    return set_global_msg(MOE_ERR_INVALID_ARG, "gdn: misaligned pointer");
  const long rows = static_cast<long>(B) * Hv * dv;
  if (rows > (1L << 33))
    return set_global_msg(MOE_ERR_INVALID_ARG, "gdn: state too large");
  GdnArgs a{q, k, v, alpha, beta, state, out, B, T, Hk, Hv, dv, 1e-6f,
            static_cast<float>(1.0 / std::sqrt(static_cast<double>(dk)))};
  const int R = pick_rows_per_warp(rows, dv, T);
  auto st = static_cast<cudaStream_t>(stream);
  cudaError_t e = dk == 64 ? launch_dk<64>(a, R, st)
                : dk == 128 ? launch_dk<128>(a, R, st) : launch_dk<256>(a, R, st);
  if (e != cudaSuccess) {
    snprintf(msg, sizeof(msg), "gdn: launch failed: %s", cudaGetErrorString(e));
    return set_global_msg(MOE_ERR_CUDA, msg);
  }
  return MOE_OK;
}
