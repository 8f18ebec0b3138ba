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

// ---- T > 1: 64 state columns per lane, token inputs staged per chunk -------
// A row is split over LPR = d_k / 64 lanes (1, 2 or 4), each holding 64 of its
// columns in registers, so a token's two recalls need log2(LPR) shuffle
// rounds.  One CTA = 4 warps = RPC consecutive rows of one (sequence, head).
// Chunks of 16 tokens: q and k (bf16), alpha and beta arrive by asynchronous
// copies into one of two raw buffers while the previous chunk is computed;
// then the CTA normalises each token once (a quarter of the tokens per warp)
// into fp32 k^ and q^ in shared memory, and every lane runs the chunk's
// tokens against its columns.  v of the next chunk is prefetched into
// registers.  Needs 16-byte aligned q and k.
template <int DK>
struct SeqGeo {
  static constexpr int LPR = DK / 64;            // lanes per row
  static constexpr int RPW = 32 / LPR;           // rows per warp
  static constexpr int RPC = RPW * kGdnWarps;    // rows per CTA
  static constexpr int TC = 16;                  // tokens per chunk
  static constexpr int VPT = TC * RPC / kGdnThreads;  // v values per thread per chunk
  static constexpr int C = DK / 32;              // columns per lane in the norms pass
};

template <int DK>
struct SeqRaw {  // one buffer of asynchronous copies
  uint16_t k[SeqGeo<DK>::TC][DK];
  uint16_t q[SeqGeo<DK>::TC][DK];
  float alpha[SeqGeo<DK>::TC], beta[SeqGeo<DK>::TC];
};

template <int DK>
struct SeqSmem {
  SeqRaw<DK> raw[2];
  float kh[SeqGeo<DK>::TC][DK];  // k / sqrt(|k|^2 + eps)
  float qh[SeqGeo<DK>::TC][DK];  // q / sqrt(|q|^2 + eps) / sqrt(d_k)
  float kq[SeqGeo<DK>::TC], al[SeqGeo<DK>::TC], be[SeqGeo<DK>::TC];
  uint16_t v[SeqGeo<DK>::TC][SeqGeo<DK>::RPC];
};

template <int DK>
__device__ __forceinline__ void seq_issue(const GdnArgs& a, SeqRaw<DK>& r, long b, int h, int j,
                                          int t0, int n) {
  constexpr int kSeg = DK * 2 / 16;  // 16-byte pieces of a q or k row
  for (int i = threadIdx.x; i < n * kSeg; i += kGdnThreads) {
    const int t = i / kSeg, p = i - t * kSeg;
    const long off = ((b * a.T + t0 + t) * a.Hk + j) * DK + p * 8;
    ptx::cp_async16(&r.k[t][p * 8], a.k + off);
    ptx::cp_async16(&r.q[t][p * 8], a.q + off);
  }
  for (int i = threadIdx.x; i < 2 * n; i += kGdnThreads) {
    const int t = i >> 1;
    const long g = (b * a.T + t0 + t) * a.Hv + h;
    if (i & 1) ptx::cp_async4(&r.beta[t], a.beta + g);
    else ptx::cp_async4(&r.alpha[t], a.alpha + g);
  }
}

template <int DK>
__device__ __forceinline__ void seq_fetch_v(const GdnArgs& a, long b, int h, int row0, int t0,
                                            int n, uint16_t (&vr)[SeqGeo<DK>::VPT]) {
  using P = SeqGeo<DK>;
#pragma unroll
  for (int i = 0; i < P::VPT; ++i) {
    const int idx = threadIdx.x + i * kGdnThreads, t = idx / P::RPC, r = idx - t * P::RPC;
    vr[i] = (t < n && row0 + r < a.dv) ? a.v[((b * a.T + t0 + t) * a.Hv + h) * a.dv + row0 + r]
                                       : (uint16_t)0;
  }
}

template <int DK>
__global__ void __launch_bounds__(kGdnThreads) gdn_sequence_kernel(GdnArgs a) {
  using P = SeqGeo<DK>;
  constexpr int TC = P::TC, C = P::C;
  extern __shared__ __align__(16) unsigned char gdn_smem[];
  SeqSmem<DK>& S = *reinterpret_cast<SeqSmem<DK>*>(gdn_smem);

  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ctas_per_head = (a.dv + P::RPC - 1) / P::RPC;
  const long bh = blockIdx.x / ctas_per_head;
  const int row0 = static_cast<int>(blockIdx.x - bh * ctas_per_head) * P::RPC;
  const int h = static_cast<int>(bh % a.Hv);
  const long b = bh / a.Hv;
  const int j = h / (a.Hv / a.Hk);
  const int rloc = warp * P::RPW + lane / P::LPR;  // this lane's row within the CTA
  const int row = row0 + rloc;
  const bool live = row < a.dv;
  const int col0 = (lane % P::LPR) * 64;
  float* srow = a.state + (bh * a.dv + (live ? row : 0)) * DK + col0;
  float s[64];
#pragma unroll
  for (int c = 0; c < 64; c += 4) {
    const float4 v4 = live ? *reinterpret_cast<const float4*>(srow + c) : make_float4(0, 0, 0, 0);
    s[c] = v4.x; s[c + 1] = v4.y; s[c + 2] = v4.z; s[c + 3] = v4.w;
  }

  const int n_chunks = (a.T + TC - 1) / TC;
  seq_issue<DK>(a, S.raw[0], b, h, j, 0, min(TC, a.T));
  ptx::cp_async_commit();
  uint16_t vr[P::VPT];
  seq_fetch_v<DK>(a, b, h, row0, 0, min(TC, a.T), vr);
  for (int ch = 0; ch < n_chunks; ++ch) {
    const int t0 = ch * TC, n = min(TC, a.T - t0);
    if (ch + 1 < n_chunks)
      seq_issue<DK>(a, S.raw[(ch + 1) & 1], b, h, j, t0 + TC, min(TC, a.T - t0 - TC));
    ptx::cp_async_commit();
    ptx::cp_async_wait<1>();
    __syncthreads();  // chunk ch landed; every lane is done with chunk ch - 1
#pragma unroll
    for (int i = 0; i < P::VPT; ++i) {
      const int idx = tid + i * kGdnThreads;
      S.v[idx / P::RPC][idx % P::RPC] = vr[i];
    }
    if (ch + 1 < n_chunks) seq_fetch_v<DK>(a, b, h, row0, t0 + TC, min(TC, a.T - t0 - TC), vr);
    const SeqRaw<DK>& R = S.raw[ch & 1];
    for (int t = warp; t < n; t += kGdnWarps) {  // the chunk's norms, once per CTA
      float kf[C], qf[C];
      load_bf16<C>(&R.k[t][lane * C], kf);
      load_bf16<C>(&R.q[t][lane * C], qf);
      float n3[3] = {0.f, 0.f, 0.f};
#pragma unroll
      for (int e = 0; e < C; ++e) {
        n3[0] = fmaf(kf[e], kf[e], n3[0]);
        n3[1] = fmaf(qf[e], qf[e], n3[1]);
        n3[2] = fmaf(kf[e], qf[e], n3[2]);
      }
      warp_sum<3>(n3);
      const float rk = 1.0f / sqrtf(n3[0] + a.eps);
      const float rq = a.inv_sqrt_dk / sqrtf(n3[1] + a.eps);
#pragma unroll
      for (int e = 0; e < C; ++e) {
        S.kh[t][lane * C + e] = __fmul_rn(kf[e], rk);
        S.qh[t][lane * C + e] = __fmul_rn(qf[e], rq);
      }
      if (lane == 0) {
        S.kq[t] = __fmul_rn(__fmul_rn(n3[2], rk), rq);
        S.al[t] = R.alpha[t];
        S.be[t] = R.beta[t];
      }
    }
    __syncthreads();
    for (int t = 0; t < n; ++t) {
      const float* kh = &S.kh[t][col0];
      const float* qh = &S.qh[t][col0];
      float sk[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(kh + c);
        const float4 q4 = *reinterpret_cast<const float4*>(qh + c);
        const int g = (c >> 2) & 3;
        sk[g] = fmaf(s[c], k4.x, sk[g]);
        sk[g] = fmaf(s[c + 1], k4.y, sk[g]);
        sk[g] = fmaf(s[c + 2], k4.z, sk[g]);
        sk[g] = fmaf(s[c + 3], k4.w, sk[g]);
        sq[g] = fmaf(s[c], q4.x, sq[g]);
        sq[g] = fmaf(s[c + 1], q4.y, sq[g]);
        sq[g] = fmaf(s[c + 2], q4.z, sq[g]);
        sq[g] = fmaf(s[c + 3], q4.w, sq[g]);
      }
      float dk = (sk[0] + sk[1]) + (sk[2] + sk[3]);
      float dq = (sq[0] + sq[1]) + (sq[2] + sq[3]);
#pragma unroll
      for (int o = 1; o < P::LPR; o <<= 1) {
        dk += __shfl_xor_sync(0xffffffffu, dk, o);
        dq += __shfl_xor_sync(0xffffffffu, dq, o);
      }
      const float alpha = S.al[t], beta = S.be[t];
      const float v = __uint_as_float(static_cast<uint32_t>(S.v[t][rloc]) << 16);
      const float u = __fmul_rn(beta, __fmaf_rn(-alpha, dk, v));
      const float o = __fmaf_rn(u, S.kq[t], __fmul_rn(alpha, dq));
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        const float4 k4 = *reinterpret_cast<const float4*>(kh + c);
        s[c] = __fmaf_rn(u, k4.x, __fmul_rn(alpha, s[c]));
        s[c + 1] = __fmaf_rn(u, k4.y, __fmul_rn(alpha, s[c + 1]));
        s[c + 2] = __fmaf_rn(u, k4.z, __fmul_rn(alpha, s[c + 2]));
        s[c + 3] = __fmaf_rn(u, k4.w, __fmul_rn(alpha, s[c + 3]));
      }
      if (live && (lane % P::LPR) == 0)
        a.out[((b * a.T + t0 + t) * a.Hv + h) * a.dv + row] = o;
    }
  }
  if (live) {
#pragma unroll
    for (int c = 0; c < 64; c += 4)
      *reinterpret_cast<float4*>(srow + c) = make_float4(s[c], s[c + 1], s[c + 2], s[c + 3]);
  }
}

template <int DK>
cudaError_t launch_seq(const GdnArgs& a, cudaStream_t st) {
  using P = SeqGeo<DK>;
  const size_t smem = sizeof(SeqSmem<DK>);
  static bool configured = false;  // the attribute is per function: set once
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gdn_sequence_kernel<DK>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg = {};
  const long ctas_per_head = (a.dv + P::RPC - 1) / P::RPC;
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<long>(a.B) * a.Hv * ctas_per_head));
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
  if (a.T > 1 && aligned(a.q, 16) && aligned(a.k, 16)) return launch_seq<DK>(a, st);
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
