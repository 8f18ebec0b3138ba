// fused_decode.cu -- the whole MoE block for one token in one launch.
//
// Decode moves ~17-22 MB of int4 expert weights per layer and token, so it is
// bound by HBM bandwidth and by latency, not by arithmetic.  One persistent
// CTA per SM runs the block in four phases separated by two bounded grid
// barriers:
//
//   P0  before waiting on the previous kernel (programmatic dependent launch):
//       bulk-copy (TMA, 1-D) this CTA's slice of the router rows, of the shared
//       expert's gate/up rows and of its down rows into shared memory -- these
//       are weights and do not depend on earlier kernels;
//   P1  router logits with their rigorous error bounds, and the shared
//       expert's gate/up + SwiGLU (neither depends on routing);
//       -- grid barrier --
//   P2  every CTA selects the top-k itself with all its warps (exact order,
//       routing_common.cuh),
//       then bulk-copies its share of the selected experts' gate/up rows and
//       its rows of their down projections;
//   P3  gate/up + SwiGLU of the selected experts from shared memory;
//       -- grid barrier --
//   P4  this CTA's rows of y: sum_j w_j (Wd_j h_j) + g (Wd_s h_s), fixed order
//       (deterministic), bf16 out.
//
// The int4 dot products fold the affine terms per 32-code chunk, with the
// codes turned into floats 1 + q/128 by one byte-permute each:
//   sum_c (s q_c + b) x_c = (128 s) * sum_c (1 + q_c/128) x_c + (b - 128 s) * sum_c x_c,
// two codes per packed fp32 FMA (FFMA2).  Each lane keeps the inputs of its
// own chunks (x, or h in P4) in registers, read once from global memory.
// Weights follow the MLX affine int4 group layout (Swiftlet README, its list
// of what was built).
#include "device_util.cuh"
#include "moe_internal.cuh"
#include "routing_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

using namespace rt;

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr uint32_t kBarSpin = 1u << 22;    // grid-barrier polls (and a 1 s limit)
constexpr uint32_t kMbarTries = 1u << 22;  // mbarrier try_waits
constexpr int kNumMbar = 10;               // 0: P0 weights, 1..8: P3 warps, 9: P4 down rows

struct FusedSmem {  // byte offsets into dynamic shared memory
  uint32_t mbar, misc, topk, lists, p1, sd, p3, p3_warp, p4, p4_expert, p4_sb, ypart, total;
  uint32_t p1_max;    // bytes reserved for router + shared gate/up rows
  uint32_t seg_max;   // row-pairs per warp segment (max)
  uint32_t nrow_max;  // P4 rows per CTA (max)
};

struct FusedArgs {
  const uint16_t* x;
  const uint16_t* router_w;
  const float* prior;
  const uint16_t* shared_gate_w;
  const uint8_t* pool;
  BlobLayout L;
  const uint8_t* shared_blob;
  BlobLayout LS;
  const int32_t* table;
  int n_slots;
  uint16_t* y;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* perm_out;
  int32_t* offsets_out;
  float* logits;
  float* bound;
  float* gate_z;
  float* h;   // [k][I]
  float* hs;  // [I]
  unsigned long long* bar;
  uint32_t bar_extra;  // test hook: arrivals the barrier waits for beyond the grid
  int32_t* err;
  int E, k, I, G;
  uint64_t inv_nc, inv_i;  // ceil(2^32 / gridDim.x), ceil(2^32 / I): see udiv
  uint64_t inv_nrow[2];    // the same for the two row counts H / gridDim.x (+1) of P4
  uint64_t inv_bar;        // ceil(2^64 / barrier arrivals): see grid_barrier
  FusedSmem sm;
};

// x / d for x * d < 2^32, with m = ceil(2^32 / d) from the host: writing
// m d = 2^32 + e (0 <= e < d), x m / 2^32 = x / d + x e / (d 2^32) and the
// excess is below 1/d, so the floor is exact.  Two instructions instead of a
// division routine; this code runs once per launch, where every instruction
// counts.
__device__ __forceinline__ int udiv(uint32_t x, uint64_t m) {
  return (int)(((uint64_t)x * m) >> 32);
}

// Start of share p of n items split into gridDim.x shares (n * p * gridDim.x
// < 2^32 here: n <= 32768 row pairs, p <= gridDim.x <= a few hundred).
__device__ __forceinline__ int part(int n, int p, uint64_t inv_nc) {
  return udiv((uint32_t)n * (uint32_t)p, inv_nc);
}

// Grid-wide barrier on a monotonic 64-bit arrival counter: barrier number b
// (counting from the last reset) is passed once the counter reaches
// (b + 1) * n, so one atomic round trip per CTA suffices, and the last
// arrival's atomic is itself the release.  b = old / n comes from a
// multiply-high with inv_n = ceil(2^64 / n) (exact while old < 2^64 / n; see
// udiv) instead of a 64-bit division routine.  Polls stop after kBarSpin
// tries or one second (no sleep between polls: each is an L2 round trip,
// and a sleep would only delay the wake-up); on expiry the sticky error word
// gets MOE_ERR_TIMEOUT and the CTA carries on (no trap, no hang).
__device__ void grid_barrier(unsigned long long* bar, uint32_t n, uint64_t inv_n, int32_t* err) {
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned long long old = ptx::atom_add_acq_rel_u64(bar, 1ull);
    const unsigned long long target = (__umul64hi(old, inv_n) + 1) * n;
    if (old + 1 < target) {
      const uint64_t t0 = ptx::globaltimer_ns();
      uint32_t it = 0;
      while (ptx::ld_acquire_u64(bar) < target) {
        if (++it > kBarSpin || ptx::globaltimer_ns() - t0 > 1000000000ull) {
          record_error(err, MOE_ERR_TIMEOUT);
          break;
        }
      }
    }
  }
  __syncthreads();
}

__device__ __forceinline__ void wait_or_flag(uint64_t* bar, uint32_t parity, int32_t* err) {
  if (!ptx::mbar_wait(bar, parity, kMbarTries)) record_error(err, MOE_ERR_TIMEOUT);
}

// sum_i (1 + q_i/128) x_i over the 32 codes of a chunk; x as 16 float2.
__device__ __forceinline__ float dot32_magic(uint4 w, const float2 (&x2)[16]) {
  float2 acc = make_float2(0.f, 0.f);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = (ws[j] & 0x0F0F0F0Fu) | 0x80808080u;         // codes 8j + 0,2,4,6
    const uint32_t hi = ((ws[j] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;  // codes 8j + 1,3,5,7
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float f0 = __uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044u | (b << 8)));
      const float f1 = __uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044u | (b << 8)));
      acc = __ffma2_rn(make_float2(f0, f1), x2[4 * j + b], acc);
    }
  }
  return acc.x + acc.y;
}

// Contribution of one 32-code chunk with packed (scale | bias << 16) and the
// chunk's input sum X.
__device__ __forceinline__ float chunk_term(uint4 w, uint32_t sb, const float2 (&x2)[16],
                                            float X) {
  const float s128 = 128.0f * bf16_lo(sb);
  return fmaf(s128, dot32_magic(w, x2), (bf16_hi(sb) - s128) * X);
}

// 32 consecutive bf16 from global memory as 16 float2, and their sum.
__device__ __forceinline__ float load_chunk_bf16(const uint16_t* src, float2 (&v)[16]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = __ldg(p + q);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      v[4 * q + r] = make_float2(bf16_lo(w[r]), bf16_hi(w[r]));
      s += v[4 * q + r].x + v[4 * q + r].y;
    }
  }
  return s;
}

// A 16-byte aligned window [lo, hi) around bytes [b0, b1) of a region whose
// size is a multiple of 16: returns lo and the padded length.
__device__ __forceinline__ void align16(uint64_t b0, uint64_t b1, uint64_t& lo, uint32_t& len) {
  lo = b0 & ~uint64_t(15);
  const uint64_t hi = (b1 + 15) & ~uint64_t(15);
  len = (uint32_t)(hi - lo);
}

template <int NJ, int MAXV>
__global__ void __launch_bounds__(kThreads, 1) fused_decode_kernel(const FusedArgs a) {
  constexpr int H = NJ * 256;
  constexpr int HC = H / 32;          // 32-code chunks per gate/up row
  constexpr int MC = (HC + 31) / 32;  // chunks per lane
  extern __shared__ __align__(1024) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nC = gridDim.x, c = blockIdx.x;
  const int E = a.E, k = a.k, I = a.I, G = a.G;
  const int lg = 31 - __clz(G);  // G is 32, 64 or 128: shifts instead of divisions
  const int HG = H >> lg, IG = I >> lg, IC = I / 32;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + a.sm.mbar);
  int* s_idx = reinterpret_cast<int*>(sm + a.sm.misc);
  float* s_w = reinterpret_cast<float*>(sm + a.sm.misc + 128);
  int* s_slot = reinterpret_cast<int*>(sm + a.sm.misc + 256);
  float* s_g = reinterpret_cast<float*>(sm + a.sm.misc + 384);
  float* ypart = reinterpret_cast<float*>(sm + a.sm.ypart);

  // unit ranges of this CTA
  const int U1 = E + I + 1;  // router rows, shared features, gate vector
  const int u0 = part(U1, c, a.inv_nc), u1 = part(U1, c + 1, a.inv_nc);
  const int re0 = min(u0, E), re1 = min(u1, E);
  const int si0 = min(max(u0 - E, 0), I), si1 = min(max(u1 - E, 0), I);
  const bool has_gv = (u0 <= E + I) && (E + I < u1);
  const int r0 = part(H, c, a.inv_nc), r1 = part(H, c + 1, a.inv_nc), nrow = r1 - r0;

  uint8_t* p1_rw = sm + a.sm.p1;
  uint8_t* p1_gq = p1_rw + (size_t)(re1 - re0) * H * 2;
  uint8_t* p1_gsb = p1_gq + (size_t)(si1 - si0) * H;
  uint8_t* p1_gv = sm + a.sm.p1 + a.sm.p1_max;
  uint8_t* sd_q = sm + a.sm.sd;
  uint8_t* sd_sb = sd_q + (size_t)a.sm.nrow_max * (I / 2);
  uint64_t dsb_lo;
  uint32_t dsb_len;  // window of rows [r0, r1) of a d_sb region (same for every expert)
  align16((uint64_t)r0 * IG * 4, (uint64_t)r1 * IG * 4, dsb_lo, dsb_len);
  const uint32_t dsb_off = (uint32_t)((uint64_t)r0 * IG * 4 - dsb_lo);

  // ---------------------------------------------------------------- P0
  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumMbar; ++i) ptx::mbar_init(&mbar[i], 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  ptx::griddep_launch_dependents();
  if (threadIdx.x == 0) {
    const uint32_t b_rw = (uint32_t)(re1 - re0) * H * 2;
    const uint32_t b_gq = (uint32_t)(si1 - si0) * H;
    const uint32_t b_gsb = (uint32_t)(si1 - si0) * 8 * HG;
    const uint32_t b_gv = has_gv ? H * 2 : 0;
    const uint32_t b_dq = (uint32_t)nrow * (I / 2);
    const uint32_t b_dsb = nrow > 0 ? dsb_len : 0;
    ptx::mbar_arrive_expect_tx(&mbar[0], b_rw + b_gq + b_gsb + b_gv + b_dq + b_dsb);
    if (b_rw) ptx::bulk_g2s(p1_rw, a.router_w + (size_t)re0 * H, b_rw, &mbar[0]);
    if (b_gq) ptx::bulk_g2s(p1_gq, a.shared_blob + a.LS.gu_q + (size_t)si0 * H, b_gq, &mbar[0]);
    if (b_gsb)
      ptx::bulk_g2s(p1_gsb, a.shared_blob + a.LS.gu_sb + (size_t)si0 * 8 * HG, b_gsb, &mbar[0]);
    if (b_gv) ptx::bulk_g2s(p1_gv, a.shared_gate_w, b_gv, &mbar[0]);
    if (b_dq) ptx::bulk_g2s(sd_q, a.shared_blob + a.LS.d_q + (size_t)r0 * (I / 2), b_dq, &mbar[0]);
    if (b_dsb) ptx::bulk_g2s(sd_sb, a.shared_blob + a.LS.d_sb + dsb_lo, b_dsb, &mbar[0]);
  }
  // everything below may read what earlier kernels wrote
  ptx::griddep_wait();

  // x in registers: router layout (8 bf16 per uint4, chunks lane + 32 j) and
  // expert layout (32 fp32 per chunk, chunks lane + 32 m, with chunk sums)
  uint4 xv[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) xv[j] = __ldg(reinterpret_cast<const uint4*>(a.x) + lane + 32 * j);
  float2 xr[MC][16];
  float xs_r[MC];
#pragma unroll
  for (int m = 0; m < MC; ++m) {
    const int ch = lane + 32 * m;
    xs_r[m] = load_chunk_bf16(a.x + (ch < HC ? ch : 0) * 32, xr[m]);
  }

  // ---------------------------------------------------------------- P1
  wait_or_flag(&mbar[0], 0, a.err);
  for (int u = u0 + warp; u < u1; u += kWarps) {
    if (u < E || u == E + I) {  // router row or the shared gate vector
      uint4 wv[NJ];
      const uint4* row =
          reinterpret_cast<const uint4*>(u < E ? p1_rw + (size_t)(u - re0) * H * 2 : p1_gv);
#pragma unroll
      for (int j = 0; j < NJ; ++j) wv[j] = row[lane + 32 * j];
      float sum, mag;
      router_row_dot_regs<NJ>(wv, xv, sum, mag);
      if (lane == 0) {
        if (u < E) {
          float l, b;
          router_logit_and_bound<NJ>(sum, mag, a.prior ? __ldg(a.prior + u) : 0.f, l, b);
          a.logits[u] = l;
          a.bound[u] = b;
        } else {
          a.gate_z[0] = sum;
        }
      }
    } else {  // shared expert feature i: gate/up + SwiGLU
      const int i = u - E;
      const uint4* q4 = reinterpret_cast<const uint4*>(p1_gq + (size_t)(i - si0) * H);
      const uint32_t* sb = reinterpret_cast<const uint32_t*>(p1_gsb + (size_t)(i - si0) * 8 * HG);
      float ag = 0.f, au = 0.f;
#pragma unroll
      for (int m = 0; m < MC; ++m) {
        const int ch = lane + 32 * m;
        if (ch < HC) {
          const int g = (ch * 32) >> lg;
          ag += chunk_term(q4[ch], sb[g], xr[m], xs_r[m]);
          au += chunk_term(q4[HC + ch], sb[HG + g], xr[m], xs_r[m]);
        }
      }
      ag = warp_sum(ag);
      au = warp_sum(au);
      if (lane == 0) a.hs[i] = silu_f(ag) * au;
    }
  }
  grid_barrier(a.bar, nC + a.bar_extra, a.inv_bar, a.err);

  // ---------------------------------------------------------------- P2
  {
    const float gz = __ldcg(a.gate_z);  // issued early: its latency overlaps the selection
    int* sel_idx;
    float* sel_val;
    topk_select_block<MAXV / kWarps>(PlainLogits{a.logits, a.bound}, E, k, a.x, a.router_w,
                                     a.prior, H, sm + a.sm.topk,
                                     reinterpret_cast<uint2*>(sm + a.sm.lists),
                                     reinterpret_cast<float*>(sm + a.sm.lists + MAXV * 32 * 8),
                                     &sel_idx, &sel_val);
    if (warp == 0) {
      const float w = renormalised_weight(sel_val, k);
      if (lane < k) {
        const int e = sel_idx[lane];
        const int slot = a.table ? __ldg(a.table + e) : e;
        const bool ok = slot >= 0 && slot < a.n_slots;
        s_idx[lane] = e;
        s_w[lane] = w;
        s_slot[lane] = ok ? slot : -1;
        if (!ok && c == 0) record_error(a.err, MOE_ERR_SLOT);
        if (c == 0) {
          a.topk_idx[lane] = e;
          a.topk_w[lane] = w;
        }
      }
      if (lane == 0) *s_g = 1.0f / (1.0f + __expf(-gz));
    }
  }
  __syncthreads();

  // P3 / P4 copies: each warp its own gate/up segment; the last warp also
  // fetches this CTA's rows of every selected expert's down projection
  const int R = k * I;
  const int R0 = part(R, c, a.inv_nc), R1 = part(R, c + 1, a.inv_nc);
  const int seg = (R1 - R0 + kWarps - 1) / kWarps;
  const int w0 = min(R1, R0 + warp * seg), w1 = min(R1, w0 + seg);
  uint8_t* p3w = sm + a.sm.p3 + (size_t)warp * a.sm.p3_warp;
  uint8_t* p3w_sb = p3w + (size_t)a.sm.seg_max * H;
  const uint32_t rp_sb = 8 * HG;  // sb bytes of one row-pair
  const int jw0 = udiv((uint32_t)w0, a.inv_i);  // expert of the segment's first row pair
  if (lane == 0) {
    uint32_t bytes = 0;
    for (int j = jw0, r = w0; r < w1; ++j) {
      const int n = min(w1, (j + 1) * I) - r;
      if (s_slot[j] >= 0) bytes += (uint32_t)n * (H + rp_sb);
      r += n;
    }
    ptx::mbar_arrive_expect_tx(&mbar[1 + warp], bytes);
    for (int j = jw0, r = w0; r < w1; ++j) {
      const int i = r - j * I, n = min(w1, (j + 1) * I) - r;
      if (s_slot[j] >= 0) {
        const uint8_t* blob = a.pool + (uint64_t)s_slot[j] * a.L.stride;
        ptx::bulk_g2s(p3w + (size_t)(r - w0) * H, blob + a.L.gu_q + (size_t)i * H,
                      (uint32_t)n * H, &mbar[1 + warp]);
        ptx::bulk_g2s(p3w_sb + (size_t)(r - w0) * rp_sb, blob + a.L.gu_sb + (size_t)i * rp_sb,
                      (uint32_t)n * rp_sb, &mbar[1 + warp]);
      }
      r += n;
    }
  }
  if (warp == kWarps - 1) {
    if (lane == 1) {
      uint32_t bytes = 0;
      for (int j = 0; j < k; ++j)
        if (s_slot[j] >= 0 && nrow > 0) bytes += (uint32_t)nrow * (I / 2) + dsb_len;
      ptx::mbar_arrive_expect_tx(&mbar[kNumMbar - 1], bytes);
    }
    __syncwarp();
    // lane j + 1 fetches expert j's down rows (lane 0 issues its own segment)
    for (int j = lane - 1; j >= 0 && j < k; j += 31) {
      if (s_slot[j] < 0 || nrow == 0) continue;
      const uint8_t* blob = a.pool + (uint64_t)s_slot[j] * a.L.stride;
      uint8_t* dst = sm + a.sm.p4 + (size_t)j * a.sm.p4_expert;
      ptx::bulk_g2s(dst, blob + a.L.d_q + (size_t)r0 * (I / 2), (uint32_t)nrow * (I / 2),
                    &mbar[kNumMbar - 1]);
      ptx::bulk_g2s(dst + a.sm.p4_sb, blob + a.L.d_sb + dsb_lo, dsb_len, &mbar[kNumMbar - 1]);
    }
  }
  // outputs of the permutation (T = 1: pair p = j)
  if (a.offsets_out) {
    for (int e = part(E + 1, c, a.inv_nc) + threadIdx.x; e < part(E + 1, c + 1, a.inv_nc);
         e += kThreads) {
      int cnt = 0;
      for (int j = 0; j < k; ++j) cnt += s_idx[j] < e;
      a.offsets_out[e] = cnt;
    }
  }
  if (a.perm_out && c == 0 && threadIdx.x < k) {
    int rank = 0;
    for (int j = 0; j < k; ++j) rank += s_idx[j] < s_idx[threadIdx.x];
    a.perm_out[rank] = threadIdx.x;
  }

  // ---------------------------------------------------------------- P3
  wait_or_flag(&mbar[1 + warp], 0, a.err);
  for (int r = w0, j = jw0, i = w0 - jw0 * I; r < w1; ++r, i = (i + 1 == I) ? 0 : i + 1,
           j += (i == 0)) {
    if (s_slot[j] < 0) continue;
    const uint4* q4 = reinterpret_cast<const uint4*>(p3w + (size_t)(r - w0) * H);
    const uint32_t* sb = reinterpret_cast<const uint32_t*>(p3w_sb + (size_t)(r - w0) * rp_sb);
    float ag = 0.f, au = 0.f;
#pragma unroll
    for (int m = 0; m < MC; ++m) {
      const int ch = lane + 32 * m;
      if (ch < HC) {
        const int g = (ch * 32) >> lg;
        ag += chunk_term(q4[ch], sb[g], xr[m], xs_r[m]);
        au += chunk_term(q4[HC + ch], sb[HG + g], xr[m], xs_r[m]);
      }
    }
    ag = warp_sum(ag);
    au = warp_sum(au);
    if (lane == 0) a.h[(size_t)j * I + i] = silu_f(ag) * au;
  }
  grid_barrier(a.bar, nC + a.bar_extra, a.inv_bar, a.err);

  // ---------------------------------------------------------------- P4
  // h of the selected experts and of the shared one into shared memory (the
  // P3 rows are dead now; 16-byte piece q of 32-float chunk c is stored at
  // piece q ^ (c & 7), so that the 16 lanes of a group reading chunks c..c+15
  // hit distinct banks), with each chunk's sum.  Then 16-lane groups take this
  // CTA's (expert, row) pairs round robin: every warp works, and a group's
  // serial chain is ~(k+1) nrow / 16 rows instead of nrow.
  {
    float4* s_h4 = reinterpret_cast<float4*>(sm + a.sm.p3);
    const int n4 = k * I / 4, ns4 = I / 4;
    for (int i = threadIdx.x; i < n4 + ns4; i += kThreads) {
      const float4 v = i < n4 ? __ldcg(reinterpret_cast<const float4*>(a.h) + i)
                              : __ldcg(reinterpret_cast<const float4*>(a.hs) + (i - n4));
      const int hc = i >> 3;
      s_h4[(hc << 3) | ((i ^ hc) & 7)] = v;
    }
  }
  wait_or_flag(&mbar[kNumMbar - 1], 0, a.err);
  __syncthreads();
  {
    const float4* s_h4 = reinterpret_cast<const float4*>(sm + a.sm.p3);
    float* s_x = reinterpret_cast<float*>(sm + a.sm.p3) + (size_t)(k + 1) * I;  // chunk sums
    for (int hc = threadIdx.x; hc < (k + 1) * IC; hc += kThreads) {
      float sum = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 u = s_h4[hc * 8 + ((q + hc) & 7)];  // rotated: distinct banks
        sum += (u.x + u.y) + (u.z + u.w);
      }
      s_x[hc] = sum;
    }
    __syncthreads();
    constexpr int kG = 16;                // lanes per pair
    constexpr int kGroups = kThreads / kG;
    const int grp = threadIdx.x / kG, sub = lane % kG;
    const int npairs = (k + 1) * nrow;
    // two pairs per group and pass (their shuffle reductions overlap); the
    // trip count depends on the warp only, so every shuffle sees all lanes
    for (int pb = 0; pb + 2 * warp < npairs; pb += 2 * kGroups) {
      float v[2];
      int jj[2], rr[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int pp = pb + u * kGroups + grp;
        v[u] = 0.f;
        jj[u] = -1;
        rr[u] = 0;
        if (pp < npairs) {
          const int j = udiv((uint32_t)pp, a.inv_nrow[nrow == a.sm.nrow_max]), rl = pp - j * nrow;
          const bool shared = j == k;
          if (shared || s_slot[j] >= 0) {
            jj[u] = j;
            rr[u] = rl;
            const uint8_t* eb = sm + a.sm.p4 + (size_t)j * a.sm.p4_expert;
            const uint4* qrow =
                reinterpret_cast<const uint4*>((shared ? sd_q : eb) + (size_t)rl * (I / 2));
            const uint32_t* sbrow = reinterpret_cast<const uint32_t*>(
                (shared ? sd_sb : eb + a.sm.p4_sb) + dsb_off + (size_t)rl * IG * 4);
            for (int ch = sub; ch < IC; ch += kG) {
              const int hc = j * IC + ch;
              float2 hr[16];
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 t = s_h4[hc * 8 + (q ^ (hc & 7))];
                hr[2 * q] = make_float2(t.x, t.y);
                hr[2 * q + 1] = make_float2(t.z, t.w);
              }
              v[u] += chunk_term(qrow[ch], sbrow[(ch * 32) >> lg], hr, s_x[hc]);
            }
          }
        }
      }
#pragma unroll
      for (int o = kG >> 1; o > 0; o >>= 1) {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        v[1] += __shfl_xor_sync(0xffffffffu, v[1], o);
      }
      if (sub == 0) {
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (jj[u] >= 0) ypart[rr[u] * (k + 1) + jj[u]] = v[u];
      }
    }
  }
  __syncthreads();
  for (int rl = threadIdx.x; rl < nrow; rl += kThreads) {
    float acc = 0.f;
    for (int j = 0; j < k; ++j)
      if (s_slot[j] >= 0) acc = fmaf(s_w[j], ypart[rl * (k + 1) + j], acc);
    acc = fmaf(*s_g, ypart[rl * (k + 1) + k], acc);
    a.y[r0 + rl] = f32_to_bf16_rne(acc);
  }
}

// Host-side shared-memory plan; false if the fused path does not fit.
bool plan_smem(const Ctx& c, int nC, FusedSmem& s) {
  const Dims& d = c.d;
  const int H = d.H, I = d.I, G = d.G, E = d.E, k = d.k;
  auto up = [](uint32_t v, uint32_t a) { return (v + a - 1) / a * a; };
  uint32_t off = 0;
  auto take = [&](uint32_t bytes) {
    const uint32_t o = off;
    off = up(off + bytes, 128);
    return o;
  };
  s.mbar = take(kNumMbar * 8);
  s.misc = take(512);
  s.topk = take((uint32_t)topk_warp_smem(E));
  // every warp's whole list (32 V entries, padding included), then the bounds
  const int mv = E <= 256 ? 8 : E <= 512 ? 16 : 32;  // MAXV of the dispatch
  s.lists = take((uint32_t)mv * 32 * 8 + kWarps * 4);
  // P1: worst CTA of router rows * 2H + shared features * (H + 8H/G)
  const int U1 = E + I + 1;
  uint32_t p1 = 0;
  for (int cc = 0; cc < nC; ++cc) {
    const int u0 = (int)(((long long)U1 * cc) / nC), u1 = (int)(((long long)U1 * (cc + 1)) / nC);
    const int nr = (u1 < E ? u1 : E) - (u0 < E ? u0 : E);
    const int a0 = u0 - E < 0 ? 0 : (u0 - E > I ? I : u0 - E);
    const int a1 = u1 - E < 0 ? 0 : (u1 - E > I ? I : u1 - E);
    const uint32_t b = (uint32_t)nr * H * 2 + (uint32_t)(a1 - a0) * (H + 8 * (H / G));
    p1 = b > p1 ? b : p1;
  }
  s.p1_max = up(p1, 128);
  s.p1 = take(s.p1_max + H * 2);
  s.nrow_max = (uint32_t)((H + nC - 1) / nC);
  const uint32_t dsb_max = up(s.nrow_max * (I / G) * 4, 16) + 16;
  s.sd = take(s.nrow_max * (I / 2) + dsb_max);
  const int R = k * I;
  const uint32_t per_cta = (uint32_t)((R + nC - 1) / nC);
  s.seg_max = (per_cta + kWarps - 1) / kWarps;
  s.p3_warp = up(s.seg_max * (H + 8 * (H / G)), 128);
  const uint32_t h_bytes = (uint32_t)(k + 1) * (I + I / 32) * 4;  // P4: h and chunk sums
  s.p3 = take(kWarps * s.p3_warp > h_bytes ? kWarps * s.p3_warp : h_bytes);
  s.p4_sb = up(s.nrow_max * (I / 2), 16);
  s.p4_expert = up(s.p4_sb + dsb_max, 128);
  s.p4 = take(s.p4_expert * k);
  s.ypart = take(s.nrow_max * (k + 1) * 4);
  s.total = off;
  return s.total <= 227 * 1024;
}

template <int NJ, int MAXV>
cudaError_t launch_fused_t(const FusedArgs& a, int nC, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nC);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.sm.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_decode_kernel<NJ, MAXV>, a);
}

template <int NJ, int MAXV>
cudaError_t prepare_t(int smem, int* occ) {
  cudaError_t e = cudaFuncSetAttribute(fused_decode_kernel<NJ, MAXV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, fused_decode_kernel<NJ, MAXV>,
                                                       kThreads, smem);
}

bool shape_ok(const Dims& d) {
  const int nj = d.H / 256;
  return d.bits == 4 && (nj == 1 || nj == 2 || nj == 4 || nj == 8) && d.I == d.Is &&
         d.I <= 1024 &&
         d.E <= kMaxE;
}

// Dispatch over (H / 256) x per-lane top-k list length.
template <template <int, int> class F, typename... Args>
cudaError_t dispatch(const Dims& d, Args... args) {
  const int mv = d.E <= 256 ? 8 : d.E <= 512 ? 16 : 32;
#define MOE_FUSED_CASE(NJ)                                     \
  case NJ:                                                     \
    return mv == 8 ? F<NJ, 8>::run(args...)                    \
                   : mv == 16 ? F<NJ, 16>::run(args...) : F<NJ, 32>::run(args...);
  switch (d.H / 256) {
    MOE_FUSED_CASE(1)
    MOE_FUSED_CASE(2)
    MOE_FUSED_CASE(4)
    MOE_FUSED_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_FUSED_CASE
}

template <int NJ, int MAXV>
struct PrepareF {
  static cudaError_t run(int smem, int* occ) { return prepare_t<NJ, MAXV>(smem, occ); }
};
template <int NJ, int MAXV>
struct LaunchF {
  static cudaError_t run(const FusedArgs* a, int nC, cudaStream_t st) {
    return launch_fused_t<NJ, MAXV>(*a, nC, st);
  }
};

}  // namespace

bool fused_decode_supported(const Ctx& c) { return shape_ok(c.d) && c.fused_ctas > 0; }

cudaError_t prepare_fused_decode(Ctx& c) {
  c.fused_ctas = 0;
  if (!shape_ok(c.d)) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  FusedSmem s;
  if (!plan_smem(c, sms, s)) return cudaSuccess;
  int occ = 0;
  e = dispatch<PrepareF>(c.d, (int)s.total, &occ);
  if (e != cudaSuccess) return e;
  if (occ >= 1) c.fused_ctas = sms;
  return cudaSuccess;
}

cudaError_t launch_fused_decode(const Ctx& c, const FwdArgs& fa, cudaStream_t st, int* launches) {
  const Dims& d = c.d;
  FusedArgs a;
  a.x = fa.x;
  a.router_w = c.router_w;
  a.prior = c.router_bias;
  a.shared_gate_w = c.shared_gate_w;
  a.pool = c.pool;
  a.L = c.ex;
  a.shared_blob = c.shared;
  a.LS = c.sh;
  a.table = fa.table;
  a.n_slots = c.n_slots;
  a.y = fa.y;
  a.topk_idx = fa.topk_idx;
  a.topk_w = fa.topk_w;
  a.perm_out = fa.perm_out;
  a.offsets_out = fa.offsets_out;
  a.logits = c.ws.logits;
  a.bound = c.ws.bound;
  a.gate_z = c.ws.gate_z;
  a.h = c.ws.h;
  a.hs = c.ws.h + (size_t)d.k * d.I;
  a.bar = c.ws.bar;
  a.bar_extra = (c.test_flags & MOE_TEST_WAIT_TIMEOUT) ? 1u : 0u;
  a.err = c.err;
  a.E = d.E;
  a.k = d.k;
  a.I = d.I;
  a.G = d.G;
  const int nC = c.fused_ctas;
  a.inv_nc = ((1ull << 32) + (uint64_t)nC - 1) / (uint64_t)nC;
  a.inv_i = ((1ull << 32) + (uint64_t)d.I - 1) / (uint64_t)d.I;
  const uint64_t nr_lo = (uint64_t)(d.H / nC), nr_hi = (uint64_t)((d.H + nC - 1) / nC);
  a.inv_nrow[0] = nr_lo ? ((1ull << 32) + nr_lo - 1) / nr_lo : 0;
  a.inv_nrow[1] = ((1ull << 32) + nr_hi - 1) / nr_hi;
  {
    const uint64_t nb = (uint64_t)nC + a.bar_extra;  // ceil(2^64 / nb) = floor((2^64 - 1) / nb) + 1
    a.inv_bar = ~0ull / nb + 1;
  }
  if (!plan_smem(c, nC, a.sm)) return cudaErrorInvalidConfiguration;
  ++*launches;
  return dispatch<LaunchF>(d, (const FusedArgs*)&a, nC, st);
}

}  // namespace moe
