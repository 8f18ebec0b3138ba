// prefill.cu -- many tokens per call: the routed and shared experts as grouped
// GEMMs on the 5th-generation tensor cores (tcgen05, fp32 accumulators in TMEM).
//
// With thousands of tokens the block is a dense contraction: each expert in
// use multiplies its dequantised weights by the activations of the tokens
// routed to it.  A work unit is one output tile D[128 weight rows][<=128
// tokens] of one expert, computed "swap-AB" (M = weight rows, N = tokens) so
// that an expert with few tokens shrinks N (any multiple of 16) instead of
// padding a token tile of 128:
//
//   gate/up : D = [Wg;Wu]_tile . X_tile^T    K = hidden.  Rows 2i and 2i+1 of
//             a blob are gate and up row i, so SwiGLU pairs neighbouring TMEM
//             lanes.  h = silu(gate) * up is stored bf16, one row per pair
//             (in permuted order) and one per token for the shared expert.
//   down    : D = Wd_tile . H_tile^T         K = inter.  The epilogue adds
//             w_tj * D into an fp32 [T][hidden] accumulator (reductions in
//             L2); the shared expert's weight is sigmoid(x . wsg).
//
// The kernel is persistent (one CTA per SM walks the units in a fixed
// stride) and warp-specialised:
//   warp 0      issues tcgen05.mma (one thread) into one of two TMEM
//               accumulators, so the epilogue of a unit overlaps the next
//               unit's main loop;
//   warps 1-7   produce K-chunks of 64: per-thread asynchronous copies bring
//               the packed int4 codes, the scale/bias words and the token rows
//               (the latter straight into the 128-byte-swizzled K-major layout
//               the tensor core reads); the codes are then dequantised (MLX
//               affine, w = s q + b; Swiftlet README, "MLX affine int4/int8
//               group quantization") to bf16 into the same layout;
//   warps 8-11  epilogue: tcgen05.ld of the accumulator, SwiGLU or the
//               weighted reduction.
// A ring of 4 shared-memory stages with full/empty mbarriers connects
// producers and MMA; the copies run two chunks ahead of the dequantisation.
// Every wait is bounded (1 s): on expiry the kernel records MOE_ERR_TIMEOUT,
// all roles leave their loops and the TMEM is released.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "moe_internal.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;       // weight rows per unit (UMMA M)
constexpr int kBN = 128;       // tokens per tile (largest UMMA N used)
constexpr int kBK = 64;        // K per chunk: one 128-byte swizzle row of bf16
constexpr int kStages = 4;
constexpr int kAhead = 2;      // chunks whose copies are in flight ahead of the dequantisation
constexpr int kProdWarps = 7;
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kEpiWarp0 = 1 + kProdWarps;       // 8: TMEM lane quarter = warp % 4
constexpr int kThreads = (kEpiWarp0 + 4) * 32;  // 384
constexpr int kAccCols = 128;  // TMEM columns per accumulator
constexpr int kTmemCols = 2 * kAccCols;
constexpr int kTileBytes = kBM * kBK * 2;  // 16 KiB (A and B alike)
constexpr int kRawCodes = kBM * kBK / 2;   // 4 KiB of packed codes per chunk
constexpr int kRawSbWords = kBM * 2;       // up to 2 scale/bias words per row per chunk
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr int kBarProd = 1, kBarEpi = 2;   // named barrier ids

static_assert(kStages >= kAhead + 2, "the stage a copy targets must be two MMAs old");
static_assert(kBN == kBM, "one producer thread per token row of B");

struct Tile {
  int slot;   // expert slot, or -1 for the shared expert
  int pos0;   // first pair position (routed) or first token (shared)
  int ntok;   // tokens in the tile, 0 < ntok <= kBN (0: skipped)
  int hrow0;  // first row of h that the tile owns
};

struct GemmArgs {
  const uint16_t* x;       // [T][H] bf16
  const int32_t* perm;     // pair ids sorted by expert
  const float* topk_w;     // [T*k]
  const float* gate;       // [T] sigmoid(x . wsg)
  const uint8_t* pool;     // routed blobs
  BlobLayout L;
  const uint8_t* shared_blob;
  BlobLayout LS;
  const Tile* tiles;
  const int32_t* n_tiles;
  uint16_t* h;             // [P + T][hstride] bf16
  float* y_acc;            // [T][H] fp32 (zero on entry to the down GEMM)
  int32_t* err;
  int k, H, I, Is, G, hstride, nm;  // nm: weight-row tiles per token tile
  int test_stall;  // MOE_TEST_WAIT_TIMEOUT: the MMA issuer first waits on a phase nothing completes
};

struct Smem {
  uint8_t a[kStages][kTileBytes];  // dequantised weights, swizzled K-major
  uint8_t b[kStages][kTileBytes];  // token rows, swizzled K-major
  uint8_t raw[kStages][kRawCodes];
  uint32_t rsb[kStages][kRawSbWords];
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int tok_t[kBN];
  float tok_w[kBN];
};

// ---- descriptors -----------------------------------------------------------
// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout: rows of 64 bf16 (128 B), 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);  // start address
  d |= (uint64_t)1 << 16;                           // leading byte offset (unused here)
  d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset: one 8-row group
  d |= (uint64_t)1 << 46;                           // descriptor version
  d |= (uint64_t)2 << 61;                           // swizzle: 128 bytes
  return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major.
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `row` in a swizzled tile.
__device__ __forceinline__ uint32_t sw128_off(int row, int ch) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4));
}

// ---- dequantisation --------------------------------------------------------
// 32 codes (one uint4; code 8j+i at bits 4i of word j) with their group's
// scale s and bias b -> 32 bf16 in four 16-byte chunks.  In fp32,
// 1 + q/128 is built by byte permutation, and s q + b = (128 s)(1 + q/128) +
// (b - 128 s): one FMA per code, then round to nearest even bf16.
__device__ __forceinline__ void dequant32(uint4 w, uint32_t sb, uint4 (&out)[4]) {
  const float s128 = 128.0f * bf16_lo(sb);
  const float off = bf16_hi(sb) - s128;
  const float2 s2 = make_float2(s128, s128), o2 = make_float2(off, off);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = (ws[j] & 0x0F0F0F0Fu) | 0x80808080u;         // codes 0, 2, 4, 6
    const uint32_t hi = ((ws[j] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;  // codes 1, 3, 5, 7
    uint32_t pk[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float f0 = __uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044u | (b << 8)));
      const float f1 = __uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044u | (b << 8)));
      const float2 v = __ffma2_rn(s2, make_float2(f0, f1), o2);
      const __nv_bfloat162 p = __floats2bfloat162_rn(v.x, v.y);
      pk[b] = *reinterpret_cast<const uint32_t*>(&p);
    }
    out[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
}

// ---- bounded waits -----------------------------------------------------------
// Wait for phase `parity` of `bar`.  Gives up when another role has aborted
// or after kWaitNs (then records MOE_ERR_TIMEOUT and aborts the CTA).
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Smem& S,
                                           int32_t* err) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (*(volatile int*)&S.abort) return false;
      if (ptx::globaltimer_ns() - t0 > kWaitNs) {
        record_error(err, MOE_ERR_TIMEOUT);
        *(volatile int*)&S.abort = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool aborted(Smem& S) { return *(volatile int*)&S.abort != 0; }

// ---- the unit walk -----------------------------------------------------------
// Units u = blockIdx.x, +gridDim.x, ...; u = tile * nm + m.  A unit is
// skipped when its tile is empty or m is past the expert's rows.  Every role
// walks the same sequence.
template <bool DOWN>
struct Walk {
  int u, U;
  Tile t;
  int m0, nk, c;
  bool live;

  __device__ __forceinline__ void seek(const GemmArgs& a) {
    live = false;
    for (; u < U; u += gridDim.x) {
      t = a.tiles[u / a.nm];
      const int inter = t.slot < 0 ? a.Is : a.I;
      const int rows = DOWN ? a.H : 2 * inter;
      m0 = (u % a.nm) * kBM;
      if (t.ntok > 0 && m0 < rows) {
        nk = (DOWN ? inter : a.H) / kBK;
        c = 0;
        live = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void start(const GemmArgs& a, int n_units) {
    u = blockIdx.x;
    U = n_units;
    seek(a);
  }
  __device__ __forceinline__ void next_unit(const GemmArgs& a) {
    u += gridDim.x;
    seek(a);
  }
  // next chunk; true when it begins a new unit (or the walk ended)
  __device__ __forceinline__ bool next(const GemmArgs& a) {
    if (++c < nk) return false;
    next_unit(a);
    return true;
  }
};

template <bool DOWN>
__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_units = *a.n_tiles * a.nm;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&S.full[s], kProdWarps);
      ptx::mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&S.acc_full[b], 1);
      ptx::mbar_init(&S.acc_empty[b], 4);
    }
    ptx::mbar_init(&S.drain, 1);
    S.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc(&S.tmem_base, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      Walk<DOWN> w;
      w.start(a, n_units);
      uint32_t g = 0, ub = 0;
      bool ok = true;
      // test hook: no arrival precedes the final commit, so this wait runs out
      if (a.test_stall) ok = wait_phase(&S.drain, 0, S, a.err);
      while (ok && w.live) {
        const int nmma = max(16, (w.t.ntok + 15) & ~15);
        const uint32_t idesc = idesc_bf16(kBM, nmma);
        const int buf = ub & 1;
        if (ub >= 2 && !wait_phase(&S.acc_empty[buf], ((ub >> 1) + 1) & 1, S, a.err)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * kAccCols;
        do {
          const int s = g % kStages;
          if (!wait_phase(&S.full[s], (g / kStages) & 1, S, a.err)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(S.a[s]), sbb = ptx::smem_u32(S.b[s]);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            ptx::tc_mma_f16(d, sw128_desc(sa + kk * 32), sw128_desc(sbb + kk * 32), idesc,
                            (w.c > 0 || kk > 0) ? 1u : 0u);
          ptx::tc_commit(&S.empty[s]);
          ++g;
        } while (!w.next(a));
        if (!ok) break;
        ptx::tc_commit(&S.acc_full[buf]);
        ++ub;
      }
      // every MMA issued has completed before the TMEM is released
      ptx::tc_commit(&S.drain);
      wait_phase(&S.drain, 0, S, a.err);
    }
    __syncwarp();
  } else if (warp < kEpiWarp0) {
    // ------------------------------------------------------------ producers
    const int pt = threadIdx.x - 32;  // 0 .. 223
    const int sbw = a.G < kBK ? kBK / a.G : 1;  // scale/bias words per row per chunk
    Walk<DOWN> wi, wp;  // issue cursor (kAhead chunks ahead) and dequantisation cursor
    wi.start(a, n_units);
    wp = wi;
    const uint16_t* brow = nullptr;  // this thread's token row (pt < kBN)
    const uint32_t* wq = nullptr;    // packed codes of row m0 of the issue unit
    const uint32_t* wsb = nullptr;
    int ldw = 0, lsb = 0;
    auto unit_setup = [&]() {
      const Tile& t = wi.t;
      const bool sh = t.slot < 0;
      const BlobLayout& B = sh ? a.LS : a.L;
      const uint8_t* blob = sh ? a.shared_blob : a.pool + (uint64_t)t.slot * a.L.stride;
      const int K = wi.nk * kBK;
      ldw = K / 8;
      lsb = K / a.G;
      wq = reinterpret_cast<const uint32_t*>(blob + (DOWN ? B.d_q : B.gu_q)) +
           (size_t)wi.m0 * ldw;
      wsb = reinterpret_cast<const uint32_t*>(blob + (DOWN ? B.d_sb : B.gu_sb)) +
            (size_t)wi.m0 * lsb;
      brow = nullptr;
      if (pt < t.ntok) {
        if (DOWN) {
          brow = a.h + (size_t)(t.hrow0 + pt) * a.hstride;
        } else {
          const int tok = sh ? t.pos0 + pt : a.perm[t.pos0 + pt] / a.k;
          brow = a.x + (size_t)tok * a.H;
        }
      }
    };
    // copies of the chunk under the issue cursor into stage gi % kStages
    auto issue = [&](uint32_t gi) {
      const int s = gi % kStages;
      const int c = wi.c;
      if (brow) {
        uint8_t* dst = S.b[s];
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
          ptx::cp_async16(dst + sw128_off(pt, ch), brow + c * kBK + ch * 8);
      }
      if (pt >= kBN) {
        for (int v = pt - kBN; v < 3 * kBM; v += kProdThreads - kBN) {
          if (v < 2 * kBM) {
            const int r = v >> 1, half = v & 1;
            ptx::cp_async16(S.raw[s] + r * 32 + half * 16,
                            wq + (size_t)r * ldw + c * 8 + half * 4);
          } else {
            const int r = v - 2 * kBM;
            const uint32_t* src = wsb + (size_t)r * lsb + (c * kBK) / a.G;
            if (sbw == 2)
              ptx::cp_async8(&S.rsb[s][2 * r], src);
            else
              ptx::cp_async4(&S.rsb[s][r], src);
          }
        }
      }
    };
    bool wi_new = true;
    uint32_t gi = 0, gp = 0;
    bool abort = false;
    for (int j = 0; j < kAhead; ++j) {
      if (wi.live) {
        if (wi_new) unit_setup();
        issue(gi++);
        wi_new = wi.next(a);
      }
      ptx::cp_async_commit();
    }
    while (wp.live) {
      // copies for the chunk kAhead ahead, once the MMA has released its stage
      if (wi.live && !abort) {
        if (gi >= kStages &&
            !wait_phase(&S.empty[gi % kStages], ((gi / kStages) + 1) & 1, S, a.err)) {
          abort = true;
        } else {
          if (wi_new) unit_setup();
          issue(gi++);
          wi_new = wi.next(a);
        }
      }
      ptx::cp_async_commit();
      ptx::cp_async_wait<kAhead>();
      // every producer's copies of chunk gp have landed, or the CTA aborts
      if (ptx::bar_any(kBarProd, kProdThreads, abort || aborted(S))) break;
      const int s = gp % kStages;
      for (int u = pt; u < 2 * kBM; u += kProdThreads) {
        const int r = u >> 1, half = u & 1;
        const uint4 w = *reinterpret_cast<const uint4*>(S.raw[s] + r * 32 + half * 16);
        const uint32_t sbv = sbw == 2 ? S.rsb[s][2 * r + half] : S.rsb[s][r];
        uint4 o[4];
        dequant32(w, sbv, o);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4*>(S.a[s] + sw128_off(r, half * 4 + j)) = o[j];
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.full[s]);
      ++gp;
      wp.next(a);
    }
    ptx::cp_async_wait_all();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                       // TMEM lane quarter
    const int et = threadIdx.x - kEpiWarp0 * 32;  // 0 .. 127
    const int r = q * 32 + lane;                  // row of the unit
    Walk<DOWN> w;
    w.start(a, n_units);
    uint32_t ub = 0;
    while (w.live) {
      const Tile t = w.t;
      if (DOWN && et < t.ntok) {
        // column -> token and routing weight
        if (t.slot < 0) {
          S.tok_t[et] = t.pos0 + et;
          S.tok_w[et] = a.gate[t.pos0 + et];
        } else {
          const int p = a.perm[t.pos0 + et];
          S.tok_t[et] = p / a.k;
          S.tok_w[et] = a.topk_w[p];
        }
      }
      const int buf = ub & 1;
      const bool ok = wait_phase(&S.acc_full[buf], (ub >> 1) & 1, S, a.err);
      // one decision for all four warps (and the table is complete)
      if (ptx::bar_any(kBarEpi, 128, !ok || aborted(S))) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + buf * kAccCols + ((uint32_t)(q * 32) << 16);
      const int grow = w.m0 + r;
      for (int n0 = 0; n0 < t.ntok; n0 += 16) {
        float v[16];
        ptx::tmem_ld16(taddr + n0, v);
        if (!DOWN) {
          // gate row 2i in an even lane, up row 2i+1 in the next lane
          uint16_t* hrow = a.h + (size_t)(t.hrow0 + n0) * a.hstride + (grow >> 1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float up = __shfl_xor_sync(0xffffffffu, v[i], 1);
            if ((lane & 1) == 0 && n0 + i < t.ntok)
              hrow[(size_t)i * a.hstride] = f32_to_bf16_rne(silu_f(v[i]) * up);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int n = n0 + i;
            if (n < t.ntok)
              atomicAdd(a.y_acc + (size_t)S.tok_t[n] * a.H + grow, S.tok_w[n] * v[i]);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.acc_empty[buf]);
      // the table is read by every warp before the next unit rewrites it
      if (DOWN) ptx::bar_any(kBarEpi, 128, false);
      ++ub;
      w.next_unit(a);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---- the tile list -------------------------------------------------------------
// One CTA: tiles of up to kBN pair positions for each expert in use (ascending
// id), then the shared expert's tiles over all T tokens.  An expert without a
// resident slot records MOE_ERR_SLOT and its tiles are left empty.
__global__ void __launch_bounds__(1024) build_tiles_kernel(
    const int32_t* __restrict__ used, const int32_t* __restrict__ n_used,
    const int32_t* __restrict__ offsets, const int32_t* __restrict__ table, int n_slots, int T,
    int P, Tile* __restrict__ tiles, int32_t* __restrict__ n_tiles, int max_tiles,
    int32_t* err) {
  __shared__ int warp_tot[32];
  const int nu = *n_used;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int cnt = 0, e = -1;
  if ((int)threadIdx.x < nu) {
    e = used[threadIdx.x];
    cnt = (offsets[e + 1] - offsets[e] + kBN - 1) / kBN;
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int nb = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += nb;
    }
    warp_tot[lane] = v;
  }
  __syncthreads();
  const int first = (warp ? warp_tot[warp - 1] : 0) + incl - cnt;
  const int routed = warp_tot[31];
  if (e >= 0) {
    const int slot = table ? table[e] : e;
    const bool bad = slot < 0 || slot >= n_slots;
    if (bad) record_error(err, MOE_ERR_SLOT);
    const int p0 = offsets[e], n_e = offsets[e + 1] - p0;
    for (int i = 0; i < cnt; ++i) {
      const int id = first + i;
      if (id < max_tiles)
        tiles[id] = Tile{bad ? 0 : slot, p0 + i * kBN, bad ? 0 : min(kBN, n_e - i * kBN),
                         p0 + i * kBN};
    }
  }
  const int nsh = (T + kBN - 1) / kBN;
  for (int i = threadIdx.x; i < nsh; i += blockDim.x) {
    const int id = routed + i;
    if (id < max_tiles) tiles[id] = Tile{-1, i * kBN, min(kBN, T - i * kBN), P + i * kBN};
  }
  if (threadIdx.x == 0) *n_tiles = min(max_tiles, routed + nsh);
}

// y = bf16(y_acc), four elements per thread step
__global__ void finalize_kernel(const float* __restrict__ y_acc, uint16_t* __restrict__ y,
                                int64_t n4) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(y_acc)[i];
    uint2 o;
    o.x = f32_to_bf16_rne(v.x) | ((uint32_t)f32_to_bf16_rne(v.y) << 16);
    o.y = f32_to_bf16_rne(v.z) | ((uint32_t)f32_to_bf16_rne(v.w) << 16);
    reinterpret_cast<uint2*>(y)[i] = o;
  }
}

constexpr size_t kGemmSmem = sizeof(Smem) + 1024;
static_assert(kGemmSmem <= 227 * 1024, "shared memory");

}  // namespace

int prefill_max_tiles(const Dims& d, int max_T) {
  const int64_t P = (int64_t)max_T * d.k;
  const int64_t routed = P / kBN + (P < d.E ? P : d.E);
  return (int)(routed + (max_T + kBN - 1) / kBN);
}

bool prefill_supported(const Dims& d) {
  return d.H % kBM == 0 && (2 * d.I) % kBM == 0 && (2 * d.Is) % kBM == 0 && d.I % kBK == 0 &&
         d.Is % kBK == 0 && d.E <= 1024;
}

cudaError_t prepare_prefill(const Ctx& c) {
  (void)c;
  cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemmSmem);
}

cudaError_t launch_prefill_experts(const Ctx& c, const FwdArgs& fa, cudaStream_t st,
                                   int* launches) {
  const Dims& d = c.d;
  const int T = fa.T, P = T * d.k;
  const int max_tiles = prefill_max_tiles(d, T);
  Tile* tiles = reinterpret_cast<Tile*>(c.ws.tiles);
  build_tiles_kernel<<<1, 1024, 0, st>>>(c.ws.used, c.ws.n_used, c.ws.offsets, fa.table,
                                         c.n_slots, T, P, tiles, c.ws.n_tiles, max_tiles, c.err);
  cudaError_t e = cudaMemsetAsync(c.ws.o, 0, (size_t)T * d.H * 4, st);
  if (e != cudaSuccess) return e;
  GemmArgs a;
  a.x = fa.x;
  a.perm = c.ws.perm;
  a.topk_w = fa.topk_w;
  a.gate = c.ws.gate;
  a.pool = c.pool;
  a.L = c.ex;
  a.shared_blob = c.shared;
  a.LS = c.sh;
  a.tiles = tiles;
  a.n_tiles = c.ws.n_tiles;
  a.h = reinterpret_cast<uint16_t*>(c.ws.h);
  a.y_acc = c.ws.o;
  a.err = c.err;
  a.k = d.k;
  a.H = d.H;
  a.I = d.I;
  a.Is = d.Is;
  a.G = d.G;
  a.hstride = d.I > d.Is ? d.I : d.Is;
  a.nm = 2 * a.hstride / kBM;
  a.test_stall = (c.test_flags & MOE_TEST_WAIT_TIMEOUT) ? 1 : 0;
  grouped_gemm_kernel<false><<<c.num_sms, kThreads, kGemmSmem, st>>>(a);
  a.nm = d.H / kBM;
  grouped_gemm_kernel<true><<<c.num_sms, kThreads, kGemmSmem, st>>>(a);
  const int64_t n4 = (int64_t)T * d.H / 4;
  finalize_kernel<<<4 * c.num_sms, 256, 0, st>>>(c.ws.o, fa.y, n4);
  *launches += 4;
  return cudaGetLastError();
}

}  // namespace moe
