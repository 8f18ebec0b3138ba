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
// Operand paths.  The token rows (B) arrive by per-thread asynchronous copies
// (any row ids; eight lanes per 128-byte row segment, so a warp moves four
// whole rows per instruction) straight into the 128-byte-swizzled K-major
// layout the tensor core reads from shared memory.  The packed int4 codes
// arrive by 3-D TMA tile copies, the scale/bias words of up to 32 groups per
// row at a time into a double-buffered window, and the weights (A) are
// dequantised (MLX affine, w = s q + b; Swiftlet README, its list of what
// was built) to bf16 straight into tensor
// memory, which the MMA reads as its A operand: A costs no shared-memory
// bandwidth and no proxy fence.
//
// The kernel is persistent (one CTA per SM walks the units in a fixed
// stride) and warp-specialised, so that no warp both waits for memory and
// computes:
//   warp 0       issues tcgen05.mma (one thread) into one of two TMEM
//                accumulators, so the epilogue of a unit overlaps the next
//                unit's main loop;
//   warps 1-8    loaders: for each K-chunk of 64, once its stage is free, the
//                copies (a ring of 8 stages; eight warps, because one warp's
//                gathers cannot keep up); each lane marks a stage full
//                kAhead chunks later, once its own copies have landed and are
//                fenced for the tensor core (the TMA copy of the codes counts
//                on the same mbarrier);
//   warps 9-16   dequantise a landed stage into the stage's TMEM A tile (two
//                warps per TMEM lane quarter, one K-half each);
//   warps 17-20  epilogue: tcgen05.ld of the accumulator, then SwiGLU (gate/
//                up) or the routing-weighted fp32 vector reductions (down),
//                both through a small shared-memory transpose so that every
//                global access is 16 bytes wide.
// Every wait is bounded (1 s): on expiry the kernel records MOE_ERR_TIMEOUT,
// all roles leave their loops and the TMEM is released.
#include <cuda.h>
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "moe_internal.cuh"
#include "sm100_ptx.cuh"
#include "tiles.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;       // weight rows per unit (UMMA M)
constexpr int kBN = kTileTokens;  // tokens per tile (largest UMMA N used)
constexpr int kBK = 64;        // K per chunk: one 128-byte swizzle row of bf16
constexpr int kStages = 8;     // token rows + packed codes + scale/bias words, and a TMEM A tile
constexpr int kAhead = 3;      // chunks of copies in flight before the loader marks one full
constexpr int kDqWarps = 8;
constexpr int kLoadWarps = 8;
constexpr int kLoad0 = 1, kDq0 = kLoad0 + kLoadWarps, kEpi0 = kDq0 + kDqWarps;  // warp roles
constexpr int kThreads = (kEpi0 + 4) * 32;  // 672
constexpr int kAccCols = 128;               // TMEM columns per accumulator
constexpr int kACols = kBK / 2;             // TMEM columns per A stage (2 bf16 per column)
constexpr int kACol0 = 2 * kAccCols;        // first A column
constexpr int kTmemCols = 512;
constexpr int kTileBytes = kBN * kBK * 2;   // 16 KiB of token rows
constexpr int kCodesOff = kTileBytes;       // in a raw stage: 4 KiB of codes
constexpr int kCodesBytes = kBM * 32;
constexpr int kRawStride = kTileBytes + kCodesBytes;  // 20 KiB, 1 KiB aligned
constexpr int kSbWin = 32;                  // scale/bias words per row in a window
constexpr int kSbPitch = kSbWin + 1;        // row pitch in the window buffer (bank spread)
constexpr int kEpiStride = 36;              // floats per transposed column (bank spread)
constexpr uint64_t kWaitNs = 1000000000ull;
constexpr int kBarEpi = 1;                  // named barrier of the epilogue warps

static_assert(kDqWarps == 8, "two dequantising warps per TMEM lane quarter");
static_assert(kACol0 + kStages * kACols <= kTmemCols, "TMEM budget");
static_assert(kAhead < kStages, "the loader must mark a stage full before it needs that stage again");
static_assert(kBK == 64 && kACols == 32, "the MMA issue loop unrolls 4 K-steps of 16");

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
  int64_t yacc_n4;  // gate/up only: float4s of y_acc it clears for the down GEMM
  int test_stall;  // MOE_TEST_WAIT_TIMEOUT: the MMA issuer first waits on a phase nothing completes
  int b_tma;       // bmap is valid: tiles whose token rows are contiguous load B by TMA
};

struct Smem {
  uint8_t raw[kStages][kRawStride];  // token rows (swizzled), codes
  uint32_t sb[2][kBM * kSbPitch];    // scale/bias windows [row][word]
  float epi[4][16 * kEpiStride];     // per epilogue warp: 16 columns x 32 rows
  uint64_t raw_full[kStages], a_full[kStages], empty[kStages], sb_full[2], sb_empty[2];
  uint64_t acc_full[2], acc_empty[2], drain;
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

// Byte offset of 16-byte chunk `ch` (0..7) of row `row` in a swizzled tile
// (the tile 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128_off(int row, int ch) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((ch ^ (row & 7)) << 4));
}

// ---- dequantisation --------------------------------------------------------
// 32 codes (one uint4; code 8j+i at bits 4i of word j) with their group's
// scale s and bias b -> 32 bf16, two per 32-bit word (lower k in the low
// half).  In fp32, 1 + q/128 is built by byte permutation, and
// s q + b = (128 s)(1 + q/128) + (b - 128 s): one FMA per code, then round to
// nearest even bf16.
__device__ __forceinline__ void dequant32(uint4 w, uint32_t sb, uint32_t (&out)[16]) {
  const float s128 = 128.0f * bf16_lo(sb);
  const float off = bf16_hi(sb) - s128;
  const float2 s2 = make_float2(s128, s128), o2 = make_float2(off, off);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t lo = (ws[j] & 0x0F0F0F0Fu) | 0x80808080u;         // codes 0, 2, 4, 6
    const uint32_t hi = ((ws[j] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;  // codes 1, 3, 5, 7
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float f0 = __uint_as_float(__byte_perm(lo, 0x3F000000u, 0x7044u | (b << 8)));
      const float f1 = __uint_as_float(__byte_perm(hi, 0x3F000000u, 0x7044u | (b << 8)));
      const float2 v = __ffma2_rn(s2, make_float2(f0, f1), o2);
      const __nv_bfloat162 p = __floats2bfloat162_rn(v.x, v.y);
      out[4 * j + b] = *reinterpret_cast<const uint32_t*>(&p);
    }
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

// cmap / cmap_sh: the packed codes of the routed pool / the shared blob,
// 3-D uint32 {K/8, rows, blobs}, box 8 x 128 x 1.  bmap: the B rows (x for
// gate/up, h for down) as 2-D bf16 {K, rows}, box 64 x kBN, 128-byte swizzle:
// a tile whose token rows are consecutive (every down tile, the shared
// expert's gate/up tiles) takes its B tile as one copy per chunk.
template <bool DOWN>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap cmap,
                        const __grid_constant__ CUtensorMap cmap_sh,
                        const __grid_constant__ CUtensorMap bmap) {
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Launched as a programmatic dependent: the prologue below (barriers, TMEM,
  // the clear of y_acc that no earlier kernel of the call uses) may overlap
  // the previous kernel; everything it produced is read after griddep_wait.
  if (!DOWN) {
    float4* y4 = reinterpret_cast<float4*>(a.y_acc);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < a.yacc_n4;
         i += (int64_t)gridDim.x * blockDim.x)
      y4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&S.raw_full[s], kLoadWarps * 32 + 1);  // loader lanes + the expect-tx arrival
      ptx::mbar_init(&S.a_full[s], kDqWarps);
      ptx::mbar_init(&S.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&S.sb_full[b], kLoadWarps * 32);  // one copy arrival per loader lane
      ptx::mbar_init(&S.sb_empty[b], kDqWarps);
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
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const uint32_t tmem = S.tmem_base;
  const int n_units = *a.n_tiles * a.nm;
  // scale/bias windows: up to kSbWin group words per row, i.e. cpw chunks
  const int cpw = kSbWin * a.G / kBK;
  const int lg = 31 - __clz(a.G);  // log2 of the group size (32, 64 or 128)

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      Walk<DOWN> w;
      w.start(a, n_units);
      uint32_t g = 0, ub = 0;
      bool ok = true;
      // test hook: no arrival precedes the final commit, so this wait runs out
      if (a.test_stall) ok = wait_phase(&S.drain, 0, S, a.err);
      // B descriptors: stage s starts kRawStride bytes after stage s-1 (the start
      // address field counts 16-byte units); a K-step of 16 advances 32 bytes
      const uint64_t bdesc0 = sw128_desc(ptx::smem_u32(S.raw[0]));
      const uint32_t acol0 = tmem + kACol0;
      while (ok && w.live) {
        const int nmma = max(16, (w.t.ntok + 15) & ~15);
        const uint32_t idesc = idesc_bf16(kBM, nmma);
        const int buf = ub & 1;
        if (ub >= 2 && !wait_phase(&S.acc_empty[buf], ((ub >> 1) + 1) & 1, S, a.err)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * kAccCols;
        do {
          const uint32_t s = g % kStages;
          // the dequantisers arrive only after the stage's copies have landed
          if (!wait_phase(&S.a_full[s], (g / kStages) & 1, S, a.err)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t at = acol0 + s * kACols;
          const uint64_t bd = bdesc0 + (uint64_t)(s * (kRawStride >> 4));
          ptx::tc_mma_f16_ta(d, at, bd, idesc, w.c > 0 ? 1u : 0u);
          ptx::tc_mma_f16_ta(d, at + 8, bd + 2, idesc, 1u);
          ptx::tc_mma_f16_ta(d, at + 16, bd + 4, idesc, 1u);
          ptx::tc_mma_f16_ta(d, at + 24, bd + 6, idesc, 1u);
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
  } else if (warp < kDq0) {
    // ------------------------------------------------------------ loaders
    const int lw = warp - kLoad0;  // rows 4 (lw + 8 i) + lane / 8, i < 4
    const int lt = lw * 32 + lane;
    Walk<DOWN> w;
    w.start(a, n_units);
    const uint32_t* wsb = nullptr;  // scale/bias words of weight row m0
    const uint16_t* bbase = DOWN ? a.h : a.x;
    const int bpitch = DOWN ? a.hstride : a.H;
    int lsb = 0, crow = 0, cblob = 0;
    int rid[4] = {-1, -1, -1, -1};  // token-row ids of this lane's rows (-1: past the tile)
    const CUtensorMap* cm = &cmap;
    bool btma = false;  // this unit's B tile by TMA, from row brow0
    int brow0 = 0;
    uint32_t g = 0, done = 0, gw = 0;  // chunks issued, chunks marked full, windows issued
    uint32_t win_start[2] = {0, 0};    // first chunk of the last two windows
    bool ok = true;
    // mark the oldest chunk in flight full once this lane's copies of it have landed
    auto mark_oldest = [&]() {
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(&S.raw_full[done % kStages]);
      ++done;
    };
    const int ch = lane & 7;  // 16-byte piece of a token row
    while (ok && w.live) {
      {
        const Tile& t = w.t;
        const bool sh = t.slot < 0;
        const BlobLayout& B = sh ? a.LS : a.L;
        const uint8_t* blob = sh ? a.shared_blob : a.pool + (uint64_t)t.slot * a.L.stride;
        lsb = w.nk * kBK / a.G;
        wsb = reinterpret_cast<const uint32_t*>(blob + (DOWN ? B.d_sb : B.gu_sb)) +
              (size_t)w.m0 * lsb;
        cm = sh ? &cmap_sh : &cmap;
        cblob = sh ? 0 : t.slot;
        crow = w.m0;
        btma = a.b_tma && (DOWN || sh);
        brow0 = DOWN ? t.hrow0 : t.pos0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int n = 4 * (lw + kLoadWarps * i) + (lane >> 3);
          rid[i] = n >= t.ntok ? -1
                   : DOWN      ? t.hrow0 + n
                   : sh        ? t.pos0 + n
                               : a.perm[t.pos0 + n] / a.k;
        }
      }
      for (int c0 = 0; ok && c0 < w.nk; c0 += cpw) {
        // a new scale/bias window: words [c0*64/G, +kSbWin) of the unit's 128 rows
        const int wb = gw & 1;
        if (gw >= 2) {
          // the dequantisers free window gw-2 only after its last chunk is marked full
          if (done < win_start[(gw - 1) & 1]) {
            ptx::cp_async_wait_all();
            while (done < g) mark_oldest();
          }
          if (!wait_phase(&S.sb_empty[wb], ((gw >> 1) + 1) & 1, S, a.err)) {
            ok = false;
            break;
          }
        }
        win_start[wb] = g;
        const int w0 = c0 * kBK / a.G, nw = min(kSbWin, lsb - w0);
        for (int j = lt; j < kBM * nw; j += kLoadWarps * 32) {
          const int row = j / nw, col = j - row * nw;
          ptx::cp_async4(&S.sb[wb][row * kSbPitch + col], wsb + (size_t)row * lsb + w0 + col);
        }
        ptx::cp_async_mbar_arrive(&S.sb_full[wb]);
        ++gw;
        const int c1 = min(w.nk, c0 + cpw);
        for (int c = c0; c < c1; ++c) {
          const int s = g % kStages;
          if (g >= kStages && !wait_phase(&S.empty[s], ((g / kStages) + 1) & 1, S, a.err)) {
            ok = false;
            break;
          }
          uint8_t* st = S.raw[s];
          if (lt == 0) {
            // the whole box lands, rows past the tile included (zeros past
            // the matrix; other tiles' rows otherwise: their columns of D
            // are never read)
            ptx::mbar_arrive_expect_tx(&S.raw_full[s], kCodesBytes + (btma ? kTileBytes : 0));
            ptx::tma_load_3d(st + kCodesOff, cm, c * 8, crow, cblob, &S.raw_full[s]);
            if (btma) ptx::tma_load_2d(st, &bmap, c * kBK, brow0, &S.raw_full[s]);
          }
          if (!btma) {
            // token rows: piece ch of rows 4 (lw + 8 i) + lane / 8
            const uint16_t* bsrc = bbase + c * kBK + ch * 8;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (rid[i] >= 0)
                ptx::cp_async16(st + sw128_off(4 * (lw + kLoadWarps * i) + (lane >> 3), ch),
                                bsrc + (size_t)rid[i] * bpitch);
            }
          }
          ptx::cp_async_commit();
          ++g;
          if (g - done > kAhead) {
            ptx::cp_async_wait<kAhead>();
            mark_oldest();
          }
        }
      }
      w.next_unit(a);
    }
    ptx::cp_async_wait_all();
    while (done < g) mark_oldest();
  } else if (warp < kEpi0) {
    // ------------------------------------------------------------ dequantisers
    const int q = warp & 3;               // TMEM lane quarter = weight rows 32 q ..
    const int kh = (warp - kDq0) >> 2;    // K-half of the chunk
    const int r = q * 32 + lane;
    const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + kACol0 + kh * 16;
    Walk<DOWN> w;
    w.start(a, n_units);
    uint32_t g = 0, gw = 0;
    bool ok = true;
    while (ok && w.live) {
      for (int c0 = 0; c0 < w.nk; c0 += cpw) {  // scale/bias windows of the unit
        const int wb = gw & 1;
        if (!wait_phase(&S.sb_full[wb], (gw >> 1) & 1, S, a.err)) {
          ok = false;
          break;
        }
        ++gw;
        const uint32_t* sbrow = &S.sb[wb][r * kSbPitch];
        const int c1 = min(w.nk, c0 + cpw);
        for (int c = c0; c < c1; ++c) {
          const int sa = g % kStages;
          // the stage's copies have landed; the MMA that read its A tile last
          // time is done (the loader waited for that before copying)
          if (!wait_phase(&S.raw_full[sa], (g / kStages) & 1, S, a.err)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint8_t* st = S.raw[sa];
          const uint4 cq = *reinterpret_cast<const uint4*>(st + kCodesOff + r * 32 + kh * 16);
          const uint32_t sb = sbrow[((c * kBK + kh * 32) >> lg) & (kSbWin - 1)];
          uint32_t o[16];
          dequant32(cq, sb, o);
          ptx::tmem_st16(tq + sa * kACols, o);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&S.a_full[sa]);
          ++g;
        }
        if (!ok) break;
        // the window's last chunk is done: its scale/bias buffer may be refilled
        if (lane == 0) ptx::mbar_arrive(&S.sb_empty[wb]);
      }
      w.next_unit(a);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;                   // TMEM lane quarter
    const int et = threadIdx.x - kEpi0 * 32;  // 0 .. 127
    float* xp = S.epi[q];                     // [16 columns][kEpiStride]
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
      // one decision for all four warps (and the column table is complete)
      if (ptx::bar_any(kBarEpi, 128, !ok || aborted(S))) break;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + buf * kAccCols + ((uint32_t)(q * 32) << 16);
      const int c = lane >> 1, hf = lane & 1;  // after the transpose: column, half
      for (int n0 = 0; n0 < t.ntok; n0 += 16) {
        float v[16];
        ptx::tmem_ld16(taddr + n0, v);
        const int n = n0 + c;
        if (!DOWN) {
          // gate row 2i in an even lane, up row 2i+1 in the next lane: the
          // even lane takes columns 0-7 of the pair, the odd lane columns
          // 8-15, and both leave h for 16 features x 16 tokens, transposed
          uint16_t* hx = reinterpret_cast<uint16_t*>(xp);  // [16 columns][16 features]
          const bool odd = lane & 1;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // even lane sends its column 8+i (gate), odd lane its column i (up)
            const float other = __shfl_xor_sync(0xffffffffu, odd ? v[i] : v[8 + i], 1);
            const float gt = odd ? other : v[i];
            const float up = odd ? v[8 + i] : other;
            const int col = odd ? 8 + i : i;
            hx[col * 16 + (lane >> 1)] = f32_to_bf16_rne(silu_f(gt) * up);
          }
          __syncwarp();
          if (n < t.ntok) {
            const uint4 hv = *reinterpret_cast<const uint4*>(hx + c * 16 + hf * 8);
            *reinterpret_cast<uint4*>(a.h + (size_t)(t.hrow0 + n) * a.hstride + (w.m0 >> 1) +
                                      q * 16 + hf * 8) = hv;
          }
          __syncwarp();
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) xp[i * kEpiStride + lane] = v[i];
          __syncwarp();
          if (n < t.ntok) {
            const float wt = S.tok_w[n];
            float* dst = a.y_acc + (size_t)S.tok_t[n] * a.H + w.m0 + q * 32 + hf * 16;
            const float* src = xp + c * kEpiStride + hf * 16;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float4 u = *reinterpret_cast<const float4*>(src + 4 * i);
              atomicAdd(reinterpret_cast<float4*>(dst + 4 * i),
                        make_float4(wt * u.x, wt * u.y, wt * u.z, wt * u.w));
            }
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&S.acc_empty[buf]);
      // the column table is read by every warp before the next unit rewrites it
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
  build_tiles_block(used, n_used, offsets, table, n_slots, T, P, tiles, n_tiles, max_tiles, err,
                    warp_tot);
}

// y = bf16(y_acc), four elements per thread step
__global__ void finalize_kernel(const float* __restrict__ y_acc, uint16_t* __restrict__ y,
                                int64_t n4) {
  ptx::griddep_wait();  // a programmatic dependent of the down GEMM
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
  return d.bits == 4 && d.H % kBM == 0 && (2 * d.I) % kBM == 0 && (2 * d.Is) % kBM == 0 && d.I % kBK == 0 &&
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

// The tile list of the grouped GEMMs (after the permutation) and a zeroed
// fp32 accumulator for y.
cudaError_t launch_prefill_plan(const Ctx& c, const FwdArgs& fa, cudaStream_t st,
                                int* launches, bool tiles_built) {
  const Dims& d = c.d;
  const int T = fa.T, P = T * d.k;
  if (!tiles_built) {
    build_tiles_kernel<<<1, 1024, 0, st>>>(c.ws.used, c.ws.n_used, c.ws.offsets, fa.table,
                                           c.n_slots, T, P, reinterpret_cast<Tile*>(c.ws.tiles),
                                           c.ws.n_tiles, prefill_max_tiles(d, T), c.err);
    ++*launches;
  }
  // (y_acc is cleared by the gate/up GEMM's prologue)
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled through the runtime's driver entry point, so that
// the library does not link the driver library (it loads without a GPU).
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

namespace {

// Packed codes of `blobs` blobs: 3-D uint32 {K/8 words, rows, blobs}, box
// 8 x 128 x 1 (the 64 codes of one K-chunk for 128 weight rows), no swizzle.
bool encode_codes(CUtensorMap* m, const uint8_t* region, int K, int rows, int blobs,
                  uint64_t blob_stride) {
  const cuuint64_t dim[3] = {(cuuint64_t)K / 8, (cuuint64_t)rows, (cuuint64_t)blobs};
  const cuuint64_t stride[2] = {(cuuint64_t)K / 2, blob_stride};
  const cuuint32_t box[3] = {8, kBM, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3,
                                const_cast<uint8_t*>(region), dim, stride, box, es,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of a bf16 matrix (row pitch `pitch` elements) as B tiles: 2-D {cols,
// rows}, box 64 x kBN, the 128-byte swizzle of the MMA's B descriptor.
bool encode_rows(CUtensorMap* m, const uint16_t* base, int cols, int rows, int pitch) {
  if (((uintptr_t)base & 15) != 0 || rows <= 0 || (pitch * 2) % 16 != 0) return false;
  const cuuint64_t dim[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t stride[1] = {(cuuint64_t)pitch * 2};
  const cuuint32_t box[2] = {kBK, kBN};
  const cuuint32_t es[2] = {1, 1};
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), dim, stride,
             box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_prefill_experts(const Ctx& c, const FwdArgs& fa, cudaStream_t st,
                                   int* launches) {
  const Dims& d = c.d;
  const int T = fa.T;
  const int hstride = d.I > d.Is ? d.I : d.Is;
  // tensor maps of the packed codes (host-side encoding, a few microseconds)
  CUtensorMap gq, gq_sh, dq, dq_sh;
  if (!encode_codes(&gq, c.pool + c.ex.gu_q, d.H, 2 * d.I, c.n_slots, c.ex.stride) ||
      !encode_codes(&gq_sh, c.shared + c.sh.gu_q, d.H, 2 * d.Is, 1, c.sh.stride) ||
      !encode_codes(&dq, c.pool + c.ex.d_q, d.I, d.H, c.n_slots, c.ex.stride) ||
      !encode_codes(&dq_sh, c.shared + c.sh.d_q, d.Is, d.H, 1, c.sh.stride))
    return cudaErrorInvalidValue;
  GemmArgs a;
  a.x = fa.x;
  a.perm = c.ws.perm;
  a.topk_w = fa.topk_w;
  a.gate = c.ws.gate;
  a.pool = c.pool;
  a.L = c.ex;
  a.shared_blob = c.shared;
  a.LS = c.sh;
  a.tiles = reinterpret_cast<const Tile*>(c.ws.tiles);
  a.n_tiles = c.ws.n_tiles;
  a.h = reinterpret_cast<uint16_t*>(c.ws.h);
  a.y_acc = c.ws.o;
  a.err = c.err;
  a.k = d.k;
  a.H = d.H;
  a.I = d.I;
  a.Is = d.Is;
  a.G = d.G;
  a.hstride = hstride;
  a.nm = 2 * hstride / kBM;
  a.test_stall = (c.test_flags & MOE_TEST_WAIT_TIMEOUT) ? 1 : 0;
  a.yacc_n4 = (int64_t)T * d.H / 4;
  // programmatic dependent launches: each kernel's prologue overlaps the
  // previous kernel, and griddepcontrol.wait orders every dependent read
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.num_sms);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // B by TMA where a tile's rows are consecutive: x rows for the shared
  // expert's gate/up tiles, h rows for every down tile (else per-lane copies)
  CUtensorMap xmap{}, hmap{};
  const bool x_tma = encode_rows(&xmap, reinterpret_cast<const uint16_t*>(fa.x), d.H, T, d.H);
  const bool h_tma = encode_rows(&hmap, a.h, hstride, T * d.k + T, hstride);
  a.b_tma = x_tma ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<false>, a, gq, gq_sh, xmap);
  if (e != cudaSuccess) return e;
  record_mark(c, MOE_MARK_GATEUP, st);
  a.nm = d.H / kBM;
  a.yacc_n4 = 0;
  a.b_tma = h_tma ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<true>, a, dq, dq_sh, hmap);
  if (e != cudaSuccess) return e;
  record_mark(c, MOE_MARK_DOWN, st);
  const int64_t n4 = (int64_t)T * d.H / 4;
  cudaLaunchConfig_t fcfg = cfg;
  fcfg.gridDim = dim3(4 * c.num_sms);
  fcfg.blockDim = dim3(256);
  fcfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&fcfg, finalize_kernel, (const float*)c.ws.o, fa.y, n4);
  if (e != cudaSuccess) return e;
  *launches += 3;
  return cudaGetLastError();
}

}  // namespace moe
