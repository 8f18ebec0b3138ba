// decode.cu -- the MoE block for one token, one persistent launch per layer
// or per stack of layers.
//
// Decode streams ~17-22 MB of int4 expert weights per layer and token; the
// block's dependency chain (router -> top-k over all E logits -> the selected
// experts' gate/up -> down) has two points where every CTA needs what all the
// others computed, and a stack adds a third (the next layer's input).  One
// CTA per SM runs the layer:
//
//   input   layer 0: the caller's x; later layers of a stack: the previous
//           layer's residual, then RMSNorm (fp32, fixed order)
//   router  this CTA's router rows from shared memory (prefetched), split over
//           all warps, and the shared gate; publish the logits; then this
//           CTA's units of the shared expert's gate/up while the others finish
//   select  every CTA reads all E logits and selects the top-k itself
//           (a histogram filter, then an exact ranking of the few candidates;
//           near-ties fall back to the exact routine of routing_common.cuh)
//   experts TMA copies of this CTA's units of the selected experts' gate/up
//           rows and of its 16-row tile of their down projections, all in
//           flight at once; gate/up + SwiGLU as the tiles land; publish h
//   down    every CTA with a down tile reads all h, then its rows of y in a
//           fixed combine order (deterministic), bf16 out; a stack also
//           publishes the next residual x + y
//
// An exchange is one release-add per CTA on a counter that only grows (pass
// p of a launch sequence waits for p x CTAs arrivals) and one acquire poll
// per CTA by a single thread, so waiting costs the memory system one word per
// CTA and the expert weights stream at full bandwidth.
//
// The int4 GEMVs run on the tensor cores (mma.sync m16n8k16, bf16 operands,
// fp32 accumulation): 16 weight rows are the M dimension and the input the
// first columns of N.  A code pair (q_j, q_j+4) of a packed word becomes the
// bf16 pair (128 + q_j, 128 + q_j+4) with one mask-and-or; the k order inside
// an MMA is permuted to match (the input is stored in the same permuted
// order), and each group of G inputs is folded as
//   sum_c (s q_c + b) x_c = s sum_c (128 + q_c) x_c + (b - 128 s) sum_c x_c.
// The down projection's input h (fp32) is split into bf16 hi + lo parts that
// ride in two columns of N, so h enters with 16 significant bits.  Weights
// are MLX affine int4 groups (Swiftlet README, wpnews page, its list of what
// was built); the routed/shared split
// and the top-k routing follow the same README, section "How it works".
#include <algorithm>

#include "device_util.cuh"
#include "gemv_mma.cuh"
#include "moe_internal.cuh"
#include "routing_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

using namespace rt;
using namespace mmag;

constexpr int kThreads = 384;
constexpr int kWarps = 12;
constexpr int kBins = 256;      // histogram of the selection filter (one bin per thread)
constexpr int kCandCap = 64;    // candidates ranked exactly on the fast path
constexpr uint32_t kSpin = 1u << 24;         // poll rounds of an exchange
constexpr uint64_t kWaitNs = 1000000000ull;  // every wait gives up after one second
static_assert(kBins <= kThreads, "the histogram is cleared one bin per thread");
static_assert(kWarps <= 16, "per-warp scratch: four fields of 16 entries");
constexpr int kRedSs = 0, kRedMx = 16, kRedMn = 32, kRedSq = 48;  // fields of s_red
constexpr int kGuSplitMax = 4;  // k-splits of a gate/up tile (8 measured slower)
constexpr int kMaxTiles = 12;  // gate/up tiles (16 rows) of one CTA
// mbarriers: 0 prologue A; 1, 2 prologue B (double); then the gate/up tiles; last the down tile
constexpr int kMbarTile0 = 3;
constexpr int kMbarDown = kMbarTile0 + kMaxTiles;
constexpr int kNumMbar = kMbarDown + 1;

struct DecSmem {  // byte offsets into dynamic shared memory
  uint32_t mbar, misc, part, hist, cand, nb, xb, xp, xg, slog, tab, pgu, pdn;
  uint32_t pa, a_sq, a_rw, a_wsg, a_nw, a_ssb, a_pr;  // prologue A (one buffer)
  uint32_t pb, pb_bytes, b_sd, b_desc, b_sdsb;        // prologue B (two buffers)
  uint32_t gu, gu_sb;                                 // routed gate/up tiles, their scales
  uint32_t dn, dn_expert, dn_sb;                      // routed down tiles, per expert
  uint32_t total;
};

struct DecArgs {
  const DecLayer* layers;  // [L] device
  int L;
  int E, k, I, G;
  const uint16_t* x;     // layer-0 input [H]
  uint16_t* x_out;       // residual after the last layer [H], or null
  uint16_t* y;           // [L][H] per-layer block outputs, or null
  uint16_t* xn_out;      // [L][H] per-layer block inputs, or null
  int32_t* topk_idx;     // [L][k]
  float* topk_w;         // [L][k]
  int32_t* perm;         // layer 0 only, or null
  int32_t* offsets;      // layer 0 only, or null
  const int32_t* tables; // [L][E] slot tables, or null (identity)
  int chain;             // 1: RMSNorm + residual between layers
  float eps;
  DecWorkspace ws;
  int32_t* err;
  uint32_t hook;               // test hook: the logits wait expects one arrival too many
  unsigned long long* stamps;  // per-phase timestamps (MOE_DECODE_STAMPS builds), or null
  uint64_t inv_nc;             // ceil(2^32 / gridDim.x)
  uint64_t inv_i;              // ceil(2^32 / inter)
  DecSmem sm;
};

// x / d for x * d < 2^32 with m = ceil(2^32 / d) from the host: writing
// m d = 2^32 + e (0 <= e < d), x m / 2^32 = x / d + x e / (d 2^32), and the
// excess is below 1/d, so the floor is exact.
__device__ __forceinline__ int udiv(uint32_t x, uint64_t m) {
  return (int)(((uint64_t)x * m) >> 32);
}
// Start of share p of n items split into gridDim.x shares.
__device__ __forceinline__ int part(int n, int p, uint64_t inv_nc) {
  return udiv((uint32_t)n * (uint32_t)p, inv_nc);
}

// Waits sleep in hardware (100 us per try, at most ~1 s in all) so that the
// warps still computing keep the issue slots.
__device__ __forceinline__ void wait_mbar(uint64_t* bar, uint32_t parity, int32_t* err) {
  for (int i = 0; i < 10000; ++i)
    if (ptx::mbar_try_wait_sleep(bar, parity, 100000u)) return;
  record_error(err, MOE_ERR_TIMEOUT);
}

// This CTA's writes so far (every thread's, ordered by the barrier) become
// visible with one release-add by thread 0.
__device__ __forceinline__ void xarrive(unsigned long long* cnt) {
  __syncthreads();
  if (threadIdx.x == 0) ptx::red_release_add_u64(cnt, 1ull);
}

// Thread 0 polls until the counter reaches `target` (bounded: after kSpin
// polls or one second the device records MOE_ERR_TIMEOUT and the CTA carries
// on), then the CTA barrier orders every thread's later reads after it.
__device__ __forceinline__ void xwait(const unsigned long long* cnt, unsigned long long target,
                                      int32_t* err) {
  if (threadIdx.x == 0 && ptx::ld_acquire_u64(cnt) < target) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 0; ptx::ld_acquire_u64(cnt) < target; ++it) {
      if (it > kSpin || ptx::globaltimer_ns() - t0 > kWaitNs) {
        record_error(err, MOE_ERR_TIMEOUT);
        break;
      }
    }
  }
  __syncthreads();
}

// x . w over 8 bf16 pairs (one uint4 of each), 8 sequential FMAs.
__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    s = fmaf(bf16_lo(aw[q]), bf16_lo(bw[q]), s);
    s = fmaf(bf16_hi(aw[q]), bf16_hi(bw[q]), s);
  }
  return s;
}

// A 16-byte aligned window [lo, lo + len) around bytes [b0, b1).
__device__ __forceinline__ void align16(uint64_t b0, uint64_t b1, uint64_t& lo, uint32_t& len) {
  lo = b0 & ~uint64_t(15);
  len = (uint32_t)(((b1 + 15) & ~uint64_t(15)) - lo);
}

// One task of a 16-row tile: chunks [c0, c1) of K (32 inputs each; c0 and c1
// multiples of max(2, chunks per group)), folded per group of 2^LCPG chunks.
// Thread (g = lane / 4, t = lane % 4) ends with rows g and g + 8 of the tile
// in out0 / out1 when t == 0.
//   tile   shared address of the tile
//   bcol   this thread's column of N: the permuted input (16 bytes per
//          (chunk, t), chunks `bstride` bytes apart), or a zeroed 16-byte
//          slot with bstride 0
//   sb0/1  (scale | bias << 16) words of rows g and g + 8, one per group
//   xg     per-group sums of the input (all columns in use, added)
template <int LCPG>
__device__ __forceinline__ void tile_task(uint32_t tile, TileGeom geo, int c0, int c1,
                                          const uint8_t* bcol, uint32_t bstride,
                                          const uint32_t* sb0, const uint32_t* sb1,
                                          const float* xg, float& out0, float& out1) {
  constexpr int CPG = 1 << LCPG;
  constexpr int STEP = CPG < 2 ? 2 : CPG;  // chunks per iteration
  // ldmatrix and mma are .aligned: the whole warp must arrive together (callers
  // come here from per-lane waits and lane-0 copy issue)
  __syncwarp();
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3;
  const int r = (lane & 7) + 8 * (mi & 1), dc = mi >> 1;
  const uint32_t rbase = tile + (uint32_t)(r >> 3) * geo.half + (uint32_t)(r & 7) * geo.pitch;
  float o0 = 0.f, o1 = 0.f;
  // row sums (columns in use added) of group gi, folded with its scale and bias
  auto fold = [&](float a0, float a1, int gi) {
    const uint32_t s0 = sb0[gi], s1 = sb1[gi];
    const float X = xg[gi];
    const float sc0 = bf16_lo(s0), sc1 = bf16_lo(s1);
    o0 = fmaf(sc0, a0, fmaf(bf16_hi(s0) - 128.0f * sc0, X, o0));
    o1 = fmaf(sc1, a1, fmaf(bf16_hi(s1) - 128.0f * sc1, X, o1));
  };
  // Four independent accumulator chains per iteration (chunk of the ldmatrix
  // pair x half of the chunk): an mma.sync result is ready only after a long
  // latency, so one chain per warp would serialise every MMA of the task.
#pragma unroll 2
  for (int c = c0; c < c1; c += STEP) {
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
    for (int cp = 0; cp < STEP; cp += 2) {
      const int cc = c + cp + dc;
      const uint32_t addr =
          geo.swz ? rbase + (uint32_t)(cc >> 3) * geo.cb_stride + ((uint32_t)((cc & 7) ^ (r & 7)) << 4)
                  : rbase + ((uint32_t)cc << 4);
      uint32_t w[4];
      ldsm_x4(addr, w[0], w[1], w[2], w[3]);  // (row g, c), (row g+8, c), (g, c+1), (g+8, c+1)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int ch = c + cp + h;
        const uint4 b = *reinterpret_cast<const uint4*>(bcol + (size_t)ch * bstride);
        const uint32_t wg = w[2 * h], wg8 = w[2 * h + 1];
        const uint32_t wg4 = wg >> 4, wg84 = wg8 >> 4;
        mma16816(acc[2 * h], code_pair(wg, 0), code_pair(wg8, 0), code_pair(wg4, 0),
                 code_pair(wg84, 0), b.x, b.y);
        mma16816(acc[2 * h + 1], code_pair(wg >> 8, 0), code_pair(wg8 >> 8, 0),
                 code_pair(wg4 >> 8, 0), code_pair(wg84 >> 8, 0), b.z, b.w);
        if (CPG == 1) {
          const float(&p)[4] = acc[2 * h];
          const float(&q)[4] = acc[2 * h + 1];
          fold((p[0] + p[1]) + (q[0] + q[1]), (p[2] + p[3]) + (q[2] + q[3]), ch);
        }
      }
    }
    if (CPG > 1)
      fold(((acc[0][0] + acc[0][1]) + (acc[1][0] + acc[1][1])) +
               ((acc[2][0] + acc[2][1]) + (acc[3][0] + acc[3][1])),
           ((acc[0][2] + acc[0][3]) + (acc[1][2] + acc[1][3])) +
               ((acc[2][2] + acc[2][3]) + (acc[3][2] + acc[3][3])),
           c >> LCPG);
  }
  out0 = o0;
  out1 = o1;
}

// Logits read back from shared memory with one uniform bound, for the exact
// selection routine.
struct SmemLogits {
  const float* l;
  float b;
  __device__ __forceinline__ void get(int e, float& logit, float& bnd) const {
    logit = l[e];
    bnd = b;
  }
  __device__ __forceinline__ int id(int e) const { return e; }
};

// Router summation of the decode kernel: a row is cut into S = min(8, NJ)
// slices of NJ / S chunks; a lane sums each 8-element chunk with 8 sequential
// FMAs and its chunks in order, a warp butterfly (5 levels) sums the slice,
// a pairwise tree (log2 S levels) the slices, and the prior is added last.
// The depth D of that tree gives the rounding-error bound 2 D u sum |x w|
// (Higham, Accuracy and Stability of Numerical Algorithms, Thm. 4.3).
template <int NJ>
struct DecRouter {
  static constexpr int S = NJ < 8 ? NJ : 8;
  static constexpr int LOG2S = S >= 8 ? 3 : S >= 4 ? 2 : S >= 2 ? 1 : 0;
  static constexpr int DEPTH = 8 + NJ / S + 5 + LOG2S + 1;
  static constexpr float kScale = 2.0f * (float)DEPTH * 5.9604644775390625e-8f;
};

#ifdef MOE_DECODE_STAMPS
// Instrumented builds: thread 0's SM cycle counter at phase s of layer l
// (32 slots per layer and CTA).
#define STAMP(s)                                                                     \
  do {                                                                               \
    if (a.stamps && threadIdx.x == 0)                                                \
      a.stamps[((size_t)l * gridDim.x + blockIdx.x) * 32 + (s)] = clock64();         \
  } while (0)
#else
#define STAMP(s) \
  do {           \
  } while (0)
#endif

template <int NJ, int LCPG>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecArgs a) {
  constexpr int V1 = kMaxE / 256;  // logits per thread in the selection
  constexpr int H = NJ * 256;
  constexpr int HC = H / 32;           // 32-element chunks of x (K chunks of gate/up)
  constexpr int XW = H / 2;            // bf16 pairs of x
  constexpr int XP = (XW + kThreads - 1) / kThreads;
  constexpr int S = DecRouter<NJ>::S;
  constexpr int NCB = H / 256;         // 128-byte column blocks of a gate/up row
  // No alignment is declared on purpose: the 128-byte swizzled TMA tiles
  // need a 1024-byte aligned base, and with a declared alignment the
  // compiler may take the padding below to be zero.  Pointer arithmetic on
  // the shared array keeps every access LDS/STS; the plan reserves the slack.
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nC = gridDim.x, c = blockIdx.x;
  const int E = a.E, k = a.k, I = a.I, L = a.L;
  constexpr int lg = LCPG + 5;     // log2 G; G is 32, 64 or 128
  const int HG = H >> lg, IG = I >> lg, IC = I / 32;
  const int need = min(k + 1, E);  // entries whose order the fast path certifies
  const int g4 = lane >> 2, tg = lane & 3;

  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + a.sm.mbar);
  float* s_red = reinterpret_cast<float*>(sm + a.sm.misc);            // [64] per-warp fields
  int* s_idx = reinterpret_cast<int*>(sm + a.sm.misc + 256);          // [32]
  float* s_w = reinterpret_cast<float*>(sm + a.sm.misc + 384);        // [32]
  int* s_slot = reinterpret_cast<int*>(sm + a.sm.misc + 512);         // [32]
  int* s_sidx = reinterpret_cast<int*>(sm + a.sm.misc + 640);         // [33] ranked candidates
  float* s_sval = reinterpret_cast<float*>(sm + a.sm.misc + 776);     // [33]
  float* s_g = reinterpret_cast<float*>(sm + a.sm.misc + 912);        // shared gate
  const uint8_t* s_zero = sm + a.sm.misc + 928;                       // 16 zero bytes
  float* s_part = reinterpret_cast<float*>(sm + a.sm.part);           // router slice sums
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(sm + a.sm.hist);     // [kBins + 1]
  uint2* s_cand = reinterpret_cast<uint2*>(sm + a.sm.cand);           // [kCandCap]
  uint32_t* s_n = reinterpret_cast<uint32_t*>(sm + a.sm.nb);          // block input, bf16 pairs
  uint32_t* s_x = reinterpret_cast<uint32_t*>(sm + a.sm.xb);          // residual, bf16 pairs
  uint8_t* s_xp = sm + a.sm.xp;                                       // permuted block input
  float* s_xg = reinterpret_cast<float*>(sm + a.sm.xg);               // its group sums
  float* s_log = reinterpret_cast<float*>(sm + a.sm.slog);            // [E]
  int* s_tab = reinterpret_cast<int*>(sm + a.sm.tab);                 // [E] slot table
  float* s_pgu = reinterpret_cast<float*>(sm + a.sm.pgu);             // gate/up task results
  float* s_pdn = reinterpret_cast<float*>(sm + a.sm.pdn);             // down task results
  const uint32_t sm_base = ptx::smem_u32(sm);

  // fixed shares of this CTA
  const int re0 = part(E, c, a.inv_nc), re1 = part(E, c + 1, a.inv_nc);
  const int nr = re1 - re0;
  const int su0 = part(I / 4, c, a.inv_nc), su1 = part(I / 4, c + 1, a.inv_nc);  // shared units
  const int nsu = su1 - su0, nst = (nsu + 1) / 2;
  const int U0 = part(k * I / 4, c, a.inv_nc), U1 = part(k * I / 4, c + 1, a.inv_nc);
  const int nunit = U1 - U0, ntile = (nunit + 1) / 2;  // gate/up units of 4 pairs, tiles of 2
  const int dt0 = part(H / 16, c, a.inv_nc), dt1 = part(H / 16, c + 1, a.inv_nc);
  const bool has_down = dt1 > dt0;  // at most one 16-row tile of y per CTA (the plan checks)
  const int r0 = 16 * dt0;
  // gate/up tasks: k-splits of whole groups and of an even number of chunks
  // (ldmatrix takes two); a down task is one expert's whole row block
  // (measured: fewer, longer down tasks cost less per chunk)
  const int nsplit_gu = min(kGuSplitMax, HC / max(2, 1 << LCPG)), nsplit_d = 1;
  const bool dswz = I / 2 >= 128;
  const int ncbd = dswz ? I / 256 : 1;
  // gate/up tiles: two units of 8 rows, each one TMA box [column block][row][128 B]
  const TileGeom geo_gu{1024u, 128u, (uint32_t)NCB * 1024u, true};
  // down tiles: one box of 16 rows, [column block][row][128 B] (or whole rows)
  const uint32_t pitch_d = dswz ? 128u : (uint32_t)(I / 2);
  const TileGeom geo_d{16u * pitch_d, pitch_d, 8u * pitch_d, dswz};
  uint64_t pr_lo;
  uint32_t pr_len;  // window of this CTA's prior entries
  align16((uint64_t)re0 * 4, (uint64_t)re1 * 4, pr_lo, pr_len);

  // prologue A of layer ll: router rows, shared gate vector, norm weight, the
  // shared expert's gate/up units -- weights only
  auto issue_pro_a = [&](int ll) {
    const DecLayer& G = a.layers[ll];
    uint8_t* pa = sm + a.sm.pa;
    const uint32_t b_pr = (G.prior && nr > 0) ? pr_len : 0;
    const uint32_t b_rw = (uint32_t)nr * H * 2;
    const uint32_t b_nw = (a.chain && G.norm_w) ? H * 2 : 0;
    const uint32_t b_sq = (uint32_t)nsu * NCB * 1024;
    const uint32_t b_ssb = (uint32_t)nsu * 32 * HG;
    ptx::fence_proxy_async_smem();  // the buffer's earlier readers were generic-proxy loads
    ptx::mbar_arrive_expect_tx(&mbar[0], b_pr + b_rw + H * 2 + b_nw + b_sq + b_ssb);
    if (b_pr)
      ptx::bulk_g2s(pa + a.sm.a_pr, reinterpret_cast<const uint8_t*>(G.prior) + pr_lo, b_pr,
                    &mbar[0]);
    if (b_rw) ptx::bulk_g2s(pa + a.sm.a_rw, G.router_w + (size_t)re0 * H, b_rw, &mbar[0]);
    ptx::bulk_g2s(pa + a.sm.a_wsg, G.shared_gate_w, H * 2, &mbar[0]);
    if (b_nw) ptx::bulk_g2s(pa + a.sm.a_nw, G.norm_w, b_nw, &mbar[0]);
#pragma unroll 1
    for (int u = 0; u < nsu; ++u)  // unit u is half (u & 1) of tile u / 2
      ptx::tma_load_4d(pa + a.sm.a_sq + (size_t)u * NCB * 1024, &a.layers[ll].map_sgu, 0,
                       8 * (su0 + u), 0, 0, &mbar[0]);
    if (b_ssb)
      ptx::bulk_g2s(pa + a.sm.a_ssb, G.shared_blob + G.gu_sb + (size_t)su0 * 32 * HG, b_ssb,
                    &mbar[0]);
  };
  // prologue B of layer ll into buffer b: its descriptor and this CTA's tile
  // of the shared expert's down projection
  auto issue_pro_b = [&](int ll, int b) {
    const DecLayer& G = a.layers[ll];
    uint8_t* pb = sm + a.sm.pb + (uint32_t)b * a.sm.pb_bytes;
    const uint32_t b_desc = (uint32_t)sizeof(DecLayer);
    const uint32_t b_sd = has_down ? (uint32_t)ncbd * 16 * pitch_d : 0;
    const uint32_t b_sdsb = has_down ? 16u * IG * 4 : 0;
    ptx::fence_proxy_async_smem();
    ptx::mbar_arrive_expect_tx(&mbar[1 + b], b_desc + b_sd + b_sdsb);
    ptx::bulk_g2s(pb + a.sm.b_desc, a.layers + ll, b_desc, &mbar[1 + b]);
    if (has_down) {
      ptx::tma_load_4d(pb + a.sm.b_sd, &a.layers[ll].map_sd, 0, r0, 0, 0, &mbar[1 + b]);
      ptx::bulk_g2s(pb + a.sm.b_sdsb, G.shared_blob + G.d_sb + (size_t)r0 * IG * 4, b_sdsb,
                    &mbar[1 + b]);
    }
  };

#ifdef MOE_DECODE_STAMPS
  if (a.stamps && tid == 0) a.stamps[(size_t)c * 32 + 31] = clock64();  // kernel entry
#endif
  if (tid == 0) {
    for (int i = 0; i < kNumMbar; ++i) ptx::mbar_init(&mbar[i], 1);
    ptx::fence_mbar_init();
  }
  if (tid < 4) reinterpret_cast<uint32_t*>(sm + a.sm.misc + 928)[tid] = 0u;
  __syncthreads();
  ptx::griddep_launch_dependents();
  if (tid == 0) {
    issue_pro_a(0);
    issue_pro_b(0, 0);
  }
  // everything below may read what earlier kernels wrote
  ptx::griddep_wait();
  const uint32_t seq = __ldcg(a.ws.seq + c);

  for (int l = 0; l < L; ++l) {
    const uint32_t pass = seq * (uint32_t)L + (uint32_t)l + 1u;  // of the logits and h exchanges
    const unsigned long long target = (unsigned long long)pass * (unsigned long long)nC;
    const int b = l & 1;
    const uint32_t par = (uint32_t)l & 1u;
    const uint32_t pb_par = (uint32_t)(l >> 1) & 1u;
    uint8_t* pa = sm + a.sm.pa;
    uint8_t* pb = sm + a.sm.pb + (uint32_t)b * a.sm.pb_bytes;
    const DecLayer& D = *reinterpret_cast<const DecLayer*>(pb + a.sm.b_desc);
    const int32_t* table = a.tables ? a.tables + (size_t)l * E : nullptr;
    STAMP(0);

    // ------------------------------------------------------------ input
    if (l > 0) {  // the previous layer's residual (stacks)
      const unsigned long long xpass =
          (unsigned long long)seq * (unsigned long long)(L - 1) + (unsigned long long)l;
      xwait(a.ws.cnt + 2 * 16, xpass * (unsigned long long)nC, a.err);
    }
    uint32_t xin[XP];
    {
      const uint32_t* src = l == 0 ? reinterpret_cast<const uint32_t*>(a.x)
                                   : reinterpret_cast<const uint32_t*>(a.ws.xt);
#pragma unroll
      for (int p = 0; p < XP; ++p) {
        const int w = tid + kThreads * p;
        xin[p] = w < XW ? __ldcg(src + w) : 0u;
      }
    }
    if (table)
      for (int e = tid; e < E; e += kThreads) s_tab[e] = __ldcg(table + e);
    if (tid < kBins) s_hist[tid] = 0u;  // histogram and candidate count of this layer
    if (tid == 0) s_hist[kBins] = 0u;
    wait_mbar(&mbar[0], par, a.err);         // router rows, norm weight, shared gate/up
    wait_mbar(&mbar[1 + b], pb_par, a.err);  // descriptor, shared down tile
    if (a.chain) {
      // RMSNorm in fp32 with a fixed order: each thread's squares in order,
      // a xor butterfly in each warp, then the warp totals left to right
      float ss = 0.f;
#pragma unroll
      for (int p = 0; p < XP; ++p) {
        if (tid + kThreads * p < XW) {
          s_x[tid + kThreads * p] = xin[p];
          const float lo = bf16_lo(xin[p]), hi = bf16_hi(xin[p]);
          ss = fmaf(lo, lo, ss);
          ss = fmaf(hi, hi, ss);
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) s_red[kRedSs + warp] = ss;
      __syncthreads();
      float tot = s_red[kRedSs];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) tot = __fadd_rn(tot, s_red[kRedSs + w]);
      const float rinv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(tot, (float)H), a.eps)));
      const uint32_t* nw = reinterpret_cast<const uint32_t*>(pa + a.sm.a_nw);
#pragma unroll
      for (int p = 0; p < XP; ++p) {
        const int w = tid + kThreads * p;
        if (w < XW) {
          const uint32_t g = D.norm_w ? nw[w] : 0x3F803F80u;  // bf16 pair (1, 1)
          const float n0 = __fmul_rn(__fmul_rn(bf16_lo(xin[p]), rinv), bf16_lo(g));
          const float n1 = __fmul_rn(__fmul_rn(bf16_hi(xin[p]), rinv), bf16_hi(g));
          s_n[w] = (uint32_t)f32_to_bf16_rne(n0) | ((uint32_t)f32_to_bf16_rne(n1) << 16);
        }
      }
    } else {
#pragma unroll
      for (int p = 0; p < XP; ++p)
        if (tid + kThreads * p < XW) s_n[tid + kThreads * p] = xin[p];
    }
    __syncthreads();
    // the block input permuted for the MMAs: entry (chunk, t) holds inputs
    // 32 chunk + 8 t + (0, 4), (1, 5), (2, 6), (3, 7); the group sums; |x|_2^2
    {
      float ssq = 0.f;
      for (int e0 = 0; e0 < H / 8; e0 += kThreads) {
        const int e = e0 + tid;
        float s8 = 0.f;
        if (e < H / 8) {
          const uint4 v = reinterpret_cast<const uint4*>(s_n)[e];
          uint4 o;
          o.x = __byte_perm(v.x, v.z, 0x5410);
          o.y = __byte_perm(v.x, v.z, 0x7632);
          o.z = __byte_perm(v.y, v.w, 0x5410);
          o.w = __byte_perm(v.y, v.w, 0x7632);
          reinterpret_cast<uint4*>(s_xp)[e] = o;
          const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float lo = bf16_lo(ww[q]), hi = bf16_hi(ww[q]);
            s8 += lo + hi;
            ssq = fmaf(lo, lo, fmaf(hi, hi, ssq));
          }
        }
        // group sums: the G/8 entries of a group sit on consecutive lanes
        for (int o = 1; o < (a.G >> 3); o <<= 1) s8 += __shfl_xor_sync(0xffffffffu, s8, o);
        if (e < H / 8 && (e & ((a.G >> 3) - 1)) == 0) s_xg[e >> (lg - 3)] = s8;
      }
      ssq = warp_sum(ssq);
      if (lane == 0) s_red[kRedSq + warp] = ssq;
    }
    if (c == 0 && a.xn_out)  // the block input, for callers that check each layer
      for (int w = tid; w < XW; w += kThreads)
        reinterpret_cast<uint32_t*>(a.xn_out + (size_t)l * H)[w] = s_n[w];
    __syncthreads();
    STAMP(1);

    // ------------------------------------------------------------ router
    // tasks (row, slice): rows re0..re1 of the router and one more for the
    // shared gate vector, each cut into S slices
    {
      const uint4* n4 = reinterpret_cast<const uint4*>(s_n);
      for (int t = warp; t < (nr + 1) * S; t += kWarps) {
        const int row = t / S, sl = t - row * S;
        const uint4* w4 = reinterpret_cast<const uint4*>(
            row < nr ? pa + a.sm.a_rw + (size_t)row * H * 2 : pa + a.sm.a_wsg);
        float acc = 0.f;
#pragma unroll
        for (int jj = 0; jj < NJ / S; ++jj) {
          const int j = sl * (NJ / S) + jj;
          acc += dot8_bf16(w4[lane + 32 * j], n4[lane + 32 * j]);
        }
        acc = warp_sum(acc);
        if (lane == 0) s_part[t] = acc;
      }
    }
    STAMP(25);
    __syncthreads();
    if (tid <= nr) {
      // the slices pairwise, then the prior
      float v[S];
#pragma unroll
      for (int i = 0; i < S; ++i) v[i] = s_part[tid * S + i];
#pragma unroll
      for (int h = S / 2; h > 0; h >>= 1) {
#pragma unroll
        for (int i = 0; i < h; ++i) v[i] += v[i + h];
      }
      if (tid < nr) {
        const float pr =
            D.prior ? reinterpret_cast<const float*>(pa + a.sm.a_pr + (re0 * 4 - pr_lo))[tid]
                    : 0.f;
        __stcg(a.ws.lt + re0 + tid, v[0] + pr);
      } else {
        *s_g = 1.0f / (1.0f + __expf(-v[0]));
      }
    }
    xarrive(a.ws.cnt);
    STAMP(2);

    // this CTA's units of the shared expert's gate/up while the logits gather
    {
      const uint32_t* ssb = reinterpret_cast<const uint32_t*>(pa + a.sm.a_ssb);
      const int span = HC / nsplit_gu;
      for (int t = warp; t < nst * nsplit_gu; t += kWarps) {
        const int ti = t / nsplit_gu, sp = t - ti * nsplit_gu;
        const uint32_t tile = sm_base + a.sm.pa + a.sm.a_sq + (uint32_t)ti * NCB * 2048;
        const int row0 = 16 * ti + g4, row1 = row0 + 8;  // rows within this CTA's units
        const uint32_t* sb0 = ssb + (size_t)min(row0, 8 * nsu - 1) * HG;
        const uint32_t* sb1 = ssb + (size_t)min(row1, 8 * nsu - 1) * HG;
        float o0, o1;
        tile_task<LCPG>(tile, geo_gu, sp * span, (sp + 1) * span,
                        g4 == 0 ? s_xp + tg * 16 : s_zero, g4 == 0 ? 64u : 0u, sb0, sb1, s_xg, o0,
                        o1);
        if (tg == 0) {
          s_pgu[t * 16 + g4] = o0;
          s_pgu[t * 16 + g4 + 8] = o1;
        }
      }
      __syncthreads();
      for (int p = tid; p < 4 * nsu; p += kThreads) {  // pairs of this CTA's shared units
        const int ti = p >> 3, m = 2 * (p & 7);
        float gsum = 0.f, usum = 0.f;
        for (int sp = 0; sp < nsplit_gu; ++sp) {
          gsum += s_pgu[(ti * nsplit_gu + sp) * 16 + m];
          usum += s_pgu[(ti * nsplit_gu + sp) * 16 + m + 1];
        }
        __stcg(a.ws.ht + (size_t)k * I + 4 * su0 + p, silu_f(gsum) * usum);
      }
    }
    xwait(a.ws.cnt, target + a.hook, a.err);
    // every warp is past its reads of prologue A: the next layer's copies
    if (tid == 0 && l + 1 < L) issue_pro_a(l + 1);
    STAMP(8);

    // ------------------------------------------------------------ select
    uint32_t key[V1];
    float lv[V1];
    uint32_t kmx = 0u, kmn = 0xFFFFFFFFu;
#pragma unroll
    for (int q = 0; q < V1; ++q) {
      const int e = tid + kThreads * q;
      float f = e < E ? __ldcg(a.ws.lt + e) : 0.f;
      if (f != f) f = -INFINITY;  // a NaN logit from bad input ranks as -inf
      lv[q] = f;
      key[q] = e < E ? f32_key(f) : 0u;
      if (e < E) {
        s_log[e] = f;
        kmx = max(kmx, key[q]);
        kmn = min(kmn, key[q]);
      }
    }
    kmx = __reduce_max_sync(0xffffffffu, kmx);
    kmn = __reduce_min_sync(0xffffffffu, kmn);
    if (lane == 0) {
      reinterpret_cast<uint32_t*>(s_red)[kRedMx + warp] = kmx;
      reinterpret_cast<uint32_t*>(s_red)[kRedMn + warp] = kmn;
    }
    __syncthreads();
    STAMP(7);
    {
      uint32_t gx = 0u, gn = 0xFFFFFFFFu;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        gx = max(gx, reinterpret_cast<uint32_t*>(s_red)[kRedMx + w]);
        gn = min(gn, reinterpret_cast<uint32_t*>(s_red)[kRedMn + w]);
      }
      const float M = key_f32(gx), mn = key_f32(gn);
      // bins of equal width over [min, max], bin 0 at the top: a monotone map,
      // so the top `need` logits lie in the first bins holding `need` entries
      const float scale = (M > mn) ? (float)(kBins - 1) / (M - mn) : 0.f;
      int bin[V1];
#pragma unroll
      for (int q = 0; q < V1; ++q) {
        bin[q] = (int)fminf((float)(kBins - 1), (M - lv[q]) * scale);
        if (tid + kThreads * q < E) atomicAdd(&s_hist[bin[q]], 1u);
      }
      __syncthreads();
      // smallest bin b* whose cumulative count reaches `need` (every warp)
      uint32_t cnt[8], run = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cnt[i] = s_hist[8 * lane + i];
        run += cnt[i];
      }
      uint32_t incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      STAMP(13);
      const uint32_t hit = __ballot_sync(0xffffffffu, incl >= (uint32_t)need);
      int bstar = kBins - 1;
      if (hit) {
        const int hl = __ffs(hit) - 1;  // the lane holding b*
        uint32_t acc = incl - run;      // exclusive prefix of this lane
        int bl = -1;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc += cnt[i];
          if (bl < 0 && acc >= (uint32_t)need) bl = i;
        }
        bstar = __shfl_sync(0xffffffffu, 8 * lane + bl, hl);
      }
#pragma unroll
      for (int q = 0; q < V1; ++q) {
        const int e = tid + kThreads * q;
        if (e < E && bin[q] <= bstar) {
          const uint32_t pos = atomicAdd(&s_hist[kBins], 1u);
          if (pos < (uint32_t)kCandCap) s_cand[pos] = make_uint2(key[q], (uint32_t)e);
        }
      }
    }
    __syncthreads();
    STAMP(14);
    int* s_ok = reinterpret_cast<int*>(sm + a.sm.misc + 944);      // fast path certified
    float* s_beta = reinterpret_cast<float*>(sm + a.sm.misc + 948);  // the uniform bound
    if (warp == 0) {
      const int nc = (int)s_hist[kBins];
      // uniform bound on every logit's rounding error: 2 D u (|x|_2 max_e |Wr_e|_2
      // + max |prior|) (Cauchy-Schwarz on sum |x w|), with 1% to spare
      float xx = lane < kWarps ? s_red[kRedSq + lane] : 0.f;
      xx = warp_sum(xx);
      const float X = sqrtf(xx) * 1.0009765625f;
      const float beta = DecRouter<NJ>::kScale * 1.01f * (X * D.wmax + D.pmax) + kBoundFloor;
      bool ok = nc >= need && nc <= kCandCap;
      if (ok) {
        for (int i = lane; i < nc; i += 32) {
          const uint2 me = s_cand[i];
          const uint64_t km = ((uint64_t)me.x << 32) | (uint32_t)~me.y;
          int rank = 0;
          for (int j = 0; j < nc; ++j) {
            const uint2 o = s_cand[j];
            rank += (((uint64_t)o.x << 32) | (uint32_t)~o.y) > km;
          }
          if (rank < need) {
            s_sidx[rank] = (int)me.y;
            s_sval[rank] = key_f32(me.x);
          }
        }
        __syncwarp();
        STAMP(21);
        // certified when consecutive computed values are more than 2 beta
        // apart over the first `need` positions
        const bool gap = lane + 1 >= need || (s_sval[lane] - s_sval[lane + 1] > 2.0f * beta);
        ok = __all_sync(0xffffffffu, gap);
      }
      if (lane == 0) {
        *s_ok = ok ? 1 : 0;
        *s_beta = beta;
      }
      STAMP(22);
    }
    __syncthreads();
    if (!*s_ok) {
      // near-ties or an overfull candidate set: the exact selection by the
      // whole CTA (rare)
      int* si;
      float* sv;
      const size_t sel = (rt::topk_warp_smem(E) + 15) & ~size_t(15);
      // the block input is read from this CTA's shared copy (generic loads)
      topk_select_block<V1>(SmemLogits{s_log, *s_beta}, E, k, reinterpret_cast<const uint16_t*>(s_n),
                            D.router_w, D.prior, H, sm + a.sm.gu,
                            reinterpret_cast<uint2*>(sm + a.sm.gu + sel),
                            reinterpret_cast<float*>(sm + a.sm.gu + sel + kThreads * V1 * 8), &si,
                            &sv);
      if (warp == 0) {
        if (lane < k) {
          s_sidx[lane] = si[lane];
          s_sval[lane] = sv[lane];
        }
        __syncwarp();
      }
    }
    // the slots first: the copies wait for them; the weights come later, off
    // the critical path
    if (warp == 0) {
      if (lane < k) {
        const int e = s_sidx[lane];
        const int slot = table ? s_tab[e] : e;
        const bool good = slot >= 0 && slot < D.n_slots;
        s_idx[lane] = e;
        s_slot[lane] = good ? slot : -1;
        if (c == 0 && !good) record_error(a.err, MOE_ERR_SLOT);
      }
      STAMP(23);
    }
    __syncthreads();
    STAMP(3);

    // ------------------------------------------------------------ experts
    // This CTA's gate/up units [U0, U1) (4 row pairs = 8 rows each; units never
    // straddle experts) in tiles of two units, tile t on its own mbarrier;
    // lane 0 of warp w issues tiles w, w + 8, ... with each unit's scales in a
    // bulk copy.  Warp 7's lanes 1..k copy this CTA's down tile of every
    // selected expert.
    {
      const DecLayer* Dg = a.layers + l;  // the tensor maps are read from global memory
      if (lane == 0) {
#pragma unroll 1
        for (int t = warp; t < ntile; t += kWarps) {
          uint32_t bytes = 0;
#pragma unroll 1
          for (int u = 2 * t; u < min(2 * t + 2, nunit); ++u) {
            const int j = udiv((uint32_t)(4 * (U0 + u)), a.inv_i);
            if (s_slot[j] >= 0) bytes += NCB * 1024 + 32 * HG;
          }
          ptx::fence_proxy_async_smem();
          ptx::mbar_arrive_expect_tx(&mbar[kMbarTile0 + t], bytes);
#pragma unroll 1
          for (int u = 2 * t; u < min(2 * t + 2, nunit); ++u) {
            const int pg = 4 * (U0 + u);  // first pair of the unit (flattened over experts)
            const int j = udiv((uint32_t)pg, a.inv_i), i = pg - j * I;
            if (s_slot[j] < 0) continue;
            ptx::tma_load_4d(sm + a.sm.gu + (size_t)u * NCB * 1024, &Dg->map_gu, 0, 2 * i, 0,
                             s_slot[j], &mbar[kMbarTile0 + t]);
            ptx::bulk_g2s(sm + a.sm.gu_sb + (size_t)u * 32 * HG,
                          D.pool + (uint64_t)s_slot[j] * D.stride + D.gu_sb + (size_t)i * 8 * HG,
                          32u * HG, &mbar[kMbarTile0 + t]);
          }
        }
      }
      if (warp == kWarps - 1) {
        if (lane == 1) {
          uint32_t bytes = 0;
          if (has_down)
            for (int j = 0; j < k; ++j)
              if (s_slot[j] >= 0) bytes += (uint32_t)ncbd * 16 * pitch_d + 16u * IG * 4;
          ptx::mbar_arrive_expect_tx(&mbar[kMbarDown], bytes);
        }
        __syncwarp();
        ptx::fence_proxy_async_smem();
        if (has_down) {
          for (int j = lane - 1; j >= 0 && j < k; j += 31) {
            if (s_slot[j] < 0) continue;
            uint8_t* dst = sm + a.sm.dn + (size_t)j * a.sm.dn_expert;
            ptx::tma_load_4d(dst, &Dg->map_d, 0, r0, 0, s_slot[j], &mbar[kMbarDown]);
            ptx::bulk_g2s(dst + a.sm.dn_sb,
                          D.pool + (uint64_t)s_slot[j] * D.stride + D.d_sb + (size_t)r0 * IG * 4,
                          16u * IG * 4, &mbar[kMbarDown]);
          }
        }
      }
    }
    // renormalised weights (read by the combine, after the h exchange)
    if (warp == 0) {
      const float w = renormalised_weight(s_sval, k);
      if (lane < k) {
        s_w[lane] = w;
        if (c == 0) {
          a.topk_idx[(size_t)l * k + lane] = s_idx[lane];
          a.topk_w[(size_t)l * k + lane] = w;
        }
      }
    }
    // permutation outputs of a single token (pair p = j), first layer only
    if (l == 0 && a.offsets) {
      for (int e = part(E + 1, c, a.inv_nc) + tid; e < part(E + 1, c + 1, a.inv_nc); e += kThreads) {
        int cnt = 0;
        for (int j = 0; j < k; ++j) cnt += s_idx[j] < e;
        a.offsets[e] = cnt;
      }
    }
    if (l == 0 && a.perm && c == 0 && tid < k) {
      int rank = 0;
      for (int j = 0; j < k; ++j) rank += s_idx[j] < s_idx[tid];
      a.perm[rank] = tid;
    }

    // gate/up: tasks (tile, k-split), tile-major so compute follows the copies
    {
      const uint32_t* gsb = reinterpret_cast<const uint32_t*>(sm + a.sm.gu_sb);
      const int span = HC / nsplit_gu;
      for (int t = warp; t < ntile * nsplit_gu; t += kWarps) {
        const int ti = t / nsplit_gu, sp = t - ti * nsplit_gu;
        wait_mbar(&mbar[kMbarTile0 + ti], par, a.err);
        const uint32_t tile = sm_base + a.sm.gu + (uint32_t)ti * NCB * 2048;
        const int row0 = 16 * ti + g4, row1 = row0 + 8;  // rows within this CTA's units
        const uint32_t* sb0 = gsb + (size_t)min(row0, 8 * nunit - 1) * HG;
        const uint32_t* sb1 = gsb + (size_t)min(row1, 8 * nunit - 1) * HG;
        float o0, o1;
        tile_task<LCPG>(tile, geo_gu, sp * span, (sp + 1) * span,
                        g4 == 0 ? s_xp + tg * 16 : s_zero, g4 == 0 ? 64u : 0u, sb0, sb1, s_xg, o0,
                        o1);
        if (tg == 0) {
          s_pgu[t * 16 + g4] = o0;
          s_pgu[t * 16 + g4 + 8] = o1;
        }
        if (t == 0) STAMP(24);
      }
      STAMP(9);
      __syncthreads();
      for (int p = tid; p < 4 * nunit; p += kThreads) {  // this CTA's pairs
        const int ti = p >> 3, m = 2 * (p & 7);
        const int pg = 4 * U0 + p, j = udiv((uint32_t)pg, a.inv_i);
        float gsum = 0.f, usum = 0.f;
        for (int sp = 0; sp < nsplit_gu; ++sp) {
          gsum += s_pgu[(ti * nsplit_gu + sp) * 16 + m];
          usum += s_pgu[(ti * nsplit_gu + sp) * 16 + m + 1];
        }
        __stcg(a.ws.ht + pg, s_slot[j] >= 0 ? silu_f(gsum) * usum : 0.f);
      }
    }
    STAMP(4);
    xarrive(a.ws.cnt + 16);
    xwait(a.ws.cnt + 16, target, a.err);
    STAMP(12);

    // ------------------------------------------------------------ down
    if (has_down) {
      // all h, permuted like x (entry (expert, chunk, t), 16 bytes) as bf16 hi
      // and lo parts, and every group's sum of hi + lo
      const int NE = (k + 1) * I / 8;
      uint8_t* hp_hi = sm + a.sm.gu;
      uint8_t* hp_lo = hp_hi + (size_t)NE * 16;
      float* hg = reinterpret_cast<float*>(hp_lo + (size_t)NE * 16);
      const float4* h4 = reinterpret_cast<const float4*>(a.ws.ht);
      constexpr int HB = 4;  // entries per thread whose loads are issued together
      for (int e0 = 0; e0 < NE; e0 += HB * kThreads) {
        float4 hu[HB], hv[HB];
#pragma unroll
        for (int q = 0; q < HB; ++q) {
          const int e = e0 + q * kThreads + tid;
          if (e < NE) {
            hu[q] = __ldcg(h4 + 2 * e);
            hv[q] = __ldcg(h4 + 2 * e + 1);
          }
        }
#pragma unroll
        for (int q = 0; q < HB; ++q) {
          const int e = e0 + q * kThreads + tid;
          float s8 = 0.f;
          if (e < NE) {
            const float f[8] = {hu[q].x, hu[q].y, hu[q].z, hu[q].w,
                                hv[q].x, hv[q].y, hv[q].z, hv[q].w};
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              hi[i] = f32_to_bf16_rne(f[i]);
              lo[i] = f32_to_bf16_rne(f[i] - __uint_as_float(hi[i] << 16));
              s8 += __uint_as_float(hi[i] << 16) + __uint_as_float(lo[i] << 16);
            }
            reinterpret_cast<uint4*>(hp_hi)[e] =
                make_uint4(hi[0] | (hi[4] << 16), hi[1] | (hi[5] << 16), hi[2] | (hi[6] << 16),
                           hi[3] | (hi[7] << 16));
            reinterpret_cast<uint4*>(hp_lo)[e] =
                make_uint4(lo[0] | (lo[4] << 16), lo[1] | (lo[5] << 16), lo[2] | (lo[6] << 16),
                           lo[3] | (lo[7] << 16));
          }
          // group sums: the G/8 entries of a group sit on consecutive lanes
          for (int o = 1; o < (a.G >> 3); o <<= 1) s8 += __shfl_xor_sync(0xffffffffu, s8, o);
          if (e < NE && (e & ((a.G >> 3) - 1)) == 0) hg[e >> (lg - 3)] = s8;
        }
      }
      __syncthreads();
      STAMP(5);
      wait_mbar(&mbar[kMbarDown], par, a.err);
      STAMP(10);
      // tasks (expert, k-split); expert k is the shared one (prologue B)
      const int span = IC / nsplit_d;
      for (int t = warp; t < (k + 1) * nsplit_d; t += kWarps) {
        const int j = t / nsplit_d, sp = t - j * nsplit_d;
        const bool shared = j == k;
        if (!shared && s_slot[j] < 0) continue;
        const uint32_t tile = sm_base + (shared ? a.sm.pb + (uint32_t)b * a.sm.pb_bytes + a.sm.b_sd
                                                : a.sm.dn + (uint32_t)j * a.sm.dn_expert);
        const uint32_t* sbt = reinterpret_cast<const uint32_t*>(
            shared ? pb + a.sm.b_sdsb : sm + a.sm.dn + (size_t)j * a.sm.dn_expert + a.sm.dn_sb);
        const size_t boff = (size_t)j * IC * 64 + tg * 16;  // expert j's permuted entries
        const uint8_t* bs = g4 == 0 ? hp_hi + boff : g4 == 1 ? hp_lo + boff : s_zero;
        float o0, o1;
        tile_task<LCPG>(tile, geo_d, sp * span, (sp + 1) * span, bs, g4 < 2 ? 64u : 0u,
                        sbt + (size_t)g4 * IG, sbt + (size_t)(g4 + 8) * IG, hg + (size_t)j * IG,
                        o0, o1);
        if (tg == 0) {
          s_pdn[t * 16 + g4] = o0;
          s_pdn[t * 16 + g4 + 8] = o1;
        }
        if (t == 0) STAMP(20);
      }
      STAMP(16);
      __syncthreads();
      STAMP(11);
      // y rows, the first 256 threads: thread (m = tid / 16, jl = tid % 16)
      // takes row m's experts jl, jl + 16, ... (the shared one is j = k), then a
      // fixed butterfly over the 16 lanes of the row (deterministic)
      if (tid < 256) {
        const int m = tid >> 4, jl = tid & 15;
        float part = 0.f;
        for (int j = jl; j <= k; j += 16) {
          if (j < k && s_slot[j] < 0) continue;
          float v = 0.f;
          for (int sp = 0; sp < nsplit_d; ++sp) v += s_pdn[(j * nsplit_d + sp) * 16 + m];
          part = fmaf(j < k ? s_w[j] : *s_g, v, part);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        const float y1 = __shfl_sync(0xffffffffu, part, 16);  // row 2 warp + 1
        if (lane == 0) {
          const uint32_t ybits =
              (uint32_t)f32_to_bf16_rne(part) | ((uint32_t)f32_to_bf16_rne(y1) << 16);
          const int wpos = r0 / 2 + warp;
          if (a.y) reinterpret_cast<uint32_t*>(a.y + (size_t)l * H)[wpos] = ybits;
          if (a.chain) {
            const uint32_t xb = s_x[wpos];
            const float n0 = __fadd_rn(bf16_lo(xb), bf16_lo(ybits));
            const float n1 = __fadd_rn(bf16_hi(xb), bf16_hi(ybits));
            const uint32_t nb =
                (uint32_t)f32_to_bf16_rne(n0) | ((uint32_t)f32_to_bf16_rne(n1) << 16);
            if (l + 1 < L)
              __stcg(reinterpret_cast<uint32_t*>(a.ws.xt) + wpos, nb);
            else if (a.x_out)
              reinterpret_cast<uint32_t*>(a.x_out)[wpos] = nb;
          }
        }
        STAMP(17);
      }
    } else {
      wait_mbar(&mbar[kMbarDown], par, a.err);  // its phase completes with no bytes
    }
    if (a.chain && l + 1 < L) xarrive(a.ws.cnt + 2 * 16);
    STAMP(18);
    // the next layer's prologue B into the other buffer (last read two layers ago)
    __syncthreads();
    STAMP(19);
    if (tid == 0 && l + 1 < L) issue_pro_b(l + 1, b ^ 1);
    STAMP(6);
  }
  if (tid == 0) a.ws.seq[c] = seq + 1u;
}

#undef STAMP

}  // namespace

// ---------------------------------------------------------------- host side
namespace {

uint64_t up_to(uint64_t v, uint64_t al) { return (v + al - 1) / al * al; }

// Host-side shared-memory plan; false if the shapes do not fit.
bool plan_smem(const Dims& d, int nC, bool chain, DecSmem& s) {
  const int H = d.H, I = d.I, G = d.G, E = d.E, k = d.k;
  const int NCB = H / 256, HG = H / G, IG = I / G;
  const bool dswz = I / 2 >= 128;
  const uint32_t pitch_d = dswz ? 128u : (uint32_t)(I / 2);
  const int ncbd = dswz ? I / 256 : 1;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes, uint64_t al) {
    off = up_to(off, al);
    const uint64_t o = off;
    off += bytes;
    return (uint32_t)o;
  };
  auto share = [&](int n, int cc) { return (int)(((long long)n * cc) / nC); };
  int rw_max = 0, su_max = 0, un_max = 0;
  for (int cc = 0; cc < nC; ++cc) {
    rw_max = std::max(rw_max, share(E, cc + 1) - share(E, cc));
    su_max = std::max(su_max, share(I / 4, cc + 1) - share(I / 4, cc));
    un_max = std::max(un_max, share(k * I / 4, cc + 1) - share(k * I / 4, cc));
    if (share(H / 16, cc + 1) - share(H / 16, cc) > 1) return false;  // one down tile per CTA
  }
  const int tiles_max = (un_max + 1) / 2, stiles_max = (su_max + 1) / 2;
  if (tiles_max > kMaxTiles || rw_max + 1 > kThreads) return false;
  const int S = std::min(8, H / 256);
  const int cpg2 = std::max(2, G / 32);
  const int nsg = std::min(kGuSplitMax, (H / 32) / cpg2), nsd = 1;
  if (nsg < 1 || (I / 32) % cpg2 != 0) return false;
  s.mbar = take(kNumMbar * 8, 16);
  s.misc = take(1024, 16);
  s.part = take((uint64_t)(rw_max + 1) * S * 4, 16);
  s.hist = take((kBins + 1) * 4, 16);
  s.cand = take(kCandCap * 8, 16);
  s.nb = take((uint64_t)H * 2, 16);
  s.xb = take((uint64_t)H * 2, 16);
  s.xp = take((uint64_t)H * 2, 16);
  s.xg = take((uint64_t)HG * 4, 16);
  s.slog = take((uint64_t)E * 4, 16);
  s.tab = take((uint64_t)E * 4, 16);
  s.pgu = take((uint64_t)std::max(tiles_max, stiles_max) * nsg * 16 * 4, 16);
  s.pdn = take((uint64_t)(k + 1) * nsd * 16 * 4, 16);
  // prologue A: the shared gate/up tiles first (1024-aligned for the swizzle)
  s.pa = take(0, 1024);
  uint64_t p = 0;
  auto ptake = [&](uint64_t bytes, uint64_t al) {
    p = up_to(p, al);
    const uint64_t o = p;
    p += bytes;
    return (uint32_t)o;
  };
  s.a_sq = ptake((uint64_t)stiles_max * NCB * 2048, 1024);
  s.a_rw = ptake((uint64_t)rw_max * H * 2, 128);
  s.a_wsg = ptake((uint64_t)H * 2, 128);
  s.a_nw = ptake(chain ? (uint64_t)H * 2 : 0, 128);
  s.a_ssb = ptake((uint64_t)su_max * 32 * HG, 128);
  s.a_pr = ptake(up_to((uint64_t)rw_max * 4, 16) + 16, 128);
  off += p;
  // prologue B, two buffers: the shared down tile first, then the descriptor
  uint64_t q = 0;
  s.b_sd = 0;
  q = (uint64_t)ncbd * 16 * pitch_d;
  q = up_to(q, 128);
  s.b_desc = (uint32_t)q;
  q += sizeof(DecLayer);
  q = up_to(q, 128);
  s.b_sdsb = (uint32_t)q;
  q += (uint64_t)16 * IG * 4;
  s.pb_bytes = (uint32_t)up_to(q, 1024);
  s.pb = take(2ull * s.pb_bytes, 1024);
  // routed gate/up tiles; later the h staging (hi, lo, group sums) and the
  // exact fallback's scratch
  const uint64_t gu_bytes = (uint64_t)tiles_max * NCB * 2048;
  const uint64_t h_bytes = (uint64_t)(k + 1) * I / 8 * 32 + (uint64_t)(k + 1) * IG * 4;
  const uint64_t sel_bytes = up_to(rt::topk_warp_smem(E), 16) + (uint64_t)kThreads * (kMaxE / 256) * 8 + 64;
  s.gu = take(std::max(gu_bytes, std::max(h_bytes, sel_bytes)), 1024);
  s.gu_sb = take((uint64_t)un_max * 32 * HG, 128);
  s.dn_sb = (uint32_t)up_to((uint64_t)ncbd * 16 * pitch_d, 128);
  s.dn_expert = (uint32_t)up_to(s.dn_sb + (uint64_t)16 * IG * 4, 1024);
  s.dn = take((uint64_t)s.dn_expert * k, 1024);
  s.total = (uint32_t)off + 1024;  // slack to align the base to 1024 bytes
  return s.total <= 227 * 1024;
}

template <int NJ, int LC>
cudaError_t launch_t(const DecArgs& a, int nC, cudaStream_t st, bool coop) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nC);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = a.sm.total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (coop) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, decode_kernel<NJ, LC>, a);
}

template <int NJ, int LC>
cudaError_t prepare_t(int smem, int* occ) {
  // the attribute is the kernel's, shared by every context and stack: set
  // the device limit, so that a smaller plan never lowers it below a larger one
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<NJ, LC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, decode_kernel<NJ, LC>, kThreads, smem);
}

template <int NJ, int LC>
struct PrepareF {
  static cudaError_t run(int smem, int* occ) { return prepare_t<NJ, LC>(smem, occ); }
};
template <int NJ, int LC>
struct LaunchF {
  static cudaError_t run(const DecArgs* a, int nC, cudaStream_t st, bool coop) {
    return launch_t<NJ, LC>(*a, nC, st, coop);
  }
};

// Dispatch over (H / 256) x (log2 of 32-input chunks per group).
template <template <int, int> class F, typename... Args>
cudaError_t dispatch(const Dims& d, Args... args) {
  const int lc = d.G == 32 ? 0 : d.G == 64 ? 1 : 2;
#define MOE_DEC_CASE(NJ)                                                               \
  case NJ:                                                                             \
    return lc == 0 ? F<NJ, 0>::run(args...) : lc == 1 ? F<NJ, 1>::run(args...)         \
                                                      : F<NJ, 2>::run(args...);
  switch (d.H / 256) {
    MOE_DEC_CASE(1)
    MOE_DEC_CASE(2)
    MOE_DEC_CASE(4)
    MOE_DEC_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_DEC_CASE
}

// max_e |Wr_e|_2 and max_e |prior_e|, both rounded up: the constants of the
// decode kernel's uniform bound on the router's rounding error.  One block;
// run once when the weights are loaded.
__global__ void router_bound_consts_kernel(const uint16_t* __restrict__ rw,
                                           const float* __restrict__ prior, int E, int H,
                                           float* out) {
  __shared__ uint32_t s_w, s_p;
  if (threadIdx.x == 0) {
    s_w = 0u;
    s_p = 0u;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  for (int e = warp; e < E; e += nw) {
    float ss = 0.f;
    for (int h = lane; h < H; h += 32) {
      const float w = bf16_val(rw[(size_t)e * H + h]);
      ss = fmaf(w, w, ss);
    }
    ss = warp_sum(ss);
    // the fp32 sum of H squares is within H u of the exact one; 2^-10 covers it
    if (lane == 0) atomicMax(&s_w, __float_as_uint(sqrtf(ss * 1.0009765625f) * 1.0009765625f));
  }
  if (prior)
    for (int e = threadIdx.x; e < E; e += blockDim.x)
      atomicMax(&s_p, __float_as_uint(fabsf(prior[e])));
  __syncthreads();
  if (threadIdx.x == 0) {
    out[0] = __uint_as_float(s_w);
    out[1] = __uint_as_float(s_p);
  }
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// A 4-D TMA map over packed-code rows of `row_bytes` bytes, ordered so that
// one box lands as [column block][row][128 B]: dims {bytes within a 128-byte
// column block, row, column block, slot} with strides {row_bytes, 128,
// slot_stride}; box {128, box_rows, all column blocks, 1}, the 128-byte
// swizzle.  Rows shorter than 128 bytes are one unswizzled column block.
bool encode_rows(CUtensorMap* m, const uint8_t* base, int row_bytes, int rows, int slots,
                 uint64_t slot_stride, int box_rows, int box_cbs = 0) {
  const EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const bool swz = row_bytes >= 128;
  const cuuint64_t inner = swz ? 128u : (cuuint64_t)row_bytes;
  const cuuint64_t ncb = (cuuint64_t)row_bytes / inner;
  // a single slot still needs a valid stride (a multiple of 16 bytes)
  const cuuint64_t sstride =
      slots > 1 ? (cuuint64_t)slot_stride : ((cuuint64_t)rows * row_bytes + 15) / 16 * 16;
  const cuuint64_t dim[4] = {inner, (cuuint64_t)rows, ncb, (cuuint64_t)slots};
  const cuuint64_t stride[3] = {(cuuint64_t)row_bytes, inner, sstride};
  // box_cbs > 0: that many column blocks per box (a part of each row)
  const cuuint32_t box[4] = {(cuuint32_t)inner, (cuuint32_t)box_rows,
                             (cuuint32_t)(box_cbs > 0 ? box_cbs : ncb), 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(base), dim, stride, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool decode_shape_ok(const Dims& d) {
  const int nj = d.H / 256;
  return d.bits == 4 && (nj == 1 || nj == 2 || nj == 4 || nj == 8) && d.I == d.Is &&
         d.E <= kMaxE &&
         d.I % 32 == 0 && d.k <= 32;
}

bool decode_fits(const Dims& d, int nC, bool chain) {
  DecSmem s;
  return decode_shape_ok(d) && plan_smem(d, nC, chain, s);
}

cudaError_t decode_router_consts(const uint16_t* router_w, const float* prior, int E, int H,
                                 float* out, cudaStream_t st) {
  router_bound_consts_kernel<<<1, 1024, 0, st>>>(router_w, prior, E, H, out);
  return cudaGetLastError();
}

bool decode_encode_maps(const Dims& d, const uint8_t* pool, const BlobLayout& ex, int n_slots,
                        const uint8_t* shared, const BlobLayout& sh, DecLayer* D) {
  return encode_rows(&D->map_gu, pool + ex.gu_q, d.H / 2, 2 * d.I, n_slots, ex.stride, 8) &&
         encode_rows(&D->map_d, pool + ex.d_q, d.I / 2, d.H, n_slots, ex.stride, 16) &&
         encode_rows(&D->map_sgu, shared + sh.gu_q, d.H / 2, 2 * d.Is, 1, sh.stride, 8) &&
         encode_rows(&D->map_sd, shared + sh.d_q, d.Is / 2, d.H, 1, sh.stride, 16) &&
         // half rows (batched decode): 8-row boxes of half the column blocks
         encode_rows(&D->map_guh, pool + ex.gu_q, d.H / 2, 2 * d.I, n_slots, ex.stride, 8,
                     std::max(1, d.H / 512)) &&
         encode_rows(&D->map_sguh, shared + sh.gu_q, d.H / 2, 2 * d.Is, 1, sh.stride, 8,
                     std::max(1, d.H / 512));
}

cudaError_t decode_prepare(const Dims& d, int nC, bool chain, int* ok) {
  *ok = 0;
  DecSmem s;
  if (!decode_shape_ok(d) || !plan_smem(d, nC, chain, s) || !encode_tiled()) return cudaSuccess;
  int occ = 0;
  cudaError_t e = dispatch<PrepareF>(d, (int)s.total, &occ);
  if (e != cudaSuccess) return e;
  *ok = occ >= 1;
  return cudaSuccess;
}

size_t decode_workspace_bytes(const Dims& d, int nC) {
  return up256((size_t)nC * 4) + up256(3 * 16 * 8) + up256((size_t)d.E * 4) +
         up256((size_t)(d.k + 1) * d.I * 4) + up256((size_t)d.H * 2);
}

void decode_workspace_carve(const Dims& d, int nC, uint8_t* base, DecWorkspace* w) {
  size_t off = 0;
  w->seq = reinterpret_cast<uint32_t*>(base + off);
  off += up256((size_t)nC * 4);
  w->cnt = reinterpret_cast<unsigned long long*>(base + off);
  off += up256(3 * 16 * 8);
  w->lt = reinterpret_cast<float*>(base + off);
  off += up256((size_t)d.E * 4);
  w->ht = reinterpret_cast<float*>(base + off);
  off += up256((size_t)(d.k + 1) * d.I * 4);
  w->xt = reinterpret_cast<uint16_t*>(base + off);
}

void decode_workspace_reset(int nC, const DecWorkspace& w) {
  cudaMemset(w.seq, 0, (size_t)nC * 4);
  cudaMemset(w.cnt, 0, 3 * 16 * 8);
}

cudaError_t decode_launch(const Dims& d, int nC, const DecLaunch& p, cudaStream_t st) {
  DecArgs a{};
  a.layers = p.layers;
  a.L = p.L;
  a.E = d.E;
  a.k = d.k;
  a.I = d.I;
  a.G = d.G;
  a.x = p.x;
  a.x_out = p.x_out;
  a.y = p.y;
  a.xn_out = p.xn_out;
  a.topk_idx = p.topk_idx;
  a.topk_w = p.topk_w;
  a.perm = p.perm;
  a.offsets = p.offsets;
  a.tables = p.tables;
  a.chain = p.chain;
  a.eps = p.eps;
  a.ws = p.ws;
  a.err = p.err;
  a.hook = p.timeout_hook ? 1u : 0u;
  a.stamps = p.stamps;
  a.inv_nc = ((1ull << 32) + (uint64_t)nC - 1) / (uint64_t)nC;
  a.inv_i = ((1ull << 32) + (uint64_t)d.I - 1) / (uint64_t)d.I;
  if (!plan_smem(d, nC, p.chain != 0, a.sm)) return cudaErrorInvalidConfiguration;
  return dispatch<LaunchF>(d, (const DecArgs*)&a, nC, st, p.cooperative);
}

}  // namespace moe
