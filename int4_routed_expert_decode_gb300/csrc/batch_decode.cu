// batch_decode.cu -- the experts of the MoE block for 2..64 tokens (batched
// decode).  After the router, top-k and permutation launches, each used
// expert's int4 weights stream from HBM once and serve all of its tokens,
// which ride in the N columns of mma.sync (8 tokens per tile):
//   bdec_prep_kernel    x in the MMA's k order (bf16) and its group sums
//   bdec_gateup_kernel  persistent; a unit is 16 interleaved gate/up rows (8
//                       pairs) of one used expert, or of the shared expert, for
//                       all of its tokens; SwiGLU; h as bf16 in the same k order
//                       plus the sum of each 8 values
//   bdec_hsum_kernel    the group sums of h (fixed order)
//   bdec_down_kernel    one CTA per 16 rows of y: those rows of every used
//                       expert's down projection against its tokens' h, then per
//                       token the routing-weighted combine plus the gated shared
//                       expert, in a fixed order (deterministic)
// The weights and the routing are the pages' block (Swiftlet README on the
// wpnews page, "How it works"; MLX affine int4 groups per its list of what was
// built); the h rounding to bf16 is the grouped GEMMs' (one bf16 operand).
#include "device_util.cuh"
#include "gemv_mma.cuh"
#include "moe_internal.cuh"
#include "routing_common.cuh"
#include "sm100_ptx.cuh"

namespace moe {

namespace {

using namespace mmag;

constexpr int kBThreads = 256;
constexpr int kBWarps = 8;
constexpr int kBMaxT = 64;
// dynamic shared memory limit of these kernels (the down kernel also has a
// little static shared memory; the sum must stay within the device's 227 KB)
constexpr int kBSmemMax = 224 * 1024;

struct BArgs {
  const DecLayer* L;  // maps and pointers of the layer (device)
  int T, k, E, I, G, P;
  const int32_t* used;     // [E] used experts, ascending
  const int32_t* n_used;   // [1]
  const int32_t* offsets;  // [E+1]
  const int32_t* perm;     // [P] pair ids sorted by expert
  const int32_t* inv;      // [P] position of pair p in perm
  const int32_t* table;    // [E] slots, or null (identity)
  const uint16_t* x;       // [T][H]
  uint16_t* xperm;         // [T][H] bf16, k-permuted
  float* xg;               // [T][H/G]
  uint16_t* hperm;         // [P + T][I] bf16, k-permuted (rows: perm positions, then shared)
  float* hs8;              // [P + T][I/8]
  float* hg;               // [P + T][I/G]
  const float* topk_w;     // [T][k]
  const float* gate;       // [T] shared-expert gate
  uint16_t* y;             // [T][H]
  int32_t* err;
  uint32_t gu_slot, gu_sb, part;       // gate/up: part slot bytes, scale buffer bytes, barriers
  uint32_t dn_slot, dn_sb, ocache;     // down: slot bytes, scales within a slot, outputs
  uint32_t smem_gu, smem_dn;
};

__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t parity, int32_t* err) {
  for (int i = 0; i < 10000; ++i)
    if (ptx::mbar_try_wait_sleep(bar, parity, 100000u)) return;
  record_error(err, MOE_ERR_TIMEOUT);
}

// A routed expert's slot, or -1 when its slot is missing or out of range.
__device__ __forceinline__ int slot_of(const BArgs& a, int e, int n_slots) {
  const int s = a.table ? a.table[e] : e;
  return (s >= 0 && s < n_slots) ? s : -1;
}

// x in the MMA's k order: entry (chunk, t) of 8 bf16 holds inputs
// 32 chunk + 8 t + (0, 4), (1, 5), (2, 6), (3, 7); and the group sums.
__global__ void __launch_bounds__(256) bdec_prep_kernel(const uint16_t* __restrict__ x, int H,
                                                       int G, uint16_t* __restrict__ xperm,
                                                       float* __restrict__ xg) {
  const int t = blockIdx.x;
  const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
  uint4* dst = reinterpret_cast<uint4*>(xperm + (size_t)t * H);
  for (int e0 = 0; e0 < H / 8; e0 += blockDim.x) {
    const int e = e0 + threadIdx.x;
    float s8 = 0.f;
    if (e < H / 8) {
      const uint4 v = src[e];
      uint4 o;
      o.x = __byte_perm(v.x, v.z, 0x5410);
      o.y = __byte_perm(v.x, v.z, 0x7632);
      o.z = __byte_perm(v.y, v.w, 0x5410);
      o.w = __byte_perm(v.y, v.w, 0x7632);
      dst[e] = o;
      const uint32_t ww[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) s8 += bf16_lo(ww[q]) + bf16_hi(ww[q]);
    }
    // a group's G/8 entries sit on consecutive lanes
    for (int o = 1; o < (G >> 3); o <<= 1) s8 += __shfl_xor_sync(0xffffffffu, s8, o);
    if (e < H / 8 && (e & ((G >> 3) - 1)) == 0) xg[(size_t)t * (H / G) + e / (G >> 3)] = s8;
  }
}

// hg[row][g] = the sum of h over group g of the row, from the sums of 8.
__global__ void __launch_bounds__(256) bdec_hsum_kernel(const float* __restrict__ hs8, int rows,
                                                       int I, int G, float* __restrict__ hg) {
  const int IG = I / G, per = G / 8;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * IG) return;
  const int row = i / IG, g = i - row * IG;
  float s = 0.f;
  for (int u = 0; u < per; ++u) s += hs8[(size_t)row * (I / 8) + g * per + u];
  hg[i] = s;
}

// Chunks [c0, c1) of a 16-row tile (local chunk indices; the tile's first
// chunk is chunk cg of the row) against NT tiles of 8 input columns at once:
// the weights' fragments are loaded and converted once per chunk pair and
// serve every column tile.  Lane (g = lane / 4, t = lane % 4) loads column g
// of each tile (input row tb[nt], or zeros when negative) and accumulates
// rows g, g + 8 x columns 2t, 2t + 1 into o[nt][0..3] (row g col 2t, row g
// col 2t + 1, row g + 8 col 2t, row g + 8 col 2t + 1), folding each group as
//   sum_c (s q_c + b) x_c = s sum_c (128 + q_c) x_c + (b - 128 s) sum_c x_c.
//   src, row_elems  the input rows (bf16, k-permuted) and their stride
//   ta, tc          input rows of columns 2t, 2t + 1 (negative: unused)
//   sb0/1           (scale | bias << 16) words of rows g and g + 8, per group
//   xg, ng          per-row group sums of the input rows, ng per row
template <int LCPG, int NT>
__device__ __forceinline__ void tile_mn(uint32_t tile, TileGeom geo, int c0, int c1, int cg,
                                        const uint16_t* src, int row_elems, const int (&tb)[NT],
                                        const int (&ta)[NT], const int (&tc)[NT],
                                        const uint32_t* sb0, const uint32_t* sb1,
                                        const float* xg, int ng, float (&o)[NT][4]) {
  constexpr int CPG = 1 << LCPG;
  constexpr int STEP = CPG < 2 ? 2 : CPG;
  const int lane = threadIdx.x & 31;
  const int mi = lane >> 3;
  const int r = (lane & 7) + 8 * (mi & 1), dc = mi >> 1;
  const int tg = lane & 3;
  const uint32_t rbase = tile + (uint32_t)(r >> 3) * geo.half + (uint32_t)(r & 7) * geo.pitch;
  auto fold = [&](const float (&acc)[NT][4], int gi) {
    const uint32_t s0 = sb0[gi], s1 = sb1[gi];
    const float sc0 = bf16_lo(s0), sc1 = bf16_lo(s1);
    const float bb0 = bf16_hi(s0) - 128.0f * sc0, bb1 = bf16_hi(s1) - 128.0f * sc1;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float XA = ta[nt] >= 0 ? xg[(size_t)ta[nt] * ng + gi] : 0.f;
      const float XB = tc[nt] >= 0 ? xg[(size_t)tc[nt] * ng + gi] : 0.f;
      o[nt][0] = fmaf(sc0, acc[nt][0], fmaf(bb0, XA, o[nt][0]));
      o[nt][1] = fmaf(sc0, acc[nt][1], fmaf(bb0, XB, o[nt][1]));
      o[nt][2] = fmaf(sc1, acc[nt][2], fmaf(bb1, XA, o[nt][2]));
      o[nt][3] = fmaf(sc1, acc[nt][3], fmaf(bb1, XB, o[nt][3]));
    }
  };
  for (int c = c0; c < c1; c += STEP) {
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int cp = 0; cp < STEP; cp += 2) {
      const int cc = c + cp + dc;
      const uint32_t addr =
          geo.swz ? rbase + (uint32_t)(cc >> 3) * geo.cb_stride + ((uint32_t)((cc & 7) ^ (r & 7)) << 4)
                  : rbase + ((uint32_t)cc << 4);
      uint32_t w[4];
      ldsm_x4(addr, w[0], w[1], w[2], w[3]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int chg = cg + c + cp + h;  // chunk of the row
        const uint32_t wg = w[2 * h], wg8 = w[2 * h + 1];
        const uint32_t wg4 = wg >> 4, wg84 = wg8 >> 4;
        const uint32_t a0 = code_pair(wg, 0), a1 = code_pair(wg8, 0), a2 = code_pair(wg4, 0),
                       a3 = code_pair(wg84, 0);
        const uint32_t a4 = code_pair(wg >> 8, 0), a5 = code_pair(wg8 >> 8, 0),
                       a6 = code_pair(wg4 >> 8, 0), a7 = code_pair(wg84 >> 8, 0);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          uint4 b = make_uint4(0u, 0u, 0u, 0u);
          if (tb[nt] >= 0)
            b = __ldg(reinterpret_cast<const uint4*>(src + (size_t)tb[nt] * row_elems) +
                      (size_t)chg * 4 + tg);
          mma16816(acc[nt], a0, a1, a2, a3, b.x, b.y);
          mma16816(acc[nt], a4, a5, a6, a7, b.z, b.w);
        }
        if (CPG == 1) {
          fold(acc, chg);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        }
      }
    }
    if (CPG > 1) fold(acc, (cg + c) >> LCPG);
  }
}

// The unit list: u / (I / 8) indexes the used experts (the last one is the
// shared expert), u % (I / 8) is a tile of 8 gate/up pairs (16 rows).
struct UnitInfo {
  int tile, pos0, n_e, hrow0, slot;  // slot: -1 missing, -2 the shared expert
};

__device__ __forceinline__ UnitInfo unit_info(const BArgs& a, int u, int n_used, int n_slots) {
  const int tpe = a.I / 8;
  const int ue = u / tpe;
  UnitInfo U;
  U.tile = u - ue * tpe;
  if (ue < n_used) {
    const int e = a.used[ue];
    U.pos0 = a.offsets[e];
    U.n_e = min(a.offsets[e + 1] - U.pos0, kBMaxT);
    U.hrow0 = U.pos0;
    U.slot = slot_of(a, e, n_slots);
  } else {
    U.pos0 = 0;
    U.n_e = a.T;
    U.hrow0 = a.P;
    U.slot = -2;
  }
  return U;
}

// Gate/up + SwiGLU.  This CTA's units u = blockIdx.x + i * gridDim.x go to
// its warps round robin (i = w, w + 8, ...); each warp streams its units in
// NH parts (halves of the rows when a row holds 2 column blocks or more)
// through two slots of its own, with every token tile of the unit's expert
// at once, and writes h itself: no CTA-wide barrier.
template <int NJ, int LCPG, int NT>
__device__ __forceinline__ void gu_unit_part(const BArgs& a, const UnitInfo& U, int part,
                                             uint32_t tile, const uint32_t* sb, float (&o)[8][4]) {
  constexpr int H = NJ * 256, NCB = H / 256, HC = H / 32;
  constexpr int NH = NCB >= 2 ? 2 : 1, PHC = HC / NH;
  const int HG = H >> (LCPG + 5);
  const int lane = threadIdx.x & 31, g4 = lane >> 2, tg = lane & 3;
  const TileGeom geo{1024u, 128u, (uint32_t)(NCB / NH) * 1024u, true};
  const bool shared = U.slot == -2;
  auto token = [&](int idx) {
    return idx < U.n_e ? (shared ? idx : a.perm[U.pos0 + idx] / a.k) : -1;
  };
  int tb[NT], ta[NT], tc[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    tb[nt] = U.slot == -1 ? -1 : token(nt * 8 + g4);
    ta[nt] = token(nt * 8 + 2 * tg);
    tc[nt] = token(nt * 8 + 2 * tg + 1);
  }
  tile_mn<LCPG, NT>(tile, geo, 0, PHC, part * PHC, a.xperm, H, tb, ta, tc, sb + g4 * HG,
                    sb + (g4 + 8) * HG, a.xg, HG, reinterpret_cast<float(&)[NT][4]>(o));
}

template <int NT>
__device__ __forceinline__ void gu_epilogue(const BArgs& a, const UnitInfo& U, float (&o)[8][4]) {
  const int I = a.I;
  const int lane = threadIdx.x & 31, g4 = lane >> 2, tg = lane & 3;
  const bool ok = U.slot != -1;
  const int i0 = 8 * U.tile;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // even g: gate rows 2m, 2m + 8 (pairs m, m + 4); lane + 4 holds their up rows
    float up[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) up[i] = __shfl_down_sync(0xffffffffu, o[nt][i], 4);
    float h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = ok ? silu_f(o[nt][i]) * up[i] : 0.f;
    const uint32_t b0 = f32_to_bf16_rne(h[0]), b1 = f32_to_bf16_rne(h[1]);
    const uint32_t b2 = f32_to_bf16_rne(h[2]), b3 = f32_to_bf16_rne(h[3]);
    // the sum of the 8 values of each column: pairs (m, m + 4) over m = 0..3
    float sa = __uint_as_float(b0 << 16) + __uint_as_float(b2 << 16);
    float sc = __uint_as_float(b1 << 16) + __uint_as_float(b3 << 16);
    sa += __shfl_xor_sync(0xffffffffu, sa, 8);
    sa += __shfl_xor_sync(0xffffffffu, sa, 16);
    sc += __shfl_xor_sync(0xffffffffu, sc, 8);
    sc += __shfl_xor_sync(0xffffffffu, sc, 16);
    if ((g4 & 1) == 0) {
      const int m = g4 >> 1;
      const int ia = nt * 8 + 2 * tg, ic = ia + 1;
      // word m of a column's 16-byte entry is the bf16 pair (h_m, h_m+4)
      if (ia < U.n_e) {
        const size_t row = (size_t)U.hrow0 + ia;
        reinterpret_cast<uint32_t*>(a.hperm + row * I + (i0 >> 5) * 32 + ((i0 & 31) >> 3) * 8)[m] =
            b0 | (b2 << 16);
        if (m == 0) a.hs8[row * (I / 8) + U.tile] = sa;
      }
      if (ic < U.n_e) {
        const size_t row = (size_t)U.hrow0 + ic;
        reinterpret_cast<uint32_t*>(a.hperm + row * I + (i0 >> 5) * 32 + ((i0 & 31) >> 3) * 8)[m] =
            b1 | (b3 << 16);
        if (m == 0) a.hs8[row * (I / 8) + U.tile] = sc;
      }
    }
  }
}

template <int NJ, int LCPG>
__global__ void __launch_bounds__(kBThreads, 1) bdec_gateup_kernel(const BArgs a) {
  constexpr int H = NJ * 256, NCB = H / 256;
  constexpr int NH = NCB >= 2 ? 2 : 1, PCB = NCB / NH;
  const int HG = H >> (LCPG + 5);
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t pslot = (uint32_t)PCB * 2048;  // one part: 16 rows x PCB column blocks
  uint8_t* slots = sm + (size_t)warp * 2 * pslot;
  uint8_t* sbuf = sm + (size_t)kBWarps * 2 * pslot + (size_t)warp * 2 * a.gu_sb;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + a.part) + warp * 2;
  const DecLayer* L = a.L;
  const int n_slots = L->n_slots;
  const int n_used = *a.n_used;
  const int U_all = (n_used + 1) * (a.I / 8);
  const int nu = (int)blockIdx.x < U_all ?
                 (U_all - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  const int nw = nu > warp ? (nu - warp + kBWarps - 1) / kBWarps : 0;  // this warp's units
  const int nitems = nw * NH;
  if (lane == 0) {
    ptx::mbar_init(&mbar[0], 1);
    ptx::mbar_init(&mbar[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  auto unit_of = [&](int q) {  // this warp's q-th item's unit index
    return (int)blockIdx.x + (warp + kBWarps * (q / NH)) * (int)gridDim.x;
  };
  auto issue = [&](int q) {  // lane 0
    const UnitInfo U = unit_info(a, unit_of(q), n_used, n_slots);
    const int part = q % NH, s = q & 1;
    uint8_t* dst = slots + (size_t)s * pslot;
    uint8_t* sdst = sbuf + (size_t)((q / NH) & 1) * a.gu_sb;
    ptx::fence_proxy_async_smem();  // the slot's previous part was read by ldmatrix
    if (U.slot == -1) {
      record_error(a.err, MOE_ERR_SLOT);
      ptx::mbar_arrive_expect_tx(&mbar[s], 0);
      return;
    }
    const bool shared = U.slot == -2;
    const CUtensorMap* map = NH == 1 ? (shared ? &L->map_sgu : &L->map_gu)
                                     : (shared ? &L->map_sguh : &L->map_guh);
    const int sl = shared ? 0 : U.slot;
    const uint32_t sbytes = part == 0 ? 16u * HG * 4 : 0u;
    ptx::mbar_arrive_expect_tx(&mbar[s], pslot + sbytes);
    ptx::tma_load_4d(dst, map, 0, 16 * U.tile, part * PCB, sl, &mbar[s]);
    ptx::tma_load_4d(dst + PCB * 1024, map, 0, 16 * U.tile + 8, part * PCB, sl, &mbar[s]);
    if (part == 0) {
      const uint8_t* sb = shared ? L->shared_blob + L->gu_sb
                                 : L->pool + (uint64_t)U.slot * L->stride + L->gu_sb;
      ptx::bulk_g2s(sdst, sb + (uint64_t)16 * U.tile * HG * 4, sbytes, &mbar[s]);
    }
  };
  if (lane == 0) {
    if (nitems > 0) issue(0);
    if (nitems > 1) issue(1);
  }
  float o[8][4];
  for (int q = 0; q < nitems; ++q) {
    const UnitInfo U = unit_info(a, unit_of(q), n_used, n_slots);
    const int part = q % NH, s = q & 1;
    if (part == 0) {
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    }
    wait_bar(&mbar[s], (uint32_t)(q >> 1) & 1u, a.err);
    __syncwarp();
    const uint32_t tile = ptx::smem_u32(slots + (size_t)s * pslot);
    const uint32_t* sb = reinterpret_cast<const uint32_t*>(sbuf + (size_t)((q / NH) & 1) * a.gu_sb);
    const int ntiles = (U.n_e + 7) >> 3;
    if (ntiles <= 1)
      gu_unit_part<NJ, LCPG, 1>(a, U, part, tile, sb, o);
    else if (ntiles <= 2)
      gu_unit_part<NJ, LCPG, 2>(a, U, part, tile, sb, o);
    else if (ntiles <= 4)
      gu_unit_part<NJ, LCPG, 4>(a, U, part, tile, sb, o);
    else
      gu_unit_part<NJ, LCPG, 8>(a, U, part, tile, sb, o);
    if (part == NH - 1) {
      if (ntiles <= 1)
        gu_epilogue<1>(a, U, o);
      else if (ntiles <= 2)
        gu_epilogue<2>(a, U, o);
      else if (ntiles <= 4)
        gu_epilogue<4>(a, U, o);
      else
        gu_epilogue<8>(a, U, o);
    }
    __syncwarp();  // every lane is past its reads of slot s
    if (lane == 0 && q + 2 < nitems) issue(q + 2);
  }
}

// Down + combine.  CTA c owns rows 16 c .. 16 c + 15 of y.  Work items: every
// used expert (all of its token tiles at once), then the shared expert one
// token tile per item; warp w takes items w, w + 8, ... through two slots of
// its own and leaves each (row, pair) output in shared memory; after one
// barrier every token's rows are combined in the order of its top-k, the
// gated shared expert last.
template <int LCPG, int NT>
__device__ __forceinline__ void dn_item(const BArgs& a, int hrow0, int n_e, int nt0, bool ok,
                                        uint32_t tile, TileGeom geo, const uint32_t* sb,
                                        float* oc) {
  const int IG = a.I >> (LCPG + 5), IC = a.I / 32;
  const int lane = threadIdx.x & 31, g4 = lane >> 2, tg = lane & 3;
  int tb[NT], ta[NT], tc[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int base = (nt0 + nt) * 8;
    tb[nt] = (ok && base + g4 < n_e) ? hrow0 + base + g4 : -1;
    ta[nt] = base + 2 * tg < n_e ? hrow0 + base + 2 * tg : -1;
    tc[nt] = base + 2 * tg + 1 < n_e ? hrow0 + base + 2 * tg + 1 : -1;
  }
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  if (ok)
    tile_mn<LCPG, NT>(tile, geo, 0, IC, 0, a.hperm, a.I, tb, ta, tc, sb + g4 * IG,
                      sb + (g4 + 8) * IG, a.hg, IG, o);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (ta[nt] >= 0) {
      oc[(size_t)ta[nt] * 16 + g4] = o[nt][0];
      oc[(size_t)ta[nt] * 16 + g4 + 8] = o[nt][2];
    }
    if (tc[nt] >= 0) {
      oc[(size_t)tc[nt] * 16 + g4] = o[nt][1];
      oc[(size_t)tc[nt] * 16 + g4 + 8] = o[nt][3];
    }
  }
}

template <int LCPG>
__global__ void __launch_bounds__(kBThreads, 1) bdec_down_kernel(const BArgs a, int H) {
  const int I = a.I, k = a.k, T = a.T, P = a.P;
  const int IG = I >> (LCPG + 5);
  const bool dswz = I / 2 >= 128;
  const uint32_t pitch = dswz ? 128u : (uint32_t)(I / 2);
  const int ncbd = dswz ? I / 256 : 1;
  const TileGeom geo{16u * pitch, pitch, 8u * pitch, dswz};
  extern __shared__ uint8_t sm_raw[];
  uint8_t* sm = sm_raw + ((1024u - (ptx::smem_u32(sm_raw) & 1023u)) & 1023u);
  float* oc = reinterpret_cast<float*>(sm + a.ocache);  // [P + T][16]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* slots = sm + (size_t)warp * 2 * a.dn_slot;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(
                       sm + a.ocache + (((size_t)(P + T) * 64 + 15) & ~size_t(15))) + warp * 2;
  const DecLayer* L = a.L;
  const int n_slots = L->n_slots;
  const int r0 = 16 * (int)blockIdx.x;
  const int n_used = *a.n_used;
  const int nitem = n_used + (T + 7) / 8;  // routed experts, then the shared expert's token tiles
  const int nw = nitem > warp ? (nitem - warp + kBWarps - 1) / kBWarps : 0;
  const uint32_t tile_bytes = (uint32_t)ncbd * 16 * pitch;
  if (lane == 0) {
    ptx::mbar_init(&mbar[0], 1);
    ptx::mbar_init(&mbar[1], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int j) {  // lane 0: this warp's j-th item into slot j & 1
    const int q = warp + kBWarps * j;
    const int s = j & 1;
    uint8_t* dst = slots + (size_t)s * a.dn_slot;
    ptx::fence_proxy_async_smem();
    if (q < n_used) {
      const int slot = slot_of(a, a.used[q], n_slots);
      if (slot < 0) {
        record_error(a.err, MOE_ERR_SLOT);
        ptx::mbar_arrive_expect_tx(&mbar[s], 0);
        return;
      }
      ptx::mbar_arrive_expect_tx(&mbar[s], tile_bytes + 16u * IG * 4);
      ptx::tma_load_4d(dst, &L->map_d, 0, r0, 0, slot, &mbar[s]);
      ptx::bulk_g2s(dst + a.dn_sb,
                    L->pool + (uint64_t)slot * L->stride + L->d_sb + (uint64_t)r0 * IG * 4,
                    16u * IG * 4, &mbar[s]);
    } else {
      ptx::mbar_arrive_expect_tx(&mbar[s], tile_bytes + 16u * IG * 4);
      ptx::tma_load_4d(dst, &L->map_sd, 0, r0, 0, 0, &mbar[s]);
      ptx::bulk_g2s(dst + a.dn_sb, L->shared_blob + L->d_sb + (uint64_t)r0 * IG * 4,
                    16u * IG * 4, &mbar[s]);
    }
  };
  if (lane == 0) {
    if (nw > 0) issue(0);
    if (nw > 1) issue(1);
  }
  for (int j = 0; j < nw; ++j) {
    const int q = warp + kBWarps * j, s = j & 1;
    wait_bar(&mbar[s], (uint32_t)(j >> 1) & 1u, a.err);
    __syncwarp();
    const uint32_t tile = ptx::smem_u32(slots + (size_t)s * a.dn_slot);
    const uint32_t* sb = reinterpret_cast<const uint32_t*>(slots + (size_t)s * a.dn_slot + a.dn_sb);
    if (q < n_used) {
      const int e = a.used[q];
      const int pos0 = a.offsets[e], n_e = min(a.offsets[e + 1] - pos0, kBMaxT);
      const bool ok = slot_of(a, e, n_slots) >= 0;
      const int ntiles = (n_e + 7) >> 3;
      if (ntiles <= 1)
        dn_item<LCPG, 1>(a, pos0, n_e, 0, ok, tile, geo, sb, oc);
      else if (ntiles <= 2)
        dn_item<LCPG, 2>(a, pos0, n_e, 0, ok, tile, geo, sb, oc);
      else if (ntiles <= 4)
        dn_item<LCPG, 4>(a, pos0, n_e, 0, ok, tile, geo, sb, oc);
      else
        dn_item<LCPG, 8>(a, pos0, n_e, 0, ok, tile, geo, sb, oc);
    } else {
      dn_item<LCPG, 1>(a, P, T, q - n_used, true, tile, geo, sb, oc);
    }
    __syncwarp();
    if (lane == 0 && j + 2 < nw) issue(j + 2);
  }
  __syncthreads();
  // combine: rows 2 q and 2 q + 1 of token t per thread
  for (int w = tid; w < T * 8; w += kBThreads) {
    const int t = w >> 3, q = w & 7;
    float yv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int m = 2 * q + h;
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int pos = a.inv[t * k + j];
        acc = fmaf(a.topk_w[t * k + j], oc[(size_t)pos * 16 + m], acc);
      }
      yv[h] = fmaf(a.gate[t], oc[(size_t)(P + t) * 16 + m], acc);
    }
    reinterpret_cast<uint32_t*>(a.y + (size_t)t * H + r0)[q] =
        (uint32_t)f32_to_bf16_rne(yv[0]) | ((uint32_t)f32_to_bf16_rne(yv[1]) << 16);
  }
}

}  // namespace
}  // namespace moe

namespace moe {
namespace {

// ---------------------------------------------------------------- routing
// Router logits of T tokens in one launch: CTA c takes its share of the E
// router rows (and CTA 0 the shared gate vector as one more row), staged in
// shared memory; warp w takes tokens w, w + 8, ...  A lane sums each 8-element
// chunk with 8 sequential FMAs and its chunks in order, a butterfly sums the
// lanes, the prior comes last: depth D = 8 + H/256 + 5 + 1, so one uniform
// bound per token, 2 D u (|x_t| max_e |Wr_e| + max|prior|) (Higham, Accuracy
// and Stability of Numerical Algorithms, Thm. 4.3, with Cauchy-Schwarz),
// covers every logit of the token.
template <int NJ>
__global__ void __launch_bounds__(256) bdec_router_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ rw,
    const float* __restrict__ prior, const uint16_t* __restrict__ wsg, int E, float wmax,
    float pmax, float* __restrict__ logits, float* __restrict__ beta, float* __restrict__ gate_z) {
  constexpr int H = NJ * 256;
  extern __shared__ uint8_t sm_raw[];
  uint4* rows = reinterpret_cast<uint4*>(sm_raw);  // [nr (+1)][H/8]
  const int nC = gridDim.x, c = blockIdx.x;
  const int re0 = (int)(((long long)E * c) / nC), re1 = (int)(((long long)E * (c + 1)) / nC);
  const int nr = re1 - re0, nrow = nr + (c == 0 ? 1 : 0);
  for (int i = threadIdx.x; i < nrow * (H / 8); i += blockDim.x) {
    const int r = i / (H / 8), j = i - r * (H / 8);
    const uint16_t* src = r < nr ? rw + (size_t)(re0 + r) * H : wsg;
    ptx::cp_async16(rows + i, reinterpret_cast<const uint4*>(src) + j);  // all in flight
  }
  ptx::cp_async_commit();
  ptx::cp_async_wait_all();
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int DEPTH = 8 + NJ + 5 + 1;
  for (int t = warp; t < T; t += blockDim.x >> 5) {
    uint4 xv[NJ];
    float ss = 0.f;
#pragma unroll
    for (int jj = 0; jj < NJ; ++jj) {
      xv[jj] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * H) + lane + 32 * jj);
      const uint32_t w4[4] = {xv[jj].x, xv[jj].y, xv[jj].z, xv[jj].w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        ss = fmaf(bf16_lo(w4[q]), bf16_lo(w4[q]), fmaf(bf16_hi(w4[q]), bf16_hi(w4[q]), ss));
    }
    for (int r = 0; r < nrow; ++r) {
      float acc = 0.f;
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const uint4 wv = rows[(size_t)r * (H / 8) + lane + 32 * jj];
        const uint32_t a4[4] = {xv[jj].x, xv[jj].y, xv[jj].z, xv[jj].w};
        const uint32_t b4[4] = {wv.x, wv.y, wv.z, wv.w};
        float sc = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          sc = fmaf(bf16_lo(a4[q]), bf16_lo(b4[q]), sc);
          sc = fmaf(bf16_hi(a4[q]), bf16_hi(b4[q]), sc);
        }
        acc += sc;
      }
      acc = warp_sum(acc);
      if (lane == 0) {
        if (r < nr)
          logits[(size_t)t * E + re0 + r] = acc + (prior ? prior[re0 + r] : 0.f);
        else
          gate_z[t] = acc;
      }
    }
    if (c == 0) {
      ss = warp_sum(ss);
      // |x_t| rounded up (the fp32 sum of squares is within H u of the exact one)
      const float X = sqrtf(ss * 1.0009765625f) * 1.0009765625f;
      if (lane == 0)
        beta[t] = 2.0f * (float)DEPTH * 5.9604644775390625e-8f * 1.01f * (X * wmax + pmax) +
                  rt::kBoundFloor;
    }
  }
}

// Logits of one token with one uniform bound, for the exact selection routine.
struct TokenLogits {
  const float* l;
  float b;
  __device__ __forceinline__ void get(int e, float& logit, float& bnd) const {
    logit = __ldcg(l + e);
    bnd = b;
  }
  __device__ __forceinline__ int id(int e) const { return e; }
};

// Exact top-k of token blockIdx.x (the CTA-wide routine of routing_common.cuh),
// renormalised weights and the shared gate.
__global__ void __launch_bounds__(256) bdec_select_kernel(
    const float* __restrict__ logits, const float* __restrict__ beta,
    const float* __restrict__ gate_z, const uint16_t* __restrict__ x,
    const uint16_t* __restrict__ rw, const float* __restrict__ prior, int E, int k, int H,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, float* __restrict__ gate) {
  constexpr int V = kMaxE / 256;
  extern __shared__ uint8_t sm_raw[];
  const int t = blockIdx.x;
  const size_t sel = (rt::topk_warp_smem(E) + 15) & ~size_t(15);
  int* si;
  float* sv;
  rt::topk_select_block<V>(TokenLogits{logits + (size_t)t * E, beta[t]}, E, k, x + (size_t)t * H,
                           rw, prior, H, sm_raw, reinterpret_cast<uint2*>(sm_raw + sel),
                           reinterpret_cast<float*>(sm_raw + sel + 256 * V * 8), &si, &sv);
  if (threadIdx.x < 32) {
    const float w = rt::renormalised_weight(sv, k);
    const int lane = threadIdx.x;
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = si[lane];
      topk_w[(size_t)t * k + lane] = w;
    }
    if (lane == 0) gate[t] = 1.0f / (1.0f + __expf(-gate_z[t]));
  }
}

// Routing of 2..64 tokens in ONE cooperative launch.
// Phase 1: CTA c computes the logits of a tile of router rows (one of ES
// expert slices; slice 0 also the shared-gate row) against a slice of at most
// kRtTok tokens, both staged in shared memory, with bdec_router_kernel's
// summation structure (so the same uniform bound per token holds).
// A bounded grid barrier (a monotonic counter: every launch adds one arrival
// per CTA), then phase 2: CTA t < T runs the exact top-k of token t.
constexpr int kRtTok = 16;                     // tokens per token slice
constexpr uint32_t kRtSpin = 1u << 26;         // barrier polls before giving up
constexpr uint64_t kRtWaitNs = 1000000000ull;  // ... or one second

template <int NJ>
__global__ void __launch_bounds__(256, 1) small_route_kernel(
    const uint16_t* __restrict__ x, int T, const uint16_t* __restrict__ rw,
    const float* __restrict__ prior, const uint16_t* __restrict__ wsg, int E, int k, float wmax,
    float pmax, float* __restrict__ logits, float* __restrict__ beta, float* __restrict__ gate_z,
    unsigned long long* __restrict__ arrive, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, float* __restrict__ gate, int32_t* __restrict__ err) {
  constexpr int H = NJ * 256, W8 = H / 8;  // 16-byte pieces per row
  extern __shared__ __align__(16) uint8_t sm_raw[];
  const int nC = gridDim.x, c = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int TS = (T + kRtTok - 1) / kRtTok, ES = nC / TS;
  if (c < ES * TS) {
    // ---- phase 1: the tile (expert slice es, token slice ts)
    const int ts = c % TS, es = c / TS;
    const int re0 = (int)(((long long)E * es) / ES), re1 = (int)(((long long)E * (es + 1)) / ES);
    const int nr = re1 - re0, nrow = nr + (es == 0 ? 1 : 0);
    const int t0 = ts * kRtTok, nt = min(kRtTok, T - t0);
    uint4* rows = reinterpret_cast<uint4*>(sm_raw);  // [nrow][W8]
    uint4* xs = rows + (size_t)nrow * W8;            // [nt][W8]
    // asynchronous copies: every piece of the tile in flight at once
    for (int i = threadIdx.x; i < nrow * W8; i += blockDim.x) {
      const int r = i / W8, j = i - r * W8;
      const uint16_t* src = r < nr ? rw + (size_t)(re0 + r) * H : wsg;
      ptx::cp_async16(rows + i, reinterpret_cast<const uint4*>(src) + j);
    }
    for (int i = threadIdx.x; i < nt * W8; i += blockDim.x)
      ptx::cp_async16(xs + i, reinterpret_cast<const uint4*>(x + (size_t)t0 * H) + i);
    ptx::cp_async_commit();
    ptx::cp_async_wait_all();
    __syncthreads();
    constexpr int DEPTH = 8 + NJ + 5 + 1;
    // a warp's tokens, each unpacked once into registers and run against
    // every row of the tile, two rows at a time (two independent sums)
    for (int i = warp; i < nt; i += blockDim.x >> 5) {
      float xf[NJ][8];
#pragma unroll
      for (int jj = 0; jj < NJ; ++jj) {
        const uint4 xv = xs[(size_t)i * W8 + lane + 32 * jj];
        const uint32_t a4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xf[jj][2 * q] = bf16_lo(a4[q]);
          xf[jj][2 * q + 1] = bf16_hi(a4[q]);
        }
      }
      for (int r = 0; r < nrow; r += 2) {
        const int r1 = min(r + 1, nrow - 1);
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
          const uint4 w0 = rows[(size_t)r * W8 + lane + 32 * jj];
          const uint4 w1 = rows[(size_t)r1 * W8 + lane + 32 * jj];
          const uint32_t b0[4] = {w0.x, w0.y, w0.z, w0.w}, b1[4] = {w1.x, w1.y, w1.z, w1.w};
          float sc0 = 0.f, sc1 = 0.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            sc0 = fmaf(xf[jj][2 * q], bf16_lo(b0[q]), sc0);
            sc0 = fmaf(xf[jj][2 * q + 1], bf16_hi(b0[q]), sc0);
            sc1 = fmaf(xf[jj][2 * q], bf16_lo(b1[q]), sc1);
            sc1 = fmaf(xf[jj][2 * q + 1], bf16_hi(b1[q]), sc1);
          }
          acc0 += sc0;
          acc1 += sc1;
        }
        acc0 = warp_sum(acc0);
        acc1 = warp_sum(acc1);
        if (lane == 0) {
          for (int h = 0; h < 2 && r + h < nrow; ++h) {
            const int rr = r + h;
            const float acc = h ? acc1 : acc0;
            if (rr < nr)
              logits[(size_t)(t0 + i) * E + re0 + rr] = acc + (prior ? prior[re0 + rr] : 0.f);
            else
              gate_z[t0 + i] = acc;
          }
        }
      }
      if (es == 0) {  // the token's norm and uniform bound (slice 0 only)
        float ss = 0.f;
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ss = fmaf(xf[jj][2 * q], xf[jj][2 * q],
                      fmaf(xf[jj][2 * q + 1], xf[jj][2 * q + 1], ss));
        ss = warp_sum(ss);
        const float X = sqrtf(ss * 1.0009765625f) * 1.0009765625f;
        if (lane == 0)
          beta[t0 + i] = 2.0f * (float)DEPTH * 5.9604644775390625e-8f * 1.01f * (X * wmax + pmax) +
                         rt::kBoundFloor;
      }
    }
  }
  // ---- grid barrier: this CTA's writes, then wait for every CTA's
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned long long old = atomicAdd(arrive, 1ull);
    const unsigned long long target = (old / (unsigned long long)nC + 1ull) * (unsigned long long)nC;
    const uint64_t tb = ptx::globaltimer_ns();
    for (uint32_t it = 0; ptx::ld_acquire_u64(arrive) < target; ++it) {
      if (it > kRtSpin || ptx::globaltimer_ns() - tb > kRtWaitNs) {
        record_error(err, MOE_ERR_TIMEOUT);
        break;
      }
    }
    __threadfence();
  }
  __syncthreads();
  if (c >= T) return;
  // ---- phase 2: top-k of token c.  Fast path (as the decode kernel's): an
  // equal-width histogram of the logits from the top finds the bins holding
  // the first k + 1 entries; those candidates are ranked by (value, id) and
  // the order is certified when consecutive values are more than 2 beta apart.
  // Otherwise the CTA-wide exact routine decides (near-ties, rare).
  constexpr int V = kMaxE / 256;
  constexpr int kBinsR = 256, kCapR = 64;
  const int tid = threadIdx.x;
  const int need = min(k + 1, E);
  const float bt = __ldcg(beta + c);  // written by another CTA in this launch: through L2
  const float* lt = logits + (size_t)c * E;
  uint32_t* s_hist = reinterpret_cast<uint32_t*>(sm_raw);        // [kBinsR + 1]
  uint2* s_cand = reinterpret_cast<uint2*>(sm_raw + 2048);       // [kCapR]
  uint32_t* s_red = reinterpret_cast<uint32_t*>(sm_raw + 2560);  // [16]
  int* s_sidx = reinterpret_cast<int*>(sm_raw + 2624);           // [33]
  float* s_sval = reinterpret_cast<float*>(sm_raw + 2768);       // [33]
  int* s_ok = reinterpret_cast<int*>(sm_raw + 2912);
  s_hist[tid] = 0u;
  if (tid == 0) s_hist[kBinsR] = 0u;
  uint32_t key[V];
  float lv[V];
  uint32_t kmx = 0u, kmn = 0xFFFFFFFFu;
#pragma unroll
  for (int q = 0; q < V; ++q) {
    const int e = tid + 256 * q;
    float f = e < E ? __ldcg(lt + e) : 0.f;
    if (f != f) f = -INFINITY;
    lv[q] = f;
    key[q] = e < E ? rt::f32_key(f) : 0u;
    if (e < E) {
      kmx = max(kmx, key[q]);
      kmn = min(kmn, key[q]);
    }
  }
  kmx = __reduce_max_sync(0xffffffffu, kmx);
  kmn = __reduce_min_sync(0xffffffffu, kmn);
  if (lane == 0) {
    s_red[warp] = kmx;
    s_red[8 + warp] = kmn;
  }
  __syncthreads();
  {
    uint32_t gx = 0u, gn = 0xFFFFFFFFu;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      gx = max(gx, s_red[w]);
      gn = min(gn, s_red[8 + w]);
    }
    const float M = rt::key_f32(gx), mn = rt::key_f32(gn);
    const float scale = (M > mn) ? (float)(kBinsR - 1) / (M - mn) : 0.f;
    int bin[V];
#pragma unroll
    for (int q = 0; q < V; ++q) {
      bin[q] = (int)fminf((float)(kBinsR - 1), (M - lv[q]) * scale);
      if (tid + 256 * q < E) atomicAdd(&s_hist[bin[q]], 1u);
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
    const uint32_t hit = __ballot_sync(0xffffffffu, incl >= (uint32_t)need);
    int bstar = kBinsR - 1;
    if (hit) {
      const int hl = __ffs(hit) - 1;
      uint32_t acc = incl - run;
      int bl = -1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        acc += cnt[i];
        if (bl < 0 && acc >= (uint32_t)need) bl = i;
      }
      bstar = __shfl_sync(0xffffffffu, 8 * lane + bl, hl);
    }
#pragma unroll
    for (int q = 0; q < V; ++q) {
      const int e = tid + 256 * q;
      if (e < E && bin[q] <= bstar) {
        const uint32_t pos = atomicAdd(&s_hist[kBinsR], 1u);
        if (pos < (uint32_t)kCapR) s_cand[pos] = make_uint2(key[q], (uint32_t)e);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int nc = (int)s_hist[kBinsR];
    bool ok = nc >= need && nc <= kCapR;
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
          s_sval[rank] = rt::key_f32(me.x);
        }
      }
      __syncwarp();
      const bool gap = lane + 1 >= need || (s_sval[lane] - s_sval[lane + 1] > 2.0f * bt);
      ok = __all_sync(0xffffffffu, gap);
    }
    if (lane == 0) *s_ok = ok ? 1 : 0;
  }
  __syncthreads();
  const int* si = s_sidx;
  const float* sv = s_sval;
  if (!*s_ok) {
    __syncthreads();  // every thread has read s_ok before the routine reuses the memory
    const size_t sel = (rt::topk_warp_smem(E) + 15) & ~size_t(15);
    int* bi;
    float* bv;
    rt::topk_select_block<V>(TokenLogits{lt, bt}, E, k, x + (size_t)c * H, rw, prior, H, sm_raw,
                             reinterpret_cast<uint2*>(sm_raw + sel),
                             reinterpret_cast<float*>(sm_raw + sel + 256 * V * 8), &bi, &bv);
    si = bi;
    sv = bv;
  }
  if (threadIdx.x < 32) {
    const float w = rt::renormalised_weight(sv, k);
    if (lane < k) {
      topk_idx[(size_t)c * k + lane] = si[lane];
      topk_w[(size_t)c * k + lane] = w;
    }
    if (lane == 0) gate[c] = 1.0f / (1.0f + __expf(-__ldcg(gate_z + c)));
  }
}

}  // namespace
}  // namespace moe

// ---------------------------------------------------------------- host side
namespace moe {
namespace {

uint32_t up_u32(uint64_t v, uint64_t al) { return (uint32_t)((v + al - 1) / al * al); }

struct BPlan {
  uint32_t gu_slot, gu_sb, part, smem_gu, dn_slot, dn_sb, ocache, smem_dn;
};

bool bplan(const Dims& d, int T, BPlan& p) {
  const int H = d.H, I = d.I, G = d.G;
  const int NCB = H / 256, HG = H / G, IG = I / G;
  const bool dswz = I / 2 >= 128;
  const uint64_t pitch = dswz ? 128 : (uint64_t)(I / 2);
  const uint64_t ncbd = dswz ? (uint64_t)(I / 256) : 1;
  // gate/up: per warp two part slots (16 rows x the column blocks of a part)
  // and two scale buffers; the barriers last
  const int NH = NCB >= 2 ? 2 : 1;
  p.gu_slot = (uint32_t)(NCB / NH) * 2048;
  p.gu_sb = up_u32(16ull * HG * 4, 16);
  p.part = kBWarps * 2 * (p.gu_slot + p.gu_sb);
  p.smem_gu = p.part + kBWarps * 2 * 8 + 1024;
  p.dn_sb = up_u32(ncbd * 16 * pitch, 128);
  p.dn_slot = up_u32((uint64_t)p.dn_sb + 16ull * IG * 4, 1024);
  p.ocache = kBWarps * 2 * p.dn_slot;  // two slots per warp, then the outputs
  const uint64_t rows = (uint64_t)T * d.k + T;
  p.smem_dn = (uint32_t)(p.ocache + ((rows * 64 + 15) & ~15ull) + kBWarps * 2 * 8 + 1024);
  return T >= 2 && T <= kBMaxT && decode_shape_ok(d) && p.smem_gu <= kBSmemMax &&
         p.smem_dn <= kBSmemMax;
}

template <int NJ, int LC>
struct GateUpF {
  static cudaError_t attr() {
    return cudaFuncSetAttribute(bdec_gateup_kernel<NJ, LC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmemMax);
  }
  static cudaError_t run(const BArgs* a, int nC, cudaStream_t st) {
    bdec_gateup_kernel<NJ, LC><<<nC, kBThreads, a->smem_gu, st>>>(*a);
    return cudaGetLastError();
  }
};

template <int LC>
cudaError_t down_run(const BArgs& a, int H, cudaStream_t st) {
  bdec_down_kernel<LC><<<H / 16, kBThreads, a.smem_dn, st>>>(a, H);
  return cudaGetLastError();
}

template <int NJ>
cudaError_t gu_dispatch_lc(int lc, bool attr_only, const BArgs* a, int nC, cudaStream_t st) {
  if (lc == 0) return attr_only ? GateUpF<NJ, 0>::attr() : GateUpF<NJ, 0>::run(a, nC, st);
  if (lc == 1) return attr_only ? GateUpF<NJ, 1>::attr() : GateUpF<NJ, 1>::run(a, nC, st);
  return attr_only ? GateUpF<NJ, 2>::attr() : GateUpF<NJ, 2>::run(a, nC, st);
}

cudaError_t gu_dispatch(const Dims& d, bool attr_only, const BArgs* a, int nC, cudaStream_t st) {
  const int lc = d.G == 32 ? 0 : d.G == 64 ? 1 : 2;
  switch (d.H / 256) {
    case 1: return gu_dispatch_lc<1>(lc, attr_only, a, nC, st);
    case 2: return gu_dispatch_lc<2>(lc, attr_only, a, nC, st);
    case 4: return gu_dispatch_lc<4>(lc, attr_only, a, nC, st);
    case 8: return gu_dispatch_lc<8>(lc, attr_only, a, nC, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool batch_decode_supported(const Ctx& c, int T) {
  BPlan p;
  return c.dec_ok && c.dec_layer && !c.pl.slots && bplan(c.d, T, p);
}

cudaError_t prepare_batch_decode(const Ctx& c) {
  {  // the fused small-T routing kernel (any shape it takes)
    const void* fns[4] = {(const void*)small_route_kernel<1>, (const void*)small_route_kernel<2>,
                          (const void*)small_route_kernel<4>, (const void*)small_route_kernel<8>};
    for (const void* f : fns) {
      cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmemMax);
      if (e != cudaSuccess) return e;
    }
  }
  BPlan p;
  if (!c.dec_ok || !bplan(c.d, 2, p)) return cudaSuccess;
  cudaError_t e = gu_dispatch(c.d, true, nullptr, 0, nullptr);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bdec_down_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBSmemMax);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bdec_down_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBSmemMax);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bdec_down_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBSmemMax);
  return e;
}

cudaError_t launch_batch_route(const Ctx& c, const FwdArgs& f, cudaStream_t st, int* launches) {
  const Dims& d = c.d;
  const int T = f.T, E = d.E, H = d.H, nC = c.num_sms;
  const size_t rsm = (size_t)(E / nC + 2) * H * 2;
  float* beta = c.ws.bound;  // [T]: one bound per token
#define MOE_BDR(NJ)                                                                            \
  bdec_router_kernel<NJ><<<nC, 256, rsm, st>>>(f.x, T, c.router_w, c.router_bias,             \
                                                c.shared_gate_w, E, c.dec_wmax, c.dec_pmax,   \
                                                c.ws.logits, beta, c.ws.gate_z)
  switch (H / 256) {
    case 1: MOE_BDR(1); break;
    case 2: MOE_BDR(2); break;
    case 4: MOE_BDR(4); break;
    case 8: MOE_BDR(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef MOE_BDR
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const size_t ssm = ((rt::topk_warp_smem(E) + 15) & ~size_t(15)) + 256 * (kMaxE / 256) * 8 + 64;
  bdec_select_kernel<<<T, 256, ssm, st>>>(c.ws.logits, beta, c.ws.gate_z, f.x, c.router_w,
                                           c.router_bias, E, d.k, H, f.topk_idx, f.topk_w,
                                           c.ws.gate);
  *launches += 2;
  return cudaGetLastError();
}

namespace {
// Shared memory of small_route_kernel: phase 1's row and token tiles, or
// phase 2's selection scratch, whichever is larger.
size_t small_route_smem(const Dims& d, int T, int nC) {
  const int TS = (T + kRtTok - 1) / kRtTok, ES = nC / TS;
  const size_t rows = (size_t)((d.E + ES - 1) / ES + 1);
  const size_t p1 = (rows + kRtTok) * (size_t)d.H * 2;
  const size_t p2 = ((rt::topk_warp_smem(d.E) + 15) & ~size_t(15)) + 256 * (kMaxE / 256) * 8 + 64;
  return p1 > p2 ? p1 : p2;
}

}  // namespace

bool small_route_supported(const Ctx& c, int T) {
  return T >= 2 && T <= 64 && c.num_sms >= T && c.num_sms >= (T + kRtTok - 1) / kRtTok &&
         c.d.H <= 2048 && c.d.H % 256 == 0 && (c.d.H / 256 & (c.d.H / 256 - 1)) == 0 &&
         c.d.E <= kMaxE && c.ws.rcnt && small_route_smem(c.d, T, c.num_sms) <= kBSmemMax;
}

cudaError_t launch_small_route(const Ctx& c, const FwdArgs& f, cudaStream_t st, int* launches) {
  const Dims& d = c.d;
  const int T = f.T;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.num_sms);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = small_route_smem(d, T, c.num_sms);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // the grid barrier needs every CTA resident
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
#define MOE_SRT(NJ)                                                                            \
  e = cudaLaunchKernelEx(&cfg, small_route_kernel<NJ>, f.x, T, (const uint16_t*)c.router_w,     \
                         (const float*)c.router_bias, (const uint16_t*)c.shared_gate_w, d.E,    \
                         d.k, c.dec_wmax, c.dec_pmax, c.ws.logits, c.ws.bound, c.ws.gate_z,     \
                         c.ws.rcnt, f.topk_idx, f.topk_w, c.ws.gate, c.err)
  switch (d.H / 256) {
    case 1: MOE_SRT(1); break;
    case 2: MOE_SRT(2); break;
    case 4: MOE_SRT(4); break;
    case 8: MOE_SRT(8); break;
    default: return cudaErrorInvalidValue;
  }
#undef MOE_SRT
  ++*launches;
  return e;
}

cudaError_t launch_batch_decode(const Ctx& c, const FwdArgs& f, cudaStream_t st, int* launches) {
  const Dims& d = c.d;
  BPlan p;
  if (!bplan(d, f.T, p)) return cudaErrorInvalidValue;
  const int T = f.T, H = d.H, I = d.I, G = d.G, P = T * d.k;
  BArgs a{};
  a.L = c.dec_layer;
  a.T = T;
  a.k = d.k;
  a.E = d.E;
  a.I = I;
  a.G = G;
  a.P = P;
  a.used = c.ws.used;
  a.n_used = c.ws.n_used;
  a.offsets = c.ws.offsets;
  a.perm = c.ws.perm;
  a.inv = c.ws.inv;
  a.table = f.table;
  a.x = f.x;
  // scratch: h in the workspace's h rows, the rest in its fp32 output rows
  a.hperm = reinterpret_cast<uint16_t*>(c.ws.h);
  uint8_t* o = reinterpret_cast<uint8_t*>(c.ws.o);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* r = o + off;
    off += (bytes + 255) & ~size_t(255);
    return r;
  };
  a.xperm = reinterpret_cast<uint16_t*>(take((size_t)T * H * 2));
  a.xg = reinterpret_cast<float*>(take((size_t)T * (H / G) * 4));
  a.hs8 = reinterpret_cast<float*>(take((size_t)(P + T) * (I / 8) * 4));
  a.hg = reinterpret_cast<float*>(take((size_t)(P + T) * (I / G) * 4));
  a.topk_w = f.topk_w;
  a.gate = c.ws.gate;
  a.y = f.y;
  a.err = c.err;
  a.gu_slot = p.gu_slot;
  a.gu_sb = p.gu_sb;
  a.part = p.part;
  a.smem_gu = p.smem_gu;
  a.dn_slot = p.dn_slot;
  a.dn_sb = p.dn_sb;
  a.ocache = p.ocache;
  a.smem_dn = p.smem_dn;
  bdec_prep_kernel<<<T, 256, 0, st>>>(f.x, H, G, a.xperm, a.xg);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = gu_dispatch(d, false, &a, c.num_sms, st);
  if (e == cudaSuccess) {
    const int n = (P + T) * (I / G);
    bdec_hsum_kernel<<<(n + 255) / 256, 256, 0, st>>>(a.hs8, P + T, I, G, a.hg);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) {
    const int lc = G == 32 ? 0 : G == 64 ? 1 : 2;
    e = lc == 0 ? down_run<0>(a, H, st) : lc == 1 ? down_run<1>(a, H, st) : down_run<2>(a, H, st);
  }
  *launches += 4;
  return e;
}

}  // namespace moe
