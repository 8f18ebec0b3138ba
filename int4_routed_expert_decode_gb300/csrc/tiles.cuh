// tiles.cuh -- the work tiles of the grouped GEMMs (prefill.cu): for each
// expert in use (ascending id) tiles of up to kTileTokens of its pair
// positions, then the shared expert's tiles over all tokens.  Built by one CTA
// of 1024 threads, either in its own launch or as the tail of the one-CTA
// permutation (permute.cu).
#pragma once

#include <stdint.h>

#include "device_util.cuh"

namespace moe {

constexpr int kTileTokens = 128;  // tokens per tile (the grouped GEMM's largest UMMA N)

struct Tile {
  int slot;   // expert slot, or -1 for the shared expert
  int pos0;   // first pair position (routed) or first token (shared)
  int ntok;   // tokens in the tile, 0 < ntok <= kTileTokens (0: skipped)
  int hrow0;  // first row of h that the tile owns
};

// One thread per used expert (blockDim.x >= *n_used, a multiple of 32, at
// most 1024); used, n_used and offsets may have been written by this CTA
// before a __syncthreads.  warp_tot: 32 ints of shared memory.  An expert
// whose slot is out of range records MOE_ERR_SLOT and gets empty tiles.
__device__ __forceinline__ void build_tiles_block(
    const int32_t* used, const int32_t* n_used, const int32_t* offsets, const int32_t* table,
    int n_slots, int T, int P, Tile* __restrict__ tiles, int32_t* __restrict__ n_tiles,
    int max_tiles, int32_t* err, int* warp_tot) {
  const int nu = *n_used;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int cnt = 0, e = -1;
  if ((int)threadIdx.x < nu) {
    e = used[threadIdx.x];
    cnt = (offsets[e + 1] - offsets[e] + kTileTokens - 1) / kTileTokens;
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
        tiles[id] = Tile{bad ? 0 : slot, p0 + i * kTileTokens,
                         bad ? 0 : min(kTileTokens, n_e - i * kTileTokens), p0 + i * kTileTokens};
    }
  }
  const int nsh = (T + kTileTokens - 1) / kTileTokens;
  for (int i = threadIdx.x; i < nsh; i += blockDim.x) {
    const int id = routed + i;
    if (id < max_tiles)
      tiles[id] = Tile{-1, i * kTileTokens, min(kTileTokens, T - i * kTileTokens),
                       P + i * kTileTokens};
  }
  if (threadIdx.x == 0) *n_tiles = min(max_tiles, routed + nsh);
}

}  // namespace moe
