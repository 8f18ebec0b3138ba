// permute.cu -- deterministic token->expert permutation (stable counting sort).
//
// The pairs p = t*k + j (token t's j-th expert) are sorted by expert id,
// keeping ascending p inside each expert: offsets[e] = number of pairs with a
// smaller expert id, perm[offsets[e] + r] = the r-th pair (in p order) that
// chose e, inv[p] = the position of p in perm.  `used` lists the experts with
// at least one pair in ascending id; the expert kernels walk it.
#include "device_util.cuh"
#include "moe_internal.cuh"
#include "tiles.cuh"

namespace moe {

namespace {

constexpr int kPairsPerBlock = 2048;
constexpr int kScatterWarps = 8;  // warps that scatter one block's pairs

// Exclusive scan of one value per thread over a CTA of up to 1024 threads.
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < nw) warp_tot[lane] = w;  // inclusive warp prefix
    if (lane == nw - 1) *total = w;
  }
  __syncthreads();
  const int before = warp ? warp_tot[warp - 1] : 0;
  const int r = before + incl - v;
  __syncthreads();
  return r;
}

// Stable placement of pairs [p0, p1) by one warp, in order, chunk by chunk:
// pos[e] holds the next free position of expert e.
__device__ void warp_stable_scatter(const int32_t* __restrict__ topk_idx, int p0, int p1,
                                    int* pos, int32_t* __restrict__ perm,
                                    int32_t* __restrict__ inv, int32_t* perm_out) {
  const int lane = threadIdx.x & 31;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    const int e = p < p1 ? topk_idx[p] : -1;
    const unsigned mask = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(mask & ((1u << lane) - 1u));
    int q = 0;
    if (e >= 0) q = pos[e] + rank;
    __syncwarp();
    if (e >= 0) {
      perm[q] = p;
      inv[p] = q;
      if (perm_out) perm_out[q] = p;
      if (lane == 31 - __clz(mask)) pos[e] += __popc(mask);
    }
    __syncwarp();
  }
}

// Stable placement of pairs [p0, p1) by the first kScatterWarps warps of the
// CTA: warp w takes a contiguous segment, counts it per expert into hist[w],
// the counts become per-warp start positions (base[e] + the counts of the
// earlier segments), and each warp places its segment in order.  Every thread
// of the CTA calls (the barriers span the CTA).  hist: kScatterWarps * E ints
// of shared memory.
__device__ void block_stable_scatter(const int32_t* __restrict__ topk_idx, int p0, int p1,
                                     const int* base, int E, int* hist,
                                     int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                     int32_t* perm_out) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = ((p1 - p0 + kScatterWarps * 32 - 1) / (kScatterWarps * 32)) * 32;
  const int w0 = min(p1, p0 + warp * seg), w1 = min(p1, w0 + seg);
  int* h = hist + (size_t)warp * E;
  if (warp < kScatterWarps)
    for (int e = lane; e < E; e += 32) h[e] = 0;
  __syncthreads();
  if (warp < kScatterWarps) {
    for (int b = w0; b < w1; b += 32) {
      const int p = b + lane;
      const int e = p < w1 ? topk_idx[p] : -1;
      const unsigned mask = __match_any_sync(0xffffffffu, e);
      if (e >= 0 && lane == 31 - __clz(mask)) h[e] += __popc(mask);
      __syncwarp();
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = base[e];
    for (int w = 0; w < kScatterWarps; ++w) {
      const int t = hist[(size_t)w * E + e];
      hist[(size_t)w * E + e] = run;
      run += t;
    }
  }
  __syncthreads();
  if (warp < kScatterWarps) warp_stable_scatter(topk_idx, w0, w1, h, perm, inv, perm_out);
}

// One CTA does everything (used when the pairs fit one block), and with
// `tiles` set also the grouped GEMMs' tile list.
struct TileArgs {
  Tile* tiles;  // null: no tile list
  int32_t* n_tiles;
  const int32_t* table;
  int n_slots, T, max_tiles;
  int32_t* err;
};

__global__ void __launch_bounds__(1024) permute_small_kernel(
    const int32_t* __restrict__ topk_idx, int P, int E, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int32_t* __restrict__ offsets, int32_t* __restrict__ used,
    int32_t* __restrict__ n_used, int32_t* perm_out, int32_t* offsets_out, TileArgs ta) {
  __shared__ int cnt[kMaxE];
  __shared__ int hist[kScatterWarps * kMaxE];
  __shared__ int warp_tot[32];
  __shared__ int total, total_used;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) atomicAdd(&cnt[topk_idx[p]], 1);
  __syncthreads();
  const int e = threadIdx.x;
  const int c = e < E ? cnt[e] : 0;
  const int excl = block_exclusive_scan(c, warp_tot, &total);
  const int uexcl = block_exclusive_scan(c > 0 ? 1 : 0, warp_tot, &total_used);
  if (e < E) {
    offsets[e] = excl;
    if (offsets_out) offsets_out[e] = excl;
    if (c > 0) used[uexcl] = e;
    cnt[e] = excl;
  }
  if (e == 0) {
    offsets[E] = total;
    if (offsets_out) offsets_out[E] = total;
    *n_used = total_used;
  }
  __syncthreads();
  block_stable_scatter(topk_idx, 0, P, cnt, E, hist, perm, inv, perm_out);
  if (ta.tiles) {
    __syncthreads();  // used, n_used and offsets are in global memory, written above
    build_tiles_block(used, n_used, offsets, ta.table, ta.n_slots, ta.T, P, ta.tiles, ta.n_tiles,
                      ta.max_tiles, ta.err, warp_tot);
  }
}

// Large P, pass 1: per-block expert counts.
__global__ void __launch_bounds__(256) permute_count_kernel(const int32_t* __restrict__ topk_idx,
                                                            int P, int E,
                                                            int32_t* __restrict__ hist) {
  __shared__ int cnt[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  const int p0 = blockIdx.x * kPairsPerBlock, p1 = min(P, p0 + kPairsPerBlock);
  for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x) atomicAdd(&cnt[topk_idx[p]], 1);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[(size_t)blockIdx.x * E + e] = cnt[e];
}

// Large P, pass 2: offsets, used list, and each block's first position per expert.
__global__ void __launch_bounds__(1024) permute_scan_kernel(
    int32_t* __restrict__ hist, int nblk, int E, int32_t* __restrict__ offsets,
    int32_t* __restrict__ used, int32_t* __restrict__ n_used, int32_t* offsets_out) {
  __shared__ int warp_tot[32];
  __shared__ int total, total_used;
  const int e = threadIdx.x;
  int running = 0;
  if (e < E) {
    for (int b = 0; b < nblk; ++b) {
      const int v = hist[(size_t)b * E + e];
      hist[(size_t)b * E + e] = running;
      running += v;
    }
  }
  const int excl = block_exclusive_scan(running, warp_tot, &total);
  const int uexcl = block_exclusive_scan(running > 0 ? 1 : 0, warp_tot, &total_used);
  if (e < E) {
    offsets[e] = excl;
    if (offsets_out) offsets_out[e] = excl;
    if (running > 0) used[uexcl] = e;
    for (int b = 0; b < nblk; ++b) hist[(size_t)b * E + e] += excl;
  }
  if (e == 0) {
    offsets[E] = total;
    if (offsets_out) offsets_out[E] = total;
    *n_used = total_used;
  }
}

// Large P, pass 3: stable scatter of each block's pairs by kScatterWarps warps.
__global__ void __launch_bounds__(kScatterWarps * 32) permute_scatter_kernel(
    const int32_t* __restrict__ topk_idx, int P, int E, const int32_t* __restrict__ hist,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* perm_out) {
  __shared__ int sh[kScatterWarps * kMaxE];
  const int p0 = blockIdx.x * kPairsPerBlock, p1 = min(P, p0 + kPairsPerBlock);
  block_stable_scatter(topk_idx, p0, p1, hist + (size_t)blockIdx.x * E, E, sh, perm, inv,
                       perm_out);
}

}  // namespace

cudaError_t launch_permute(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches,
                           bool with_tiles, bool* tiles_built) {
  const int P = a.T * c.d.k, E = c.d.E;
  *tiles_built = false;
  if (P <= kPairsPerBlock) {
    TileArgs ta{nullptr, nullptr, nullptr, 0, 0, 0, nullptr};
    if (with_tiles) {
      ta = TileArgs{reinterpret_cast<Tile*>(c.ws.tiles), c.ws.n_tiles, a.table, c.n_slots, a.T,
                    prefill_max_tiles(c.d, a.T), c.err};
      *tiles_built = true;
    }
    permute_small_kernel<<<1, 1024, 0, st>>>(a.topk_idx, P, E, c.ws.perm, c.ws.inv,
                                              c.ws.offsets, c.ws.used, c.ws.n_used, a.perm_out,
                                              a.offsets_out, ta);
    ++*launches;
    return cudaGetLastError();
  }
  const int nblk = (P + kPairsPerBlock - 1) / kPairsPerBlock;
  permute_count_kernel<<<nblk, 256, 0, st>>>(a.topk_idx, P, E, c.ws.hist);
  permute_scan_kernel<<<1, 1024, 0, st>>>(c.ws.hist, nblk, E, c.ws.offsets, c.ws.used,
                                           c.ws.n_used, a.offsets_out);
  permute_scatter_kernel<<<nblk, kScatterWarps * 32, 0, st>>>(a.topk_idx, P, E, c.ws.hist,
                                                                c.ws.perm, c.ws.inv, a.perm_out);
  *launches += 3;
  return cudaGetLastError();
}

}  // namespace moe
