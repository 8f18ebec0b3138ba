// pool.cu -- a bounded pool of resident expert slots, filled on the stream.
//
// The pages stream routed experts from storage into a pool of bounded size
// that evicts by use frequency and recency (Swiftlet README on the wpnews
// page, "How it works"; creativeainews, "How Expert Streaming Works").  Here every expert's
// blob lives in pinned, device-mapped host memory (reached over NVLink-C2C)
// and the device holds S < E slots.  After the routing of each forward call
// and before any expert runs:
//   pool_update_kernel  one CTA: counts the pairs per expert, marks hits
//                       (frequency += pairs, last use = this step), then for
//                       each miss in ascending expert id takes an empty slot,
//                       else evicts the slot (not needed this step) with the
//                       lowest frequency, then the least recent use, then the
//                       lowest id; writes the list of fills and the table
//   pool_copy_kernel    all SMs: copies the filled blobs from host memory
// No host synchronisation: the table the expert kernels read is updated on
// the stream.  Frequencies saturate at 2^23 - 1, steps at 2^24 - 1 and slots
// are fewer than 2^16 - 1, so that a slot's (occupied, frequency, step, slot)
// key packs into 64 bits below the "not evictable" key ~0.
#include "moe_internal.cuh"

namespace moe {

namespace {

constexpr int kPoolThreads = 1024;
constexpr uint32_t kFreqMax = (1u << 23) - 1;
constexpr uint32_t kStepMax = (1u << 24) - 1;

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long t = __shfl_xor_sync(0xffffffffu, v, o);
    v = t < v ? t : v;
  }
  return v;
}

// state: [0] step, [1] hits, [2] misses, [3] evictions, [4] overflows,
// [5] fills of the last step
__global__ void __launch_bounds__(kPoolThreads) pool_update_kernel(
    const int32_t* __restrict__ topk_idx, int P, int E, int S, int32_t* __restrict__ table,
    int32_t* __restrict__ owner, uint32_t* __restrict__ freq, uint32_t* __restrict__ last,
    uint32_t* __restrict__ state, int32_t* __restrict__ fill_expert,
    int32_t* __restrict__ fill_slot) {
  __shared__ uint32_t cnt[kMaxE];
  __shared__ unsigned long long wmin[kPoolThreads / 32];
  __shared__ int s_victim;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kPoolThreads) cnt[e] = 0u;
  __syncthreads();
  for (int p = tid; p < P; p += kPoolThreads) {
    const int e = topk_idx[p];
    if (e >= 0 && e < E) atomicAdd(&cnt[e], 1u);
  }
  __syncthreads();
  const uint32_t step = min(state[0] + 1u, kStepMax);
  // hits
  uint32_t hits = 0;
  for (int e = tid; e < E; e += kPoolThreads) {
    const int s = table[e];
    if (cnt[e] && s >= 0) {
      freq[s] = min(freq[s] + cnt[e], kFreqMax);
      last[s] = step;
      ++hits;
    }
  }
  __syncthreads();
  // misses in ascending expert id, one block-wide arg-min per miss
  uint32_t misses = 0, evictions = 0, overflows = 0;
  for (int e = 0; e < E; ++e) {
    if (!cnt[e] || table[e] >= 0) continue;  // uniform: shared and global reads after a barrier
    unsigned long long best = ~0ull;
    for (int s = tid; s < S; s += kPoolThreads) {
      const int o = owner[s];
      unsigned long long key;
      if (o < 0)
        key = (unsigned long long)s;  // empty slots first
      else if (cnt[o])
        key = ~0ull;                   // needed by this step: not evictable
      else
        key = (1ull << 63) | ((unsigned long long)freq[s] << 40) |
              ((unsigned long long)last[s] << 16) | (unsigned long long)s;
      best = key < best ? key : best;
    }
    best = warp_min_u64(best);
    if (lane == 0) wmin[warp] = best;
    __syncthreads();
    if (tid == 0) {
      unsigned long long b = wmin[0];
      for (int w = 1; w < kPoolThreads / 32; ++w) b = wmin[w] < b ? wmin[w] : b;
      s_victim = b == ~0ull ? -1 : (int)(b & 0xFFFFull);
    }
    __syncthreads();
    const int v = s_victim;
    if (tid == 0) {
      if (v < 0) {
        ++overflows;
      } else {
        const int o = owner[v];
        if (o >= 0) {
          table[o] = -1;
          ++evictions;
        }
        owner[v] = e;
        table[e] = v;
        freq[v] = min(cnt[e], kFreqMax);
        last[v] = step;
        fill_expert[misses] = e;
        fill_slot[misses] = v;
        ++misses;
      }
    }
    __syncthreads();  // the table and owner updates are seen by the next miss
  }
  // totals (thread 0 holds the miss counts; every thread its share of hits)
  for (int o = 16; o > 0; o >>= 1) hits += __shfl_xor_sync(0xffffffffu, hits, o);
  if (lane == 0 && hits) atomicAdd(&state[1], hits);
  if (tid == 0) {
    state[0] = step;
    state[2] += misses;
    state[3] += evictions;
    state[4] += overflows;
    state[5] = misses;
  }
}

// Copies the fills of the last step: work item i = (fill, 16 KB chunk).
__global__ void __launch_bounds__(256) pool_copy_kernel(
    const uint8_t* __restrict__ store, uint8_t* __restrict__ pool, uint64_t stride,
    const uint32_t* __restrict__ state, const int32_t* __restrict__ fill_expert,
    const int32_t* __restrict__ fill_slot) {
  const uint32_t nfill = state[5];
  const uint64_t chunks = (stride + 16383) / 16384;
  for (uint64_t w = blockIdx.x; w < (uint64_t)nfill * chunks; w += gridDim.x) {
    const uint64_t f = w / chunks, c = w - f * chunks;
    const uint4* src =
        reinterpret_cast<const uint4*>(store + (uint64_t)fill_expert[f] * stride + c * 16384);
    uint4* dst = reinterpret_cast<uint4*>(pool + (uint64_t)fill_slot[f] * stride + c * 16384);
    const uint64_t n = (c + 1) * 16384 <= stride ? 1024 : (stride - c * 16384) / 16;
    for (uint64_t i = threadIdx.x; i < n; i += blockDim.x) dst[i] = src[i];
  }
}

}  // namespace

cudaError_t launch_pool_update(const Ctx& c, const int32_t* topk_idx, int P, cudaStream_t st,
                               int* launches) {
  const PoolState& p = c.pl;
  pool_update_kernel<<<1, kPoolThreads, 0, st>>>(topk_idx, P, c.d.E, p.slots, p.table, p.owner,
                                                 p.freq, p.last, p.state, p.fill_expert,
                                                 p.fill_slot);
  ++*launches;
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pool_copy_kernel<<<c.num_sms * 4, 256, 0, st>>>(p.store_dev, c.pool, c.ex.stride, p.state,
                                                  p.fill_expert, p.fill_slot);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace moe
