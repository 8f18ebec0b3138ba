// repack.cu -- canonical MLX affine int4 / int8 tensors <-> fixed-stride expert blobs.
//
// The Swiftlet README (wpnews page, "How it works") repacks the routed
// experts into records of one fixed stride, so that one expert is one
// contiguous record addressed by a 64-bit offset.  Here a blob holds, for one
// expert (c = 32/bits codes per packed word: 8 for int4, 4 for int8):
//   gu_q  [I][2][H/c]  gate row i and up row i side by side (one SwiGLU
//                      output needs both, so a warp streams them together)
//   gu_sb [I][2][H/G]  scale | bias << 16 per group, same row order
//   d_q   [H][I/c]     down rows
//   d_sb  [H][I/G]     scale | bias << 16
// Region offsets are 256-byte aligned, the blob stride 4 KiB aligned.
#include "moe_internal.cuh"

namespace moe {

static uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

BlobLayout make_blob_layout(int H, int I, int G, int bits) {
  BlobLayout L{};
  const int cpw = 32 / bits;  // codes per word
  uint64_t off = 0;
  L.gu_q = off;
  off = align_up(off + (uint64_t)I * 2 * (H / cpw) * 4, 256);
  L.gu_sb = off;
  off = align_up(off + (uint64_t)I * 2 * (H / G) * 4, 256);
  L.d_q = off;
  off = align_up(off + (uint64_t)H * (I / cpw) * 4, 256);
  L.d_sb = off;
  off = align_up(off + (uint64_t)H * (I / G) * 4, 256);
  L.stride = align_up(off, 4096);
  return L;
}

// One thread per output word of the four regions of expert `blockIdx.y`.
__global__ void repack_kernel(const uint32_t* __restrict__ gq, const uint16_t* __restrict__ gs,
                              const uint16_t* __restrict__ gb, const uint32_t* __restrict__ uq,
                              const uint16_t* __restrict__ us, const uint16_t* __restrict__ ub,
                              const uint32_t* __restrict__ dq, const uint16_t* __restrict__ ds,
                              const uint16_t* __restrict__ db, int H, int I, int G, int bits,
                              uint8_t* __restrict__ blobs, BlobLayout L) {
  const int64_t e = blockIdx.y;
  const int64_t cpw = 32 / bits;
  const int64_t wq = (int64_t)H / cpw, wg = (int64_t)H / G;  // words per gate/up row
  const int64_t dw = (int64_t)I / cpw, dg = (int64_t)I / G;  // words per down row
  const int64_t n_guq = (int64_t)I * 2 * wq, n_gusb = (int64_t)I * 2 * wg;
  const int64_t n_dq = (int64_t)H * dw, n_dsb = (int64_t)H * dg;
  uint8_t* blob = blobs + (uint64_t)e * L.stride;
  uint32_t* o_guq = (uint32_t*)(blob + L.gu_q);
  uint32_t* o_gusb = (uint32_t*)(blob + L.gu_sb);
  uint32_t* o_dq = (uint32_t*)(blob + L.d_q);
  uint32_t* o_dsb = (uint32_t*)(blob + L.d_sb);
  const int64_t total = n_guq + n_gusb + n_dq + n_dsb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < n_guq) {
      int64_t row = i / wq, c = i % wq, f = row >> 1;
      const uint32_t* src = (row & 1) ? uq : gq;
      o_guq[i] = src[(e * I + f) * wq + c];
    } else if (i < n_guq + n_gusb) {
      int64_t j = i - n_guq, row = j / wg, c = j % wg, f = row >> 1;
      const uint16_t* s = (row & 1) ? us : gs;
      const uint16_t* b = (row & 1) ? ub : gb;
      int64_t src = (e * I + f) * wg + c;
      o_gusb[j] = (uint32_t)s[src] | ((uint32_t)b[src] << 16);
    } else if (i < n_guq + n_gusb + n_dq) {
      int64_t j = i - n_guq - n_gusb;
      o_dq[j] = dq[e * n_dq + j];
    } else {
      int64_t j = i - n_guq - n_gusb - n_dq;
      o_dsb[j] = (uint32_t)ds[e * n_dsb + j] | ((uint32_t)db[e * n_dsb + j] << 16);
    }
  }
}

__global__ void unpack_kernel(const uint8_t* __restrict__ blob, int H, int I, int G, int bits,
                              BlobLayout L, uint32_t* gq, uint16_t* gs, uint16_t* gb, uint32_t* uq,
                              uint16_t* us, uint16_t* ub, uint32_t* dq, uint16_t* ds,
                              uint16_t* db) {
  const int64_t cpw = 32 / bits;
  const int64_t wq = (int64_t)H / cpw, wg = (int64_t)H / G;
  const int64_t dw = (int64_t)I / cpw, dg = (int64_t)I / G;
  const int64_t n_guq = (int64_t)I * 2 * wq, n_gusb = (int64_t)I * 2 * wg;
  const int64_t n_dq = (int64_t)H * dw, n_dsb = (int64_t)H * dg;
  const uint32_t* guq = (const uint32_t*)(blob + L.gu_q);
  const uint32_t* gusb = (const uint32_t*)(blob + L.gu_sb);
  const uint32_t* dqq = (const uint32_t*)(blob + L.d_q);
  const uint32_t* dsb = (const uint32_t*)(blob + L.d_sb);
  const int64_t total = n_guq + n_gusb + n_dq + n_dsb;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < n_guq) {
      int64_t row = i / wq, c = i % wq, f = row >> 1;
      ((row & 1) ? uq : gq)[f * wq + c] = guq[i];
    } else if (i < n_guq + n_gusb) {
      int64_t j = i - n_guq, row = j / wg, c = j % wg, f = row >> 1;
      uint32_t v = gusb[j];
      ((row & 1) ? us : gs)[f * wg + c] = (uint16_t)(v & 0xFFFF);
      ((row & 1) ? ub : gb)[f * wg + c] = (uint16_t)(v >> 16);
    } else if (i < n_guq + n_gusb + n_dq) {
      int64_t j = i - n_guq - n_gusb;
      dq[j] = dqq[j];
    } else {
      int64_t j = i - n_guq - n_gusb - n_dq;
      uint32_t v = dsb[j];
      ds[j] = (uint16_t)(v & 0xFFFF);
      db[j] = (uint16_t)(v >> 16);
    }
  }
}

cudaError_t launch_repack_expert(const uint32_t* gq, const uint16_t* gs, const uint16_t* gb,
                                 const uint32_t* uq, const uint16_t* us, const uint16_t* ub,
                                 const uint32_t* dq, const uint16_t* ds, const uint16_t* db,
                                 int n, int H, int I, int G, int bits, uint8_t* blobs,
                                 const BlobLayout& L, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  dim3 grid(256, n);
  repack_kernel<<<grid, 256, 0, st>>>(gq, gs, gb, uq, us, ub, dq, ds, db, H, I, G, bits, blobs,
                                      L);
  return cudaGetLastError();
}

cudaError_t launch_unpack_expert(const uint8_t* blob, int H, int I, int G, int bits,
                                 const BlobLayout& L, uint32_t* gq, uint16_t* gs, uint16_t* gb,
                                 uint32_t* uq, uint16_t* us, uint16_t* ub, uint32_t* dq,
                                 uint16_t* ds, uint16_t* db, cudaStream_t st) {
  unpack_kernel<<<256, 256, 0, st>>>(blob, H, I, G, bits, L, gq, gs, gb, uq, us, ub, dq, ds, db);
  return cudaGetLastError();
}

}  // namespace moe
