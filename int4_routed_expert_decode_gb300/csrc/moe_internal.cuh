// moe_internal.cuh -- shared declarations of the CUDA library (host + device).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxH = 8192;
constexpr int kMaxInter = 4096;
constexpr int kSyncWords = 1;  // counters of the fused decode kernel
// hidden sizes the router kernels are instantiated for: 256 * 2^j up to kMaxH
inline bool hidden_supported(int H) {
  return H >= 256 && H <= kMaxH && H % 256 == 0 && ((H / 256) & (H / 256 - 1)) == 0;
}
constexpr int kTileRouterMinT = 16;  // from this many tokens the router is a tiled GEMM
constexpr int kPathFusedV1 = 4;  // the earlier barrier-based fused decode kernel (comparison)
// Floats of the router's slice sums: the slices are only used while
// slices x tiles <= 2 x SMs, and a tile covers 64 x 128 logits.
inline int64_t tile_router_part_floats(int num_sms) { return (int64_t)2 * num_sms * 64 * 128; }

// Byte offsets of the four regions of one expert blob.  Layout of a blob
// (all words uint32, offsets 256-byte aligned, 64-bit throughout):
//   gu_q  [I][2][H/8]   row 2i = gate row i, row 2i+1 = up row i (packed codes)
//   gu_sb [I][2][H/G]   (bf16 scale) | (bf16 bias) << 16, same row order
//   d_q   [H][I/8]      down rows
//   d_sb  [H][I/G]
struct BlobLayout {
  uint64_t gu_q, gu_sb, d_q, d_sb, stride;
};

// bits: code width (4 or 8), 32/bits codes per packed word.
BlobLayout make_blob_layout(int H, int I, int G, int bits);

struct Dims {
  int E, k, H, I, Is, G;
  int bits = 4;  // expert code width: 4 (every path) or 8 (the general path)
};

// cuTensorMapEncodeTiled, reached through the runtime (null if unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled();

// ---- persistent decode kernel (decode.cu): one token, one launch per layer
// or per stack of layers chained through RMSNorm and a residual add.
// Per-layer resident weights and constants, read by the kernel from device
// memory (and copied into shared memory with each layer's prologue).
struct alignas(64) DecLayer {
  // 4-D TMA maps of the packed codes {bytes of a 128-byte column block, row,
  // column block, slot} (128-byte swizzle; rows under 128 bytes are one
  // unswizzled block), one box per copy landing as [column block][row][bytes]:
  // routed gate/up 2I rows of H/2 bytes, box 8 rows; routed down H rows of
  // I/2 bytes, box 16 rows; the shared expert's the same with one slot
  CUtensorMap map_gu, map_d, map_sgu, map_sd;
  // the same gate/up maps with boxes of half the column blocks (batched decode)
  CUtensorMap map_guh, map_sguh;
  const uint16_t* router_w;       // [E][H]
  const float* prior;             // [E] or null
  const uint16_t* shared_gate_w;  // [H]
  const uint16_t* norm_w;         // [H] or null (stacks)
  const uint8_t* pool;            // routed blobs
  const uint8_t* shared_blob;     // the shared expert (same layout: inter == shared_inter)
  uint64_t stride, gu_q, gu_sb, d_q, d_sb;
  int n_slots;
  float wmax, pmax;  // max_e |Wr_e|_2 and max_e |prior_e|, rounded up
};
// Exchange state of one decode launch sequence (zeroed once, never reset:
// the counters only grow).
struct DecWorkspace {
  uint32_t* seq;             // [CTAs] launch counters
  unsigned long long* cnt;   // logits, h and residual counters, 128 bytes apart
  float* lt;                 // [E] logits
  float* ht;                 // [(k + 1) I] SwiGLU activations (shared expert last)
  uint16_t* xt;              // [H] residual (stacks)
};

// Workspace carved out of one allocation by moe_reserve.
struct Workspace {
  float* logits;      // [max_T][E]  fp32 router logits
  float* bound;       // [max_T][E]  rigorous bound on their rounding error
  float* gate_z;      // [max_T]     x . wsg (shared gate pre-activation)
  float* gate;        // [max_T]     sigmoid(x . wsg)
  float* xnorm;       // [max_T]     upper bound of |x_t|_2 (many-token router)
  float* wnorm;       // [E]         upper bound of |Wr_e|_2
  float* rpart;       // many-token router: slice sums [slices][T][E]
  int32_t* perm;      // [max_T*k]   pair ids sorted by expert
  int32_t* inv;       // [max_T*k]   position of pair p in perm
  int32_t* offsets;   // [E+1]
  int32_t* used;      // [E]         experts with at least one pair, ascending
  int32_t* n_used;    // [1]
  int32_t* hist;      // [nblk][E]   per-block expert counts (large T)
  float* h;           // [max_T*k + max_T][maxI] fp32 SwiGLU activations
  float* o;           // [max_T*k + max_T][H]    fp32 expert outputs
  unsigned long long* bar;  // fused kernel: grid-barrier arrival counter (monotonic)
  uint32_t* rstats;   // tensor-core router check: [0] max observed error / (|x| max|Wr|)
                      // (float bits), [1] tokens that fell back to certifying every expert
  unsigned long long* rcnt;  // small-T routing: grid-barrier arrivals (monotonic)
  uint8_t* rovf;      // tensor-core router: per-token overflow of the candidate selection
  void* tiles;        // [max tiles] prefill work tiles (16 bytes each)
  int32_t* n_tiles;   // [1]
};

// Bounded slot pool (pool.cu): every expert blob in pinned, device-mapped
// host memory, `slots` of them resident in the device pool.
struct PoolState {
  int slots = 0;                  // 0: no pool (the caller's table or the identity)
  uint8_t* store = nullptr;       // host: E blobs (cudaHostAlloc, mapped)
  const uint8_t* store_dev = nullptr;  // its device address
  void* dev = nullptr;            // one device allocation for the arrays below
  int32_t* table = nullptr;       // [E] expert -> slot or -1
  int32_t* owner = nullptr;       // [slots] slot -> expert or -1
  uint32_t* freq = nullptr;       // [slots]
  uint32_t* last = nullptr;       // [slots]
  uint32_t* state = nullptr;      // [8] step, hits, misses, evictions, overflows, last fills
  int32_t* fill_expert = nullptr; // [E]
  int32_t* fill_slot = nullptr;   // [E]
};

struct Ctx {
  int device = -1;
  Dims d{};
  int n_slots = 0;
  int path = MOE_PATH_AUTO;
  // resident weights
  uint16_t* router_w = nullptr;       // [E][H]
  float* router_bias = nullptr;       // [E] or null
  uint16_t* shared_gate_w = nullptr;  // [H]
  uint8_t* pool = nullptr;            // n_slots routed blobs
  BlobLayout ex{};
  uint8_t* shared = nullptr;          // one blob (inner size Is)
  BlobLayout sh{};
  int64_t weight_bytes = 0;
  // workspace
  int max_T = 0;
  void* ws_base = nullptr;
  int64_t ws_bytes = 0;
  Workspace ws{};
  int32_t* err = nullptr;             // sticky device error word
  int num_sms = 0;                    // multiprocessors of the device
  int fused_ctas = 0;                 // CTAs of the fused decode kernel (0: unavailable)
  float dec_wmax = 0.f, dec_pmax = 0.f;  // router bound constants (with the weights)
  DecLayer* dec_layer = nullptr;      // this layer's descriptor (in the workspace)
  DecWorkspace dec_ws{};              // decode exchange state (in the workspace)
  int dec_ok = 0;                     // the persistent decode kernel fits these shapes
  // Launch a single layer with the cooperative attribute?  Measured: it keeps
  // the next launch from starting until this one has fully drained (about
  // 2.5 us per layer), so single-layer launches go without it (stacks use it).
  bool cooperative = false;
  unsigned long long* dec_stamps = nullptr;  // phase timestamps (instrumented builds only)
  PoolState pl{};                     // bounded slot pool (moe_pool_enable)
  int test_flags = 0;                 // MOE_TEST_* hooks
  cudaEvent_t marks[MOE_MARK_COUNT] = {};  // borrowed stage events (moe_set_stage_events)
  int n_marks = 0;
  int last_launches = 0;
  char msg[512] = {0};
};

// ---- kernels' host launchers (return cudaError_t of the last launch) ----
cudaError_t launch_repack_expert(const uint32_t* gq, const uint16_t* gs, const uint16_t* gb,
                                 const uint32_t* uq, const uint16_t* us, const uint16_t* ub,
                                 const uint32_t* dq, const uint16_t* ds, const uint16_t* db,
                                 int n, int H, int I, int G, int bits, uint8_t* blobs,
                                 const BlobLayout& L, cudaStream_t st);
cudaError_t launch_unpack_expert(const uint8_t* blob, int H, int I, int G, int bits,
                                 const BlobLayout& L,
                                 uint32_t* gq, uint16_t* gs, uint16_t* gb, uint32_t* uq,
                                 uint16_t* us, uint16_t* ub, uint32_t* dq, uint16_t* ds,
                                 uint16_t* db, cudaStream_t st);

cudaError_t launch_pool_update(const Ctx& c, const int32_t* topk_idx, int P, cudaStream_t st,
                               int* launches);
struct FwdArgs;
// Batched decode (batch_decode.cu): 2 <= T <= 64 tokens, after routing and the permutation.
bool batch_decode_supported(const Ctx& c, int T);
cudaError_t prepare_batch_decode(const Ctx& c);
cudaError_t launch_batch_route(const Ctx& c, const FwdArgs& f, cudaStream_t st, int* launches);
// Routing of 2..64 tokens (logits, exact top-k, weights, shared gate) in one
// cooperative launch, for hidden <= 2048.
bool small_route_supported(const Ctx& c, int T);
cudaError_t launch_small_route(const Ctx& c, const FwdArgs& f, cudaStream_t st, int* launches);
cudaError_t launch_batch_decode(const Ctx& c, const FwdArgs& f, cudaStream_t st, int* launches);

struct FwdArgs {
  const uint16_t* x;
  int T;
  const int32_t* table;
  uint16_t* y;
  int32_t* topk_idx;
  float* topk_w;
  int32_t* perm_out;     // may be null
  int32_t* offsets_out;  // may be null
};

// One-time kernel attributes (dynamic shared memory limits); called by
// moe_reserve so that moe_forward makes no such call (graph capture).
cudaError_t prepare_router(const Ctx& c);
cudaError_t prepare_general_experts(const Ctx& c);

// Fused single-launch decode (T = 1): availability, one-time set-up, launch.
bool fused_decode_supported(const Ctx& c);
cudaError_t prepare_fused_decode(Ctx& c);
cudaError_t launch_fused_decode(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches);

// ---- persistent decode kernel (decode.cu), continued
struct DecLaunch {
  const DecLayer* layers;
  int L;
  const uint16_t* x;
  uint16_t* x_out;
  uint16_t* y;
  uint16_t* xn_out;  // [L][H] block inputs (after the RMSNorm), or null
  int32_t* topk_idx;
  float* topk_w;
  int32_t* perm;
  int32_t* offsets;
  const int32_t* tables;
  int chain;
  float eps;
  DecWorkspace ws;
  int32_t* err;
  int timeout_hook;
  unsigned long long* stamps;
  bool cooperative;
};
bool decode_shape_ok(const Dims& d);
bool decode_fits(const Dims& d, int nC, bool chain);
cudaError_t decode_prepare(const Dims& d, int nC, bool chain, int* ok);
size_t decode_workspace_bytes(const Dims& d, int nC);
void decode_workspace_carve(const Dims& d, int nC, uint8_t* base, DecWorkspace* w);
// Zero the launch and arrival counters (synchronous; nothing may be in flight).
void decode_workspace_reset(int nC, const DecWorkspace& w);
cudaError_t decode_router_consts(const uint16_t* router_w, const float* prior, int E, int H,
                                 float* out, cudaStream_t st);
// The four TMA maps of a layer's descriptor (host-side encoding).
bool decode_encode_maps(const Dims& d, const uint8_t* pool, const BlobLayout& ex, int n_slots,
                        const uint8_t* shared, const BlobLayout& sh, DecLayer* D);
cudaError_t decode_launch(const Dims& d, int nC, const DecLaunch& p, cudaStream_t st);

// Tensor-core grouped GEMM path for many tokens: availability, workspace
// size (tiles for max_T tokens), one-time set-up, launch (after router, top-k
// and permutation).
bool prefill_supported(const Dims& d);
int prefill_max_tiles(const Dims& d, int max_T);
cudaError_t prepare_prefill(const Ctx& c);
// The grouped GEMMs' tile list (unless the permutation already built it) and
// a cleared y accumulator.
cudaError_t launch_prefill_plan(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches,
                                bool tiles_built);
cudaError_t launch_prefill_experts(const Ctx& c, const FwdArgs& a, cudaStream_t st,
                                   int* launches);

// Router for many tokens: approximate logits on the tensor cores, then
// certified logits of each token's candidates and the exact selection.
bool router_tc_supported(const Dims& d, int T);
// Workspace bytes for the candidate selection's per-token overflow (0 when the
// router is never used for up to max_T tokens).
size_t router_tc_overflow_bytes(const Dims& d, int max_T);
cudaError_t prepare_router_tc();
cudaError_t launch_router_tc(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches);
cudaError_t launch_router_candidates(const Ctx& c, const FwdArgs& a, cudaStream_t st,
                                     int* launches);

cudaError_t launch_router(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches);
cudaError_t launch_topk(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches);
// with_tiles: also build the grouped GEMMs' tile list when the one-CTA
// permutation runs (then *tiles_built is set).
cudaError_t launch_permute(const Ctx& c, const FwdArgs& a, cudaStream_t st, int* launches,
                           bool with_tiles, bool* tiles_built);
cudaError_t launch_general_experts(const Ctx& c, const FwdArgs& a, cudaStream_t st,
                                   int* launches);

// Record stage event `m` on `st` if the caller set one (moe_set_stage_events).
inline void record_mark(const Ctx& c, int m, cudaStream_t st) {
  if (m < c.n_marks && c.marks[m]) cudaEventRecord(c.marks[m], st);
}

// Set the message returned by moe_last_error(NULL); returns `code`.
int set_global_msg(int code, const char* text);

}  // namespace moe
