// api.cu -- the C ABI declared in include/moe.h: argument checks, device
// memory, weight loading/repacking and the launch sequence of moe_forward.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "moe_internal.cuh"

using namespace moe;

struct moe_ctx {
  Ctx c;
};

struct moe_stack {
  int device = -1;
  Dims d{};
  int L = 0;
  int num_sms = 0;
  int n_slots_min = 1 << 30;  // smallest n_slots over the layers
  float eps = 1e-6f;
  int test_flags = 0;
  void* base = nullptr;       // one device allocation: descriptors, workspace, error word
  DecLayer* layers = nullptr;  // [L]
  DecWorkspace ws{};
  int32_t* err = nullptr;
  unsigned long long* stamps = nullptr;  // phase timestamps (instrumented builds only)
};

namespace {

thread_local char g_create_msg[512];

int set_msg(moe_ctx* ctx, int code, const char* fmt, ...) {
  char* buf = ctx ? ctx->c.msg : g_create_msg;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, 512, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(moe_ctx* ctx, cudaError_t e, const char* what) {
  const int code = (e == cudaErrorMemoryAllocation) ? MOE_ERR_OOM : MOE_ERR_CUDA;
  return set_msg(ctx, code, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) == cudaSuccess && prev != dev && dev >= 0) {
      changed = cudaSetDevice(dev) == cudaSuccess;
    }
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

template <typename T>
void free_dev(T*& p) {
  if (p) cudaFree(p);
  p = nullptr;
}

void free_pool(Ctx& c) {
  if (c.pl.store) cudaFreeHost(c.pl.store);
  if (c.pl.dev) cudaFree(c.pl.dev);
  c.pl = PoolState{};
}

void free_weights(Ctx& c) {
  free_pool(c);
  free_dev(c.router_w);
  free_dev(c.router_bias);
  free_dev(c.shared_gate_w);
  free_dev(c.pool);
  free_dev(c.shared);
  c.n_slots = 0;
  c.weight_bytes = 0;
}

void free_workspace(Ctx& c) {
  if (c.ws_base) cudaFree(c.ws_base);
  c.ws_base = nullptr;
  c.ws_bytes = 0;
  c.ws = Workspace{};
  c.err = nullptr;
  c.max_T = 0;
  c.dec_layer = nullptr;
  c.dec_ws = DecWorkspace{};
  c.dec_ok = 0;
}

// The descriptor of this layer for the persistent decode kernel (host copy;
// false if a TMA map could not be encoded).
bool fill_decode_layer(const Ctx& c, DecLayer& D) {
  D = DecLayer{};
  D.router_w = c.router_w;
  D.prior = c.router_bias;
  D.shared_gate_w = c.shared_gate_w;
  D.norm_w = nullptr;
  D.pool = c.pool;
  D.shared_blob = c.shared;
  D.wmax = c.dec_wmax;
  D.pmax = c.dec_pmax;
  D.stride = c.ex.stride;
  D.gu_q = c.ex.gu_q;
  D.gu_sb = c.ex.gu_sb;
  D.d_q = c.ex.d_q;
  D.d_sb = c.ex.d_sb;
  D.n_slots = c.n_slots;
  return decode_encode_maps(c.d, c.pool, c.ex, c.n_slots, c.shared, c.sh, &D);
}

// The descriptor the persistent decode kernel reads for this layer (written
// once the weights and the workspace both exist).
cudaError_t refresh_decode_layer(Ctx& c) {
  if (!c.pool || !c.dec_layer || !c.dec_ok) return cudaSuccess;
  DecLayer D;
  if (!fill_decode_layer(c, D)) return cudaErrorInvalidValue;
  return cudaMemcpy(c.dec_layer, &D, sizeof D, cudaMemcpyHostToDevice);
}

uint64_t align256(uint64_t v) { return (v + 255) & ~uint64_t(255); }

bool qm_ok(const moe_qmatrix& m) { return m.q && m.s && m.b; }

// Sizes in bytes of one canonical expert's nine arrays.
struct CanonSizes {
  size_t gq, gsb, dq, dsb;  // q words of gate (= up), s (= b) of gate, q of down, s of down
};
CanonSizes canon_sizes(int H, int I, int G, int bits) {
  CanonSizes s;
  const int cpw = 32 / bits;  // codes per packed word
  s.gq = (size_t)I * (H / cpw) * 4;
  s.gsb = (size_t)I * (H / G) * 2;
  s.dq = (size_t)H * (I / cpw) * 4;
  s.dsb = (size_t)H * (I / G) * 2;
  return s;
}

// Copy `n` experts starting at index e0 of the canonical arrays (host or
// device) into blobs[0..n), staging host data through device memory.
int load_experts(moe_ctx* ctx, const moe_qmatrix& g, const moe_qmatrix& u, const moe_qmatrix& d,
                 int e0, int n, int on_device, int H, int I, int G, int bits, uint8_t* blobs,
                 const BlobLayout& L, cudaStream_t st) {
  const CanonSizes cs = canon_sizes(H, I, G, bits);
  if (on_device) {
    cudaError_t e = launch_repack_expert(
        g.q + (size_t)e0 * cs.gq / 4, g.s + (size_t)e0 * cs.gsb / 2, g.b + (size_t)e0 * cs.gsb / 2,
        u.q + (size_t)e0 * cs.gq / 4, u.s + (size_t)e0 * cs.gsb / 2, u.b + (size_t)e0 * cs.gsb / 2,
        d.q + (size_t)e0 * cs.dq / 4, d.s + (size_t)e0 * cs.dsb / 2, d.b + (size_t)e0 * cs.dsb / 2,
        n, H, I, G, bits, blobs, L, st);
    if (e != cudaSuccess) return cuda_fail(ctx, e, "repack");
    return MOE_OK;
  }
  const size_t per = 2 * cs.gq + 4 * cs.gsb + cs.dq + 2 * cs.dsb;
  const int chunk = (int)((256ull << 20) / per > 0 ? (256ull << 20) / per : 1);
  uint8_t* stage = nullptr;
  const int cap = chunk < n ? chunk : n;
  cudaError_t e = cudaMalloc(&stage, per * (size_t)cap);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "staging allocation");
  int rc = MOE_OK;
  for (int s0 = 0; s0 < n && rc == MOE_OK; s0 += cap) {
    const int m = (n - s0) < cap ? (n - s0) : cap;
    const size_t E0 = (size_t)(e0 + s0);
    uint8_t* p = stage;
    auto put = [&](const void* src, size_t bytes_each) -> uint8_t* {
      uint8_t* dst = p;
      const size_t bytes = bytes_each * m;
      if (cudaMemcpyAsync(dst, (const uint8_t*)src + E0 * bytes_each, bytes,
                          cudaMemcpyHostToDevice, st) != cudaSuccess)
        rc = MOE_ERR_CUDA;
      p += bytes;
      return dst;
    };
    uint8_t* gq = put(g.q, cs.gq);
    uint8_t* gs = put(g.s, cs.gsb);
    uint8_t* gb = put(g.b, cs.gsb);
    uint8_t* uq = put(u.q, cs.gq);
    uint8_t* us = put(u.s, cs.gsb);
    uint8_t* ub = put(u.b, cs.gsb);
    uint8_t* dq = put(d.q, cs.dq);
    uint8_t* ds = put(d.s, cs.dsb);
    uint8_t* db = put(d.b, cs.dsb);
    if (rc != MOE_OK) {
      rc = set_msg(ctx, MOE_ERR_CUDA, "host-to-device copy of expert weights failed");
      break;
    }
    e = launch_repack_expert((uint32_t*)gq, (uint16_t*)gs, (uint16_t*)gb, (uint32_t*)uq,
                             (uint16_t*)us, (uint16_t*)ub, (uint32_t*)dq, (uint16_t*)ds,
                             (uint16_t*)db, m, H, I, G, bits, blobs + (size_t)s0 * L.stride, L,
                             st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) rc = cuda_fail(ctx, e, "repack");
  }
  cudaFree(stage);
  return rc;
}

}  // namespace

namespace moe {
// Message of a context-free entry point, read back by moe_last_error(NULL).
int set_global_msg(int code, const char* text) {
  snprintf(g_create_msg, sizeof(g_create_msg), "%s", text);
  return code;
}
}  // namespace moe

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_NOT_LOADED: return "weights not loaded";
    case MOE_ERR_NOT_RESERVED: return "workspace not reserved for this many tokens";
    case MOE_ERR_SLOT: return "a selected expert has no valid slot";
    case MOE_ERR_TIMEOUT: return "a bounded device wait expired";
    case MOE_ERR_UNSUPPORTED: return "unsupported sizes";
    default: return "unknown status";
  }
}

const char* moe_last_error(const moe_ctx* ctx) { return ctx ? ctx->c.msg : g_create_msg; }

int moe_create(int E, int k, int hidden, int inter, int shared_inter, int group, moe_ctx** out) {
  return moe_create_quant(E, k, hidden, inter, shared_inter, group, 4, out);
}

int moe_create_quant(int E, int k, int hidden, int inter, int shared_inter, int group, int bits,
                     moe_ctx** out) {
  if (!out) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (bits != 4 && bits != 8)
    return set_msg(nullptr, MOE_ERR_UNSUPPORTED, "bits=%d not in {4, 8}", bits);
  if (E < 1 || E > kMaxE) return set_msg(nullptr, MOE_ERR_UNSUPPORTED, "E=%d not in [1, %d]", E, kMaxE);
  if (k < 1 || k > E || k > kMaxK)
    return set_msg(nullptr, MOE_ERR_INVALID_ARG, "k=%d not in [1, min(E, %d)]", k, kMaxK);
  if (group != 32 && group != 64 && group != 128)
    return set_msg(nullptr, MOE_ERR_UNSUPPORTED, "group=%d not in {32, 64, 128}", group);
  if (!hidden_supported(hidden))
    return set_msg(nullptr, MOE_ERR_UNSUPPORTED,
                   "hidden=%d not in {256, 512, 1024, 2048, 4096, 8192}", hidden);
  if (inter < group || inter > kMaxInter || inter % group != 0 || shared_inter < group ||
      shared_inter > kMaxInter || shared_inter % group != 0)
    return set_msg(nullptr, MOE_ERR_UNSUPPORTED,
                   "inter=%d / shared_inter=%d must be multiples of group=%d in [group, %d]", inter,
                   shared_inter, group, kMaxInter);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_msg(nullptr, MOE_ERR_CUDA, "no CUDA device: %s", cudaGetErrorString(e));
  moe_ctx* ctx = new (std::nothrow) moe_ctx();
  if (!ctx) return set_msg(nullptr, MOE_ERR_OOM, "host allocation failed");
  ctx->c.device = dev;
  ctx->c.d = Dims{E, k, hidden, inter, shared_inter, group, bits};
  ctx->c.ex = make_blob_layout(hidden, inter, group, bits);
  ctx->c.sh = make_blob_layout(hidden, shared_inter, group, bits);
  *out = ctx;
  return MOE_OK;
}

int moe_load_weights(moe_ctx* ctx, const moe_weights* w, int n_slots, void* stream) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (!w) return set_msg(ctx, MOE_ERR_INVALID_ARG, "weights is NULL");
  if (n_slots < 1 || n_slots > 65536)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "n_slots=%d not in [1, 65536]", n_slots);
  if (!w->router_w || !w->shared_gate_w || !qm_ok(w->shared_gate) || !qm_ok(w->shared_up) ||
      !qm_ok(w->shared_down) || !qm_ok(w->gate) || !qm_ok(w->up) || !qm_ok(w->down))
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "a weight pointer is NULL");
  DeviceGuard guard(ctx->c.device);
  Ctx& c = ctx->c;
  const Dims& d = c.d;
  cudaStream_t st = (cudaStream_t)stream;
  cudaStreamSynchronize(st);
  free_weights(c);
  cudaError_t e;
  const size_t rw_bytes = (size_t)d.E * d.H * 2;
  if ((e = cudaMalloc(&c.router_w, rw_bytes)) != cudaSuccess) return cuda_fail(ctx, e, "router alloc");
  if ((e = cudaMalloc(&c.shared_gate_w, (size_t)d.H * 2)) != cudaSuccess)
    return cuda_fail(ctx, e, "shared gate alloc");
  if (w->router_bias && (e = cudaMalloc(&c.router_bias, (size_t)d.E * 4)) != cudaSuccess)
    return cuda_fail(ctx, e, "prior alloc");
  if ((e = cudaMalloc(&c.pool, (size_t)n_slots * c.ex.stride)) != cudaSuccess) {
    free_weights(c);
    return cuda_fail(ctx, e, "expert pool alloc");
  }
  if ((e = cudaMalloc(&c.shared, c.sh.stride)) != cudaSuccess) {
    free_weights(c);
    return cuda_fail(ctx, e, "shared expert alloc");
  }
  const cudaMemcpyKind kind = w->on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
  e = cudaMemcpyAsync(c.router_w, w->router_w, rw_bytes, kind, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c.shared_gate_w, w->shared_gate_w, (size_t)d.H * 2, kind, st);
  if (e == cudaSuccess && w->router_bias)
    e = cudaMemcpyAsync(c.router_bias, w->router_bias, (size_t)d.E * 4, kind, st);
  if (e != cudaSuccess) {
    free_weights(c);
    return cuda_fail(ctx, e, "router copy");
  }
  int rc = load_experts(ctx, w->gate, w->up, w->down, 0, n_slots, w->on_device, d.H, d.I, d.G,
                        d.bits, c.pool, c.ex, st);
  if (rc == MOE_OK) {  // the decode kernel's bound constants, kept on the host
    float* tmp = nullptr;
    float hv[2] = {0.f, 0.f};
    e = cudaMalloc(&tmp, 2 * sizeof(float));
    if (e == cudaSuccess) e = decode_router_consts(c.router_w, c.router_bias, d.E, d.H, tmp, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(hv, tmp, sizeof hv, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (tmp) cudaFree(tmp);
    if (e != cudaSuccess) rc = cuda_fail(ctx, e, "router bound constants");
    c.dec_wmax = hv[0];
    c.dec_pmax = hv[1];
  }
  if (rc == MOE_OK)
    rc = load_experts(ctx, w->shared_gate, w->shared_up, w->shared_down, 0, 1, w->on_device, d.H,
                      d.Is, d.G, d.bits, c.shared, c.sh, st);
  if (rc == MOE_OK && (e = cudaStreamSynchronize(st)) != cudaSuccess) rc = cuda_fail(ctx, e, "load");
  if (rc != MOE_OK) {
    free_weights(c);
    return rc;
  }
  c.n_slots = n_slots;
  if ((e = refresh_decode_layer(c)) != cudaSuccess) return cuda_fail(ctx, e, "decode descriptor");
  c.weight_bytes = (int64_t)rw_bytes + d.H * 2 + (w->router_bias ? d.E * 4 : 0) +
                   (int64_t)n_slots * c.ex.stride + (int64_t)c.sh.stride;
  return MOE_OK;
}

int moe_reserve(moe_ctx* ctx, int max_T) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (max_T < 1 || max_T > (1 << 20))
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "max_T=%d not in [1, 2^20]", max_T);
  DeviceGuard guard(ctx->c.device);
  Ctx& c = ctx->c;
  const Dims& d = c.d;
  cudaDeviceSynchronize();
  free_workspace(c);
  const uint64_t P = (uint64_t)max_T * d.k;
  const uint64_t rows = P + max_T;
  const int maxI = d.I > d.Is ? d.I : d.Is;
  const uint64_t nblk = (P + 2047) / 2048;
  uint64_t off = 0;
  auto take = [&](uint64_t bytes) {
    const uint64_t o = off;
    off = align256(off + bytes);
    return o;
  };
  const uint64_t o_logits = take((uint64_t)max_T * d.E * 4);
  const uint64_t o_bound = take((uint64_t)max_T * d.E * 4);
  const uint64_t o_gz = take((uint64_t)max_T * 4);
  const uint64_t o_gate = take((uint64_t)max_T * 4);
  const uint64_t o_xnorm = take((uint64_t)max_T * 4);
  const uint64_t o_wnorm = take((uint64_t)d.E * 4);
  int n_sms = 0;
  if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, c.device) != cudaSuccess)
    n_sms = 160;
  const uint64_t o_rpart = take((uint64_t)tile_router_part_floats(n_sms) * 4);
  const uint64_t o_perm = take(P * 4);
  const uint64_t o_inv = take(P * 4);
  const uint64_t o_off = take((uint64_t)(d.E + 1) * 4);
  const uint64_t o_used = take((uint64_t)d.E * 4);
  const uint64_t o_nused = take(4);
  const uint64_t o_hist = take(nblk * d.E * 4);
  const uint64_t o_h = take(rows * maxI * 4);
  const uint64_t o_o = take(rows * d.H * 4);
  const uint64_t o_err = take(4);
  const uint64_t o_bar = take(kSyncWords * 8);
  const uint64_t o_rstats = take(8);
  const uint64_t o_rcnt = take(16);
  const uint64_t o_rovf = take(router_tc_overflow_bytes(d, max_T) + 16);
  const uint64_t o_tiles = take((uint64_t)prefill_max_tiles(d, max_T) * 16);
  const uint64_t o_ntiles = take(4);
  const uint64_t o_dlayer = take(sizeof(DecLayer));
  const uint64_t o_dws = take(decode_workspace_bytes(d, n_sms));
  uint8_t* base = nullptr;
  cudaError_t e = cudaMalloc(&base, off);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "workspace alloc");
  e = cudaMemset(base, 0, off);
  if (e != cudaSuccess) {
    cudaFree(base);
    return cuda_fail(ctx, e, "workspace clear");
  }
  c.ws_base = base;
  c.ws_bytes = (int64_t)off;
  c.ws.logits = (float*)(base + o_logits);
  c.ws.bound = (float*)(base + o_bound);
  c.ws.gate_z = (float*)(base + o_gz);
  c.ws.gate = (float*)(base + o_gate);
  c.ws.xnorm = (float*)(base + o_xnorm);
  c.ws.wnorm = (float*)(base + o_wnorm);
  c.ws.rpart = (float*)(base + o_rpart);
  c.ws.perm = (int32_t*)(base + o_perm);
  c.ws.inv = (int32_t*)(base + o_inv);
  c.ws.offsets = (int32_t*)(base + o_off);
  c.ws.used = (int32_t*)(base + o_used);
  c.ws.n_used = (int32_t*)(base + o_nused);
  c.ws.hist = (int32_t*)(base + o_hist);
  c.ws.h = (float*)(base + o_h);
  c.ws.o = (float*)(base + o_o);
  c.err = (int32_t*)(base + o_err);
  c.ws.bar = (unsigned long long*)(base + o_bar);
  c.ws.rstats = (uint32_t*)(base + o_rstats);
  c.ws.rcnt = (unsigned long long*)(base + o_rcnt);
  c.ws.rovf = base + o_rovf;
  c.ws.tiles = base + o_tiles;
  c.ws.n_tiles = (int32_t*)(base + o_ntiles);
  c.dec_layer = (DecLayer*)(base + o_dlayer);
#ifdef MOE_DECODE_STAMPS
  cudaMalloc(&c.dec_stamps, (size_t)n_sms * 32 * 8);
  cudaMemset(c.dec_stamps, 0, (size_t)n_sms * 32 * 8);
#endif
  decode_workspace_carve(d, n_sms, base + o_dws, &c.dec_ws);
  c.max_T = max_T;
  if ((e = cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, c.device)) !=
      cudaSuccess) {
    free_workspace(c);
    return cuda_fail(ctx, e, "device attributes");
  }
  if ((e = prepare_router(c)) != cudaSuccess || (e = prepare_general_experts(c)) != cudaSuccess ||
      (e = prepare_fused_decode(c)) != cudaSuccess ||
      (e = decode_prepare(d, c.num_sms, false, &c.dec_ok)) != cudaSuccess ||
      (e = refresh_decode_layer(c)) != cudaSuccess || (e = prepare_batch_decode(c)) != cudaSuccess ||
      (prefill_supported(d) && (e = prepare_prefill(c)) != cudaSuccess)) {
    free_workspace(c);
    return cuda_fail(ctx, e, "kernel attributes");
  }
  return MOE_OK;
}

int moe_forward(moe_ctx* ctx, const void* x, int T, const int32_t* expert_slot_table, void* y,
                int32_t* topk_idx, float* topk_w, int32_t* perm, int32_t* offsets, void* stream) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  Ctx& c = ctx->c;
  c.last_launches = 0;
  if (T < 0) return set_msg(ctx, MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (T == 0) return MOE_OK;
  if (!c.pool) return set_msg(ctx, MOE_ERR_NOT_LOADED, "moe_load_weights has not been called");
  if (!c.ws_base) return set_msg(ctx, MOE_ERR_NOT_RESERVED, "moe_reserve has not been called");
  if (T > c.max_T) return set_msg(ctx, MOE_ERR_NOT_RESERVED, "T=%d > reserved max_T=%d", T, c.max_T);
  if (!x || !y || !topk_idx || !topk_w)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "x, y, topk_idx and topk_w must be non-NULL");
  if (c.pl.slots && expert_slot_table)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "the slot pool keeps its own table: pass NULL");
  if (!c.pl.slots && !expert_slot_table && c.n_slots < c.d.E)
    return set_msg(ctx, MOE_ERR_INVALID_ARG,
                   "identity slot table needs n_slots (%d) >= E (%d)", c.n_slots, c.d.E);
  if (c.pl.slots) expert_slot_table = c.pl.table;
  if (((uintptr_t)x & 15) != 0)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  const size_t xb = (size_t)T * c.d.H * 2;
  const uint8_t* xp = (const uint8_t*)x;
  const uint8_t* yp = (const uint8_t*)y;
  if (xp < yp + xb && yp < xp + xb) return set_msg(ctx, MOE_ERR_INVALID_ARG, "x and y overlap");
  DeviceGuard guard(c.device);
  cudaStream_t st = (cudaStream_t)stream;
  FwdArgs a{(const uint16_t*)x, T, expert_slot_table, (uint16_t*)y, topk_idx, topk_w, perm, offsets};
  int launches = 0;
  // the slot pool updates the table between routing and the experts: not in
  // the single-launch decode kernels
  const bool fused_ok = T == 1 && !c.pl.slots && (c.dec_ok || fused_decode_supported(c));
  // 2..64 tokens: the batched decode kernels (weights streamed once per used
  // expert, its tokens in the MMA's columns)
  const bool bdec_ok = T >= 2 && batch_decode_supported(c, T);
  const bool prefill_ok = prefill_supported(c.d);
  if (c.path == MOE_PATH_DECODE && !fused_ok && !bdec_ok)
    return set_msg(ctx, MOE_ERR_UNSUPPORTED,
                   "the decode path needs T <= 64, no slot pool and supported sizes");
  if (c.path == MOE_PATH_PREFILL && !prefill_ok)
    return set_msg(ctx, MOE_ERR_UNSUPPORTED,
                   "the prefill path needs hidden and 2*inter multiples of 128");
  // measured on GB300: from two tokens on, the grouped GEMMs beat the general
  // CUDA-core kernels (at T = 64 by 30x), so AUTO uses them whenever the sizes allow
  // (AUTO keeps the grouped GEMMs for T >= 2 until the batched kernels beat them)
  const bool use_bdec = bdec_ok && c.path == MOE_PATH_DECODE;
  const bool use_prefill = !use_bdec && (c.path == MOE_PATH_PREFILL ||
                                         (c.path == MOE_PATH_AUTO && prefill_ok && T > 1));
  cudaError_t e;
  record_mark(c, MOE_MARK_START, st);
  if (fused_ok && c.dec_ok && c.path == MOE_PATH_DECODE) {
    DecLaunch p{};
    p.layers = c.dec_layer;
    p.L = 1;
    p.x = a.x;
    p.y = a.y;
    p.topk_idx = a.topk_idx;
    p.topk_w = a.topk_w;
    p.perm = a.perm_out;
    p.offsets = a.offsets_out;
    p.tables = a.table;
    p.ws = c.dec_ws;
    p.err = c.err;
    p.timeout_hook = (c.test_flags & MOE_TEST_WAIT_TIMEOUT) != 0;
    p.cooperative = c.cooperative;
#ifdef MOE_DECODE_STAMPS
    p.stamps = c.dec_stamps;
#endif
    ++launches;
    e = decode_launch(c.d, c.num_sms, p, st);
  } else if (fused_ok && (c.path == MOE_PATH_AUTO || c.path == MOE_PATH_DECODE ||
                          c.path == kPathFusedV1)) {
    e = launch_fused_decode(c, a, st, &launches);
  } else {
    if (T <= 64 && small_route_supported(c, T)) {
      // up to 64 tokens: logits, exact top-k and the shared gate in one launch
      e = launch_small_route(c, a, st, &launches);
    } else if (use_bdec) {  // logits, exact top-k and the shared gate in two launches
      e = launch_batch_route(c, a, st, &launches);
    } else {
      e = launch_router(c, a, st, &launches);
      record_mark(c, MOE_MARK_LOGITS, st);
      if (e == cudaSuccess) e = launch_topk(c, a, st, &launches);
    }
    if (e == cudaSuccess && c.pl.slots) e = launch_pool_update(c, a.topk_idx, T * c.d.k, st, &launches);
    record_mark(c, MOE_MARK_ROUTED, st);
    bool tiles_built = false;
    if (e == cudaSuccess) e = launch_permute(c, a, st, &launches, use_prefill, &tiles_built);
    if (e == cudaSuccess && use_prefill)
      e = launch_prefill_plan(c, a, st, &launches, tiles_built);
    record_mark(c, MOE_MARK_PERMUTED, st);
    if (e == cudaSuccess)
      e = use_bdec      ? launch_batch_decode(c, a, st, &launches)
          : use_prefill ? launch_prefill_experts(c, a, st, &launches)
                        : launch_general_experts(c, a, st, &launches);
  }
  record_mark(c, MOE_MARK_END, st);
  c.last_launches = launches;
  if (e != cudaSuccess) return cuda_fail(ctx, e, "moe_forward launch");
  return MOE_OK;
}

int moe_get_status(moe_ctx* ctx, void* stream) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  DeviceGuard guard(ctx->c.device);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "stream synchronise");
  if (!ctx->c.err) return MOE_OK;
  int32_t v = 0;
  e = cudaMemcpy(&v, ctx->c.err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "status read");
  if (v != 0) {
    cudaMemset(ctx->c.err, 0, 4);
    // a timed-out grid barrier leaves its counter off the multiple of the
    // grid size that every barrier expects: start it afresh
    if (ctx->c.ws.bar) cudaMemset(ctx->c.ws.bar, 0, kSyncWords * 8);
    // the persistent decode kernel's exchanges: launch counters and arrival
    // counters back to zero together (a launch reads both afresh, so CUDA
    // graphs captured earlier replay correctly after the reset)
    if (ctx->c.dec_ws.seq) decode_workspace_reset(ctx->c.num_sms, ctx->c.dec_ws);
    return set_msg(ctx, v, "device reported: %s", moe_status_string(v));
  }
  return MOE_OK;
}

int moe_read_expert(moe_ctx* ctx, int slot, uint32_t* gate_q, uint16_t* gate_s, uint16_t* gate_b,
                    uint32_t* up_q, uint16_t* up_s, uint16_t* up_b, uint32_t* down_q,
                    uint16_t* down_s, uint16_t* down_b) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  Ctx& c = ctx->c;
  if (!c.pool) return set_msg(ctx, MOE_ERR_NOT_LOADED, "no weights loaded");
  if (slot < -1 || slot >= c.n_slots)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "slot=%d not in [-1, %d)", slot, c.n_slots);
  if (!gate_q || !gate_s || !gate_b || !up_q || !up_s || !up_b || !down_q || !down_s || !down_b)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "an output pointer is NULL");
  DeviceGuard guard(c.device);
  const int I = slot < 0 ? c.d.Is : c.d.I;
  const BlobLayout& L = slot < 0 ? c.sh : c.ex;
  const uint8_t* blob = slot < 0 ? c.shared : c.pool + (uint64_t)slot * L.stride;
  const CanonSizes cs = canon_sizes(c.d.H, I, c.d.G, c.d.bits);
  const size_t total = 2 * cs.gq + 4 * cs.gsb + cs.dq + 2 * cs.dsb;
  uint8_t* stage = nullptr;
  cudaError_t e = cudaMalloc(&stage, total);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "staging alloc");
  uint8_t* p = stage;
  uint8_t* dgq = p; p += cs.gq;
  uint8_t* dgs = p; p += cs.gsb;
  uint8_t* dgb = p; p += cs.gsb;
  uint8_t* duq = p; p += cs.gq;
  uint8_t* dus = p; p += cs.gsb;
  uint8_t* dub = p; p += cs.gsb;
  uint8_t* ddq = p; p += cs.dq;
  uint8_t* dds = p; p += cs.dsb;
  uint8_t* ddb = p;
  e = launch_unpack_expert(blob, c.d.H, I, c.d.G, c.d.bits, L, (uint32_t*)dgq, (uint16_t*)dgs,
                           (uint16_t*)dgb, (uint32_t*)duq, (uint16_t*)dus, (uint16_t*)dub,
                           (uint32_t*)ddq, (uint16_t*)dds, (uint16_t*)ddb, 0);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  struct {
    void* dst;
    const void* src;
    size_t n;
  } cp[9] = {{gate_q, dgq, cs.gq}, {gate_s, dgs, cs.gsb}, {gate_b, dgb, cs.gsb},
             {up_q, duq, cs.gq},   {up_s, dus, cs.gsb},   {up_b, dub, cs.gsb},
             {down_q, ddq, cs.dq}, {down_s, dds, cs.dsb}, {down_b, ddb, cs.dsb}};
  for (int i = 0; i < 9 && e == cudaSuccess; ++i)
    e = cudaMemcpy(cp[i].dst, cp[i].src, cp[i].n, cudaMemcpyDeviceToHost);
  cudaFree(stage);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "read back");
  return MOE_OK;
}

int moe_set_path(moe_ctx* ctx, int path) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (path < MOE_PATH_AUTO || path > kPathFusedV1)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "path=%d unknown", path);
  ctx->c.path = path;
  return MOE_OK;
}

int moe_set_test_flags(moe_ctx* ctx, int flags) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (flags & ~MOE_TEST_WAIT_TIMEOUT)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "unknown test flag %d", flags);
  ctx->c.test_flags = flags;
  return MOE_OK;
}

int moe_set_stage_events(moe_ctx* ctx, void* const* events, int n_events) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  if (n_events < 0 || n_events > MOE_MARK_COUNT || (n_events > 0 && !events))
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "n_events=%d not in [0, %d] or events NULL",
                   n_events, (int)MOE_MARK_COUNT);
  Ctx& c = ctx->c;
  for (int i = 0; i < MOE_MARK_COUNT; ++i)
    c.marks[i] = i < n_events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
  c.n_marks = n_events;
  return MOE_OK;
}

int64_t moe_expert_blob_bytes(const moe_ctx* ctx) { return ctx ? (int64_t)ctx->c.ex.stride : 0; }

int64_t moe_device_bytes(const moe_ctx* ctx) {
  return ctx ? ctx->c.weight_bytes + ctx->c.ws_bytes : 0;
}

int moe_last_launch_count(const moe_ctx* ctx) { return ctx ? ctx->c.last_launches : 0; }

void moe_destroy(moe_ctx* ctx) {
  if (!ctx) return;
  {
    DeviceGuard guard(ctx->c.device);
    cudaDeviceSynchronize();
    free_weights(ctx->c);
    free_workspace(ctx->c);
  }
  delete ctx;
}

int moe_pool_enable(moe_ctx* ctx, int slots) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  Ctx& c = ctx->c;
  const int E = c.d.E;
  if (!c.pool) return set_msg(ctx, MOE_ERR_NOT_LOADED, "moe_load_weights has not been called");
  if (c.pl.slots) return set_msg(ctx, MOE_ERR_INVALID_ARG, "the slot pool is already enabled");
  if (c.n_slots < E)
    return set_msg(ctx, MOE_ERR_INVALID_ARG,
                   "the pool takes its store from the loaded experts: n_slots (%d) must be >= E (%d)",
                   c.n_slots, E);
  if (slots < 1 || slots >= E || slots > 65534)
    return set_msg(ctx, MOE_ERR_INVALID_ARG, "slots=%d not in [1, min(E - 1, 65534)]", slots);
  DeviceGuard guard(c.device);
  cudaDeviceSynchronize();
  const size_t blob = c.ex.stride, store_bytes = (size_t)E * blob;
  PoolState p{};
  p.slots = slots;
  cudaError_t e = cudaHostAlloc(&p.store, store_bytes, cudaHostAllocMapped);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "pinned expert store");
  void* dptr = nullptr;
  e = cudaHostGetDevicePointer(&dptr, p.store, 0);
  if (e == cudaSuccess) e = cudaMemcpy(p.store, c.pool, store_bytes, cudaMemcpyDeviceToHost);
  const size_t arr = align256((uint64_t)E * 4) * 3 + align256((uint64_t)slots * 4) * 3 + 256;
  if (e == cudaSuccess) e = cudaMalloc(&p.dev, arr);
  uint8_t* newpool = nullptr;
  if (e == cudaSuccess) e = cudaMalloc(&newpool, (size_t)slots * blob);
  if (e != cudaSuccess) {
    if (newpool) cudaFree(newpool);
    c.pl = p;
    free_pool(c);
    return cuda_fail(ctx, e, "slot pool");
  }
  p.store_dev = (const uint8_t*)dptr;
  uint8_t* b = (uint8_t*)p.dev;
  size_t o = 0;
  auto take = [&](size_t n) {
    uint8_t* r = b + o;
    o += align256(n);
    return r;
  };
  p.table = (int32_t*)take((size_t)E * 4);
  p.fill_expert = (int32_t*)take((size_t)E * 4);
  p.fill_slot = (int32_t*)take((size_t)E * 4);
  p.owner = (int32_t*)take((size_t)slots * 4);
  p.freq = (uint32_t*)take((size_t)slots * 4);
  p.last = (uint32_t*)take((size_t)slots * 4);
  p.state = (uint32_t*)take(8 * 4);
  e = cudaMemset(p.dev, 0, arr);
  if (e == cudaSuccess) e = cudaMemset(p.table, 0xFF, (size_t)E * 4);  // every expert unmapped
  if (e == cudaSuccess) e = cudaMemset(p.owner, 0xFF, (size_t)slots * 4);  // every slot empty
  if (e != cudaSuccess) {
    cudaFree(newpool);
    c.pl = p;
    free_pool(c);
    return cuda_fail(ctx, e, "slot pool init");
  }
  cudaFree(c.pool);
  c.pool = newpool;
  c.n_slots = slots;
  c.pl = p;
  c.weight_bytes -= (int64_t)(E - slots) * (int64_t)blob;
  // the persistent decode kernel is not used with a pool (it reads no table
  // updated between its phases); its descriptor would name the old pool
  c.dec_ok = 0;
  return MOE_OK;
}

int moe_pool_stats(moe_ctx* ctx, int64_t* out) {
  if (!ctx || !out) return set_msg(ctx, MOE_ERR_INVALID_ARG, "ctx or out is NULL");
  Ctx& c = ctx->c;
  if (!c.pl.slots) return set_msg(ctx, MOE_ERR_INVALID_ARG, "no slot pool (moe_pool_enable)");
  DeviceGuard guard(c.device);
  uint32_t v[8];
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(v, c.pl.state, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "slot pool stats");
  for (int i = 0; i < 5; ++i) out[i] = (int64_t)v[i];
  return MOE_OK;
}

int moe_pool_table(moe_ctx* ctx, int32_t* table_out) {
  if (!ctx || !table_out) return set_msg(ctx, MOE_ERR_INVALID_ARG, "ctx or table_out is NULL");
  Ctx& c = ctx->c;
  if (!c.pl.slots) return set_msg(ctx, MOE_ERR_INVALID_ARG, "no slot pool (moe_pool_enable)");
  DeviceGuard guard(c.device);
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess)
    e = cudaMemcpy(table_out, c.pl.table, (size_t)c.d.E * 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "slot pool table");
  return MOE_OK;
}

int moe_router_check_stats(moe_ctx* ctx, float* max_error_ratio, int* fallback_tokens) {
  if (!ctx) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "ctx is NULL");
  Ctx& c = ctx->c;
  if (!c.ws.rstats) return set_msg(ctx, MOE_ERR_NOT_RESERVED, "moe_reserve has not been called");
  DeviceGuard guard(c.device);
  uint32_t v[2] = {0, 0};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(v, c.ws.rstats, 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(c.ws.rstats, 0, 8);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "router check stats");
  float r;
  std::memcpy(&r, &v[0], 4);
  if (max_error_ratio) *max_error_ratio = r;
  if (fallback_tokens) *fallback_tokens = (int)v[1];
  return MOE_OK;
}

// ---------------------------------------------------------------- stacks
// moe_stack_*: L layers of one shape run for one token by a single
// cooperative launch of the persistent decode kernel.

int moe_stack_create(moe_ctx* const* layers, int L, const uint16_t* const* norm_w, float eps,
                     moe_stack** out) {
  if (!out) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!layers || L < 1 || L > MOE_STACK_MAX_LAYERS)
    return set_msg(nullptr, MOE_ERR_INVALID_ARG, "layers is NULL or L=%d not in [1, %d]", L,
                   MOE_STACK_MAX_LAYERS);
  if (!(eps > 0.f) || !(eps < 1.f))
    return set_msg(nullptr, MOE_ERR_INVALID_ARG, "eps must lie in (0, 1)");
  for (int l = 0; l < L; ++l) {
    if (!layers[l]) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "layers[%d] is NULL", l);
    const Ctx& c = layers[l]->c;
    if (!c.pool) return set_msg(nullptr, MOE_ERR_NOT_LOADED, "layers[%d] has no weights", l);
    if (c.pl.slots)
      return set_msg(nullptr, MOE_ERR_INVALID_ARG, "layers[%d] has a slot pool (not in stacks)", l);
    const Dims& a = layers[0]->c.d;
    if (c.d.E != a.E || c.d.k != a.k || c.d.H != a.H || c.d.I != a.I || c.d.Is != a.Is ||
        c.d.G != a.G || c.device != layers[0]->c.device)
      return set_msg(nullptr, MOE_ERR_INVALID_ARG,
                     "layers[%d] differs from layers[0] in shape or device", l);
    if (norm_w && norm_w[l] && ((uintptr_t)norm_w[l] & 15) != 0)
      return set_msg(nullptr, MOE_ERR_INVALID_ARG, "norm_w[%d] must be 16-byte aligned", l);
  }
  const Ctx& c0 = layers[0]->c;
  DeviceGuard guard(c0.device);
  int nC = 0;
  cudaError_t e = cudaDeviceGetAttribute(&nC, cudaDevAttrMultiProcessorCount, c0.device);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "device attributes");
  int ok = 0;
  if ((e = decode_prepare(c0.d, nC, true, &ok)) != cudaSuccess)
    return cuda_fail(nullptr, e, "kernel attributes");
  if (!ok)
    return set_msg(nullptr, MOE_ERR_UNSUPPORTED,
                   "the persistent decode kernel does not fit these sizes (hidden %d, inter %d, "
                   "shared_inter %d, E %d, k %d)",
                   c0.d.H, c0.d.I, c0.d.Is, c0.d.E, c0.d.k);
  moe_stack* s = new (std::nothrow) moe_stack;
  if (!s) return set_msg(nullptr, MOE_ERR_OOM, "host allocation");
  s->device = c0.device;
  s->d = c0.d;
  s->L = L;
  s->num_sms = nC;
  s->eps = eps;
  for (int l = 0; l < L; ++l) s->n_slots_min = std::min(s->n_slots_min, layers[l]->c.n_slots);
  const size_t b_layers = align256((uint64_t)L * sizeof(DecLayer));
  const size_t b_ws = decode_workspace_bytes(c0.d, nC);
  e = cudaMalloc(&s->base, b_layers + b_ws + 256);
  if (e != cudaSuccess) {
    delete s;
    return cuda_fail(nullptr, e, "stack workspace");
  }
  uint8_t* base = (uint8_t*)s->base;
  s->layers = (DecLayer*)base;
  decode_workspace_carve(c0.d, nC, base + b_layers, &s->ws);
  s->err = (int32_t*)(base + b_layers + b_ws);
  DecLayer* host = new (std::nothrow) DecLayer[L];
  bool good = host != nullptr;
  for (int l = 0; good && l < L; ++l) {
    good = fill_decode_layer(layers[l]->c, host[l]);
    host[l].norm_w = norm_w ? norm_w[l] : nullptr;
  }
  if (good) {
    e = cudaMemset(s->base, 0, b_layers + b_ws + 256);
    if (e == cudaSuccess) e = cudaMemcpy(s->layers, host, (size_t)L * sizeof(DecLayer),
                                         cudaMemcpyHostToDevice);
  }
  delete[] host;
  if (!good || e != cudaSuccess) {
    cudaFree(s->base);
    delete s;
    return good ? cuda_fail(nullptr, e, "stack descriptors")
                : set_msg(nullptr, MOE_ERR_CUDA, "TMA descriptor encoding failed");
  }
#ifdef MOE_DECODE_STAMPS
  cudaMalloc(&s->stamps, (size_t)L * nC * 32 * 8);
  cudaMemset(s->stamps, 0, (size_t)L * nC * 32 * 8);
#endif
  *out = s;
  return MOE_OK;
}

int moe_stack_forward(moe_stack* s, const void* x, const int32_t* expert_slot_tables, void* x_out,
                      void* y, void* xn, int32_t* topk_idx, float* topk_w, void* stream) {
  if (!s) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "stack is NULL");
  if (!x || !topk_idx || !topk_w)
    return set_msg(nullptr, MOE_ERR_INVALID_ARG, "x, topk_idx and topk_w must be non-NULL");
  if (((uintptr_t)x & 15) != 0 || ((uintptr_t)x_out & 15) != 0 || ((uintptr_t)y & 15) != 0 ||
      ((uintptr_t)xn & 15) != 0)
    return set_msg(nullptr, MOE_ERR_INVALID_ARG, "x, x_out, y and xn must be 16-byte aligned");
  if (!expert_slot_tables && s->n_slots_min < s->d.E)
    return set_msg(nullptr, MOE_ERR_INVALID_ARG,
                   "identity slot tables need n_slots (%d) >= E (%d) in every layer",
                   s->n_slots_min, s->d.E);
  DeviceGuard guard(s->device);
  DecLaunch p{};
  p.layers = s->layers;
  p.L = s->L;
  p.x = (const uint16_t*)x;
  p.x_out = (uint16_t*)x_out;
  p.y = (uint16_t*)y;
  p.xn_out = (uint16_t*)xn;
  p.topk_idx = topk_idx;
  p.topk_w = topk_w;
  p.tables = expert_slot_tables;
  p.chain = 1;
  p.eps = s->eps;
  p.ws = s->ws;
  p.err = s->err;
  p.timeout_hook = s->test_flags & MOE_TEST_WAIT_TIMEOUT;
  p.stamps = s->stamps;
  // every CTA of the grid exchanges data with every other: the cooperative
  // attribute makes the launch fail rather than start with CTAs not resident
  p.cooperative = true;
  const cudaError_t e = decode_launch(s->d, s->num_sms, p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "moe_stack_forward launch");
  return MOE_OK;
}

int moe_stack_get_status(moe_stack* s, void* stream) {
  if (!s) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "stack is NULL");
  DeviceGuard guard(s->device);
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "stream synchronise");
  int32_t v = 0;
  e = cudaMemcpy(&v, s->err, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "status read");
  if (v != 0) {
    cudaMemset(s->err, 0, 4);
    decode_workspace_reset(s->num_sms, s->ws);
    return set_msg(nullptr, v, "device reported: %s", moe_status_string(v));
  }
  return MOE_OK;
}

int moe_stack_set_test_flags(moe_stack* s, int flags) {
  if (!s) return set_msg(nullptr, MOE_ERR_INVALID_ARG, "stack is NULL");
  if (flags & ~MOE_TEST_WAIT_TIMEOUT)
    return set_msg(nullptr, MOE_ERR_INVALID_ARG, "unknown test flags 0x%x", flags);
  s->test_flags = flags;
  return MOE_OK;
}

void moe_stack_destroy(moe_stack* s) {
  if (!s) return;
  {
    DeviceGuard guard(s->device);
    cudaDeviceSynchronize();
    if (s->base) cudaFree(s->base);
    if (s->stamps) cudaFree(s->stamps);
  }
  delete s;
}

}  // extern "C"

#ifdef MOE_DECODE_STAMPS
extern "C" int moe_debug_stack_stamps(moe_stack* s, unsigned long long* host, int n) {
  if (!s || !s->stamps) return MOE_ERR_INVALID_ARG;
  return cudaMemcpy(host, s->stamps, (size_t)n * 8, cudaMemcpyDeviceToHost) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
// Instrumented builds only: the per-CTA phase timestamps of the last decode
// launch ([CTA][32] SM cycle counts) and the launch attribute knob.
extern "C" int moe_debug_decode_stamps(moe_ctx* ctx, unsigned long long* host, int n) {
  if (!ctx || !ctx->c.dec_stamps) return MOE_ERR_INVALID_ARG;
  return cudaMemcpy(host, ctx->c.dec_stamps, (size_t)n * 8, cudaMemcpyDeviceToHost) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
extern "C" int moe_debug_set_cooperative(moe_ctx* ctx, int on) {
  if (!ctx) return MOE_ERR_INVALID_ARG;
  ctx->c.cooperative = on != 0;
  return MOE_OK;
}
#endif
