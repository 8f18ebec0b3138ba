/*
 * moe.h -- C ABI of the int4 routed-expert MoE block for GB300 (sm_103a).
 *
 * The block is the sparse Mixture-of-Experts layer of the Qwen3-Next /
 * Qwen3.5-3.6 hybrid decoders described in the Swiftlet project README
 * ("Show HN: Run an 80B Qwen in 4.3 GB of RAM on a Mac and a 35B on an
 * iPhone", wpnews), section "How it works": each layer routes every token to
 * k of E experts (8 of 256 for Qwen3.6-35B-A3B, 10 of 512 for
 * Qwen3-Next-80B-A3B), keeps a shared expert resident, and stores the experts
 * in MLX's affine int4 group quantisation, addressed with 64-bit byte
 * offsets (same README, its list of what was built).  For every token t:
 *
 *   l[t,e]  = x_t . Wr_e (+ prior_e)                        router
 *   idx, w  = top-k of softmax(l[t,:]) (descending, ties -> lowest e),
 *             renormalised to sum to one                     routing
 *   p       = t*k + j, stable counting sort by idx[t,j]      permutation
 *   o[t,j]  = Wd (silu(Wg x_t) * (Wu x_t)), W = s*q + b      routed experts
 *   y_t     = sum_j w[t,j] o[t,j] + sigmoid(x_t . wsg) S(x_t)  combine
 *
 * where S is the shared expert (same form, inner size shared_inter) and the
 * int4 codes q are grouped in `group` consecutive inputs sharing one bf16
 * scale s and bias b.  Expert selection ranks the exact real values of the
 * logits (bf16 x bf16 products summed without rounding), so the selected
 * indices do not depend on any summation order.
 *
 * Conventions
 *   - bf16 tensors are passed as uint16_t bit patterns.
 *   - Packed int4: code 8c+j of a row is bits 4j..4j+3 of uint32 word c;
 *     packed int8 (moe_create_quant with bits = 8): code 4c+j is bits
 *     8j..8j+7 of word c.
 *   - Every function returns a moe_status (0 = MOE_OK, negative = error);
 *     moe_last_error(ctx) gives a one-line message.  Nothing here throws,
 *     aborts or prints.
 *   - A context is bound to the CUDA device that is current at moe_create;
 *     all later calls must be made with that device current.
 *   - Device pointers are plain CUDA device addresses; `stream` is a
 *     cudaStream_t (NULL = legacy default stream).
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* a size, pointer or option is out of range       */
  MOE_ERR_CUDA = -2,         /* a CUDA runtime call failed (message has details)  */
  MOE_ERR_OOM = -3,          /* device memory could not be allocated             */
  MOE_ERR_NOT_LOADED = -4,   /* moe_forward before moe_load_weights              */
  MOE_ERR_NOT_RESERVED = -5, /* moe_forward before moe_reserve, or T > max_T     */
  MOE_ERR_SLOT = -6,         /* device: a selected expert maps to no valid slot  */
  MOE_ERR_TIMEOUT = -7,      /* device: a bounded wait inside a kernel expired   */
  MOE_ERR_UNSUPPORTED = -8   /* sizes outside what the kernels were built for    */
} moe_status;

typedef struct moe_ctx moe_ctx;

/* One int4 matrix [rows][cols] in MLX affine layout:
 *   q  uint32 [rows][cols/8]      packed codes
 *   s  bf16   [rows][cols/group]  scales
 *   b  bf16   [rows][cols/group]  biases            w = s*q + b
 * For a stack of matrices the arrays carry one more leading dimension. */
typedef struct moe_qmatrix {
  const uint32_t* q;
  const uint16_t* s;
  const uint16_t* b;
} moe_qmatrix;

/* Canonical weights of one MoE layer.  With on_device = 1 every pointer is a
 * device address, with 0 a host address.  E, H = hidden, I = inter,
 * Is = shared_inter, n = n_slots.
 *   router_w       bf16 [E][H]
 *   router_bias    fp32 [E], or NULL (no additive prior on the logits)
 *   shared_gate_w  bf16 [H]   (sigmoid gate of the shared expert)
 *   shared_gate, shared_up   [Is][H] int4 (leading dim 1 allowed, ignored)
 *   shared_down              [H][Is] int4
 *   gate, up                 [n][I][H] int4, slot-major
 *   down                     [n][H][I] int4, slot-major                    */
typedef struct moe_weights {
  int on_device;
  const uint16_t* router_w;
  const float* router_bias;
  const uint16_t* shared_gate_w;
  moe_qmatrix shared_gate, shared_up, shared_down;
  moe_qmatrix gate, up, down;
} moe_weights;

/* Create a context for one MoE layer (the sparse block of a decoder layer:
 * routed experts, a resident shared expert; README "How it works").
 *   E in [1, 1024]; k in [1, min(E, 32)]; hidden in {256, 512, 1024, 2048,
 *   4096, 8192}; inter and shared_inter multiples of group, at most 4096;
 *   group in {32, 64, 128}.  Nothing is allocated on the device yet.
 * Errors: MOE_ERR_INVALID_ARG for k or a NULL `out`; MOE_ERR_UNSUPPORTED for
 * E, hidden, inter, shared_inter or group outside those sets; MOE_ERR_CUDA if
 * no device is current. */
int moe_create(int E, int k, int hidden, int inter, int shared_inter, int group, moe_ctx** out);

/* As moe_create, with the experts' code width `bits` in {4, 8} (the pages'
 * MLX affine quantisation comes in int4 and int8 widths: README, its list of
 * what was built).  bits = 4 is moe_create.  With bits = 8 the packed words
 * of every moe_qmatrix hold 4 codes (code 4c+j of a row is bits 8j..8j+7 of
 * word c, low byte first), q is uint32 [rows][cols/4], w = s*q + b with q in
 * [0, 255]; such a context runs the general CUDA-core path for every T (the
 * decode, batched and grouped-GEMM kernels and stacks are int4 only:
 * MOE_PATH_DECODE and MOE_PATH_PREFILL return MOE_ERR_UNSUPPORTED and
 * moe_stack_create refuses it).  Errors: as moe_create, and
 * MOE_ERR_UNSUPPORTED for another `bits`. */
int moe_create_quant(int E, int k, int hidden, int inter, int shared_inter, int group, int bits,
                     moe_ctx** out);

/* Copy and repack the weights into library-owned device memory (on the pages
 * the routed experts sit in a container of equal-stride records, one per
 * expert, README "How it works"; MLX affine int4 layout per its list of
 * what was built): the routed experts become n_slots fixed-stride blobs (slot s holds the s-th expert of
 * `w`, 64-bit byte offsets), the router, prior, shared gate vector and shared
 * expert stay resident beside them.  Synchronous: when it returns the caller
 * may free or reuse every buffer of `w`.  May be called again to replace the
 * weights (the previous ones are freed).  n_slots in [1, 65536].
 * Errors: INVALID_ARG (null pointers, n_slots), OOM, CUDA. */
int moe_load_weights(moe_ctx* ctx, const moe_weights* w, int n_slots, void* stream);

/* Size the device workspace for up to max_T tokens per moe_forward call
 * (the pages have no counterpart: it keeps moe_forward free of allocations)
 * (max_T in [1, 1<<20]).  Must be called before moe_forward and before any
 * CUDA-graph capture of it; moe_forward never allocates.  Synchronous.
 * Errors: INVALID_ARG, OOM. */
int moe_reserve(moe_ctx* ctx, int max_T);

/* One pass of the block over T tokens, enqueued on `stream` (asynchronous,
 * no host synchronisation, no allocation: capturable in a CUDA graph): the
 * router, top-k, shared expert and routed experts of README "How it works",
 * with the slot table standing for the pages' bounded expert pool.
 *   x                  bf16 [T][H] device, 16-byte aligned, read only
 *   expert_slot_table  int32 [E] device: slot holding expert e, or NULL for
 *                      the identity (requires n_slots >= E).  A selected
 *                      expert whose slot is negative or >= n_slots makes the
 *                      device record MOE_ERR_SLOT and skip that expert.
 *   y                  bf16 [T][H] device, written
 *   topk_idx           int32 [T][k] device, written: expert ids, descending
 *                      exact logit, ties to the lowest id
 *   topk_w             fp32 [T][k] device, written: renormalised weights
 *   perm               int32 [T*k] device or NULL: pair ids p = t*k+j sorted
 *                      stably by expert
 *   offsets            int32 [E+1] device or NULL: expert e's pairs are
 *                      perm[offsets[e] .. offsets[e+1])
 * T = 0 is a no-op.  x and y must not overlap.
 * Errors (host side, nothing launched): INVALID_ARG, NOT_LOADED,
 * NOT_RESERVED (T > max_T), CUDA (launch failure).  Errors found on the
 * device are sticky and reported by moe_get_status.
 *
 * Co-residency: for T = 1 the single-launch decode kernels run one CTA per
 * SM and exchange data between all of them through counters in device
 * memory.  They are launched without the cooperative attribute (it would
 * keep each layer from overlapping the previous one's tail, about 2.5 us per
 * layer), so they need every SM free of other work while they run: a kernel
 * of another stream, or an MPS client, holding an SM makes the exchange wait
 * out its bound (about one second), the device records MOE_ERR_TIMEOUT and y
 * of that call is not valid.  moe_stack_forward launches cooperatively
 * instead (one launch per token).  The exchange counters only grow and every
 * launch reads them afresh, so a CUDA graph captured around moe_forward keeps
 * replaying correctly; moe_get_status zeroes them after a device error. */
int moe_forward(moe_ctx* ctx, const void* x, int T, const int32_t* expert_slot_table, void* y,
                int32_t* topk_idx, float* topk_w, int32_t* perm, int32_t* offsets, void* stream);

/* Synchronise `stream`, then return and clear the sticky device error word
 * (MOE_OK, MOE_ERR_SLOT or MOE_ERR_TIMEOUT), or MOE_ERR_CUDA if the
 * synchronisation itself failed.  After a device error it also zeroes the
 * decode kernels' exchange counters (synchronously; nothing of this context
 * may be in flight on another stream).  No counterpart on the pages. */
int moe_get_status(moe_ctx* ctx, void* stream);

/* Read slot `slot` (or the shared expert when slot == -1) back from the
 * device pool (MLX affine int4, list of what was built) into host buffers in
 * the canonical layout of moe_weights
 * (gate/up [I][H], down [H][I]; I = shared_inter for the shared expert).
 * Synchronous.  Used to verify the repacking byte for byte. */
int moe_read_expert(moe_ctx* ctx, int slot, uint32_t* gate_q, uint16_t* gate_s, uint16_t* gate_b,
                    uint32_t* up_q, uint16_t* up_s, uint16_t* up_b, uint32_t* down_q,
                    uint16_t* down_s, uint16_t* down_b);

/* Kernel path of moe_forward (an implementation choice; the pages run one
 * Metal shader sequence).  MOE_PATH_AUTO uses the fused single-launch
 * decode kernel for T = 1 when the sizes allow it (hidden in {256, 512,
 * 1024, 2048}, inter == shared_inter <= 1024), the tensor-core grouped GEMMs
 * for T >= 2 when hidden, 2*inter and 2*shared_inter are multiples of 128,
 * and the general kernels otherwise.  MOE_PATH_DECODE insists on the fused
 * kernel and MOE_PATH_PREFILL on the grouped GEMMs (any T >= 1); either
 * returns MOE_ERR_UNSUPPORTED if its sizes do not allow it.
 * MOE_PATH_GENERAL forces the general kernels.  The grouped GEMMs round the
 * dequantised weights and the SwiGLU activations to bf16 (tensor-core
 * operands) and sum the expert outputs with fp32 atomic additions, so their
 * y is not bitwise reproducible from run to run; the routing outputs are. */
enum { MOE_PATH_AUTO = 0, MOE_PATH_DECODE = 1, MOE_PATH_GENERAL = 2, MOE_PATH_PREFILL = 3 };
int moe_set_path(moe_ctx* ctx, int path);

/* Test hooks, off by default (failure injection on the host side of a
 * bounded device wait; no counterpart on the pages).  MOE_TEST_WAIT_TIMEOUT makes the grid
 * barriers of the fused decode kernel wait for one arrival more than the
 * grid has, and the MMA issuer of each grouped-GEMM CTA wait on an mbarrier
 * phase that nothing completes: each bounded wait runs out (about one
 * second), the device records MOE_ERR_TIMEOUT, every role of the CTA leaves
 * its loop, and moe_get_status reports it and resets the barrier counter so
 * that the context stays usable.  flags = 0 turns every hook off. */
enum { MOE_TEST_WAIT_TIMEOUT = 1 };
int moe_set_test_flags(moe_ctx* ctx, int flags);

/* Optional device timing of moe_forward's stages.  `events` holds
 * n_events (<= MOE_MARK_COUNT) cudaEvent_t handles that the caller created
 * with timing enabled.  While they are set, moe_forward records events[m] on
 * its stream at each mark m that its path has:
 *   MOE_MARK_START     before the first launch (every path)
 *   MOE_MARK_LOGITS    router logits written
 *   MOE_MARK_ROUTED    top-k indices and weights written
 *   MOE_MARK_PERMUTED  permutation (and the grouped GEMMs' tile list) done
 *   MOE_MARK_GATEUP    gate/up projections and SwiGLU done
 *   MOE_MARK_DOWN      down projections done
 *   MOE_MARK_END       y written (every path)
 * The fused decode kernel has START and END only.  The handles are borrowed
 * until the next call; n_events = 0 turns the marks off.  Inside a stream
 * capture the records become event-record nodes of the graph.
 * MOE_ERR_INVALID_ARG if n_events is out of range or events is NULL with
 * n_events > 0. */
enum {
  MOE_MARK_START = 0,
  MOE_MARK_LOGITS = 1,
  MOE_MARK_ROUTED = 2,
  MOE_MARK_PERMUTED = 3,
  MOE_MARK_GATEUP = 4,
  MOE_MARK_DOWN = 5,
  MOE_MARK_END = 6,
  MOE_MARK_COUNT = 7
};
int moe_set_stage_events(moe_ctx* ctx, void* const* events, int n_events);

/* Bytes of one routed-expert blob (codes + scales + biases, padded: the
 * pages' fixed-stride blob, README "How it works") and the number of
 * resident device bytes of the context (weights + workspace). */
int64_t moe_expert_blob_bytes(const moe_ctx* ctx);
int64_t moe_device_bytes(const moe_ctx* ctx);

/* Number of kernel launches the last moe_forward enqueued (the pages' decode
 * loop is dispatch bound, README "Status"). */
int moe_last_launch_count(const moe_ctx* ctx);

/* ---------------------------------------------------------------- slot pool
 * The pages keep the routed experts in storage and cache the frequently used
 * ones in a pool of bounded size whose eviction combines use frequency with
 * recency (README "How it works"; creativeainews, "How Expert Streaming
 * Works").  moe_pool_enable moves the
 * loaded experts (n_slots >= E, slot e = expert e) into pinned, device-mapped
 * host memory -- the store, read by the GPU over NVLink-C2C -- and keeps
 * `slots` of them (1 <= slots < E, at most 65534) in the device pool, empty
 * at first.  From then on every moe_forward (expert_slot_table must be NULL)
 * routes, then updates the pool on the stream with no host synchronisation:
 *   - a selected expert in the pool is a hit: its frequency grows by the
 *     number of (token, expert) pairs routed to it, its last use is this call;
 *   - the misses, in ascending expert id, take an empty slot (lowest first),
 *     else evict among the slots this call does not need the one with the
 *     lowest frequency, then the least recent use, then the lowest slot;
 *     the evicted expert leaves the table, the new one is copied in;
 *   - a call that needs more distinct experts than there are slots leaves the
 *     excess unmapped (counted as overflows; the device records MOE_ERR_SLOT
 *     and those experts are skipped).
 * y is the same as with every expert resident.  Calls with a pool use the
 * multi-launch path (router, top-k, pool, permutation, experts), also for
 * T = 1; stacks do not take pooled layers.  Synchronous.
 * Errors: INVALID_ARG (sizes, already enabled, n_slots < E), NOT_LOADED,
 * OOM/CUDA (allocations). */
int moe_pool_enable(moe_ctx* ctx, int slots);

/* Counters since moe_pool_enable, synchronising the device: out[0] calls,
 * out[1] hits, out[2] misses (fills), out[3] evictions, out[4] overflows.
 * The hit rate is hits / (hits + misses). */
int moe_pool_stats(moe_ctx* ctx, int64_t* out);

/* The pool's current table (int32 [E], host): slot of expert e or -1. */
int moe_pool_table(moe_ctx* ctx, int32_t* table_out);

/* The tensor-core router (T >= 128 tokens, E a multiple of 128) filters
 * candidates with a margin d = 2^-10 |x|_2 max_e |Wr_e|_2 + 2^-22 max|prior|
 * around approximate logits and certifies the candidates; a token whose
 * measured approximation error on a candidate exceeds d/8 has every expert
 * certified instead.  This reads (synchronising the device) and resets what
 * the calls since the last read saw: the largest |approximate - certified
 * fp32 logit| over the candidates, divided by |x|_2 max_e |Wr_e|_2, and the
 * number of tokens that fell back.  Either
 * pointer may be NULL.  A diagnostic; the pages have no counterpart.
 * Errors: INVALID_ARG, NOT_RESERVED, CUDA. */
int moe_router_check_stats(moe_ctx* ctx, float* max_error_ratio, int* fallback_tokens);

/* Allocation-free routing: router logits, exact top-k with renormalised
 * weights, and the shared-expert sigmoid gate for T tokens, with no context
 * and no device allocation of any kind.  The pages have no counterpart: this
 * entry point exists for callers that cannot call cudaMalloc -- code whose
 * device memory belongs to a host application's own allocator, code that
 * must not trigger the device synchronisation an allocation can cause, or
 * code that may only enqueue work on streams it is given.
 *   x              bf16 [T][hidden] device, 16-byte aligned
 *   router_w       bf16 [E][hidden] device, 16-byte aligned
 *   router_bias    fp32 [E] device, or NULL (no prior)
 *   shared_gate_w  bf16 [hidden] device, 16-byte aligned
 *   topk_idx       int32 [T][k] device, written (same contract as moe_forward)
 *   topk_w         fp32 [T][k] device, written
 *   shared_gate    fp32 [T] device, written: sigmoid(x_t . shared_gate_w)
 * Sizes: E in [1, 1024], k in [1, min(E, 32)], hidden in {256, 512, 1024,
 * 2048, 4096, 8192}, T in [0, MOE_STATIC_ROUTE_MAX_T] and
 * T*E <= MOE_STATIC_ROUTE_MAX_LOGITS.  A hidden outside that set returns
 * MOE_ERR_UNSUPPORTED; every other size out of range returns
 * MOE_ERR_INVALID_ARG; both leave a message for moe_last_error(NULL) and
 * launch nothing.
 * Scratch: the intermediates live in one file-scope device array of
 * (2 * MOE_STATIC_ROUTE_MAX_LOGITS + MOE_STATIC_ROUTE_MAX_T) floats (1 MiB +
 * 16 KiB), held by every device that loads the library until the process
 * exits.  The first call on a device looks up that array's device address
 * and sets kernel attributes; make it before any stream capture.  Every call
 * shares the one array: calls whose kernels overlap on the GPU (different
 * streams without ordering between them) race and give undefined results;
 * calls in one stream, or otherwise ordered, are safe.  Asynchronous on
 * `stream`. */
#define MOE_STATIC_ROUTE_MAX_LOGITS 131072
#define MOE_STATIC_ROUTE_MAX_T 4096
int moe_route_static(const void* x, int T, const uint16_t* router_w, const float* router_bias,
                     const uint16_t* shared_gate_w, int E, int k, int hidden, int32_t* topk_idx,
                     float* topk_w, float* shared_gate, void* stream);

/* ---------------------------------------------------------------- stacks
 * A stack chains L MoE layers of one shape for ONE token in a single
 * persistent launch, as a decoder runs them one after another (the Swiftlet
 * README on the wpnews page, paragraph "Status": the decode loop is bound by
 * dispatch, not by IO).  There is no attention between the blocks here:
 * layer l's input is the previous residual, normalised, and its output is
 * added back:
 *
 *   n_l     = bf16( x_l / sqrt(mean_h x_l[h]^2 + eps) * norm_w_l )   RMSNorm
 *   y_l     = MoE block of layer l on n_l (as moe_forward, T = 1)
 *   x_{l+1} = bf16( x_l + y_l )                       residual (y_l in bf16)
 *
 * with x_0 the caller's x and x_L the result.  The RMSNorm runs in fp32 (the
 * sum of squares in a fixed order, so results are reproducible bit for bit).
 *
 * The launch is cooperative: all of its CTAs, one per SM, must be resident
 * together, and it fails with MOE_ERR_CUDA rather than start otherwise
 * (other work occupying SMs, MPS limits).  Its CTAs exchange data through
 * counters in the stack's workspace that only grow (each launch reads the
 * launch count afresh), so a CUDA graph captured around moe_stack_forward
 * replays correctly, also after moe_stack_get_status has reset the counters.
 * A stack borrows its layers' weights: destroy it before any of them, and
 * do not reload their weights while it exists.  One stack runs on one
 * stream at a time (its launches must be ordered). */
#define MOE_STACK_MAX_LAYERS 1024
typedef struct moe_stack moe_stack;

/* Create a stack over `layers` [L] (L in [1, MOE_STACK_MAX_LAYERS]), every
 * one created with the same sizes on the same device and already loaded
 * (moe_reserve is not needed).
 *   norm_w  NULL, or L device pointers (16-byte aligned) to bf16 [hidden]
 *           RMSNorm weights; a NULL entry means all ones
 *   eps     RMSNorm epsilon in (0, 1)
 * Errors: INVALID_ARG (pointers, L, eps, mismatched layers), NOT_LOADED,
 * UNSUPPORTED (sizes the persistent kernel does not fit: hidden up to 2048,
 * inter == shared_inter, shared memory), OOM, CUDA.  Messages go to
 * moe_last_error(NULL). */
int moe_stack_create(moe_ctx* const* layers, int L, const uint16_t* const* norm_w, float eps,
                     moe_stack** out);

/* Run the stack for one token (asynchronous on `stream`, no allocation).
 *   x                   bf16 [hidden] device, 16-byte aligned, read
 *   expert_slot_tables  int32 [L][E] device, or NULL for identity tables
 *                       (every layer needs n_slots >= E); as moe_forward
 *   x_out               bf16 [hidden] device, or NULL: x_L; may equal x
 *   y                   bf16 [L][hidden] device, or NULL: every y_l
 *   xn                  bf16 [L][hidden] device, or NULL: every n_l
 *   topk_idx, topk_w    int32 / fp32 [L][k] device, written as moe_forward
 * Errors (host side): INVALID_ARG, CUDA (launch failure, including a grid
 * that cannot be co-resident).  Device errors are sticky: see
 * moe_stack_get_status. */
int moe_stack_forward(moe_stack* s, const void* x, const int32_t* expert_slot_tables, void* x_out,
                      void* y, void* xn, int32_t* topk_idx, float* topk_w, void* stream);

/* As moe_get_status, for the stack's own error word; after a device error it
 * also zeroes the stack's exchange counters (synchronous). */
int moe_stack_get_status(moe_stack* s, void* stream);

/* As moe_set_test_flags: MOE_TEST_WAIT_TIMEOUT makes every layer's logits
 * exchange wait for one arrival more than the grid has. */
int moe_stack_set_test_flags(moe_stack* s, int flags);

/* Free the stack's device memory (synchronises the device).  NULL is a no-op. */
void moe_stack_destroy(moe_stack* s);

/* ---- Gated DeltaNet recurrence --------------------------------------------
 * The linear-attention layers of the same hybrid stack (three quarters of its
 * layers: wpnews page, Swiftlet README, "How it works"; creativeainews page,
 * "How Expert Streaming Works") carry a fixed-size state per value head
 * instead of a KV cache.  The pages print no equations; this call computes
 * the plain gated delta rule, for each value head h and token t:
 *   k^ = k / sqrt(|k|^2 + 1e-6),  q^ = q / sqrt(|q|^2 + 1e-6) / sqrt(dk)
 *   S  = alpha S + beta (v - alpha S k^) k^T,   o = S q^   (S after the update)
 * where value head h reads key head h / (Hv / Hk).  The gates alpha and beta,
 * the short convolution before it and the norm and projection after it belong
 * to the rest of the layer: alpha and beta arrive computed.
 *   q, k    bf16 [B][T][Hk][dk] device, aligned to dk/16 bytes
 *   v       bf16 [B][T][Hv][dv] device
 *   alpha   fp32 [B][T][Hv] device (decay, normally in [0, 1])
 *   beta    fp32 [B][T][Hv] device (write strength, normally in [0, 1])
 *   state   fp32 [B][Hv][dv][dk] device, 16-byte aligned, row i of a head's
 *           state holds its dk columns contiguously; read, then overwritten
 *           with the state after token T-1 (in place)
 *   out     fp32 [B][T][Hv][dv] device, written; must not overlap the inputs
 * B independent sequences of T tokens each (T = 1 is a decode step; T > 1
 * runs the tokens in order, the state kept in registers in between).
 * Sizes: dk in {64, 128, 256} (else MOE_ERR_UNSUPPORTED); B, T >= 0 (either 0:
 * nothing happens); Hk >= 1; Hv a multiple of Hk; dv in [1, 4096];
 * B*Hv*dv <= 2^33.  Other sizes, a NULL or misaligned pointer return
 * MOE_ERR_INVALID_ARG with a message for moe_last_error(NULL) and launch
 * nothing; a launch failure returns MOE_ERR_CUDA.  No context, no allocation;
 * asynchronous on `stream`; calls on different streams over disjoint states
 * may overlap. */
int moe_gdn_recurrence(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const float* alpha, const float* beta, float* state, float* out,
                       int B, int T, int Hk, int Hv, int dk, int dv, void* stream);

/* The last message of `ctx` (NULL: of the calls without a context), and the
 * name of a status code.  Never NULL. */
const char* moe_last_error(const moe_ctx* ctx);
const char* moe_status_string(int status);

/* Free every device allocation of the context (synchronises the device
 * first).  NULL is a no-op. */
void moe_destroy(moe_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
