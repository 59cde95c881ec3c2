/*
 * ft.h -- C ABI of libft, a single-GPU (sm_103a) implementation of the
 * FreeToken MoE layer's data-parallel hot path: the per-layer routing-control
 * pass over an all-layer, slot-indexed GPU expert cache, the cache fills, the
 * expert SwiGLU computation over resident slots merged with a supplied
 * CPU-set partial sum, the full-layer double-buffered prefill, and cache
 * resize.
 *
 * Conventions (all entry points):
 *   - Every call returns an ft_status; nothing throws across the ABI.
 *   - Pointers are plain host or device addresses as stated per argument;
 *     sizes are element counts unless stated.  No ownership is transferred
 *     unless stated: the library owns the slot pool, residency maps, LRU
 *     stamps, worklists and scratch; the caller owns the host expert pool and
 *     every input/output buffer.
 *   - Calls marked "async" enqueue work on the context's compute stream (and,
 *     for prefill, its transfer stream) and return without a host
 *     synchronisation.  Calls marked "syncs" block until the context's
 *     streams are idle.
 *   - Problems detected on the device (an out-of-range or duplicated expert id,
 *     a non-finite logit, a bounded wait that ran out) latch a sticky error
 *     word; ft_get_status() returns and clears it.
 *   - A context must be used from one host thread at a time.
 */
#ifndef FT_H
#define FT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ft_status;
#define FT_OK             0
#define FT_ERR_ARG       -1   /* invalid argument (checked on the host)              */
#define FT_ERR_CUDA      -2   /* a CUDA runtime / driver call failed                  */
#define FT_ERR_OOM       -3   /* device or pinned memory could not be allocated       */
#define FT_ERR_CAPACITY  -4   /* the cache is too small for the request (prefill <2E) */
#define FT_ERR_TIMEOUT   -5   /* a bounded device wait gave up                        */
#define FT_ERR_STATE     -6   /* call not allowed in the current state                */
#define FT_ERR_DEVICE    -7   /* invalid input detected on the device (ids, logits)   */

#define FT_FMT_BF16   0       /* bf16 banks                                           */
#define FT_FMT_NVFP4  1       /* e2m1 values + e4m3 block-16 scales + fp32 global     */
#define FT_FMT_MXFP4  2       /* e2m1 values + E8M0 block-32 scales (OCP MX v1.0)     */
#define FT_FMT_FP8    3       /* E4M3 values + fp32 scale per 128 x 128 block         */

typedef struct ft_ctx ft_ctx; /* opaque; created by ft_layer_init, freed by ft_destroy */

/* Result summary of the last control pass (ft_get_last_ctl). */
typedef struct {
    int32_t layer;     /* MoE layer of the pass                                      */
    int32_t T;         /* tokens                                                     */
    int32_t u;         /* unique experts routed (|U|)                                */
    int32_t h;         /* hits                                                       */
    int32_t m;         /* misses                                                     */
    int32_t q0;        /* round(m*B_P/B_H), halves away from zero                    */
    int32_t q1;        /* q0 clamped to [1, m] (0 when m = 0)                        */
    int32_t q;         /* fills after the capacity clamp min(q1, S-h)                */
    int32_t nC;        /* experts left to the CPU set C (m - q)                      */
    int32_t u_gpu;     /* experts computed on the GPU (h + q)                        */
    int32_t n_assign;  /* routed (token, expert) pairs computed on the GPU           */
    uint32_t clock;    /* LRU clock value of the pass                                */
} ft_ctl_info;

/* Cumulative counters since init (ft_get_counters).  calls: control passes;
 * unique/hits/misses/fills/cpu: sums of u, h, m, q, m-q; assign: routed pairs
 * computed on the GPU (sum of n_assign). */
typedef struct {
    uint64_t calls, unique, hits, misses, fills, cpu, assign;
} ft_counters;

/* Kernel ids of the profile (ft_profile_read). */
#define FT_K_ROUTE_CTL    0   /* control pass                                   */
#define FT_K_FILL         1   /* cache fills (host pool -> slots)               */
#define FT_K_EXPERT       2   /* decode expert FFN: gate/up + SwiGLU, down,     */
                              /* gated merge + partial_C (one fused kernel)     */
#define FT_K_PF_ROUTE     4   /* prefill routing + counting sort                */
#define FT_K_PF_PERMUTE   5   /* prefill token gather into expert order         */
#define FT_K_PF_GEMM1     6   /* prefill gate/up grouped GEMM + SwiGLU          */
#define FT_K_PF_GEMM2     7   /* prefill down grouped GEMM                      */
#define FT_K_PF_COMBINE   8   /* prefill gated combine                          */
#define FT_K_PF_H2D       9   /* prefill layer copy (transfer stream)           */
#define FT_K_PF_DEQUANT  10   /* prefill NVFP4 layer -> bf16 staging            */
#define FT_K_COUNT       16
typedef struct {
    double ms[FT_K_COUNT];          /* summed device time of the launches       */
    uint64_t launches[FT_K_COUNT];  /* launches recorded                        */
} ft_profile;

/* ABI version of this header; ft_abi_version() returns the library's. */
#define FT_ABI_VERSION 1
int32_t ft_abi_version(void);
const char* ft_status_str(ft_status s);

/*
 * ft_layer_init -- create a context: the slot cache and control state for L
 * MoE layers of E experts each (top-k routing, hidden size H, expert ffn size
 * F), with S slots.  FreeToken deepmox chapter "The Expert Cache That Follows
 * the Router", section "One logical expert, two physical levels of memory":
 * the host pool is the source of truth and holds one complete record per flat
 * id layer*E+expert; a GPU slot holds one complete record; one cache is shared
 * by all layers.
 *
 *   L, E, k, H, F  sizes; need E <= 1024, k <= 16, k <= E, H % 64 == 0,
 *                  F % 64 == 0 (H, F >= 64).
 *   S              number of slots (>= 1).  Prefill needs S >= 2E.
 *   fmt            FT_FMT_BF16, FT_FMT_NVFP4 or FT_FMT_MXFP4 (record layout in
 *                  ft_record_bytes); NVFP4 needs H % 256 == 0, F % 256 == 0
 *                  and nvfp4_global; MXFP4 needs H % 256 == 0, F % 512 == 0
 *                  (the W_d scale rows of a CTA's output rows are copied as
 *                  16-byte multiples) and nvfp4_global == NULL.  The pages
 *                  list MXFP4 among the bank layouts (deepmox, "One logical
 *                  expert, two physical levels of memory").  MXFP4 contexts
 *                  with prefill hold the same bf16 staging copy as NVFP4.
 *                  FP8 (block-FP8, the same section's "FP8 weights and
 *                  block-scale data") needs H % 128 == 0, F % 128 == 0,
 *                  (H/128)*(F/128) a multiple of 4 (so that every record and
 *                  each of its three scale matrices starts on a 16-byte
 *                  boundary, as the kernels' bulk copies and 16-byte loads
 *                  require), nvfp4_global == NULL and T_max*k*ceil(H/SMs)*4 bytes of
 *                  shared memory (at most 227 KiB); its decode streams the
 *                  pending fills inside the gate/up kernel, as the other
 *                  formats do, and its prefill stages the layer in bf16 (one
 *                  rounding of e4m3 * scale).
 *   T_max          largest T of a decode call (ft_route_ctl), 1..256, with
 *                  T_max*k <= 4096 and T_max*H <= 32768 (the tokens of a
 *                  decode call are staged in shared memory); the decode
 *                  kernel of the format must have a shared-memory plan for
 *                  every T <= T_max (BF16: two ring slots of 16 rows of H,
 *                  so H up to about 3400), else FT_ERR_ARG.
 *   T_prefill_max  largest T of a prefill layer call; 0 disables prefill (no
 *                  prefill scratch is allocated).  Prefill needs H % 256 == 0,
 *                  2F % 256 == 0 and E <= 256.  NVFP4 contexts with prefill
 *                  also hold a bf16 staging copy of one layer (E*6*H*F bytes).
 *   host_pool      HOST address of the caller's expert pool: L*E records of
 *                  ft_record_bytes(H,F,fmt) bytes, record l*E+e at offset
 *                  (l*E+e)*record_bytes.  Must be page-locked (cudaHostAlloc /
 *                  cudaHostRegister) or otherwise device-accessible, its
 *                  device address 16-byte aligned (FT_ERR_ARG otherwise: the
 *                  fills read it with bulk copies), and stay valid and
 *                  unchanged until ft_destroy.  Not copied.
 *   nvfp4_global   HOST array of L*E fp32 per-record global scales (NVFP4), or
 *                  NULL for BF16, MXFP4 and FP8.  Copied to device memory at init (the pages:
 *                  small per-expert values stay GPU-resident).
 *   compute_stream, transfer_stream
 *                  cudaStream_t handles owned by the caller (NULL = legacy
 *                  default stream for compute; transfer must then differ only
 *                  if prefill is used).  They must outlive the context.
 *   out            receives the context.
 * Errors: FT_ERR_ARG (sizes, NULL pool), FT_ERR_OOM, FT_ERR_CUDA.  Syncs.
 */
ft_status ft_layer_init(ft_ctx** out, int32_t L, int32_t E, int32_t k, int32_t H, int32_t F,
                        int32_t S, int32_t fmt, int32_t T_max, int32_t T_prefill_max,
                        const void* host_pool, const float* nvfp4_global,
                        void* compute_stream, void* transfer_stream);

/* Bytes of one complete layer-expert record.
 * BF16 : [W_gu 2F x H bf16, row-major, gate/up rows interleaved in groups of 16
 *         (16 gate rows, the 16 matching up rows, ...)] [W_d H x F bf16 row-major].
 * NVFP4: [W_gu values 2F x H e2m1, 2 per byte, low nibble first, same row order]
 *        [W_d values H x F] [W_gu e4m3 scales 2F x H/16] [W_d scales H x F/16].
 * MXFP4: the NVFP4 layout with one E8M0 scale (value 2^(code-127), 0xFF NaN)
 *        per 32 values along K: [W_gu values] [W_d values]
 *        [W_gu scales 2F x H/32] [W_d scales H x F/32]; no global.
 * FP8  : [W_gu values 2F x H E4M3, one byte each, same row order]
 *        [W_d values H x F] [W_g scales F/128 x H/128 fp32]
 *        [W_u scales F/128 x H/128] [W_d scales H/128 x F/128], row-major;
 *        w = e4m3 * scale(row / 128, k / 128).
 * Returns 0 for an unknown fmt. */
size_t ft_record_bytes(int32_t H, int32_t F, int32_t fmt);

/*
 * ft_route_ctl -- the per-layer control pass and the cache fills, async.
 * FreeToken explainer sections 4-10 and deepmox section "How residency
 * follows demand without leaving the device": dedup the routed experts, look
 * each flat id up in slot_for_id (resident = hit), q = clamp(round(m*B_P/B_H),
 * 1, m) for m >= 1 (explainer section 5; txtmix: at least one fill), the fill
 * set F = the first q misses by routed-token count (descending, lower id
 * first), the rest is the CPU set C; victims = the q least recently used slots
 * not holding a hit of this call (smallest (stamp, slot)); hits and fills get
 * the pass's clock as stamp; route ids are rewritten to slot ids; then the q
 * complete records are copied from the host pool into their victim slots.
 * All of it runs on the device: no host synchronisation.  The copies are
 * enqueued with the next ft_moe_forward of the context, fused into its
 * expert kernel (the fill overlaps the computation on the hits); every other
 * call of the context that reads or changes the slots (ft_route_ctl,
 * ft_read_slot, ft_get/set_ctl_state, ft_cache_resize, ft_prefill_begin,
 * ft_get_status) first completes a pending fill with a standalone copy.
 *
 *   layer     0..L-1.
 *   T         tokens, 1..T_max.
 *   logits    DEVICE fp32 [T, E] router logits, or NULL when top-k is given.
 *             Top-k is taken by value (descending), lower id first on ties;
 *             gates are the softmax over the k selected logits (fp32).
 *   topk_ids  DEVICE int32 [T, k] expert ids (distinct within a token), or NULL.
 *   topk_w    DEVICE fp32 [T, k] gate weights matching topk_ids, or NULL.
 *             Exactly one of logits / (topk_ids and topk_w) must be given.
 *   B_P, B_H  host-to-device expert-transfer and host-side expert bandwidths
 *             (any common unit, B_P > 0, B_H > 0).  q uses (m*B_P)/B_H in fp64.
 * Errors: FT_ERR_ARG (host checks), FT_ERR_STATE (a prefill chunk is open).
 * Invalid ids or non-finite logits latch FT_ERR_DEVICE; the pass then routes
 * nothing to the GPU and changes no residency.
 */
ft_status ft_route_ctl(ft_ctx* ctx, int32_t layer, int32_t T, const float* logits,
                       const int32_t* topk_ids, const float* topk_w, double B_P, double B_H);

/*
 * ft_moe_forward -- expert computation for the layer of the last
 * ft_route_ctl, async.  For every routed pair (t, j) whose expert is a hit or
 * a fill: FFN(x_t) = W_d (SiLU(W_g x_t) * (W_u x_t)) over the slot's record;
 * y_t = sum_j g_tj FFN_{e_tj}(x_t) (j ascending) + partial_C_t.  The METAL
 * MEDIA page, Figure 2 caption, and explainer section 14: GPU and CPU partial
 * outputs merge exactly.
 *
 *   x          DEVICE bf16 [T, H] (T of the last ft_route_ctl).
 *   partial_C  DEVICE fp32 [T, H] partial sum of the CPU set C, or NULL (zeros).
 *   y          DEVICE fp32 [T, H] output; must not alias x or partial_C.
 * Errors: FT_ERR_STATE if no control pass preceded it.
 */
ft_status ft_moe_forward(ft_ctx* ctx, const void* x, const float* partial_C, float* y);

/*
 * ft_prefill_begin -- open a prefill chunk, async.  FreeToken explainer
 * section 2 and deepmox section "How residency follows demand...": prefill
 * streams whole layers through two full-layer buffers carved from the first
 * two expert-layer regions of the slot pool (buffer b = slots [b*E, (b+1)*E)).
 * A begin fence orders the transfer after earlier decode work; the owners of
 * buffer (layer & 1) are invalidated (slot_for_id cleared, stamp 0) and the
 * E records of `layer` are copied host-to-device on the transfer stream.
 *   layer  first layer of the chunk.
 * Errors: FT_ERR_CAPACITY (S < 2E), FT_ERR_STATE (chunk already open or
 * prefill disabled).
 */
ft_status ft_prefill_begin(ft_ctx* ctx, int32_t layer);

/*
 * ft_prefill_layer -- one prefill layer, async.  Waits for buffer `buffer` to
 * hold `layer`; if next_layer >= 0, invalidates the other buffer and streams
 * next_layer into it on the transfer stream once the previous layer's GEMMs
 * released it (release event); routes T tokens (top-k of logits, softmax
 * gates), runs the grouped SwiGLU FFN over the buffer with tensor cores and
 * writes y_t = sum_j g_tj FFN_{e_tj}(x_t) (j ascending).  next_layer = -1
 * closes the chunk; the buffer slots are left empty afterwards.
 *
 *   buffer      0 or 1: the i-th layer of a chunk (counting from 0 at
 *               ft_prefill_begin) is held by buffer i & 1.
 *   layer       layer held by `buffer`.
 *   next_layer  layer to stream next, or -1.
 *   T           tokens, 1..T_prefill_max.
 *   x           DEVICE bf16 [T, H];  logits DEVICE fp32 [T, E];
 *   y           DEVICE fp32 [T, H].
 * Errors: FT_ERR_STATE (no open chunk / wrong buffer), FT_ERR_ARG.
 */
ft_status ft_prefill_layer(ft_ctx* ctx, int32_t buffer, int32_t layer, int32_t next_layer,
                           int32_t T, const void* x, const float* logits, float* y);

/*
 * ft_cache_resize -- rebuild the slot cache with S_new slots, syncs.
 * FreeToken explainer section 11 and txtmix section on "ft ctl cache": the
 * cache is rebuilt for a new VRAM budget at a safe point without restarting;
 * the host pool keeps results correct.  Shrinking evicts in LRU order
 * (smallest (stamp, slot) first) until min(S_new, occupied) entries remain and
 * packs the survivors, in ascending old slot order, into slots 0..n-1;
 * growing keeps every slot and adds empty ones.  Stamps and clock are kept.
 * On any failure the old cache is left unchanged.
 * Errors: FT_ERR_ARG (S_new < 1), FT_ERR_STATE (prefill chunk open), FT_ERR_OOM.
 */
ft_status ft_cache_resize(ft_ctx* ctx, int32_t S_new);

/*
 * ft_measure_link -- measure B_P, the record-copy bandwidth over the host
 * link, with the library's own fill path; syncs.
 * FreeToken explainer section 5 "Deriving q*": B_P is the measured transfer
 * bandwidth of expert records; the txtmix write-up describes a one-off
 * on-machine measurement of it ("ft bench bw") whose result drives q.
 * Copies n_records complete records of the host pool (flat ids spread evenly
 * over the pool) into a temporary device buffer with the fill kernel, reps
 * times, and stores the best repetition's rate in *gbps (1e9 bytes per
 * second).  The cache, its state and the statistics are not touched; a
 * pending fill is performed first.  The temporary buffer (n_records *
 * ft_record_bytes bytes) is allocated and freed inside the call.
 * Errors: FT_ERR_ARG (n_records < 1 or > L*E, reps < 1 or > 1000, gbps
 * NULL), FT_ERR_STATE (prefill chunk open), FT_ERR_OOM, FT_ERR_CUDA.
 */
ft_status ft_measure_link(ft_ctx* ctx, int32_t n_records, int32_t reps, double* gbps);

/*
 * ft_expert_ffn_noalloc -- the decode expert FFN without a context and
 * without allocating anything.  The pages have no counterpart to this entry
 * point.  It exists for callers that may not allocate device memory once
 * they run: serving engines that carve all device memory into their own
 * pools at start-up and forbid later allocations, and latency-critical paths
 * that cannot afford the device synchronisation of cudaMalloc / cudaFree.
 * ft_layer_init allocates, so such callers use this.
 *
 * For every route (t, j) with route_records[t*k+j] >= 0 it computes
 * FFN(x_t) = W_d (SiLU(W_g x_t) * (W_u x_t)) over that BF16 record and writes
 * y_t = sum_j gates[t*k+j] FFN_{route_records[t*k+j]}(x_t) (j ascending) +
 * partial_C_t -- the same kernel and arithmetic as ft_moe_forward.
 *
 *   records        DEVICE array of n_records BF16 records (ft_record_bytes
 *                  layout), 16-byte aligned; read only.
 *   route_records  DEVICE int32 [T, k]: record index of each route, or -1 for a
 *                  route computed elsewhere (the CPU set).  An index outside
 *                  [-1, n_records) is an error found on the device: the call
 *                  then routes nothing (y = partial_C, or 0 without it) and
 *                  latches FT_ERR_DEVICE for ft_noalloc_status.
 *   gates          DEVICE fp32 [T, k].
 *   x              DEVICE bf16 [T, H];  partial_C DEVICE fp32 [T, H] or NULL;
 *   y              DEVICE fp32 [T, H], not aliasing x or partial_C.
 *   T, k, H, F     T*k <= 1024, k <= 16, H and F multiples of 64, T*H <= 32768,
 *                  65536 + T*k*F*4 <= FT_NOALLOC_SCRATCH_BYTES, and a
 *                  shared-memory plan of the expert kernel for these sizes
 *                  (as ft_layer_init's BF16 check; else FT_ERR_ARG).
 *   stream         cudaStream_t to run on (NULL = legacy default stream).
 * Scratch: one file-scope device array of FT_NOALLOC_SCRATCH_BYTES per device
 * that loads the library, held until the process exits; no cudaMalloc,
 * cudaFree or allocating library call is made.  The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress) with that device
 * current.  Every call shares the array and leaves its contents behind; each
 * call rewrites what it reads.  Calls that overlap on the GPU (several streams
 * or host threads) race on the array: serialise them.  Async; returns
 * FT_ERR_ARG (host checks) or FT_ERR_CUDA; problems found on the device are
 * reported by ft_noalloc_status.
 */
#define FT_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u + 65536u)
ft_status ft_expert_ffn_noalloc(const void* records, int32_t n_records, const int32_t* route_records,
                                const float* gates, const void* x, const float* partial_C, float* y,
                                int32_t T, int32_t k, int32_t H, int32_t F, void* stream);

/*
 * ft_noalloc_status -- synchronise `stream` (a cudaStream_t, NULL = legacy
 * default stream) and return, then clear, the error word that the
 * ft_expert_ffn_noalloc calls on the current device latched since the last
 * ft_noalloc_status: FT_OK, FT_ERR_DEVICE (an out-of-range record index) or
 * FT_ERR_TIMEOUT (a bounded wait in the expert kernel gave up; that call's y
 * is not valid).  Allocates nothing.  FT_ERR_CUDA if a CUDA call fails.
 */
ft_status ft_noalloc_status(void* stream);

/* ---- observability and test surface (all sync) ------------------------- */

/* Copy the control state to HOST buffers: slot_for_id [L*E], id_for_slot [S],
 * stamps [S], clock [1].  Any pointer may be NULL to skip it. */
ft_status ft_get_ctl_state(ft_ctx* ctx, int32_t* slot_for_id, int32_t* id_for_slot,
                           uint32_t* stamps, uint32_t* clock);

/* Replace the control state from HOST buffers (same shapes).  Checked: maps
 * form a bijection on occupied slots, ids and slots in range, stamps <= clock.
 * Slot CONTENTS are not touched: use only with a state whose occupied slots
 * already hold the named records, or right after init with an all-empty map. */
ft_status ft_set_ctl_state(ft_ctx* ctx, const int32_t* slot_for_id, const int32_t* id_for_slot,
                           const uint32_t* stamps, uint32_t clock);

/* Details of the last control pass, into HOST buffers (any may be NULL):
 * F [q] fill experts (fill order), C [nC] CPU-set experts (same order),
 * victims [q] slots (ascending (stamp, slot); victims[i] received F[i]),
 * topk_ids [T*k], gates [T*k] (routing used), slots_topk [T*k] (slot or -1). */
ft_status ft_get_last_ctl(ft_ctx* ctx, ft_ctl_info* info, int32_t* F, int32_t* C,
                          int32_t* victims, int32_t* topk_ids, float* gates, int32_t* slots_topk);

/* Copy slot `slot`'s record (ft_record_bytes bytes) to a HOST buffer. */
ft_status ft_read_slot(ft_ctx* ctx, int32_t slot, void* host_dst);

/* Cumulative counters into a HOST struct. */
ft_status ft_get_counters(ft_ctx* ctx, ft_counters* out);

/* Per-kernel device timing.  While enabled, the library records a CUDA event
 * pair around each of its own launches on the stream the launch uses;
 * ft_profile_read (syncs) sums the elapsed times per kernel id and clears the
 * records.  Enabling resets the sums.  Inside a stream capture the records
 * become external event-record nodes of the graph: read the profile after the
 * graph ran once.  ft_kernel_name returns a static name for an id (NULL if
 * unknown). */
ft_status ft_profile_enable(ft_ctx* ctx, int32_t enable);
/* Suspend (paused != 0) or resume recording without synchronising or
 * resetting: usable between the calls of a stream capture to time a sample
 * of the captured launches. */
ft_status ft_profile_pause(ft_ctx* ctx, int32_t paused);
ft_status ft_profile_read(ft_ctx* ctx, ft_profile* out);
const char* ft_kernel_name(int32_t id);

/* Current number of slots. */
int32_t ft_num_slots(const ft_ctx* ctx);

/* Synchronise the context's streams and return (and clear) the sticky device
 * error word: FT_OK, FT_ERR_DEVICE or FT_ERR_TIMEOUT; FT_ERR_CUDA if a CUDA
 * error is pending.  On FT_ERR_TIMEOUT the outputs of the calls since the
 * last status read are not valid, and, because a wait that gave up may have
 * left a fill record incomplete, every slot is evicted (maps emptied, stamps
 * 0, clock kept): later calls refill from the host pool, which stays the
 * source of truth (deepmox, "How residency follows demand without leaving
 * the device"). */
ft_status ft_get_status(ft_ctx* ctx);

/* Limit, in nanoseconds of GPU global time, of the BF16 decode expert
 * kernel's waits on the progress of its other warps and CTAs (ring slots,
 * fill chunks, completion counters); each such wait that runs out latches
 * FT_ERR_TIMEOUT and the kernel winds down.  Waits for a thread's own copies
 * in flight keep the 2 s default, so a kernel never exits with a copy
 * landing in its shared memory.  ns = 0 restores the default (2e9); else
 * 1000 <= ns <= 2e9 (FT_ERR_ARG otherwise).  Host only; applies to the
 * launches that follow.  The other kernels always use the default. */
ft_status ft_set_wait_limit(ft_ctx* ctx, uint64_t ns);

/* Free every library-owned resource.  Syncs.  ctx may be NULL. */
void ft_destroy(ft_ctx* ctx);

#ifdef __cplusplus
}
#endif
#endif /* FT_H */
