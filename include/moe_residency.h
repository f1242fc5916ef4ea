/*
 * moe_residency.h -- C ABI of the split-residency routed MoE layer for one
 * GB300 GPU (sm_103a).
 *
 * The layer (write-up "vLLM: Pin Hot Experts", section "Results, September 17"
 * and "The one open door: two tensors and a row map"): each MoE layer keeps
 * its experts in two banks -- a hot bank in HBM and a cold bank in pinned host
 * memory that the GPU reads in place through a mapped (UVA) device pointer --
 * plus a device row map from global expert id to (bank, row).  A layer-step
 * routes each token to its top-k experts, splits the picks by residency
 * (counting them into a usage table, write-up "We Built the Counter",
 * section 2), runs the MXFP4 expert FFN once per bank without finalize, and
 * finalizes each token's k expert rows in fixed k order.  Between steps, rows
 * move between banks by true swaps ("vLLM: Pin Hot Experts", section "Making
 * it follow the traffic"; "We Built the Counter", section 2).
 *
 * Conventions for every entry point:
 *  - Return value: MOE_OK (0) or a negative MOE_E* code; moe_last_error()
 *    gives a message for the calling thread.  Nothing throws across the ABI.
 *  - "device" pointers are CUDA device (or mapped) addresses on the context's
 *    device; "host" pointers are ordinary CPU memory.  The caller owns every
 *    pointer it passes; the library owns the banks, row maps, usage table,
 *    swap staging rows and swap stream it allocates in moe_create /
 *    moe_init_banks.
 *  - stream: a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Calls marked "async" only enqueue work on it.
 *  - bf16 tensors are passed as uint16_t bit patterns.
 *  - Expert weights use the logical MXFP4 layout (OCP MX v1.0): for one
 *    expert, w13_q [2I][H/2] and w2_q [H][I/2] bytes, where byte b of a row
 *    holds K elements 2b (low nibble) and 2b+1 (high nibble); w13_s [2I][H/32]
 *    and w2_s [H][I/32] are e8m0 scales, one per 32 contiguous K elements.
 *    Rows 0..I-1 of W13 are the gate projection, rows I..2I-1 the up one.
 *  - Row map encoding: row_map[e] >= 0 is hot-bank row row_map[e];
 *    row_map[e] < 0 is cold-bank row -1 - row_map[e].
 */
#ifndef MOE_RESIDENCY_H
#define MOE_RESIDENCY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    MOE_OK = 0,
    MOE_EINVAL = -1,    /* bad argument, shape or id                        */
    MOE_ENOMEM = -2,    /* a device or pinned-host allocation failed         */
    MOE_ECUDA = -3,     /* a CUDA runtime call failed                        */
    MOE_ESTALE = -4,    /* (per swap pair) the rows moved since the decision */
    MOE_ETIMEOUT = -5,  /* a bounded device wait gave up                     */
    MOE_ESTATE = -6     /* call out of order (e.g. layer has no banks yet)   */
};

enum { MOE_BANK_HOT = 0, MOE_BANK_COLD = 1, MOE_BANK_BOTH = 2 };

/* FFN kernel implementation: tensor cores (tcgen05 + TMEM, default) or a
 * CUDA-core kernel kept for cross-checking. */
enum { MOE_FFN_TCGEN05 = 0, MOE_FFN_SIMT = 1 };

typedef struct moe_ctx moe_ctx;

typedef struct moe_geom {
    int32_t layers;      /* L: MoE layers managed by this context            */
    int32_t experts;     /* E: routed experts per layer (<= 1024)             */
    int32_t top_k;       /* k: experts per token (1..16)                      */
    int32_t hidden;      /* H: model width, a multiple of 128 (of 256 unless
                            I is a multiple of 128)                         */
    int32_t inter;       /* I: expert intermediate width, a multiple of 64    */
    int32_t count_tmax;  /* count only steps with T <= count_tmax (256)       */
    int32_t max_tokens;  /* T_max: largest T any call will pass               */
} moe_geom;

/* Message for the last failing call on this thread (never NULL). */
const char *moe_last_error(void);

/* Bytes of one expert (weights + scales); 18,800,640 at H=4096, I=2880
 * ("vLLM: Pin Hot Experts": 17.93 MiB per MXFP4 expert). */
int64_t moe_expert_bytes(int32_t hidden, int32_t inter);

/* Pack one expert, given in the logical MXFP4 layout above, into the bytes of
 * a bank row (what moe_init_banks places and moe_read_bank_row returns).
 * Host memory only; no device is touched.  out: moe_expert_bytes(hidden,
 * inter) bytes.  The row is the W13 part, then the W2 part.  Each part is a
 * sequence of 8704-byte blocks, one per (128-row M-tile, 128-wide K group):
 * the tile's 128 rows of 64 code bytes in the logical nibble order, then a
 * 512-byte scale atom holding the scale of tile row m and 32-wide K block kb
 * at byte (m%32)*16 + 4*(m/32) + kb.  W13 tile mt row 32w+l holds W13 row
 * (l<16 ? 0 : I) + 64mt + 16w + l%16; W2 tile mt row m holds W2 row 128mt+m.
 * A tile's blocks follow in K order, tiles in order.  When I % 128 == 64, W2
 * tiles 2p and 2p+1 are stored as a pair: 2p's full groups, then 2p+1's, then
 * one shared group whose K blocks 0-1 are 2p's last 64 columns and whose
 * blocks 2-3 are 2p+1's.  The geometry must satisfy moe_create's rules for
 * H and I, and the scale bytes moe_init_banks' range; otherwise MOE_EINVAL. */
int moe_pack_expert(int32_t hidden, int32_t inter, const uint8_t *w13_q, const uint8_t *w13_s,
                    const uint8_t *w2_q, const uint8_t *w2_s, uint8_t *out);

/* Create a context on CUDA device `device`: validates the geometry and
 * allocates the [L x E] int32 usage table (zeroed), two HBM staging rows for
 * swaps, and the swap stream with its events.  *out receives the context.
 * MOE_EINVAL on a bad geometry (the rules above), a null argument or no such
 * device; on a failed allocation the error of that call, with nothing left
 * allocated. */
int moe_create(const moe_geom *geom, int device, moe_ctx **out);

/* Free everything the context allocated (its banks included).  Synchronizes
 * the device.  NULL is a no-op. */
int moe_destroy(moe_ctx *ctx);

/* Select the FFN kernel implementation (MOE_FFN_*) for later calls.
 * MOE_EINVAL for another value. */
int moe_set_ffn_impl(moe_ctx *ctx, int impl);

/* Activation format of the tensor-core FFN on prefill-sized steps (more
 * than 256 tokens; decode-sized steps always use MOE_ACT_E4M3X2), for later
 * calls.  The pages leave the activation format of the routed MXFP4 kernel
 * unstated ("vLLM: Pin Hot Experts", Where the experts live today).
 *  MOE_ACT_E4M3X2 (default): each token row and h row is scaled by a power
 *    of two and carried as two e4m3 pieces (bf16-class precision, about 2^-8
 *    of each value); two MMAs per product.
 *  MOE_ACT_MXFP8: OCP MXFP8 -- each 32-element block of a row shares an e8m0
 *    scale (the smallest 2^e with max|v| 2^-e <= 448) and its elements are
 *    e4m3, rounded to nearest even; one MMA per product, at e4m3 precision
 *    (rows within about 8e-2 relative L2 of the exact FFN).
 * MOE_EINVAL for another value. */
enum { MOE_ACT_E4M3X2 = 0, MOE_ACT_MXFP8 = 1 };
int moe_set_act_format(moe_ctx *ctx, int format);

/* Place one layer's experts ("vLLM: Pin Hot Experts", The one open door):
 * experts with is_hot[e] != 0 go to an HBM bank, the rest to a pinned host
 * bank mapped into the device address space; hot rows are assigned in
 * increasing expert id, cold rows likewise, and the device row map written.
 * Inputs are HOST pointers to all E experts stacked ([E][...] each, logical
 * layout above); the library repacks them into its tiled device layout and
 * does not keep the pointers.  Re-initialising a layer frees its old banks.
 * Scale bytes must lie in [104, 140] (scales 2^-23 .. 2^13); other values
 * return MOE_EINVAL.  Synchronous. */
int moe_init_banks(moe_ctx *ctx, int layer, const uint8_t *w13_q, const uint8_t *w13_s,
                   const uint8_t *w2_q, const uint8_t *w2_s, const uint8_t *is_hot,
                   void *stream);

/* Bytes of the caller-owned device workspace that serves every step of at
 * most T tokens (split lists, per-bank scratch for the FFN's intermediate
 * rows); non-decreasing in T.  MOE_EINVAL unless 0 <= T <= T_max and bytes
 * is non-null. */
int moe_workspace_bytes(const moe_ctx *ctx, int T, size_t *bytes);

/* Big-batch cold staging ("We Built the Counter", section 6: copying an
 * expert on a miss is a tool for big batches; "Should a GB300 Prefetch Its
 * Cold Experts?", section 6: staging offloaded experts for prefill-sized
 * steps).  The FFN streams a unit's weights once per token tile (8, 16 or
 * 32 tokens by step size; on steps of more than 256 tokens 144, or 160 in
 * the MXFP8 format), so a cold expert with picks in several tiles
 * would cross the host link once per tile.  With a pool of `slots` expert
 * rows in HBM (0..64; 0 frees it and turns staging off, the default), every
 * later FFN call that covers the cold bank of a step of more than 16 tokens
 * first picks the cold rows with more picks than one tile -- most picks
 * first, ties to the lower row, at most `slots` -- and copies each once into
 * the pool; their units then read the pool.  Same bytes, same arithmetic: the
 * rows of Y are bit-identical to unstaged steps.  The pool belongs to the
 * context and is rewritten by each such call, so calls of different layers
 * that use it must not overlap on the GPU.  Synchronizes the device;
 * MOE_ENOMEM if the pool cannot be allocated (staging is then off). */
int moe_set_cold_staging(moe_ctx *ctx, int slots);

/* After a staged FFN call: the cold-bank row copied into each pool slot, or
 * -1 (rows: host int32 [64]).  ws and T as in the call.  Synchronizes
 * stream. */
int moe_read_stage(moe_ctx *ctx, const void *ws, int T, int32_t *rows, void *stream);

/* Route, split and count (async).  "vLLM: Pin Hot Experts", Results (split
 * each token's k ids by residency); "We Built the Counter", section 2 (one
 * masked relaxed atomic add per pick into the usage table; only steps of at
 * most count_tmax tokens are counted).
 *   logits: device fp32 [T][E].  Top-k per token (ties: lower expert id
 *           first); w = softmax over the k picked logits in fp32.  A NaN
 *           logit is read as -infinity (ranked last, weight 0 beside a
 *           finite first pick), so ids are always valid expert ids.
 *   ids:    device int32 [T][k] out, descending logit order (the k order).
 *   w:      device fp32  [T][k] out.
 *   ws:     device workspace (moe_workspace_bytes) receiving both banks'
 *           pick lists grouped by (bank row, slot t*k+j).
 *   count_on: nonzero adds 1 per pick to usage[layer][id] when
 *           T <= count_tmax.
 * T == 0 writes empty lists.  MOE_EINVAL on a layer or T outside [0, T_max],
 * a null pointer or a workspace not 256-byte aligned; MOE_ESTATE if the
 * layer has no banks. */
int moe_route_split_count(moe_ctx *ctx, int layer, const float *logits, int T, int count_on,
                          int32_t *ids, float *w, void *ws, void *stream);

/* Copy one bank's pick lists from a routed workspace to host memory and
 * synchronize `stream`: *n_act active rows (increasing), act_off [n_act+1]
 * offsets into picks, picks [n_picks] slot indices t*k+j.  Host arrays must
 * hold T*k (+1) entries.  T must be the routed step's T. */
int moe_read_split(moe_ctx *ctx, const void *ws, int T, int bank, int32_t *n_act, int32_t *n_picks,
                   int32_t *act_row, int32_t *act_off, int32_t *picks, void *stream);

/* Expert FFN over one bank without finalize (async).  "vLLM: Pin Hot
 * Experts", Results: the routed MXFP4 expert kernel runs once on the hot
 * tensor and once on the cold one, unfinalized.  For every pick (t, j) whose
 * expert lives in `bank`: Y[t][j][:] = bf16( W2 (silu(W_gate x_t) * (W_up x_t)) ).
 * Rows of the other bank are not touched, so the two banks' calls may run on
 * two streams at once (each uses its own part of ws).  A bank with no picks
 * is a no-op on the device.
 *   bank: MOE_BANK_HOT, MOE_BANK_COLD, or MOE_BANK_BOTH.  MOE_BANK_BOTH runs
 *   both banks' FFNs in one launch per GEMM: the first CTA on each SM takes
 *   cold-bank work first (keeping the host link streaming from every SM),
 *   the others hot-bank work, and each turns to the other bank when its own
 *   runs out.  The rows equal those of the two one-bank calls bit for bit.
 *   Do not run a MOE_BANK_BOTH call concurrently with a one-bank call on the
 *   same workspace.
 *   x: device bf16 [T][H];  Y: device bf16 [T][k][H] out (x and Y 16-byte
 *   aligned);  ws as routed, 256-byte aligned.
 * T == 0 is a no-op.  MOE_EINVAL on a bad bank, layer or T, a null or
 * misaligned pointer; MOE_ESTATE if the layer has no banks.  A device wait
 * that runs out (moe_set_wait_limit) is reported by moe_device_status as
 * MOE_ETIMEOUT, not by this call's return value. */
int moe_expert_ffn_bank(moe_ctx *ctx, int layer, int bank, const uint16_t *x, int T, void *ws,
                        uint16_t *Y, void *stream);

/* Allocation-free variant of moe_expert_ffn_bank (async).  The write-ups
 * have no counterpart: this serves callers that may not allocate device
 * memory -- a plugin given a fixed memory budget by its host framework, or a
 * serving loop that must not call cudaMalloc because it can synchronize the
 * device and fail under memory pressure.  Instead of the FFN scratch part of
 * a caller workspace it uses one library-owned area in a __device__ array of
 * moe_static_scratch_bytes() (16 MiB) on every GPU that loads the library,
 * held until the process exits.
 *   split_ws: the caller's workspace after moe_route_split_count for this
 *   step (only its pick lists are read).  x, T, Y as moe_expert_ffn_bank; Y
 *   receives the same rows moe_expert_ffn_bank would write.
 * Returns MOE_EINVAL if the step's scratch would exceed the area (about
 * T*k*(6H + 14I) bytes, fp32 partial-sum rows included: at H=4096, I=2880,
 * k=6 steps of up to 43 tokens fit).  The first call on a device looks up the area's
 * device address; make that first call before any stream capture.  Every
 * call shares the one area and leaves its contents behind: calls whose work
 * overlaps on the GPU race, so run the two banks' calls one after the other
 * on one stream.  Allocates nothing (no cudaMalloc, cudaFree or allocating
 * library call). */
int moe_expert_ffn_bank_static(moe_ctx *ctx, int layer, int bank, const uint16_t *x, int T,
                               const void *split_ws, uint16_t *Y, void *stream);
size_t moe_static_scratch_bytes(void);

/* One whole layer-step from host buffers: the call an application that holds
 * its logits, hidden states and output rows in (pinned) host memory makes.
 * "vLLM: Pin Hot Experts", Results: route and split each token's k picks,
 * run the routed FFN over both banks, finalize the k weighted rows.  In order
 * on `stream`: the logits and hidden states are copied host -> device, then
 * moe_route_split_count (count_on as there), moe_expert_ffn_bank over both
 * banks and moe_finalize run on the scratch area, then the output rows are
 * copied device -> host.  The result is bit-identical to those calls made on
 * device buffers.
 *   logits: host fp32 [T][E]; x: host bf16 [T][H]; out: host bf16 [T][H] out.
 * Pinned host memory (cudaHostAlloc) makes the copies asynchronous; with
 * pageable memory they still complete, but they synchronize with the host.
 * out is written when the stream reaches the end of the call: synchronize the
 * stream before reading it.  scratch: device memory of at least
 * moe_step_scratch_bytes(ctx, Tcap) bytes, 256-byte aligned, for any T <=
 * Tcap; caller-owned, and calls that share it must not overlap on the GPU.
 * T == 0 is a no-op.  MOE_EINVAL on a bad argument; errors of the inner calls
 * are returned as they come. */
int moe_step_scratch_bytes(const moe_ctx *ctx, int T, size_t *bytes);
int moe_layer_step_host(moe_ctx *ctx, int layer, const float *logits, const uint16_t *x, int T, int count_on,
                        uint16_t *out, void *scratch, void *stream);

/* Router GEMM (async): the logits the routing call reads.  "vLLM: Pin Hot
 * Experts", Where the experts live today: each MoE layer's router scores all
 * experts for every token, whatever bank they sit in.
 *   logits[t][e] = bias[e] + sum_h x[t][h] * w_router[e][h]
 * x: device bf16 [T][H] (16-byte aligned); w_router: device bf16 [E][H]
 * (16-byte aligned); bias: device fp32 [E] or NULL (zero); logits: device
 * fp32 [T][E] out.  Exact products, fp32 sums: up to 32 tokens on the CUDA
 * cores (in a fixed order), beyond that on the tensor cores (kind::f16, fp32
 * accumulator), so a logit may differ from the exactly rounded sum in its
 * last bits.  H % 8 == 0, 1 <= E <= 2^20; T == 0 is a no-op.  The context
 * gives the device and the status word a bounded wait sets on timeout
 * (moe_device_status).  All other pointers are caller-owned.  MOE_EINVAL on
 * a bad shape or a null or misaligned pointer. */
int moe_router_logits(moe_ctx *ctx, const uint16_t *x, const uint16_t *w_router, const float *bias, int T, int E,
                      int H, float *logits, void *stream);

/* Finalize (async).  "vLLM: Pin Hot Experts", Results: accumulate each
 * token's k bf16 expert rows in fp32 with fma in the original k order and
 * cast once:  out[t][c] = bf16(fma(w[t][k-1], Y[t][k-1][c], ... fma(w[t][0],
 * Y[t][0][c], 0.0f))).  Y device bf16 [T][k][H], w device fp32 [T][k],
 * out device bf16 [T][H], all caller-owned; Y and out 16-byte aligned.
 * Takes no context: it runs on the calling thread's current device, which
 * must hold the three buffers.  1 <= k <= 16, H % 8 == 0; T == 0 is a no-op.
 * MOE_EINVAL on a bad shape or a null or misaligned pointer. */
int moe_finalize(const uint16_t *Y, const float *w, int T, int k, int H, uint16_t *out,
                 void *stream);

/* True swaps between steps ("vLLM: Pin Hot Experts", Making it follow the
 * traffic and E4/E4b; "We Built the Counter", section 2).  For each pair i in
 * order: promote[i] must be cold and demote[i] hot in the library's CPU copy
 * of the placement, else applied[i] = 0 (stale, nothing changes).  An applied
 * pair enqueues on `stream`: hot row -> HBM staging, cold row -> the hot
 * slot, then staging -> the cold slot (weights and scales together) on the
 * context's own swap stream, ordered after the first two, so that it runs
 * beside the next pair's copy into HBM (the host link carries both
 * directions at once; consecutive pairs alternate between two staging
 * rows); then a two-element device row-map write on `stream`, ordered after
 * all three copies.  Work enqueued on `stream` after the call sees every
 * applied pair complete.  promote,
 * demote: host int32 [n]; applied: host int32 [n] out (may be NULL).  Returns
 * the number applied (>= 0) or an error code.  Never call it while a step of
 * this layer is in flight on another stream.  If enqueuing a pair's copies or
 * map write fails, the call returns that error (MOE_ECUDA or MOE_ENOMEM),
 * applied[] marks only the pairs completed before it, and the layer is left
 * unplaced: every later call on it returns MOE_ESTATE until moe_init_banks
 * places it again (a bank row may hold neither expert whole). */
int moe_swap_rows(moe_ctx *ctx, int layer, int n, const int32_t *promote, const int32_t *demote,
                  int32_t *applied, void *stream);

/* Copy the [L][E] usage table to host_out and synchronize `stream` (the
 * counts are exact after the sync).  Counts only grow; a reader uses deltas. */
int moe_read_counts(moe_ctx *ctx, int32_t *host_out, void *stream);

/* Zero the usage table (async). */
int moe_reset_counts(moe_ctx *ctx, void *stream);

/* Placement queries.  moe_get_rowmap gives the library's CPU copy;
 * moe_read_rowmap_device copies the device row map (synchronizes stream). */
int moe_bank_rows(moe_ctx *ctx, int layer, int32_t *n_hot, int32_t *n_cold);
int moe_get_rowmap(moe_ctx *ctx, int layer, int32_t *host_out);
int moe_read_rowmap_device(moe_ctx *ctx, int layer, int32_t *host_out, void *stream);

/* Copy one bank row (one expert in the library's device layout,
 * moe_expert_bytes long) to host memory; synchronizes stream. */
int moe_read_bank_row(moe_ctx *ctx, int layer, int bank, int row, uint8_t *host_out,
                      void *stream);

/* Host-link probe: a kernel that reads `bytes` of the layer-independent
 * pinned probe buffer (mapped host memory) with 16-byte loads, `iters`
 * times; *gbps receives the best read rate.  Also measures an HBM read of
 * the same size into *hbm_gbps (may be NULL).  Synchronous. */
int moe_probe_link(moe_ctx *ctx, size_t bytes, int iters, double *gbps, double *hbm_gbps);

/* Read and clear the device status word that bounded device waits set
 * (MOE_OK or MOE_ETIMEOUT).  Synchronizes the device. */
int moe_device_status(moe_ctx *ctx, int32_t *status);

/* Number of kernels this library has launched in this process. */
int64_t moe_kernel_launches(void);

/* Bytes of device memory and of pinned host memory the library holds in
 * this process (banks, row maps, usage tables, staging rows, probe buffers of
 * every live context).  Either pointer may be NULL.  Lets a caller check that
 * a failed call left nothing behind. */
int moe_memory_in_use(int64_t *device_bytes, int64_t *pinned_bytes);

/* ---- failure handling (no GPU fault is ever raised on purpose) ----
 * Every pipeline wait of the FFN kernels is bounded by wall-clock time.  A
 * wait that runs out sets the status word to MOE_ETIMEOUT (read it with
 * moe_device_status), raises an abort flag that ends the CTA's other roles'
 * waits, lets the copies and MMAs the CTA already issued finish, frees its
 * tensor memory and returns; the rows of that call are then incomplete.
 * The next call needs no reset: each call re-initialises its work counters
 * and partial-sum rows.
 * moe_set_wait_limit: the bound in nanoseconds for this context's later FFN
 * calls (default 1 s; 0 restores the default). */
int moe_set_wait_limit(moe_ctx *ctx, uint64_t ns);

/* Host-set test hook for that path.  MOE_FAULT_WITHHOLD_COPY: in the next
 * FFN call's gate/up GEMM, the CTA that takes the first unit of a bank skips
 * the copies of its first K group, so every role waiting for them runs out
 * its wait.  MOE_FAULT_NONE clears a pending injection.  The allocation
 * failure path is tested through the environment instead: while
 * MOE_INJECT_ALLOC_FAIL names an allocation site ("cold_bank", "hot_bank",
 * "rowmap", "init_staging", "create_counts", "create_staging",
 * "create_status", "probe"), that site reports an
 * allocation failure without allocating (MOE_ENOMEM; moe_init_banks then
 * leaves the layer unplaced and frees what it had allocated). */
enum { MOE_FAULT_NONE = 0, MOE_FAULT_WITHHOLD_COPY = 1 };
int moe_inject_fault(moe_ctx *ctx, int kind);

/* ---- adaptive policy (host, between steps) ----
 * "We Built the Counter", sections 2 and 9: read the usage table every N
 * steps, keep a decaying average, queue swaps decided against a CPU copy of
 * the hot/cold lists.  At each read, per expert: delta = counts - last
 * (uint32), acc = d*acc + delta, wsum = d*wsum + 1 with
 * d = 0.5^(read_every/half_life); avg = acc/wsum (picks per read).  Cold
 * experts with avg >= min_avg (descending avg) pair with hot experts
 * (ascending avg), ties by lower expert id, while avg_cold > hysteresis *
 * avg_hot and fewer than max_pairs pairs were taken. */
typedef struct moe_policy moe_policy;
int moe_policy_create(int experts, double read_every, double half_life, double hysteresis,
                      double min_avg, int max_pairs, const int32_t *counts_now,
                      moe_policy **out);
int moe_policy_destroy(moe_policy *p);
/* counts: host int32 [E] of one layer; row_map: host int32 [E] (the CPU
 * copy); promote/demote: host int32 [E] out.  Returns the pair count. */
int moe_policy_read(moe_policy *p, const int32_t *counts, const int32_t *row_map,
                    int32_t *promote, int32_t *demote);

/* ---- restore a saved placement (host, between steps) ----
 * "We Built the Counter", section 2: an operator may ask for the start-up
 * placement back, and a round trip of swaps back to the start-up hot set
 * leaves the output unchanged.  A map is saved with
 * moe_get_rowmap.  moe_plan_restore gives the swaps that bring row_map's hot
 * set back to target's: the experts cold in row_map and hot in target, in
 * ascending id, are promoted, the i-th against the i-th expert hot in row_map
 * and cold in target (ascending id).  Only the hot SET is restored; the row an
 * expert takes inside a bank changes no output.  At most max_pairs pairs are
 * written (call again after applying them with moe_swap_rows to continue;
 * a step budget of 8 swaps keeps the restore off the step's critical path).
 * row_map, target: host int32 [experts] (negative = cold); promote, demote:
 * host int32 [max_pairs] out.  Returns the pair count (0 = restored), or
 * MOE_EINVAL when the maps hold different numbers of hot experts or an
 * argument is invalid. */
int moe_plan_restore(int experts, const int32_t *row_map, const int32_t *target, int max_pairs,
                     int32_t *promote, int32_t *demote);

#ifdef __cplusplus
}
#endif
#endif /* MOE_RESIDENCY_H */
