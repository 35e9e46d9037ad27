/*
 * ep.h -- C ABI of the single-GPU MoE expert-parallel token shuffle
 * (get_dispatch_layout -> dispatch -> combine) for GB300 (sm_103a).
 *
 * The operations are the high-throughput expert-parallel kernels described in
 * "[Not ready] MSCCLPP EP implementation" (mscclpp pull request 852), section
 * "Scope": get_dispatch_layout, intranode_dispatch and intranode_combine (the
 * DeepEP kernels, there ported onto MSCCL++ channels), plus the kUseFP8
 * payload cast of the low-latency dispatch<kUseFP8,...> kernel.  Here all R
 * logical ranks live on one GPU: rank s owns tokens [s*T_r, (s+1)*T_r) of
 * one call and experts [s*E_l, (s+1)*E_l), and every destination rank's
 * receive buffer is a range of rows of one packed device buffer.  The
 * "exchange" is the scatter kernel's own HBM writes; there is no peer
 * traffic and no collective.
 *
 * Notation: T tokens (T % R == 0, T_r = T/R), K top-k slots, E experts
 * (E % R == 0, E_l = E/R), H hidden channels, R ranks, P = number of
 * (token, destination rank) pairs = rows of the receive buffer.
 * src(t) = t / T_r, rank(e) = e / E_l.
 *
 * Conventions shared by every entry point
 *   - Pointers marked "device" are CUDA device pointers (or managed memory);
 *     "host" pointers are ordinary host memory.  The library never
 *     allocates or frees memory: the caller owns every buffer.
 *   - Every call is enqueued on `stream` (NULL = the legacy default stream)
 *     and returns without synchronising, except ep_layout_total_rows.
 *   - Argument checks are done on the host before anything is enqueued; a
 *     failed check returns EP_ERR_INVALID_ARG and enqueues nothing.
 *   - Problems that only the data reveal are reported through an optional
 *     device error word (int32, nullable): the kernels OR EP_ERRBIT_* bits
 *     into it with atomicOr.  The caller zeroes it; the library never clears
 *     it.  No kernel traps.
 *   - All buffers must be 16-byte aligned; x / recv_x / y / out rows are
 *     moved in 16-byte vectors and 1-D bulk (TMA) copies.
 *   - Limits: 1 <= R <= EP_MAX_RANKS, 1 <= K <= EP_MAX_TOPK,
 *     1 <= E <= EP_MAX_EXPERTS, H % 8 == 0 (H % 128 == 0 for FP8),
 *     T * R < 2^31.
 *   - The first call of each kind on a device does a one-time set-up on
 *     the host (kernel attributes, occupancy and cluster-size queries,
 *     cached per device; thread-safe).  Later calls repeat none of it: they
 *     check arguments and launch, so a sequence of calls can be captured
 *     into a CUDA graph once each kind has run eagerly on that device.
 */
#ifndef EP_H_
#define EP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same opaque type as cudaStream_t / CUstream, so no CUDA header is needed. */
typedef struct CUstream_st* ep_stream_t;

typedef enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1, /* a host-side argument check failed; nothing enqueued */
  EP_ERR_CAPACITY = 2,    /* a caller-provided buffer is too small (host-visible size) */
  EP_ERR_CUDA = 3,        /* a CUDA runtime call failed (launch, copy, sync) */
  EP_ERR_TIMEOUT = 4      /* reserved: a bounded device wait ran out (see EP_ERRBIT_TIMEOUT) */
} ep_status_t;

/* Bits OR-ed into the device error word. */
#define EP_ERRBIT_BAD_EXPERT 1 /* a topk_idx entry outside [-1, E): treated as masked */
#define EP_ERRBIT_CAPACITY 2   /* a slot >= recv_capacity_rows: that row was not written */
#define EP_ERRBIT_TIMEOUT 4    /* a bounded shared-memory pipeline wait ran out */
#define EP_ERRBIT_SCHED 8      /* a scheduled combine found its counters in use by another
                                  launch, or not zero at launch: tokens may be missing */

#define EP_MAX_RANKS 64
#define EP_MAX_TOPK 32
#define EP_MAX_EXPERTS 4096

/* Human-readable name of a status code (static storage; never NULL). */
const char* ep_status_string(ep_status_t status);

/*
 * Bytes of device scratch that ep_get_dispatch_layout needs for T tokens,
 * R ranks and E experts.  Returns 0 for invalid sizes.  The scratch holds
 * one 64-bit rank mask per token and per-block partial counts; its contents
 * need no initialisation and are dead after the call's kernels finish.
 */
size_t ep_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts);

/*
 * get_dispatch_layout + slot assignment ("Scope", Intranode:
 * get_dispatch_layout; the internode-combine commit: combine must use the
 * receiver-side prefix matrices, i.e. the slot order is fixed by prefix sums
 * over source rank and token order).
 *
 * In  (device): topk_idx [T, K] int64, row-major; -1 = masked slot.
 * Out (device), every element written:
 *   num_tokens_per_rank   [R, R] int32: [s][r] = tokens of source s sent to r
 *   num_tokens_per_expert [R, E] int32: [s][e] = slots (t,k) with src(t)=s, e_k = e
 *   is_token_in_rank      [T, R] uint8 (0/1; torch.bool storage)
 *   slot                  [T, R] int32: row of (t, r) in the receive buffer,
 *                         -1 if token t is not sent to rank r.  Rows are packed
 *                         destination-major: destination r owns rows
 *                         [recv_base[r], recv_base[r+1]), ordered by source
 *                         rank and then token index.
 *   recv_base             [R + 1] int32: exclusive prefix of rows per
 *                         destination; recv_base[R] = P.
 * err_word (device, nullable): EP_ERRBIT_BAD_EXPERT if some id is outside
 *   [-1, E) (the slot is then treated as masked).
 * workspace (device): at least ep_workspace_bytes(T, R, E) bytes, passed as
 *   workspace_bytes; a smaller value returns EP_ERR_CAPACITY.  Unused (may be
 *   NULL, with workspace_bytes 0) when ep_layout_auto_single_launch(T, R, E):
 *   such batches take the single-launch form described below.
 * T = 0 is valid (counts and recv_base are zeroed).
 * Same as ep_get_dispatch_layout_path(..., EP_LAYOUT_AUTO, stream).
 */
ep_status_t ep_get_dispatch_layout(const int64_t* topk_idx, int64_t num_tokens, int num_topk,
                                   int num_experts, int num_ranks, int32_t* num_tokens_per_rank,
                                   int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
                                   int32_t* slot, int32_t* recv_base, int32_t* err_word,
                                   void* workspace, size_t workspace_bytes, ep_stream_t stream);

/*
 * Which kernels compute the layout.  Both forms give identical outputs.
 *
 * EP_LAYOUT_MULTI_LAUNCH: two or three launches spread over the whole GPU
 *   (counts per block of tokens, block offsets, slots), with scratch in the
 *   caller's workspace.  Any size.
 * EP_LAYOUT_SINGLE_LAUNCH: one launch of one thread-block cluster of up to
 *   16 CTAs (8 where the device does not schedule 16), which exchange their
 *   counts through distributed shared memory; no workspace.  For small
 *   batches only (ep_layout_single_launch_fits): T <= 16384 and
 *   R * E <= 16384.  At decode sizes the layout is bound by latency, and
 *   this form removes the round trips between kernels.  The pages run layout, count exchange (notify_dispatch,
 *   cached_notify) and data movement as separate kernels ("Scope",
 *   Internode HT); this fused form has no counterpart there.
 * EP_LAYOUT_AUTO: the single-launch form where it is the faster one
 *   (ep_layout_auto_single_launch: it fits and T <= 8192), else multi-launch.
 *   Should the device refuse the cluster launch (a partition with too few
 *   free SMs, say), AUTO runs the multi-launch form instead if a usable
 *   workspace was passed, and returns EP_ERR_CUDA if not.
 */
typedef enum {
  EP_LAYOUT_AUTO = 0,
  EP_LAYOUT_MULTI_LAUNCH = 1,
  EP_LAYOUT_SINGLE_LAUNCH = 2
} ep_layout_path_t;

/* 1 if the single-launch form applies to (T, R, E), else 0 (also for invalid sizes). */
int ep_layout_single_launch_fits(int64_t num_tokens, int num_ranks, int num_experts);

/* 1 if EP_LAYOUT_AUTO takes the single-launch form for (T, R, E), else 0. */
int ep_layout_auto_single_launch(int64_t num_tokens, int num_ranks, int num_experts);

/*
 * ep_get_dispatch_layout with an explicit choice of kernels (`path`, an
 * ep_layout_path_t).  Arguments and outputs as ep_get_dispatch_layout.
 * Returns EP_ERR_INVALID_ARG, with nothing enqueued, for an unknown path or
 * for EP_LAYOUT_SINGLE_LAUNCH when the batch does not fit it (T = 0
 * included).  The workspace is needed only when the multi-launch form runs.
 */
ep_status_t ep_get_dispatch_layout_path(const int64_t* topk_idx, int64_t num_tokens,
                                        int num_topk, int num_experts, int num_ranks,
                                        int32_t* num_tokens_per_rank,
                                        int32_t* num_tokens_per_expert,
                                        uint8_t* is_token_in_rank, int32_t* slot,
                                        int32_t* recv_base, int32_t* err_word, void* workspace,
                                        size_t workspace_bytes, int path, ep_stream_t stream);

/*
 * The same layout as ep_get_dispatch_layout, for callers that cannot
 * allocate device memory when they call it (the MSCCL++ EP pages have no counterpart to
 * this entry point).  Such callers include plugin or custom-op hosts that
 * hand the library only tensors they already own, C callers with no device
 * allocator of their own, and serving loops whose device-memory budget is
 * fixed at start-up (cudaMalloc may also stall every stream on the device).
 * The scratch comes from a fixed array of EP_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library holds until the process
 * exits; nothing is allocated or freed.
 *
 * Arguments, outputs and error word: as ep_get_dispatch_layout, without the
 * workspace.  It always runs the multi-launch form (EP_LAYOUT_MULTI_LAUNCH),
 * whatever the batch size; the outputs are the same as those of every other
 * form.  Returns EP_ERR_CAPACITY, with nothing enqueued, when
 * ep_workspace_bytes(T, R, E) exceeds EP_NOALLOC_SCRATCH_BYTES (about 8 bytes
 * per token plus a small per-block term: roughly 800k tokens at 256 experts).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array, so calls that
 * overlap on the GPU (two streams, or two threads enqueueing at once) race
 * and must be serialised by the caller.  The array needs no clearing: each
 * call writes every scratch word before reading it.
 */
#define EP_NOALLOC_SCRATCH_BYTES (8u << 20)
ep_status_t ep_get_dispatch_layout_noalloc(const int64_t* topk_idx, int64_t num_tokens,
                                           int num_topk, int num_experts, int num_ranks,
                                           int32_t* num_tokens_per_rank,
                                           int32_t* num_tokens_per_expert,
                                           uint8_t* is_token_in_rank, int32_t* slot,
                                           int32_t* recv_base, int32_t* err_word,
                                           ep_stream_t stream);

/*
 * Copies P = recv_base[R] (device) into *host_total_rows and synchronises
 * `stream`.  The only synchronising call; use it to size the receive buffer
 * exactly, or skip it and pass a worst-case capacity of
 * T * min(K, R) rows to ep_dispatch.
 */
ep_status_t ep_layout_total_rows(const int32_t* recv_base, int num_ranks, int32_t* host_total_rows,
                                 ep_stream_t stream);

/*
 * dispatch ("Scope", Intranode: intranode_dispatch; the low-latency port:
 * dispatch<kUseFP8,...>).  For every pair (t, r) with slot[t][r] >= 0:
 *   use_fp8 == 0:  recv_x[slot] = x[t]                      (bf16 bit copy)
 *   use_fp8 == 1:  for each block b of 128 channels,
 *                    amax  = max |x[t][b*128 .. b*128+127]|   (float32)
 *                    a     = max(amax, 1e-4f)
 *                    recv_scales[slot][b] = a / 448          (float32, rounded once)
 *                    recv_x[slot][i] = E4M3(x[t][i] * (448 / a)),
 *                    with 448/a rounded once, one float32 multiply, and the
 *                    E4M3 conversion rounding to nearest even and saturating
 *                    to +-448; dequantise as code * scale.
 *   recv_src_idx[slot]         = t
 *   recv_topk_idx[slot][k]     = e_k - r*E_l if rank(e_k) == r, else -1
 *   recv_topk_weights[slot][k] = w[t][k]     if rank(e_k) == r, else 0.0f
 * In (device): x [T, H] bf16; topk_idx [T, K] int64; topk_weights [T, K]
 *   float32; slot [T, R] int32 from ep_get_dispatch_layout.
 *   num_tokens_per_expert [R, E] int32 from ep_get_dispatch_layout (nullable;
 *   only read to fill num_recv_tokens_per_expert).
 * Out (device): recv_x [capacity, H] bf16, or [capacity, H] E4M3 bytes with
 *   recv_scales [capacity, H/128] float32 (FP8 only, else may be NULL);
 *   recv_src_idx [capacity] int32, recv_topk_idx [capacity, K] int64,
 *   recv_topk_weights [capacity, K] float32 (each nullable: skipped if NULL);
 *   num_recv_tokens_per_expert [R, E_l] int32 (nullable): rows each
 *   destination rank receives per local expert, summed over source ranks.
 *   Rows >= P are not touched.
 * recv_capacity_rows: rows the caller allocated; a pair whose slot is >= it
 *   is skipped and sets EP_ERRBIT_CAPACITY in err_word.  With 0 rows nothing
 *   is written, and recv_x / recv_scales may be NULL (a shard whose tokens
 *   all go nowhere has an empty send buffer).
 * T need not be a multiple of R here (the slots place the rows), so the
 * sharded form below dispatches one rank's own tokens with this call.
 */
ep_status_t ep_dispatch(const void* x, int hidden, const int64_t* topk_idx,
                        const float* topk_weights, int64_t num_tokens, int num_topk,
                        int num_experts, int num_ranks, const int32_t* slot,
                        const int32_t* num_tokens_per_expert, int64_t recv_capacity_rows,
                        int use_fp8, void* recv_x, float* recv_scales, int32_t* recv_src_idx,
                        int64_t* recv_topk_idx, float* recv_topk_weights,
                        int32_t* num_recv_tokens_per_expert, int32_t* err_word,
                        ep_stream_t stream);

/*
 * combine ("Scope", Intranode: intranode_combine; the bench-accounting
 * commit: combine moves one copy per dispatched (token, rank) row back to
 * its owner).  For every token t:
 *   out[t] = bf16_rne( sum over k with e_k != -1 of
 *                      w[t][k] * float(y[slot[t][rank(e_k)]]) )
 * accumulated in float32; a token whose slots are all masked gives +0.
 * A rank named by several slots contributes its row once per slot.
 * With topk_weights == NULL the combine is the unweighted rank sum of the
 * high-throughput kernels (the expert stage has applied the weights):
 *   out[t] = bf16_rne( sum over ranks r with slot[t][r] >= 0 of y[slot[t][r]] ),
 * each destination rank's row once.
 * In (device): y [rows, H] bf16 in dispatch's row layout (expert outputs,
 *   one row per (token, rank) pair), with rows >= P = recv_base[R] (every
 *   row a slot names; the call takes no row count, so this is not checked);
 *   topk_idx [T, K] int64; topk_weights [T, K] float32 (nullable, see
 *   above); slot [T, R] int32 from ep_get_dispatch_layout.
 * Out (device): out [T, H] bf16, every element written.
 * err_word (device, nullable): EP_ERRBIT_BAD_EXPERT for ids outside [-1, E)
 *   (skipped), EP_ERRBIT_TIMEOUT if a bounded pipeline wait ran out (the
 *   output is then incomplete).
 * y rows are staged through shared memory with 1-D bulk (TMA) copies; y and
 * out must not overlap.  T need not be a multiple of R here.
 */
ep_status_t ep_combine(const void* y, int hidden, const int64_t* topk_idx,
                       const float* topk_weights, int64_t num_tokens, int num_topk,
                       int num_experts, int num_ranks, const int32_t* slot, void* out,
                       int32_t* err_word, ep_stream_t stream);

/* ------------------------------------------------------------------------
 * Layout and dispatch in one launch, for small (decode-size) batches.
 *
 * The same outputs as ep_get_dispatch_layout followed by ep_dispatch, from
 * one kernel launch: the pages run layout, the count exchange that fixes
 * the receive offsets (notify_dispatch, cached_notify: "[Not ready] MSCCLPP
 * EP implementation", section "Scope", Internode HT) and the data movement
 * as separate kernels; on one GPU the exchange becomes a wait inside one
 * grid.  The first blocks of the grid to start (picked by an atomic ticket,
 * so that no block waits on one that has not started) compute the layout
 * and meet at a bounded barrier; every block loads its share of x at once
 * and waits, bounded, for the layout before it scatters.  At these sizes the
 * layout is bound by latency, and the fused launch hides the x loads behind
 * it and saves the launches between the kernels.
 *
 * Fits (ep_layout_dispatch_fused_fits): 1 <= T <= 16384 and at most 8192
 * ballots, R * R * ceil(T_r / 32) <= 8192 (one 32-bit ballot per
 * destination and group of 32 tokens, groups never straddling two source
 * ranks): the 4096-token decode batch at 32 ranks, or 16384 tokens at 8
 * ranks.  Other sizes return EP_ERR_INVALID_ARG with nothing enqueued.
 * Arguments: those of ep_get_dispatch_layout (its outputs, all required)
 *   and of ep_dispatch (slot is written here and read back by the scatter;
 *   num_recv_tokens_per_expert is computed here, nullable), plus:
 * workspace (device): ep_layout_dispatch_fused_workspace_bytes(T, R, E)
 *   bytes (about 8 * R * R * ceil(T_r / 32)); EP_ERR_CAPACITY if smaller.
 *   No initialisation needed.
 * sync (device, EP_FUSED_SYNC_WORDS 64-bit words, 8-byte aligned): the
 *   grid's counters (start ticket, barrier, layout done, blocks left) and
 *   release flags, spread over 256-byte lines.  The caller zeroes them once;
 *   every launch leaves them zero again when its last block exits,
 *   including a launch whose waits ran out.  Launches that can overlap on
 *   the GPU need separate states.
 * err_word: as ep_get_dispatch_layout and ep_dispatch, plus
 *   EP_ERRBIT_TIMEOUT if a bounded wait (1 s) ran out: the layout or its
 *   barrier did not complete, and no row was dispatched.
 * ------------------------------------------------------------------------ */
#define EP_FUSED_SYNC_WORDS 640

/* 1 if (T, R, E) fits the one-launch layout + dispatch, else 0. */
int ep_layout_dispatch_fused_fits(int64_t num_tokens, int num_ranks, int num_experts);

/* Bytes of workspace ep_layout_dispatch_fused needs (0 if it does not fit). */
size_t ep_layout_dispatch_fused_workspace_bytes(int64_t num_tokens, int num_ranks,
                                                int num_experts);

ep_status_t ep_layout_dispatch_fused(
    const void* x, int hidden, const int64_t* topk_idx, const float* topk_weights,
    int64_t num_tokens, int num_topk, int num_experts, int num_ranks,
    int32_t* num_tokens_per_rank, int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank,
    int32_t* slot, int32_t* recv_base, int64_t recv_capacity_rows, int use_fp8, void* recv_x,
    float* recv_scales, int32_t* recv_src_idx, int64_t* recv_topk_idx, float* recv_topk_weights,
    int32_t* num_recv_tokens_per_expert, void* workspace, size_t workspace_bytes,
    uint64_t* sync, int32_t* err_word, ep_stream_t stream);

/*
 * Test hook for the bounded waits of ep_layout_dispatch_fused: the next
 * launch from this host thread leaves the first layout block's barrier
 * arrival out, so the barrier and the wait for the layout run out after
 * about 1 s each; the launch then reports EP_ERRBIT_TIMEOUT, dispatches
 * nothing, and still returns its state to zero.  One-shot; 0 cancels it.
 */
void ep_debug_set_fused_stall(int on);

/* ------------------------------------------------------------------------
 * Sharded form: one process and one GPU per rank ("[Not ready] MSCCLPP EP
 * implementation", section "Scope", Intranode: get_dispatch_layout on every
 * rank, then dispatch and combine over peer buffers; the internode
 * notify_dispatch commit: the count exchange that fixes the receiver-side
 * prefix matrices).  Rank s holds its own T tokens.  Per rank:
 *   1. ep_shard_layout: the rank's tokens as the one source of a layout
 *      with R destinations.  Its send buffer is packed destination-major in
 *      token order: destination r's rows are [send_base[r], send_base[r+1]).
 *   2. an all-gather of every rank's send_counts row gives counts [R, R]
 *      (counts[s][r] = tokens of rank s sent to rank r); ep_shard_offsets
 *      turns it into this rank's send and receive offsets.
 *   3. ep_dispatch with slot = send_slot (T need not be a multiple of R)
 *      fills the send buffer; an all-to-all-v moves run r to rank r, which
 *      stores the runs in source-rank order at its receive offsets.  Those
 *      are exactly the rows that destination r holds in the single-call
 *      layout (rows ordered by source rank, then token).  recv_src_idx then
 *      holds each row's token index within its source rank.
 *   4. combine: the reverse all-to-all-v brings every row back into the
 *      send buffer's layout, and ep_combine with slot = send_slot reduces it.
 * The collectives are the caller's (the Python package uses
 * torch.distributed); the library computes the layout, the offsets and the
 * rows.
 * ------------------------------------------------------------------------ */

/* Device scratch for ep_shard_layout (0 for invalid sizes). */
size_t ep_shard_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts);

/*
 * The layout of one rank's T tokens (any T >= 0) over R destinations.
 * In (device): topk_idx [T, K] int64.
 * Out (device), every element written:
 *   send_counts   [R] int32: tokens sent to each destination
 *   expert_counts [E] int32: slots naming each expert
 *   is_token_in_rank [T, R] uint8, send_slot [T, R] int32 (-1: not sent)
 *   send_base [R + 1] int32: exclusive prefix of send_counts
 * err_word, workspace (ep_shard_workspace_bytes), errors: as
 * ep_get_dispatch_layout.  Always the multi-launch kernels.
 */
ep_status_t ep_shard_layout(const int64_t* topk_idx, int64_t num_tokens, int num_topk,
                            int num_experts, int num_ranks, int32_t* send_counts,
                            int32_t* expert_counts, uint8_t* is_token_in_rank,
                            int32_t* send_slot, int32_t* send_base, int32_t* err_word,
                            void* workspace, size_t workspace_bytes, ep_stream_t stream);

/*
 * Host function (no GPU work).  counts (host) [R, R] int32: counts[s][r] =
 * tokens of rank s sent to rank r (every rank's send_counts, gathered).
 * Out (host): send_offsets [R + 1] int64, the exclusive prefix of
 * counts[rank][.] (this rank's runs in its send buffer); recv_offsets
 * [R + 1] int64, the exclusive prefix of counts[.][rank] (where the run
 * from each source rank lands in this rank's receive buffer;
 * recv_offsets[R] = rows received).  EP_ERR_INVALID_ARG for a negative
 * count or a rank outside [0, R).
 */
ep_status_t ep_shard_offsets(const int32_t* counts, int num_ranks, int rank,
                             int64_t* send_offsets, int64_t* recv_offsets);

/*
 * Host function (no GPU work).  expert_counts (host) [R, E] int32: every
 * rank's expert_counts row, gathered.  Out (host) [E/R] int32: the rows
 * this rank receives for each of its local experts (summed over sources),
 * the rank's row of ep_dispatch's num_recv_tokens_per_expert.
 */
ep_status_t ep_shard_recv_tokens_per_expert(const int32_t* expert_counts, int num_experts,
                                            int num_ranks, int rank, int32_t* out);

/* ------------------------------------------------------------------------
 * Low-latency (expert-major) layout: the receive layout of the low-latency
 * kernels ("[Not ready] MSCCLPP EP implementation", the low-latency port:
 * dispatch<kUseFP8,...> and combine over per-expert buffers indexed
 * [local_expert * num_ranks + dst_rank]).  Every unmasked top-k slot (t, k)
 * has its own row in the buffer of expert e = topk_idx[t][k]; expert e owns
 * rows [e*cap, (e+1)*cap) of one packed buffer of E*cap rows, packed by
 * source rank, then token, then k.
 * ------------------------------------------------------------------------ */

/* Device scratch for ep_ll_get_dispatch_layout (0 for invalid sizes). */
size_t ep_ll_workspace_bytes(int64_t num_tokens, int num_ranks, int num_experts);

/*
 * In (device): topk_idx [T, K] int64, -1 = masked.
 * expert_capacity: rows per expert (cap); cap * E < 2^31.  T is the largest
 *   count any expert can receive when each token names distinct experts.
 * Out (device):
 *   ll_slot [T, K] int32: row of slot (t, k), i.e.
 *     e*cap + ll_src_offset[e][src(t)]
 *     + #{(t', k') of src(t) before (t, k) in (token, k) order naming e};
 *     -1 for masked slots, ids outside [-1, E) (EP_ERRBIT_BAD_EXPERT) and
 *     positions >= cap (EP_ERRBIT_CAPACITY).
 *   ll_count [E] int32: slots naming each expert, over all sources
 *   ll_src_offset [E, R] int32 (nullable): first row of source s within
 *     expert e's rows (relative to e*cap).
 * workspace: ep_ll_workspace_bytes(T, R, E) bytes (EP_ERR_CAPACITY if less);
 *   unused (may be NULL) when ep_ll_layout_auto_single_launch(T, K, R, E).
 * Same as ep_ll_get_dispatch_layout_path(..., EP_LAYOUT_AUTO, stream).
 */
ep_status_t ep_ll_get_dispatch_layout(const int64_t* topk_idx, int64_t num_tokens, int num_topk,
                                      int num_experts, int num_ranks, int64_t expert_capacity,
                                      int32_t* ll_slot, int32_t* ll_count, int32_t* ll_src_offset,
                                      int32_t* err_word, void* workspace, size_t workspace_bytes,
                                      ep_stream_t stream);

/*
 * The expert-major layout's kernels, as for the rank-major layout
 * (ep_layout_path_t):
 *   EP_LAYOUT_MULTI_LAUNCH: three launches over the whole GPU (ranks within
 *     chunks of 16..128 tokens, a prefix over chunks per expert, rows), with
 *     scratch in the caller's workspace.  Any size.
 *   EP_LAYOUT_SINGLE_LAUNCH: one launch of one thread-block cluster of up to
 *     16 CTAs that exchange per-expert counts through distributed shared
 *     memory; no workspace.  Small batches only
 *     (ep_ll_layout_single_launch_fits): E <= 1024, and every warp of a
 *     cluster of 8 CTAs walks at most 2048 slots (roughly T * K <= 131072
 *     when R divides 64).
 *   EP_LAYOUT_AUTO: the single launch whenever it fits (measured faster
 *     at every size it takes); ep_ll_layout_auto_single_launch says which.
 *     As for the rank-major layout, AUTO falls back to the three launches
 *     if the device refuses the cluster and a usable workspace was passed.
 * Both give identical outputs.  EP_LAYOUT_SINGLE_LAUNCH on a batch that does
 * not fit (T = 0 included) returns EP_ERR_INVALID_ARG with nothing enqueued.
 */
int ep_ll_layout_single_launch_fits(int64_t num_tokens, int num_topk, int num_ranks,
                                    int num_experts);
int ep_ll_layout_auto_single_launch(int64_t num_tokens, int num_topk, int num_ranks,
                                    int num_experts);
ep_status_t ep_ll_get_dispatch_layout_path(const int64_t* topk_idx, int64_t num_tokens,
                                           int num_topk, int num_experts, int num_ranks,
                                           int64_t expert_capacity, int32_t* ll_slot,
                                           int32_t* ll_count, int32_t* ll_src_offset,
                                           int32_t* err_word, void* workspace,
                                           size_t workspace_bytes, int path, ep_stream_t stream);

/*
 * Low-latency dispatch: for every slot with ll_slot[t][k] >= 0, row
 * ll_slot[t][k] of recv_x receives token t, as a bf16 copy or (use_fp8) as
 * E4M3 codes with recv_scales per 128 channels, with the same rounding as
 * ep_dispatch; recv_src_idx[row] = t (nullable).  A token named by K experts
 * is written K times.
 * In (device): x [T, H] bf16, ll_slot [T, K].  Out (device): recv_x
 * [capacity, H] (bf16 or bytes), recv_scales [capacity, H/128] f32 (FP8),
 * recv_src_idx [capacity] int32.  Rows >= recv_capacity_rows are skipped
 * and set EP_ERRBIT_CAPACITY; with 0 rows recv_x / recv_scales may be NULL.
 */
ep_status_t ep_ll_dispatch(const void* x, int hidden, int64_t num_tokens, int num_topk,
                           const int32_t* ll_slot, int64_t recv_capacity_rows, int use_fp8,
                           void* recv_x, float* recv_scales, int32_t* recv_src_idx,
                           int32_t* err_word, ep_stream_t stream);

/*
 * Low-latency combine: out[t] = bf16_rne( sum over slots k with
 * ll_slot[t][k] >= 0 of w[t][k] * float(y[ll_slot[t][k]]) ), accumulated in
 * float32 (each expert's output row read once; with topk_weights == NULL
 * every slot weighs 1).  In (device): y [rows, H] bf16 in the expert-major
 * layout, with rows above every row ll_slot names (E * cap suffices; not
 * checked), topk_weights [T, K] f32 (nullable), ll_slot [T, K].  Out
 * (device): out [T, H] bf16, every element written.  Staging as ep_combine.
 */
ep_status_t ep_ll_combine(const void* y, int hidden, const float* topk_weights,
                          int64_t num_tokens, int num_topk, const int32_t* ll_slot, void* out,
                          int32_t* err_word, ep_stream_t stream);

/* ------------------------------------------------------------------------
 * Dynamically scheduled combine.  The combine grid is persistent, and its
 * blocks take the tokens in batches of a few.  Each block's first batch is
 * fixed.  ep_combine and ep_ll_combine hand out the rest statically (block b
 * takes every grid-th batch).  The _sched forms below hand out the rest on
 * demand from a counter in device memory, so a block that the memory system
 * serves faster takes more batches, and all blocks finish together.  On one
 * GB300 this took skewed routing (131072 tokens) from 1586 to 1550 us per
 * layout -> dispatch -> combine step, and Mixtral-shaped routing from 978 to
 * 945 us.  The outputs are identical: each token is summed in the same
 * order whichever block takes it.
 *
 * sched (device, EP_COMBINE_SCHED_WORDS 64-bit words, 8-byte aligned): the
 * counter state.  The caller zeroes it once after allocating it.  Every
 * launch leaves it zero again when its last block exits, including a launch
 * that ran out of a bounded wait.  So one state serves any number of
 * launches in order on one stream, and inside a CUDA graph.  Two combines
 * that can run at the same time (other streams, a graph replayed beside
 * eager calls) need separate states: a shared state would split the tokens
 * between them and leave both outputs incomplete.  A launch checks, as its
 * blocks leave, that it made exactly the claims a launch alone makes and
 * that no claim or exit came from elsewhere; if not (a shared state, or one
 * that was not zero at launch) it sets EP_ERRBIT_SCHED in err_word, and its
 * output may be missing tokens.  A shared state is not always caught (a
 * launch that runs entirely between the other's claims sees nothing amiss,
 * but then neither output is affected).  A NULL sched is the static
 * schedule of ep_combine.  A batch small enough that every block has only
 * its first batch is scheduled statically too, and leaves the state
 * untouched.  Other arguments and errors: as ep_combine and ep_ll_combine.
 * ------------------------------------------------------------------------ */
#define EP_COMBINE_SCHED_WORDS 2

ep_status_t ep_combine_sched(const void* y, int hidden, const int64_t* topk_idx,
                             const float* topk_weights, int64_t num_tokens, int num_topk,
                             int num_experts, int num_ranks, const int32_t* slot, void* out,
                             uint64_t* sched, int32_t* err_word, ep_stream_t stream);
ep_status_t ep_ll_combine_sched(const void* y, int hidden, const float* topk_weights,
                                int64_t num_tokens, int num_topk, const int32_t* ll_slot,
                                void* out, uint64_t* sched, int32_t* err_word,
                                ep_stream_t stream);

/*
 * Test hook for the bounded waits of the combine pipeline (ep_combine,
 * ep_ll_combine and their _sched forms).  The next combine launched from this host thread leaves
 * pipeline unit `unit` of CTA 0 unarmed, so the waits on it run out after
 * about 1 s.  The launch then reports EP_ERRBIT_TIMEOUT in the error word,
 * its output is incomplete, and it returns.  The hook is one-shot; -1
 * cancels it.  It faults, traps and hangs nothing, and exists only so that
 * tests can exercise the timeout path.
 */
void ep_debug_set_combine_stall(int unit);

/*
 * Test hook for the FP8 payload conversion (the pages give the FP8 cast only
 * by name, kUseFP8 in the low-latency port of "[Not ready] MSCCLPP EP
 * implementation"; this hook has no counterpart there).  out[i] receives the
 * E4M3 code that the FP8 dispatch's conversion (round to nearest even,
 * saturating to +-448) gives the float32 whose bit pattern is first + i, for
 * 0 <= i < n, so that a test can compare the oracle's encoder with the
 * device on every float32.  n % 4 == 0 and first + n <= 2^32, else
 * EP_ERR_INVALID_ARG; out: device, n bytes, 4-byte aligned.  Asynchronous
 * on `stream`.
 */
ep_status_t ep_debug_e4m3_range(uint32_t first, int64_t n, uint8_t* out, ep_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_H_ */
