/*
 * kvm.h - C ABI of libkvm.so: the chunked forward of a Key-Value Means (KVM)
 * attention layer on one NVIDIA GB300 GPU (sm_103a).
 *
 * Source of the operation: "Key-Value Means" (gist.science technical
 * summary, Methodology and Core mechanisms 1-5; chatpaper.ai abstract).
 * A KVM layer is one softmax attention layer whose keys are
 *   - a block-sliding window of recent tokens with RoPE on both sides
 *     (Core mechanism 1 and 4), and
 *   - a compressed state of slots read "just in time": key = LayerNorm of the
 *     slot's mean key with the rotary dims zeroed, value = the slot's read
 *     radius rho_i times the unit direction of its value sum (Core
 *     mechanisms 2 and 4), read with the unrotated query,
 * combined in one softmax.  Each chunk of C tokens that leaves the window is
 * folded into the state (Core mechanism 1): the first S tokens of the
 * sequence found protected sink slots (Core mechanism 5); the most surprising
 * tokens (lowest best cosine to the current slots) are appended as new slots
 * up to the growth schedule's capacity (Core mechanism 3); every other token
 * goes to the slot whose LayerNorm'd key has the highest cosine with it (ties
 * to the lowest slot index) and adds its gate-weighted key and value to that
 * slot's raw sums and 1 to its count (Core mechanism 2; lay part "smart
 * merge").
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers, contiguous, row-major.
 *     Prefill tensors are [B, H, N, d]; decode tensors are [B, H, d];
 *     gates are fp32 [B, H, N] / [B, H].  Element type of q, k, v, out and of
 *     the window ring is the config's dtype (bf16 or fp32).  Keys are passed
 *     UNROTATED: the library applies RoPE itself (the state needs raw keys).
 *   - The caller owns every buffer, including the workspace.  The layer owns
 *     only host-side metadata.
 *   - Calls enqueue work on the given CUDA stream (NULL = legacy default
 *     stream) and return without synchronising.  Arguments are validated
 *     before anything is enqueued: a call that fails validation enqueued
 *     nothing; one that returns KVM_ERR_CUDA may have enqueued its earlier
 *     launches.  Errors raised on the device are latched in a status word in
 *     the workspace and reported by kvm_layer_sync.
 *   - No entry point aborts the process.  kvm_last_error gives a message.
 *   - A layer may be used from one host thread at a time.
 */
#ifndef KVM_H
#define KVM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVM_OK = 0,
    KVM_ERR_INVALID_ARG = 1,   /* bad pointer, size, shape or config value */
    KVM_ERR_UNSUPPORTED = 2,   /* valid config this library does not implement */
    KVM_ERR_CAPACITY = 3,      /* the growth schedule would exceed max_slots / max_tokens */
    KVM_ERR_WORKSPACE = 4,     /* workspace too small or misaligned */
    KVM_ERR_CUDA = 5,          /* a CUDA runtime call failed */
    KVM_ERR_TIMEOUT = 6,       /* a bounded device-side wait expired */
    KVM_ERR_DEVICE = 7         /* a device-side check failed */
} kvm_status;

typedef enum { KVM_BF16 = 0, KVM_FP32 = 1 } kvm_dtype;

/* Growth schedule (Core mechanism 3).  FIXED: capacity = max_slots.
 * POWER: capacity after t overflowed tokens = n_sinks + ceil(coef * t^expo)
 * (the "sqrt" state is expo = 0.5, coef = 4).  Capacities count sink slots. */
typedef enum { KVM_SCHED_FIXED = 0, KVM_SCHED_POWER = 1 } kvm_sched;

/* Ablation switches ("Key-Value Means", technical summary, Experimental
 * results, ablation studies: removing the value-length normalisation, the sink
 * protection or the merge gate).  KVM_FLAG_NO_VALUE_NORM: the state's read
 * value is the mean of its gate-weighted members, sum_v / count, instead of
 * rho * unit(sum_v).  No sink protection is n_sinks = 0 (every overflowed token
 * is an ordinary merge or append candidate); no merge gate is a gate of ones. */
#define KVM_FLAG_NO_VALUE_NORM 1

typedef struct {
    int32_t batch;       /* B >= 1 */
    int32_t heads;       /* H >= 1; one state per (batch, head) */
    int32_t head_dim;    /* d; this library supports 64 */
    int32_t rope_dims;   /* r: RoPE on dims [0, r), rotate-half pairs (i, i + r/2); even, 0..d */
    float rope_theta;    /* RoPE base, e.g. 10000 */
    int32_t chunk;       /* C: multiple of 16, 16..256 */
    int32_t window;      /* W: multiple of C, >= 0; a query in chunk c sees chunks c-W/C..c */
    int32_t n_sinks;     /* S: 0..C protected sink slots (the first S tokens) */
    int32_t sched;       /* kvm_sched */
    int32_t max_slots;   /* M: slot rows reserved per (batch, head), S+1..4096 */
    float coef, expo;    /* POWER schedule parameters (coef > 0, 0 < expo <= 1) */
    float ln_eps;        /* LayerNorm epsilon for the state keys, e.g. 1e-5 */
    int32_t dtype;       /* kvm_dtype of q, k, v, out and the window ring */
    int32_t max_tokens;  /* longest sequence the layer will see (prefill + decode) */
    int32_t flags;       /* KVM_FLAG_* ablation switches; 0 = the method as described */
} kvm_config;

typedef struct kvm_layer kvm_layer;

/* State of every (batch, head), for export/import (checkpoint / resume).
 * Device buffers owned by the caller:
 *   sum_k, sum_v : fp32 [B, H, max_slots, d] raw gate-weighted sums
 *   counts       : int32 [B, H, max_slots]  member tokens per slot
 *   rho          : fp32 [B, H, max_slots]   read radius per slot
 *   ring_k, ring_v : dtype [B, H, W + C, d] unrotated window tokens; the token
 *                  at position p sits in row p mod (W + C)
 *   ring_g       : fp32 [B, H, W + C]        their merge gates
 * Host scalars (identical for every (batch, head): the schedule is data
 * independent): n_slots, n_overflow (tokens folded so far), pos (next
 * position).  Rows >= n_slots of the slot arrays, and ring rows that hold no
 * token (positions outside n_overflow .. pos-1), are unspecified on export
 * and ignored on import. */
typedef struct {
    float* sum_k;
    float* sum_v;
    int32_t* counts;
    float* rho;
    void* ring_k;
    void* ring_v;
    float* ring_g;
    int64_t n_slots;
    int64_t n_overflow;
    int64_t pos;
} kvm_state_bufs;

/* Optional per-fold-event record of a prefill (device buffers, may be NULL
 * individually).  Event e folds chunk e (tokens e*C .. e*C+C-1); only events
 * e < max_events are recorded.  Shapes [B, H, max_events, C]:
 *   assign  : int32 slot the token went to
 *   kind    : int32 0 merged, 1 appended as a new slot, 2 founded a sink slot
 *   max_sim : fp32 surprise score (best cosine to the slots that existed
 *             before this event's appends; -inf if none; NaN for sinks)
 *   gap     : fp32 top-2 cosine gap of a merged token's argmax (+inf with a
 *             single candidate slot; NaN for appended tokens and sinks) */
typedef struct {
    int32_t* assign;
    int32_t* kind;
    float* max_sim;
    float* gap;
    int64_t max_events;
    /* Test hook of the failure path: when nonzero, the on-chip fold chain (bf16,
     * chunk <= 128, max_slots <= 256) waits for a chunk copy that is never
     * issued; its bounded wait expires after about two seconds, the kernel
     * drains and exits, and kvm_layer_sync reports KVM_ERR_TIMEOUT.  The
     * prefill's outputs are then meaningless; the context stays usable. */
    int32_t test_stall;
} kvm_debug;

/* Bytes of device workspace a layer with this config needs (0 if the config
 * is invalid; kvm_last_error(NULL) then says why).  Alignment: 256 bytes. */
size_t kvm_workspace_bytes(const kvm_config* cfg);

/* Validate cfg, carve the caller's workspace (device pointer, >= the size
 * above, 256-byte aligned) and build the RoPE and schedule tables in it
 * (synchronous copies on the legacy stream).  On success *out receives a new
 * layer in the empty state at position 0. */
kvm_status kvm_layer_create(const kvm_config* cfg, void* dev_workspace, size_t bytes,
                            kvm_layer** out);

/* Chunked prefill (Core mechanism 1; abstract: chunk-wise parallel prefill).
 * Resets the layer to the empty state at position 0, then computes, for
 * every (b, h) and token p < n_tokens, the KVM attention output of query p
 * into out, folding chunk c - W/C - 1 into the state before chunk c runs.
 * q, k, v, out: dtype [B, H, n_tokens, d]; gate: fp32 [B, H, n_tokens].
 * 0 <= n_tokens <= max_tokens.  On return of the work the layer holds the
 * state and window ring after n_tokens tokens (ready for kvm_decode_step).
 * dbg may be NULL.  KVM_ERR_CAPACITY if the schedule exceeds max_slots. */
kvm_status kvm_prefill(kvm_layer* layer, const void* q, const void* k, const void* v,
                       const float* gate, int64_t n_tokens, void* out, void* cuda_stream,
                       const kvm_debug* dbg);

/* One decode step at the layer's position p (then p + 1): if p is the first
 * token of chunk c >= W/C + 1, chunk c - W/C - 1 is folded from the window
 * ring first; the new unrotated k, v and gate enter the ring; the query
 * attends to the state and to tokens (c - W/C)*C .. p.  Equal to row p of a
 * prefill of p + 1 tokens.  q, k, v, out: dtype [B, H, d]; gate fp32 [B, H]. */
kvm_status kvm_decode_step(kvm_layer* layer, const void* q, const void* k, const void* v,
                           const float* gate, void* out, void* cuda_stream);

/* Copy the layer's state and window ring into dst (device-to-device, async
 * on the stream) and fill dst's host scalars. */
kvm_status kvm_state_export(const kvm_layer* layer, kvm_state_bufs* dst, void* cuda_stream);

/* Replace the layer's state and window ring by src (device-to-device, async)
 * and recompute the state's read view.  src->n_slots <= max_slots,
 * 0 <= src->n_overflow <= src->pos <= max_tokens, counts >= 1 for rows < n_slots. */
kvm_status kvm_state_import(kvm_layer* layer, const kvm_state_bufs* src, void* cuda_stream);

/* Wait for the layer's last stream, then report (and clear) the device-side
 * status word: KVM_OK, KVM_ERR_TIMEOUT or KVM_ERR_DEVICE. */
kvm_status kvm_layer_sync(kvm_layer* layer);

/* Message of the layer's last error (or, with NULL, of the last failed
 * kvm_workspace_bytes / kvm_layer_create on this thread).  Never NULL. */
const char* kvm_last_error(const kvm_layer* layer);

/* Device time of the layer's kernels, by phase, accumulated between
 * kvm_layer_set_timing(layer, 1) and kvm_layer_get_timing.  Measured with CUDA
 * events recorded on the launch stream immediately before and after each
 * kernel: a phase's time is its kernels' device duration (the start event
 * completes only when the stream reaches the kernel, so queueing behind earlier
 * work is not counted).  In an overlapped prefill (kvm_layer_set_overlap) one
 * fold interval spans the whole chain, from the start of its first segment to
 * the end of its last, and the attention, split over several launches that
 * run beside the chain, is not timed. */
typedef struct {
    double fold_ms;      /* fold-chain kernels (prefill chains and decode-boundary folds) */
    double attn_ms;      /* prefill attention kernels (sequential prefill only) */
    double decode_ms;    /* decode attention kernels */
    double other_ms;     /* ring fill, state renormalisation */
    int64_t fold_launches, attn_launches, decode_launches, other_launches;  /* timed intervals */
    int64_t kernels;     /* every kernel the layer launched, timed or not */
    double proj_ms;      /* projection GEMMs of kvm_layer_forward */
    int64_t proj_launches;
} kvm_timing;

/* Enable (1) or disable (0) per-kernel timing; enabling resets the totals.
 * Timing adds two event records per kernel launch. */
kvm_status kvm_layer_set_timing(kvm_layer* layer, int enable);

/* Wait for the recorded events and return the totals since timing was enabled. */
kvm_status kvm_layer_get_timing(kvm_layer* layer, kvm_timing* out);

/* Overlapped prefill.  The fold chain runs one CTA per (b,h) row, each on an SM
 * of its own, for the whole chain, while the attention of chunk c needs only
 * the fold events before it ("Key-Value Means", technical summary, Core
 * mechanism 4: attention of a chunk overlaps the state update from the chunk
 * that left the window).  With overlap on, kvm_prefill splits the GPU's SMs
 * into two disjoint partitions (CUDA green contexts): the chain runs in
 * `segments` launches on the first (at least B*H SMs), and after each segment
 * the attention of every chunk it has made ready runs on the second; what is
 * left of the attention then runs on all SMs.  Results are identical to the
 * sequential prefill (same kernels, same per-tile arithmetic).
 *
 * segments: 0 = never overlap; n > 0 = n fold segments (at most 16, at most
 * the number of fold events); < 0 = automatic (the default: 2 segments when
 * the state fits on chip (max_slots <= 256, chunk 128), where each segment
 * restart reloads the state; 8 with the streamed state, which restarts for
 * free).  Overlap applies only to the tensor-core paths (bf16, chunk 128 or
 * 256, max_slots <= 4096), without a debug record, with at least 2 fold
 * events, and when the device leaves at least one SM partition beside B*H
 * SMs, and not while a CUDA injection library (a profiler) is attached;
 * otherwise the prefill runs sequentially.  The partition is made on first
 * use and released by kvm_layer_destroy. */
kvm_status kvm_layer_set_overlap(kvm_layer* layer, int32_t segments);

/* Fold segments the layer's last kvm_prefill ran with (0: sequential). */
kvm_status kvm_layer_get_overlap(const kvm_layer* layer, int32_t* last_segments);

/* Whole-layer forward ("Key-Value Means", technical summary, Methodology: the
 * layer's own projections around the KVM attention; the merge gate is produced
 * inside the layer from its input).  For x [B, n_tokens, d_model] bf16:
 *   [q | k | v | gate_logit] = x * w_in^T, w_in [3*H*64 + H, d_model] bf16
 *     (rows: q of heads 0..H-1, then k, then v, each 64 rows per head, then one
 *     gate row per head); gate = sigmoid(gate_logit), fused in the GEMM epilogue;
 *   o = the KVM attention of this layer (kvm_prefill) on q, k, v, gate;
 *   y = o_flat * w_out^T, o_flat [B, n_tokens, H*64] (head-major features),
 *     w_out [d_model, H*64] bf16, y [B, n_tokens, d_model] bf16.
 * Only for bf16 layers; d_model a positive multiple of 64; x, w_in, w_out and y
 * 16-byte aligned.  The projections run on the tensor cores (tcgen05, fp32
 * accumulation).  scratch (device, 256-byte aligned, at least
 * kvm_forward_scratch_bytes) receives, in order and each 256-byte aligned:
 * q, k, v, o (bf16 [B, H, n_tokens, 64]) and gate (fp32 [B, H, n_tokens]); they
 * stay readable after the call.  The layer's state afterwards is that of
 * kvm_prefill.  Asynchronous on the stream; 0 on invalid arguments. */
size_t kvm_forward_scratch_bytes(const kvm_config* cfg, int32_t d_model, int64_t n_tokens);
kvm_status kvm_layer_forward(kvm_layer* layer, int32_t d_model, const void* x, const void* w_in,
                             const void* w_out, int64_t n_tokens, void* y, void* scratch,
                             size_t scratch_bytes, void* cuda_stream);

/* Size of the static device scratch behind kvm_prefill_noalloc: 32 MiB. */
#define KVM_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* kvm_prefill_noalloc - a one-shot prefill that allocates no memory.
 * This entry point has no counterpart in the paper; it exists for callers
 * that may not allocate device memory themselves: a plugin running inside an
 * inference server or host framework that owns all device memory through
 * its own pool and forbids direct cudaMalloc/cudaFree, or a latency-critical
 * loop that cannot afford the device synchronisation an allocation implies.
 * Such callers cannot hand kvm_layer_create a workspace.
 *
 * Computes what kvm_prefill computes into out, with the same kernels and the
 * same RoPE and schedule tables, so the outputs are identical bit for bit,
 * for q, k, v, out: dtype [B, H, n_tokens, d] and gate fp32 [B, H, n_tokens]
 * buffers owned by the caller, but keeps no layer: nothing is left for a
 * later decode, export or debug record.  The call runs on the CURRENT device
 * (cudaGetDevice): every buffer must be device memory of that device, else
 * KVM_ERR_INVALID_ARG before anything is enqueued.  Its scratch (state,
 * read-view snapshots, RoPE and schedule tables) is a file-scope device array
 * of KVM_NOALLOC_SCRATCH_BYTES bytes that every GPU loading this library
 * holds until the process exits; with CUDA's lazy module loading the array
 * may be reserved only when this library's device code is first used on the
 * device (possibly this call).  A call whose scratch would exceed it (or that
 * would fold more than 1024 chunks) returns KVM_ERR_WORKSPACE with the
 * required size in kvm_last_error(NULL), before enqueuing anything.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any CUDA
 * stream capture.  Every call reuses the same array and clears what must
 * start at zero; calls whose GPU work overlaps in time (several streams or
 * host threads) race on it and must be serialised by the caller.  Calls no
 * cudaMalloc, cudaFree or other allocating routine.  Errors are reported
 * through kvm_last_error(NULL); device-side status (a bounded wait that
 * expired) is not reported, and the outputs of such a call are undefined. */
kvm_status kvm_prefill_noalloc(const kvm_config* cfg, const void* q, const void* k, const void* v,
                               const float* gate, int64_t n_tokens, void* out, void* cuda_stream);

/* Backward of kvm_prefill for chunk-parallel training ("Key-Value Means",
 * technical summary, Contributions: the layer trains chunk-parallel).  The
 * pages do not say how the gradient passes the winner-take-all assignment;
 * here the fold's discrete decisions (the slot of every merged token, the
 * surprise-selected appends, the sinks) are constants from the forward, and
 * the gradient flows through the attention, RoPE, the just-in-time read of
 * the state (LayerNorm(sum_k / count) with the rotary dims zeroed,
 * rho * unit(sum_v)), the gate-weighted member sums and the founders' read
 * radius rho = |v|.  Counts carry no gradient.
 *
 * Call it after the layer's kvm_prefill of the same q, k, v, gate and
 * n_tokens, with no other prefill on the layer in between (it reads the
 * forward's per-event read rows from the workspace): out is that prefill's
 * output, record its debug record (assign and kind of every fold event; NULL
 * allowed when no event folded), dout the loss gradient with respect to out
 * (dtype [B, H, n_tokens, d]).  Outputs fp32: dq, dk, dv [B, H, n_tokens, d],
 * dgate [B, H, n_tokens]; every element is written.  scratch: device memory of
 * kvm_backward_scratch_bytes(cfg, n_tokens) bytes, 256-byte aligned.  Chunks of
 * at most 256 tokens and rope_dims a multiple of 4 (else KVM_ERR_UNSUPPORTED).
 * KVM_ERR_INVALID_ARG when the layer's last prefill was not of n_tokens tokens
 * or the record is missing or shorter than the fold events; a record entry
 * that names no slot of its event's state is skipped and makes kvm_layer_sync
 * report KVM_ERR_DEVICE. */
size_t kvm_backward_scratch_bytes(const kvm_config* cfg, int64_t n_tokens);
kvm_status kvm_prefill_backward(kvm_layer* layer, const void* q, const void* k, const void* v,
                                const float* gate, const void* out, const void* dout,
                                const kvm_debug* record, int64_t n_tokens, float* dq, float* dk,
                                float* dv, float* dgate, void* scratch, size_t scratch_bytes,
                                void* cuda_stream);

/* Free the layer's host metadata.  The workspace stays the caller's. */
void kvm_layer_destroy(kvm_layer* layer);

#ifdef __cplusplus
}
#endif

#endif /* KVM_H */
