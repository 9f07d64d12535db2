/*
 * moe.h -- C ABI of the GB300 (sm_103a) gated Mixture-of-Experts FFN layer, forward pass.
 *
 * One layer, one GPU, every expert resident in device memory:
 *
 *   gate      logits[t,e] = sum_i x[t,i] Wg[i,e] (fp32), softmax over experts, top-1 or
 *             top-2 by logit.  Each token is sent to experts by a gating function
 *             (DeepSpeed-MoE review, "MoE based NLG Model Architecture").
 *   dispatch  capacity C = ceil(cf T / E) per expert; assignments taken in token order,
 *             those past an expert's capacity are dropped; compact slots per expert.
 *   experts   FFN_e(x) = GeLU_tanh(x W1[e]) W2[e], fp16 operands, fp32 accumulation.
 *   combine   out[t] = sum_j w[t,j] FFN_{e_j}(x_t) over kept assignments: Top2-MoE sums the
 *             outputs of two experts (same review, "Phenomenon2").
 *   residual  mlp_type 'residual' (DeepSpeed-MoE Inference wiki, "PR-MoE 최적화로 더 낮은 비용";
 *             PR-MoE in the review) adds a fixed dense MLP GeLU(x Wr1) Wr2 to the routed
 *             expert's output (review, "Phenomenon2": Residual-MoE).
 *
 * The pages fix none of the exact formulas; the readings used are stated beside each call
 * (no biases; fp32 fused-multiply-add chain for the logits; ties go to the lower expert
 * index; top-1 weight = softmax probability of the chosen expert; top-2 weights are the two
 * probabilities renormalised to sum 1 before drops and not after; capacity independent of
 * k; dropped assignments contribute zero; GeLU in its tanh form).
 *
 * Conventions for every call:
 *   - Matrices are dense row-major.  Shapes are given as [rows, cols].
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless stated.  The
 *     library never allocates or frees device memory, keeps no pointer after a call
 *     returns, and never synchronises `stream` (moe_status_read excepted).
 *   - All work is enqueued on `stream` (a cudaStream_t; 0 is the legacy default stream);
 *     calls return once the work is enqueued.
 *   - Return value: a moe_status.  Argument errors are detected on the host before anything
 *     is enqueued, and nothing is written then.  MOE_ERR_CUDA reports a failed launch.
 *     Errors found on the device while a call runs (a bounded wait that gave up) are
 *     recorded in the workspace's status word and read with moe_status_read.
 *   - No call throws across this boundary; all are safe to call from any host thread as
 *     long as concurrent calls use different workspaces and outputs.
 *   - T = 0 (an empty batch) is valid: the call enqueues nothing and returns MOE_OK.
 *
 * Supported shapes: E <= 1024, k in {1, 2}, k <= E.  MOE_F16 (tensor-core path): d, f and
 * f_res multiples of 128.  MOE_F32 (SIMT path): d and f multiples of 4.  Every pointer
 * 16-byte aligned.  Otherwise MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t; /* same type as cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* a size, pointer, k, capacity factor or enum is invalid */
  MOE_ERR_UNSUPPORTED = 2,    /* valid, but a shape / alignment this build does not run */
  MOE_ERR_WORKSPACE = 3,      /* workspace missing or smaller than moe_workspace_size */
  MOE_ERR_CUDA = 4,           /* a CUDA launch or API call failed */
  MOE_ERR_TIMEOUT = 5,        /* device side: a bounded wait gave up (status word) */
  MOE_ERR_DEVICE_BOUNDS = 6   /* device side: an index failed its bounds check (status word):
                                 the expert FFN's offsets left [0, S_max] or decreased, or a
                                 perm entry left [0, T).  The offending index is clamped (no
                                 access leaves its buffer) and the outputs are unspecified.
                                 moe_combine's slot_of is not checked (the call has no bound
                                 for it): pass it as moe_dispatch writes it */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_F16 = 1 } moe_dtype;           /* activations and expert weights */
typedef enum { MOE_MLP_STANDARD = 0, MOE_MLP_RESIDUAL = 1 } moe_mlp_type;

/*
 * Capacity per expert: C = ceil(cf * T / E), with cf*T and the division evaluated in
 * double.  The pages define no per-expert token capacity: the "expert capacity" of the
 * DeepSpeed-MoE review ("Phenomenon2") is the number of experts each token passes through
 * (k here; Top2-MoE doubles it).  The token capacity of an expert is therefore a reading:
 * the capacity-factor rule above, with overflow dropped in token order.  Host only.
 * cf = +INFINITY selects the dropless mode: C = T, so no assignment is dropped and a hot
 * expert's rows are spread over as many tiles as it needs (the single-GPU counterpart of the
 * physical expert replicas of "Fast MoE Inference via Predictive Prefetching and Expert
 * Replication", methodology).  Every entry taking a capacity factor accepts it.
 * Returns C (0 when T = 0), or -1 when T < 0, E < 1, cf <= 0 or NaN, or C > 2^31-1.
 */
MOE_API int moe_capacity(int T, int E, float capacity_factor);

/*
 * Bytes of workspace that moe_layer_forward needs for this shape (and enough for
 * moe_expert_ffn of the same shape).  Host only; writes *bytes.  f_res is ignored for
 * MOE_MLP_STANDARD.  Returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED as the calls would.
 */
MOE_API moe_status moe_workspace_size(int T, int d, int f, int E, int k, float capacity_factor,
                              moe_mlp_type mlp_type, int f_res, moe_dtype dtype, size_t* bytes);

/*
 * Gate: logits, softmax and top-k (DeepSpeed-MoE review, "MoE based NLG Model
 * Architecture": tokens reach experts through a gating function; "Phenomenon2": Top2).
 *   tokens     [T, d] in `dtype` (f16 values are widened exactly to f32).
 *   Wg         [d, E] float32.
 *   logits_in  nullable [T, E] float32: when given, the logits are taken from here and
 *              tokens / Wg are not read (may be NULL then).
 *   logits_out [T, E] float32: the logits used; required when logits_in is NULL (it holds
 *              them), otherwise nullable (a copy of logits_in).
 *   probs_out  nullable [T, E] float32: softmax over E.
 *   topk_idx   [T, k] int32: experts by descending logit, ties to the lower index.
 *   topk_w     [T, k] float32: k = 1: p[e1]; k = 2: p[e_j] / (p[e1] + p[e2]).
 * The logits are the fp32 chain acc = fmaf(x[t,i], Wg[i,e], acc), i ascending from +0, so
 * they (and hence routing) are reproducible bit for bit by any IEEE implementation.
 */
MOE_API moe_status moe_gate_topk(const void* tokens, moe_dtype dtype, const float* Wg,
                                 const float* logits_in, int T, int d, int E, int k, float* logits_out,
                         float* probs_out, int32_t* topk_idx, float* topk_w, moe_stream_t stream);

/*
 * Capacity-limited dispatch (reading: token-major order, capacity ceil(cf T / E)).
 *   topk_idx   [T, k] int32 experts; an index outside [0, E) is not counted and its
 *              assignment is dropped (slot_of = -1).
 *   counts_raw [E]    assignments per expert before the capacity cut.
 *   kept       [E]    min(counts_raw, C).
 *   offsets    [E+1]  exclusive scan of kept; offsets[E] = S, the number of kept slots.
 *   perm       [min(T k, E C)]  perm[s] = token of slot s; expert e owns slots
 *                               offsets[e] .. offsets[e+1]-1 in token order.  Entries >= S
 *                               are not written.
 *   slot_of    [T, k] slot of assignment (t, j), or -1 when it was dropped.
 * Pure integer work: results are unique and bit-exact.  One thread block; no atomics.
 */
MOE_API moe_status moe_dispatch(const int32_t* topk_idx, int T, int E, int k, float capacity_factor,
                        int32_t* counts_raw, int32_t* kept, int32_t* offsets, int32_t* perm,
                        int32_t* slot_of, moe_stream_t stream);

/*
 * Dispatch of one shard of a token-sharded batch, with the whole batch's capacity rule.
 * The pages have no multi-GPU data-parallel layout of this layer (their own design is expert
 * parallelism); this entry is the one exchange step that token sharding needs so that
 * routing does not depend on how the batch is split (capacity as moe_capacity computes it,
 * ceil(cf T / E) of the whole batch, with drops in token order).
 *   The batch of T_global tokens is split over n_ranks callers in token order; this call
 *   holds shard `rank` (T tokens).  counts_all [n_ranks, E] int32 (device; nullable when
 *   rank == 0): the counts_raw of every shard in rank order, exchanged by the caller (for
 *   example an all_gather of each shard's counts_raw from moe_dispatch).
 *   C = ceil(cf T_global / E).  An assignment is kept iff (assignments to its expert in
 *   earlier shards) + (its rank within this shard) < C, so the kept / dropped decisions are
 *   those of moe_dispatch on the whole batch.
 *   Outputs as moe_dispatch, local to the shard: counts_raw / kept per expert for this
 *   shard, offsets / perm / slot_of over this shard's compact slots (perm holds local token
 *   indices), perm sized min(T k, E C).
 * Errors: MOE_ERR_INVALID_ARG for T_global < T, rank outside [0, n_ranks), or counts_all
 * NULL with rank > 0; otherwise as moe_dispatch.  T = 0 is a valid no-op.
 */
MOE_API moe_status moe_dispatch_sharded(const int32_t* topk_idx, int T, int E, int k,
                                        float capacity_factor, int T_global,
                                        const int32_t* counts_all, int n_ranks, int rank,
                                        int32_t* counts_raw, int32_t* kept, int32_t* offsets,
                                        int32_t* perm, int32_t* slot_of, moe_stream_t stream);

/*
 * Grouped expert FFN over the dispatched slots, unscaled:
 *   expert_out[s, :] = GeLU_tanh(tokens[perm[s], :] W1[e]) W2[e]   for s in expert e's slots.
 *   tokens [T, d], W1 [E, d, f], W2 [E, f, d], expert_out [S_max, d]: all in `dtype`.
 *   perm, offsets: as written by moe_dispatch.  S_max >= offsets[E] bounds the slot count
 *   (min(T k, E C) always suffices).  Rows >= offsets[E] of expert_out are not written.
 *   Bounds: the kernels clamp offsets to [0, S_max], so no row >= S_max of expert_out or of
 *   the workspace is ever written; offsets outside that range or decreasing, and perm
 *   entries outside [0, T), record MOE_ERR_DEVICE_BOUNDS in the workspace's status word
 *   (moe_status_read).
 *   workspace: >= 256 + S_max * f * sizeof(dtype) bytes, rounded up to a multiple of 256
 *   (the status word, then the hidden activations H [S_max, f]); moe_workspace_size of the
 *   same layer shape is always enough for S_max = min(T k, E C).
 * f16: hidden activations are rounded to f16 between the two GEMMs.
 */
MOE_API moe_status moe_expert_ffn(const void* tokens, const int32_t* perm, const int32_t* offsets,
                          const void* W1, const void* W2, moe_dtype dtype, int T, int d, int f,
                          int E, int S_max, void* expert_out, void* workspace, size_t ws_bytes,
                          moe_stream_t stream);

/*
 * Gate-weighted combine back to token order (DeepSpeed-MoE review, "Phenomenon2": the
 * outputs of the experts a token visits are summed; Residual-MoE adds a fixed MLP):
 *   out[t, :] = sum_j [slot_of[t,j] >= 0] topk_w[t,j] expert_out[slot_of[t,j], :]
 *               (+ residual_in[t, :] when residual_in is not NULL)
 * in fp32, j ascending, the residual added last, rounded once to `dtype`.
 *   expert_out [S, d], residual_in nullable [T, d], out [T, d]: all in `dtype`.
 */
MOE_API moe_status moe_combine(const void* expert_out, const int32_t* slot_of, const float* topk_w,
                       const void* residual_in, moe_dtype dtype, int T, int d, int k, void* out,
                       moe_stream_t stream);

/*
 * The whole layer, fused: gate, dispatch, expert GEMM1 + GeLU, expert GEMM2 with the
 * gate-weighted combine in its epilogue, and for MOE_MLP_RESIDUAL the dense MLP
 *   out[t] += GeLU(x_t Wr1) Wr2,   Wr1 [d, f_res], Wr2 [f_res, d]   (NULL for STANDARD),
 * computed by the same grouped-GEMM kernels as an extra group of all T tokens.
 *   tokens [T, d], W1 [E, d, f], W2 [E, f, d], out [T, d]: `dtype`.  Wg [d, E]: float32.
 *   topk_idx_out nullable [T, k], slot_of_out nullable [T, k]: routing, as moe_gate_topk /
 *   moe_dispatch define it.
 *   workspace >= moe_workspace_size(...) bytes; contents need no initialisation.
 *   out must not overlap tokens or the workspace: it is cleared before the experts' outputs
 *   are added into it.
 * Deterministic: repeated calls give identical bits.  Top-1 standard layers write each
 * output row once.  Where an output element has two addends (top-2, or one expert plus the
 * residual MLP), each is rounded to `dtype` and added into the cleared output: 0 + a is exact
 * and a + b commutes, so the order of the additions does not matter.  Top-2 with the residual
 * MLP (three addends) sums in fp32 in a fixed order and rounds once.
 */
MOE_API moe_status moe_layer_forward(const void* tokens, const float* Wg, const void* W1, const void* W2,
                             const void* Wr1, const void* Wr2, moe_dtype dtype, int T, int d,
                             int f, int E, int k, float capacity_factor, moe_mlp_type mlp_type,
                             int f_res, void* out, int32_t* topk_idx_out, int32_t* slot_of_out,
                             void* workspace, size_t ws_bytes, moe_stream_t stream);

/*
 * Synchronises `stream`, then returns the device-side status word of the most recent
 * moe_expert_ffn / moe_layer_forward call on this workspace (MOE_OK, MOE_ERR_TIMEOUT or
 * MOE_ERR_DEVICE_BOUNDS), or MOE_ERR_CUDA if the synchronisation or the read failed.
 * The word is cleared at the start of each of those calls.
 */
MOE_API moe_status moe_status_read(const void* workspace, moe_stream_t stream);

/* Static, human-readable name of a status code ("MOE_OK", ...). */
MOE_API const char* moe_status_string(moe_status status);

/*
 * Self-test of the device-side bounded wait that every pipeline wait in the library uses:
 * launches one block that waits on an mbarrier nothing ever arrives on, with a budget of
 * timeout_ns nanoseconds (1 .. 10^10) instead of the library's default of 2 s.  The wait
 * gives up, records MOE_ERR_TIMEOUT in the workspace's status word and the kernel returns
 * normally, leaving the context usable; read the result with moe_status_read.
 * workspace: >= 256 bytes.
 */
MOE_API moe_status moe_selftest_wait(void* workspace, uint64_t timeout_ns, moe_stream_t stream);

/*
 * Measurement hook (the pages have no counterpart): when `events` is not NULL, the calling
 * thread's next moe_layer_forward calls record events[0 .. 6] (cudaEvent_t handles created
 * by the caller) on their stream at the stage boundaries: [0] start, [1] after the gate
 * logits, [2] after softmax / top-k, [3] after dispatch, [4] after the first expert GEMM
 * (+ GeLU), [5] after the second expert GEMM (+ combine), [6] at the end.  n_events must be
 * 7, or 0 with events NULL to stop recording.  Thread-local; host only.
 */
#define MOE_STAGE_EVENTS 7
MOE_API moe_status moe_set_stage_events(void* const* events, int n_events);

/*
 * Measurement hook (the pages have no counterpart): the number of kernels this library has
 * enqueued in this process so far, counted on the host at each successful launch.  Inside a
 * stream capture a launch is counted once when captured (not per graph replay), so the
 * difference across a capture is the number of kernels per replay.  Never fails.
 */
MOE_API unsigned long long moe_kernel_launches(void);

/*
 * Allocation-free variant of moe_expert_ffn (the pages have no counterpart).
 *
 * For callers that cannot allocate device memory where they run the layer: a plugin or
 * custom operator inside a host framework that owns all device memory and gives its
 * plugins no workspace, or a serving loop that forbids cudaMalloc after start-up because it
 * can synchronise the device.  They pass inputs and outputs only; the scratch (the hidden
 * activations H [S_max, f]) lives in a fixed 64 MiB array compiled into the library, which
 * every GPU that loads the library keeps until the process exits.
 *   Arguments and results: as moe_expert_ffn, without the workspace.
 *   Limit: S_max * f * sizeof(dtype) <= 64 MiB, else MOE_ERR_WORKSPACE (nothing runs).
 *   The first call on each device looks up the array's device address (with that device
 *   current) and keeps it; make that first call before any stream capture, and make no call
 *   on a device after a reset of it (cudaDeviceReset), which invalidates the kept address.
 *   All calls share the one array and it keeps the last call's contents: calls that
 *   overlap on the GPU race on it (order them on one stream).  Device-side wait timeouts
 *   are not reported by this variant (it has no status word to read).
 *   Calls no cudaMalloc, cudaFree or other allocating routine.
 */
MOE_API moe_status moe_expert_ffn_noalloc(const void* tokens, const int32_t* perm,
                                          const int32_t* offsets, const void* W1, const void* W2,
                                          moe_dtype dtype, int T, int d, int f, int E, int S_max,
                                          void* expert_out, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
