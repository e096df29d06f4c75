/*
 * moe.h - C ABI of a single-GPU (B300, sm_103a) forward pass of the
 * sparsely-gated Mixture-of-Experts layer with noisy top-k gating.
 *
 * The operation is the one described in "Mixture of Experts: Outrageously
 * Large Neural Networks" (intuitivepapers.ai, an explainer of Shazeer et al.
 * 2017): noisy logits H = x W_g + eps * Softplus(x W_noise) (section "Noisy
 * top-k gating", eq (4)), KeepTopK and a softmax over the kept logits
 * (eqs (3)/(5)), per-expert ReLU feed-forward experts whose gate-weighted
 * outputs are summed (section "How a mixture-of-experts layer works",
 * eq (1)), and the two balancing losses: CV^2 of the Importance (section "Why
 * experts collapse, and the balancing losses", eqs (6)-(7)) and CV^2 of the
 * smooth Load built from P(x, i) = Phi((x W_g)_i - kth_excluding(H, k, i)) /
 * Softplus((x W_noise)_i)) (section "A differentiable count of examples",
 * eqs (8)-(10)).  The order of the steps follows the forward-pass listing in
 * the page's "Implementation notes".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller (the one
 *   exception, moe_ep_plan, takes host pointers and says so); the
 *   library never allocates device memory and never frees caller memory.
 * - Tensors are dense, row-major, with the shapes given in [brackets];
 *   element types are stated per argument ("x dtype" = cfg->x_dtype,
 *   "expert dtype" = cfg->expert_dtype).  bf16 is IEEE bfloat16 stored in
 *   uint16.  Pointers to bf16/fp32 data must be 16-byte aligned.
 * - Scratch memory is a caller-supplied workspace of at least
 *   moe_workspace_size(cfg) bytes, 256-byte aligned.  Its contents need not
 *   be initialised and are clobbered.
 * - All work is enqueued on the caller's CUDA stream; no entry point
 *   synchronises the host except moe_get_device_error.  Calls on one stream
 *   run in order; two calls sharing a workspace must not overlap.
 * - Errors are returned as moe_status; no C++ exception crosses the ABI.
 *   Argument checks happen on the host before anything is enqueued, so an
 *   error other than MOE_ERR_CUDA leaves the stream untouched.
 * - Results are deterministic: no floating-point atomics; every reduction
 *   is in a fixed order, so repeated calls give bitwise-identical outputs.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* NULL pointer, k < 1, k > n, a size <= 0   */
    MOE_ERR_UNSUPPORTED = 2,   /* shape/dtype outside what the kernels take */
    MOE_ERR_WORKSPACE = 3,     /* workspace too small or misaligned         */
    MOE_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed      */
    MOE_ERR_TIMEOUT = 5,       /* a device-side bounded wait expired        */
    MOE_ERR_RANGE = 6          /* a value beyond what its output can hold:  */
                               /* an fp16 expert output of |v| >= 65520 or  */
                               /* NaN; more taken pairs than the batchwise  */
                               /* threshold mode's workspace holds          */
} moe_status;

typedef enum moe_dtype {
    MOE_F32 = 0,
    MOE_BF16 = 1
} moe_dtype;

/* Shapes and settings of one flat MoE layer call.
 *   T  tokens in the batch            d  input/output size of an expert
 *   n  experts                        h  hidden size of an expert
 *   k  experts kept per token (1 <= k <= n, k <= 8)
 * x_dtype:      MOE_F32 or MOE_BF16 (x and the dispatched rows x_perm)
 * expert_dtype: MOE_F32 (then x_dtype must be MOE_F32) or MOE_BF16
 *               (W_in, W_out, y_perm; fp32 accumulation)
 * std_floor:    added to Softplus((x W_noise)_i); 0 is eq (4) as written,
 *               0.01 the floor of the official implementation.
 * w_importance, w_load: loss weights (0.1 in the 1 Billion Word models).
 * flags:        0 or a combination of MOE_FLAG_FFN_ROW_TILES or
 *               MOE_FLAG_FFN_SIZED_TILES (not both), MOE_FLAG_SWITCH_GATE and
 *               MOE_FLAG_DEVICE_NOISE.
 * capacity:     0 = every routed row is processed (the layer as the paper
 *               defines it).  C > 0 = an expert processes at most C of its
 *               routed rows, the first C in routed-row order; the others add
 *               nothing to y (a fixed per-expert capacity whose overflow passes
 *               through the caller's residual connection, as in GShard: "From
 *               LSTMs to Switch and Mixtral").  The gate's outputs and the
 *               balancing losses do not depend on it.
 * noise_seed:   with MOE_FLAG_DEVICE_NOISE, the seed of the noise the layer draws.
 * Supported sizes: d and h multiples of 64, n <= 16384, T*k < 2^31.  */
typedef struct moe_config {
    int T, d, n, h, k;
    moe_dtype x_dtype;
    moe_dtype expert_dtype;
    float std_floor;
    float w_importance;
    float w_load;
    unsigned flags;
    int capacity;
    unsigned long long noise_seed;
} moe_config;

/* Tile kind of the bf16 expert FFN (d, h multiples of 256).  By default (and with
 * MOE_FLAG_FFN_ROW_TILES) the library runs 256-row tiles, every expert's last tile
 * padded to 256 rows; MOE_FLAG_FFN_SIZED_TILES runs tiles sized to each expert's
 * rows (rounded up to 32, operands exchanged so the rows are the MMA's N), which
 * measured slower on the workloads tried.  Setting both is an error; results agree
 * up to fp32 summation order.  Every other bit of flags is reserved and must be 0. */
#define MOE_FLAG_FFN_ROW_TILES 1u
#define MOE_FLAG_FFN_SIZED_TILES 2u

/* The Switch gate ("From LSTMs to Switch and Mixtral": Switch Transformers run the
 * softmax over all n logits first and multiply the chosen expert's output by its
 * probability, a number below 1 that still depends on W_g; used with k = 1).  The
 * kept experts are the same k largest noisy logits; gates[t,j] is the softmax of
 * H_t over all n experts at the j-th kept expert (not renormalised over the kept);
 * load[i] is the number of routed rows sent to expert i; importance[i] the sum over
 * the batch of expert i's probability; and the single balancing loss is
 *   L = n * sum_i f_i P_i,  f_i = load_i / (T k),  P_i = importance_i / T
 * (1 under uniform routing), returned as losses = (L, 0, w_importance * L).  Flat
 * layer only (moe_gate, moe_forward); moe_balance_losses answers
 * MOE_ERR_UNSUPPORTED. */
#define MOE_FLAG_SWITCH_GATE 4u

/* The gate's noise drawn by the layer ("Noisy top-k gating", eq (4): one standard
 * normal draw per token and expert).  The caller passes eps = NULL to moe_gate,
 * moe_forward(_timed) and moe_backward(_timed) (non-NULL: MOE_ERR_INVALID_ARG); the
 * layer writes the draws for cfg->noise_seed into its workspace (T*n floats more,
 * included in moe_workspace_size) and uses them as eps, so a batch's noise never
 * crosses the host link.  The draws are moe_draw_noise's for the same seed, element
 * t*n + e for token t and expert e, so a backward call with the same cfg sees the
 * forward call's noise.  moe_batchwise_forward and moe_batchwise_threshold_forward
 * answer MOE_ERR_UNSUPPORTED. */
#define MOE_FLAG_DEVICE_NOISE 8u

/* eps[i], i < count: the standard normal draws of a counter-based generator for seed
 * (device pointer, 16-byte aligned for count >= 4; written on stream).  Elements 2j and
 * 2j + 1 are the two normals of Box-Muller pair j:
 *   z  = seed + (j + 1) * 0x9E3779B97F4A7C15 mod 2^64, then the SplitMix64 finaliser
 *        (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
 *        OOPSLA 2014): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
 *        z *= 0x94D049BB133111EB; z ^= z >> 31;
 *   u1 = ((z >> 40) + 1) / 2^24,  u2 = (z mod 2^24) / 2^24,  r = sqrt(-2 ln u1),
 *   eps[2j] = r cos(2 pi u2),  eps[2j+1] = r sin(2 pi u2)   (|eps| <= 5.77),
 * in fp32 (CUDA's logf, sqrtf and sincospif).  count < 0 or a NULL eps with count > 0:
 * MOE_ERR_INVALID_ARG. */
moe_status moe_draw_noise(unsigned long long seed, long long count, float* eps,
                          cudaStream_t stream);

/* Human-readable name of a status code (static storage, never NULL). */
const char* moe_status_string(moe_status s);

/* Bytes of workspace every entry point below needs for cfg, written to
 * *bytes.  One workspace of this size serves every call for cfg. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes);

/* Noisy top-k gate ("Noisy top-k gating", eqs (3)-(5); "A differentiable
 * count of examples", eqs (8)-(10)).
 *   x        [T,d]  x dtype
 *   W_g      [d,n]  fp32         W_noise [d,n] fp32
 *   eps      [T,n]  fp32  standard normal draws, one per token and expert;
 *                   NULL (or all zeros) = no noise: inference, or the
 *                   noiseless gate of later layers such as Mixtral's ("From
 *                   LSTMs to Switch and Mixtral"); NULL reads nothing
 *   b_g      [n]    fp32  optional per-expert logit bias added to the clean
 *                   logit (NULL = none)
 * Outputs:
 *   idx      [T,k]  int32  kept experts, largest noisy logit first; equal
 *                   logits rank the lower expert index first
 *   gates    [T,k]  fp32   softmax over the kept noisy logits
 *   tie      [T]    uint8  1 where H_(k) - H_(k+1) < 1e-5 (a near tie at the
 *                   k-th place, where fp32 and exact arithmetic may keep
 *                   different experts); 0 otherwise and when k = n.  May be NULL.
 *   load     [n]    fp32   Load_i = sum over the batch of P(x, i), with
 *                   kth_excluding = the (k+1)-th largest H when i is kept,
 *                   the k-th largest otherwise (-inf when k = n).
 *   logits   [3,T,n] fp32  optional debug copy of (clean, std, H); NULL = none.
 * Logits are computed in fp32 from the exact x and W values. */
moe_status moe_gate(const moe_config* cfg, const void* x, const float* W_g,
                    const float* W_noise, const float* eps, const float* b_g,
                    int32_t* idx, float* gates, uint8_t* tie, float* load,
                    float* logits, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/* Dispatch: group the T*k routed rows by expert (the per-expert row lists of
 * the forward-pass listing).  Routed row r = t*k + j is token t's j-th kept
 * slot; rows are grouped by ascending expert and keep ascending r inside a
 * group (a stable counting sort).
 *   idx      [T,k]  int32 in [0,n)   (distinct per row is not required)
 *   x        [T,d]  x dtype
 * Outputs:
 *   offsets  [n+1]  int32  expert e owns positions [offsets[e], offsets[e+1])
 *   perm     [T*k]  int32  perm[p] = r, the routed row at position p
 *   inv      [T*k]  int32  inv[r] = p
 *   x_perm   [T*k,d] x dtype  x_perm[p] = x[perm[p] / k]
 * With cfg->capacity = C > 0, expert e keeps the first min(count_e, C) of its
 * rows: offsets[e+1] - offsets[e] = min(count_e, C), offsets[n] = the rows kept,
 * and a dropped row r has inv[r] = -1 and no position (perm and x_perm hold the
 * kept rows only).
 * An idx value outside [0,n) is reported as MOE_ERR_INVALID_ARG by
 * moe_get_device_error (the row is dropped, nothing is written out of bounds). */
moe_status moe_dispatch(const moe_config* cfg, const int32_t* idx, const void* x,
                        int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* moe_dispatch for callers that cannot allocate device memory.  The paper has
 * no counterpart to this entry point; it exists for code that may not call
 * cudaMalloc: a plugin running inside a host framework whose memory pool owns
 * all of the GPU's memory and lends it none, or a serving loop that must never
 * let cudaFree's implicit device-wide synchronisation stall other streams.
 * Such a caller often has no spare buffer to offer as a workspace either.
 *
 * Same arguments, results and errors as moe_dispatch (bit-identical outputs),
 * minus the workspace: the counting sort's per-tile expert counts live in a
 * 1 MiB array of the library's own device memory (MOE_NOALLOC_DISPATCH_INTS
 * int32), which every GPU that loads the library holds until the process exits.
 *   - Limit: (tiles + 1) * n <= MOE_NOALLOC_DISPATCH_INTS, with tiles the
 *     counting sort's row tiles, today min(256, ceil(T*k / 1024)) (the check
 *     uses the sort's own tiling, so it follows any change of it).  Larger shapes return
 *     MOE_ERR_WORKSPACE before anything is enqueued.  n <= 1020 always fits;
 *     n = 4096 fits up to T*k = 64512, n = 16384 up to T*k = 15360.
 *   - Nothing is allocated: the call makes no cudaMalloc/cudaFree or other
 *     allocating call.  The first call on each device looks up the array's
 *     device address (cudaGetSymbolAddress) with that device current and keeps
 *     it for the life of the process; make that first call before any stream
 *     capture, and do not call this entry point on a device after
 *     cudaDeviceReset (the kept address belongs to the old context).
 *   - Every call on a device shares the one array: calls whose GPU work
 *     overlaps (other streams, other host threads) race and corrupt each
 *     other's results.  Serialise them, e.g. on one stream.  No entry of the
 *     array has to start at zero; each call overwrites what it reads. */
#define MOE_NOALLOC_DISPATCH_INTS 262144
moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* idx, const void* x,
                                int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm,
                                cudaStream_t stream);

/* Experts ("How a mixture-of-experts layer works"): for every expert e and
 * every position p in [offsets[e], offsets[e+1]):
 *     y_perm[p] = ReLU(x_perm[p] W_in[e]) W_out[e]
 * Experts that own no row are never run.
 *   x_perm   [T*k,d]  x dtype (must equal expert dtype)
 *   offsets  [n+1]    int32, non-decreasing, offsets[0] = 0, offsets[n] <= T*k
 *                     (rows past offsets[n] are not read)
 *   W_in     [n,d,h]  expert dtype      W_out [n,h,d] expert dtype
 * Output:
 *   y_perm   [T*k,d]  fp16 for bf16 experts, fp32 for fp32 experts
 * bf16 experts run on the tensor cores (tcgen05): bf16 operands, fp32
 * accumulation, the hidden layer rounded to bf16 (it is the second product's
 * operand) and each expert output rounded to fp16, whose 11-bit significand
 * keeps the combined layer output within 2e-2 RMS of exact arithmetic where a
 * bf16 output would not.  fp16's largest finite value is 65504: an expert output
 * of magnitude 65520 or more (which rounds to infinity), or a NaN, is stored as
 * such and sets the device error word to MOE_ERR_RANGE (read by
 * moe_get_device_error; the call itself returns MOE_OK).  fp32 experts: fp32
 * throughout (CUDA cores), no such limit. */
moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const void* W_in, const void* W_out, void* y_perm,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Combine, eq (1): y[t] = sum_j gates[t,j] * y_perm[inv[t*k+j]], summed in
 * slot order j = 0..k-1 in fp32.
 *   y_perm [T*k,d] fp16 (bf16 experts) or fp32 (fp32 experts), as written by
 *   moe_expert_ffn;  inv [T*k] int32 (-1: a row its expert dropped, which adds
 *   nothing);  gates [T,k] fp32
 * Output: y [T,d] fp32. */
moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* inv,
                       const float* gates, float* y, cudaStream_t stream);

/* Balancing losses, eqs (6), (7) and (10).
 *   gates [T,k] fp32, perm [T*k] int32, offsets [n+1] int32 (from moe_dispatch
 *   on the same idx), load [n] fp32 (from moe_gate)
 * Outputs:
 *   importance [n] fp32   Importance_e = sum of the gates routed to e, summed
 *                         in ascending routed-row order
 *   losses     [3] fp32   CV^2(Importance), CV^2(Load),
 *                         w_importance*CV^2(Importance) + w_load*CV^2(Load)
 * CV^2 = population variance / mean^2 (0 when the mean is 0 or n = 1).
 * Needs the dispatch of every routed row: MOE_ERR_UNSUPPORTED when
 * cfg->capacity > 0 (moe_forward forms the same losses from the gate), and with
 * MOE_FLAG_SWITCH_GATE (whose Importance covers every expert's probability). */
moe_status moe_balance_losses(const moe_config* cfg, const float* gates, const int32_t* perm,
                              const int32_t* offsets, const float* load, float* importance,
                              float* losses, cudaStream_t stream);

/* ---- Sharding the layer over several GPUs ----------------------------------
 *
 * "Keeping each expert's batch large" (the paragraph on mixing data parallelism
 * and model parallelism): the gate and the other layers are replicated and each
 * device takes its own share of the batch (data parallel); the experts are spread
 * over the devices, each device holding n / world of them, and every routed row
 * travels to the device that holds its expert and its output travels back
 * (expert parallel).  The collectives themselves (an all-reduce, an all-gather and
 * two all-to-alls) are the caller's, e.g. NCCL through torch.distributed; these
 * entry points are the steps around them.
 *
 * Balancing losses of the whole batch from sums the caller formed.  Eqs (6)-(7)
 * and (10) are batch quantities, and the CV^2 of one shard's sums is not that of
 * the whole batch's, so a data-parallel caller adds every rank's Importance and
 * Load vectors (moe_forward's importance / load outputs; one all-reduce of 2n
 * floats when both sit in one buffer) and forms the losses from the totals here.
 *   importance [n], load [n] fp32   the whole batch's sums
 *   cfg->T   tokens of the whole batch (read by the Switch gate's loss only)
 * Output: losses [3] fp32, as moe_forward's (MOE_FLAG_SWITCH_GATE: the Switch
 * loss, with load = routed-row counts and importance = summed probabilities). */
moe_status moe_losses_from_sums(const moe_config* cfg, const float* importance,
                                const float* load, float* losses, cudaStream_t stream);

/* Expert-parallel exchange plan of one rank.  HOST-ONLY: every pointer is a host
 * pointer, nothing is enqueued and no GPU is needed.  Rank r holds experts
 * [r * n_local, (r+1) * n_local), n_local = n / world (n must be a multiple of
 * world, else MOE_ERR_UNSUPPORTED).  Each rank dispatches its own tokens with
 * moe_dispatch, so its x_perm holds the rows bound for rank r contiguously, in
 * expert order; the caller all-gathers every rank's offsets and calls this.
 *   all_offsets [world][n+1] int32   moe_dispatch's offsets of every rank
 *                                    (each starting at 0, non-decreasing, else
 *                                    MOE_ERR_INVALID_ARG)
 * Outputs (host int32, caller-owned):
 *   send_rows [world]   rows this rank sends to each rank (its x_perm rows
 *                       offsets[r n_local] .. offsets[(r+1) n_local])
 *   recv_rows [world]   rows it receives from each rank, which arrive source
 *                       rank major, each source's rows in expert order
 *   plan [2 B + n_local + 2], B = world * n_local:
 *     plan[e*world + s]          arrival position of the first row that source s
 *                                sends for local expert e
 *     plan[B + e*world + s]      its position in expert-major order (every source's
 *                                rows of expert e together, sources ascending);
 *     plan[2B]                   rows received in all
 *     plan[2B + 1 + e]           local expert offsets [n_local + 1] in expert-major
 *                                order: the offsets moe_expert_ffn takes for the
 *                                rank's n_local experts
 * Expert-major order is the order a single-GPU dispatch of the concatenated batch
 * (rank 0's tokens first) gives these experts' rows.  MOE_ERR_UNSUPPORTED when the
 * rows received reach 2^31. */
moe_status moe_ep_plan(int world, int rank, int n, const int32_t* all_offsets,
                       int32_t* send_rows, int32_t* recv_rows, int32_t* plan);

/* Rows between arrival order and expert-major order on the device, by the plan
 * of moe_ep_plan (copied to the device by the caller):
 *   to_expert_major = 1: out[p] = in[arrival position of expert-major row p]
 *   to_expert_major = 0: the inverse (expert outputs back to arrival order, the
 *                        order the return all-to-all sends them in).
 *   plan   [2 B + n_local + 2] int32 (device)
 *   in, out [plan[2B], row_bytes] (device, 16-byte aligned, not overlapping);
 *   row_bytes a positive multiple of 16 (else MOE_ERR_UNSUPPORTED). */
moe_status moe_ep_regroup(int world, int n_local, const int32_t* plan, const void* in,
                          void* out, size_t row_bytes, int to_expert_major,
                          cudaStream_t stream);

/* The whole layer: moe_gate, moe_dispatch, moe_expert_ffn, moe_combine and
 * moe_balance_losses in one call on one stream.
 * Inputs as for moe_gate plus W_in [n,d,h], W_out [n,h,d] (expert dtype).
 * Outputs: y [T,d] fp32, losses [3] fp32 (as moe_balance_losses).
 * Optional outputs (NULL = kept in the workspace only): idx [T,k] int32,
 * gates [T,k] fp32, tie [T] uint8, importance [n] fp32, load [n] fp32. */
moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_g,
                       const float* W_noise, const float* eps, const float* b_g,
                       const void* W_in, const void* W_out, float* y, float* losses,
                       int32_t* idx, float* gates, uint8_t* tie, float* importance,
                       float* load, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Backward pass of the whole layer ("Implementation notes" of the paper's explainer:
 * which parameters receive gradient and by which path).  Gradients of
 *   L = sum(dy * y) + w_importance CV(Importance)^2 + w_load CV(Load)^2
 * (the task loss's gradient dy with respect to y, plus the two balancing losses
 * moe_forward returns in losses[2]) with respect to x, W_g, W_noise, b_g, W_in and
 * W_out, with the kept experts held fixed (the selection passes no gradient).  The
 * load loss reaches clean_i and std_i of every expert through eq (9), and the
 * threshold kth_excluding(H, k, i), the noisy logit of the expert at the k-th or
 * (k+1)-th place, passes its gradient to that expert's logit.  The forward pass is
 * recomputed inside the call (the experts' hidden layer included, the memory saving
 * the paper describes), so the inputs are those of moe_forward.  ReLU'(u) = [hidden >
 * 0] on the stored (bf16 for bf16 experts) hidden layer.
 *   dy [T,d] fp32 (device)
 * Outputs (device, fp32, overwritten): dx [T,d], dW_g [d,n], dW_noise [d,n],
 * db_g [n] (NULL = not wanted), dW_in [n,d,h], dW_out [n,h,d] (zero for an expert
 * without rows).  workspace: moe_backward_workspace_size bytes.  Not with
 * cfg->capacity > 0 or MOE_FLAG_SWITCH_GATE (MOE_ERR_UNSUPPORTED). */
moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes);
moe_status moe_backward(const moe_config* cfg, const void* x, const float* W_g,
                        const float* W_noise, const float* eps, const float* b_g,
                        const void* W_in, const void* W_out, const float* dy, float* dx,
                        float* dW_g, float* dW_noise, float* db_g, float* dW_in, float* dW_out,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);
/* moe_backward that also records six caller-created CUDA events on `stream`: before
 * the forward recompute and after it, after the combine and gate backward, after the
 * expert data gradients (dx's share included), after the expert weight gradients and
 * after the gate's weight gradients (a profiling aid, like moe_forward_timed). */
moe_status moe_backward_timed(const moe_config* cfg, const void* x, const float* W_g,
                              const float* W_noise, const float* eps, const float* b_g,
                              const void* W_in, const void* W_out, const float* dy, float* dx,
                              float* dW_g, float* dW_noise, float* db_g, float* dW_in,
                              float* dW_out, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream, cudaEvent_t* stage_events);

/* The layer with the batchwise top-m gate the paper's single-pair translation models
 * use (its Appendix F, as the explainer's "What the paper measured" describes it):
 * during training each expert takes exactly the m = floor(k T / n) tokens of the batch
 * with its largest noisy logits H (eq (4); equal H -> the lower token index), so every
 * expert gets the same batch size; a token's gates over the experts that took it are
 * the softmax of their H, and a token no expert took gets y = 0.
 * Inputs as for moe_forward (eps NULL = no noise).  Outputs: y [T,d] fp32; losses [3]
 * fp32 = (CV^2(Importance), CV^2(load) = 0, w_importance CV^2(Importance)), Importance_i
 * being the gates expert i received; sel [n,m] int32 (NULL = not wanted): the tokens
 * each expert took, ascending.  workspace: moe_batchwise_workspace_size bytes.  Needs
 * 1 <= k T / n, cfg->capacity = 0 and no MOE_FLAG_SWITCH_GATE (else
 * MOE_ERR_UNSUPPORTED).  The inference mode is moe_batchwise_threshold_forward. */
moe_status moe_batchwise_workspace_size(const moe_config* cfg, size_t* bytes);
moe_status moe_batchwise_forward(const moe_config* cfg, const void* x, const float* W_g,
                                 const float* W_noise, const float* eps, const float* b_g,
                                 const void* W_in, const void* W_out, float* y, float* losses,
                                 int32_t* sel, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* The batchwise gate at inference: the page says a learned per-expert threshold
 * replaces the batch-wise top-m choice.  Expert i takes every token t whose noisy
 * logit H_ti (eq (4)) exceeds threshold[i] (strictly), so the experts' batch sizes
 * vary; gates and output are formed as in moe_batchwise_forward (softmax of H over
 * the experts that took the token, y = 0 for a token none took).
 *   threshold [n] fp32 (device)
 * Outputs: y [T,d] fp32; losses [3] fp32 = (CV^2(Importance), CV^2(counts),
 * w_importance CV^2(Importance) + w_load CV^2(counts)); counts [n] int32 (NULL =
 * not wanted): the tokens each expert took.  The workspace
 * (moe_batchwise_workspace_size) holds k T taken (token, expert) pairs in all, k
 * acting as the expected experts a token: thresholds that admit more fill the
 * first k T positions in expert order, drop the rest and set the device error word
 * to MOE_ERR_RANGE (moe_get_device_error), y then covering only the pairs kept.
 * cfg->capacity = 0 and no MOE_FLAG_SWITCH_GATE (else MOE_ERR_UNSUPPORTED). */
moe_status moe_batchwise_threshold_forward(const moe_config* cfg, const void* x,
                                           const float* W_g, const float* W_noise,
                                           const float* eps, const float* b_g,
                                           const float* threshold, const void* W_in,
                                           const void* W_out, float* y, float* losses,
                                           int32_t* counts, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);

/* moe_forward that also records six caller-created CUDA events on `stream`: before
 * the gate and after the gate, the dispatch, the experts, the combine and the
 * losses, so a caller can time each stage of the one-call forward pass with
 * cudaEventElapsedTime.  A profiling aid with no counterpart in the layer's
 * definition.  stage_events: host array of 6 events (none NULL), owned by the
 * caller; results and errors as moe_forward (MOE_ERR_INVALID_ARG for a NULL
 * array or event). */
moe_status moe_forward_timed(const moe_config* cfg, const void* x, const float* W_g,
                             const float* W_noise, const float* eps, const float* b_g,
                             const void* W_in, const void* W_out, float* y, float* losses,
                             int32_t* idx, float* gates, uint8_t* tie, float* importance,
                             float* load, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream, cudaEvent_t* stage_events);

/* ---- Hierarchical MoE ("Hierarchical MoE" section of the page) --------------
 *
 * A primary noisy top-k1 gate over a groups chooses groups; inside each chosen
 * group i a secondary noisy top-k2 gate over that group's b experts chooses
 * experts; the gate of expert (i, j) is the product G_primary(x)_i * G_i(x)_j and
 * y = sum over the k1*k2 chosen (i, j) of that product times E_{i,j}(x).  Expert
 * (i, j) is flat expert i*b + j of W_in / W_out.  The secondary gate of group i
 * has its own weights W_g2[i], W_noise2[i] and sees only the tokens routed to
 * group i; a token's noise for the secondary gate of its s-th chosen group is
 * eps2[t, s, :].  (The page's formula is lost in extraction; this is the reading
 * its prose supports.)
 *
 *   T tokens, d model size, a groups of b experts, h hidden size,
 *   k1 groups kept per token (1 <= k1 <= a), k2 experts kept per group
 *   (1 <= k2 <= b), k1*k2 <= 8.
 * x_dtype = expert_dtype = MOE_BF16 (both gates run on the tensor cores with the
 * exact three-term split of fp32 weights).  Supported: a <= 256, b <= 256,
 * a*b <= 16384, d and h multiples of 64. */
typedef struct moe_hier_config {
    int T, d, a, b, h, k1, k2;
    moe_dtype x_dtype;
    moe_dtype expert_dtype;
    float std_floor;           /* as in moe_config, for both gates */
    float w_importance;
    float w_load;
    unsigned flags;            /* as in moe_config, without MOE_FLAG_SWITCH_GATE */
} moe_hier_config;

/* Workspace bytes of moe_hier_forward for cfg, written to *bytes. */
moe_status moe_hier_workspace_size(const moe_hier_config* cfg, size_t* bytes);

/* The hierarchical layer's forward pass on one stream.
 *   x        [T,d]        bf16
 *   W_g1, W_noise1 [d,a]  fp32   primary gate         eps1 [T,a] fp32
 *   W_g2, W_noise2 [a,d,b] fp32  secondary gates      eps2 [T,k1,b] fp32
 *   W_in [a*b,d,h], W_out [a*b,h,d]  bf16
 * Outputs:
 *   y        [T,d]  fp32
 *   losses   [3]    fp32  CV^2(Importance1), CV^2(Load1) and
 *                   w_importance*CV^2(Importance1) + w_load*CV^2(Load1) of the
 *                   primary gate over the a groups (the page gives no loss of
 *                   its own for the hierarchy)
 * Optional outputs (NULL = kept in the workspace only):
 *   idx      [T,k1*k2] int32  flat expert ids, slot s*k2 + j = the j-th expert
 *                   of the s-th kept group (groups and experts by descending H)
 *   gates    [T,k1*k2] fp32   product gates (each row sums to 1)
 *   tie1     [T]     uint8    near tie at the k1-th place of the primary gate
 *   tie2     [T,k1]  uint8    near tie at the k2-th place of each secondary gate
 *   importance1, load1 [a]    fp32  primary Importance and Load over groups
 *   importance, load2  [a*b]  fp32  Importance of the product gates over the
 *                   flat experts, and each secondary gate's Load (sum over the
 *                   group's rows of P) at its experts' flat ids
 * Errors as moe_forward. */
moe_status moe_hier_forward(const moe_hier_config* cfg, const void* x, const float* W_g1,
                            const float* W_noise1, const float* eps1, const float* W_g2,
                            const float* W_noise2, const float* eps2, const void* W_in,
                            const void* W_out, float* y, float* losses, int32_t* idx,
                            float* gates, uint8_t* tie1, uint8_t* tie2, float* importance1,
                            float* load1, float* importance, float* load2, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream);

/* Waits for `stream`, then reads and clears the device error word that the
 * kernels set instead of trapping (bounded waits that expired, idx values out
 * of range, fp16 expert outputs out of range).  Returns MOE_OK, MOE_ERR_TIMEOUT,
 * MOE_ERR_INVALID_ARG, MOE_ERR_RANGE or MOE_ERR_CUDA; the first error since the
 * last read is the one reported.  This is the only entry point that blocks the
 * host. */
moe_status moe_get_device_error(cudaStream_t stream);

/* Failure-detection self-test, with no counterpart in the layer's definition.
 * Enqueues one CTA on `stream` whose bounded waits, the same code as the waits of
 * the tensor-core kernels, wait for an mbarrier that nothing ever completes: the
 * first gives up after budget_cycles SM cycles (1 .. 1e9) and records a timeout,
 * the second sees the CTA's abort flag and returns, and the CTA exits normally.
 * moe_get_device_error(stream) then returns MOE_ERR_TIMEOUT (and clears it); the
 * context stays usable.  Nothing faults, traps or hangs. */
moe_status moe_selftest_timeout(long long budget_cycles, cudaStream_t stream);

/* Name of the CUDA error behind the last MOE_ERR_CUDA that an entry point
 * returned on the calling host thread ("cudaSuccess" if none); static storage.
 * A diagnostic with no counterpart in the layer's definition. */
const char* moe_last_cuda_error(void);

/* Number of CUDA kernels this library has enqueued in this process so far
 * (all devices and streams).  A diagnostic for counting launches per call;
 * it has no counterpart in the layer's definition. */
unsigned long long moe_launch_counter(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
