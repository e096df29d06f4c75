// Host-side launch wrappers of the kernels, one translation unit each.
// Internal to the library; the public boundary is include/moe.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace moe {

// Counts one enqueued kernel (read back through moe_launch_counter).
void note_launch();

// ---- gate (gate_simt.cu) ---------------------------------------------------
// clean/std/H [T,n] fp32 from x [T,d] (fp32 or bf16), W_g, W_noise [d,n], eps [T,n].
cudaError_t launch_gate_logits(const void* x, bool x_bf16, const float* W_g, const float* W_noise,
                               const float* eps, const float* b_g, int T, int d, int n,
                               float std_floor, float* clean, float* stdv, float* H,
                               cudaStream_t s);
// Per-token top-(k+1) over H: idx/gates [T,k], tie [T] (nullable), thr [T,2] = (H_(k+1), H_(k)).
cudaError_t launch_gate_select(const float* H, int T, int n, int k, int32_t* idx, float* gates,
                               uint8_t* tie, float* thr, cudaStream_t s, bool sw = false,
                               int32_t* next_idx = nullptr);
// The Switch gate's sums (after launch_gate_select with sw): load [n] = routed rows per
// expert, importance [n] (nullable) = summed probabilities; part, imp_part scratch
// [gate_load_chunks(T), n].
cudaError_t launch_gate_switch_sums(const float* H, const int32_t* idx, const float* thr, int T,
                                    int n, int k, float* part, float* load, float* imp_part,
                                    float* importance, cudaStream_t s);
// Load partial sums part [ceil(T/chunk), n] of P(t,e), then load [n] in fixed chunk order.
// With imp_part and importance non-null, also the Importance (sum of kept gates)
// the same way: imp_part [ceil(T/chunk), n] scratch, importance [n].
int gate_load_chunks(int T);
cudaError_t launch_gate_load(const float* clean, const float* stdv, const int32_t* idx,
                             const float* gates, const float* thr, int T, int n, int k, float* part,
                             float* load, float* imp_part, float* importance, cudaStream_t s);
// load[e] (and importance[e] when imp_part is non-null) = fp64 sum over the
// `chunks` rows of part [chunks, n] (imp_part likewise), in a fixed order.
cudaError_t launch_partial_reduce(const float* part, const float* imp_part, int chunks, int n,
                                  float* load, float* importance, cudaStream_t s);

// ---- gate on the tensor cores (gate_tc.cu, gate_fused.cu), bf16 x only ------
// W3 scratch: 3*d x 2*gate_tc_n_pad(n) bf16 (the exact three-term split of W_g | W_noise).
int gate_tc_n_pad(int n);
cudaError_t launch_gate_split_weights(const float* W_g, const float* W_noise, int d, int n,
                                      void* W3, cudaStream_t s);
// Tensor map of a row-major bf16 [rows, cols] matrix, boxes of 64 cols x box_rows rows,
// 128-byte swizzle; false when the driver entry point is missing or rejects it.
bool gate_bf16_map(CUtensorMap* m, const void* base, long long rows, long long cols,
                   int box_rows);
int gate_sm_count();
// clean/std/H [T,n] fp32 written to memory (debug logits, and n > 256).
cudaError_t launch_gate_logits_tc(const void* x, const float* W_g, const float* W_noise,
                                  const float* eps, const float* b_g, int T, int d, int n,
                                  float std_floor, void* W3, float* clean, float* stdv, float* H,
                                  int* err, cudaStream_t s);
// Per-group split: W_g, W_noise [groups][d][n] -> W3 [groups][3d][2 n_pad].
cudaError_t launch_gate_split_weights_grouped(const float* W_g, const float* W_noise, int groups,
                                              int d, int n, void* W3, cudaStream_t s);
// The fused gate (logits never leave the SM) takes n_pad <= 256.
bool gate_tc_fusable(int n);
// idx/gates/tie [T,k]/[T]; load_part, imp_part scratch [ceil(T/128), n]; load [n];
// importance [n] optional.  load == nullptr: the partials are left for the caller to
// reduce (the dispatch's column scan).  tile_counts (nullable) [ceil(T/128), n] receives, per
// 128-token tile, how many of its routed rows go to each expert (the counting sort's
// histograms, so the dispatch can skip its counting pass).  sw: the Switch gate (the
// gates are the softmax over all n; load_part holds kept counts, imp_part the summed
// probabilities of every expert).
cudaError_t launch_gate_fused_tc(const void* x, const float* W_g, const float* W_noise,
                                 const float* eps, const float* b_g, int T, int d, int n, int k,
                                 float std_floor, void* W3, int32_t* idx, float* gates,
                                 uint8_t* tie, float* load_part, float* imp_part, float* load,
                                 float* importance, int* err, cudaStream_t s,
                                 int32_t* tile_counts = nullptr, bool sw = false);
// Gate for n > 256 (gate_big.cu): selection in the GEMM's epilogue over 128-expert
// chunks; writes clean (with the bias) and 1/std fp32 in the blocked layout
// (gate_big_blocked_floats(T, n) floats each) for launch_gate_load_blocked, and
// idx/gates [T,k], tie [T] (nullable), thr [T,2] = (H_(k+1), H_(k)).
size_t gate_big_blocked_floats(int T, int n);
int gate_big_tiles(int T);
// Load (and Importance when non-null) from the blocked clean / (1/std): per-tile partials
// load_part, imp_part [gate_big_tiles(T), n], then the fixed-order reduction.
cudaError_t launch_gate_load_blocked(const float* clean, const float* stdv, const int32_t* idx,
                                     const float* gates, const float* thr, int T, int n, int k,
                                     float* load_part, float* imp_part, float* load,
                                     float* importance, cudaStream_t s);
cudaError_t launch_gate_big_tc(const void* x, const float* W_g, const float* W_noise,
                               const float* eps, const float* b_g, int T, int d, int n, int k,
                               float std_floor, void* W3, float* clean, float* stdv, int32_t* idx,
                               float* gates, uint8_t* tie, float* thr, int* err, cudaStream_t s);
// Tokens per tile of the fused gate (the tiles of its load partials and counts).
int gate_fused_tile_tokens();

// Grouped fused gate (the secondary gates of the hierarchical layer): rows
// [offsets[g], offsets[g+1]) of x_rows [rows, d] (bf16) go through group g's gate
// (W_g, W_noise [groups][d][n], n_pad <= 256) with noise eps [routed rows][n] at
// routed row perm[p]; writes at that routed row idx [.,k] (flat ids g*n + j),
// gates [.,k] = gate_scale[row] * softmax, tie [.]; load / importance [groups*n]
// are the per-group sums of P and of the product gates.  blk_prefix [groups+1] is
// the prefix of ceil(rows_g / 128); load_part / imp_part hold
// gate_grouped_max_tiles(rows, groups) x n floats; W3 [groups][3d][2 n_pad] bf16.
int gate_grouped_max_tiles(long long rows, int groups);
cudaError_t launch_gate_grouped_tc(const void* x_rows, long long rows, const int32_t* offsets,
                                   const int32_t* blk_prefix, const int32_t* perm, int groups,
                                   const float* W_g, const float* W_noise, const float* eps,
                                   const float* gate_scale, int d, int n, int k, float std_floor,
                                   void* W3, int32_t* idx, float* gates, uint8_t* tie,
                                   float* load_part, float* imp_part, float* load,
                                   float* importance, int* err, cudaStream_t s);

// ---- dispatch (dispatch.cu) ------------------------------------------------
struct DispatchPlan {
    int tiles;   // number of row tiles of the counting sort
    int chunk;   // routed rows per tile (multiple of 32)
};
DispatchPlan dispatch_plan(long long R);
// x (row_bytes per row, a multiple of 16, required): the scatter launch also copies
// every routed row's input into x_perm (x_perm[p] = x[perm[p] / k]).  cap > 0: expert e keeps
// its first min(count_e, cap) rows; a dropped row gets inv[r] = -1 and no position.
cudaError_t launch_dispatch(const int32_t* idx, int T, int k, int n, int32_t* tile_counts,
                            int32_t* offsets, int32_t* perm, int32_t* inv, int* err,
                            cudaStream_t s, const void* x = nullptr, size_t row_bytes = 0,
                            void* x_perm = nullptr, int cap = 0);
// out[g] = sum over g' < g of ceil((offsets[g'+1] - offsets[g']) / block), out[n] = total;
// with units (nullable, int4 [total]): units[u] = (group, first row, end of the group's
// rows, 0) for every block u of that schedule.
cudaError_t launch_row_block_prefix(const int32_t* offsets, int n, int block, int32_t* out,
                                    cudaStream_t s, void* units = nullptr);
// int4 entries of the unit table for R rows over n groups in blocks of `block` rows.
inline size_t row_block_units(long long R, int n, int block) {
    return (size_t)((R + block - 1) / block) + (size_t)n + 1;
}
// The dispatch from per-tile counts already in tile_counts [tiles, n] (tile t owning
// routed rows [t*chunk, (t+1)*chunk)): column scan, offsets and the stable scatter.
// tile_counts needs (tiles + 1) * n int32 (the last n hold the totals); n <= 256 (the
// column scan is one cluster of at most eight CTAs).  With x, as launch_dispatch.
// The rest of the forward pass's bookkeeping in the same launches, all optional: with
// tail.load_part, the column scan's CTAs also sum the gate's per-tile Load / Importance
// partials (tile_sums_512 order) into tail.load / tail.importance and form the losses
// (losses_512 order); with tail.blk, they also write the expert FFN's block prefix and
// work-unit table (launch_row_block_prefix's, block tail.block).
struct DispatchTail {
    const float* load_part = nullptr;
    const float* imp_part = nullptr;
    float* load = nullptr;
    float* importance = nullptr;
    float w_imp = 0.0f, w_load = 0.0f;
    double switch_scale = 0.0;
    float* losses = nullptr;
    int32_t* blk = nullptr;
    void* units = nullptr;
    int block = 0;
};
cudaError_t launch_dispatch_counted(const int32_t* idx, long long R, int n, int tiles, int chunk,
                                    int32_t* tile_counts, int32_t* offsets, int32_t* perm,
                                    int32_t* inv, cudaStream_t s,
                                    const void* x = nullptr, int k = 1, int T = 0,
                                    size_t row_bytes = 0, void* x_perm = nullptr, int cap = 0,
                                    int* err = nullptr, const DispatchTail* tail = nullptr);

// ---- experts ---------------------------------------------------------------
// SIMT grouped FFN for fp32 experts (ffn_simt.cu); hidden [R,h] fp32 scratch.
cudaError_t launch_ffn_simt(const float* x_perm, const int32_t* offsets, const float* W_in,
                            const float* W_out, float* y_perm, float* hidden, long long R, int d,
                            int h, int n, cudaStream_t s);
// Both products in one persistent tcgen05 kernel with the hidden layer kept in L2
// between them (ffn_fused.cu): hidden [R,h] bf16 scratch, y_perm fp16, blk [n+1] and
// done [ffn_fused_count_entries(R, n)] int32 scratch.
int ffn_fused_count_entries(long long R, int n);
cudaError_t launch_ffn_fused(const void* x_perm, const int32_t* offsets, const void* W_in,
                             const void* W_out, void* y_perm, void* hidden, int32_t* blk,
                             int32_t* done, long long R, int d, int h, int n, int* err,
                             cudaStream_t s);

// The same on pairs of SMs (ffn_pair.cu, tcgen05 cta_group::2, 256-row tiles), for
// d and h multiples of 256: hidden [R,h] bf16 scratch, y_perm fp16, blk [n+1] scratch.
bool ffn_pair_supported(int d, int h);
// units: scratch of row_block_units(R, n, 256) int4 (the unit table of the 256-row blocks);
// prefix_done: blk and units were already written (the dispatch's column scan wrote
// them with block ffn_pair_block()).
int ffn_pair_block();
cudaError_t launch_ffn_pair(const void* x_perm, const int32_t* offsets, const void* W_in,
                            const void* W_out, void* y_perm, void* hidden, int32_t* blk,
                            void* units, long long R, int d, int h, int n, int* err,
                            cudaStream_t s, bool prefix_done = false);
// The backward's expert data gradients on the same kernel (d, h multiples of 256): dE
// [R,d] bf16 at the forward's routed positions -> dU [R,h] bf16 = (dE W_out[e]^T)
// [hidden_fwd > 0] and dX [R,d] fp16 = dU W_in[e]^T.
cudaError_t launch_ffn_pair_dgrad(const void* dE, const int32_t* offsets, const void* W_in,
                                  const void* W_out, const void* hidden_fwd, void* dU, void* dX,
                                  int32_t* blk, void* units, long long R, int d, int h, int n,
                                  int* err, cudaStream_t s);
// The backward's expert weight gradients on SM pairs (M, N multiples of 256): dW [n,M,N]
// fp32 with dW[e] = A_e^T B_e over expert e's rows of A [R,M] and B [R,N] (bf16);
// btail: scratch of wgrad_tail_bytes(n, N) bytes.
size_t wgrad_tail_bytes(int n, int cols);
cudaError_t launch_ffn_wgrad(const void* A, const void* B, void* btail, const int32_t* offsets,
                             long long R, int M, int N, int n, float* dW, int* err,
                             cudaStream_t s);
// Same contract with the operands exchanged (D^T = W^T x^T): each unit's MMA N is its
// expert's rows in the 256-row block rounded up to 32, so the last block of an expert
// costs what its rows need.
cudaError_t launch_ffn_swap(const void* x_perm, const int32_t* offsets, const void* W_in,
                            const void* W_out, void* y_perm, void* hidden, int32_t* blk,
                            void* units, long long R, int d, int h, int n, int* err,
                            cudaStream_t s);

// ---- backward (backward.cu) -------------------------------------------------
int backward_row_block();   // rows per unit of the expert data-gradient GEMM (64)
// g_imp / g_load [n] = w * dCV^2/dv of importance / load.
cudaError_t launch_cv2_grad(const float* importance, const float* load, int n, float w_imp,
                            float w_load, float* g_imp, float* g_load, cudaStream_t s);
// dG [T*k] = <dy_t, y_perm[inv]>, dE [T*k, d] fp32 = gates dy_t at the routed positions.
cudaError_t launch_combine_backward(const float* dy, const void* y_perm, bool half_rows,
                                    const int32_t* inv, const float* gates, int T, int k, int d,
                                    float* dG, void* dE, bool dE_bf16, cudaStream_t s);
// dclean, dnz [T,n] from the logits (clean, std), the selection (idx, gates, thr, next_idx)
// and dG, g_imp, g_load.
// split (nullable): [T][4n] bf16 = (dclean hi, lo, dnz hi, lo), the exact two-term split
// the tensor-core weight gradients take.
cudaError_t launch_gate_backward(const float* clean, const float* stdv, const float* eps,
                                 const int32_t* idx, const float* gates, const float* dG,
                                 const float* thr, const int32_t* next_idx, const float* g_imp,
                                 const float* g_load, int T, int n, int k, float std_floor,
                                 float* dclean, float* dnz, void* split, cudaStream_t s);
// dW_g, dW_noise on SM pairs (d % 256 == 0, n % 64 == 0): x^T split over 1024-token
// chunks (each a group of launch_ffn_wgrad), then a fixed-order sum of the chunks and of
// the two terms.  chunk_offsets: ceil(T/1024)+1 int32; btail: wgrad_tail_bytes(chunks, 4n);
// part: chunks * d * 4n floats.
int gate_tc_chunk();
cudaError_t launch_gate_tc_weight_grads(const void* x, const void* split, int T, int d, int n,
                                        int32_t* chunk_offsets, void* btail, float* part,
                                        float* dW_g, float* dW_noise, int* err, cudaStream_t s);
// dx += dclean W_g^T + dnz W_noise^T on the CUDA cores.
cudaError_t launch_gate_dx(const float* W_g, const float* W_noise, const float* dclean,
                           const float* dnz, int T, int d, int n, float* dx, cudaStream_t s);
// dx[t] = sum_j dXp[inv[t*k+j]] (overwrites dx).
cudaError_t launch_gather_dx(const void* dxp, bool half_rows, const int32_t* inv, int T, int k,
                             int d, float* dx, cudaStream_t s);
// out[i] = sum over t of v[t][i]; part: column_sum_scratch_floats(T, n) floats.
size_t column_sum_scratch_floats(int T, int n);
cudaError_t launch_column_sum(const float* v, int T, int n, float* out, float* part,
                              cudaStream_t s);
// dU [R,h] = (dE W_out[e]^T)[hidden > 0], dXp [R,d] = dU W_in[e]^T; units / blk from
// launch_row_block_prefix(offsets, n, backward_row_block(), blk, s, units).
cudaError_t launch_expert_dgrad(const float* dE, const void* W_in, const void* W_out,
                                const void* hidden, bool bf16, const void* units,
                                const int32_t* blk, long long R, int d, int h, int n, float* dU,
                                float* dXp, cudaStream_t s);
// dW_out [n,h,d] = hidden_e^T dE_e, dW_in [n,d,h] = x_perm_e^T dU_e (fp32, every expert).
cudaError_t launch_expert_wgrad(const void* x_perm, const void* hidden, bool bf16, const void* dE,
                                const void* dU, bool grads_bf16, const int32_t* offsets, int d,
                                int h, int n, float* dW_in, float* dW_out, cudaStream_t s);
// dW_g = x^T dclean, dW_noise = x^T dnz; dx += dclean W_g^T + dnz W_noise^T.  part:
// scratch of gate_splitk(T) * d * n floats (the split contraction's partial sums).
int gate_splitk(int T);
cudaError_t launch_gate_weight_grads(const void* x, bool x_bf16, const float* W_g,
                                     const float* W_noise, const float* dclean, const float* dnz,
                                     int T, int d, int n, float* dW_g, float* dW_noise, float* dx,
                                     float* part, cudaStream_t s);

// ---- batchwise top-m gate (batchwise.cu) -------------------------------------
// From the noisy logits H [T,n]: Ht [n,T] scratch, sel [n,m] (the tokens each expert
// takes, ascending), rowmap [T,n] (routed row i m + position, or -1), gates_r [n m]
// (softmax over the experts that took the token), importance [n], load [n] (= m).
cudaError_t launch_batch_select(const float* H, int T, int n, int m, float* Ht, int32_t* sel,
                                int32_t* rowmap, float* gates_r, float* importance, float* load,
                                cudaStream_t s);
// The inference mode: expert i takes the tokens with H > threshold[i]: counts [n],
// offsets [n+1] (clamped to cap rows, an excess raising DEV_RANGE), sel [cap] expert-major
// ascending tokens, rowmap, gates_r [cap], importance / load [n] (load = rows taken).
cudaError_t launch_threshold_select(const float* H, int T, int n, const float* threshold,
                                    long long cap, float* Ht, int32_t* counts, int32_t* offsets,
                                    int32_t* sel, int32_t* rowmap, float* gates_r,
                                    float* importance, float* load, int* err, cudaStream_t s);
// x_perm [n m, d] = x[sel], offsets [n+1] = e m; with given_rows_cap > 0 the offsets are
// read instead (rows = offsets[n] <= given_rows_cap).
cudaError_t launch_batch_gather(const void* x, size_t row_bytes, const int32_t* sel, int n, int m,
                                void* x_perm, int32_t* offsets, cudaStream_t s,
                                long long given_rows_cap = 0);
// y [T,d] = per token, over the experts that took it in ascending order, gates_r y_perm.
cudaError_t launch_batch_combine(const void* y_perm, bool half_rows, const int32_t* rowmap,
                                 const float* gates_r, int T, int n, int d, float* y,
                                 cudaStream_t s);

// ---- combine (combine.cu) --------------------------------------------------
// y_perm is fp16 when half_rows, else fp32.
cudaError_t launch_combine(const void* y_perm, bool half_rows, const int32_t* inv,
                           const float* gates, int T, int k, int d, float* y, cudaStream_t s);

// ---- balance (balance.cu) --------------------------------------------------
// importance [n] = the kept gates summed per expert in the dispatch's grouped order;
// launch_cv2_losses: losses [3] from importance and load (one 512-thread CTA,
// losses_512 order).  switch_scale > 0: the Switch loss
// switch_scale * sum_i load_i importance_i instead of the CV^2 losses.
cudaError_t launch_importance(const float* gates, const int32_t* perm, const int32_t* offsets,
                              int n, float* importance, cudaStream_t s);
cudaError_t launch_cv2_losses(const float* importance, const float* load, int n, float w_imp,
                              float w_load, float* losses, cudaStream_t s,
                              double switch_scale = 0.0);

// ---- the gate's share of dx on the tensor cores (gate_dx.cu) -------------------
// dx [T,d] += dclean W_g^T + dnz W_noise^T from the gate backward's split [T][4n] bf16
// (clean hi, clean lo, noise hi, noise lo); W2: gate_dx_split_bytes(d, n) of scratch.
bool gate_dx_tc_supported(int d, int n);
size_t gate_dx_split_bytes(int d, int n);
cudaError_t launch_gate_dx_tc(const float* W_g, const float* W_noise, const void* split, int T,
                              int d, int n, void* W2, float* dx, int* err, cudaStream_t s);

// ---- the gate's noise drawn on the device (noise.cu) ---------------------------
// eps[i] = the standard normal draw of element i (i < count) for `seed` (the
// counter-based generator of noise.cu; element t n + e is token t's draw for expert e).
// wait = false only for the layer's own draw into its workspace (see noise.cu).
cudaError_t launch_noise(unsigned long long seed, long long count, float* eps, cudaStream_t s,
                         bool wait = true);

// ---- sharding over several GPUs (shards.cu) ----------------------------------
// Host only: the exchange plan of `rank` from every rank's dispatch offsets offs
// [world][n+1] (n a multiple of world, rank r holding experts [r n/world, (r+1) n/world)).
// send_rows / recv_rows [world]; plan [2 B + 1 + n/world + 1], B = world * n/world:
// source-major start of block (e, s) at e*world + s, then the expert-major starts of
// the same blocks and the total, then the local expert offsets.  Returns 0, 1 for
// offsets that do not start at 0 or decrease, 2 when the rows received reach 2^31.
int ep_plan_host(int world, int rank, int n, const int32_t* offs, int32_t* send_rows,
                 int32_t* recv_rows, int32_t* plan);
// Rows between the arrival order (source major) and the FFN order (expert major):
// to_expert_major: out[p] = in[src(p)]; else out[src(p)] = in[p].  plan on the device.
cudaError_t launch_ep_regroup(int world, int n_local, const int32_t* plan, const void* in,
                              void* out, size_t row_bytes, int to_expert_major, int sms,
                              cudaStream_t s);

// ---- failure detection (selftest.cu) ----------------------------------------
// One CTA whose bounded waits run out after budget_cycles: DEV_TIMEOUT in *err.
cudaError_t launch_timeout_probe(long long budget_cycles, int* err, cudaStream_t s);

}  // namespace moe
