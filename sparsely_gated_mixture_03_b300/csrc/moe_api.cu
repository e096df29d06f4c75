// C ABI of the MoE forward pass: argument checks, workspace layout and the
// launch sequence of each entry point.  Declarations and contracts: include/moe.h.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "moe.h"
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {
std::atomic<unsigned long long> g_launches{0};
}
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
}  // namespace moe

namespace {

// The device error word the kernels set instead of trapping (see moe_get_device_error).
__device__ int g_moe_error_word;

int* device_error_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_error_word) != cudaSuccess) return nullptr;
    return static_cast<int*>(p);
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

size_t dtype_bytes(moe_dtype t) { return t == MOE_BF16 ? 2 : 4; }

// Byte offsets of every scratch region inside the workspace.
struct Layout {
    size_t clean, stdv, H, thr, load_part, imp_part, w3;
    size_t idx, gates, tie, load, importance;
    size_t tile_counts, offsets, perm, inv;
    size_t x_perm, hidden, y_perm, mt_prefix, units, ffn_done, noise;
    size_t total;
};

Layout make_layout(const moe_config& c) {
    Layout L{};
    const size_t T = c.T, n = c.n, R = (size_t)c.T * c.k;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    // clean / std / H: [T,n] each for the CUDA-core gate (fp32 x); the blocked clean and
    // std of the large-n tensor-core gate; nothing when the whole gate is one fused kernel
    const bool tc_gate = c.x_dtype == MOE_BF16;
    const bool sw = (c.flags & MOE_FLAG_SWITCH_GATE) != 0;
    // the logits path (CUDA-core gate, or the Switch gate above 256 experts) keeps all three
    const bool logits_path = !tc_gate || (sw && !moe::gate_tc_fusable(c.n));
    const size_t tn = logits_path ? T * n
                      : moe::gate_tc_fusable(c.n) ? 0 : moe::gate_big_blocked_floats(c.T, c.n);
    L.clean = take(tn * 4);
    L.stdv = take(tn * 4);
    L.H = take(logits_path ? T * n * 4 : 0);
    L.thr = take(T * 2 * 4);
    L.load_part = take((size_t)moe::gate_load_chunks(c.T) * n * 4);
    L.imp_part = take((size_t)moe::gate_load_chunks(c.T) * n * 4);
    L.w3 = take(c.x_dtype == MOE_BF16 ? (size_t)3 * c.d * 2 * moe::gate_tc_n_pad(c.n) * 2 : 0);
    L.idx = take(R * 4);
    L.gates = take(R * 4);
    L.tie = take(T);
    L.load = take(n * 4);
    L.importance = take(n * 4);
    const moe::DispatchPlan dp = moe::dispatch_plan((long long)R);
    const size_t gate_tiles =
        (c.T + moe::gate_fused_tile_tokens() - 1) / moe::gate_fused_tile_tokens();
    L.tile_counts = take(((size_t)(dp.tiles > (int)gate_tiles ? dp.tiles : gate_tiles) + 1) * n * 4);
    L.offsets = take((n + 1) * 4);
    L.perm = take(R * 4);
    L.inv = take(R * 4);
    L.x_perm = take(R * c.d * dtype_bytes(c.x_dtype));
    L.hidden = take(R * c.h * dtype_bytes(c.expert_dtype));
    L.y_perm = take(R * c.d * dtype_bytes(c.expert_dtype));   // fp16 for bf16 experts
    L.mt_prefix = take((n + 1) * 4);
    L.units = take(moe::row_block_units((long long)R, c.n, 256) * 16);
    L.ffn_done = take((size_t)moe::ffn_fused_count_entries((long long)R, c.n) * 4);
    L.noise = take((c.flags & MOE_FLAG_DEVICE_NOISE) ? T * n * 4 : 0);   // the drawn eps [T,n]
    L.total = o;
    return L;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_config(const moe_config* c) {
    if (c == nullptr) return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->d < 1 || c->n < 1 || c->h < 1 || c->k < 1 || c->k > c->n)
        return MOE_ERR_INVALID_ARG;
    if ((c->flags & ~(MOE_FLAG_FFN_ROW_TILES | MOE_FLAG_FFN_SIZED_TILES | MOE_FLAG_SWITCH_GATE |
                      MOE_FLAG_DEVICE_NOISE)) != 0 ||
        (c->flags & MOE_FLAG_FFN_ROW_TILES && c->flags & MOE_FLAG_FFN_SIZED_TILES))
        return MOE_ERR_INVALID_ARG;
    if (c->x_dtype != MOE_F32 && c->x_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->expert_dtype != MOE_F32 && c->expert_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->k > 8 || c->n > 16384 || c->d % 64 != 0 || c->h % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if ((long long)c->T * c->k >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    if (c->x_dtype != c->expert_dtype) return MOE_ERR_UNSUPPORTED;
    if (!(c->std_floor >= 0.0f)) return MOE_ERR_INVALID_ARG;
    if (c->capacity < 0) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

// MOE_FLAG_DEVICE_NOISE: the caller passes no eps; the layer draws it into the
// workspace (noise.cu's generator, seed c.noise_seed) and points eps there.
moe_status draw_noise_into(const moe_config& c, const float*& eps, void* ws, cudaStream_t s) {
    if ((c.flags & MOE_FLAG_DEVICE_NOISE) == 0) return MOE_OK;
    if (eps != nullptr) return MOE_ERR_INVALID_ARG;
    float* out = reinterpret_cast<float*>(static_cast<char*>(ws) + make_layout(c).noise);
    const cudaError_t e = moe::launch_noise(c.noise_seed, (long long)c.T * c.n, out, s, false);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    eps = out;
    return MOE_OK;
}

moe_status check_workspace(const moe_config* c, const void* ws, size_t bytes) {
    if (ws == nullptr) return MOE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return MOE_ERR_WORKSPACE;
    if (bytes < make_layout(*c).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

// The last CUDA error an entry point returned MOE_ERR_CUDA for, per host thread.
thread_local cudaError_t g_last_cuda_error = cudaSuccess;

moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    g_last_cuda_error = e;
    return MOE_ERR_CUDA;
}

#define MOE_TRY(expr)                          \
    do {                                       \
        const moe_status _st = (expr);         \
        if (_st != MOE_OK) return _st;         \
    } while (0)

#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// ---- stage bodies (arguments already checked) ---------------------------------

// importance: optional; when given, the Importance is summed in the same pass as
// the Load (per token chunk in fp32, then over chunks in fp64).
// bf16 x runs the gate GEMM on the tensor cores: fused (nothing [T,n] leaves the SM)
// for n <= 256 unless the debug logits are requested, else logits to memory first.
moe_status gate_body(const moe_config& c, const void* x, const float* W_g, const float* W_noise,
                     const float* eps, const float* b_g, int32_t* idx, float* gates, uint8_t* tie,
                     float* load, float* importance, float* logits, void* ws, cudaStream_t s) {
    const Layout L = make_layout(c);
    const size_t tn = (size_t)c.T * c.n;
    float* clean = logits != nullptr ? logits : at<float>(ws, L.clean);
    float* stdv = logits != nullptr ? logits + tn : at<float>(ws, L.stdv);
    float* H = logits != nullptr ? logits + 2 * tn : at<float>(ws, L.H);
    float* thr = at<float>(ws, L.thr);
    const bool sw = (c.flags & MOE_FLAG_SWITCH_GATE) != 0;
    if (c.x_dtype == MOE_BF16) {
        int* err = device_error_word();
        if (err == nullptr) return MOE_ERR_CUDA;
        if (logits == nullptr && moe::gate_tc_fusable(c.n)) {
            MOE_CUDA(moe::launch_gate_fused_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.k,
                                               c.std_floor, at<void>(ws, L.w3), idx, gates, tie,
                                               at<float>(ws, L.load_part),
                                               at<float>(ws, L.imp_part), load, importance, err,
                                               s, nullptr, sw));
            return MOE_OK;
        }
        if (logits == nullptr && !sw) {
            // more than 256 experts: selection in the GEMM's epilogue, clean and std to
            // memory for the Load pass (the noisy logits never reach memory)
            MOE_CUDA(moe::launch_gate_big_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.k,
                                             c.std_floor, at<void>(ws, L.w3), clean, stdv, idx,
                                             gates, tie, thr, err, s));
            MOE_CUDA(moe::launch_gate_load_blocked(clean, stdv, idx, gates, thr, c.T, c.n, c.k,
                                                   at<float>(ws, L.load_part),
                                                   at<float>(ws, L.imp_part), load, importance,
                                                   s));
            return MOE_OK;
        }
        MOE_CUDA(moe::launch_gate_logits_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.std_floor,
                                            at<void>(ws, L.w3), clean, stdv, H, err, s));
    } else {
        MOE_CUDA(moe::launch_gate_logits(x, false, W_g, W_noise, eps, b_g, c.T, c.d, c.n,
                                         c.std_floor, clean, stdv, H, s));
    }
    MOE_CUDA(moe::launch_gate_select(H, c.T, c.n, c.k, idx, gates, tie, thr, s, sw));
    if (sw)
        MOE_CUDA(moe::launch_gate_switch_sums(H, idx, thr, c.T, c.n, c.k,
                                              at<float>(ws, L.load_part), load,
                                              at<float>(ws, L.imp_part), importance, s));
    else
        MOE_CUDA(moe::launch_gate_load(clean, stdv, idx, gates, thr, c.T, c.n, c.k,
                                       at<float>(ws, L.load_part), load,
                                       at<float>(ws, L.imp_part), importance, s));
    return MOE_OK;
}

moe_status dispatch_body(const moe_config& c, const int32_t* idx, const void* x, int32_t* offsets,
                         int32_t* perm, int32_t* inv, void* x_perm, void* ws, cudaStream_t s) {
    const Layout L = make_layout(c);
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    MOE_CUDA(moe::launch_dispatch(idx, c.T, c.k, c.n, at<int32_t>(ws, L.tile_counts), offsets,
                                  perm, inv, err, s, x, (size_t)c.d * dtype_bytes(c.x_dtype),
                                  x_perm, c.capacity));
    return MOE_OK;
}

// 256-row tiles unless tiles sized to each expert's rows are asked for: measured on
// one B300, the 256-row kernel is the faster one at 512 rows per expert (0.263 ms
// against 0.332 ms) and at 64 (1.73 ms against 1.84 ms at a lower clock): both stream
// the same weight bytes, and the sized tiles pay a transposing epilogue and
// cluster-scope hand-offs of the hidden blocks.
bool ffn_row_tiles(unsigned flags, long long /*R*/, long long /*n*/) {
    return (flags & MOE_FLAG_FFN_SIZED_TILES) == 0;
}

// The FFN runs the SM-pair kernel with its 256-row unit table.
bool ffn_uses_pairs(const moe_config& c) {
    return c.expert_dtype == MOE_BF16 && moe::ffn_pair_supported(c.d, c.h) &&
           ffn_row_tiles(c.flags, (long long)c.T * c.k, c.n);
}

// prefix_done: the unit table of the pair kernel is already in the workspace (the
// dispatch's column scan wrote it).
moe_status ffn_body(const moe_config& c, const void* x_perm, const int32_t* offsets,
                    const void* W_in, const void* W_out, void* y_perm, void* ws, cudaStream_t s,
                    bool prefix_done = false) {
    const Layout L = make_layout(c);
    const long long R = (long long)c.T * c.k;
    if (c.expert_dtype == MOE_BF16) {
        int* err = device_error_word();
        if (err == nullptr) return MOE_ERR_CUDA;
        if (moe::ffn_pair_supported(c.d, c.h) && ffn_row_tiles(c.flags, R, c.n))
            MOE_CUDA(moe::launch_ffn_pair(x_perm, offsets, W_in, W_out, y_perm,
                                          at<void>(ws, L.hidden), at<int32_t>(ws, L.mt_prefix),
                                          at<void>(ws, L.units), R, c.d, c.h, c.n, err, s,
                                          prefix_done));
        else if (moe::ffn_pair_supported(c.d, c.h))
            MOE_CUDA(moe::launch_ffn_swap(x_perm, offsets, W_in, W_out, y_perm,
                                          at<void>(ws, L.hidden), at<int32_t>(ws, L.mt_prefix),
                                          at<void>(ws, L.units), R, c.d, c.h, c.n, err, s));
        else
            MOE_CUDA(moe::launch_ffn_fused(x_perm, offsets, W_in, W_out, y_perm,
                                           at<void>(ws, L.hidden), at<int32_t>(ws, L.mt_prefix),
                                           at<int32_t>(ws, L.ffn_done), R, c.d, c.h, c.n, err,
                                           s));
    } else {
        MOE_CUDA(moe::launch_ffn_simt(static_cast<const float*>(x_perm), offsets,
                                      static_cast<const float*>(W_in),
                                      static_cast<const float*>(W_out), static_cast<float*>(y_perm),
                                      at<float>(ws, L.hidden), R, c.d, c.h, c.n, s));
    }
    return MOE_OK;
}

// ---- hierarchical layer ----------------------------------------------------------

struct HierLayout {
    size_t w3_1, idx1, gates1, tie1, load_part1, imp_part1, load1, importance1;
    size_t tile_counts1, offsets1, perm1, inv1, x1_perm, blk1, w3_2, tie2;
    size_t load_part2, imp_part2, load2, importance;
    size_t idx, gates, tile_counts, offsets, perm, inv, x_perm, hidden, y_perm, mt_prefix, units;
    size_t ffn_done;
    size_t total;
};

HierLayout make_hier_layout(const moe_hier_config& c) {
    HierLayout L{};
    const size_t T = c.T, a = c.a, nb = (size_t)c.a * c.b;
    const size_t R1 = (size_t)c.T * c.k1, K = (size_t)c.k1 * c.k2, R = T * K;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    L.w3_1 = take((size_t)3 * c.d * 2 * moe::gate_tc_n_pad(c.a) * 2);
    L.idx1 = take(R1 * 4);
    L.gates1 = take(R1 * 4);
    L.tie1 = take(T);
    L.load_part1 = take((size_t)moe::gate_load_chunks(c.T) * a * 4);
    L.imp_part1 = take((size_t)moe::gate_load_chunks(c.T) * a * 4);
    L.load1 = take(a * 4);
    L.importance1 = take(a * 4);
    const moe::DispatchPlan dp1 = moe::dispatch_plan((long long)R1);
    L.tile_counts1 = take(((size_t)dp1.tiles + 1) * a * 4);
    L.offsets1 = take((a + 1) * 4);
    L.perm1 = take(R1 * 4);
    L.inv1 = take(R1 * 4);
    L.x1_perm = take(R1 * c.d * 2);
    L.blk1 = take((a + 1) * 4);
    L.w3_2 = take(a * 3 * c.d * 2 * moe::gate_tc_n_pad(c.b) * 2);
    L.tie2 = take(R1);
    const size_t tiles2 = (size_t)moe::gate_grouped_max_tiles((long long)R1, c.a);
    L.load_part2 = take(tiles2 * c.b * 4);
    L.imp_part2 = take(tiles2 * c.b * 4);
    L.load2 = take(nb * 4);
    L.importance = take(nb * 4);
    L.idx = take(R * 4);
    L.gates = take(R * 4);
    const moe::DispatchPlan dp = moe::dispatch_plan((long long)R);
    L.tile_counts = take(((size_t)dp.tiles + 1) * nb * 4);
    L.offsets = take((nb + 1) * 4);
    L.perm = take(R * 4);
    L.inv = take(R * 4);
    L.x_perm = take(R * c.d * 2);
    L.hidden = take(R * c.h * 2);
    L.y_perm = take(R * c.d * 2);
    L.mt_prefix = take((nb + 1) * 4);
    L.units = take(moe::row_block_units((long long)R, (int)nb, 256) * 16);
    L.ffn_done = take((size_t)moe::ffn_fused_count_entries((long long)R, (int)nb) * 4);
    L.total = o;
    return L;
}

moe_status check_hier_config(const moe_hier_config* c) {
    if (c == nullptr) return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->d < 1 || c->a < 1 || c->b < 1 || c->h < 1 || c->k1 < 1 || c->k2 < 1 ||
        c->k1 > c->a || c->k2 > c->b)
        return MOE_ERR_INVALID_ARG;
    if ((c->flags & ~(MOE_FLAG_FFN_ROW_TILES | MOE_FLAG_FFN_SIZED_TILES)) != 0 ||
        (c->flags & MOE_FLAG_FFN_ROW_TILES && c->flags & MOE_FLAG_FFN_SIZED_TILES))
        return MOE_ERR_INVALID_ARG;
    if (c->x_dtype != MOE_F32 && c->x_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->expert_dtype != MOE_F32 && c->expert_dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (!(c->std_floor >= 0.0f)) return MOE_ERR_INVALID_ARG;
    if (c->x_dtype != MOE_BF16 || c->expert_dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (c->k1 * c->k2 > 8 || c->d % 64 != 0 || c->h % 64 != 0) return MOE_ERR_UNSUPPORTED;
    if (!moe::gate_tc_fusable(c->a) || !moe::gate_tc_fusable(c->b)) return MOE_ERR_UNSUPPORTED;
    if ((long long)c->a * c->b > 16384) return MOE_ERR_UNSUPPORTED;
    if ((long long)c->T * c->k1 * c->k2 >= (1LL << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

}  // namespace

// Scratch of moe_dispatch_noalloc: the counting sort's per-tile expert counts
// ((tiles + 1) * n int32) for callers that cannot hand the library any device
// memory.  Every device that loads the library holds these 1 MiB until exit.
static __device__ __align__(256) int32_t g_noalloc_dispatch_scratch[MOE_NOALLOC_DISPATCH_INTS];

namespace {

constexpr int kMaxDevices = 64;

// Looks the array's device address up once per device, on the first call made
// with that device current, and caches it; no memory is allocated.  The cache
// lives as long as the process: a cudaDeviceReset (a new primary context, which
// may load the module elsewhere) leaves it stale.
moe_status noalloc_scratch(int32_t** out) {
    static std::mutex mu;
    static int32_t* addr[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_dispatch_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        addr[dev] = static_cast<int32_t*>(p);
    }
    *out = addr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: invalid argument";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape or dtype not supported";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace too small or misaligned";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call failed";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT: a device-side bounded wait expired";
        case MOE_ERR_RANGE: return "MOE_ERR_RANGE: a value beyond what its output holds";
    }
    return "unknown moe_status";
}

moe_status moe_workspace_size(const moe_config* cfg, size_t* bytes) {
    MOE_TRY(check_config(cfg));
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *bytes = make_layout(*cfg).total;
    return MOE_OK;
}

moe_status moe_draw_noise(unsigned long long seed, long long count, float* eps,
                          cudaStream_t stream) {
    if (count < 0 || (count > 0 && eps == nullptr)) return MOE_ERR_INVALID_ARG;
    return cuda_status(moe::launch_noise(seed, count, eps, stream));
}

moe_status moe_gate(const moe_config* cfg, const void* x, const float* W_g, const float* W_noise,
                    const float* eps, const float* b_g, int32_t* idx, float* gates, uint8_t* tie,
                    float* load, float* logits, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!x || !W_g || !W_noise || !idx || !gates || !load) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_g) || !aligned16(W_noise) || (eps && !aligned16(eps)))
        return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_workspace(cfg, workspace, workspace_bytes));
    MOE_TRY(draw_noise_into(*cfg, eps, workspace, stream));
    return gate_body(*cfg, x, W_g, W_noise, eps, b_g, idx, gates, tie, load, nullptr, logits,
                     workspace,
                     stream);
}

moe_status moe_dispatch(const moe_config* cfg, const int32_t* idx, const void* x,
                        int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!idx || !x || !offsets || !perm || !inv || !x_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_workspace(cfg, workspace, workspace_bytes));
    return dispatch_body(*cfg, idx, x, offsets, perm, inv, x_perm, workspace, stream);
}

moe_status moe_dispatch_noalloc(const moe_config* cfg, const int32_t* idx, const void* x,
                                int32_t* offsets, int32_t* perm, int32_t* inv, void* x_perm,
                                cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!idx || !x || !offsets || !perm || !inv || !x_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_UNSUPPORTED;
    // the scratch launch_dispatch uses: (tiles + 1) * n counts of the same plan
    const long long tiles = moe::dispatch_plan((long long)cfg->T * cfg->k).tiles;
    if ((tiles + 1) * cfg->n > MOE_NOALLOC_DISPATCH_INTS) return MOE_ERR_WORKSPACE;
    int32_t* scratch = nullptr;
    MOE_TRY(noalloc_scratch(&scratch));
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    MOE_CUDA(moe::launch_dispatch(idx, cfg->T, cfg->k, cfg->n, scratch, offsets, perm, inv, err,
                                  stream, x, (size_t)cfg->d * dtype_bytes(cfg->x_dtype), x_perm,
                                  cfg->capacity));
    return MOE_OK;
}

moe_status moe_expert_ffn(const moe_config* cfg, const void* x_perm, const int32_t* offsets,
                          const void* W_in, const void* W_out, void* y_perm, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!x_perm || !offsets || !W_in || !W_out || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(W_in) || !aligned16(W_out) || !aligned16(y_perm))
        return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_workspace(cfg, workspace, workspace_bytes));
    return ffn_body(*cfg, x_perm, offsets, W_in, W_out, y_perm, workspace, stream);
}

moe_status moe_combine(const moe_config* cfg, const void* y_perm, const int32_t* inv,
                       const float* gates, float* y, cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!y_perm || !inv || !gates || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_perm) || !aligned16(y)) return MOE_ERR_UNSUPPORTED;
    return cuda_status(moe::launch_combine(y_perm, cfg->expert_dtype == MOE_BF16, inv, gates,
                                           cfg->T, cfg->k, cfg->d, y, stream));
}

moe_status moe_balance_losses(const moe_config* cfg, const float* gates, const int32_t* perm,
                              const int32_t* offsets, const float* load, float* importance,
                              float* losses, cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!gates || !perm || !offsets || !load || !importance || !losses) return MOE_ERR_INVALID_ARG;
    if (cfg->capacity > 0) return MOE_ERR_UNSUPPORTED;   // perm lists the kept rows only
    if (cfg->flags & MOE_FLAG_SWITCH_GATE) return MOE_ERR_UNSUPPORTED;   // needs every probability
    MOE_CUDA(moe::launch_importance(gates, perm, offsets, cfg->n, importance, stream));
    MOE_CUDA(moe::launch_cv2_losses(importance, load, cfg->n, cfg->w_importance, cfg->w_load,
                                    losses, stream));
    return MOE_OK;
}

moe_status moe_losses_from_sums(const moe_config* cfg, const float* importance, const float* load,
                                float* losses, cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!importance || !load || !losses) return MOE_ERR_INVALID_ARG;
    const moe_config& c = *cfg;
    const double switch_scale = (c.flags & MOE_FLAG_SWITCH_GATE)
                                    ? (double)c.n / ((double)c.T * c.k * (double)c.T) : 0.0;
    MOE_CUDA(moe::launch_cv2_losses(importance, load, c.n, c.w_importance, c.w_load, losses,
                                    stream, switch_scale));
    return MOE_OK;
}

moe_status moe_ep_plan(int world, int rank, int n, const int32_t* all_offsets,
                       int32_t* send_rows, int32_t* recv_rows, int32_t* plan) {
    if (world < 1 || rank < 0 || rank >= world || n < 1) return MOE_ERR_INVALID_ARG;
    if (!all_offsets || !send_rows || !recv_rows || !plan) return MOE_ERR_INVALID_ARG;
    if (n % world != 0) return MOE_ERR_UNSUPPORTED;
    const int r = moe::ep_plan_host(world, rank, n, all_offsets, send_rows, recv_rows, plan);
    return r == 0 ? MOE_OK : (r == 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_UNSUPPORTED);
}

moe_status moe_ep_regroup(int world, int n_local, const int32_t* plan, const void* in, void* out,
                          size_t row_bytes, int to_expert_major, cudaStream_t stream) {
    if (world < 1 || n_local < 1 || !plan || !in || !out) return MOE_ERR_INVALID_ARG;
    if (row_bytes == 0 || row_bytes % 16 != 0 || !aligned16(in) || !aligned16(out))
        return MOE_ERR_UNSUPPORTED;
    if ((long long)world * n_local >= (1LL << 30)) return MOE_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    MOE_CUDA(cudaGetDevice(&dev));
    MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    MOE_CUDA(moe::launch_ep_regroup(world, n_local, plan, in, out, row_bytes, to_expert_major,
                                    sms > 0 ? sms : 148, stream));
    return MOE_OK;
}

}  // extern "C"

namespace {

// One forward pass; events (six, or null) are recorded on the stream before the gate,
// after the gate, the dispatch, the experts, the combine and the losses.
moe_status forward_body(const moe_config* cfg, const void* x, const float* W_g,
                        const float* W_noise, const float* eps, const float* b_g, const void* W_in,
                        const void* W_out, float* y, float* losses, int32_t* idx, float* gates,
                        uint8_t* tie, float* importance, float* load, void* workspace,
                        size_t workspace_bytes, cudaStream_t stream, cudaEvent_t* ev) {
    MOE_TRY(check_config(cfg));
    if (!x || !W_g || !W_noise || !W_in || !W_out || !y || !losses)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_g) || !aligned16(W_noise) || (eps && !aligned16(eps)) ||
        !aligned16(W_in) || !aligned16(W_out) || !aligned16(y))
        return MOE_ERR_UNSUPPORTED;
    MOE_TRY(check_workspace(cfg, workspace, workspace_bytes));
    const moe_config& c = *cfg;
    const Layout L = make_layout(c);
    void* ws = workspace;
    const bool sw = (c.flags & MOE_FLAG_SWITCH_GATE) != 0;
    // the Switch loss n * sum_i (load_i / (T k)) (importance_i / T)
    const double switch_scale = sw ? (double)c.n / ((double)c.T * c.k * (double)c.T) : 0.0;
    if (!idx) idx = at<int32_t>(ws, L.idx);
    if (!gates) gates = at<float>(ws, L.gates);
    if (!tie) tie = at<uint8_t>(ws, L.tie);
    if (!importance) importance = at<float>(ws, L.importance);
    if (!load) load = at<float>(ws, L.load);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* perm = at<int32_t>(ws, L.perm);
    int32_t* inv = at<int32_t>(ws, L.inv);
    void* x_perm = at<void>(ws, L.x_perm);
    void* y_perm = at<void>(ws, L.y_perm);
    auto mark = [&](int i) -> moe_status {
        return ev != nullptr ? cuda_status(cudaEventRecord(ev[i], stream)) : MOE_OK;
    };
    MOE_TRY(mark(0));
    MOE_TRY(draw_noise_into(c, eps, ws, stream));
    if (c.x_dtype == MOE_BF16 && moe::gate_tc_fusable(c.n)) {
        // the fused gate also counts each 128-token tile's routed rows per expert (the
        // dispatch starts from its scan) and leaves its Load / Importance partials to
        // the last kernel, which reduces them and forms the losses
        int* err = device_error_word();
        if (err == nullptr) return MOE_ERR_CUDA;
        const int tt = moe::gate_fused_tile_tokens();
        const int tiles = (c.T + tt - 1) / tt;
        MOE_CUDA(moe::launch_gate_fused_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.k,
                                           c.std_floor, at<void>(ws, L.w3), idx, gates, tie,
                                           at<float>(ws, L.load_part), at<float>(ws, L.imp_part),
                                           nullptr, nullptr, err, stream,
                                           at<int32_t>(ws, L.tile_counts), sw));
        MOE_TRY(mark(1));
        // the column scan of the counting sort also reduces the gate's Load / Importance
        // partials and forms the losses in its last CTA (which also writes the FFN's unit
        // table when the pair kernel runs): nothing is left for the end of the pass
        moe::DispatchTail tail;
        tail.load_part = at<float>(ws, L.load_part);
        tail.imp_part = at<float>(ws, L.imp_part);
        tail.load = load;
        tail.importance = importance;
        tail.w_imp = c.w_importance;
        tail.w_load = c.w_load;
        tail.switch_scale = switch_scale;
        tail.losses = losses;
        const bool pairs = ffn_uses_pairs(c);
        if (pairs) {
            tail.blk = at<int32_t>(ws, L.mt_prefix);
            tail.units = at<void>(ws, L.units);
            tail.block = moe::ffn_pair_block();
        }
        MOE_CUDA(moe::launch_dispatch_counted(idx, (long long)c.T * c.k, c.n, tiles, tt * c.k,
                                              at<int32_t>(ws, L.tile_counts), offsets, perm, inv,
                                              stream, x, c.k, c.T,
                                              (size_t)c.d * dtype_bytes(c.x_dtype), x_perm,
                                              c.capacity, err, &tail));
        MOE_TRY(mark(2));
        MOE_TRY(ffn_body(c, x_perm, offsets, W_in, W_out, y_perm, ws, stream, pairs));
        MOE_TRY(mark(3));
        MOE_CUDA(moe::launch_combine(y_perm, true, inv, gates, c.T, c.k, c.d, y, stream));
        MOE_TRY(mark(4));
        MOE_TRY(mark(5));          // the losses were formed with the dispatch
        return MOE_OK;
    }
    // Importance is summed inside the gate pass, in the same fixed order as the Load.
    MOE_TRY(gate_body(c, x, W_g, W_noise, eps, b_g, idx, gates, tie, load, importance, nullptr, ws,
                      stream));
    MOE_TRY(mark(1));
    MOE_TRY(dispatch_body(c, idx, x, offsets, perm, inv, x_perm, ws, stream));
    MOE_TRY(mark(2));
    MOE_TRY(ffn_body(c, x_perm, offsets, W_in, W_out, y_perm, ws, stream));
    MOE_TRY(mark(3));
    MOE_CUDA(moe::launch_combine(y_perm, c.expert_dtype == MOE_BF16, inv, gates, c.T, c.k, c.d, y,
                                 stream));
    MOE_TRY(mark(4));
    MOE_CUDA(moe::launch_cv2_losses(importance, load, c.n, c.w_importance, c.w_load, losses,
                                    stream, switch_scale));
    MOE_TRY(mark(5));
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward(const moe_config* cfg, const void* x, const float* W_g,
                       const float* W_noise, const float* eps, const float* b_g, const void* W_in,
                       const void* W_out, float* y, float* losses, int32_t* idx, float* gates,
                       uint8_t* tie, float* importance, float* load, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
    return forward_body(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, y, losses, idx, gates, tie,
                        importance, load, workspace, workspace_bytes, stream, nullptr);
}

moe_status moe_forward_timed(const moe_config* cfg, const void* x, const float* W_g,
                             const float* W_noise, const float* eps, const float* b_g,
                             const void* W_in, const void* W_out, float* y, float* losses,
                             int32_t* idx, float* gates, uint8_t* tie, float* importance,
                             float* load, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream, cudaEvent_t* stage_events) {
    if (stage_events == nullptr) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (stage_events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    return forward_body(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, y, losses, idx, gates, tie,
                        importance, load, workspace, workspace_bytes, stream, stage_events);
}

}  // extern "C"

namespace {

// The gate's weight gradients go to SM pairs for bf16 x with d a multiple of 256 and n
// of 64 (the split operand [T][4n] then has 4n a multiple of 256).
bool gate_grads_on_pairs(const moe_config& c) {
    return c.x_dtype == MOE_BF16 && c.d % 256 == 0 && c.n % 64 == 0;
}

// The backward's scratch: the forward's layout (its recompute) followed by the logits,
// the selection's extra outputs and the gradient buffers.
struct BwdLayout {
    Layout F;
    size_t clean, stdv, H, next_idx, dG, g_imp, g_load, dE, dU, dXp, dclean, dnz, blk, units,
        gate_part, wg_tail, gsplit, gchunks, gtail, gdx_w2, colsum;
    size_t total;
};

BwdLayout make_bwd_layout(const moe_config& c) {
    BwdLayout L{};
    L.F = make_layout(c);
    const size_t T = c.T, n = c.n, R = (size_t)c.T * c.k;
    size_t o = L.F.total;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    L.clean = take(T * n * 4);
    L.stdv = take(T * n * 4);
    L.H = take(T * n * 4);
    L.next_idx = take(T * 4);
    L.dG = take(R * 4);
    L.g_imp = take(n * 4);
    L.g_load = take(n * 4);
    L.dE = take(R * c.d * 4);
    L.dU = take(R * c.h * 4);
    L.dXp = take(R * c.d * 4);
    L.dclean = take(T * n * 4);
    L.dnz = take(T * n * 4);
    L.blk = take((n + 1) * 4);
    L.units = take(moe::row_block_units((long long)R, c.n, moe::backward_row_block()) * 16);
    L.gate_part = take((size_t)moe::gate_splitk(c.T) * c.d * n * 4);
    L.wg_tail = take(moe::wgrad_tail_bytes(c.n, c.d > c.h ? c.d : c.h));
    L.colsum = take(moe::column_sum_scratch_floats(c.T, c.n) * 4);
    if (gate_grads_on_pairs(c)) {
        const int chunks = (c.T + moe::gate_tc_chunk() - 1) / moe::gate_tc_chunk();
        L.gsplit = take(T * 4 * n * 2);
        L.gdx_w2 = take(moe::gate_dx_split_bytes(c.d, c.n));
        L.gchunks = take((size_t)(chunks + 1) * 4);
        L.gtail = take(moe::wgrad_tail_bytes(chunks, 4 * c.n));
        // the chunk partials share gate_part's region, sized for the larger of the two
        const size_t need = (size_t)chunks * c.d * 4 * n * 4;
        const size_t have = (size_t)moe::gate_splitk(c.T) * c.d * n * 4;
        if (need > have) L.gate_part = take(need);
    }
    L.total = o;
    return L;
}

}  // namespace

extern "C" {

moe_status moe_backward_workspace_size(const moe_config* cfg, size_t* bytes) {
    MOE_TRY(check_config(cfg));
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *bytes = make_bwd_layout(*cfg).total;
    return MOE_OK;
}

}  // extern "C"

namespace {

// The backward; events (six, or null) are recorded before the recompute and after the
// recompute, the combine / gate backward, the expert data gradients (with dx's share),
// the expert weight gradients and the gate gradients.
moe_status backward_body(const moe_config* cfg, const void* x, const float* W_g,
                         const float* W_noise, const float* eps, const float* b_g,
                         const void* W_in, const void* W_out, const float* dy, float* dx,
                         float* dW_g, float* dW_noise, float* db_g, float* dW_in, float* dW_out,
                         void* workspace, size_t workspace_bytes, cudaStream_t stream,
                         cudaEvent_t* ev) {
    auto mark = [&](int i) -> moe_status {
        if (ev != nullptr && cudaEventRecord(ev[i], stream) != cudaSuccess) return MOE_ERR_CUDA;
        return MOE_OK;
    };
    MOE_TRY(check_config(cfg));
    if (!x || !W_g || !W_noise || !W_in || !W_out || !dy || !dx || !dW_g || !dW_noise || !dW_in ||
        !dW_out)
        return MOE_ERR_INVALID_ARG;
    if (cfg->capacity > 0 || (cfg->flags & MOE_FLAG_SWITCH_GATE)) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(W_g) || !aligned16(W_noise) || (eps && !aligned16(eps)) ||
        !aligned16(W_in) || !aligned16(W_out))
        return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_WORKSPACE;
    const moe_config& c = *cfg;
    const BwdLayout B = make_bwd_layout(c);
    if (workspace_bytes < B.total) return MOE_ERR_WORKSPACE;
    const Layout& L = B.F;
    void* ws = workspace;
    cudaStream_t s = stream;
    const long long R = (long long)c.T * c.k;
    const bool bf16 = c.x_dtype == MOE_BF16;
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    MOE_TRY(mark(0));
    MOE_TRY(draw_noise_into(c, eps, ws, s));
    float* clean = at<float>(ws, B.clean);
    float* stdv = at<float>(ws, B.stdv);
    float* H = at<float>(ws, B.H);
    int32_t* idx = at<int32_t>(ws, L.idx);
    float* gates = at<float>(ws, L.gates);
    float* thr = at<float>(ws, L.thr);
    float* load = at<float>(ws, L.load);
    float* importance = at<float>(ws, L.importance);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* perm = at<int32_t>(ws, L.perm);
    int32_t* inv = at<int32_t>(ws, L.inv);
    void* x_perm = at<void>(ws, L.x_perm);
    void* y_perm = at<void>(ws, L.y_perm);
    // ---- the forward pass again: logits to memory, selection, Load / Importance,
    //      dispatch and the experts (the hidden layer recomputed)
    if (bf16)
        MOE_CUDA(moe::launch_gate_logits_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.std_floor,
                                            at<void>(ws, L.w3), clean, stdv, H, err, s));
    else
        MOE_CUDA(moe::launch_gate_logits(x, false, W_g, W_noise, eps, b_g, c.T, c.d, c.n,
                                         c.std_floor, clean, stdv, H, s));
    MOE_CUDA(moe::launch_gate_select(H, c.T, c.n, c.k, idx, gates, nullptr, thr, s, false,
                                     at<int32_t>(ws, B.next_idx)));
    MOE_CUDA(moe::launch_gate_load(clean, stdv, idx, gates, thr, c.T, c.n, c.k,
                                   at<float>(ws, L.load_part), load, at<float>(ws, L.imp_part),
                                   importance, s));
    MOE_TRY(dispatch_body(c, idx, x, offsets, perm, inv, x_perm, ws, s));
    MOE_TRY(ffn_body(c, x_perm, offsets, W_in, W_out, y_perm, ws, s));
    MOE_TRY(mark(1));
    // ---- gradients
    float* dG = at<float>(ws, B.dG);
    float* dE = at<float>(ws, B.dE);     // bf16 / bf16 / fp16 on the tensor-core path
    float* dU = at<float>(ws, B.dU);
    float* dXp = at<float>(ws, B.dXp);
    float* dclean = at<float>(ws, B.dclean);
    float* dnz = at<float>(ws, B.dnz);
    MOE_CUDA(moe::launch_cv2_grad(importance, load, c.n, c.w_importance, c.w_load,
                                  at<float>(ws, B.g_imp), at<float>(ws, B.g_load), s));
    // bf16 experts with d, h multiples of 256: the data gradients on the tensor cores (the
    // forward's pair kernel, B read K-contiguous), with dE and dU in bf16 and dX in fp16
    const bool tc_grads = c.expert_dtype == MOE_BF16 && moe::ffn_pair_supported(c.d, c.h);
    MOE_CUDA(moe::launch_combine_backward(dy, y_perm, c.expert_dtype == MOE_BF16, inv, gates, c.T,
                                          c.k, c.d, dG, dE, tc_grads, s));
    MOE_CUDA(moe::launch_gate_backward(clean, stdv, eps, idx, gates, dG, thr,
                                       at<int32_t>(ws, B.next_idx), at<float>(ws, B.g_imp),
                                       at<float>(ws, B.g_load), c.T, c.n, c.k, c.std_floor, dclean,
                                       dnz, gate_grads_on_pairs(c) ? at<void>(ws, B.gsplit) : nullptr,
                                       s));
    MOE_TRY(mark(2));
    const void* hidden = at<void>(ws, L.hidden);
    if (tc_grads) {
        MOE_CUDA(moe::launch_ffn_pair_dgrad(dE, offsets, W_in, W_out, hidden, dU, dXp,
                                            at<int32_t>(ws, L.mt_prefix), at<void>(ws, L.units),
                                            R, c.d, c.h, c.n, err, s));
    } else {
        MOE_CUDA(moe::launch_row_block_prefix(offsets, c.n, moe::backward_row_block(),
                                              at<int32_t>(ws, B.blk), s, at<void>(ws, B.units)));
        MOE_CUDA(moe::launch_expert_dgrad(dE, W_in, W_out, hidden, c.expert_dtype == MOE_BF16,
                                          at<void>(ws, B.units), at<int32_t>(ws, B.blk), R, c.d,
                                          c.h, c.n, dU, dXp, s));
    }
    MOE_CUDA(moe::launch_gather_dx(dXp, tc_grads, inv, c.T, c.k, c.d, dx, s));
    MOE_TRY(mark(3));
    if (tc_grads) {     // weight gradients on SM pairs too
        MOE_CUDA(moe::launch_ffn_wgrad(hidden, dE, at<void>(ws, B.wg_tail), offsets, R, c.h, c.d,
                                       c.n, dW_out, err, s));
        MOE_CUDA(moe::launch_ffn_wgrad(x_perm, dU, at<void>(ws, B.wg_tail), offsets, R, c.d, c.h,
                                       c.n, dW_in, err, s));
    } else {
        MOE_CUDA(moe::launch_expert_wgrad(x_perm, hidden, c.expert_dtype == MOE_BF16, dE, dU,
                                          false, offsets, c.d, c.h, c.n, dW_in, dW_out, s));
    }
    MOE_TRY(mark(4));
    if (gate_grads_on_pairs(c)) {
        MOE_CUDA(moe::launch_gate_tc_weight_grads(x, at<void>(ws, B.gsplit), c.T, c.d, c.n,
                                                  at<int32_t>(ws, B.gchunks), at<void>(ws, B.gtail),
                                                  at<float>(ws, B.gate_part), dW_g, dW_noise, err,
                                                  s));
        // the gate's share of dx on the tensor cores, from the same split
        MOE_CUDA(moe::launch_gate_dx_tc(W_g, W_noise, at<void>(ws, B.gsplit), c.T, c.d, c.n,
                                        at<void>(ws, B.gdx_w2), dx, err, s));
    } else {
        MOE_CUDA(moe::launch_gate_weight_grads(x, bf16, W_g, W_noise, dclean, dnz, c.T, c.d, c.n,
                                               dW_g, dW_noise, dx, at<float>(ws, B.gate_part), s));
    }
    if (db_g != nullptr)
        MOE_CUDA(moe::launch_column_sum(dclean, c.T, c.n, db_g, at<float>(ws, B.colsum), s));
    MOE_TRY(mark(5));
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_backward(const moe_config* cfg, const void* x, const float* W_g,
                        const float* W_noise, const float* eps, const float* b_g,
                        const void* W_in, const void* W_out, const float* dy, float* dx,
                        float* dW_g, float* dW_noise, float* db_g, float* dW_in, float* dW_out,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    return backward_body(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, dy, dx, dW_g, dW_noise,
                         db_g, dW_in, dW_out, workspace, workspace_bytes, stream, nullptr);
}

moe_status moe_backward_timed(const moe_config* cfg, const void* x, const float* W_g,
                              const float* W_noise, const float* eps, const float* b_g,
                              const void* W_in, const void* W_out, const float* dy, float* dx,
                              float* dW_g, float* dW_noise, float* db_g, float* dW_in,
                              float* dW_out, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream, cudaEvent_t* stage_events) {
    if (stage_events == nullptr) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (stage_events[i] == nullptr) return MOE_ERR_INVALID_ARG;
    return backward_body(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, dy, dx, dW_g, dW_noise,
                         db_g, dW_in, dW_out, workspace, workspace_bytes, stream, stage_events);
}

}  // extern "C"

namespace {

// The batchwise gate's scratch: the forward's layout (x_perm, hidden, y_perm, the FFN's
// tables, W3), then the logits, their transpose, the selection and the gates.
struct BatchLayout {
    Layout F;
    size_t clean, stdv, H, Ht, rowmap, sel, gates_r, offsets, importance, load, counts;
    size_t total;
};

BatchLayout make_batch_layout(const moe_config& c) {
    BatchLayout L{};
    L.F = make_layout(c);
    const size_t T = c.T, n = c.n;
    const size_t m = (size_t)c.k * c.T / c.n;
    size_t o = L.F.total;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    L.clean = take(T * n * 4);
    L.stdv = take(T * n * 4);
    L.H = take(T * n * 4);
    L.Ht = take(T * n * 4);
    L.rowmap = take(T * n * 4);
    const size_t rows = std::max(n * m, (size_t)c.k * c.T);   // the inference mode's cap
    L.sel = take(rows * 4);
    L.gates_r = take(rows * 4);
    L.offsets = take((n + 1) * 4);
    L.importance = take(n * 4);
    L.load = take(n * 4);
    L.counts = take(n * 4);
    L.total = o;
    return L;
}

}  // namespace

extern "C" {

moe_status moe_batchwise_workspace_size(const moe_config* cfg, size_t* bytes) {
    MOE_TRY(check_config(cfg));
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *bytes = make_batch_layout(*cfg).total;
    return MOE_OK;
}

moe_status moe_batchwise_forward(const moe_config* cfg, const void* x, const float* W_g,
                                 const float* W_noise, const float* eps, const float* b_g,
                                 const void* W_in, const void* W_out, float* y, float* losses,
                                 int32_t* sel, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!x || !W_g || !W_noise || !W_in || !W_out || !y || !losses) return MOE_ERR_INVALID_ARG;
    if (cfg->capacity > 0 || (cfg->flags & (MOE_FLAG_SWITCH_GATE | MOE_FLAG_DEVICE_NOISE)))
        return MOE_ERR_UNSUPPORTED;
    const long long m = (long long)cfg->k * cfg->T / cfg->n;
    if (m < 1) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(W_g) || !aligned16(W_noise) || (eps && !aligned16(eps)) ||
        !aligned16(W_in) || !aligned16(W_out) || !aligned16(y))
        return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_WORKSPACE;
    const moe_config& c = *cfg;
    const BatchLayout B = make_batch_layout(c);
    if (workspace_bytes < B.total) return MOE_ERR_WORKSPACE;
    const Layout& L = B.F;
    void* ws = workspace;
    cudaStream_t s = stream;
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    float* H = at<float>(ws, B.H);
    if (c.x_dtype == MOE_BF16)
        MOE_CUDA(moe::launch_gate_logits_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.std_floor,
                                            at<void>(ws, L.w3), at<float>(ws, B.clean),
                                            at<float>(ws, B.stdv), H, err, s));
    else
        MOE_CUDA(moe::launch_gate_logits(x, false, W_g, W_noise, eps, b_g, c.T, c.d, c.n,
                                         c.std_floor, at<float>(ws, B.clean),
                                         at<float>(ws, B.stdv), H, s));
    int32_t* sel_ws = sel != nullptr ? sel : at<int32_t>(ws, B.sel);
    int32_t* rowmap = at<int32_t>(ws, B.rowmap);
    float* gates_r = at<float>(ws, B.gates_r);
    float* importance = at<float>(ws, B.importance);
    float* load = at<float>(ws, B.load);
    MOE_CUDA(moe::launch_batch_select(H, c.T, c.n, (int)m, at<float>(ws, B.Ht), sel_ws, rowmap,
                                      gates_r, importance, load, s));
    int32_t* offsets = at<int32_t>(ws, B.offsets);
    void* x_perm = at<void>(ws, L.x_perm);
    void* y_perm = at<void>(ws, L.y_perm);
    MOE_CUDA(moe::launch_batch_gather(x, (size_t)c.d * dtype_bytes(c.x_dtype), sel_ws, c.n,
                                      (int)m, x_perm, offsets, s));
    MOE_TRY(ffn_body(c, x_perm, offsets, W_in, W_out, y_perm, ws, s));
    MOE_CUDA(moe::launch_batch_combine(y_perm, c.expert_dtype == MOE_BF16, rowmap, gates_r, c.T,
                                       c.n, c.d, y, s));
    MOE_CUDA(moe::launch_cv2_losses(importance, load, c.n, c.w_importance, c.w_load, losses, s));
    return MOE_OK;
}

moe_status moe_batchwise_threshold_forward(const moe_config* cfg, const void* x,
                                           const float* W_g, const float* W_noise,
                                           const float* eps, const float* b_g,
                                           const float* threshold, const void* W_in,
                                           const void* W_out, float* y, float* losses,
                                           int32_t* counts, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_config(cfg));
    if (!x || !W_g || !W_noise || !threshold || !W_in || !W_out || !y || !losses)
        return MOE_ERR_INVALID_ARG;
    if (cfg->capacity > 0 || (cfg->flags & (MOE_FLAG_SWITCH_GATE | MOE_FLAG_DEVICE_NOISE)))
        return MOE_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(W_g) || !aligned16(W_noise) || (eps && !aligned16(eps)) ||
        !aligned16(W_in) || !aligned16(W_out) || !aligned16(y))
        return MOE_ERR_UNSUPPORTED;
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0)
        return MOE_ERR_WORKSPACE;
    const moe_config& c = *cfg;
    const BatchLayout B = make_batch_layout(c);
    if (workspace_bytes < B.total) return MOE_ERR_WORKSPACE;
    const Layout& L = B.F;
    void* ws = workspace;
    cudaStream_t s = stream;
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    float* H = at<float>(ws, B.H);
    if (c.x_dtype == MOE_BF16)
        MOE_CUDA(moe::launch_gate_logits_tc(x, W_g, W_noise, eps, b_g, c.T, c.d, c.n, c.std_floor,
                                            at<void>(ws, L.w3), at<float>(ws, B.clean),
                                            at<float>(ws, B.stdv), H, err, s));
    else
        MOE_CUDA(moe::launch_gate_logits(x, false, W_g, W_noise, eps, b_g, c.T, c.d, c.n,
                                         c.std_floor, at<float>(ws, B.clean),
                                         at<float>(ws, B.stdv), H, s));
    const long long cap = (long long)c.k * c.T;
    int32_t* sel = at<int32_t>(ws, B.sel);
    int32_t* rowmap = at<int32_t>(ws, B.rowmap);
    float* gates_r = at<float>(ws, B.gates_r);
    float* importance = at<float>(ws, B.importance);
    float* load = at<float>(ws, B.load);
    int32_t* offsets = at<int32_t>(ws, B.offsets);
    MOE_CUDA(moe::launch_threshold_select(H, c.T, c.n, threshold, cap, at<float>(ws, B.Ht),
                                          counts != nullptr ? counts : at<int32_t>(ws, B.counts),
                                          offsets, sel, rowmap, gates_r, importance, load, err,
                                          s));
    void* x_perm = at<void>(ws, L.x_perm);
    void* y_perm = at<void>(ws, L.y_perm);
    MOE_CUDA(moe::launch_batch_gather(x, (size_t)c.d * dtype_bytes(c.x_dtype), sel, c.n, 0,
                                      x_perm, offsets, s, cap));
    MOE_TRY(ffn_body(c, x_perm, offsets, W_in, W_out, y_perm, ws, s));
    MOE_CUDA(moe::launch_batch_combine(y_perm, c.expert_dtype == MOE_BF16, rowmap, gates_r, c.T,
                                       c.n, c.d, y, s));
    MOE_CUDA(moe::launch_cv2_losses(importance, load, c.n, c.w_importance, c.w_load, losses, s));
    return MOE_OK;
}

moe_status moe_hier_workspace_size(const moe_hier_config* cfg, size_t* bytes) {
    MOE_TRY(check_hier_config(cfg));
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *bytes = make_hier_layout(*cfg).total;
    return MOE_OK;
}

moe_status moe_hier_forward(const moe_hier_config* cfg, const void* x, const float* W_g1,
                            const float* W_noise1, const float* eps1, const float* W_g2,
                            const float* W_noise2, const float* eps2, const void* W_in,
                            const void* W_out, float* y, float* losses, int32_t* idx,
                            float* gates, uint8_t* tie1, uint8_t* tie2, float* importance1,
                            float* load1, float* importance, float* load2, void* workspace,
                            size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_hier_config(cfg));
    if (!x || !W_g1 || !W_noise1 || !eps1 || !W_g2 || !W_noise2 || !eps2 || !W_in || !W_out ||
        !y || !losses)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(W_g1) || !aligned16(W_noise1) || !aligned16(eps1) ||
        !aligned16(W_g2) || !aligned16(W_noise2) || !aligned16(eps2) || !aligned16(W_in) ||
        !aligned16(W_out) || !aligned16(y))
        return MOE_ERR_UNSUPPORTED;
    const moe_hier_config& c = *cfg;
    const HierLayout L = make_hier_layout(c);
    if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0 ||
        workspace_bytes < L.total)
        return MOE_ERR_WORKSPACE;
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    void* ws = workspace;
    cudaStream_t s = stream;
    const int K = c.k1 * c.k2, nb = c.a * c.b;
    const long long R1 = (long long)c.T * c.k1, R = (long long)c.T * K;
    if (!idx) idx = at<int32_t>(ws, L.idx);
    if (!gates) gates = at<float>(ws, L.gates);
    if (!tie1) tie1 = at<uint8_t>(ws, L.tie1);
    if (!tie2) tie2 = at<uint8_t>(ws, L.tie2);
    if (!importance1) importance1 = at<float>(ws, L.importance1);
    if (!load1) load1 = at<float>(ws, L.load1);
    if (!importance) importance = at<float>(ws, L.importance);
    if (!load2) load2 = at<float>(ws, L.load2);
    int32_t* idx1 = at<int32_t>(ws, L.idx1);
    float* gates1 = at<float>(ws, L.gates1);
    int32_t* offsets1 = at<int32_t>(ws, L.offsets1);
    int32_t* perm1 = at<int32_t>(ws, L.perm1);
    int32_t* blk1 = at<int32_t>(ws, L.blk1);
    void* x1_perm = at<void>(ws, L.x1_perm);
    int32_t* offsets = at<int32_t>(ws, L.offsets);
    int32_t* perm = at<int32_t>(ws, L.perm);
    int32_t* inv = at<int32_t>(ws, L.inv);
    void* x_perm = at<void>(ws, L.x_perm);
    void* y_perm = at<void>(ws, L.y_perm);
    // primary gate over the a groups (Importance and Load over groups in the same pass)
    MOE_CUDA(moe::launch_gate_fused_tc(x, W_g1, W_noise1, eps1, nullptr, c.T, c.d, c.a, c.k1,
                                       c.std_floor, at<void>(ws, L.w3_1), idx1, gates1, tie1,
                                       at<float>(ws, L.load_part1), at<float>(ws, L.imp_part1),
                                       load1, importance1, err, s));
    // group the routed rows (t, s) by group and copy their inputs
    MOE_CUDA(moe::launch_dispatch(idx1, c.T, c.k1, c.a, at<int32_t>(ws, L.tile_counts1),
                                  offsets1, perm1, at<int32_t>(ws, L.inv1), err, s, x,
                                  (size_t)c.d * 2, x1_perm));
    MOE_CUDA(moe::launch_row_block_prefix(offsets1, c.a, 128, blk1, s));
    // secondary gates, one per group, on that group's rows: flat ids and product gates
    MOE_CUDA(moe::launch_gate_grouped_tc(x1_perm, R1, offsets1, blk1, perm1, c.a, W_g2, W_noise2,
                                         eps2, gates1, c.d, c.b, c.k2, c.std_floor,
                                         at<void>(ws, L.w3_2), idx, gates, tie2,
                                         at<float>(ws, L.load_part2), at<float>(ws, L.imp_part2),
                                         load2, importance, err, s));
    // the flat layer over a*b experts with k1*k2 kept per token
    MOE_CUDA(moe::launch_dispatch(idx, c.T, K, nb, at<int32_t>(ws, L.tile_counts), offsets, perm,
                                  inv, err, s, x, (size_t)c.d * 2, x_perm));
    if (moe::ffn_pair_supported(c.d, c.h) && ffn_row_tiles(c.flags, R, nb))
        MOE_CUDA(moe::launch_ffn_pair(x_perm, offsets, W_in, W_out, y_perm, at<void>(ws, L.hidden),
                                      at<int32_t>(ws, L.mt_prefix), at<void>(ws, L.units), R,
                                      c.d, c.h, nb, err, s));
    else if (moe::ffn_pair_supported(c.d, c.h))
        MOE_CUDA(moe::launch_ffn_swap(x_perm, offsets, W_in, W_out, y_perm, at<void>(ws, L.hidden),
                                      at<int32_t>(ws, L.mt_prefix), at<void>(ws, L.units), R,
                                      c.d, c.h, nb, err, s));
    else
        MOE_CUDA(moe::launch_ffn_fused(x_perm, offsets, W_in, W_out, y_perm,
                                       at<void>(ws, L.hidden), at<int32_t>(ws, L.mt_prefix),
                                       at<int32_t>(ws, L.ffn_done), R, c.d, c.h, nb, err, s));
    MOE_CUDA(moe::launch_combine(y_perm, true, inv, gates, c.T, K, c.d, y, s));
    MOE_CUDA(moe::launch_cv2_losses(importance1, load1, c.a, c.w_importance, c.w_load, losses, s));
    return MOE_OK;
}

moe_status moe_selftest_timeout(long long budget_cycles, cudaStream_t stream) {
    if (budget_cycles < 1 || budget_cycles > 1000000000LL) return MOE_ERR_INVALID_ARG;
    int* err = device_error_word();
    if (err == nullptr) return MOE_ERR_CUDA;
    MOE_CUDA(moe::launch_timeout_probe(budget_cycles, err, stream));
    return MOE_OK;
}

const char* moe_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda_error); }

unsigned long long moe_launch_counter(void) {
    return moe::g_launches.load(std::memory_order_relaxed);
}

moe_status moe_get_device_error(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    int code = 0;
    if (cudaMemcpyFromSymbol(&code, g_moe_error_word, sizeof(int)) != cudaSuccess)
        return MOE_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_moe_error_word, &zero, sizeof(int)) != cudaSuccess)
        return MOE_ERR_CUDA;
    switch (code) {
        case moe::DEV_OK: return MOE_OK;
        case moe::DEV_TIMEOUT: return MOE_ERR_TIMEOUT;
        case moe::DEV_BAD_INDEX: return MOE_ERR_INVALID_ARG;
        case moe::DEV_RANGE: return MOE_ERR_RANGE;
        default: return MOE_ERR_CUDA;
    }
}

}  // extern "C"
