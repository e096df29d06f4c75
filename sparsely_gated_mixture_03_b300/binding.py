"""Thin Python binding of libmoe_b300.so (include/moe.h), via ctypes.

Argument marshalling only: every function takes torch tensors that already
live on the GPU (or None for optional arguments), checks their dtype, device,
contiguity and size, and passes raw device pointers and the CUDA stream to the
C entry point of the same name.  All computation happens in the library's CUDA
kernels; there is no fallback of any kind.  A missing library or a non-OK
status raises MoeError.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_b300.so")

MOE_F32, MOE_BF16 = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
          3: "MOE_ERR_WORKSPACE", 4: "MOE_ERR_CUDA", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_RANGE"}

# Every symbol include/moe.h declares, in declaration order.
EXPORTS = ["moe_status_string", "moe_workspace_size", "moe_gate", "moe_dispatch",
           "moe_dispatch_noalloc", "moe_expert_ffn", "moe_combine", "moe_balance_losses",
           "moe_losses_from_sums", "moe_ep_plan", "moe_ep_regroup",
           "moe_forward", "moe_backward_workspace_size", "moe_backward", "moe_backward_timed",
           "moe_batchwise_workspace_size", "moe_batchwise_forward",
           "moe_batchwise_threshold_forward",
           "moe_forward_timed", "moe_draw_noise",
           "moe_hier_workspace_size", "moe_hier_forward",
           "moe_get_device_error", "moe_selftest_timeout", "moe_last_cuda_error",
           "moe_launch_counter"]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("n", ctypes.c_int),
                ("h", ctypes.c_int), ("k", ctypes.c_int), ("x_dtype", ctypes.c_int),
                ("expert_dtype", ctypes.c_int), ("std_floor", ctypes.c_float),
                ("w_importance", ctypes.c_float), ("w_load", ctypes.c_float),
                ("flags", ctypes.c_uint), ("capacity", ctypes.c_int),
                ("noise_seed", ctypes.c_ulonglong)]


class MoeHierConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int), ("d", ctypes.c_int), ("a", ctypes.c_int),
                ("b", ctypes.c_int), ("h", ctypes.c_int), ("k1", ctypes.c_int),
                ("k2", ctypes.c_int), ("x_dtype", ctypes.c_int), ("expert_dtype", ctypes.c_int),
                ("std_floor", ctypes.c_float), ("w_importance", ctypes.c_float),
                ("w_load", ctypes.c_float), ("flags", ctypes.c_uint)]


def _dtype_code(dt):
    if dt == torch.float32:
        return MOE_F32
    if dt == torch.bfloat16:
        return MOE_BF16
    raise ValueError(f"unsupported dtype {dt}")


# moe_config.flags bits forcing the tile kind of the bf16 expert FFN: 256-row tiles
# (every expert's last tile padded to 256 rows) or tiles sized to each expert's rows.
# Neither: chosen by the average rows per expert.
FLAG_FFN_ROW_TILES = 1
FLAG_FFN_SIZED_TILES = 2
# moe_config.flags bit: the Switch gate (softmax over all n logits, a kept expert's
# gate is its probability; the single Switch balancing loss).
FLAG_SWITCH_GATE = 4
# moe_config.flags bit: the layer draws the gate's noise itself (eps = None) from
# cfg.noise_seed, with moe_draw_noise's generator.
FLAG_DEVICE_NOISE = 8


def make_hier_config(T, d, a, b, h, k1, k2, x_dtype=torch.bfloat16, expert_dtype=torch.bfloat16,
                     std_floor=0.0, w_importance=0.1, w_load=0.1, flags=0) -> MoeHierConfig:
    return MoeHierConfig(T, d, a, b, h, k1, k2, _dtype_code(x_dtype), _dtype_code(expert_dtype),
                         std_floor, w_importance, w_load, flags)


def make_config(T, d, n, h, k, x_dtype=torch.bfloat16, expert_dtype=torch.bfloat16,
                std_floor=0.0, w_importance=0.1, w_load=0.1, flags=0, capacity=0,
                noise_seed=0) -> MoeConfig:
    """capacity: 0, or the most routed rows one expert processes (the first in
    routed-row order; the rest add nothing to y).  noise_seed: the seed of the noise
    the layer draws with FLAG_DEVICE_NOISE."""
    return MoeConfig(T, d, n, h, k, _dtype_code(x_dtype), _dtype_code(expert_dtype), std_floor,
                     w_importance, w_load, flags, capacity, noise_seed)


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe_b300.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoeError(-1, f"{LIB_PATH} is missing; build it with "
                               "`python -m sparsely_gated_mixture_03_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, S, C = ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(MoeConfig)
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_gate.argtypes = [C] + [P] * 11 + [S, P]
        L.moe_dispatch.argtypes = [C] + [P] * 7 + [S, P]
        L.moe_dispatch_noalloc.argtypes = [C] + [P] * 7
        L.moe_expert_ffn.argtypes = [C] + [P] * 6 + [S, P]
        L.moe_combine.argtypes = [C] + [P] * 5
        L.moe_balance_losses.argtypes = [C] + [P] * 7
        L.moe_losses_from_sums.argtypes = [C] + [P] * 4
        I = ctypes.c_int
        L.moe_ep_plan.argtypes = [I, I, I] + [P] * 4
        L.moe_ep_regroup.argtypes = [I, I, P, P, P, S, I, P]
        L.moe_forward.argtypes = [C] + [P] * 15 + [S, P]
        L.moe_forward_timed.argtypes = [C] + [P] * 15 + [S, P, P]
        L.moe_backward_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_backward.argtypes = [C] + [P] * 15 + [S, P]
        L.moe_backward_timed.argtypes = [C] + [P] * 15 + [S, P, P]
        L.moe_batchwise_workspace_size.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_batchwise_forward.argtypes = [C] + [P] * 11 + [S, P]
        L.moe_batchwise_threshold_forward.argtypes = [C] + [P] * 12 + [S, P]
        HC = ctypes.POINTER(MoeHierConfig)
        L.moe_hier_workspace_size.argtypes = [HC, ctypes.POINTER(ctypes.c_size_t)]
        L.moe_hier_forward.argtypes = [HC] + [P] * 20 + [S, P]
        L.moe_draw_noise.argtypes = [ctypes.c_ulonglong, ctypes.c_longlong, P, P]
        L.moe_get_device_error.argtypes = [P]
        L.moe_selftest_timeout.argtypes = [ctypes.c_longlong, P]
        for name in EXPORTS[1:-2]:
            getattr(L, name).restype = ctypes.c_int
        L.moe_last_cuda_error.restype = ctypes.c_char_p
        L.moe_last_cuda_error.argtypes = []
        L.moe_launch_counter.restype = ctypes.c_ulonglong
        L.moe_launch_counter.argtypes = []
        _lib = L
    return _lib


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, numel=None, required=True):
    if t is None:
        if required:
            raise ValueError(f"{name} is required")
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return t.data_ptr()


def _check(status: int, where: str):
    if status == 4:      # MOE_ERR_CUDA: name the CUDA error behind it
        raise MoeError(status, f"{where} ({lib().moe_last_cuda_error().decode()})")
    if status != 0:
        raise MoeError(status, where)


def _xdt(cfg):
    return torch.bfloat16 if cfg.x_dtype == MOE_BF16 else torch.float32


def _edt(cfg):
    return torch.bfloat16 if cfg.expert_dtype == MOE_BF16 else torch.float32


def expert_rows_dtype(cfg):
    """dtype of y_perm, the expert outputs: fp16 for bf16 experts, else fp32."""
    return torch.float16 if cfg.expert_dtype == MOE_BF16 else torch.float32


def workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def alloc_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    return torch.empty(max(workspace_size(cfg), 256), dtype=torch.uint8, device=device)


def backward_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return n.value


def alloc_backward_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    return torch.empty(max(backward_workspace_size(cfg), 256), dtype=torch.uint8, device=device)


def moe_backward(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, dy, dx, dW_g, dW_noise, db_g,
                 dW_in, dW_out, workspace, stream=None):
    """Gradients of sum(dy * y) + the balancing losses (include/moe.h, moe_backward)."""
    T, d, n, h = cfg.T, cfg.d, cfg.n, cfg.h
    f, e = torch.float32, _edt(cfg)
    st = lib().moe_backward(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(W_in, "W_in", e, n * d * h),
        _ptr(W_out, "W_out", e, n * h * d), _ptr(dy, "dy", f, T * d), _ptr(dx, "dx", f, T * d),
        _ptr(dW_g, "dW_g", f, d * n), _ptr(dW_noise, "dW_noise", f, d * n),
        _ptr(db_g, "db_g", f, n, required=False), _ptr(dW_in, "dW_in", f, n * d * h),
        _ptr(dW_out, "dW_out", f, n * h * d), _ptr(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream))
    _check(st, "moe_backward")


def moe_backward_timed(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, dy, dx, dW_g, dW_noise,
                       db_g, dW_in, dW_out, workspace, events, stream=None):
    """moe_backward recording six torch.cuda.Event(enable_timing=True) at its stage
    boundaries (include/moe.h, moe_backward_timed)."""
    T, d, n, h = cfg.T, cfg.d, cfg.n, cfg.h
    f, e = torch.float32, _edt(cfg)
    if len(events) != 6:
        raise ValueError("moe_backward_timed takes six events")
    st_ = stream if stream is not None else torch.cuda.current_stream()
    for ev in events:
        if not ev.cuda_event:
            ev.record(st_)
    arr = (ctypes.c_void_p * 6)(*[ctypes.c_void_p(ev.cuda_event) for ev in events])
    st = lib().moe_backward_timed(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(W_in, "W_in", e, n * d * h),
        _ptr(W_out, "W_out", e, n * h * d), _ptr(dy, "dy", f, T * d), _ptr(dx, "dx", f, T * d),
        _ptr(dW_g, "dW_g", f, d * n), _ptr(dW_noise, "dW_noise", f, d * n),
        _ptr(db_g, "db_g", f, n, required=False), _ptr(dW_in, "dW_in", f, n * d * h),
        _ptr(dW_out, "dW_out", f, n * h * d), _ptr(workspace, "workspace", torch.uint8),
        workspace.numel(), _stream(stream), arr)
    _check(st, "moe_backward_timed")


def batchwise_workspace_size(cfg: MoeConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_batchwise_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_batchwise_workspace_size")
    return n.value


def alloc_batchwise_workspace(cfg: MoeConfig, device="cuda") -> torch.Tensor:
    return torch.empty(max(batchwise_workspace_size(cfg), 256), dtype=torch.uint8, device=device)


def moe_batchwise_forward(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, y, losses, sel=None,
                          workspace=None, stream=None):
    """The layer with the batchwise top-m gate (include/moe.h, moe_batchwise_forward);
    sel, if given, receives [n, m] int32, m = k T // n."""
    T, d, n, h, k = cfg.T, cfg.d, cfg.n, cfg.h, cfg.k
    f, e = torch.float32, _edt(cfg)
    if workspace is None:
        workspace = alloc_batchwise_workspace(cfg, device=x.device)
    st = lib().moe_batchwise_forward(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(W_in, "W_in", e, n * d * h),
        _ptr(W_out, "W_out", e, n * h * d), _ptr(y, "y", f, T * d), _ptr(losses, "losses", f, 3),
        _ptr(sel, "sel", torch.int32, n * (k * T // n), required=False),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_batchwise_forward")


def moe_batchwise_threshold_forward(cfg, x, W_g, W_noise, eps, b_g, threshold, W_in, W_out, y,
                                    losses, counts=None, workspace=None, stream=None):
    """The batchwise gate at inference (include/moe.h): expert i takes the tokens whose
    noisy logit exceeds threshold[i]; counts, if given, receives [n] int32."""
    T, d, n, h = cfg.T, cfg.d, cfg.n, cfg.h
    f, e = torch.float32, _edt(cfg)
    if workspace is None:
        workspace = alloc_batchwise_workspace(cfg, device=x.device)
    st = lib().moe_batchwise_threshold_forward(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(threshold, "threshold", f, n),
        _ptr(W_in, "W_in", e, n * d * h), _ptr(W_out, "W_out", e, n * h * d),
        _ptr(y, "y", f, T * d), _ptr(losses, "losses", f, 3),
        _ptr(counts, "counts", torch.int32, n, required=False),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_batchwise_threshold_forward")


def moe_gate(cfg, x, W_g, W_noise, eps, b_g, idx, gates, tie, load, logits, workspace,
             stream=None):
    T, d, n, k = cfg.T, cfg.d, cfg.n, cfg.k
    f = torch.float32
    st = lib().moe_gate(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(idx, "idx", torch.int32, T * k),
        _ptr(gates, "gates", f, T * k), _ptr(tie, "tie", torch.uint8, T, required=False),
        _ptr(load, "load", f, n), _ptr(logits, "logits", f, 3 * T * n, required=False),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_gate")


def moe_dispatch(cfg, idx, x, offsets, perm, inv, x_perm, workspace, stream=None):
    T, d, n, k = cfg.T, cfg.d, cfg.n, cfg.k
    i32 = torch.int32
    st = lib().moe_dispatch(
        ctypes.byref(cfg), _ptr(idx, "idx", i32, T * k), _ptr(x, "x", _xdt(cfg), T * d),
        _ptr(offsets, "offsets", i32, n + 1), _ptr(perm, "perm", i32, T * k),
        _ptr(inv, "inv", i32, T * k), _ptr(x_perm, "x_perm", _xdt(cfg), T * k * d),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_dispatch")


def moe_dispatch_noalloc(cfg, idx, x, offsets, perm, inv, x_perm, stream=None):
    """moe_dispatch without a workspace, for callers that may not allocate
    device memory (see include/moe.h): the counting sort's scratch is the
    library's own 1 MiB device array, shared by every call on the device."""
    T, d, n, k = cfg.T, cfg.d, cfg.n, cfg.k
    i32 = torch.int32
    st = lib().moe_dispatch_noalloc(
        ctypes.byref(cfg), _ptr(idx, "idx", i32, T * k), _ptr(x, "x", _xdt(cfg), T * d),
        _ptr(offsets, "offsets", i32, n + 1), _ptr(perm, "perm", i32, T * k),
        _ptr(inv, "inv", i32, T * k), _ptr(x_perm, "x_perm", _xdt(cfg), T * k * d),
        _stream(stream))
    _check(st, "moe_dispatch_noalloc")


def moe_expert_ffn(cfg, x_perm, offsets, W_in, W_out, y_perm, workspace, stream=None):
    T, d, n, h, k = cfg.T, cfg.d, cfg.n, cfg.h, cfg.k
    e = _edt(cfg)
    st = lib().moe_expert_ffn(
        ctypes.byref(cfg), _ptr(x_perm, "x_perm", _xdt(cfg), T * k * d),
        _ptr(offsets, "offsets", torch.int32, n + 1), _ptr(W_in, "W_in", e, n * d * h),
        _ptr(W_out, "W_out", e, n * h * d),
        _ptr(y_perm, "y_perm", expert_rows_dtype(cfg), T * k * d),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_expert_ffn")


def moe_combine(cfg, y_perm, inv, gates, y, stream=None):
    T, d, k = cfg.T, cfg.d, cfg.k
    st = lib().moe_combine(
        ctypes.byref(cfg), _ptr(y_perm, "y_perm", expert_rows_dtype(cfg), T * k * d),
        _ptr(inv, "inv", torch.int32, T * k), _ptr(gates, "gates", torch.float32, T * k),
        _ptr(y, "y", torch.float32, T * d), _stream(stream))
    _check(st, "moe_combine")


def moe_balance_losses(cfg, gates, perm, offsets, load, importance, losses, stream=None):
    T, n, k = cfg.T, cfg.n, cfg.k
    f = torch.float32
    st = lib().moe_balance_losses(
        ctypes.byref(cfg), _ptr(gates, "gates", f, T * k), _ptr(perm, "perm", torch.int32, T * k),
        _ptr(offsets, "offsets", torch.int32, n + 1), _ptr(load, "load", f, n),
        _ptr(importance, "importance", f, n), _ptr(losses, "losses", f, 3), _stream(stream))
    _check(st, "moe_balance_losses")


def moe_draw_noise(seed, eps, stream=None):
    """eps (fp32 CUDA tensor, any shape): the layer's noise draws for seed, element i of
    the flattened tensor being draw i (FLAG_DEVICE_NOISE's eps[t, e] is draw t*n + e)."""
    count = eps.numel()
    _check(lib().moe_draw_noise(int(seed), count, _ptr(eps, "eps", torch.float32, count),
                                _stream(stream)), "moe_draw_noise")


def moe_losses_from_sums(cfg, importance, load, losses, stream=None):
    """The balancing losses from whole-batch Importance / Load sums (e.g. every
    data-parallel rank's vectors after an all-reduce); cfg.T = the whole batch's
    tokens."""
    n, f = cfg.n, torch.float32
    st = lib().moe_losses_from_sums(
        ctypes.byref(cfg), _ptr(importance, "importance", f, n), _ptr(load, "load", f, n),
        _ptr(losses, "losses", f, 3), _stream(stream))
    _check(st, "moe_losses_from_sums")


def ep_plan_size(world: int, n_local: int) -> int:
    """int32 entries of moe_ep_plan's plan array."""
    return 2 * world * n_local + n_local + 2


def moe_ep_plan(world: int, rank: int, n: int, all_offsets):
    """Host-only exchange plan of `rank` (include/moe.h).  all_offsets: host
    int32 array-like [world, n+1] (every rank's moe_dispatch offsets).  Returns
    numpy int32 arrays (send_rows [world], recv_rows [world], plan)."""
    import numpy as np
    offs = np.ascontiguousarray(np.asarray(all_offsets, dtype=np.int32).reshape(world, n + 1))
    n_local = n // world if world > 0 else 0
    send = np.zeros(max(world, 1), dtype=np.int32)
    recv = np.zeros(max(world, 1), dtype=np.int32)
    plan = np.zeros(max(ep_plan_size(world, n_local), 1), dtype=np.int32)
    st = lib().moe_ep_plan(world, rank, n, offs.ctypes.data, send.ctypes.data, recv.ctypes.data,
                           plan.ctypes.data)
    _check(st, "moe_ep_plan")
    return send, recv, plan


def moe_ep_regroup(world, n_local, plan, inp, out, to_expert_major, stream=None):
    """Rows between arrival order and expert-major order (plan on the device)."""
    rows = inp.shape[0]
    row_bytes = inp[0].numel() * inp.element_size() if rows else 16
    if out.shape != inp.shape or out.dtype != inp.dtype:
        raise ValueError("out must match in")
    st = lib().moe_ep_regroup(
        world, n_local, _ptr(plan, "plan", torch.int32, ep_plan_size(world, n_local)),
        _ptr(inp, "in"), _ptr(out, "out"), row_bytes, 1 if to_expert_major else 0,
        _stream(stream))
    _check(st, "moe_ep_regroup")


def moe_forward(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, y, losses, idx=None, gates=None,
                tie=None, importance=None, load=None, workspace=None, stream=None):
    T, d, n, h, k = cfg.T, cfg.d, cfg.n, cfg.h, cfg.k
    f, e = torch.float32, _edt(cfg)
    st = lib().moe_forward(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(W_in, "W_in", e, n * d * h),
        _ptr(W_out, "W_out", e, n * h * d), _ptr(y, "y", f, T * d), _ptr(losses, "losses", f, 3),
        _ptr(idx, "idx", torch.int32, T * k, required=False),
        _ptr(gates, "gates", f, T * k, required=False),
        _ptr(tie, "tie", torch.uint8, T, required=False),
        _ptr(importance, "importance", f, n, required=False),
        _ptr(load, "load", f, n, required=False),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_forward")


def hier_workspace_size(cfg: MoeHierConfig) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_hier_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_hier_workspace_size")
    return n.value


def alloc_hier_workspace(cfg: MoeHierConfig, device="cuda") -> torch.Tensor:
    return torch.empty(max(hier_workspace_size(cfg), 256), dtype=torch.uint8, device=device)


def moe_hier_forward(cfg, x, W_g1, W_noise1, eps1, W_g2, W_noise2, eps2, W_in, W_out, y, losses,
                     idx=None, gates=None, tie1=None, tie2=None, importance1=None, load1=None,
                     importance=None, load2=None, workspace=None, stream=None):
    T, d, a, b, h, k1, k2 = cfg.T, cfg.d, cfg.a, cfg.b, cfg.h, cfg.k1, cfg.k2
    f, bf, K, nb = torch.float32, torch.bfloat16, k1 * k2, a * b
    st = lib().moe_hier_forward(
        ctypes.byref(cfg), _ptr(x, "x", bf, T * d), _ptr(W_g1, "W_g1", f, d * a),
        _ptr(W_noise1, "W_noise1", f, d * a), _ptr(eps1, "eps1", f, T * a),
        _ptr(W_g2, "W_g2", f, a * d * b), _ptr(W_noise2, "W_noise2", f, a * d * b),
        _ptr(eps2, "eps2", f, T * k1 * b), _ptr(W_in, "W_in", bf, nb * d * h),
        _ptr(W_out, "W_out", bf, nb * h * d), _ptr(y, "y", f, T * d),
        _ptr(losses, "losses", f, 3),
        _ptr(idx, "idx", torch.int32, T * K, required=False),
        _ptr(gates, "gates", f, T * K, required=False),
        _ptr(tie1, "tie1", torch.uint8, T, required=False),
        _ptr(tie2, "tie2", torch.uint8, T * k1, required=False),
        _ptr(importance1, "importance1", f, a, required=False),
        _ptr(load1, "load1", f, a, required=False),
        _ptr(importance, "importance", f, nb, required=False),
        _ptr(load2, "load2", f, nb, required=False),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    _check(st, "moe_hier_forward")


def moe_forward_timed(cfg, x, W_g, W_noise, eps, b_g, W_in, W_out, y, losses, events, idx=None,
                      gates=None, tie=None, importance=None, load=None, workspace=None,
                      stream=None):
    """moe_forward recording six torch.cuda.Event objects (created with
    enable_timing=True) at its stage boundaries on the stream."""
    if len(events) != 6:
        raise ValueError("moe_forward_timed takes 6 events")
    for ev in events:           # torch creates an event's CUDA handle at its first record
        if not ev.cuda_event:
            ev.record(torch.cuda.current_stream() if stream is None else stream)
    T, d, n, h, k = cfg.T, cfg.d, cfg.n, cfg.h, cfg.k
    f, e = torch.float32, _edt(cfg)
    ev = (ctypes.c_void_p * 6)(*[int(x.cuda_event) for x in events])
    st = lib().moe_forward_timed(
        ctypes.byref(cfg), _ptr(x, "x", _xdt(cfg), T * d), _ptr(W_g, "W_g", f, d * n),
        _ptr(W_noise, "W_noise", f, d * n), _ptr(eps, "eps", f, T * n, required=False),
        _ptr(b_g, "b_g", f, n, required=False), _ptr(W_in, "W_in", e, n * d * h),
        _ptr(W_out, "W_out", e, n * h * d), _ptr(y, "y", f, T * d), _ptr(losses, "losses", f, 3),
        _ptr(idx, "idx", torch.int32, T * k, required=False),
        _ptr(gates, "gates", f, T * k, required=False),
        _ptr(tie, "tie", torch.uint8, T, required=False),
        _ptr(importance, "importance", f, n, required=False),
        _ptr(load, "load", f, n, required=False),
        _ptr(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream),
        ctypes.cast(ev, ctypes.c_void_p))
    _check(st, "moe_forward_timed")


def moe_launch_counter() -> int:
    """Kernels the library has enqueued in this process so far."""
    return int(lib().moe_launch_counter())


def moe_selftest_timeout(budget_cycles: int, stream=None):
    """Enqueue the failure-detection self-test (a CTA whose bounded waits run out)."""
    _check(lib().moe_selftest_timeout(int(budget_cycles), _stream(stream)), "moe_selftest_timeout")


def moe_get_device_error(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device error status."""
    return lib().moe_get_device_error(_stream(stream))
