"""The C-ABI library loads on a machine without a GPU, exports every symbol
include/moe.h declares, and rejects bad arguments on the host before any
CUDA call (these tests make no compute call)."""
import ctypes
import os
import re

import pytest

import sparsely_gated_mixture_03_b300 as moe
from sparsely_gated_mixture_03_b300 import binding
from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ["moe_gate", "moe_dispatch", "moe_expert_ffn", "moe_combine",
                 "moe_balance_losses", "moe_forward", "moe_workspace_size"]:
        assert name in syms
    assert sorted(binding.EXPORTS) == syms


def test_library_exports_every_declared_symbol():
    L = moe.lib()
    nm = os.popen(f"nm -D --defined-only {binding.LIB_PATH}").read()
    for name in declared_symbols():
        assert re.search(rf"\bT {name}\b", nm), f"{name} not exported"
        assert getattr(L, name) is not None


def test_flag_values_match_header():
    text = open(HEADER).read()
    for name, value in [("FFN_ROW_TILES", moe.FLAG_FFN_ROW_TILES),
                        ("FFN_SIZED_TILES", moe.FLAG_FFN_SIZED_TILES),
                        ("SWITCH_GATE", moe.FLAG_SWITCH_GATE),
                        ("DEVICE_NOISE", moe.FLAG_DEVICE_NOISE)]:
        m = re.search(rf"#define\s+MOE_FLAG_{name}\s+(\d+)u", text)
        assert m and int(m.group(1)) == value


def test_tile_flags_accepted():
    make = lambda f: binding.MoeConfig(64, 256, 8, 256, 2, 1, 1, 0.0, 0.1, 0.1, f)
    assert _ws(make(moe.FLAG_FFN_ROW_TILES))[0] == 0
    assert _ws(make(moe.FLAG_FFN_SIZED_TILES))[0] == 0
    assert _ws(make(moe.FLAG_FFN_ROW_TILES | moe.FLAG_FFN_SIZED_TILES))[0] == 1
    assert _ws(make(moe.FLAG_SWITCH_GATE | moe.FLAG_FFN_ROW_TILES))[0] == 0
    assert _ws(make(16))[0] == 1                      # a reserved bit
    # the drawn noise [T, n] fp32 lives in the workspace
    plain, drawn = _ws(make(0)), _ws(make(moe.FLAG_DEVICE_NOISE))
    assert plain[0] == 0 and drawn[0] == 0 and drawn[1] - plain[1] >= 64 * 8 * 4


def test_status_strings():
    L = moe.lib()
    for code in range(7):
        s = L.moe_status_string(code).decode()
        assert s.startswith(binding.STATUS[code])
    assert L.moe_status_string(99).decode() == "unknown moe_status"


def _ws(cfg):
    n = ctypes.c_size_t(0)
    st = moe.lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), 1), (dict(k=0), 1), (dict(k=9, n=9), 2), (dict(k=5, n=4), 1), (dict(d=100), 2),
    (dict(h=96), 2), (dict(n=16385), 2), (dict(x_dtype=0, expert_dtype=1), 2),
    (dict(std_floor=-1.0), 1), (dict(flags=16), 1), (dict(flags=8), 0), (dict(x_dtype=7), 1),
    (dict(capacity=-1), 1)])
def test_config_validation(kw, status):
    base = dict(T=64, d=64, n=8, h=64, k=2, x_dtype=1, expert_dtype=1, std_floor=0.0,
                w_importance=0.1, w_load=0.1, flags=0)
    base.update(kw)
    cfg = binding.MoeConfig(**base)
    assert _ws(cfg)[0] == status


def test_workspace_size_grows_with_the_batch():
    a = _ws(moe.make_config(1024, 512, 256, 1024, 4))
    b = _ws(moe.make_config(2048, 512, 256, 1024, 4))
    assert a[0] == 0 and b[0] == 0 and 0 < a[1] < b[1]
    assert a[1] % 256 == 0


def test_null_and_workspace_checks_before_any_cuda_call():
    L = moe.lib()
    cfg = moe.make_config(64, 64, 8, 64, 2)
    _, need = _ws(cfg)
    dummy = 256 * 1024                      # an aligned fake device address, never dereferenced
    p = ctypes.c_void_p
    # missing required pointer
    st = L.moe_gate(ctypes.byref(cfg), None, p(dummy), p(dummy), p(dummy), None, p(dummy), p(dummy),
                    None, p(dummy), None, p(dummy), need, None)
    assert st == 1
    # misaligned x
    st = L.moe_gate(ctypes.byref(cfg), p(dummy + 2), p(dummy), p(dummy), p(dummy), None, p(dummy),
                    p(dummy), None, p(dummy), None, p(dummy), need, None)
    assert st == 2
    # workspace too small, NULL, misaligned
    for ws, size in [(dummy, need - 1), (None, need), (dummy + 16, need)]:
        st = L.moe_gate(ctypes.byref(cfg), p(dummy), p(dummy), p(dummy), p(dummy), None, p(dummy),
                        p(dummy), None, p(dummy), None, p(ws) if ws else None, size, None)
        assert st == 3
    st = L.moe_forward(ctypes.byref(cfg), *([p(dummy)] * 4), None, p(dummy), p(dummy), None,
                       p(dummy), *([None] * 5), p(dummy), need, None)
    assert st == 1
    st = L.moe_combine(None, p(dummy), p(dummy), p(dummy), p(dummy), None)
    assert st == 1


def test_backward_and_batchwise_host_checks():
    """moe_backward and moe_batchwise_forward reject bad arguments on the host before
    any CUDA call, and their workspaces hold the forward's."""
    L = moe.lib()
    dummy = 256 * 1024                      # an aligned fake device address, never dereferenced
    p = ctypes.c_void_p
    cfg = moe.make_config(64, 64, 8, 64, 2)
    fwd = _ws(cfg)[1]
    nb, nw = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(nb)) == 0
    assert L.moe_batchwise_workspace_size(ctypes.byref(cfg), ctypes.byref(nw)) == 0
    assert nb.value > fwd and nw.value > fwd
    full = [p(dummy)] * 14                  # x .. dW_out, db_g included

    def bwd(c, ptrs, size):
        return L.moe_backward(ctypes.byref(c), *ptrs, p(dummy), size, None)
    assert bwd(cfg, [None] + full[1:], nb.value) == 1            # x missing
    assert bwd(cfg, full, nb.value - 1) == 3                     # workspace too small
    for c in (moe.make_config(64, 64, 8, 64, 2, capacity=4),
              moe.make_config(64, 64, 8, 64, 1, flags=moe.FLAG_SWITCH_GATE)):
        assert bwd(c, full, 1 << 40) == 2                        # capacity / Switch: unsupported

    def bw(c, ptrs, size):
        return L.moe_batchwise_forward(ctypes.byref(c), *ptrs, p(dummy), size, None)
    ten = [p(dummy)] * 10                   # x .. sel
    assert bw(cfg, ten[:7] + [None] + ten[8:], nw.value) == 1     # y missing
    assert bw(cfg, ten, nw.value - 1) == 3
    assert bw(moe.make_config(4, 64, 8, 64, 1), ten, 1 << 40) == 2   # k T / n < 1
    assert bw(moe.make_config(64, 64, 8, 64, 2, capacity=4), ten, 1 << 40) == 2


def test_binding_rejects_host_tensors():
    import torch
    cfg = moe.make_config(8, 64, 4, 64, 2, torch.float32, torch.float32)
    with pytest.raises(ValueError):
        moe.moe_combine(cfg, torch.zeros(16, 64), torch.zeros(16, dtype=torch.int32),
                        torch.zeros(8, 2), torch.zeros(8, 64))


def _hier_ws(cfg):
    n = ctypes.c_size_t(0)
    st = moe.lib().moe_hier_workspace_size(ctypes.byref(cfg), ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("kw,status", [
    (dict(T=0), 1), (dict(k1=0), 1), (dict(k2=0), 1), (dict(k1=5, a=4), 1), (dict(k2=3, b=2), 1),
    (dict(k1=3, k2=3), 2), (dict(a=257), 2), (dict(b=300), 2), (dict(a=200, b=100), 2),
    (dict(d=96), 2), (dict(h=32), 2), (dict(x_dtype=0, expert_dtype=0), 2),
    (dict(x_dtype=0), 2), (dict(std_floor=-0.5), 1), (dict(flags=3), 1), (dict(flags=4), 1),
    (dict(x_dtype=3), 1)])
def test_hier_config_validation(kw, status):
    base = dict(T=256, d=64, a=8, b=16, h=64, k1=2, k2=2, x_dtype=1, expert_dtype=1,
                std_floor=0.0, w_importance=0.1, w_load=0.1, flags=0)
    base.update(kw)
    assert _hier_ws(binding.MoeHierConfig(**base))[0] == status


def test_hier_workspace_and_null_checks_before_any_cuda_call():
    L = moe.lib()
    cfg = moe.make_hier_config(128, 64, 8, 16, 64, 2, 2)
    st, need = _hier_ws(cfg)
    assert st == 0 and need % 256 == 0
    big = _hier_ws(moe.make_hier_config(65536, 512, 128, 128, 1024, 2, 2))
    assert big[0] == 0 and big[1] > need
    dummy = 256 * 1024
    p = ctypes.c_void_p
    args = [p(dummy)] * 11 + [None] * 8
    # a missing required input, then a short, NULL and misaligned workspace
    bad = list(args)
    bad[3] = None                                   # eps1
    assert L.moe_hier_forward(ctypes.byref(cfg), *bad, p(dummy), need, None) == 1
    for ws, size in [(dummy, need - 1), (None, need), (dummy + 64, need)]:
        st = L.moe_hier_forward(ctypes.byref(cfg), *args, p(ws) if ws else None, size, None)
        assert st == 3
    mis = list(args)
    mis[0] = p(dummy + 4)                           # x not 16-byte aligned
    assert L.moe_hier_forward(ctypes.byref(cfg), *mis, p(dummy), need, None) == 2
