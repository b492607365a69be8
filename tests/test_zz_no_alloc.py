"""mi_block_forward_static_ws: the block forward for callers that cannot allocate device memory
(its workspace is a static device array inside the library).  Called through the C ABI and
checked against mi_block_forward with a caller workspace, on two calls in a row with different
inputs (the static array keeps the previous call's contents).  This file sorts last so that a run
stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import mi_synth
from tests._gpu import assert_parity, require_gpu, to_dev, to_dev_bf16, to_f64

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else t.data_ptr()


def _inputs(g, seed):
    inp = mi_synth.block_inputs(g, seed)
    return dict(x=to_dev_bf16(inp.x), mod=to_dev_bf16(inp.mod), cos=to_dev(inp.rope_cos), sin=to_dev(inp.rope_sin),
                mask=to_dev(inp.key_mask), weights=inp.weights)


def test_static_workspace_forward_matches_caller_workspace():
    mi = require_gpu()
    lib = mi.lib()
    g = mi_synth.GEOMETRIES["small_cfg_b2"]
    first = _inputs(g, 11)
    w = first["weights"]
    blk = mi.Block(to_dev_bf16(w.w_qkv), to_dev_bf16(w.w_o), to_dev_bf16(w.w_gu), to_dev_bf16(w.w_d),
                   to_dev_bf16(w.q_norm_w), to_dev_bf16(w.k_norm_w), g.n_heads, g.eps)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    ws = torch.empty(blk.workspace_size(g.batch, g.seq), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (11, 12):  # two calls in a row, different activations and modulation
        a = first if seed == 11 else _inputs(g, seed)
        y_ref = torch.empty_like(a["x"])
        y_static = torch.empty_like(a["x"])
        st = lib.mi_block_forward(blk.handle, ctypes.byref(layout), _ptr(a["x"]), _ptr(y_ref), _ptr(a["mod"]),
                                  _ptr(a["cos"]), _ptr(a["sin"]), 0, _ptr(a["mask"]), _ptr(ws),
                                  ws.numel(), stream)
        assert st == 0, lib.mi_last_error()
        st = lib.mi_block_forward_static_ws(blk.handle, ctypes.byref(layout), _ptr(a["x"]), _ptr(y_static),
                                            _ptr(a["mod"]), _ptr(a["cos"]), _ptr(a["sin"]), 0, _ptr(a["mask"]),
                                            stream)
        assert st == 0, lib.mi_last_error()
        torch.cuda.synchronize()
        assert mi.device_error() == 0
        assert_parity(to_f64(y_static), to_f64(y_ref), f"static-workspace forward, call with seed {seed}")


def test_static_workspace_refuses_a_geometry_that_does_not_fit():
    mi = require_gpu()
    lib = mi.lib()
    g = mi_synth.GEOMETRIES["block_1024"]  # needs about 300 MB of workspace
    H, I = g.hidden, g.mlp_inter
    inp = mi_synth.block_inputs(mi_synth.Geometry("zeros", 1, g.text_pad, g.n_text, g.grid_h, g.grid_w, 256, 2, 128), 0)
    x = torch.zeros(g.batch, g.seq, H, dtype=torch.bfloat16, device="cuda")
    mod = torch.zeros(g.batch, 6, H, dtype=torch.bfloat16, device="cuda")
    cos = to_dev(inp.rope_cos)
    sin = to_dev(inp.rope_sin)
    w_qkv = torch.zeros(3 * H, H, dtype=torch.bfloat16, device="cuda")
    w_o = torch.zeros(H, H, dtype=torch.bfloat16, device="cuda")
    w_gu = torch.zeros(2 * I, H, dtype=torch.bfloat16, device="cuda")
    w_d = torch.zeros(H, I, dtype=torch.bfloat16, device="cuda")
    gain = torch.ones(128, dtype=torch.bfloat16, device="cuda")
    blk = mi.Block(w_qkv, w_o, w_gu, w_d, gain, gain, g.n_heads, g.eps)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    assert blk.workspace_size(g.batch, g.seq) > mi.lib().mi_abi_version() * (64 << 20)
    st = lib.mi_block_forward_static_ws(blk.handle, ctypes.byref(layout), x.data_ptr(), x.data_ptr(),
                                        mod.data_ptr(), cos.data_ptr(), sin.data_ptr(), 0, None, None)
    assert st == 3 and b"static one holds" in lib.mi_last_error()
    torch.cuda.synchronize()
