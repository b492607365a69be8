"""mi_block_forward_static_ws: the block forward for callers that cannot allocate device memory
(its workspace is a static device array inside the library).  Called through the C ABI and
checked against mi_block_forward with a caller workspace, byte for byte, on two calls in a row
with different inputs (the static array keeps the previous call's contents), and against the
float64 oracle.  This file sorts last so that a run stopping at the first failure has already
run every other test."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import mi_synth
from oracle import mi_oracle as O
from tests._gpu import assert_parity, require_gpu, to_dev, to_dev_bf16, to_f64

pytestmark = pytest.mark.gpu

# The size of the static workspace, MI_STATIC_WS_BYTES in include/mi_block.h.
STATIC_WS_BYTES = 64 << 20

# A batch-2 geometry whose down projection (K = 8448, 132 k-blocks over one 256-column tile per
# 128-row block) takes the GEMM's stream-K tail: its k-blocks are split over two CTAs per tile,
# whose fp32 partial sums and arrival counters live in the workspace.  The counters must start at
# zero on every call, which is what a second call through the shared static array checks.
STREAM_K_GEOM = mi_synth.GEOMETRIES["small_cfg_b2_streamk"]


def _ptr(t):
    return None if t is None else t.data_ptr()


def _inputs(g, seed):
    inp = mi_synth.block_inputs(g, seed)
    return inp, dict(x=to_dev_bf16(inp.x), mod=to_dev_bf16(inp.mod), cos=to_dev(inp.rope_cos),
                     sin=to_dev(inp.rope_sin), mask=to_dev(inp.key_mask))


def _tensor_bytes(mi, blk, g):
    """End of the last intermediate tensor inside the workspace (the rest is GEMM scratch)."""
    end = 0
    for which in mi.TENSORS.values():
        off, nbytes = ctypes.c_size_t(), ctypes.c_size_t()
        st = mi.lib().mi_block_tensor_offset(blk.handle, g.batch, g.seq, which, ctypes.byref(off),
                                             ctypes.byref(nbytes))
        if st == 0:
            end = max(end, off.value + nbytes.value)
    return end


@pytest.mark.parametrize("geom", [mi_synth.GEOMETRIES["small_cfg_b2"], STREAM_K_GEOM], ids=lambda g: g.name)
def test_static_workspace_forward_matches_caller_workspace(geom):
    mi = require_gpu()
    lib = mi.lib()
    g = geom
    first_np, first = _inputs(g, 11)
    w = first_np.weights
    blk = mi.Block(to_dev_bf16(w.w_qkv), to_dev_bf16(w.w_o), to_dev_bf16(w.w_gu), to_dev_bf16(w.w_d),
                   to_dev_bf16(w.q_norm_w), to_dev_bf16(w.k_norm_w), g.n_heads, g.eps)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    ws_bytes = blk.workspace_size(g.batch, g.seq)
    assert ws_bytes <= STATIC_WS_BYTES
    if g is STREAM_K_GEOM:
        # the plan reserves stream-K scratch (at least one 128 x 256 fp32 partial tile)
        assert ws_bytes - _tensor_bytes(mi, blk, g) >= 128 * 256 * 4
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for seed in (11, 12):  # two calls in a row, different activations and modulation
        inp, a = (first_np, first) if seed == 11 else _inputs(g, seed)
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
        # the same kernels on the same inputs: the same bytes
        assert torch.equal(y_static.view(torch.int16), y_ref.view(torch.int16)), \
            f"static-workspace forward differs from the caller-workspace forward (seed {seed})"
        # the block holds the first call's weights; the second call changes activations and modulation
        ref = O.block_forward_inputs(dataclasses.replace(inp, weights=w))["y"]
        assert_parity(to_f64(y_static), ref, f"static-workspace forward against the oracle, seed {seed}")


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
    assert blk.workspace_size(g.batch, g.seq) > STATIC_WS_BYTES
    st = lib.mi_block_forward_static_ws(blk.handle, ctypes.byref(layout), x.data_ptr(), x.data_ptr(),
                                        mod.data_ptr(), cos.data_ptr(), sin.data_ptr(), 0, None, None)
    assert st == 3 and b"static one holds" in lib.mi_last_error()
    torch.cuda.synchronize()
