"""Failure detection on the GPU without a fault: a pipeline wait that can never complete runs out
after its limit, the kernel reports the timeout through the device error flag and returns, and the
context stays usable for the next block."""
import numpy as np
import pytest
import torch

import mi_synth
from tests._gpu import require_gpu, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    mi = require_gpu()
    assert mi.device_error() == 0
    mi.selftest_wait_timeout(20000)  # 20 ms
    torch.cuda.synchronize()
    assert mi.device_error() == 0x300
    assert mi.device_error() == 0  # read-and-clear
    # the context still runs a block
    g = mi_synth.GEOMETRIES["tiny_8x8"]
    inp = mi_synth.block_inputs(g, 0)
    w = inp.weights
    blk = mi.Block(to_dev_bf16(w.w_qkv), to_dev_bf16(w.w_o), to_dev_bf16(w.w_gu), to_dev_bf16(w.w_d),
                   to_dev_bf16(w.q_norm_w), to_dev_bf16(w.k_norm_w), g.n_heads, g.eps)
    x = to_dev_bf16(inp.x)
    y = torch.empty_like(x)
    ws = torch.empty(blk.workspace_size(g.batch, g.seq), dtype=torch.uint8, device="cuda")
    blk.forward(mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w), x, y, to_dev_bf16(inp.mod),
                to_dev(inp.rope_cos), to_dev(inp.rope_sin), to_dev(inp.key_mask), ws)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    assert torch.isfinite(y.float()).all()


def test_selftest_argument_checks():
    mi = require_gpu()
    with pytest.raises(mi.MiError):
        mi.selftest_wait_timeout(0)
    with pytest.raises(mi.MiError):
        mi.selftest_wait_timeout(2_000_000)
