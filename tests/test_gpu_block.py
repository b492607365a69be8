"""Whole-block parity through mi_block_forward against the float64 oracle, every intermediate
tensor, plus the invariants that must hold bit for bit on the GPU."""
import hashlib

import numpy as np
import pytest
import torch

import mi_synth
from oracle import mi_oracle as O
from tests._gpu import assert_parity, bf16_to_bits, require_gpu, to_dev, to_dev_bf16, to_f64

pytestmark = pytest.mark.gpu
BF = torch.bfloat16

_ORACLE_CACHE = {}


def oracle_block(name, seed=0):
    key = (name, seed)
    if key not in _ORACLE_CACHE:
        _ORACLE_CACHE[key] = O.block_forward_inputs(mi_synth.block_inputs(mi_synth.GEOMETRIES[name], seed))
    return _ORACLE_CACHE[key]


class GpuBlock:
    def __init__(self, mi, inp, fused=True):
        g = inp.geom
        w = inp.weights
        self.g = g
        self.w = [to_dev_bf16(a) for a in (w.w_qkv, w.w_o, w.w_gu, w.w_d, w.q_norm_w, w.k_norm_w)]
        self.blk = mi.Block(*self.w, n_heads=g.n_heads, eps=g.eps, fuse_epilogues=fused)
        self.layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
        self.x = to_dev_bf16(inp.x)
        self.mod = to_dev_bf16(inp.mod)
        self.cos = to_dev(inp.rope_cos)
        self.sin = to_dev(inp.rope_sin)
        self.mask = to_dev(inp.key_mask)
        self.ws = torch.empty(self.blk.workspace_size(g.batch, g.seq), dtype=torch.uint8, device="cuda")
        self.y = torch.empty_like(self.x)

    def run(self, x=None, y=None):
        self.blk.forward(self.layout, self.x if x is None else x, self.y if y is None else y, self.mod, self.cos,
                         self.sin, self.mask, self.ws)
        return self.y if y is None else y

    def tensor(self, name, shape):
        off, nb = self.blk.tensor_offset(self.g.batch, self.g.seq, name)
        return self.ws[off:off + nb].view(BF).view(*shape)


def _check_all(gb, ref, fused):
    g = gb.g
    B, S, H, I = g.batch, g.seq, g.hidden, g.mlp_inter
    names = [("h", (B, S, H)), ("qkv", (B, S, 3 * H)), ("qp", (B, g.n_heads, S, 128)),
             ("kp", (B, g.n_heads, S, 128)), ("o", (B, S, H)), ("x1", (B, S, H)), ("h2", (B, S, H)),
             ("m", (B, S, I))]
    if not fused:
        names += [("a", (B, S, H)), ("gu", (B, S, 2 * I)), ("dn", (B, S, H))]
    key = {"qp": "q", "kp": "k"}
    report = {}
    for n, shp in names:
        got = to_f64(gb.tensor(n, shp))
        want = ref[key.get(n, n)]
        if n == "qkv" and fused:  # the fused projection writes only the v columns
            got, want = got[..., 2 * H:], want[..., 2 * H:]
        report[n] = assert_parity(got, want, n)
    report["y"] = assert_parity(to_f64(gb.y), ref["y"], "y")
    return report


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "unfused"])
@pytest.mark.parametrize("name", ["tiny_8x8", "small_ragged_17x19", "small_cfg_b2"])
def test_block_parity_small(name, fused):
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES[name], 0)
    gb = GpuBlock(mi, inp, fused)
    gb.run()
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    _check_all(gb, oracle_block(name), fused)


def test_fused_and_unfused_blocks_give_identical_bytes():
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES["small_cfg_b2"], 3)
    a = GpuBlock(mi, inp, True)
    b = GpuBlock(mi, inp, False)
    assert torch.equal(a.run().view(torch.int16), b.run().view(torch.int16))


@pytest.mark.parametrize("name", ["block_1024", "block_1200x880"])
def test_block_parity_full_size(name):
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES[name], 0)
    gb = GpuBlock(mi, inp, True)
    gb.run()
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    _check_all(gb, oracle_block(name), True)


@pytest.mark.parametrize("name", ["small_cfg_b2_streamk", "block_1024_cfg_b2"])
def test_fused_and_unfused_give_identical_bytes_at_batch_2(name):
    # small_cfg_b2_streamk: the down projection (4 row tiles, 132 k-blocks) spreads its k-blocks
    # over twice as many CTAs in both paths (the stream-K tail), and the partial sums are added in a
    # fixed order; block_1024_cfg_b2: the guided step's block (8260 rows), every projection on the
    # CTA-pair kernel.  Either way the two paths agree exactly, and so do repeats.
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES[name], 3)
    a = GpuBlock(mi, inp, True)
    b = GpuBlock(mi, inp, False)
    ya = a.run().clone()
    assert torch.equal(ya.view(torch.int16), b.run().view(torch.int16))
    assert torch.equal(ya.view(torch.int16), a.run().view(torch.int16))
    assert mi.device_error() == 0


def test_block_repeats_bit_for_bit():
    # the same block twice, with another geometry run in between, gives identical bytes
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES["block_1024"], 1)
    other = GpuBlock(mi, mi_synth.block_inputs(mi_synth.GEOMETRIES["small_cfg_b2"], 1), True)
    gb = GpuBlock(mi, inp, True)
    h1 = hashlib.sha256(bf16_to_bits(gb.run()).tobytes()).hexdigest()
    other.run()
    h2 = hashlib.sha256(bf16_to_bits(gb.run()).tobytes()).hexdigest()
    assert h1 == h2


def test_zero_gates_return_the_input_exactly():
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES["small_ragged_17x19"], 2)
    mod = inp.mod.copy()
    mod[:, 2] = 0
    mod[:, 5] = 0
    inp.mod = mod
    gb = GpuBlock(mi, inp, True)
    assert np.array_equal(bf16_to_bits(gb.run()), inp.x)


def test_in_place_equals_out_of_place():
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES["small_cfg_b2"], 4)
    gb = GpuBlock(mi, inp, True)
    y = gb.run().clone()
    x = gb.x.clone()
    gb.run(x=x, y=x)
    assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_zero_modulation_matches_plain_prenorm_block():
    mi = require_gpu()
    g = mi_synth.GEOMETRIES["small_ragged_17x19"]
    inp = mi_synth.block_inputs(g, 5)
    mod = np.zeros_like(inp.mod)
    mod[:, 2] = mi_synth.bf16_bits(np.ones(g.hidden))
    mod[:, 5] = mi_synth.bf16_bits(np.ones(g.hidden))
    inp.mod = mod
    inp.key_mask[:] = 1
    gb = GpuBlock(mi, inp, True)
    w = inp.weights
    ref = O.plain_prenorm_block(O.widen(inp.x[0]), O.widen(w.w_qkv), O.widen(w.w_o), O.widen(w.w_gu), O.widen(w.w_d),
                                O.widen(w.q_norm_w), O.widen(w.k_norm_w), inp.rope_cos.astype(np.float64),
                                inp.rope_sin.astype(np.float64), g.n_heads)
    assert_parity(to_f64(gb.run())[0], ref, "y")


def test_workspace_too_small_is_refused():
    mi = require_gpu()
    inp = mi_synth.block_inputs(mi_synth.GEOMETRIES["tiny_8x8"], 0)
    gb = GpuBlock(mi, inp, True)
    small = gb.ws[: gb.ws.numel() // 2]
    with pytest.raises(mi.MiError) as e:
        gb.blk.forward(gb.layout, gb.x, gb.y, gb.mod, gb.cos, gb.sin, gb.mask, small)
    assert e.value.status == 3
