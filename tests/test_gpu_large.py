"""Full-size geometries: the long-sequence block (34 + 128x128 rows) on sampled rows, the guided step
at the 1024x1024 geometry (two blocks, and all 24 blocks, against the oracle; all 24 blocks for
repeatability), and the guided step captured in a CUDA graph."""
import os
import time

import numpy as np
import pytest
import torch

import mi_synth
from oracle import mi_oracle as O
from tests._gpu import (assert_parity, assert_parity_combination, parity_stats, require_gpu, to_dev, to_dev_bf16,
                        to_f64)

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def test_block_2048_sampled_rows():
    mi = require_gpu()
    g = mi_synth.GEOMETRIES["block_2048"]
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
    rng = np.random.default_rng(1)
    rows = np.unique(np.r_[0:8, 30:40, g.seq - 8:g.seq, rng.integers(0, g.seq, 40)])
    ref = O.block_forward_rows(O.widen(inp.x), O.widen(inp.mod), O.widen(w.w_qkv), O.widen(w.w_o),
                               O.widen(w.w_gu), O.widen(w.w_d), O.widen(w.q_norm_w), O.widen(w.k_norm_w),
                               inp.rope_cos.astype(np.float64), inp.rope_sin.astype(np.float64), rows,
                               inp.key_mask, g.n_heads, g.eps)
    assert_parity(to_f64(y)[0][rows], ref, "y on sampled rows of the 16418-row block")


def test_step_full_geometry_two_blocks():
    # the guided step at the 1024x1024 geometry (batch 2: prompt 34 rows, negative 10 rows padded
    # to 34 with a key mask) with two blocks, against the oracle's step
    mi = require_gpu()
    from tests.test_gpu_step import GpuStep, _oracle_step

    base = mi_synth.GEOMETRIES["step_1024_cfg"]
    g = mi_synth.Geometry("step_1024_cfg_2blocks", base.batch, base.text_pad, base.n_text, base.grid_h,
                          base.grid_w, base.hidden, base.n_heads, base.mlp_inter, n_blocks=2)
    si = mi_synth.step_inputs(g, 0)
    gs = GpuStep(mi, si)
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    gs.step(lat, 1.0, 3.0)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    _, vp, vn = _oracle_step(si, 1.0, 3.0)
    assert_parity_combination(to_f64(lat) - O.widen(si.latent), [(-2.0, vn), (3.0, vp)],
                              "guided velocity, 1024x1024 geometry, 2 blocks")


@pytest.mark.slow
def test_step_full_24_blocks_against_oracle():
    """The whole guided step at full size (24 blocks of the 1024x1024 geometry, batch 2: the prompt's
    34 rows and the empty negative's 10 rows padded to 34 with a key mask, guidance 3) against the
    oracle's step on the same seeded bf16 inputs.  Each branch velocity (guidance 1 and 0), the
    guided velocity and the latent after one step of the default schedule are compared at the
    per-tensor bar.  The oracle widens one block's weights at a time (24 blocks in float64 would
    be 21.7 GB) and takes several minutes on the host cores; its time is printed."""
    mi = require_gpu()
    from tests.test_gpu_step import GpuStep

    g = mi_synth.GEOMETRIES["step_1024_cfg"]
    t0 = time.perf_counter()
    si = mi_synth.step_inputs(g, 0)
    t_draw = time.perf_counter() - t0
    gs = GpuStep(mi, si)
    lat0 = to_dev(mi_synth.bits_to_f32(si.latent))
    vel = {}
    for name, guidance in (("guided", 3.0), ("prompt", 1.0), ("negative", 0.0)):
        lat = lat0.clone()
        gs.step(lat, 1.0, guidance)  # dt = 1: the latent moves by the velocity
        vel[name] = to_f64(lat) - O.widen(si.latent)
    ts = mi_synth.euler_schedule(50)
    dt = float(ts[1] - ts[0])  # the default schedule's step, -0.02
    lat = lat0.clone()
    gs.step(lat, dt, 3.0)
    lat_new = to_f64(lat)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    del gs

    a = O.step_inputs_widened_lazy(si)
    t0 = time.perf_counter()
    _, vp, vn = O.denoise_step(**a, dt=1.0, guidance=3.0)
    t_oracle = time.perf_counter() - t0
    print(f"oracle guided step at full size (24 blocks, batch 2): {t_oracle:.1f} s on {os.cpu_count()} host "
          f"cores (inputs drawn in {t_draw:.1f} s)")
    v = O.cfg_combine(vp, vn, 3.0)
    for name, got, ref in (("prompt velocity", vel["prompt"], vp), ("negative velocity", vel["negative"], vn),
                           ("latent after one step", lat_new, O.euler_update(O.widen(si.latent), v, dt))):
        cos, err, mref = parity_stats(got, ref)
        print(f"{name}: cosine {cos:.6f}, max|err|/max|ref| {err / mref:.3e}")
        assert_parity(got, ref, f"{name}, full-size guided step")
    # the guided velocity is a derived tensor, (1 - g) v_neg + g v_pos: held to the bound its branches
    # give it (its plain-bar figures are printed)
    assert_parity_combination(vel["guided"], [(-2.0, vn), (3.0, vp)], "guided velocity, full-size guided step")


def _gpu_step_weights(g, seed):
    """Seeded weights drawn on the GPU with the synthetic recipe's distributions (24 blocks at full
    size are 5.4 GB; drawing them on the host would dominate the test)."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    H, I, C, B = g.hidden, g.mlp_inter, g.latent_ch, g.batch

    def rn(*shape, std=1.0, mean=0.0):
        return (torch.randn(*shape, generator=gen, device="cuda") * std + mean).to(BF)

    blocks = [dict(w_qkv=rn(3 * H, H, std=0.02), w_o=rn(H, H, std=0.02), w_gu=rn(2 * I, H, std=0.02),
                   w_d=rn(H, I, std=0.02), q_norm_w=rn(128, std=0.02, mean=1.0), k_norm_w=rn(128, std=0.02, mean=1.0))
              for _ in range(g.n_blocks)]
    mods = rn(g.n_blocks, 1, 6, H, std=0.1).expand(g.n_blocks, B, 6, H).contiguous()
    return dict(blocks=blocks, mods=mods, w_in=rn(H, C, std=0.02), w_out=rn(C, H, std=0.02),
                mod_final=rn(1, 2, H, std=0.1).expand(B, 2, H).contiguous(),
                text=rn(B, g.text_pad, H), latent=torch.randn(g.n_img, C, generator=gen, device="cuda").to(BF).float())


def test_step_full_24_blocks_repeats_and_graph_capture():
    mi = require_gpu()
    g = mi_synth.GEOMETRIES["step_1024_cfg"]
    p = _gpu_step_weights(g, 7)
    model = mi.Model(p["blocks"], p["w_in"], p["w_out"], g.n_heads, g.eps)
    layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
    ws = torch.empty(model.workspace_size(layout), dtype=torch.uint8, device="cuda")
    cos, sin = (to_dev(t) for t in mi_synth.rope_tables(g))
    mask = to_dev(mi_synth.key_mask(g))

    def step(lat):
        model.denoise_step(layout, lat, p["text"], p["mods"], p["mod_final"], cos, sin, mask, -0.02, 3.0, ws)

    lat1 = p["latent"].clone()
    step(lat1)
    lat2 = p["latent"].clone()
    step(lat2)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    assert torch.isfinite(lat1).all()
    assert torch.equal(lat1.view(torch.int32), lat2.view(torch.int32))
    # the same step captured in a CUDA graph and replayed
    lat3 = p["latent"].clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(lat3)
    lat3.copy_(p["latent"])
    graph.replay()
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    assert torch.equal(lat3.view(torch.int32), lat1.view(torch.int32))
