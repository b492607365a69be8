"""The guided denoising step (mi_denoise_step) against the float64 oracle's step."""
import numpy as np
import pytest
import torch

import mi_synth
from oracle import mi_oracle as O
from tests._gpu import (COS_MIN, REL_MAX, assert_parity, assert_parity_combination, require_gpu, to_dev,
                        to_dev_bf16, to_f64)

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


class GpuStep:
    def __init__(self, mi, si, fused=True):
        g = si.geom
        self.g = g
        self.blocks = [dict(w_qkv=to_dev_bf16(b.w_qkv), w_o=to_dev_bf16(b.w_o), w_gu=to_dev_bf16(b.w_gu),
                            w_d=to_dev_bf16(b.w_d), q_norm_w=to_dev_bf16(b.q_norm_w),
                            k_norm_w=to_dev_bf16(b.k_norm_w)) for b in si.blocks]
        self.w_in = to_dev_bf16(si.w_in)
        self.w_out = to_dev_bf16(si.w_out)
        self.model = mi.Model(self.blocks, self.w_in, self.w_out, g.n_heads, g.eps, fused)
        self.layout = mi.SeqLayout(g.batch, g.text_pad, g.grid_h, g.grid_w)
        self.text = to_dev_bf16(si.text_rows)
        self.mods = to_dev_bf16(np.stack(si.mods))
        self.mod_final = to_dev_bf16(si.mod_final)
        self.cos = to_dev(si.rope_cos)
        self.sin = to_dev(si.rope_sin)
        self.mask = to_dev(si.key_mask)
        self.ws = torch.empty(self.model.workspace_size(self.layout), dtype=torch.uint8, device="cuda")

    def step(self, latent, dt, guidance, skip_neg=None):
        sk = None if skip_neg is None else np.asarray(skip_neg, dtype=np.uint8)
        self.model.denoise_step(self.layout, latent, self.text, self.mods, self.mod_final, self.cos, self.sin,
                                self.mask, dt, guidance, self.ws, skip_neg=sk)


def _oracle_step(si, dt, guidance, skip_neg=None, latent=None):
    a = O.step_inputs_widened(si)
    if latent is not None:
        a["latent"] = latent
    return O.denoise_step(**a, dt=dt, guidance=guidance, skip_neg=skip_neg)


def test_step_velocity_parity():
    # dt = 1 makes the latent change equal to the guided velocity
    mi = require_gpu()
    si = mi_synth.step_inputs(mi_synth.GEOMETRIES["step_tiny_cfg"], 0)
    gs = GpuStep(mi, si)
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    gs.step(lat, 1.0, 3.0)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    _, vp, vn = _oracle_step(si, 1.0, 3.0)
    # v = (1 - g) v_neg + g v_pos: each branch carries the per-tensor bar, the combination their sum
    assert_parity_combination(to_f64(lat) - O.widen(si.latent), [(-2.0, vn), (3.0, vp)], "guided velocity")


def test_step_parity_default_schedule():
    mi = require_gpu()
    si = mi_synth.step_inputs(mi_synth.GEOMETRIES["step_tiny_cfg"], 1)
    gs = GpuStep(mi, si)
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    gs.step(lat, -0.02, 3.0)
    new, _, _ = _oracle_step(si, -0.02, 3.0)
    assert_parity(to_f64(lat), new, "latent")


def test_step_skip_negative_block():
    mi = require_gpu()
    si = mi_synth.step_inputs(mi_synth.GEOMETRIES["step_tiny_cfg"], 2)
    skip = np.zeros(si.geom.n_blocks, dtype=bool)
    skip[22] = True
    gs = GpuStep(mi, si)
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    gs.step(lat, 1.0, 3.0, skip_neg=skip)
    _, vp, vn = _oracle_step(si, 1.0, 3.0, skip_neg=skip)
    assert_parity_combination(to_f64(lat) - O.widen(si.latent), [(-2.0, vn), (3.0, vp)],
                              "velocity with block 22 skipped")


def test_step_batch_one_is_the_prompt_velocity():
    mi = require_gpu()
    g2 = mi_synth.GEOMETRIES["step_tiny_cfg"]
    si = mi_synth.step_inputs(g2, 3)
    gs = GpuStep(mi, si)
    g1 = mi_synth.Geometry("b1", 1, g2.text_pad, g2.n_text[:1], g2.grid_h, g2.grid_w, g2.hidden, g2.n_heads,
                           g2.mlp_inter, n_blocks=g2.n_blocks)
    gs.layout = mi.SeqLayout(1, g2.text_pad, g2.grid_h, g2.grid_w)
    gs.mods = to_dev_bf16(np.stack([m[:1] for m in si.mods]))
    gs.mod_final = to_dev_bf16(si.mod_final[:1])
    gs.mask = to_dev(si.key_mask[:1])
    gs.text = to_dev_bf16(si.text_rows[:1])
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    gs.step(lat, 1.0, 3.0)
    _, vp, _ = _oracle_step(si, 1.0, 3.0)
    assert_parity(to_f64(lat) - O.widen(si.latent), vp, "prompt velocity")
    assert g1.batch == 1


@pytest.mark.parametrize("guidance", [1.0, 0.0], ids=["prompt_branch", "negative_branch"])
def test_step_branch_velocities(guidance):
    # guidance 1 gives v = v_pos and guidance 0 gives v = v_neg: each branch alone at the bar
    mi = require_gpu()
    si = mi_synth.step_inputs(mi_synth.GEOMETRIES["step_tiny_cfg"], 6)
    gs = GpuStep(mi, si)
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    gs.step(lat, 1.0, guidance)
    _, vp, vn = _oracle_step(si, 1.0, guidance)
    assert_parity(to_f64(lat) - O.widen(si.latent), vp if guidance == 1.0 else vn, "branch velocity")


def test_euler_loop_50_steps():
    # every step is checked against the oracle step taken from the same (GPU) latent; the whole
    # chain is then compared with the oracle's own 50-step chain
    mi = require_gpu()
    g = mi_synth.GEOMETRIES["loop_tiny_cfg50"]
    si = mi_synth.step_inputs(g, 4)
    gs = GpuStep(mi, si)
    ts = mi_synth.euler_schedule(g.n_steps)
    lat = to_dev(mi_synth.bits_to_f32(si.latent))
    hist = [to_f64(lat)]
    for i in range(g.n_steps):
        gs.step(lat, float(ts[i + 1] - ts[i]), g.guidance)
        hist.append(to_f64(lat))
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    a = O.step_inputs_widened(si)
    gd = g.guidance
    for i in range(g.n_steps):
        a["latent"] = hist[i]
        dt = ts[i + 1] - ts[i]
        _, vp, vn = O.denoise_step(**a, dt=dt, guidance=gd)
        assert_parity_combination(hist[i + 1] - hist[i], [(dt * (1 - gd), vn), (dt * gd, vp)],
                                  f"step {i} displacement")

    # the oracle's own chain; first-order bound: the per-step velocity bounds summed over the steps
    x = O.widen(si.latent)
    l2_bound = max_bound = 0.0
    rel_l2 = np.sqrt(2.0 * (1.0 - COS_MIN))
    for i in range(g.n_steps):
        a["latent"] = x
        dt = ts[i + 1] - ts[i]
        x, vp, vn = O.denoise_step(**a, dt=dt, guidance=gd)
        l2_bound += abs(dt) * rel_l2 * (abs(1 - gd) * np.linalg.norm(vn) + abs(gd) * np.linalg.norm(vp))
        max_bound += abs(dt) * REL_MAX * (abs(1 - gd) * np.abs(vn).max() + abs(gd) * np.abs(vp).max())
    e = hist[-1] - x
    print(f"50-step chain: |err|_2 {np.linalg.norm(e):.4g} (bound {l2_bound:.4g}), "
          f"max|err| {np.abs(e).max():.4g} (bound {max_bound:.4g})")
    assert np.linalg.norm(e) <= l2_bound and np.abs(e).max() <= max_bound
    assert_parity(hist[-1], x, "latent after 50 steps")


def test_step_repeats_bit_for_bit():
    mi = require_gpu()
    si = mi_synth.step_inputs(mi_synth.GEOMETRIES["step_tiny_cfg"], 5)
    gs = GpuStep(mi, si)
    outs = []
    for _ in range(2):
        lat = to_dev(mi_synth.bits_to_f32(si.latent))
        gs.step(lat, -0.02, 3.0)
        outs.append(lat.cpu().numpy().copy())
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
