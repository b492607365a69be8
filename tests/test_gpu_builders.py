"""Device-side builders: rotary tables, timestep -> modulation, and a guided loop that runs with no
host input per step (modulation, step and time advance all on the device, captured in a graph)."""
import numpy as np
import pytest
import torch

import mi_synth
from oracle import mi_oracle as O
from tests._gpu import assert_parity, assert_parity_combination, require_gpu, to_dev, to_dev_bf16, to_f64

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


@pytest.mark.parametrize("name", ["small_cfg_b2", "block_1024", "block_1200x880"])
def test_rope_tables_on_device(name):
    mi = require_gpu()
    g = mi_synth.GEOMETRIES[name]
    cos = torch.empty(g.seq, 64, dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    mi.rope_tables(g.text_pad, g.grid_h, g.grid_w, cos, sin)
    rc, rs = O.rope_angle_tables(g.text_pad, g.grid_h, g.grid_w)
    for got, ref in ((cos, rc), (sin, rs)):
        got = got.cpu().numpy().astype(np.float64)
        err = np.abs(got - ref)
        assert err.max() <= 1.2e-7  # within one fp32 ulp of the fp64 value (|value| <= 1)
        assert (got == ref.astype(np.float32)).mean() > 0.999  # almost always the correctly rounded fp32


def test_timestep_modulation_on_device():
    mi = require_gpu()
    g = mi_synth.GEOMETRIES["step_tiny_cfg"]
    tw = mi_synth.timestep_weights(g, 3)
    tm = mi.TimestepModulation(to_dev_bf16(tw.w_t1), to_dev_bf16(tw.w_t2), to_dev_bf16(tw.w_mod), g.n_blocks)
    t = torch.tensor([0.37, 0.37], dtype=torch.float32, device="cuda")
    mods = torch.empty(g.n_blocks, 2, 6, g.hidden, dtype=BF, device="cuda")
    fin = torch.empty(2, 2, g.hidden, dtype=BF, device="cuda")
    ws = torch.empty(tm.workspace_size(2), dtype=torch.uint8, device="cuda")
    tm(t, mods, fin, ws)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    rm, rf = O.timestep_modulation(np.array([0.37, 0.37], dtype=np.float32).astype(np.float64), O.widen(tw.w_t1),
                                   O.widen(tw.w_t2), O.widen(tw.w_mod), g.n_blocks)
    assert_parity(to_f64(mods), rm, "block modulation")
    assert_parity(to_f64(fin), rf, "final modulation")


def test_guided_loop_with_device_builders_in_a_graph():
    mi = require_gpu()
    from tests.test_gpu_step import GpuStep

    g = mi_synth.GEOMETRIES["step_tiny_cfg"]
    si = mi_synth.step_inputs(g, 8)
    tw = mi_synth.timestep_weights(g, 9)
    gs = GpuStep(mi, si)
    tm = mi.TimestepModulation(to_dev_bf16(tw.w_t1), to_dev_bf16(tw.w_t2), to_dev_bf16(tw.w_mod), g.n_blocks)
    n_steps = 5
    ts = mi_synth.euler_schedule(50)
    dt = float(ts[1] - ts[0])
    t = torch.full((2,), 1.0, dtype=torch.float32, device="cuda")
    mods = torch.empty(g.n_blocks, 2, 6, g.hidden, dtype=BF, device="cuda")
    fin = torch.empty(2, 2, g.hidden, dtype=BF, device="cuda")
    tws = torch.empty(tm.workspace_size(2), dtype=torch.uint8, device="cuda")
    cos = torch.empty(g.seq, 64, dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    mi.rope_tables(g.text_pad, g.grid_h, g.grid_w, cos, sin)
    lat0 = to_dev(mi_synth.bits_to_f32(si.latent))
    lat = lat0.clone()

    def step():
        tm(t, mods, fin, tws)
        gs.model.denoise_step(gs.layout, lat, gs.text, mods, fin, cos, sin, gs.mask, dt, 3.0, gs.ws)
        mi.time_advance(t, dt)

    # eager loop, recording every latent
    hist = [to_f64(lat)]
    for _ in range(n_steps):
        step()
        hist.append(to_f64(lat))
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    # the same loop from a CUDA graph of one step
    lat.copy_(lat0)
    t.fill_(1.0)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    lat.copy_(lat0)
    t.fill_(1.0)
    for _ in range(n_steps):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(lat.view(torch.int32), torch.from_numpy(hist[-1].astype(np.float32)).cuda().view(torch.int32))
    # every step against the oracle step from the same latent and timestep
    a = O.step_inputs_widened(si)
    a["rope_cos"], a["rope_sin"] = O.rope_angle_tables(g.text_pad, g.grid_h, g.grid_w)
    tcur = np.float32(1.0)
    for i in range(n_steps):
        rm, rf = O.timestep_modulation(np.array([tcur, tcur], dtype=np.float64), O.widen(tw.w_t1), O.widen(tw.w_t2),
                                       O.widen(tw.w_mod), g.n_blocks)
        a["latent"], a["mods"], a["mod_final"] = hist[i], list(rm), rf
        _, vp, vn = O.denoise_step(**a, dt=dt, guidance=3.0)
        assert_parity_combination(hist[i + 1] - hist[i], [(dt * -2.0, vn), (dt * 3.0, vp)], f"step {i}")
        tcur = np.float32(tcur + np.float32(dt))
