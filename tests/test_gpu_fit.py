"""One planned workspace serving several geometries (the pages' serving run: 1024x1024, 1280x1024
and 1408x1024 served from one scratch, 1536x1024 refused with an out-of-memory status, and the
next 1024x1024 request answered with the same bytes).  A two-block model at full width, batch 2
(prompt and empty negative), latent grids of 64 rows and 64, 80, 88 or 96 columns."""
import pytest
import torch

import mi_synth
from tests._gpu import require_gpu, to_dev
from tests.test_gpu_large import _gpu_step_weights

pytestmark = pytest.mark.gpu

GRIDS = [(64, 64), (64, 80), (64, 88), (64, 96)]  # 1024x1024, 1280x1024, 1408x1024, 1536x1024 pictures


def _geometry(gh, gw):
    return mi_synth.Geometry(f"fit_{gh}x{gw}", 2, 34, (34, 10), gh, gw, 3072, 24, 8192, n_blocks=2)


class _Serving:
    def __init__(self, mi):
        self.mi = mi
        g0 = _geometry(*GRIDS[0])
        self.p = _gpu_step_weights(g0, 11)
        self.model = mi.Model(self.p["blocks"], self.p["w_in"], self.p["w_out"], g0.n_heads, g0.eps)
        self.layouts = [mi.SeqLayout(2, 34, gh, gw) for gh, gw in GRIDS]

    def inputs(self, i, seed):
        g = _geometry(*GRIDS[i])
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        latent = torch.randn(g.n_img, g.latent_ch, generator=gen, device="cuda").to(torch.bfloat16).float()
        cos, sin = (to_dev(t) for t in mi_synth.rope_tables(g))
        return latent, cos, sin, to_dev(mi_synth.key_mask(g))

    def step(self, i, latent, cos, sin, mask, ws):
        self.model.denoise_step(self.layouts[i], latent, self.p["text"], self.p["mods"], self.p["mod_final"], cos,
                                sin, mask, -0.02, 3.0, ws)


def test_one_workspace_serves_several_geometries_and_refuses_the_rest():
    mi = require_gpu()
    sv = _Serving(mi)
    needs = [sv.model.workspace_size(L) for L in sv.layouts]
    assert needs == sorted(needs) and needs[2] < needs[3]
    nbytes, served = sv.model.plan(sv.layouts, needs[2])
    assert served == [True, True, True, False]
    assert nbytes == needs[2]
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")

    first = {}
    for i in range(3):  # every served geometry inside the one workspace
        lat, cos, sin, mask = sv.inputs(i, 100 + i)
        out = lat.clone()
        sv.step(i, out, cos, sin, mask, ws)
        torch.cuda.synchronize()
        assert mi.device_error() == 0
        assert torch.isfinite(out).all()
        first[i] = (lat, out)
        # the same step in a workspace of exactly its own size gives the same bytes
        own = torch.empty(needs[i], dtype=torch.uint8, device="cuda")
        out2 = lat.clone()
        sv.step(i, out2, cos, sin, mask, own)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int32), out2.view(torch.int32))
        del own

    # the geometry that does not fit is refused with the out-of-memory status, nothing enqueued
    lat, cos, sin, mask = sv.inputs(3, 103)
    out = lat.clone()
    with pytest.raises(mi.MiError) as e:
        sv.step(3, out, cos, sin, mask, ws)
    assert e.value.status == 3
    assert torch.equal(out, lat)

    # and the engine keeps serving: the first geometry again, the same bytes
    lat0, out0 = first[0]
    _, cos, sin, mask = sv.inputs(0, 100)
    again = lat0.clone()
    sv.step(0, again, cos, sin, mask, ws)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    assert torch.equal(again.view(torch.int32), out0.view(torch.int32))


def test_plan_with_no_geometry_in_budget_is_an_out_of_memory_refusal():
    mi = require_gpu()
    sv = _Serving(mi)
    need0 = sv.model.workspace_size(sv.layouts[0])
    with pytest.raises(mi.MiError) as e:
        sv.model.plan(sv.layouts, need0 - 1)
    assert e.value.status == 3
    nbytes, served = sv.model.plan(sv.layouts[:1], need0)
    assert served == [True] and nbytes == need0
