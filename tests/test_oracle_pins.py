"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each pin is a closed form, an invariant of the operation, a special case that
reduces to a textbook result, a value printed on the MOSS-Image pages, or a
scalar-loop brute force written directly from the definition.  The planted
mistakes at the end show that a plausible slip in the oracle fails at least one
pin.
"""
import json
import math
import os

import numpy as np
import pytest

import mi_synth
import oracle.mi_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ RMSNorm and modulation
def pin_unit_rms():
    x = _rng(1).standard_normal((7, 384)) * 3.0
    h = O.modulated_rms_norm(x, np.zeros(384), np.zeros(384), 1e-6)
    m = (x * x).mean(axis=1)
    rms_h = np.sqrt((h * h).mean(axis=1))
    np.testing.assert_allclose(rms_h, np.sqrt(m / (m + 1e-6)), rtol=0, atol=1e-14)


def pin_scale_invariance():
    x = _rng(2).standard_normal((5, 256))
    np.testing.assert_allclose(O.rms_norm(17.5 * x, 0.0), O.rms_norm(x, 0.0), atol=1e-14)


def pin_constant_row():
    # a constant row c*1 normalises to c / sqrt(c^2 + eps) in every entry
    for c in (0.5, -3.0, 1e-3):
        h = O.rms_norm(np.full((1, 64), c), 1e-6)
        np.testing.assert_allclose(h, c / math.sqrt(c * c + 1e-6), rtol=1e-15, atol=0)


def pin_modulation_affine():
    # shift and scale enter as (1 + scale) * n + shift per column
    x = _rng(3).standard_normal((4, 128))
    shift = _rng(4).standard_normal(128)
    scale = _rng(5).standard_normal(128)
    n = x / np.sqrt((x ** 2).mean(axis=1, keepdims=True) + 1e-6)
    h = O.modulated_rms_norm(x, shift, scale, 1e-6)
    np.testing.assert_allclose(h[:, 7], n[:, 7] * (1 + scale[7]) + shift[7], atol=1e-14)


def test_unit_rms():
    pin_unit_rms()


def test_scale_invariance():
    pin_scale_invariance()


def test_constant_row():
    pin_constant_row()


def test_modulation_affine():
    pin_modulation_affine()


# ------------------------------------------------------------------ block-level special cases
def _tiny_widened(seed=0, geom="tiny_8x8"):
    g = mi_synth.GEOMETRIES[geom]
    inp = mi_synth.block_inputs(g, seed)
    w = inp.weights
    args = dict(x=O.widen(inp.x), mod=O.widen(inp.mod), w_qkv=O.widen(w.w_qkv), w_o=O.widen(w.w_o),
                w_gu=O.widen(w.w_gu), w_d=O.widen(w.w_d), q_norm_w=O.widen(w.q_norm_w),
                k_norm_w=O.widen(w.k_norm_w), rope_cos=inp.rope_cos.astype(np.float64),
                rope_sin=inp.rope_sin.astype(np.float64), key_mask=inp.key_mask, n_heads=g.n_heads)
    return g, args


def pin_zero_modulation_is_plain_block():
    g, a = _tiny_widened(0)
    H = g.hidden
    mod = np.zeros((1, 6, H))
    mod[0, 2] = 1.0   # gate1
    mod[0, 5] = 1.0   # gate2
    a["mod"] = mod
    y = O.block_forward(**a)["y"][0]
    ref = O.plain_prenorm_block(a["x"][0], a["w_qkv"], a["w_o"], a["w_gu"], a["w_d"], a["q_norm_w"],
                                a["k_norm_w"], a["rope_cos"], a["rope_sin"], g.n_heads)
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-11)


def pin_zero_gates_identity():
    g, a = _tiny_widened(1)
    a["mod"] = a["mod"].copy()
    a["mod"][:, 2] = 0.0
    a["mod"][:, 5] = 0.0
    y = O.block_forward(**a)["y"]
    assert np.array_equal(y, a["x"])


def test_zero_modulation_is_plain_block():
    pin_zero_modulation_is_plain_block()


def test_zero_gates_identity():
    pin_zero_gates_identity()


# ------------------------------------------------------------------ rotary
def _angles(pos, n=64):
    j = np.arange(n, dtype=np.float64)
    freq = 0.37 ** (j / 8.0)      # any frequencies: the invariants hold for every table
    ang = pos[:, None] * freq[None, :]
    return np.cos(ang), np.sin(ang)


def pin_rope_norm_and_identity():
    t = _rng(6).standard_normal((9, 3, 128))
    c, s = _angles(np.arange(9, dtype=np.float64) * 1.7)
    r = O.rope(t, c, s)
    # every pair keeps its length, hence every head keeps its norm
    pair_in = t[..., 0::2] ** 2 + t[..., 1::2] ** 2
    pair_out = r[..., 0::2] ** 2 + r[..., 1::2] ** 2
    np.testing.assert_allclose(pair_out, pair_in, rtol=1e-13, atol=1e-14)
    # cos = 1, sin = 0 is the identity
    assert np.array_equal(O.rope(t, np.ones((9, 64)), np.zeros((9, 64))), t)


def pin_rope_relative_position():
    # <rope(q, p + c), rope(k, p' + c)> does not depend on c
    rng = _rng(7)
    q = rng.standard_normal((6, 1, 128))
    k = rng.standard_normal((6, 1, 128))
    pos = np.array([0, 1, 2, 5, 9, 14], dtype=np.float64)
    base = None
    for shift in (0.0, 3.0, 11.0):
        c, s = _angles(pos + shift)
        sc = O.rope(q, c, s)[:, 0] @ O.rope(k, c, s)[:, 0].T
        if base is None:
            base = sc
        else:
            np.testing.assert_allclose(sc, base, rtol=1e-12, atol=1e-12)


def pin_rope_pair_direction():
    # the pair (1, 0) rotated by angle a is (cos a, sin a): interleaved pairs, counter-clockwise
    t = np.zeros((1, 1, 128))
    t[0, 0, 0] = 1.0
    a = 0.3
    c = np.full((1, 64), math.cos(a))
    s = np.full((1, 64), math.sin(a))
    r = O.rope(t, c, s)
    assert abs(r[0, 0, 0] - math.cos(a)) < 1e-15 and abs(r[0, 0, 1] - math.sin(a)) < 1e-15
    assert np.all(r[0, 0, 2:] == 0)


def test_rope_norm_and_identity():
    pin_rope_norm_and_identity()


def test_rope_relative_position():
    pin_rope_relative_position()


def test_rope_pair_direction():
    pin_rope_pair_direction()


def test_rope_tables_reading():
    # the input tables follow the stated reading: image token (r, c) rotates its first 32 pairs
    # by r * 10000^(-j/32) and the last 32 by c * 10000^(-j/32); text row t uses t on both halves
    g = mi_synth.GEOMETRIES["small_ragged_17x19"]
    cos, sin = mi_synth.rope_tables(g)
    r, c, j = 5, 11, 7
    row = g.text_pad + r * g.grid_w + c
    w = 10000.0 ** (-j / 32)
    assert abs(cos[row, j] - np.float32(math.cos(r * w))) == 0
    assert abs(sin[row, 32 + j] - np.float32(math.sin(c * w))) == 0
    assert abs(cos[4, 32 + j] - np.float32(math.cos(4 * w))) == 0


# ------------------------------------------------------------------ attention
def pin_attention_bruteforce():
    rng = _rng(8)
    q = rng.standard_normal((7, 2, 128))
    k = rng.standard_normal((7, 2, 128))
    v = rng.standard_normal((7, 2, 128))
    valid = np.array([1, 1, 0, 1, 1, 1, 0], dtype=bool)
    np.testing.assert_allclose(O.attention(q, k, v, valid), O.attention_loops(q, k, v, valid),
                               rtol=0, atol=1e-12)


def pin_attention_two_keys():
    # two keys: weights are the logistic function of the score gap / sqrt(d)
    d = 128
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 2.0
    k = np.zeros((2, 1, d))
    k[0, 0, 0] = 1.5
    k[1, 0, 0] = -0.5
    v = np.zeros((2, 1, d))
    v[0, 0, 3] = 1.0
    v[1, 0, 3] = -1.0
    gap = (2.0 * 1.5 - 2.0 * -0.5) / math.sqrt(d)
    w0 = 1.0 / (1.0 + math.exp(-gap))
    o = O.attention(q, k, v)
    assert abs(o[0, 0, 3] - (w0 - (1 - w0))) < 1e-15


def pin_attention_equal_scores_cancellation():
    # q = 0 gives equal scores: o is the mean of V over the valid keys.  V rows of +-2^10 that
    # cancel stress the accumulation (the pages' adversarial attention gate, PR #1512).
    S = 33
    q = np.zeros((S, 1, 128))
    k = _rng(9).standard_normal((S, 1, 128))
    v = np.zeros((S, 1, 128))
    v[0::2, 0, :] = 1024.0
    v[1::2, 0, :] = -1024.0
    v[:, 0, 5] += np.arange(S)
    valid = np.ones(S, dtype=bool)
    valid[-1] = False  # leaves 16 of each sign
    o = O.attention(q, k, v, valid)
    assert np.allclose(o[:, 0, 0], 0.0, atol=1e-10)
    assert np.allclose(o[:, 0, 5], np.arange(S - 1).mean(), atol=1e-10)


def pin_attention_masked_huge_values():
    rng = _rng(10)
    q = rng.standard_normal((6, 2, 128))
    k = rng.standard_normal((6, 2, 128))
    v = rng.standard_normal((6, 2, 128))
    valid = np.array([1, 0, 1, 1, 0, 1], dtype=bool)
    o1 = O.attention(q, k, v, valid)
    v2 = v.copy()
    v2[~valid] = 1e30
    k2 = k.copy()
    k2[~valid] = 1e3
    assert np.array_equal(O.attention(q, k2, v2, valid), o1)


def test_attention_bruteforce():
    pin_attention_bruteforce()


def test_attention_two_keys():
    pin_attention_two_keys()


def test_attention_equal_scores_cancellation():
    pin_attention_equal_scores_cancellation()


def test_attention_masked_huge_values():
    pin_attention_masked_huge_values()


def test_attention_no_valid_key_is_zero():
    q = np.ones((3, 1, 128))
    assert np.array_equal(O.attention(q, q, q, np.zeros(3, dtype=bool)), np.zeros((3, 1, 128)))


# ------------------------------------------------------------------ SiLU
def pin_silu_knee():
    with open(os.path.join(GOLDEN, "silu_knee.json")) as f:
        gold = json.load(f)
    # locate the minimum on a fine grid, then compare with the printed 3-digit values
    z = np.linspace(-3, 0, 300001)
    s = O.silu(z)
    i = int(np.argmin(s))
    tol = 0.5 * 10.0 ** (-gold["printed_digits"])
    assert abs(z[i] - gold["z_min"]) <= tol + 1e-5
    assert abs(s[i] - gold["silu_min"]) <= tol
    # closed form at the minimum: d/dz [z sigma(z)] = 0 gives z sigma(z) = 1 + z
    lo, hi = -2.0, -1.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        sig = 1.0 / (1.0 + math.exp(-mid))
        if 1.0 + mid * (1.0 - sig) > 0:
            hi = mid
        else:
            lo = mid
    zs = 0.5 * (lo + hi)
    assert abs(O.silu(np.array([zs]))[0] - (1.0 + zs)) < 1e-14


def pin_silu_special():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu(np.array([40.0]))[0] - 40.0) < 1e-14
    assert abs(O.silu(np.array([-40.0]))[0] - (-40.0 * math.exp(-40.0))) < 1e-30
    z = np.array([0.7, -2.3])
    np.testing.assert_allclose(O.silu(z), z / (1 + np.exp(-z)), rtol=1e-15)
    assert np.isfinite(O.silu(np.array([-1000.0, 1000.0]))).all()


def test_silu_knee_golden():
    pin_silu_knee()


def test_silu_special():
    pin_silu_special()


# ------------------------------------------------------------------ projections (orientation)
def pin_projection_one_hot():
    # W_qkv one-hot: qkv column i copies h column perm[i]; W_gu one-hot makes gate/up copies of h2
    g, a = _tiny_widened(2)
    H, I = g.hidden, g.mlp_inter
    perm = _rng(11).permutation(3 * H) % H
    w = np.zeros((3 * H, H))
    w[np.arange(3 * H), perm] = 1.0
    a["w_qkv"] = w
    out = O.block_forward(**a)
    assert np.array_equal(out["qkv"][0], out["h"][0][:, perm])
    wg = np.zeros((2 * I, H))
    cols = _rng(12).integers(0, H, size=2 * I)
    wg[np.arange(2 * I), cols] = 1.0
    a["w_gu"] = wg
    out = O.block_forward(**a)
    assert np.array_equal(out["gu"][0], out["h2"][0][:, cols])
    # and the SiLU gate reads gate from the first I columns
    gu = out["gu"][0]
    np.testing.assert_allclose(out["m"][0], O.silu(gu[:, :I]) * gu[:, I:], rtol=1e-15)


def test_projection_one_hot():
    pin_projection_one_hot()


# ------------------------------------------------------------------ whole block by scalar loops
def _block_loops(x, mod, w_qkv, w_o, w_gu, w_d, gq, gk, cos, sin, valid, nh, eps):
    """The block for one batch element, written with Python loops over scalars."""
    S, H = len(x), len(x[0])
    d = H // nh
    inter = len(w_d[0])

    def matvec_t(row, W):  # row . W^T
        return [sum(row[c] * W[r][c] for c in range(len(row))) for r in range(len(W))]

    def mnorm(row, shift, scale):
        ms = sum(v * v for v in row) / len(row)
        r = 1.0 / math.sqrt(ms + eps)
        return [row[c] * r * (1.0 + scale[c]) + shift[c] for c in range(len(row))]

    shift1, scale1, gate1, shift2, scale2, gate2 = mod
    h = [mnorm(x[s], shift1, scale1) for s in range(S)]
    qkv = [matvec_t(h[s], w_qkv) for s in range(S)]
    qh = [[None] * nh for _ in range(S)]
    kh = [[None] * nh for _ in range(S)]
    for s in range(S):
        for j in range(nh):
            for which, store, gain in ((0, qh, gq), (1, kh, gk)):
                seg = qkv[s][which * H + j * d: which * H + (j + 1) * d]
                ms = sum(v * v for v in seg) / d
                r = 1.0 / math.sqrt(ms + eps)
                nv = [seg[e] * r * gain[e] for e in range(d)]
                rot = [0.0] * d
                for p in range(d // 2):
                    a_, b_ = nv[2 * p], nv[2 * p + 1]
                    rot[2 * p] = a_ * cos[s][p] - b_ * sin[s][p]
                    rot[2 * p + 1] = a_ * sin[s][p] + b_ * cos[s][p]
                store[s][j] = rot
    o = [[0.0] * H for _ in range(S)]
    for j in range(nh):
        for s in range(S):
            sc = [(t, sum(qh[s][j][e] * kh[t][j][e] for e in range(d)) / math.sqrt(d))
                  for t in range(S) if valid[t]]
            mx = max(v for _, v in sc)
            den = sum(math.exp(v - mx) for _, v in sc)
            for e in range(d):
                o[s][j * d + e] = sum(math.exp(v - mx) / den * qkv[t][2 * H + j * d + e]
                                      for t, v in sc)
    y = []
    for s in range(S):
        a_row = matvec_t(o[s], w_o)
        x1 = [x[s][c] + gate1[c] * a_row[c] for c in range(H)]
        h2 = mnorm(x1, shift2, scale2)
        gu = matvec_t(h2, w_gu)
        m = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[inter + i] for i in range(inter)]
        dn = matvec_t(m, w_d)
        y.append([x1[c] + gate2[c] * dn[c] for c in range(H)])
    return y


def pin_block_loops():
    rng = _rng(13)
    S, H, nh, I = 5, 256, 2, 6
    x = rng.standard_normal((1, S, H))
    mod = rng.standard_normal((1, 6, H)) * 0.3
    w_qkv = rng.standard_normal((3 * H, H)) * 0.05
    w_o = rng.standard_normal((H, H)) * 0.05
    w_gu = rng.standard_normal((2 * I, H)) * 0.05
    w_d = rng.standard_normal((H, I)) * 0.05
    gq = 1 + 0.1 * rng.standard_normal(128)
    gk = 1 + 0.1 * rng.standard_normal(128)
    ang = rng.uniform(-3, 3, size=(S, 64))
    cos, sin = np.cos(ang), np.sin(ang)
    mask = np.array([[1, 1, 0, 1, 1]], dtype=np.uint8)
    y = O.block_forward(x, mod, w_qkv, w_o, w_gu, w_d, gq, gk, cos, sin, mask, nh, 1e-6)["y"][0]
    ref = _block_loops(x[0].tolist(), mod[0].tolist(), w_qkv.tolist(), w_o.tolist(), w_gu.tolist(),
                       w_d.tolist(), gq.tolist(), gk.tolist(), cos.tolist(), sin.tolist(),
                       mask[0].tolist(), nh, 1e-6)
    np.testing.assert_allclose(y, np.array(ref), rtol=0, atol=1e-12)


def test_block_loops():
    pin_block_loops()


# ------------------------------------------------------------------ guidance and Euler
def pin_guidance_identities():
    rng = _rng(14)
    vp = rng.standard_normal((10, 4))
    vn = rng.standard_normal((10, 4))
    np.testing.assert_allclose(O.cfg_combine(vp, vn, 1.0), vp, rtol=0, atol=1e-15)
    assert np.array_equal(O.cfg_combine(vp, vp, 3.0), vp)
    np.testing.assert_allclose(O.cfg_combine(vp, vn, 3.0), 3 * vp - 2 * vn, atol=1e-14)


def pin_euler_schedule():
    ts = mi_synth.euler_schedule(50)
    dts = np.diff(ts)
    assert abs(dts.sum() + 1.0) < 1e-15
    assert np.allclose(dts, -0.02, atol=1e-15)
    v = _rng(15).standard_normal((8, 3))
    x0 = _rng(16).standard_normal((8, 3))
    xf = O.euler_loop(x0, ts, lambda x, dt: O.euler_update(x, v, dt))
    np.testing.assert_allclose(xf, x0 - v, rtol=0, atol=1e-13)


def test_guidance_identities():
    pin_guidance_identities()


def test_euler_schedule():
    pin_euler_schedule()


def test_denoise_step_guidance_one_ignores_negative():
    si = mi_synth.step_inputs(mi_synth.Geometry("t", 2, 10, (10, 4), 4, 4, 256, 2, 256, n_blocks=2), 3)
    a = O.step_inputs_widened(si)
    lat1, vp, vn = O.denoise_step(**a, dt=-0.02, guidance=1.0)
    np.testing.assert_allclose(lat1, a["latent"] - 0.02 * vp, atol=1e-14)
    # a different negative prompt changes v_neg but not the guidance-1 update
    a2 = dict(a)
    a2["text_rows"] = a["text_rows"].copy()
    a2["text_rows"][1] *= -1
    lat2, vp2, vn2 = O.denoise_step(**a2, dt=-0.02, guidance=1.0)
    assert np.array_equal(vp2, vp) and not np.allclose(vn2, vn)
    np.testing.assert_allclose(lat2, lat1, atol=1e-14)


def test_denoise_step_skip_negative_block():
    si = mi_synth.step_inputs(mi_synth.Geometry("t", 2, 10, (10, 4), 4, 4, 256, 2, 256, n_blocks=2), 4)
    a = O.step_inputs_widened(si)
    _, vp, vn = O.denoise_step(**a, dt=-0.02, guidance=3.0, skip_neg=[True, True])
    # with every block skipped the negative branch's velocity is the head applied to W_in-embedded latent
    u = a["latent"] @ a["w_in"].T
    ref = O.modulated_rms_norm(u, a["mod_final"][1, 0], a["mod_final"][1, 1]) @ a["w_out"].T
    np.testing.assert_allclose(vn, ref, atol=1e-12)
    _, vp_ns, _ = O.denoise_step(**a, dt=-0.02, guidance=3.0)
    assert np.array_equal(vp, vp_ns)


def test_padded_negative_rows_do_not_leak():
    # the masked padded rows of the negative element never reach the image rows
    g = mi_synth.GEOMETRIES["small_cfg_b2"]
    inp = mi_synth.block_inputs(g, 5)
    out1 = O.block_forward_inputs(inp)
    x2 = inp.x.copy()
    x2[1, g.n_text[1]: g.text_pad] = mi_synth.bf16_bits(np.full((g.text_pad - g.n_text[1], g.hidden), 7.0))
    inp2 = mi_synth.BlockInputs(g, x2, inp.mod, inp.weights, inp.rope_cos, inp.rope_sin, inp.key_mask)
    out2 = O.block_forward_inputs(inp2)
    valid = inp.key_mask[1] != 0
    np.testing.assert_allclose(out2["y"][1][valid], out1["y"][1][valid], rtol=0, atol=1e-12)


# ------------------------------------------------------------------ planted mistakes
def _mut_rope_reflect(t, cos, sin):
    out = np.empty_like(t)
    a, b = t[..., 0::2], t[..., 1::2]
    out[..., 0::2] = a * cos[:, None, :] - b * sin[:, None, :]
    out[..., 1::2] = a * sin[:, None, :] - b * cos[:, None, :]
    return out


def _mut_rms_sum(x, eps=1e-6):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _mut_mod_no_one(x, shift, scale, eps=1e-6):
    return O.rms_norm(x, eps) * scale + shift


_ATTENTION = O.attention


def _mut_attention_noscale(q, k, v, valid=None):
    return _ATTENTION(q * math.sqrt(q.shape[-1]), k, v, valid)


def _mut_silu_gate_swapped(gu, inter):
    return O.silu(gu[..., inter:]) * gu[..., :inter]


def _mut_silu_sign(z):
    return np.asarray(z) / (1.0 + np.exp(np.asarray(z)))


MUTANTS = [
    ("rope", _mut_rope_reflect, [pin_rope_relative_position, pin_block_loops]),
    ("rms_norm", _mut_rms_sum, [pin_unit_rms, pin_block_loops]),
    ("modulated_rms_norm", _mut_mod_no_one, [pin_zero_modulation_is_plain_block, pin_block_loops]),
    ("attention", _mut_attention_noscale, [pin_attention_bruteforce, pin_block_loops]),
    ("silu_gate", _mut_silu_gate_swapped, [pin_block_loops, pin_projection_one_hot]),
    ("silu", _mut_silu_sign, [pin_silu_knee, pin_silu_special]),
]


@pytest.mark.parametrize("name,mutant,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, mutant, pins):
    monkeypatch.setattr(O, name, mutant)
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()


def test_row_subset_forward_matches_full_forward():
    g = mi_synth.GEOMETRIES["small_ragged_17x19"]
    inp = mi_synth.block_inputs(g, 7)
    full = O.block_forward_inputs(inp)["y"][0]
    w = inp.weights
    rows = np.array([0, 5, 12, 13, 200, g.seq - 1])
    sub = O.block_forward_rows(O.widen(inp.x), O.widen(inp.mod), O.widen(w.w_qkv), O.widen(w.w_o),
                               O.widen(w.w_gu), O.widen(w.w_d), O.widen(w.q_norm_w), O.widen(w.k_norm_w),
                               inp.rope_cos.astype(np.float64), inp.rope_sin.astype(np.float64), rows,
                               inp.key_mask, g.n_heads)
    np.testing.assert_allclose(sub, full[rows], rtol=0, atol=1e-12)


# ------------------------------------------------------------------ device-side builders
def test_rope_angle_tables_pins():
    cos, sin = O.rope_angle_tables(3, 4, 5)
    np.testing.assert_allclose(cos ** 2 + sin ** 2, 1.0, atol=1e-15)
    # pair 0 has frequency 1: the angle is the position itself
    assert abs(cos[2, 0] - math.cos(2.0)) < 1e-15 and abs(sin[2, 32] - math.sin(2.0)) < 1e-15
    # image token (r, c) = (1, 3): row axis on the first half, column axis on the second
    s = 3 + 1 * 5 + 3
    w = 10000.0 ** (-5 / 32)
    assert abs(cos[s, 5] - math.cos(1 * w)) < 1e-15 and abs(cos[s, 37] - math.cos(3 * w)) < 1e-15
    # text row t and image token (t, t) share every angle
    t = 2
    assert np.array_equal(cos[t], cos[3 + t * 5 + t]) and np.array_equal(sin[t], sin[3 + t * 5 + t])
    # consecutive columns differ by one rotation step: angle addition on the column half
    a = 3 + 2 * 5
    j = 40
    w = 10000.0 ** (-(j - 32) / 32)
    rot = cos[a, j] * math.cos(w) - sin[a, j] * math.sin(w)
    assert abs(rot - cos[a + 1, j]) < 1e-14


def test_rope_angle_tables_match_the_input_tables():
    g = mi_synth.GEOMETRIES["small_ragged_17x19"]
    cos, sin = O.rope_angle_tables(g.text_pad, g.grid_h, g.grid_w)
    c32, s32 = mi_synth.rope_tables(g)
    assert np.array_equal(cos.astype(np.float32), c32) and np.array_equal(sin.astype(np.float32), s32)


def test_timestep_embedding_pins():
    e0 = O.timestep_embedding([0.0])
    assert np.all(e0[0, :128] == 1.0) and np.all(e0[0, 128:] == 0.0)
    e = O.timestep_embedding([0.37, 0.8])
    np.testing.assert_allclose((e ** 2).sum(axis=1), 128.0, rtol=1e-13)
    assert abs(e[0, 0] - math.cos(370.0)) < 1e-12 and abs(e[1, 128] - math.sin(800.0)) < 1e-12
    assert abs(e[0, 127] - math.cos(370.0 * 10000.0 ** (-127 / 128))) < 1e-12


def test_timestep_modulation_pins():
    rng = _rng(21)
    H, n = 256, 3
    w1 = rng.standard_normal((H, 256)) * 0.05
    w2 = rng.standard_normal((H, H)) * 0.05
    wm = rng.standard_normal(((6 * n + 2) * H, H)) * 0.05
    mods, fin = O.timestep_modulation([0.25, 0.25], w1, w2, wm, n)
    assert mods.shape == (n, 2, 6, H) and fin.shape == (2, 2, H)
    assert np.array_equal(mods[:, 0], mods[:, 1])  # the same timestep gives the same vectors
    # block i's k-th vector is rows [(6 i + k) H, (6 i + k + 1) H) of W_mod applied to silu(c)
    c = O.silu(w1 @ O.timestep_embedding([0.25])[0]) @ w2.T
    sc = O.silu(c)
    np.testing.assert_allclose(mods[1, 0, 4], wm[(6 + 4) * H:(6 + 5) * H] @ sc, atol=1e-13)
    np.testing.assert_allclose(fin[0, 1], wm[(6 * n + 1) * H:(6 * n + 2) * H] @ sc, atol=1e-13)
    # zero projection gives zero modulation
    m0, f0 = O.timestep_modulation([0.5], w1, w2, np.zeros_like(wm), n)
    assert not m0.any() and not f0.any()
