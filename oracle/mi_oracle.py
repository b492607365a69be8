"""Float64 CPU oracle of the MOSS-Image-style diffusion-transformer block.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module.  The CUDA library
never calls it and shares no code with it; the only thing both sides share is
the seeded input generator ``mi_synth`` (which holds none of the arithmetic).

What is computed follows the TensorFold "MOSS-Image transformer on CUDA" page
(PR #1528, "What it adds": modulated RMSNorm, q/k norm and rotary into packed
rows, the SiLU gate, gated add; projections as GEMMs with fp32 sums; full
head-128 attention; "Precision": bf16 weights/activations with fp32 sums, norms
and softmax) and the MOSS-Image host on PR #2281 ("What this changes": the
pipeline's schedule, empty negative prompt, classifier-free guidance).  The
pages give the kernel list, not the formulas; every formula below is the plain
textbook definition of the named operation, with these readings where the pages
are silent:

* RMSNorm eps = 1e-6; modulation is ``norm(x) * (1 + scale) + shift`` with no
  learned gain; the six vectors per batch element are ordered
  shift1, scale1, gate1, shift2, scale2, gate2 and apply to text and image rows.
* q/k RMSNorm over each 128-wide head with one gain vector for q and one for k
  (shared by all heads), applied before the rotary.
* Rotary acts on interleaved pairs (2p, 2p+1): (a, b) -> (a cos - b sin, a sin + b cos)
  with cos/sin taken from the input tables at (row, p).
* Attention is non-causal softmax(q k^T / sqrt(128)) v; a key whose mask byte
  is 0 gets weight 0.  A query row with no valid key returns zeros.
* No biases.  MLP: silu(gate) * up, then down; gate rows come first in W_gu.
* The oracle keeps every intermediate in float64 (no bf16 rounding between
  steps); inputs are the bf16 tensors widened exactly.

Pins (tests/test_oracle_pins.py): unit RMS after RMSNorm, scale invariance,
zero modulation equals a separately written plain pre-norm block, zero gates
give the identity, rotary norm preservation / identity / relative-position
invariance, scalar-loop brute force of the whole block on a tiny input, equal
scores giving the mean of V, masked keys carrying huge values leaving the
output unchanged, the SiLU minimum printed on PR #2281 ("Three findings"),
one-hot projections, and the guidance / Euler identities.  Parity unpinned:
the numeric value of a random block under the readings above (the pages give
no per-block numbers and no weights are available); which of the readings the
real checkpoint uses.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

EPS_DEFAULT = 1e-6


# ----------------------------------------------------------------------------------------------
# decoding of the bf16 inputs (exact widening)
# ----------------------------------------------------------------------------------------------
def widen(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64, exactly (a bf16 is the top half of an IEEE binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------------------------
# normalisation (PR #1528 "What it adds": modulated RMSNorm; q/k norm)
# ----------------------------------------------------------------------------------------------
def rms_norm(x: np.ndarray, eps: float = EPS_DEFAULT) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def modulated_rms_norm(x, shift, scale, eps: float = EPS_DEFAULT):
    """adaLN: rms_norm(x) * (1 + scale) + shift; shift/scale broadcast over rows."""
    return rms_norm(x, eps) * (1.0 + scale) + shift


def head_rms_norm(t: np.ndarray, gain: np.ndarray, n_heads: int, eps: float = EPS_DEFAULT):
    """Per-head RMSNorm of [..., n_heads*d] rows with a shared gain [d]; returns [..., n_heads, d]."""
    d = gain.shape[0]
    th = t.reshape(t.shape[:-1] + (n_heads, d))
    return rms_norm(th, eps) * gain


# ----------------------------------------------------------------------------------------------
# rotary (PR #1528: "q/k norm and rotary into packed rows")
# ----------------------------------------------------------------------------------------------
def rope(t: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate interleaved pairs of t [S, n_heads, d] by the angles of cos/sin [S, d/2]."""
    a = t[..., 0::2]
    b = t[..., 1::2]
    c = cos[:, None, :]
    s = sin[:, None, :]
    out = np.empty_like(t)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out


# ----------------------------------------------------------------------------------------------
# attention (PR #1528: full, non-causal attention at head dim 128, fp32 softmax)
# ----------------------------------------------------------------------------------------------
def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, valid: Optional[np.ndarray] = None):
    """softmax(q k^T / sqrt(d)) v per head.

    q, k, v: [S, n_heads, d]; valid: bool [S] over keys (None = all valid).
    Returns [S, n_heads, d]."""
    S, nh, d = q.shape
    out = np.zeros_like(q)
    if valid is None:
        valid = np.ones(k.shape[0], dtype=bool)
    kv = k[valid]
    vv = v[valid]
    if kv.shape[0] == 0:
        return out
    for h in range(nh):
        z = q[:, h, :] @ kv[:, h, :].T / np.sqrt(d)
        z = z - z.max(axis=1, keepdims=True)
        p = np.exp(z)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ vv[:, h, :]
    return out


def attention_loops(q, k, v, valid=None):
    """The same attention with explicit Python loops over scalars (tiny inputs only)."""
    import math

    S, nh, d = q.shape
    Sk = k.shape[0]
    out = np.zeros_like(q)
    for h in range(nh):
        for i in range(S):
            scores = []
            for j in range(Sk):
                if valid is not None and not valid[j]:
                    continue
                dot = 0.0
                for e in range(d):
                    dot += float(q[i, h, e]) * float(k[j, h, e])
                scores.append((j, dot / math.sqrt(d)))
            if not scores:
                continue
            mx = max(s for _, s in scores)
            den = sum(math.exp(s - mx) for _, s in scores)
            for e in range(d):
                acc = 0.0
                for j, s in scores:
                    acc += math.exp(s - mx) / den * float(v[j, h, e])
                out[i, h, e] = acc
    return out


# ----------------------------------------------------------------------------------------------
# MLP (PR #1528: the SiLU gate kernel; PR #2281 "Three findings": silu is not monotone)
# ----------------------------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """z * sigmoid(z) = z / (1 + exp(-z)), written to avoid overflow for very negative z."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = z[pos] / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = z[~pos] * ez / (1.0 + ez)
    return out


def silu_gate(gu: np.ndarray, inter: int) -> np.ndarray:
    """m = silu(gate) * up for gu = [..., 2I] with gate columns [0, I) and up columns [I, 2I)."""
    return silu(gu[..., :inter]) * gu[..., inter:]


# ----------------------------------------------------------------------------------------------
# projections (PR #1528: bf16 GEMMs with fp32 sums; here exact in float64)
# ----------------------------------------------------------------------------------------------
def project(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """x W^T for rows x [..., K] and a weight W [N, K] (no bias)."""
    return x @ w.T


def gated_residual(x, gate, y):
    """x + gate * y (gate broadcast over rows)."""
    return x + gate * y


# ----------------------------------------------------------------------------------------------
# the block (the step list of PR #1528's kernels, with projections between them)
# ----------------------------------------------------------------------------------------------
def block_forward(x, mod, w_qkv, w_o, w_gu, w_d, q_norm_w, k_norm_w, rope_cos, rope_sin,
                  key_mask=None, n_heads=None, eps=EPS_DEFAULT) -> Dict[str, np.ndarray]:
    """One block over every batch element; float64 in and out.

    x [B, S, H]; mod [B, 6, H]; weights as in mi_synth.BlockWeights (widened);
    rope_cos/sin [S, 64]; key_mask [B, S] (nonzero = valid) or None.
    Returns every intermediate: h, q, k (after norm+rotary, [B, nh, S, d]), v, o, a, x1,
    h2, gu, m, dn, y."""
    B, S, H = x.shape
    d = q_norm_w.shape[0]
    nh = n_heads if n_heads is not None else H // d
    I = w_d.shape[1]
    outs = {k: [] for k in ("h", "qkv", "q", "k", "v", "o", "a", "x1", "h2", "gu", "m", "dn", "y")}
    for b in range(B):
        shift1, scale1, gate1, shift2, scale2, gate2 = mod[b]
        xb = x[b]
        h = modulated_rms_norm(xb, shift1, scale1, eps)                      # step 1
        qkv = project(h, w_qkv)                                               # step 2
        q, k, v = qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:]
        qn = rope(head_rms_norm(q, q_norm_w, nh, eps), rope_cos, rope_sin)   # steps 3-4
        kn = rope(head_rms_norm(k, k_norm_w, nh, eps), rope_cos, rope_sin)
        vh = v.reshape(S, nh, d)
        valid = None if key_mask is None else np.asarray(key_mask[b]) != 0
        o = attention(qn, kn, vh, valid).reshape(S, H)                       # step 5
        a = project(o, w_o)
        x1 = gated_residual(xb, gate1, a)                                     # step 6
        h2 = modulated_rms_norm(x1, shift2, scale2, eps)                     # step 7
        gu = project(h2, w_gu)
        m = silu_gate(gu, I)                                                  # step 8
        dn = project(m, w_d)
        y = gated_residual(x1, gate2, dn)                                     # step 9
        for name, val in (("h", h), ("qkv", qkv), ("q", qn.transpose(1, 0, 2)),
                          ("k", kn.transpose(1, 0, 2)), ("v", vh.transpose(1, 0, 2)), ("o", o),
                          ("a", a), ("x1", x1), ("h2", h2), ("gu", gu), ("m", m), ("dn", dn),
                          ("y", y)):
            outs[name].append(val)
    return {k: np.stack(v) for k, v in outs.items()}


def block_forward_rows(x, mod, w_qkv, w_o, w_gu, w_d, q_norm_w, k_norm_w, rope_cos, rope_sin, rows,
                       key_mask=None, n_heads=None, eps=EPS_DEFAULT) -> np.ndarray:
    """The block output y for the query rows `rows` of batch element 0 only ([len(rows), H]).

    Same step list as block_forward; keys and values are still formed from every row (attention
    reads all of them), but the query-side steps run for the selected rows alone.  Used to time
    the oracle on a bounded sample of a large workload."""
    S, H = x.shape[1], x.shape[2]
    d = q_norm_w.shape[0]
    nh = n_heads if n_heads is not None else H // d
    inter = w_d.shape[1]
    shift1, scale1, gate1, shift2, scale2, gate2 = mod[0]
    xb = x[0]
    h = modulated_rms_norm(xb, shift1, scale1, eps)
    k = project(h, w_qkv[H:2 * H])
    v = project(h, w_qkv[2 * H:])
    q = project(h[rows], w_qkv[:H])
    qn = rope(head_rms_norm(q, q_norm_w, nh, eps), rope_cos[rows], rope_sin[rows])
    kn = rope(head_rms_norm(k, k_norm_w, nh, eps), rope_cos, rope_sin)
    valid = None if key_mask is None else np.asarray(key_mask[0]) != 0
    o = attention(qn, kn, v.reshape(S, nh, d), valid).reshape(len(rows), H)
    x1 = gated_residual(xb[rows], gate1, project(o, w_o))
    h2 = modulated_rms_norm(x1, shift2, scale2, eps)
    m = silu_gate(project(h2, w_gu), inter)
    return gated_residual(x1, gate2, project(m, w_d))


def block_forward_inputs(inp, eps=None) -> Dict[str, np.ndarray]:
    """block_forward on a mi_synth.BlockInputs (bf16 bits widened here)."""
    g = inp.geom
    w = inp.weights
    return block_forward(widen(inp.x), widen(inp.mod), widen(w.w_qkv), widen(w.w_o), widen(w.w_gu),
                         widen(w.w_d), widen(w.q_norm_w), widen(w.k_norm_w),
                         inp.rope_cos.astype(np.float64), inp.rope_sin.astype(np.float64),
                         inp.key_mask, g.n_heads, g.eps if eps is None else eps)


def plain_prenorm_block(x, w_qkv, w_o, w_gu, w_d, q_norm_w, k_norm_w, rope_cos, rope_sin,
                        n_heads, eps=EPS_DEFAULT):
    """A pre-norm transformer block with no modulation, written on its own (batch 1, [S, H]).

    y = x1 + MLP(RMSNorm(x1)),  x1 = x + Attn(RMSNorm(x)).  Used to pin that zero modulation
    (shift = scale = 0, gate = 1) reduces the modulated block to this one."""
    S, H = x.shape
    d = H // n_heads
    inter = w_d.shape[1]

    def norm(t):
        return t / np.sqrt((t ** 2).sum(axis=1, keepdims=True) / t.shape[1] + eps)

    hq = norm(x)
    q = hq @ w_qkv[:H].T
    k = hq @ w_qkv[H:2 * H].T
    v = hq @ w_qkv[2 * H:].T
    att = np.zeros((S, H))
    for hd in range(n_heads):
        sl = slice(hd * d, (hd + 1) * d)
        qh = q[:, sl] / np.sqrt((q[:, sl] ** 2).mean(axis=1, keepdims=True) + eps) * q_norm_w
        kh = k[:, sl] / np.sqrt((k[:, sl] ** 2).mean(axis=1, keepdims=True) + eps) * k_norm_w
        # rotate as complex numbers: (a + ib) * e^{i angle}
        qc = (qh[:, 0::2] + 1j * qh[:, 1::2]) * (rope_cos + 1j * rope_sin)
        kc = (kh[:, 0::2] + 1j * kh[:, 1::2]) * (rope_cos + 1j * rope_sin)
        qr = np.stack([qc.real, qc.imag], axis=-1).reshape(S, d)
        kr = np.stack([kc.real, kc.imag], axis=-1).reshape(S, d)
        sc = qr @ kr.T / np.sqrt(d)
        e = np.exp(sc - sc.max(axis=1, keepdims=True))
        att[:, sl] = (e / e.sum(axis=1, keepdims=True)) @ v[:, sl]
    x1 = x + att @ w_o.T
    h2 = norm(x1)
    g = h2 @ w_gu[:inter].T
    u = h2 @ w_gu[inter:].T
    return x1 + ((g / (1.0 + np.exp(-g))) * u) @ w_d.T


# ----------------------------------------------------------------------------------------------
# the guided denoising step (PR #2281 "What this changes": the pipeline's schedule, noise and CFG;
# PR #1528 "Measured": 50 Euler steps, guidance 3)
# ----------------------------------------------------------------------------------------------
def cfg_combine(v_pos, v_neg, guidance):
    """Classifier-free guidance: v = v_neg + g (v_pos - v_neg)."""
    return v_neg + guidance * (v_pos - v_neg)


def euler_update(latent, v, dt):
    """One explicit Euler step of the flow ODE: x <- x + dt v."""
    return latent + dt * v


def denoise_step(latent, text_rows, w_in, w_out, mod_final, mods, blocks, rope_cos, rope_sin,
                 key_mask, n_heads, dt, guidance, skip_neg=None, eps=EPS_DEFAULT):
    """One guided step, float64 throughout.

    latent [N, C]; text_rows [B, T, H] (B = 2: element 0 the prompt, 1 the negative);
    mods: list of [B, 6, H]; blocks: list of dicts with w_qkv, w_o, w_gu, w_d, q_norm_w, k_norm_w;
    mod_final [B, 2, H] (shift_f, scale_f).  skip_neg: optional bools per block; a True entry
    makes the negative branch bypass that block.  Returns (new latent, v_pos, v_neg).

    u = latent W_in^T; sequence = [text rows; u]; the blocks; velocity =
    (RMSNorm(image rows) (1 + scale_f) + shift_f) W_out^T; guidance; Euler."""
    B, T, H = text_rows.shape
    u = latent @ w_in.T
    x = np.concatenate([text_rows, np.broadcast_to(u, (B,) + u.shape)], axis=1).copy()
    for i, (mod, w) in enumerate(zip(mods, blocks)):
        y = block_forward(x, mod, w["w_qkv"], w["w_o"], w["w_gu"], w["w_d"], w["q_norm_w"],
                          w["k_norm_w"], rope_cos, rope_sin, key_mask, n_heads, eps)["y"]
        if skip_neg is not None and skip_neg[i]:
            y[1] = x[1]
        x = y
    img = x[:, T:, :]
    vel = modulated_rms_norm(img, mod_final[:, 0:1, :], mod_final[:, 1:2, :], eps) @ w_out.T
    v = cfg_combine(vel[0], vel[1], guidance)
    return euler_update(latent, v, dt), vel[0], vel[1]


def step_inputs_widened(si):
    """Widen a mi_synth.StepInputs into the float64 arguments of denoise_step."""
    blocks = [dict(w_qkv=widen(b.w_qkv), w_o=widen(b.w_o), w_gu=widen(b.w_gu), w_d=widen(b.w_d),
                   q_norm_w=widen(b.q_norm_w), k_norm_w=widen(b.k_norm_w)) for b in si.blocks]
    return dict(latent=widen(si.latent), text_rows=widen(si.text_rows), w_in=widen(si.w_in),
                w_out=widen(si.w_out), mod_final=widen(si.mod_final),
                mods=[widen(m) for m in si.mods], blocks=blocks,
                rope_cos=si.rope_cos.astype(np.float64), rope_sin=si.rope_sin.astype(np.float64),
                key_mask=si.key_mask, n_heads=si.geom.n_heads)


def step_inputs_widened_lazy(si):
    """step_inputs_widened, with each block's weights widened only when denoise_step reaches that
    block (a generator), so a many-block full-size step holds one block in float64 at a time."""
    a = step_inputs_widened(_StepBlocksDeferred(si))
    a["blocks"] = (dict(w_qkv=widen(b.w_qkv), w_o=widen(b.w_o), w_gu=widen(b.w_gu), w_d=widen(b.w_d),
                        q_norm_w=widen(b.q_norm_w), k_norm_w=widen(b.k_norm_w)) for b in si.blocks)
    return a


class _StepBlocksDeferred:
    """A view of a mi_synth.StepInputs without its blocks (they are widened lazily)."""

    def __init__(self, si):
        self._si = si
        self.blocks = []

    def __getattr__(self, name):
        return getattr(self._si, name)


# ----------------------------------------------------------------------------------------------
# device-side builders (PR #1528 "What it adds": the config, rotary tables and the timestep's
# modulation are computed by host code shared with the Metal family; here they are computed on
# the device, and these are their definitions)
# ----------------------------------------------------------------------------------------------
def rope_angle_tables(text_pad, grid_h, grid_w, theta=10000.0):
    """cos/sin [S, 64] of the 2-D rotary: pair j < 32 turns by (row position) * theta^(-j/32), pair
    j >= 32 by (column position) * theta^(-(j-32)/32); text row t has position t on both axes,
    image token (r, c) (row-major after the text) has (r, c)."""
    S = text_pad + grid_h * grid_w
    cos = np.empty((S, 64))
    sin = np.empty((S, 64))
    for s in range(S):
        if s < text_pad:
            pa = pb = float(s)
        else:
            pa, pb = divmod(s - text_pad, grid_w)
        for j in range(64):
            pos = pa if j < 32 else pb
            ang = pos * theta ** (-(j % 32) / 32.0)
            cos[s, j] = np.cos(ang)
            sin[s, j] = np.sin(ang)
    return cos, sin


def timestep_embedding(t, dim=256, scale=1000.0, max_period=10000.0):
    """Sinusoidal embedding of scale * t: [cos(scale t f_k) for k < dim/2, sin(scale t f_k) for
    k < dim/2] with f_k = max_period^(-k / (dim/2)).  t: [B] -> [B, dim]."""
    t = np.asarray(t, dtype=np.float64)
    half = dim // 2
    f = max_period ** (-np.arange(half, dtype=np.float64) / half)
    ang = scale * t[:, None] * f[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


def timestep_modulation(t, w_t1, w_t2, w_mod, n_blocks):
    """Modulation of every block and of the final norm from the timestep:
    c = W_t2 silu(W_t1 emb(t)); all = W_mod silu(c) with W_mod [(6 n_blocks + 2) H, H].
    Returns (mods [n_blocks, B, 6, H], mod_final [B, 2, H])."""
    H = w_t2.shape[0]
    c = project(silu(project(timestep_embedding(t, w_t1.shape[1]), w_t1)), w_t2)
    allv = project(silu(c), w_mod)
    B = allv.shape[0]
    mods = allv[:, : 6 * n_blocks * H].reshape(B, n_blocks, 6, H).transpose(1, 0, 2, 3)
    final = allv[:, 6 * n_blocks * H:].reshape(B, 2, H)
    return mods, final


def euler_loop(latent, timesteps, step_fn):
    """Run step_fn(latent, dt) over the schedule's consecutive differences dt_i = t_{i+1} - t_i."""
    x = latent
    for i in range(len(timesteps) - 1):
        x = step_fn(x, timesteps[i + 1] - timesteps[i])
    return x
