"""Seeded synthetic inputs for the diffusion-transformer block.

This module is shared by the oracle (``oracle/``) and the CUDA path (tests and
``bench.py``). It draws random tensors and lays them out; it holds none of the
block's arithmetic. Everything it returns is either raw bf16 bit patterns
(``uint16`` arrays), fp32 rotary tables, or ``uint8`` key masks.

Recipe (one ``numpy.random.default_rng(seed)`` per call, float64 draws, rounded
to bf16 with round-to-nearest-even):

* activations and latents ~ N(0, 1)
* projection weights ~ N(0, 0.02)
* adaLN modulation vectors (shift, scale, gate for attention and MLP) ~ N(0, 0.1)
* q/k RMSNorm gains ~ 1 + N(0, 0.02)

The geometry follows the MOSS-Image transformer pages (TensorFold PR #1528,
"Measured": a 1024x1024 picture with a 34-row prompt and a 1200x880 picture with
a 63-row prompt; PR #2281: an empty negative prompt for guidance).  The rotary
tables are inputs to the block ("the config, rotary tables and the timestep's
modulation are shared", PR #1528 "What it adds"); they are built here by the
reading stated in ``rope_tables``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Tuple

import numpy as np

HEAD_DIM = 128
ROPE_THETA = 10000.0


@dataclass(frozen=True)
class Geometry:
    """One workload: sequence layout plus block dimensions."""

    name: str
    batch: int
    text_pad: int                 # T: text rows per batch element (padded)
    n_text: Tuple[int, ...]       # valid text rows per batch element (<= T)
    grid_h: int
    grid_w: int
    hidden: int
    n_heads: int
    mlp_inter: int
    n_blocks: int = 1
    latent_ch: int = 64
    eps: float = 1e-6
    guidance: float = 3.0
    n_steps: int = 1

    @property
    def head_dim(self) -> int:
        return HEAD_DIM

    @property
    def n_img(self) -> int:
        return self.grid_h * self.grid_w

    @property
    def seq(self) -> int:
        return self.text_pad + self.n_img

    @property
    def rows(self) -> int:
        return self.batch * self.seq


# The workloads.  Names say what they are.
GEOMETRIES: Dict[str, Geometry] = {
    # tiny block the oracle finishes instantly: 10 text rows + 8x8 latent grid
    "tiny_8x8": Geometry("tiny_8x8", 1, 10, (10,), 8, 8, 256, 2, 1024),
    # a small block with several 128-row tiles and a ragged tail (S = 336 = 2*128 + 80)
    "small_ragged_17x19": Geometry("small_ragged_17x19", 1, 13, (13,), 17, 19, 512, 4, 1024),
    # small batch-2 guidance layout: masked padded negative prompt (S = 210)
    "small_cfg_b2": Geometry("small_cfg_b2", 2, 18, (18, 5), 12, 16, 512, 4, 1536),
    # single block at 1024x1024 picture scale: 34 text rows + 64x64 grid
    "block_1024": Geometry("block_1024", 1, 34, (34,), 64, 64, 3072, 24, 8192),
    # single block at 1200x880 (75 wide x 55 high grid), 63 text rows: ragged tiles
    "block_1200x880": Geometry("block_1200x880", 1, 63, (63,), 55, 75, 3072, 24, 8192),
    # small batch-2 layout with a deep MLP (I = 8448): its down projection has 4 row tiles of
    # 132 k-blocks, fewer tiles than SMs, which the GEMM spreads along k (its stream-K tail)
    "small_cfg_b2_streamk": Geometry("small_cfg_b2_streamk", 2, 18, (18, 5), 12, 16, 256, 2, 8448),
    # the guided step's block on its own (batch 2: prompt 34 rows, negative 10 rows padded to 34)
    "block_1024_cfg_b2": Geometry("block_1024_cfg_b2", 2, 34, (34, 10), 64, 64, 3072, 24, 8192),
    # long sequence: 128x128 grid (about 2048x2048 picture) + 34 text rows
    "block_2048": Geometry("block_2048", 1, 34, (34,), 128, 128, 3072, 24, 8192),
    # one guided denoising step: 24 blocks, batch 2 (prompt 34 rows; empty negative 10 rows padded)
    "step_1024_cfg": Geometry("step_1024_cfg", 2, 34, (34, 10), 64, 64, 3072, 24, 8192, n_blocks=24),
    # the same step at the tiny block geometry (24 blocks) for whole-step parity
    "step_tiny_cfg": Geometry("step_tiny_cfg", 2, 10, (10, 4), 8, 8, 256, 2, 1024, n_blocks=24),
    # 50 guided Euler steps of the tiny step (loop parity)
    "loop_tiny_cfg50": Geometry("loop_tiny_cfg50", 2, 10, (10, 4), 8, 8, 256, 2, 1024,
                                n_blocks=24, n_steps=50),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float64/float32 values to bf16 (round to nearest even) and return the uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    # round to nearest even on the 16 dropped bits; NaN never occurs in these draws
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def rope_tables(g: Geometry) -> Tuple[np.ndarray, np.ndarray]:
    """cos/sin tables, fp32 [S, 64], shared by every batch element.

    Reading (the pages only say "2-D rotary over (row, col) for image tokens and
    1-D positions for text"): theta = 10000, omega_j = theta^(-j/32) for
    j in [0, 32); rotary pair p in [0, 32) carries the row axis and pair
    p in [32, 64) the column axis.  Text row t uses position t on both halves;
    image token (r, c) uses r on the first half and c on the second.  Positions
    start at 0.  Angles are formed in float64 and stored as fp32.
    """
    j = np.arange(32, dtype=np.float64)
    omega = ROPE_THETA ** (-j / 32.0)
    pos_a = np.empty(g.seq, dtype=np.float64)
    pos_b = np.empty(g.seq, dtype=np.float64)
    t = np.arange(g.text_pad, dtype=np.float64)
    pos_a[: g.text_pad] = t
    pos_b[: g.text_pad] = t
    r, c = np.meshgrid(np.arange(g.grid_h), np.arange(g.grid_w), indexing="ij")
    pos_a[g.text_pad:] = r.reshape(-1)
    pos_b[g.text_pad:] = c.reshape(-1)
    ang = np.concatenate([pos_a[:, None] * omega[None, :], pos_b[:, None] * omega[None, :]], axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def key_mask(g: Geometry) -> np.ndarray:
    """uint8 [B, S]: 1 for a key row that attention may read, 0 for a padded text row.

    Padded rows sit at the end of each element's text segment."""
    m = np.ones((g.batch, g.seq), dtype=np.uint8)
    for b, nt in enumerate(g.n_text):
        m[b, nt: g.text_pad] = 0
    return m


@dataclass
class BlockWeights:
    w_qkv: np.ndarray   # bf16 bits [3H, H] (q rows, then k rows, then v rows)
    w_o: np.ndarray     # bf16 bits [H, H]
    w_gu: np.ndarray    # bf16 bits [2I, H] (gate rows, then up rows)
    w_d: np.ndarray     # bf16 bits [H, I]
    q_norm_w: np.ndarray  # bf16 bits [128]
    k_norm_w: np.ndarray  # bf16 bits [128]


@dataclass
class BlockInputs:
    geom: Geometry
    x: np.ndarray          # bf16 bits [B, S, H]
    mod: np.ndarray        # bf16 bits [B, 6, H]: shift1, scale1, gate1, shift2, scale2, gate2
    weights: BlockWeights
    rope_cos: np.ndarray   # fp32 [S, 64]
    rope_sin: np.ndarray   # fp32 [S, 64]
    key_mask: np.ndarray   # uint8 [B, S]


def _normal(rng, shape, std, mean=0.0):
    return rng.standard_normal(shape) * std + mean


def _draw_weights(rng, g: Geometry) -> BlockWeights:
    H, I = g.hidden, g.mlp_inter
    return BlockWeights(
        w_qkv=bf16_bits(_normal(rng, (3 * H, H), 0.02)),
        w_o=bf16_bits(_normal(rng, (H, H), 0.02)),
        w_gu=bf16_bits(_normal(rng, (2 * I, H), 0.02)),
        w_d=bf16_bits(_normal(rng, (H, I), 0.02)),
        q_norm_w=bf16_bits(_normal(rng, (HEAD_DIM,), 0.02, 1.0)),
        k_norm_w=bf16_bits(_normal(rng, (HEAD_DIM,), 0.02, 1.0)),
    )


def block_inputs(g: Geometry, seed: int = 0) -> BlockInputs:
    """Inputs of one block forward, drawn in the order x, mod, W_qkv, W_o, W_gu, W_d, w_q, w_k."""
    rng = np.random.default_rng(seed)
    B, S, H = g.batch, g.seq, g.hidden
    x = bf16_bits(_normal(rng, (B, S, H), 1.0))
    mod = bf16_bits(_normal(rng, (B, 6, H), 0.1))
    w = _draw_weights(rng, g)
    cos, sin = rope_tables(g)
    return BlockInputs(g, x, mod, w, cos, sin, key_mask(g))


@dataclass
class StepInputs:
    """Inputs of one guided denoising step (every block, the embedders, the latent)."""

    geom: Geometry
    latent: np.ndarray       # bf16 bits [N, C]
    text_rows: np.ndarray    # bf16 bits [B, T, H] (padded rows are drawn too; they are masked)
    w_in: np.ndarray         # bf16 bits [H, C]
    w_out: np.ndarray        # bf16 bits [C, H]
    mod_final: np.ndarray    # bf16 bits [B, 2, H]: shift_f, scale_f
    mods: list = field(default_factory=list)      # per block bf16 bits [B, 6, H]
    blocks: list = field(default_factory=list)    # per block BlockWeights
    rope_cos: np.ndarray = None
    rope_sin: np.ndarray = None
    key_mask: np.ndarray = None


def step_inputs(g: Geometry, seed: int = 0) -> StepInputs:
    """Inputs of a guided step, drawn in the order: per block (mod, W_qkv, W_o, W_gu, W_d, w_q, w_k),
    then W_in, W_out, mod_final, latent, text rows.

    The modulation is a function of the timestep alone, so both guidance branches get the same
    vectors: one [6, H] draw per block, repeated over the batch.  It is held fixed across steps."""
    rng = np.random.default_rng(seed)
    B, H, C = g.batch, g.hidden, g.latent_ch
    mods, blocks = [], []
    for _ in range(g.n_blocks):
        m = bf16_bits(_normal(rng, (1, 6, H), 0.1))
        mods.append(np.repeat(m, B, axis=0))
        blocks.append(_draw_weights(rng, g))
    w_in = bf16_bits(_normal(rng, (H, C), 0.02))
    w_out = bf16_bits(_normal(rng, (C, H), 0.02))
    mf = bf16_bits(_normal(rng, (1, 2, H), 0.1))
    mod_final = np.repeat(mf, B, axis=0)
    latent = bf16_bits(_normal(rng, (g.n_img, C), 1.0))
    text = bf16_bits(_normal(rng, (B, g.text_pad, H), 1.0))
    cos, sin = rope_tables(g)
    return StepInputs(g, latent, text, w_in, w_out, mod_final, mods, blocks, cos, sin, key_mask(g))


def euler_schedule(n_steps: int) -> np.ndarray:
    """Timesteps t_i = 1 - i/n for i = 0..n (linear in [1, 0]); step i moves by t_{i+1} - t_i."""
    return 1.0 - np.arange(n_steps + 1, dtype=np.float64) / n_steps


@dataclass
class TimestepWeights:
    """Weights of the timestep -> modulation path: W_t1 [H, 256], W_t2 [H, H] and the stacked
    projection W_mod [(6 n_blocks + 2) H, H], all ~ N(0, 0.02) (bf16 bits)."""

    w_t1: np.ndarray
    w_t2: np.ndarray
    w_mod: np.ndarray


def timestep_weights(g: Geometry, seed: int = 0) -> TimestepWeights:
    rng = np.random.default_rng(seed)
    H = g.hidden
    return TimestepWeights(bf16_bits(_normal(rng, (H, 256), 0.02)), bf16_bits(_normal(rng, (H, H), 0.02)),
                           bf16_bits(_normal(rng, ((6 * g.n_blocks + 2) * H, H), 0.02)))
