"""Per-kernel parity through the C ABI against the float64 oracle's step functions.

Each kernel gets seeded bf16 inputs; the oracle gets the same bits widened exactly.  Sizes span
several 128-row tiles with ragged tails; the largest cases use the 1024x1024 block's shapes and
check sampled rows that the oracle computes one by one."""
import numpy as np
import pytest
import torch

import mi_synth
from oracle import mi_oracle as O
from tests._gpu import (assert_parity, bf16_to_bits, require_gpu, to_dev, to_dev_bf16, to_f64)

pytestmark = pytest.mark.gpu
BF = torch.bfloat16


def _bits(rng, shape, std=1.0, mean=0.0):
    return mi_synth.bf16_bits(rng.standard_normal(shape) * std + mean)


# ------------------------------------------------------------------------------ GEMM
@pytest.mark.parametrize("m,n,k", [(128, 256, 64), (333, 768, 256), (1, 512, 128), (300, 200, 192),
                                   (4130, 9216, 3072), (4130, 3072, 8192)])
def test_gemm_parity(m, n, k):
    mi = require_gpu()
    rng = np.random.default_rng(m * 7 + n * 3 + k)
    a = _bits(rng, (m, k))
    w = _bits(rng, (n, k), 0.02)
    c = torch.empty(m, n, dtype=BF, device="cuda")
    mi.gemm(to_dev_bf16(a), to_dev_bf16(w), c)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    rows = np.arange(m) if m * n * k < 2e9 else np.unique(np.r_[0:64, m - 64:m, rng.integers(0, m, 128)])
    ref = O.project(O.widen(a[rows]), O.widen(w))
    got = to_f64(c)[rows]
    assert_parity(got, ref, f"gemm {m}x{n}x{k}")
    # each output is one bf16 rounding of an fp32 sum: well inside 1% of the row scale
    scale = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(got - ref) <= 1e-2 * np.abs(ref) + 2e-3 * scale)


def test_gemm_one_hot_is_exact():
    mi = require_gpu()
    rng = np.random.default_rng(5)
    m, n, k = 200, 512, 256
    a = _bits(rng, (m, k))
    perm = rng.integers(0, k, size=n)
    w = np.zeros((n, k))
    w[np.arange(n), perm] = 1.0
    c = torch.empty(m, n, dtype=BF, device="cuda")
    mi.gemm(to_dev_bf16(a), to_dev_bf16(mi_synth.bf16_bits(w)), c)
    assert np.array_equal(bf16_to_bits(c), a[:, perm])


def test_gemm_repeats_bit_for_bit():
    mi = require_gpu()
    rng = np.random.default_rng(6)
    a = to_dev_bf16(_bits(rng, (1000, 1024)))
    w = to_dev_bf16(_bits(rng, (2048, 1024), 0.02))
    c1 = torch.empty(1000, 2048, dtype=BF, device="cuda")
    c2 = torch.empty_like(c1)
    mi.gemm(a, w, c1)
    mi.gemm(a[:500].contiguous(), w, c2[:500])
    mi.gemm(a, w, c2)
    assert torch.equal(c1.view(torch.int16), c2.view(torch.int16))


@pytest.mark.parametrize("m,n,k,seq", [(336, 512, 512, 336), (420, 256, 1024, 210)])
def test_fused_gated_residual_matches_unfused_bytes(m, n, k, seq):
    mi = require_gpu()
    rng = np.random.default_rng(m + n)
    a = to_dev_bf16(_bits(rng, (m, k)))
    w = to_dev_bf16(_bits(rng, (n, k), 0.02))
    x = to_dev_bf16(_bits(rng, (m, n)))
    mod = to_dev_bf16(_bits(rng, (m // seq, 6, n), 0.1))
    c = torch.empty(m, n, dtype=BF, device="cuda")
    out1 = torch.empty_like(c)
    out2 = torch.empty_like(c)
    mi.gemm(a, w, c)
    mi.gated_add(x, c, mod, 2, out1, m // seq, seq)
    mi.gemm_gated_residual(a, w, x, mod, 2, out2, seq)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))
    ref = O.gated_residual(to_f64(x).reshape(m // seq, seq, n), to_f64(mod)[:, 2:3, :],
                           O.project(to_f64(a), to_f64(w)).reshape(m // seq, seq, n))
    assert_parity(to_f64(out2).reshape(ref.shape), ref, "gemm+gated residual")


@pytest.mark.parametrize("m,inter,k", [(336, 1024, 512), (74, 256, 256)])
def test_fused_silu_gate_matches_unfused_bytes(m, inter, k):
    mi = require_gpu()
    rng = np.random.default_rng(m + inter)
    a = to_dev_bf16(_bits(rng, (m, k)))
    w = to_dev_bf16(_bits(rng, (2 * inter, k), 0.05))
    gu = torch.empty(m, 2 * inter, dtype=BF, device="cuda")
    m1 = torch.empty(m, inter, dtype=BF, device="cuda")
    m2 = torch.empty_like(m1)
    mi.gemm(a, w, gu)
    mi.silu_gate(gu, m1)
    mi.gemm_silu_gate(a, w, m2)
    assert torch.equal(m1.view(torch.int16), m2.view(torch.int16))
    ref = O.silu_gate(O.project(to_f64(a), to_f64(w)), inter)
    assert_parity(to_f64(m2), ref, "gemm+silu gate")


def test_gemm_rows_do_not_depend_on_the_launch():
    """A row's result does not depend on the launch it is computed in: 4130 rows in one launch (CTA
    pairs, the last 256-row pair tile holding 34 rows) give the bytes of two launches over rows
    0-4095 (CTA pairs, no ragged tile) and 4096-4129 (34 rows: the one-CTA kernel), and sampled
    rows on both sides of the boundary match the oracle.  Both pair launches end in a partial wave
    that runs as half-width tiles (the last 24 of 1088 tiles, and the last 36 of 1024), on
    different tiles, so the half-width tiles are checked against whole ones too."""
    mi = require_gpu()
    m, inter, k, top_rows = 4130, 8192, 3072, 4096
    rng = np.random.default_rng(4130)
    a = to_dev_bf16(_bits(rng, (m, k)))
    w = to_dev_bf16(_bits(rng, (2 * inter, k), 0.05))
    full = torch.empty(m, inter, dtype=BF, device="cuda")
    top = torch.empty(top_rows, inter, dtype=BF, device="cuda")
    bottom = torch.empty(m - top_rows, inter, dtype=BF, device="cuda")
    mi.gemm_silu_gate(a, w, full)
    mi.gemm_silu_gate(a[:top_rows].contiguous(), w, top)
    mi.gemm_silu_gate(a[top_rows:].contiguous(), w, bottom)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    assert torch.equal(full[:top_rows].view(torch.int16), top.view(torch.int16))
    assert torch.equal(full[top_rows:].view(torch.int16), bottom.view(torch.int16))
    rows = np.r_[0:4, top_rows - 6:top_rows + 6, m - 4:m]
    ref = O.silu_gate(O.project(to_f64(a)[rows], to_f64(w)), inter)
    assert_parity(to_f64(full)[rows], ref, "gemm+silu gate, rows across launches")


@pytest.mark.parametrize("batch,seq,heads", [(1, 74, 2), (2, 210, 4), (1, 4130, 24)])
def test_fused_qkv_rope_matches_unfused_bytes(batch, seq, heads):
    mi = require_gpu()
    H = heads * 128
    rng = np.random.default_rng(seq + 17 * heads)
    h = to_dev_bf16(_bits(rng, (batch * seq, H)))
    w = to_dev_bf16(_bits(rng, (3 * H, H), 0.02))
    wq = to_dev_bf16(_bits(rng, (128,), 0.02, 1.0))
    wk = to_dev_bf16(_bits(rng, (128,), 0.02, 1.0))
    g = mi_synth.Geometry("t", batch, 10, (10,) * batch, 1, seq - 10, H, heads, 256)
    cos, sin = mi_synth.rope_tables(g)
    cos, sin = to_dev(cos), to_dev(sin)
    qkv = torch.empty(batch * seq, 3 * H, dtype=BF, device="cuda")
    qp1 = torch.empty(batch, heads, seq, 128, dtype=BF, device="cuda")
    kp1 = torch.empty_like(qp1)
    mi.gemm(h, w, qkv)
    mi.qk_norm_rope(qkv, wq, wk, cos, sin, qp1, kp1, batch, seq, heads)
    qkv2 = torch.zeros_like(qkv)
    qp2 = torch.empty_like(qp1)
    kp2 = torch.empty_like(qp1)
    mi.gemm_qkv_rope(h, w, wq, wk, cos, sin, qp2, kp2, qkv2, batch, seq, heads)
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    assert torch.equal(qp1.view(torch.int16), qp2.view(torch.int16))
    assert torch.equal(kp1.view(torch.int16), kp2.view(torch.int16))
    assert torch.equal(qkv[:, 2 * H:].contiguous().view(torch.int16), qkv2[:, 2 * H:].contiguous().view(torch.int16))
    assert not qkv2[:, :2 * H].any()  # q/k columns are not written


# ------------------------------------------------------------------------------ element-wise
@pytest.mark.parametrize("batch,seq,hidden", [(1, 74, 256), (2, 210, 512), (1, 4130, 3072)])
def test_mod_rmsnorm_parity(batch, seq, hidden):
    mi = require_gpu()
    rng = np.random.default_rng(seq)
    x = _bits(rng, (batch, seq, hidden), 1.5)
    mod = _bits(rng, (batch, 6, hidden), 0.1)
    out = torch.empty(batch * seq, hidden, dtype=BF, device="cuda")
    mi.mod_rmsnorm(to_dev_bf16(x).view(batch * seq, hidden), to_dev_bf16(mod), 3, 4, out, batch, seq)
    xf, mf = O.widen(x), O.widen(mod)
    ref = np.stack([O.modulated_rms_norm(xf[b], mf[b, 3], mf[b, 4]) for b in range(batch)])
    assert_parity(to_f64(out).reshape(ref.shape), ref, "mod_rmsnorm")


@pytest.mark.parametrize("batch,seq,heads", [(1, 74, 2), (2, 210, 4), (1, 4130, 24)])
def test_qk_norm_rope_parity(batch, seq, heads):
    mi = require_gpu()
    H = heads * 128
    rng = np.random.default_rng(seq + heads)
    qkv = _bits(rng, (batch * seq, 3 * H), 1.1)
    wq = _bits(rng, (128,), 0.02, 1.0)
    wk = _bits(rng, (128,), 0.02, 1.0)
    g = mi_synth.Geometry("t", batch, 10, (10,) * batch, 1, seq - 10, H, heads, 256)
    cos, sin = mi_synth.rope_tables(g)
    qp = torch.empty(batch, heads, seq, 128, dtype=BF, device="cuda")
    kp = torch.empty_like(qp)
    mi.qk_norm_rope(to_dev_bf16(qkv), to_dev_bf16(wq), to_dev_bf16(wk), to_dev(cos), to_dev(sin), qp, kp, batch,
                    seq, heads)
    f = O.widen(qkv).reshape(batch, seq, 3 * H)
    c64, s64 = cos.astype(np.float64), sin.astype(np.float64)
    for b in range(batch):
        rq = O.rope(O.head_rms_norm(f[b, :, :H], O.widen(wq), heads), c64, s64)
        rk = O.rope(O.head_rms_norm(f[b, :, H:2 * H], O.widen(wk), heads), c64, s64)
        assert_parity(to_f64(qp[b]), rq.transpose(1, 0, 2), "q")
        assert_parity(to_f64(kp[b]), rk.transpose(1, 0, 2), "k")


def test_gated_add_and_silu_gate_parity():
    mi = require_gpu()
    rng = np.random.default_rng(11)
    batch, seq, hidden, inter = 2, 210, 512, 1024
    x = _bits(rng, (batch * seq, hidden))
    y = _bits(rng, (batch * seq, hidden))
    mod = _bits(rng, (batch, 6, hidden), 0.1)
    out = torch.empty(batch * seq, hidden, dtype=BF, device="cuda")
    mi.gated_add(to_dev_bf16(x), to_dev_bf16(y), to_dev_bf16(mod), 5, out, batch, seq)
    mf = O.widen(mod)
    ref = O.gated_residual(O.widen(x).reshape(batch, seq, hidden), mf[:, 5:6, :], O.widen(y).reshape(batch, seq, hidden))
    assert_parity(to_f64(out).reshape(ref.shape), ref, "gated_add")
    gu = _bits(rng, (batch * seq, 2 * inter), 2.0)
    m = torch.empty(batch * seq, inter, dtype=BF, device="cuda")
    mi.silu_gate(to_dev_bf16(gu), m)
    assert_parity(to_f64(m), O.silu_gate(O.widen(gu), inter), "silu_gate")


def test_gated_add_zero_gate_is_identity():
    mi = require_gpu()
    rng = np.random.default_rng(12)
    x = _bits(rng, (300, 256))
    y = _bits(rng, (300, 256), 100.0)
    mod = np.zeros((1, 6, 256), dtype=np.uint16)
    out = torch.empty(300, 256, dtype=BF, device="cuda")
    mi.gated_add(to_dev_bf16(x), to_dev_bf16(y), to_dev_bf16(mod), 2, out, 1, 300)
    assert np.array_equal(bf16_to_bits(out), x)


# ------------------------------------------------------------------------------ attention
def _attn_inputs(rng, batch, seq, heads, q_std=1.0):
    H = heads * 128
    qp = _bits(rng, (batch, heads, seq, 128), q_std)
    kp = _bits(rng, (batch, heads, seq, 128))
    qkv = _bits(rng, (batch * seq, 3 * H), 1.1)
    return qp, kp, qkv


def _attn_ref(qp, kp, qkv, mask, b, heads, rows=None):
    H = heads * 128
    seq = qp.shape[2]
    q = O.widen(qp[b]).transpose(1, 0, 2)
    k = O.widen(kp[b]).transpose(1, 0, 2)
    v = O.widen(qkv).reshape(-1, seq, 3 * H)[b, :, 2 * H:].reshape(seq, heads, 128)
    if rows is not None:
        q = q[rows]
    valid = None if mask is None else mask[b] != 0
    return O.attention(q, k, v, valid).reshape(q.shape[0], H)


def _attn_ws(mi, batch, seq, heads, split):
    """The split schedule's workspace (None: one CTA per query-tile pair)."""
    if not split:
        return None
    return torch.empty(mi.attention_workspace_size(batch, seq, heads), dtype=torch.uint8, device="cuda")


@pytest.mark.parametrize("split", [False, True], ids=["unit_per_cta", "split_per_sm"])
@pytest.mark.parametrize("batch,seq,heads,masked,q_std", [
    (1, 74, 2, False, 1.0), (1, 336, 4, False, 1.0), (2, 210, 4, True, 1.0), (1, 300, 2, False, 4.0),
    (1, 128, 2, False, 1.0), (1, 1, 2, False, 1.0), (1, 4130, 24, False, 1.0), (1, 4188, 24, True, 1.0),
    (2, 1000, 40, True, 1.0)])
def test_attention_parity(batch, seq, heads, masked, q_std, split):
    # (2, 1000, 40): 320 query-tile pairs on the split schedule, whose CTA boundaries fall inside
    # pairs of both batch elements (the key mask is rebuilt when a CTA moves to the second)
    mi = require_gpu()
    rng = np.random.default_rng(seq * 13 + heads)
    qp, kp, qkv = _attn_inputs(rng, batch, seq, heads, q_std)
    mask = None
    if masked:
        mask = np.ones((batch, seq), dtype=np.uint8)
        mask[:, 5:20] = 0
        mask[-1, 100:140] = 0
    o = torch.empty(batch * seq, heads * 128, dtype=BF, device="cuda")
    mi.attention(to_dev_bf16(qp), to_dev_bf16(kp), to_dev_bf16(qkv), None if mask is None else to_dev(mask), o,
                 batch, seq, heads, ws=_attn_ws(mi, batch, seq, heads, split))
    torch.cuda.synchronize()
    assert mi.device_error() == 0
    got = to_f64(o).reshape(batch, seq, -1)
    for b in range(batch):
        rows = None if seq <= 1024 else np.unique(np.r_[0:40, seq - 40:seq, rng.integers(0, seq, 100)])
        ref = _attn_ref(qp, kp, qkv, mask, b, heads, rows)
        assert_parity(got[b] if rows is None else got[b][rows], ref, f"attention b={b}")


def test_attention_split_parts_repeat_and_agree():
    """The split schedule at the 1024x1024 block's shape (408 query-tile pairs on one CTA per SM):
    repeats bit for bit, agrees with the one-CTA-per-pair schedule within the bar (the two add
    partial sums in different places), and a key mask covering the first half of the keys leaves
    some split parts with no valid key at all (their weight in the combination is zero)."""
    mi = require_gpu()
    rng = np.random.default_rng(77)
    batch, seq, heads = 1, 4130, 24
    qp, kp, qkv = (to_dev_bf16(a) for a in _attn_inputs(rng, batch, seq, heads))
    ws = _attn_ws(mi, batch, seq, heads, True)
    assert ws.numel() > 0
    outs = []
    for masked in (False, True):
        mask = np.ones((batch, seq), dtype=np.uint8)
        if masked:
            mask[:, :2048] = 0
        m = to_dev(mask)
        o1 = torch.empty(batch * seq, heads * 128, dtype=BF, device="cuda")
        o2 = torch.empty_like(o1)
        o3 = torch.empty_like(o1)
        mi.attention(qp, kp, qkv, m, o1, batch, seq, heads, ws=ws)
        mi.attention(qp, kp, qkv, m, o2, batch, seq, heads, ws=ws)
        mi.attention(qp, kp, qkv, m, o3, batch, seq, heads)
        torch.cuda.synchronize()
        assert mi.device_error() == 0
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
        assert_parity(to_f64(o1), to_f64(o3), f"split against unsplit schedule, masked={masked}")
        outs.append((mask, o1))
    mask, o = outs[1]
    rows = np.unique(np.r_[0:20, seq - 20:seq, rng.integers(0, seq, 60)])
    ref = _attn_ref(*(bf16_to_bits(t) for t in (qp, kp, qkv)), mask, 0, heads, rows)
    assert_parity(to_f64(o)[rows], ref, "split schedule, first half of the keys masked")


def test_attention_long_sequence_reads_the_mask_per_tile():
    """Past 65536 keys the key-validity bitmask no longer fits in shared memory and every key tile
    takes its validity from the mask in global memory: parity on sampled rows, with masked keys
    on both sides of key 65536 and in the ragged last tile."""
    mi = require_gpu()
    batch, seq, heads = 1, 66000, 1
    rng = np.random.default_rng(66000)
    qp, kp, qkv = _attn_inputs(rng, batch, seq, heads)
    mask = np.ones((batch, seq), dtype=np.uint8)
    mask[:, 3:40] = 0
    mask[:, 65500:65600] = 0
    mask[:, 65950:65990] = 0
    for split in (False, True):  # 258 query-tile pairs: the split schedule cuts pairs of 516 key tiles
        o = torch.empty(batch * seq, heads * 128, dtype=BF, device="cuda")
        mi.attention(to_dev_bf16(qp), to_dev_bf16(kp), to_dev_bf16(qkv), to_dev(mask), o, batch, seq, heads,
                     ws=_attn_ws(mi, batch, seq, heads, split))
        torch.cuda.synchronize()
        assert mi.device_error() == 0
        got = to_f64(o).reshape(batch, seq, -1)
        rows = np.unique(np.r_[0:16, 65520:65540, seq - 16:seq, rng.integers(0, seq, 24)])
        assert_parity(got[0][rows], _attn_ref(qp, kp, qkv, mask, 0, heads, rows), f"attention, 66000 keys, split={split}")


def test_attention_equal_scores_cancel():
    # q = 0: every valid key weighs the same; V rows of +-2^10 cancel (the pages' adversarial gate)
    mi = require_gpu()
    batch, seq, heads = 1, 300, 2
    rng = np.random.default_rng(21)
    qp = np.zeros((batch, heads, seq, 128), dtype=np.uint16)
    kp = _bits(rng, (batch, heads, seq, 128))
    H = heads * 128
    v = np.zeros((seq, 3 * H))
    v[0::2, 2 * H:] = 1024.0
    v[1::2, 2 * H:] = -1024.0
    v[:, 2 * H + 7] += np.arange(seq) % 16
    qkv = mi_synth.bf16_bits(v)
    mask = np.ones((batch, seq), dtype=np.uint8)
    mask[0, -1] = 0
    mask[0, -2] = 0
    o = torch.empty(seq, H, dtype=BF, device="cuda")
    mi.attention(to_dev_bf16(qp), to_dev_bf16(kp), to_dev_bf16(qkv), to_dev(mask), o, batch, seq, heads)
    ref = _attn_ref(qp, kp, qkv, mask, 0, heads)
    got = to_f64(o)
    assert np.allclose(got[:, 0], 0.0, atol=1e-6)
    assert np.allclose(got[:, 7], ref[:, 7], rtol=1e-2)


def test_attention_masked_keys_carry_nothing():
    mi = require_gpu()
    batch, seq, heads = 2, 200, 2
    rng = np.random.default_rng(22)
    qp, kp, qkv = _attn_inputs(rng, batch, seq, heads)
    mask = np.ones((batch, seq), dtype=np.uint8)
    mask[:, 3:30] = 0
    H = heads * 128
    big = qkv.copy().reshape(batch, seq, 3 * H)
    big[:, 3:30, 2 * H:] = mi_synth.bf16_bits(np.full((batch, 27, H), 3.0e30))
    kbig = kp.copy()
    kbig[:, :, 3:30, :] = mi_synth.bf16_bits(np.full((batch, heads, 27, 128), 1.0e4))
    o1 = torch.empty(batch * seq, H, dtype=BF, device="cuda")
    o2 = torch.empty_like(o1)
    m = to_dev(mask)
    mi.attention(to_dev_bf16(qp), to_dev_bf16(kp), to_dev_bf16(qkv), m, o1, batch, seq, heads)
    mi.attention(to_dev_bf16(qp), to_dev_bf16(kbig), to_dev_bf16(big.reshape(batch * seq, 3 * H)), m, o2, batch,
                 seq, heads)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("batch,seq,heads", [(2, 150, 2), (2, 700, 48)], ids=["unit_per_cta", "split_per_sm"])
def test_attention_all_keys_masked_gives_zero(batch, seq, heads):
    # (2, 700, 48): 288 query-tile pairs on the split schedule; the pairs of the masked element
    # that are split have two parts with no valid key
    mi = require_gpu()
    rng = np.random.default_rng(23)
    qp, kp, qkv = _attn_inputs(rng, batch, seq, heads)
    mask = np.ones((batch, seq), dtype=np.uint8)
    mask[1, :] = 0
    o = torch.empty(batch * seq, heads * 128, dtype=BF, device="cuda")
    mi.attention(to_dev_bf16(qp), to_dev_bf16(kp), to_dev_bf16(qkv), to_dev(mask), o, batch, seq, heads,
                 ws=_attn_ws(mi, batch, seq, heads, heads > 2))
    got = to_f64(o).reshape(batch, seq, -1)
    assert np.all(got[1] == 0.0)
    assert_parity(got[0], _attn_ref(qp, kp, qkv, mask, 0, heads), "attention b=0")
