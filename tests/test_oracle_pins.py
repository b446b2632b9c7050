"""Pins for the CPU oracle: each test checks it against something other than itself
(hand-worked examples, closed forms, brute force, library routines, invariants the
pages state).  No GPU is needed."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from ternary_weight_moe_02_b300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f32_bits_to_bf16_bits(values):
    a = np.asarray(values, dtype=np.float32)
    bits = a.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "fixture values must be bf16-exact"
    return (bits >> 16).astype(np.uint16)


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([p.strip() for p in line.split("|")])
    return rows


# ---------------------------------------------------------------- pack / unpack

def test_pack_golden_examples():
    """Hand-computed bytes ("The 5.31 GB claim reconciles": 5 trits per byte)."""
    for K, trits, expected in _read_fixture("pack_examples.txt"):
        K = int(K)
        q = np.array([int(v) for v in trits.split()], dtype=np.int8).reshape(1, K)
        want = np.array([int(v) for v in expected.split()], dtype=np.uint8)
        got = oracle.pack(q)
        assert got.shape == (1, (K + 4) // 5)
        np.testing.assert_array_equal(got[0], want)
        np.testing.assert_array_equal(oracle.unpack(got, K), q)


def test_pack_is_a_bijection_onto_243_codes():
    """All 3^5 trit patterns map to distinct codes 0..242 and back; 243 <= 256."""
    patterns = np.array(list(itertools.product((-1, 0, 1), repeat=5)), dtype=np.int8)
    assert patterns.shape == (243, 5) and 3 ** 5 == 243 <= 256
    codes = oracle.pack(patterns)[:, 0]
    assert sorted(codes.tolist()) == list(range(243))
    # brute force of the digit rule: code = sum (q_i + 1) 3^i
    brute = [sum((int(t) + 1) * 3 ** i for i, t in enumerate(p)) for p in patterns]
    assert codes.tolist() == brute
    np.testing.assert_array_equal(oracle.unpack(codes.reshape(243, 1), 5), patterns)


def test_unpack_rejects_codes_243_to_255():
    for code in range(243, 256):
        q, st = oracle.unpack(np.array([[code]], np.uint8), 5, check=False)
        assert st == oracle.BAD_CODE
    _, st = oracle.unpack(np.array([[242]], np.uint8), 5, check=False)
    assert st == oracle.OK


def test_k_tail_trits_are_zero():
    rng = np.random.default_rng(1)
    for K in (1, 2, 3, 4, 6, 13, 2047):
        q = rng.integers(-1, 2, size=(3, K)).astype(np.int8)
        p = oracle.pack(q)
        full = np.zeros((3, p.shape[1] * 5), np.int8)
        full[:, :K] = q
        np.testing.assert_array_equal(p, oracle.pack(full))
        np.testing.assert_array_equal(oracle.unpack(p, K), q)


# ------------------------------------------------------------ bits per weight

def test_bits_per_weight_and_census():
    """"The 5.31 GB claim reconciles": log2 3 floor, 1.65 bit/weight, census."""
    assert oracle.packed_row_bytes(2048) == 410
    assert oracle.packed_row_bytes(512) == 103
    assert oracle.packed_row_bytes(2045) == 409 and 8 * 409 / 2045 == pytest.approx(1.6)
    floor = math.log2(3)
    assert floor == pytest.approx(1.585, abs=5e-4)
    for K in (2048, 512):
        bits = 8 * oracle.packed_row_bytes(K) / K
        assert floor <= bits < 2.0
    assert 8 * 410 / 2048 == pytest.approx(1.6016, abs=1e-4)
    assert 8 * 103 / 512 == pytest.approx(1.6094, abs=1e-4)
    # one 2048 -> 512 -> 2048 expert: gate + up + down bytes + fp32 row scales
    H, I = 2048, 512
    expert_bytes = 2 * I * oracle.packed_row_bytes(H) + H * oracle.packed_row_bytes(I) + 4 * (2 * I + H)
    assert expert_bytes == 643072
    bits = 8 * expert_bytes / (3 * H * I)
    assert bits == pytest.approx(1.635, abs=1e-3)
    assert abs(bits - 1.65) / 1.65 < 0.01  # the pages' 1.65 within a percent
    # parameter census: bf16 checkpoint bytes / 2 = ternary + full-precision params
    assert 40_428_060_672 / 2 / 1e9 == pytest.approx(19.58 + 0.64, abs=0.01)
    assert 24 * 256 * 3 * H * I <= 19.58e9
    assert (5.31 - 1.27) * 8 / 19.58 == pytest.approx(1.65, abs=0.01)


# ------------------------------------------------------------------ ternarize

def test_ternarize_golden_examples():
    """Hand-worked rows ("The claim, verified from the bytes")."""
    for wtxt, stxt, qtxt in _read_fixture("ternarize_examples.txt"):
        w = [float(v) for v in wtxt.split()]
        bits = _f32_bits_to_bf16_bits(w).reshape(1, -1)
        q, s = oracle.ternarize(bits)
        assert s[0] == np.float32(float(Fraction(stxt)))
        np.testing.assert_array_equal(q[0], [int(v) for v in qtxt.split()])


def test_ternary_exact_golden_examples():
    """Hand-worked already-ternary rows ("The claim, verified from the bytes")."""
    for wtxt, stxt, qtxt, flag in _read_fixture("ternary_exact_examples.txt"):
        w = [float(v) for v in wtxt.split()]
        bits = _f32_bits_to_bf16_bits(w).reshape(1, -1)
        q, s, bad = oracle.ternary_exact(bits)
        assert s[0] == np.float32(float(stxt))
        np.testing.assert_array_equal(q[0], [int(v) for v in qtxt.split()])
        assert bad == int(flag)


def test_ternary_exact_recovers_constructed_rows_and_relates_to_absmean():
    """Rows built as a_r * q_r (q random trits with a random zero share, a a bf16
    magnitude) come back as exactly q and a, none flagged.  Absmean ternarization of
    the same rows gives the same trits and the scale (1 - z_r) a_r, z_r the row's zero
    fraction (mean |w| over a row of a and 0 values)."""
    rng = np.random.default_rng(5)
    rows, K = 64, 517
    q = rng.choice([-1, 0, 1], size=(rows, K), p=[0.3, 0.4, 0.3]).astype(np.int8)
    q[3] = 0                   # an all-zero row: s = 0
    q[4] = 0
    q[4, 100] = -1             # a single nonzero weight
    a = torch.tensor(rng.uniform(0.001, 2.0, rows), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    w = (a[:, None] * q).astype(np.float32)  # products of a bf16 value and +-1 / 0: bf16-exact
    bits = _f32_bits_to_bf16_bits(w.reshape(-1)).reshape(rows, K)
    qe, se, bad = oracle.ternary_exact(bits)
    np.testing.assert_array_equal(qe, q)
    expect_s = np.where(np.any(q != 0, axis=1), a, 0.0).astype(np.float32)
    np.testing.assert_array_equal(se, expect_s)
    assert bad == 0
    np.testing.assert_array_equal(oracle.pack(qe), oracle.pack(q))
    qa, sa = oracle.ternarize(bits)
    np.testing.assert_array_equal(qa, q)
    z = (q == 0).mean(axis=1)
    np.testing.assert_allclose(sa, (1 - z) * expect_s, rtol=1e-6)


def test_ternary_exact_flags_a_row_one_ulp_off():
    """One nonzero magnitude moved by one bf16 ulp makes its row not ternary; sign trits
    and the max scale stay."""
    w = np.array([[0.5, -0.5, 0.0, 0.5], [0.5, -0.5, 0.0, 0.5]], np.float32)
    bits = _f32_bits_to_bf16_bits(w.reshape(-1)).reshape(2, 4)
    bits[1, 3] += 1  # 0.5 -> 0.50390625
    q, s, bad = oracle.ternary_exact(bits)
    assert bad == 1
    np.testing.assert_array_equal(q, [[1, -1, 0, 1], [1, -1, 0, 1]])
    assert s[0] == np.float32(0.5) and s[1] == np.float32(0.50390625)


def test_ternarize_invariants_gaussian():
    """Three symmetric values per row, all present; closed-form scale and zero share."""
    rows, K, std = 256, 2048, 0.02
    w = synth.bf16_normal((rows, K), std, seed=11)
    bits = synth.bf16_bits(w)
    q, s = oracle.ternarize(bits)
    wf = synth.bits_to_float(bits).astype(np.float64)
    for r in range(rows):
        vals = np.unique(q[r].astype(np.float64) * s[r])
        np.testing.assert_array_equal(vals, [-s[r], 0.0, s[r]])
    # s = mean |w| (checked against numpy on the same values)
    np.testing.assert_allclose(s, np.abs(wf).mean(axis=1), rtol=1e-7)
    # scale ~ sigma sqrt(2/pi): per-row sampling sd is sigma sqrt(1-2/pi)/sqrt(K)
    sd = std * math.sqrt(1 - 2 / math.pi) / math.sqrt(K)
    assert np.all(np.abs(s - std * math.sqrt(2 / math.pi)) < 6 * sd)
    assert abs(s.mean() - std * math.sqrt(2 / math.pi)) < 6 * sd / math.sqrt(rows)
    # zero share: P(|z| <= sqrt(2/pi)/2) = 2 Phi(0.3989) - 1 = 0.3101 for Gaussian rows
    closed = math.erf(0.5 * math.sqrt(2 / math.pi) / math.sqrt(2))
    assert closed == pytest.approx(0.3101, abs=1e-4)
    zero_share = (q == 0).mean()
    assert abs(zero_share - closed) < 0.004
    # sign symmetry
    assert abs((q == 1).mean() - (q == -1).mean()) < 0.01


def test_ternarize_zero_share_laplace_rows_in_pages_band():
    """Heavier-tailed rows land in the pages' 38-43% band: 1 - e^-1/2 = 39.3%."""
    w = synth.laplace_bf16((256, 2048), 0.014, seed=3)
    q, s = oracle.ternarize(synth.bf16_bits(w))
    share = (q == 0).mean()
    assert 0.38 <= share <= 0.43
    assert share == pytest.approx(1 - math.exp(-0.5), abs=0.006)


def test_ternarize_is_idempotent_on_trits():
    """A row that is already ternary keeps its trits; its new scale is 1 - zero share."""
    rng = np.random.default_rng(5)
    q0 = rng.integers(-1, 2, size=(32, 517)).astype(np.int8)
    q0[0] = 0  # all-zero row: s = 0, trits 0
    bits = _f32_bits_to_bf16_bits(q0.astype(np.float32))
    q1, s1 = oracle.ternarize(bits.reshape(q0.shape))
    np.testing.assert_array_equal(q1, q0)
    np.testing.assert_array_equal(s1, (q0 != 0).mean(axis=1).astype(np.float32))


# ----------------------------------------------------------------------- route

def test_route_hand_example_ties_go_to_lower_index():
    """logits [0.5, 0.25, 0.5, -1]: ties rank the lower expert first."""
    x = _f32_bits_to_bf16_bits([1.0, 0.0]).reshape(1, 2)
    wr = _f32_bits_to_bf16_bits([0.5, 0, 0.25, 0, 0.5, 0, -1.0, 0]).reshape(4, 2)
    logits, idx, w = oracle.route(x, wr, None, 3)
    np.testing.assert_array_equal(logits[0], [0.5, 0.25, 0.5, -1.0])
    np.testing.assert_array_equal(idx[0], [0, 2, 1])
    e = [1.0, 1.0, math.exp(-0.25)]
    np.testing.assert_allclose(w[0], [v / sum(e) for v in e], rtol=1e-15)
    # a bias moves expert 3 to the top
    logits, idx, w = oracle.route(x, wr, np.array([0.0, 0.0, 0.0, 2.0]), 2)
    np.testing.assert_array_equal(idx[0], [3, 0])
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-0.5)), 1 - 1 / (1 + math.exp(-0.5))],
                               rtol=1e-15)


def test_route_matches_full_sort_and_softmax():
    """Top-8 = first 8 of a full sort of numpy's fp64 logits; weights sum to 1."""
    T, H, E, k = 16, 2048, 256, 8
    x = synth.bf16_bits(synth.tokens(T, H, seed=2))
    wr = synth.bf16_bits(synth.router_weights(E, H, seed=2))
    bias = synth.bias_normal(E, seed=2).double().numpy()
    logits, idx, w = oracle.route(x, wr, bias, k)
    ref = synth.bits_to_float(x).astype(np.float64) @ synth.bits_to_float(wr).astype(np.float64).T + bias
    np.testing.assert_allclose(logits, ref, rtol=1e-12, atol=1e-12)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-ref[t, e], e))[:k]
        assert idx[t].tolist() == order
        z = np.exp(ref[t, order] - ref[t, order[0]])
        np.testing.assert_allclose(w[t], z / z.sum(), rtol=1e-12)
        assert abs(w[t].sum() - 1.0) < 1e-12
        assert np.all(np.diff(w[t]) <= 0)


# ----------------------------------------------------------------------- group

def test_group_matches_brute_force():
    rng = np.random.default_rng(7)
    for T, k, E in ((1, 8, 256), (5, 3, 4), (64, 8, 256), (300, 8, 32)):
        idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        counts, offsets, perm = oracle.group(idx, E)
        flat = idx.reshape(-1)
        want = sorted(range(T * k), key=lambda s: (flat[s], s))
        assert perm.tolist() == want
        assert counts.tolist() == [int((flat == e).sum()) for e in range(E)]
        assert offsets[0] == 0 and offsets[-1] == T * k
        np.testing.assert_array_equal(np.diff(offsets), counts)


# ------------------------------------------------------------------------- FFN

def _silu(z):
    return z / (1.0 + math.exp(-z))


def _hand_case(scale_x=1.0):
    """Two experts, H=5, I=2, k=2; trits chosen by hand (see the closed form below)."""
    H, I, E = 5, 2, 2
    gate_q = np.array([[[1, 0, 0, 0, 0], [0, -1, 0, 0, 1]],
                       [[0, 0, 0, 1, 0], [-1, 0, 0, 0, 0]]], np.int8)
    up_q = np.array([[[0, 0, 1, 0, 0], [1, 1, 1, 1, 1]],
                     [[0, 1, 0, 0, 0], [0, 0, 0, 0, -1]]], np.int8)
    down_q = np.array([[[1, 0], [0, 1], [1, -1], [0, 0], [-1, -1]],
                       [[0, 1], [1, 0], [0, 0], [1, 1], [-1, 0]]], np.int8)
    s_gate = np.array([[0.5, 1.0], [0.25, 2.0]], np.float32)
    s_up = np.array([[2.0, 1.0], [1.0, 0.5]], np.float32)
    s_down = np.array([[1.0, 0.5, 2.0, 3.0, 1.0], [0.5, 1.0, 1.0, 1.0, 4.0]], np.float32)
    x = np.array([1.0, 2.0, 3.0, 4.0, 5.0]) * scale_x
    packed = (oracle.pack(gate_q.reshape(E * I, H)).reshape(E, I, -1),
              oracle.pack(up_q.reshape(E * I, H)).reshape(E, I, -1),
              oracle.pack(down_q.reshape(E * H, I)).reshape(E, H, -1))
    return H, I, E, gate_q, up_q, down_q, s_gate, s_up, s_down, x, packed


@pytest.mark.parametrize("scale_x", [1.0, 50.0])
def test_ffn_hand_example_closed_form(scale_x):
    """y = sum_i w_i down_e(silu(min(g, 7)) * clamp(u, -7, 7)), element by element.
    scale_x = 50 makes both clamps bind ("The shipped code does no quantization")."""
    H, I, E, gq, uq, dq, sg, su, sd, x, (gp, up, dp) = _hand_case(scale_x)
    xbits = _f32_bits_to_bf16_bits(x).reshape(1, H)
    idx = np.array([[1, 0]], np.int32)
    w = np.array([[0.75, 0.25]])
    y = oracle.moe_ffn(gp, up, dp, sg, su, sd, xbits, idx, w, clamp=7.0)
    c = 7.0
    x1, x2, x3, x4, x5 = x
    # expert 0
    g = [0.5 * x1, 1.0 * (x5 - x2)]
    u = [2.0 * x3, 1.0 * (x1 + x2 + x3 + x4 + x5)]
    h0 = [_silu(min(g[r], c)) * max(-c, min(u[r], c)) for r in range(2)]
    y0 = [1.0 * h0[0], 0.5 * h0[1], 2.0 * (h0[0] - h0[1]), 0.0, -(h0[0] + h0[1])]
    # expert 1
    g = [0.25 * x4, 2.0 * (-x1)]
    u = [1.0 * x2, 0.5 * (-x5)]
    h1 = [_silu(min(g[r], c)) * max(-c, min(u[r], c)) for r in range(2)]
    y1 = [0.5 * h1[1], 1.0 * h1[0], 0.0, h1[0] + h1[1], -4.0 * h1[0]]
    want = [0.75 * a + 0.25 * b for a, b in zip(y1, y0)]
    np.testing.assert_allclose(y[0], want, rtol=1e-14, atol=1e-14)
    if scale_x == 50.0:
        assert 50.0 * 3 > c  # g of expert 0 row 1 is 150 before the clamp


def test_ffn_all_zero_weights_give_zero():
    E, H, I, T, k = 3, 11, 6, 2, 2
    gp = np.full((E, I, (H + 4) // 5), 121, np.uint8)
    dp = np.full((E, H, (I + 4) // 5), 121, np.uint8)
    x = synth.bf16_bits(synth.tokens(T, H, seed=1))
    y = oracle.moe_ffn(gp, gp, dp, np.ones((E, I), np.float32), np.ones((E, I), np.float32),
                       np.ones((E, H), np.float32), x, np.array([[0, 2], [1, 0]], np.int32),
                       np.full((T, k), 0.5), clamp=7.0)
    assert np.all(y == 0.0)


def _dequant_numpy(packed, K, scales):
    """Independent dequantizer: base-3 digits by numpy vector ops, times row scales."""
    p = packed.astype(np.int64)
    digits = np.stack([(p // 3 ** i) % 3 for i in range(5)], axis=-1).reshape(*p.shape[:-1], -1)
    return (digits[..., :K] - 1).astype(np.float64) * scales.astype(np.float64)[..., None]


@pytest.mark.parametrize("clamp", [7.0, math.inf, 0.3])
def test_ffn_equals_dense_fp64_on_tiny_shapes(clamp):
    """Brute-force dense fp64 matmuls on dequantized weights (K tails: H=13, I=7)."""
    E, H, I, T, k = 16, 13, 7, 3, 8
    wts = synth.expert_weights(E, H, I, seed=4, std=0.3)
    pk = {}
    for name in ("gate", "up", "down"):
        b = synth.bf16_bits(wts[name])
        pm, s = oracle.ternarize_pack(b.reshape(-1, b.shape[-1]))
        pk[name] = (pm.reshape(*b.shape[:-1], -1), s.reshape(b.shape[:-1]))
    x = synth.tokens(T, H, seed=4)
    xbits = synth.bf16_bits(x)
    rng = np.random.default_rng(4)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T)
    y = oracle.moe_ffn(pk["gate"][0], pk["up"][0], pk["down"][0], pk["gate"][1], pk["up"][1],
                       pk["down"][1], xbits, idx, w, clamp=clamp)
    Wg = _dequant_numpy(pk["gate"][0], H, pk["gate"][1])
    Wu = _dequant_numpy(pk["up"][0], H, pk["up"][1])
    Wd = _dequant_numpy(pk["down"][0], I, pk["down"][1])
    xf = synth.bits_to_float(xbits).astype(np.float64)
    silu = lambda z: z / (1 + np.exp(-z))
    ref = np.zeros((T, H))
    for t in range(T):
        for i in range(k):
            e = idx[t, i]
            g = Wg[e] @ xf[t]
            u = Wu[e] @ xf[t]
            h = silu(np.minimum(g, clamp)) * np.clip(u, -clamp, clamp)
            ref[t] += w[t, i] * (Wd[e] @ h)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
