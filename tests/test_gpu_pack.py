"""GPU parity of maple_ternarize_pack / maple_unpack against the CPU oracle.

Bytes are bit-exact except trits on the 0.5 rounding boundary (counted), scales agree
to 1e-6 relative ("Maple-Preview ...", sections "The claim, verified from the bytes"
and "The 5.31 GB claim reconciles")."""
import numpy as np
import pytest
import torch

import oracle
from support import pack_compare
from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


def _gpu_pack(w):
    from ternary_weight_moe_02_b300 import maple
    rows, K = w.shape
    packed = torch.full((rows, (K + 4) // 5), 255, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    maple.maple_ternarize_pack(w, packed, scales)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy()


@pytest.mark.parametrize("rows,K", [(1, 1), (3, 4), (5, 5), (4, 13), (7, 16), (33, 2047),
                                    (64, 2048), (130, 512), (17, 1000), (9, 4101), (11, 8),
                                    (600, 16), (77, 4104), (50, 520), (3, 16384), (2, 49152)])
def test_pack_parity_shapes(rows, K):
    w = synth.bf16_normal((rows, K), 0.02, seed=rows * 1000 + K).cuda()
    gp, gs = _gpu_pack(w)
    pack_compare(synth.bf16_bits(w), gp, gs)  # bit-exact up to counted boundary trits


def test_pack_special_rows():
    K = 40
    rows = [np.zeros(K, np.float32), np.full(K, 0.25, np.float32), -np.full(K, 3.0, np.float32)]
    exact_tie = np.array([0.75, 0.25] * (K // 2), np.float32)  # s = 0.5: 0.25 -> 0, 0.75 -> 1
    rows.append(exact_tie)
    rows.append(-exact_tie)
    signed_zero = np.zeros(K, np.float32)
    signed_zero[::2] = -0.0
    signed_zero[5] = 1.0
    rows.append(signed_zero)
    # row sums of |w| must stay below the fp32 maximum (the kernel sums in fp32)
    big = np.linspace(-1e36, 1e36, K).astype(np.float32)
    rows.append(big)
    tiny = np.linspace(-1e-38, 1e-38, K).astype(np.float32)
    rows.append(tiny)
    w32 = torch.tensor(np.stack(rows))
    w = w32.to(torch.bfloat16).cuda()
    gp, gs = _gpu_pack(w)
    excluded, ref_p, ref_s = pack_compare(synth.bf16_bits(w), gp, gs)
    assert excluded == 0
    np.testing.assert_array_equal(gp, ref_p)
    assert gs[0] == 0 and np.all(gp[0] == 121)  # all-zero row: s = 0, trits 0
    q = oracle.unpack(gp[3:4], K)[0]
    np.testing.assert_array_equal(q, [1, 0] * (K // 2))


def test_pack_full_layer_sampled_against_oracle():
    """One Maple layer (256 experts x gate/up/down) packed in the bench's per-layer
    launch; 6 sampled matrices checked against the oracle byte by byte."""
    from ternary_weight_moe_02_b300 import maple
    E, H, I = 256, 2048, 512
    w = synth.expert_weights(E, H, I, seed=77, device="cuda")
    out = {}
    for name, (R, K) in (("gate", (E * I, H)), ("up", (E * I, H)), ("down", (E * H, I))):
        p = torch.empty((R, (K + 4) // 5), dtype=torch.uint8, device="cuda")
        s = torch.empty((R,), dtype=torch.float32, device="cuda")
        maple.maple_ternarize_pack(w[name].view(R, K), p, s)
        out[name] = (p, s)
    torch.cuda.synchronize()
    total_excl = 0
    for name, e in (("gate", 0), ("up", 131), ("down", 255), ("gate", 200), ("down", 17), ("up", 64)):
        rows = w[name].shape[1]
        K = w[name].shape[2]
        p, s = out[name]
        gp = p[e * rows:(e + 1) * rows].cpu().numpy()
        gs = s[e * rows:(e + 1) * rows].cpu().numpy()
        excl, _, ref_s = pack_compare(synth.bf16_bits(w[name][e]), gp, gs)
        total_excl += excl
        # three symmetric values per row and the Gaussian zero share (~31%)
        q = oracle.unpack(gp, K)
        assert abs((q == 0).mean() - 0.3101) < 0.01
    assert total_excl <= 50


def test_unpack_roundtrip_and_bad_codes():
    from ternary_weight_moe_02_b300 import maple
    rng = np.random.default_rng(9)
    rows, K = 37, 23
    q = rng.integers(-1, 2, size=(rows, K)).astype(np.int8)
    p = oracle.pack(q)
    s = rng.uniform(0.001, 2.0, size=rows).astype(np.float32)
    p_bad = p.copy()
    p_bad[3, 1] = 243
    p_bad[10, 4] = 255
    for packed, nbad in ((p, 0), (p_bad, 2)):
        out = torch.empty((rows, K), dtype=torch.float32, device="cuda")
        bad = torch.zeros(1, dtype=torch.int32, device="cuda")
        maple.maple_unpack(torch.from_numpy(packed).cuda(), torch.from_numpy(s).cuda(), K, out, bad)
        torch.cuda.synchronize()
        assert int(bad.item()) == nbad
        ref_q, st = oracle.unpack(packed, K, check=False)
        np.testing.assert_array_equal(out.cpu().numpy(), ref_q.astype(np.float32) * s[:, None])
