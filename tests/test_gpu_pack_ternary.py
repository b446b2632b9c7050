"""GPU parity of maple_pack_ternary against the CPU oracle (oracle.ternary_exact +
oracle.pack): for rows that are already ternary, as in the released bf16 checkpoint
("Maple-Preview ...", section "The claim, verified from the bytes"), the packed bytes
are bit-exact, the scales (the rows' largest magnitudes) exactly equal, and the count
of rows that are not ternary equal."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _ternary_rows(rows, K, seed, off_rows=()):
    """bf16 bits of rows a_r * q_r (a bf16 magnitude, trits with ~40 % zeros), some
    special rows, and the rows in off_rows moved one ulp off ternary."""
    rng = np.random.default_rng(seed)
    q = rng.choice([-1, 0, 1], size=(rows, K), p=[0.3, 0.4, 0.3]).astype(np.float32)
    a = torch.tensor(rng.uniform(1e-3, 4.0, rows), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    w = a[:, None] * q
    if rows > 3:
        w[0] = 0.0                            # all zero: s = 0
        w[1] = 0.0
        w[1, K - 1] = -0.5                    # one nonzero, at the K tail
        w[2] = np.where(q[2] != 0, q[2] * np.float32(2.0 ** -130), np.float32(-0.0))  # bf16 subnormals, -0
    bits = (w.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), w.astype(np.float32))
    for r in off_rows:
        nz = np.nonzero(bits[r] & 0x7FFF)[0]
        bits[r, nz[len(nz) // 2]] += 1      # one magnitude one ulp up
    return bits


def _to_gpu(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _gpu_pack_ternary(w):
    from ternary_weight_moe_02_b300 import maple
    rows, K = w.shape
    packed = torch.full((rows, (K + 4) // 5), 255, dtype=torch.uint8, device="cuda")
    scales = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    maple.maple_pack_ternary(w, packed, scales, bad)
    torch.cuda.synchronize()
    return packed.cpu().numpy(), scales.cpu().numpy(), int(bad.item())


@pytest.mark.parametrize("rows,K,off", [(7, 1, ()), (5, 13, (4,)), (11, 8, ()), (64, 2048, (5, 63)),
                                        (300, 512, (7, 8, 299)), (9, 4101, (3,)), (33, 517, ()),
                                        (2, 49152, (1,))])
def test_pack_ternary_parity(rows, K, off):
    bits = _ternary_rows(rows, K, seed=rows * 7 + K, off_rows=off)
    gp, gs, gbad = _gpu_pack_ternary(_to_gpu(bits))
    q, s, bad = oracle.ternary_exact(bits)
    np.testing.assert_array_equal(gp, oracle.pack(q))
    np.testing.assert_array_equal(gs, s)
    assert gbad == bad == len(off)


def test_pack_ternary_matches_absmean_bytes_on_ternary_rows():
    """On rows that are exactly ternary, absmean ternarization gives the same trits (only
    its scale differs), so both entry points write the same bytes."""
    from ternary_weight_moe_02_b300 import maple
    bits = _ternary_rows(256, 2048, seed=3)
    w = _to_gpu(bits)
    gp, _, gbad = _gpu_pack_ternary(w)
    packed = torch.empty((256, 410), dtype=torch.uint8, device="cuda")
    scales = torch.empty(256, dtype=torch.float32, device="cuda")
    maple.maple_ternarize_pack(w, packed, scales)
    torch.cuda.synchronize()
    assert gbad == 0
    np.testing.assert_array_equal(gp, packed.cpu().numpy())


def test_pack_ternary_counter_is_optional():
    from ternary_weight_moe_02_b300 import maple
    bits = _ternary_rows(16, 100, seed=9, off_rows=(6,))
    w = _to_gpu(bits)
    packed = torch.empty((16, 20), dtype=torch.uint8, device="cuda")
    scales = torch.empty(16, dtype=torch.float32, device="cuda")
    maple.maple_pack_ternary(w, packed, scales)
    torch.cuda.synchronize()
    q, s, _ = oracle.ternary_exact(bits)
    np.testing.assert_array_equal(packed.cpu().numpy(), oracle.pack(q))
    np.testing.assert_array_equal(scales.cpu().numpy(), s)
