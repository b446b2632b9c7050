"""GPU parity of the grouped tensor-core FFN path (tcgen05 fp8 MMAs: trits decoded to
e4m3, each bf16 activation row split exactly into two e4m3 rows under a power-of-two
scale) against the CPU oracle, element by element: |y_gpu - y| <= 2e-3 * max|y| + 1e-5
("Maple-Preview ...", section "The shipped code does no quantization").  This path
rounds h to bf16 before the down projection; the bound above covers it.

maple_moe_ffn_ex names the path, so the tensor path also runs on shapes where the
automatic choice would take the CUDA-core kernels, and both paths run on the same
inputs."""
import numpy as np
import pytest
import torch

import oracle
from support import assert_ffn_close, oracle_pack_layer, run_ffn, upload_experts
from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


def _layer(E, H, I, seed, std=0.02):
    w = synth.expert_weights(E, H, I, seed=seed, std=std, device="cuda")
    packed = oracle_pack_layer(w)
    return packed, upload_experts(packed)


def _oracle(packed, x, idx, w32, clamp=7.0):
    return oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                          packed["s_up"], packed["s_down"], synth.bf16_bits(x), idx,
                          w32.astype(np.float64), clamp=clamp)


def _run(ex, x, idx, w32, path=None):
    y = run_ffn(ex, x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w32).cuda(), path)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def _random_routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w32 = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    return idx, w32


@pytest.mark.parametrize("E,H,I,T,k", [(8, 256, 128, 40, 4), (4, 384, 192, 33, 3),
                                       (6, 128, 128, 17, 6), (16, 2048, 512, 24, 8),
                                       (4, 384, 192, 200, 2), (2, 256, 2048, 150, 2),
                                       (2, 2048, 2048, 40, 1)])
def test_tensor_path_shapes(E, H, I, T, k):
    """Ragged token tiles (n_e not a multiple of the tile width), K tails (H = 384: 77
    packed bytes per row, the last 320-value stage 64 values long; I = 192: 39 bytes),
    the smallest shape the path takes (H = I = 128), the Maple expert shape, the same
    K tails on 64-token tiles (400 slots over 4 experts), a wide intermediate dimension
    (I = 2048: down rows of 410 packed bytes, two packed-row buffers) on 64-token tiles,
    and H = I = 2048 on 16-token tiles."""
    packed, ex = _layer(E, H, I, seed=E + H + T)
    x = synth.tokens(T, H, seed=T)
    idx, w32 = _random_routing(T, E, k, seed=T)
    y = _run(ex, x, idx, w32, "tensor")
    assert_ffn_close(y, _oracle(packed, x, idx, w32), f"tensor E={E} H={H} I={I}")


def test_tensor_path_several_token_tiles_per_expert():
    """Four experts, 300 tokens, top-2: about 150 tokens per expert, so each expert
    spans three 64-token tiles; expert 0 gets exactly 128 + 1 tokens (its last tile
    holds one token)."""
    E, H, I, T, k = 4, 256, 128, 300, 2
    packed, ex = _layer(E, H, I, seed=11)
    x = synth.tokens(T, H, seed=11)
    idx, w32 = _random_routing(T, E, k, seed=11)
    idx[:129, 0] = 0
    idx[:129, 1] = 1 + (np.arange(129) % 3)
    idx[129:, 0] = 1 + (np.arange(T - 129) % 3)
    idx[129:, 1] = 1 + ((np.arange(T - 129) + 1) % 3)
    assert np.bincount(idx.reshape(-1), minlength=E)[0] == 129
    y = _run(ex, x, idx, w32, "tensor")
    assert_ffn_close(y, _oracle(packed, x, idx, w32), "two token tiles")


def test_tensor_path_many_slots_chunked_grouping():
    """5600 slots (700 tokens, top-8, 16 experts): the grouping runs over six chunks of
    1024 slots (the last one partial) and the tiles are 64 tokens wide."""
    E, H, I, T, k = 16, 256, 128, 700, 8
    packed, ex = _layer(E, H, I, seed=17)
    x = synth.tokens(T, H, seed=17)
    idx, w32 = _random_routing(T, E, k, seed=17)
    idx[5, 3] = -1  # an invalid slot inside the first chunk
    w32[5, 3] = 0.0
    y1 = _run(ex, x, idx, w32)
    y2 = _run(ex, x, idx, w32)
    assert np.array_equal(y1, y2)
    valid = (idx >= 0) & (idx < E)
    y_ref = _oracle(packed, x, np.where(valid, idx, 0).astype(np.int32), np.where(valid, w32, 0))
    assert_ffn_close(y1, y_ref, "chunked grouping")


def test_tensor_path_is_the_automatic_choice_for_dense_loads():
    """With the automatic choice (maple_moe_ffn), 96 tokens on 16 experts (48 slots per
    expert) take the tensor path; the result matches the oracle and repeats bit for bit."""
    E, H, I, T, k = 16, 2048, 512, 96, 8
    packed, ex = _layer(E, H, I, seed=3)
    x = synth.tokens(T, H, seed=3)
    idx, w32 = _random_routing(T, E, k, seed=3)
    y1 = _run(ex, x, idx, w32)
    y2 = _run(ex, x, idx, w32)
    assert np.array_equal(y1, y2)
    assert_ffn_close(y1, _oracle(packed, x, idx, w32), "automatic tensor path")


def test_tensor_and_core_paths_agree():
    E, H, I, T, k = 8, 2048, 512, 20, 8
    packed, ex = _layer(E, H, I, seed=21)
    x = synth.tokens(T, H, seed=21)
    idx, w32 = _random_routing(T, E, k, seed=21)
    y_t = _run(ex, x, idx, w32, "tensor")
    y_c = _run(ex, x, idx, w32, "cores")
    y_ref = _oracle(packed, x, idx, w32)
    assert_ffn_close(y_t, y_ref, "tensor")
    assert_ffn_close(y_c, y_ref, "cores")
    assert np.abs(y_t - y_c).max() <= 4e-3 * np.abs(y_ref).max()


def test_tensor_path_invalid_ids_and_clamp():
    """Out-of-range ids add nothing; x scaled by 50 makes both clamps bind."""
    E, H, I, T, k = 6, 256, 128, 5, 4
    packed, ex = _layer(E, H, I, seed=8, std=0.2)
    x = (synth.tokens(T, H, seed=8).float() * 50).to(torch.bfloat16)
    idx = np.array([[0, 0, 5, 2], [-1, 3, E, 1], [4, 4, 4, 4], [1, 2, 3, 5], [5, -7, 0, 2]], np.int32)
    w32 = np.full((T, k), 0.25, np.float32)
    y = _run(ex, x, idx, w32, "tensor")
    valid = (idx >= 0) & (idx < E)
    y_ref = _oracle(packed, x, np.where(valid, idx, 0).astype(np.int32), np.where(valid, w32, 0))
    assert_ffn_close(y, y_ref, "tensor invalid ids, clamped")


def test_tensor_path_rows_of_very_different_magnitude():
    """Each token row gets its own split scale: rows scaled by 2^-24 .. 2^9 (and one
    all-zero row): the whole output meets the FFN bound 2e-3 max|y| + 1e-5 element by
    element, and each row matches the oracle within 4e-3 of that row's own largest
    output.  One scale shared by the tile would flush the small rows to zero (errors of
    order one).  The per-row bound is twice the whole-output one because, taken row by
    row, the rounding of h to bf16 alone reaches 2.1e-3 of a row's largest output on
    these inputs (fp64 model of that single rounding; over the whole output it is
    0.96e-3 of max|y|)."""
    E, H, I, T, k = 8, 256, 128, 12, 4
    packed, ex = _layer(E, H, I, seed=31)
    scale = torch.tensor([2.0 ** (3 * t - 24) for t in range(T)]).unsqueeze(1)
    x = (synth.tokens(T, H, seed=31).float() * scale).to(torch.bfloat16)
    x[4] = 0
    idx, w32 = _random_routing(T, E, k, seed=31)
    y = _run(ex, x, idx, w32, "tensor")
    y_ref = _oracle(packed, x, idx, w32)
    assert np.all(y[4] == 0)
    assert_ffn_close(y, y_ref, "rows of very different magnitude")
    for t in range(T):
        tol = 4e-3 * np.abs(y_ref[t]).max() + 1e-30
        assert np.abs(y[t] - y_ref[t]).max() <= tol, (t, np.abs(y[t] - y_ref[t]).max(), tol)


def test_tensor_path_all_zero_weights_give_zero():
    E, H, I, T, k = 2, 256, 128, 3, 2
    Bh, Bi = (H + 4) // 5, (I + 4) // 5
    packed = {"gate": np.full((E, I, Bh), 121, np.uint8), "up": np.full((E, I, Bh), 121, np.uint8),
              "down": np.full((E, H, Bi), 121, np.uint8), "s_gate": np.ones((E, I), np.float32),
              "s_up": np.ones((E, I), np.float32), "s_down": np.ones((E, H), np.float32)}
    ex = upload_experts(packed)
    y = _run(ex, synth.tokens(T, H, seed=1), np.array([[0, 1]] * T, np.int32),
             np.full((T, k), 0.5, np.float32), "tensor")
    assert np.all(y == 0)


def test_device_status_is_clean_after_the_tensor_cases():
    from ternary_weight_moe_02_b300 import maple
    maple.maple_check_device_status()
