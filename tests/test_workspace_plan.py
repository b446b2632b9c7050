"""Workspace sizing of maple_moe_ffn, on the host (no GPU needed): the size a call asks
for follows the FFN path the call will take.  The CUDA-core layout is counts, offsets,
the slot permutation, the active-expert list and h fp32 [T*k][I], each region 256-byte
aligned; the grouped tensor-core path adds its own regions.  That path is taken for
T*k >= 32 and 8*T*k >= E on shapes it accepts (maple_moe_ffn_workspace_size_ex names a path), and
never when its tile count would pass 65535 (a cap on its operand workspace); asking
for the tensor path where it cannot run sizes nothing (0: the call would be rejected)."""
import ctypes

import pytest

from ternary_weight_moe_02_b300 import maple


def _align(v, a=256):
    return (v + a - 1) // a * a


def cores_bytes(T, k, E, I):
    S = T * k
    o = _align(4 * E)             # counts
    o = _align(o + 4 * (E + 1))   # offsets
    o = _align(o + 4 * S)         # perm
    o = _align(o + 4 * E)         # active experts
    o = _align(o + 4)             # their number
    return _align(o + 4 * S * I)  # h fp32


def ws(T, k, E, H, I, path=None):
    ex = maple.maple_experts(None, None, None, None, None, None, E, H, I, 7.0)
    if path is None:
        return maple._lib.maple_moe_ffn_workspace_size(T, k, ctypes.byref(ex))
    return maple._lib.maple_moe_ffn_workspace_size_ex(T, k, ctypes.byref(ex), maple._path(path))


@pytest.mark.parametrize("T,k,E,H,I", [(1, 8, 256, 2048, 512), (64, 8, 256, 2048, 512),
                                       (3, 8, 16, 13, 7), (5000, 3, 1024, 384, 192)])
def test_cuda_core_layout(T, k, E, H, I):
    assert ws(T, k, E, H, I, "cores") == cores_bytes(T, k, E, I)


def test_static_scratch_limit_is_127_tokens_at_the_maple_shape():
    """The allocation-free entry point runs the CUDA-core kernels in a 2 MiB array."""
    assert ws(127, 8, 16, 2048, 512, "cores") <= 2 << 20 < ws(128, 8, 16, 2048, 512, "cores")


def test_default_choice_follows_the_slot_count():
    assert ws(1, 8, 256, 2048, 512) == cores_bytes(1, 8, 256, 512)        # 8 slots < 256 / 8
    assert ws(3, 8, 256, 2048, 512) == cores_bytes(3, 8, 256, 512)        # 24 slots
    assert ws(4, 8, 256, 2048, 512) > cores_bytes(4, 8, 256, 512)         # 32 slots: tensor path
    assert ws(4, 8, 256, 2048, 512) == ws(4, 8, 256, 2048, 512, "tensor")
    assert ws(4, 8, 256, 2048, 512) == ws(4, 8, 256, 2048, 512, "auto")


def test_unknown_path_sizes_nothing():
    assert ws(16, 8, 256, 2048, 512, 3) == 0
    assert ws(16, 8, 256, 2048, 512, -1) == 0


def test_shapes_the_tensor_path_rejects_stay_on_cuda_cores():
    for H, I in ((2000, 512), (2048, 520), (2176, 512), (64, 128)):
        assert ws(64, 8, 256, H, I) == cores_bytes(64, 8, 256, I)
        assert ws(64, 8, 256, H, I, "tensor") == 0


def test_calls_beyond_the_grid_limit_take_cuda_cores():
    """64-token tiles: at most S/64 + E tiles.  2^18 tokens x 8 slots (33,024 tiles)
    fit; 2^19 tokens (65,792 tiles) and the API's maximum of 2^24 slots do not."""
    E, H, I, k = 256, 2048, 512, 8
    assert ws(1 << 18, k, E, H, I, "tensor") > cores_bytes(1 << 18, k, E, I)
    for T in (1 << 19, 1 << 21):
        assert ws(T, k, E, H, I) == cores_bytes(T, k, E, I)
        assert ws(T, k, E, H, I, "tensor") == 0
