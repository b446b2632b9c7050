"""maple_moe_ffn_static_scratch: the FFN entry point that allocates nothing.

It serves callers that cannot allocate device memory (a plugin whose host owns all
device allocations, code running inside CUDA graph capture, a loop that must not
enter an allocator).  Its scratch is a static 2 MiB array per GPU.  This file is
collected last on purpose, and it must pass alone in a fresh process as well as
after the other tests: the first call on the device performs the one-time look-up
of the array's device address.

Checks, through the C-ABI, against the CPU oracle on the same packed bytes, idx and w,
within the FFN tolerance |y - y_oracle| <= 2e-3 max|y_oracle| + 1e-5 ("Maple-Preview
...", section "The shipped code does no quantization"): two calls in a row with
different inputs (so stale contents of the shared array would show); the largest
accepted size; and the next size up, which is rejected with MAPLE_ERR_WORKSPACE and
leaves the output untouched."""
import numpy as np
import pytest
import torch

import oracle
from support import assert_ffn_close, oracle_moe_ffn_rows, oracle_pack_layer, upload_experts

pytestmark = pytest.mark.gpu


def _layer(E, H, I, seed):
    """bf16 N(0, 0.02) experts packed by the oracle, uploaded."""
    from ternary_weight_moe_02_b300 import synth
    w = synth.expert_weights(E, H, I, seed=seed, device="cuda")
    packed = oracle_pack_layer(w)
    return packed, upload_experts(packed)


def _inputs(T, E, H, k, seed):
    from ternary_weight_moe_02_b300 import synth
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    x = synth.tokens(T, H, seed=seed, device="cuda")
    return x, idx, w


def _oracle(packed, x, idx, w):
    from ternary_weight_moe_02_b300 import synth
    return oracle_moe_ffn_rows(packed, synth.bf16_bits(x), idx, w, np.arange(x.shape[0]))


def test_static_scratch_matches_the_oracle_twice_in_a_row():
    from ternary_weight_moe_02_b300 import maple
    E, H, I, k = 64, 2048, 512, 8
    packed, ex = _layer(E, H, I, seed=21)
    for call, (T, seed) in enumerate(((48, 1), (5, 2))):
        x, idx, w = _inputs(T, E, H, k, seed)
        y = torch.full((T, H), float("nan"), device="cuda")
        maple.maple_moe_ffn_static_scratch(ex, x, torch.from_numpy(idx).cuda(),
                                           torch.from_numpy(w).cuda(), y)
        torch.cuda.synchronize()
        assert_ffn_close(y.cpu().numpy(), _oracle(packed, x, idx, w), f"static scratch, call {call}")


def test_static_scratch_rejects_sizes_beyond_the_array():
    from ternary_weight_moe_02_b300 import maple
    E, H, I, k = 16, 2048, 512, 8
    packed, ex = _layer(E, H, I, seed=3)
    # the entry point runs the CUDA-core kernels: 127 tokens fit, 128 tokens x 8 slots x
    # 512 rows x 4 B = 2 MiB of h alone do not
    x, idx, w = _inputs(127, E, H, k, seed=4)
    y = torch.full((127, H), float("nan"), device="cuda")
    maple.maple_moe_ffn_static_scratch(ex, x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), y)
    torch.cuda.synchronize()
    assert_ffn_close(y.cpu().numpy(), _oracle(packed, x, idx, w), "static scratch, 127 tokens")
    T = 128
    x, idx, w = _inputs(T, E, H, k, seed=3)
    y = torch.full((T, H), 7.0, device="cuda")
    with pytest.raises(maple.MapleError) as err:
        maple.maple_moe_ffn_static_scratch(ex, x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda(), y)
    assert err.value.status == maple.MAPLE_ERR_WORKSPACE
    assert "static array" in str(err.value)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
