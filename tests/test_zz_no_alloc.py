"""maple_moe_ffn_static_scratch: the FFN entry point that allocates nothing.

It serves callers that cannot allocate device memory (a plugin whose host owns all
device allocations, code running inside CUDA graph capture, a loop that must not
enter an allocator).  Its scratch is a static 2 MiB array per GPU.  This file is
collected last on purpose, and it must pass alone in a fresh process as well as
after the other tests: the first call on the device performs the one-time look-up
of the array's device address.

Checks, through the C-ABI: two calls in a row (different inputs, so stale contents
of the shared array would show) match maple_moe_ffn with a caller-provided workspace
within the FFN tolerance |y - y_ref| <= 2e-3 max|y_ref| + 1e-5 (the entry point always
takes the CUDA-core kernels; the workspace call takes the tensor-core path at these
sizes); the largest accepted size works and the next one is rejected with
MAPLE_ERR_WORKSPACE, leaving the output untouched."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _experts(E, H, I, seed):
    from ternary_weight_moe_02_b300 import maple, synth
    w = synth.expert_weights(E, H, I, seed=seed, device="cuda")
    Bh, Bi = (H + 4) // 5, (I + 4) // 5
    gate = torch.empty((E, I, Bh), dtype=torch.uint8, device="cuda")
    up = torch.empty_like(gate)
    down = torch.empty((E, H, Bi), dtype=torch.uint8, device="cuda")
    sg, su = torch.empty((E, I), device="cuda"), torch.empty((E, I), device="cuda")
    sd = torch.empty((E, H), device="cuda")
    maple.maple_ternarize_pack(w["gate"].view(E * I, H), gate.view(E * I, Bh), sg.view(-1))
    maple.maple_ternarize_pack(w["up"].view(E * I, H), up.view(E * I, Bh), su.view(-1))
    maple.maple_ternarize_pack(w["down"].view(E * H, I), down.view(E * H, Bi), sd.view(-1))
    return maple.Experts(gate, up, down, sg, su, sd, clamp=7.0)


def _inputs(T, E, H, k, seed):
    from ternary_weight_moe_02_b300 import synth
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    x = synth.tokens(T, H, seed=seed, device="cuda")
    return x, torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()


def _with_workspace(ex, x, idx, w):
    from ternary_weight_moe_02_b300 import maple
    T, k = idx.shape
    y = torch.empty((T, ex.H), device="cuda")
    ws = torch.empty(maple.maple_moe_ffn_workspace_size(T, k, ex), dtype=torch.uint8, device="cuda")
    maple.maple_moe_ffn(ex, x, idx, w, y, ws)
    return y


def test_static_scratch_matches_workspace_entry_point_twice_in_a_row():
    from ternary_weight_moe_02_b300 import maple
    E, H, I, k = 64, 2048, 512, 8
    ex = _experts(E, H, I, seed=21)
    for call, (T, seed) in enumerate(((48, 1), (5, 2))):
        x, idx, w = _inputs(T, E, H, k, seed)
        y_ref = _with_workspace(ex, x, idx, w)
        y = torch.full((T, H), float("nan"), device="cuda")
        maple.maple_moe_ffn_static_scratch(ex, x, idx, w, y)
        torch.cuda.synchronize()
        ref = y_ref.cpu().numpy().astype(np.float64)
        got = y.cpu().numpy().astype(np.float64)
        tol = 2e-3 * np.abs(ref).max() + 1e-5
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        assert np.abs(got - ref).max() <= tol, f"call {call}: {np.abs(got - ref).max()} > {tol}"


def test_static_scratch_rejects_sizes_beyond_the_array():
    from ternary_weight_moe_02_b300 import maple
    E, H, I, k = 16, 2048, 512, 8
    ex = _experts(E, H, I, seed=3)
    # the entry point runs the CUDA-core kernels: 127 tokens fit, 128 tokens x 8 slots x
    # 512 rows x 4 B = 2 MiB of h alone do not
    x, idx, w = _inputs(127, E, H, k, seed=4)
    y_ref = _with_workspace(ex, x, idx, w)
    y = torch.full((127, H), float("nan"), device="cuda")
    maple.maple_moe_ffn_static_scratch(ex, x, idx, w, y)
    torch.cuda.synchronize()
    ref = y_ref.cpu().numpy().astype(np.float64)
    assert np.abs(y.cpu().numpy() - ref).max() <= 2e-3 * np.abs(ref).max() + 1e-5
    T = 128
    x, idx, w = _inputs(T, E, H, k, seed=3)
    y = torch.full((T, H), 7.0, device="cuda")
    with pytest.raises(maple.MapleError) as err:
        maple.maple_moe_ffn_static_scratch(ex, x, idx, w, y)
    assert err.value.status == maple.MAPLE_ERR_WORKSPACE
    assert "static array" in str(err.value)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
