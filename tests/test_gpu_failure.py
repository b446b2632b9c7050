"""Failure detection on the GPU without faulting it (no trap, no bad address, no
unbounded wait).  Every device wait in the library is a bounded poll; these tests make
one of them run out on purpose and check that the library reports it and recovers:

  * MAPLE_INJECT_COPY_STALL: the next fused single-token layer launch arms one
    bulk-copy barrier for 16 bytes more than its copies deliver, with a short poll
    limit.  The wait gives up, maple_check_device_status reports MAPLE_ERR_TIMEOUT
    (and clears it), the rows of the stalled CTA come out NaN, and the very next call,
    with the same workspace and no clean-up, matches the result of an undisturbed call
    bit for bit.
  * MAPLE_INJECT_LAUNCH_ERROR: the next launching call reports MAPLE_ERR_CUDA and
    launches nothing (its outputs stay untouched); the call after it works."""
import numpy as np
import pytest
import torch

from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def layer():
    from ternary_weight_moe_02_b300 import maple
    E, H, I = 32, 2048, 512
    w = synth.expert_weights(E, H, I, seed=77, device="cuda")
    Bh, Bi = (H + 4) // 5, (I + 4) // 5
    t = {"gate": torch.empty((E, I, Bh), dtype=torch.uint8, device="cuda"),
         "up": torch.empty((E, I, Bh), dtype=torch.uint8, device="cuda"),
         "down": torch.empty((E, H, Bi), dtype=torch.uint8, device="cuda")}
    s = {"gate": torch.empty((E, I), device="cuda"), "up": torch.empty((E, I), device="cuda"),
         "down": torch.empty((E, H), device="cuda")}
    for name, K in (("gate", H), ("up", H), ("down", I)):
        maple.maple_ternarize_pack(w[name].view(-1, K), t[name].view(-1, (K + 4) // 5), s[name].view(-1))
    ex = maple.Experts(t["gate"], t["up"], t["down"], s["gate"], s["up"], s["down"], clamp=7.0)
    return ex, synth.router_weights(E, H, seed=77, device="cuda")


def _call(ex, router, x, ws, k=8):
    from ternary_weight_moe_02_b300 import maple
    E = router.shape[0]
    out = (torch.full((1, E), float("nan"), device="cuda"),
           torch.full((1, k), -7, dtype=torch.int32, device="cuda"),
           torch.full((1, k), float("nan"), device="cuda"),
           torch.full((1, ex.H), 123.0, device="cuda"))
    maple.maple_moe_layer(x, router, None, ex, k, *out, ws)
    return out


def test_copy_stall_times_out_reports_and_recovers(layer):
    from ternary_weight_moe_02_b300 import maple
    ex, router = layer
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(1, 8, ex), dtype=torch.uint8, device="cuda")
    x = synth.tokens(1, ex.H, seed=5, device="cuda")
    maple.maple_check_device_status()  # clean before
    ref = _call(ex, router, x, ws)
    maple.maple_check_device_status()
    maple.maple_test_inject(maple.MAPLE_INJECT_COPY_STALL, 20)
    bad = _call(ex, router, x, ws)
    with pytest.raises(maple.MapleError) as err:
        maple.maple_check_device_status()
    assert err.value.status == maple.MAPLE_ERR_TIMEOUT
    y_bad = bad[3].cpu().numpy()
    assert np.isnan(y_bad).any(), "the stalled CTA's rows should be NaN"
    maple.maple_check_device_status()  # the report cleared the word
    # the next call needs no clean-up: counters were left at zero
    again = _call(ex, router, x, ws)
    maple.maple_check_device_status()
    for a, b in zip(ref, again):
        assert torch.equal(a, b)


def test_injected_launch_error_launches_nothing(layer):
    from ternary_weight_moe_02_b300 import maple
    ex, router = layer
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(1, 8, ex), dtype=torch.uint8, device="cuda")
    x = synth.tokens(1, ex.H, seed=6, device="cuda")
    maple.maple_test_inject(maple.MAPLE_INJECT_LAUNCH_ERROR)
    with pytest.raises(maple.MapleError) as err:
        out = _call(ex, router, x, ws)
    assert err.value.status == maple.MAPLE_ERR_CUDA and "injected" in str(err.value)
    torch.cuda.synchronize()
    out = _call(ex, router, x, ws)
    maple.maple_check_device_status()
    assert torch.isfinite(out[3]).all()
    # the failed call wrote nothing: its output buffers keep their fill values
    from ternary_weight_moe_02_b300 import maple as m
    y = torch.full((1, ex.H), 123.0, device="cuda")
    m.maple_test_inject(m.MAPLE_INJECT_LAUNCH_ERROR)
    with pytest.raises(m.MapleError):
        m.maple_moe_layer(x, router, None, ex, 8, torch.empty((1, router.shape[0]), device="cuda"),
                          torch.empty((1, 8), dtype=torch.int32, device="cuda"),
                          torch.empty((1, 8), device="cuda"), y, ws)
    torch.cuda.synchronize()
    assert torch.all(y == 123.0)
