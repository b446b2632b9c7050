"""GPU parity of maple_moe_layer (route + FFN in one call; a single token runs the
fused one-launch path) against the CPU oracle's route followed by its FFN.

Tolerances as for the separate calls: logits within their fp32 bound, top-k exact
unless a near tie, softmax weights within the derived bound, y within
2e-3 max|y| + 1e-5 ("Maple-Preview ...", sections "The claim, verified from the
bytes" and "The shipped code does no quantization")."""
import numpy as np
import pytest
import torch

import oracle
from support import assert_ffn_close, check_route, logit_bounds, oracle_pack_layer, upload_experts
from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


def _layer_call(ex, x, router, bias, k, ws=None):
    from ternary_weight_moe_02_b300 import maple
    T, E = x.shape[0], router.shape[0]
    logits = torch.full((T, E), float("nan"), device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), device="cuda")
    y = torch.full((T, ex.H), float("nan"), device="cuda")
    if ws is None:
        ws = torch.zeros(maple.maple_moe_layer_workspace_size(T, k, ex), dtype=torch.uint8, device="cuda")
    maple.maple_moe_layer(x, router, bias, ex, k, logits, idx, w, y, ws)
    return logits, idx, w, y, ws


def _check_against_oracle(packed, x, router, bias, k, logits, idx, w, y):
    xb, rb = synth.bf16_bits(x), synth.bf16_bits(router)
    bnp = None if bias is None else bias.double().cpu().numpy()
    ref_logits, ref_idx, ref_w = oracle.route(xb, rb, bnp, k)
    bounds = logit_bounds(xb, rb, bnp)
    near = check_route(ref_logits, ref_idx, bounds, logits.cpu().numpy(), idx.cpu().numpy(),
                       w.cpu().numpy(), k)
    assert near == 0, "seeded tokens chosen without near ties"
    y_ref = oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                           packed["s_up"], packed["s_down"], xb, ref_idx, ref_w)
    return assert_ffn_close(y.cpu().numpy(), y_ref, "layer")


@pytest.fixture(scope="module")
def layer256():
    w = synth.expert_weights(256, 2048, 512, seed=0, device="cuda")
    packed = oracle_pack_layer(w)
    del w
    torch.cuda.empty_cache()
    return packed, upload_experts(packed), synth.router_weights(256, 2048, seed=0, device="cuda")


@pytest.mark.parametrize("seed,biased", [(1, False), (2, False), (3, True), (4, True)])
def test_layer_single_token_full_layer(layer256, seed, biased):
    packed, ex, router = layer256
    x = synth.tokens(1, 2048, seed=seed, device="cuda")
    bias = synth.bias_normal(256, seed=seed).cuda() if biased else None
    logits, idx, w, y, _ = _layer_call(ex, x, router, bias, 8)
    torch.cuda.synchronize()
    _check_against_oracle(packed, x, router, bias, 8, logits, idx, w, y)


def test_layer_fused_matches_separate_calls_bitwise(layer256):
    """Same logits and selection as maple_route_topk (same accumulation order), and y
    within the FFN tolerance of maple_moe_ffn."""
    from ternary_weight_moe_02_b300 import maple
    packed, ex, router = layer256
    x = synth.tokens(1, 2048, seed=11, device="cuda")
    logits, idx, w, y, _ = _layer_call(ex, x, router, None, 8)
    l2 = torch.empty_like(logits)
    i2 = torch.empty_like(idx)
    w2 = torch.empty_like(w)
    maple.maple_route_topk(x, router, None, 8, l2, i2, w2)
    y2 = torch.empty_like(y)
    ws2 = torch.empty(maple.maple_moe_ffn_workspace_size(1, 8, ex), dtype=torch.uint8, device="cuda")
    maple.maple_moe_ffn(ex, x, i2, w2, y2, ws2)
    torch.cuda.synchronize()
    assert torch.equal(logits, l2) and torch.equal(idx, i2) and torch.equal(w, w2)
    assert_ffn_close(y.cpu().numpy(), y2.cpu().numpy().astype(np.float64), "fused vs separate")


def test_layer_repeated_calls_reuse_the_workspace(layer256):
    """The barrier counters are left at zero: many calls in a row on one workspace (and
    in a CUDA graph) give the same answer as a fresh call."""
    from ternary_weight_moe_02_b300 import maple
    packed, ex, router = layer256
    xs = synth.tokens(6, 2048, seed=5, device="cuda")
    first = [_layer_call(ex, xs[t:t + 1], router, None, 8)[3].clone() for t in range(6)]
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(1, 8, ex), dtype=torch.uint8, device="cuda")
    for rep in range(20):
        for t in range(6):
            y = _layer_call(ex, xs[t:t + 1], router, None, 8, ws=ws)[3]
            assert torch.equal(y, first[t])
    assert int(ws[:256].count_nonzero().item()) == 0
    # and captured in a graph, replayed
    outs = [torch.empty((1, 2048), device="cuda") for _ in range(6)]
    logits = torch.empty((1, 256), device="cuda")
    idx = torch.empty((1, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((1, 8), device="cuda")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        maple.maple_moe_layer(xs[0:1], router, None, ex, 8, logits, idx, w, outs[0], ws, stream=s)
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            for t in range(6):
                maple.maple_moe_layer(xs[t:t + 1], router, None, ex, 8, logits, idx, w, outs[t], ws,
                                      stream=s)
        for _ in range(3):
            g.replay()
    s.synchronize()
    for t in range(6):
        assert torch.equal(outs[t], first[t])
    maple.maple_check_device_status()


def test_layer_reduced_E32_single_token():
    """Fewer experts than CTAs: most CTAs own no router row."""
    E, H, I, k = 32, 2048, 512, 8
    w = synth.expert_weights(E, H, I, seed=0, device="cuda")
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    router = synth.router_weights(E, H, seed=0, device="cuda")
    for seed in (0, 1):
        x = synth.tokens(1, H, seed=seed, device="cuda")
        logits, idx, w32, y, _ = _layer_call(ex, x, router, None, k)
        torch.cuda.synchronize()
        _check_against_oracle(packed, x, router, None, k, logits, idx, w32, y)


@pytest.mark.parametrize("T", [2, 4])
def test_layer_batches_take_the_separate_path(T):
    E, H, I, k = 32, 2048, 512, 8
    w = synth.expert_weights(E, H, I, seed=0, device="cuda")
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    router = synth.router_weights(E, H, seed=0, device="cuda")
    x = synth.tokens(T, H, seed=3, device="cuda")
    logits, idx, w32, y, _ = _layer_call(ex, x, router, None, k)
    torch.cuda.synchronize()
    _check_against_oracle(packed, x, router, None, k, logits, idx, w32, y)


def test_layer_small_shapes_single_token():
    """A small shape the fused path accepts (H=160, I=40) and one it does not (H=40)."""
    for E, H, I, k in ((12, 160, 40, 4), (6, 40, 24, 3)):
        w = synth.expert_weights(E, H, I, seed=7, std=0.2, device="cuda")
        packed = oracle_pack_layer(w)
        ex = upload_experts(packed)
        router = synth.router_weights(E, H, seed=7, device="cuda")
        x = synth.tokens(1, H, seed=7, device="cuda")
        logits, idx, w32, y, _ = _layer_call(ex, x, router, None, k)
        torch.cuda.synchronize()
        _check_against_oracle(packed, x, router, None, k, logits, idx, w32, y)


def test_layer_host_buffers_match_the_device_call(layer256):
    """maple_moe_layer_host (token copied in from pinned host memory; y written to it by
    the fused launch, or copied out for pageable buffers) gives the device call's results
    bit for bit, twice in a row, in y and in y_host; the bound form too, and pageable
    host buffers."""
    from ternary_weight_moe_02_b300 import maple
    packed, ex, router = layer256
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(1, 8, ex), dtype=torch.uint8, device="cuda")
    for seed in (21, 22):
        x = synth.tokens(1, 2048, seed=seed, device="cuda")
        logits, idx, w, y, _ = _layer_call(ex, x, router, None, 8, ws)
        x_host = x.cpu().pin_memory()
        y_host = torch.full((1, 2048), float("nan")).pin_memory()
        x_dev = torch.empty_like(x)
        l2, i2, w2, y2 = (torch.empty_like(logits), torch.empty_like(idx), torch.empty_like(w),
                          torch.empty_like(y))
        y2.fill_(float("nan"))
        maple.maple_moe_layer_host(x_host, x_dev, router, None, ex, 8, l2, i2, w2, y2, y_host, ws)
        torch.cuda.synchronize()
        assert torch.equal(logits, l2) and torch.equal(idx, i2) and torch.equal(w, w2)
        assert torch.equal(y.cpu(), y_host) and torch.equal(y, y2)
        y_host.fill_(float("nan"))
        maple.bind_moe_layer_host(x_host, x_dev, router, None, ex, 8, l2, i2, w2, y2, y_host, ws)()
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), y_host)
        # pageable host buffers take asynchronous copies instead of the copy kernels
        x_page, y_page = x.cpu(), torch.full((1, 2048), float("nan"))
        maple.maple_moe_layer_host(x_page, x_dev, router, None, ex, 8, l2, i2, w2, y2, y_page, ws)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), y_page)


def test_layer_host_buffers_several_tokens(layer256):
    """Three tokens through maple_moe_layer_host (the route + FFN calls, copy kernels on
    pinned buffers) against the device call, bit for bit."""
    from ternary_weight_moe_02_b300 import maple
    packed, ex, router = layer256
    T = 3
    ws = torch.zeros(maple.maple_moe_layer_workspace_size(T, 8, ex), dtype=torch.uint8, device="cuda")
    x = synth.tokens(T, 2048, seed=31, device="cuda")
    logits, idx, w, y, _ = _layer_call(ex, x, router, None, 8, ws)
    x_host = x.cpu().pin_memory()
    y_host = torch.full((T, 2048), float("nan")).pin_memory()
    x_dev = torch.empty_like(x)
    l2, i2, w2, y2 = (torch.empty_like(logits), torch.empty_like(idx), torch.empty_like(w), torch.empty_like(y))
    maple.maple_moe_layer_host(x_host, x_dev, router, None, ex, 8, l2, i2, w2, y2, y_host, ws)
    torch.cuda.synchronize()
    assert torch.equal(logits, l2) and torch.equal(idx, i2) and torch.equal(w, w2)
    assert torch.equal(y.cpu(), y_host)
