"""GPU parity of maple_route_topk and maple_group_tokens against the CPU oracle.

Router ("Maple-Preview ...", section "The claim, verified from the bytes": full
precision, 8 of 256 experts by logit margin): logits within their fp32 error bound,
top-k sets exact except counted near ties, softmax weights within the derived bound.
Grouping: bit-exact."""
import zlib

import numpy as np
import pytest
import torch

import oracle
from support import check_route, logit_bounds
from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


def _route_gpu(x, wr, bias, k):
    from ternary_weight_moe_02_b300 import maple
    T, E = x.shape[0], wr.shape[0]
    logits = torch.full((T, E), float("nan"), device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), float("nan"), device="cuda")
    maple.maple_route_topk(x, wr, bias, k, logits, idx, w)
    torch.cuda.synchronize()
    return logits.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy()


CASES = {
    # name: (T, H, E, k, bias kind)
    "reduced_layer_T4_E32": (4, 2048, 32, 8, None),
    "decode_T1_E256": (1, 2048, 256, 8, None),
    "decode_T64_E256_bias": (64, 2048, 256, 8, "normal"),
    "prefill_T4096_E256_zipf": (4096, 2048, 256, 8, "zipf"),
    "k_equals_E": (3, 64, 5, 5, None),
    "scalar_path_H13": (9, 13, 20, 3, "normal"),
    "single_expert": (2, 16, 1, 1, None),
    "E1024_k32": (5, 256, 1024, 32, "normal"),
    "ragged_T_and_E": (19, 2048, 250, 8, None),
    "tiled_ragged_T_and_E": (37, 2048, 250, 8, "normal"),
    "tiled_E1024": (33, 512, 1024, 32, None),
    "tensor_ragged_T_and_E": (300, 2048, 250, 8, "normal"),
    "tensor_E1024_H512": (520, 512, 1024, 32, None),
}

# More than this many tokens (H a multiple of 8) route on the tensor cores.
STAGED_MAX_T = 256


@pytest.mark.parametrize("name", list(CASES))
def test_route_parity(name):
    T, H, E, k, bias_kind = CASES[name]
    seed = zlib.crc32(name.encode()) % 10000
    x = synth.tokens(T, H, seed=seed, device="cuda")
    wr = synth.router_weights(E, H, seed=seed, device="cuda")
    bias = None
    if bias_kind == "normal":
        bias = synth.bias_normal(E, seed=seed)
    elif bias_kind == "zipf":
        bias = synth.bias_zipf(E, seed=seed, gamma=1.0)
    xb, wb = synth.bf16_bits(x), synth.bf16_bits(wr)
    bnp = None if bias is None else bias.double().numpy()
    ref_logits, ref_idx, ref_w = oracle.route(xb, wb, bnp, k)
    g_logits, g_idx, g_w = _route_gpu(x, wr, None if bias is None else bias.cuda(), k)
    bounds = logit_bounds(xb, wb, bnp, tensor=T > STAGED_MAX_T and H % 8 == 0)
    near = check_route(ref_logits, ref_idx, bounds, g_logits, g_idx, g_w, k)
    assert near <= max(1, T // 50), f"{near} near-tie tokens of {T}"
    assert np.all(np.abs(g_w.sum(axis=1) - 1) < 1e-5)


@pytest.mark.parametrize("T,H,E", [(256, 2048, 256), (250, 520, 33), (37, 4096, 250)])
def test_route_logits_do_not_depend_on_the_token_grouping(T, H, E):
    """Up to 256 tokens the logits come from the staged kernel, whose FMA chain per logit
    does not depend on which tokens share a CTA: the logits of one call equal, bit for
    bit, those of the same tokens routed in smaller groups (they are also the bits of
    the fused batch-1 layer, checked in test_gpu_layer)."""
    x = synth.tokens(T, H, seed=T + E, device="cuda")
    wr = synth.router_weights(E, H, seed=T + E, device="cuda")
    bias = synth.bias_normal(E, seed=T).cuda()
    whole, _, _ = _route_gpu(x, wr, bias, 8)
    for step in (1, 8, 100):
        parts = [_route_gpu(x[t:t + step].contiguous(), wr, bias, 8)[0] for t in range(0, T, step)]
        np.testing.assert_array_equal(whole, np.concatenate(parts))


def test_route_exact_ties_go_to_lower_index():
    """Identical router rows give identical logits: lower ids must win."""
    T, H, E, k = 6, 64, 40, 8
    x = synth.tokens(T, H, seed=1, device="cuda")
    base = synth.router_weights(4, H, seed=1, device="cuda")
    wr = base.repeat(E // 4, 1).contiguous()  # rows e and e+4 are identical
    xb, wb = synth.bf16_bits(x), synth.bf16_bits(wr)
    ref_logits, ref_idx, _ = oracle.route(xb, wb, None, k)
    _, g_idx, g_w = _route_gpu(x, wr, None, k)
    np.testing.assert_array_equal(g_idx, ref_idx)
    for t in range(T):
        assert np.all(np.diff(g_w[t]) <= 1e-7)


@pytest.mark.parametrize("T,k,E", [(2, 8, 256), (64, 8, 256), (4096, 8, 256), (5000, 3, 1024),
                                   (1000, 8, 32), (7, 64, 64)])
def test_group_parity(T, k, E):
    from ternary_weight_moe_02_b300 import maple
    rng = np.random.default_rng(T * 31 + E)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    # skewed loads: a third of the slots go to a few experts
    hot = rng.random((T, k)) < 0.3
    idx[hot] = rng.integers(0, 4, size=int(hot.sum()))
    counts, offsets, perm = oracle.group(idx, E)
    g = [torch.full(s, -1, dtype=torch.int32, device="cuda") for s in ((E,), (E + 1,), (T * k,))]
    maple.maple_group_tokens(torch.from_numpy(idx).cuda(), E, *g)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(g[0].cpu().numpy(), counts)
    np.testing.assert_array_equal(g[1].cpu().numpy(), offsets)
    np.testing.assert_array_equal(g[2].cpu().numpy(), perm)


def test_group_skips_out_of_range_ids():
    from ternary_weight_moe_02_b300 import maple
    E = 16
    idx = np.array([[0, 3, -1], [16, 3, 5], [5, 5, 99]], np.int32)
    valid = [(s, e) for s, e in enumerate(idx.reshape(-1)) if 0 <= e < E]
    g = [torch.full(s, -1, dtype=torch.int32, device="cuda") for s in ((E,), (E + 1,), (9,))]
    maple.maple_group_tokens(torch.from_numpy(idx).cuda(), E, *g)
    torch.cuda.synchronize()
    counts = g[0].cpu().numpy()
    assert counts.tolist() == [sum(1 for _, e in valid if e == x) for x in range(E)]
    perm = g[2].cpu().numpy()[: len(valid)]
    assert perm.tolist() == [s for s, _ in sorted(valid, key=lambda p: (p[1], p[0]))]
