"""GPU parity of maple_moe_ffn against the CPU oracle, element by element:
|y_gpu - y| <= 2e-3 * max|y| + 1e-5 ("Maple-Preview ...", section "The shipped code
does no quantization": down(act(clamp(gate x, max=7)) * clamp(up x, -7, 7)), weighted
over the k routed experts).

Every case feeds both sides the same packed bytes (packed by the oracle) and the same
idx / fp32 w, so a mismatch points at the FFN kernels alone."""
import math

import numpy as np
import pytest
import torch

import oracle
from support import assert_ffn_close, oracle_pack_layer, run_ffn, upload_experts
from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


def _route_oracle(x, wr, bias, k):
    _, idx, w = oracle.route(synth.bf16_bits(x), synth.bf16_bits(wr),
                             None if bias is None else bias.double().numpy(), k)
    return idx, w.astype(np.float32)


def _compare(packed, ex, x, idx, w32, clamp=7.0, rows=None, what=""):
    y_gpu = run_ffn(ex, x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w32).cuda())
    torch.cuda.synchronize()
    y_gpu = y_gpu.cpu().numpy()
    sel = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    y_ref = oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                           packed["s_up"], packed["s_down"], synth.bf16_bits(x[sel]),
                           idx[sel], w32[sel].astype(np.float64), clamp=clamp)
    return assert_ffn_close(y_gpu[sel], y_ref, what), y_gpu


@pytest.fixture(scope="module")
def layer256():
    """One full Maple MoE layer: 256 experts 2048->512->2048, bf16 N(0, 0.02) drawn on
    the GPU, packed by the oracle, uploaded."""
    w = synth.expert_weights(256, 2048, 512, seed=0, device="cuda")
    packed = oracle_pack_layer(w)
    del w
    torch.cuda.empty_cache()
    return packed, upload_experts(packed)


@pytest.fixture(scope="module")
def router256():
    return synth.router_weights(256, 2048, seed=0, device="cuda")


@pytest.mark.parametrize("T", [1, 2, 3])
def test_ffn_tiny_shapes_with_k_tails(T):
    E, H, I, k = 16, 13, 7, 8
    w = synth.expert_weights(E, H, I, seed=4, std=0.3)
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    rng = np.random.default_rng(T)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w32 = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    x = synth.tokens(T, H, seed=4)
    _compare(packed, ex, x, idx, w32, what=f"tiny T={T}")


def test_ffn_reduced_layer_E32_T4():
    """Reduced MoE layer: hidden 2048, 32 experts, top-8, intermediate 512, 4 tokens."""
    E, H, I, T, k = 32, 2048, 512, 4, 8
    w = synth.expert_weights(E, H, I, seed=0, device="cuda")
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    wr = synth.router_weights(E, H, seed=0)
    x = synth.tokens(T, H, seed=0)
    idx, w32 = _route_oracle(x, wr, None, k)
    _compare(packed, ex, x, idx, w32, what="reduced layer")


def test_ffn_clamps_bind():
    """x scaled by 50: gate and up sums far beyond +-7, so both clamps bind."""
    E, H, I, T, k = 8, 2048, 512, 3, 4
    w = synth.expert_weights(E, H, I, seed=5, device="cuda")
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    x = (synth.tokens(T, H, seed=5).float() * 50).to(torch.bfloat16)
    rng = np.random.default_rng(5)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w32 = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    _compare(packed, ex, x, idx, w32, what="clamped")
    # the clamp changes the answer: an unclamped oracle disagrees
    y_free = oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                            packed["s_up"], packed["s_down"], synth.bf16_bits(x), idx,
                            w32.astype(np.float64), clamp=math.inf)
    y_c = oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                         packed["s_up"], packed["s_down"], synth.bf16_bits(x), idx,
                         w32.astype(np.float64), clamp=7.0)
    assert np.abs(y_free - y_c).max() > 0.1 * np.abs(y_c).max()
    # and the plain SwiGLU reading (clamp = inf) is matched by the GPU too
    ex_free = upload_experts(packed, clamp=math.inf)
    _compare(packed, ex_free, x, idx, w32, clamp=math.inf, what="no clamp")


def test_ffn_decode_T1_full_layer(layer256, router256):
    """Full Maple layer, batch-1 decode, three distinct tokens one at a time."""
    packed, ex = layer256
    for seed in (1, 2, 3):
        x = synth.tokens(1, 2048, seed=seed)
        idx, w32 = _route_oracle(x, router256.cpu(), None, 8)
        _compare(packed, ex, x, idx, w32, what=f"T=1 seed {seed}")


@pytest.mark.parametrize("T", [8, 32, 64])
def test_ffn_decode_batches_full_layer(layer256, router256, T):
    """Decode batches with a per-expert router bias ~ N(0, 0.5)."""
    packed, ex = layer256
    x = synth.tokens(T, 2048, seed=10 + T)
    idx, w32 = _route_oracle(x, router256.cpu(), synth.bias_normal(256, seed=T), 8)
    _compare(packed, ex, x, idx, w32, what=f"T={T}")


def test_ffn_prefill_4096_every_tile(layer256, router256):
    """4096-token prefill, Zipf(1.1) router bias; the GPU runs all tokens in one call
    (grouped tensor-core path, 64-token tiles).  The oracle checks, for every expert
    with a non-zero load, the first and the last token of each of its 64-token tiles
    (tiles follow the stable grouping of slots by expert, which the oracle's own
    grouping gives), plus the first tokens of the busiest and the idlest expert, the
    first and last token of the call and random picks: every tile record of the call,
    including the experts spanning several tiles and the tiles past the first chunk of
    the grouping, has at least one checked token."""
    from support import oracle_moe_ffn_rows
    packed, ex = layer256
    T, k, E, NT = 4096, 8, 256, 64
    x = synth.tokens(T, 2048, seed=42)
    idx, w32 = _route_oracle(x, router256.cpu(), synth.bias_zipf(E, seed=0, gamma=1.0), k)
    counts, offsets, perm = oracle.group(idx, E)
    assert counts.max() >= 200  # several hundred tokens on the busiest expert
    rows, tiles = set(), 0
    for e in np.nonzero(counts)[0]:
        for j in range(0, int(counts[e]), NT):
            last = min(j + NT, int(counts[e])) - 1
            rows.add(int(perm[offsets[e] + j]) // k)
            rows.add(int(perm[offsets[e] + last]) // k)
            tiles += 1
    rng = np.random.default_rng(0)
    busiest, idlest = np.argmax(counts), np.argmin(np.where(counts > 0, counts, 10**9))
    rows |= set(np.nonzero((idx == busiest).any(axis=1))[0][:6].tolist())
    rows |= set(np.nonzero((idx == idlest).any(axis=1))[0][:6].tolist())
    rows |= {0, T - 1}
    rows |= set(rng.choice(T, size=24, replace=False).tolist())
    rows = sorted(rows)
    print(f"prefill parity: {tiles} tiles of {int((counts > 0).sum())} loaded experts, "
          f"{len(rows)} tokens checked")
    y_gpu = run_ffn(ex, x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w32).cuda())
    torch.cuda.synchronize()
    y_gpu = y_gpu.cpu().numpy()
    y_ref = oracle_moe_ffn_rows(packed, synth.bf16_bits(x), idx, w32, rows)
    # the tolerance is taken over the checked rows (max|y| of the whole output is not
    # known without the oracle on every token; over a subset it can only be smaller)
    assert_ffn_close(y_gpu[rows], y_ref, "prefill, every tile")
    # every tile has a checked token
    checked = np.zeros(T, bool)
    checked[rows] = True
    for e in np.nonzero(counts)[0]:
        for j in range(0, int(counts[e]), NT):
            toks = perm[offsets[e] + j: offsets[e] + min(j + NT, int(counts[e]))] // k
            assert checked[toks].any()


@pytest.mark.parametrize("E,H,I", [(6, 40, 24), (8, 2048, 512)])
def test_ffn_invalid_and_duplicate_ids(E, H, I):
    """Generic path (H=40, I=24) and bulk-copy path (H=2048, I=512)."""
    T, k = 3, 4
    w = synth.expert_weights(E, H, I, seed=8, std=0.2, device="cuda")
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    x = synth.tokens(T, H, seed=8)
    idx = np.array([[0, 0, 5, 2], [-1, 3, E, 1], [4, 4, 4, 4]], np.int32)
    w32 = np.array([[0.4, 0.3, 0.2, 0.1], [0.5, 0.2, 0.2, 0.1], [0.25] * 4], np.float32)
    y_gpu = run_ffn(ex, x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w32).cuda())
    torch.cuda.synchronize()
    # an out-of-range id contributes nothing: the oracle sees weight 0 on a valid id
    idx_ref = np.where((idx >= 0) & (idx < E), idx, 0).astype(np.int32)
    w_ref = np.where((idx >= 0) & (idx < E), w32, 0).astype(np.float64)
    y_ref = oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                           packed["s_up"], packed["s_down"], synth.bf16_bits(x), idx_ref, w_ref)
    assert_ffn_close(y_gpu.cpu().numpy(), y_ref, "invalid/duplicate ids")


@pytest.mark.parametrize("k,T", [(12, 3), (13, 2), (1, 5)])
def test_ffn_k_range_full_shape(k, T):
    """k = 12 is the largest k of the bulk-copy down kernel; 13 falls back to the
    generic down kernel; k = 1 is a single expert per token."""
    E, H, I = 16, 2048, 512
    w = synth.expert_weights(E, H, I, seed=30 + k, device="cuda")
    packed = oracle_pack_layer(w)
    ex = upload_experts(packed)
    rng = np.random.default_rng(k)
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w32 = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    _compare(packed, ex, synth.tokens(T, H, seed=k), idx, w32, what=f"k={k}")


def test_ffn_all_zero_weights_give_zero():
    E, H, I, T, k = 4, 2048, 512, 2, 2
    packed = {
        "gate": np.full((E, I, 410), 121, np.uint8), "up": np.full((E, I, 410), 121, np.uint8),
        "down": np.full((E, H, 103), 121, np.uint8), "s_gate": np.ones((E, I), np.float32),
        "s_up": np.ones((E, I), np.float32), "s_down": np.ones((E, H), np.float32)}
    ex = upload_experts(packed)
    y = run_ffn(ex, synth.tokens(T, H, seed=1).cuda(), torch.tensor([[0, 1], [2, 3]], dtype=torch.int32).cuda(),
                torch.full((T, k), 0.5).cuda())
    torch.cuda.synchronize()
    assert torch.all(y == 0)


def test_device_status_is_clean_after_the_suite():
    """No bounded device wait gave up in any kernel launched so far in this process."""
    from ternary_weight_moe_02_b300 import maple
    maple.maple_check_device_status()


def test_ffn_is_deterministic(layer256, router256):
    packed, ex = layer256
    x = synth.tokens(64, 2048, seed=99)
    idx, w32 = _route_oracle(x, router256.cpu(), None, 8)
    args = (x.cuda(), torch.from_numpy(idx).cuda(), torch.from_numpy(w32).cuda())
    y1 = run_ffn(ex, *args)
    y2 = run_ffn(ex, *args)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_route_then_ffn_chain(layer256, router256):
    """The decode chain through both calls: GPU route feeding GPU FFN against oracle
    route feeding oracle FFN, on tokens that are not near ties."""
    from support import check_route, logit_bounds
    from ternary_weight_moe_02_b300 import maple
    packed, ex = layer256
    T, k = 16, 8
    x = synth.tokens(T, 2048, seed=123).cuda()
    logits = torch.empty((T, 256), device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), device="cuda")
    maple.maple_route_topk(x, router256, None, k, logits, idx, w)
    y = run_ffn(ex, x, idx, w)
    torch.cuda.synchronize()
    xb, wb = synth.bf16_bits(x), synth.bf16_bits(router256)
    ref_logits, ref_idx, ref_w = oracle.route(xb, wb, None, k)
    near = check_route(ref_logits, ref_idx, logit_bounds(xb, wb, None), logits.cpu().numpy(),
                       idx.cpu().numpy(), w.cpu().numpy(), k)
    assert near == 0
    y_ref = oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                           packed["s_up"], packed["s_down"], xb, ref_idx, ref_w)
    # same experts; the weights differ from the oracle's by a few fp32 ulps
    assert_ffn_close(y.cpu().numpy(), y_ref, "route -> ffn chain")
