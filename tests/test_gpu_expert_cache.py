"""Host-resident experts streamed into an HBM cache (maple_cache_fetch), through the
C-ABI: the experts of a layer live in pinned host memory, C slots in device memory; each
step's routed experts are made resident (least recently used slot on a miss) and the
FFN runs on the cache ("Maple Preview 接入 Mference：M4 MacBook 上 500MB 内存跑 20B MoE",
section "接入 Mference 后的实测结果": experts read on demand from outside the
accelerator).

Checked every step against a host model of the policy (which slot each routed expert
lands in, the tables, the hit and miss counts), and the FFN on the cache against the
CPU oracle on the pool's experts (|y - y_oracle| <= 2e-3 max|y_oracle| + 1e-5) and, bit
for bit, against the FFN on a device copy of the pool (the same path pinned on both
sides with maple_moe_ffn_ex)."""
import numpy as np
import pytest
import torch

import oracle
from support import assert_ffn_close, oracle_moe_ffn_rows, oracle_pack_layer
from ternary_weight_moe_02_b300 import synth

pytestmark = pytest.mark.gpu


class LruModel:
    """The cache policy restated on the host."""

    def __init__(self, E, C):
        self.slot_of = [-1] * E
        self.expert_of = [-1] * C
        self.last = [0] * C
        self.step = 0
        self.hits = self.misses = 0

    def fetch(self, idx):
        E, C = len(self.slot_of), len(self.expert_of)
        self.step += 1
        need = sorted({int(e) for e in idx.reshape(-1) if 0 <= e < E})
        hits = [e for e in need if self.slot_of[e] >= 0]
        in_use = {self.slot_of[e] for e in hits}
        for e in hits:
            self.last[self.slot_of[e]] = self.step
        misses = [e for e in need if self.slot_of[e] < 0]
        free = sorted((s for s in range(C) if s not in in_use), key=lambda s: (self.last[s], s))
        for r, e in enumerate(misses):
            v = free[r]
            if self.expert_of[v] >= 0:
                self.slot_of[self.expert_of[v]] = -1
            self.expert_of[v] = e
            self.slot_of[e] = v
            self.last[v] = self.step
        self.hits += len(hits)
        self.misses += len(misses)
        return np.array([[self.slot_of[e] if 0 <= e < E else -1 for e in row] for row in idx], np.int32)


@pytest.fixture(scope="module")
def pool32():
    """32 Maple-shaped experts packed by the oracle: numpy, pinned host tensors, and a
    device copy."""
    from ternary_weight_moe_02_b300 import maple
    w = synth.expert_weights(32, 2048, 512, seed=61, device="cuda")
    packed = oracle_pack_layer(w)
    names = ("gate", "up", "down", "s_gate", "s_up", "s_down")
    host = [torch.from_numpy(packed[n]).pin_memory() for n in names]
    dev = [t.cuda() for t in host]
    return packed, maple.Experts(*host, clamp=7.0), maple.Experts(*dev, clamp=7.0)


def _routing(rng, T, E, k):
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.dirichlet(np.ones(k), size=T).astype(np.float32)
    return idx, w


def test_streamed_steps_match_the_policy_and_the_oracle(pool32):
    from ternary_weight_moe_02_b300 import maple
    packed, pool, dev = pool32
    E, H, I, k, C = 32, 2048, 512, 8, 12
    cache = maple.ExpertCache(C, E, H, I)
    model = LruModel(E, C)
    ws = torch.empty(maple.maple_cache_fetch_workspace_size(2, k), dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(5)
    for step in range(12):
        T = 1 if step % 3 else 1
        idx, w = _routing(rng, T, E, k)
        if step == 4:
            idx[0, 2] = -1  # an id outside [0, E): no slot, contributes nothing
            idx[0, 5] = E
        x = synth.tokens(T, H, seed=100 + step, device="cuda")
        idx_d, w_d = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
        idx_slot = torch.full((T, k), -9, dtype=torch.int32, device="cuda")
        maple.maple_cache_fetch(pool, cache, idx_d, idx_slot, ws)
        # the same FFN path on both sides (the automatic choice depends on E: 12 slots
        # against 32 pool experts would pick different paths)
        y = torch.full((T, H), float("nan"), device="cuda")
        wsf = torch.empty(maple.maple_moe_ffn_workspace_size_ex(T, k, cache.experts, "cores"), dtype=torch.uint8,
                          device="cuda")
        maple.maple_moe_ffn_ex(cache.experts, x, idx_slot, w_d, y, "cores", wsf)
        y_ref_dev = torch.full_like(y, float("nan"))
        wsd = torch.empty(maple.maple_moe_ffn_workspace_size_ex(T, k, dev, "cores"), dtype=torch.uint8, device="cuda")
        maple.maple_moe_ffn_ex(dev, x, idx_d, w_d, y_ref_dev, "cores", wsd)
        torch.cuda.synchronize()
        want = model.fetch(idx)
        assert np.array_equal(idx_slot.cpu().numpy(), want), f"step {step}"
        assert cache.slot_of.cpu().tolist() == model.slot_of
        assert cache.expert_of.cpu().tolist() == model.expert_of
        assert torch.equal(y, y_ref_dev), f"step {step}: cache FFN differs from the FFN on the pool"
        valid = (idx >= 0) & (idx < E)
        y_ref = oracle_moe_ffn_rows(packed, synth.bf16_bits(x), np.where(valid, idx, 0).astype(np.int32),
                                    np.where(valid, w, 0), np.arange(T))
        assert_ffn_close(y.cpu().numpy(), y_ref, f"streamed step {step}")
    got = cache.counters()
    assert got["steps"] == 12 and got["hits"] == model.hits and got["misses"] == model.misses
    assert got["experts_copied"] == model.misses and model.hits > 0 and model.misses > C
    maple.maple_check_device_status()


def test_streamed_batch_and_graph_replay(pool32):
    """T = 2 tokens with k = 4 (8 routed slots, C = 8); the fetch + FFN of a step
    captured in a CUDA graph and replayed gives the same result as the direct calls."""
    from ternary_weight_moe_02_b300 import maple
    packed, pool, dev = pool32
    E, H, I, k, C, T = 32, 2048, 512, 4, 8, 2
    rng = np.random.default_rng(9)
    idx, w = _routing(rng, T, E, k)
    x = synth.tokens(T, H, seed=9, device="cuda")
    idx_d, w_d = torch.from_numpy(idx).cuda(), torch.from_numpy(w).cuda()
    outs = []
    for mode in ("direct", "graph"):
        cache = maple.ExpertCache(C, E, H, I)
        ws = torch.empty(maple.maple_cache_fetch_workspace_size(T, k), dtype=torch.uint8, device="cuda")
        idx_slot = torch.empty((T, k), dtype=torch.int32, device="cuda")
        y = torch.empty((T, H), device="cuda")
        wsf = torch.empty(maple.maple_moe_ffn_workspace_size(T, k, cache.experts), dtype=torch.uint8, device="cuda")

        def step(s=None):
            maple.maple_cache_fetch(pool, cache, idx_d, idx_slot, ws, stream=s)
            maple.maple_moe_ffn(cache.experts, x, idx_slot, w_d, y, wsf, stream=s)
        if mode == "direct":
            step()
        else:
            s = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    step(s)
                g.replay()
        torch.cuda.synchronize()
        outs.append(y.clone())
    assert torch.equal(outs[0], outs[1])
    y_ref = oracle_moe_ffn_rows(packed, synth.bf16_bits(x), idx, w, np.arange(T))
    assert_ffn_close(outs[0].cpu().numpy(), y_ref, "streamed batch")
