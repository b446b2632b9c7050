"""Helpers shared by the GPU parity tests: oracle-side packing of expert layers,
exclusion bookkeeping at the rounding boundaries, and the tolerances.

Tolerances (derived, and written where they are used):
  * packed bytes: bit-exact, except trits whose |w|/s lies within 1e-6 relative of the
    0.5 rounding boundary (using the oracle's s); those are excluded and counted;
  * scales: relative difference <= 1e-6 (the kernel's compensated fp32 row sum is
    within ~10 ulp of the exact sum);
  * router logits: |l_gpu - l| <= gamma_n * (sum_j |x_j W_ej| + |bias_e|), n = H/32 + 7
    (per-lane FMA chain of H/32 exact products, 5 butterfly levels, the bias add),
    gamma_n = n u / (1 - n u), u = 2^-24;
  * top-k: a token whose k-th and (k+1)-th oracle logits are closer than the two
    bounds together is a near tie: its index set is not compared (counted instead);
    inside the top-k, positions may swap only between logits within their bounds;
  * softmax weights: relative error <= 4 * max bound + 1e-6 (a perturbation d of every
    logit moves log w_i by at most 2d, and the normaliser by at most 2d);
  * FFN output: |y_gpu - y| <= 2e-3 * max|y| + 1e-5, element by element.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from ternary_weight_moe_02_b300 import synth

U32 = 2.0 ** -24


def gamma(n: int) -> float:
    return n * U32 / (1 - n * U32)


# A row can have excluded trits only if some bf16 magnitude lies within the window
# ||w|/s - 0.5| <= 0.5e-6, i.e. within 0.5e-6 s of s/2.  bf16 magnitudes near s/2 are
# 2^(e-7) apart for s/2 in [2^e, 2^(e+1)), so the window (width 1e-6 s) holds one with
# probability at most 1e-6 s / 2^(e-7) < 1e-6 * 512 = 5.12e-4 per row.
ROW_EXCLUSION_RATE = 5.12e-4


def pack_compare(w_bits: np.ndarray, gpu_packed: np.ndarray, gpu_scales: np.ndarray):
    """Compare GPU ternarize+pack with the oracle.  Returns (n_excluded_trits,
    oracle_packed, oracle_scales); raises AssertionError on a real mismatch.
    Excluded trits are checked against their expected rate: within a row they all
    share one magnitude (the bf16 value next to s/2), and the rows holding any stay
    within a 4-sigma Poisson bound of ROW_EXCLUSION_RATE per row."""
    rows, K = w_bits.shape
    ref_q, ref_s = oracle.ternarize(w_bits)
    ref_p = oracle.pack(ref_q)
    rel = np.abs(gpu_scales.astype(np.float64) - ref_s) / np.maximum(np.abs(ref_s), 1e-30)
    assert np.all((rel <= 1e-6) | (ref_s == 0) & (gpu_scales == 0)), f"scale rel err {rel.max()}"
    diff_rows = np.nonzero(np.any(gpu_packed != ref_p, axis=1))[0]
    excluded = 0
    if len(diff_rows):
        gq = oracle.unpack(gpu_packed[diff_rows], K)
        rq = ref_q[diff_rows]
        wv = synth.bits_to_float(w_bits[diff_rows]).astype(np.float64)
        r_idx, c_idx = np.nonzero(gq != rq)
        ratio = np.abs(wv[r_idx, c_idx]) / ref_s[diff_rows][r_idx].astype(np.float64)
        near = np.abs(ratio - 0.5) <= 0.5e-6
        assert np.all(near), (
            f"{int((~near).sum())} trits differ away from the rounding boundary; first ratio "
            f"{ratio[~near][:4]}")
        excluded = len(r_idx)
        mag = np.abs(wv[r_idx, c_idx])
        for r in np.unique(r_idx):
            assert np.unique(mag[r_idx == r]).size == 1, f"row {diff_rows[r]}: excluded trits of two magnitudes"
        lam = ROW_EXCLUSION_RATE * rows
        assert len(diff_rows) <= lam + 4 * np.sqrt(lam) + 2, (
            f"{len(diff_rows)} of {rows} rows hold excluded trits (expected about {lam:.3f})")
    return excluded, ref_p, ref_s


def oracle_pack_layer(w: dict, experts=None):
    """Oracle ternarize+pack of a layer's bf16 weights (torch tensors on any device).
    Only `experts` are packed (default: all); the others get five-zero bytes (121)
    and zero scales, which the FFN never reads for unrouted experts."""
    E, I, H = w["gate"].shape
    sel = range(E) if experts is None else sorted(set(int(e) for e in experts))
    out = {
        "gate": np.full((E, I, oracle.packed_row_bytes(H)), 121, np.uint8),
        "up": np.full((E, I, oracle.packed_row_bytes(H)), 121, np.uint8),
        "down": np.full((E, H, oracle.packed_row_bytes(I)), 121, np.uint8),
        "s_gate": np.zeros((E, I), np.float32),
        "s_up": np.zeros((E, I), np.float32),
        "s_down": np.zeros((E, H), np.float32),
    }
    for name in ("gate", "up", "down"):
        for e in sel:
            bits = synth.bf16_bits(w[name][e])
            p, s = oracle.ternarize_pack(bits)
            out[name][e] = p
            out["s_" + name][e] = s
    return out


def upload_experts(packed: dict, clamp: float = 7.0, device="cuda"):
    from ternary_weight_moe_02_b300 import maple
    t = {k: torch.from_numpy(v).to(device) for k, v in packed.items()}
    return maple.Experts(t["gate"], t["up"], t["down"], t["s_gate"], t["s_up"], t["s_down"],
                         clamp=clamp)


def run_ffn(ex, x, idx, w, path=None):
    """maple_moe_ffn (path None) or maple_moe_ffn_ex on the named path."""
    from ternary_weight_moe_02_b300 import maple
    T = x.shape[0]
    k = idx.shape[1]
    y = torch.full((T, ex.H), float("nan"), device=x.device, dtype=torch.float32)
    if path is None:
        ws = torch.empty(max(1, maple.maple_moe_ffn_workspace_size(T, k, ex)), dtype=torch.uint8,
                         device=x.device)
        maple.maple_moe_ffn(ex, x, idx, w, y, ws)
    else:
        need = maple.maple_moe_ffn_workspace_size_ex(T, k, ex, path)
        assert need > 0, f"path {path} cannot take T={T} k={k} on this shape"
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
        maple.maple_moe_ffn_ex(ex, x, idx, w, y, path, ws)
    return y


def oracle_moe_ffn_rows(packed: dict, x_bits: np.ndarray, idx: np.ndarray, w: np.ndarray,
                        rows, clamp: float = 7.0, workers: int | None = None) -> np.ndarray:
    """oracle.moe_ffn on the given token rows, the rows split over a pool of host
    threads.  Each oracle call is the plain single-threaded C routine on a chunk of
    rows (ctypes releases the GIL during it); the threads only run several such calls
    at once.  Returns y fp64 [len(rows), H] in the order of `rows`."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    rows = np.asarray(rows, dtype=np.int64)
    n = len(rows)
    if workers is None:
        workers = max(1, min(16, os.cpu_count() or 1))
    chunks = [c for c in np.array_split(np.arange(n), min(n, 4 * workers)) if len(c)]

    def one(c):
        r = rows[c]
        return c, oracle.moe_ffn(packed["gate"], packed["up"], packed["down"], packed["s_gate"],
                                 packed["s_up"], packed["s_down"], x_bits[r], idx[r],
                                 np.asarray(w, np.float64)[r], clamp=clamp)
    out = np.empty((n, packed["down"].shape[1]), np.float64)
    with ThreadPoolExecutor(max_workers=workers) as pool:
        for c, y in pool.map(one, chunks):
            out[c] = y
    return out


def assert_ffn_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    tol = 2e-3 * np.abs(y_ref).max() + 1e-5
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    assert err.max() <= tol, f"{what}: max err {err.max():.3e} > tol {tol:.3e}"
    return err.max() / max(np.abs(y_ref).max(), 1e-30)


def logit_bounds(x_bits, wr_bits, bias, tensor=False):
    """Bound on |l_gpu - l_exact| for every (t, e).  CUDA-core kernels: a lane's FMA
    chain of H/32 terms, a 5-level butterfly and the bias add, rounded to nearest
    (rigorous).  Tensor-core kernel (tensor=True): H/16 MMA accumulations, each adding
    16 exact products, taken as 16 more rounding steps, plus the bias add, with the
    unit doubled (2^-23) so that truncating additions are covered too; the hardware's
    internal order is not published, so this one is a model, checked here."""
    H = x_bits.shape[1]
    mag = np.abs(synth.bits_to_float(x_bits).astype(np.float64)) @ \
        np.abs(synth.bits_to_float(wr_bits).astype(np.float64)).T
    if bias is not None:
        mag = mag + np.abs(np.asarray(bias, np.float64))[None, :]
    if tensor:
        n = (H + 15) // 16 + 16 + 8
        u = 2.0 ** -23
        return n * u / (1 - n * u) * mag + 1e-30
    n = (H + 31) // 32 + 7
    return gamma(n) * mag + 1e-30


def check_route(ref_logits, ref_idx, bounds, g_logits, g_idx, g_w, k):
    """Returns the number of near-tie tokens (index sets not compared)."""
    T, E = ref_logits.shape
    assert np.all(np.abs(g_logits - ref_logits) <= bounds), "logit outside its error bound"
    near = 0
    for t in range(T):
        order = np.lexsort((np.arange(E), -ref_logits[t]))
        lk, lk1 = order[k - 1], order[k] if k < E else None
        boundary_tie = lk1 is not None and \
            ref_logits[t, lk] - ref_logits[t, lk1] <= bounds[t, lk] + bounds[t, lk1]
        if boundary_tie:
            near += 1
        else:
            assert set(g_idx[t].tolist()) == set(order[:k].tolist()), f"token {t}: top-k set"
        # order inside the selection: non-increasing up to the bounds
        for i in range(k - 1):
            a, b = g_idx[t, i], g_idx[t, i + 1]
            assert ref_logits[t, a] - ref_logits[t, b] >= -(bounds[t, a] + bounds[t, b])
            if ref_logits[t, a] == ref_logits[t, b] and bounds[t, a] < 1e-29:
                assert a < b
        # softmax weights of the GPU's own selection
        sel = g_idx[t]
        z = np.exp(ref_logits[t, sel] - ref_logits[t, sel].max())
        w_ref = z / z.sum()
        tol = 4 * bounds[t, sel].max() + 1e-6
        rel = np.abs(g_w[t].astype(np.float64) - w_ref) / w_ref
        assert rel.max() <= tol, f"token {t}: softmax weight rel err {rel.max():.3e} > {tol:.3e}"
    return near
