"""CPU model of the bulk-copy (TMA) plan of the FFN kernels.

For every shape the dispatch predicates accept, enumerate each 1-D bulk copy and L2
bulk prefetch the kernels issue (offsets relative to 16-byte aligned bases, sizes) and
check that all of them start on a 16-byte boundary, have a size that is a multiple of
16 and stay inside their buffer.  The formulas restate those in csrc/ffn_decode.cu;
a misaligned bulk copy faults the GPU, so this runs on the CPU first."""
import itertools

import numpy as np
import torch

GU_ROWS = 8      # row pairs per gate/up CTA
DN_ROWS = 16     # output rows per down CTA
DN_MAX_K = 12
MAX_LANE_BYTES = 13


def nbytes(K):
    return (K + 4) // 5


def gateup_ok(H, I):
    Bh = nbytes(H)
    return I % GU_ROWS == 0 and Bh % 2 == 0 and H % 8 == 0 and (Bh + 31) // 32 <= MAX_LANE_BYTES


def down_ok(H, I, k):
    Bi = nbytes(I)
    return H % DN_ROWS == 0 and I % 4 == 0 and k <= DN_MAX_K and (Bi + 31) // 32 <= MAX_LANE_BYTES


def prefetch_down(H, I):
    return (H * nbytes(I)) % 16 == 0 and H % 4 == 0


def _check(off, size, buf_bytes, what):
    assert off % 16 == 0, f"{what}: offset {off} not 16-byte aligned"
    assert size % 16 == 0 and size > 0, f"{what}: size {size}"
    assert off + size <= buf_bytes, f"{what}: [{off}, {off + size}) past {buf_bytes}"


def gateup_transfers(E, H, I, T, k):
    Bh = nbytes(H)
    gate_bytes = E * I * Bh
    x_bytes = T * H * 2
    down_bytes = E * H * nbytes(I)
    wbytes = GU_ROWS * Bh
    grid_x = I // GU_ROWS
    for e, bx, t in itertools.product(range(E), range(grid_x), range(T)):
        r0 = bx * GU_ROWS
        yield (e * I + r0) * Bh, wbytes, gate_bytes, "gate rows"
        yield (e * I + r0) * Bh, wbytes, gate_bytes, "up rows"
        yield (e * I + r0) * 4, 4 * GU_ROWS, E * I * 4, "gate scales"
        yield (e * I + r0) * 4, 4 * GU_ROWS, E * I * 4, "up scales"
        yield t * H * 2, 2 * H, x_bytes, "x row"
        if prefetch_down(H, I):
            total = H * nbytes(I)
            part = ((total + grid_x - 1) // grid_x + 15) // 16 * 16
            start = bx * part
            if start < total:
                yield e * total + start, min(part, total - start), down_bytes, "down prefetch"
            if bx == 0:
                yield e * H * 4, 4 * H, E * H * 4, "s_down prefetch"


def down_transfers(E, H, I, T, k):
    Bi = nbytes(I)
    down_bytes = E * H * Bi
    h_bytes = T * k * I * 4
    dbytes = DN_ROWS * Bi
    for e, by, t, i in itertools.product(range(E), range(H // DN_ROWS), range(T), range(k)):
        c0 = by * DN_ROWS
        yield (e * H + c0) * Bi, dbytes, down_bytes, "down rows"
        yield (t * k + i) * I * 4, 4 * I, h_bytes, "h row"
        yield (e * H + c0) * 4, 4 * DN_ROWS, E * H * 4, "down scales"


SHAPES = [(H, I) for H in (8, 16, 40, 80, 96, 160, 512, 1000, 2048, 2064, 2080)
          for I in (4, 8, 16, 24, 40, 64, 100, 512, 520, 2048)]


def test_tma_plan_is_aligned_and_in_bounds():
    checked = 0
    for H, I in SHAPES:
        E, T = 2, 2
        for k in (1, 3, 8, 12, 13):
            if gateup_ok(H, I):
                for off, size, buf, what in gateup_transfers(E, H, I, T, k):
                    _check(off, size, buf, f"H={H} I={I} {what}")
                    checked += 1
            if down_ok(H, I, k):
                for off, size, buf, what in down_transfers(E, H, I, T, k):
                    _check(off, size, buf, f"H={H} I={I} k={k} {what}")
                    checked += 1
    assert checked > 10000


def test_maple_shapes_take_the_bulk_copy_path():
    assert gateup_ok(2048, 512) and down_ok(2048, 512, 8) and prefetch_down(2048, 512)
    assert not down_ok(2048, 512, 13)
    # the shape that once issued a misaligned prefetch: the prefetch must now be off
    assert gateup_ok(40, 24) and not prefetch_down(40, 24)


# ---------------------------------------------------------------- fused layer kernel
# restates csrc/layer_decode.cu: C 16-CTA clusters (one CTA per SM, 16 warps); slot c < C
# on cluster c, slots C..k-1 split over the clusters by ranges of 40 intermediate columns
LC_CS, LC_WARPS, LC_CHUNKS, LC_MAX_E, LC_MAX_K, LC_MAX_SPLIT = 16, 16, 4, 256, 16, 2
LC_MAX_DOWN_LANE_BYTES, LC_UNIT, LC_MAX_UNITS, LC_SPLIT_COPY_ROWS = 4, 40, 4, 24
LUT16_BYTES = 243 * 16 * 8


def _a16(v):
    return (v + 15) // 16 * 16


def split_range(I, C, c):
    nu = (I + LC_UNIT - 1) // LC_UNIT
    u0, u1 = c * nu // C, (c + 1) * nu // C
    return u0 * LC_UNIT, min(u1 * LC_UNIT, I)


def split_pairs(n, r):
    per = (n + LC_CS - 1) // LC_CS
    p0 = min(r * per, n)
    p1 = min(p0 + per, n)
    return p0, p1, p0 // 8 * 8


def layer_smem(H, I, E):
    """Offsets of the union region and inside it, and the total bytes."""
    Bh, Bi = nbytes(H), nbytes(I)
    MB = (Bh + 31) // 32
    rg, rd = I // LC_CS, H // LC_CS
    o = (LUT16_BYTES + _a16(2 * H) + 4 * 32 * MB * 5 + 4 * 32 * LC_MAX_DOWN_LANE_BYTES * 5
         + 4 * LC_MAX_SPLIT * _a16(I) + 4 * LC_MAX_E + 4 * (rg + LC_MAX_SPLIT * LC_CS))
    un = _a16(o)
    cr = rg // LC_CHUNKS
    chunk = 2 * cr * Bh + 8 * cr
    dn = LC_CHUNKS * chunk
    dn_bytes = rd * Bi + 4 * rd
    sp = dn + dn_bytes
    sp_gu = 2 * LC_SPLIT_COPY_ROWS * Bh + 8 * LC_SPLIT_COPY_ROWS
    sp_bytes = sp_gu + dn_bytes
    total = un + sp + LC_MAX_SPLIT * sp_bytes
    return dict(un=un, cr=cr, chunk=chunk, dn=dn, sp=sp, sp_gu=sp_gu, sp_bytes=sp_bytes, total=total)


def layer_ok(H, I, E, k, C, smem_optin=232448):
    Bh, Bi = nbytes(H), nbytes(I)
    if H % 8 or H % (LC_CS * LC_WARPS) or H // LC_CS // LC_WARPS > 8:
        return False
    rd = H // LC_CS
    if (rd * Bi) % 16 or (H * Bi) % 16 or (Bi + 31) // 32 > LC_MAX_DOWN_LANE_BYTES:
        return False
    if I % 8 or I % (LC_CS * LC_WARPS) or I // LC_CS // LC_WARPS > 4:
        return False
    cr = I // LC_CS // LC_CHUNKS
    if (cr * Bh) % 16 or (I * Bh) % 16 or (8 * Bh) % 16 or (Bh + 31) // 32 > 13:
        return False
    if k < 1 or k > LC_MAX_K or k > E or E > LC_MAX_E or (E + LC_CS - 1) // LC_CS > LC_WARPS:
        return False
    C = min(k, C)
    nsplit = k - C
    if nsplit > LC_MAX_SPLIT:
        return False
    if nsplit:
        nu = (I + LC_UNIT - 1) // LC_UNIT
        if (nu + C - 1) // C > LC_MAX_UNITS:
            return False
        for c in range(C):
            c0, c1 = split_range(I, C, c)
            per = (c1 - c0 + LC_CS - 1) // LC_CS
            if per > LC_WARPS or per + 7 > LC_SPLIT_COPY_ROWS:
                return False
    return layer_smem(H, I, E)["total"] + 1024 <= smem_optin


def layer_transfers(E, H, I, k, C):
    """Every bulk copy of every CTA (global offset, size, global buffer size, what,
    shared destination, shared end), for any top-k outcome (experts 0 and E - 1 stand
    for all)."""
    Bh, Bi = nbytes(H), nbytes(I)
    L = layer_smem(H, I, E)
    un, total = L["un"], L["total"]
    C = min(k, C)
    nsplit = k - C
    rg, rd = I // LC_CS, H // LC_CS
    cr = L["cr"]
    for c in range(C):
        col0, col1 = split_range(I, C, c)
        for r in range(LC_CS):
            yield 0, LUT16_BYTES, LUT16_BYTES, "table", 0, total
            for e in (0, E - 1):
                for q in range(LC_CHUNKS):
                    r0 = e * I + r * rg + q * cr
                    base = un + q * L["chunk"]
                    yield r0 * Bh, cr * Bh, E * I * Bh, "gate chunk", base, total
                    yield r0 * Bh, cr * Bh, E * I * Bh, "up chunk", base + cr * Bh, total
                    yield r0 * 4, 4 * cr, E * I * 4, "gate scales", base + 2 * cr * Bh, total
                    yield r0 * 4, 4 * cr, E * I * 4, "up scales", base + 2 * cr * Bh + 4 * cr, total
                d0 = e * H + r * rd
                yield d0 * Bi, rd * Bi, E * H * Bi, "down rows", un + L["dn"], total
                yield d0 * 4, 4 * rd, E * H * 4, "down scales", un + L["dn"] + rd * Bi, total
                p0, p1, g0 = split_pairs(col1 - col0, r)
                for s in range(nsplit):
                    sp = un + L["sp"] + s * L["sp_bytes"]
                    if p1 > p0:
                        nrows = min(LC_SPLIT_COPY_ROWS, I - col0 - g0)
                        assert nrows % 8 == 0 and p1 - g0 <= nrows, (c, r, p0, p1, g0, nrows)
                        r0 = e * I + col0 + g0
                        yield r0 * Bh, nrows * Bh, E * I * Bh, "split gate rows", sp, sp + LC_SPLIT_COPY_ROWS * Bh
                        yield (r0 * Bh, nrows * Bh, E * I * Bh, "split up rows", sp + LC_SPLIT_COPY_ROWS * Bh,
                               sp + 2 * LC_SPLIT_COPY_ROWS * Bh)
                        sc = sp + 2 * LC_SPLIT_COPY_ROWS * Bh
                        yield r0 * 4, 4 * nrows, E * I * 4, "split gate scales", sc, sc + 4 * LC_SPLIT_COPY_ROWS
                        yield (r0 * 4, 4 * nrows, E * I * 4, "split up scales", sc + 4 * LC_SPLIT_COPY_ROWS,
                               sc + 8 * LC_SPLIT_COPY_ROWS)
                    d0 = e * H + r * rd
                    yield d0 * Bi, rd * Bi, E * H * Bi, "split down rows", sp + L["sp_gu"], total
                    yield d0 * 4, 4 * rd, E * H * 4, "split down scales", sp + L["sp_gu"] + rd * Bi, total


def test_fused_layer_plan_is_aligned_and_in_bounds():
    """Source and shared-memory destination of every copy 16-byte aligned, sizes multiples
    of 16, both inside their buffers, for cluster counts that take every slot whole
    (C >= k) or split one or two slots; the copies of one barrier stay below the 2^20 - 1
    byte count; a router row fits the 9 16-byte chunks per lane a warp holds in
    registers."""
    checked = 0
    for H, I in [(2048, 512), (1024, 512), (2048, 256), (4096, 512), (2048, 768)]:
        for E, k in [(256, 8), (32, 8), (8, 8), (250, 3), (16, 9), (256, 1), (256, 16)]:
            for C in (7, 8, 6, 5, 16):
                if k > E or not layer_ok(H, I, E, k, C):
                    continue
                assert LUT16_BYTES < 1 << 20 and (H // 8 + 31) // 32 <= 9
                for off, size, buf, what, dst, dst_end in layer_transfers(E, H, I, k, C):
                    _check(off, size, buf, f"layer H={H} I={I} E={E} k={k} C={C} {what}")
                    assert dst % 16 == 0 and dst + size <= dst_end, f"{what}: smem [{dst}, {dst + size})"
                    checked += 1
    assert checked > 5000
    assert layer_ok(2048, 512, 256, 8, 7) and layer_ok(2048, 512, 32, 8, 7) and layer_ok(2048, 512, 256, 8, 8)


def test_fused_layer_split_ranges_cover_every_column_once():
    """Split slot: the clusters' column ranges tile [0, I) in order, each range starts on
    a 40-column unit (8 whole gate/up row groups, 8 whole down-row bytes), and the CTAs'
    pair ranges tile each cluster's range."""
    for I in (512, 256):
        for C in (5, 6, 7, 8):
            cols = []
            for c in range(C):
                c0, c1 = split_range(I, C, c)
                assert c0 % LC_UNIT == 0 and c0 < c1 or c0 == c1
                pairs = []
                for r in range(LC_CS):
                    p0, p1, g0 = split_pairs(c1 - c0, r)
                    pairs += list(range(c0 + p0, c0 + p1))
                assert pairs == list(range(c0, c1))
                cols += list(range(c0, c1))
            assert cols == list(range(I))


def test_fused_layer_is_one_cta_per_sm_at_the_maple_shape():
    """The Maple layer's CTA (shared memory plus the SM's 1 KB reserve per CTA) does not
    fit twice into an SM's 228 KB, so the clusters never share SMs."""
    total = layer_smem(2048, 512, 256)["total"]
    assert 228 * 1024 < 2 * (total + 3440 + 1024) and total + 3440 + 1024 <= 227 * 1024


PK_MAX_WARPS = 8
PK_STAGE_BYTES = 4096
PK_MAX_K = 49152
PK_PAD = 32


def pack_plan(K, smem_optin=232448):
    """(rows per stage R, warps per CTA, dynamic shared memory) of the bulk-copy pack
    path, or None where the generic path runs; restates the launcher in csrc/pack.cu."""
    if K % 8 or K > PK_MAX_K:
        return None
    rowbytes = 2 * K
    R = 1
    while R < 32 and 2 * R * rowbytes <= PK_STAGE_BYTES:
        R *= 2
    per_warp = 2 * R * (rowbytes + PK_PAD)
    warps = min(PK_MAX_WARPS, (smem_optin - 1024) // per_warp)
    if warps < 1:
        return None
    return R, warps, per_warp * warps


def test_pack_plan_is_aligned_and_in_bounds():
    """ternarize_pack's bulk-copy path: warps stream blocks of R rows (one 2K-byte copy
    per row, into row slots of 2K + PK_PAD bytes) into one of two stages; every shared-
    memory read of a row (16-byte chunks for the sum, five words per ten-weight unit)
    stays inside its slot, and the ragged unit reads only the slot's zeroed pad."""
    for K in (8, 16, 40, 512, 520, 2048, 4104, 8192, 16384, 49152):
        R, warps, smem = pack_plan(K)
        assert R in (1, 2, 4, 8, 16, 32) and (R == 1 or R * 2 * K <= PK_STAGE_BYTES)
        assert smem + 128 + 1024 <= 232448
        stage = R * 2 * K  # bytes copied per full block
        for rows in (1, R - 1, R, 3 * R + 1, 37):
            if rows < 1:
                continue
            nblk = -(-rows // R)
            for b in range(nblk):
                n = min(R, rows - b * R)
                _check(b * R * 2 * K, n * 2 * K, rows * 2 * K, f"pack K={K} block {b}")
                assert n * 2 * K <= stage
        slot = 2 * K + PK_PAD
        assert slot % 16 == 0
        for w in range(warps):
            for st in (0, 1):
                for q in range(R):
                    off = (w * 2 + st) * R * slot + q * slot
                    assert off % 16 == 0 and off + slot <= smem
        assert 16 * (K // 8) <= 2 * K                  # row-sum chunks
        nb = nbytes(K)
        units = (nb + 1) // 2
        assert units == -(-K // 10)
        assert 4 * (5 * (units - 1) + 4) + 4 <= slot   # last unit's fifth word
    assert pack_plan(49160) is None and pack_plan(2052) is None
    assert pack_plan(512)[0] == 4 and pack_plan(2048)[0] == 1 and pack_plan(8)[0] == 32


def _trit_field(x, c2):
    y = ((x & 0x7FFF7FFF) + c2) & 0xFFFFFFFF
    return (y & ~x & 0x80008000) | ((~y >> 1) & 0x40004000)


def _mad_hi(a, b, c):
    return (((a * b) >> 32) + c) & 0xFFFFFFFF


def _pk_mul(lo, hi):
    return (lo << 18) | (hi << 2)


def _model_pack_unit(words, thr):
    """The integer packing of ten bf16 weights (five 32-bit words) at threshold thr,
    as csrc/pack.cu computes it; returns the two code bytes."""
    t16 = (int(np.float32(thr).view(np.uint32)) >> 16) & 0x7FFF
    c2 = (0x7FFF - t16) * 0x10001
    f = [_trit_field(int(w), c2) for w in words]
    a = _mad_hi(f[0], _pk_mul(1, 3), 0)
    a = _mad_hi(f[1], _pk_mul(9, 27), a)
    a = _mad_hi(f[2], _pk_mul(81, 0), a)
    b = _mad_hi(f[2], _pk_mul(0, 1), 0)
    b = _mad_hi(f[3], _pk_mul(3, 9), b)
    b = _mad_hi(f[4], _pk_mul(27, 81), b)
    return a & 0xFF, b & 0xFF


def test_integer_pack_unit_matches_the_oracle_packing():
    """The bit trick (bf16 threshold, digit fields, mad.hi sums) against the oracle's
    five-trits-per-byte packing of the trits q = sign(w) [|w| > thr], compared in fp32;
    thresholds are set on, just above and just below weight magnitudes."""
    import oracle
    rng = np.random.default_rng(5)
    checked = 0
    for trial in range(3000):
        kind = trial % 4
        if kind == 0:
            w = rng.normal(0, 0.02, 10).astype(np.float32)
        elif kind == 1:
            w = rng.choice([0.0, -0.0, 1e-38, -3e-39, 5.0, -5.0, np.inf, -np.inf], 10).astype(np.float32)
        else:
            w = (rng.normal(0, 1, 10) * 10.0 ** rng.integers(-30, 30)).astype(np.float32)
        bits = (w.view(np.uint32) >> 16).astype(np.uint32)  # truncate to bf16
        wb = (bits << 16).view(np.float32)
        mags = np.abs(wb[np.isfinite(wb)])
        base = float(mags[rng.integers(len(mags))]) if len(mags) else 0.0
        thr = np.float32(base)
        if kind == 3:
            thr = np.nextafter(thr, np.float32(np.inf)) if trial % 8 == 3 else np.nextafter(
                thr, np.float32(0))
        if not np.isfinite(thr):
            continue
        q = np.where(np.abs(wb) > thr, np.sign(wb), 0).astype(np.int8)
        words = [int(bits[2 * i]) | (int(bits[2 * i + 1]) << 16) for i in range(5)]
        got = _model_pack_unit(words, thr)
        want = oracle.pack(q[None, :])[0]
        assert got == (int(want[0]), int(want[1])), (w, thr, q)
        checked += 1
    assert checked > 2500


TC_ROWS, TC_KTILE = 128, 160
TC_LUT = 256 * 16 * 8        # 256 entries x 16 copies x 8 bytes
TC_STATIC_SMEM = 2048        # static shared memory of the streaming kernels, rounded up (ptxas -v)
TC_SMEM_OPTIN = 232448       # 227 KB of dynamic shared memory per CTA
PS_SUPER = 2                 # K tiles per ring stage
PS_KS = PS_SUPER * TC_KTILE  # K values per stage: 64 packed bytes of a row
PS_MAX_PACKED = 4


def tc_shape_ok(H, I):
    return (H % TC_ROWS == 0 and I % (TC_ROWS // 2) == 0 and H >= 128 and I >= 128
            and H <= 2080 and I <= 2080)


def ps_stage_b(nt):
    """A B stage: PS_KS / 16 core-matrix columns of 16 e4m3 values for 2 NT rows (hi, lo)."""
    return PS_KS // 16 * 2 * nt * 16


def ps_stages(nt):
    return 3 if nt <= 16 else 2


def ps_accs(nt):
    return min(256 // (2 * nt), 4)


def ps_pk_stride(rb):
    return -(-(TC_ROWS * rb) // 128) * 128


def ps_smem(rb, nt, npk):
    return TC_LUT + npk * ps_pk_stride(rb) + ps_stages(nt) * ps_stage_b(nt)


def ps_npk(rb, nt):
    """Packed-row buffers the launcher picks: as many as fit, from 4 down to 2."""
    n = PS_MAX_PACKED
    while n > 2 and ps_smem(rb, nt, n) > 227 * 1024:
        n -= 1
    return n


def test_streaming_tensor_plan_fits_and_is_aligned():
    """The streaming tcgen05 kernels (csrc/ffn_tensor.cu), for both token-tile widths
    (16 for decode batches, 64 for prefill) and every accepted shape: shared memory
    (decode table, 2-4 packed-row buffers, the B ring) within the opt-in limit with at
    least two packed buffers; the producers' word loads inside the allocation (five
    aligned words from byte 16 part + 64 st of a row, reading up to 3 bytes past);
    every MMA read of a B stage (2 core-matrix columns at 2NT * 16 B, 2NT / 8 row groups
    at 128 B) inside the stage; the tensor-memory plan (A stages of 80 columns below
    column 256, the accumulators of 2NT columns from 256 on, within 512); and each
    item's packed-row bulk copies (64 gate rows and 64 up rows, or 128 down rows)
    16-byte aligned and inside the expert's matrix."""
    shapes = [(H, I) for H in range(128, 2081, 128) for I in range(128, 2081, 64)]
    for nt in (16, 64):
        n = 2 * nt
        sb = ps_stage_b(nt)
        assert ps_stages(nt) * (PS_KS // 4) <= 256            # A stages below column 256
        assert 256 + ps_accs(nt) * n <= 512 and ps_accs(nt) >= 2
        for q in range(PS_KS // 32):
            assert q * 2 * n * 16 + n * 16 + (n // 8 - 1) * 128 + 127 < sb
        for H, I in shapes:
            assert tc_shape_ok(H, I)
            for rb, rows, mtot, K in ((nbytes(H), TC_ROWS // 2, I, H), (nbytes(I), TC_ROWS, H, I)):
                npk = ps_npk(rb, nt)
                total = ps_smem(rb, nt, npk)
                assert npk >= 2 and total + TC_STATIC_SMEM <= TC_SMEM_OPTIN, (H, I, nt, total)
                assert K % 32 == 0                             # MMAs cover whole K = 32 steps
                ns = -(-K // PS_KS)
                # farthest producer read: last row of the last buffer, last stage, last part
                far = TC_LUT + (npk - 1) * ps_pk_stride(rb) + ((127 * rb + PS_KS // 5 * (ns - 1) + 48) & ~3) + 20
                assert far <= total, (H, I, nt)
                size = rows * rb
                assert size % 16 == 0
                for e in (0, 1, 7):
                    for m0 in range(0, mtot, rows):
                        _check((e * mtot + m0) * rb, size, (e + 1) * mtot * rb, f"stream H={H} I={I}")
    assert not tc_shape_ok(2080, 512) and not tc_shape_ok(2048, 520) and not tc_shape_ok(40, 24)
    assert not tc_shape_ok(128, 64)


def test_tensor_path_operand_blocks_are_aligned_and_in_bounds():
    """The B operand of a tile lives in global memory as [K / 16][2NT][16] e4m3 bytes
    (the split kernels write x and h that way: hi rows 0..NT-1, lo rows NT..2NT-1); each
    ring stage is one bulk copy of up to PS_KS / 16 chunks, fewer at the K tail.  Every
    copy starts on a 16-byte boundary, has a multiple of 16 bytes and stays inside its
    tile's block, and the split kernels' 8-byte stores stay inside the block too."""
    for nt in (16, 64):
        for K in (128, 192, 384, 512, 2048):
            block = K * 2 * nt
            ns = -(-K // PS_KS)
            covered = 0
            for st in range(ns):
                left = K // 16 - st * (PS_KS // 16)
                nb = min(left, PS_KS // 16) * 2 * nt * 16
                off = st * ps_stage_b(nt)
                for tile in (0, 1, 5):
                    _check(tile * block + off, nb, (tile + 1) * block, f"B nt={nt} K={K} st={st}")
                assert nb <= ps_stage_b(nt)
                covered += nb
            assert covered == block
            for c in range(K // 8):
                for row in (0, nt - 1, nt, 2 * nt - 1):
                    off = (c >> 1) * 2 * nt * 16 + (c & 1) * 8 + row * 16
                    assert off % 8 == 0 and off + 8 <= block


def _e4m3(v):
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).float().numpy()


def test_two_e4m3_split_is_exact_for_bf16_rows():
    """The grouped kernels feed bf16 rows to fp8 MMAs as v = s (hi + lo), with s a power
    of two that puts the row's largest magnitude in [2^7, 2^8), hi = e4m3(v / s) and lo =
    e4m3(v / s - hi) (round to nearest even).  Over every finite bf16 value of that
    range and below: the split is exact once |v / s| >= 2^-2, and below that it loses at
    most half of e4m3's smallest step, 2^-10."""
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # every non-negative finite bf16
    v = (bits << 16).view(np.float32)
    v = v[v < 256.0]
    v = np.concatenate([v, -v])
    hi = _e4m3(v)
    lo = _e4m3(v - hi)
    err = np.abs(hi.astype(np.float64) + lo - v)
    big = np.abs(v) >= 0.25
    assert np.all(err[big] == 0)
    assert err.max() <= 2.0 ** -10
    assert np.abs(hi).max() <= 256.0


def test_grouped_decode_table_matches_the_oracle_unpack():
    """The grouped kernels decode a packed byte c through a 256-entry table whose entry
    c holds the e4m3 values of the five trits (0xB8 = -1, 0x00 = 0, 0x38 = +1) in bytes
    0-4, and five zeros for the invalid codes 243..255; a word of the row's four next
    e4m3 values is assembled by byte permutes.  The table's construction (digits by
    repeated division) against oracle.unpack for every byte value, and the permutes
    against plain concatenation."""
    import oracle

    e4m3_of = {-1: 0xB8, 0: 0x00, 1: 0x38}
    table = []
    for c in range(256):
        b = [0] * 5
        if c < 243:
            code = c
            for t in range(5):
                b[t] = e4m3_of[code % 3 - 1]
                code //= 3
        table.append(b)
    for c in range(256):
        if c > 242:
            assert table[c] == [0] * 5
            continue
        trits = oracle.unpack(np.array([[c]], np.uint8), 5)[0]
        assert table[c] == [e4m3_of[int(t)] for t in trits], c

    def perm(x, y, sel):
        src = [(x >> (8 * i)) & 0xFF for i in range(4)] + [(y >> (8 * i)) & 0xFF for i in range(4)]
        return sum(src[(sel >> (4 * i)) & 7] << (8 * i) for i in range(4))

    def word(bs):
        return sum(v << (8 * i) for i, v in enumerate(bs))
    rng = np.random.default_rng(0)
    for _ in range(300):
        codes = rng.integers(0, 256, 4)
        en = [(word(table[c][:4]), table[c][4]) for c in codes]
        flat = sum((table[c] for c in codes), [])
        words = [en[0][0], perm(en[0][1], en[1][0], 0x6540),
                 perm(perm(en[1][0], en[1][1], 0x0043), en[2][0], 0x5410),
                 perm(perm(en[2][0], en[2][1], 0x0432), en[3][0], 0x4210),
                 perm(en[3][0], en[3][1], 0x4321)]
        assert words == [word(flat[4 * i:4 * i + 4]) for i in range(5)]


def test_grouped_decode_81_entry_table_matches_the_oracle_unpack():
    """The alternative decode that was measured (slower, not used by the kernels): a byte
    c = low + 81 q4 with q4 = (c * 203) >> 14, the first four trits from entry `low` of
    an 82-entry table (entry 81 all zero, taken for the invalid codes 243..255), the
    fifth from q4 (byte q4 of 0x003800B8 as e4m3: -1, 0, +1, and 0 for q4 = 3).  Every
    byte value against oracle.unpack, so the comparison of the two decodes compared
    correct ones."""
    import oracle

    e4m3_of = {-1: 0xB8, 0: 0x00, 1: 0x38}
    table = []
    for low in range(82):
        vals = [0] * 4
        if low < 81:
            code = low
            for t in range(4):
                vals[t] = e4m3_of[code % 3 - 1]
                code //= 3
        table.append(vals)
    for c in range(256):
        q4 = (c * 203) >> 14
        entry = 81 if c > 242 else c - 81 * q4
        assert 0 <= entry < 82 and q4 <= 3
        vals = table[entry] + [(0x003800B8 >> (8 * q4)) & 0xFF]
        if c > 242:
            assert vals == [0] * 5, c
            continue
        trits = oracle.unpack(np.array([[c]], np.uint8), 5)[0]
        assert vals == [e4m3_of[int(t)] for t in trits], (c, vals, trits)


def test_packed_magnitude_fold_has_no_cross_half_borrow():
    """The already-ternary pack folds a word of two bf16 into packed 16-bit minima of
    (|w| - 1) mod 2^16 as ((w | 0x80008000) - 0x00010001) ^ 0x80008000: every magnitude
    in either half (any sign bit, any value in the other half) maps to |w| - 1, and 0 to
    0xffff, above every other."""
    m = np.arange(0x8000, dtype=np.uint64)
    for sign in (0, 1):
        for other in (0x0000, 0x0001, 0x7fff, 0x8000, 0xffff):
            for low_half in (True, False):
                h = (m | (sign << 15)).astype(np.uint64)
                w = (h | (other << 16)) if low_half else ((h << 16) | other)
                f = (((w | 0x80008000) - 0x00010001) ^ 0x80008000) & 0xffffffff
                got = (f & 0xffff) if low_half else (f >> 16)
                want = np.where(m == 0, 0xffff, m - 1)
                assert np.array_equal(got, want), (sign, other, low_half)
