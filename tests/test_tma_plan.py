"""CPU model of the bulk-copy (TMA) plan of the FFN kernels.

For every shape the dispatch predicates accept, enumerate each 1-D bulk copy and L2
bulk prefetch the kernels issue (offsets relative to 16-byte aligned bases, sizes) and
check that all of them start on a 16-byte boundary, have a size that is a multiple of
16 and stay inside their buffer.  The formulas restate those in csrc/ffn_decode.cu;
a misaligned bulk copy faults the GPU, so this runs on the CPU first."""
import itertools

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
LD_ITEM_ROWS, LD_DOWN_ROWS, LD_MAX_ITEMS, LD_MAX_ROUTER_ROWS, LD_MAX_K, LD_WARPS = 8, 16, 8, 8, 12, 16


def layer_ok(H, I, E, k, G=148, smem_optin=232448):
    Bh, Bi = nbytes(H), nbytes(I)
    if H % LD_DOWN_ROWS or H // LD_DOWN_ROWS > G:
        return False
    if I % LD_ITEM_ROWS or I % 4 or Bh % 2 or (Bh + 31) // 32 > 13:
        return False
    nr = (E + G - 1) // G
    nitems = (k * (I // LD_ITEM_ROWS) + G - 1) // G
    if k > LD_MAX_K or E > 1024 or nr > LD_MAX_ROUTER_ROWS or nr > LD_WARPS or nitems > LD_MAX_ITEMS:
        return False
    if (Bi + 31) // 32 > 4:
        return False
    MB = (Bh + 31) // 32
    total = (31104 + nr * 2 * H + 2 * H + 4 * 32 * MB * 5 + nitems * (2 * LD_ITEM_ROWS * Bh + 8 * LD_ITEM_ROWS)
             + k * (LD_DOWN_ROWS * Bi + 4 * LD_DOWN_ROWS) + k * 4 * I + 4 * ((E + 3) // 4 * 4))
    return total <= smem_optin - 1024


def layer_transfers(E, H, I, k, G=148):
    """Every bulk copy of every CTA, for any top-k outcome (all experts e < E)."""
    Bh, Bi = nbytes(H), nbytes(I)
    ngroups = I // LD_ITEM_ROWS
    nr = (E + G - 1) // G
    nitems = (k * ngroups + G - 1) // G
    for c in range(G):
        for j in range(nr):
            if c + j * G < E:
                yield (c + j * G) * H * 2, 2 * H, E * H * 2, "router row"
        yield 0, 2 * H, H * 2, "x"
        for n in range(nitems):
            jj = c + n * G
            if jj >= k * ngroups:
                continue
            r0 = (jj % ngroups) * LD_ITEM_ROWS
            for e in (0, E - 1):
                yield (e * I + r0) * Bh, LD_ITEM_ROWS * Bh, E * I * Bh, "gate item"
                yield (e * I + r0) * 4, 4 * LD_ITEM_ROWS, E * I * 4, "gate scales"
        if c < H // LD_DOWN_ROWS:
            c0 = c * LD_DOWN_ROWS
            for e in (0, E - 1):
                yield (e * H + c0) * Bi, LD_DOWN_ROWS * Bi, E * H * Bi, "down group"
                yield (e * H + c0) * 4, 4 * LD_DOWN_ROWS, E * H * 4, "down scales"
            for i in range(k):
                yield i * I * 4, 4 * I, k * I * 4, "h"


def test_fused_layer_plan_is_aligned_and_in_bounds():
    checked = 0
    for H, I in [(2048, 512), (160, 40), (512, 64), (2080, 520), (1024, 640), (96, 16)]:
        for E, k in [(256, 8), (32, 8), (8, 8), (1024, 12), (300, 3)]:
            if k > E or not layer_ok(H, I, E, k):
                continue
            for off, size, buf, what in layer_transfers(E, H, I, k):
                _check(off, size, buf, f"layer H={H} I={I} E={E} k={k} {what}")
                checked += 1
    assert checked > 1000
    assert layer_ok(2048, 512, 256, 8) and layer_ok(2048, 512, 32, 8)


def test_pack_plan_is_aligned_and_in_bounds():
    """ternarize_pack's bulk-copy path: one copy of 2K bytes per row (K % 8 == 0, base
    16-byte aligned), into one of two row buffers of a warp; the last byte's third
    32-bit load may read up to 4 bytes past the row, inside the 16-byte pad."""
    for K in (8, 16, 40, 512, 520, 2048, 4104, 8192):
        rows = 37
        for r in range(rows):
            _check(r * 2 * K, 2 * K, rows * 2 * K, f"pack K={K} row {r}")
        nb = nbytes(K)
        last_word = (5 * (nb - 1)) // 2 + 2          # third word of the last byte
        assert 4 * (last_word + 1) <= 2 * K + 16 + 2 * K  # within the two buffers + pad
        assert 4 * (last_word + 1) - 2 * K <= 16       # at most 16 bytes past one row
