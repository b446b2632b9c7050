"""C-ABI tests that need no GPU: the library loads, exports every symbol the header
declares, names every status, and rejects bad arguments on the host before any CUDA
call (so these run on a machine without a GPU)."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "maple.h")


@pytest.fixture(scope="module")
def lib():
    from ternary_weight_moe_02_b300 import build_lib
    path = build_lib.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"MAPLE_API\s+[\w\s\*]+?\b(maple_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("maple_ternarize_pack", "maple_route_topk", "maple_moe_ffn",
                     "maple_group_tokens", "maple_moe_ffn_workspace_size", "maple_unpack",
                     "maple_status_string", "maple_last_error", "maple_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_exposes_every_declared_symbol():
    from ternary_weight_moe_02_b300 import maple
    for name in declared_functions():
        assert name in maple.EXPORTED and callable(getattr(maple, name)), name


def test_library_exports_only_the_boundary():
    import subprocess
    from ternary_weight_moe_02_b300 import build_lib
    out = subprocess.run(["nm", "-D", "--defined-only", build_lib.LIB], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    lib.maple_status_string.restype = ctypes.c_char_p
    names = {0: b"MAPLE_OK", -1: b"MAPLE_ERR_INVALID_ARG", -2: b"MAPLE_ERR_UNSUPPORTED_SHAPE",
             -3: b"MAPLE_ERR_MISALIGNED", -4: b"MAPLE_ERR_CUDA", -5: b"MAPLE_ERR_TIMEOUT",
             -6: b"MAPLE_ERR_BAD_CODE", -7: b"MAPLE_ERR_WORKSPACE"}
    for code, name in names.items():
        assert lib.maple_status_string(code) == name
    assert lib.maple_status_string(-99) == b"MAPLE_ERR_UNKNOWN"
    lib.maple_version.restype = ctypes.c_int
    assert lib.maple_version() >= 100


# Fake device addresses: validation must reject or accept them without dereferencing.
A16 = 0x10000
MIS = 0x10001
P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64


def _last(lib):
    lib.maple_last_error.restype = ctypes.c_char_p
    return lib.maple_last_error().decode()


def test_ternarize_pack_validation(lib):
    f = lib.maple_ternarize_pack
    f.argtypes = [P, I64, I64, P, P, P]
    assert f(A16, 4, 0, A16, A16, None) == -1
    assert "K=0" in _last(lib)
    assert f(A16, -1, 8, A16, A16, None) == -1
    assert f(A16, 4, (1 << 24) + 1, A16, A16, None) == -2
    assert f(None, 4, 8, A16, A16, None) == -1
    assert f(MIS, 4, 8, A16, A16, None) == -3
    assert f(A16, 4, 8, A16, A16 + 2, None) == -3
    assert f(A16, 0, 8, None, None, None) == 0  # empty: a no-op, no CUDA call


def test_route_topk_validation(lib):
    f = lib.maple_route_topk
    f.argtypes = [P, P, P, I32, I32, I32, I32, P, P, P, P]
    assert f(A16, A16, None, 4, 2048, 256, 0, A16, A16, A16, None) == -1
    assert f(A16, A16, None, 4, 2048, 8, 9, A16, A16, A16, None) == -1  # k > E
    assert f(A16, A16, None, 4, 2048, 2048, 8, A16, A16, A16, None) == -2  # E > 1024
    assert f(A16, A16, None, 4, 2048, 256, 33, A16, A16, A16, None) == -2  # k > 32
    assert f(A16, A16, None, 4, 2048, 256, 8, None, A16, A16, None) == -1
    assert f(A16 + 8, A16, None, 4, 2048, 256, 8, A16, A16, A16, None) == -3
    assert f(A16, A16, None, 0, 2048, 256, 8, None, None, None, None) == 0


def test_group_tokens_validation(lib):
    f = lib.maple_group_tokens
    f.argtypes = [P, I32, I32, I32, P, P, P, P]
    assert f(A16, 4, 0, 256, A16, A16, A16, None) == -1
    assert f(A16, 4, 8, 2000, A16, A16, A16, None) == -2
    assert f(A16, 4, 8, 256, None, A16, A16, None) == -1
    assert f(A16 + 2, 4, 8, 256, A16, A16, A16, None) == -3


def _experts(lib, E=256, H=2048, I=512, clamp=7.0, gate=A16):
    from ternary_weight_moe_02_b300.maple import maple_experts
    return maple_experts(gate, A16, A16, A16, A16, A16, E, H, I, clamp)


def test_moe_ffn_validation(lib):
    from ternary_weight_moe_02_b300.maple import maple_experts
    ws_size = lib.maple_moe_ffn_workspace_size
    ws_size.argtypes = [I32, I32, ctypes.POINTER(maple_experts)]
    ws_size.restype = ctypes.c_size_t
    f = lib.maple_moe_ffn
    f.argtypes = [ctypes.POINTER(maple_experts), P, P, P, I32, I32, P, P, ctypes.c_size_t, P]
    ex = _experts(lib)
    need = ws_size(64, 8, ctypes.byref(ex))
    # h for 512 slots x 512 rows fp32 dominates
    assert need >= 64 * 8 * 512 * 4
    assert need % 256 == 0
    assert ws_size(1, 8, ctypes.byref(ex)) < need
    ok_args = (A16, A16, A16, 64, 8, A16, A16, need, None)
    assert f(None, *ok_args) == -1
    assert f(ctypes.byref(_experts(lib, clamp=0.0)), *ok_args) == -1
    assert f(ctypes.byref(_experts(lib, clamp=float("nan"))), *ok_args) == -1
    assert f(ctypes.byref(_experts(lib, H=4096)), *ok_args) == -2
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 65, A16, A16, need, None) == -2
    assert f(ctypes.byref(_experts(lib, gate=A16 + 8)), *ok_args) == -3
    assert f(ctypes.byref(ex), A16 + 8, A16, A16, 64, 8, A16, A16, need, None) == -3
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 8, A16, A16, need - 1, None) == -7
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 8, A16, None, need, None) == -7
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 8, None, A16, need, None) == -1
    assert f(ctypes.byref(ex), None, None, None, 0, 8, None, None, 0, None) == 0
    assert f(ctypes.byref(_experts(lib, clamp=math.inf)), None, None, None, 0, 8, None, None, 0,
             None) == 0


def test_moe_layer_validation(lib):
    from ternary_weight_moe_02_b300.maple import maple_experts
    wsz = lib.maple_moe_layer_workspace_size
    wsz.argtypes = [I32, I32, ctypes.POINTER(maple_experts)]
    wsz.restype = ctypes.c_size_t
    f = lib.maple_moe_layer
    f.argtypes = [P, P, P, ctypes.POINTER(maple_experts), I32, I32, P, P, P, P, P, ctypes.c_size_t, P]
    ex = _experts(lib)
    need = wsz(1, 8, ctypes.byref(ex))
    ffn = lib.maple_moe_ffn_workspace_size
    ffn.argtypes = [I32, I32, ctypes.POINTER(maple_experts)]
    ffn.restype = ctypes.c_size_t
    # 256 bytes of counters, then the larger of the FFN workspace and the fused kernel's
    # per-slot outputs: C (1 + k - C) rows of H fp32 for C clusters, bounded over C <= k
    groups = max(C * (1 + 8 - C) for C in range(1, 9))
    assert groups == 20
    assert need == 256 + max(ffn(1, 8, ctypes.byref(ex)), groups * 2048 * 4)
    assert wsz(64, 8, ctypes.byref(ex)) == 256 + ffn(64, 8, ctypes.byref(ex))
    good = (A16, A16, None, ctypes.byref(ex), 1, 8, A16, A16, A16, A16, A16, need, None)
    assert f(*good[:3], None, *good[4:]) == -1
    assert f(A16, A16, None, ctypes.byref(ex), 1, 0, A16, A16, A16, A16, A16, need, None) == -1
    assert f(A16, A16, None, ctypes.byref(ex), 1, 257, A16, A16, A16, A16, A16, need, None) == -1
    assert f(A16, A16, None, ctypes.byref(ex), 1, 33, A16, A16, A16, A16, A16, need, None) == -2
    assert f(A16 + 8, A16, None, ctypes.byref(ex), 1, 8, A16, A16, A16, A16, A16, need, None) == -3
    assert f(A16, A16, None, ctypes.byref(ex), 1, 8, A16, A16, A16, A16, A16, need - 1, None) == -7
    assert f(A16, A16, None, ctypes.byref(ex), 1, 8, None, A16, A16, A16, A16, need, None) == -1
    assert f(None, None, None, ctypes.byref(ex), 0, 8, None, None, None, None, None, 0, None) == 0


def test_moe_ffn_ex_path_validation(lib):
    """maple_moe_ffn_ex: an unknown path is an invalid argument; the tensor path on a
    shape its kernels do not take is an unsupported shape (both before any launch)."""
    from ternary_weight_moe_02_b300.maple import maple_experts
    wsz = lib.maple_moe_ffn_workspace_size_ex
    wsz.argtypes = [I32, I32, ctypes.POINTER(maple_experts), I32]
    wsz.restype = ctypes.c_size_t
    f = lib.maple_moe_ffn_ex
    f.argtypes = [ctypes.POINTER(maple_experts), P, P, P, I32, I32, P, I32, P, ctypes.c_size_t, P]
    ex = _experts(lib)
    need = max(wsz(64, 8, ctypes.byref(ex), p) for p in (0, 1, 2))
    assert wsz(64, 8, ctypes.byref(ex), 1) < wsz(64, 8, ctypes.byref(ex), 2)
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 8, A16, 3, A16, need, None) == -1
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 8, A16, -1, A16, need, None) == -1
    odd = _experts(lib, H=2000)
    assert wsz(64, 8, ctypes.byref(odd), 2) == 0
    assert f(ctypes.byref(odd), A16, A16, A16, 64, 8, A16, 2, A16, need, None) == -2
    # the workspace check follows the named path
    cores = wsz(64, 8, ctypes.byref(ex), 1)
    assert f(ctypes.byref(ex), A16, A16, A16, 64, 8, A16, 2, A16, cores, None) == -7


def test_test_inject_validation_and_launch_error(lib):
    """maple_test_inject rejects unknown kinds and poll counts; an injected launch error
    is reported by the next launching call (before any CUDA call) and only once."""
    f = lib.maple_test_inject
    f.argtypes = [I32, I32]
    assert f(7, 0) == -1
    assert f(1, 0) == -1 and f(1, 100001) == -1
    assert f(0, 0) == 0
    route = lib.maple_route_topk
    route.argtypes = [P, P, P, I32, I32, I32, I32, P, P, P, P]
    last = lib.maple_last_error
    last.restype = ctypes.c_char_p
    assert f(2, 0) == 0
    assert route(A16, A16, None, 1, 64, 8, 2, A16, A16, A16, None) == -4
    assert b"injected launch failure" in last()
    # consumed: the next call gets past the hook (here it then fails on the missing GPU
    # or launches, but not with the injected message)
    route(A16, A16, None, 1, 64, 8, 2, A16, A16, A16, None)
    assert b"injected" not in last()
    # validation errors come first and leave a pending injection in place
    assert f(2, 0) == 0
    assert route(A16, A16, None, 1, 64, 0, 2, A16, A16, A16, None) == -1
    assert route(A16, A16, None, 1, 64, 8, 2, A16, A16, A16, None) == -4
    assert f(0, 0) == 0


def test_cache_fetch_validation(lib):
    """maple_cache_fetch rejects, before any launch: a null pool or cache, pool and slots
    of different H or I, more routed slots than cache slots, arrays that are not whole
    16-byte chunks, misaligned arrays and a short workspace."""
    from ternary_weight_moe_02_b300.maple import maple_expert_cache, maple_experts
    wsz = lib.maple_cache_fetch_workspace_size
    wsz.argtypes = [I32, I32]
    wsz.restype = ctypes.c_size_t
    assert wsz(1, 8) == 4 * (1 + 16) and wsz(0, 8) == 4
    f = lib.maple_cache_fetch
    f.argtypes = [ctypes.POINTER(maple_experts), ctypes.POINTER(maple_expert_cache), P, I32, I32, P, P,
                  ctypes.c_size_t, P]

    def cache(C=12, H=2048, I=512, gate=A16):
        return maple_expert_cache(maple_experts(gate, A16, A16, A16, A16, A16, C, H, I, 7.0), A16, A16, A16, A16)
    pool = _experts(lib, E=32)
    good = (ctypes.byref(pool), ctypes.byref(cache()), A16, 1, 8, A16, A16, wsz(1, 8), None)
    assert f(None, *good[1:]) == -1
    assert f(good[0], None, *good[2:]) == -1
    assert f(good[0], ctypes.byref(cache(H=1024)), *good[2:]) == -1
    assert f(good[0], ctypes.byref(cache(C=7)), *good[2:]) == -2       # T*k = 8 > C
    assert f(ctypes.byref(_experts(lib, E=2000)), *good[1:]) == -2
    odd = _experts(lib, E=32, H=13, I=7)
    assert f(ctypes.byref(odd), ctypes.byref(cache(H=13, I=7)), *good[2:]) == -2
    assert f(good[0], ctypes.byref(cache(gate=A16 + 8)), *good[2:]) == -3
    assert f(*good[:7], wsz(1, 8) - 4, None) == -7
    assert f(good[0], good[1], A16, 0, 8, A16, A16, 0, None) == 0
