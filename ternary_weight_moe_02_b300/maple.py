"""Thin ctypes binding of libmaple.so (C-ABI in include/maple.h).

Argument marshalling only: every step runs in the library's CUDA kernels.  Functions
carry the C names; tensors are caller-owned torch CUDA tensors, passed by data
pointer, and work is enqueued on the given stream (default: torch's current stream).
A non-OK status raises MapleError.  Importing this module fails loudly when the
library has not been built (python -m ternary_weight_moe_02_b300.build_lib).
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmaple.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libmaple.so is missing at {_LIB_PATH}; build it with "
        "`python -m ternary_weight_moe_02_b300.build_lib` (there is no fallback path)")
_lib = ctypes.CDLL(_LIB_PATH)

MAPLE_OK = 0
MAPLE_ERR_INVALID_ARG = -1
MAPLE_ERR_UNSUPPORTED_SHAPE = -2
MAPLE_ERR_MISALIGNED = -3
MAPLE_ERR_CUDA = -4
MAPLE_ERR_TIMEOUT = -5
MAPLE_ERR_BAD_CODE = -6
MAPLE_ERR_WORKSPACE = -7

MAPLE_INJECT_NONE = 0
MAPLE_INJECT_COPY_STALL = 1
MAPLE_INJECT_LAUNCH_ERROR = 2

MAPLE_FFN_AUTO = 0
MAPLE_FFN_CORES = 1
MAPLE_FFN_TENSOR = 2
_FFN_PATHS = {"auto": MAPLE_FFN_AUTO, "cores": MAPLE_FFN_CORES, "tensor": MAPLE_FFN_TENSOR}

EXPORTED = ("maple_version", "maple_status_string", "maple_last_error",
            "maple_check_device_status", "maple_ternarize_pack", "maple_pack_ternary",
            "maple_unpack", "maple_route_topk", "maple_group_tokens",
            "maple_moe_ffn_workspace_size", "maple_moe_ffn", "maple_moe_ffn_workspace_size_ex",
            "maple_moe_ffn_ex", "maple_moe_layer_workspace_size",
            "maple_moe_layer", "maple_moe_layer_host", "maple_moe_ffn_static_scratch",
            "maple_test_inject", "maple_cache_fetch_workspace_size", "maple_cache_fetch")


class maple_experts(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("s_gate", ctypes.c_void_p), ("s_up", ctypes.c_void_p), ("s_down", ctypes.c_void_p),
                ("E", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
                ("clamp", ctypes.c_float)]


class maple_expert_cache(ctypes.Structure):
    _fields_ = [("slots", maple_experts), ("slot_of", ctypes.c_void_p), ("expert_of", ctypes.c_void_p),
                ("last_use", ctypes.c_void_p), ("stats", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_lib.maple_version.restype = ctypes.c_int
_lib.maple_status_string.restype = ctypes.c_char_p
_lib.maple_status_string.argtypes = [ctypes.c_int]
_lib.maple_last_error.restype = ctypes.c_char_p
_lib.maple_check_device_status.argtypes = [_P]
_lib.maple_check_device_status.restype = ctypes.c_int
_lib.maple_ternarize_pack.argtypes = [_P, _I64, _I64, _P, _P, _P]
_lib.maple_unpack.argtypes = [_P, _P, _I64, _I64, _P, _P, _P]
_lib.maple_pack_ternary.argtypes = [_P, _I64, _I64, _P, _P, _P, _P]
_lib.maple_route_topk.argtypes = [_P, _P, _P, _I32, _I32, _I32, _I32, _P, _P, _P, _P]
_lib.maple_group_tokens.argtypes = [_P, _I32, _I32, _I32, _P, _P, _P, _P]
_lib.maple_moe_ffn_workspace_size.argtypes = [_I32, _I32, ctypes.POINTER(maple_experts)]
_lib.maple_moe_ffn_workspace_size.restype = ctypes.c_size_t
_lib.maple_moe_ffn.argtypes = [ctypes.POINTER(maple_experts), _P, _P, _P, _I32, _I32, _P, _P,
                               ctypes.c_size_t, _P]
_lib.maple_moe_ffn_workspace_size_ex.argtypes = [_I32, _I32, ctypes.POINTER(maple_experts), _I32]
_lib.maple_moe_ffn_workspace_size_ex.restype = ctypes.c_size_t
_lib.maple_moe_ffn_ex.argtypes = [ctypes.POINTER(maple_experts), _P, _P, _P, _I32, _I32, _P, _I32, _P,
                                  ctypes.c_size_t, _P]
_lib.maple_moe_layer_workspace_size.argtypes = [_I32, _I32, ctypes.POINTER(maple_experts)]
_lib.maple_moe_layer_workspace_size.restype = ctypes.c_size_t
_lib.maple_moe_layer.argtypes = [_P, _P, _P, ctypes.POINTER(maple_experts), _I32, _I32, _P, _P, _P,
                                 _P, _P, ctypes.c_size_t, _P]
_lib.maple_moe_layer.restype = ctypes.c_int
_lib.maple_moe_layer_host.argtypes = [_P, _P, _P, _P, ctypes.POINTER(maple_experts), _I32, _I32, _P, _P, _P,
                                      _P, _P, _P, ctypes.c_size_t, _P]
_lib.maple_moe_layer_host.restype = ctypes.c_int
_lib.maple_moe_ffn_static_scratch.argtypes = [ctypes.POINTER(maple_experts), _P, _P, _P, _I32,
                                              _I32, _P, _P]
_lib.maple_cache_fetch_workspace_size.argtypes = [_I32, _I32]
_lib.maple_cache_fetch_workspace_size.restype = ctypes.c_size_t
_lib.maple_cache_fetch.argtypes = [ctypes.POINTER(maple_experts), ctypes.POINTER(maple_expert_cache), _P, _I32,
                                   _I32, _P, _P, ctypes.c_size_t, _P]
_lib.maple_cache_fetch.restype = ctypes.c_int
_lib.maple_test_inject.argtypes = [_I32, _I32]
_lib.maple_test_inject.restype = ctypes.c_int
for _n in ("maple_ternarize_pack", "maple_unpack", "maple_route_topk", "maple_group_tokens",
           "maple_moe_ffn", "maple_moe_ffn_ex", "maple_moe_ffn_static_scratch"):
    getattr(_lib, _n).restype = ctypes.c_int


class MapleError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.maple_last_error().decode(errors="replace")
        name = _lib.maple_status_string(status).decode()
        super().__init__(f"{where}: {name}: {msg}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def _check(status: int, where: str):
    if status != MAPLE_OK:
        raise MapleError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _expect(t, dtype, shape, name):
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


def packed_row_bytes(K: int) -> int:
    return (K + 4) // 5


def maple_version() -> int:
    return _lib.maple_version()


def maple_status_string(status: int) -> str:
    return _lib.maple_status_string(status).decode()


def maple_last_error() -> str:
    return _lib.maple_last_error().decode(errors="replace")


def maple_check_device_status(stream=None):
    """Synchronise the stream and raise if a kernel recorded a device-side error."""
    _check(_lib.maple_check_device_status(_stream(stream)), "maple_check_device_status")


def maple_test_inject(kind: int, value: int = 0):
    """One-shot failure injection for tests (MAPLE_INJECT_*; see include/maple.h)."""
    _check(_lib.maple_test_inject(kind, value), "maple_test_inject")


def maple_ternarize_pack(W, packed, scales, stream=None):
    """W bf16 [rows, K] -> packed uint8 [rows, ceil(K/5)], scales fp32 [rows]."""
    rows, K = W.shape
    _expect(W, torch.bfloat16, (rows, K), "W")
    _expect(packed, torch.uint8, (rows, packed_row_bytes(K)), "packed")
    _expect(scales, torch.float32, (rows,), "scales")
    _check(_lib.maple_ternarize_pack(_ptr(W), rows, K, _ptr(packed), _ptr(scales), _stream(stream)),
           "maple_ternarize_pack")


def maple_pack_ternary(W, packed, scales, bad_rows=None, stream=None):
    """W bf16 [rows, K] with already-ternary rows -> packed uint8 [rows, ceil(K/5)],
    scales fp32 [rows] = max|w|; bad_rows: optional int32 [1] counter of rows that are
    not ternary (added to)."""
    rows, K = W.shape
    _expect(W, torch.bfloat16, (rows, K), "W")
    _expect(packed, torch.uint8, (rows, packed_row_bytes(K)), "packed")
    _expect(scales, torch.float32, (rows,), "scales")
    if bad_rows is not None:
        _expect(bad_rows, torch.int32, (1,), "bad_rows")
    _check(_lib.maple_pack_ternary(_ptr(W), rows, K, _ptr(packed), _ptr(scales), _ptr(bad_rows),
                                   _stream(stream)), "maple_pack_ternary")


def maple_unpack(packed, scales, K, W_out, bad_codes=None, stream=None):
    rows = packed.shape[0]
    _expect(packed, torch.uint8, (rows, packed_row_bytes(K)), "packed")
    _expect(scales, torch.float32, (rows,), "scales")
    _expect(W_out, torch.float32, (rows, K), "W_out")
    if bad_codes is not None:
        _expect(bad_codes, torch.int32, (1,), "bad_codes")
    _check(_lib.maple_unpack(_ptr(packed), _ptr(scales), rows, K, _ptr(W_out), _ptr(bad_codes),
                             _stream(stream)), "maple_unpack")


def maple_route_topk(x, Wr, bias, k, logits, idx, w, stream=None):
    """x bf16 [T,H], Wr bf16 [E,H], bias fp32 [E] or None -> logits [T,E], idx [T,k], w [T,k]."""
    T, H = x.shape
    E = Wr.shape[0]
    _expect(x, torch.bfloat16, (T, H), "x")
    _expect(Wr, torch.bfloat16, (E, H), "Wr")
    if bias is not None:
        _expect(bias, torch.float32, (E,), "bias")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(w, torch.float32, (T, k), "w")
    _check(_lib.maple_route_topk(_ptr(x), _ptr(Wr), _ptr(bias), T, H, E, k, _ptr(logits), _ptr(idx),
                                 _ptr(w), _stream(stream)), "maple_route_topk")


def maple_group_tokens(idx, E, counts, offsets, perm, stream=None):
    T, k = idx.shape
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(counts, torch.int32, (E,), "counts")
    _expect(offsets, torch.int32, (E + 1,), "offsets")
    _expect(perm, torch.int32, (T * k,), "perm")
    _check(_lib.maple_group_tokens(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm),
                                   _stream(stream)), "maple_group_tokens")


class Experts:
    """Packed expert weights of one layer (caller-owned tensors) and their C struct."""

    def __init__(self, gate, up, down, s_gate, s_up, s_down, clamp: float = 7.0):
        E, I, bh = gate.shape
        H = down.shape[1]
        _expect(gate, torch.uint8, (E, I, packed_row_bytes(H)), "gate")
        _expect(up, torch.uint8, (E, I, packed_row_bytes(H)), "up")
        _expect(down, torch.uint8, (E, H, packed_row_bytes(I)), "down")
        _expect(s_gate, torch.float32, (E, I), "s_gate")
        _expect(s_up, torch.float32, (E, I), "s_up")
        _expect(s_down, torch.float32, (E, H), "s_down")
        self.tensors = (gate, up, down, s_gate, s_up, s_down)
        self.E, self.H, self.I, self.clamp = E, H, I, clamp
        self.struct = maple_experts(gate.data_ptr(), up.data_ptr(), down.data_ptr(),
                                    s_gate.data_ptr(), s_up.data_ptr(), s_down.data_ptr(), E, H, I,
                                    clamp)

    @property
    def packed_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in self.tensors)


class ExpertCache:
    """C expert slots in device memory plus the cache's tables (caller-owned tensors,
    initialised as include/maple.h asks: slot_of and expert_of -1, last_use and stats
    0).  `experts` is the slots seen as a layer of C experts, for maple_moe_ffn."""

    def __init__(self, C: int, E: int, H: int, I: int, clamp: float = 7.0, device="cuda"):
        bh, bi = packed_row_bytes(H), packed_row_bytes(I)
        self.C, self.E, self.H, self.I = C, E, H, I
        self.gate = torch.empty((C, I, bh), dtype=torch.uint8, device=device)
        self.up = torch.empty((C, I, bh), dtype=torch.uint8, device=device)
        self.down = torch.empty((C, H, bi), dtype=torch.uint8, device=device)
        self.s_gate = torch.empty((C, I), dtype=torch.float32, device=device)
        self.s_up = torch.empty((C, I), dtype=torch.float32, device=device)
        self.s_down = torch.empty((C, H), dtype=torch.float32, device=device)
        self.experts = Experts(self.gate, self.up, self.down, self.s_gate, self.s_up, self.s_down, clamp=clamp)
        self.slot_of = torch.full((E,), -1, dtype=torch.int32, device=device)
        self.expert_of = torch.full((C,), -1, dtype=torch.int32, device=device)
        self.last_use = torch.zeros((C,), dtype=torch.int32, device=device)  # uint32 bits
        self.stats = torch.zeros((4,), dtype=torch.int32, device=device)     # uint32 bits
        self.struct = maple_expert_cache(self.experts.struct, self.slot_of.data_ptr(), self.expert_of.data_ptr(),
                                         self.last_use.data_ptr(), self.stats.data_ptr())

    def counters(self) -> dict:
        st = self.stats.cpu().tolist()
        return {"steps": st[0], "hits": st[1], "misses": st[2], "experts_copied": st[3]}


def maple_cache_fetch_workspace_size(T: int, k: int) -> int:
    return int(_lib.maple_cache_fetch_workspace_size(T, k))


def maple_cache_fetch(pool: Experts, cache: ExpertCache, idx, idx_slot, ws, stream=None):
    """Make the experts idx routes to resident in the cache; idx_slot (int32 [T, k]) gets
    their slots.  pool: Experts whose tensors the device can read (pinned host memory or
    device memory)."""
    T, k = idx.shape
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(idx_slot, torch.int32, (T, k), "idx_slot")
    if pool.H != cache.H or pool.I != cache.I or pool.E != cache.E:
        raise ValueError("pool and cache differ in E, H or I")
    for t in pool.tensors:
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("a host pool must be pinned memory")
    _check(_lib.maple_cache_fetch(ctypes.byref(pool.struct), ctypes.byref(cache.struct), _ptr(idx), T, k,
                                  _ptr(idx_slot), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream(stream)), "maple_cache_fetch")


def maple_moe_ffn_workspace_size(T: int, k: int, experts: Experts) -> int:
    return int(_lib.maple_moe_ffn_workspace_size(T, k, ctypes.byref(experts.struct)))


def maple_moe_ffn(experts: Experts, x, idx, w, y, ws, stream=None):
    """y fp32 [T,H] = sum_i w[t,i] * expert_{idx[t,i]}(x_t); ws = uint8 workspace tensor."""
    T, H = x.shape
    k = idx.shape[1]
    _expect(x, torch.bfloat16, (T, experts.H), "x")
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(w, torch.float32, (T, k), "w")
    _expect(y, torch.float32, (T, experts.H), "y")
    _check(_lib.maple_moe_ffn(ctypes.byref(experts.struct), _ptr(x), _ptr(idx), _ptr(w), T, k,
                              _ptr(y), _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                              _stream(stream)), "maple_moe_ffn")


def _path(path) -> int:
    return _FFN_PATHS[path] if isinstance(path, str) else int(path)


def maple_moe_ffn_workspace_size_ex(T: int, k: int, experts: Experts, path) -> int:
    """Workspace of maple_moe_ffn_ex on `path` ("auto", "cores", "tensor" or the
    MAPLE_FFN_* value); 0 when the call would be rejected."""
    return int(_lib.maple_moe_ffn_workspace_size_ex(T, k, ctypes.byref(experts.struct), _path(path)))


def maple_moe_ffn_ex(experts: Experts, x, idx, w, y, path, ws, stream=None):
    """maple_moe_ffn on the named path ("auto", "cores", "tensor" or MAPLE_FFN_*)."""
    T, H = x.shape
    k = idx.shape[1]
    _expect(x, torch.bfloat16, (T, experts.H), "x")
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(w, torch.float32, (T, k), "w")
    _expect(y, torch.float32, (T, experts.H), "y")
    _check(_lib.maple_moe_ffn_ex(ctypes.byref(experts.struct), _ptr(x), _ptr(idx), _ptr(w), T, k,
                                 _ptr(y), _path(path), _ptr(ws),
                                 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "maple_moe_ffn_ex")


def maple_moe_layer_workspace_size(T: int, k: int, experts: Experts) -> int:
    return int(_lib.maple_moe_layer_workspace_size(T, k, ctypes.byref(experts.struct)))


def maple_moe_layer(x, Wr, bias, experts: Experts, k, logits, idx, w, y, ws, stream=None):
    """Route + FFN for one layer step.  ws: uint8 tensor of maple_moe_layer_workspace_size
    bytes whose first 256 bytes are zero before the first call (torch.zeros does it)."""
    _check_layer(x, Wr, bias, experts, k, logits, idx, w, y)
    T = x.shape[0]
    _check(_lib.maple_moe_layer(_ptr(x), _ptr(Wr), _ptr(bias), ctypes.byref(experts.struct), T, k,
                                _ptr(logits), _ptr(idx), _ptr(w), _ptr(y), _ptr(ws),
                                0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "maple_moe_layer")


def _check_layer(x, Wr, bias, experts, k, logits, idx, w, y):
    T = x.shape[0]
    E = Wr.shape[0]
    _expect(x, torch.bfloat16, (T, experts.H), "x")
    _expect(Wr, torch.bfloat16, (experts.E, experts.H), "Wr")
    if bias is not None:
        _expect(bias, torch.float32, (E,), "bias")
    _expect(logits, torch.float32, (T, E), "logits")
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(w, torch.float32, (T, k), "w")
    _expect(y, torch.float32, (T, experts.H), "y")


def _layer_host_args(x_host, x_dev, Wr, bias, experts, k, logits, idx, w, y, y_host, ws, stream):
    _check_layer(x_dev, Wr, bias, experts, k, logits, idx, w, y)
    T = x_dev.shape[0]
    _expect(x_host, torch.bfloat16, (T, experts.H), "x_host")
    _expect(y_host, torch.float32, (T, experts.H), "y_host")
    if x_host.is_cuda or y_host.is_cuda:
        raise ValueError("x_host and y_host must be host tensors (pinned for asynchronous copies)")
    return (_ptr(x_host), _ptr(x_dev), _ptr(Wr), _ptr(bias), ctypes.byref(experts.struct), T, k, _ptr(logits),
            _ptr(idx), _ptr(w), _ptr(y), _ptr(y_host), _ptr(ws),
            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream))


def maple_moe_layer_host(x_host, x_dev, Wr, bias, experts: Experts, k, logits, idx, w, y, y_host, ws,
                         stream=None):
    """maple_moe_layer with the tokens in host memory: x_host (bf16 [T,H]) is copied
    into x_dev, the layer runs, and y reaches y_host (fp32 [T,H]) as well, all enqueued
    on the stream; pinned host buffers are copied by kernels chained with the layer's
    (a single token's fused launch writes y_host itself)."""
    _check(_lib.maple_moe_layer_host(*_layer_host_args(x_host, x_dev, Wr, bias, experts, k, logits, idx, w,
                                                       y, y_host, ws, stream)), "maple_moe_layer_host")


class BoundCall:
    """One C call with its arguments checked and marshalled once: calling the object
    makes the C call and nothing else (for decode loops, where per-call checks would
    take longer than the microseconds-long step).  The tensors must stay alive and
    unchanged in shape while the object is used."""

    def __init__(self, fn, args, where, keep):
        self._fn, self._args, self._where, self._keep = fn, args, where, keep

    def __call__(self):
        st = self._fn(*self._args)
        if st != MAPLE_OK:
            raise MapleError(st, self._where)


def bind_moe_layer_host(x_host, x_dev, Wr, bias, experts: Experts, k, logits, idx, w, y, y_host, ws,
                        stream=None) -> BoundCall:
    """maple_moe_layer_host with its arguments bound (see BoundCall)."""
    args = _layer_host_args(x_host, x_dev, Wr, bias, experts, k, logits, idx, w, y, y_host, ws, stream)
    return BoundCall(_lib.maple_moe_layer_host, args, "maple_moe_layer_host",
                     (x_host, x_dev, Wr, bias, experts, logits, idx, w, y, y_host, ws))


def maple_moe_ffn_static_scratch(experts: Experts, x, idx, w, y, stream=None):
    """maple_moe_ffn for callers that cannot allocate: the library's static per-GPU
    scratch array stands in for the workspace (maple_moe_ffn_workspace_size must not
    exceed 2 MiB).  Calls that overlap on the GPU share that array and must be
    serialised by the caller."""
    T, H = x.shape
    k = idx.shape[1]
    _expect(x, torch.bfloat16, (T, experts.H), "x")
    _expect(idx, torch.int32, (T, k), "idx")
    _expect(w, torch.float32, (T, k), "w")
    _expect(y, torch.float32, (T, experts.H), "y")
    _check(_lib.maple_moe_ffn_static_scratch(ctypes.byref(experts.struct), _ptr(x), _ptr(idx),
                                             _ptr(w), T, k, _ptr(y), _stream(stream)),
           "maple_moe_ffn_static_scratch")


def clamp_none() -> float:
    """Clamp value that turns the Maple clamps off (plain SwiGLU)."""
    return math.inf
