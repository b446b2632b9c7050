"""CPU oracle for the ternary MoE FFN step (plain C, fp64), with numpy wrappers.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU-baseline leg
of the benchmark may import this package; the product library never does.  The C
source (``maple_oracle.c``) shares no code with the CUDA library.

Passages each function follows are cited in the C source; in short:
  * ternarize / ternary_exact / pack / unpack -- "Maple-Preview: a 20B reasoning model where 97% of
    the weights are -1, 0, or +1", sections "The claim, verified from the bytes" and
    "The 5.31 GB claim reconciles";
  * route -- same page, "The claim, verified from the bytes" (router kept in full
    precision, 8 of 256 experts);
  * moe_ffn -- same page, "The shipped code does no quantization" (MapleMLP forward)
    and "IA de 20B Rodando a 120 tok/s no iPhone", "Pesos ternarios" (skip / add /
    subtract).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "maple_oracle.c")
_LIB = os.path.join(_HERE, "libmaple_oracle.so")
_lock = threading.Lock()
_lib = None

OK = 0
BAD_ARG = -1
BAD_CODE = -6


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (single-threaded, -O2, strict IEEE double)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
             "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            lib.oracle_ternarize.argtypes = [P, I64, I64, P, P]
            lib.oracle_ternary_exact.argtypes = [P, I64, I64, P, P, P]
            lib.oracle_pack.argtypes = [P, I64, I64, P]
            lib.oracle_unpack.argtypes = [P, I64, I64, P]
            lib.oracle_route.argtypes = [P, P, P, I64, I64, I64, I64, P, P, P]
            lib.oracle_group.argtypes = [P, I64, I64, I64, P, P, P]
            lib.oracle_moe_ffn.argtypes = [P, P, P, P, P, P, I64, I64, I64, ctypes.c_double,
                                           P, P, P, I64, I64, P]
            lib.oracle_packed_row_bytes.argtypes = [I64]
            lib.oracle_packed_row_bytes.restype = I64
            for name in ("oracle_ternarize", "oracle_ternary_exact", "oracle_pack", "oracle_unpack", "oracle_route",
                         "oracle_group", "oracle_moe_ffn"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return a


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: oracle status {status}")
        self.status = status


def packed_row_bytes(K: int) -> int:
    return int(_load().oracle_packed_row_bytes(K))


def ternarize(w_bits: np.ndarray):
    """bf16 bits [rows, K] -> (trits int8 [rows, K], scales fp32 [rows])."""
    w = _bf16_bits(w_bits)
    rows, K = w.shape
    q = np.empty((rows, K), np.int8)
    s = np.empty(rows, np.float32)
    st = _load().oracle_ternarize(_ptr(w), rows, K, _ptr(q), _ptr(s))
    if st != OK:
        raise OracleError(st, "ternarize")
    return q, s


def ternary_exact(w_bits: np.ndarray):
    """bf16 bits [rows, K] of already-ternary rows -> (trits int8 [rows, K] = sign(w),
    scales fp32 [rows] = max|w|, number of rows that are not ternary)."""
    w = _bf16_bits(w_bits)
    rows, K = w.shape
    q = np.empty((rows, K), np.int8)
    s = np.empty(rows, np.float32)
    bad = np.zeros(1, np.int64)
    st = _load().oracle_ternary_exact(_ptr(w), rows, K, _ptr(q), _ptr(s), _ptr(bad))
    if st != OK:
        raise OracleError(st, "ternary_exact")
    return q, s, int(bad[0])


def pack(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.int8)
    rows, K = q.shape
    out = np.empty((rows, packed_row_bytes(K)), np.uint8)
    st = _load().oracle_pack(_ptr(q), rows, K, _ptr(out))
    if st != OK:
        raise OracleError(st, "pack")
    return out


def unpack(packed: np.ndarray, K: int, check: bool = True):
    """Packed bytes [rows, ceil(K/5)] -> trits int8 [rows, K] (and the status)."""
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    rows = p.shape[0]
    assert p.shape[1] == packed_row_bytes(K)
    q = np.empty((rows, K), np.int8)
    st = _load().oracle_unpack(_ptr(p), rows, K, _ptr(q))
    if check and st != OK:
        raise OracleError(st, "unpack")
    return (q, st) if not check else q


def ternarize_pack(w_bits: np.ndarray):
    q, s = ternarize(w_bits)
    return pack(q), s


def route(x_bits: np.ndarray, wr_bits: np.ndarray, bias, k: int):
    """x bf16 [T,H], Wr bf16 [E,H], bias fp64 [E] or None -> (logits fp64 [T,E],
    idx int32 [T,k], w fp64 [T,k])."""
    x = _bf16_bits(x_bits)
    wr = _bf16_bits(wr_bits)
    T, H = x.shape
    E, H2 = wr.shape
    assert H == H2
    logits = np.empty((T, E), np.float64)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    st = _load().oracle_route(_ptr(x), _ptr(wr), None if b is None else _ptr(b), T, H, E, k,
                              _ptr(logits), _ptr(idx), _ptr(w))
    if st != OK:
        raise OracleError(st, "route")
    return logits, idx, w


def group(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(T * k, np.int32)
    st = _load().oracle_group(_ptr(idx), T, k, E, _ptr(counts), _ptr(offsets), _ptr(perm))
    if st != OK:
        raise OracleError(st, "group")
    return counts, offsets, perm


def moe_ffn(gate, up, down, s_gate, s_up, s_down, x_bits, idx, w, clamp: float = 7.0):
    """Packed experts (gate/up [E,I,ceil(H/5)], down [E,H,ceil(I/5)], fp32 scales),
    x bf16 [T,H], idx int32 [T,k], w [T,k] -> y fp64 [T,H]."""
    gate = np.ascontiguousarray(gate, np.uint8)
    up = np.ascontiguousarray(up, np.uint8)
    down = np.ascontiguousarray(down, np.uint8)
    s_gate = np.ascontiguousarray(s_gate, np.float32)
    s_up = np.ascontiguousarray(s_up, np.float32)
    s_down = np.ascontiguousarray(s_down, np.float32)
    x = _bf16_bits(x_bits)
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    E, I, _ = gate.shape
    H = down.shape[1]
    T, k = idx.shape
    assert x.shape == (T, H) and w.shape == (T, k)
    assert gate.shape == (E, I, packed_row_bytes(H)) and up.shape == gate.shape
    assert down.shape == (E, H, packed_row_bytes(I))
    assert s_gate.shape == (E, I) and s_up.shape == (E, I) and s_down.shape == (E, H)
    y = np.empty((T, H), np.float64)
    st = _load().oracle_moe_ffn(_ptr(gate), _ptr(up), _ptr(down), _ptr(s_gate), _ptr(s_up),
                                _ptr(s_down), E, H, I, float(clamp), _ptr(x), _ptr(idx), _ptr(w),
                                T, k, _ptr(y))
    if st != OK:
        raise OracleError(st, "moe_ffn")
    return y
