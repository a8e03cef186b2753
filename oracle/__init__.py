"""CPU oracle for the quantized KV cache -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It is a ctypes wrapper around the plain
C file ``kvq_oracle.c`` (scalar fp32 quantization exactly as the formula
states it, fp64 attention), which shares no code with the CUDA library and
never calls it.  The state of one head (one batch entry, one KV head) lives in
numpy arrays owned by :class:`OracleHead`; every method maps to one C routine.

The C code cites the pages it follows; the numbers checked against it are in
``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_HDR = os.path.join(_HERE, "kvq_oracle.h")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "libkvq_oracle.so")

KIVI = 0
INNERQ = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle (default: oracle/_build/libkvq_oracle.so), gcc with
    no floating-point contraction and no fast-math."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    newest = max(os.path.getmtime(src), os.path.getmtime(_HDR))
    if force or not os.path.exists(out) or os.path.getmtime(out) < newest:
        tmp = out + ".%d.tmp" % os.getpid()
        cmd = ["cc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-I", _HERE, "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


class _Head(ctypes.Structure):
    _fields_ = [
        ("d", ctypes.c_int32), ("bits", ctypes.c_int32), ("scheme", ctypes.c_int32),
        ("k_group", ctypes.c_int32), ("v_group", ctypes.c_int32),
        ("residual", ctypes.c_int32), ("n_sink", ctypes.c_int32), ("k_normalize", ctypes.c_int32),
        ("cap", ctypes.c_int64), ("n_quant", ctypes.c_int64), ("n_resid", ctypes.c_int64),
        ("n_sink_used", ctypes.c_int64), ("n_flush", ctypes.c_int64),
        ("k_u", ctypes.c_void_p), ("v_u", ctypes.c_void_p),
        ("k_scale", ctypes.c_void_p), ("k_zero", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p),
        ("k_sym", ctypes.c_void_p), ("v_sym", ctypes.c_void_p),
        ("k_res", ctypes.c_void_p), ("v_res", ctypes.c_void_p),
        ("k_sink", ctypes.c_void_p), ("v_sink", ctypes.c_void_p),
        ("k_norm", ctypes.c_void_p),
        ("v_queue", ctypes.c_int32), ("n_vquant", ctypes.c_int64),
        ("meta_f16", ctypes.c_int32), ("outliers", ctypes.c_int32),
        ("k_oidx", ctypes.c_void_p), ("v_oidx", ctypes.c_void_p),
        ("k_oval", ctypes.c_void_p), ("v_oval", ctypes.c_void_p),
    ]


def _declare(L):
    P = ctypes.c_void_p
    L.orc_rounding_is_nearest.restype = ctypes.c_int
    L.orc_half_to_float.argtypes = [ctypes.c_uint16]
    L.orc_half_to_float.restype = ctypes.c_float
    L.orc_float_to_half.argtypes = [ctypes.c_float]
    L.orc_float_to_half.restype = ctypes.c_uint16
    L.orc_quant_asym_f16.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int64]
    L.orc_quant_sym_f16.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int64]
    L.orc_quant_asym.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int64]
    L.orc_quant_sym.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P, ctypes.c_int64]
    L.orc_choose_symmetric.argtypes = [ctypes.c_float, ctypes.c_float, ctypes.c_int]
    L.orc_choose_symmetric.restype = ctypes.c_int
    L.orc_prefill.argtypes = [ctypes.POINTER(_Head), P, P, ctypes.c_int64]
    L.orc_append.argtypes = [ctypes.POINTER(_Head), P, P]
    L.orc_attend.argtypes = [ctypes.POINTER(_Head), P, ctypes.c_double, P]
    L.orc_attend_rope.argtypes = [ctypes.POINTER(_Head), P, ctypes.c_double, ctypes.c_double,
                                  ctypes.c_int64, P]
    L.orc_pack.argtypes = [P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P]
    L.orc_select_outliers.argtypes = [P, ctypes.c_int, ctypes.c_int, P]
    L.orc_pack_modes.argtypes = [P, ctypes.c_int64, P]
    if not L.orc_rounding_is_nearest():
        raise RuntimeError("oracle needs round-to-nearest-even")
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every oracle call to another build of the C file for the duration
    (used by the tests that plant mistakes in a copy of the oracle)."""
    global _lib
    lib()
    old = _lib
    _lib = _declare(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = old


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def _f16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float16:
        raise TypeError("expected fp16, got %s" % a.dtype)
    return a


def half_to_float(h: int) -> float:
    return lib().orc_half_to_float(int(h))


def float_to_half(f: float) -> int:
    """IEEE binary32 -> binary16 bits, round to nearest even."""
    return int(lib().orc_float_to_half(float(f)))


def quant_asym(x, bits: int, meta_f16: bool = False):
    """Asymmetric quantization of one group x (float32): (scale, zero, codes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s, z = ctypes.c_float(), ctypes.c_float()
    u = np.zeros(x.size, dtype=np.uint8)
    fn = lib().orc_quant_asym_f16 if meta_f16 else lib().orc_quant_asym
    fn(_ptr(x), x.size, bits, ctypes.addressof(s), ctypes.addressof(z), _ptr(u), 1)
    return np.float32(s.value), np.float32(z.value), u


def quant_sym(x, bits: int, meta_f16: bool = False):
    """Symmetric quantization of one group x (float32): (scale, zero, codes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    s, z = ctypes.c_float(), ctypes.c_float()
    u = np.zeros(x.size, dtype=np.uint8)
    fn = lib().orc_quant_sym_f16 if meta_f16 else lib().orc_quant_sym
    fn(_ptr(x), x.size, bits, ctypes.addressof(s), ctypes.addressof(z), _ptr(u), 1)
    return np.float32(s.value), np.float32(z.value), u


def choose_symmetric(mn: float, mx: float, bits: int) -> bool:
    return bool(lib().orc_choose_symmetric(float(mn), float(mx), bits))


def select_outliers(row, k: int) -> np.ndarray:
    """Channels (ascending) of the k largest-magnitude elements of one fp16 row."""
    row = _f16(row)
    idx = np.zeros(k, np.uint16)
    lib().orc_select_outliers(_ptr(row.view(np.uint16)), row.size, k, _ptr(idx))
    return idx


def pack(u: np.ndarray, bits: int) -> np.ndarray:
    """Pack code rows [n][d] (one code per byte) into [n][d*bits/8] bytes."""
    u = np.ascontiguousarray(u, dtype=np.uint8)
    n, d = u.shape
    out = np.zeros((n, d * bits // 8), dtype=np.uint8)
    lib().orc_pack(_ptr(u), n, d, bits, _ptr(out))
    return out


def pack_modes(sym: np.ndarray, n_words: int | None = None) -> np.ndarray:
    """Pack mode flags (token-major, one per group) into uint32 words."""
    sym = np.ascontiguousarray(sym, dtype=np.uint8).reshape(-1)
    n = sym.size
    words = (n + 31) // 32 if n_words is None else n_words
    out = np.zeros(max(words, (n + 31) // 32), dtype=np.uint32)
    lib().orc_pack_modes(_ptr(sym), n, _ptr(out))
    return out[:words]


class OracleHead:
    """Cache state of one head, driven through the C oracle."""

    def __init__(self, d, bits, scheme, k_group, v_group, residual, n_sink, cap, k_norm=False,
                 v_queue=False, meta_f16=False, outliers=0):
        if d > 256 or bits not in (2, 4, 8) or d % (8 // bits):
            raise ValueError("unsupported head_dim / bits")
        if k_norm and scheme != INNERQ:
            raise ValueError("key normalization is an InnerQ option")
        if v_queue and scheme != KIVI:
            raise ValueError("the value queue is a KIVI option")
        if outliers and (scheme != KIVI or not 0 < outliers <= 8 or outliers >= d):
            raise ValueError("outliers: KIVI only, 1..8 per token")
        self.d, self.bits, self.scheme = d, bits, scheme
        self.k_group, self.v_group = k_group, v_group
        self.residual, self.n_sink, self.cap = residual, n_sink, cap
        if scheme == KIVI:
            kg_rows, kg_cols = (cap + k_group - 1) // k_group, d
        else:
            kg_rows, kg_cols = cap, d // k_group
        self.k_u = np.zeros((cap, d), np.uint8)
        self.v_u = np.zeros((cap, d), np.uint8)
        self.k_scale = np.zeros((kg_rows, kg_cols), np.float32)
        self.k_zero = np.zeros((kg_rows, kg_cols), np.float32)
        self.v_scale = np.zeros((cap, d // v_group), np.float32)
        self.v_zero = np.zeros((cap, d // v_group), np.float32)
        self.k_sym = np.zeros((cap, d // k_group if scheme == INNERQ else 1), np.uint8)
        self.v_sym = np.zeros((cap, d // v_group), np.uint8)
        self.k_res = np.zeros((max(residual, 1), d), np.uint16)
        self.v_res = np.zeros((max(residual, 1), d), np.uint16)
        self.k_sink = np.zeros((max(n_sink, 1), d), np.uint16)
        self.v_sink = np.zeros((max(n_sink, 1), d), np.uint16)
        self.k_norm = np.ones(d, np.float32)  # per-channel key factors (InnerQ option)
        no = max(outliers, 1)
        self.k_oidx = np.zeros((cap, no), np.uint16)   # per-token outlier channels
        self.v_oidx = np.zeros((cap, no), np.uint16)
        self.k_oval = np.zeros((cap, no), np.uint16)   # and their fp16 values
        self.v_oval = np.zeros((cap, no), np.uint16)
        s = _Head()
        s.d, s.bits, s.scheme = d, bits, scheme
        s.k_group, s.v_group, s.residual, s.n_sink = k_group, v_group, residual, n_sink
        s.cap = cap
        s.k_normalize = 1 if k_norm else 0
        s.v_queue = 1 if v_queue else 0
        s.meta_f16 = 1 if meta_f16 else 0
        s.outliers = int(outliers)
        for name in ("k_u", "v_u", "k_scale", "k_zero", "v_scale", "v_zero", "k_sym",
                     "v_sym", "k_res", "v_res", "k_sink", "v_sink", "k_norm", "k_oidx", "v_oidx",
                     "k_oval", "v_oval"):
            setattr(s, name, _ptr(getattr(self, name)))
        self._s = s

    @classmethod
    def for_workload(cls, w, cap=None):
        cap = w.max_ctx() if cap is None else cap
        return cls(w.head_dim, w.bits, w.scheme, w.k_group, w.v_group, w.residual,
                   w.n_sink, cap, k_norm=getattr(w, "k_norm", False),
                   v_queue=getattr(w, "v_queue", False),
                   meta_f16=getattr(w, "meta_f16", False),
                   outliers=getattr(w, "outliers", 0))

    # counters
    def save_state(self):
        """The counters and fp16 residual/window rows (enough to rewind appends:
        the rows they overwrite are rewritten in the same order)."""
        s = self._s
        return ((s.n_quant, s.n_resid, s.n_sink_used, s.n_flush, s.n_vquant),
                self.k_res.copy(), self.v_res.copy())

    def load_state(self, state) -> None:
        (nq, nr, ns, nf, nvq), kr, vr = state
        s = self._s
        s.n_quant, s.n_resid, s.n_sink_used, s.n_flush, s.n_vquant = nq, nr, ns, nf, nvq
        self.k_res[...] = kr
        self.v_res[...] = vr

    n_quant = property(lambda self: self._s.n_quant)
    n_resid = property(lambda self: self._s.n_resid)
    n_sink_used = property(lambda self: self._s.n_sink_used)
    n_flush = property(lambda self: self._s.n_flush)

    @property
    def n_vquant(self) -> int:
        """Values held quantized (the keys' count unless KIVI's value queue)."""
        return self._s.n_vquant if self._s.v_queue else self._s.n_quant

    def prefill(self, K, V) -> None:
        K, V = _f16(K), _f16(V)
        if lib().orc_prefill(ctypes.byref(self._s), _ptr(K.view(np.uint16)),
                             _ptr(V.view(np.uint16)), K.shape[0]) != 0:
            raise ValueError("prefill exceeds capacity")

    def append(self, k, v) -> None:
        k, v = _f16(k), _f16(v)
        if lib().orc_append(ctypes.byref(self._s), _ptr(k.view(np.uint16)),
                            _ptr(v.view(np.uint16))) != 0:
            raise ValueError("append exceeds capacity")

    def attend(self, q, tau: float) -> np.ndarray:
        """fp64 attention output [d] of one query head q ([d] fp16)."""
        q = _f16(q)
        out = np.zeros(self.d, np.float64)
        if lib().orc_attend(ctypes.byref(self._s), _ptr(q.view(np.uint16)), float(tau),
                            _ptr(out)) != 0:
            raise MemoryError("oracle attention")
        return out

    def attend_rope(self, q, tau: float, base: float, pos0: int = 0) -> np.ndarray:
        """fp64 attention output [d] over keys cached before the rotary
        embedding: the j-th token held sits at position pos0 + j, the query
        (pre-RoPE, [d] fp16) at pos0 + n - 1."""
        q = _f16(q)
        out = np.zeros(self.d, np.float64)
        if lib().orc_attend_rope(ctypes.byref(self._s), _ptr(q.view(np.uint16)), float(tau),
                                 float(base), int(pos0), _ptr(out)) != 0:
            raise MemoryError("oracle attention")
        return out

    # views in the library's storage layout, for byte-for-byte comparison
    def packed_k(self) -> np.ndarray:
        return pack(self.k_u[: self.n_quant], self.bits)

    def packed_v(self) -> np.ndarray:
        return pack(self.v_u[: self.n_vquant], self.bits)

    def k_meta(self):
        """(scale, zero) of the quantized keys: KIVI [n_quant/G][d], InnerQ [n_quant][d/G]."""
        rows = self.n_quant // self.k_group if self.scheme == KIVI else self.n_quant
        return self.k_scale[:rows], self.k_zero[:rows]

    def key_norms(self) -> np.ndarray:
        """Per-channel key factors of the one-shot normalization ([d] fp32)."""
        return self.k_norm.copy()

    def v_meta(self):
        return self.v_scale[: self.n_vquant], self.v_zero[: self.n_vquant]

    def residual_tokens(self):
        """fp16 residual (KIVI) or window (InnerQ) keys and values, oldest first
        (with KIVI's value queue the values are value_queue())."""
        n = self.n_resid
        return self.k_res[:n].view(np.float16), self.v_res[:n].view(np.float16)

    def value_queue(self) -> np.ndarray:
        """fp16 values not yet quantized, oldest first."""
        n = self.n_quant + self.n_resid - self.n_vquant
        return self.v_res[:n].view(np.float16)

    def sink_tokens(self):
        n = self.n_sink_used
        return self.k_sink[:n].view(np.float16), self.v_sink[:n].view(np.float16)
