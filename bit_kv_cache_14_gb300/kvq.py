"""Python binding of libkvq (argument marshalling only).

Every call goes through the C ABI declared in include/kvq.h; all arithmetic
runs in the library's CUDA kernels.  PyTorch provides device memory and the
current stream.  There is no fallback: if ``_build/libkvq.so`` is missing the
first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

KVQ_OK = 0
KVQ_EINVAL = -1
KVQ_EUNSUPPORTED = -2
KVQ_ECAPACITY = -3
KVQ_EALIGN = -4
KVQ_ECUDA = -5
KVQ_ETIMEOUT = -6
KIVI = 0
INNERQ = 1
INNERQ_KNORM = 2  # InnerQ with the one-shot per-channel key normalization
META_F16 = 1      # config.flags: scales and zero points stored in fp16
VALUE_QUEUE = 2   # config.flags: KIVI values leave the fp16 residual one at a time
RAGGED = 4        # config.flags: every sequence has its own prompt length
CAP_ALIGN = 128  # token-stride granularity of the cache layout

# Every entry point declared in include/kvq.h.
EXPORTS = (
    "kvq_cache_sizes", "kvq_workspace_bytes", "kvq_quantize_prefill", "kvq_append",
    "kvq_decode_attention", "kvq_decode_step_host", "kvq_get_device_status",
    "kvq_last_launch_count", "kvq_strerror", "kvq_debug_stall_waits",
    "kvq_decode_attention_noalloc", "kvq_append_decode", "kvq_decode_attention_rope",
    "kvq_decode_kernel_name", "kvq_quantize_prefill_ragged", "kvq_rope_kernel_name",
)


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "n_q_heads", "n_kv_heads", "head_dim", "bits", "scheme", "k_group",
        "v_group", "residual", "n_sink")] + [("max_ctx", ctypes.c_int64),
                                             ("flags", ctypes.c_uint32),
                                             ("outliers", ctypes.c_int32)]


class Sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "blocks", "k_meta", "k_mode", "v_mode", "k_res", "v_res", "k_sink", "v_sink", "status",
        "seq_prompt")]


class Cache(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "blocks", "k_meta", "k_mode", "v_mode", "k_res", "v_res", "k_sink", "v_sink")] + [
        (n, ctypes.c_int64) for n in ("n_quant", "n_resid", "n_sink", "ring_head")] + [
        ("dev_status", ctypes.c_void_p), ("seq_prompt", ctypes.c_void_p),
        ("n_appended", ctypes.c_int64)]


class KVQError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__("%s: %s (%d)" % (what, strerror(code), code))


_lib = None
_lock = threading.Lock()


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libkvq is not built (%s missing); run "
                                   "python -m bit_kv_cache_14_gb300.build_lib" % LIB_PATH)
            L = ctypes.CDLL(LIB_PATH)
            P, I64, C = ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(Config)
            CA = ctypes.POINTER(Cache)
            L.kvq_cache_sizes.argtypes = [C, ctypes.POINTER(Sizes)]
            L.kvq_workspace_bytes.argtypes = [C, ctypes.POINTER(ctypes.c_size_t)]
            L.kvq_quantize_prefill.argtypes = [C, CA, P, P, I64, P]
            L.kvq_quantize_prefill_ragged.argtypes = [C, CA, P, P, I64, P, P]
            L.kvq_append.argtypes = [C, CA, P, P, P]
            L.kvq_decode_attention.argtypes = [C, CA, P, P, ctypes.c_float, P, ctypes.c_size_t, P]
            L.kvq_decode_step_host.argtypes = [C, CA, P, P, P, P, ctypes.c_float, P,
                                               ctypes.c_size_t, P]
            L.kvq_decode_attention_rope.argtypes = [C, CA, P, P, ctypes.c_float, ctypes.c_double,
                                                    P, ctypes.c_size_t, P]
            L.kvq_decode_attention_noalloc.argtypes = [C, CA, P, P, ctypes.c_float, P]
            L.kvq_append_decode.argtypes = [C, CA, P, P, P, P, ctypes.c_float, P,
                                            ctypes.c_size_t, P]
            L.kvq_decode_kernel_name.argtypes = [C, I64, ctypes.c_char_p, ctypes.c_size_t]
            L.kvq_rope_kernel_name.argtypes = [C, I64, ctypes.c_char_p, ctypes.c_size_t]
            L.kvq_get_device_status.argtypes = [CA, P]
            L.kvq_last_launch_count.argtypes = []
            L.kvq_debug_stall_waits.argtypes = [ctypes.c_int64]
            L.kvq_debug_stall_waits.restype = None
            L.kvq_strerror.argtypes = [ctypes.c_int]
            L.kvq_strerror.restype = ctypes.c_char_p
            for name in EXPORTS:
                if name not in ("kvq_strerror", "kvq_debug_stall_waits"):
                    getattr(L, name).restype = ctypes.c_int
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().kvq_strerror(int(code)).decode()


def _check(code: int, what: str) -> None:
    if code != KVQ_OK:
        raise KVQError(code, what)


def make_config(batch, n_q_heads, n_kv_heads, head_dim, bits, scheme, k_group, v_group,
                residual, n_sink, max_ctx, flags=0, outliers=0) -> Config:
    return Config(batch, n_q_heads, n_kv_heads, head_dim, bits, scheme, k_group, v_group,
                  residual, n_sink, max_ctx, flags, outliers)


def config_of(w, max_ctx: int | None = None) -> Config:
    """Config of a synth.Workload (max_ctx defaults to prompt + streamed tokens)."""
    scheme = INNERQ_KNORM if getattr(w, "k_norm", False) else w.scheme
    flags = ((META_F16 if getattr(w, "meta_f16", False) else 0)
             | (VALUE_QUEUE if getattr(w, "v_queue", False) else 0)
             | (RAGGED if getattr(w, "ragged", False) else 0))
    return make_config(w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.bits, scheme,
                       w.k_group, w.v_group, w.residual, w.n_sink,
                       w.max_ctx() if max_ctx is None else max_ctx, flags,
                       getattr(w, "outliers", 0))


def decode_kernel_name(cfg: Config, n_quant: int) -> str:
    """The decode kernel instantiation the library launches for this
    configuration with n_quant quantized tokens (host only)."""
    buf = ctypes.create_string_buffer(128)
    _check(lib().kvq_decode_kernel_name(ctypes.byref(cfg), int(n_quant), buf, len(buf)),
           "kvq_decode_kernel_name")
    return buf.value.decode()


def rope_kernel_name(cfg: Config, n_quant: int) -> str:
    """The kernel kvq_decode_attention_rope launches for this configuration
    with n_quant quantized tokens (host only)."""
    buf = ctypes.create_string_buffer(128)
    _check(lib().kvq_rope_kernel_name(ctypes.byref(cfg), int(n_quant), buf, len(buf)),
           "kvq_rope_kernel_name")
    return buf.value.decode()


def cache_sizes(cfg: Config) -> Sizes:
    s = Sizes()
    _check(lib().kvq_cache_sizes(ctypes.byref(cfg), ctypes.byref(s)), "kvq_cache_sizes")
    return s


def workspace_bytes(cfg: Config) -> int:
    n = ctypes.c_size_t()
    _check(lib().kvq_workspace_bytes(ctypes.byref(cfg), ctypes.byref(n)), "kvq_workspace_bytes")
    return n.value


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _ptr(t: torch.Tensor) -> int:
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous (the library reads plain row-major buffers)")
    return t.data_ptr()


def _need_f16(*ts) -> None:
    for t in ts:
        if t.dtype != torch.float16:
            raise TypeError("expected a float16 tensor, got %s" % t.dtype)


class QuantizedKVCache:
    """Device buffers (torch-allocated) of one quantized cache plus its C view."""

    _BUFS = ("blocks", "k_meta", "k_mode", "v_mode", "k_res", "v_res", "k_sink", "v_sink")

    def __init__(self, cfg: Config, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        sizes = cache_sizes(cfg)
        self.bufs = {}
        view = Cache()
        for name in self._BUFS:
            n = getattr(sizes, name)
            t = torch.zeros(max(n, 16), dtype=torch.uint8, device=self.device)
            self.bufs[name] = t
            setattr(view, name, t.data_ptr() if n else None)
        self.status = torch.zeros(4, dtype=torch.int32, device=self.device)
        view.dev_status = self.status.data_ptr()
        # per-sequence prompt lengths (KVQ_RAGGED), written by the prefill
        self.seq_prompt = torch.zeros(max(cfg.batch, 4), dtype=torch.int32, device=self.device)
        view.seq_prompt = self.seq_prompt.data_ptr() if sizes.seq_prompt else None
        self.view = view
        self.ws_bytes = workspace_bytes(cfg)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=self.device)
        self.sizes = sizes

    # counters
    n_appended = property(lambda self: self.view.n_appended)
    n_quant = property(lambda self: self.view.n_quant)
    n_resid = property(lambda self: self.view.n_resid)
    n_sink = property(lambda self: self.view.n_sink)
    ring_head = property(lambda self: self.view.ring_head)

    def prefill(self, K: torch.Tensor, V: torch.Tensor, stream=None) -> None:
        """K, V: fp16 [B][H][T][d] on the device."""
        _need_f16(K, V)
        if K.shape != V.shape:
            raise ValueError("K and V shapes differ: %s vs %s" % (tuple(K.shape), tuple(V.shape)))
        _check(lib().kvq_quantize_prefill(ctypes.byref(self.cfg), ctypes.byref(self.view),
                                          _ptr(K), _ptr(V), K.shape[2], _stream(stream)),
               "kvq_quantize_prefill")

    def prefill_ragged(self, K: torch.Tensor, V: torch.Tensor, lens, stream=None) -> None:
        """K, V: fp16 [B][H][T_max][d] on the device; sequence b's prompt is its
        first lens[b] rows (KVQ_RAGGED)."""
        _need_f16(K, V)
        if K.shape != V.shape:
            raise ValueError("K and V shapes differ: %s vs %s" % (tuple(K.shape), tuple(V.shape)))
        lens = (ctypes.c_int32 * self.cfg.batch)(*[int(x) for x in lens])
        _check(lib().kvq_quantize_prefill_ragged(ctypes.byref(self.cfg), ctypes.byref(self.view),
                                                 _ptr(K), _ptr(V), K.shape[2], lens,
                                                 _stream(stream)),
               "kvq_quantize_prefill_ragged")

    def seq_lengths(self):
        """Tokens each sequence holds (host arithmetic: prompt + appended)."""
        c = self.cfg
        if not c.flags & RAGGED:
            n = self.n_quant + self.n_resid + self.n_sink
            return [n] * c.batch
        return [int(x) + self.n_appended for x in self.seq_prompt[: c.batch].tolist()]

    def append(self, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        """k, v: fp16 [B][H][d] on the device."""
        _need_f16(k, v)
        _check(lib().kvq_append(ctypes.byref(self.cfg), ctypes.byref(self.view), _ptr(k),
                                _ptr(v), _stream(stream)), "kvq_append")

    def decode(self, q: torch.Tensor, out: torch.Tensor | None = None, scale: float | None = None,
               stream=None) -> torch.Tensor:
        """q: fp16 [B][Hq][d]; returns fp32 [B][Hq][d]."""
        _need_f16(q)
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if scale is None:
            scale = 1.0 / math.sqrt(self.cfg.head_dim)
        _check(lib().kvq_decode_attention(ctypes.byref(self.cfg), ctypes.byref(self.view),
                                          _ptr(q), _ptr(out), float(scale), self.ws.data_ptr(),
                                          self.ws_bytes, _stream(stream)),
               "kvq_decode_attention")
        return out

    def decode_rope(self, q: torch.Tensor, base: float = 10000.0, out: torch.Tensor | None = None,
                    scale: float | None = None, stream=None) -> torch.Tensor:
        """Attention over keys cached before the rotary embedding: q (fp16
        [B][Hq][d], un-rotated) belongs to the newest token; every key is
        rotated by its position inside the kernel.  Returns fp32 [B][Hq][d]."""
        _need_f16(q)
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if scale is None:
            scale = 1.0 / math.sqrt(self.cfg.head_dim)
        _check(lib().kvq_decode_attention_rope(ctypes.byref(self.cfg), ctypes.byref(self.view),
                                               _ptr(q), _ptr(out), float(scale), float(base),
                                               self.ws.data_ptr(), self.ws_bytes,
                                               _stream(stream)),
               "kvq_decode_attention_rope")
        return out

    def append_decode(self, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor,
                      out: torch.Tensor | None = None, scale: float | None = None,
                      stream=None) -> torch.Tensor:
        """One decode step on device tensors: append k, v ([B][H][d] fp16), then
        attend with q; a single launch when the append needs no flush."""
        _need_f16(k, v, q)
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if scale is None:
            scale = 1.0 / math.sqrt(self.cfg.head_dim)
        _check(lib().kvq_append_decode(ctypes.byref(self.cfg), ctypes.byref(self.view), _ptr(k),
                                       _ptr(v), _ptr(q), _ptr(out), float(scale),
                                       self.ws.data_ptr(), self.ws_bytes, _stream(stream)),
               "kvq_append_decode")
        return out

    def decode_step_host(self, h_in, h_out, d_in, d_out, scale=None, stream=None) -> None:
        """One append + decode from pinned host tensors: h_in holds the step's
        k, v ([B][H][d] each) and q ([B][Hq][d]) back to back as fp16 (see
        step_input_halves), copied in one piece to d_in; the fp32 output
        [B][Hq][d] comes back to h_out through d_out."""
        _need_f16(h_in, d_in)
        n = self.step_input_halves()
        if h_in.numel() != n or d_in.numel() != n:
            raise ValueError("step input holds %d halves, expected %d" % (h_in.numel(), n))
        if scale is None:
            scale = 1.0 / math.sqrt(self.cfg.head_dim)
        _check(lib().kvq_decode_step_host(
            ctypes.byref(self.cfg), ctypes.byref(self.view), _ptr(h_in), _ptr(h_out), _ptr(d_in),
            _ptr(d_out), float(scale), self.ws.data_ptr(), self.ws_bytes, _stream(stream)),
            "kvq_decode_step_host")

    def step_input_halves(self) -> int:
        """fp16 elements of one step's [k | v | q] input block."""
        c = self.cfg
        return (2 * c.n_kv_heads + c.n_q_heads) * c.batch * c.head_dim

    def device_status(self, stream=None) -> int:
        """Synchronizes, reads and clears the status word.  After an error the
        decode workspace is zero-filled again (its counters are undefined)."""
        code = lib().kvq_get_device_status(ctypes.byref(self.view), _stream(stream))
        if code != KVQ_OK:
            self.ws.zero_()
            torch.cuda.synchronize(self.device)
        return code

    # ---- typed views of the buffers (for tests and inspection) ------------
    @property
    def cap(self) -> int:
        """Per-head token stride of every buffer: max_ctx rounded up to 128."""
        return (self.cfg.max_ctx + CAP_ALIGN - 1) // CAP_ALIGN * CAP_ALIGN

    # Byte offsets inside a 32-token block (include/kvq.h, "Packed layout").
    def _block_layout(self):
        c = self.cfg
        rb = c.head_dim * c.bits // 8
        m = 2 if c.flags & META_F16 else 4
        ngv = c.head_dim // c.v_group
        ngk = c.head_dim // c.k_group if c.scheme in (INNERQ, INNERQ_KNORM) else 0
        off = {"k_codes": 0, "v_codes": 32 * rb, "v_scale": 64 * rb}
        off["v_zero"] = off["v_scale"] + 32 * m * ngv
        off["k_scale"] = off["v_zero"] + 32 * m * ngv
        off["k_zero"] = off["k_scale"] + 32 * m * ngk
        end = off["k_zero"] + 32 * m * ngk
        if c.scheme == KIVI and c.k_group <= 32:
            off["k_stats"] = off["k_scale"]          # 32/G groups x (scale row, zero row)
            end = off["k_stats"] + (32 // c.k_group) * 2 * c.head_dim * m
        off["k_outliers"] = end
        off["v_outliers"] = end + 32 * 4 * c.outliers
        bb = off["v_outliers"] + 32 * 4 * c.outliers
        return off, bb, rb, ngv, ngk

    def _meta_dtype(self):
        return torch.float16 if self.cfg.flags & META_F16 else torch.float32

    def _block_field(self, name: str, width: int) -> torch.Tensor:
        """Bytes [off, off + 32*width) of every block as [B][H][cap][width] (a copy)."""
        c = self.cfg
        off, bb, _, _, _ = self._block_layout()
        nb = self.cap // 32
        blocks = self.bufs["blocks"][: c.batch * c.n_kv_heads * nb * bb]
        f = blocks.view(c.batch, c.n_kv_heads, nb, bb)[..., off[name]: off[name] + 32 * width]
        return f.reshape(c.batch, c.n_kv_heads, self.cap, width)

    def codes(self, which: str) -> torch.Tensor:
        """Packed code rows as u8 [B][H][cap][d*bits/8] (a copy)."""
        _, _, rb, _, _ = self._block_layout()
        return self._block_field(which + "_codes", rb)

    def meta(self, name: str) -> torch.Tensor:
        """scale / zero statistics as fp32 [B][H][rows * cols] (a copy; fp16
        statistics are widened exactly): KIVI keys [cap/G][d], per-token
        statistics [cap][groups]."""
        c = self.cfg
        dt = self._meta_dtype()
        m = 2 if dt == torch.float16 else 4
        if name.startswith("k") and c.scheme == KIVI:
            rows = self.cap // c.k_group
            which = 0 if name == "k_scale" else 1
            if c.k_group <= 32:
                per = 32 // c.k_group
                f = self._block_field("k_stats", per * 2 * c.head_dim * m // 32)
                f = f.contiguous().view(dt).float()
                f = f.reshape(c.batch, c.n_kv_heads, self.cap // 32, per, 2, c.head_dim)
                return f[:, :, :, :, which, :].reshape(c.batch, c.n_kv_heads, -1)
            n = c.batch * c.n_kv_heads * rows * 2 * c.head_dim
            km = self.bufs["k_meta"][: n * m].view(dt).float()
            km = km.view(c.batch, c.n_kv_heads, rows, 2, c.head_dim)
            return km[:, :, :, which, :].reshape(c.batch, c.n_kv_heads, -1)
        _, _, _, ngv, ngk = self._block_layout()
        cols = ngk if name.startswith("k") else ngv
        f = self._block_field(name, m * cols).contiguous().view(dt).float()
        return f.reshape(c.batch, c.n_kv_heads, -1)

    def outlier_lists(self, which: str):
        """Per-token outlier lists (KIVI with outliers): channels and fp16 bit
        patterns, each int32 [B][H][cap][outliers] (copies)."""
        c = self.cfg
        w = self._block_field(which + "_outliers", 4 * c.outliers).contiguous().view(torch.int32)
        w = w.reshape(c.batch, c.n_kv_heads, self.cap, c.outliers)
        return (w >> 16) & 0xFFFF, w & 0xFFFF

    def key_norms(self) -> torch.Tensor:
        """Per-channel key factors fp32 [B][H][d] (INNERQ_KNORM), stored after
        the last head's blocks (a copy)."""
        c = self.cfg
        if c.scheme != INNERQ_KNORM:
            raise ValueError("the configuration has no key normalization")
        _, bb, _, _, _ = self._block_layout()
        off = c.batch * c.n_kv_heads * (self.cap // 32) * bb
        n = c.batch * c.n_kv_heads * c.head_dim
        f = self.bufs["blocks"][off: off + 4 * n].view(torch.float32)
        return f.reshape(c.batch, c.n_kv_heads, c.head_dim)

    def modes(self, which: str) -> torch.Tensor:
        c = self.cfg
        n = getattr(self.sizes, which + "_mode") // 4
        return self.bufs[which + "_mode"][: n * 4].view(torch.int32).view(c.batch, c.n_kv_heads, -1)

    def fp16_rows(self, name: str, rows: int) -> torch.Tensor:
        c = self.cfg
        n = getattr(self.sizes, name) // 2
        return self.bufs[name][: n * 2].view(torch.float16).view(c.batch, c.n_kv_heads, rows,
                                                                 c.head_dim)

    def last_launch_count(self) -> int:
        return lib().kvq_last_launch_count()


def debug_stall_waits(iterations: int) -> None:
    """Force the decode kernel's timeout path (iterations > 0) or switch it off (0)."""
    lib().kvq_debug_stall_waits(int(iterations))
