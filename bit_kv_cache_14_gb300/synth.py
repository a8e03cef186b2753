"""Seeded synthetic workloads for the quantized KV cache.

This module is the one piece shared by the CUDA path and the CPU oracle: it
only draws random fp16 tensors and names the five workload shapes.  It holds
none of the method's arithmetic (no quantization, no attention).

Every head (b, h) draws its keys and values from its own PCG64 stream, keyed by
(seed, tensor, b, h, part), so any single head can be regenerated on its own
and heads can be generated in parallel threads.  ``part`` 0 is the prompt
(prefill) and part 1 the tokens streamed in later by decode steps.  Values are
drawn in float32 and rounded to fp16 with numpy's round-to-nearest-even.

Workload shapes follow the pages' settings: the Llama-2-7B layer (32 heads,
head_dim 128) of the KIVI experiments and of the per-token cache-size table in
the HF quantized-cache how-to (section 3.2), KIVI's group size 32 and residual
length 128 (KIVI ablation section), 4-bit groups of 64 channels with four fp16
sink tokens and a 32-token recent window for InnerQ (InnerQ method section),
and a 1M-token context as in the KVQuant abstract.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

KIVI = 0
INNERQ = 1

_TENSOR_K = 1
_TENSOR_V = 2
_TENSOR_Q = 3
_TENSOR_OUTLIER = 7
_TENSOR_OFFSET = 8
_TENSOR_LENGTH = 9


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ctx: int               # prompt length T quantized by prefill
    bits: int
    scheme: int            # KIVI or INNERQ
    k_group: int           # KIVI: tokens per key group; InnerQ: channels per group
    v_group: int           # channels per value group
    residual: int          # KIVI: residual length R; InnerQ: recent window W
    n_sink: int            # fp16 sink tokens (InnerQ)
    n_append: int          # decode tokens streamed in after the prompt
    seed: int
    dist: str              # "normal" or "student_t"
    k_outlier_frac: float = 0.0    # fraction of (head, channel) key channels scaled
    k_outlier_count: int = 0       # explicit count (overrides the fraction when > 0)
    k_outlier_mult: float = 1.0
    k_offset_sigma: float = 0.0    # per-(head, channel) key offset ~ N(0, sigma)
    data_scale: float = 1.0          # multiplier on every key and value
    first_token_k_mult: float = 1.0
    k_norm: bool = False             # InnerQ: one-shot per-channel key normalization
    v_queue: bool = False            # KIVI: values leave fp16 one at a time (a queue)
    meta_f16: bool = False           # scales and zeros stored in fp16
    outliers: int = 0                # KIVI: fp16 outliers kept per token and tensor
    ragged: bool = False             # every sequence has its own prompt length

    @property
    def group_ratio(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def n_outliers(self) -> int:
        if self.k_outlier_count > 0:
            return self.k_outlier_count
        return int(round(self.k_outlier_frac * self.n_kv_heads * self.head_dim))

    def max_ctx(self, extra: int = 0) -> int:
        return self.ctx + self.n_append + extra


WORKLOADS = {
    # 1 KV head, head_dim 64, 256 tokens, 2-bit, G=32, Gv=32, R=32; 4 fixed K
    # channels x10; one decode step.
    "tiny": Workload("tiny", 1, 1, 1, 64, 256, 2, KIVI, 32, 32, 32, 0, 1, 0,
                     "normal", k_outlier_count=4, k_outlier_mult=10.0),
    # Llama-2-7B-shaped layer: batch 8, 32 heads, head_dim 128, 4096 tokens,
    # 2-bit, G=32, R=128; 2% of key channels x8; 256 streamed appends.
    "llama2_7b_2bit": Workload("llama2_7b_2bit", 8, 32, 32, 128, 4096, 2, KIVI,
                               32, 32, 128, 0, 256, 1, "normal",
                               k_outlier_frac=0.02, k_outlier_mult=8.0),
    # 4-bit: batch 32, 32 heads, 8192 tokens, G=64, Gv=64, R=128; Student-t(4)
    # scaled 0.5 with per-channel key offsets ~ N(0, 2).
    "kivi_4bit": Workload("kivi_4bit", 32, 32, 32, 128, 8192, 4, KIVI, 64, 64,
                          128, 0, 1, 2, "student_t", k_offset_sigma=2.0,
                          data_scale=0.5),
    # GQA: batch 64, 32 query heads over 8 KV heads, 16384 tokens, 2-bit,
    # G=32, Gv=32, R=128; 2% of key channels x10.
    "gqa_2bit": Workload("gqa_2bit", 64, 32, 8, 128, 16384, 2, KIVI, 32, 32,
                         128, 0, 1, 3, "normal", k_outlier_frac=0.02,
                         k_outlier_mult=10.0),
    # Long context, InnerQ-style: batch 1, 32 heads, 1M tokens, 4-bit groups of
    # 64 channels with per-group sym/asym, 4 sinks + 32 recent fp16 tokens;
    # first-token K x20.
    "innerq_1m": Workload("innerq_1m", 1, 32, 32, 128, 1 << 20, 4, INNERQ, 64,
                          64, 32, 4, 1, 4, "normal", first_token_k_mult=20.0),
}


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (smaller parity cases)."""
    return dataclasses.replace(w, **changes)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(k) for k in key]))


def _draw(rng: np.random.Generator, w: Workload, shape) -> np.ndarray:
    if w.dist == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
    elif w.dist == "student_t":
        x = rng.standard_t(4.0, shape).astype(np.float32)
    else:
        raise ValueError(w.dist)
    return x


def outlier_channels(w: Workload) -> np.ndarray:
    """Fixed (kv_head, channel) pairs whose keys are scaled, as flat indices
    h*head_dim + c, drawn without replacement; shared by every batch entry."""
    n = w.n_outliers()
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    rng = _rng(w.seed, _TENSOR_OUTLIER)
    return np.sort(rng.choice(w.n_kv_heads * w.head_dim, size=n, replace=False))


def key_offsets(w: Workload) -> np.ndarray:
    """Per-(kv_head, channel) key offsets, float32 [H][d] (zeros if unused)."""
    if w.k_offset_sigma == 0.0:
        return np.zeros((w.n_kv_heads, w.head_dim), dtype=np.float32)
    rng = _rng(w.seed, _TENSOR_OFFSET)
    return (rng.standard_normal((w.n_kv_heads, w.head_dim), dtype=np.float32)
            * np.float32(w.k_offset_sigma))


def head_tokens(w: Workload, b: int, h: int, part: int, n: int,
                first_token: int = 0):
    """Keys and values of head (b, h): fp16 arrays [n][head_dim].

    part 0 = prompt tokens 0..n-1; part 1 = streamed tokens, the i-th of which
    is absolute token ctx + i.  ``first_token`` is the absolute index of row 0
    (only used for the first-token key multiplier).
    """
    d = w.head_dim
    rk = _rng(w.seed, _TENSOR_K, b, h, part)
    rv = _rng(w.seed, _TENSOR_V, b, h, part)
    k = _draw(rk, w, (n, d))
    v = _draw(rv, w, (n, d))
    if w.data_scale != 1.0:
        k *= np.float32(w.data_scale)
        v *= np.float32(w.data_scale)
    out = outlier_channels(w)
    chans = out[out // d == h] % d
    if chans.size:
        k[:, chans] *= np.float32(w.k_outlier_mult)
    if w.k_offset_sigma != 0.0:
        k += key_offsets(w)[h][None, :]
    if w.first_token_k_mult != 1.0 and first_token == 0 and n > 0:
        k[0, :] *= np.float32(w.first_token_k_mult)
    return k.astype(np.float16), v.astype(np.float16)


def prompt_lengths(w: Workload) -> np.ndarray:
    """Prompt length of each sequence, int32 [B]: all ctx, or (ragged) drawn
    uniformly from [0, ctx] per sequence from the workload's seed, with the
    first sequence at ctx (the longest) and, from four sequences on, the
    second empty and the third shorter than the residual / window."""
    if not w.ragged:
        return np.full(w.batch, w.ctx, np.int32)
    rng = _rng(w.seed, _TENSOR_LENGTH)
    lens = rng.integers(0, w.ctx + 1, size=w.batch).astype(np.int32)
    lens[0] = w.ctx
    if w.batch >= 4:
        lens[1] = 0
        lens[2] = min(w.ctx, max(0, w.residual - 1))
    return lens


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def prompt(w: Workload, T: int | None = None):
    """Prompt keys and values for every head: fp16 [B][H][T][d] each."""
    T = w.ctx if T is None else T
    B, H, d = w.batch, w.n_kv_heads, w.head_dim
    K = np.empty((B, H, T, d), dtype=np.float16)
    V = np.empty((B, H, T, d), dtype=np.float16)

    def one(idx):
        b, h = divmod(idx, H)
        K[b, h], V[b, h] = head_tokens(w, b, h, 0, T)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(one, range(B * H)))
    return K, V


def streamed(w: Workload, n: int | None = None):
    """Tokens streamed in after the prompt: fp16 [n][B][H][d] keys and values."""
    n = w.n_append if n is None else n
    B, H, d = w.batch, w.n_kv_heads, w.head_dim
    K = np.empty((n, B, H, d), dtype=np.float16)
    V = np.empty((n, B, H, d), dtype=np.float16)
    for b in range(B):
        for h in range(H):
            k, v = head_tokens(w, b, h, 1, n, first_token=w.ctx)
            K[:, b, h], V[:, b, h] = k, v
    return K, V


def queries(w: Workload, step: int = 0) -> np.ndarray:
    """Decode queries for one step: fp16 [B][H_q][d], N(0, 1)."""
    rng = _rng(w.seed, _TENSOR_Q, step)
    q = rng.standard_normal((w.batch, w.n_q_heads, w.head_dim), dtype=np.float32)
    return q.astype(np.float16)
