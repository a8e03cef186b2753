"""Pins of the CPU oracle against facts fixed outside it (no GPU).

Each pin checks the oracle against something other than its own code: the
hand-worked rows and the page-printed numbers under tests/golden/, numpy's
IEEE fp16 conversion, closed-form round-trip bounds, grid-exact data (where
quantization is lossless, so attention must equal a library softmax-attention
call on the raw fp16 data), torch's scaled_dot_product_attention in fp64,
perturbation bounds, and the residual-flush cadence.  The last test plants
mistakes in copies of the oracle's C file and checks that every one of them
fails at least one pin.
"""
import math
import os
import shutil
import tempfile

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_14_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# --------------------------------------------------------------------------
# scalar pins
# --------------------------------------------------------------------------

def pin_half_to_float():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    for b in list(range(0, 1 << 16, 97)) + [0, 1, 0x3ff, 0x400, 0x3c00, 0x7bff, 0x8001, 0xfbff]:
        got = np.float32(oracle.half_to_float(int(b)))
        r = ref[b]
        assert (np.isnan(got) and np.isnan(r)) or got.tobytes() == r.tobytes(), hex(b)


def pin_worked_examples():
    for row in _golden_rows("asym_worked_examples.txt"):
        head, xs, scale, zero, codes = [c.strip() for c in row.split("|")]
        mode, bits = head.split()
        x = np.array([float(v) for v in xs.split()], np.float32)
        fn = oracle.quant_asym if mode == "asym" else oracle.quant_sym
        s, z, u = fn(x, int(bits))
        assert s == np.float32(float(scale)), (row, s)
        assert z == np.float32(float(zero)), (row, z)
        assert list(u) == [int(c) for c in codes.split()], (row, u)


def pin_float_to_half():
    """fp32 -> fp16, nearest-even, against numpy's IEEE conversion: every
    midpoint between consecutive halves (ties) and its two neighbours, both
    signs, subnormals, the overflow boundary, infinities and zeros."""
    h = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mid = ((h[:-1] + h[1:]) / 2).astype(np.float32)
    vals = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)),
                           np.nextafter(mid, np.float32(0)),
                           np.float32([0.0, 65504, 65519, 65520, 1e9, 2.0 ** -25, 2.0 ** -26,
                                       1e-30, np.inf])])
    vals = np.concatenate([vals, -vals])
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    for i in list(range(0, vals.size, 7)) + list(range(vals.size - 20, vals.size)):
        assert oracle.float_to_half(vals[i]) == ref[i], (vals[i], hex(ref[i]))


def pin_f16_meta_worked_examples():
    for row in _golden_rows("f16_meta_worked_examples.txt"):
        head, xs, scale, zero, codes = [c.strip() for c in row.split("|")]
        mode, bits = head.split()
        x = np.array([float(v) for v in xs.split()], np.float32)
        fn = oracle.quant_asym if mode == "asym" else oracle.quant_sym
        s, z, u = fn(x, int(bits), meta_f16=True)
        assert s == np.float32(float(scale)), (row, s)
        assert z == np.float32(float(zero)), (row, z)
        assert list(u) == [int(c) for c in codes.split()], (row, u)


def pin_f16_meta_round_trip_bound():
    """With fp16 metadata the stored scale and zero are fp16 values, and every
    element reconstructs within half a stored step plus what rounding the
    scale and the zero moved the grid: |x - x_hat| <= s16/2 + |min - z16| +
    (2^b - 1)|s32 - s16| (+ fp32 slack), for fp16 and for arbitrary fp32
    groups (normalized keys)."""
    rng = np.random.default_rng(42)
    for bits in (2, 4):
        top = (1 << bits) - 1
        for trial in range(400):
            n = int(rng.integers(2, 70))
            x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 2)).astype(np.float32)
            if trial % 2:
                x = x.astype(np.float16).astype(np.float32)
            s, z, u = oracle.quant_asym(x, bits, meta_f16=True)
            assert np.float32(s).astype(np.float16).astype(np.float32) == s
            assert np.float32(z).astype(np.float16).astype(np.float32) == z
            mn, mx = float(x.min()), float(x.max())
            s32 = (mx - mn) / top
            xh = u.astype(np.float64) * float(s) + float(z)
            bound = float(s) / 2 + abs(mn - float(z)) + top * abs(s32 - float(s)) \
                + 4 * np.spacing(np.float32(max(abs(mn), abs(mx))))
            assert np.abs(x.astype(np.float64) - xh).max() <= bound, (bits, trial)


def pin_mode_choice():
    # midpoint 0 -> symmetric; far from zero -> asymmetric; equality -> symmetric
    assert oracle.choose_symmetric(-1.0, 1.0, 4)
    assert not oracle.choose_symmetric(0.0, 3.0, 2)
    assert oracle.choose_symmetric(-1.0, 2.0, 2)        # |1| <= 3/3
    assert not oracle.choose_symmetric(-1.0, 2.25, 2)   # |1.25| > 3.25/3
    assert not oracle.choose_symmetric(2.0, 2.0, 4)     # constant group


def pin_pack_layout():
    for row in _golden_rows("pack_layout_example.txt"):
        bits, codes, hexes = [c.strip() for c in row.split("|")]
        u = np.array([[int(c) for c in codes.split()]], np.uint8)
        got = oracle.pack(u, int(bits))[0]
        assert [int(h, 16) for h in hexes.split()] == list(got), row


def pin_llama2_bytes_per_token():
    # layers * (K and V) * heads * bytes of one packed head row (codes only);
    # the 16-bit row is the fp16 residual row the cache keeps unquantized.
    L, H, d = 32, 32, 128
    for row in _golden_rows("llama2_7b_bytes_per_token.txt"):
        bits, expect = map(int, row.split())
        if bits == 16:
            row_bytes = d * np.dtype(np.float16).itemsize
        else:
            row_bytes = oracle.pack(np.zeros((1, d), np.uint8), bits).nbytes
        assert L * 2 * H * row_bytes == expect
    # "10k tokens about 5 GB" for fp16
    assert abs(10_000 * 524288 / 1e9 - 5.0) < 0.3


def _rand_groups(rng, n_groups, n, bits):
    x = rng.standard_normal((n_groups, n)).astype(np.float16).astype(np.float32)
    x[::7] *= 20.0
    x[1::5] += 3.0
    return x


def pin_round_trip_bound():
    rng = np.random.default_rng(11)
    for bits in (2, 4, 8):
        for n in (4, 32, 64):
            for x in _rand_groups(rng, 60, n, bits):
                for fn in (oracle.quant_asym, oracle.quant_sym):
                    s, z, u = fn(x, bits)
                    xh = u.astype(np.float64) * np.float64(s) + np.float64(z)
                    amax = float(np.max(np.abs(x)))
                    slack = 4 * np.spacing(np.float32(amax))
                    assert np.all(np.abs(x - xh) <= float(s) / 2 + slack), (fn, bits, n)


def pin_endpoints():
    rng = np.random.default_rng(12)
    for bits in (2, 4):
        top, lim = (1 << bits) - 1, (1 << (bits - 1)) - 1
        for x in _rand_groups(rng, 50, 32, bits):
            s, z, u = oracle.quant_asym(x, bits)
            assert u[np.argmin(x)] == 0 and u[np.argmax(x)] == top
            assert z == x.min()
            s, z, u = oracle.quant_sym(x, bits)
            i = np.argmax(np.abs(x))
            assert int(u[i]) - (1 << (bits - 1)) == (lim if x[i] > 0 else -lim)


def pin_grid_exact_round_trip():
    rng = np.random.default_rng(13)
    for bits in (2, 4):
        top = (1 << bits) - 1
        for _ in range(200):
            e = int(rng.integers(1, 6))
            step = 2.0 ** -e
            base = float(rng.integers(-40, 40)) * step
            u = rng.integers(0, top + 1, 32)
            u[rng.integers(0, 16)] = 0
            u[16 + rng.integers(0, 16)] = top
            x = (base + u * step).astype(np.float32)
            s, z, got = oracle.quant_asym(x, bits)
            assert s == np.float32(step) and z == np.float32(base)
            assert np.array_equal(got, u)


# --------------------------------------------------------------------------
# cache state machine pins
# --------------------------------------------------------------------------

def _randn16(rng, *shape, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


def pin_kivi_flush_cadence():
    rng = np.random.default_rng(14)
    d, G, R = 16, 8, 32
    for T in (0, 5, 31, 32, 100, 120):
        h = oracle.OracleHead(d, 2, oracle.KIVI, G, 8, R, 0, 1024)
        K, V = _randn16(rng, T, d), _randn16(rng, T, d)
        h.prefill(K, V)
        assert h.n_resid == T % R and h.n_quant == T - T % R
        n0 = h.n_resid
        for n in range(1, 140):
            h.append(_randn16(rng, d), _randn16(rng, d))
            assert h.n_flush == (n0 + n) // R
            assert 0 <= h.n_resid < R and h.n_quant % G == 0
            assert h.n_quant + h.n_resid == T + n
        # the residual always holds the newest tokens, oldest first
        kr, _ = h.residual_tokens()
        assert kr.shape[0] == (T + 139) % R


def pin_kivi_residual_is_exact_and_tail():
    rng = np.random.default_rng(15)
    d, G, R, T = 16, 8, 32, 77
    K, V = _randn16(rng, T, d), _randn16(rng, T, d)
    h = oracle.OracleHead(d, 2, oracle.KIVI, G, 8, R, 0, 256)
    h.prefill(K, V)
    kr, vr = h.residual_tokens()
    assert np.array_equal(kr.view(np.uint16), K[64:].view(np.uint16))
    assert np.array_equal(vr.view(np.uint16), V[64:].view(np.uint16))


def pin_kivi_cache_round_trip():
    """Every quantized element of a prefilled + appended cache reconstructs
    within scale/2 through the storage layout (key meta per (G-token group,
    channel), value meta per (token, channel group))."""
    rng = np.random.default_rng(16)
    d, G, Gv, R, T, n_app = 32, 8, 16, 16, 64, 40
    K, V = _randn16(rng, T + n_app, d, scale=2.0), _randn16(rng, T + n_app, d)
    for bits in (2, 4):
        h = oracle.OracleHead(d, bits, oracle.KIVI, G, Gv, R, 0, 256)
        h.prefill(K[:T], V[:T])
        for i in range(T, T + n_app):
            h.append(K[i], V[i])
        n = h.n_quant
        t = np.arange(n)
        ks = h.k_scale[t // G]                       # [n][d]
        kz = h.k_zero[t // G]
        kh = h.k_u[:n] * ks.astype(np.float64) + kz
        vs = np.repeat(h.v_scale[:n], Gv, axis=1)
        vz = np.repeat(h.v_zero[:n], Gv, axis=1)
        vh = h.v_u[:n] * vs.astype(np.float64) + vz
        kx, vx = K[:n].astype(np.float64), V[:n].astype(np.float64)
        assert np.all(np.abs(kx - kh) <= ks / 2 + 1e-5)
        assert np.all(np.abs(vx - vh) <= vs / 2 + 1e-5)
        # key groups: code 0 at the channel minimum of each group
        kg = K[:n].astype(np.float32).reshape(n // G, G, d)
        assert np.array_equal(h.k_zero[: n // G], kg.min(axis=1))


def pin_innerq_windows():
    rng = np.random.default_rng(17)
    d, S, W = 128, 4, 8
    for T in (0, 2, 4, 9, 12, 50):
        K, V = _randn16(rng, T + 30, d), _randn16(rng, T + 30, d)
        h = oracle.OracleHead(d, 4, oracle.INNERQ, 64, 64, W, S, 256)
        h.prefill(K[:T], V[:T])
        for i in range(T, T + 30):
            h.append(K[i], V[i])
            n = i + 1
            assert h.n_sink_used == min(S, n)
            assert h.n_resid == min(W, max(0, n - S))
            assert h.n_quant == max(0, n - S - W)
        ks, _ = h.sink_tokens()
        kw, vw = h.residual_tokens()
        n = T + 30
        assert np.array_equal(ks.view(np.uint16), K[:S].view(np.uint16))
        assert np.array_equal(kw.view(np.uint16), K[n - W:n].view(np.uint16))
        assert np.array_equal(vw.view(np.uint16), V[n - W:n].view(np.uint16))
        # quantized tokens are S .. n-W-1 in order: each reconstructs within scale/2
        q = h.n_quant
        src = K[S:S + q].astype(np.float64)
        sc = np.repeat(h.k_scale[:q], 64, axis=1).astype(np.float64)
        zz = np.repeat(h.k_zero[:q], 64, axis=1).astype(np.float64)
        assert np.all(np.abs(src - (h.k_u[:q] * sc + zz)) <= sc / 2 + 1e-5)


def pin_innerq_modes():
    """Group modes follow the min/max rule, codes reach the symmetric limits."""
    rng = np.random.default_rng(18)
    d = 128
    K = _randn16(rng, 40, d)
    K[:, 64:] += np.float16(3.0)     # second group is far from zero: asymmetric
    V = _randn16(rng, 40, d)
    h = oracle.OracleHead(d, 4, oracle.INNERQ, 64, 64, 0, 0, 64)
    h.prefill(K, V)
    assert h.n_quant == 40
    x = K.astype(np.float32)
    for t in range(40):
        for j in range(2):
            g = x[t, 64 * j:64 * j + 64]
            mn, mx = g.min(), g.max()
            sym = abs(np.float32(mx + mn)) <= np.float32((mx - mn) / np.float32(15))
            assert bool(h.k_sym[t, j]) == bool(sym)
        assert h.k_sym[t, 1] == 0


def pin_innerq_key_norms():
    """One-shot per-channel key normalization: the factor of channel c is the
    largest |K[t][c]| over the whole prompt (1 for an all-zero channel or an
    empty prompt), and scaling a key channel by a power of two scales its
    factor and leaves every code, scale, zero and mode unchanged (appended
    keys included)."""
    rng = np.random.default_rng(23)
    d, S, W = 128, 2, 8
    for T in (0, 1, 40):
        K, V = _randn16(rng, T + 20, d), _randn16(rng, T + 20, d)
        if T:
            K[:, 5] = 0                           # an all-zero channel
            K[0, 7] = np.float16(-9.5)            # a channel whose extreme is a sink
        e = rng.integers(0, 4, d)          # up-scaling: exact in fp16 (no subnormals)
        K2 = (K.astype(np.float32) * np.exp2(e).astype(np.float32)).astype(np.float16)
        assert np.array_equal(K2.astype(np.float32), K.astype(np.float32) * np.exp2(e))
        hs = []
        for KK in (K, K2):
            h = oracle.OracleHead(d, 4, oracle.INNERQ, 32, 64, W, S, 128, k_norm=True)
            h.prefill(KK[:T], V[:T])
            for i in range(T, T + 20):
                h.append(KK[i], V[i])
            hs.append(h)
        if T == 0:
            assert np.array_equal(hs[0].key_norms(), np.ones(d, np.float32))
            continue
        amax = np.abs(K[:T].astype(np.float32)).max(axis=0)
        want = np.where(amax > 0, amax, np.float32(1))
        assert np.array_equal(hs[0].key_norms(), want)
        assert want[5] == 1 and want[7] == np.float32(9.5)
        want2 = np.where(amax > 0, want * np.exp2(e).astype(np.float32), np.float32(1))
        assert np.array_equal(hs[1].key_norms(), want2)
        n = hs[0].n_quant
        assert n == hs[1].n_quant and n > 0
        for a, b in ((hs[0].k_u, hs[1].k_u), (hs[0].k_scale, hs[1].k_scale),
                     (hs[0].k_zero, hs[1].k_zero), (hs[0].k_sym, hs[1].k_sym)):
            assert np.array_equal(a[:n], b[:n])
        # the normalized keys reconstruct within half a step of K / factor
        x = K[S:S + n].astype(np.float32) * (np.float32(1) / hs[0].key_norms())
        sc = np.repeat(hs[0].k_scale[:n], 32, axis=1).astype(np.float64)
        zz = np.repeat(hs[0].k_zero[:n], 32, axis=1).astype(np.float64)
        assert np.all(np.abs(x - (hs[0].k_u[:n] * sc + zz)) <= sc / 2 + 1e-5)


# --------------------------------------------------------------------------
# attention pins
# --------------------------------------------------------------------------

def _sdpa(q, K, V, tau):
    """torch scaled_dot_product_attention in fp64 on the CPU, one query."""
    qt = torch.from_numpy(q.astype(np.float64))[None, None, None, :]
    kt = torch.from_numpy(K.astype(np.float64))[None, None]
    vt = torch.from_numpy(V.astype(np.float64))[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=tau)
    return o[0, 0, 0].numpy()


def pin_attention_unquantized_is_sdpa():
    rng = np.random.default_rng(19)
    d, T = 64, 50
    K, V = _randn16(rng, T + 20, d, scale=2.0), _randn16(rng, T + 20, d)
    q = _randn16(rng, d)
    h = oracle.OracleHead(d, 2, oracle.KIVI, 32, 32, 128, 0, 256)   # R > T + steps
    h.prefill(K[:T], V[:T])
    for i in range(T, T + 20):
        h.append(K[i], V[i])
    assert h.n_quant == 0
    tau = 1 / math.sqrt(d)
    np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K, V, tau), rtol=0, atol=1e-12)


def _grid_tokens(rng, T, d, bits, k_rows, v_cols, sym_groups=False):
    """fp16 tokens that every group quantizes losslessly.  Keys: groups of
    k_rows consecutive tokens per channel (k_rows=1: per token over v_cols
    channels, like values).  Values: per token, groups of v_cols channels."""
    top = (1 << bits) - 1

    def grid(n):
        e = int(rng.integers(1, 5))
        step = 2.0 ** -e
        if sym_groups and rng.integers(0, 2):
            lim = (1 << (bits - 1)) - 1
            u = rng.integers(-lim, lim + 1, n)
            u[0], u[-1] = -lim, lim
            return rng.permutation(u) * step
        base = float(rng.integers(-24, 24)) * step
        if sym_groups:
            base = abs(base) + 4.0          # clearly off-centre: asymmetric
        u = rng.integers(0, top + 1, n)
        u[0], u[-1] = 0, top
        return base + rng.permutation(u) * step

    K = np.empty((T, d), np.float64)
    V = np.empty((T, d), np.float64)
    if k_rows > 1:
        for g in range(T // k_rows):
            for c in range(d):
                K[g * k_rows:(g + 1) * k_rows, c] = grid(k_rows)
    else:
        for t in range(T):
            for j in range(d // v_cols):
                K[t, j * v_cols:(j + 1) * v_cols] = grid(v_cols)
    for t in range(T):
        for j in range(d // v_cols):
            V[t, j * v_cols:(j + 1) * v_cols] = grid(v_cols)
    K16, V16 = K.astype(np.float16), V.astype(np.float16)
    assert np.array_equal(K16.astype(np.float64), K) and np.array_equal(V16.astype(np.float64), V)
    return K16, V16


def pin_attention_grid_exact_kivi():
    rng = np.random.default_rng(20)
    d, G, Gv, R = 32, 8, 16, 16
    for bits in (2, 4):
        T = 64 + 7
        K, V = _grid_tokens(rng, 64 + 16, d, bits, G, Gv)
        Kx, Vx = _randn16(rng, 40, d), _randn16(rng, 40, d)
        h = oracle.OracleHead(d, bits, oracle.KIVI, G, Gv, R, 0, 256)
        h.prefill(K[:T], V[:T])              # 64 quantized, 7 residual
        for i in range(T, 80):
            h.append(K[i], V[i])             # flush at 80: all 80 quantized
        assert h.n_quant == 80 and h.n_resid == 0
        q = _randn16(rng, d)
        tau = 1 / math.sqrt(d)
        np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K[:80], V[:80], tau),
                                   rtol=0, atol=1e-12)
        # with a non-empty fp16 residual next to the quantized part
        h.append(Kx[0], Vx[0])
        Kall = np.concatenate([K[:80], Kx[:1]])
        Vall = np.concatenate([V[:80], Vx[:1]])
        np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, Kall, Vall, tau),
                                   rtol=0, atol=1e-12)


def pin_attention_grid_exact_innerq():
    rng = np.random.default_rng(21)
    d, S, W, T = 128, 4, 8, 60
    K, V = _grid_tokens(rng, T, d, 4, 1, 64, sym_groups=True)
    K[0] *= np.float16(8)                      # loud sink token, kept fp16
    h = oracle.OracleHead(d, 4, oracle.INNERQ, 64, 64, W, S, 256)
    h.prefill(K, V)
    assert h.n_quant == T - S - W
    assert 0 < h.k_sym[:h.n_quant].sum() < h.k_sym[:h.n_quant].size
    q = _randn16(rng, d)
    tau = 1 / math.sqrt(d)
    np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K, V, tau), rtol=0, atol=1e-12)


def pin_attention_grid_exact_innerq_key_norm():
    """Normalized keys with power-of-two factors stay grid-exact, so attention
    with the factor folded into q equals plain attention on the raw tokens."""
    rng = np.random.default_rng(24)
    d, S, W, T = 128, 2, 8, 60
    K, V = _grid_tokens(rng, T, d, 4, 1, 64, sym_groups=True)
    assert np.abs(K.astype(np.float32)).max() < 32
    q = _randn16(rng, d)
    # the sink carries each channel's extreme (factors 32 and 128) and scores
    # far below the rest, so the quantized tokens decide the output
    sgn = np.where(q.astype(np.float32) > 0, -1, 1)
    K[0] = (np.repeat(np.float32([32, 128]), 64) * sgn).astype(np.float16)
    h = oracle.OracleHead(d, 4, oracle.INNERQ, 64, 64, W, S, 256, k_norm=True)
    h.prefill(K, V)
    assert h.n_quant == T - S - W
    assert np.array_equal(h.key_norms(), np.repeat(np.float32([32, 128]), 64))
    tau = 1 / math.sqrt(d)
    np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K, V, tau), rtol=0, atol=1e-12)


def pin_attention_grid_exact_f16_meta():
    """Grid data has power-of-two steps and fp16 bases, which fp16 metadata
    stores exactly: attention over KIVI and InnerQ caches with fp16 scales
    and zeros equals torch's fp64 SDPA on the raw tokens."""
    rng = np.random.default_rng(25)
    d, G, Gv, R = 32, 8, 16, 16
    K, V = _grid_tokens(rng, 80, d, 2, G, Gv)
    h = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 256, meta_f16=True)
    h.prefill(K[:71], V[:71])
    for i in range(71, 80):
        h.append(K[i], V[i])
    q = _randn16(rng, d)
    tau = 1 / math.sqrt(d)
    np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K, V, tau), rtol=0, atol=1e-12)
    d, S, W, T = 128, 4, 8, 60
    K, V = _grid_tokens(rng, T, d, 4, 1, 64, sym_groups=True)
    h = oracle.OracleHead(d, 4, oracle.INNERQ, 64, 64, W, S, 256, meta_f16=True)
    h.prefill(K, V)
    assert 0 < h.k_sym[:h.n_quant].sum() < h.k_sym[:h.n_quant].size
    q = _randn16(rng, d)
    tau = 1 / math.sqrt(d)
    np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K, V, tau), rtol=0, atol=1e-12)


def pin_attention_identical_keys_mean():
    rng = np.random.default_rng(22)
    d, G, Gv, R, T = 32, 8, 8, 16, 48
    krow = _randn16(rng, d)
    K = np.repeat(krow[None], T + 3, axis=0)
    V = _randn16(rng, T + 3, d)
    h = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 128)
    h.prefill(K[:T], V[:T])
    for i in range(T, T + 3):
        h.append(K[i], V[i])
    n = h.n_quant
    # constant key groups are lossless; output = mean of the values as stored
    vh = h.v_u[:n] * np.repeat(h.v_scale[:n], Gv, axis=1).astype(np.float64) \
        + np.repeat(h.v_zero[:n], Gv, axis=1)
    _, vr = h.residual_tokens()
    expect = np.concatenate([vh, vr.astype(np.float64)]).mean(axis=0)
    np.testing.assert_allclose(h.attend(_randn16(rng, d), 0.3), expect, rtol=0, atol=1e-12)


def pin_attention_error_bound():
    """Random data: the quantized-cache output stays within the perturbation
    bound implied by |x - x_hat| <= scale/2 of the fp64 attention over the
    raw fp16 cache."""
    rng = np.random.default_rng(23)
    d, G, Gv, R, T = 64, 16, 16, 32, 200
    for bits in (2, 4):
        K, V = _randn16(rng, T, d), _randn16(rng, T, d)
        h = oracle.OracleHead(d, bits, oracle.KIVI, G, Gv, R, 0, 256)
        h.prefill(K, V)
        n = h.n_quant
        q = _randn16(rng, d)
        tau = 1 / math.sqrt(d)
        ks = h.k_scale[np.arange(n) // G].astype(np.float64)
        delta = tau * (np.abs(q.astype(np.float64))[None, :] * ks / 2).sum(axis=1).max()
        vs = np.repeat(h.v_scale[:n], Gv, axis=1).astype(np.float64)
        vmax = np.abs(V.astype(np.float64)).max() + vs.max() / 2
        bound = (math.exp(2 * delta) - 1) * vmax + vs.max() / 2 + 1e-9
        err = np.abs(h.attend(q, tau) - _sdpa(q, K, V, tau)).max()
        assert err <= bound, (bits, err, bound)
        assert err > 0


# --------------------------------------------------------------------------
# KIVI's value queue (values leave the fp16 queue one at a time)
# --------------------------------------------------------------------------

def pin_kivi_value_queue_cadence():
    """After n tokens the queue holds the last min(n, R - 1) values in fp16
    (oldest first) and the rest are quantized per token; the keys flush
    exactly as in the batch reading; every value token quantized under both
    readings has the same codes, scales and zeros."""
    rng = np.random.default_rng(40)
    d, G, Gv, R = 32, 8, 16, 16
    for T in (0, 5, 15, 16, 17, 40, 48):
        K, V = _randn16(rng, T + 40, d), _randn16(rng, T + 40, d)
        hq = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 256, v_queue=True)
        hb = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 256)
        hq.prefill(K[:T], V[:T])
        hb.prefill(K[:T], V[:T])
        for n in range(T, T + 40):
            if n > T:
                hq.append(K[n - 1], V[n - 1])
                hb.append(K[n - 1], V[n - 1])
            assert hq.n_vquant == max(0, n - R + 1), (T, n, hq.n_vquant)
            assert np.array_equal(hq.value_queue().view(np.uint16),
                                  V[hq.n_vquant:n].view(np.uint16)), (T, n)
            assert (hq.n_quant, hq.n_resid) == (hb.n_quant, hb.n_resid)
            nq = hq.n_quant
            assert np.array_equal(hq.k_u[:nq], hb.k_u[:nq])
            m = min(hq.n_vquant, hb.n_vquant)
            assert np.array_equal(hq.v_u[:m], hb.v_u[:m]), (T, n)
            assert np.array_equal(hq.v_scale[:m].view(np.uint32), hb.v_scale[:m].view(np.uint32))
            assert np.array_equal(hq.v_zero[:m].view(np.uint32), hb.v_zero[:m].view(np.uint32))


def pin_kivi_value_queue_selector():
    """One token whose score leads all others by hundreds of nats makes the
    attention output that token's value as stored: the exact fp16 row while
    it waits in the queue (also when its key is already quantized) and the
    dequantized row once it has left.  Under the batch reading the same
    token's value is already quantized (the two readings differ)."""
    rng = np.random.default_rng(41)
    d, G, Gv, R, T = 32, 8, 16, 16, 40       # keys: 32 quantized; values: 25
    q = np.zeros(d, np.float16)
    q[0] = 64
    for sel, where in ((28, "queue, key quantized"), (36, "queue and residual"),
                       (10, "quantized")):
        K = (rng.standard_normal((T, d)) * 0.5).astype(np.float16)
        K[sel, 0] = 8
        V = _randn16(rng, T, d)
        hq = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 64, v_queue=True)
        hb = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 64)
        hq.prefill(K, V)
        hb.prefill(K, V)
        assert (hq.n_quant, hq.n_vquant, hb.n_vquant) == (32, 25, 32)
        out = hq.attend(q, 1.0)
        if sel >= hq.n_vquant:
            np.testing.assert_allclose(out, V[sel].astype(np.float64), rtol=0, atol=1e-12,
                                       err_msg=where)
        else:
            vh = hq.v_u[sel] * np.repeat(hq.v_scale[sel], Gv).astype(np.float64) \
                + np.repeat(hq.v_zero[sel], Gv)
            np.testing.assert_allclose(out, vh, rtol=0, atol=1e-12, err_msg=where)
        if 25 <= sel < 32:
            assert np.abs(hb.attend(q, 1.0) - V[sel].astype(np.float64)).max() > 1e-3


# --------------------------------------------------------------------------
# dense-and-sparse outliers (KVQuant per-vector), KIVI layout
# --------------------------------------------------------------------------

def pin_outlier_selection():
    """A token's outliers are its k largest magnitudes, equal magnitudes going
    to the lower channel: numpy's stable sort agrees on rows full of ties."""
    rng = np.random.default_rng(50)
    for trial in range(300):
        d = int(rng.choice([16, 32, 64, 128]))
        k = int(rng.integers(1, 5))
        row = (rng.integers(-6, 7, d) * 0.5).astype(np.float16)   # many ties, +-0
        if trial % 3 == 0:
            row = _randn16(rng, d, scale=3.0)
        order = np.argsort(-np.abs(row.astype(np.float32)), kind="stable")[:k]
        assert list(oracle.select_outliers(row, k)) == sorted(order.tolist()), (row, k)


def _outlier_head(d, bits, G, Gv, R, k, cap=256):
    return oracle.OracleHead(d, bits, oracle.KIVI, G, Gv, R, 0, cap, outliers=k)


def pin_outlier_statistics():
    """Every quantized token stores its own outliers (channels and exact fp16
    values); each key group's per-channel statistics and each value group's
    come from the inliers alone (the quantizer applied to the elements left
    after removing the outliers); outlier positions hold code 0."""
    rng = np.random.default_rng(51)
    d, G, Gv, R, k = 32, 8, 16, 16, 2
    T = 70
    K, V = _randn16(rng, T + 20, d), _randn16(rng, T + 20, d)
    for arr in (K, V):
        for t in range(T + 20):
            c = rng.integers(0, d, 3)
            arr[t, c] = (rng.choice([-1, 1], 3) * rng.uniform(20, 60, 3)).astype(np.float16)
    h = _outlier_head(d, 2, G, Gv, R, k)
    h.prefill(K[:T], V[:T])
    for i in range(T, T + 20):
        h.append(K[i], V[i])
    n = h.n_quant
    assert n == 80
    for name, X, oidx, oval in (("k", K, h.k_oidx, h.k_oval), ("v", V, h.v_oidx, h.v_oval)):
        for t in range(n):
            sel = oracle.select_outliers(X[t], k)
            assert np.array_equal(oidx[t], sel), (name, t)
            assert np.array_equal(oval[t], X[t, sel].view(np.uint16)), (name, t)
    for g in range(n // G):
        for c in range(d):
            toks = [t for t in range(g * G, (g + 1) * G) if c not in h.k_oidx[t]]
            s_, z_, u_ = oracle.quant_asym(K[toks, c].astype(np.float32), 2)
            assert h.k_scale[g, c] == s_ and h.k_zero[g, c] == z_, (g, c)
            assert list(h.k_u[toks, c]) == list(u_)
            outs = [t for t in range(g * G, (g + 1) * G) if c in h.k_oidx[t]]
            assert all(h.k_u[t, c] == 0 for t in outs)
    for t in range(n):
        for j in range(d // Gv):
            chans = [c for c in range(j * Gv, (j + 1) * Gv) if c not in h.v_oidx[t]]
            s_, z_, u_ = oracle.quant_asym(V[t, chans].astype(np.float32), 2)
            assert h.v_scale[t, j] == s_ and h.v_zero[t, j] == z_, (t, j)
            assert list(h.v_u[t, chans]) == list(u_)


def pin_attention_grid_exact_outliers():
    """Inliers on a grid that every group still spans after its outliers are
    removed, plus one loud outlier per token and tensor: the dense part is
    lossless and the outliers are restored exactly, so attention equals
    torch's fp64 SDPA on the raw tokens (prompt, flushes, residual)."""
    rng = np.random.default_rng(52)
    d, G, Gv, R, k, top = 32, 8, 16, 16, 1, 3
    T = 96
    K = np.empty((T, d), np.float64)
    V = np.empty((T, d), np.float64)
    kout = np.empty(T, int)
    for g in range(T // G):
        while True:   # each channel keeps at least two inlier tokens in the group
            cs = rng.integers(0, d, G)
            if np.bincount(cs, minlength=d).max() <= G - 2:
                break
        kout[g * G:(g + 1) * G] = cs
        for c in range(d):
            step = 2.0 ** -int(rng.integers(1, 4))
            u = rng.integers(0, top + 1, G)
            inl = [i for i in range(G) if cs[i] != c]
            u[inl[0]], u[inl[1]] = 0, top
            K[g * G:(g + 1) * G, c] = float(rng.integers(-8, 8)) * step + u * step
    for t in range(T):
        K[t, kout[t]] = float(rng.choice([-1, 1])) * (64 + int(rng.integers(0, 64)))
        vo = []
        for j in range(d // Gv):
            step = 2.0 ** -int(rng.integers(1, 4))
            u = rng.integers(0, top + 1, Gv)
            u[0], u[1] = 0, top
            V[t, j * Gv:(j + 1) * Gv] = float(rng.integers(-8, 8)) * step + u * step
            vo.append(j * Gv + int(rng.integers(2, Gv)))
        V[t, vo[int(rng.integers(0, len(vo)))]] = float(rng.choice([-1, 1])) * 96
    K16, V16 = K.astype(np.float16), V.astype(np.float16)
    assert np.array_equal(K16.astype(np.float64), K) and np.array_equal(V16.astype(np.float64), V)
    q = (_randn16(rng, d).astype(np.float32) / 16).astype(np.float16)
    tau = 1 / math.sqrt(d)
    # also combined with the value queue and with fp16 metadata (grid steps
    # and bases are fp16 values, so both stay lossless)
    for v_queue, meta_f16 in ((False, False), (True, False), (False, True), (True, True)):
        h = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 256, outliers=k, v_queue=v_queue,
                              meta_f16=meta_f16)
        h.prefill(K16[:75], V16[:75])
        for i in range(75, 91):
            h.append(K16[i], V16[i])
        assert (h.n_quant, h.n_resid) == (80, 11)
        assert h.n_vquant == (91 - 15 if v_queue else 80)
        np.testing.assert_allclose(h.attend(q, tau), _sdpa(q, K16[:91], V16[:91], tau), rtol=0,
                                   atol=1e-12, err_msg=str((v_queue, meta_f16)))


def pin_outlier_isolation_bounds_the_error():
    """Gaussian tokens with a few loud elements: keeping k outliers per token
    apart bounds every other element's error by its group's inlier half-step,
    and the largest error falls well below that of the plain cache."""
    rng = np.random.default_rng(53)
    d, G, Gv, R, k = 64, 16, 32, 32, 2
    K, V = _randn16(rng, 64, d), _randn16(rng, 64, d)
    for t in range(64):
        c = rng.choice(d, 2, replace=False)
        K[t, c] = (rng.choice([-1, 1], 2) * 40).astype(np.float16)
        V[t, c] = (rng.choice([-1, 1], 2) * 40).astype(np.float16)
    ho, hp = _outlier_head(d, 4, G, Gv, R, k), oracle.OracleHead(d, 4, oracle.KIVI, G, Gv, R, 0, 256)
    ho.prefill(K, V)
    hp.prefill(K, V)
    err = {}
    for name, h in (("sparse", ho), ("plain", hp)):
        kh = h.k_u[:64] * np.repeat(h.k_scale[:4], G, axis=0).astype(np.float64) \
            + np.repeat(h.k_zero[:4], G, axis=0)
        if name == "sparse":
            for t in range(64):
                inl = np.ones(d, bool)
                inl[h.k_oidx[t]] = False
                sc = np.repeat(h.k_scale[:4], G, axis=0)[t].astype(np.float64)
                e = np.abs(kh[t] - K[t].astype(np.float64))[inl]
                assert np.all(e <= sc[inl] / 2 + 1e-5), t
                kh[t, h.k_oidx[t]] = K[t, h.k_oidx[t]]
        err[name] = np.abs(kh - K.astype(np.float64)).max()
    assert err["sparse"] * 10 < err["plain"], err


# --------------------------------------------------------------------------
# keys cached before the rotary position embedding
# --------------------------------------------------------------------------

def _rope_sdpa(q, K, V, tau, base, pos0=0):
    """Attention with RoPE in complex form, independent of the oracle's code:
    channel pair (2i, 2i+1) is the complex number x_2i + 1j*x_2i+1, multiplied
    by exp(1j * p * base^(-2i/d)) at position p; a score is Re(sum z_q conj(z_k)).
    Token t sits at pos0 + t, the query at pos0 + T - 1 (T tokens)."""
    d, T = q.size, K.shape[0]
    theta = float(base) ** (-2.0 * np.arange(d // 2) / d)
    pos = pos0 + np.arange(T, dtype=np.float64)
    K64, q64 = K.astype(np.float64), q.astype(np.float64)
    zk = (K64[:, 0::2] + 1j * K64[:, 1::2]) * np.exp(1j * np.outer(pos, theta))
    zq = (q64[0::2] + 1j * q64[1::2]) * np.exp(1j * (pos0 + T - 1) * theta)
    sc = tau * np.real(zk.conj() @ zq)
    p = np.exp(sc - sc.max())
    return (p / p.sum()) @ V.astype(np.float64)


def pin_rope_closed_form():
    """Three fp16 tokens at positions 0, 1, 2, base 100 (theta = 1, 0.1 for
    d = 4), query (1, 0, 1, 0) at position 2: the scores are sin 2 (pair 0
    turned by 2 rad), sin 0.1 (pair 1 turned by one step of 0.1 rad) and 1
    (same position); one-hot values read the softmax weights back."""
    h = oracle.OracleHead(4, 2, oracle.KIVI, 4, 4, 8, 0, 8)      # R > T: all fp16
    K = np.array([[0, 1, 0, 0], [0, 0, 0, 1], [0, 0, 1, 0]], np.float16)
    V = np.eye(3, 4).astype(np.float16)
    h.prefill(K, V)
    q = np.array([1, 0, 1, 0], np.float16)
    for tau in (1.0, 0.7):
        sc = tau * np.array([math.sin(2.0), math.sin(0.1), 1.0])
        p = np.exp(sc - sc.max())
        expect = np.append(p / p.sum(), 0.0)
        np.testing.assert_allclose(h.attend_rope(q, tau, 100.0), expect, rtol=0, atol=1e-12)


def pin_rope_grid_exact_kivi():
    """Lossless KIVI cache (quantized tokens, a flush, then an fp16 residual):
    RoPE attention equals the complex-form attention on the raw tokens."""
    rng = np.random.default_rng(30)
    d, G, Gv, R = 32, 8, 16, 16
    K, V = _grid_tokens(rng, 80, d, 2, G, Gv)
    Kx, Vx = _randn16(rng, 5, d), _randn16(rng, 5, d)
    h = oracle.OracleHead(d, 2, oracle.KIVI, G, Gv, R, 0, 256)
    h.prefill(K[:71], V[:71])
    for i in range(71, 80):
        h.append(K[i], V[i])
    for i in range(5):
        h.append(Kx[i], Vx[i])
    assert h.n_quant == 80 and h.n_resid == 5
    Kall, Vall = np.concatenate([K, Kx]), np.concatenate([V, Vx])
    q = _randn16(rng, d)
    tau = 1 / math.sqrt(d)
    for base in (10000.0, 50.0):
        np.testing.assert_allclose(h.attend_rope(q, tau, base), _rope_sdpa(q, Kall, Vall, tau, base),
                                   rtol=0, atol=1e-11)


def pin_rope_grid_exact_innerq():
    """Lossless InnerQ cache with sinks, quantized tokens and a window that
    has wrapped (tokens evicted into the quantized region by appends), with
    and without the key normalization (power-of-two factors)."""
    rng = np.random.default_rng(31)
    d, S, W, T, n_app = 128, 4, 8, 60, 13
    for k_norm in (False, True):
        K, V = _grid_tokens(rng, T + n_app, d, 4, 1, 64, sym_groups=True)
        if k_norm:
            K[0] = np.repeat(np.float16([32, 128]), 64) * np.where(rng.integers(0, 2, d), 1, -1)
        h = oracle.OracleHead(d, 4, oracle.INNERQ, 64, 64, W, S, 256, k_norm=k_norm)
        h.prefill(K[:T], V[:T])
        for i in range(T, T + n_app):
            h.append(K[i], V[i])
        assert h.n_quant == T + n_app - S - W and h.n_resid == W
        q = _randn16(rng, d)
        tau = 1 / math.sqrt(d)
        np.testing.assert_allclose(h.attend_rope(q, tau, 10000.0),
                                   _rope_sdpa(q, K, V, tau, 10000.0), rtol=0, atol=1e-11)


def pin_rope_shift_invariance():
    """Scores depend on positions only through their differences: moving
    every token and the query by the same offset leaves the output unchanged
    (random, lossy data: quantized, sink and window tokens)."""
    rng = np.random.default_rng(32)
    d = 64
    K, V = _randn16(rng, 200, d), _randn16(rng, 200, d)
    q = _randn16(rng, d)
    for head in (oracle.OracleHead(d, 2, oracle.KIVI, 16, 32, 32, 0, 256),
                 oracle.OracleHead(d, 4, oracle.INNERQ, 32, 32, 16, 3, 256)):
        head.prefill(K[:180], V[:180])
        for i in range(180, 200):
            head.append(K[i], V[i])
        a = head.attend_rope(q, 0.125, 10000.0)
        b = head.attend_rope(q, 0.125, 10000.0, pos0=12345)
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-9)
        assert np.abs(a - head.attend(q, 0.125)).max() > 1e-3   # RoPE does change it


def pin_workload_shapes():
    """The named workloads have the shapes their descriptions give."""
    w = synth.WORKLOADS["llama2_7b_2bit"]
    assert (w.batch, w.n_kv_heads, w.head_dim, w.ctx, w.bits, w.k_group, w.residual) == \
        (8, 32, 128, 4096, 2, 32, 128)
    assert w.n_outliers() == 82
    assert synth.WORKLOADS["gqa_2bit"].n_outliers() == 20
    assert synth.WORKLOADS["innerq_1m"].ctx == 1048576


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# --------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin
# --------------------------------------------------------------------------

MUTANTS = [
    ("ties away from zero", "float r = rintf((x[i] - mn) / s);", "float r = roundf((x[i] - mn) / s);"),
    ("zero = max", "*zero = mn;\n  if (mx == mn)", "*zero = mx;\n  if (mx == mn)"),
    ("2^b levels", "const float s = (mx - mn) / top;", "const float s = (mx - mn) / (top + 1.0f);"),
    ("sym zero off by one", "*zero = -(float)half * s;\n  for (int i = 0; i < n; ++i) {\n    float r = rintf(x[i] / s);",
     "*zero = -(float)(half - 1) * s;\n  for (int i = 0; i < n; ++i) {\n    float r = rintf(x[i] / s);"),
    ("strict mode rule", "return fabsf(mx + mn) <= step;", "return fabsf(mx + mn) < step;"),
    ("key meta by token", "const int64_t i = (t / s->k_group) * d + c;", "const int64_t i = (t % s->k_group) * d + c;"),
    ("value zero dropped", "return (double)s->v_u[t * d + c] * (double)s->v_scale[i] + (double)s->v_zero[i];",
     "return (double)s->v_u[t * d + c] * (double)s->v_scale[i];"),
    ("flush one early", "if (s->n_resid == R) {", "if (s->n_resid == R - 1) {"),
    ("prefill split by G", "const int64_t nq = T - T % R;", "const int64_t nq = T - T % G;"),
    ("softmax sign", "sc[j] = exp(sc[j] - m); l += sc[j]; }\n\n  i = 0;",
     "sc[j] = exp(m - sc[j]); l += sc[j]; }\n\n  i = 0;"),
    ("rope softmax sign", "sc[j] = exp(sc[j] - m); l += sc[j]; }\n  for (int64_t j = 0; j < n; ++j) {\n    token_row",
     "sc[j] = exp(m - sc[j]); l += sc[j]; }\n  for (int64_t j = 0; j < n; ++j) {\n    token_row"),
    ("tau dropped", "acc += qd[c] * (s->k_normalize ? (double)s->k_norm[c] : 1.0) * key_hat(s, t, c);\n    sc[i] = tau * acc;",
     "acc += qd[c] * (s->k_normalize ? (double)s->k_norm[c] : 1.0) * key_hat(s, t, c);\n    sc[i] = acc;"),
    ("key factor not folded into q", "acc += qd[c] * (s->k_normalize ? (double)s->k_norm[c] : 1.0)",
     "acc += qd[c] * 1.0"),
    ("key factor over the quantized tokens only", "for (int64_t t = 0; t < T; ++t) {\n      const float x = fabsf",
     "for (int64_t t = s->n_sink < T ? s->n_sink : T; t < T; ++t) {\n      const float x = fabsf"),
    ("zero channel factor 0", "s->k_norm[c] = a > 0.0f ? a : 1.0f;", "s->k_norm[c] = a;"),
    ("big-endian pack", "<< ((c % per) * bits)", "<< ((per - 1 - c % per) * bits)"),
    ("evict newest", "innerq_quant_kv(s, s->k_res, s->v_res, s->n_quant);", "innerq_quant_kv(s, k, v, s->n_quant);"),
    ("half exponent bias", "expo - 25", "expo - 24"),
    ("rope query one position late", "rope_rotate(qd, d, base, (double)(pos0 + n - 1));",
     "rope_rotate(qd, d, base, (double)(pos0 + n));"),
    ("rope pairs as halves", "const int ca = 2 * i, cb = 2 * i + 1;", "const int ca = i, cb = i + d / 2;"),
    ("rope keys turned backwards", "rope_rotate(row, d, base, (double)(pos0 + j));",
     "rope_rotate(row, d, base, -(double)(pos0 + j));"),
    ("rope theta exponent", "pow(base, -2.0 * i / d)", "pow(base, -1.0 * i / d)"),
    ("rope key factor dropped", "row[c] = k ? (s->k_normalize ? (double)s->k_norm[c] : 1.0) * key_hat(s, j, c)",
     "row[c] = k ? key_hat(s, j, c)"),
    ("rope window newest first", "const uint16_t *src = (k ? s->k_res : s->v_res) + j * d;",
     "const uint16_t *src = (k ? s->k_res : s->v_res) + (s->n_resid - 1 - j) * d;"),
    ("queue holds R values after the prompt", "(T >= R ? T - (R - 1) : 0)", "(T >= R ? T - R : 0)"),
    ("queue pops newest", "kivi_quant_value_token(s, s->v_res, s->n_vquant);",
     "kivi_quant_value_token(s, s->v_res + (int64_t)(R - 1) * d, s->n_vquant);"),
    ("queue ignored by attention", "return s->v_queue ? s->n_vquant : s->n_quant;", "return s->n_quant;"),
    ("f16 codes from the fp32 scale", "float r = s == 0.0f ? 0.0f : rintf((x[i] - z) / s);",
     "float r = s == 0.0f ? 0.0f : rintf((x[i] - z) / ((mx - mn) / top));"),
    ("f16 symmetric codes from the fp32 scale", "float r = s == 0.0f ? 0.0f : rintf(x[i] / s);",
     "float r = s == 0.0f ? 0.0f : rintf(x[i] / (a / lim));"),
    ("fp32 to fp16 truncates", "if (rem > half || (rem == half && (q & 1u))) q += 1;", "if (0) q += 1;"),
    ("fp32 to fp16 ties away", "(rem == half && (q & 1u))", "(rem == half)"),
    ("outliers are the smallest", "if (!taken[c] && m > bm) {", "if (!taken[c] && (bm < 0.0f || m < bm)) {"),
    ("outlier ties to the higher channel", "if (!taken[c] && m > bm) {", "if (!taken[c] && m >= bm) {"),
    ("outliers kept in the statistics", "if (!is_out[i]) in[m++] = x[i];", "in[m++] = x[i];"),
    ("key outlier not restored", "if (o >= 0) return (double)orc_half_to_float(s->k_oval[t * s->outliers + o]);",
     "if (0) return (double)orc_half_to_float(s->k_oval[t * s->outliers + o]);"),
    ("value outlier not restored", "if (o >= 0) return (double)orc_half_to_float(s->v_oval[t * s->outliers + o]);",
     "if (0) return (double)orc_half_to_float(s->v_oval[t * s->outliers + o]);"),
    ("value group transposed", "x[i] = orc_half_to_float(src[j * Gv + i]);", "x[i] = orc_half_to_float(src[i * (d / Gv) + j]);"),
]


def test_planted_mistakes_are_caught():
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kvq_oracle.c")).read()
    tmp = tempfile.mkdtemp(prefix="orc_mut_")
    try:
        survivors = []
        for i, (name, old, new) in enumerate(MUTANTS):
            assert src.count(old) == 1, name
            path = os.path.join(tmp, "m%d.c" % i)
            with open(path, "w") as f:
                f.write(src.replace(old, new))
            so = oracle.build(force=True, src=path, out=os.path.join(tmp, "m%d.so" % i))
            failed = False
            with oracle.using_library(so):
                for pin in PINS:
                    try:
                        pin()
                    except (AssertionError, ValueError):
                        failed = True
                        break
            if not failed:
                survivors.append(name)
        assert not survivors, "mutants not caught: %s" % survivors
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
