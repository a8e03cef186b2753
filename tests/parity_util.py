"""Shared helpers of the GPU parity tests: drive the CUDA path (through the C
ABI binding) and the CPU oracle on the same seeded inputs and compare.

Bit-exact: packed codes, scales, zeros, mode bits, fp16 residual / sink /
window rows.  Attention output: max-abs error against the oracle's fp64
result <= ATOL (fp32 accumulation on the device).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from bit_kv_cache_14_gb300 import kvq, synth

ATOL = 2e-3


def new_cache(w, max_ctx=None):
    return kvq.QuantizedKVCache(kvq.config_of(w, max_ctx), "cuda")


def oracle_head(w, b, h, max_ctx, T=None):
    """Oracle state of head (b, h) after the prefill of its T prompt tokens
    (default: the workload's ctx)."""
    T = w.ctx if T is None else int(T)
    head = oracle.OracleHead.for_workload(w, cap=max_ctx)
    K, V = synth.head_tokens(w, b, h, 0, w.ctx)
    head.prefill(K[:T], V[:T])
    head.nq_prefill = head.n_quant  # evictions since the prefill give the window's ring offset
    return head


def _same_bits(got, exp, what):
    assert got.size == exp.size, (what, got.shape, exp.shape)
    assert np.array_equal(got.reshape(-1).view(np.uint32), exp.reshape(-1).view(np.uint32)), what


def check_head_state(cache, w, b, h, head):
    """Byte-for-byte comparison of one head's cache contents with the oracle.
    The oracle's counters say which rows of the cache are live (under ragged
    lengths the host counters describe the longest sequence only)."""
    ragged = getattr(w, "ragged", False)
    if not ragged:
        assert cache.n_quant == head.n_quant, (cache.n_quant, head.n_quant)
        assert cache.n_resid == head.n_resid
    n, nvq = head.n_quant, head.n_vquant
    where = "(b=%d h=%d)" % (b, h)
    kc = cache.codes("k")[b, h, :n].cpu().numpy()
    vc = cache.codes("v")[b, h, :nvq].cpu().numpy()
    assert np.array_equal(kc, head.packed_k()), "key codes differ " + where
    assert np.array_equal(vc, head.packed_v()), "value codes differ " + where
    ks_o, kz_o = head.k_meta()
    vs_o, vz_o = head.v_meta()
    ks = cache.meta("k_scale")[b, h, : ks_o.size].cpu().numpy()
    kz = cache.meta("k_zero")[b, h, : kz_o.size].cpu().numpy()
    vs = cache.meta("v_scale")[b, h, : vs_o.size].cpu().numpy()
    vz = cache.meta("v_zero")[b, h, : vz_o.size].cpu().numpy()
    for got, exp, name in ((ks, ks_o, "k_scale"), (kz, kz_o, "k_zero"), (vs, vs_o, "v_scale"),
                           (vz, vz_o, "v_zero")):
        _same_bits(got, exp, "%s differs %s" % (name, where))
    if getattr(w, "outliers", 0):
        for which, rows, oidx, oval in (("k", n, head.k_oidx, head.k_oval),
                                        ("v", nvq, head.v_oidx, head.v_oval)):
            idx, bits = cache.outlier_lists(which)
            idx = idx[b, h, :rows].cpu().numpy()
            bits = bits[b, h, :rows].cpu().numpy()
            assert np.array_equal(idx, oidx[:rows].astype(np.int32)), \
                "%s outlier channels differ %s" % (which, where)
            assert np.array_equal(bits, oval[:rows].astype(np.int32)), \
                "%s outlier values differ %s" % (which, where)
    if getattr(w, "k_norm", False):
        kn = cache.key_norms()[b, h].cpu().numpy()
        assert np.array_equal(kn.view(np.uint32), head.key_norms().view(np.uint32)), \
            "key factors differ " + where
    kr_o, vr_o = head.residual_tokens()
    nr = head.n_resid
    if w.scheme == synth.KIVI:
        R = w.residual
        kr = cache.fp16_rows("k_res", R)[b, h, :nr].cpu().numpy()
        if getattr(w, "v_queue", False):
            # the queue's values, oldest first: token t sits in ring slot t mod R
            vr_o = head.value_queue()
            slots = [(nvq + i) % R for i in range(len(vr_o))]
            vr = cache.fp16_rows("v_res", R)[b, h].cpu().numpy()[slots]
        else:
            vr = cache.fp16_rows("v_res", R)[b, h, :nr].cpu().numpy()
    else:
        # window ring: slot (ring_head + i) % W holds the i-th oldest token, and
        # the ring moves one slot per eviction since the prefill
        W = w.residual
        ring_head = (head.n_quant - head.nq_prefill) % W if W > 0 else 0
        if not ragged:
            assert cache.ring_head == ring_head
        order = [(ring_head + i) % W for i in range(nr)] if nr == W else list(range(nr))
        if W > 0:
            kr = cache.fp16_rows("k_res", W)[b, h].cpu().numpy()[order]
            vr = cache.fp16_rows("v_res", W)[b, h].cpu().numpy()[order]
        else:
            kr = vr = np.zeros((0, w.head_dim), np.float16)
        ns = head.n_sink_used
        if not ragged:
            assert cache.n_sink == ns
        if ns:
            ksk_o, vsk_o = head.sink_tokens()
            ksk = cache.fp16_rows("k_sink", w.n_sink)[b, h, :ns].cpu().numpy()
            vsk = cache.fp16_rows("v_sink", w.n_sink)[b, h, :ns].cpu().numpy()
            assert np.array_equal(ksk.view(np.uint16), ksk_o.view(np.uint16))
            assert np.array_equal(vsk.view(np.uint16), vsk_o.view(np.uint16))
        for which, ng, sym in (("k", w.head_dim // w.k_group, head.k_sym),
                               ("v", w.head_dim // w.v_group, head.v_sym)):
            nbits = n * ng
            words = cache.modes(which)[b, h].cpu().numpy().view(np.uint32)
            exp = oracle.pack_modes(sym[:n, :ng].reshape(-1))
            full = nbits // 32
            assert np.array_equal(words[:full], exp[:full]), "%s mode bits differ" % which
            if nbits % 32:
                mask = np.uint32((1 << (nbits % 32)) - 1)
                assert (words[full] & mask) == (exp[full] & mask), "%s mode tail" % which
    assert np.array_equal(kr.view(np.uint16), kr_o.view(np.uint16)), "key residual differs " + where
    assert np.array_equal(vr.view(np.uint16), vr_o.view(np.uint16)), \
        "value residual differs " + where


def check_decode(out, q, w, b, h, head, tau, rope_base=None):
    """Attention output of the query heads of KV head (b, h) vs the oracle
    (keys cached before the rotary embedding when rope_base is given)."""
    rg = w.group_ratio
    worst = 0.0
    for hq in range(h * rg, (h + 1) * rg):
        if rope_base is None:
            exp = head.attend(q[b, hq], tau)
        else:
            exp = head.attend_rope(q[b, hq], tau, rope_base)
        got = out[b, hq].astype(np.float64)
        err = float(np.max(np.abs(got - exp)))
        worst = max(worst, err)
        assert err <= ATOL, "attention error %.3g > %g (b=%d hq=%d)" % (err, ATOL, b, hq)
    return worst


def run_workload(w, heads=None, n_append=None, decode_every=None, max_ctx=None,
                 check_steps=None, rope_base=None):
    """Prefill + appends + decodes on the GPU; oracle on `heads` (default: all).
    With rope_base, the decodes are kvq_decode_attention_rope (keys and
    queries cached / given before the rotary embedding).  Returns the worst
    attention error seen."""
    n_append = w.n_append if n_append is None else n_append
    max_ctx = w.ctx + n_append if max_ctx is None else max_ctx
    if heads is None:
        heads = [(b, h) for b in range(w.batch) for h in range(w.n_kv_heads)]
    K, V = synth.prompt(w)
    lens = synth.prompt_lengths(w)
    cache = new_cache(w, max_ctx)
    if getattr(w, "ragged", False):
        cache.prefill_ragged(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(), lens)
    else:
        cache.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    del K, V
    heads_o = {bh: oracle_head(w, bh[0], bh[1], max_ctx, lens[bh[0]]) for bh in heads}
    torch.cuda.synchronize()
    for (b, h), ho in heads_o.items():
        check_head_state(cache, w, b, h, ho)
    tau = 1.0 / math.sqrt(w.head_dim)
    worst = 0.0
    Ks, Vs = synth.streamed(w, n_append) if n_append else (None, None)
    steps = set(check_steps or [])
    if decode_every is None:
        steps |= {n_append}
    else:
        steps |= set(range(0, n_append + 1, decode_every)) | {n_append}
    for s in range(n_append + 1):
        if s > 0:
            cache.append(torch.from_numpy(Ks[s - 1]).cuda(), torch.from_numpy(Vs[s - 1]).cuda())
            for (b, h), ho in heads_o.items():
                ho.append(Ks[s - 1, b, h], Vs[s - 1, b, h])
        if s in steps:
            q = synth.queries(w, s)
            qd = torch.from_numpy(q).cuda()
            out = (cache.decode(qd) if rope_base is None
                   else cache.decode_rope(qd, rope_base)).cpu().numpy()
            for (b, h), ho in heads_o.items():
                check_head_state(cache, w, b, h, ho)
                worst = max(worst, check_decode(out, q, w, b, h, ho, tau, rope_base))
    assert cache.device_status() == 0
    return worst
