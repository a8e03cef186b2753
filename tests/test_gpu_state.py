"""Cache state on the device (needs a GB300).

Guard bands: every cache buffer, the scratch and the output sit inside a
larger allocation whose margins hold a canary byte; prefill, appends with
flushes and window evictions, and every decode path (tensor-core MHA,
grouped-query, general, pre-RoPE, one-launch append + decode) must leave the
margins untouched.  This stands in for a device memory checker, which is
closed on this pool: it catches writes past either end of a buffer.

Checkpoint / resume: the cache is plain caller-owned buffers plus the host
counters, so copying both makes a checkpoint; the copy, resumed, must
evolve bit for bit like the original.
"""
import numpy as np
import pytest
import torch

from bit_kv_cache_14_gb300 import kvq, synth
from parity_util import new_cache

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
S = synth.scaled
PAD = 4096          # bytes of margin on each side (keeps 16-byte alignment)
CANARY = 0xA5


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


def _guarded(nbytes, device):
    """A zeroed uint8 buffer of nbytes inside canary margins: (inner, whole)."""
    whole = torch.full((PAD + nbytes + PAD,), CANARY, dtype=torch.uint8, device=device)
    inner = whole[PAD:PAD + nbytes]
    inner.zero_()
    return inner, whole


def guard_cache(cache):
    """Moves every buffer of a QuantizedKVCache (and its scratch and status
    word) into guarded allocations; returns the list of whole allocations."""
    wholes = []
    for name in cache._BUFS:
        n = getattr(cache.sizes, name)
        inner, whole = _guarded(max(n, 16), cache.device)
        cache.bufs[name] = inner
        setattr(cache.view, name, inner.data_ptr() if n else None)
        wholes.append((name, whole))
    ws, whole = _guarded(cache.ws_bytes, cache.device)
    cache.ws = ws
    wholes.append(("workspace", whole))
    st, whole = _guarded(16, cache.device)
    cache.status = st.view(torch.int32)
    cache.view.dev_status = st.data_ptr()
    wholes.append(("status", whole))
    return wholes


def guarded_out(shape, device):
    n = int(np.prod(shape)) * 4
    inner, whole = _guarded(n, device)
    return inner.view(torch.float32).view(*shape), whole


def check_margins(wholes):
    torch.cuda.synchronize()
    for name, whole in wholes:
        head, tail = whole[:PAD], whole[-PAD:]
        assert bool((head == CANARY).all()), "write before %s" % name
        assert bool((tail == CANARY).all()), "write past %s" % name


GUARD_CASES = {
    "tc_mha": (S(W["llama2_7b_2bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=700,
                 residual=64, n_append=70), "fused"),
    "gqa": (S(W["gqa_2bit"], batch=1, n_q_heads=8, n_kv_heads=2, ctx=800, n_append=130), "plain"),
    "general_d64": (S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2, head_dim=64,
                      ctx=300, k_group=16, v_group=16, residual=48, n_append=50), "plain"),
    "innerq_window": (S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=400,
                        n_append=40, k_norm=True), "plain"),
    "kivi_rope": (S(W["llama2_7b_2bit"], batch=1, n_q_heads=4, n_kv_heads=2, ctx=500,
                    n_append=130), "rope"),
}


@pytest.mark.parametrize("name", sorted(GUARD_CASES))
def test_guard_bands_stay_untouched(name):
    w, mode = GUARD_CASES[name]
    max_ctx = w.ctx + w.n_append
    cache = new_cache(w, max_ctx)
    wholes = guard_cache(cache)
    K, V = synth.prompt(w)
    Kd, Vd = torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda()
    cache.prefill(Kd, Vd)
    check_margins(wholes)
    Ks, Vs = synth.streamed(w, w.n_append)
    out, whole_out = guarded_out((w.batch, w.n_q_heads, w.head_dim), cache.device)
    wholes.append(("output", whole_out))
    for s in range(w.n_append):
        k, v = torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda()
        q = torch.from_numpy(synth.queries(w, s)).cuda()
        if mode == "fused":
            cache.append_decode(k, v, q, out=out)
        else:
            cache.append(k, v)
            if mode == "rope":
                cache.decode_rope(q, 10000.0, out=out)
            else:
                cache.decode(q, out=out)
        if s % 16 == 15 or s == w.n_append - 1:
            check_margins(wholes)
    assert cache.device_status() == 0
    check_margins(wholes)


def _checkpoint(cache):
    c = kvq.QuantizedKVCache(cache.cfg, cache.device)
    for name in cache._BUFS:
        c.bufs[name].copy_(cache.bufs[name])
    for f in ("n_quant", "n_resid", "n_sink", "ring_head"):
        setattr(c.view, f, getattr(cache.view, f))
    return c


@pytest.mark.parametrize("name", ["kivi", "innerq"])
def test_checkpoint_resume_is_bit_exact(name):
    w = (S(W["llama2_7b_2bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=600, residual=64,
           n_append=150) if name == "kivi" else
         S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=500, n_append=60))
    cache = new_cache(w, w.ctx + w.n_append)
    K, V = synth.prompt(w)
    cache.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    Ks, Vs = synth.streamed(w, w.n_append)
    half = w.n_append // 3
    for s in range(half):
        cache.append(torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda())
    torch.cuda.synchronize()
    resumed = _checkpoint(cache)
    for s in range(half, w.n_append):
        k, v = torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda()
        q = torch.from_numpy(synth.queries(w, s)).cuda()
        cache.append(k, v)
        resumed.append(k, v)
        a, b = cache.decode(q), resumed.decode(q)
        assert torch.equal(a, b), s
    for f in ("n_quant", "n_resid", "n_sink", "ring_head"):
        assert getattr(cache.view, f) == getattr(resumed.view, f)
    torch.cuda.synchronize()
    for name in cache._BUFS:
        assert torch.equal(cache.bufs[name], resumed.bufs[name]), name
    assert cache.device_status() == 0 and resumed.device_status() == 0
