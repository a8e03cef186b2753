"""CUDA path vs the CPU oracle, through the C ABI (needs a GB300).

Small cases run the oracle on every head; they span several key tiles and
decode splits, ragged residuals, flushes, and the degenerate cache states.
The full-size cases use the five named workloads at their own sizes, in the
launch configuration the benchmark times, and compare sampled heads.
"""
import math

import numpy as np
import pytest
import torch

from bit_kv_cache_14_gb300 import kvq, synth
from parity_util import ATOL, check_decode, check_head_state, new_cache, run_workload

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
S = synth.scaled


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


SMALL = {
    "tiny": W["tiny"],
    "llama_small": S(W["llama2_7b_2bit"], batch=2, n_q_heads=3, n_kv_heads=3, ctx=1000,
                     n_append=300),
    "kivi4_small": S(W["kivi_4bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=777, n_append=200),
    "gqa_small": S(W["gqa_2bit"], batch=2, n_q_heads=16, n_kv_heads=4, ctx=1500, n_append=140),
    "innerq_small": S(W["innerq_1m"], batch=1, n_q_heads=4, n_kv_heads=4, ctx=3000, n_append=60),
    "kivi_d64_g16": S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2, head_dim=64,
                      ctx=600, k_group=16, v_group=16, residual=48, n_append=100),
    "kivi_g128_r128": S(W["kivi_4bit"], batch=1, n_q_heads=2, n_kv_heads=1, ctx=700,
                        k_group=128, v_group=128, residual=128, n_append=140),
    "kivi_r_eq_g": S(W["llama2_7b_2bit"], batch=1, n_q_heads=8, n_kv_heads=1, ctx=333,
                     k_group=32, residual=32, n_append=70),
    "innerq_d64_g16_2bit": S(W["innerq_1m"], batch=2, n_q_heads=2, n_kv_heads=2, head_dim=64,
                             bits=2, k_group=16, v_group=32, ctx=500, n_sink=3, residual=8,
                             n_append=20),
    "innerq_gqa": S(W["innerq_1m"], batch=1, n_q_heads=8, n_kv_heads=2, ctx=900, n_append=40),
    # head_dim 128 MHA shapes that take the tensor-core decode path
    "kivi_g16_mha": S(W["llama2_7b_2bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=1100,
                      k_group=16, residual=64, n_append=90),
    "kivi_g128_mha_4bit": S(W["kivi_4bit"], batch=1, n_q_heads=3, n_kv_heads=3, ctx=1500,
                            k_group=128, v_group=32, residual=128, n_append=140),
    "innerq_g32_2bit": S(W["innerq_1m"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=700, bits=2,
                         k_group=32, v_group=32, n_append=30),
    # grouped-query tensor-core path: 2 query heads per KV head, G 64, two
    # value groups (the gqa_small case covers 4 heads per KV head, G 32)
    "gqa_rg2_g64": S(W["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=4, ctx=900, k_group=64,
                     v_group=64, residual=128, n_append=150),
    # InnerQ with the one-shot per-channel key normalization: MHA (tensor-core
    # kernel), 2-bit with 32-channel key groups, and grouped-query (general kernel)
    "innerq_knorm": S(W["innerq_1m"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=900, n_append=40,
                      k_norm=True),
    "innerq_knorm_2bit": S(W["innerq_1m"], batch=1, n_q_heads=3, n_kv_heads=3, ctx=700, bits=2,
                           k_group=32, v_group=32, n_append=30, k_norm=True),
    "innerq_knorm_gqa": S(W["innerq_1m"], batch=1, n_q_heads=8, n_kv_heads=2, ctx=600,
                          n_append=40, k_norm=True),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workload_all_heads(name):
    w = SMALL[name]
    worst = run_workload(w, decode_every=max(1, w.n_append // 4))
    assert worst <= ATOL


EDGE = {
    # nothing quantized: the residual holds everything (textbook attention)
    "kivi_short_prompt": S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=100,
                           n_append=20),
    # empty prompt, every token streamed in (first flush at R)
    "kivi_empty_prompt": S(W["llama2_7b_2bit"], batch=1, n_q_heads=1, n_kv_heads=1, ctx=0,
                           n_append=260),
    # prompt exactly R: no residual left after prefill
    "kivi_prompt_eq_r": S(W["llama2_7b_2bit"], batch=1, n_q_heads=1, n_kv_heads=1, ctx=128,
                          n_append=3),
    # InnerQ prompt shorter than the sinks
    "innerq_prompt_lt_sink": S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=2,
                               n_append=50),
    # InnerQ without a recent window: every token past the sinks is quantized
    "innerq_no_window": S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=300,
                          residual=0, n_append=10),
    # InnerQ without sinks
    "innerq_no_sink": S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=300, n_sink=0,
                        n_append=10),
    # the grouped-query kernel's corners: quantized tokens arriving one at a
    # time (a single short tile of 1, 2, ... tokens), no fp16 rows at all, and
    # a KIVI prompt shorter than R that reaches its first flush
    "innerq_gqa_prompt_lt_sink": S(W["innerq_1m"], batch=2, n_q_heads=8, n_kv_heads=2, ctx=2,
                                   n_append=50),
    "innerq_gqa_no_window_no_sink": S(W["innerq_1m"], batch=2, n_q_heads=8, n_kv_heads=2, ctx=300,
                                      residual=0, n_sink=0, n_append=10),
    "kivi_gqa_short_prompt": S(W["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=2, ctx=100,
                               n_append=40),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(name):
    w = EDGE[name]
    run_workload(w, decode_every=max(1, w.n_append // 5))


def test_empty_cache_decodes_to_zero():
    w = S(W["tiny"], ctx=0)
    cache = new_cache(w, 64)
    q = torch.from_numpy(synth.queries(w)).cuda()
    cache.prefill(torch.zeros(1, 1, 0, 64, dtype=torch.float16, device="cuda"),
                  torch.zeros(1, 1, 0, 64, dtype=torch.float16, device="cuda"))
    out = cache.decode(q)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_grid_exact_equals_sdpa():
    """Lossless data: the fused kernel equals plain fp64 softmax attention on
    the raw fp16 keys and values (independent of the oracle)."""
    rng = np.random.default_rng(5)
    B, H, T, d, G = 2, 2, 512, 128, 32
    K = np.empty((B, H, T, d), np.float64)
    V = np.empty((B, H, T, d), np.float64)
    for b in range(B):
        for h in range(H):
            for g in range(T // G):
                for c in range(d):
                    u = rng.integers(0, 4, G)
                    u[0], u[1] = 0, 3
                    K[b, h, g * G:(g + 1) * G, c] = float(rng.integers(-8, 8)) / 4 + u / 4.0
            for t in range(T):
                for j in range(d // 32):
                    u = rng.integers(0, 4, 32)
                    u[0], u[1] = 0, 3
                    V[b, h, t, j * 32:(j + 1) * 32] = float(rng.integers(-8, 8)) / 8 + u / 8.0
    w = S(W["llama2_7b_2bit"], batch=B, n_q_heads=H, n_kv_heads=H, ctx=T, n_append=0)
    cache = new_cache(w, T)
    cache.prefill(torch.from_numpy(K.astype(np.float16)).cuda(),
                  torch.from_numpy(V.astype(np.float16)).cuda())
    q = rng.standard_normal((B, H, d)).astype(np.float16)
    out = cache.decode(torch.from_numpy(q).cuda()).cpu().double()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[:, :, None, :], torch.from_numpy(K),
        torch.from_numpy(V), scale=1 / math.sqrt(d))[:, :, 0, :]
    assert (out - ref).abs().max().item() <= ATOL


def test_decode_step_host_matches_device_path():
    w = S(W["llama2_7b_2bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=600, n_append=4)
    K, V = synth.prompt(w)
    Ks, Vs = synth.streamed(w, 4)
    a, b = new_cache(w), new_cache(w)
    for c in (a, b):
        c.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    shape_q = (w.batch, w.n_q_heads, w.head_dim)
    d_in = torch.empty(a.step_input_halves(), dtype=torch.float16, device="cuda")
    d_out = torch.empty(shape_q, dtype=torch.float32, device="cuda")
    h_out = torch.empty(shape_q, dtype=torch.float32).pin_memory()
    for s in range(4):
        q = synth.queries(w, s)
        h_in = torch.from_numpy(np.concatenate([Ks[s].ravel(), Vs[s].ravel(), q.ravel()]))
        h_in = h_in.pin_memory()
        a.decode_step_host(h_in, h_out, d_in, d_out)
        torch.cuda.synchronize()
        b.append(torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda())
        ref = b.decode(torch.from_numpy(q).cuda()).cpu()
        assert torch.equal(h_out, ref)


def test_fused_append_decode_matches_two_launches():
    """kvq_append_decode (one launch unless the append flushes) leaves the same
    cache and returns the same output as kvq_append + kvq_decode_attention."""
    w = S(W["llama2_7b_2bit"], batch=2, n_q_heads=3, n_kv_heads=3, ctx=600, residual=64,
          n_append=70)
    K, V = synth.prompt(w)
    Ks, Vs = synth.streamed(w, w.n_append)
    a, b = new_cache(w), new_cache(w)
    for c in (a, b):
        c.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    fused = flushed = 0
    for s in range(w.n_append):
        q = torch.from_numpy(synth.queries(w, s)).cuda()
        k, v = torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda()
        will_flush = a.n_resid + 1 == w.residual
        got = a.append_decode(k, v, q)
        n = a.last_launch_count()
        assert n == (2 if will_flush else 1)
        fused += n == 1
        flushed += n == 2
        b.append(k, v)
        ref = b.decode(q)
        assert torch.equal(got, ref), s
        assert (a.n_quant, a.n_resid) == (b.n_quant, b.n_resid)
    assert fused > 0 and flushed > 0
    torch.cuda.synchronize()
    for name in ("k_res", "v_res"):
        assert torch.equal(a.bufs[name], b.bufs[name])
    assert torch.equal(a.bufs["blocks"], b.bufs["blocks"])
    assert a.device_status() == 0


def test_errors_leave_state_unchanged():
    w = S(W["tiny"], ctx=64)
    cache = new_cache(w, 64)
    K, V = synth.prompt(w)
    cache.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    k = torch.zeros(1, 1, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(kvq.KVQError) as e:
        cache.append(k, k)                     # cache is full (max_ctx = 64)
    assert e.value.code == kvq.KVQ_ECAPACITY
    assert cache.n_quant == 64 and cache.n_resid == 0
    with pytest.raises(kvq.KVQError) as e:
        cache.append(k[..., 1:], k[..., 1:])   # misaligned device pointer
    assert e.value.code in (kvq.KVQ_EALIGN, kvq.KVQ_ECAPACITY)
    assert cache.device_status() == 0


# ---------------------------------------------------------------------------
# full-size workloads, sampled heads
# ---------------------------------------------------------------------------

def _sample_heads(w, n=3):
    B, H = w.batch, w.n_kv_heads
    picks = [(0, 0), (B - 1, H - 1), (B // 2, H // 2)]
    return sorted(set(picks))[:n]


# the named workloads, the grouped-query layer with 4-bit codes and the
# InnerQ cache on the grouped-query layer's shape (the benchmark's derived
# shapes)
FULL_SIZE = {n: W[n] for n in ("llama2_7b_2bit", "kivi_4bit", "gqa_2bit", "innerq_1m")}
FULL_SIZE["gqa_4bit"] = S(W["gqa_2bit"], bits=4)
FULL_SIZE["innerq_gqa"] = S(W["innerq_1m"], batch=64, n_q_heads=32, n_kv_heads=8, ctx=16384)


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(FULL_SIZE))
def test_full_size_sampled(name):
    w = FULL_SIZE[name]
    heads = _sample_heads(w, 2 if name == "innerq_1m" else 3)
    n_append = w.n_append
    steps = [1, n_append] if n_append > 1 else [n_append]
    run_workload(w, heads=heads, n_append=n_append, decode_every=None, check_steps=steps)


def test_forced_timeout_is_reported_and_recoverable():
    """The decode kernel's bounded pipeline wait gives up on a barrier that
    nothing completes, records KVQ_ETIMEOUT, drains its own copies and
    returns; the context stays usable and the next decode is correct."""
    w = S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=512, n_append=0)
    K, V = synth.prompt(w)
    cache = new_cache(w, 512)
    cache.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    q = torch.from_numpy(synth.queries(w)).cuda()
    good = cache.decode(q).clone()
    assert cache.device_status() == 0
    try:
        kvq.debug_stall_waits(1000)
        cache.decode(q)
        assert cache.device_status() == kvq.KVQ_ETIMEOUT
    finally:
        kvq.debug_stall_waits(0)
    again = cache.decode(q)
    assert cache.device_status() == 0
    assert torch.equal(again, good)
