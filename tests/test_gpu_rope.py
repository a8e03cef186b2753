"""Decode attention over keys cached before the rotary position embedding
(kvq_decode_attention_rope) vs the CPU oracle, through the C ABI (needs a
GB300).  The cases span several 32-token sub-tiles and splits, ragged
tails, flushes, a wrapped InnerQ window, two key groups per sub-tile
(G = 16), 4-bit codes with separate key statistics (G = 64), grouped-query
heads, the key normalization, and the degenerate cache states.
"""
import math

import numpy as np
import pytest
import torch

from bit_kv_cache_14_gb300 import kvq, synth
from parity_util import ATOL, new_cache, run_workload

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
S = synth.scaled
BASE = 10000.0


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


CASES = {
    "llama_small": S(W["llama2_7b_2bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=1000,
                     n_append=140),
    "kivi4_g64": S(W["kivi_4bit"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=777, n_append=130),
    "gqa_rg4": S(W["gqa_2bit"], batch=1, n_q_heads=8, n_kv_heads=2, ctx=1500, n_append=40),
    "kivi_d64_g16": S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2, head_dim=64,
                      ctx=600, k_group=16, v_group=16, residual=48, n_append=60),
    "innerq_wrap": S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=3000, n_append=45),
    "innerq_knorm_rg2": S(W["innerq_1m"], batch=1, n_q_heads=4, n_kv_heads=2, ctx=900,
                          n_append=40, k_norm=True),
    "innerq_d64_g16_2bit": S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, head_dim=64,
                             bits=2, k_group=16, v_group=32, ctx=500, n_sink=3, residual=8,
                             n_append=20),
    # degenerate states: nothing quantized; empty prompt; prompt shorter than the sinks
    "kivi_short_prompt": S(W["llama2_7b_2bit"], batch=1, n_q_heads=1, n_kv_heads=1, ctx=100,
                           n_append=10),
    "kivi_empty_prompt": S(W["llama2_7b_2bit"], batch=1, n_q_heads=1, n_kv_heads=1, ctx=0,
                           n_append=130),
    "innerq_prompt_lt_sink": S(W["innerq_1m"], batch=1, n_q_heads=1, n_kv_heads=1, ctx=2,
                               n_append=40),
}

# the tensor-core form: every instantiation (bits x value groups x key
# statistics inside the block (G 32) or beside it (G 64)), ragged residuals,
# flushes between the decodes
TC_CASES = {}
for _bits in (2, 4):
    for _ngv in (2, 4):
        for _g in (32, 64):
            TC_CASES["tc_b%d_ngv%d_g%d" % (_bits, _ngv, _g)] = S(
                W["llama2_7b_2bit"] if _bits == 2 else W["kivi_4bit"], batch=2, n_q_heads=2,
                n_kv_heads=2, ctx=700, k_group=_g, v_group=128 // _ngv, residual=64,
                n_append=74)
CASES.update(TC_CASES)


@pytest.mark.parametrize("name", sorted(CASES))
def test_rope_small_workload_all_heads(name):
    w = CASES[name]
    worst = run_workload(w, decode_every=max(1, w.n_append // 3), rope_base=BASE)
    assert worst <= ATOL


def test_rope_empty_cache_decodes_to_zero():
    w = S(W["tiny"], ctx=0)
    cache = new_cache(w, 64)
    cache.prefill(torch.zeros(1, 1, 0, 64, dtype=torch.float16, device="cuda"),
                  torch.zeros(1, 1, 0, 64, dtype=torch.float16, device="cuda"))
    out = cache.decode_rope(torch.from_numpy(synth.queries(w)).cuda(), BASE)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0


def test_rope_grid_exact_equals_rotated_sdpa():
    """Lossless keys and values: the kernel equals plain fp64 attention over
    keys and query rotated explicitly (complex form of the embedding, on the
    CPU), independent of the oracle."""
    rng = np.random.default_rng(6)
    B, H, T, d, G = 1, 2, 700, 128, 32
    K = np.empty((B, H, T, d), np.float64)
    V = np.empty((B, H, T, d), np.float64)
    for b in range(B):
        for h in range(H):
            for g in range(T // G):
                for c in range(d):
                    u = rng.integers(0, 4, G)
                    u[0], u[1] = 0, 3
                    K[b, h, g * G:(g + 1) * G, c] = float(rng.integers(-8, 8)) / 4 + u / 4.0
            K[b, h, T // G * G:] = rng.standard_normal((T % G, d)).astype(np.float16)
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
    out = cache.decode_rope(torch.from_numpy(q).cuda(), BASE).cpu().double()
    theta = BASE ** (-2.0 * np.arange(d // 2) / d)
    rot_k = np.exp(1j * np.outer(np.arange(T), theta))          # [T][d/2]
    rot_q = np.exp(1j * (T - 1) * theta)
    zk = (K[..., 0::2] + 1j * K[..., 1::2]) * rot_k
    zq = (q.astype(np.float64)[..., 0::2] + 1j * q.astype(np.float64)[..., 1::2]) * rot_q
    kr = np.empty_like(K)
    kr[..., 0::2], kr[..., 1::2] = zk.real, zk.imag
    qr = np.empty(q.shape)
    qr[..., 0::2], qr[..., 1::2] = zq.real, zq.imag
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qr)[:, :, None, :], torch.from_numpy(kr), torch.from_numpy(V),
        scale=1 / math.sqrt(d))[:, :, 0, :]
    assert (out - ref).abs().max().item() <= ATOL


def test_rope_rejects_bad_base_and_unsupported_groups():
    w = S(W["tiny"], ctx=64)
    cache = new_cache(w, 64)
    q = torch.from_numpy(synth.queries(w)).cuda()
    for base in (0.0, -1.0, float("inf"), float("nan")):
        with pytest.raises(kvq.KVQError) as e:
            cache.decode_rope(q, base)
        assert e.value.code == kvq.KVQ_EINVAL
    w8 = S(W["gqa_2bit"], batch=1, n_q_heads=8, n_kv_heads=1, ctx=64, n_append=0)
    c8 = new_cache(w8, 64)
    with pytest.raises(kvq.KVQError) as e:
        c8.decode_rope(torch.from_numpy(synth.queries(w8)).cuda(), BASE)
    assert e.value.code == kvq.KVQ_EUNSUPPORTED


@pytest.mark.slow
def test_rope_full_size_llama_sampled():
    """The Llama-2-7B-shaped layer at full size (the benchmark's launch), three
    sampled heads, at the first step and after a flush."""
    w = W["llama2_7b_2bit"]
    heads = [(0, 0), (w.batch // 2, w.n_kv_heads // 2), (w.batch - 1, w.n_kv_heads - 1)]
    run_workload(w, heads=heads, n_append=130, decode_every=None, check_steps=[1, 130],
                 rope_base=BASE)
