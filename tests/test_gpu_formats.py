"""Cache-format options on the device against the CPU oracle: scales and zero
points stored in fp16, KIVI's value queue, dense-and-sparse outliers (each
token's largest elements kept in fp16), and per-sequence prompt lengths --
alone and combined, on every decode path they reach.

Codes, statistics, outlier lists, fp16 rows and mode bits are compared bit
for bit; attention within ATOL of the oracle's fp64 result.  One case with
lossless data (grid inliers, loud outliers restored exactly) is compared with
torch's fp64 attention on the raw tokens, independently of the oracle.
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

LLAMA = dict(batch=2, n_q_heads=2, n_kv_heads=2, ctx=700, residual=64, n_append=80)

CASES = {
    # scales and zeros in fp16
    "f16_kivi2_g32": S(W["llama2_7b_2bit"], meta_f16=True, **LLAMA),
    "f16_kivi2_g16_ngv2": S(W["llama2_7b_2bit"], k_group=16, v_group=64, meta_f16=True, **LLAMA),
    "f16_kivi4_g64": S(W["kivi_4bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=777,
                       n_append=140, meta_f16=True),
    "f16_kivi2_d64_g16": S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2, head_dim=64,
                           ctx=600, k_group=16, v_group=16, residual=48, n_append=60,
                           meta_f16=True),
    "f16_innerq4": S(W["innerq_1m"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=700, n_append=40,
                     meta_f16=True),
    "f16_innerq2_g32": S(W["innerq_1m"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=700, bits=2,
                         k_group=32, v_group=32, n_append=40, meta_f16=True),
    "f16_innerq_knorm_gqa": S(W["innerq_1m"], batch=1, n_q_heads=8, n_kv_heads=2, ctx=600,
                              n_append=40, k_norm=True, meta_f16=True),
    "f16_gqa": S(W["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=2, ctx=900, n_append=140,
                 meta_f16=True),
    # the value queue
    "vq_kivi2": S(W["llama2_7b_2bit"], v_queue=True, **LLAMA),
    "vq_kivi4_g64": S(W["kivi_4bit"], batch=2, n_q_heads=2, n_kv_heads=2, ctx=777,
                      n_append=140, v_queue=True),
    "vq_gqa_d64": S(W["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=2, head_dim=64, ctx=500,
                    residual=32, n_append=70, v_queue=True),
    # dense-and-sparse outliers (1 % of 128 channels rounded up = 2)
    "out2_kivi2": S(W["llama2_7b_2bit"], outliers=2, **LLAMA),
    "out1_kivi2_d64_g16": S(W["llama2_7b_2bit"], batch=1, n_q_heads=2, n_kv_heads=2,
                            head_dim=64, ctx=600, k_group=16, v_group=16, residual=48,
                            n_append=60, outliers=1),
    "out8_kivi4_g128": S(W["kivi_4bit"], batch=1, n_q_heads=2, n_kv_heads=2, ctx=700,
                         k_group=128, v_group=32, residual=128, n_append=140, outliers=8),
    "out2_gqa": S(W["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=2, ctx=900, n_append=140,
                  outliers=2),
    # combined
    "out2_vq_f16": S(W["llama2_7b_2bit"], outliers=2, v_queue=True, meta_f16=True, **LLAMA),
    # per-sequence prompt lengths (one sequence empty, one shorter than R)
    "ragged_kivi2": S(W["llama2_7b_2bit"], batch=5, n_q_heads=2, n_kv_heads=2, ctx=700,
                      residual=64, n_append=80, ragged=True),
    "ragged_innerq4": S(W["innerq_1m"], batch=5, n_q_heads=2, n_kv_heads=2, ctx=700,
                        n_append=40, ragged=True),
    "ragged_innerq_knorm_d64": S(W["innerq_1m"], batch=4, n_q_heads=2, n_kv_heads=2,
                                 head_dim=64, bits=2, k_group=16, v_group=32, n_sink=3,
                                 residual=8, ctx=300, n_append=20, k_norm=True, ragged=True),
    "ragged_gqa_all_options": S(W["gqa_2bit"], batch=4, n_q_heads=8, n_kv_heads=2, ctx=900,
                                n_append=140, ragged=True, v_queue=True, meta_f16=True,
                                outliers=2),
}


@pytest.fixture(autouse=True, scope="module")
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield


@pytest.mark.parametrize("name", sorted(CASES))
def test_format_matches_oracle(name):
    w = CASES[name]
    worst = run_workload(w, decode_every=max(1, w.n_append // 4))
    assert worst <= ATOL


@pytest.mark.parametrize("T", [0, 1, 15, 16, 17, 31, 32, 48])
def test_value_queue_cadence(T):
    """Prompts of 0 .. 48 tokens, then 40 appends with R = 16: the queue's
    contents, the quantized values and attention after every step."""
    w = S(W["llama2_7b_2bit"], batch=1, n_q_heads=1, n_kv_heads=1, head_dim=64, ctx=T,
          k_group=16, v_group=32, residual=16, n_append=40, v_queue=True)
    run_workload(w, decode_every=1)


def _lossless_outlier_tokens(rng, T, d, G, Gv, top=3):
    """Keys and values (fp64, exactly fp16) whose inliers lie on a grid that
    every group still spans after its outliers are removed, with one loud key
    outlier and one loud value outlier per token: quantization with one
    outlier per token loses nothing."""
    K = np.empty((T, d))
    V = np.empty((T, d))
    kout = np.empty(T, int)
    for g in range(T // G):
        while True:  # each channel keeps at least two inliers in the group
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
    assert np.array_equal(K.astype(np.float16).astype(np.float64), K)
    assert np.array_equal(V.astype(np.float16).astype(np.float64), V)
    return K, V


@pytest.mark.parametrize("v_queue,meta_f16", [(False, False), (True, False), (False, True),
                                              (True, True)])
def test_lossless_outliers_equal_sdpa(v_queue, meta_f16):
    rng = np.random.default_rng(7)
    B, H, d, G, Gv, R = 1, 2, 128, 32, 32, 64
    T0, n_app = 600, 100
    KV = [_lossless_outlier_tokens(rng, T0 + n_app + 4, d, G, Gv) for _ in range(B * H)]
    K = np.stack([k for k, _ in KV]).reshape(B, H, -1, d)
    V = np.stack([v for _, v in KV]).reshape(B, H, -1, d)
    w = S(W["llama2_7b_2bit"], batch=B, n_q_heads=H, n_kv_heads=H, ctx=T0, k_group=G,
          v_group=Gv, residual=R, n_append=n_app, outliers=1, v_queue=v_queue,
          meta_f16=meta_f16)
    cache = new_cache(w, T0 + n_app)
    cache.prefill(torch.from_numpy(K[:, :, :T0].astype(np.float16)).cuda(),
                  torch.from_numpy(V[:, :, :T0].astype(np.float16)).cuda())
    for i in range(T0, T0 + n_app):
        cache.append(torch.from_numpy(K[:, :, i].astype(np.float16)).cuda(),
                     torch.from_numpy(V[:, :, i].astype(np.float16)).cuda())
    n = T0 + n_app
    q = (rng.standard_normal((B, H, d)) / 16).astype(np.float16)
    out = cache.decode(torch.from_numpy(q).cuda()).cpu().double()
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[:, :, None, :], torch.from_numpy(K[:, :, :n]),
        torch.from_numpy(V[:, :, :n]), scale=1 / math.sqrt(d))[:, :, 0, :]
    assert (out - ref).abs().max().item() <= ATOL
    assert cache.device_status() == 0


def test_ragged_sequences_match_their_uniform_caches():
    """Each sequence of a ragged batch attends like a uniform cache holding
    only that sequence: the same kernel (head_dim 64 runs the general one for
    both), so the outputs differ only by the fp32 summation order of the two
    launches' token splits."""
    w = S(W["llama2_7b_2bit"], batch=4, n_q_heads=2, n_kv_heads=2, head_dim=64, ctx=500,
          residual=64, n_append=70, ragged=True)
    lens = synth.prompt_lengths(w)
    K, V = synth.prompt(w)
    Ks, Vs = synth.streamed(w)
    rag = new_cache(w)
    rag.prefill_ragged(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda(), lens)
    singles = []
    for b in range(w.batch):
        wb = S(w, batch=1, ragged=False)
        c = new_cache(wb, w.ctx + w.n_append)
        c.prefill(torch.from_numpy(np.ascontiguousarray(K[b:b + 1, :, :lens[b]])).cuda(),
                  torch.from_numpy(np.ascontiguousarray(V[b:b + 1, :, :lens[b]])).cuda())
        singles.append(c)
    for s in range(w.n_append):
        rag.append(torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda())
        for b, c in enumerate(singles):
            c.append(torch.from_numpy(np.ascontiguousarray(Ks[s, b:b + 1])).cuda(),
                     torch.from_numpy(np.ascontiguousarray(Vs[s, b:b + 1])).cuda())
        if s % 23 == 0 or s == w.n_append - 1:
            q = synth.queries(w, s)
            got = rag.decode(torch.from_numpy(q).cuda()).cpu()
            for b, c in enumerate(singles):
                one = c.decode(torch.from_numpy(np.ascontiguousarray(q[b:b + 1])).cuda()).cpu()
                assert (got[b:b + 1] - one).abs().max().item() <= 1e-4, (s, b)
    assert rag.seq_lengths() == [int(x) + w.n_append for x in lens]
    assert rag.device_status() == 0


@pytest.mark.slow
@pytest.mark.parametrize("opts", [dict(meta_f16=True), dict(outliers=2),
                                  dict(v_queue=True), dict(ragged=True)])
def test_full_size_llama_layer_options(opts):
    """The Llama-2-7B-shaped layer at full size with each option, sampled heads."""
    w = S(W["llama2_7b_2bit"], **opts)
    heads = [(0, 0), (w.batch - 1, w.n_kv_heads - 1), (w.batch // 2, w.n_kv_heads // 2)]
    run_workload(w, heads=heads, n_append=w.n_append, decode_every=None,
                 check_steps=[1, w.n_append])
    assert kvq.decode_kernel_name(kvq.config_of(w), 4096)
