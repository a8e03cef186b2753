"""kvq_decode_attention_noalloc: decode attention for callers that cannot give
the library a scratch buffer (no device allocator reachable from where they
run).  Its scratch is a fixed device array inside the library; the same kernel
then runs on the same inputs as the regular entry point, so the two outputs
must be identical bit for bit.

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It passes alone in a fresh process too.
"""
import ctypes
import math

import pytest
import torch

from bit_kv_cache_14_gb300 import build_lib, kvq, synth
from parity_util import new_cache

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
S = synth.scaled


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build_lib.build()
    yield


CASES = {
    # head_dim 128 MHA: the tensor-core decode kernel
    "tensor_core": S(W["llama2_7b_2bit"], batch=2, n_q_heads=4, n_kv_heads=4, ctx=900,
                     n_append=5),
    # 2-bit KIVI, 4 query heads per KV head: the grouped-query tensor-core kernel
    "grouped_query": S(W["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=2, ctx=700, n_append=5),
    # head_dim 64: the general (CUDA-core) decode kernel
    "general": S(W["llama2_7b_2bit"], batch=2, n_q_heads=2, n_kv_heads=2, head_dim=64, ctx=600,
                 n_append=5),
}

KERNEL_PREFIX = {"tensor_core": "tc_decode_kernel", "grouped_query": "tc_gqa_kernel",
                 "general": "decode_kernel"}


def _noalloc(cache, q, out, scale):
    return kvq.lib().kvq_decode_attention_noalloc(
        ctypes.byref(cache.cfg), ctypes.byref(cache.view), q.data_ptr(), out.data_ptr(),
        ctypes.c_float(scale), torch.cuda.current_stream().cuda_stream)


def _filled_cache(w):
    K, V = synth.prompt(w)
    cache = new_cache(w)
    cache.prefill(torch.from_numpy(K).cuda(), torch.from_numpy(V).cuda())
    Ks, Vs = synth.streamed(w)
    for s in range(w.n_append):
        cache.append(torch.from_numpy(Ks[s]).cuda(), torch.from_numpy(Vs[s]).cuda())
    return cache


@pytest.mark.parametrize("name", sorted(CASES))
def test_noalloc_matches_regular_decode_twice(name):
    w = CASES[name]
    cache = _filled_cache(w)
    assert kvq.decode_kernel_name(cache.cfg, cache.n_quant).startswith(KERNEL_PREFIX[name] + "<")
    scale = 1.0 / math.sqrt(w.head_dim)
    qs = [torch.from_numpy(synth.queries(w, s)).cuda() for s in (0, 1)]
    outs = [torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda") for q in qs]
    # two allocation-free calls in a row, then the regular entry point
    for q, out in zip(qs, outs):
        assert _noalloc(cache, q, out, scale) == kvq.KVQ_OK
    torch.cuda.synchronize()
    assert cache.device_status() == kvq.KVQ_OK
    for q, out in zip(qs, outs):
        ref = cache.decode(q, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert cache.device_status() == kvq.KVQ_OK


def test_noalloc_recovers_after_a_call_that_stopped_early():
    """A decode that gave up (bounded wait, KVQ_ETIMEOUT) leaves the shared
    array in an unknown state; the next call clears what it uses and is exact."""
    w = CASES["tensor_core"]
    cache = _filled_cache(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    q = torch.from_numpy(synth.queries(w, 0)).cuda()
    ref = cache.decode(q, scale=scale)
    assert cache.device_status() == kvq.KVQ_OK
    out = torch.empty_like(ref)
    try:
        kvq.debug_stall_waits(1000)
        assert _noalloc(cache, q, out, scale) == kvq.KVQ_OK
        assert cache.device_status() == kvq.KVQ_ETIMEOUT
    finally:
        kvq.debug_stall_waits(0)
    out.fill_(float("nan"))
    assert _noalloc(cache, q, out, scale) == kvq.KVQ_OK
    assert cache.device_status() == kvq.KVQ_OK
    assert torch.equal(out, ref)


def test_noalloc_rejects_configurations_beyond_its_scratch():
    w = W["kivi_4bit"]                 # its decode workspace is larger than 16 MiB
    cfg = kvq.config_of(w)
    assert kvq.workspace_bytes(cfg) > (16 << 20)
    view = kvq.Cache()
    q = torch.zeros(8, dtype=torch.float16, device="cuda")
    out = torch.zeros(8, dtype=torch.float32, device="cuda")
    rc = kvq.lib().kvq_decode_attention_noalloc(ctypes.byref(cfg), ctypes.byref(view),
                                                q.data_ptr(), out.data_ptr(),
                                                ctypes.c_float(1.0), None)
    assert rc == kvq.KVQ_ECAPACITY


def test_noalloc_rejects_what_the_regular_decode_rejects():
    """A call the regular decode would reject (here: a misaligned output) is
    rejected the same way, and the next call is exact."""
    w = CASES["tensor_core"]
    cache = _filled_cache(w)
    scale = 1.0 / math.sqrt(w.head_dim)
    q = torch.from_numpy(synth.queries(w, 0)).cuda()
    big = torch.zeros(q.numel() + 4, dtype=torch.float32, device="cuda")
    rc = kvq.lib().kvq_decode_attention_noalloc(
        ctypes.byref(cache.cfg), ctypes.byref(cache.view), q.data_ptr(), big.data_ptr() + 4,
        ctypes.c_float(scale), torch.cuda.current_stream().cuda_stream)
    assert rc == kvq.KVQ_EALIGN
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    assert _noalloc(cache, q, out, scale) == kvq.KVQ_OK
    assert torch.equal(out, cache.decode(q, scale=scale))
