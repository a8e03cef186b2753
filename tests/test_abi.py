"""The C-ABI library builds, loads without a GPU, exports every entry point
that include/kvq.h declares, and its host-side logic (sizes, validation,
error strings) behaves as documented.  No compute call is made here."""
import ctypes
import os
import re

import pytest

from bit_kv_cache_14_gb300 import build_lib, kvq, synth

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "kvq.h")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib.build()
    yield


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_\w+)\s*\(", src)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 9
    L = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert sorted(kvq.EXPORTS) == names


def _cfg(**kw):
    base = dict(batch=8, n_q_heads=32, n_kv_heads=32, head_dim=128, bits=2, scheme=kvq.KIVI,
                k_group=32, v_group=32, residual=128, n_sink=0, max_ctx=4352)
    base.update(kw)
    return kvq.make_config(**base)


def test_sizes_follow_layout():
    s = kvq.cache_sizes(_cfg(max_ctx=4300))
    BH, T, d = 8 * 32, 4352, 128      # per-head capacity: 4300 rounded up to 128
    # a 32-token block: K codes, V codes (32 B a row), V scale, V zero (4 groups),
    # then the scale and zero rows of its one 32-token key group
    assert s.blocks == BH * (T // 32) * (2 * 32 * 32 + 2 * 32 * 4 * 4 + 2 * d * 4)
    assert s.k_meta == 0
    s64 = kvq.cache_sizes(_cfg(max_ctx=4300, k_group=64))
    assert s64.blocks == BH * (T // 32) * (2 * 32 * 32 + 2 * 32 * 4 * 4)
    assert s64.k_meta == BH * (T // 64) * 2 * d * 4 + 64
    assert s.k_res == BH * 128 * d * 2
    assert s.k_mode == 0 and s.k_sink == 0
    si = kvq.cache_sizes(_cfg(scheme=kvq.INNERQ, bits=4, k_group=64, v_group=64, residual=32,
                              n_sink=4, batch=1, max_ctx=1 << 20))
    # 4-bit rows of 64 B; two value groups and two key groups per token
    assert si.blocks == 32 * ((1 << 20) // 32) * (2 * 32 * 64 + 4 * 32 * 2 * 4)
    assert si.k_meta == 0
    assert si.k_mode == 32 * ((1 << 20) * 2 // 32) * 4
    assert si.k_sink == 32 * 4 * 128 * 2
    # the key normalization adds the fp32 factors [B][H][d] after the blocks
    sn = kvq.cache_sizes(_cfg(scheme=kvq.INNERQ_KNORM, bits=4, k_group=64, v_group=64,
                              residual=32, n_sink=4, batch=1, max_ctx=1 << 20))
    assert sn.blocks == si.blocks + 32 * 128 * 4
    assert (sn.k_mode, sn.v_mode, sn.k_res, sn.k_sink) == (si.k_mode, si.v_mode, si.k_res, si.k_sink)


def test_per_token_bytes_match_llama2_table():
    # codes of one token, all 32 layers x 32 heads, keys and values
    for bits, expect in ((2, 65536), (4, 131072)):
        s = kvq.cache_sizes(_cfg(bits=bits, batch=1, max_ctx=128, v_group=128))
        meta = 32 * (128 * 2 * 4 + 4 * 2 * 128 * 4)  # 32 heads: value + key statistics
        assert 32 * (s.blocks - meta) // 128 == expect


def test_workspace_bytes():
    n = kvq.workspace_bytes(_cfg())
    assert n > 8 * 32 * 3 * 130 * 4


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), kvq.KVQ_EUNSUPPORTED),
    (dict(bits=3), kvq.KVQ_EUNSUPPORTED),
    (dict(residual=100), kvq.KVQ_EINVAL),
    (dict(n_q_heads=30), kvq.KVQ_EINVAL),
    (dict(n_q_heads=96), kvq.KVQ_EUNSUPPORTED),
    (dict(n_sink=4), kvq.KVQ_EINVAL),
    (dict(v_group=24), kvq.KVQ_EUNSUPPORTED),
    (dict(batch=0), kvq.KVQ_EINVAL),
    (dict(max_ctx=0), kvq.KVQ_EINVAL),
    (dict(scheme=7), kvq.KVQ_EINVAL),
    (dict(scheme=kvq.INNERQ, k_group=48), kvq.KVQ_EUNSUPPORTED),
    (dict(scheme=kvq.INNERQ_KNORM, k_group=48), kvq.KVQ_EUNSUPPORTED),
    (dict(scheme=3), kvq.KVQ_EINVAL),
    (dict(max_ctx=(1 << 30) + 1), kvq.KVQ_EUNSUPPORTED),
    (dict(max_ctx=1 << 62), kvq.KVQ_EUNSUPPORTED),
])
def test_config_validation(kw, code):
    with pytest.raises(kvq.KVQError) as e:
        kvq.cache_sizes(_cfg(**kw))
    assert e.value.code == code


def test_calls_validate_before_touching_the_device():
    L = kvq.lib()
    cfg = _cfg()
    empty = kvq.Cache()
    assert L.kvq_quantize_prefill(ctypes.byref(cfg), ctypes.byref(empty), None, None, 0,
                                  None) == kvq.KVQ_EINVAL
    assert L.kvq_append(ctypes.byref(cfg), None, None, None, None) == kvq.KVQ_EINVAL
    assert L.kvq_decode_attention(ctypes.byref(cfg), ctypes.byref(empty), None, None, 1.0, None,
                                  0, None) == kvq.KVQ_EINVAL
    bad = _cfg(head_dim=80)
    assert L.kvq_append(ctypes.byref(bad), ctypes.byref(empty), None, None,
                        None) == kvq.KVQ_EUNSUPPORTED
    # misaligned cache buffer pointers are rejected before any launch
    c = kvq.Cache()
    for name in ("blocks", "k_meta", "k_res", "v_res"):
        setattr(c, name, 0x1000)
    c.blocks = 0x1001
    assert L.kvq_quantize_prefill(ctypes.byref(cfg), ctypes.byref(c), None, None, 0,
                                  None) == kvq.KVQ_EALIGN
    c.blocks = 0x1000
    c.k_meta = None          # needed only for key groups longer than a block
    cfg64 = _cfg(k_group=64)
    assert L.kvq_quantize_prefill(ctypes.byref(cfg64), ctypes.byref(c), None, None, 0,
                                  None) == kvq.KVQ_EINVAL
    assert L.kvq_quantize_prefill(ctypes.byref(cfg), ctypes.byref(c), ctypes.c_void_p(0x2000),
                                  ctypes.c_void_p(0x2000), 5000, None) == kvq.KVQ_ECAPACITY
    assert L.kvq_decode_attention(ctypes.byref(cfg), ctypes.byref(c), ctypes.c_void_p(0x2000),
                                  ctypes.c_void_p(0x3000), 1.0, ctypes.c_void_p(0x4000), 16,
                                  None) == kvq.KVQ_ECAPACITY


def test_noalloc_decode_rejects_oversized_configs_on_the_host():
    L = kvq.lib()
    big = kvq.config_of(synth.WORKLOADS["kivi_4bit"])
    assert kvq.workspace_bytes(big) > (16 << 20)
    c = kvq.Cache()
    assert L.kvq_decode_attention_noalloc(ctypes.byref(big), ctypes.byref(c),
                                          ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000),
                                          1.0, None) == kvq.KVQ_ECAPACITY


def test_strerror():
    assert kvq.strerror(0) == "ok"
    assert "capacity" in kvq.strerror(kvq.KVQ_ECAPACITY)
    assert kvq.strerror(12345) == "unknown error"


def test_workload_configs_are_accepted():
    for w in synth.WORKLOADS.values():
        kvq.cache_sizes(kvq.config_of(w))


def test_rope_decode_validates_before_touching_the_device():
    """kvq_decode_attention_rope: the decode's checks, then the base (finite,
    > 0) and the supported shapes (1, 2 or 4 query heads per KV head;
    max_ctx <= 2^24 so positions are exact in fp32), all on the host."""
    L = kvq.lib()
    cfg = _cfg()
    c = kvq.Cache()
    c.blocks, c.k_res, c.v_res = 0x1000, 0x1000, 0x1000
    q, out = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    ws, ws_n = ctypes.c_void_p(0x4000), kvq.workspace_bytes(cfg)

    def call(cfg_, base, n=ws_n):
        return L.kvq_decode_attention_rope(ctypes.byref(cfg_), ctypes.byref(c), q, out, 1.0,
                                           base, ws, n, None)

    assert L.kvq_decode_attention_rope(ctypes.byref(cfg), ctypes.byref(kvq.Cache()), q, out, 1.0,
                                       10000.0, ws, ws_n, None) == kvq.KVQ_EINVAL
    assert call(cfg, 10000.0, 16) == kvq.KVQ_ECAPACITY
    for base in (0.0, -2.0, float("inf"), float("nan")):
        assert call(cfg, base) == kvq.KVQ_EINVAL, base
    rg8 = _cfg(n_q_heads=32, n_kv_heads=4)
    assert call(rg8, 10000.0, kvq.workspace_bytes(rg8)) == kvq.KVQ_EUNSUPPORTED
    long_ctx = _cfg(batch=1, n_q_heads=1, n_kv_heads=1, max_ctx=(1 << 24) + 1)
    assert call(long_ctx, 10000.0, kvq.workspace_bytes(long_ctx)) == kvq.KVQ_EUNSUPPORTED
    bad = kvq.Cache()
    bad.blocks, bad.k_res, bad.v_res = 0x1001, 0x1000, 0x1000
    assert L.kvq_decode_attention_rope(ctypes.byref(cfg), ctypes.byref(bad), q, out, 1.0,
                                       10000.0, ws, ws_n, None) == kvq.KVQ_EALIGN


def test_binding_rejects_bad_tensors_before_any_call():
    """The binding checks dtype and layout itself (not with asserts, which
    python -O strips): a wrong dtype or a non-contiguous tensor raises
    before the library sees a pointer."""
    import torch
    with pytest.raises(ValueError):
        kvq._ptr(torch.zeros(4, 4).t())
    with pytest.raises(TypeError):
        kvq._need_f16(torch.zeros(2, dtype=torch.float32))
    kvq._need_f16(torch.zeros(2, dtype=torch.float16))
    assert kvq._ptr(torch.zeros(3)) != 0


def test_binding_block_layout_matches_the_library():
    """The binding's mirror of the block layout (used to read codes and
    statistics back) gives the same block size as kvq_cache_sizes, for every
    supported bits / scheme / group combination and cache-format option."""
    cases = []
    for bits in (2, 4):
        for d in (64, 128):
            for gv in (16, 32, 64, 128):
                if d % gv:
                    continue
                for G in (16, 32, 64, 128):
                    for flags in (0, kvq.META_F16, kvq.VALUE_QUEUE | kvq.RAGGED):
                        for o in (0, 1, 8):
                            cases.append(dict(head_dim=d, bits=bits, v_group=gv, k_group=G,
                                              residual=G * 2, scheme=kvq.KIVI, flags=flags,
                                              outliers=o))
                for gk in (16, 32, 64, 128):
                    if d % gk == 0:
                        for sch in (kvq.INNERQ, kvq.INNERQ_KNORM):
                            for flags in (0, kvq.META_F16 | kvq.RAGGED):
                                cases.append(dict(head_dim=d, bits=bits, v_group=gv, k_group=gk,
                                                  residual=8, n_sink=2, scheme=sch, flags=flags))
    for kw in cases:
        cfg = _cfg(batch=2, n_q_heads=3, n_kv_heads=3, max_ctx=300, **kw)
        s = kvq.cache_sizes(cfg)
        view = kvq.QuantizedKVCache.__new__(kvq.QuantizedKVCache)
        view.cfg = cfg
        off, bb, rb, ngv, ngk = view._block_layout()
        BH, cap = 6, 384
        extra = BH * cfg.head_dim * 4 if cfg.scheme == kvq.INNERQ_KNORM else 0
        assert s.blocks == BH * (cap // 32) * bb + extra, kw
        assert rb == cfg.head_dim * cfg.bits // 8 and bb % 128 == 0, kw
        assert s.seq_prompt == (2 * 4 if cfg.flags & kvq.RAGGED else 0), kw
        m = 2 if cfg.flags & kvq.META_F16 else 4
        if cfg.scheme == kvq.KIVI and cfg.k_group > 32:
            assert s.k_meta == BH * (cap // cfg.k_group) * 2 * cfg.head_dim * m + 64, kw


def test_format_options_sizes_and_refusals():
    """fp16 statistics cut the Llama-2-7B layer's 2-bit tokens from 128 to 96
    bytes per token-head (codes 64 + statistics 32); outlier lists add 8 bytes
    per outlier (key and value word); options outside their scheme, unknown
    flag bits and more than 8 outliers are refused; the pre-RoPE decode
    refuses every option."""
    per_tok = lambda s: s.blocks / (8 * 32 * 4352)  # noqa: E731
    assert per_tok(kvq.cache_sizes(_cfg(max_ctx=4300))) == 128
    assert per_tok(kvq.cache_sizes(_cfg(max_ctx=4300, flags=kvq.META_F16))) == 96
    assert per_tok(kvq.cache_sizes(_cfg(max_ctx=4300, outliers=2))) == 128 + 16
    for kw in (dict(flags=8), dict(outliers=9), dict(outliers=-1),
               dict(scheme=kvq.INNERQ, k_group=64, residual=32, n_sink=4, outliers=1),
               dict(scheme=kvq.INNERQ, k_group=64, residual=32, n_sink=4,
                    flags=kvq.VALUE_QUEUE)):
        with pytest.raises(kvq.KVQError) as e:
            kvq.cache_sizes(_cfg(**kw))
        assert e.value.code == kvq.KVQ_EINVAL, kw
    # the workload fields map onto the options
    base = synth.scaled(synth.WORKLOADS["tiny"])
    cfg = kvq.config_of(synth.scaled(base, v_queue=True, meta_f16=True, outliers=1, ragged=True))
    assert cfg.flags == kvq.META_F16 | kvq.VALUE_QUEUE | kvq.RAGGED and cfg.outliers == 1
    L = kvq.lib()
    c = kvq.Cache()
    for name in ("blocks", "k_meta", "k_res", "v_res"):
        setattr(c, name, 0x1000)
    for kw in (dict(flags=kvq.META_F16), dict(outliers=1)):
        cfg = _cfg(**kw)
        assert L.kvq_decode_attention_rope(ctypes.byref(cfg), ctypes.byref(c),
                                           ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000), 1.0,
                                           10000.0, ctypes.c_void_p(0x4000), 1 << 40,
                                           None) == kvq.KVQ_EUNSUPPORTED


def test_ragged_prefill_validates_on_the_host():
    """The ragged prefill needs the option, a seq_prompt buffer and lengths in
    [0, T_max]; each is checked before anything is enqueued."""
    L = kvq.lib()
    c = kvq.Cache()
    for name in ("blocks", "k_meta", "k_res", "v_res"):
        setattr(c, name, 0x1000)
    lens = (ctypes.c_int32 * 8)(*([100] * 8))
    K = ctypes.c_void_p(0x2000)
    plain = _cfg()
    assert L.kvq_quantize_prefill_ragged(ctypes.byref(plain), ctypes.byref(c), K, K, 100, lens,
                                         None) == kvq.KVQ_EINVAL
    rag = _cfg(flags=kvq.RAGGED)
    assert L.kvq_quantize_prefill_ragged(ctypes.byref(rag), ctypes.byref(c), K, K, 100, lens,
                                         None) == kvq.KVQ_EINVAL   # no seq_prompt buffer
    c.seq_prompt = 0x1000
    assert L.kvq_quantize_prefill_ragged(ctypes.byref(rag), ctypes.byref(c), K, K, 100, None,
                                         None) == kvq.KVQ_EINVAL
    bad = (ctypes.c_int32 * 8)(*([100] * 7 + [101]))
    assert L.kvq_quantize_prefill_ragged(ctypes.byref(rag), ctypes.byref(c), K, K, 100, bad,
                                         None) == kvq.KVQ_EINVAL
    neg = (ctypes.c_int32 * 8)(*([100] * 7 + [-1]))
    assert L.kvq_quantize_prefill_ragged(ctypes.byref(rag), ctypes.byref(c), K, K, 100, neg,
                                         None) == kvq.KVQ_EINVAL
    assert L.kvq_quantize_prefill_ragged(ctypes.byref(rag), ctypes.byref(c), K, K, 5000, lens,
                                         None) == kvq.KVQ_ECAPACITY


def test_corrupted_counters_are_rejected_before_any_launch():
    """Counters that no sequence of calls can produce (too many sinks or
    residual tokens, a quantized count off the flush grid or past the
    capacity, a ring head past the window) make every call but prefill return
    KVQ_EINVAL instead of steering a kernel past the buffers."""
    L = kvq.lib()
    q, out = ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    ws = ctypes.c_void_p(0x4000)
    kivi = _cfg()
    innerq = _cfg(scheme=kvq.INNERQ, bits=4, k_group=64, v_group=64, residual=32, n_sink=4)
    for cfg, bad in ((kivi, dict(n_resid=128)), (kivi, dict(n_quant=100)),
                     (kivi, dict(n_quant=4352 + 128)), (kivi, dict(n_quant=4352, n_resid=1)),
                     (innerq, dict(n_sink=5)), (innerq, dict(n_resid=33)),
                     (innerq, dict(ring_head=32))):
        c = kvq.Cache()
        for name in ("blocks", "k_meta", "k_mode", "v_mode", "k_res", "v_res", "k_sink",
                     "v_sink"):
            setattr(c, name, 0x1000)
        for k, v in bad.items():
            setattr(c, k, v)
        n = kvq.workspace_bytes(cfg)
        assert L.kvq_decode_attention(ctypes.byref(cfg), ctypes.byref(c), q, out, 1.0, ws, n,
                                      None) == kvq.KVQ_EINVAL, bad
        assert L.kvq_decode_attention_rope(ctypes.byref(cfg), ctypes.byref(c), q, out, 1.0,
                                           10000.0, ws, n, None) == kvq.KVQ_EINVAL, bad
        assert L.kvq_append(ctypes.byref(cfg), ctypes.byref(c), q, q, None) == kvq.KVQ_EINVAL, bad
