"""Every tensor-core decode instantiation the library can dispatch to, against
the CPU oracle (all heads, ragged residuals, at least one flush or window
eviction), and a host-side check that the dispatch table has no entry
without such a case.

The tensor-core kernels are templates over the code width, the scheme, the
value groups per head, the key groups per head (InnerQ) or where the KIVI key
statistics live (G 16 / 32 inside the block, G >= 64 beside it), and for the
grouped-query kernel the query heads per KV head.  kvq_decode_kernel_name
reports which instantiation a configuration reaches, so the coverage check
asks the library itself rather than a copy of its rule.
"""
import itertools

import pytest
import torch

from bit_kv_cache_14_gb300 import build_lib, kvq, synth
from parity_util import ATOL, run_workload

W = synth.WORKLOADS
S = synth.scaled


def _kivi(bits, ngv, G, mf=False, out=0, ragged=False):
    base = W["llama2_7b_2bit"] if bits == 2 else W["kivi_4bit"]
    R = 64 if G <= 64 else 128
    return S(base, batch=4 if ragged else 2, n_q_heads=2, n_kv_heads=2, ctx=700, k_group=G,
             v_group=128 // ngv, residual=R, n_append=R + 10, meta_f16=mf, outliers=out,
             ragged=ragged)


def _innerq(bits, ngv, ngk, mf=False, ragged=False):
    return S(W["innerq_1m"], batch=4 if ragged else 2, n_q_heads=2, n_kv_heads=2, ctx=700,
             bits=bits, k_group=128 // ngk, v_group=128 // ngv, n_append=40, meta_f16=mf,
             ragged=ragged)


def _gqa_iq(bits, ngv, ngk, rg, knorm=False, mf=False):
    # 700 prompt tokens: 4 sinks, a 32-token window, 664 quantized (a short
    # last tile), and every append moves one more token into the quantized
    # region
    return S(W["innerq_1m"], batch=2, n_q_heads=2 * rg, n_kv_heads=2, ctx=700, bits=bits,
             k_group=128 // ngk, v_group=128 // ngv, n_append=40, k_norm=knorm, meta_f16=mf)


def _gqa(bits, ngv, G, rg, mf=False):
    return S(W["gqa_2bit"], batch=2, n_q_heads=2 * rg, n_kv_heads=2, ctx=900, bits=bits,
             k_group=G, v_group=128 // ngv, residual=128, n_append=140, meta_f16=mf)


CASES = {}
for mf in (False, True):
    sfx = "_f16" if mf else ""
    for bits, ngv, G in itertools.product((2, 4), (2, 4), (16, 32, 64)):
        CASES["tc_kivi_b%d_ngv%d_g%d%s" % (bits, ngv, G, sfx)] = _kivi(bits, ngv, G, mf)
    for bits, ngv, ngk in itertools.product((2, 4), (2, 4), (2, 4)):
        CASES["tc_innerq_b%d_ngv%d_ngk%d%s" % (bits, ngv, ngk, sfx)] = _innerq(bits, ngv, ngk, mf)
    # the extended kernel: KIVI with outlier lists (1, 2 and 8 per token spread
    # over the shapes); per-sequence lengths only: KIVI and InnerQ
    for i, (bits, ngv, G) in enumerate(itertools.product((2, 4), (2, 4), (16, 32, 64))):
        CASES["tc_kivi_b%d_ngv%d_g%d%s_out" % (bits, ngv, G, sfx)] = _kivi(bits, ngv, G, mf,
                                                                         (1, 2, 8)[i % 3])
        CASES["tc_kivi_b%d_ngv%d_g%d%s_ragged" % (bits, ngv, G, sfx)] = _kivi(bits, ngv, G, mf,
                                                                            ragged=True)
    for bits, ngv, ngk in itertools.product((2, 4), (2, 4), (2, 4)):
        CASES["tc_innerq_b%d_ngv%d_ngk%d%s_ragged" % (bits, ngv, ngk, sfx)] = _innerq(
            bits, ngv, ngk, mf, ragged=True)
for mf in (False, True):
    sfx = "_f16" if mf else ""
    for bits, ngv, G, rg in itertools.product((2, 4), (2, 4), (32, 64), (2, 4)):
        CASES["gqa_b%d_ngv%d_g%d_rg%d%s" % (bits, ngv, G, rg, sfx)] = _gqa(bits, ngv, G, rg, mf)
        # InnerQ keys: the same four axes, with G read as 128 / key channel groups
        CASES["gqa_innerq_b%d_ngv%d_ngk%d_rg%d%s" % (bits, ngv, 128 // G, rg, sfx)] = _gqa_iq(
            bits, ngv, 128 // G, rg, mf=mf)
# InnerQ's folded key normalization on the grouped-query kernel (a run-time
# flag of the same instantiations)
CASES["gqa_innerq_knorm_b2_ngv4_ngk4_rg2"] = _gqa_iq(2, 4, 4, 2, knorm=True)
CASES["gqa_innerq_knorm_b4_ngv2_ngk2_rg4"] = _gqa_iq(4, 2, 2, 4, knorm=True)


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib.build()
    yield


def _name(w):
    return kvq.decode_kernel_name(kvq.config_of(w), 1)


def dispatched_tensor_core_names():
    """Every tensor-core instantiation reachable from a valid configuration."""
    names = set()
    for d, bits, rg, gk, gv in itertools.product((64, 128), (2, 4), (1, 2, 4, 8),
                                                 (16, 32, 64, 128), (16, 32, 64, 128)):
        if gv > d:
            continue
        cfgs = []
        for fl in (0, kvq.META_F16, kvq.META_F16 | kvq.RAGGED, kvq.RAGGED,
                   kvq.VALUE_QUEUE):
            for o in (0, 2):
                cfgs.append(kvq.make_config(2, 2 * rg, 2, d, bits, kvq.KIVI, gk, gv, 128, 0, 4096,
                                            fl, o))
            if gk <= d and not fl & kvq.VALUE_QUEUE:
                cfgs += [kvq.make_config(2, 2 * rg, 2, d, bits, s, gk, gv, 32, 4, 4096, fl)
                         for s in (kvq.INNERQ, kvq.INNERQ_KNORM)]
        for cfg in cfgs:
            name = kvq.decode_kernel_name(cfg, 1)
            if name.startswith("tc_"):
                names.add(name)
    return names


def test_every_dispatched_instantiation_has_a_parity_case():
    dispatched = dispatched_tensor_core_names()
    # MHA: 20 shapes with fp32 and with fp16 statistics, each plain and with
    # per-sequence lengths only, and the 12 KIVI shapes extended (outlier lists,
    # value queue; InnerQ has neither); grouped-query: 8 for each code width
    # with KIVI keys, 8 with InnerQ keys, each with fp32 and fp16 statistics
    assert len(dispatched) == 2 * (2 * 20 + 12) + 64, sorted(dispatched)
    covered = {_name(w) for w in CASES.values()}
    assert dispatched <= covered, sorted(dispatched - covered)
    # and each named case reaches the instantiation its name says
    for name, w in CASES.items():
        got = _name(w)
        if name.startswith("gqa"):
            assert got.startswith("tc_gqa_kernel<"), (name, got)
        else:
            assert got.startswith("tc_decode_kernel<"), (name, got)


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_instantiation_matches_oracle(name):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = CASES[name]
    worst = run_workload(w, decode_every=max(1, w.n_append // 4))
    assert worst <= ATOL


def test_every_rotary_instantiation_has_a_parity_case():
    """The tensor-core form of the decode over keys cached before RoPE: every
    instantiation a valid configuration reaches is one of the rotary parity
    cases in test_gpu_rope.py, and the other shapes name the general kernel."""
    import test_gpu_rope
    dispatched = set()
    for d, bits, rg, gk, gv in itertools.product((64, 128), (2, 4), (1, 2, 4), (16, 32, 64, 128),
                                                 (16, 32, 64, 128)):
        if gv > d:
            continue
        for fl in (0, kvq.META_F16):
            cfg = kvq.make_config(2, 2 * rg, 2, d, bits, kvq.KIVI, gk, gv, 128, 0, 4096, fl)
            name = kvq.rope_kernel_name(cfg, 1)
            if name.startswith("tc_"):
                dispatched.add(name)
                assert d == 128 and rg == 1 and gk >= 32 and not fl, name
            else:
                assert name.startswith("rope_decode_kernel<"), name
    assert len(dispatched) == 8, sorted(dispatched)
    covered = {kvq.rope_kernel_name(kvq.config_of(w), 1) for w in test_gpu_rope.TC_CASES.values()}
    assert dispatched == covered, sorted(dispatched ^ covered)
