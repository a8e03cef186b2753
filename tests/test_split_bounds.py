"""Workspace bound of the tensor-core MHA decode's warp-level split, checked
on the host for every reachable cache state of the named workloads (and
edge shapes): the warps whose unit ranges touch one head never outnumber the
partial slots a head owns in the scratch.

The slot count and the block size come from the library itself
(kvq_workspace_bytes, kvq_cache_sizes); the split below restates the
kernel's own arithmetic: a head is 2 empty units + one unit per 32-token
tile + two units per fp16 chunk, the concatenated units of all heads are
cut into nw equal ranges (warp w holds [w*total/nw, (w+1)*total/nw)), and
nw = min(8 * blocks, total) with blocks = min(SMs * resident, 1024)."""
import ctypes

import pytest

from bit_kv_cache_14_gb300 import build_lib, kvq, synth


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_lib.build()
    yield


def _part_stride(cfg):
    """Partial slots per head of the scratch, from kvq_workspace_bytes."""
    BH, d = cfg.batch * cfg.n_kv_heads, cfg.head_dim
    rg = cfg.n_q_heads // cfg.n_kv_heads
    cnt = (BH * 4 + 255) & ~255
    ws = kvq.workspace_bytes(cfg)
    return (ws - cnt - 256) // (BH * rg * (d + 2) * 4)


def _fp16_chunk(cfg):
    s = kvq.cache_sizes(cfg)
    BH = cfg.batch * cfg.n_kv_heads
    cap = (cfg.max_ctx + 127) // 128 * 128
    block_bytes = (s.blocks - (BH * cfg.head_dim * 4 if cfg.scheme == kvq.INNERQ_KNORM else 0)) \
        // (BH * (cap // 32))
    kmb = 2 * cfg.head_dim * 4 if cfg.scheme == kvq.KIVI and cfg.k_group > 32 else 0
    return min(8, (block_bytes + kmb) // (4 * cfg.head_dim))


def _max_parts(BH, n_quant, n_fp16, ch, blocks):
    nch = -(-n_fp16 // ch) if n_fp16 else 0
    U = 2 + -(-n_quant // 32) + 2 * nch
    total = BH * U
    nw = max(1, min(8 * blocks, total))

    def owner(x):
        return ((x + 1) * nw - 1) // total

    worst = 0
    for bh in range(BH):
        base = bh * U
        worst = max(worst, owner(base + U - 1) - owner(base) + 1)
    return worst, nw, total


CASES = [synth.WORKLOADS[n] for n in ("llama2_7b_2bit", "kivi_4bit", "innerq_1m")] + [
    synth.scaled(synth.WORKLOADS["llama2_7b_2bit"], batch=1, n_q_heads=1, n_kv_heads=1,
                 ctx=64, k_group=16, residual=16),
    synth.scaled(synth.WORKLOADS["innerq_1m"], batch=3, n_q_heads=5, n_kv_heads=5, ctx=5000,
                 bits=2, k_group=32, v_group=32, n_sink=1024, residual=1024),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_tc_split_never_exceeds_the_partial_slots(w):
    cfg = kvq.config_of(w)
    assert kvq.lib().kvq_workspace_bytes(ctypes.byref(cfg), ctypes.byref(ctypes.c_size_t())) == 0
    stride, ch = _part_stride(cfg), _fp16_chunk(cfg)
    BH = cfg.batch * cfg.n_kv_heads
    cap = (cfg.max_ctx + 127) // 128 * 128
    fp16_max = cfg.residual + cfg.n_sink
    quant = sorted({1, 31, 32, 33, 4096, cap // 2, cap - 1, cap} & set(range(1, cap + 1)))
    for n_quant in quant:
        for n_fp16 in sorted({0, 1, ch, fp16_max}):
            for blocks in (1, 8, 152, 304, 608, 1024):
                worst, nw, total = _max_parts(BH, n_quant, n_fp16, ch, blocks)
                assert nw <= total
                assert worst <= stride, (w.name, n_quant, n_fp16, blocks, worst, stride)


def _gqa_max_parts(cfg, BH, n_quant, n_fp16, blocks):
    """Partial slots the grouped-query kernel's block-level split gives its
    busiest head: 8 per block holding quantized units of the head, plus one
    per warp with at least one of a block's fp16 chunks (the kernel's own
    count).  Units: 128 quantized tokens, or CPU fp16 chunks of CH tokens."""
    s = kvq.cache_sizes(cfg)
    cap = (cfg.max_ctx + 127) // 128 * 128
    block_bytes = s.blocks // (BH * (cap // 32))
    ch = _fp16_chunk(cfg)
    kmb = 2 * 128 * 4 if cfg.scheme == kvq.KIVI and cfg.k_group > 32 else 0
    cpu = max(1, (128 // 32) * (block_bytes + kmb) // (ch * 4 * 128))
    nch = -(-n_fp16 // ch) if n_fp16 else 0
    S_h, F_h = -(-n_quant // 128), -(-nch // cpu)
    U = S_h + F_h
    total = BH * U
    nc = max(1, min(blocks, 1024, total))

    def owner(x):
        return ((x + 1) * nc - 1) // total

    worst = 0
    for bh in range(BH):
        base, npart = bh * U, 0
        if S_h:
            npart = 8 * (owner(base + S_h - 1) - owner(base) + 1)
        if F_h:
            for x in range(owner(base + S_h), owner(base + U - 1) + 1):
                x0, x1 = x * total // nc, (x + 1) * total // nc
                fa, fb = max(x0 - base - S_h, 0), min(x1 - base - S_h, F_h)
                c0 = fa * cpu
                c1 = min(fb * cpu, nch) if fa < fb else c0
                npart += min(8, c1 - c0)
        worst = max(worst, npart)
    return worst


GQA_CASES = [synth.WORKLOADS["gqa_2bit"],
             synth.scaled(synth.WORKLOADS["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=4,
                          ctx=900, k_group=64, v_group=64),
             synth.scaled(synth.WORKLOADS["gqa_2bit"], batch=1, n_q_heads=4, n_kv_heads=1,
                          ctx=1 << 20),
             synth.scaled(synth.WORKLOADS["gqa_2bit"], batch=2, n_q_heads=8, n_kv_heads=2,
                          ctx=900, bits=4),
             synth.scaled(synth.WORKLOADS["gqa_2bit"], batch=1, n_q_heads=4, n_kv_heads=1,
                          ctx=1 << 20, bits=4, k_group=64),
             synth.scaled(synth.WORKLOADS["innerq_1m"], batch=2, n_q_heads=8, n_kv_heads=2,
                          ctx=700),
             synth.scaled(synth.WORKLOADS["innerq_1m"], batch=1, n_q_heads=8, n_kv_heads=4,
                          bits=2, k_group=32),
             # fp16 statistics: smaller blocks, so other chunk and unit counts
             synth.scaled(synth.WORKLOADS["gqa_2bit"], meta_f16=True),
             synth.scaled(synth.WORKLOADS["innerq_1m"], batch=2, n_q_heads=8, n_kv_heads=2,
                          ctx=700, meta_f16=True)]


@pytest.mark.parametrize("w", GQA_CASES,
                         ids=lambda w: "%s_B%d_T%d_b%d%s" % (w.name, w.batch, w.ctx, w.bits,
                                                             "_f16" if w.meta_f16 else ""))
def test_gqa_split_never_exceeds_the_partial_slots(w):
    """Block counts up to 8 resident blocks on each of 152 SMs (the kernel
    fits at most 2: 112 KB of shared memory per block; 4-bit codes, 1)."""
    cfg = kvq.config_of(w)
    stride = _part_stride(cfg)
    BH = cfg.batch * cfg.n_kv_heads
    cap = (cfg.max_ctx + 127) // 128 * 128
    quant = sorted({1, 127, 128, 129, cap // 3, cap - 1, cap} & set(range(1, cap + 1)))
    for n_quant in quant:
        for n_fp16 in (0, 1, 9, cfg.residual):
            for blocks in (1, 7, 152, 304, 608, 1216):
                worst = _gqa_max_parts(cfg, BH, n_quant, n_fp16, blocks)
                assert worst <= stride, (n_quant, n_fp16, blocks, worst, stride)
