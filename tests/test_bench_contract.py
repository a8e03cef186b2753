"""The benchmark's GPU-arm JSON line keeps its contract, checked on the CPU:
bench.main() runs with the GPU leg replaced by fixed figures (and the rank
reduction on the CPU), and the one line it prints carries every key the
contract names, with the whole-job value, the roofline of the timed kernel
(traffic from the committed ncu summary while its source hash matches), the
end-to-end figure, the launch count, the clocks and the oracle baseline."""
import contextlib
import io
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

BYTES = 134348800  # one decode launch on the Llama-2-7B-shaped layer, 4096 + 1 tokens


def _fake_gpu(args, w, rank, world):
    return dict(warmup_steps=1280, elapsed_ms=600.0, total_bytes=args.steps * BYTES,
                decode_ms=0.0274, timed_launches=args.steps + args.steps // 128,
                dstate_bytes=BYTES, plain_ms=0.031, e2e_ms=12.0, e2e_bytes=256 * BYTES,
                n_e2e=256, h2d=196608, d2h=131072,
                clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 9},
                copies=5, cache_bytes=1, prefill_ms=0.65, prompt_bytes_in=536870912,
                l2=136e6, ws_cache_total=5, append={"store": {"us_median": 3.0, "launches": 9}})


@pytest.fixture
def line(monkeypatch):
    monkeypatch.setattr(bench, "run_gpu", _fake_gpu)
    monkeypatch.setattr(bench, "run_configs",
                        lambda names, peak, base=None: {n: {"us": 1.0, "frac": 0.5}
                                                        for n in names})
    real = bench.max_over_ranks
    monkeypatch.setattr(bench, "max_over_ranks", lambda v, world, device: real(v, world, "cpu"))

    def run(*argv):
        monkeypatch.setattr(sys, "argv", ["bench.py", *argv])
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            bench.main()
        rows = [r for r in out.getvalue().splitlines() if r.strip()]
        assert len(rows) == 1
        return json.loads(rows[0])
    return run


REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "roofline",
            "e2e", "gpu_launches", "clocks")


def test_decode_bytes_match_the_layout_arithmetic():
    """Bytes per decode (the roofline's numerator) for the Llama layer: 128 B
    per quantized token-head (64 of codes, 64 of fp32 statistics), 96 with
    fp16 statistics, + 16 with two outliers per token and tensor, 512 per fp16
    token-head; the value queue keeps up to R - 1 values fp16 (256 B each
    instead of 64); ragged sequences each count their own tokens."""
    w = bench.synth.WORKLOADS["llama2_7b_2bit"]
    S = bench.synth.scaled
    assert bench.decode_bytes(w, 4096, 1, 0) == BYTES
    assert bench.decode_bytes(S(w, meta_f16=True), 4096, 1, 0) == 256 * (4096 * 96 + 512)
    assert bench.decode_bytes(S(w, outliers=2), 4096, 1, 0) == 256 * (4096 * 144 + 512)
    vq = S(w, v_queue=True)
    # 4097 tokens, R = 128: values of tokens 3970 .. 4096 (127) still fp16
    assert bench.decode_bytes(vq, 4096, 1, 0) == 256 * (4096 * 64 + 3970 * 64 + 256 + 127 * 256)
    rg = S(w, ragged=True)
    assert bench.decode_bytes_ragged(rg, [4097] * 8) == BYTES
    assert bench.decode_bytes_ragged(rg, [0] * 8) == 0


@pytest.mark.parametrize("rope", [False, True])
def test_gpu_line_contract(line, rope):
    argv = ["--steps", "2000", "--warmup", "5", "--cpu-seconds", "0.5"]
    if rope:
        argv += ["--rope-base", "10000"]
    d = line(*argv)
    for k in REQUIRED:
        assert k in d, k
    assert d["steps"] == 2000 and d["n_gpus"] == 1 and d["scaling"] == "weak"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] == pytest.approx(2000 * BYTES / 0.6 / 1e9)
    assert d["config"]["workload"] == "llama2_7b_2bit"
    assert ("variant" in d["config"]) == rope
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(BYTES / 0.0274e-3 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    # (the tensor-core kernel in both: its rotary form for keys cached before RoPE)
    assert r["kernel"] == "tc_decode_kernel"
    # from the committed ncu summary while its source hash matches (then at
    # least the algorithmic bytes), else null
    assert r["traffic"] is None or r["traffic"] > BYTES
    e = d["e2e"]
    assert set(("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step")) <= set(e)
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] > 0
    assert set(("sm_mhz", "sm_max_mhz", "reasons")) <= set(d["clocks"])
    if rope:
        assert "configs" not in d
    else:
        # the other named workloads, each with its own decode-kernel line
        assert sorted(d["configs"]) == ["gqa_2bit", "innerq_1m", "kivi_4bit", "tiny"]
        # and each cache-format option on the headline layer
        assert sorted(d["formats"]) == ["meta_f16", "outliers_2", "ragged", "value_queue"]
        # and the derived shapes (the grouped-query layer with 4-bit codes)
        assert sorted(d["variants"]) == ["gqa_4bit", "innerq_gqa"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1 and cb["sample"]
