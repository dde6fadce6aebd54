"""The bench line's contract, on the CPU.

With the GPU measurement replaced by fixed times, bench.main() prints one
JSON line holding every key of the contract, and the derived figures (the
whole-job value, the end-to-end value, the dominant kernel and its roofline
fraction, the launch count) follow from those times.  The reference arm's
line is checked the same way, with the oracle sample replaced by a fixed
time.
"""
import json
import sys

import pytest

import bench

STEPS = 10
PER = dict(gdn=0.0080, attn=0.0275, accept=0.0168, commit=0.0150, conv=0.0025, conv_commit=0.0091, ddtree=0.0294)


def fake_run_gpu(args, rank, world):
    return dict(ms=0.862 * args.steps, per=dict(PER), dist={k: [v, v, v] for k, v in PER.items()},
                step_pct=[0.860, 0.862, 0.870],
                scale={"gdn_b8_n64": {"ms_per_launch": 0.134, "nodes_per_s_per_layer": 512 / 0.134e-3,
                                      "algorithmic_bytes_per_launch": 63209472,
                                      "achieved": 63209472 / 0.134e-3 / 1e9, "unit": "GB/s"}},
                clocks={"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 5},
                L=8, e2e_ms=1.1 * args.steps, h2d=41182976, d2h=96, launches=68, dev_name="fake", host=None)


def _line(capsys):
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1, out
    return json.loads(out[0])


def test_bench_line_has_every_key_and_consistent_figures(monkeypatch, capsys):
    monkeypatch.setattr(bench, "run_gpu", fake_run_gpu)
    monkeypatch.setattr(bench, "cpu_baseline", lambda host: {"value": 1000.0, "unit": bench.UNIT, "cores": 16,
                                                             "kind": "oracle", "sample": "a block"})
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", str(STEPS), "--warmup", "3"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main()
    line = _line(capsys)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["n_gpus"] == 1 and line["steps"] == STEPS and line["warmup"] == 3
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert "workload" in line["config"]
    # nodes verified per second per layer: 22 nodes x 64 layers per step
    assert line["value"] == pytest.approx(22 * 64 * STEPS / (0.862 * STEPS * 1e-3))
    assert line["ms_per_step"] == pytest.approx(0.862)
    assert line["e2e"]["value"] == pytest.approx(22 * 64 * STEPS / (1.1 * STEPS * 1e-3))
    assert line["e2e"]["h2d_bytes_per_step"] == 41182976 and line["e2e"]["d2h_bytes_per_step"] == 96
    assert line["gpu_launches"] == 68 * STEPS
    # the dominant kernel is the one with the largest share of the step:
    # attention 16 x 27.5 us against GDN 48 x 8.0 us
    roof = line["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in roof, k
    assert roof["kernel"] == "attn" and roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert roof["achieved"] == pytest.approx(bench.attn_bytes() / (PER["attn"] * 1e-3) / 1e9)
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert roof["traffic"] is None or isinstance(roof["traffic"], int)
    cb = line["cpu_baseline"]
    for k in ("value", "unit", "cores", "kind", "sample"):
        assert k in cb, k
    assert line["nodes_per_s_per_layer"]["attn"] == pytest.approx(22 / (PER["attn"] * 1e-3))
    assert line["at_scale"]["gdn_b8_n64"]["frac"] == pytest.approx(
        line["at_scale"]["gdn_b8_n64"]["achieved"] / roof["peak"])
    assert set(line["clocks"]) >= {"sm_mhz", "sm_max_mhz", "reasons"}


def test_reference_arm_line(monkeypatch, capsys):
    import oracle

    monkeypatch.setattr(bench, "oracle_block_sample", lambda host: 0.25)
    monkeypatch.setattr(bench, "make_host_inputs", lambda rng, n_layers=4: None)
    monkeypatch.setattr(oracle, "set_threads", lambda n: 4)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "4", "--warmup", "3"])
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    bench.main()
    line = _line(capsys)
    assert line["impl"] == "reference" and line["steps"] == 4
    # one 4-layer block of 22 nodes per step, 0.25 s each
    assert line["value"] == pytest.approx(22 * 4 / 0.25)
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["cores"] == 4
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
