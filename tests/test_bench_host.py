"""Host-side helpers of bench.py (no GPU): the watchdog and the device record."""
import os
import subprocess
import sys
import threading

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_watchdog_fires_and_reports(capsys):
    fired = threading.Event()
    t = bench.start_watchdog(0.05, on_timeout=fired.set)
    assert fired.wait(5.0)
    t.join(5.0)
    assert "bench watchdog: no result after" in capsys.readouterr().err


def test_watchdog_cancelled_in_time_stays_quiet():
    fired = threading.Event()
    t = bench.start_watchdog(30.0, on_timeout=fired.set)
    t.cancel()
    t.join(5.0)
    assert not fired.is_set()


def test_device_info_never_raises():
    class NoCuda:
        class cuda:
            @staticmethod
            def current_device():
                raise RuntimeError("no device")

    info = bench.device_info(NoCuda)
    assert info["gpu"] is None and info["sms"] is None and info["host_cores"] == os.cpu_count()


def test_cli_parses_without_a_gpu():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--help"], capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and "--watchdog-s" in r.stdout


def test_timed_step_accounting_counts_active_rows_and_their_kv():
    """Batch-4 slots: row 2 retires at step 64, row 3 (900 prefilled) writes its last position at
    step 123; tokens and KV bytes of the timed steps follow that row by row."""
    from workloads import full2b_b4_workload
    wl = full2b_b4_workload()
    c = wl.cfg
    per_pos = c.n_layers * 2 * c.n_kv_heads * c.head_dim * 2
    tok, kv = bench.timed_steps_accounting(wl, 20)
    assert tok == 80
    assert kv == per_pos * sum(p + t + 1 for p in wl.prefill for t in range(20))
    tok, kv = bench.timed_steps_accounting(wl, wl.steps)
    assert tok == bench.tokens_per_generation(wl) == 128 + 128 + 64 + 124


def test_oracle_leg_times_whole_steps():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-leg", "tiny", "--oracle-steps", "2",
                        "--oracle-budget-s", "30"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    import json
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["steps"] == 2 and len(d["s_per_step"]) == 2 and d["extrapolated"] is False and d["tok_per_s"] > 0


def test_projection_flop_counts_every_layer_projection():
    """2 flops per weight and token over QKV, O, gate_up and down of every layer (2B shapes:
    4096 x 2048 + 2048 x 2048 + 12288 x 2048 + 2048 x 6144 weights per layer)."""
    import bench
    from workloads import layer2b_config
    cfg = layer2b_config(slots=1, n_layers=28)
    per_layer = 4096 * 2048 + 2048 * 2048 + 12288 * 2048 + 2048 * 6144
    assert bench.projection_flop(cfg, 512) == 2.0 * per_layer * 512 * 28
    assert bench.projection_flop(cfg, 0) == 0.0


def test_prefill_record_reports_flop_rate_and_speedup():
    """The prefill object: the projections' flops over the default path's time, its fraction of
    the measured bf16 peak, and the warp-level path's time and the speedup over it."""
    import bench
    from workloads import layer2b_config
    cfg = layer2b_config(slots=1, n_layers=28)
    r = {"prefill": {"tokens": 512, "ms": 4.0, "tok_s": 128000.0}, "prefill_mma": {"ms": 8.0}}
    rec = bench.prefill_record(r, cfg, {"bf16_tflops": 1854.8})
    flop = bench.projection_flop(cfg, 512)
    assert rec["kernel"] == "tcgen05" and rec["tokens"] == 512 and rec["ms"] == 4.0
    assert abs(rec["projection_tflops_whole_prefill"] - round(flop / 4e-3 / 1e12, 1)) < 1e-9
    assert abs(rec["frac_of_bf16_peak"] - round(flop / 4e-3 / 1e12 / 1854.8, 3)) < 1e-9
    assert rec["warp_mma_ms"] == 8.0 and rec["speedup_over_warp_mma"] == 2.0
    assert bench.prefill_record(r, cfg, {})["frac_of_bf16_peak"] is None
