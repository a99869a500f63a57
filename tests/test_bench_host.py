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
