"""Per-phase timeline of the persistent decode step (diagnostic).

Needs a library built with the step's trace hooks compiled in:

    KMR_NVCC_FLAGS=-DKMR_STEP_TRACE python -c "import __graft_entry__ as g; g.build()"
    python -m int4_weight_only_group_gb300.steptrace [B]

It runs a few persistent decode steps of the seeded 28-layer 2B-shaped workload (batch 1 or 4)
and reads the %globaltimer stamps thread 0 of every CTA wrote for the last step: per phase (QKV,
attention, O, gate_up, down of each layer) its start after the phase barrier and its end, and
points inside the projection and attention phases.  Prints, per phase kind averaged over the
layers, the barrier wait and the work time, then the projection and attention timelines.
"""
from __future__ import annotations

import ctypes
import sys

import numpy as np

PHASES = ("qkv", "attn", "o", "gate_up", "down")
MAX_CTAS = 160
MAX_LAYERS = 64


def main(batch: int = 1) -> None:
    import torch

    import int4_weight_only_group_gb300 as kmr
    from int4_weight_only_group_gb300 import driver
    from workloads import SyntheticModel, full2b_b1_workload, full2b_b4_workload, initial_state

    L = kmr.lib()
    if not hasattr(L, "kmr_step_trace"):
        raise SystemExit("the library has no step trace: build it with KMR_NVCC_FLAGS=-DKMR_STEP_TRACE")
    wl = full2b_b1_workload() if batch == 1 else full2b_b4_workload()
    cfg = wl.cfg
    syn = SyntheticModel(cfg, wl.seed)
    m = kmr.Model.from_config(cfg, max_batch=batch)
    driver.load_weights(m, syn, cfg.n_layers, cfg.qk_norm)
    for b in range(batch):
        driver.load_kv(m, syn, cfg.n_layers, wl.slot_ids[b], wl.prefill[b])
    m.set_persistent_step(True)
    dev = [torch.tensor(np.asarray(v), device="cuda") for v in initial_state(wl)]
    for _ in range(6):
        m.decode_step(*dev, batch, None)
    torch.cuda.synchronize()
    assert m.sync_status() == 0
    nph = len(PHASES) * MAX_LAYERS
    marks = np.zeros((MAX_CTAS, 2 + 2 * nph), np.uint64)
    subs = np.zeros((MAX_CTAS, nph, 5), np.uint64)
    L.kmr_step_trace.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert L.kmr_step_trace(marks.ctypes.data, subs.ctypes.data) == 0
    m.close()

    G = int(torch.cuda.get_device_properties(0).multi_processor_count)
    t = marks[:G].astype(np.int64)
    t0 = t[:, 0].min()
    t = (t - t0) / 1000.0                               # us from the first CTA's start
    sub = subs[:G].astype(np.int64)
    nl = cfg.n_layers
    print(f"batch {batch}: {G} CTAs, start spread {t[:, 0].max():.2f} us, copy schedule built "
          f"(median / max) {np.median(t[:, 1]):.2f} / {t[:, 1].max():.2f} us, "
          f"last phase ends {t[:, 3 + 2 * (nl * len(PHASES) - 1)].max():.1f} us")
    rows = {n: [] for n in PHASES}
    for layer in range(nl):
        for k, name in enumerate(PHASES):
            idx = layer * len(PHASES) + k
            prev_leave = t[:, 3 + 2 * (idx - 1)].max() if idx > 0 else t[:, 1].max()
            ent, lv = t[:, 2 + 2 * idx], t[:, 3 + 2 * idx]
            rows[name].append((np.median(ent) - prev_leave, ent.max() - prev_leave, lv.max() - ent.max(),
                               np.median(lv - ent)))
    print("phase    barrier wait (median / max, us)   slowest end after last start   work (median, us)")
    for name in PHASES:
        a = np.array(rows[name]).mean(axis=0)
        print(f"{name:8s} {a[0]:6.2f} / {a[1]:6.2f}                       {a[2]:6.2f}                 {a[3]:6.2f}")
    print("projection timeline, us after the phase start (median over CTAs with work, layers 2..):")
    for k, name in enumerate(PHASES):
        if name == "attn":
            continue
        acc = []
        for layer in range(2, nl):
            idx = layer * len(PHASES) + k
            ent = t[:, 2 + 2 * idx] * 1000.0 + t0
            lv = t[:, 3 + 2 * idx] * 1000.0 + t0
            a = sub[:, idx, :].astype(np.float64)
            ok = a[:, 0] > 0
            if not ok.any():
                continue
            e = ent[ok]
            acc.append([np.median((a[ok, j] - e) / 1000.0) for j in range(5)] + [np.median((lv[ok] - e) / 1000.0)])
        v = np.array(acc).mean(axis=0)
        print(f"  {name:8s} body {v[0]:.2f}, x staged {v[1]:.2f}, weight slots ready {v[2]:.2f}, "
              f"products {v[3]:.2f}, epilogue end {v[4]:.2f}, leave {v[5]:.2f}")
    vals = []
    for layer in range(2, nl):
        idx = layer * len(PHASES) + 1
        ent = t[:, 2 + 2 * idx] * 1000.0 + t0
        a = sub[:, idx, :].astype(np.float64)
        ok = a[:, 4] > 0
        d = (a[ok] - ent[ok][:, None]) / 1000.0
        vals.append([np.median(d[:, j]) for j in range(5)] + [d[:, 4].max(), ok.sum()])
    v = np.array(vals).mean(axis=0)
    print(f"attention items, us after the phase start: start {v[0]:.2f}, prologue done {v[1]:.2f}, "
          f"scoring done {v[2]:.2f}, state written {v[3]:.2f}, item end median {v[4]:.2f} max {v[5]:.2f} "
          f"({v[6]:.0f} CTAs with an item)")


if __name__ == "__main__":
    main(int(sys.argv[1]) if len(sys.argv) > 1 else 1)
