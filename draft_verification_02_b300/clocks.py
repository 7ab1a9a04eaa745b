"""Read-only GPU clock sampler (NVML), run as a separate process so that it
never competes with the benchmark's launch thread.

    python -m draft_verification_02_b300.clocks --pci 0000:1b:00.0 --interval-ms 5 --out f

Writes one line per sample: wall time (s), SM MHz, max SM MHz, power (W),
active clock-event reason bits.  It only reads; it changes no GPU setting.
"""
from __future__ import annotations

import argparse
import statistics
import sys
import time

REASONS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
    0x100: "display_clock_setting",
}
REJECT = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def _handle(pynvml, pci):
    if pci:
        try:
            return pynvml.nvmlDeviceGetHandleByPciBusId(pci.encode())
        except Exception:
            pass
    return pynvml.nvmlDeviceGetHandleByIndex(0)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--pci", default="")
    ap.add_argument("--interval-ms", type=float, default=5.0)
    ap.add_argument("--out", required=True)
    ap.add_argument("--max-seconds", type=float, default=600.0)
    a = ap.parse_args(argv)
    with open(a.out, "w", buffering=1) as f:
        try:
            import pynvml
            pynvml.nvmlInit()
            h = _handle(pynvml, a.pci)
        except Exception as e:
            print(f"# nvml unavailable: {e}", file=f)
            return 1
        t_end = time.time() + a.max_seconds
        while time.time() < t_end:
            t = time.time()
            try:
                sm = pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM)
                smax = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
                pw = pynvml.nvmlDeviceGetPowerUsage(h) / 1000.0
                rs = pynvml.nvmlDeviceGetCurrentClocksEventReasons(h)
            except Exception as e:  # pragma: no cover
                print(f"# nvml query failed: {e}", file=f)
                break
            f.write(f"{t:.6f} {sm} {smax} {pw:.1f} {int(rs)}\n")
            time.sleep(a.interval_ms / 1000.0)
    return 0


def summarize(path: str, t0: float, t1: float) -> dict:
    """Samples taken inside [t0, t1] (the nearest ones if none fall inside)."""
    rows = []
    notes = []
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("#"):
                    notes.append(line[1:].strip())
                    continue
                p = line.split()
                if len(p) == 5:
                    rows.append((float(p[0]), int(p[1]), int(p[2]), float(p[3]), int(p[4])))
    except FileNotFoundError:
        return {"samples": 0, "error": "no clock samples"}
    if not rows:
        return {"samples": 0, "error": "; ".join(notes) or "no clock samples"}
    inside = [r for r in rows if t0 <= r[0] <= t1]
    note = None
    if not inside:
        inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        note = "timed region shorter than the sampling interval: nearest samples"
    reasons = set()
    for r in inside:
        for bit, name in REASONS.items():
            if r[4] & bit:
                reasons.add(name)
    out = {"sm_mhz": statistics.median(r[1] for r in inside),
           "sm_max_mhz": max(r[2] for r in inside),
           "power_w_max": max(r[3] for r in inside),
           "reasons": sorted(reasons - {"gpu_idle"}),
           "samples": len(inside)}
    if note:
        out["note"] = note
    out["rejected"] = bool(reasons & REJECT)
    return out


if __name__ == "__main__":
    sys.exit(main())
