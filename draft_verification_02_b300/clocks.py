"""Read-only GPU clock sampler, run beside the benchmark: it starts
`nvidia-smi --query-gpu ... -lms N` for one GPU and keeps its output, and
`summarize` reduces the samples that fall inside the timed region.  It only
reads; it changes no GPU setting.

    python -m draft_verification_02_b300.clocks --gpu 00000000:1B:00.0 --interval-ms 50 --out f

Each sample line: timestamp, SM MHz, max SM MHz, power (W), active event
reasons (bit mask), then hw_slowdown, hw_thermal_slowdown,
sw_thermal_slowdown and sw_power_cap as Active / Not Active.
"""
from __future__ import annotations

import argparse
import datetime
import statistics
import subprocess
import sys

QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
NAMED = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
REASON_BITS = {
    0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
    0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
    0x100: "display_clock_setting",
}
REJECT = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


def command(gpu: str, interval_ms: int) -> list:
    cmd = ["nvidia-smi", f"--query-gpu={QUERY}", "--format=csv,noheader,nounits",
           f"--loop-ms={int(interval_ms)}"]
    if gpu:
        cmd.append(f"--id={gpu}")
    return cmd


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpu", default="", help="PCI bus id or index for nvidia-smi --id")
    ap.add_argument("--interval-ms", type=int, default=50)
    ap.add_argument("--out", required=True)
    a = ap.parse_args(argv)
    with open(a.out, "w", buffering=1) as f:
        try:
            p = subprocess.Popen(command(a.gpu, a.interval_ms), stdout=f,
                                 stderr=subprocess.STDOUT)
        except OSError as e:
            print(f"# nvidia-smi unavailable: {e}", file=f)
            return 1
        return p.wait()


def _parse_time(s: str) -> float:
    s = s.strip()
    for fmt in ("%Y/%m/%d %H:%M:%S.%f", "%Y/%m/%d %H:%M:%S"):
        try:
            return datetime.datetime.strptime(s, fmt).timestamp()
        except ValueError:
            pass
    raise ValueError(s)


def parse(path: str):
    """(samples, notes): samples are (t, sm, max, power, reasons set)."""
    rows, notes = [], []
    try:
        with open(path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) != 9:
                    if line.strip():
                        notes.append(line.strip()[:200])
                    continue
                try:
                    t = _parse_time(p[0])
                    sm, smax = int(float(p[1])), int(float(p[2]))
                    pw = float(p[3]) if p[3] not in ("[N/A]", "N/A") else 0.0
                    bits = int(p[4], 16) if p[4].lower().startswith("0x") else 0
                except ValueError:
                    notes.append(line.strip()[:200])
                    continue
                reasons = {name for bit, name in REASON_BITS.items() if bits & bit}
                for name, v in zip(NAMED, p[5:9]):
                    if v == "Active":
                        reasons.add(name)
                rows.append((t, sm, smax, pw, reasons))
    except FileNotFoundError:
        notes.append("no clock file")
    return rows, notes


def summarize(path: str, t0: float, t1: float) -> dict:
    """Samples taken inside [t0, t1] (the nearest ones if none fall inside)."""
    rows, notes = parse(path)
    if not rows:
        return {"samples": 0, "error": "; ".join(notes) or "no clock samples"}
    inside = [r for r in rows if t0 <= r[0] <= t1]
    note = None
    if not inside:
        inside = sorted(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))[:2]
        note = "timed region shorter than the sampling interval: nearest samples"
    reasons = set()
    for r in inside:
        reasons |= r[4]
    out = {"sm_mhz": statistics.median(r[1] for r in inside),
           "sm_max_mhz": max(r[2] for r in inside),
           "power_w_max": max(r[3] for r in inside),
           "reasons": sorted(reasons - {"gpu_idle"}),
           "samples": len(inside),
           "source": "nvidia-smi --query-gpu"}
    if note:
        out["note"] = note
    out["rejected"] = bool(reasons & REJECT)
    return out


if __name__ == "__main__":
    sys.exit(main())
