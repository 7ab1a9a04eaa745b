"""The bench's clock sampler on CPU: parsing nvidia-smi's query lines and
flagging the throttle reasons that reject a measurement."""
import datetime
import time

from draft_verification_02_b300 import clocks


def _line(sm, reasons_hex, named):
    t = datetime.datetime.now().strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{t}, {sm}, 2032, 640.50, {reasons_hex}, " + ", ".join(named) + "\n"


def test_summary_of_samples_inside_the_timed_region(tmp_path):
    p = tmp_path / "c.txt"
    na = ["Not Active"] * 4
    p.write_text(_line(1900, "0x0000000000000000", na) +
                 _line(1950, "0x0000000000000004", na[:3] + ["Active"]))
    s = clocks.summarize(str(p), time.time() - 60, time.time() + 60)
    assert s["samples"] == 2 and s["sm_mhz"] == 1925 and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"] and s["rejected"] is False


def test_thermal_slowdown_rejects(tmp_path):
    p = tmp_path / "c.txt"
    p.write_text(_line(1500, "0x0000000000000040", ["Not Active", "Active", "Not Active",
                                                    "Not Active"]))
    s = clocks.summarize(str(p), time.time() - 60, time.time() + 60)
    assert s["rejected"] is True and "hw_thermal_slowdown" in s["reasons"]


def test_errors_are_reported(tmp_path):
    p = tmp_path / "c.txt"
    p.write_text("nvidia-smi unavailable: not found\n")
    s = clocks.summarize(str(p), 0, 1)
    assert s["samples"] == 0 and "unavailable" in s["error"]


def test_command_is_read_only():
    cmd = clocks.command("00000000:1B:00.0", 50)
    assert cmd[0] == "nvidia-smi" and any(c.startswith("--query-gpu=") for c in cmd)
    assert not any(c in cmd for c in ("-lgc", "-ac", "-pm", "-rgc", "-r"))
