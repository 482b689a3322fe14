"""Host logic of bench.py on the CPU: the algorithmic work it divides by, the ncu traffic
it attaches to the roofline, the peaks it falls back to and the clock record it reads.

These are the numbers behind every bench line, so each is checked against its own
definition on small cases written out by hand.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_tiled_attention_20_gb300 import inputs  # noqa: E402


def test_decode_bytes_counts_valid_rows_q_o_and_lse():
    wd = inputs.DecodeWorkload("t", B=2, Hq=4, Hkv=2, D=64, Smax=100, len_lo=1, len_hi=100)
    lens = [10, 0]
    kv = (10 + 0) * 2 * 64 * 2 * 2            # K and V rows actually read, 2 bytes each
    q_o = 2 * 4 * 64 * 2 * 2                  # one query and one output row per head
    lse = 2 * 4 * 4
    assert bench.decode_bytes(wd, lens) == kv + q_o + lse


def test_row_flops_non_causal_and_causal():
    wf = inputs.FwdWorkload("t", B=1, Sq=4, Sk=6, Hq=1, Hkv=1, D=8, causal=False)
    rows = np.array([[0, 0, 0], [0, 0, 3]])
    assert bench._row_flops(wf, rows) == 2 * 4.0 * 6 * 8
    wc = inputs.FwdWorkload("t", B=1, Sq=4, Sk=6, Hq=1, Hkv=1, D=8, causal=True)
    # bottom-right alignment: row i sees keys j <= i + Sk - Sq, i.e. i + 3 of them
    assert bench._row_flops(wc, rows) == 4.0 * 8 * (3 + 6)


def test_ncu_traffic_only_for_the_sources_it_was_taken_on(monkeypatch):
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        stored = json.load(f)
    entry = stored["fa_fwd_kernel"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: entry["source_hash"])
    assert bench.ncu_traffic("fa_fwd_kernel") == entry["bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 16)
    assert bench.ncu_traffic("fa_fwd_kernel") is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_traffic_hash_covers_each_kernel_and_the_shared_layer_only():
    fwd = bench.kernel_source_files("fa_fwd_kernel")
    dec = bench.kernel_source_files("fa_decode_split_kernel")
    assert "fa_fwd.cuh" in fwd and "fa_decode.cuh" in dec
    assert not any(n.startswith("fa_decode") for n in fwd)
    assert not any(n.startswith("fa_fwd") for n in dec)
    for shared in ("fa_ptx.cuh", "fa_api.cu"):
        assert shared in fwd and shared in dec


def test_source_hash_ignores_comments_only():
    a = 'int x = 1; // one\n/* block */ asm("mov.u32 %0, 1; // not a comment");\n'
    b = 'int x = 1;\n asm("mov.u32 %0, 1; // not a comment");'
    c = 'int x = 2;\n asm("mov.u32 %0, 1; // not a comment");'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert "// not a comment" in bench._code_only(a)


def test_stored_traffic_is_close_to_the_algorithmic_bytes():
    """The committed forward capture, scaled to the full launch, is within 10 % of the
    algorithmic bytes 2 (|Q| + |K| + |V| + |O|) + 4 B Hq S; the decode's within 2 %."""
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        stored = json.load(f)
    wf = inputs.PREFILL_LONG[0]
    n = wf.B * wf.Sq * wf.Hq * wf.D
    alg = 2.0 * 4 * n + 4.0 * wf.B * wf.Hq * wf.Sq
    assert abs(stored["fa_fwd_kernel"]["bytes_per_launch"] / alg - 1) < 0.10
    wd = inputs.DECODE
    _, _, _, lens = inputs.decode_inputs(wd)
    alg_d = bench.decode_bytes(wd, lens.tolist())
    assert abs(stored["fa_decode_split_kernel"]["bytes_per_launch"] / alg_d - 1) < 0.02


def test_peaks_fall_back_when_the_measured_file_is_absent(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, source = bench.load_peaks()
    assert source == "fallback"
    assert peaks == bench.FALLBACK_PEAKS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1.0}))
    peaks, source = bench.load_peaks()
    assert source == "measured" and peaks == {"hbm_gbs": 1.0}


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_record_median_and_throttle_reasons(tmp_path):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1950, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1395.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    with open(s.path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.fh = open(s.path, "a")
    s.proc = _FakeProc()
    rec = s.stop()
    # the three samples are all above the 300 W load threshold
    assert rec == {"sm_mhz": 1980.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                   "samples": 3, "samples_under_load": 3, "power_cap_frac": round(2 / 3, 3),
                   "power_w_max": 1395.0}
    assert not os.path.exists(s.path)


def test_clock_record_keeps_only_samples_under_load():
    lines = ["0, 1987, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2070, 2070, 640.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 2070, 2070, 650.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1987, 2070, [N/A], 0x0, Not Active, Not Active, Not Active, Not Active"]
    rec = bench.parse_clock_csv(lines)
    assert rec["sm_mhz"] == 2070.0 and rec["samples_under_load"] == 2 and rec["samples"] == 4
    assert rec["power_cap_frac"] == 0.0 and rec["reasons"] == []
    # with no sample under load, every sample counts
    rec = bench.parse_clock_csv(lines[:1])
    assert rec["sm_mhz"] == 1987.0 and rec["samples_under_load"] == 1


def test_peak_follows_the_clock_record():
    peaks = {"bf16_tflops": 1939.8, "bf16_tflops_sustained": 1703.7, "hbm_gbs": 6788.3}
    burst = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_cap_frac": 0.1}
    capped = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "power_cap_frac": 0.8}
    slow = {"sm_mhz": 1485.0, "sm_max_mhz": 2070.0, "power_cap_frac": 0.0}
    assert bench.choose_tensor_peak(peaks, "measured", burst)[0] == 1939.8
    assert bench.choose_tensor_peak(peaks, "measured", capped)[0] == 1703.7
    assert bench.choose_tensor_peak(peaks, "measured", slow)[0] == 1703.7
    assert bench.choose_tensor_peak(peaks, "measured", None)[0] == 1703.7
    r = bench.tensor_roofline(1637.0, peaks, "measured", burst, num_sms=152)
    assert r["frac"] == round(1637.0 / 1939.8, 4) and "burst" in r["peak_kind"]
    assert r["frac_of_sustained"] == round(1637.0 / 1703.7, 4)
    nominal = 152 * 8192 * 2070e6 / 1e12
    assert r["clock_nominal"]["peak"] == round(nominal, 1)


def test_visible_keys_causal_and_window():
    # bottom-right causal with Sq = 4, Sk = 6: row i sees i + 3 keys
    assert [bench.visible_keys(i, 4, 6, True) for i in range(4)] == [3, 4, 5, 6]
    assert [bench.visible_keys(i, 4, 6, False) for i in range(4)] == [6] * 4
    # window (2, 0) with causal, Sq = Sk = 5: row i sees min(i + 1, 3) keys
    assert [bench.visible_keys(i, 5, 5, True, (2, 0)) for i in range(5)] == [1, 2, 3, 3, 3]
    # a row whose window lies before key 0 sees nothing (Sq > Sk, causal)
    assert bench.visible_keys(0, 5, 2, True) == 0


def test_clock_record_absent_without_nvidia_smi():
    s = bench.ClockSampler(0)
    assert s.stop() is None  # never started
