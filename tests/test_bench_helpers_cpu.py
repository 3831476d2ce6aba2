"""Host logic of bench.py that decides what the bench line reports: the DRAM
traffic read from profiles/ (only while the kernel sources keep the hash the
counters were taken with), the rejection of a timed region by its clock
record, and the parsing of the sampled clocks."""
import os
import shutil

import bench


REPO = bench.ROOT


def _tree(tmp_path, lines):
    csrc = tmp_path / "bf16_causal_prefill_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.ATTN_SOURCES:
        shutil.copy(os.path.join(REPO, "bf16_causal_prefill_gb300", "csrc", name), csrc / name)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "attn.md").write_text("\n".join(lines) + "\n")
    return csrc


def test_traffic_is_read_only_for_the_current_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    csrc = _tree(tmp_path, [])
    h = bench.source_hash(*bench.ATTN_SOURCES)
    (tmp_path / "profiles" / "attn.md").write_text(
        "# summary\n"
        f"traffic[attn_fwd_fp8:w32k]: 586435328 bytes/launch src={h}\n"
        "traffic[attn_fwd_bf16:w32k]: 897987925 bytes/launch src=0123456789abcdef\n")
    assert bench.traffic_from_profiles(bench.ATTN_SOURCES, "attn_fwd_fp8:w32k") == 586435328.0
    # counters taken with other sources, or for another tag: none
    assert bench.traffic_from_profiles(bench.ATTN_SOURCES, "attn_fwd_bf16:w32k") is None
    assert bench.traffic_from_profiles(bench.ATTN_SOURCES, "attn_fwd_fp8:w8k") is None
    # any change to a kernel source (a comment included) retires the figure
    with open(csrc / bench.ATTN_SOURCES[0], "a") as f:
        f.write("\n// changed\n")
    assert bench.source_hash(*bench.ATTN_SOURCES) != h
    assert bench.traffic_from_profiles(bench.ATTN_SOURCES, "attn_fwd_fp8:w32k") is None


def test_committed_traffic_lines_are_well_formed():
    """Every traffic line under profiles/ names a kernel and workload, a
    positive byte count and a 16-digit source hash."""
    import re
    pat = re.compile(r"^traffic\[(attn_fwd_(fp8|bf16)):([a-z0-9_]+)\]:\s*([0-9]+)\s+bytes/launch\s+src=([0-9a-f]{16})$")
    n = 0
    pdir = os.path.join(REPO, "profiles")
    for name in os.listdir(pdir):
        for line in open(os.path.join(pdir, name)):
            if line.startswith("traffic["):
                m = pat.match(line.strip())
                assert m, line
                assert int(m.group(4)) > 0
                n += 1
    assert n >= 2


def test_clock_records_that_reject_a_run():
    ok = {"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}
    assert not bench.clocks_rejected(ok)
    assert not bench.clocks_rejected(None)
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert bench.clocks_rejected({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": [r]})
    # clocks stuck far below the maximum with no reason: a leftover lock
    assert bench.clocks_rejected({"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": []})
    # low clocks under the power cap are kept
    assert not bench.clocks_rejected({"sm_mhz": 900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]})


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_samples_are_summarised_over_the_loaded_ones(tmp_path):
    csv = tmp_path / "clocks.csv"
    csv.write_text(
        "0, 2070, 2070, 120.5, 0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "0, 1950, 2070, 1390.2, 100, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 1965, 2070, 1385.0, 100, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
        "0, 1980, 2070, 1370.8, 99, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
        "garbled line\n")
    cs = bench.ClockSampler(0)
    cs.proc, cs.path = _Done(), str(csv)
    c = cs.stop()
    assert c["samples"] == 3                      # the idle sample is left out
    assert c["sm_mhz"] == 1965.0 and c["sm_max_mhz"] == 2070.0
    assert c["power_w_max"] == 1390.2
    assert c["reasons"] == ["sw_power_cap"]
    assert not os.path.exists(csv)
