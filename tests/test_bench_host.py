"""Host-side logic of bench.py (no GPU): the work conventions its metrics use
and the rule that a recorded DRAM figure is reported only while the kernel
sources it was captured on are unchanged."""

import re

import pytest

import bench


def test_forward_flops_convention():
    # 4 * B * H * L^2 * D: 2.199 TFLOP at B8 H32 L4096 D128 (the headline workload)
    full = bench.fwd_flops(8, 32, 4096, 128, False)
    assert full == 4.0 * 8 * 32 * 4096 * 4096 * 128
    assert round(full / 1e12, 3) == 2.199
    # causal counts half the square
    assert bench.fwd_flops(8, 32, 4096, 128, True) == full / 2
    # queries as the last Lq of Lk positions: Lq*(Lk-Lq) fully visible pairs + Lq^2/2
    assert bench.fwd_flops(1, 1, 2, 1, True, Lk=6) == 4.0 * (2 * 4 + 2 * 2 / 2)
    assert bench.fwd_flops(1, 1, 2, 1, False, Lk=6) == 4.0 * 2 * 6


def test_step_is_forward_plus_two_and_a_half_backward():
    f = bench.fwd_flops(4, 8, 1024, 64, True)
    assert bench.step_flops(4, 8, 1024, 64, True) == 3.5 * f


def test_decode_bytes_by_hand():
    # Q and O: 1 x 1 x 2 x 64 halves each; K and V: 1 x 128 x 1 x 64 halves each; LSE: 2 floats
    want = 2 * (1 * 1 * 2 * 64) * 2 + 2 * (1 * 128 * 1 * 64) * 2 + 4 * 2
    assert bench.decode_bytes(1, 1, 128, 2, 1, 64) == want


def test_traffic_records_cover_every_kernel():
    text = open(bench.os.path.join(bench.ROOT, "profiles", "traffic.txt")).read()
    recs = {}
    for line in text.splitlines():
        if line.startswith("kernel="):
            f = dict(kv.split("=", 1) for kv in line.split())
            recs[f["kernel"]] = f
    assert set(recs) == set(bench.KERNEL_SOURCES)
    for k, f in recs.items():
        assert re.fullmatch(r"[0-9a-f]{16}", f["src"]), k
        rd, wr, tot = (int(f[x]) for x in ("read", "write", "dram_bytes_per_launch"))
        assert rd > 0 and wr >= 0 and abs(rd + wr - tot) <= 1, k


def test_recorded_traffic_needs_the_recorded_sources(monkeypatch):
    # whatever the record says, a different source hash hides it
    monkeypatch.setattr(bench, "source_hash", lambda kernel: "0" * 16)
    for k in bench.KERNEL_SOURCES:
        assert bench.recorded_traffic(k) is None


def test_recorded_traffic_reads_the_matching_line(monkeypatch, tmp_path):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.txt").write_text(
        "# comment line\n"
        "kernel=fa_fwd_kernel src=aaaaaaaaaaaaaaaa dram_bytes_per_launch=100 read=60 write=40\n"
        "kernel=fa_fwd_kernel src=bbbbbbbbbbbbbbbb dram_bytes_per_launch=200 read=150 write=50\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda kernel: "bbbbbbbbbbbbbbbb")
    assert bench.recorded_traffic("fa_fwd_kernel") == 200.0
    assert bench.recorded_traffic("fa_bwd_kernel") is None


@pytest.mark.parametrize("kernel", sorted(bench.KERNEL_SOURCES))
def test_source_hash_covers_the_kernel_sources(kernel, monkeypatch, tmp_path):
    # editing any listed source changes the hash
    import shutil
    for p in bench.KERNEL_SOURCES[kernel]:
        dst = tmp_path / p
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(bench.os.path.join(bench.ROOT, p), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    before = bench.source_hash(kernel)
    last = tmp_path / bench.KERNEL_SOURCES[kernel][-1]
    last.write_text(last.read_text() + "\n// edit\n")
    assert bench.source_hash(kernel) != before


def test_clock_samples_count_only_inside_the_timed_region():
    import datetime
    t0 = datetime.datetime(2026, 1, 1, 12, 0, 0)
    t1 = t0 + datetime.timedelta(seconds=1)
    idle = ["Not Active"] * 4
    capped = ["Not Active"] * 3 + ["Active"]
    rows = [
        ["2026/01/01 11:59:59.900", "0", "2070", "2070", "300", "0x0"] + idle,   # before
        ["2026/01/01 12:00:00.200", "0", "1700", "2070", "1390", "0x4"] + capped,
        ["2026/01/01 12:00:00.600", "0", "1750", "2070", "1395", "0x4"] + capped,
        ["2026/01/01 12:00:00.900", "0", "1800", "2070", "1380", "0x4"] + capped,
        ["2026/01/01 12:00:01.300", "0", "2070", "2070", "350", "0x0"] + idle,   # after
        ["garbled"],
    ]
    c = bench.ClockSampler.summarize(rows, t0, t1)
    assert c["sm_mhz"] == 1750.0 and c["samples"] == 3 and c["samples_outside"] == 2
    assert c["reasons"] == ["sw_power_cap"] and c["sm_max_mhz"] == 2070.0
    # a region with no sample inside says so instead of quoting idle clocks
    c = bench.ClockSampler.summarize(rows[:1], t0, t1)
    assert c["sm_mhz"] is None and c["reasons"] == ["no sample inside the timed region"]
