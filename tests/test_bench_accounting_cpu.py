"""The bench's byte accounting and its traffic record, on the CPU.

The algorithmic bytes behind every `hbm_frac` and `roofline.achieved` are
checked against byte counts worked out by hand from the formats (a Q2S
superblock of 256 weights is 84 bytes, a Q8_0 block of 32 weights 34 bytes;
the router is 256 Q8_0 rows of 4096). The ncu traffic record is reported only
while the kernel sources it was captured on are unchanged."""
import json
import os
import shutil

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_one_token_step_bytes_by_hand():
    # per routed expert: gate and up 2048 rows x 16 superblocks x 84 B each,
    # down 4096 rows x 8 superblocks x 84 B
    routed = 2 * 2048 * 16 * 84 + 4096 * 8 * 84
    assert routed == 8_257_536
    # shared expert (Q8_0): gate and up 2048 rows x 128 blocks x 34 B, down
    # 4096 rows x 64 blocks x 34 B
    shared = 2 * 2048 * 128 * 34 + 4096 * 64 * 34
    assert shared == 26_738_688
    router = 256 * 128 * 34 + 256 * 4
    xy = 3 * 4096 * 4  # x read, y read and written
    assert bench.step_bytes(synth.DS4, 1, 6) == 6 * routed + shared + router + xy == 77_448_192


def test_one_token_gateup_bytes_by_hand():
    weights = 6 * 2 * 2048 * 16 * 84 + 2 * 2048 * 128 * 34
    act_in = 4096 + 4096 // 32 * 4 + 4096 // 16 * 2  # codes, scales, group sums of x
    act_out = 7 * (2048 + 2048 // 32 * 4 + 2048 // 16 * 2)  # SwiGLU codes of 6 + 1 slots
    assert bench.gateup_bytes(synth.DS4, 1, 6) == weights + act_in + act_out == 50_878_976


def test_traffic_record_follows_its_sources(tmp_path, monkeypatch):
    rec_path = os.path.join(ROOT, "profiles", "ds4_decode1_gateup_traffic.json")
    with open(rec_path) as f:
        rec = json.load(f)
    # a copy of the tree's record and sources: reported as recorded
    for rel in ["profiles/ds4_decode1_gateup_traffic.json"] + rec["sources"]:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, rel), dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    got = bench.recorded_traffic()
    assert got == float(rec["dram_bytes_per_launch"])
    # the capture is of the gate/up launch whose algorithmic bytes the bench
    # reports; DRAM bytes at or just above them mean nothing is re-read
    assert 1.0 <= got / bench.gateup_bytes(synth.DS4, 1, 6) < 1.01
    # any change to a kernel source makes the record stale: no traffic
    src = tmp_path / rec["sources"][0]
    src.write_bytes(src.read_bytes() + b"\n")
    assert bench.recorded_traffic() is None
