"""The host arithmetic behind bench.py's roofline figures: algorithmic bytes
and FLOPs per decode row, worked by hand for the batch-32 x 32k workload
(ratio 4, budget 2048, H_I 64 x d_I 128, Hq 32 / Hkv 4, D 128)."""
import pytest

import bench
from indexer_selected_sparse_gb300 import synth as S


@pytest.fixture(scope="module")
def sh():
    return S.workload(2).shapes


def test_decode_row_at_32k(sh):
    # V = 32769 visible tokens: 8192 complete blocks, 512 of them selected plus a tail of 1
    w = bench.row_work(sh, 32769)
    assert (w["n_blk"], w["n_tok"]) == (8192, 2049)
    # keys 8192 x 128 x 2 B, the row's index queries 64 x 128 x 2 B, its 64 fp32 weights
    assert w["score_bytes"] == 2_097_152 + 16_384 + 256 == 2_113_792
    # K and V of 2049 tokens x 4 heads x 128 x 2 B, then q and o (32 x 128 x 2 B each)
    assert w["attn_bytes"] == 2049 * 4 * 128 * 2 * 2 + 2 * 32 * 128 * 2 == 4_212_736
    # the appended token: K and V rows (4 x 128 x 2 B each) and its raw index key (128 x 2 B)
    assert w["append_bytes"] == 2_304
    assert w["score_flops"] == 2 * 64 * 128 * 8192
    assert w["attn_flops"] == 4 * 32 * 128 * 2049
    # a step of 32 rows at that prefix
    step = 32 * (w["score_bytes"] + w["attn_bytes"] + w["append_bytes"])
    assert step == 202_522_624


def test_mx_planes_count_their_own_key_bytes(sh):
    assert bench.key_bytes(sh, "bf16") == 256
    assert bench.key_bytes(sh, "mxfp8") == 128 + 4      # E4M3 elements + one scale byte per 32
    assert bench.key_bytes(sh, "mxfp4") == 64 + 4       # E2M1 pairs + one scale byte per 32
    for fmt, kb in (("mxfp8", 132), ("mxfp4", 68)):
        w = bench.row_work(sh, 32769, fmt)
        assert w["score_bytes"] == 8192 * kb + 16_384 + 256
        assert w["attn_bytes"] == bench.row_work(sh, 32769)["attn_bytes"]


def test_rows_at_the_inert_bound_score_nothing(sh):
    # up to budget + ratio - 1 = 2051 visible tokens every block is selected: no scoring
    w = bench.row_work(sh, 2051)
    assert w["score_bytes"] == 0 and w["score_flops"] == 0 and w["n_tok"] == 2051
    w = bench.row_work(sh, 2052)   # one block past it: 513 blocks scored, 512 kept, no tail
    assert w["score_bytes"] == 513 * 256 + 16_384 + 256 and w["n_tok"] == 2048
    tot = bench.sum_work(sh, [2051, 2052])
    assert tot["n_tok"] == 2051 + 2048


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the CPU oracle arm) on a tiny run: one JSON
    line with the contract's keys; a rank other than 0 prints nothing."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "4", "--warmup", "3"]
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "rows/s"
    assert d["value"] > 0 and d["steps"] == 4 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    env1 = dict(env, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res1 = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env1)
    assert res1.returncode == 0 and res1.stdout.strip() == ""


def test_clock_summary_keeps_the_timed_window_and_its_reasons():
    """The clock record is parsed from nvidia-smi's CSV lines: only samples
    inside the timed window count; a reason counts when it is Active there."""
    from datetime import datetime
    cs = bench.ClockSampler.__new__(bench.ClockSampler)   # no nvidia-smi process
    cs.proc = None
    t0 = datetime(2026, 1, 5, 12, 0, 0).timestamp()

    def line(dt, sm, reasons=("Not Active",) * 4):
        ts = datetime.fromtimestamp(t0 + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return f"{ts}, 0, {sm}, 2070, 905.25, 0x0000000000000004, " + ", ".join(reasons)
    cs.lines = [line(-1.0, 800, ("Active",) * 4),                          # before the window
                line(0.1, 2070), line(0.2, 2055),
                line(0.3, 2070, ("Not Active", "Not Active", "Not Active", "Active")),
                line(5.0, 600, ("Active",) * 4)]                            # after it
    s = cs.summary(t0, t0 + 1.0)
    assert s["samples"] == 3 and s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    cs.lines = [line(0.5, 1900, ("Not Active", "Active", "Not Active", "Not Active"))]
    assert cs.summary(t0, t0 + 1.0)["reasons"] == ["hw_thermal_slowdown"]
    cs.lines = ["garbage", line(3.0, 2000)]
    assert cs.summary(t0, t0 + 1.0)["samples"] == 0


def test_packed_step_inputs_are_aligned_disjoint_views():
    import torch
    ts = [torch.randn(3, 5).to(torch.bfloat16), torch.randn(7), torch.arange(10, dtype=torch.int32).view(2, 5),
          torch.randn(32, 4, 128).to(torch.bfloat16)]
    buf, views = bench.packed(torch, ts, "cpu")
    assert buf.dtype == torch.uint8 and buf.numel() == 256 + 256 + 256 + 32 * 4 * 128 * 2
    for v, t in zip(views, ts):
        assert v.shape == t.shape and v.dtype == t.dtype and v.is_contiguous()
        assert (v.data_ptr() - buf.data_ptr()) % 256 == 0       # the C ABI wants 16-byte aligned inputs
        v.copy_(t)
    for v, t in zip(views, ts):                                  # nothing overwrote another view
        assert torch.equal(v, t)


def test_pool_rate_ignores_worker_start_skew():
    import bench
    # two workers, 10 rows each at 0.1 s per row, the second starting 5 s later:
    # 20 rows/s in all, whatever the skew
    w1 = [(0.1 * i, 0.1 * (i + 1)) for i in range(10)]
    w2 = [(5 + 0.1 * i, 5 + 0.1 * (i + 1)) for i in range(10)]
    assert abs(bench.pool_rate([w1, w2]) - 20.0) < 1e-9


def test_token_count_is_the_union_of_the_rows_sets():
    import bench
    # ratio 4: row A (V = 10: blocks 0, 1 complete, tail 8..9) selected block 1;
    # row B (V = 13: 3 blocks, tail 12) selected blocks 1 and 2, -1 padded
    assert bench.token_count([[1, -1], [1, 2]], [10, 13], 4) == len(set(range(4, 8)) | {8, 9} | set(range(4, 12)) | {12})
