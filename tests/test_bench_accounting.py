"""bench.py's algorithmic work per call, on CPU: the per-unit byte and flop
counts behind every reported roofline fraction, against the totals they must
give on the serving workloads, and the peak lookup's fallback."""
import json

import bench
import workloads as W

KIB = 1024
TOKEN_HEAD = 4 * 128 * 2 + 2 + 128 * 2  # q, k, v, raw gate (bf16) + raw beta + o (bf16)


def test_per_unit_bytes():
    assert TOKEN_HEAD == 1282
    # decode: the state read and written once, one token's activations and output
    assert bench.decode_work(1, 1) == 2 * 64 * KIB + 1282
    assert bench.decode_work(1, 1, sb=32 * KIB) == 2 * 32 * KIB + 1282  # 16-bit pool
    # verify: the checkpoint once; per position the activations, the bf16 output, fp32 u
    # and the bf16 key / raw-gate record
    assert bench.verify_work(1, 7, 1) == 64 * KIB + 7 * (1026 + 256 + 512 + 512)
    # commit: requests with a > 0 read the checkpoint and write the state and read a
    # records; every request reads 2K ids and writes its length and next token
    K = 7
    ids = 2 * K * 4 + 2 * 4
    assert bench.commit_work([0], 1, K) == ids
    assert bench.commit_work([3, 0], 2, K) == 2 * ids + 2 * (128 * KIB + 3 * (512 + 512))


def test_prefill_bytes_and_flops():
    byts, flops = bench.prefill_work([64, 100], H=2, M=1)
    assert byts == 164 * 2 * TOKEN_HEAD + 2 * 2 * 3 * 64 * KIB  # S_0, S_final, 1 snapshot
    assert flops == 164 * 2 * (10 * 64 * 128 + 6 * 128 * 128 + 64 * 64 / 3)


def test_workload_totals():
    # 256 requests x 32 heads of decode: 1.084 GB per call
    assert bench.decode_work(256, 32) == 1_084_243_968
    # 64 requests x K = 7 x 32 heads of verify: 167 MB per call
    assert bench.verify_work(64, 7, 32) == 167_276_544
    # the batched prefill: 8 sequences, 32 heads, one snapshot each
    lengths = W.batched_prefill_lengths()
    byts, _ = bench.prefill_work(lengths, 32, 1)
    assert byts == sum(lengths) * 32 * 1282 + 8 * 32 * 3 * 64 * KIB
    assert 1.6e9 < byts < 1.9e9
    # the long prefill: 131072 tokens x 16 heads, 31 snapshots + S_0 + S_final
    byts4, _ = bench.prefill_work([131072], 16, 31)
    assert byts4 == 131072 * 16 * 1282 + 16 * 33 * 64 * KIB


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    hbm, tc, kind = bench.load_peaks()
    assert (hbm, tc, kind) == (6800.0, 1900.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6790.3,
                                                               "bf16_tflops": 1890.2}))
    assert bench.load_peaks() == (6790.3, 1890.2, "measured")


def test_traffic_stamp_belongs_to_the_kernel_source():
    # the DRAM traffic figure is charged only while the prefill source is the one it was
    # captured on; the committed stamp must name the committed source
    th = 41460 * 32
    t = bench.prefill_traffic(th)
    assert t is not None
    assert abs(t - bench.PREFILL_TRAFFIC["bytes_per_token_head"] * th) < 1.0
    # between the algorithmic bytes and ten times them
    assert 1282 < bench.PREFILL_TRAFFIC["bytes_per_token_head"] < 12820


def test_traffic_is_null_once_the_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "prefill_2p.cu"
    src.write_text("// another kernel source\n")
    monkeypatch.setitem(bench.PREFILL_TRAFFIC, "source", str(src))
    assert bench.prefill_traffic(1000) is None
    monkeypatch.setitem(bench.PREFILL_TRAFFIC, "source", str(tmp_path / "missing.cu"))
    assert bench.prefill_traffic(1000) is None
