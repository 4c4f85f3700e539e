"""bench.py's host logic on the CPU: arguments, per-op algorithmic bytes, the
traffic record check, and the multi-rank path (two gloo ranks: barrier and
max over ranks; the reference arm runs on rank 0 only)."""

import json
import os
import socket

import pytest

import bench


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_defaults_and_validation():
    a = bench.parse_args([])
    assert a.op == "scan_exclusive" and a.gpus == 1 and a.warmup >= 3 and a.impl == "ours"
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.parse_args(["--steps", "0"])


def test_algorithmic_bytes_per_op():
    n28, n26, n27, n25 = 1 << 28, 1 << 26, 1 << 27, 1 << 25
    assert bench.make_op(bench.parse_args([])).algorithmic_bytes() == 8 * n28
    assert bench.make_op(bench.parse_args(["--op", "scan_inclusive"])).algorithmic_bytes() == 8 * n28
    seg = bench.make_op(bench.parse_args(["--op", "segscan"]))
    seg.nseg = 5
    assert seg.algorithmic_bytes() == 12 * n26
    red = bench.make_op(bench.parse_args(["--op", "segreduce", "--heads", "regular4"]))
    red.nseg = n26 // 4
    assert red.algorithmic_bytes() == 8 * n26 + 4 * (n26 // 4) + 4
    seg8 = bench.make_op(bench.parse_args(["--op", "segscan", "--u8heads"]))
    seg8.nseg = 5
    assert seg8.algorithmic_bytes() == 9 * n26
    assert bench.make_op(bench.parse_args(["--op", "compact"])).algorithmic_bytes() == 12 * n27 + 4
    assert bench.make_op(bench.parse_args(["--op", "radix"])).algorithmic_bytes() == 60 * n25
    assert bench.make_op(bench.parse_args(["--op", "radix", "--ties"])).algorithmic_bytes() == 12 * n25
    assert bench.make_op(bench.parse_args(["--op", "radix", "--sort", "pairs"])).algorithmic_bytes() == 64 * n25
    assert bench.make_op(bench.parse_args(["--op", "radix", "--sort", "keys"])).algorithmic_bytes() == 36 * n25
    assert bench.make_op(bench.parse_args(["--op", "radix", "--sort", "keys", "--ties"])).algorithmic_bytes() == 12 * n25
    cv = bench.make_op(bench.parse_args(["--op", "compact", "--project", "values", "--log2n", "12"]))
    f = cv.host_inputs()["flags"]
    assert cv.kept == int((f != 0).sum()) and cv.algorithmic_bytes() == 8 * (1 << 12) + 4 * cv.kept + 4
    cz = bench.make_op(bench.parse_args(["--op", "compact", "--project", "nonzero", "--log2n", "12"]))
    v = cz.host_inputs()["values"]
    assert cz.kept == int((v != 0).sum()) and cz.algorithmic_bytes() == 4 * (1 << 12) + 4 * cz.kept + 4
    runs = bench.make_op(bench.parse_args(["--op", "runs", "--log2n", "12"]))
    c = runs.host_inputs()["counts"]
    assert runs.entries == int(c.sum()) and runs.algorithmic_bytes() == 4 * (1 << 12) + 4 * runs.entries
    assert bench.make_op(bench.parse_args(["--op", "scan64"])).algorithmic_bytes() == 16 * n27
    assert bench.make_op(bench.parse_args(["--log2n", "20"])).n == 1 << 20


def test_traffic_record_must_match_source_and_size(tmp_path, monkeypatch):
    op = bench.make_op(bench.parse_args([]))
    f = tmp_path / "t.json"
    monkeypatch.setattr(type(op), "traffic_file", property(lambda self: f))
    assert bench.load_traffic(op) is None  # no record
    rec = {"source_hash": bench.source_hash(op.kernel_sources), "scaled_to_n": op.n, "dram_bytes_per_launch": 123.0}
    f.write_text(json.dumps(rec))
    assert bench.load_traffic(op) == 123.0
    f.write_text(json.dumps({**rec, "source_hash": "stale"}))
    assert bench.load_traffic(op) is None  # the kernel changed since the capture
    f.write_text(json.dumps({**rec, "scaled_to_n": op.n // 2}))
    assert bench.load_traffic(op) is None


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(1.5 + rank, world)
        ref = bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3",
                                                    "--log2n", "12"]), rank)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as fh:
            json.dump({"max": got, "ref": None if ref is None else ref["impl"]}, fh)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_max_and_reference_on_rank0(tmp_path):
    import torch.multiprocessing as mp

    world = 2
    mp.spawn(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    r0 = json.loads((tmp_path / "rank0.json").read_text())
    r1 = json.loads((tmp_path / "rank1.json").read_text())
    assert r0["max"] == r1["max"] == 2.5  # the slowest rank's time
    assert r0["ref"] == "reference" and r1["ref"] is None


def test_scan_under_several_ranks_is_one_sharded_scan():
    args = bench.parse_args([])
    args.world, args.rank = 4, 2
    op = bench.make_op(args)
    assert op.sharded and op.is_marked() and op.launches_per_step == 3
    assert "4 x 2^28" in op.workload()
    # rank 2's shard continues the seed-2 stream where rank 1's ends
    from u32_prefix_scan_gb300 import inputs

    args.log2n = 10
    op = bench.make_op(args)
    whole = inputs.splitmix_u32(2, 0, 4 << 10)
    assert (op.host_inputs()["data"] == whole[2 << 10: 3 << 10]).all()
    args.world, args.rank = 1, 0
    assert not bench.make_op(args).sharded


def test_compaction_under_several_ranks_is_one_sharded_compaction():
    args = bench.parse_args(["--op", "compact", "--log2n", "10"])
    args.world, args.rank = 2, 1
    op = bench.make_op(args)
    assert op.sharded and op.is_marked() and op.launches_per_step == 4
    assert "2 x 2^10" in op.workload()
    from u32_prefix_scan_gb300 import inputs

    whole = inputs.compact_flags(2 << 10, 4, 0.1)
    assert (op.host_inputs()["flags"] == whole[1 << 10:]).all()


def test_segmented_scan_under_several_ranks_is_one_sharded_scan():
    from u32_prefix_scan_gb300 import inputs

    args = bench.parse_args(["--op", "segscan", "--log2n", "10"])
    args.world, args.rank = 3, 2
    op = bench.make_op(args)
    assert op.sharded and op.is_marked()
    h = op.host_inputs()
    whole_f = inputs.segment_heads_geometric(3 << 10, 3)
    assert (h["flags"] == whole_f[2 << 10:]).all() and (h["data"] == inputs.splitmix_u32(3, 0, 3 << 10)[2 << 10:]).all()
    args = bench.parse_args(["--op", "segscan_sums"])
    args.world, args.rank = 2, 0
    assert not bench.make_op(args).sharded  # only the plain segmented scan shards


def test_parse_cpulist_reads_sysfs_ranges():
    import bench

    assert bench.parse_cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench.parse_cpulist("5") == {5}
    assert bench.parse_cpulist("") == set()


def test_other_rows_cover_every_primitive_workload():
    """The default line's other rows: the segmented forms at both segment
    mixes, compaction at both keep rates, the radix permutation on both key
    sets, each at its workload's full size with its own byte count."""
    seen = set()
    for argv in bench.ROW_WORKLOADS:
        a = bench.parse_args(argv)
        a.world, a.rank = 1, 0
        op = bench.make_op(a)
        assert op.n == 1 << op.log2n and not getattr(op, "sharded", False)
        seen.add(op.name)
    assert seen == {"segscan_geometric", "segscan_sums_geometric", "segscan_sums_regular4", "segreduce_geometric",
                    "segreduce_regular4", "compact_p0.1", "compact_p0.9", "radix_sort_perm_u32",
                    "radix_sort_perm_u32_ties"}
    assert not bench.parse_args([]).no_rows and bench.parse_args(["--no-rows"]).no_rows
