"""Host-side logic of bench.py on CPU: the byte model against the pages' printed figures
(tests/golden/pages_bandwidth.txt), and the multi-rank path (max over ranks, whole-job
aggregate, independent per-rank batches) on two gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "pages_bandwidth.txt")


def golden_rows():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        f = [c.strip() for c in line.split("|")]
        out.append(dict(source=f[0], op=f[1], rows=int(f[2]), hidden=int(f[3]), e=int(f[4]),
                        ms=float(f[5]), digits=int(f[6]), gbs=float(f[7]),
                        expect=f[8].split()[0]))
    return out


@pytest.mark.parametrize("row", golden_rows(), ids=lambda r: r["source"][:40])
def test_byte_model_against_printed_figures(row):
    nbytes = bench.algorithmic_bytes(row["op"], row["rows"], row["hidden"], row["e"])
    half = 0.5 * 10.0 ** -row["digits"]
    lo_ms, hi_ms = row["ms"] - half, row["ms"] + half
    implied_ms = nbytes / (row["gbs"] * 1e9) * 1e3
    consistent = lo_ms <= implied_ms <= hi_ms
    assert consistent == (row["expect"] == "consistent"), (implied_ms, lo_ms, hi_ms)


def test_byte_model_values():
    # the large prefill step: 1,073,758,208 B plain, 2,147,500,032 B fused
    assert bench.algorithmic_bytes("rms_norm", 32768, 8192, 2) == 1073758208
    assert bench.algorithmic_bytes("fused_add_rms_norm", 32768, 8192, 2) == 2147500032
    assert bench.algorithmic_bytes("fused_add_rms_norm", 4, 1536, 2) == 52224


def test_whole_job_aggregate():
    assert bench.whole_job_gbs(1, 10 ** 9, 1000, 1000.0) == pytest.approx(1000.0)
    assert bench.whole_job_gbs(4, 10 ** 9, 1000, 1000.0) == pytest.approx(4000.0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
        worst = bench.max_over_ranks(local_ms)
        seeds = [torch.tensor([bench.rank_seed(1234, rank)]) for _ in range(world)]
        dist.all_gather(seeds, torch.tensor([bench.rank_seed(1234, rank)]))
        dist.barrier()
        q.put((rank, worst, [int(s) for s in seeds]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_draw_independent_batches():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, seeds in results:
        assert worst == 15.0
        assert len(set(seeds)) == world  # every rank draws its own batch


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_kernel_hash_ignores_comments_and_layout():
    """The recorded DRAM traffic stays valid across comment edits, not across code edits."""
    src = 'int f(int a) { // sum\n  return a + 1; /* one */\n}\nconst char *s = "// kept";\n'
    same = '/* header */\nint f(int a)   {\n\n  return a + 1;\n}  // trailing\nconst char *s = "// kept";'
    changed = 'int f(int a) { return a + 2; }\nconst char *s = "// kept";'
    assert bench.code_only(src) == bench.code_only(same)
    assert bench.code_only(src) != bench.code_only(changed)
    assert '"// kept"' in bench.code_only(src)



def test_recorded_traffic_only_for_the_recorded_shape():
    """The committed ncu bytes are per launch of the full workload: a smaller --rows/--hidden
    case reports no traffic, and its config names its own shape."""
    assert bench.recorded_traffic("fused_add_rms_norm", 8192, 8192) is None
    assert bench.recorded_traffic("rms_norm", bench.FULL_ROWS, 4096) is None
    assert "[8192,8192]" in bench.workload(8192, 8192) and "128 MiB" in bench.workload(8192, 8192)
    assert bench.workload(bench.FULL_ROWS, bench.FULL_HIDDEN).startswith("large prefill bf16")
    l2 = 126 << 20
    assert "larger than L2" in bench.l2_note(bench.FULL_ROWS, bench.FULL_HIDDEN, l2)
    assert "not a bench figure" in bench.l2_note(1024, 1024, l2)


def test_recorded_traffic_follows_the_sources(tmp_path, monkeypatch):
    """The DRAM-traffic record is data: it is used only while the kernel and plan sources hash
    to the value it was taken on, only for the shape it records, and only while the library
    picks the recorded plan for that shape."""
    import json
    from row_wise_rmsnorm_ks_gb300 import _abi
    try:
        _abi.load()
    except OSError as e:
        pytest.skip(f"libks.so not built: {e}")
    R, H = bench.FULL_ROWS, bench.FULL_HIDDEN
    now = _abi.ks_plan_launch(1, R, H, _abi.KS_DTYPE_BF16, True, 152, 0)[1]
    plan = {k: getattr(now, k) for k in bench.PLAN_FIELDS}
    rec = {"sources_sha": bench.kernel_source_sha(),
           "launches": {"fused_add_rms_norm": {"shape": [R, H], "plan": plan,
                                               "dram_read_bytes": 1000,
                                               "dram_write_bytes": 900}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_RECORD", str(path))
    assert bench.recorded_traffic("fused_add_rms_norm", R, H, now) == 1900
    assert bench.recorded_traffic("fused_add_rms_norm", R, H) is None  # no plan to check
    other = _abi.ks_plan_launch(1, R, H, _abi.KS_DTYPE_BF16, True, 152, 0)[1]
    other.vec_per_thread = 4
    assert bench.recorded_traffic("fused_add_rms_norm", R, H, other) is None
    assert bench.recorded_traffic("rms_norm", R, H, now) is None
    assert bench.recorded_traffic("fused_add_rms_norm", 4096, H, now) is None
    rec["sources_sha"] = "0" * 16
    path.write_text(json.dumps(rec))
    assert bench.recorded_traffic("fused_add_rms_norm", R, H, now) is None
    # the plan code is part of the hash, but not its generated band table
    assert any(s.endswith("ks_abi.cu") for s in bench.KERNEL_SOURCES)
    src = "int a;\n// BEGIN GENERATED ROW BANDS\nint b;\n// END GENERATED ROW BANDS\nint c;\n"
    assert bench.code_only(bench.GENERATED_BANDS.sub("", src)) == "int a; int c;"


def test_committed_traffic_record_is_current():
    """The committed record matches the current sources and the library's headline plans, so
    the bench line carries its traffic."""
    from row_wise_rmsnorm_ks_gb300 import _abi
    try:
        _abi.load()
    except OSError as e:
        pytest.skip(f"libks.so not built: {e}")
    R, H = bench.FULL_ROWS, bench.FULL_HIDDEN
    for op, code in (("rms_norm", 0), ("fused_add_rms_norm", 1)):
        now = _abi.ks_plan_launch(code, R, H, _abi.KS_DTYPE_BF16, True, 152, 0)[1]
        assert bench.recorded_traffic(op, R, H, now) is not None, op


def test_host_cpu_model_names_the_cpu():
    import bench
    name = bench.host_cpu_model()
    assert isinstance(name, str) and name.strip()


def test_oracle_all_cores_figure():
    """The all-cores CPU figure runs the oracle on row slices in threads; it must cover the
    requested rows and report the threads it used."""
    import bench
    from row_wise_rmsnorm_ks_gb300 import synth
    R, H = 40, 256
    x = synth.cast(synth.normal_np((R, H), 5), "bf16")
    r = synth.cast(synth.normal_np((R, H), 6), "bf16")
    w = synth.weight(H, "bf16")
    d = bench.oracle_all_cores({"x": x, "xf": x.clone(), "r": r, "w": w}, R, H, 1e-5)
    assert d["value"] > 0 and 1 <= d["cores"] <= min(R, os.cpu_count())
    assert d["sample"].startswith(f"first {R} rows")


def test_kernel_times_table_joins_the_launch_list(tmp_path):
    """The kernel-times summary pairs each case with its own launches from an ncu launch list
    (this library's kernels only, in order; the untimed first launch of each case left out) and
    refuses a list from another command."""
    import json
    hdr = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream",'
           '"Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit",'
           '"Metric Value"\n')

    def row(i, name, ns):
        return (f'"{i}","1","python3","h","{name}","1","7","(256, 1, 1)","(152, 1, 1)","0","10.3",'
                f'"Command line profiler metrics","gpu__time_duration.sum","ns","{ns}"\n')
    csv_text = "==PROF== Connected\n" + hdr
    csv_text += row(0, "void at::native::reduce_kernel<...>", 500)  # not this library's
    times = [9000, 2000, 2200, 2100, 30000, 10000, 10400, 10200]
    for i, ns in enumerate(times):
        csv_text += row(i + 1, "void rows_vec_kernel<bf16, 4, 0, 0, 0>(RowArgs)", ns)
    (tmp_path / "l.csv").write_text(csv_text)
    plan = {"kernel_name": "cta_row", "cluster": 0}
    cases = [{"kernel_times": "small", "dtype": "bf16", "op": "rms_norm", "rows": 128,
              "hidden": 1024, "launches": 4, "event_p50_us": 6.8, "event_frac_of_peak": 0.01,
              "bytes": 526336, "plan": plan},
             {"kernel_times": "fused", "dtype": "bf16", "op": "fused_add_rms_norm", "rows": 512,
              "hidden": 4096, "launches": 4, "event_p50_us": 12.0, "event_frac_of_peak": 0.2,
              "bytes": 16785408, "plan": plan}]
    (tmp_path / "k.jsonl").write_text("".join(json.dumps(c) + "\n" for c in cases))
    table = bench.kernel_times_table(str(tmp_path / "k.jsonl"), str(tmp_path / "l.csv"))
    lines = table.splitlines()
    assert len(lines) == 4
    assert "| 2.10 | 6.80 |" in lines[2] and "| 10.20 | 12.00 |" in lines[3]
    (tmp_path / "k.jsonl").write_text(json.dumps(cases[0]) + "\n")
    with pytest.raises(SystemExit):
        bench.kernel_times_table(str(tmp_path / "k.jsonl"), str(tmp_path / "l.csv"))
