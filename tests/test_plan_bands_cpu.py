"""The RMSNorm launch heuristic's band table for many rows of 1..2048 16-byte vectors, against the
measured record it is generated from (no GPU: the plan is host code).

The record (csrc/bands/rms_norm_plan_bands.json) holds, per dtype, op and measured width, the score
of every launch the table can name (the worse of steady state and right after a large-shared-
memory kernel, in thousandths of the measured copy peak). The tests check that the library's table
is exactly what the committed rule derives from it, that the library's default plan at every
measured width scores within 2 points of that width's best launch, and that each band code
launches what it names.
"""
import json
import os
import re

import pytest

import bench
from row_wise_rmsnorm_ks_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BANDS = os.path.join(ROOT, "row_wise_rmsnorm_ks_gb300", "csrc", "bands")
RECORD = os.path.join(BANDS, "rms_norm_plan_bands.json")
SOURCE = os.path.join(ROOT, "row_wise_rmsnorm_ks_gb300", "csrc", "ks_abi.cu")
DTYPES = {"bf16": _abi.KS_DTYPE_BF16, "fp16": _abi.KS_DTYPE_F16, "fp32": _abi.KS_DTYPE_F32}
OPS = {"rms_norm": 0, "fused_add_rms_norm": 1}
NO_PF = _abi.KS_PLAN_NO_PREFETCH


@pytest.fixture(scope="module", autouse=True)
def lib():
    try:
        return _abi.load()
    except OSError as e:
        pytest.skip(f"libks.so not built: {e}")


@pytest.fixture(scope="module")
def record():
    with open(RECORD) as f:
        return json.load(f)


def plan(op, rows, hidden, dtype, sms, bps=0):
    st, p = _abi.ks_plan_launch(op, rows, hidden, dtype, True, sms, bps)
    assert st == _abi.KS_SUCCESS, _abi.ks_last_error()
    return p


def code_of(p):
    """The band code of a library plan."""
    if p.kernel == _abi.KS_KERNEL_WARP_ROW:
        c = {8: "E", 16: "H", 32: "W"}[p.team]
        return c.lower() if p.flags & NO_PF else c
    if p.kernel == _abi.KS_KERNEL_CTA_ROW:
        c = {2: "T", 4: "F"}[p.vec_per_thread]
        return c.lower() if p.flags & NO_PF else c
    if p.kernel == _abi.KS_KERNEL_BULK_ROW:
        return "R"
    if p.kernel == _abi.KS_KERNEL_TWOPASS_ROW and p.cluster <= 1:
        return "P"
    raise AssertionError(f"not a band launch: {p.as_dict()}")


def up32(n):
    return -(-n // 32) * 32


def hidden_of(dt, hv):
    return hv * (4 if dt == "fp32" else 8)


def test_record_covers_every_dtype_and_op(record):
    assert set(record["tables"]) == {f"{d}/{o}" for d in DTYPES for o in OPS}
    for key, t in record["tables"].items():
        assert t["hv"] == sorted(t["hv"]) and t["hv"][0] == 1 and t["hv"][-1] == 2048, key
        assert min(t["rows"]) >= 4 * record["sm_count"], key  # every width measured with many rows
        for c in bench.PLAN_BAND_CODES:
            assert len(t[c]) == len(t["hv"]), (key, c)


def test_library_table_is_the_derivation_of_the_record(record):
    src = open(SOURCE).read()
    m = re.search(r"// BEGIN GENERATED ROW BANDS\n(.*?)\n// END GENERATED ROW BANDS", src, re.S)
    assert m, "generated block not found"
    assert m.group(1) == bench.plan_bands_cpp(bench.derive_plan_bands(record))


def test_default_plan_within_two_points_of_the_measured_best(record):
    sms = record["sm_count"]
    worst = []
    for key, t in record["tables"].items():
        dt, op = key.split("/")
        for i, hv in enumerate(t["hv"]):
            p = plan(OPS[op], t["rows"][i], hidden_of(dt, hv), DTYPES[dt], sms)
            c = code_of(p)
            scores = {k: t[k][i] for k in bench.PLAN_BAND_CODES if t[k][i] is not None}
            assert t[c][i] is not None, (key, hv, c)
            loss = max(scores.values()) - t[c][i]
            worst.append((loss, key, hv, c, max(scores, key=scores.get)))
            assert loss <= 20, (key, hv, c, scores)
    # and the derivation's own tolerance holds everywhere: a point of the copy peak
    assert max(worst)[0] <= 10, max(worst)


def test_derivation_rule_on_a_small_record():
    """The rule on a hand-made record: fewest bands within the tolerance, best mean among the
    codes a band allows, the fallback of a two-pass band, the last band to 2048 vectors."""
    n = None
    t = {"hv": [100, 200, 300, 400], "rows": [10 ** 5] * 4,
         #      a narrow warp row, then CTA rows, then the two-pass kernel
         "W": [950, 900, n, n], "w": [940, 800, n, n], "T": [800, 945, 900, 850],
         "t": [700, 940, 930, 800], "F": [600, 700, 800, 880], "f": [600, 700, 800, 870],
         "R": [n, n, n, n], "P": [n, 500, 700, 960]}
    bands = bench.derive_plan_bands({"tables": {"bf16/rms_norm": t}})["bf16/rms_norm"]
    # 100: W (w within a point too); 200: T or t (within a point), not W (45 below);
    # 300: t (T is 30 below); 400: P, falling back to F (the better one-pass code there)
    assert bands == [(100, "W", "W"), (300, "t", "t"), (2048, "P", "F")]


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("op", list(OPS))
def test_every_band_width_gets_a_plan_the_library_accepts(dt, op):
    # what each code launches, for every width of the table, with many rows (4 CTAs per SM)
    for hv in range(1, 2049):
        p = plan(OPS[op], 32768, hidden_of(dt, hv), DTYPES[dt], 152, bps=4)
        c = code_of(p)
        if c in "EeHhWw":
            team = {"E": 8, "H": 16, "W": 32}[c.upper()]
            v = next(v for v in (1, 2, 4, 6, 8) if team * v >= hv)  # the fewest that cover
            assert (p.vec_per_thread, p.team) == (v, team)
            assert p.block == (256 if v <= 4 else 128)
            assert p.rows_per_pass == p.grid * p.block // team
        elif c in "TtFf":
            v = 2 if c in "Tt" else 4
            assert p.vec_per_thread == v and p.block == up32(-(-hv // v))
            assert p.block <= (1024 if v == 2 else 512) and p.team == p.block
        elif c == "R":
            assert p.stages == 2 and p.vec_per_thread == 4 and p.block * 4 >= hv
        else:
            assert p.flags == NO_PF and p.block in (256, 512)
        assert p.grid <= 152 * 4


def test_ring_and_two_pass_need_four_rows_per_sm(record):
    """Bands of the staged ring or the two-pass kernel take their one-pass fallback with fewer
    than 4 rows per SM."""
    bands = bench.derive_plan_bands(record)
    seen = 0
    for key, bl in bands.items():
        dt, op = key.split("/")
        for hv, code, fb in bl:
            many = plan(OPS[op], 4 * 152, hidden_of(dt, hv), DTYPES[dt], 152)
            few = plan(OPS[op], 4 * 152 - 1, hidden_of(dt, hv), DTYPES[dt], 152)
            assert code_of(many) == code, (key, hv)
            assert code_of(few) == fb, (key, hv)
            seen += code in "RP"
    assert seen >= 1  # the record has at least one such band


def test_latency_regime_is_outside_the_table():
    # at most SMs rows: the latency rules (warp rows up to 128 vectors, CTA rows beyond)
    for hv in (1, 8, 64, 128):
        p = plan(0, 152, hv * 8, _abi.KS_DTYPE_BF16, 152)
        assert p.kernel == _abi.KS_KERNEL_WARP_ROW and p.team == 32 and p.block == 32
        assert p.vec_per_thread == next(v for v in (1, 2, 4) if 32 * v >= hv)
    p = plan(0, 152, 1032, _abi.KS_DTYPE_BF16, 152)  # 129 vectors
    assert p.kernel == _abi.KS_KERNEL_CTA_ROW and p.vec_per_thread == 2


def test_team_rows_spread_over_sms():
    """Sub-warp teams hold 4 (8 lanes) or 2 (16 lanes) rows per warp: a CTA takes up to 8 warps
    of rows, but never so many that fewer CTAs than SMs get rows."""
    for rows in (153, 1000, 4864, 10 ** 6):
        for dt, hv in (("bf16", 8), ("bf16", 40), ("fp32", 16)):
            p = plan(0, rows, hidden_of(dt, hv), DTYPES[dt], 152)
            assert p.kernel == _abi.KS_KERNEL_WARP_ROW and p.team in (8, 16)
            per_warp = 32 // p.team
            warps = min(8, max(1, -(-rows // (152 * per_warp))))
            assert p.block == 32 * warps
            assert p.grid == -(-rows // (warps * per_warp))


def test_next_op_tables_are_the_derivation_of_their_record():
    """The Softmax and LayerNorm width bands in the library are exactly what the committed rule
    derives from the committed record of --ops-bands runs."""
    with open(os.path.join(BANDS, "softmax_layer_norm_bands.json")) as f:
        rec = json.load(f)
    src = open(os.path.join(ROOT, "row_wise_rmsnorm_ks_gb300", "csrc", "ks_ops.cu")).read()
    m = re.search(r"// BEGIN GENERATED OP BANDS\n(.*?)\n// END GENERATED OP BANDS", src, re.S)
    assert m, "generated block not found"
    want = "\n".join(bench.bands_cpp(name, bench.derive_bands(rec, op, dts))
                     for name, op, dts in bench.OPS_BAND_TABLES)
    assert m.group(1) == want


def _op_name(p):
    """The ops-bands candidate name of a library Softmax or LayerNorm plan."""
    K = _abi
    n = "n" if p.flags & NO_PF else ""
    if p.kernel == K.KS_KERNEL_WARP_ROW:
        return (f"w{p.vec_per_thread}" if p.team in (0, 32) else f"t{p.team}v{p.vec_per_thread}") + n
    if p.kernel == K.KS_KERNEL_CTA_ROW:
        return f"c{p.vec_per_thread}{n}"
    if p.kernel == K.KS_KERNEL_BULK_ROW:
        return f"r{p.stages}" + ("a" if p.flags & K.KS_PLAN_AFFINE_SMEM else "")
    if p.kernel == K.KS_KERNEL_TWOPASS_ROW:
        return f"x{p.block}"
    raise AssertionError(p.as_dict())


def test_next_op_default_plans_follow_the_record():
    """At every width the record measured with many rows, the library's default Softmax or
    LayerNorm plan is the derived band's launch (the general rule's where the band says so), and
    scores within 2 points of the measured best in its worst dtype."""
    with open(os.path.join(BANDS, "softmax_layer_norm_bands.json")) as f:
        rec = json.load(f)
    codes = {"softmax": _abi.OP_SOFTMAX, "layer_norm": _abi.OP_LAYER_NORM}
    scored = 0
    for _, op, dts in bench.OPS_BAND_TABLES:
        bands = bench.derive_bands(rec, op, dts)
        by_w = {}
        for ln in rec["lines"]:
            if ln["op"] == op and ln["dtype"] in dts:
                by_w.setdefault(ln["hv"], {})[ln["dtype"]] = ln
        for hv, per in by_w.items():
            band = next(b for b in bands if hv <= b[0])
            names = set()
            for dt in per:
                p = _abi.ks_plan_launch(codes[op], 100000, hidden_of(dt, hv), DTYPES[dt], True,
                                        152, 0)[1]
                if band[1] != "g":
                    kind = {_abi.KS_KERNEL_WARP_ROW: "w", _abi.KS_KERNEL_CTA_ROW: "c",
                            _abi.KS_KERNEL_BULK_ROW: "r", _abi.KS_KERNEL_TWOPASS_ROW: "x"}[p.kernel]
                    if kind == "r" and p.flags & _abi.KS_PLAN_AFFINE_SMEM:
                        kind = "R"  # the ring with the weight and bias rows in shared memory
                    assert kind == band[1], (op, dt, hv, band, p.as_dict())
                    if kind in "rR":
                        assert p.stages == band[2], (op, dt, hv, band, p.as_dict())
                names.add(_op_name(p))
            assert len(names) == 1, (op, hv, names)  # one table, one launch for its dtypes
            name = names.pop()

            def score(l2):
                # where the run's default launch was this one, it measured this launch twice
                sc = l2["scores"][name]
                return max(sc, l2["scores"]["default"]) if l2["default_name"] == name else sc

            if all(name in l2["scores"] for l2 in per.values()):
                # scored as the rule scores: each candidate by its worst dtype
                common = set.intersection(*(set(l2["scores"]) for l2 in per.values()))
                best = max(min(l2["scores"][n] for l2 in per.values()) for n in common)
                assert min(score(l2) for l2 in per.values()) >= best - 20, (op, hv, name)
                scored += 1
    assert scored >= 100


WIDE = os.path.join(BANDS, "rms_norm_wide_bands.json")


def test_wide_tables_are_the_derivation_of_their_record():
    with open(WIDE) as f:
        rec = json.load(f)
    src = open(SOURCE).read()
    m = re.search(r"// BEGIN GENERATED WIDE BANDS\n(.*?)\n// END GENERATED WIDE BANDS", src, re.S)
    assert m, "generated block not found"
    assert m.group(1) == bench.wide_bands_cpp(bench.derive_wide_bands(rec))


def _wide_name(p, hv):
    """The plan-sweep candidate name of a library plan for a row of hv vectors."""
    K = _abi
    npf = p.flags & NO_PF
    if p.kernel == K.KS_KERNEL_TWOPASS_ROW and p.cluster < 2:
        return f"t{p.block}u{p.vec_per_thread}" + ("n" if npf else "")
    if p.kernel == K.KS_KERNEL_TWOPASS_ROW:
        sfx = "p" if p.stages == 2 else ("n" if npf else "")
        return f"s{p.cluster}b{p.block}u{p.vec_per_thread}{sfx}"
    if p.kernel == K.KS_KERNEL_CLUSTER_ROW:
        return f"c{p.cluster}"
    if p.kernel == K.KS_KERNEL_BULK_ROW and p.cluster >= 2:
        return (f"b{p.cluster}s{p.stages}" + ("v8" if p.vec_per_thread == 8 else "")
                + ("m" if p.flags & K.KS_PLAN_SMEM_ROWS else ""))
    raise AssertionError(p.as_dict())


def test_wide_default_plans_within_two_points_of_the_measured_best():
    with open(WIDE) as f:
        rec = json.load(f)
    for key, lines in rec["tables"].items():
        dt, op = key.split("/")
        for ln in lines:
            p = plan(OPS[op], ln["rows"], hidden_of(dt, ln["hv"]), DTYPES[dt], rec["sm_count"])
            name = _wide_name(p, ln["hv"])
            sc = {n: v for n, v in ln["scores"].items() if n != "default"}
            assert name in sc, (key, ln["hv"], name)
            assert sc[name] >= max(sc.values()) - 20, (key, ln["hv"], name, max(sc.values()))


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("op", list(OPS))
def test_every_wide_width_gets_a_plan_the_library_accepts(dt, op):
    """Every width of the wide table, with many rows past L2: the plan meets the rules the planned
    entry points check (covered slices, no CTA without vectors, blocks and rings within bounds:
    512 threads, 1024 for the shared-memory rows kernel at 4 vectors; portable clusters of 2..8,
    whole clusters in the grid)."""
    fused = op != "rms_norm"
    for hv in range(2049, 32769, 3):
        rows = max(4 * 152, -(-(160 << 20) // (hv * 32)) + 1)
        p = plan(OPS[op], rows, hidden_of(dt, hv), DTYPES[dt], 152, bps=1)
        C = p.cluster if p.cluster >= 2 else 1
        sl = -(-hv // C)
        assert (C - 1) * sl < hv
        if p.kernel == _abi.KS_KERNEL_TWOPASS_ROW:
            assert p.vec_per_thread in (2, 4) and p.block <= 1024
        else:
            assert p.kernel in (_abi.KS_KERNEL_BULK_ROW, _abi.KS_KERNEL_CLUSTER_ROW), p.as_dict()
            smem_rows = p.kernel == _abi.KS_KERNEL_BULK_ROW and p.flags & _abi.KS_PLAN_SMEM_ROWS
            bound = 1024 if smem_rows and p.vec_per_thread == 4 else 512
            assert 2 <= C <= 8 and p.block <= bound and p.block * p.vec_per_thread >= sl
            assert not smem_rows or (not fused and p.stages >= 2)
            if p.kernel == _abi.KS_KERNEL_BULK_ROW:
                assert p.vec_per_thread == 4 or (p.vec_per_thread == 8 and not fused)
                assert p.smem_bytes == 128 + p.stages * sl * 16 * (2 if fused else 1)
                assert p.smem_bytes <= 226 * 1024
        assert p.grid % C == 0 and p.grid >= C


def _sweep_line(dt, hv, scores):
    line = {"plan_sweep": dt, "op": "rms_norm", "hv": hv, "hidden": hv * 8, "rows": 1000,
            "default_plan": {}, "default": scores["default"]}
    line.update({k: v for k, v in scores.items() if k != "default"})
    return json.dumps(line)


def test_wide_record_keeps_the_last_run_per_width(tmp_path):
    """A width measured by a later run takes that run's lines alone (it may time candidates the
    earlier runs did not); a width measured twice in one run keeps the mean."""
    a, b = tmp_path / "a.log", tmp_path / "b.log"
    a.write_text("\n".join([
        _sweep_line("bf16", 4096, {"default": 0.90, "b4s2": 0.90, "t512u2": 0.80}),
        _sweep_line("bf16", 8192, {"default": 0.80, "b4s2": 0.85, "t512u2": 0.70}),
        _sweep_line("bf16", 8192, {"default": 0.82, "b4s2": 0.87, "t512u2": 0.72}),
    ]) + "\n")
    b.write_text(_sweep_line("bf16", 4096, {"default": 0.91, "b4s2": 0.92, "b4s3m": 0.95}) + "\n")
    rec = bench.wide_bands_record([str(a), str(b)], 152)
    lines = {ln["hv"]: ln["scores"] for ln in rec["tables"]["bf16/rms_norm"]}
    assert lines[4096] == {"default": 910, "b4s2": 920, "b4s3m": 950}  # the later run only
    assert lines[8192] == {"default": 810, "b4s2": 860}  # mean of one run; t512u2 > 5 points behind


def test_wide_derivation_takes_portable_clusters_only():
    """A cluster of 16 is never a band's launch, however it scores: the default launch must not
    depend on the device placing a non-portable cluster."""
    rec = {"tables": {"bf16/rms_norm": [
        {"hv": 4096, "rows": 1000, "scores": {"default": 900, "b16s3m": 990, "b8s2": 920}},
        {"hv": 8192, "rows": 1000, "scores": {"default": 900, "b16s3v8m": 990, "b4s3m": 930}},
    ]}}
    bands = bench.derive_wide_bands(rec)["bf16/rms_norm"]
    assert [n for _, n in bands] == ["b8s2", "b4s3m"]
    assert bands[-1][0] == bench.WIDE_HI


def test_candidate_names_of_default_launches():
    """The record's default-launch names match the band sweep's candidate names for every
    kernel kind, including a ring plan from a run that did not report its stages."""
    name = bench.ops_candidate_name
    assert name({"kernel_name": "warp_row", "vec_per_thread": 4, "flags": 0, "team": 32}, 100) == "w4"
    assert name({"kernel_name": "warp_row", "vec_per_thread": 2, "flags": 1, "team": 8}, 16) == "t8v2n"
    assert name({"kernel_name": "cta_row", "vec_per_thread": 4, "flags": 1, "block": 160}, 640) == "c4n"
    assert name({"kernel_name": "bulk_row", "vec_per_thread": 4, "flags": 4, "stages": 2}, 1280) == "r2a"
    # no stages reported: the ring's own rule, 64 KiB of rows per CTA (2..8 stages)
    assert name({"kernel_name": "bulk_row", "vec_per_thread": 4, "flags": 0}, 1024) == "r4"
    assert name({"kernel_name": "twopass_row", "vec_per_thread": 4, "flags": 0, "block": 256}, 4096) == "x256"


def test_every_wide_band_launch_has_a_gpu_parity_variant():
    """Each kind of launch the wide band tables name (kernel, vectors per thread, rows kept in
    shared memory, two rows in flight) is among the explicit-plan variants the GPU parity test
    runs on ragged shapes, so a re-derived table cannot pick a form no parity case covers."""
    with open(os.path.join(ROOT, "tests", "test_gpu_parity.py")) as f:
        src = f.read()
    variants = set(re.findall(r'"((?:bulk_row|split|splitp|twopass|cluster_row)[a-z0-9_]*)"', src))
    with open(WIDE) as f:
        bands = bench.derive_wide_bands(json.load(f))
    for key, table in bands.items():
        for _, name in table:
            kernel, cluster, block, v, stages, flags = bench.wide_plan_fields(name)
            if kernel == _abi.KS_KERNEL_BULK_ROW:
                smem_rows = bool(flags & _abi.KS_PLAN_SMEM_ROWS)
                want = [x for x in variants if x.startswith("bulk_row_c")
                        and ("_v8" in x) == (v == 8) and x.endswith("_m") == smem_rows]
            elif kernel == _abi.KS_KERNEL_TWOPASS_ROW and cluster >= 2:
                prefix = "splitp_" if stages == 2 else "split_"
                want = [x for x in variants if x.startswith(prefix) and x.endswith(f"_u{v}")]
            elif kernel == _abi.KS_KERNEL_TWOPASS_ROW:
                want = [x for x in variants if x.startswith("twopass_") and x.endswith(f"_u{v}")]
            else:
                want = [x for x in variants if x.startswith("cluster_row")]
            assert want, (key, name)
