"""bench.py's link between the committed DRAM counters and the kernel sources
(CPU only): a record counts only while the kernel code it was taken on is
unchanged, else the bench line reports null traffic; comments do not count
as code."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_comments_and_blank_lines_do_not_change_the_code():
    a = "int f(int x) {\n  return x + 1;  // add one\n}\n"
    b = "/* a comment\n   over lines */\nint f(int x) {\n\n  return x + 1;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)


def test_a_code_edit_changes_the_code():
    a = "int f(int x) { return x + 1; }  // one\n"
    b = "int f(int x) { return x + 2; }  // one\n"
    assert bench._code_only(a) != bench._code_only(b)


def test_a_record_is_used_only_while_its_kernel_code_is_unchanged():
    """A committed record gives the bench line its traffic only while the
    kernel code it was taken on is unchanged; a stale record gives null."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        records = json.load(f)
    assert records
    for name, rec in records.items():
        sources = bench.BWD_SOURCES if name.endswith("_bwd") else None
        current = rec["kernel_sha"] == bench._kernel_sha(sources)
        got = bench._traffic(name, sources)
        assert got == (rec["bytes_per_launch"] if current else None), name
        assert os.path.exists(os.path.join(ROOT, rec["source"].split(" ")[0].split(":")[0]))


def test_each_line_names_the_workload_it_measured():
    """The headline forward keeps the benchmark's own metric name; every other
    forward or backward line names its own shape, dtype and mask."""
    import synthetic
    assert bench.metric_for(synthetic.HEADLINE) == bench.METRIC
    names = set()
    for w in synthetic.WORKLOADS + synthetic.FP8_WORKLOADS:
        for pass_ in ("fwd", "bwd"):
            m = bench.metric_for(w, pass_)
            names.add(m)
            assert ("bwd" in m) == (pass_ == "bwd")
            if not (w is synthetic.HEADLINE and pass_ == "fwd"):
                assert w.describe() in m
    assert len(names) == 2 * len(synthetic.WORKLOADS + synthetic.FP8_WORKLOADS)


def test_default_run_covers_every_named_configuration():
    """The default bench line carries, besides the headline, a record for each
    of the other named forward workloads and the headline's backward pass."""
    import synthetic
    keys = {n if p == "fwd" else n + "_bwd" for n, p in bench.EXTRA_CONFIGS}
    want = {w.name for w in synthetic.WORKLOADS + synthetic.FP8_WORKLOADS} - {
        synthetic.HEADLINE.name}
    assert want <= keys and synthetic.HEADLINE.name + "_bwd" in keys
