"""bench.py's roofline `traffic` field comes from the committed ncu summaries under
profiles/: each summary carries the hash of the kernel sources it was captured on and
the DRAM bytes per full-size launch of the workloads it was scaled to.  On CPU: every
summary bench.py names exists and states its capture command; where its hash matches
the current sources, its figures are plausible (at least the compulsory bytes of inputs
and outputs), and otherwise the field is null; the lookup is null for a workload the
summary does not list, and turns null once a source changes."""
import hashlib
import os
import re

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# workloads the summaries are scaled to, with their compulsory DRAM bytes (inputs read and
# outputs written once, bf16 with fp32 lse): the figure must not be below them
COMPULSORY = {
    ("fwd", 128, "fwd_b8h32_t4096_d128_causal"): 8 * 32 * 4096 * (4 * 128 * 2 + 4),
    ("fwd", 256, "fwd_b1h24_t32768_d256_causal"): 24 * 32768 * (4 * 256 * 2 + 4),
    ("fwd", 64, "fwdbwd_b1h16_t65536_d64"): 16 * 65536 * (4 * 64 * 2 + 4),
    ("bwd_main", 128, "bwd_b8h32_t4096_d128_causal"): 8 * 32 * 4096 * 6 * 128 * 2,
    ("bwd_main", 64, "fwdbwd_b1h16_t65536_d64"): 16 * 65536 * 6 * 64 * 2,
}


def _sha(srcs):
    h = hashlib.sha256()
    for f in srcs:
        with open(os.path.join(ROOT, "exact_io_aware_05_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _current(kernel, d):
    path, srcs = bench.PROFILE_OF[(kernel, d)]
    with open(os.path.join(ROOT, path)) as fh:
        text = fh.read()
    m = re.search(r"source-sha256-16:\s*([0-9a-f]{16})", text)
    assert m, path
    return m.group(1) == _sha(srcs)


def test_summaries_exist_and_state_their_command():
    for (kernel, d), (path, srcs) in bench.PROFILE_OF.items():
        with open(os.path.join(ROOT, path)) as fh:
            text = fh.read()
        assert re.search(r"source-sha256-16:\s*[0-9a-f]{16}", text), path
        assert "ncu " in text and "--clock-control none" in text, path


def test_traffic_figures_are_plausible_or_null():
    for (kernel, d, key), floor in COMPULSORY.items():
        v = bench.ncu_traffic(kernel, d, key)
        if not _current(kernel, d):
            assert v is None, (kernel, d, key)
            continue
        assert v is not None, (kernel, d, key)
        assert floor <= v <= 8 * floor, (kernel, d, key, v, floor)
    # the headline's figures are those of its two workloads
    assert bench.ncu_traffic("fwd") == bench.ncu_traffic("fwd", 128, "fwd_b8h32_t4096_d128_causal")
    assert bench.ncu_traffic("bwd_main") == bench.ncu_traffic("bwd_main", 128, "bwd_b8h32_t4096_d128_causal")


def test_traffic_is_null_where_unknown(monkeypatch, tmp_path):
    assert bench.ncu_traffic("fwd", 128, "no_such_workload") is None
    assert bench.ncu_traffic("fwd", 32) is None
    # a summary captured on other sources gives no figure
    path, srcs = bench.PROFILE_OF[("fwd", 128)]
    with open(os.path.join(ROOT, path)) as fh:
        text = fh.read()
    stale = tmp_path / "stale.md"
    stale.write_text(re.sub(r"(source-sha256-16:\s*)[0-9a-f]{16}", r"\g<1>0000000000000000", text))
    monkeypatch.setitem(bench.PROFILE_OF, ("fwd", 128), (str(stale), srcs))
    assert bench.ncu_traffic("fwd") is None
