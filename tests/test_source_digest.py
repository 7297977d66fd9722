"""The recorded DRAM traffic of a workload's dominant kernel goes stale with a
change of that kernel's code, and only then (no GPU)."""
import os
import shutil

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "segmented_gathered_rank_gb300",
                    "csrc")


def _copy(tmp_path):
    d = tmp_path / "csrc"
    shutil.copytree(CSRC, d)
    return str(d)


def _edit(folder, name, old, new):
    p = os.path.join(folder, name)
    with open(p, encoding="utf-8") as f:
        text = f.read()
    with open(p, "w", encoding="utf-8") as f:
        f.write(text.replace(old, new, 1) if old else text + new)


def test_digest_ignores_comments_and_blank_lines(tmp_path):
    d = _copy(tmp_path)
    before = {w: bench.source_digest(w, d) for w in bench.KERNEL_SOURCES}
    _edit(d, "bgmv.cu", None, "\n// a new comment\n\n/* and a block\n comment */\n")
    _edit(d, "sgmv.cu", None, "\n\n// trailing note\n")
    assert {w: bench.source_digest(w, d) for w in bench.KERNEL_SOURCES} == before


def test_code_change_stales_only_the_workloads_built_from_that_file(tmp_path):
    d = _copy(tmp_path)
    single = [w for w, names in bench.KERNEL_SOURCES.items() if names is not None]
    before = {w: bench.source_digest(w, d) for w in single}
    all_before = bench.source_digest(None, d)
    fused_before = bench.source_digest("fused_layer", d)
    assert fused_before == all_before      # the fused layer's unit is a call over every kernel
    _edit(d, "layer_tc.cu", None, "\nstatic int unused_marker_for_the_test = 1;\n")
    assert {w: bench.source_digest(w, d) for w in single} == before   # no single-kernel record there
    assert bench.source_digest(None, d) != all_before
    assert bench.source_digest("fused_layer", d) != fused_before
    _edit(d, "sgmv.cu", None, "\nstatic int another_marker = 2;\n")
    after = {w: bench.source_digest(w, d) for w in single}
    assert after["decode_bgmv"] == before["decode_bgmv"]
    assert after["prefill_sgmv"] != before["prefill_sgmv"]
    assert after["encoder_mixed_rank"] != before["encoder_mixed_rank"]
    assert after["prefill_sgmv.shrink"] != before["prefill_sgmv.shrink"]

