"""Planted mistakes in the oracle must be caught by its pins (no GPU).

Each mutant is a copy of ``oracle/lora_oracle.c`` with one plausible slip
(a dropped scale, a wrong sign, a transposed operand, a wrong index, an
off-by-one range, a lost error flag, single-precision accumulation).  It is
compiled to a temporary library and every pin in ``tests/oracle_pins.py`` is
run against it in a subprocess; at least one pin must fail (a crash counts
as caught).  The real oracle is never modified.
"""
import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "drop_scale_layer": [("yi[n] += scale[a] * acc;", "yi[n] += acc;")],
    "drop_scale_expand": [("y[(size_t)i * h_out + n] += scale[a] * acc;", "y[(size_t)i * h_out + n] += acc;")],
    "sign_flip_layer": [("yi[n] += scale[a] * acc;", "yi[n] -= scale[a] * acc;")],
    "transposed_base": [("W[(size_t)n * h_in + k]", "W[(size_t)k * h_out + n]")],
    "wrong_x_index": [("acc += xt[k] * at[(size_t)j * h_in + k];", "acc += xt[j] * at[(size_t)j * h_in + k];")],
    "b_row_stride": [("acc += vt[j] * b[(size_t)j * h_out + n];", "acc += vt[j] * b[(size_t)j * h_in + n];")],
    "rank_short_by_one": [("for (int j = 0; j < r; ++j) {", "for (int j = 0; j + 1 < r; ++j) {"),
                          ("for (int j = 0; j < rank[a]; ++j) {", "for (int j = 0; j + 1 < rank[a]; ++j) {")],
    "segment_skips_first": [("for (int t = seg_starts[s]; t < seg_starts[s + 1]; ++t)",
                             "for (int t = seg_starts[s] + 1; t < seg_starts[s + 1]; ++t)")],
    "neighbour_token_id": [("int a = token_adapter[t];", "int a = token_adapter[t > 0 ? t - 1 : 0];")],
    "none_as_adapter0": [("if (a < 0)\n        return -1;", "if (a < 0)\n        a = 0;")],
    "lost_error_flag": [("*status |= ORC_ERR_ADAPTER;", "(void)0;")],
    "float_accumulator": [("double acc = 0.0;", "float acc = 0.0f;")],
}


def _mutate(src: str, edits) -> str:
    for old, new in edits:
        assert old in src, f"mutation anchor not found: {old!r}"
        src = src.replace(old, new)
    return src


def _run(name, edits, tmp):
    with open(oracle.SRC) as f:
        src = _mutate(f.read(), edits)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"lib{name}.so")
    with open(c, "w") as f:
        f.write(src)
    oracle.build(force=True, src=c, out=so)
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, os.path.join(HERE, "oracle_pins.py"), so],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    if r.returncode != 0:
        return name, {"crash": f"exit {r.returncode}"}
    return name, json.loads(r.stdout.strip().splitlines()[-1])


@pytest.fixture(scope="module")
def verdicts(tmp_path_factory):
    tmp = str(tmp_path_factory.mktemp("mutants"))
    with ThreadPoolExecutor(max_workers=4) as ex:
        return dict(ex.map(lambda kv: _run(kv[0], kv[1], tmp), MUTANTS.items()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(verdicts, name):
    v = verdicts[name]
    failed = [k for k, s in v.items() if s != "ok"]
    assert failed, f"mutant {name} passed every pin: {v}"
