"""The bench's host-side bookkeeping on CPU: the DSA workloads' FLOP and byte
counts against hand counts, and both reference arms (the CPU oracle timed on
a bounded sample) printing a well-formed JSON line."""
import contextlib
import io
import json

import numpy as np
import pytest

import bench
from tiled_online_softmax_02_gb300.inputs import DsaWorkload, make_dsa_inputs


def test_dsa_allowed_counts_and_flops():
    w = DsaWorkload("t", B=2, S=3, H=5, D=8, T=10, top_k=4, dtype="bf16", bias="causal")
    x = make_dsa_inputs(w)
    cnt = bench.dsa_allowed_counts(x)
    # causal: row s allows keys t <= T - S + s
    exp = np.array([[w.T - w.S + s + 1 for s in range(w.S)]] * w.B)
    assert np.array_equal(cnt, exp)
    assert bench.dsa_flops(w, cnt) == 2 * w.H * w.D * int(exp.sum())


def test_dsa_algorithmic_bytes():
    w = DsaWorkload("t", B=2, S=3, H=5, D=8, T=10, top_k=4, dtype="bf16")
    rows = 6
    exp = (rows * 5 * 8 * 2 + 2 * 10 * 8 * 2 + rows * 5 * 2  # query, key, weights
           + rows * 10 * 4 + 2 * rows * 10 * 4 + rows * 4 * 8)  # bias, scores twice, indices
    assert bench.dsa_algorithmic_bytes(w) == exp
    assert bench.dsa_algorithmic_bytes(w.replace(dtype="f32")) == exp + rows * 5 * 8 * 2 + 2 * 10 * 8 * 2 + rows * 5 * 2


def _reference_line(argv):
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main(argv) == 0
    lines = [l for l in buf.getvalue().splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", ["dsa_decode_bf16", "tiny_f32"])
def test_reference_arm_prints_one_line(workload):
    d = _reference_line(["--impl", "reference", "--workload", workload, "--steps", "1", "--warmup", "3",
                         "--ref-seconds", "2"])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == workload
    assert d["steps"] == 1 and d["warmup"] == 3
