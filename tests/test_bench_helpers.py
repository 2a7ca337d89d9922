"""Host helpers of bench.py that the reported figures rest on (no GPU).

- `_pairs`: allowed (i, j) pairs of the causal mask, with and without packed
  documents, against a brute-force count over the mask's definition
  (j <= i and the same document);
- `_flops`: the forward FLOP count of the N=65536 workload against the
  figure the survey's measurement table states for it (3.52e13);
- `ClockSampler.summary`: median clock, maximum and throttle reasons parsed
  from a synthetic `nvidia-smi --format=csv,noheader,nounits` log.
"""
import os
import types

import numpy as np
import pytest

import bench
from ulysses_inputs import WORKLOADS, cu_seqlens_from_lengths, doc_lengths


def _pairs_brute(N, cu):
    doc = np.zeros(N, dtype=np.int64)
    if cu is not None:
        lengths = np.diff(np.asarray(cu, dtype=np.int64))
        doc = np.repeat(np.arange(len(lengths)), lengths)
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    return int(((j <= i) & (doc[:, None] == doc[None, :])).sum())


@pytest.mark.parametrize("N,cu", [
    (1, None),
    (300, None),
    (700, [0, 100, 101, 350, 700]),
    (600, [0, 0, 128, 128, 300, 600, 600]),   # zero-length documents
    (2048, "recipe"),
])
def test_pairs_match_the_mask(N, cu):
    if cu == "recipe":
        cu = list(cu_seqlens_from_lengths(doc_lengths(N, 4, seed=3, lo=64, hi=512)))
    assert bench._pairs(N, cu) == _pairs_brute(N, cu)


def test_forward_flops_of_the_64k_workload():
    w = WORKLOADS["qwen3_4b_n65536"]
    fwd, bwd = bench._flops(w, None)
    assert bench._pairs(w.N, None) == 2_147_516_416
    assert fwd == pytest.approx(3.518e13, rel=1e-3)
    assert bwd == pytest.approx(2.5 * fwd)


def _sampler_with(tmp_path, lines):
    path = os.path.join(str(tmp_path), "clocks.csv")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")
    s = bench.ClockSampler(0, str(tmp_path))
    s.path = path
    s.proc = types.SimpleNamespace()  # as if nvidia-smi had run
    return s


def test_clock_summary_parses_samples(tmp_path):
    lines = [
        "0, 1965, 2070, 1180.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1205.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1199.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    out = _sampler_with(tmp_path, lines).summary()
    assert out["sm_mhz"] == 1980.0
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 3


def test_clock_summary_reports_slowdowns(tmp_path):
    lines = ["0, 1500, 2070, 900.0, 0x8, Active, Not Active, Active, Not Active"]
    out = _sampler_with(tmp_path, lines).summary()
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples(tmp_path):
    out = _sampler_with(tmp_path, ["not a sample"]).summary()
    assert out["reasons"] == ["no samples"]
