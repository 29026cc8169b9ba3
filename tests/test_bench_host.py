"""Host logic of bench.py that needs no GPU: the acceptance bytes counted
from a finished walk, the traffic figure's source-hash guard and the peaks
file fallback."""

import json
import os

import numpy as np

import bench


class _W:
    V = 10


def test_walk_bytes_counts_visited_rows():
    # tree: 0 -> {1, 2}, 1 -> {3}; walks: root only, root -> 1, root -> 1 -> 3
    parent = np.array([[-1, 0, 0, 1]] * 3, np.int32)
    path = np.array([[0, -1, -1, -1], [0, 1, -1, -1], [0, 1, 3, -1]], np.int32)
    alen = np.array([0, 1, 2], np.int32)
    row = _W.V * 4
    # the root and node 1 have children (target + draft rows); node 3 is a leaf
    expect = 2 * row + (2 * row + 2 * row) + (2 * row + 2 * row + row)
    assert bench.walk_bytes(_W, parent, path, alen) == expect


def test_walk_bytes_chain_reads_every_visited_row_pair():
    N = 5
    parent = np.array([[-1] + list(range(N - 1))], np.int32)
    path = np.array([list(range(N))], np.int32)
    # every node but the last has a child: 2 rows each, the last 1
    assert bench.walk_bytes(_W, parent, path, np.array([N - 1])) == (2 * (N - 1) + 1) * _W.V * 4


def test_committed_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    entry = {"dram_bytes_per_launch": 1234, "source": "k.cu",
             "source_hash": bench.source_hash("k.cu")}
    one_chunk = dict(entry, dram_bytes_per_launch=99)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"w": entry, "w@1": one_chunk}))
    assert bench.committed_traffic("w") == 1234.0
    assert bench.committed_traffic("w", 1) == 99.0     # captured with one chunk
    assert bench.committed_traffic("w", 2) is None     # no capture with two
    assert bench.committed_traffic("other") is None
    src.write_text("kernel v2")                 # the kernel changed since the capture
    assert bench.committed_traffic("w") is None


def test_measured_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_peaks() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.5}))
    assert bench.measured_peaks() == (7000.5, "measured")
