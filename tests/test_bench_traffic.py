"""bench.py reports an ncu traffic figure only for the kernel sources it was
captured on: the committed summary's hash must match the current sources
(the kernel's .cu file and the headers compiled into it)."""
from __future__ import annotations

import json
import os
import shutil

import bench


def make_tree(tmp_path, kernel):
    name, sources = bench.KERNEL_FILES[kernel]
    csrc = tmp_path / "sparse_mla_decode_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in sources:
        shutil.copy(os.path.join(bench.ROOT, "sparse_mla_decode_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return name, sources, csrc


def test_traffic_counts_only_for_the_sources_it_was_captured_on(tmp_path, monkeypatch):
    name, sources, csrc = make_tree(tmp_path, 2)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    digest = bench.source_digest(sources)
    path = tmp_path / "profiles" / f"{name}_throughput.json"
    path.write_text(json.dumps({"kernel_source_sha256_16": digest, "dram_bytes_per_launch": 123}))
    assert bench.load_traffic("throughput", 2) == 123
    # any source compiled into the kernel changes: the figure is stale
    hdr = csrc / sources[-1]
    hdr.write_text(hdr.read_text() + "\n// changed\n")
    assert bench.source_digest(sources) != digest
    assert bench.load_traffic("throughput", 2) is None
    assert bench.load_traffic("no_such_workload", 2) is None


def test_every_kernel_lists_its_sources():
    for kernel, (name, sources) in bench.KERNEL_FILES.items():
        assert sources[0].endswith(".cu") and "smd_internal.h" in sources and "smd_ptx.cuh" in sources
        for f in sources:
            assert os.path.exists(os.path.join(bench.ROOT, "sparse_mla_decode_gb300", "csrc", f)), f
        text = open(os.path.join(bench.ROOT, "sparse_mla_decode_gb300", "csrc", sources[0])).read()
        for f in sources[1:]:
            assert f'#include "{f}"' in text, (sources[0], f)
