"""Host-side pieces of bench.py that need no GPU.

The roofline line carries the DRAM traffic of the committed ncu capture only
while the kernel sources are the ones that capture ran on; the check is a hash
of the sources' code (comments dropped). These tests pin that rule: a comment
edit keeps the hash, a code edit changes it, and a record taken on other
sources is not used.
"""

import json
import os
import shutil

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _copy_csrc(tmp_path):
    dst = tmp_path / "invariant_sparse_mla_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "invariant_sparse_mla_gb300", "csrc"), dst)
    return dst


def _sha_at(monkeypatch, root):
    monkeypatch.setattr(bench, "ROOT", str(root))
    return bench.kernel_source_sha()


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    csrc = _copy_csrc(tmp_path)
    base = _sha_at(monkeypatch, tmp_path)
    f = csrc / "attention.cu"
    text = f.read_text()
    f.write_text("// a new leading comment\n/* and a block\n   comment */\n" +
                 text.replace("constexpr int kStages = 2;",
                              "constexpr int kStages = 2;   // trailing note"))
    assert _sha_at(monkeypatch, tmp_path) == base
    f.write_text(text.replace("constexpr int kStages = 2;", "constexpr int kStages = 3;"))
    assert _sha_at(monkeypatch, tmp_path) != base


def test_traffic_record_is_used_only_for_its_own_sources(tmp_path, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    for r in rec["records"].values():
        if "split_kernel_bytes" in r:
            assert r["bytes_per_launch"] == r["split_kernel_bytes"] + r["combine_kernel_bytes"]
    key = next(iter(rec["records"]))
    wl, kern = key.split(":")
    csrc = _copy_csrc(tmp_path)
    (tmp_path / "profiles").mkdir()
    rec["source_sha"] = _sha_at(monkeypatch, tmp_path)
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic(wl, kern) == rec["records"][key]["bytes_per_launch"]
    assert bench.ncu_traffic(wl, "no_such_kernel") is None
    f = csrc / "combine_note.h"
    f.write_text("#pragma once\nconstexpr int kChanged = 1;\n")
    assert bench.ncu_traffic(wl, kern) is None


def test_warmup_and_steps_are_honoured_exactly():
    # Replayer runs whole passes over the input sets as one graph (captured
    # once per starting set) and the rest one set at a time, continuing from
    # where the last call stopped.
    class G:
        def __init__(self, log, name):
            self.log, self.name = log, name

        def replay(self):
            self.log.append(self.name)

    log = []
    rep = bench.Replayer.__new__(bench.Replayer)
    rep.stream, rep.n, rep.pos = None, 4, 0
    rep.cycles = [G(log, f"all@{k}") for k in range(4)]
    rep.single = [G(log, i) for i in range(4)]
    import contextlib
    import torch
    orig = torch.cuda.stream
    torch.cuda.stream = lambda s: contextlib.nullcontext()
    try:
        rep.run(5)      # warm-up of 5 steps
        assert log == ["all@0", 0] and rep.pos == 1
        log.clear()
        rep.run(20)     # 20 timed steps, continuing at set 1: five whole passes
        assert log == ["all@1"] * 5 and rep.pos == 1
        log.clear()
        rep.run(6)
        assert log == ["all@1", 1, 2] and rep.pos == 3
    finally:
        torch.cuda.stream = orig
