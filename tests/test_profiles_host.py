"""The DRAM traffic that bench.py reports comes from profiles/, never from a
hand-kept constant: every row of profiles/dram_traffic.md names the ncu
summary it was copied from, that summary holds the same byte counts, and the
row carries the hash of the kernel sources it was captured with, so a bench
line reports null (with the reason) once those sources change."""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def rows():
    return bench.traffic_rows()


def test_table_exists_and_parses():
    assert os.path.exists(bench.TRAFFIC_TABLE)
    assert len(rows()) >= 1


def test_rows_are_unique_and_well_formed():
    keys = [(r["op"], r["workload"], r["tokens"]) for r in rows()]
    assert len(keys) == len(set(keys)), "one capture per (op, workload, tokens)"
    for r in rows():
        assert r["op"] in bench.KERNEL_SOURCES, r
        assert re.fullmatch(r"[0-9a-f]{12}", r["hash"]), r
        assert r["read"] > 0 and r["write"] >= 0, r


def test_each_row_matches_its_summary():
    for r in rows():
        path = os.path.join(ROOT, "profiles", r["summary"])
        assert os.path.exists(path), f"{r['summary']} is missing"
        text = open(path).read().replace(",", "")
        for field in ("read", "write"):
            assert str(r[field]) in text, f"{r['summary']} does not show the {field} bytes {r[field]}"
        assert r["hash"] in text, f"{r['summary']} does not name the source hash {r['hash']}"


def test_lookup_follows_the_source_hash(monkeypatch):
    r = rows()[0]
    monkeypatch.setattr(bench, "source_hash", lambda op: r["hash"])
    val, note = bench.ncu_traffic(r["op"], r["workload"], r["tokens"])
    assert val == r["read"] + r["write"] and r["summary"] in note
    monkeypatch.setattr(bench, "source_hash", lambda op: "0" * 12)
    val, note = bench.ncu_traffic(r["op"], r["workload"], r["tokens"])
    assert val is None and "changed" in note
    val, note = bench.ncu_traffic(r["op"], "no-such-workload", 1)
    assert val is None and "no ncu capture" in note


def test_source_hash_is_stable_and_covers_every_op():
    for op in bench.KERNEL_SOURCES:
        h = bench.source_hash(op)
        assert re.fullmatch(r"[0-9a-f]{12}", h) and h == bench.source_hash(op)
