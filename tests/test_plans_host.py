"""Saved plans (memory_bound_weight_gb300.plans) on the CPU, against an
in-memory stand-in for the library's plan API: a round trip restores every
plan, and a file from another identity, an index out of range, an index that
now describes another plan, and a damaged file restore nothing wrong."""
import json

import pytest

from memory_bound_weight_gb300 import plans


class FakePlanAPI:
    """Candidate lists per shape and the current choice, like the library's cache."""

    def __init__(self, candidates):
        self.cand = {k: list(v) for k, v in candidates.items()}
        self.cur = {k: 0 for k in candidates}

    def plan_candidates(self, op, M, N, K):
        return len(self.cand.get((op, M, N, K), []))

    def plan_index(self, op, M, N, K):
        return self.cur.get((op, M, N, K), -1)

    def plan_select(self, op, M, N, K, i):
        assert 0 <= i < self.plan_candidates(op, M, N, K)
        self.cur[(op, M, N, K)] = i

    def plan_describe(self, op, M, N, K):
        return self.cand[(op, M, N, K)][self.cur[(op, M, N, K)]]


SHAPES = {(2, 1, 11264, 2048): ["lat a", "lat b", "mma2 c"], (4, 64, 18944, 3584): ["tc x", "tc y"]}
IDENT = {"gpu": "GB300", "sms": 152, "cc": "10.3", "library": "abc"}


@pytest.fixture
def api(monkeypatch):
    fake = FakePlanAPI(SHAPES)
    for name in ("plan_candidates", "plan_index", "plan_select", "plan_describe"):
        monkeypatch.setattr(plans.B, name, getattr(fake, name))
    monkeypatch.setattr(plans, "identity", lambda: dict(IDENT))
    return fake


def test_round_trip(api, tmp_path):
    api.cur = {(2, 1, 11264, 2048): 2, (4, 64, 18944, 3584): 1}
    path = str(tmp_path / "plans.json")
    assert plans.save_plans(path, list(SHAPES) + [(9, 1, 8, 64)]) == 2  # the unknown shape is left out
    api.cur = {k: 0 for k in SHAPES}
    assert plans.load_plans(path) == (2, [])
    assert api.cur == {(2, 1, 11264, 2048): 2, (4, 64, 18944, 3584): 1}


def test_other_identity_restores_nothing(api, tmp_path, monkeypatch):
    api.cur[(2, 1, 11264, 2048)] = 1
    path = str(tmp_path / "plans.json")
    plans.save_plans(path, SHAPES)
    api.cur[(2, 1, 11264, 2048)] = 0
    monkeypatch.setattr(plans, "identity", lambda: dict(IDENT, sms=148))
    n, why = plans.load_plans(path)
    assert n == 0 and "identity differs" in why[0]
    assert api.cur[(2, 1, 11264, 2048)] == 0


def test_stale_entries_are_skipped_and_leave_the_plan_alone(api, tmp_path):
    api.cur = {(2, 1, 11264, 2048): 2, (4, 64, 18944, 3584): 1}
    path = str(tmp_path / "plans.json")
    plans.save_plans(path, SHAPES)
    doc = json.load(open(path))
    doc["plans"][0]["index"] = 7            # out of range now
    doc["plans"][1]["plan"] = "tc z"        # index 1 describes another plan now
    doc["plans"].append({"op": 2, "M": 1})  # malformed
    json.dump(doc, open(path, "w"))
    api.cur = {(2, 1, 11264, 2048): 1, (4, 64, 18944, 3584): 0}
    n, why = plans.load_plans(path)
    assert n == 0 and len(why) == 3
    assert "out of range" in why[0] and "no longer" in why[1] and "malformed" in why[2]
    assert api.cur == {(2, 1, 11264, 2048): 1, (4, 64, 18944, 3584): 0}


def test_damaged_or_foreign_files(api, tmp_path):
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    assert plans.load_plans(str(bad))[0] == 0
    other = tmp_path / "other.json"
    other.write_text(json.dumps({"format": 99, "plans": []}))
    assert plans.load_plans(str(other)) == (0, ["not a plan file of this format"])
    assert plans.load_plans(str(tmp_path / "missing.json"))[0] == 0


def test_library_hash_covers_the_sources():
    h = plans.library_sources_sha()
    assert len(h) == 16 and h == plans.library_sources_sha()
