"""The cold-L2 rotation of bench.py's small workloads (host logic, CPU tensors): the copies of a
step's cache-side inputs hold at least 3x the L2 together, each copy is its own storage with the
original's values, and the inputs a step does not read from the cache (q, lengths) are shared."""

import torch

import bench


def _inputs():
    g = torch.Generator().manual_seed(5)
    return {"q": torch.randn(2, 8, 64, generator=g),
            "kv_len": torch.tensor([300, 7], dtype=torch.int32),
            "seq_of": torch.tensor([0, 1], dtype=torch.int32),
            "k": torch.randn(2, 320, 2, 64, generator=g).half(),
            "v": torch.randn(2, 320, 2, 64, generator=g).half(),
            "ids": None}


def test_copies_cover_three_l2(monkeypatch):
    monkeypatch.setattr(bench, "L2_BYTES", 1 << 20)  # a 1 MiB stand-in keeps the test small
    x = _inputs()
    rot = bench._rotation(x, torch)
    per_copy = x["k"].nbytes + x["v"].nbytes
    assert len(rot) * per_copy >= 3 * bench.L2_BYTES
    assert (len(rot) - 1) * per_copy < 3 * bench.L2_BYTES  # no more copies than that needs
    ptrs = {r["k"].data_ptr() for r in rot} | {r["v"].data_ptr() for r in rot}
    assert len(ptrs) == 2 * len(rot)  # every copy its own storage
    for r in (rot[0], rot[len(rot) // 2], rot[-1]):
        assert torch.equal(r["k"], x["k"]) and torch.equal(r["v"], x["v"])
        assert r["q"] is x["q"] and r["kv_len"] is x["kv_len"] and r["ids"] is None


def test_at_least_two_copies(monkeypatch):
    monkeypatch.setattr(bench, "L2_BYTES", 1)  # any input already exceeds 3x this
    rot = bench._rotation(_inputs(), torch)
    assert len(rot) == 2
