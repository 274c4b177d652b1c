"""Host-side pieces of bench.py on CPU: the reference arm's JSON line (the
oracle timed on the host cores on the 131K-context workload) and the packed
input/output buffers of the end-to-end leg."""
import json
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_reference_arm_json_line(capsys, monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.main(["--impl", "reference", "--workload", "131k", "--steps", "2", "--warmup", "0"]) == 0
    d = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is False and d["n_gpus"] == 1 and d["steps"] == 2
    assert d["value"] > 0 and d["dtype"] == "f64" and d["data"] == "synthetic"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert "131K" in d["config"]["workload"]


def test_packed_views_are_aligned_disjoint_and_complete():
    parts = [(torch.bfloat16, (6, 1, 2, 256)), (torch.bfloat16, (6, 1, 2, 256)),
             (torch.bfloat16, (6, 1, 1, 16, 256)), (torch.int32, (1,)), (torch.float32, (3, 5))]
    buf, views = bench.packed("cpu", parts)
    base = buf.data_ptr()
    spans = []
    for v, (dt, shape) in zip(views, parts):
        assert v.dtype == dt and tuple(v.shape) == shape and v.is_contiguous()
        off = v.data_ptr() - base
        assert off % 256 == 0
        spans.append((off, off + v.numel() * v.element_size()))
    assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:]))  # in order, no overlap
    assert spans[-1][1] <= buf.numel()
    for i, v in enumerate(views):  # writes land in their own bytes only
        v.fill_(i + 1)
    for i, v in enumerate(views):
        assert torch.all(v == i + 1)
