"""Host logic of bench.py, on the CPU: the segment lengths its FLOP count
uses equal the oracle's packing of the same documents, the traffic record is
reported only for the kernel sources and workload it was captured on, and the
CPU oracle table runs."""
import json

import numpy as np
import pytest

import bench
from oracle import attention as OA


@pytest.mark.parametrize("name", ["tiny", "c2", "c3", "c3_unpack", "c4", "c5"])
def test_segment_lengths_match_the_oracle_pack(name):
    w, lens, toks = bench.workload_docs(name)
    segs = bench.segment_lengths(lens, w)
    ref = OA.pack(toks, lens, w.micro_bsz, w.seq_len, w.use_packed_dataset)
    np.testing.assert_array_equal(segs, np.diff(ref["cu_seqlens"]))
    f = bench.flops(segs, w.Hq, w.head_dim)
    assert f["bwd"] == 2.5 * f["fwd"] and f["total"] == f["fwd"] + f["bwd"]
    assert f["pairs"] == float(np.sum(segs.astype(np.float64) * (segs + 1) / 2))


def test_traffic_record_follows_sources_and_workload(tmp_path):
    from sample_packing_document_gb300 import workloads as W
    w = W.WORKLOADS["c5"]
    rec = {"source": bench.kernel_source_hash(bench.BWD_SOURCES), "docs": "c5", "hq": 1, "group": 1, "d": 128,
           "dram_bytes": 1000}
    p = tmp_path / "rec.json"
    p.write_text(json.dumps(rec))
    assert bench.recorded_traffic(str(p), bench.BWD_SOURCES, w) == 1000 * w.Hq
    assert bench.recorded_traffic(str(p), bench.BWD_SOURCES, W.WORKLOADS["c2"]) is None   # other documents
    p.write_text(json.dumps(dict(rec, source="0" * 16)))
    assert bench.recorded_traffic(str(p), bench.BWD_SOURCES, w) is None                  # sources changed
    assert bench.recorded_traffic(str(tmp_path / "missing.json"), bench.BWD_SOURCES, w) is None


def test_committed_traffic_record_is_well_formed():
    rec = json.load(open(bench.TRAFFIC_RECORD))
    for key in ("source", "docs", "hq", "group", "d", "dram_bytes", "command"):
        assert key in rec
    assert rec["dram_bytes"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]


def test_committed_traffic_record_matches_the_current_sources():
    """The bench reports roofline.traffic only while the backward kernel's
    sources hash to the recorded value: a source change must come with a new
    capture, or the reported traffic goes null."""
    from sample_packing_document_gb300 import workloads as W
    rec = json.load(open(bench.TRAFFIC_RECORD))
    assert rec["source"] == bench.kernel_source_hash(bench.BWD_SOURCES)
    assert bench.recorded_traffic(bench.TRAFFIC_RECORD, bench.BWD_SOURCES, W.WORKLOADS["c5"]) == \
        rec["dram_bytes"] * W.WORKLOADS["c5"].Hq


def test_replica_value_is_the_whole_job():
    assert bench.replica_value(4, 2e12, 1000.0) == pytest.approx(4 * 2e12 / 1.0 / 1e12)


def test_cpu_table_runs_on_the_tiny_workload(capsys):
    assert bench.cpu_table(["tiny"]) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["kind"] == "oracle" and line["fwd_s"] > 0 and line["bwd_s"] > 0
