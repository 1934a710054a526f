"""Host-side checks of the trace buffer reader and the trace ABI's sizes (no GPU needed).

A buffer is assembled by hand in the layout include/tl.h documents for
tl_ctx_set_trace, and the reader's decoding, drop accounting, ordering, summary and
Chrome export are checked against it.
"""
import json
import struct

import numpy as np
import pytest

from communication_overlapped_gemm_gb300 import trace


def make_buffer(grid, held, cap, spans):
    """spans: {(cta, warp): [(t0, dur, kind, index), ...]} (beyond cap: counted, not stored)."""
    hdr = struct.pack("<8I", trace.MAGIC, 1, grid, trace.WARPS, cap, held, 0, 0)
    counts = np.zeros((held, trace.WARPS), dtype="<u4")
    rec = np.zeros((held, trace.WARPS, cap), dtype=[("t0", "<u8"), ("dur", "<u4"), ("tag", "<u4")])
    for (c, w), lst in spans.items():
        counts[c, w] = len(lst)
        for i, (t0, dur, kind, index) in enumerate(lst[:cap]):
            rec[c, w, i] = (t0, dur, (kind << 24) | index)
    return hdr + counts.tobytes() + rec.tobytes()


def test_trace_bytes_matches_documented_layout():
    import communication_overlapped_gemm_gb300 as tl
    tl.build()
    for ctas, cap in [(1, 1), (152, 256), (7, 3)]:
        assert tl.tl_trace_bytes(ctas, cap) == 32 + ctas * (16 * 4 + 16 * 16 * cap)
    assert tl.tl_trace_bytes(0, 4) == 0 and tl.tl_trace_bytes(4, 0) == 0
    # a null context is rejected without touching a device
    assert tl.lib().tl_ctx_set_trace(None, None, 0, 1) == tl.TL_ERR_INVALID


def test_parse_decodes_spans_counts_and_drops():
    spans = {
        (0, 0): [(1000, 50, 1, 7), (900, 10, 2, 7)],
        (0, 1): [(1200, 300, 4, 0), (1600, 200, 4, 5), (1900, 100, 4, 9), (2100, 5, 4, 12), (2500, 1, 4, 99)],
        (1, 2): [(1100, 400, 7, 3)],
    }
    raw = make_buffer(grid=2, held=3, cap=4, spans=spans)
    tr = trace.parse(raw)
    assert (tr["grid"], tr["cap"], tr["ctas"]) == (2, 4, 2)
    assert tr["counts"][0, 1] == 5 and tr["dropped"] == 1
    sp = tr["spans"]
    assert sp.size == 2 + 4 + 1
    assert np.all(np.diff(sp["t0"].astype(np.int64)) >= 0)  # sorted by start
    first = sp[0]
    assert (int(first["cta"]), int(first["warp"]), int(first["kind"]), int(first["index"])) == (0, 0, 2, 7)
    mma = sp[sp["kind"] == 4]
    assert sorted(mma["index"].tolist()) == [0, 5, 9, 12]  # the fifth span (index 99) was dropped
    epi = sp[sp["kind"] == 7]
    assert (int(epi[0]["cta"]), int(epi[0]["warp"]), int(epi[0]["dur"])) == (1, 2, 400)


def test_summary_and_chrome_export(tmp_path):
    spans = {(0, 1): [(1000, 2000, 4, 0), (3000, 1000, 4, 1)], (0, 2): [(3100, 1500, 7, 0)]}
    tr = trace.parse(make_buffer(grid=1, held=1, cap=2, spans=spans))
    s = trace.summary(tr)
    assert s["mma tile"]["count"] == 2 and s["mma tile"]["total_us"] == pytest.approx(3.0)
    assert s["extent_us"] == pytest.approx(3.6)  # 1000 .. 4600 ns
    path = tmp_path / "t.json"
    ev = trace.to_chrome(tr, str(path))
    assert len(ev) == 3 and ev[0]["ts"] == 0.0 and ev[0]["ph"] == "X"
    data = json.loads(path.read_text())
    assert {e["name"] for e in data["traceEvents"]} == {"mma tile", "epilogue tile"}


def test_parse_rejects_foreign_buffers():
    with pytest.raises(ValueError):
        trace.parse(b"\0" * 64)
    raw = make_buffer(grid=1, held=1, cap=2, spans={})
    with pytest.raises(ValueError):
        trace.parse(raw[:-16])  # truncated
