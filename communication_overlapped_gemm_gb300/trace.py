"""Reader of the trace buffer that ``tl_ctx_set_trace`` makes the persistent kernels fill.

The buffer layout is the one ``include/tl.h`` documents for ``tl_ctx_set_trace``: a
header of eight uint32 words, a uint32 span count per (CTA, warp), then 16-byte spans
``(uint64 t0_ns, uint32 dur_ns, uint32 kind << 24 | index)`` per (CTA, warp).  This module
only decodes that layout (host memory in, numpy records out) and writes the Chrome
trace-event JSON that chrome://tracing and Perfetto display: one process per CTA, one
thread per warp.
"""
from __future__ import annotations

import json

import numpy as np

MAGIC = 0x544C5452
HDR_WORDS = 8
WARPS = 16

KINDS = {
    1: "producer tile",
    2: "producer signal wait",
    3: "producer ring stall (total)",
    4: "mma tile",
    5: "mma starve (total)",
    6: "mma accumulator wait",
    7: "epilogue tile",
    8: "epilogue accumulator wait",
    9: "mover chunk",
    10: "side unit",
    11: "side wait",
}
# Kinds whose duration is a per-tile total of many short waits, not one interval.
TOTAL_KINDS = (3, 5)

SPAN_DTYPE = np.dtype([("cta", np.int32), ("warp", np.int32), ("kind", np.int32), ("index", np.int32),
                       ("t0", np.uint64), ("dur", np.uint32)])


def parse(raw) -> dict:
    """Decode a trace buffer copied to the host (bytes, bytearray or a uint8 array).

    Returns ``{"grid", "warps", "cap", "ctas", "counts", "dropped", "spans"}``: ``counts`` is
    the (ctas, 16) array of spans each warp recorded (dropped ones included), ``spans`` a
    structured array (cta, warp, kind, index, t0, dur) sorted by t0.  Raises ValueError
    when the header is not a trace header.
    """
    buf = np.frombuffer(bytes(raw), dtype=np.uint8)
    if buf.size < 4 * HDR_WORDS:
        raise ValueError("buffer smaller than the trace header")
    hdr = buf[: 4 * HDR_WORDS].view("<u4")
    if int(hdr[0]) != MAGIC or int(hdr[1]) != 1:
        raise ValueError("no trace header (magic/version mismatch): was a persistent kernel traced?")
    grid, warps, cap, held = (int(x) for x in hdr[2:6])
    if warps != WARPS or cap < 1:
        raise ValueError("malformed trace header")
    ctas = min(grid, held)
    cnt_off = 4 * HDR_WORDS
    rec_off = cnt_off + 4 * WARPS * held
    need = rec_off + 16 * WARPS * cap * held
    if buf.size < need:
        raise ValueError(f"trace buffer truncated: {buf.size} < {need} bytes")
    counts = buf[cnt_off: cnt_off + 4 * WARPS * ctas].view("<u4").reshape(ctas, WARPS).astype(np.int64)
    rec = buf[rec_off: rec_off + 16 * WARPS * cap * ctas].view(
        np.dtype([("t0", "<u8"), ("dur", "<u4"), ("tag", "<u4")])).reshape(ctas, WARPS, cap)
    kept = np.minimum(counts, cap)
    n = int(kept.sum())
    out = np.empty(n, dtype=SPAN_DTYPE)
    pos = 0
    for c in range(ctas):
        for w in range(WARPS):
            k = int(kept[c, w])
            if k == 0:
                continue
            r = rec[c, w, :k]
            sl = slice(pos, pos + k)
            out["cta"][sl] = c
            out["warp"][sl] = w
            out["kind"][sl] = (r["tag"] >> 24).astype(np.int32)
            out["index"][sl] = (r["tag"] & 0xFFFFFF).astype(np.int32)
            out["t0"][sl] = r["t0"]
            out["dur"][sl] = r["dur"]
            pos += k
    out = out[np.argsort(out["t0"], kind="stable")]
    return {"grid": grid, "warps": warps, "cap": cap, "ctas": ctas, "counts": counts,
            "dropped": int((counts - kept).sum()), "spans": out}


def summary(tr: dict) -> dict:
    """Per kind: span count and total / mean duration in microseconds, plus the traced
    kernel's extent (first span start to last span end) in microseconds."""
    sp = tr["spans"]
    res = {}
    for k, name in KINDS.items():
        m = sp["kind"] == k
        if not m.any():
            continue
        d = sp["dur"][m].astype(np.float64) / 1e3
        res[name] = {"count": int(m.sum()), "total_us": float(d.sum()), "mean_us": float(d.mean())}
    if sp.size:
        t0 = int(sp["t0"].min())
        t1 = int((sp["t0"] + sp["dur"].astype(np.uint64)).max())
        res["extent_us"] = (t1 - t0) / 1e3
    return res


def to_chrome(tr: dict, path: str | None = None) -> list:
    """Chrome trace-event list (complete "X" events, microseconds from the first span);
    written as JSON to ``path`` when given.  Per-tile totals (ring stall, MMA starve) are
    emitted as counter-free "X" events starting at their tile's start."""
    sp = tr["spans"]
    base = int(sp["t0"].min()) if sp.size else 0
    ev = []
    for s in sp:
        k = int(s["kind"])
        ev.append({"name": KINDS.get(k, f"kind {k}"), "ph": "X", "pid": int(s["cta"]), "tid": int(s["warp"]),
                   "ts": (int(s["t0"]) - base) / 1e3, "dur": int(s["dur"]) / 1e3,
                   "args": {"index": int(s["index"]), "total": k in TOTAL_KINDS}})
    if path is not None:
        with open(path, "w") as f:
            json.dump({"traceEvents": ev, "displayTimeUnit": "ns"}, f)
    return ev
