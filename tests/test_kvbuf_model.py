"""Pin for the reference reuse state machine: a trace written from the rules
of sglang PR #45909 (SparsePrefillKVBuffer.get_with_head)."""
import json
import os

import pytest

from oracle.kvbuf_model import KVBufModel

# a source is (layout, pool, pool_rows, ids); "A2" shares A's pool, not its ids
SOURCES = {"A": (1, 0x1000, 4096, 0x9000), "B": (1, 0x2000, 4096, 0xA000),
           "A2": (1, 0x1000, 4096, 0xB000)}


def run_trace(buf, ops):
    hits = []
    for op in ops:
        if op[0] == "begin_forward":
            buf.begin_forward()
        elif op[0] == "get":
            buf.get(op[1])
        elif op[0] == "realloc":
            buf.realloc(op[1])
        else:
            layout, pool, rows, ids = SOURCES[op[1]]
            hits.append((buf.get_with_head(layout, pool, rows, ids, op[2]), op[3]))
    return hits


def test_trace_from_the_page(golden_dir):
    with open(os.path.join(golden_dir, "kvbuf_trace.json")) as f:
        g = json.load(f)
    buf = KVBufModel(g["capacity"])
    for got, want in run_trace(buf, g["ops"]):
        assert got == want
    assert buf.dequants == g["dequants"]


def test_capacity_errors_leave_state():
    buf = KVBufModel(10)
    assert buf.get_with_head(1, 1, 1, 1, 10) is False
    with pytest.raises(ValueError):
        buf.get_with_head(1, 1, 1, 1, 11)
    assert buf.get_with_head(1, 1, 1, 1, 10) is True
