"""The frozen per-shape plan table compiled into the library
(transformer_encoder_layer_gb300/csrc/tune_table.inc, written by
tests/tune_plan_table.py): well formed, and covering the five workloads."""
import os
import re

from transformer_encoder_layer_gb300.inputs import SHAPES

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "transformer_encoder_layer_gb300", "csrc", "tune_table.inc")
DTYPE = {"f32": 0, "f16": 1, "bf16": 2}


def entries():
    out = []
    for line in open(TABLE):
        m = re.match(r"\s*\{([-\d,\s]+)\},\s*$", line)
        if m:
            out.append(tuple(int(v) for v in m.group(1).split(",")))
    return out


def test_entries_are_well_formed():
    es = entries()
    assert es
    keys = set()
    for dtype, d, H, dff, nl, B, L, path, split in es:
        assert dtype in (0, 1, 2) and d % H == 0 and d >= 16 and dff >= 16 and nl >= 1
        assert B >= 1 and L >= 1 and path in (1, 2, 3, 4)
        assert split in (0, 8, 16, 32, 64) if path == 2 else split == -1
        key = (dtype, d, H, dff, nl, B, L)
        assert key not in keys  # one plan per shape
        keys.add(key)


def test_every_workload_has_a_frozen_plan():
    keys = {e[:7] for e in entries()}
    for s in SHAPES.values():
        assert (DTYPE[s.dtype], s.d_model, s.n_heads, s.d_ff, s.n_layers, s.batch, s.seq_len) in keys, s.name
