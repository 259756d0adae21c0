#!/usr/bin/env python
"""Writes the library's frozen per-shape plan table by proving, then timing
("KernelForge", section "What it does": every candidate is first proven
against the gate over several seeds and input scales, only survivors are
timed, and the winner is frozen into a table that the run time merely looks
up -- no autotuning at run time).

Run on the GPU it is tuned for (one GB300):

    python tests/tune_plan_table.py [--out PATH] [--rounds N]

For each shape below, the candidates are every execution path that can run
it and, on the layered path, the split-K attention chunk sizes {off, 8, 16,
32, 64} key tiles.  Proof: each candidate's output passes the gate against
the fp64 oracle for seeds {0, 1, 2} x input scales {1e-3, 1, 1e3}, on a
subsample the oracle finishes in seconds (the first sequences, and for very
long sequences the same layer on 4096 tokens).  Timing: the survivors at full
size, interleaved round-robin with the order rotated every round, an L2
flush before each timed forward, CUDA events; the median wins.  The output
is a C++ include (transformer_encoder_layer_gb300/csrc/tune_table.inc) that
paths.cu compiles in.  This script lives with the tests because the proof
stage runs the oracle; the library never runs it.
"""
from __future__ import annotations

import argparse
import datetime
import os
import statistics
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from transformer_encoder_layer_gb300.gate import gate  # noqa: E402
from transformer_encoder_layer_gb300.inputs import (  # noqa: E402
    SHAPES, from_storage, make_inputs, tiny_shape, to_storage)

DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}
PATH_CODE = {"simt": 1, "layered": 2, "mega": 3, "dag": 4}
SPLITS = (0, 8, 16, 32, 64)


def tuned_shapes():
    long64 = SHAPES["long_d64_L100k_B8"]
    wide = SHAPES["wide_d1024_L1024_B32"]
    return [
        SHAPES["tiny_d32_L32"], SHAPES["short_d128_L64_B4096"], SHAPES["batch1_d256_L512"],
        wide, long64,
        long64.with_(name="long_d64_B1_L8192", batch=1, seq_len=8192, vl_lo=7400, vl_hi=8192),
        long64.with_(name="long_d64_B1_L16384", batch=1, seq_len=16384, vl_lo=14800, vl_hi=16384),
        long64.with_(name="long_d64_B1_L32768", batch=1, seq_len=32768, vl_lo=29500, vl_hi=32768),
        tiny_shape(name="d256_dh64_B1_L4096", dtype="bf16", batch=1, seq_len=4096, vl_lo=3700,
                   vl_hi=4096, d_model=256, n_heads=4, d_ff=1024, n_layers=2),
        wide.with_(name="wide_d1024_B1_L4096", batch=1, seq_len=4096, vl_lo=3700, vl_hi=4096),
    ]


def proof_shape(s):
    """The subsample a candidate is proven on: at most 4 sequences of at most
    4096 tokens (valid lengths scaled to the same fraction of L)."""
    b = min(s.batch, 2 if s.d_model >= 512 else 4)
    if s.seq_len <= 4096:
        return s.with_(batch=b)
    f = 4096 / s.seq_len
    return s.with_(batch=b, seq_len=4096, vl_lo=max(1, int(s.vl_lo * f)), vl_hi=int(s.vl_hi * f))


def candidates(binding, s):
    enc = binding.Encoder(make_inputs(s.with_(batch=1, seq_len=1, vl_lo=1, vl_hi=1)).layers,
                          s.d_model, s.n_heads, s.d_ff, s.dtype)
    out = []
    for p in ("mega", "dag", "layered", "simt"):
        enc.set_path(p)
        try:
            enc.plan(s.batch, s.seq_len)
        except binding.TLError:
            continue
        if p == "simt" and s.dtype != "f32":
            continue  # the generic CUDA-core path is never faster on 16-bit shapes
        if p == "layered":
            out += [(p, k) for k in SPLITS]
        else:
            out.append((p, -1))
    enc.close()
    return out


def _dev(inp, torch):
    st = to_storage(inp.x, inp.shape.dtype)
    x = (torch.from_numpy(st.view(np.int16)).view(torch.bfloat16) if inp.shape.dtype == "bf16"
         else torch.from_numpy(st))
    return x.cuda(), torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()


def _f64(t, dtype, torch):
    o = t.cpu()
    if dtype == "bf16":
        return from_storage(o.view(torch.int16).numpy().view(np.uint16), "bf16")
    return from_storage(o.numpy(), dtype)


def make_encoder(binding, inp, cand):
    s = inp.shape
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    enc.set_path(cand[0])
    if cand[0] == "layered":
        enc.set_attention_split(cand[1])
    return enc


def prove(binding, torch, s, cands):
    ps = proof_shape(s)
    worst = {c: 0.0 for c in cands}
    for seed in (0, 1, 2):
        for scale in (1e-3, 1.0, 1e3):
            inp = make_inputs(ps, seed=seed, input_scale=scale)
            ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, ps.n_heads, check=False)
            x, vl = _dev(inp, torch)
            for c in cands:
                if worst[c] > 1.0:
                    continue
                enc = make_encoder(binding, inp, c)
                got = _f64(enc.forward(x, vl), ps.dtype, torch)
                enc.close()
                worst[c] = max(worst[c], gate(got, ref)[1])
    return worst


def time_candidates(binding, torch, s, cands, rounds):
    inp = make_inputs(s, seed=0)
    x, vl = _dev(inp, torch)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    encs, outs, wss = [], [], []
    for c in cands:
        enc = make_encoder(binding, inp, c)
        wss.append(torch.empty(max(enc.workspace_size(s.batch, s.seq_len), 256), dtype=torch.uint8,
                               device="cuda"))
        outs.append(torch.empty_like(x))
        for _ in range(3):
            enc.forward(x, vl, out=outs[-1], workspace=wss[-1], check=False)
        encs.append(enc)
    torch.cuda.synchronize()
    times = {c: [] for c in cands}
    for r in range(rounds):
        order = list(range(len(cands)))
        order = order[r % len(order):] + order[:r % len(order)]
        for i in order:
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            encs[i].forward(x, vl, out=outs[i], workspace=wss[i], check=False)
            b.record()
            torch.cuda.synchronize()
            times[cands[i]].append(a.elapsed_time(b))
    for e in encs:
        assert e.get_status() == 0
        e.close()
    return {c: statistics.median(v) for c, v in times.items()}


def main():
    import torch
    from transformer_encoder_layer_gb300 import binding, build
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", default=os.path.join(ROOT, "transformer_encoder_layer_gb300", "csrc",
                                                  "tune_table.inc"))
    ap.add_argument("--rounds", type=int, default=9)
    args = ap.parse_args()
    build.build()
    binding.load()
    torch.cuda.set_device(0)
    gpu = torch.cuda.get_device_name(0)
    lines = []
    for s in tuned_shapes():
        cands = candidates(binding, s)
        worst = prove(binding, torch, s, cands)
        proven = [c for c in cands if worst[c] <= 1.0]
        med = time_candidates(binding, torch, s, proven, args.rounds) if proven else {}
        best = min(med, key=med.get)
        report = ", ".join(f"{p}{'' if k < 0 else f'/kc{k}'}: {med[(p, k)]:.4f} ms"
                           f" (envelope {worst[(p, k)]:.3f})" for p, k in proven)
        rejected = [c for c in cands if worst[c] > 1.0]
        print(f"{s.name}: best {best} {med[best]:.4f} ms; {report}; rejected {rejected}", flush=True)
        lines.append(f"// {s.name}: {report}" + (f"; failed the gate: {rejected}" if rejected else ""))
        lines.append("{%d, %d, %d, %d, %d, %d, %d, %d, %d}," % (
            DTYPE_CODE[s.dtype], s.d_model, s.n_heads, s.d_ff, s.n_layers, s.batch, s.seq_len,
            PATH_CODE[best[0]], max(best[1], -1)))
    head = [
        "// Frozen per-shape plan table: {dtype, d_model, n_heads, d_ff, n_layers, B, L, path,",
        "// attention split (key tiles per chunk; 0 = unsplit, -1 = not the layered path)}.",
        f"// Written by tests/tune_plan_table.py on {gpu}, "
        f"{datetime.date.today().isoformat()}: each candidate proven",
        "// against the fp64 oracle (seeds 0-2 x input scales 1e-3, 1, 1e3), then the survivors",
        f"// timed at full size, {args.rounds} interleaved rounds, median (ms per forward).",
    ]
    with open(args.out, "w") as f:
        f.write("\n".join(head + lines) + "\n")
    print("wrote", args.out)


if __name__ == "__main__":
    main()
