"""Calibration of the per-segment layout cost model (kvq_layout_cost).

The BitLLM summary ("How it works") scores a layout as
    alpha1 * Bytes / BW + alpha2 * UnpackOps
with the two weights fitted once per GPU by a short microbenchmark.  Here a
segment is read by the split-KV attention kernel, so:
  Bytes     HBM bytes the kernel's copies move for the segment: whole
            16-token tiles for KVQ_LAYOUT_TILES, exactly the filled rows for
            KVQ_LAYOUT_ROWS (scale rows in pairs);
  UnpackOps warp-instructions spent turning the staged bytes into the tile
            order: 0 for tiles, `ops_rows` per staged tile for rows (the
            in-shared-memory permute; counted with ncu as the difference of
            executed instructions between the two layouts on the same cache,
            passed in with --ops-rows).
This script times decode steps over one sequence of 256 kv heads whose cache
is 60 segments of n tokens each, in either layout, for several n, rotating
over enough cache copies that no step reads L2-resident bytes, and fits
    t = t0 + a_bytes * Bytes + a_ops * UnpackOps
by least squares.  It writes layout_model.json beside this file (the
coefficients kvq_layout_cost defaults to) with every measured point.

    python -m quantized_kv_cache_03_gb300.layout_calib --ops-rows 56 [--out PATH]
"""
from __future__ import annotations

import argparse
import json
import os

import numpy as np
import torch

from . import kvq

HEADS = 256
N_SEGS = 60
N_LIST = (1, 2, 4, 8, 12, 15, 16, 24, 32)
L2_BYTES = 129 * 1024 * 1024
BYTES_PER_ROW = {kvq.V_Q4_0: 128 + 8 + 64 + 8, kvq.V_Q8_0: 128 + 8 + 128 + 8}


def seg_bytes(layout: int, v_type: int, n: int) -> int:
    """HBM bytes the attention kernel moves for one kv head of a segment of n
    tokens (read as one piece)."""
    row = BYTES_PER_ROW[v_type]
    if layout == kvq.LAYOUT_TILES:
        return -(-n // 16) * 16 * row
    code = row - 16                               # K and V code bytes of a row
    return n * code + (n + (n & 1)) * 16          # scale rows copied in pairs


def seg_tiles(n: int) -> int:
    return -(-n // 16)


def build_copy(layout, v_type, n, dev):
    c = kvq.Cache(1, HEADS, v_type, max_segs=N_SEGS, device=dev)
    L = N_SEGS * n
    g = torch.Generator(device="cpu").manual_seed(1234)
    k = torch.randn(L, HEADS, 128, generator=g).half().to(dev)
    v = torch.randn(L, HEADS, 128, generator=g).half().to(dev)
    for s in range(N_SEGS):
        c.add_segment(0, n, layout)
        kvq.kvq_append(c, [0], [n], k[s * n:(s + 1) * n].contiguous(), v[s * n:(s + 1) * n].contiguous())
    return c, L


def time_config(layout, v_type, n, dev, reps=200):
    per_copy = HEADS * N_SEGS * seg_bytes(layout, v_type, n)
    n_rot = int(min(64, max(3, -(-3 * L2_BYTES // per_copy))))
    copies = [build_copy(layout, v_type, n, dev) for _ in range(n_rot)]
    L = copies[0][1]
    q = torch.randn(1, 1, HEADS, 128, device=dev).half()
    lens = torch.tensor([L], dtype=torch.int32, device=dev)
    out = torch.empty(1, 1, HEADS, 128, device=dev)
    lse = torch.empty(1, 1, HEADS, device=dev)
    nws = max(kvq.kvq_decode_workspace_size(c, HEADS, 1, L) for c, _ in copies)
    ws = torch.empty(max(1, nws), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(c):
        kvq.kvq_decode_attn(c, q, HEADS, 1, False, lens, L, None, 0.088, out, lse, ws if nws else None, stream)

    with torch.cuda.stream(stream):
        for c, _ in copies:
            step(c)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c, _ in copies:
            step(c)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        torch.cuda._sleep(2_000_000)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    us = 1e3 * e0.elapsed_time(e1) / (reps * n_rot)
    del copies
    torch.cuda.empty_cache()
    return us, n_rot


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--ops-rows", type=float, required=True,
                    help="warp-instructions of the rows-to-tile permute per staged tile (ncu difference)")
    ap.add_argument("--v-type", type=int, default=kvq.V_Q4_0)
    ap.add_argument("--out", default=os.path.join(os.path.dirname(os.path.abspath(__file__)), "layout_model.json"))
    args = ap.parse_args()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    points = []
    for n in N_LIST:
        for layout in (kvq.LAYOUT_TILES, kvq.LAYOUT_ROWS):
            us, n_rot = time_config(layout, args.v_type, n, dev)
            b = HEADS * N_SEGS * seg_bytes(layout, args.v_type, n)
            ops = HEADS * N_SEGS * seg_tiles(n) * (args.ops_rows if layout == kvq.LAYOUT_ROWS else 0.0)
            points.append(dict(n=n, layout=layout, us=us, bytes=b, unpack_ops=ops, copies=n_rot))
            print(json.dumps(points[-1]), flush=True)
    A = np.array([[1.0, p["bytes"], p["unpack_ops"]] for p in points])
    t = np.array([p["us"] for p in points])
    coef, *_ = np.linalg.lstsq(A, t, rcond=None)
    model = dict(v_type=args.v_type, heads=HEADS, segments=N_SEGS, t0_us=float(coef[0]),
                 us_per_byte=float(coef[1]), us_per_op=float(coef[2]), ops_rows_per_tile=args.ops_rows,
                 bytes_per_row=BYTES_PER_ROW[args.v_type], points=points,
                 gpu=torch.cuda.get_device_name(dev))
    with open(args.out, "w") as f:
        json.dump(model, f, indent=1)
        f.write("\n")
    print(json.dumps({k: v for k, v in model.items() if k != "points"}))


if __name__ == "__main__":
    main()
