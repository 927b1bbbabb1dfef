"""Command line of the oracle: the CPU reference results of a workload's
layer steps on its seeded inputs (test infrastructure, like the package).

    python -m oracle --workload tiny --steps 3
    python -m oracle --workload mlp7b --rows 256 --cols 1024 --steps 2 --current

Each step takes the workload's seeded X, W and dY for that step, drawn by
its generators at M = ``--rows`` tokens and N = ``--cols`` output features
when given (all K input features; X and W are then the first rows of the
full tensors), runs the forward, the backward and the scale update of one
FP8 linear layer, and prints one JSON line: the five slots' amax, scale and
scale_inv (values and binary32 bit patterns, the state after the update)
and SHA-256 digests of every FP8 array (X8, X8t, W8, W8t, dY8, dY8t) and
BF16 output (Y, dX, dW) as stored bytes.  The inputs are drawn on the CPU;
the bench and the GPU tests draw theirs on the device, whose generator gives
other values, and hand copies of them to the oracle.  The same tensors run
through the GPU library's Fp8Linear give the same FP8 arrays and the same
X, W and dY state bit for bit; its BF16 outputs (and so the Y and dX amax)
match within the GEMM tolerance, since the GPU accumulates in fp32.
"""
import argparse
import dataclasses
import hashlib
import json
import sys

import numpy as np

import fp8_workloads as wl

from . import (SLOT_DX, SLOT_DY, SLOT_W, SLOT_X, SLOT_Y, Recipe, State, layer_bwd, layer_fwd,
               layer_update)

SLOT_NAMES = {SLOT_X: "X", SLOT_W: "W", SLOT_Y: "Y", SLOT_DY: "dY", SLOT_DX: "dX"}


def _digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def _bits(v) -> str:
    return f"0x{int(np.float32(v).view(np.uint32)):08x}"


def run(workload: str, steps: int, rows=None, cols=None, current: bool = False):
    """The per-step records (dicts) of ``steps`` oracle layer steps."""
    w = wl.WORKLOADS[workload]
    s = dataclasses.replace(w, M=rows or w.M, N=cols or w.N)
    rc = Recipe(margin=w.margin, history_len=w.history_len, hybrid=w.hybrid, current=current)
    st = State.initial(w.history_len)
    W = wl.bf16_bits(wl.layer_weight(s))
    out = []
    for t in range(steps):
        X = wl.bf16_bits(wl.layer_x(s, t))
        dY = wl.bf16_bits(wl.layer_dy(s, t))
        fo = layer_fwd(st, rc, X, W)
        bo = layer_bwd(st, rc, dY, fo["X8t"], fo["W8t"])
        amax_seen = st.amax.copy()
        layer_update(st, rc)
        rec = {"step": t, "workload": workload, "M": s.M, "K": s.K, "N": s.N,
               "scaling": "just-in-time" if current else "delayed",
               "slots": {SLOT_NAMES[k]: {"amax": float(amax_seen[k]),
                                         "amax_bits": _bits(amax_seen[k]),
                                         "scale": float(st.scale[k]),
                                         "scale_bits": _bits(st.scale[k]),
                                         "scale_inv": float(st.scale_inv[k]),
                                         "scale_inv_bits": _bits(st.scale_inv[k])}
                         for k in sorted(SLOT_NAMES)},
               "sha256": {name: _digest(arr) for name, arr in
                          (("X8", fo["X8"]), ("X8t", fo["X8t"]), ("W8", fo["W8"]),
                           ("W8t", fo["W8t"]), ("dY8", bo["dY8"]), ("dY8t", bo["dY8t"]),
                           ("Y", fo["Y"]), ("dX", bo["dX"]), ("dW", bo["dW"]))}}
        out.append(rec)
    return out


def main(argv=None) -> int:
    p = argparse.ArgumentParser(prog="python -m oracle", description=__doc__.split("\n\n")[0])
    p.add_argument("--workload", default="tiny", choices=sorted(wl.WORKLOADS))
    p.add_argument("--steps", type=int, default=1)
    p.add_argument("--rows", type=int, default=None, help="tokens of the slice (default: all)")
    p.add_argument("--cols", type=int, default=None,
                   help="output features of the slice (default: all)")
    p.add_argument("--current", action="store_true", help="just-in-time scaling")
    a = p.parse_args(argv)
    for v, name in ((a.rows, "--rows"), (a.cols, "--cols")):
        if v is not None and (v <= 0 or v % 16):
            p.error(f"{name} must be a positive multiple of 16")
    if a.steps < 1:
        p.error("--steps must be at least 1")
    for rec in run(a.workload, a.steps, a.rows, a.cols, a.current):
        print(json.dumps(rec))
    return 0


if __name__ == "__main__":
    sys.exit(main())
