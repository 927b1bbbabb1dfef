"""The oracle's command line (python -m oracle): its records are those of the
oracle's own layer functions called directly on the workload's seeded inputs
(the state after each step, bit for bit, and the FP8 arrays' digests), for
delayed and just-in-time scaling and for a slice of a larger workload; bad
arguments are refused."""
import dataclasses
import hashlib
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import fp8_workloads as wl
import oracle as o

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cli(*args):
    r = subprocess.run([sys.executable, "-m", "oracle", *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    return r.returncode, [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")], r.stderr


def _direct(workload, steps, rows=None, cols=None, current=False):
    w = wl.WORKLOADS[workload]
    s = dataclasses.replace(w, M=rows or w.M, N=cols or w.N)
    rc = o.Recipe(margin=w.margin, history_len=w.history_len, hybrid=w.hybrid, current=current)
    st = o.State.initial(w.history_len)
    W = wl.bf16_bits(wl.layer_weight(s))
    recs = []
    for t in range(steps):
        fo = o.layer_fwd(st, rc, wl.bf16_bits(wl.layer_x(s, t)), W)
        bo = o.layer_bwd(st, rc, wl.bf16_bits(wl.layer_dy(s, t)), fo["X8t"], fo["W8t"])
        o.layer_update(st, rc)
        recs.append((st.copy(), {k: hashlib.sha256(np.ascontiguousarray(v).tobytes()).hexdigest()
                                 for k, v in (("X8", fo["X8"]), ("W8t", fo["W8t"]),
                                              ("dY8t", bo["dY8t"]), ("Y", fo["Y"]))}))
    return recs


@pytest.mark.parametrize("args,kw", [(("--workload", "tiny", "--steps", "3"), {}),
                                     (("--workload", "tiny", "--steps", "2", "--current"),
                                      {"current": True}),
                                     (("--workload", "mlp7b", "--rows", "32", "--cols", "64"),
                                      {"rows": 32, "cols": 64})])
def test_cli_records_are_the_oracle_steps(args, kw):
    rc, recs, err = _cli(*args)
    assert rc == 0, err
    workload = args[1]
    steps = int(args[args.index("--steps") + 1]) if "--steps" in args else 1
    direct = _direct(workload, steps, **kw)
    assert len(recs) == steps
    names = ["X", "W", "Y", "dY", "dX"]
    for rec, (st, dig) in zip(recs, direct):
        for k, name in enumerate(names):
            slot = rec["slots"][name]
            assert slot["scale_bits"] == f"0x{int(st.scale[k].view(np.uint32)):08x}", name
            assert slot["scale_inv_bits"] == f"0x{int(st.scale_inv[k].view(np.uint32)):08x}", name
            assert np.float32(slot["scale"]) == st.scale[k]
        for name, h in dig.items():
            assert rec["sha256"][name] == h, name
        assert rec["scaling"] == ("just-in-time" if kw.get("current") else "delayed")


@pytest.mark.parametrize("args", [("--rows", "24"), ("--cols", "0"), ("--steps", "0"),
                                  ("--workload", "nope")])
def test_cli_refuses_bad_arguments(args):
    rc, recs, err = _cli(*args)
    assert rc == 2 and not recs
