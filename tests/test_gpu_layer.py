"""GPU parity of the whole FP8 linear-layer step against the oracle, on the
layer workloads of fp8_workloads.py, through the same Fp8Linear.step that
bench.py times (fp8_linear_fwd, fp8_linear_bwd, fp8_amax_scale_update).

Every step:
  * bit-exact: amax of X, W, dY; every FP8 byte of X8, X8t, W8, W8t, dY8,
    dY8t (the oracle's cast through its 65,536-entry code table at that
    step's scale, compared on the device); history, scale and scale_inv of
    the X, W and dY slots, before and after the update;
  * Y and dX slots: the fused amax equals max |output| of the GPU's own BF16
    output exactly, the history holds those amaxes newest first, and the
    scale follows from them by the recipe's formula.
On the GEMM-check steps (every ``gemm_every`` steps, listed extra steps and
the last), Y, dX and dW within the tolerance of helpers.py: whole tensors on
small shapes; at full size three 16-row blocks (every column tile) and 16
columns over all rows (every row tile) of each output.
"""
import numpy as np
import pytest
import torch

import fp8_workloads as wl
import oracle as o
from helpers import (assert_codes_on_device, assert_fp8_equal, assert_gemm_close, bf16_values,
                     device_absmax_bits, f32_bits, host_bf16_bits, host_u8, oracle_code_table)

pytestmark = pytest.mark.gpu


def _lib():
    import fp8_mixed_precision_amax_gb300 as f
    return f


def _row_blocks(n, width=16):
    return sorted({0, (n // 2 // 16) * 16 + 48 if n > 128 else 0, n - width})


def _col_sample(n, count=16):
    """``count`` output columns spread over [0, n), first and last included."""
    return np.unique(np.linspace(0, n - 1, count).round().astype(np.int64))


def _gpu_slot_checks(lin, f, gpu_amax_hist, fmts, margin, g_amax):
    """Y / dX slots: properties that hold at any size (g_amax: the amax slots
    as the step left them, before the update consumed and cleared them)."""
    hist = lin.meta.history.cpu().numpy()
    scale = lin.meta.scale.cpu().numpy()
    assert not lin.meta.amax.cpu().numpy().any()       # cleared by the update
    for slot, out in ((f.SLOT_Y, lin.Y), (f.SLOT_DX, lin.dX)):
        a = float(g_amax[slot])
        mx = device_absmax_bits(out)                    # NaN skipped
        assert f32_bits(np.float32(a)) == f32_bits(mx), (slot, a, mx)
        gpu_amax_hist[slot].insert(0, np.float32(a))
        L = hist.shape[1]
        seq = (gpu_amax_hist[slot] + [np.float32(0)] * L)[:L]
        assert np.array_equal(hist[slot].view(np.uint32), np.array(seq, np.float32).view(np.uint32))
        m = np.float32(max(seq))
        if 0 < m < np.inf:
            fmax = np.float32(448.0 if fmts[slot] == o.E4M3 else 57344.0)
            expect = np.float32(np.float32(fmax / m) * np.float32(2.0 ** -margin))
            assert f32_bits(scale[slot]) == f32_bits(expect)


class _HostCopy:
    """Pinned host buffers reused across steps for the BF16 inputs' bits."""

    def __init__(self):
        self.bufs = {}

    def bits(self, name, t):
        b = self.bufs.get(name)
        if b is None or b.shape != t.shape:
            b = torch.empty(t.shape, dtype=torch.int16, pin_memory=True)
            self.bufs[name] = b
        b.copy_(t.view(torch.int16))
        return b.numpy().view(np.uint16)


def _check_gemms(gemms, full, step, report):
    """gemms: (name, GPU output, A codes, fa, B codes, fb, sa_inv, sb_inv, K)."""
    for name, out, A, fa, B, fb, sa, sb, K in gemms:
        gout = host_bf16_bits(out)
        if full:
            ref = o.epilogue(o.gemm_tn(A, fa, B, fb), sa, sb)
            report.append((step, name, assert_gemm_close(gout, ref, K, f"step {step} {name}")))
            continue
        for r0 in _row_blocks(A.shape[0]):
            ref = o.epilogue(o.gemm_tn(A, fa, B, fb, r0, 16), sa, sb)
            report.append((step, name, assert_gemm_close(gout[r0:r0 + 16], ref, K,
                                                         f"step {step} {name} rows {r0}")))
        cols = _col_sample(B.shape[0])
        ref = o.epilogue(o.gemm_tn(A, fa, np.ascontiguousarray(B[cols]), fb), sa, sb)
        report.append((step, name, assert_gemm_close(np.ascontiguousarray(gout[:, cols]), ref, K,
                                                     f"step {step} {name} columns")))


def run_layer(w: wl.Workload, steps, gemm_every=1, full=True, hybrid=None, extra_checks=(),
              current=False):
    f = _lib()
    hybrid = w.hybrid if hybrid is None else hybrid
    W = wl.layer_weight(w, "cuda")
    rc_gpu = f.Recipe(margin=w.margin, history_len=w.history_len, hybrid=hybrid, current=current)
    lin = f.Fp8Linear(W, w.M, rc_gpu)
    rc = o.Recipe(margin=w.margin, history_len=w.history_len, hybrid=hybrid, current=current)
    st = o.State.initial(w.history_len)
    fm = rc.formats()
    Wb = host_bf16_bits(W)
    w_amax = o.amax(Wb)
    host = _HostCopy()
    gpu_amax_hist = {f.SLOT_Y: [], f.SLOT_DX: []}
    report = []
    for step in range(steps):
        X = wl.layer_x(w, step, "cuda")
        dY = wl.layer_dy(w, step, "cuda")
        lin.forward(X)
        lin.backward(dY)
        torch.cuda.synchronize()
        g_amax = lin.meta.amax.cpu().numpy().copy()
        g_scale = lin.meta.scale.cpu().numpy().copy()
        g_scale_inv = lin.meta.scale_inv.cpu().numpy().copy()
        Xb, dYb = host.bits("X", X), host.bits("dY", dY)
        # the oracle's view of this step: amaxes (and just-in-time scales)
        st.amax[o.SLOT_X] = o.amax(Xb)
        st.amax[o.SLOT_W] = w_amax
        st.amax[o.SLOT_DY] = o.amax(dYb)
        if current:
            for slot in (o.SLOT_X, o.SLOT_W, o.SLOT_DY):
                o.just_in_time_scale(st, rc, slot, fm[slot])
        for slot in (o.SLOT_X, o.SLOT_W, o.SLOT_DY):
            assert f32_bits(g_amax[slot]) == f32_bits(st.amax[slot]), (step, slot)
            # the scales the casts of this step used
            assert f32_bits(g_scale[slot]) == f32_bits(st.scale[slot]), (step, slot)
            assert f32_bits(g_scale_inv[slot]) == f32_bits(st.scale_inv[slot]), (step, slot)
        # every FP8 byte, against the oracle's cast at this step's scales
        tables = {slot: oracle_code_table(st.scale[slot], fm[slot])
                  for slot in (o.SLOT_X, o.SLOT_W, o.SLOT_DY)}
        for name, g, x, slot, tr in [("X8", lin.X8, X, o.SLOT_X, False),
                                     ("X8t", lin.X8t, X, o.SLOT_X, True),
                                     ("W8", lin.W8, W, o.SLOT_W, False),
                                     ("W8t", lin.W8t, W, o.SLOT_W, True),
                                     ("dY8", lin.dY8, dY, o.SLOT_DY, False),
                                     ("dY8t", lin.dY8t, dY, o.SLOT_DY, True)]:
            assert_codes_on_device(g, x, tables[slot], fm[slot], tr, f"step {step} {name}")
        if (step % gemm_every == 0) or step in extra_checks or step == steps - 1:
            X8 = tables[o.SLOT_X][Xb]
            W8 = tables[o.SLOT_W][Wb]
            dY8 = tables[o.SLOT_DY][dYb]
            X8t, W8t, dY8t = (np.ascontiguousarray(a.T) for a in (X8, W8, dY8))
            si = st.scale_inv
            _check_gemms([("Y", lin.Y, X8, fm[0], W8, fm[1], si[0], si[1], w.K),
                          ("dX", lin.dX, dY8, fm[3], W8t, fm[1], si[3], si[1], w.N),
                          ("dW", lin.dW, dY8t, fm[3], X8t, fm[0], si[3], si[0], w.M)],
                         full, step, report)
        # the delayed-scaling update
        lin.update()
        torch.cuda.synchronize()
        st.amax[o.SLOT_Y] = st.amax[o.SLOT_DX] = 0.0   # checked by property below
        o.layer_update(st, rc)
        hist = lin.meta.history.cpu().numpy()
        for slot in (o.SLOT_X, o.SLOT_W, o.SLOT_DY):
            assert np.array_equal(hist[slot].view(np.uint32), st.history[slot].view(np.uint32))
            assert f32_bits(lin.meta.scale[slot].item()) == f32_bits(st.scale[slot]), (step, slot)
            assert f32_bits(lin.meta.scale_inv[slot].item()) == f32_bits(st.scale_inv[slot])
        _gpu_slot_checks(lin, f, gpu_amax_hist, fm, w.margin, g_amax)
    f.fp8_sync_status()
    return report


def test_tiny_layer_four_steps_whole_tensors():
    w = wl.WORKLOADS["tiny"]
    run_layer(w, w.steps, full=True)


@pytest.mark.parametrize("hybrid", [True, False])
def test_tiny_shape_long_run_history_window(hybrid):
    """1000 drifting steps at a small shape with history 512: spikes enter,
    persist exactly 512 steps and leave; all-zero steps keep the scale."""
    d = wl.WORKLOADS["drift"]
    small = wl.Workload("drift_small", 128, 256, 256, "drift", 1.0, 1 / 16, 1.0, 512, 0, True,
                        1000)
    run_layer(small, 1000, gemm_every=50, full=True, hybrid=hybrid,
              extra_checks=(49, 50, 51, 75, 76, 150, 562, 563))
    assert d.history_len == 512


def test_mlp7b_full_size_100_steps():
    """The 7B-shaped layer's 100 steps: state and every FP8 byte each step,
    the GEMMs (row blocks and column samples) every 10th step."""
    w = wl.WORKLOADS["mlp7b"]
    run_layer(w, w.steps, gemm_every=10, full=False)


def test_mlp70b_full_size_50_steps():
    """The 70B-shaped layer's 50 steps (Student-t X with outlier channels,
    margin 1): state and every FP8 byte each step, the GEMMs every 10th."""
    w = wl.WORKLOADS["mlp70b"]
    run_layer(w, w.steps, gemm_every=10, full=False)


@pytest.mark.parametrize("hybrid", [True, False])
def test_drift_full_size_1000_steps(hybrid):
    """The drifting-scale stress at full size (4096^3) through all 1000
    steps, in both the HYBRID and the E4M3-everywhere arms: state and every
    FP8 byte each step (the x1000 spikes at t % 100 == 50, the all-zero steps
    at t % 100 == 75, the history window of 512), GEMMs every 50th step and
    around the spikes and zero steps."""
    w = wl.WORKLOADS["drift"]
    run_layer(w, w.steps, gemm_every=50, full=False, hybrid=hybrid,
              extra_checks=(49, 51, 75, 76, 562, 563, 950, 951))


def test_ragged_layer_shape():
    """A layer whose M, N, K are not multiples of the GEMM tiles."""
    w = wl.Workload("ragged", 144, 272, 400, "normal", 1.0, 0.05, 0.01, 16, 0, True, 3)
    run_layer(w, 3, full=True)


@pytest.mark.parametrize("M,K,N", [(128, 400, 272), (16, 48, 32), (512, 16, 1040)])
def test_small_and_thin_layer_shapes(M, K, N):
    """Shapes where some GEMMs fit one 128-row tile (single-CTA variant, also
    inside the grouped backward launch), K = 16, and tiny layers."""
    w = wl.Workload("thin", M, K, N, "normal", 1.0, 0.05, 0.01, 8, 0, True, 2)
    run_layer(w, 2, full=True)


def test_just_in_time_scaling_tiny_and_drift():
    """Just-in-time scaling: X, W and dY are cast with scales from their own
    amax in the same step (including the all-zero and x1000 steps)."""
    run_layer(wl.WORKLOADS["tiny"], 4, full=True, current=True)
    small = wl.Workload("drift_small", 128, 256, 256, "drift", 1.0, 1 / 16, 1.0, 512, 0, True,
                        120)
    run_layer(small, 120, gemm_every=10, full=True, current=True,
              extra_checks=(49, 50, 51, 75, 76))


def test_just_in_time_scaling_mlp7b_full_size():
    run_layer(wl.WORKLOADS["mlp7b"], 2, full=False, current=True)


def test_just_in_time_scaling_mlp70b_full_size():
    """Just-in-time scaling at the 70B shape, where X, W and dY are all larger
    than the 96 MB that the amax pass leaves in L2 (its streaming loads)."""
    run_layer(wl.WORKLOADS["mlp70b"], 2, full=False, current=True)


def test_graph_replay_matches_eager_steps():
    """A captured step replays exactly what eager steps compute: two layers
    from the same state, one stepping eagerly, one through graph replays, stay
    bit-identical (outputs and scaling state) over several steps."""
    f = _lib()
    w = wl.Workload("graph", 384, 512, 272, "normal", 1.0, 0.05, 1e-2, 16, 0, True, 4)
    W = wl.layer_weight(w, "cuda")
    X, dY = wl.layer_x(w, 0, "cuda"), wl.layer_dy(w, 0, "cuda")
    a = f.Fp8Linear(W, w.M, f.Recipe(w.margin, w.history_len, w.hybrid))
    b = f.Fp8Linear(W, w.M, f.Recipe(w.margin, w.history_len, w.hybrid))
    g = b.capture_step(X, dY)      # includes one eager warm-up step
    a.step(X, dY)
    for _ in range(4):
        a.step(X, dY)
        g.replay()
        torch.cuda.synchronize()
        for t1, t2 in [(a.Y, b.Y), (a.dX, b.dX), (a.dW, b.dW), (a.meta.history, b.meta.history),
                       (a.meta.scale, b.meta.scale), (a.meta.scale_inv, b.meta.scale_inv)]:
            assert torch.equal(t1.view(torch.uint8), t2.view(torch.uint8))
    f.fp8_sync_status()


@pytest.mark.parametrize("K,current", [(512, False), (512, True), (4112, False)])
def test_graph_replay_of_the_layernorm_linear(K, current):
    """The same for LayerNorm + FP8 linear: the one-pass LayerNorm cast and the
    byte transpose (K = 512, delayed scaling), the statistics kernel and the
    cast kernel's LayerNorm branch (just-in-time scaling; K = 4112, past the
    one-pass limit) replay bit-identically, mean and rstd included."""
    f = _lib()
    w = wl.Workload("graph_ln", 384, K, 272, "normal", 1.0, 0.05, 1e-2, 16, 0, True, 4)
    W = wl.layer_weight(w, "cuda")
    X, dY = wl.layer_x(w, 0, "cuda"), wl.layer_dy(w, 0, "cuda")
    gen = torch.Generator().manual_seed(K)
    gamma = (1 + 0.1 * torch.randn(K, generator=gen)).to(torch.bfloat16).cuda()
    beta = (0.1 * torch.randn(K, generator=gen)).to(torch.bfloat16).cuda()
    rec = lambda: f.Recipe(w.margin, w.history_len, w.hybrid, current=current)
    a = f.Fp8LayerNormLinear(W, w.M, gamma, beta, 1e-5, rec())
    b = f.Fp8LayerNormLinear(W, w.M, gamma, beta, 1e-5, rec())
    g = b.capture_step(X, dY)      # includes one eager warm-up step
    a.step(X, dY)
    for _ in range(3):
        a.step(X, dY)
        g.replay()
        torch.cuda.synchronize()
        for t1, t2 in [(a.Y, b.Y), (a.dX, b.dX), (a.dW, b.dW), (a.X8, b.X8), (a.X8t, b.X8t),
                       (a.mean, b.mean), (a.rstd, b.rstd), (a.meta.history, b.meta.history),
                       (a.meta.scale, b.meta.scale), (a.meta.scale_inv, b.meta.scale_inv)]:
            assert torch.equal(t1.view(torch.uint8), t2.view(torch.uint8))
    f.fp8_sync_status()


def test_special_values_through_the_layer():
    """Degenerate inputs through whole steps: X holds +-inf, NaN and the
    largest BF16 values.  The amax of X is inf, so the X history holds inf
    and X's scale is kept (reading: a non-finite history max keeps the
    scale); inf and huge values saturate to the largest E4M3 code, NaN stays
    a NaN code; Y is NaN exactly in the rows (and dW in the columns) a NaN
    reaches, and the fused output amaxes skip NaN."""
    f = _lib()
    w = wl.Workload("special", 144, 272, 256, "normal", 1.0, 0.05, 0.01, 4, 0, True, 3)
    W = wl.layer_weight(w, "cuda")
    lin = f.Fp8Linear(W, w.M, f.Recipe(w.margin, w.history_len, w.hybrid))
    rc = o.Recipe(margin=w.margin, history_len=w.history_len, hybrid=w.hybrid)
    st = o.State.initial(w.history_len)
    fm = rc.formats()
    Wb = host_bf16_bits(W)
    for step in range(3):
        X = wl.layer_x(w, step, "cuda").clone()
        X[3, 5] = float("inf")
        X[100, 7] = -float("inf")
        X[17, 200] = float("nan")
        X[40, :] = 3.3895e38          # near the largest BF16 value
        dY = wl.layer_dy(w, step, "cuda")
        lin.step(X, dY)
        torch.cuda.synchronize()
        Xb, dYb = host_bf16_bits(X), host_bf16_bits(dY)
        fo = o.layer_fwd(st, rc, Xb, Wb)
        bo = o.layer_bwd(st, rc, dYb, fo["X8t"], fo["W8t"])
        for name, ref, fmt in [("X8", fo["X8"], fm[0]), ("X8t", fo["X8t"], fm[0]),
                               ("W8", fo["W8"], fm[1]), ("dY8", bo["dY8"], fm[3])]:
            assert_fp8_equal(host_u8(getattr(lin, name)), ref, fmt, f"step {step} {name}")
        assert (host_u8(lin.X8)[3, 5] & 0x7F) == 0x7E and (host_u8(lin.X8)[100, 7] == 0xFE)
        assert (host_u8(lin.X8)[17, 200] & 0x7F) == 0x7F
        for name, ref, K in [("Y", fo["Y"], w.K), ("dX", bo["dX"], w.N), ("dW", bo["dW"], w.M)]:
            assert_gemm_close(host_bf16_bits(getattr(lin, name)), ref, K, f"step {step} {name}")
        y = bf16_values(host_bf16_bits(lin.Y))
        assert np.isnan(y[17]).all() and not np.isnan(np.delete(y, 17, axis=0)).any()
        dw = bf16_values(host_bf16_bits(lin.dW))
        assert np.isnan(dw[:, 200]).all()
        o.layer_update(st, rc)
        hist = lin.meta.history.cpu().numpy()
        for slot in (o.SLOT_X, o.SLOT_W, o.SLOT_DY):
            assert np.array_equal(hist[slot].view(np.uint32), st.history[slot].view(np.uint32))
            assert f32_bits(lin.meta.scale[slot].item()) == f32_bits(st.scale[slot])
        assert hist[o.SLOT_X, 0] == np.inf and lin.meta.scale[o.SLOT_X].item() == 1.0
    f.fp8_sync_status()


def test_gradient_accumulation_records_the_max_over_micro_batches():
    """Two forward + backward passes before one update (gradient
    accumulation over two micro-batches): both passes cast with the same,
    not yet updated scales; the amax slots hold the max over both passes
    (X, W, dY against the oracle, Y and dX against the GPU's own outputs);
    the update pushes exactly that max into each history and clears the
    slots."""
    f = _lib()
    w = wl.Workload("accum", 256, 512, 384, "normal", 1.0, 0.05, 0.01, 16, 0, True, 2)
    W = wl.layer_weight(w, "cuda")
    lin = f.Fp8Linear(W, w.M, f.Recipe(w.margin, w.history_len, w.hybrid))
    lin.step(wl.layer_x(w, 5, "cuda"), wl.layer_dy(w, 5, "cuda"))   # scales away from 1.0
    torch.cuda.synchronize()
    scale0 = lin.meta.scale.cpu().numpy().copy()
    hist0 = lin.meta.history.cpu().numpy().copy()
    passes = []
    for k in (0, 1):
        X, dY = wl.layer_x(w, k, "cuda"), wl.layer_dy(w, k, "cuda")
        Y = torch.empty((w.M, w.N), dtype=torch.bfloat16, device="cuda")
        dX = torch.empty((w.M, w.K), dtype=torch.bfloat16, device="cuda")
        dW = torch.empty((w.N, w.K), dtype=torch.bfloat16, device="cuda")
        lin.forward(X, Y=Y)
        X8 = lin.X8.clone()
        lin.backward(dY, dX=dX, dW=dW)
        passes.append((host_bf16_bits(X), host_bf16_bits(dY), Y, dX, X8, lin.dY8.clone()))
    torch.cuda.synchronize()
    assert np.array_equal(lin.meta.scale.cpu().numpy().view(np.uint32), scale0.view(np.uint32))
    amax = lin.meta.amax.cpu().numpy().copy()
    absmax = lambda t: np.float32(np.max(np.abs(bf16_values(host_bf16_bits(t)))))
    expect = {
        f.SLOT_X: max(o.amax(p[0]) for p in passes),
        f.SLOT_W: o.amax(host_bf16_bits(W)),
        f.SLOT_DY: max(o.amax(p[1]) for p in passes),
        f.SLOT_Y: max(absmax(p[2]) for p in passes),
        f.SLOT_DX: max(absmax(p[3]) for p in passes),
    }
    for slot, v in expect.items():
        assert f32_bits(np.float32(amax[slot])) == f32_bits(np.float32(v)), slot
    for xb, dyb, _, _, X8, dY8 in passes:
        q, _ = o.quantize(xb, np.float32(scale0[f.SLOT_X]), o.E4M3)
        assert np.array_equal(host_u8(X8), q)
        q, _ = o.quantize(dyb, np.float32(scale0[f.SLOT_DY]), o.E5M2)
        assert np.array_equal(host_u8(dY8), q)
    lin.update()
    torch.cuda.synchronize()
    hist = lin.meta.history.cpu().numpy()
    assert np.array_equal(hist[:, 0].view(np.uint32), amax.view(np.uint32))
    assert np.array_equal(hist[:, 1:].view(np.uint32), hist0[:, :-1].view(np.uint32))
    assert not lin.meta.amax.cpu().numpy().any()
    f.fp8_sync_status()


def test_two_layers_on_two_streams_match_sequential_runs():
    """The library keeps no hidden per-call state: two layers stepping
    concurrently on two streams produce, bit for bit, what each produces when
    run alone (every output, every FP8 buffer and the whole scaling state)."""
    f = _lib()
    wa = wl.Workload("sa", 1040, 1024, 784, "normal", 1.0, 0.03, 1e-2, 16, 0, True, 3)
    wb = wl.Workload("sb", 512, 784, 1040, "normal", 1.0, 0.05, 1e-2, 16, 1, True, 3, seed=1)
    works = (wa, wb)
    inputs = {w.name: [(wl.layer_x(w, s, "cuda"), wl.layer_dy(w, s, "cuda")) for s in range(3)]
              for w in works}

    def make():
        return [f.Fp8Linear(wl.layer_weight(w, "cuda"), w.M,
                            f.Recipe(w.margin, w.history_len, w.hybrid)) for w in works]

    seq = make()
    for lin, w in zip(seq, works):
        for X, dY in inputs[w.name]:
            lin.step(X, dY)
    torch.cuda.synchronize()
    con = make()
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    for k in range(3):
        for lin, w, s in zip(con, works, streams):
            with torch.cuda.stream(s):
                X, dY = inputs[w.name][k]
                lin.step(X, dY)
    for s in streams:
        torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    bits = lambda t: t.view(torch.int16) if t.dtype == torch.bfloat16 else \
        (t.view(torch.int32) if t.dtype == torch.float32 else t)
    for a, b in zip(seq, con):
        for name in ("Y", "dX", "dW", "X8", "X8t", "W8", "W8t", "dY8", "dY8t"):
            assert torch.equal(bits(getattr(a, name)), bits(getattr(b, name))), name
        for name in ("history", "amax", "scale", "scale_inv"):
            assert torch.equal(bits(getattr(a.meta, name)), bits(getattr(b.meta, name))), name
    f.fp8_sync_status()
