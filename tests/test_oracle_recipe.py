"""Pins for the oracle's amax, scaled cast and delayed-scaling update (CPU only).

Sources: "NVIDIA Transformer Engine and FP8 mixed precision: implementation
guide", section "Dynamic scaling and the FP8 recipe" (margin, Format.HYBRID,
amax_history_len; facts in tests/golden/recipe.txt), the Absolute-Max
statistic of "FP8 quantization with NVIDIA TensorRT", and the scale formula
(fmax / max(history)) / 2^margin of the delayed-scaling recipe.
"""
import io
import os

import numpy as np
import pytest
import torch

import oracle as o

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "recipe.txt")
F32_MAX = np.finfo(np.float32).max


def _golden():
    d = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            d[k] = v
    return d


def bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


# --------------------------------------------------------------------- amax --

def test_amax_planted_maximum_every_position_class():
    rng = np.random.default_rng(0)
    for n in [1, 7, 64, 1000, 4097]:
        x = rng.standard_normal(n).astype(np.float32)
        for pos in sorted({0, n // 2, n - 1}):
            y = x.copy()
            y[pos] = -1000.0 if pos % 2 else 1000.0
            assert o.amax(bf16_bits(y)) == np.float32(1000.0)


def test_amax_matches_numpy_and_specials():
    rng = np.random.default_rng(1)
    x = bf16_bits(rng.standard_normal(10000) * 3)
    ref = np.max(np.abs(torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()))
    assert o.amax(x) == ref
    assert o.amax(bf16_bits(np.zeros(100))) == 0
    negz = np.full(10, 0x8000, np.uint16)
    a = o.amax(negz)
    assert a == 0 and not np.signbit(a)
    with_nan = bf16_bits([1.0, np.nan, -2.0, np.nan])
    assert o.amax(with_nan) == 2.0                     # NaN skipped
    assert o.amax(bf16_bits([1.0, -np.inf])) == np.inf


# ----------------------------------------------------------------- the cast --

@pytest.mark.parametrize("fmt", [o.E4M3, o.E5M2])
def test_quantize_is_scaled_encode_with_transpose(fmt):
    rng = np.random.default_rng(3)
    x = bf16_bits(rng.standard_normal((48, 80)) * 10)
    s = np.float32(37.123)
    q, qt = o.quantize(x, s, fmt)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()
    v = (xf * s).astype(np.float32)                      # numpy binary32 multiply
    limit = 464.0 if fmt == o.E4M3 else 61440.0
    inr = np.abs(v) < limit
    tq = torch.from_numpy(np.where(inr, v, 0)).to(
        torch.float8_e4m3fn if fmt == o.E4M3 else torch.float8_e5m2).view(torch.uint8).numpy()
    top = 0x7E if fmt == o.E4M3 else 0x7B
    ref = np.where(inr, tq, np.where(v > 0, top, top | 0x80)).astype(np.uint8)
    assert np.array_equal(q, ref)
    assert np.array_equal(qt, q.T)


# -------------------------------------------------------------- the recipe --

def test_recipe_defaults_and_format_routing():
    g = _golden()
    rc = o.Recipe()
    assert rc.margin == int(g["margin_default"])
    assert rc.history_len == int(g["amax_history_len_default"])
    names = {o.E4M3: "E4M3", o.E5M2: "E5M2"}
    f = rc.formats()
    assert [names[f[i]] for i in (o.SLOT_X, o.SLOT_W, o.SLOT_Y)] == [g["hybrid_forward"]] * 3
    assert [names[f[i]] for i in (o.SLOT_DY, o.SLOT_DX)] == [g["hybrid_backward"]] * 2
    assert o.Recipe(hybrid=False).formats() == [o.E4M3] * 5


@pytest.mark.parametrize("fmt,fmax", [(o.E4M3, 448.0), (o.E5M2, 57344.0)])
def test_scale_closed_forms(fmt, fmax):
    h = np.zeros(16, np.float32)
    _, s, si = o.history_update(h, fmax, 1.0, 1.0, fmt, 0)
    assert s == 1.0 and si == 1.0
    _, s, si = o.history_update(h, 1.0, 1.0, 1.0, fmt, 0)
    assert s == fmax and si == np.float32(1.0) / np.float32(fmax)
    _, s, _ = o.history_update(h, 1.0, 1.0, 1.0, fmt, 1)
    assert s == fmax / 2
    _, s, _ = o.history_update(h, 2.0, 1.0, 1.0, fmt, 3)
    assert s == fmax / 16


def test_scale_margin_halves_exactly_and_inverse_is_f32_division():
    rng = np.random.default_rng(4)
    for a in (rng.standard_normal(200) * 10.0 ** rng.integers(-30, 30, 200)).astype(np.float32):
        a = np.float32(abs(a)) or np.float32(1.0)
        prev = None
        for margin in range(0, 6):
            _, s, si = o.history_update(np.zeros(4, np.float32), a, 1, 1, o.E4M3, margin)
            assert si == np.float32(1.0) / s                 # numpy binary32 division
            if prev is not None and np.isfinite(prev) and prev < F32_MAX and s > 2.0 ** -120:
                assert s == prev / 2
            prev = s


def test_largest_element_lands_on_largest_code():
    """With margin 0 and the current amax equal to max(history), the largest
    element of the tensor casts to the largest finite code."""
    rng = np.random.default_rng(5)
    for fmt, top in [(o.E4M3, 0x7E), (o.E5M2, 0x7B)]:
        for trial in range(20):
            x = bf16_bits(rng.standard_normal((8, 32)) * 10.0 ** rng.uniform(-5, 5))
            a = o.amax(x)
            _, s, _ = o.history_update(np.zeros(8, np.float32), a, 1, 1, fmt, 0)
            q, _ = o.quantize(x, s, fmt)
            assert (q & 0x7F).max() == top


def test_margin_trades_overflow_for_underflow():
    """A larger margin gives no more saturated elements and no fewer flushed
    to zero (the recipe section's description of margin)."""
    rng = np.random.default_rng(6)
    x = bf16_bits(rng.standard_normal((64, 64)) * np.exp(rng.standard_normal((64, 64)) * 3))
    stale = np.float32(o.amax(x) / 8)           # history lags behind the tensor
    sat, under = [], []
    for margin in range(6):
        _, s, _ = o.history_update(np.zeros(4, np.float32), stale, 1, 1, o.E4M3, margin)
        q, _ = o.quantize(x, s, o.E4M3)
        xf = o.bf16_to_f32(x)
        sat.append(int(np.sum((q & 0x7F) == 0x7E)))
        under.append(int(np.sum(((q & 0x7F) == 0) & (xf != 0))))
    assert all(a >= b for a, b in zip(sat, sat[1:])) and sat[0] > sat[-1]
    assert all(a <= b for a, b in zip(under, under[1:])) and under[-1] > under[0]


def test_history_window_spike_enters_persists_and_leaves():
    L = 16
    h = np.zeros(L, np.float32)
    s, si = np.float32(1), np.float32(1)
    seq = [1.0] * 5 + [100.0] + [1.0] * 30
    scales = []
    for a in seq:
        h, s, si = o.history_update(h, a, s, si, o.E4M3, 0)
        scales.append(s)
    assert h[0] == 1.0 and h.max() == 1.0 and h.size == L
    assert scales[4] == 448.0
    spike = [i for i, v in enumerate(scales) if v == np.float32(448.0) / np.float32(100.0)]
    assert spike == list(range(5, 5 + L))        # exactly L steps
    assert scales[5 + L] == 448.0


def test_zero_and_nonfinite_history_keep_scale_and_overflow_clamps():
    h = np.zeros(8, np.float32)
    h2, s, si = o.history_update(h, 0.0, 3.0, np.float32(1 / 3), o.E4M3, 0)
    assert s == 3.0 and si == np.float32(1 / 3) and h2[0] == 0
    _, s, si = o.history_update(h, np.inf, 3.0, 0.5, o.E4M3, 0)
    assert s == 3.0 and si == 0.5
    tiny = np.float32(2.0 ** -133)               # smallest BF16 subnormal
    _, s, si = o.history_update(h, tiny, 1.0, 1.0, o.E4M3, 0)
    assert s == F32_MAX and si == np.float32(1.0) / F32_MAX


def test_state_save_restore_gives_identical_next_scales():
    """The scaling state is checkpointed with the model; restoring it must give
    bit-identical scales and histories afterwards."""
    rng = np.random.default_rng(7)
    rc = o.Recipe(margin=0, history_len=8)
    amaxes = (np.abs(rng.standard_normal((12, 5))) * 10.0 ** rng.integers(-3, 3, (12, 1))
              ).astype(np.float32)

    def run(st, rows):
        for a in rows:
            st.amax[:] = a
            o.layer_update(st, rc)
        return st

    full = run(o.State.initial(8), amaxes)
    part = run(o.State.initial(8), amaxes[:5])
    buf = io.BytesIO()
    np.savez(buf, h=part.history, s=part.scale, si=part.scale_inv)
    buf.seek(0)
    z = np.load(buf)
    resumed = run(o.State(z["h"].copy(), np.zeros(5, np.float32), z["s"].copy(), z["si"].copy()),
                  amaxes[5:])
    assert np.array_equal(full.history.view(np.uint32), resumed.history.view(np.uint32))
    assert np.array_equal(full.scale.view(np.uint32), resumed.scale.view(np.uint32))
    assert np.array_equal(full.scale_inv.view(np.uint32), resumed.scale_inv.view(np.uint32))


# -------------------------------------------------- just-in-time scaling --

def test_just_in_time_scaling_uses_this_steps_amax():
    """Under just-in-time scaling (margin 0) the scale is fmax / amax of the
    tensor being cast, so its largest element lands on the largest code at
    every step, including the first; an all-zero tensor keeps the scale."""
    rng = np.random.default_rng(8)
    rc = o.Recipe(margin=0, history_len=4, hybrid=True, current=True)
    st = o.State.initial(4)
    W = bf16_bits(rng.standard_normal((16, 32)) / 4)
    for step, mag in enumerate([1.0, 300.0, 1e-3, 0.0, 7.0]):
        X = bf16_bits(rng.standard_normal((16, 32)) * mag)
        dY = bf16_bits(rng.standard_normal((16, 16)) * mag * 1e-2)
        prev_x = st.scale[o.SLOT_X]
        fo = o.layer_fwd(st, rc, X, W)
        bo = o.layer_bwd(st, rc, dY, fo["X8t"], fo["W8t"])
        if mag == 0.0:
            assert st.scale[o.SLOT_X] == prev_x and np.all((fo["X8"] & 0x7F) == 0)
        else:
            assert st.scale[o.SLOT_X] == np.float32(448.0) / o.amax(X)
            assert (fo["X8"] & 0x7F).max() == 0x7E
            assert (bo["dY8"] & 0x7F).max() == 0x7B
            assert st.scale_inv[o.SLOT_DY] == np.float32(1.0) / st.scale[o.SLOT_DY]
        assert (fo["W8"] & 0x7F).max() == 0x7E
        o.layer_update(st, rc)


def test_just_in_time_differs_from_delayed_only_by_the_scale_source():
    """The same step under the two recipes: delayed scaling casts with the
    scale left by the previous update, just-in-time with fmax / amax now."""
    rng = np.random.default_rng(9)
    X = bf16_bits(rng.standard_normal((16, 32)) * 50)
    W = bf16_bits(rng.standard_normal((16, 32)))
    d = o.State.initial(4)
    c = o.State.initial(4)
    fd = o.layer_fwd(d, o.Recipe(history_len=4), X, W)
    fc = o.layer_fwd(c, o.Recipe(history_len=4, current=True), X, W)
    assert d.scale[o.SLOT_X] == 1.0
    q, _ = o.quantize(X, np.float32(1.0), o.E4M3)
    assert np.array_equal(fd["X8"], q)
    q, _ = o.quantize(X, np.float32(448.0) / o.amax(X), o.E4M3)
    assert np.array_equal(fc["X8"], q)
