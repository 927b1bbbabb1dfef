"""Pins for the oracle's decoupled-precision Adam (CPU only).

Sources: "Mixed-precision training" wiki note, bullet "precision decoupling"
(first moment FP8, second moment FP16, master weights FP16 with tensor
scaling; 16 -> 6 bytes per parameter) and its "Definition" table (FP16 max
65,504).  Pins: numpy float16 for the FP16 codec, torch.optim.AdamW (a library
routine, run in float64 on the decoded states) for the update, the closed
form of Adam's first step (sign descent), and the scale rule."""
import numpy as np
import torch

import oracle as o


def _bf16(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)


def _bf16_vals(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def test_f16_codec_matches_numpy():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(20000) * 10.0 ** rng.uniform(-9, 4.8, 20000)).astype(np.float32)
    v = v[np.abs(v) < 65504]
    assert np.array_equal(o.f16_encode(v), v.astype(np.float16).view(np.uint16))
    codes = np.arange(0, 0x7c00, 7, dtype=np.uint16)
    assert np.array_equal(o.f16_decode(codes), codes.view(np.float16).astype(np.float32))
    assert list(o.f16_encode(np.array([1e6, -1e6, np.inf], np.float32))) == [0x7bff, 0xfbff, 0x7bff]
    assert o.f16_decode(np.array([0x7bff], np.uint16))[0] == 65504.0


def _fresh_state(n, rng, wmag=0.05):
    w = (rng.standard_normal(n) * wmag).astype(np.float32)
    w_scale = np.float32(65504.0 / np.abs(w).max())
    return dict(m1=np.zeros(n, np.uint8), m1_scale=np.float32(1), m1_scale_inv=np.float32(1),
                m2=np.zeros(n, np.uint16), w16=o.f16_encode(w * w_scale), w_scale=w_scale,
                w_scale_inv=np.float32(1) / w_scale)


def test_first_step_is_sign_descent():
    """t = 1 from zero moments: m = (1-b1) g, v = (1-b2) g^2, so the update is
    g / (|g| + eps): a step of lr against the sign of g."""
    rng = np.random.default_rng(1)
    n = 4096
    st = _fresh_state(n, rng)
    g = _bf16(rng.standard_normal(n) * 1e-2)
    hp = o.AdamHyper(lr=1e-3)
    w0 = o.f16_decode(st["w16"]).astype(np.float64) * st["w_scale_inv"]
    m1, ms, msi, m2, w16, ws, wsi, wb, am = o.adam_step(g, st["m1"], st["m1_scale"],
                                                        st["m1_scale_inv"], st["m2"], st["w16"],
                                                        st["w_scale"], st["w_scale_inv"], hp, 1)
    gd = _bf16_vals(g)
    w1 = _bf16_vals(wb)
    assert np.allclose(w1, w0 - 1e-3 * np.sign(gd), rtol=0, atol=2 ** -8 * np.abs(w0).max() + 1e-7)
    assert np.isclose(am[0], 0.1 * np.abs(gd).max(), rtol=1e-6)
    # new first-moment codes: the largest lands on 448's code, the scale is 448 / amax
    assert (m1 & 0x7F).max() == 0x7E and ms == np.float32(448.0) / am[0]
    assert msi == np.float32(1.0) / ms and wsi == np.float32(1.0) / ws


def test_steps_match_torch_adamw():
    """Several steps, each compared with torch.optim.AdamW in float64 started
    from the oracle's decoded states: the moments agree to their storage
    precision (FP8 / FP16) and the weights to BF16 / FP16 rounding."""
    rng = np.random.default_rng(2)
    n = 8192
    st = _fresh_state(n, rng)
    hp = o.AdamHyper(lr=3e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    table = o.fp8_decode_table(o.E4M3)
    for t in range(1, 6):
        g = _bf16(rng.standard_normal(n) * 1e-2 * (1 + t))
        m_in = table[st["m1"]] * np.float64(st["m1_scale_inv"])
        v_in = o.f16_decode(st["m2"]).astype(np.float64)
        w_in = o.f16_decode(st["w16"]).astype(np.float64) * np.float64(st["w_scale_inv"])
        p = torch.nn.Parameter(torch.from_numpy(w_in.copy()))
        opt = torch.optim.AdamW([p], lr=hp.lr, betas=(hp.beta1, hp.beta2), eps=hp.eps,
                                weight_decay=hp.weight_decay)
        opt.state[p] = {"step": torch.tensor(float(t - 1)),
                        "exp_avg": torch.from_numpy(m_in.copy()),
                        "exp_avg_sq": torch.from_numpy(v_in.copy())}
        p.grad = torch.from_numpy(_bf16_vals(g))
        opt.step()
        out = o.adam_step(g, st["m1"], st["m1_scale"], st["m1_scale_inv"], st["m2"], st["w16"],
                          st["w_scale"], st["w_scale_inv"], hp, t)
        m1, ms, msi, m2, w16, ws, wsi, wb, am = out
        m_ref = opt.state[p]["exp_avg"].numpy()
        v_ref = opt.state[p]["exp_avg_sq"].numpy()
        w_ref = p.detach().numpy()
        m_got = table[m1] * np.float64(msi)
        assert np.all(np.abs(m_got - m_ref) <= 2 ** -4 * np.abs(m_ref) + 2 ** -9 / ms + 1e-12)
        v_got = o.f16_decode(m2).astype(np.float64)
        assert np.all(np.abs(v_got - v_ref) <= 2 ** -11 * np.abs(v_ref) + 2 ** -24)
        assert np.allclose(_bf16_vals(wb), w_ref, rtol=2 ** -8, atol=1e-9)
        w_got = o.f16_decode(w16).astype(np.float64) * np.float64(wsi)
        assert np.allclose(w_got, w_ref, rtol=2 ** -10, atol=1e-9)
        assert np.isclose(am[1], np.abs(w_ref).max(), rtol=1e-5)
        st = dict(m1=m1, m1_scale=ms, m1_scale_inv=msi, m2=m2, w16=w16, w_scale=ws,
                  w_scale_inv=wsi)


def test_zero_gradient_keeps_first_moment_scale():
    rng = np.random.default_rng(3)
    n = 256
    st = _fresh_state(n, rng)
    g = np.zeros(n, np.uint16)
    out = o.adam_step(g, st["m1"], np.float32(5.0), np.float32(0.2), st["m2"], st["w16"],
                      st["w_scale"], st["w_scale_inv"], o.AdamHyper(), 1)
    assert out[1] == 5.0 and out[2] == np.float32(0.2) and out[8][0] == 0.0


def _np_f16_bits(v32):
    """numpy's binary32 -> binary16 conversion (round to nearest even), after
    clipping to the largest finite FP16 value (the saturating reading)."""
    return np.clip(v32, -65504.0, 65504.0).astype(np.float16).view(np.uint16)


def test_initial_state_of_a_weight_tensor():
    """The initial master weights are the FP16 codes of w under the tensor
    scale that puts w's largest magnitude on FP16's largest finite value
    (65504, the wiki table): numpy's float16 conversion of the binary32
    product gives every code, the largest element lands on 0x7bff (or its
    negative), the decoded weights are within FP16 rounding of w, and the
    moments start at zero with unit scales."""
    rng = np.random.default_rng(4)
    for n, mag in ((4096, 0.02), (1000 * 16, 3.0), (16, 1e-3)):
        wb = _bf16(rng.standard_normal(n) * mag)
        w = _bf16_vals(wb)
        m1, ms, msi, m2, w16, ws, wsi, am = o.adam_init(wb, margin=0)
        assert not m1.any() and not m2.any() and ms == 1.0 and msi == 1.0
        assert am[0] == 0.0 and am[1] == np.float32(np.abs(w).max())
        assert np.array_equal(w16, _np_f16_bits(w.astype(np.float32) * ws))
        top = int(np.argmax(np.abs(w)))
        assert w16[top] & 0x7FFF == 0x7BFF
        back = o.f16_decode(w16).astype(np.float64) * np.float64(wsi)
        assert np.all(np.abs(back - w) <= 2 ** -11 * np.abs(w) + 2 ** -24 * float(wsi))
        assert wsi == np.float32(1.0) / ws


def test_initial_state_margin_and_zero_weights():
    rng = np.random.default_rng(5)
    wb = _bf16(rng.standard_normal(256) * 0.1)
    s0 = o.adam_init(wb, margin=0)[5]
    s1 = o.adam_init(wb, margin=1)
    assert s1[5] == s0 / 2
    top = int(np.argmax(np.abs(_bf16_vals(wb))))
    assert s1[4][top] & 0x7FFF == 0x77FF          # 32752 = 65504 / 2
    z = o.adam_init(np.zeros(64, np.uint16))
    assert z[5] == 1.0 and z[6] == 1.0 and not z[4].any() and z[7][1] == 0.0
