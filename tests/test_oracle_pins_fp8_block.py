"""Pins of the oracle's FP8 mode: E4M3 block linears with delayed per-tensor scaling (CPU only).

"FP8 training for Flux models", §Configuration › FP8 model configuration: E4M3 operands, a
per-tensor scale from the most recent amax (margin 0), attention kept out of FP8.  The pins
fix what that mode computes without re-using its code:
* scales divide out exactly when they are powers of two and no value leaves the normal range;
* a linear's error stays inside the E4M3 rounding bound (half a step, 2^-4 relative, per
  operand);
* the tensor names map to the right tensors (the recorded amax of each weight is that weight's
  max |w|, of the QKV input the max of the LayerNorm-modulated stream);
* the image and text streams keep separate scales (a text-only scale leaves the image output
  untouched after the joint attention);
* the output projection reads the attention output in the activation type (bf16 values).
"""
import numpy as np

from diffusion_transformer_flux_gb300 import synth
from oracle import e4m3 as E
from oracle import flux as O

RNG = np.random.default_rng(23)
NAMES = ("qkv", "o", "fc1", "fc2")


def test_power_of_two_scales_divide_out_exactly():
    # |x|, |w| in [0.1, 10]: with scales 2^a, 2^b (a, b <= 4) every scaled value stays a normal
    # E4M3 number below 448, so quantize(v * 2^a) / 2^a == quantize(v) and the result matches
    # the unscaled one bit for bit.  A kernel that multiplied by the scales instead of dividing,
    # or used one scale twice, would not.
    x = RNG.uniform(0.1, 10, (7, 33)) * RNG.choice([-1, 1], (7, 33))
    w = RNG.uniform(0.1, 10, (5, 33)) * RNG.choice([-1, 1], (5, 33))
    b = RNG.standard_normal(5)
    ref = E.fp8_linear(x, w, b, 1.0, 1.0)
    for a, c in ((4, -3), (-2, 2), (3, 3)):
        np.testing.assert_array_equal(E.fp8_linear(x, w, b, 2.0 ** a, 2.0 ** c), ref)


def test_fp8_linear_error_within_the_e4m3_rounding_bound():
    # Normal-range E4M3 rounding moves a value by at most half a step, 2^-4 of its magnitude,
    # so |x_q w_q - x w| <= (2 * 2^-4 + 2^-8) |x| |w| term by term.
    x = RNG.standard_normal((9, 64))
    w = RNG.standard_normal((11, 64)) * 0.05
    sx = E.delayed_scale(np.abs(x).max())
    sw = E.delayed_scale(np.abs(w).max())
    got = E.fp8_linear(x, w, None, sx, sw)
    bound = (2 * 2.0 ** -4 + 2.0 ** -8) * (np.abs(x) @ np.abs(w).T)
    # values that fall below the normal range (2^-6 / s) may lose up to half a subnormal step
    tiny = 2.0 ** -10 * (np.abs(x).sum(1, keepdims=True) / sw + np.abs(w).sum(1)[None, :] / sx)
    assert np.all(np.abs(got - x @ w.T) <= bound + tiny)
    # and the error is not trivially zero: the cast really happened
    assert np.abs(got - x @ w.T).max() > 1e-4 * np.abs(x @ w.T).max()


def test_delayed_scale_puts_the_amax_element_at_448():
    ds = E.DelayedScaling()
    x = RNG.standard_normal((6, 32))
    w = RNG.standard_normal((4, 32))
    ds.linear("t", x, w, None)
    nxt = ds.next_scales()
    assert set(nxt) == {"t.x", "t.w"}
    for name, a in (("t.x", x), ("t.w", w)):
        q = E.e4m3_quantize(a * nxt[name])
        assert np.abs(q).max() == 448.0
        assert np.all((np.abs(q) == 448.0) == (np.abs(a) == np.abs(a).max()))


def _case(D=32, H=2, F=64, S_i=9, S_t=5, B=2, seed=3):
    rng = np.random.default_rng(seed)
    wi = synth.stream_weights(rng, D, H, D // H, F, "bf16", 0.2)
    wt = synth.stream_weights(rng, D, H, D // H, F, "bf16", 0.2)
    inp = synth.block_inputs(B, S_i, S_t, D, "bf16", seed)
    ax = (4, 6, 6)
    cos, sin = O.rope_cos_sin(inp.ids, ax)
    return inp, wi, wt, cos, sin, H


def test_tensor_names_record_the_right_tensors():
    inp, wi, wt, cos, sin, H = _case()
    ds = E.DelayedScaling()
    O.double_block(inp.x_img, inp.x_txt, inp.vec, cos, sin, wi, wt, H, mm_cast=O.round_bf16, fp8=ds)
    assert set(ds.amax) == {f"{s}.{n}.{o}" for s in ("img", "txt") for n in NAMES for o in "xw"}
    for s, w in (("img", wi), ("txt", wt)):
        for n, key in zip(NAMES, ("w_qkv", "w_o", "w_1", "w_2")):
            assert ds.amax[f"{s}.{n}.w"] == np.abs(w[key]).max()
    for s, x, w in (("img", inp.x_img, wi), ("txt", inp.x_txt, wt)):
        m = O.modulation(inp.vec, w["w_mod"], w["b_mod"], mm_cast=O.round_bf16)
        assert ds.amax[f"{s}.qkv.x"] == np.abs(O.modulate(x, m[0], m[1])).max()
        # the output projection reads bf16 values (the attention's output type)
        a = ds.amax[f"{s}.o.x"]
        assert O.round_bf16(a) == a
    ds1 = E.DelayedScaling()
    x = np.concatenate([inp.x_img, inp.x_txt], axis=1)
    O.single_block(x, inp.vec, cos, sin, wi, H, mm_cast=O.round_bf16, fp8=ds1)
    assert set(ds1.amax) == {f"single.{n}.{o}" for n in NAMES for o in "xw"}


def test_streams_keep_separate_scales():
    inp, wi, wt, cos, sin, H = _case(seed=5)
    ds = E.DelayedScaling()
    args = (inp.x_img, inp.x_txt, inp.vec, cos, sin, wi, wt, H)
    O.double_block(*args, mm_cast=O.round_bf16, fp8=ds)
    scales = ds.next_scales()
    base = O.double_block(*args, mm_cast=O.round_bf16, fp8=E.DelayedScaling(scales))
    # a text-stream tensor after the attention: only the text output moves
    for name in ("txt.o.x", "txt.fc1.w", "txt.fc2.x"):
        sc = dict(scales, **{name: scales[name] * 0.37})
        y = O.double_block(*args, mm_cast=O.round_bf16, fp8=E.DelayedScaling(sc))
        np.testing.assert_array_equal(y[0], base[0])
        assert np.abs(y[1] - base[1]).max() > 0
    # the image stream's QKV input feeds the joint attention: both outputs move
    sc = dict(scales, **{"img.qkv.x": scales["img.qkv.x"] * 0.37})
    y = O.double_block(*args, mm_cast=O.round_bf16, fp8=E.DelayedScaling(sc))
    assert np.abs(y[0] - base[0]).max() > 0 and np.abs(y[1] - base[1]).max() > 0


def test_fp8_block_stays_near_the_exact_block():
    # Each operand rounding errs by at most 2^-4 relative (RMS 2^-3/sqrt(12) ~ 3.6%), so each
    # linear deviates by ~5% norm-wise and the block, whose branches here are of the size of the
    # residual, by well under 15%.  A scale applied the wrong way round errs by orders more.
    inp, wi, wt, cos, sin, H = _case(D=64, H=4, F=128, S_i=20, S_t=7, seed=9)
    args = (inp.x_img, inp.x_txt, inp.vec, cos, sin, wi, wt, H)
    ref = O.double_block(*args)
    ds = E.DelayedScaling()
    O.double_block(*args, mm_cast=O.round_bf16, fp8=ds)
    y = O.double_block(*args, mm_cast=O.round_bf16, fp8=E.DelayedScaling(ds.next_scales()))
    for a, r in zip(y, ref):
        rel = np.linalg.norm(a - r) / np.linalg.norm(r)
        assert 1e-4 < rel < 0.15, rel


def test_history_scale_algorithms_and_margin():
    hist = [3.0, 10.0, 0.5, 2.0]
    assert E.history_scale(hist, "most_recent") == 448.0 / 2.0
    assert E.history_scale(hist, "max") == 448.0 / 10.0
    # the margin halves the scale per unit, exactly
    assert E.history_scale(hist, "max", margin=2) == 448.0 / 10.0 / 4.0
    assert E.history_scale([], "max") == 1.0 and E.history_scale([0.0, 0.0], "max") == 1.0
    # most_recent over a run of evaluations is what DelayedScaling.next_scales gives
    rng = np.random.default_rng(4)
    seen = []
    for f in (1.0, 5.0, 0.25):
        ds = E.DelayedScaling()
        ds.linear("t", rng.standard_normal((4, 16)) * f, rng.standard_normal((3, 16)), None)
        seen.append(ds.amax["t.x"])
        assert E.history_scale(seen, "most_recent") == ds.next_scales()["t.x"]
    # max never lets a value that was seen saturate: 448 / max keeps every recorded amax <= 448
    s = E.history_scale(seen, "max")
    assert all(a * s <= 448.0 * (1 + 1e-15) for a in seen)
