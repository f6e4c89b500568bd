"""Pins of the oracle's parallel-branch single block (CPU only).

The parallel block shares one LayerNorm-modulate between the attention and the MLP and adds
both through one gated residual.  Its two halves are pinned against the sequential single
block, whose own pins fix the attention and MLP branches:
* with the MLP silenced (W_1 = 0, b_1 = 0, so GELU(0) = 0; b_2 = 0) it equals the sequential
  block whose MLP gate is zero;
* with the attention projection silenced (W_o = 0, b_o = 0) it equals the sequential block
  whose attention gate is zero and whose second LayerNorm takes the same shift and scale;
* a zero gate gives the identity; the row-sampled form equals the full one at those rows.
"""
import numpy as np

from diffusion_transformer_flux_gb300 import synth
from oracle import flux as O

AX = (4, 6, 6)


def _case(seed, B=2, S=13, D=32, H=2, F=64):
    rng = np.random.default_rng(seed)
    w = synth.stream_weights(rng, D, H, D // H, F, "f32", 0.2, gain_jitter=0.1)
    w["w_mod"], w["b_mod"] = w["w_mod"][:3 * D], w["b_mod"][:3 * D]
    x = rng.standard_normal((B, S, D))
    vec = rng.standard_normal((B, D))
    ids = synth.position_ids(B, 3, 3, S - 9)
    cos, sin = O.rope_cos_sin(ids, AX)
    return w, x, vec, cos, sin, H, D, rng


def _sequential_weights(w, D, rng, chunks):
    """A 6-chunk modulation whose rows reproduce the given chunk choice: 'p0' / 'p1' / 'p2' take
    the parallel block's shift / scale / gate rows, 0 a zero chunk."""
    ws = dict(w)
    rows_w, rows_b = [], []
    for ch in chunks:
        if ch == 0:
            rows_w.append(np.zeros((D, D))), rows_b.append(np.zeros(D))
        else:
            i = int(ch[1])
            rows_w.append(w["w_mod"][i * D:(i + 1) * D]), rows_b.append(w["b_mod"][i * D:(i + 1) * D])
    ws["w_mod"], ws["b_mod"] = np.concatenate(rows_w), np.concatenate(rows_b)
    return ws


def test_attention_half_is_the_sequential_attention_branch():
    w, x, vec, cos, sin, H, D, rng = _case(1)
    w = dict(w, w_1=np.zeros_like(w["w_1"]), b_1=np.zeros_like(w["b_1"]), b_2=np.zeros_like(w["b_2"]))
    got = O.single_block_parallel(x, vec, cos, sin, w, H)
    seq = O.single_block(x, vec, cos, sin, _sequential_weights(w, D, rng, ["p0", "p1", "p2", "p0", "p1", 0]), H)
    np.testing.assert_allclose(got, seq, atol=1e-12)
    assert np.abs(got - x).max() > 1e-2  # the branch is really there


def test_mlp_half_is_the_sequential_mlp_branch():
    w, x, vec, cos, sin, H, D, rng = _case(2)
    w = dict(w, w_o=np.zeros_like(w["w_o"]), b_o=np.zeros_like(w["b_o"]))
    got = O.single_block_parallel(x, vec, cos, sin, w, H)
    seq = O.single_block(x, vec, cos, sin, _sequential_weights(w, D, rng, ["p0", "p1", 0, "p0", "p1", "p2"]), H)
    np.testing.assert_allclose(got, seq, atol=1e-12)
    assert np.abs(got - x).max() > 1e-2


def test_zero_gate_and_row_sampling():
    w, x, vec, cos, sin, H, D, rng = _case(3)
    w0 = dict(w, w_mod=w["w_mod"].copy(), b_mod=w["b_mod"].copy())
    w0["w_mod"][2 * D:], w0["b_mod"][2 * D:] = 0, 0
    np.testing.assert_array_equal(O.single_block_parallel(x, vec, cos, sin, w0, H), x)
    full = O.single_block_parallel(x, vec, cos, sin, w, H)
    rows = np.array([0, 5, 12, 7])
    np.testing.assert_allclose(O.single_block_parallel(x, vec, cos, sin, w, H, rows=rows), full[:, rows], atol=1e-13)


def test_both_branches_read_the_same_input():
    # full = attention-only + MLP-only - x: the branches add, both computed from x (a block whose
    # MLP read the attention-updated stream, as the sequential one does, fails this)
    w, x, vec, cos, sin, H, D, rng = _case(4)
    full = O.single_block_parallel(x, vec, cos, sin, w, H)
    attn = O.single_block_parallel(x, vec, cos, sin, dict(w, w_1=np.zeros_like(w["w_1"]),
                                                          b_1=np.zeros_like(w["b_1"]),
                                                          b_2=np.zeros_like(w["b_2"])), H)
    mlp = O.single_block_parallel(x, vec, cos, sin, dict(w, w_o=np.zeros_like(w["w_o"]),
                                                         b_o=np.zeros_like(w["b_o"])), H)
    np.testing.assert_allclose(full, attn + mlp - x, atol=1e-12)
    seq_like = O.single_block(x, vec, cos, sin, _sequential_weights(w, D, rng, ["p0", "p1", "p2", "p0", "p1", "p2"]), H)
    assert np.abs(seq_like - full).max() > 1e-3
