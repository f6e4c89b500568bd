"""GPU parity of the FP8 E4M3 path: the cast, the FP8 linear, and the blocks with E4M3 linears.

"FP8 training for Flux models", §Configuration › FP8 model configuration: the four linears
of each stream run on E4M3 operands with per-tensor delayed scaling (most_recent, margin 0);
attention stays bf16.

What is compared, and why:
* The cast is bit-exact: both sides round the float32 product x * scale to E4M3.
* The FP8 linear, fed the same codes (power-of-two scales make the products exact on both
  sides), agrees to fp32-accumulation level.
* In a block, every E4M3 cast turns a difference smaller than one E4M3 step into a whole-step
  difference in some codes, so two correct evaluations whose attention outputs differ at the
  bf16 level already differ by ~0.3 x RMS element-wise at the output (measured on the oracle).
  So the block is checked
    - element-wise wherever both sides take the same decisions: the LayerNorm-modulate codes,
      Q, K, V^T after the FP8 QKV linear, the attention output, and, with V = 0 (an attention
      output of exact zeros), the whole chain after the attention;
    - norm-wise at the output: ||y - y64|| / ||y64|| <= 6e-2 against the float64 block, and
      no more than 1.5x the deviation of an exact FP8 evaluation (the oracle's) at the same
      scales;
    - in max norm at the output: max|y - y64| / RMS at most 1.5x the exact FP8 evaluation's,
      and max|y - y8| / RMS (GPU against the exact FP8 evaluation) at most the exact FP8
      evaluation's own max|y8 - y64| / RMS.
* The delayed-scaling state: the recorded amax of every weight is its max |w| exactly, that of
  the QKV input matches the oracle, and scale = 448 / amax afterwards.
"""
import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import synth
from oracle import e4m3 as E
from oracle import flux as O

from gpu_util import BlockCase, assert_parity, dev, host, upload_weights, workspace_view

pytestmark = pytest.mark.gpu
NAMES = ("qkv", "o", "fc1", "fc2")
HIST = 1024


@pytest.fixture(scope="module", autouse=True)
def _lib_loaded():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()


def _codes_f32(x, s):
    """E4M3 codes of x * s with the product rounded to float32 first (the kernels' order)."""
    p = (np.asarray(x, np.float32) * np.float32(s)).astype(np.float64)
    return E.e4m3_encode(p)


_DEC = np.array([E.e4m3_decode(c) for c in range(256)])


# ----------------------------------------------------------------------------- the cast
@pytest.mark.parametrize("n", [16, 16 * 1001, 16384 * 3 + 48])
@pytest.mark.parametrize("scale", [1.0, 448.0 / 3.7, 2.0 ** -5])
def test_quantize_e4m3_bit_exact(n, scale):
    rng = np.random.default_rng(n)
    mag = rng.choice([1e-4, 1e-2, 1.0, 30.0, 3000.0], size=n)
    x = synth.bf16_round(rng.standard_normal(n) * mag)
    x[:8] = [0.0, -0.0, 448.0 / scale, -1e30, 2.0 ** -12, -2.0 ** -10, 1.0625, 1e-38]
    x = synth.bf16_round(x)
    xt = torch.from_numpy(x).cuda().to(torch.bfloat16)
    s = torch.tensor([scale], dtype=torch.float32, device="cuda")
    amax = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    L.mmdit_fp8_quantize_e4m3(xt, s, amax, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), _codes_f32(x, np.float32(scale)))
    assert amax.item() == max(0.5, float(np.abs(x).max()))


def test_quantize_keeps_a_larger_recorded_amax():
    x = torch.ones(32, dtype=torch.bfloat16, device="cuda")
    s = torch.ones(1, device="cuda")
    amax = torch.tensor([7.0], device="cuda")
    out = torch.empty(32, dtype=torch.uint8, device="cuda")
    L.mmdit_fp8_quantize_e4m3(x, s, amax, out)
    assert amax.item() == 7.0
    assert (out == 0x38).all()  # 1.0


# ----------------------------------------------------------------------------- the linear
def _pow2_scale(a):
    """The largest power of two s with amax * s <= 448."""
    return 2.0 ** np.floor(np.log2(448.0 / a))


@pytest.mark.parametrize("M,N,K", [(300, 256, 3072), (130, 384, 112), (1, 128, 16), (257, 3072, 3072)])
def test_fp8_linear_matches_oracle(M, N, K):
    rng = np.random.default_rng(M + N + K)
    x = synth.bf16_round(rng.standard_normal((M, K)))
    w = synth.bf16_round(rng.standard_normal((N, K)) * 0.02)
    b = synth.bf16_round(rng.standard_normal(N) * 0.02)
    sx, sw = _pow2_scale(np.abs(x).max()), _pow2_scale(np.abs(w).max())
    scales = torch.tensor([sx, sw], dtype=torch.float32, device="cuda")
    amax = torch.zeros(2, device="cuda")
    xq = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    wq = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    L.mmdit_fp8_quantize_e4m3(dev(x), scales[0:1], amax[0:1], xq)
    L.mmdit_fp8_quantize_e4m3(dev(w), scales[1:2], amax[1:2], wq)
    y = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    ws = L.mmdit_fp8_linear_fwd(xq, wq, scales[0:1], scales[1:2], dev(b), y)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    ref = E.fp8_linear(x, w, b, sx, sw)
    # the same codes on both sides: only the fp32 accumulation order and the bf16 output differ
    assert_parity(host(y), ref, 2e-3, "FP8 linear", out_bf16=True)


# ----------------------------------------------------------------------------- blocks
def _fp8_dims(case):
    return L.make_dims(case.B, case.S_i, case.S_t, case.D, case.H, case.F, L.MMDIT_BF16,
                       rope_interleaved=case.interleaved, gelu_tanh=case.gelu_tanh,
                       gemm=L.MMDIT_GEMM_FP8_E4M3)


class Fp8Run:
    """A block case run through the C ABI with E4M3 linears, two calls in a row on the same
    inputs: the first with the empty-history scales (1), the second with the scales the first
    recorded (the delayed-scaling protocol)."""

    def __init__(self, case: BlockCase, calls=2):
        self.case = case
        c = case
        self.dims = _fp8_dims(c)
        n_t = 8 if c.single else 16
        self.hist = torch.zeros(n_t, HIST, device="cuda")
        self.scale = torch.ones(n_t, device="cuda")
        ids = torch.from_numpy(c.ids).cuda()
        cos = torch.empty(c.B, c.S, 64, device="cuda")
        sin = torch.empty_like(cos)
        L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
        vec = dev(c.vec)
        wi = upload_weights(c.w_img, "bf16")
        self.scales_used = []
        for call in range(calls):
            self.scales_used.append(self.scale.cpu().numpy().copy())
            st = L.make_fp8_state(self.hist, self.scale, pos=call)
            if c.single:
                x = dev(c.x_joint())
                y = torch.empty_like(x)
                ws = L.mmdit_single_block_fwd(self.dims, wi, vec, cos, sin, x, y, fp8=st)
                outs = (y,)
            else:
                wt = upload_weights(c.w_txt, "bf16")
                xi, xt = dev(c.x_img), dev(c.x_txt)
                yi, yt = torch.empty_like(xi), torch.empty_like(xt)
                ws = L.mmdit_double_block_fwd(self.dims, wi, wt, vec, cos, sin, xi, xt, yi, yt, fp8=st)
                outs = (yi, yt)
            torch.cuda.synchronize()
            assert L.mmdit_workspace_status(ws) == 0
        self.ws = ws
        self.y = tuple(host(o) for o in outs)
        self.amax = self.hist.cpu().numpy()  # [n_t, HIST]
        self.scale_after = self.scale.cpu().numpy()

    def slots(self):
        return [("single", 0)] if self.case.single else [("img", 0), ("txt", 1)]

    def name_of(self, t):
        slot, rem = divmod(t, 8)
        s = self.slots()[slot][0] if slot < len(self.slots()) else None
        return f"{s}.{NAMES[rem // 2]}.{'xw'[rem % 2]}"


def _oracle_fp8(case, scales=None, rows=None):
    """The oracle with E4M3 linears (bf16 elsewhere) at the given scales; returns (outputs, ds)."""
    ds = E.DelayedScaling(scales or {})
    args = dict(mm_cast=O.round_bf16, fp8=ds, interleaved=case.interleaved, gelu_tanh=case.gelu_tanh)
    if case.single:
        x = case.x_joint()
        if rows is None:
            y = (O.single_block(x, case.vec, case.cos, case.sin, case.w_img, case.H, **args),)
        else:
            y = (O.single_block_rows(x, case.vec, case.cos, case.sin, case.w_img, case.H, rows[0], **args),)
    elif rows is None:
        y = O.double_block(case.x_img, case.x_txt, case.vec, case.cos, case.sin, case.w_img, case.w_txt,
                           case.H, **args)
    else:
        y = O.double_block_rows(case.x_img, case.x_txt, case.vec, case.cos, case.sin, case.w_img,
                                case.w_txt, case.H, rows[0], rows[1], **args)
    return y, ds


def _oracle_two_calls(case, rows=None):
    _, ds1 = _oracle_fp8(case, rows=rows)
    sc = ds1.next_scales()
    y, ds2 = _oracle_fp8(case, sc, rows=rows)
    return y, sc, ds1


def _check_state(run: Fp8Run, ds1, tol=None, sampled=False):
    """The amax the first call recorded (column 0) and the scales the last call left.

    Weights: max |w| exactly.  Inputs: within tol[linear] (relative) of the oracle's amax; with
    `sampled` rows the oracle saw only some rows after the attention, so there the recorded
    amax must only be at least the oracle's (less a bf16-level margin)."""
    tol = dict({"qkv": 1e-5, "o": 0.1, "fc1": 0.1, "fc2": 0.1}, **(tol or {}))
    a0 = run.amax[:, 0]
    for t in range(len(a0)):
        name = run.name_of(t)
        ref = ds1.amax[name]
        lin = name.split(".")[1]
        if name.endswith(".w"):
            assert a0[t] == np.float32(ref), (name, a0[t], ref)  # max |w| of bf16 values, exact
        elif sampled and lin != "qkv":
            assert a0[t] >= ref * (1 - 1e-2), (name, a0[t], ref)
        else:
            assert abs(a0[t] - ref) <= tol[lin] * ref, (name, a0[t], ref)
    # scale after the last call = 448 / its recorded amax (float32 division)
    last = run.amax[:, len(run.scales_used) - 1]
    for t in range(len(last)):
        if last[t] > 0:
            assert run.scale_after[t] == np.float32(448.0) / np.float32(last[t]), run.name_of(t)
        else:
            assert run.scale_after[t] == run.scales_used[-1][t]


def _check_codes(got, h, s_gpu, s_oracle, what):
    """E4M3 codes `got` of the values h: each is a valid rounding of h * s_gpu (half an E4M3
    step, or half a subnormal step, plus float32 rounding of h), and the oracle's decisions at
    its own scale agree almost everywhere."""
    hs = h * s_gpu
    err = np.abs(_DEC[got] - hs)
    assert np.all(err <= 2.0 ** -4 * np.abs(hs) * (1 + 1e-5) + 2.0 ** -10 + 1e-6 * np.abs(hs)), what
    same = np.mean(got == E.e4m3_encode(h * s_oracle))
    assert same >= 0.999, (what, same)


def _check_pre_attention(run: Fp8Run, sc):
    """Q, K, V^T after the FP8 QKV linear, and the attention output, of the last call."""
    case = run.case
    offs = L.mmdit_block_workspace_offsets(run.dims, case.single)
    B, H, S, D = case.B, case.H, case.S, case.D
    S_pad = (S + 7) // 8 * 8
    streams = [("single" if case.single else "img", case.x_joint() if case.single else case.x_img,
                case.w_img)]
    if not case.single:
        streams.append(("txt", case.x_txt, case.w_txt))
    qs, ks, vs = [], [], []
    for name, x, w in streams:
        m = O.modulation(case.vec, w["w_mod"], w["b_mod"], mm_cast=O.round_bf16)
        q, kk, v = O.qkv_heads(x, m[0], m[1], w, H, mm_cast=O.round_bf16, fp8=E.DelayedScaling(sc),
                               name=name)
        qs.append(q), ks.append(kk), vs.append(v)
    q, k, v = (np.concatenate(a, axis=2) for a in (qs, ks, vs))
    cs, sn = case.cos[:, None], case.sin[:, None]
    q = O.apply_rope(q, cs, sn, case.interleaved)
    k = O.apply_rope(k, cs, sn, case.interleaved)
    gq = host(workspace_view(run.ws, offs[2], (B, H, S, 128), torch.bfloat16))
    gk = host(workspace_view(run.ws, offs[3], (B, H, S, 128), torch.bfloat16))
    gvt = host(workspace_view(run.ws, offs[4], (B, H, 128, S_pad), torch.float16))[..., :S]
    assert_parity(gq, q, 2e-2, "Q after FP8 QKV + RMSNorm + RoPE", out_bf16=True)
    assert_parity(gk, k, 2e-2, "K after FP8 QKV + RMSNorm + RoPE", out_bf16=True)
    assert_parity(gvt, np.swapaxes(v, -1, -2), 2e-2, "V^T after FP8 QKV", out_bf16=True)
    o = O.attention(q, k, v, O.round_bf16).transpose(0, 2, 1, 3).reshape(B, S, D)
    rows_i = B * (S if case.single else case.S_i)
    go = host(workspace_view(run.ws, offs[5], (rows_i, D), torch.bfloat16)).reshape(B, -1, D)
    assert_parity(go, o if case.single else o[:, :case.S_i], 2e-2, "attention output", out_bf16=True)


def _check_norm_wise(got, y8, y64, what, factor=1.5):
    """Norm-wise and max-norm bars of a whole FP8 block (y8: the exact-E4M3 oracle at the GPU's
    scales; y64: the float64 block).  Max norm: the GPU's largest element error against float64
    may be at most `factor` x the exact-E4M3 evaluation's own, and the GPU may sit no further
    from the exact-E4M3 evaluation than that evaluation sits from float64 -- so a mistake confined
    to a few rows or heads, which a norm would average away, still fails."""
    for g, a, r, n in zip(got, y8, y64, ("first", "second")):
        if r.size == 0:
            continue
        e_gpu = np.linalg.norm(g - r) / np.linalg.norm(r)
        e_fp8 = np.linalg.norm(a - r) / np.linalg.norm(r)
        rms = float(np.sqrt(np.mean(np.asarray(r, np.float64) ** 2)))
        m_gpu = float(np.abs(g - r).max()) / rms
        m_fp8 = float(np.abs(a - r).max()) / rms
        m_gpu_fp8 = float(np.abs(g - a).max()) / rms
        print(f"[fp8] {what} ({n} output): norm-wise vs float64: GPU {e_gpu:.4e}, exact FP8 {e_fp8:.4e}; "
              f"max|err|/RMS vs float64: GPU {m_gpu:.4e}, exact FP8 {m_fp8:.4e}; GPU vs exact FP8 "
              f"{m_gpu_fp8:.4e}")
        assert e_gpu <= 6e-2, f"{what} ({n} output): ||y - y64|| / ||y64|| = {e_gpu:.3e} > 6e-2"
        assert e_gpu <= factor * e_fp8, (f"{what} ({n} output): {e_gpu:.3e} vs exact-FP8 "
                                         f"{e_fp8:.3e}")
        assert m_gpu <= factor * m_fp8, (f"{what} ({n} output): max|err|/RMS {m_gpu:.3e} vs exact-FP8 "
                                         f"{m_fp8:.3e}")
        assert m_gpu_fp8 <= m_fp8, (f"{what} ({n} output): max|GPU - exact FP8|/RMS {m_gpu_fp8:.3e} > "
                                    f"exact FP8's own {m_fp8:.3e}")


SMALL = [
    # B, S_i, S_t, D, H, F, single
    (2, 300, 45, 256, 2, 1024, False),
    (1, 200, 77, 512, 4, 1536, False),
    (2, 300, 45, 256, 2, 1024, True),
]


@pytest.mark.parametrize("B,S_i,S_t,D,H,F,single", SMALL)
def test_fp8_block_small(B, S_i, S_t, D, H, F, single):
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=31 + S_i + D, std=0.05, single=single)
    run = Fp8Run(case)
    y8, sc, ds1 = _oracle_two_calls(case)
    _check_state(run, ds1)
    _check_pre_attention(run, sc)
    _check_norm_wise(run.y, y8, case.oracle(None), "FP8 block")


@pytest.mark.parametrize("single", [False, True])
def test_fp8_block_after_attention_elementwise(single):
    """V = 0 makes the attention output exactly zero on both sides, so the output projection,
    LayerNorm-modulate -> E4M3, fc1 + GELU -> E4M3 and fc2 take the same decisions as the oracle
    and can be held to the element-wise bar."""
    case = BlockCase(2, 300, 45, 256, 2, 1024, "bf16", seed=77, std=0.05, single=single)
    for w in [case.w_img] + ([] if single else [case.w_txt]):
        D = case.D
        w["w_qkv"][2 * D:] = 0.0
        w["b_qkv"][2 * D:] = 0.0
    run = Fp8Run(case)
    y8, sc, ds1 = _oracle_two_calls(case)
    # every amax, o's (exactly 0) included, is now decided like the oracle's
    _check_state(run, ds1, tol={"o": 0.0, "fc1": 1e-5, "fc2": 1e-3})
    xs = [case.x_joint()] if single else [case.x_img, case.x_txt]
    ws_names = ["single"] if single else ["img", "txt"]
    wsets = [case.w_img] if single else [case.w_img, case.w_txt]
    offs = L.mmdit_block_workspace_offsets(run.dims, single)
    for k, (x, w, name) in enumerate(zip(xs, wsets, ws_names)):
        # the MLP branch's LayerNorm-modulate codes (the h slot holds them after the call): the
        # attention output is zero, so the output projection is its bias
        m = O.modulation(case.vec, w["w_mod"], w["b_mod"], mm_cast=O.round_bf16)
        x1 = O.gated_residual(x, m[2], np.broadcast_to(np.asarray(w["b_o"], np.float64), x.shape))
        h2 = O.modulate(x1, m[3], m[4])
        got = workspace_view(run.ws, offs[10 + k], (x.shape[0] * x.shape[1], case.D), torch.uint8)
        _check_codes(got.cpu().numpy().reshape(h2.shape), h2, run.scales_used[-1][8 * k + 4],
                     sc[f"{name}.fc1.x"], f"{name} MLP-branch LayerNorm codes")
    for g, r, x in zip(run.y, y8, xs):
        e = assert_parity(g, r, 2e-2, "FP8 block output (V = 0)", out_bf16=True)
        print(f"[fp8] V = 0 block output: max|err| / RMS beyond bf16 rounding = {e:.3e}")
        assert_parity(g - x, r - x, 0.1, "FP8 block branch (V = 0)", out_bf16=True)


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(n, size=min(k, n), replace=False))
    return np.unique(np.concatenate([rows, [0, n - 1]]))


@pytest.mark.parametrize("single", [False, True])
def test_fp8_blocks_at_2048px_sampled_rows(single):
    """The 12B block shapes at 2048 px (16384 image + 512 text tokens, batch 1) with E4M3
    linears, in the launch configuration the benchmark times, on seeded rows."""
    case = BlockCase(1, 128 * 128, 512, 3072, 24, 12288, "bf16", seed=1004 + single, std=0.02,
                     gain_jitter=0.0, lat_hw=(128, 128), single=single)
    run = Fp8Run(case)
    rows = (_sample(case.S, 96, 5),) if single else (_sample(case.S_i, 64, 5), _sample(case.S_t, 32, 6))
    y8, sc, ds1 = _oracle_two_calls(case, rows=rows)
    _check_state(run, ds1, sampled=True)
    y64 = case.oracle_rows(*rows, mm_cast=None)
    got = [g[:, r] for g, r in zip(run.y, rows)]
    _check_norm_wise(got, y8, y64, "FP8 block at 2048 px")


@pytest.mark.parametrize("algo,margin", [(L.AMAX_MAX, 0), (L.AMAX_MOST_RECENT, 1), (L.AMAX_MAX, 2)])
def test_scale_update_over_three_calls(algo, margin):
    """Three calls recording into history columns 0, 1, 2 with a conditioning vector scaled by
    1, 3 and 0.5 (so the casts' amax differ from call to call); after each call every recorded
    tensor's scale is 448 / amax / 2^margin, with amax the latest column (most_recent) or the
    row's largest entry (max), in float32 as the pages' formula gives it (oracle.e4m3)."""
    case = BlockCase(1, 200, 40, 256, 2, 512, "bf16", seed=5, std=0.05)
    dims = _fp8_dims(case)
    hist = torch.zeros(16, HIST, device="cuda")
    scale = torch.ones(16, device="cuda")
    ids = torch.from_numpy(case.ids).cuda()
    cos = torch.empty(case.B, case.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
    wi, wt = upload_weights(case.w_img, "bf16"), upload_weights(case.w_txt, "bf16")
    xi, xt = dev(case.x_img), dev(case.x_txt)
    yi, yt = torch.empty_like(xi), torch.empty_like(xt)
    name = "max" if algo == L.AMAX_MAX else "most_recent"
    for call, f in enumerate((1.0, 3.0, 0.5)):
        vec = dev(synth.bf16_round(case.vec * np.float32(f)))
        st = L.make_fp8_state(hist, scale, pos=call, algo=algo, margin=margin)
        ws = L.mmdit_double_block_fwd(dims, wi, wt, vec, cos, sin, xi, xt, yi, yt, fp8=st)
        torch.cuda.synchronize()
        assert L.mmdit_workspace_status(ws) == 0
        h = hist.cpu().numpy()[:, :call + 1]
        sc = scale.cpu().numpy()
        assert np.all(h > 0), "every tensor records an amax in every call"
        for t in range(16):
            a = np.float32(h[t, -1] if name == "most_recent" else h[t].max())
            expect = np.float32(np.ldexp(np.float32(448.0) / a, -margin))
            assert sc[t] == expect, (call, t, sc[t], expect)
            # the same rule as the oracle's, to float32 rounding
            assert abs(sc[t] - E.history_scale(h[t], name, margin)) <= 1e-6 * sc[t]
    assert not np.all(hist.cpu().numpy()[:, 0] == hist.cpu().numpy()[:, 1]), "the calls differ"


# ----------------------------------------------------------------------------- tensorwise recipe
def _tensorwise_run(case, margin=0):
    """One call of the block with gemm = MMDIT_GEMM_FP8_TENSORWISE (current per-tensor scaling);
    returns (outputs, recorded amax [n_t], scales after the call [n_t])."""
    dims = L.make_dims(case.B, case.S_i, case.S_t, case.D, case.H, case.F, L.MMDIT_BF16,
                       rope_interleaved=case.interleaved, gelu_tanh=case.gelu_tanh,
                       gemm=L.MMDIT_GEMM_FP8_TENSORWISE)
    n_t = 8 if case.single else 16
    hist = torch.zeros(n_t, 4, device="cuda")
    scale = torch.full((n_t,), 123.0, device="cuda")  # overwritten: the recipe keeps no history
    st = L.make_fp8_state(hist, scale, pos=2, margin=margin)
    ids = torch.from_numpy(case.ids).cuda()
    cos = torch.empty(case.B, case.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
    wi = upload_weights(case.w_img, "bf16")
    if case.single:
        x = dev(case.x_joint())
        y = torch.empty_like(x)
        ws = L.mmdit_single_block_fwd(dims, wi, dev(case.vec), cos, sin, x, y, fp8=st)
        outs = (y,)
    else:
        wt = upload_weights(case.w_txt, "bf16")
        xi, xt = dev(case.x_img), dev(case.x_txt)
        yi, yt = torch.empty_like(xi), torch.empty_like(xt)
        ws = L.mmdit_double_block_fwd(dims, wi, wt, dev(case.vec), cos, sin, xi, xt, yi, yt, fp8=st)
        outs = (yi, yt)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    h = hist.cpu().numpy()
    assert np.all(h[:, [0, 1, 3]] == 0), "only history column pos is written"
    return tuple(host(o) for o in outs), h[:, 2], scale.cpu().numpy()


@pytest.mark.parametrize("B,S_i,S_t,D,H,F,single", SMALL)
def test_fp8_tensorwise_block_small(B, S_i, S_t, D, H, F, single):
    """The tensorwise recipe ("FP8 training for Flux models", §Configuration, fp8_recipe
    "tensorwise"): one call, no history.  Recorded amax: every weight's max |w| exactly, every input
    within a bf16 step of the oracle's (the GPU takes the amax of its own bf16 LayerNorm, attention
    and GELU outputs); each scale 448 / that amax in float32; the block output under the FP8 bars
    against the exact tensorwise evaluation (oracle.fp8_recipes.TensorwiseScaling on bf16-stored
    inputs) and the float64 block."""
    from oracle import fp8_recipes as R
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=41 + S_i + D, std=0.05, single=single)
    y, amax, scale = _tensorwise_run(case)
    tw = R.TensorwiseScaling(act_cast=O.round_bf16)
    args = dict(mm_cast=O.round_bf16, fp8=tw, interleaved=case.interleaved, gelu_tanh=case.gelu_tanh)
    if single:
        y8 = (O.single_block(case.x_joint(), case.vec, case.cos, case.sin, case.w_img, case.H, **args),)
        slots = [("single", 0)]
    else:
        y8 = O.double_block(case.x_img, case.x_txt, case.vec, case.cos, case.sin, case.w_img, case.w_txt,
                            case.H, **args)
        slots = [("img", 0), ("txt", 1)]
    for name, slot in slots:
        for g, lin in enumerate(NAMES):
            for op, tag in ((1, "w"), (0, "x")):
                t = 8 * slot + 2 * g + op
                ref = tw.amax[f"{name}.{lin}.{tag}"]
                if tag == "w":
                    assert amax[t] == np.float32(ref), (name, lin, amax[t], ref)
                else:
                    assert abs(amax[t] - ref) <= 2.0 ** -7 * ref, (name, lin, amax[t], ref)
                assert scale[t] == np.float32(448.0) / np.float32(amax[t]), (name, lin)
    _check_norm_wise(y, y8, case.oracle(None), "FP8 tensorwise block")



# ----------------------------------------------------------------------------- FP8 linear backward
@pytest.mark.parametrize("recipe", ["e4m3", "hybrid"])
@pytest.mark.parametrize("fp8_wgrad", [True, False])
@pytest.mark.parametrize("M,N,K", [(300, 256, 384), (4608, 3072, 3072), (77, 48, 128)])
def test_fp8_linear_backward_matches_oracle(recipe, fp8_wgrad, M, N, K):
    """mmdit_fp8_linear_bwd against oracle.fp8_backward.fp8_linear_bwd ("FP8 training for Flux
    models", §Configuration: fp8 "e4m3" / "hybrid", fp8_wgrad).  The forward casts come from the
    library's bit-exact E4M3 cast at power-of-two scales, and dy's scale is a power of two too, so
    both sides multiply the same codes: dx and dW agree to fp32 accumulation (2e-3 x RMS, the FP8
    linear's bar), db to 1e-5.  The recorded amax of dy is max |dy| exactly."""
    from oracle import fp8_backward as FB
    rng = np.random.default_rng(M + N + K + (recipe == "hybrid"))
    x = synth.bf16_round(rng.standard_normal((M, K)))
    w = synth.bf16_round(rng.standard_normal((N, K)) * 0.02)
    dy = synth.bf16_round(rng.standard_normal((M, N)) * 1e-3)
    fmax = 448.0 if recipe == "e4m3" else 57344.0
    sx, sw = _pow2_scale(np.abs(x).max()), _pow2_scale(np.abs(w).max())
    sdy = 2.0 ** np.floor(np.log2(fmax / np.abs(dy).max()))
    scales = torch.tensor([sx, sw, sdy], dtype=torch.float32, device="cuda")
    amax = torch.zeros(3, device="cuda")
    xq = torch.empty(M, K, dtype=torch.uint8, device="cuda")
    wq = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    L.mmdit_fp8_quantize_e4m3(dev(x), scales[0:1], amax[0:1], xq)
    L.mmdit_fp8_quantize_e4m3(dev(w), scales[1:2], amax[1:2], wq)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device="cuda")
    dw = torch.full((N, K), float("nan"), device="cuda")
    db = torch.full((N,), float("nan"), device="cuda")
    ws = L.mmdit_fp8_linear_bwd(dev(dy), xq, wq, scales[0:1], scales[1:2], scales[2:3], amax[2:3], dx, dw, db,
                                x=dev(x), recipe=recipe, fp8_wgrad=fp8_wgrad)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    rdx, rdw, rdb = FB.fp8_linear_bwd(dy, x, w, sx, sw, sdy, recipe, fp8_wgrad)
    assert amax[2].item() == np.float32(np.abs(dy).max())
    assert_parity(host(dx), rdx, 2e-3, f"FP8 dgrad ({recipe})", out_bf16=True)
    # without fp8_wgrad the weight gradient is the bf16 product dy^T x, held to the linear
    # backward's bar
    assert_parity(host(dw), rdw, 2e-3 if fp8_wgrad else 2e-2, f"wgrad ({recipe}, fp8_wgrad={fp8_wgrad})")
    assert_parity(host(db), rdb, 1e-5, "db")


# ----------------------------------------------------------------------------- FP8 attention
@pytest.mark.parametrize("B,H,S", [(1, 2, 100), (2, 3, 128), (2, 3, 300), (1, 4, 1000), (1, 24, 4608)])
def test_fp8_attention_matches_oracle(B, H, S):
    """mmdit_fp8_attention_fwd (the opt-in fp8_dot_product_attention) against
    oracle.fp8_attention.fp8_attention at the same per-tensor scales (powers of two, so both sides
    cast the same codes).  With one key tile (S <= 128) the running maximum is the row maximum and
    the two agree to the exp2 rounding: 1e-2 x RMS.  With more tiles a row whose maximum arrives
    late casts its earlier probabilities against a smaller maximum, so the codes differ by E4M3
    rounding: the GPU must then sit no further from the FP8 oracle than the FP8 oracle sits from
    exact attention (max norm and norm-wise)."""
    from oracle import fp8_attention as FA
    rng = np.random.default_rng(S + 7 * H)
    q = synth.bf16_round(rng.standard_normal((B, H, S, 128)) * 1.5)
    k = synth.bf16_round(rng.standard_normal((B, H, S, 128)))
    v = synth.bf16_round(rng.standard_normal((B, H, S, 128)))
    sq, sk, sv = (_pow2_scale(np.abs(a).max()) for a in (q, k, v))
    scales = torch.tensor([sq, sk, sv], dtype=torch.float32, device="cuda")
    out = torch.empty(B, S, H * 128, device="cuda", dtype=torch.bfloat16)
    ws = L.mmdit_fp8_attention_fwd(dev(q), dev(k), dev(v), scales[0:1], scales[1:2], scales[2:3], out)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    rows = np.sort(np.random.default_rng(1).choice(S, 160, replace=False)) if S > 1000 else np.arange(S)
    ref8 = FA.fp8_attention(q[:, :, rows], k, v, sq, sk, sv).transpose(0, 2, 1, 3).reshape(B, len(rows), H * 128)
    ref64 = O.attention(q[:, :, rows], k, v).transpose(0, 2, 1, 3).reshape(B, len(rows), H * 128)
    got = host(out)[:, rows]
    assert np.all(np.isfinite(got))
    rms = float(np.sqrt(np.mean(ref64 ** 2)))
    m_gpu8 = float(np.abs(got - ref8).max()) / rms
    m_864 = float(np.abs(ref8 - ref64).max()) / rms
    n_gpu8 = np.linalg.norm(got - ref8) / np.linalg.norm(ref8)
    n_864 = np.linalg.norm(ref8 - ref64) / np.linalg.norm(ref64)
    print(f"[fp8 attention] B={B} H={H} S={S}: max/RMS GPU-FP8 {m_gpu8:.3e}, FP8-exact {m_864:.3e}; "
          f"norm-wise GPU-FP8 {n_gpu8:.3e}, FP8-exact {n_864:.3e}")
    if S <= 128:
        assert_parity(got, ref8, 1e-2, f"FP8 attention S={S}", out_bf16=True)
    else:
        assert m_gpu8 <= m_864, (m_gpu8, m_864)
        assert n_gpu8 <= n_864, (n_gpu8, n_864)


# ----------------------------------------------------------------------------- blockwise recipe
def _ru256(n):
    return (n + 255) // 256 * 256


def _blockwise_parts(ws, M, N, K):
    """The codes and scales the call leaves in its workspace (layout stated in include/mmdit.h)."""
    raw = ws.cpu().numpy().view(np.uint8)
    off = 256
    xq = raw[off:off + M * K].reshape(M, K)
    off += _ru256(M * K)
    wq = raw[off:off + N * K].reshape(N, K)
    off += _ru256(N * K)
    sx = raw[off:off + (K // 128) * M * 4].view(np.float32).reshape(K // 128, M)
    off += _ru256((K // 128) * M * 4)
    sw = raw[off:off + (N // 128) * (K // 128) * 4].view(np.float32).reshape(N // 128, K // 128)
    return xq, wq, sx, sw


def _f32_tile_cast(t):
    """The stated float32 cast of one tile: s = 448 / amax (IEEE float32), codes of (x s) rounded to
    float32 first, then to E4M3 (the oracle's encoder: nearest even, saturating)."""
    t = np.asarray(t, np.float32)
    amax = np.float32(np.abs(t).max())
    s = np.float32(448.0) / amax if amax > 0 else np.float32(1.0)
    return E.e4m3_encode((t * s).astype(np.float64)), s


@pytest.mark.parametrize("M,N,K", [(300, 256, 512), (1024, 3072, 3072)])
def test_blockwise_fp8_linear(M, N, K):
    """[FP8] §Configuration, fp8_recipe "blockwise" (oracle.fp8_recipes.blockwise_linear): the casts
    are bit-exact against a float32 emulation of the stated arithmetic (codes and scales, with an
    outlier, a tile of zeros and a ragged last row tile); the GEMM, fed the GPU's codes and scales,
    agrees with their float64 product to fp32 accumulation and the bf16 output rounding; and the
    whole linear sits far closer to the oracle's float64 recipe than that recipe sits to the exact
    product (max norm, so a mistake in one tile's scale fails)."""
    from oracle import fp8_recipes as R
    rng = np.random.default_rng(M + N)
    x = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    x[7, 200] = 300.0                            # an outlier owns its 1 x 128 tile's scale
    w = synth.bf16_round((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    w[128:256, K - 128:] = 0.0                   # a tile of zeros: scale 1, codes 0
    b = synth.bf16_round((rng.standard_normal(N) * 0.1).astype(np.float32))
    y = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    ws = L.mmdit_fp8_blockwise_linear_fwd(dev(x), dev(w), dev(b), y)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    xq, wq, sx, sw = _blockwise_parts(ws, M, N, K)
    # casts, bit-exact
    for m in range(0, M, max(1, M // 64)):
        for j in range(K // 128):
            codes, s = _f32_tile_cast(x[m, 128 * j:128 * (j + 1)])
            assert sx[j, m] == s, (m, j)
            assert np.array_equal(xq[m, 128 * j:128 * (j + 1)], codes), (m, j)
    for i in range(N // 128):
        for j in range(K // 128):
            codes, s = _f32_tile_cast(w[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)])
            assert sw[i, j] == s, (i, j)
            assert np.array_equal(wq[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)], codes), (i, j)
    assert sw[1, K // 128 - 1] == 1.0 and not wq[128:256, K - 128:].any()
    # the GEMM from the GPU's own codes and scales, in float64
    dec = np.array([E.e4m3_decode(c) for c in range(256)])
    ref = np.zeros((M, N))
    tile_row = np.arange(N) // 128
    for j in range(K // 128):
        sl = slice(128 * j, 128 * (j + 1))
        ref += (dec[xq[:, sl]] @ dec[wq[:, sl]].T) / (sx[j][:, None].astype(np.float64) *
                                                      sw[tile_row, j][None, :].astype(np.float64))
    ref += b
    got = host(y)
    assert_parity(got, ref, 1e-3, f"blockwise GEMM {M}x{N}x{K}", out_bf16=True)
    # the whole linear against the oracle's recipe and the exact product
    y_or = R.blockwise_linear(x, w, b)
    y_ex = x.astype(np.float64) @ w.astype(np.float64).T + b
    rms = float(np.sqrt(np.mean(y_ex ** 2)))
    d_gpu = float(np.abs(got - y_or).max()) / rms
    d_fp8 = float(np.abs(y_or - y_ex).max()) / rms
    print(f"[fp8 blockwise] {M}x{N}x{K}: max|GPU - recipe|/RMS {d_gpu:.3e}, max|recipe - exact|/RMS {d_fp8:.3e}")
    assert d_gpu <= 0.25 * d_fp8


def _blockwise_block_run(case, gemm=L.MMDIT_GEMM_FP8_BLOCKWISE):
    """One call of the block with a stateless recipe (gemm = MMDIT_GEMM_FP8_BLOCKWISE or
    MMDIT_GEMM_FP8_MXFP8; no FP8 state)."""
    dims = L.make_dims(case.B, case.S_i, case.S_t, case.D, case.H, case.F, L.MMDIT_BF16,
                       rope_interleaved=case.interleaved, gelu_tanh=case.gelu_tanh, gemm=gemm)
    ids = torch.from_numpy(case.ids).cuda()
    cos = torch.empty(case.B, case.S, 64, device="cuda")
    sin = torch.empty_like(cos)
    L.rope3d_freqs(ids, (16, 56, 56), 10000.0, cos, sin)
    wi = upload_weights(case.w_img, "bf16")
    if case.single:
        x = dev(case.x_joint())
        y = torch.empty_like(x)
        ws = L.mmdit_single_block_fwd(dims, wi, dev(case.vec), cos, sin, x, y)
        outs = (y,)
    else:
        wt = upload_weights(case.w_txt, "bf16")
        xi, xt = dev(case.x_img), dev(case.x_txt)
        yi, yt = torch.empty_like(xi), torch.empty_like(xt)
        ws = L.mmdit_double_block_fwd(dims, wi, wt, dev(case.vec), cos, sin, xi, xt, yi, yt)
        outs = (yi, yt)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    return tuple(host(o) for o in outs)


@pytest.mark.parametrize("B,S_i,S_t,D,H,F,single", SMALL)
def test_fp8_blockwise_block_small(B, S_i, S_t, D, H, F, single):
    """The blockwise recipe inside the blocks ("FP8 training for Flux models", §Configuration,
    fp8_recipe "blockwise"): every linear's bf16 input cast per 1 x 128 tile and its weight per
    128 x 128 tile, no state.  The block output under the FP8 bars against the exact blockwise
    evaluation (oracle.fp8_recipes.BlockwiseScaling on bf16-stored inputs) and the float64 block."""
    from oracle import fp8_recipes as R
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=51 + S_i + D, std=0.05, single=single)
    y = _blockwise_block_run(case)
    bw = R.BlockwiseScaling(act_cast=O.round_bf16)
    args = dict(mm_cast=O.round_bf16, fp8=bw, interleaved=case.interleaved, gelu_tanh=case.gelu_tanh)
    if single:
        y8 = (O.single_block(case.x_joint(), case.vec, case.cos, case.sin, case.w_img, case.H, **args),)
    else:
        y8 = O.double_block(case.x_img, case.x_txt, case.vec, case.cos, case.sin, case.w_img, case.w_txt,
                            case.H, **args)
    _check_norm_wise(y, y8, case.oracle(None), "FP8 blockwise block")


# ----------------------------------------------------------------------------- MXFP8 recipe
def _mx_parts(ws, M, N, K):
    """The represented values, codes and scale codes the call leaves in its workspace (layout
    stated in include/mmdit.h)."""
    raw = ws.cpu().numpy().view(np.uint8)

    def bf16_at(off, n):
        return (raw[off:off + 2 * n].view(np.uint16).astype(np.uint32) << 16).view(np.float32)

    off = 256
    xd = bf16_at(off, M * K).reshape(M, K)
    off += _ru256(2 * M * K)
    wd = bf16_at(off, N * K).reshape(N, K)
    off += _ru256(2 * N * K)
    xq = raw[off:off + M * K].reshape(M, K)
    off += _ru256(M * K)
    wq = raw[off:off + N * K].reshape(N, K)
    off += _ru256(N * K)
    xs = raw[off:off + M * (K // 32)].reshape(M, K // 32)
    off += _ru256(M * (K // 32))
    wsc = raw[off:off + N * (K // 32)].reshape(N, K // 32)
    return xd, wd, xq, wq, xs, wsc


@pytest.mark.parametrize("M,N,K", [(300, 96, 512), (1024, 3072, 3072)])
def test_mxfp8_linear(M, N, K):
    """[FP8] §Configuration, fp8_recipe "mxfp8" (oracle.fp8_recipes.mxfp8_quantize / mxfp8_linear,
    the OCP MX v1.0 reading): the casts are bit-exact against the oracle's -- the E4M3 codes, the
    E8M0 scale codes and the represented values P 2^e -- with an outlier, a quotient above 448
    that saturates, a block of zeros and a block near 2^-100; the GEMM agrees with the float64
    product of the GPU's represented values to fp32 accumulation and the bf16 output rounding;
    and the whole linear sits far closer to the oracle's recipe than that recipe sits to the
    exact product (max norm)."""
    from oracle import fp8_recipes as R
    rng = np.random.default_rng(M + 3 * N)
    x = synth.bf16_round(rng.standard_normal((M, K)).astype(np.float32))
    x[7, 200] = 300.0                               # an outlier owns its block's exponent
    x[9, 96] = 480.0                                # e = 0 and 480 > 448: saturates
    x[3, 64:96] = 0.0                               # a block of zeros: e = -127, codes 0
    x[5, 32:64] = synth.bf16_round(x[5, 32:64] * np.float32(2.0 ** -100))
    w = synth.bf16_round((rng.standard_normal((N, K)) * 0.02).astype(np.float32))
    w[10, :32] = 0.0
    b = synth.bf16_round((rng.standard_normal(N) * 0.1).astype(np.float32))
    y = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    ws = L.mmdit_fp8_mxfp8_linear_fwd(dev(x), dev(w), dev(b), y)
    torch.cuda.synchronize()
    assert L.mmdit_workspace_status(ws) == 0
    xd, wd, xq, wq, xs, wsc = _mx_parts(ws, M, N, K)
    dec = np.array([E.e4m3_decode(c) for c in range(256)])
    for name, src, vals, codes, scales in (("x", x, xd, xq, xs), ("W", w, wd, wq, wsc)):
        p, e = R.mxfp8_quantize(src.astype(np.float64))
        assert np.array_equal(scales.astype(np.int64) - 127, e), name
        assert np.array_equal(dec[codes], p), name
        assert np.array_equal(vals.astype(np.float64), R.mxfp8_dequantize(p, e)), name
    assert xs[3, 2] == 0 and not xq[3, 64:96].any() and dec[xq[9, 96]] == 448.0
    # the GEMM from the GPU's represented values, in float64
    got = host(y)
    ref = xd.astype(np.float64) @ wd.astype(np.float64).T + b
    assert_parity(got, ref, 1e-3, f"MXFP8 GEMM {M}x{N}x{K}", out_bf16=True)
    # the whole linear against the oracle's recipe and the exact product
    y_or = R.mxfp8_linear(x, w, b)
    y_ex = x.astype(np.float64) @ w.astype(np.float64).T + b
    rms = float(np.sqrt(np.mean(y_ex ** 2)))
    d_gpu = float(np.abs(got - y_or).max()) / rms
    d_fp8 = float(np.abs(y_or - y_ex).max()) / rms
    print(f"[fp8 mxfp8] {M}x{N}x{K}: max|GPU - recipe|/RMS {d_gpu:.3e}, max|recipe - exact|/RMS {d_fp8:.3e}")
    assert d_gpu <= 0.25 * d_fp8


@pytest.mark.parametrize("B,S_i,S_t,D,H,F,single", SMALL)
def test_fp8_mxfp8_block_small(B, S_i, S_t, D, H, F, single):
    """The MXFP8 recipe inside the blocks ("FP8 training for Flux models", §Configuration,
    fp8_recipe "mxfp8"): every linear's bf16 input and its weight cast per 32 elements along K,
    no state.  The block output under the FP8 bars against the exact MXFP8 evaluation
    (oracle.fp8_recipes.MxScaling on bf16-stored inputs) and the float64 block."""
    from oracle import fp8_recipes as R
    case = BlockCase(B, S_i, S_t, D, H, F, "bf16", seed=61 + S_i + D, std=0.05, single=single)
    y = _blockwise_block_run(case, gemm=L.MMDIT_GEMM_FP8_MXFP8)
    mx = R.MxScaling(act_cast=O.round_bf16)
    args = dict(mm_cast=O.round_bf16, fp8=mx, interleaved=case.interleaved, gelu_tanh=case.gelu_tanh)
    if single:
        y8 = (O.single_block(case.x_joint(), case.vec, case.cos, case.sin, case.w_img, case.H, **args),)
    else:
        y8 = O.double_block(case.x_img, case.x_txt, case.vec, case.cos, case.sin, case.w_img, case.w_txt,
                            case.H, **args)
    _check_norm_wise(y, y8, case.oracle(None), "FP8 MXFP8 block")


@pytest.mark.parametrize("recipe,single", [("mxfp8", False), ("blockwise", True)])
def test_stateless_fp8_blocks_at_2048px_sampled_rows(recipe, single):
    """The 12B block shapes at 2048 px (16384 image + 512 text tokens, batch 1) under the MXFP8
    and blockwise recipes, in the launch configuration the benchmark times, on seeded rows.  Both
    recipes scale activations within a row (1 x 32 or 1 x 128 blocks along K) and weights as a
    whole, so the oracle evaluated on the sampled rows casts exactly what the GPU cast there."""
    from oracle import fp8_recipes as R
    case = BlockCase(1, 128 * 128, 512, 3072, 24, 12288, "bf16", seed=1014 + single, std=0.02,
                     gain_jitter=0.0, lat_hw=(128, 128), single=single)
    gemm = L.MMDIT_GEMM_FP8_MXFP8 if recipe == "mxfp8" else L.MMDIT_GEMM_FP8_BLOCKWISE
    y = _blockwise_block_run(case, gemm=gemm)
    rows = (_sample(case.S, 96, 7),) if single else (_sample(case.S_i, 64, 7), _sample(case.S_t, 32, 8))
    obj = (R.MxScaling if recipe == "mxfp8" else R.BlockwiseScaling)(act_cast=O.round_bf16)
    args = dict(mm_cast=O.round_bf16, fp8=obj, interleaved=case.interleaved, gelu_tanh=case.gelu_tanh)
    if single:
        y8 = (O.single_block_rows(case.x_joint(), case.vec, case.cos, case.sin, case.w_img, case.H, rows[0],
                                  **args),)
    else:
        y8 = O.double_block_rows(case.x_img, case.x_txt, case.vec, case.cos, case.sin, case.w_img, case.w_txt,
                                 case.H, rows[0], rows[1], **args)
    y64 = case.oracle_rows(*rows, mm_cast=None)
    got = [g[:, r] for g, r in zip(y, rows)]
    _check_norm_wise(got, y8, y64, f"FP8 {recipe} block at 2048 px")
