"""Runs one library entry point on one seeded case, for profiling a kernel with ncu.

    python -m diffusion_transformer_flux_gb300.profile_case attention --batch 2 --seq 4608
    python -m diffusion_transformer_flux_gb300.profile_case double_block --seq-img 4096 --seq-txt 512
    python -m diffusion_transformer_flux_gb300.profile_case linear --m 4608 --n 12288 --k 3072
    python -m diffusion_transformer_flux_gb300.profile_case double_block_bwd --seq-img 4096 --seq-txt 512
    python -m diffusion_transformer_flux_gb300.profile_case fp8_attention --seq 4608
    python -m diffusion_transformer_flux_gb300.profile_case head_loss --seq-img 4096
    python -m diffusion_transformer_flux_gb300.profile_case modulation --jobs 4
    python -m diffusion_transformer_flux_gb300.profile_case blockwise_linear --m 4608 --n 12288 --k 3072
    python -m diffusion_transformer_flux_gb300.profile_case mxfp8_linear --m 4608 --n 12288 --k 3072

Inputs are drawn on the device (N(0,1) activations, N(0,0.02) weights); the case runs
--iters times and exits 0 only if every kernel finished its waits.
"""
from __future__ import annotations

import argparse

import torch

from . import _lib as L


def _w(*shape, std=0.02):
    return (torch.randn(*shape, device="cuda") * std).to(torch.bfloat16)


def _stream_w(D, F, d=128):
    return {"w_mod": _w(6 * D, D), "b_mod": _w(6 * D), "w_qkv": _w(3 * D, D), "b_qkv": _w(3 * D),
            "g_q": torch.ones(d, device="cuda", dtype=torch.bfloat16),
            "g_k": torch.ones(d, device="cuda", dtype=torch.bfloat16),
            "w_o": _w(D, D), "b_o": _w(D), "w_1": _w(F, D), "b_1": _w(F), "w_2": _w(D, F), "b_2": _w(D)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["attention", "double_block", "single_block", "linear", "double_block_bwd",
                                     "fp8_attention", "head_loss", "modulation", "blockwise_linear",
                                     "mxfp8_linear"])
    ap.add_argument("--jobs", type=int, default=4)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--seq", type=int, default=4608)
    ap.add_argument("--seq-img", type=int, default=4096)
    ap.add_argument("--seq-txt", type=int, default=512)
    ap.add_argument("--hidden", type=int, default=3072)
    ap.add_argument("--mlp", type=int, default=12288)
    ap.add_argument("--m", type=int, default=4608)
    ap.add_argument("--n", type=int, default=12288)
    ap.add_argument("--k", type=int, default=3072)
    ap.add_argument("--iters", type=int, default=3)
    a = ap.parse_args()
    torch.manual_seed(0)
    L.load()
    wss = []
    if a.case == "fp8_attention":
        H = a.hidden // 128
        q, k, v = (torch.randn(a.batch, H, a.seq, 128, device="cuda").to(torch.bfloat16) for _ in range(3))
        scales = torch.full((3,), 32.0, device="cuda")
        out = torch.empty(a.batch, a.seq, a.hidden, device="cuda", dtype=torch.bfloat16)
        run = lambda: wss.append(L.mmdit_fp8_attention_fwd(q, k, v, scales[0:1], scales[1:2], scales[2:3], out))
    elif a.case == "head_loss":
        B, Si, D = a.batch, a.seq_img, a.hidden
        hw = int(round(Si ** 0.5))
        dims = L.make_dims(B, Si, 0, D, D // 128, a.mlp, L.MMDIT_BF16)
        x, vec = _w(B, Si, D, std=1.0), _w(B, D, std=1.0)
        z0, z1 = (torch.randn(B, 64, hw, hw, device="cuda") for _ in range(2))
        loss = torch.zeros(1, device="cuda")
        args = (dims, hw, hw, x, vec, _w(2 * D, D), _w(2 * D), _w(64, D), _w(64), z0, z1, loss)
        run = lambda: wss.append(L.mmdit_final_layer_loss_fwd(*args))
    elif a.case == "modulation":
        D = a.hidden
        vec = _w(a.batch, D, std=1.0)
        jobs = [(_w(6 * D, D), _w(6 * D), torch.empty(a.batch, 6 * D, device="cuda")) for _ in range(a.jobs)]
        run = lambda: L.mmdit_modulation_batched_fwd(vec, jobs)
    elif a.case == "attention":
        H = a.hidden // 128
        q, k, v = (torch.randn(a.batch, H, a.seq, 128, device="cuda").to(torch.bfloat16) for _ in range(3))
        out = torch.empty(a.batch, a.seq, a.hidden, device="cuda", dtype=torch.bfloat16)
        run = lambda: wss.append(L.mmdit_attention_fwd(q, k, v, out))
    elif a.case == "linear":
        x, w, b = _w(a.m, a.k, std=1.0), _w(a.n, a.k), _w(a.n)
        y = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
        run = lambda: wss.append(L.mmdit_linear_fwd(x, w, b, y))
    elif a.case == "blockwise_linear":
        x, w, b = _w(a.m, a.k, std=1.0), _w(a.n, a.k), _w(a.n)
        y = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
        run = lambda: wss.append(L.mmdit_fp8_blockwise_linear_fwd(x, w, b, y))
    elif a.case == "mxfp8_linear":
        x, w, b = _w(a.m, a.k, std=1.0), _w(a.n, a.k), _w(a.n)
        y = torch.empty(a.m, a.n, device="cuda", dtype=torch.bfloat16)
        run = lambda: wss.append(L.mmdit_fp8_mxfp8_linear_fwd(x, w, b, y))
    else:
        B, Si, St, D, F = a.batch, a.seq_img, a.seq_txt, a.hidden, a.mlp
        S = Si + St
        dims = L.make_dims(B, Si, St, D, D // 128, F, L.MMDIT_BF16)
        vec = _w(B, D, std=1.0)
        cos, sin = torch.rand(B, S, 64, device="cuda"), torch.rand(B, S, 64, device="cuda")
        if a.case == "double_block_bwd":
            wi, wt = _stream_w(D, F), _stream_w(D, F)
            xi, xt = _w(B, Si, D, std=1.0), _w(B, St, D, std=1.0)
            dyi, dyt = _w(B, Si, D, std=1e-3), _w(B, St, D, std=1e-3)
            dxi, dxt = torch.empty_like(xi), torch.empty_like(xt)
            dvec = torch.empty(B, D, device="cuda")
            g = [{n: torch.empty(tuple(w[n].shape), device="cuda") for n in L.STREAM_W_FIELDS} for w in (wi, wt)]
            ws = L.workspace(L.mmdit_double_block_bwd_workspace_size(dims))
            run = lambda: wss.append(L.mmdit_double_block_bwd(dims, wi, wt, vec, cos, sin, xi, xt, dyi, dyt, dxi, dxt,
                                                              dvec, g[0], g[1], ws=ws))
        elif a.case == "double_block":
            wi, wt = _stream_w(D, F), _stream_w(D, F)
            xi, xt = _w(B, Si, D, std=1.0), _w(B, St, D, std=1.0)
            yi, yt = torch.empty_like(xi), torch.empty_like(xt)
            ws = L.workspace(L.mmdit_double_block_workspace_size(dims))
            run = lambda: wss.append(L.mmdit_double_block_fwd(dims, wi, wt, vec, cos, sin, xi, xt, yi, yt, ws=ws))
        else:
            w = _stream_w(D, F)
            x = _w(B, S, D, std=1.0)
            y = torch.empty_like(x)
            ws = L.workspace(L.mmdit_single_block_workspace_size(dims))
            run = lambda: wss.append(L.mmdit_single_block_fwd(dims, w, vec, cos, sin, x, y, ws=ws))
    for _ in range(a.iters):
        run()
    torch.cuda.synchronize()
    for ws in wss:
        if L.mmdit_workspace_status(ws) != 0:
            raise SystemExit("a kernel gave up a bounded wait")
    print(f"{a.case}: {a.iters} iterations ok")


if __name__ == "__main__":
    main()
