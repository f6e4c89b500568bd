"""The C ABI without a GPU: the library builds and loads, exports every function that
include/mmdit.h declares, sizes workspaces, and rejects bad arguments before touching CUDA."""
import ctypes as C
import os
import re

import pytest

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return L.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mmdit.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b([A-Za-z_][A-Za-z0-9_]*)\s*\([^;{]*\)\s*;", src)
    return sorted(set(n for n in names if not n.startswith("typedef")))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("mmdit_double_block_fwd", "mmdit_single_block_fwd", "rope3d_freqs",
              "flow_match_noise_and_loss"):
        assert n in names
    assert sorted(L.EXPORTED) == names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared_functions():
        assert hasattr(lib, n), n


def _dims(**kw):
    base = dict(batch=1, seq_img=4096, seq_txt=512, hidden=3072, heads=24, mlp_hidden=12288,
                act=L.MMDIT_BF16)
    base.update(kw)
    return L.make_dims(**base)


def test_workspace_sizes(lib):
    d = _dims()
    ws = L.mmdit_double_block_workspace_size(d)
    B, S, Si, St, D, F = 1, 4608, 4096, 512, 3072, 12288
    # at least: modulation, LN outputs, Q, K, V^T, attention outputs, fp32 x1, MLP hidden
    floor = 2 * 6 * D * 4 + S * D * 2 * (1 + 3 + 1) + S * D * 4 + S * F * 2
    assert ws >= floor
    assert ws < floor * 1.01 + 64 * 1024
    single = L.mmdit_single_block_workspace_size(d)
    assert single >= S * D * 2 * 5 + S * D * 4 + S * F * 2
    assert L.mmdit_double_block_workspace_size(_dims(head_dim=64)) == 0
    offs = L.mmdit_block_workspace_offsets(d, False)
    assert len(offs) == 17 and offs[0] == 256
    assert all(o % 256 == 0 for o in offs if o >= 0)
    assert sorted(offs[:10]) == offs[:10]  # carved in order
    assert offs[13:] == [-1, -1, -1, -1]  # E4M3 slots only in FP8 mode
    so = L.mmdit_block_workspace_offsets(d, True)
    assert so[1] == -1 and so[6] == -1 and so[8] == -1 and so[11] == -1 and so[12] == -1
    # FP8 mode: the LayerNorm and GELU outputs shrink to one byte per element, and the E4M3
    # attention output and weights (12 D^2 bytes with F = 4D) are added
    f8 = _dims(gemm=1)
    ws8 = L.mmdit_double_block_workspace_size(f8)
    assert ws8 >= ws - S * (D + F) + S * D + 2 * (4 * D * D + 2 * F * D)
    o8 = L.mmdit_block_workspace_offsets(f8, False)
    assert all(o >= 0 and o % 256 == 0 for o in o8)
    assert o8[16] + 4 * D * D + 2 * F * D <= ws8
    assert L.flow_match_workspace_size(4, 64 * 32 * 32) >= 256 + 4
    assert lib.mmdit_linear_workspace_size(1, 4096, 3072, 3072) == 256  # wide: no split
    assert lib.mmdit_linear_workspace_size(1, 512, 3072, 4096) > 512 * 3072 * 4  # narrow: split K


def test_validation_errors_before_any_launch(lib):
    d = _dims()
    w = L.StreamW()
    st = lib.mmdit_double_block_fwd(C.byref(d), C.byref(w), C.byref(w), None, None, None, None, None,
                                    None, None, None, None, 0, None)
    assert st == 1 and "NULL" in L.last_error()
    bad = _dims(head_dim=64)
    assert lib.mmdit_single_block_fwd(C.byref(bad), C.byref(w), None, None, None, None, None, None,
                                      None, 0, None) == 2
    fp8_f32 = _dims(gemm=1, act=0)  # FP8 linears need bf16 activations
    assert lib.mmdit_double_block_fwd(C.byref(fp8_f32), C.byref(w), C.byref(w), None, None, None, None,
                                      None, None, None, None, None, 0, None) == 2
    assert "FP8" in L.last_error()
    fp8 = _dims(gemm=1, act=1)
    assert lib.mmdit_double_block_fwd(C.byref(fp8), C.byref(w), C.byref(w), None, None, None, None,
                                      None, None, None, None, None, 0, None) == 1
    assert "fp8 state" in L.last_error()
    # the blockwise recipe keeps no state: one given is an error
    bwd = _dims(gemm=L.MMDIT_GEMM_FP8_BLOCKWISE, act=1)
    stb = L.Fp8State(0x1000, 0x2000, 1024, 16, 0, 0, 0)
    assert lib.mmdit_double_block_fwd(C.byref(bwd), C.byref(w), C.byref(w), None, None, None, None,
                                      None, None, None, C.byref(stb), None, 0, None) == 1
    assert "blockwise" in L.last_error()
    # nor does the MXFP8 recipe
    mxd = _dims(gemm=L.MMDIT_GEMM_FP8_MXFP8, act=1)
    assert lib.mmdit_double_block_fwd(C.byref(mxd), C.byref(w), C.byref(w), None, None, None, None,
                                      None, None, None, C.byref(stb), None, 0, None) == 1
    assert "MXFP8" in L.last_error()
    # and the modes after it are unknown
    assert lib.mmdit_double_block_fwd(C.byref(_dims(gemm=5, act=1)), C.byref(w), C.byref(w), None, None, None,
                                      None, None, None, None, None, None, 0, None) == 1
    assert "gemm mode" in L.last_error()
    # an FP8 state with too few tensors for a double block, or a position outside the history
    st8 = L.Fp8State(0x1000, 0x2000, 1024, 8, 0, 0, 0)
    assert lib.mmdit_double_block_fwd(C.byref(fp8), C.byref(w), C.byref(w), None, None, None, None,
                                      None, None, None, C.byref(st8), None, 0, None) == 1
    assert "tensors" in L.last_error()
    st8 = L.Fp8State(0x1000, 0x2000, 1024, 16, 1024, 0, 0)
    assert lib.mmdit_single_block_fwd(C.byref(fp8), C.byref(w), None, None, None, None, None,
                                      C.byref(st8), None, 0, None) == 1
    # a state given with the native linears
    st8 = L.Fp8State(0x1000, 0x2000, 1024, 16, 0, 0, 0)
    assert lib.mmdit_single_block_fwd(C.byref(d), C.byref(w), None, None, None, None, None,
                                      C.byref(st8), None, 0, None) == 1
    # an unknown amax algorithm, a margin out of range
    for algo, margin in ((2, 0), (0, -1), (1, 17)):
        st8 = L.Fp8State(0x1000, 0x2000, 1024, 16, 0, algo, margin)
        assert lib.mmdit_double_block_fwd(C.byref(fp8), C.byref(w), C.byref(w), None, None, None, None,
                                          None, None, None, C.byref(st8), None, 0, None) == 1
    # E4M3 cast and FP8 linear shapes
    assert lib.mmdit_fp8_quantize_e4m3(0x1000, 24, 0x2000, 0x3000, 0x4000, None) == 2
    assert lib.mmdit_fp8_quantize_e4m3(0x1000, 0, None, None, None, None) == 0
    assert lib.mmdit_fp8_linear_fwd(8, 96, 64, 0x1000, 0x2000, 0x3000, 0x3004, None, 0x4000, 0x5000,
                                    256, None) == 2
    assert lib.mmdit_fp8_linear_fwd(8, 128, 64, 0x1000, 0x2000, None, 0x3004, None, 0x4000, 0x5000,
                                    256, None) == 1
    mism = _dims(heads=23)
    assert lib.mmdit_double_block_fwd(C.byref(mism), C.byref(w), C.byref(w), None, None, None, None,
                                      None, None, None, None, None, 0, None) == 1
    # odd axes_dim and oversize tables
    axes = (C.c_int32 * 3)(16, 55, 56)
    assert lib.rope3d_freqs(None, 1, 4, axes, 1e4, None, None, None) == 1
    axes = (C.c_int32 * 3)(128, 128, 2)
    assert lib.rope3d_freqs(None, 1, 4, axes, 1e4, None, None, None) == 2
    # empty RoPE call is a no-op
    axes = (C.c_int32 * 3)(16, 56, 56)
    assert lib.rope3d_freqs(None, 0, 4, axes, 1e4, None, None, None) == 0
    # misaligned pointer
    assert lib.mmdit_linear_fwd(1, 8, 32, 8, 0x1001, 0x2000, None, 0x3000, 0x4000, 256, None) == 1
    # shape the tensor-core path does not take
    assert lib.mmdit_linear_fwd(1, 8, 33, 8, 0x1000, 0x2000, None, 0x3000, 0x4000, 256, None) == 2
    # workspace too small / misaligned
    assert lib.mmdit_linear_fwd(1, 8, 32, 8, 0x1000, 0x2000, None, 0x3000, 0x4000, 16, None) == 3
    assert lib.mmdit_linear_fwd(1, 8, 32, 8, 0x1000, 0x2000, None, 0x3000, 0x4010, 4096, None) == 3
    # flow matching: loss needs both pred and loss, n multiple of 8
    assert lib.flow_match_noise_and_loss(0, 0x1000, 0x2000, 0x3000, 1, 12, None, None, None, 0x4000,
                                         4096, None) == 2
    assert lib.flow_match_noise_and_loss(0, 0x1000, 0x2000, 0x3000, 1, 16, None, 0x5000, None,
                                         0x4000, 4096, None) == 1
    assert lib.mmdit_attention_fwd(1, 1, 1, 16, 64, 0x1000, 0x1000, 0x1000, 0x1000, 0x4000, 1 << 20,
                                   None) == 2
    # sampling step: n a multiple of 8, aligned pointers, v_uncond optional
    assert lib.flow_match_euler_step(1, 12, 0x1000, 0x2000, None, 3.5, 0.1, 0x3000, None) == 2
    assert lib.flow_match_euler_step(1, 16, 0x1000, 0x2000, 0x2008, 3.5, 0.1, 0x3000, None) == 1
    assert lib.flow_match_euler_step(0, 0, None, None, None, 1.0, 0.1, None, None) == 0


def test_library_does_not_fall_back(tmp_path, monkeypatch):
    monkeypatch.setattr(build_ext, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(L, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        L.load()


def _flux_cfg(**kw):
    d = _dims(batch=kw.pop("batch", 1), seq_img=1024, seq_txt=512, gemm=kw.pop("gemm", 0))
    base = dict(n_double=19, n_single=38, lat_h=32, lat_w=32)
    base.update(kw)
    return L.make_flux_config(d, **base)


def test_whole_model_workspace_and_validation(lib):
    D, Si, St = 3072, 1024, 512
    cfg = _flux_cfg()
    ws = L.mmdit_flux_workspace_size(cfg)
    # one block region plus vec, 76 modulations and the joint sequence (batch 1: the streams
    # live inside it)
    block = max(L.mmdit_double_block_workspace_size(cfg.block), L.mmdit_single_block_workspace_size(cfg.block))
    floor = block + D * 2 + 76 * 6 * D * 4 + (Si + St) * D * 2
    assert floor <= ws < floor + 64 * 1024
    # batch 2 adds separate image and text streams
    ws2 = L.mmdit_flux_workspace_size(_flux_cfg(batch=2))
    assert ws2 > 2 * ws - block
    # unsupported or inconsistent configurations size to 0 and are rejected before any launch
    assert L.mmdit_flux_workspace_size(_flux_cfg(gemm=1)) == 0
    assert L.mmdit_flux_workspace_size(_flux_cfg(lat_h=16)) == 0
    assert L.mmdit_flux_workspace_size(_flux_cfg(time_dim=1024)) == 0
    assert L.mmdit_flux_workspace_size(_flux_cfg(n_double=-1)) == 0
    fw = L.FluxW()
    for bad, status in ((_flux_cfg(gemm=1), 2), (_flux_cfg(lat_w=31), 1), (_flux_cfg(channels=48), 2)):
        assert lib.mmdit_flux_forward(C.byref(bad), C.byref(fw), 16, 16, 16, 16, None, 16, 16, 16, 16,
                                      1 << 30, None) == status
    # NULL weights are reported, not dereferenced
    assert lib.mmdit_flux_forward(C.byref(cfg), C.byref(fw), 16, 16, 16, 16, None, 16, 16, 16, 16,
                                  1 << 30, None) == 1
    assert "NULL" in L.last_error()


def test_conditioning_and_batched_modulation_validation(lib):
    assert lib.mmdit_conditioning_workspace_size(1, 2, 3072, 256) >= 256 + 2 * 256 * 2 + 2 * 3072 * (2 + 2 + 4)
    cw = L.CondW()
    # odd or oversized time_dim, misaligned widths: unsupported before the weights are looked at
    assert lib.mmdit_conditioning_fwd(1, 2, 3072, 1024, 768, C.byref(cw), 16, 16, None, 16, 16, 1 << 20, None) == 2
    assert lib.mmdit_conditioning_fwd(1, 2, 3072, 256, 770, C.byref(cw), 16, 16, None, 16, 16, 1 << 20, None) == 2
    assert lib.mmdit_conditioning_fwd(1, 2, 3072, 256, 768, C.byref(cw), 16, 16, None, 16, 16, 1 << 20, None) == 1
    job = L.GemvJob(16, None, 16, -1)
    assert lib.mmdit_modulation_batched_fwd(1, 1, 3072, 16, 1, C.byref(job), None) == 1
    assert lib.mmdit_modulation_batched_fwd(1, 1, 3070, 16, 1, C.byref(job), None) == 2
    assert lib.mmdit_modulation_batched_fwd(1, 1, 3072, 16, 1, None, None) == 1
    # nothing to do: no jobs, or an empty batch
    assert lib.mmdit_modulation_batched_fwd(1, 1, 3072, 16, 0, None, None) == 0
    assert lib.mmdit_modulation_batched_fwd(1, 0, 3072, 16, 1, C.byref(job), None) == 0


def test_parallel_single_block_validation(lib):
    sw = L.StreamW()
    # FP8 is not offered for the parallel block; NULL weights are reported
    assert lib.mmdit_single_block_parallel_fwd(C.byref(_dims(gemm=1)), C.byref(sw), 16, 16, 16, 16, 16, 16,
                                               1 << 30, None) == 2
    assert lib.mmdit_single_block_parallel_fwd(C.byref(_dims()), C.byref(sw), 16, 16, 16, 16, 16, 16,
                                               1 << 30, None) == 1


def test_linear_bwd_embedding_head_and_modulation_validation(lib):
    # every case below is rejected before any CUDA call (no launch, no memset)
    ws = L.mmdit_linear_bwd_workspace_size(1, 64, 128, 256)
    assert ws >= 256 + 256 * 128 * 2 + 128 * 64 * 2 + 256 * 64 * 2
    assert lib.mmdit_linear_bwd(7, 64, 128, 256, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mmdit_linear_bwd(1, -1, 128, 256, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mmdit_linear_bwd(1, 64, 128, 48, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 2
    assert lib.mmdit_linear_bwd(1, 64, 100, 256, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 2
    assert lib.mmdit_linear_bwd(1, 64, 128, 256, 0x1008, 16, 16, 16, None, None, 16, 1 << 30, None) == 1
    assert lib.mmdit_linear_bwd(1, 64, 128, 256, 16, None, 16, None, 16, None, 16, 1 << 30, None) == 1
    assert "linear backward x" in L.last_error()
    assert lib.mmdit_linear_bwd(1, 64, 128, 256, 16, 16, 16, None, None, 0x1004, 16, 1 << 30, None) == 1
    assert lib.mmdit_linear_bwd(1, 64, 128, 256, 16, 16, 16, 16, 16, 16, 16, ws - 1, None) == 3
    # img_in: channels a multiple of 8, hidden of 32, every pointer given, workspace big enough
    assert lib.mmdit_img_in_fwd(1, 1, 12, 8, 8, 256, 16, 16, 16, 16, 16, 1 << 30, None) == 2
    assert lib.mmdit_img_in_fwd(1, 1, 64, 8, 8, 48, 16, 16, 16, 16, 16, 1 << 30, None) == 2
    assert lib.mmdit_img_in_fwd(1, 0, 64, 8, 8, 256, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mmdit_img_in_fwd(1, 1, 64, 8, 8, 256, None, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mmdit_img_in_fwd(1, 1, 64, 8, 8, 256, 16, 16, 16, 16, 16, 16, None) == 3
    # output head: seq_img must be lat_h * lat_w; channels a multiple of 32, hidden of 256
    d = _dims(seq_img=64, hidden=256, heads=2, mlp_hidden=1024)
    assert lib.mmdit_final_layer_fwd(C.byref(d), 64, 8, 7, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mmdit_final_layer_fwd(C.byref(d), 48, 8, 8, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 2
    d2 = _dims(seq_img=64, hidden=384, heads=3, mlp_hidden=1536)
    assert lib.mmdit_final_layer_fwd(C.byref(d2), 64, 8, 8, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 2
    assert lib.mmdit_final_layer_fwd(C.byref(d), 64, 8, 8, 16, None, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    assert lib.mmdit_final_layer_fwd(None, 64, 8, 8, 16, 16, 16, 16, 16, 16, 16, 16, 1 << 30, None) == 1
    # output head with the fused loss: the same shape rules; z0, z1 and loss required; pred optional
    # but never aliasing a latent; workspace at least its own size (larger than the head's alone)
    fl = lib.mmdit_final_layer_loss_fwd
    assert fl(C.byref(d), 64, 8, 7, 16, 16, 16, 16, 16, 16, 32, 48, 64, 80, None, 256, 1 << 30, None) == 1
    assert fl(C.byref(d), 48, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, 64, 80, None, 256, 1 << 30, None) == 2
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, None, 48, 64, 80, None, 256, 1 << 30, None) == 1
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, 64, None, None, 256, 1 << 30, None) == 1
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, 64, 82, None, 256, 1 << 30, None) == 1
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, 32, 80, None, 256, 1 << 30, None) == 1
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, 0x1004, 80, None, 256, 1 << 30, None) == 1
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, 64, 80, 0x1004, 256, 1 << 30, None) == 1
    need = L.mmdit_final_layer_loss_workspace_size(d, 64)
    assert need > L.mmdit_final_layer_workspace_size(d, 64)
    assert fl(C.byref(d), 64, 8, 8, 16, 16, 16, 16, 16, 16, 32, 48, None, 80, None, 256, need - 1, None) == 3
    # img_in with the noise fused: z0, z1, t required; z_t optional, never aliasing a latent
    fi = lib.mmdit_img_in_noise_fwd
    assert fi(1, 1, 12, 8, 8, 256, 16, 32, 48, 16, 16, 16, None, 256, 1 << 30, None) == 2
    assert fi(1, 1, 64, 8, 8, 256, 16, None, 48, 16, 16, 16, None, 256, 1 << 30, None) == 1
    assert fi(1, 1, 64, 8, 8, 256, 16, 32, None, 16, 16, 16, None, 256, 1 << 30, None) == 1
    assert fi(1, 1, 64, 8, 8, 256, 16, 32, 48, 16, 16, 16, 32, 256, 1 << 30, None) == 1
    assert fi(1, 1, 64, 8, 8, 256, 16, 32, 48, 16, 16, 16, None, 256, 16, None) == 3
    # modulation GEMV: dim a multiple of 8 and at most 6144; an empty batch does nothing
    assert lib.mmdit_modulation_fwd(1, 1, 6 * 3072, 3070, 16, 16, 16, 16, None) == 2
    assert lib.mmdit_modulation_fwd(1, 1, 6 * 3072, 6152, 16, 16, 16, 16, None) == 2
    assert lib.mmdit_modulation_fwd(1, -1, 6 * 3072, 3072, 16, 16, 16, 16, None) == 1
    assert lib.mmdit_modulation_fwd(1, 1, 6 * 3072, 3072, None, 16, 16, 16, None) == 1
    assert lib.mmdit_modulation_fwd(1, 0, 6 * 3072, 3072, None, None, None, None, None) == 0


def test_block_backward_rejects_bad_arguments_before_any_cuda_call(lib):
    d = _dims(seq_img=256, seq_txt=45, hidden=256, heads=2, mlp_hidden=1024)
    need = L.mmdit_double_block_bwd_workspace_size(d)
    assert need > L.mmdit_double_block_workspace_size(d)
    assert L.mmdit_single_block_bwd_workspace_size(d) > 0
    w = L.StreamW(*([16] * 12), None)
    bad_w = L.StreamW(*([16] * 11 + [0x1004]), None)
    g_bad = L.StreamGrads(*([None] * 6 + [0x1004] + [None] * 5))
    ptrs = [16] * 9  # vec, cos, sin, x_img, x_txt, dy_img, dy_txt, dx_img, dx_txt
    db = lib.mmdit_double_block_bwd

    def call(dims=d, wi=w, wt=w, p=ptrs, dvec=None, gi=None, gt=None, ws=256, nbytes=1 << 40):
        return db(C.byref(dims), C.byref(wi), C.byref(wt), *p, dvec, gi, gt, ws, nbytes, None)

    assert call(dims=_dims(seq_img=256, seq_txt=45, hidden=256, heads=2, mlp_hidden=1024, act=L.MMDIT_F32)) == 2
    assert call(dims=_dims(seq_img=256, seq_txt=0, hidden=256, heads=2, mlp_hidden=1024)) == 2
    assert call(dims=_dims(batch=9, seq_img=256, seq_txt=45, hidden=256, heads=2, mlp_hidden=1024)) == 2
    assert call(dims=_dims(seq_img=256, seq_txt=45, hidden=256, heads=2, mlp_hidden=1024, gemm=1)) == 2
    assert call(wi=bad_w) == 1
    assert call(p=[16] * 8 + [None]) == 1
    assert call(dvec=0x1004) == 1
    assert call(gi=C.byref(g_bad)) == 1
    assert "gradient 6" in L.last_error()
    assert call(nbytes=need - 1) == 3
    sb = lib.mmdit_single_block_bwd
    assert sb(C.byref(d), C.byref(w), 16, 16, 16, 16, 16, None, None, None, 256, 1 << 40, None) == 1
    assert sb(C.byref(d), C.byref(w), 16, 16, 16, 16, 16, 16, None, None, 256, 16, None) == 3


def test_blockwise_fp8_linear_rejects_bad_arguments_before_any_cuda_call(lib):
    need = L.mmdit_fp8_blockwise_linear_workspace_size(300, 256, 512)
    # status word, codes of x and W, both scale arrays, each on a 256-byte boundary
    assert need == 256 + 153600 + 131072 + 4864 + 256
    f = lib.mmdit_fp8_blockwise_linear_fwd
    assert f(300, 200, 512, 16, 16, None, 16, 256, 1 << 30, None) == 2      # N % 128
    assert f(300, 256, 500, 16, 16, None, 16, 256, 1 << 30, None) == 2      # K % 128
    assert f(-1, 256, 512, 16, 16, None, 16, 256, 1 << 30, None) == 1
    assert f(300, 256, 512, None, 16, None, 16, 256, 1 << 30, None) == 1
    assert "blockwise FP8 linear" in L.last_error()
    assert f(300, 256, 512, 16, 16, 0x1008, 16, 256, 1 << 30, None) == 1   # bias alignment
    assert f(300, 256, 512, 16, 16, None, 16, 256, need - 1, None) == 3


def test_mxfp8_linear_rejects_bad_arguments_before_any_cuda_call(lib):
    need = L.mmdit_fp8_mxfp8_linear_workspace_size(300, 96, 512)
    # status word; bf16 values of x and W; codes of x and W; E8M0 scales of x and W; each part on
    # a 256-byte boundary
    assert need == 256 + 307200 + 98304 + 153600 + 49152 + 4864 + 1536
    f = lib.mmdit_fp8_mxfp8_linear_fwd
    assert f(300, 80, 512, 16, 16, None, 16, 256, 1 << 30, None) == 2       # N % 32
    assert f(300, 96, 500, 16, 16, None, 16, 256, 1 << 30, None) == 2       # K % 32
    assert f(-1, 96, 512, 16, 16, None, 16, 256, 1 << 30, None) == 1
    assert f(300, 96, 512, 16, None, None, 16, 256, 1 << 30, None) == 1
    assert "MXFP8 linear" in L.last_error()
    assert f(300, 96, 512, 16, 16, 0x1008, 16, 256, 1 << 30, None) == 1    # bias alignment
    assert f(300, 96, 512, 16, 16, None, 16, 256, need - 1, None) == 3


def test_training_pair_rejects_bad_arguments_before_any_cuda_call(lib):
    # the split backward: same checks as the one-call backward; the forward half needs the
    # outputs y, the backward half dy and dx, both a backward-sized `saved` buffer
    d = _dims(seq_img=256, seq_txt=45, hidden=256, heads=2, mlp_hidden=1024)
    need = L.mmdit_double_block_bwd_workspace_size(d)
    w = L.StreamW(*([16] * 12), None)
    ft, bs = lib.mmdit_double_block_fwd_train, lib.mmdit_double_block_bwd_saved
    # fwd_train(dims, w_img, w_txt, vec, cos, sin, x_img, x_txt, y_img, y_txt, saved, bytes, stream)
    assert ft(C.byref(d), C.byref(w), C.byref(w), 16, 16, 16, 16, 16, None, 16, 256, 1 << 40, None) == 1
    assert "training forward" in L.last_error()
    assert ft(C.byref(d), C.byref(w), C.byref(w), 16, 16, 16, 16, 16, 16, 16, 256, need - 1, None) == 3
    f32 = _dims(seq_img=256, seq_txt=45, hidden=256, heads=2, mlp_hidden=1024, act=L.MMDIT_F32)
    assert ft(C.byref(f32), C.byref(w), C.byref(w), 16, 16, 16, 16, 16, 16, 16, 256, 1 << 40, None) == 2
    # bwd_saved(dims, w_img, w_txt, vec, cos, sin, x_img, x_txt, dy_img, dy_txt, dx_img, dx_txt, dvec,
    #           g_img, g_txt, saved, bytes, stream)
    assert bs(C.byref(d), C.byref(w), C.byref(w), 16, 16, 16, 16, 16, 16, 16, 16, None, None, None, None,
              256, 1 << 40, None) == 1
    assert "saved forward" in L.last_error()
    assert bs(C.byref(d), C.byref(w), C.byref(w), 16, 16, 16, 16, 16, 16, 16, 16, 16, 0x1004, None, None,
              256, 1 << 40, None) == 1
    assert bs(C.byref(d), C.byref(w), C.byref(w), 16, 16, 16, 16, 16, 16, 16, 16, 16, None, None, None,
              256, need - 1, None) == 3
    sft, sbs = lib.mmdit_single_block_fwd_train, lib.mmdit_single_block_bwd_saved
    assert sft(C.byref(d), C.byref(w), 16, 16, 16, 16, None, 256, 1 << 40, None) == 1
    assert sbs(C.byref(d), C.byref(w), 16, 16, 16, 16, 16, None, None, None, 256, 1 << 40, None) == 1
    assert sbs(C.byref(d), C.byref(w), 16, 16, 16, 16, 16, 16, None, None, 256,
               L.mmdit_single_block_bwd_workspace_size(d) - 1, None) == 3


def test_binding_refuses_host_tensors():
    # a host tensor's address would reach a kernel as if it were device memory
    import torch
    with pytest.raises(ValueError, match="CUDA tensor"):
        L._ptr(torch.zeros(8))
    assert L._ptr(None) is None and L._ptr(0x1000) == 0x1000
