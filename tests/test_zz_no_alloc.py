"""flow_match_noise_and_loss_noalloc: the flow-matching noise and loss for callers that cannot
allocate device memory (a plug-in under another framework's allocator, or a host whose memory is
fixed at start-up).  Its partial sums live in a static device array instead of a caller
workspace; its results must equal the workspace entry point's bit for bit, and a call must not
change the memory torch has allocated.

This file is collected last so that a run stopping at the first failure has run every other
test first.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from diffusion_transformer_flux_gb300 import _lib as L
from diffusion_transformer_flux_gb300 import build_ext, synth


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    build_ext.build()
    lib = L.load()
    # 4 x 64 x 128 x 128 = 4,194,304 elements > 2,097,152: rejected before any CUDA call
    st = lib.flow_match_noise_and_loss_noalloc(0, 0x1000, 0x2000, 0x3000, 4, 64 * 128 * 128, None,
                                               0x4000, 0x5000, None)
    assert st == 2
    assert "2,097,152" in L.last_error()
    # a per-sample count whose product with the batch overflows int64 is rejected the same way
    # (the limit is checked before the product is formed)
    st = lib.flow_match_noise_and_loss_noalloc(0, 0x1000, 0x2000, 0x3000, 4, (1 << 62) + 8, None,
                                               0x4000, 0x5000, None)
    assert st == 2
    assert "2,097,152" in L.last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_no_alloc_matches_workspace_entry_point_twice(dtype):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    L.load()
    for call, shape in enumerate([(4, 64, 32, 32), (2, 64, 64, 64)]):
        rng = np.random.default_rng(100 + call)
        z0, z1 = synth.latent_pair(rng, *shape)
        t = torch.from_numpy(synth.timesteps(rng, shape[0], "logit_normal")).cuda()
        d0 = torch.from_numpy(z0).cuda().to(dtype)
        d1 = torch.from_numpy(z1).cuda().to(dtype)
        pred = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).cuda().to(dtype)
        zt_ref, loss_ref = torch.empty_like(d0), torch.zeros(1, device="cuda")
        L.flow_match_noise_and_loss(d0, d1, t, z_t=zt_ref, pred=pred, loss=loss_ref)
        zt, loss = torch.full_like(d0, float("nan")), torch.full((1,), float("nan"), device="cuda")
        torch.cuda.synchronize()
        allocated = torch.cuda.memory_allocated()
        L.flow_match_noise_and_loss_noalloc(d0, d1, t, z_t=zt, pred=pred, loss=loss)
        torch.cuda.synchronize()
        assert torch.cuda.memory_allocated() == allocated, "the call allocated device memory"
        # same kernels, same grid, same reduction order: bit-equal results
        assert torch.equal(zt, zt_ref), f"call {call}: z_t differs"
        assert loss.item() == loss_ref.item(), f"call {call}: loss {loss.item()} vs {loss_ref.item()}"
        assert np.isfinite(loss.item())
