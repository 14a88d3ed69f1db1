"""gs2d_loss_l2_noalloc: the L2 loss for callers that cannot allocate device
memory (for instance code handed its buffers by another framework, with no
allocator of its own, or a loop that must not call cudaMalloc because it
synchronises the device).  It keeps its partial sums in a fixed array inside
the library instead of a caller workspace.

Checked through the C ABI against gs2d_loss_l2 (the workspace version), on
two calls in a row with different images, so that the shared array's
leftovers from the first call cannot leak into the second.  This file is
named to be collected last; it passes alone in a fresh process (where its
first call also looks the array's address up) and after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from raster_gaussian_02_b300 import gs2d

pytestmark = pytest.mark.gpu


def _loss_with_workspace(lib, h, w, img, tgt, stream):
    ws = torch.empty(gs2d.gs2d_workspace_size(gs2d.make_config(w, h), 0, 0), dtype=torch.uint8,
                     device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    d = torch.empty_like(img)
    st = lib.gs2d_loss_l2(h, w, img.data_ptr(), tgt.data_ptr(), loss.data_ptr(), d.data_ptr(),
                          ws.data_ptr(), stream)
    assert st == gs2d.GS2D_OK
    return loss, d


def test_noalloc_loss_matches_workspace_loss_on_two_calls():
    lib = gs2d.lib()
    stream = torch.cuda.current_stream().cuda_stream
    # the first size takes the vectorised path, the second the scalar one
    for h, w, seed in [(512, 768, 11), (37, 101, 12)]:
        g = torch.Generator().manual_seed(seed)
        img = torch.rand(3, h, w, generator=g).cuda()
        tgt = torch.rand(3, h, w, generator=g).cuda()
        loss_ref, d_ref = _loss_with_workspace(lib, h, w, img, tgt, stream)
        loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        d = torch.full_like(img, float("nan"))
        st = lib.gs2d_loss_l2_noalloc(h, w, img.data_ptr(), tgt.data_ptr(), loss.data_ptr(),
                                      d.data_ptr(), stream)
        assert st == gs2d.GS2D_OK
        torch.cuda.synchronize()
        a, b = float(loss.item()), float(loss_ref.item())
        assert abs(a - b) <= 1e-5 * abs(b), (a, b)
        np.testing.assert_allclose(d.cpu().numpy(), d_ref.cpu().numpy(), rtol=1e-5,
                                   atol=1e-7 * float(d_ref.abs().max()))
        # and against the definition, in double on the host
        e = (img.double() - tgt.double())
        assert abs(a - float((e * e).mean())) <= 1e-5 * abs(a)


def test_noalloc_loss_rejects_images_beyond_the_limit():
    lib = gs2d.lib()
    fake = C.c_void_p(0x10000)
    assert lib.gs2d_loss_l2_noalloc(40000, 16, fake, fake, fake, fake, None) == gs2d.GS2D_ERR_INVALID_ARG
    assert lib.gs2d_loss_l2_noalloc(16, 0, fake, fake, fake, fake, None) == gs2d.GS2D_ERR_INVALID_ARG
    assert lib.gs2d_loss_l2_noalloc(16, 16, None, fake, fake, fake, None) == gs2d.GS2D_ERR_INVALID_ARG
