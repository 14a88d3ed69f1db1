"""The selective Adam kernel (gs2d_adam_step) against the oracle's Adam in
double: several steps on random parameters and gradients of widely spread
magnitudes, rows of width 1, 2 and 3, with and without a pair-count
selection.  FP32 against double: each element within a few ulp of the
parameter's size; the rows a selection skips must not change at all."""
import numpy as np
import pytest
import torch

import oracle
from raster_gaussian_02_b300 import gs2d

pytestmark = pytest.mark.gpu

# The call takes FP32 hyperparameters; the oracle gets the same values widened.
LR, B1, B2, EPS = (float(np.float32(x)) for x in (1e-2, 0.9, 0.999, 1e-8))


@pytest.mark.parametrize("width", [1, 2, 3])
@pytest.mark.parametrize("selective", [False, True])
def test_adam_matches_oracle_over_steps(width, selective):
    rng = np.random.default_rng(10 * width + selective)
    n = 5003
    shape = (n,) if width == 1 else (n, width)
    p = rng.normal(size=shape).astype(np.float32)
    m = np.zeros(shape, np.float32)
    v = np.zeros(shape, np.float32)
    count = (rng.integers(0, 4, n) * (rng.random(n) < 0.7)).astype(np.int32) if selective else None
    dev = torch.device("cuda")
    tp, tm, tv = (torch.from_numpy(a.copy()).to(dev) for a in (p, m, v))
    tc = None if count is None else torch.from_numpy(count).to(dev)
    rp, rm, rv = p.astype(np.float64), m.astype(np.float64), v.astype(np.float64)
    for step in range(1, 6):
        g = (rng.normal(size=shape) * 10.0 ** rng.uniform(-4, 2, shape)).astype(np.float32)
        gs2d.adam_step(tp, torch.from_numpy(g).to(dev), tm, tv, step, lr=LR, beta1=B1, beta2=B2, eps=EPS,
                       count=tc)
        m_scale = 0.9 * np.abs(rm) + 0.1 * np.abs(g.astype(np.float64))  # size of m's two terms
        rp, rm, rv = oracle.adam_step(rp, g, rm, rv, step, LR, B1, B2, EPS, count=count)
        # the oracle continues from the kernel's FP32 state so errors do not compound
        torch.cuda.synchronize()
        gp, gm, gv = (t.cpu().numpy().astype(np.float64) for t in (tp, tm, tv))
        assert np.all(np.abs(gm - rm) <= 2e-6 * m_scale), (np.abs(gm - rm) / np.maximum(m_scale, 1e-300)).max()
        assert np.allclose(gv, rv, rtol=2e-6, atol=0), np.abs(gv - rv).max()
        # one step moves p by at most lr (1 + rounding): compare relative to that scale
        err = np.abs(gp - rp) / (np.abs(rp) + 1e-2)
        assert err.max() <= 1e-5, err.max()
        rp, rm, rv = gp, gm, gv
    if selective:
        off = count == 0
        assert np.array_equal(tp.cpu().numpy()[off], p[off])
        assert not tm.cpu().numpy()[off].any() and not tv.cpu().numpy()[off].any()


def test_first_step_closed_form():
    """From zero moments the first step moves every element by lr g/(|g| + eps)."""
    n = 1000
    rng = np.random.default_rng(5)
    g = (rng.normal(size=(n, 2)) * 10.0 ** rng.uniform(-3, 3, (n, 2))).astype(np.float32)
    dev = torch.device("cuda")
    tp = torch.zeros((n, 2), device=dev)
    tm, tv = torch.zeros_like(tp), torch.zeros_like(tp)
    gs2d.adam_step(tp, torch.from_numpy(g).to(dev), tm, tv, 1, lr=0.5, eps=EPS)
    got = tp.cpu().numpy().astype(np.float64)
    g64 = g.astype(np.float64)
    want = -0.5 * g64 / (np.abs(g64) + EPS)
    assert np.allclose(got, want, rtol=1e-5, atol=0), np.abs(got - want).max()


def test_rejects_bad_arguments():
    dev = torch.device("cuda")
    t = torch.zeros((4, 2), device=dev)
    for kw in (dict(step=0, lr=1.0), dict(step=1, lr=-1.0), dict(step=1, lr=1.0, beta1=1.0),
               dict(step=1, lr=1.0, beta2=-0.1), dict(step=1, lr=1.0, eps=0.0)):
        with pytest.raises(gs2d.Gs2dError):
            gs2d.adam_step(t, t.clone(), t.clone(), t.clone(), **kw)
