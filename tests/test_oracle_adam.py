"""Pins of the oracle's selective Adam step (oracle.adam_step) against closed
forms of Adam's recurrences (the pages name a selective Adam on row-aligned
state, DrawingWithGaussians README, MLX-specific notes, and give no
formula).  Each pin follows from the definition by algebra, not by
re-running it:
  - from zero moments, step 1 gives mhat = g and vhat = g^2 exactly;
  - a constant gradient keeps mhat = g and vhat = g^2 at every step (the
    bias corrections undo the moments' warm-up);
  - +g then -g gives mhat_2 = -(1 - beta1)/(1 + beta1) g and vhat_2 = g^2;
  - beta1 = beta2 = 0 reduces to p - lr g / (|g| + eps) whatever the state;
  - count 0 rows keep parameters and moments; the other rows are unchanged
    by the selection;
  - a zero gradient from zero moments moves nothing.
A set of planted mistakes checks that every one of them trips a pin."""
import numpy as np
import pytest

import oracle

LR, B1, B2, EPS = 0.01, 0.9, 0.999, 1e-8


def _data(seed=0, shape=(64, 3)):
    rng = np.random.default_rng(seed)
    p0 = rng.normal(size=shape)
    g = rng.normal(size=shape) * 10.0 ** rng.uniform(-3, 2, shape)
    return p0, g


def pins(adam):
    """Name -> whether `adam` (oracle.adam_step's signature) meets the pin."""
    p0, g = _data()
    z = np.zeros_like(p0)
    out = {}
    p1, m1, v1 = adam(p0, g, z, z, 1, LR, B1, B2, EPS)
    out["first step"] = (np.allclose(p1, p0 - LR * g / (np.abs(g) + EPS), rtol=0, atol=1e-13)
                         and np.allclose(m1, (1 - B1) * g, rtol=1e-14, atol=0)
                         and np.allclose(v1, (1 - B2) * g * g, rtol=1e-14, atol=0))
    p, m, v = p0, z, z
    for t in range(1, 8):
        p, m, v = adam(p, g, m, v, t, LR, B1, B2, EPS)
    out["constant gradient"] = np.allclose(p, p0 - 7 * LR * g / (np.abs(g) + EPS), rtol=0, atol=1e-12)
    pa, ma, va = adam(p0, g, z, z, 1, LR, B1, B2, EPS)
    pb, _, _ = adam(pa, -g, ma, va, 2, LR, B1, B2, EPS)
    mhat2 = -(1 - B1) / (1 + B1) * g
    out["alternating sign"] = np.allclose(pb, pa - LR * mhat2 / (np.abs(g) + EPS), rtol=0, atol=1e-12)
    rng = np.random.default_rng(3)
    rm, rv = rng.normal(size=p0.shape), rng.uniform(0, 4, p0.shape)
    pz, mz, vz = adam(p0, g, rm, rv, 5, LR, 0.0, 0.0, EPS)
    out["zero betas"] = (np.allclose(pz, p0 - LR * g / (np.abs(g) + EPS), rtol=0, atol=1e-13)
                         and np.allclose(mz, g, rtol=1e-15, atol=0) and np.allclose(vz, g * g, rtol=1e-15, atol=0))
    count = (np.arange(p0.shape[0]) % 3 != 0).astype(np.int32)
    ps, ms, vs = adam(p0, g, rm, rv, 4, LR, B1, B2, EPS, count=count)
    pf, mf, vf = adam(p0, g, rm, rv, 4, LR, B1, B2, EPS)
    off, on = count == 0, count != 0
    out["selective rows"] = (np.array_equal(ps[off], p0[off]) and np.array_equal(ms[off], rm[off])
                             and np.array_equal(vs[off], rv[off]) and np.array_equal(ps[on], pf[on])
                             and np.array_equal(ms[on], mf[on]) and np.array_equal(vs[on], vf[on])
                             and not np.allclose(ps[off], pf[off]))
    p0z, m0z, v0z = adam(p0, z, z, z, 1, LR, B1, B2, EPS)
    out["zero gradient"] = np.array_equal(p0z, p0) and not m0z.any() and not v0z.any()
    return out


def test_oracle_meets_every_pin():
    got = pins(oracle.adam_step)
    assert all(got.values()), {k: v for k, v in got.items() if not v}


def test_one_dimensional_rows():
    p0, g = _data(shape=(40,))
    z = np.zeros_like(p0)
    p1, _, _ = oracle.adam_step(p0, g, z, z, 1, LR, B1, B2, EPS, count=np.ones(40, np.int32))
    assert np.allclose(p1, p0 - LR * g / (np.abs(g) + EPS), rtol=0, atol=1e-13)


def _mutant(kind):
    @np.errstate(divide="ignore", invalid="ignore")
    def adam(param, grad, m, v, step, lr, beta1=0.9, beta2=0.999, eps=1e-8, count=None):
        p = np.array(param, np.float64)
        g = np.asarray(grad, np.float64)
        m = np.array(m, np.float64)
        v = np.array(v, np.float64)
        b1, b2 = (1 - beta1, 1 - beta2) if kind == "betas swapped" else (beta1, beta2)
        mn = b1 * m + (1 - b1) * g
        vn = b2 * v + (1 - b2) * (np.abs(g) if kind == "first power in v" else g * g)
        bc1 = 1.0 if kind == "no bias correction" else 1 - b1 ** step
        bc2 = 1.0 if kind == "no bias correction" else 1 - b2 ** step
        if kind == "eps inside the root":
            pn = p - lr * (mn / bc1) / np.sqrt(vn / bc2 + eps)
        else:
            pn = p - lr * (mn / bc1) / (np.sqrt(vn / bc2) + eps)
        if kind == "sign":
            pn = 2 * p - pn
        if count is None or kind == "selection ignored":
            return pn, mn, vn
        sel = (np.asarray(count) != 0).reshape((-1,) + (1,) * (p.ndim - 1))
        return np.where(sel, pn, p), np.where(sel, mn, m), np.where(sel, vn, v)
    return adam


@pytest.mark.parametrize("kind", ["betas swapped", "first power in v", "no bias correction",
                                  "eps inside the root", "sign", "selection ignored"])
def test_each_planted_mistake_trips_a_pin(kind):
    assert not all(pins(_mutant(kind)).values())
