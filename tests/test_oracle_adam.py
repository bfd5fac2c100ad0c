"""Pins of the oracle's optimizer and compaction.

- dense Adam in fp64 equals torch.optim.Adam (the library routine) in fp64;
- deferred Adam (catch-up of skipped zero-gradient steps, then the step) equals
  dense Adam stepped every iteration, bit for bit in fp32, over random masks;
- from a zero state with zero gradients the update is exactly zero;
- flush brings every Gaussian to the current step;
- compaction equals numpy's flatnonzero.
"""
import numpy as np
import pytest
import torch

import oracle


def test_dense_adam_matches_torch_fp64():
    rng = np.random.default_rng(0)
    rows, n = 5, 40
    p = rng.standard_normal((rows, n))
    lr = np.array([1e-3, 2e-2, 5e-4, 1e-1, 3e-3])
    b1, b2, eps = 0.9, 0.999, 1e-8
    m = np.zeros_like(p); v = np.zeros_like(p)
    tp = [torch.tensor(p[r].copy(), dtype=torch.float64, requires_grad=True) for r in range(rows)]
    opt = torch.optim.Adam([{"params": [tp[r]], "lr": float(lr[r])} for r in range(rows)], betas=(b1, b2), eps=eps)
    for t in range(1, 16):
        g = rng.standard_normal((rows, n)) * (rng.uniform(size=(rows, n)) < 0.7)
        oracle.adam_dense_step(p, m, v, g.copy(), lr, t, b1, b2, eps, prec="f64")
        for r in range(rows):
            tp[r].grad = torch.tensor(g[r], dtype=torch.float64)
        opt.step()
        ref = np.stack([x.detach().numpy() for x in tp])
        assert np.allclose(p, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("prec", ["f32", "f64"])
def test_deferred_equals_dense_bitwise(prec):
    dt = np.float32 if prec == "f32" else np.float64
    rng = np.random.default_rng(1)
    rows, n = 6, 300
    p0 = rng.standard_normal((rows, n)).astype(dt)
    lr = np.linspace(1e-3, 5e-2, rows).astype(dt)
    b1, b2, eps = 0.9, 0.999, 1e-8
    pd, md, vd = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    pf, mf, vf = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    last = np.zeros(n, np.int32)
    gbuf = np.zeros_like(p0)
    for t in range(1, 14):
        mask = rng.uniform(size=n) < (0.05 if t < 4 else 0.4)
        g = (rng.standard_normal((rows, n)) * mask[None, :]).astype(dt)
        oracle.adam_dense_step(pd, md, vd, g, lr, t, b1, b2, eps, prec=prec)
        gbuf[:] = g
        idx = np.flatnonzero(mask).astype(np.uint32)
        oracle.adam_deferred(pf, mf, vf, gbuf, last, lr, idx, t, b1, b2, eps, prec=prec)
        assert not gbuf[:, idx].any()                 # consumed gradients are cleared
        assert (last[idx] == t).all()
        touched = last == t
        assert np.array_equal(pf[:, touched], pd[:, touched])
        assert np.array_equal(mf[:, touched], md[:, touched]) and np.array_equal(vf[:, touched], vd[:, touched])
    oracle.adam_deferred(pf, mf, vf, gbuf, last, lr, None, 13, b1, b2, eps, flush=True, prec=prec)
    assert (last == 13).all()
    assert np.array_equal(pf, pd) and np.array_equal(mf, md) and np.array_equal(vf, vd)


def test_zero_state_zero_gradient_is_a_fixed_point():
    rows, n = 3, 10
    p = np.random.default_rng(2).standard_normal((rows, n)).astype(np.float32)
    p0 = p.copy()
    m = np.zeros_like(p); v = np.zeros_like(p); g = np.zeros_like(p)
    last = np.zeros(n, np.int32)
    oracle.adam_deferred(p, m, v, g, last, np.full(rows, 0.1, np.float32), np.arange(n, dtype=np.uint32),
                         25, 0.9, 0.999, 1e-8)
    assert np.array_equal(p, p0) and not m.any() and not v.any()


def test_compaction_is_flatnonzero():
    t = (np.random.default_rng(3).uniform(size=10007) < 0.3).astype(np.uint8)
    assert np.array_equal(oracle.compact(t), np.flatnonzero(t).astype(np.uint32))
    assert oracle.compact(np.zeros(5, np.uint8)).size == 0
