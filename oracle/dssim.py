"""D-SSIM loss term and its gradient, fp64 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It shares no code with the CUDA path.

The training loss on the pages ("Grendel: scaling 3D Gaussian Splatting
training", summary of the loss) is the standard 3DGS one, L1 plus a D-SSIM
term, without restating SSIM.  The reading taken here is the usual one
(Wang et al., "Image quality assessment: from error visibility to structural
similarity", with the 3DGS settings), written out from its definition:

* each colour channel separately, window w = 11 x 11 Gaussian of standard
  deviation 1.5, normalised to sum 1 over its 121 taps;
* windowed moments with the image zero-padded outside its borders
  (the window is not renormalised near a border):
  mu_x = w * x, mu_y = w * y, s_xx = w * x^2 - mu_x^2, s_yy = w * y^2 - mu_y^2,
  s_xy = w * (x y) - mu_x mu_y;
* SSIM map (2 mu_x mu_y + C1)(2 s_xy + C2) / ((mu_x^2 + mu_y^2 + C1)(s_xx + s_yy + C2))
  with C1 = 0.01^2, C2 = 0.03^2 (dynamic range 1);
* SSIM = mean of the map over channels and pixels;
* loss = (1 - lambda) L1 + lambda (1 - SSIM), lambda = 0.2, L1 the mean absolute
  error over channels and pixels.

The gradient is the chain rule through the three windowed moments that depend
on x (mu_x, E[x^2] = w * x^2, E[xy] = w * (x y)); because w is symmetric, the
adjoint of "window sum around p" is again a window sum, so

  dSSIM/dx_q = (1/N) [ w * dS/dmu_x + 2 x_q (w * dS/dE[x^2]) + y_q (w * dS/dE[xy]) ](q)

with N = 3 H W and, writing A = 2 mu_x mu_y + C1, B = 2 s_xy + C2,
C = mu_x^2 + mu_y^2 + C1, D = s_xx + s_yy + C2, S = A B / (C D):

  dS/dmu_x  = 2 mu_y (B - A) / (C D) - 2 mu_x S (D - C) / (C D)
  dS/dE[x^2] = -S / D
  dS/dE[xy]  = 2 A / (C D)

(no division by B, which may be zero or negative).  The window sums are
written as plain 121-tap double loops over shifted, zero-padded copies.
"""
from __future__ import annotations

import numpy as np

WINDOW = 11
SIGMA = 1.5
C1 = 0.01 ** 2
C2 = 0.03 ** 2
LAMBDA = 0.2


def window() -> np.ndarray:
    """The 11 x 11 Gaussian window (outer product of the normalised 1-D one)."""
    r = WINDOW // 2
    t = np.arange(-r, r + 1, dtype=np.float64)
    g = np.exp(-t * t / (2.0 * SIGMA * SIGMA))
    g /= g.sum()
    return np.outer(g, g)


def wsum(img: np.ndarray) -> np.ndarray:
    """Window sum around every pixel of [..., H, W], zero outside the image."""
    w = window()
    r = WINDOW // 2
    H, W = img.shape[-2:]
    pad = np.zeros(img.shape[:-2] + (H + 2 * r, W + 2 * r), np.float64)
    pad[..., r:r + H, r:r + W] = img
    out = np.zeros(img.shape, np.float64)
    for dy in range(WINDOW):
        for dx in range(WINDOW):
            out += w[dy, dx] * pad[..., dy:dy + H, dx:dx + W]
    return out


def ssim_map(x: np.ndarray, y: np.ndarray) -> np.ndarray:
    """Per-channel, per-pixel SSIM of images [3, H, W]."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    mx, my = wsum(x), wsum(y)
    exx, eyy, exy = wsum(x * x), wsum(y * y), wsum(x * y)
    A = 2.0 * mx * my + C1
    B = 2.0 * (exy - mx * my) + C2
    C = mx * mx + my * my + C1
    D = (exx - mx * mx) + (eyy - my * my) + C2
    return (A * B) / (C * D)


def ssim(x, y) -> float:
    return float(ssim_map(x, y).mean())


def ssim_terms(x, y) -> dict:
    """Every intermediate of the SSIM map and of its derivatives, per channel and pixel:
    the moments, A, B, C, D, S and the three derivative maps dS/dmu_x, dS/dE[x^2],
    dS/dE[xy]."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    mx, my = wsum(x), wsum(y)
    exx, eyy, exy = wsum(x * x), wsum(y * y), wsum(x * y)
    A = 2.0 * mx * my + C1
    B = 2.0 * (exy - mx * my) + C2
    C = mx * mx + my * my + C1
    D = (exx - mx * mx) + (eyy - my * my) + C2
    CD = C * D
    S = (A * B) / CD
    return dict(mx=mx, my=my, exx=exx, eyy=eyy, exy=exy, A=A, B=B, C=C, D=D, S=S,
                d_mu=2.0 * my * (B - A) / CD - 2.0 * mx * S * (D - C) / CD,
                d_exx=-S / D, d_exy=2.0 * A / CD)


def ssim_grad(x, y) -> np.ndarray:
    """d SSIM / d x for images [3, H, W] (SSIM = mean of the map)."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    t = ssim_terms(x, y)
    return (wsum(t["d_mu"]) + 2.0 * x * wsum(t["d_exx"]) + y * wsum(t["d_exy"])) / float(x.size)


def loss(x, y, lam: float = LAMBDA) -> float:
    """(1 - lam) L1 + lam (1 - SSIM) of images [3, H, W]."""
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    return (1.0 - lam) * float(np.abs(x - y).mean()) + lam * (1.0 - ssim(x, y))


def dssim_dldc(x, y, lam: float = LAMBDA) -> np.ndarray:
    """The D-SSIM term's share of dL/dC: -lam d SSIM / d x.  The L1 share
    ((1 - lam) sign(x - y) / N) is added by the renderer."""
    return -lam * ssim_grad(x, y)
