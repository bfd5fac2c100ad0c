"""Seeded synthetic scenes for the five workloads (tiny, small, medium, large, batched).

This module only draws inputs: Gaussian parameters, cameras, training targets of
the uniform-noise kind, and the perturbed parameter set that a "perturbed-scene
render" target is rendered from. It contains none of the rasterizer's arithmetic
(no projection, no compositing, no spherical-harmonic evaluation), so both the
CPU oracle and the CUDA path can take their inputs from it without sharing code.

Parameter layout (float32, row-major ``[P, N]``, one row per scalar parameter):

====== ===========================================================
rows   meaning
====== ===========================================================
0..2   mean x, y, z (world units)
3..5   log-scale along the three local axes
6..9   rotation quaternion (w, x, y, z), stored normalised
10     opacity logit (opacity = sigmoid(logit))
11..13 RGB (degree 0)                          -- P = 14
11..58 SH coefficient k (0..15), channel c at row 11 + 3k + c -- P = 59
====== ===========================================================

The workloads stand in for the evaluation scenes of the pages (ByteSplat's six
datasets, Grendel's Rubble, the "large-scale datasets" of GS-Scale and Splaxel),
which are not available; sizes follow the configurations listed with the task.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

PARAM_ROWS = {0: 14, 3: 59}
ROW_MEAN, ROW_LOGSCALE, ROW_QUAT, ROW_OPACITY, ROW_COLOUR = 0, 3, 6, 10, 11

SEEDS = {"tiny": 0, "small": 1, "medium": 2, "large": 3, "batched": 4}

# Render options shared by every workload: near plane, EWA low-pass (px^2),
# alpha skip threshold, alpha clamp, transmittance stop, background colour.
DEFAULT_OPTS = dict(near_z=0.2, lowpass=0.3, alpha_min=np.float32(1.0) / np.float32(255.0),
                    alpha_max=0.99, t_min=1e-4, bg=(0.0, 0.0, 0.0), exclude_crossing=0)

# Adam hyper-parameters: per parameter group learning rates
# (mean, log-scale, quaternion, opacity logit, colour) and moments.
DEFAULT_LR = (1.6e-4, 5e-3, 1e-3, 5e-2, 2.5e-3)
ADAM_BETAS = (0.9, 0.999)
ADAM_EPS = 1e-8


@dataclasses.dataclass
class Camera:
    R: np.ndarray        # (3, 3) float32, world -> camera rotation (rows = camera x, y, z axes)
    t: np.ndarray        # (3,) float32, world -> camera translation
    fx: float
    fy: float
    cx: float
    cy: float
    width: int
    height: int


@dataclasses.dataclass
class Scene:
    name: str
    params: np.ndarray            # (P, N) float32
    sh_degree: int
    cameras: list                 # list[Camera]
    target_kind: str              # "uniform" or "perturbed"
    target_uniform: np.ndarray | None   # (V, 3, H, W) float32 for "uniform"
    perturbed_params: np.ndarray | None # (P, N) float32 for "perturbed"
    lr: tuple                     # per-group learning rates, already batch-scaled
    opts: dict

    @property
    def n(self) -> int:
        return self.params.shape[1]

    @property
    def n_views(self) -> int:
        return len(self.cameras)


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def _look_at(centre, target, up=(0.0, 0.0, 1.0)):
    """Camera looking from ``centre`` at ``target``; image x right, y down."""
    centre = np.asarray(centre, np.float64)
    f = np.asarray(target, np.float64) - centre
    f /= np.linalg.norm(f)
    x = np.cross(f, np.asarray(up, np.float64))
    x /= np.linalg.norm(x)
    y = np.cross(f, x)
    R = np.stack([x, y, f])
    t = -R @ centre
    return _f32(R), _f32(t)


def _common_params(rng, n, means, log_lo, log_hi, logit_mu, logit_sigma, sh_degree):
    P = PARAM_ROWS[sh_degree]
    p = np.empty((P, n), np.float32)
    p[0:3] = means
    p[3:6] = rng.uniform(log_lo, log_hi, size=(3, n))
    q = rng.standard_normal(size=(4, n))
    q /= np.linalg.norm(q, axis=0, keepdims=True)
    p[6:10] = q
    p[10] = rng.normal(logit_mu, logit_sigma, size=n)
    if sh_degree == 0:
        p[11:14] = rng.uniform(0.0, 1.0, size=(3, n))
    else:
        # DC coefficient uniform on [-sqrt(pi), sqrt(pi)]: with the higher bands at
        # zero this makes the view-independent colour U(0, 1) per channel.
        s = math.sqrt(math.pi)
        p[11:14] = rng.uniform(-s, s, size=(3, n))
        p[14:59] = rng.normal(0.0, 0.1, size=(45, n))
    return p


def _perturbed(rng, params, sigma=0.01):
    q = params.copy()
    q[0:3] += rng.normal(0.0, sigma, size=(3, params.shape[1])).astype(np.float32)
    return q


def make_scene(name: str, seed: int | None = None, n: int | None = None) -> Scene:
    """Build one of the five workloads.  ``n`` overrides the Gaussian count (tests)."""
    if seed is None:
        seed = SEEDS[name]
    rng = np.random.default_rng(seed)
    opts = dict(DEFAULT_OPTS)
    lr_scale = 1.0
    if name == "tiny":
        n = 1000 if n is None else n
        means = np.stack([rng.uniform(-1, 1, n), rng.uniform(-1, 1, n), rng.uniform(2, 4, n)])
        params = _common_params(rng, n, means, -4.0, -2.0, 0.0, 1.0, 0)
        cams = [Camera(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), 64.0, 64.0, 32.0, 32.0, 64, 64)]
        target = rng.uniform(0.0, 1.0, size=(1, 3, 64, 64)).astype(np.float32)
        return Scene(name, params, 0, cams, "uniform", target, None, DEFAULT_LR, opts)
    if name == "small":
        n = 100_000 if n is None else n
        means = np.stack([rng.uniform(-5, 5, n), rng.uniform(-5, 5, n), rng.uniform(3, 20, n)])
        params = _common_params(rng, n, means, -5.0, -2.5, 0.0, 1.0, 0)
        cams = [Camera(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), 1000.0, 1000.0, 640.0, 360.0, 1280, 720)]
        sh = 0
    elif name == "medium":
        n = 1_000_000 if n is None else n
        centres = np.stack([rng.uniform(-20, 20, 64), rng.uniform(-20, 20, 64), rng.uniform(30, 70, 64)])
        which = rng.integers(0, 64, size=n)
        means = centres[:, which] + rng.normal(0.0, 1.5, size=(3, n))
        params = _common_params(rng, n, means, -6.0, -3.0, 0.0, 1.0, 3)
        cams = [Camera(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), 1400.0, 1400.0, 960.0, 540.0, 1920, 1080)]
        sh = 3
    elif name == "large":
        n = 11_200_000 if n is None else n
        means = np.stack([rng.uniform(-100, 100, n), rng.uniform(-100, 100, n), rng.uniform(0, 50, n)])
        params = _common_params(rng, n, means, -7.0, -3.0, -1.0, 1.5, 3)
        tilt = math.radians(30.0)
        centre = (0.0, 0.0, 110.0)
        look = (0.0, 110.0 * math.tan(tilt), 0.0)   # 30 degrees off nadir toward +y
        R, t = _look_at(centre, look)
        cams = [Camera(R, t, 3000.0, 3000.0, 2048.0, 1080.0, 4096, 2160)]
        sh = 3
    elif name == "batched":
        n = 20_000_000 if n is None else n
        means = rng.uniform(-75, 75, size=(3, n))
        params = _common_params(rng, n, means, -7.0, -3.0, -1.0, 1.5, 3)
        cams = []
        for k in range(16):
            a = 2.0 * math.pi * k / 16.0
            R, t = _look_at((80.0 * math.cos(a), 80.0 * math.sin(a), 40.0), (0.0, 0.0, 0.0))
            cams.append(Camera(R, t, 1400.0, 1400.0, 960.0, 540.0, 1920, 1080))
        sh = 3
        lr_scale = math.sqrt(16.0)   # Grendel: learning rate x sqrt(batch size)
    else:
        raise KeyError(name)
    pert = _perturbed(rng, params)
    lr = tuple(float(x) * lr_scale for x in DEFAULT_LR)
    return Scene(name, params, sh, cams, "perturbed", None, pert, lr, opts)


def lr_rows(lr, sh_degree) -> np.ndarray:
    """Expand the five group learning rates to one value per parameter row."""
    P = PARAM_ROWS[sh_degree]
    out = np.empty(P, np.float32)
    out[0:3] = lr[0]
    out[3:6] = lr[1]
    out[6:10] = lr[2]
    out[10] = lr[3]
    out[11:] = lr[4]
    return out


def random_small_scene(seed, n, width, height, sh_degree, fx=None, log_lo=-2.5, log_hi=-1.0,
                       logit_mu=0.5, logit_sigma=1.0, depth=(2.0, 4.0), spread=0.8):
    """A handful of large, overlapping Gaussians for gradient checks (not one of the five workloads)."""
    rng = np.random.default_rng(seed)
    fx = float(width) if fx is None else fx
    means = np.stack([rng.uniform(-spread, spread, n) * 0.5, rng.uniform(-spread, spread, n) * 0.5 * height / width,
                      rng.uniform(depth[0], depth[1], n)])
    params = _common_params(rng, n, means, log_lo, log_hi, logit_mu, logit_sigma, sh_degree)
    if sh_degree == 3:
        params[14:59] = rng.normal(0.0, 0.3, size=(45, n))
    cam = Camera(np.eye(3, dtype=np.float32), np.zeros(3, np.float32), fx, fx, width / 2.0, height / 2.0, width, height)
    target = rng.uniform(0.0, 1.0, size=(1, 3, height, width)).astype(np.float32)
    return Scene("grad-check", params, sh_degree, [cam], "uniform", target, None, DEFAULT_LR, dict(DEFAULT_OPTS))
