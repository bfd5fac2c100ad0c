"""One training step of the tile-based 3DGS rasterizer on one GPU.

``GaussianTrainer`` owns the device buffers (torch tensors used as plain device
memory) and calls the five C-ABI entry points in order on one stream:

    gs_project -> gs_bin_sort -> gs_raster_fused_fwd_bwd -> gs_grad_compact -> gs_adam_deferred

With ``dssim_lambda`` set, the loss is (1 - lambda) L1 + lambda (1 - SSIM) and the
fused call is replaced by three: gs_raster_forward_state -> gs_dssim_loss_grad ->
gs_raster_backward_state (the SSIM window reaches into neighbouring tiles).

Buffer layout in HBM (fp32 unless stated):
    params, grads, adam_m, adam_v   [n, stride]      stride = 16 (RGB, P = 14) or 64 (SH 3, P = 59);
                                                     one aligned block per Gaussian (grads: valid for
                                                     the Gaussians of the current step's union only)
    last_step                       [n] int32
    rec                             [V, n, 12]       3 float4 per (view, Gaussian)
    depth, tiles_touched, rect      [V, n], [V, n], [V, n, 4] uint16
    keys, ids                       [capacity] u64, u32 (sorted instances)
    ranges                          [V * tiles, 2] u32
    image                           [V, 3, H, W];  loss [V] fp64
    grad2d                          [V, n, 12]  (kept all-zero between steps)
    touched                         [V, n] u8   (kept all-zero between steps)
    idx, n_idx                      [V + 1, n] u32, [V + 1] int64 (per-view lists + union)
    t_final, last_idx, dldc         [V, H, W], [V, H, W] int32, [V, 3, H, W]  (D-SSIM loss only)
    bits_ws                         [(capacity + 32 V tiles) * 8] u32: saved pass bits (the raster's scratch)
The sizes follow the workload: nothing is allocated per step once the instance
capacity has been reached (it grows by 25 % headroom when a step needs more).
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import abi


class GaussianTrainer:
    def __init__(self, params: np.ndarray | torch.Tensor, sh_degree: int, cameras, opts: dict, lr,
                 betas=(0.9, 0.999), eps=1e-8, device="cuda", capacity: int | None = None,
                 dssim_lambda: float | None = None, tile_budget: int | None = None):
        self.device = torch.device(device)
        if tile_budget is None:
            tile_budget = opts.get("tile_budget", 0)
        self.tile_budget = int(tile_budget) if tile_budget else None
        self.dssim_lambda = None if dssim_lambda is None else float(dssim_lambda)
        self.sh_degree = sh_degree
        self.P = abi.gs_param_rows(sh_degree)
        self.stride = abi.gs_param_stride(sh_degree)
        p = torch.as_tensor(params, dtype=torch.float32)
        assert p.shape[0] == self.P, (p.shape, self.P)
        self.n = int(p.shape[1])
        self.V = len(cameras)
        self.W, self.H = cameras[0].width, cameras[0].height
        self.tiles = abi.gs_num_tiles(self.W, self.H)
        self.cams = abi.cameras(cameras)
        self.opts = abi.render_opts(opts)
        self._opts_dict = dict(opts)
        self.lr = tuple(float(x) for x in lr)
        self.betas = betas
        self.eps = eps
        self.t = 0
        dev = self.device
        n, V = self.n, self.V
        self.params = self.to_device_layout(p)
        self.grads = torch.zeros_like(self.params)
        self.adam_m = torch.zeros_like(self.params)
        self.adam_v = torch.zeros_like(self.params)
        self.last_step = torch.zeros(n, dtype=torch.int32, device=dev)
        self.rec = torch.empty((V, n, 12), dtype=torch.float32, device=dev)
        self.depth = torch.empty((V, n), dtype=torch.float32, device=dev)
        self.rect = torch.empty((V, n, 4), dtype=torch.int16, device=dev)
        self.tiles_touched = torch.empty((V, n), dtype=torch.int32, device=dev)
        self.ranges = torch.empty((V * self.tiles, 2), dtype=torch.int32, device=dev)
        self.image = torch.empty((V, 3, self.H, self.W), dtype=torch.float32, device=dev)
        self.loss = torch.zeros(V, dtype=torch.float64, device=dev)
        self.grad2d = torch.zeros((V, n, abi.GS_GRAD2D_STRIDE), dtype=torch.float32, device=dev)
        self.touched = torch.zeros((V, n), dtype=torch.uint8, device=dev)
        self.idx = torch.empty((V + 1, n), dtype=torch.int32, device=dev)
        self.n_idx = torch.zeros(V + 1, dtype=torch.int64, device=dev)
        self.eval_counts = torch.zeros(3, dtype=torch.int64, device=dev)
        self.compact_ws = torch.empty(abi.gs_grad_compact_ws_bytes(n), dtype=torch.uint8, device=dev)
        if self.dssim_lambda is not None:
            self.t_final = torch.empty((V, self.H, self.W), dtype=torch.float32, device=dev)
            self.last_idx = torch.empty((V, self.H, self.W), dtype=torch.int32, device=dev)
            self.dldc = torch.empty((V, 3, self.H, self.W), dtype=torch.float32, device=dev)
        self.proj = abi.proj_struct(self.rec.data_ptr(), self.depth.data_ptr(), self.rect.data_ptr(),
                                    self.tiles_touched.data_ptr())
        self.capacity = 0
        self.n_instances = 0
        self._alloc_instances(capacity if capacity is not None else max(1024, 4 * n * V // 8))

    # ------------------------------------------------------------------ layout
    def to_device_layout(self, rows) -> torch.Tensor:
        """[P, n] parameter rows (numpy or torch) -> device [n, stride] blocks (padding zero)."""
        r = torch.as_tensor(rows, dtype=torch.float32)
        out = torch.zeros((r.shape[1], self.stride), dtype=torch.float32, device=self.device)
        out[:, :self.P] = r.to(self.device).t()
        return out

    def rows(self, blocks: torch.Tensor) -> torch.Tensor:
        """Device [n, stride] blocks -> [P, n] rows (a copy), the generator's layout."""
        return blocks[:, :self.P].t().contiguous()

    # ------------------------------------------------------------------ buffers
    def _alloc_instances(self, capacity: int):
        capacity = int(min(capacity, 2 ** 32 - 1))
        self.capacity = capacity
        self.keys = torch.empty(capacity, dtype=torch.int64, device=self.device)
        self.ids = torch.empty(capacity, dtype=torch.int32, device=self.device)
        # the fused raster's saved-pass-bits scratch (32 B per instance)
        self.bits_ws = torch.empty(abi.raster_bits_ws_words(capacity, self.V * self.tiles), dtype=torch.int32,
                                   device=self.device)
        nbytes = abi.gs_bin_sort_ws_bytes(self.n, self.V, self.W, self.H, capacity)
        self.sort_ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)

    def kernel_launches_per_step(self) -> int:
        """Kernels the library launches for one train_step, from its launch structure:
        projection 1; binning: count 1, scan 3, bucket stats 1, scatter 1, warp sort 1,
        sort of 257..2048 1 (these three queued before the count is known), and one
        more sort kernel for each of the size classes 2049..16384 and over 16384 that
        occurs; pruning (with a
        tile budget) 1; fused raster 1
        (with the D-SSIM loss: forward, D-SSIM and backward, 3); compaction: 3 per
        view-list scan, then (several views) union 1 and union scan 3, VJP 1; Adam 2.
        Memsets and copies are not kernels.  Reads the last step's ranges."""
        V, n = self.V, self.n
        r = self.ranges.view(-1, 2).to(torch.int64)
        c = r[:, 1] - r[:, 0]
        sort = (1 if n * V else 0) + 3 + 1 + (3 if n else 0)
        if self.n_instances:
            sort += sum(int(((c > lo) & (c <= hi)).any().item()) for lo, hi in ((2048, 16384), (16384, 1 << 62)))
        compact = (3 * V + (1 + 3 if V > 1 else 0) + 1) if n else 0
        raster = 1 if self.dssim_lambda is None else 3
        prune = 1 if self.tile_budget else 0
        return (1 if n else 0) + sort + prune + raster + compact + (2 if n else 0)

    def stream_handle(self):
        return torch.cuda.current_stream(self.device).cuda_stream

    # ------------------------------------------------------------------ stages
    def project(self, params=None):
        params = self.params if params is None else params
        abi.gs_project(params.data_ptr(), self.n, self.sh_degree, self.cams, self.V, self.opts, self.proj,
                       self.stream_handle())

    def bin_sort(self):
        while True:
            st, cnt = abi.gs_bin_sort(self.proj, self.n, self.V, self.W, self.H, self.capacity, self.keys.data_ptr(),
                                      self.ids.data_ptr(), self.ranges.data_ptr(), self.sort_ws.data_ptr(),
                                      self.sort_ws.numel(), self.stream_handle())
            self.n_instances = cnt
            if st == abi.GS_OK:
                if self.tile_budget:
                    abi.gs_prune_tiles(self.proj, self.n, self.V, self.W, self.H, self.tile_budget,
                                       self.ids.data_ptr(), self.ranges.data_ptr(), self.stream_handle())
                return cnt
            self._alloc_instances(int(math.ceil(cnt * 1.25)) + 1024)

    def raster(self, target=None, count_evals=True):
        if target is not None and self.dssim_lambda is not None:
            return self.raster_dssim(target, count_evals)
        abi.gs_raster_fused_fwd_bwd(self.proj, self.n, self.ranges.data_ptr(), self.ids.data_ptr(), self.cams, self.V,
                                    self.opts, target.data_ptr() if target is not None else None,
                                    self.image.data_ptr(), self.loss.data_ptr(), self.grad2d.data_ptr(),
                                    self.touched.data_ptr(), self.eval_counts.data_ptr() if count_evals else None,
                                    self.stream_handle(), self.bits_ws.data_ptr(), self.bits_ws.numel())

    def work_counts(self, target) -> dict:
        """One fused raster launch in its counting variant (gs_raster_work_counts) on
        the current projection and lists: the same outputs as raster(target), plus
        what the kernel executed (candidates tested, exponentials, composites,
        backward entries and warp steps, chunks staged).  grad2d and touched are left
        filled as after raster(); compact() consumes them."""
        work = torch.zeros(abi.GS_RASTER_WORK_COUNTERS, dtype=torch.int64, device=self.device)
        abi.gs_raster_work_counts(self.proj, self.n, self.ranges.data_ptr(), self.ids.data_ptr(), self.cams, self.V,
                                  self.opts, target.data_ptr(), self.image.data_ptr(), self.loss.data_ptr(),
                                  self.grad2d.data_ptr(), self.touched.data_ptr(), work.data_ptr(),
                                  self.stream_handle(), self.bits_ws.data_ptr(), self.bits_ws.numel())
        return dict(zip(abi.RASTER_WORK_NAMES, (int(x) for x in work.cpu().tolist())))

    def raster_dssim(self, target, count_evals=True, events=None):
        """L1 + D-SSIM: forward with stored per-pixel state, loss and dL/dC, backward.
        events: None or two CUDA events recorded after the forward and after the loss."""
        sh = self.stream_handle()
        abi.gs_raster_forward_state(self.proj, self.n, self.ranges.data_ptr(), self.ids.data_ptr(), self.cams, self.V,
                                    self.opts, self.image.data_ptr(), self.t_final.data_ptr(),
                                    self.last_idx.data_ptr(), self.bits_ws.data_ptr(), self.bits_ws.numel(),
                                    self.eval_counts.data_ptr() if count_evals else None, sh)
        if events is not None:
            events[0].record(torch.cuda.current_stream(self.device))
        abi.gs_dssim_loss_grad(self.image.data_ptr(), target.data_ptr(), self.V, self.W, self.H, self.dssim_lambda,
                               self.loss.data_ptr(), self.dldc.data_ptr(), sh)
        if events is not None:
            events[1].record(torch.cuda.current_stream(self.device))
        abi.gs_raster_backward_state(self.proj, self.n, self.ranges.data_ptr(), self.ids.data_ptr(), self.cams,
                                     self.V, self.opts, self.t_final.data_ptr(), self.last_idx.data_ptr(),
                                     self.bits_ws.data_ptr(), self.bits_ws.numel(), self.dldc.data_ptr(),
                                     self.grad2d.data_ptr(), self.touched.data_ptr(), sh)

    def compact(self):
        abi.gs_grad_compact(self.grad2d.data_ptr(), self.touched.data_ptr(), self.params.data_ptr(), self.n,
                            self.sh_degree, self.cams, self.V, self.opts, self.idx.data_ptr(), self.n_idx.data_ptr(),
                            self.grads.data_ptr(), self.compact_ws.data_ptr(), self.compact_ws.numel(),
                            self.stream_handle())

    def adam(self, t, flush=False):
        union = self.idx[self.V]
        abi.gs_adam_deferred(self.params.data_ptr(), self.grads.data_ptr(), self.adam_m.data_ptr(),
                             self.adam_v.data_ptr(), self.last_step.data_ptr(), self.n, self.sh_degree,
                             union.data_ptr(), self.n_idx[self.V:].data_ptr(), t, self.lr, self.betas[0],
                             self.betas[1], self.eps, flush, self.stream_handle())

    # ------------------------------------------------------------------ steps
    def train_step(self, target: torch.Tensor, count_evals=True):
        """One full step (device-resident target [V, 3, H, W]); returns the loss tensor (device)."""
        self.t += 1
        self.project()
        self.bin_sort()
        self.raster(target, count_evals)
        self.compact()
        self.adam(self.t)
        return self.loss

    def train_step_host(self, target_host: torch.Tensor, target_dev: torch.Tensor, loss_host: torch.Tensor):
        """End-to-end step from pinned host memory: copy the target in, step, copy the loss out."""
        target_dev.copy_(target_host, non_blocking=True)
        self.train_step(target_dev)
        loss_host.copy_(self.loss, non_blocking=True)
        return loss_host

    def train_steps_host(self, targets_host, loss_host: torch.Tensor) -> torch.Tensor:
        """End-to-end steps from pinned host memory, pipelined: while step k runs, the
        target of step k + 1 is copied in on a second stream (two device buffers), and
        each step's loss is copied out right after it.

        targets_host: sequence of pinned [V, 3, H, W] fp32 tensors, one per step (the
        same tensor may repeat).  loss_host: pinned [steps, V] fp64; row k receives
        step k's loss.  Returns loss_host (valid once the current stream is synced)."""
        steps = len(targets_host)
        if steps == 0:
            return loss_host
        main = torch.cuda.current_stream(self.device)
        if getattr(self, "_copy_stream", None) is None:
            self._copy_stream = torch.cuda.Stream(self.device)
        shape = tuple(targets_host[0].shape)
        bufs = getattr(self, "_target_bufs", None)
        if bufs is None or tuple(bufs[0].shape) != shape:
            bufs = self._target_bufs = [torch.empty(shape, dtype=torch.float32, device=self.device) for _ in range(2)]
        copy = self._copy_stream
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]
        copy.wait_stream(main)   # copies start after everything already queued on the main stream
        with torch.cuda.stream(copy):
            bufs[0].copy_(targets_host[0], non_blocking=True)
            copied[0].record(copy)
        for k in range(steps):
            b = k % 2
            main.wait_event(copied[b])
            if k + 1 < steps:
                nb = (k + 1) % 2
                with torch.cuda.stream(copy):
                    if k >= 1:
                        copy.wait_event(consumed[nb])   # step k - 1 has finished reading that buffer
                    bufs[nb].copy_(targets_host[k + 1], non_blocking=True)
                    copied[nb].record(copy)
            self.train_step(bufs[b])
            consumed[b].record(main)
            loss_host[k].copy_(self.loss, non_blocking=True)
        return loss_host

    def render(self, params=None) -> torch.Tensor:
        """Forward only (no loss, gradients or touched flags); returns the image tensor."""
        self.project(params)
        self.bin_sort()
        self.raster(None, count_evals=False)
        return self.image

    def render_partial(self, depth_splits, params=None):
        """Forward only, as S = len(depth_splits[0]) + 1 depth slabs rendered on their own
        (zero background) and composed front to back; returns the composed image.
        depth_splits: [V][S-1] ascending positive depths.  The slabs' (C, T) stay in
        self.c_parts [S, V, 3, H, W] and self.t_parts [S, V, H, W]."""
        S = len(depth_splits[0]) + 1
        V, H, W = self.V, self.H, self.W
        dev = self.device
        if getattr(self, "c_parts", None) is None or self.c_parts.shape[0] != S:
            self.c_parts = torch.empty((S, V, 3, H, W), dtype=torch.float32, device=dev)
            self.t_parts = torch.empty((S, V, H, W), dtype=torch.float32, device=dev)
            self.l_parts = torch.empty((S, V, H, W), dtype=torch.int32, device=dev)
            self.sub_ranges = torch.empty((S, V * self.tiles, 2), dtype=torch.int32, device=dev)
            self.t_composed = torch.empty((V, H, W), dtype=torch.float32, device=dev)
        budget, self.tile_budget = self.tile_budget, None   # slabs split the unpruned lists
        try:
            self.project(params)
            self.bin_sort()
        finally:
            self.tile_budget = budget
        sh = self.stream_handle()
        abi.gs_split_ranges(self.keys.data_ptr(), self.ranges.data_ptr(), V, W, H, S, depth_splits,
                            self.sub_ranges.data_ptr(), sh)
        zero_bg = abi.render_opts(dict(self._opts_dict, bg=(0.0, 0.0, 0.0)))
        for s in range(S):
            abi.gs_raster_forward_state(self.proj, self.n, self.sub_ranges[s].data_ptr(), self.ids.data_ptr(),
                                        self.cams, V, zero_bg, self.c_parts[s].data_ptr(),
                                        self.t_parts[s].data_ptr(), self.l_parts[s].data_ptr(), None, 0, None, sh)
        abi.gs_compose(self.c_parts.data_ptr(), self.t_parts.data_ptr(), S, V, W, H, self._opts_dict["bg"],
                       self.image.data_ptr(), self.t_composed.data_ptr(), sh)
        return self.image

    def flush(self):
        """Bring every Gaussian's optimizer state to the current step (before reading params)."""
        if self.t > 0:
            self.adam(self.t, flush=True)

    def state_dict(self):
        self.flush()
        return dict(params=self.params.clone(), m=self.adam_m.clone(), v=self.adam_v.clone(),
                    last_step=self.last_step.clone(), t=self.t)

    def load_state_dict(self, sd):
        self.params.copy_(sd["params"])
        self.adam_m.copy_(sd["m"])
        self.adam_v.copy_(sd["v"])
        self.last_step.copy_(sd["last_step"])
        self.t = int(sd["t"])
