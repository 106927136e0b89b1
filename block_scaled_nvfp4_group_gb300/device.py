"""Device-resident problems: the buffers of one grouped call and the two
launches of the hot path (scale relayout, grouped GEMM).

PyTorch only allocates memory and supplies the stream; both steps run in the
library's kernels through ``ops``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import ops


def _dev(a: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
    return t.reshape(-1) if t.numel() else torch.empty(0, dtype=torch.uint8, device=device)


class DeviceProblem:
    """A, B, row-major SFA/SFB, tiled SFA/SFB and C for every group.

    ``step()`` runs the whole path: one grouped relayout launch for every
    SFA and SFB, then the grouped GEMM.  ``gemm()`` runs the GEMM alone on
    the tiled scales already produced."""

    def __init__(self, groups, device="cuda"):
        self.device = torch.device(device)
        self.shapes = [(g.M, g.N, g.K) for g in groups]
        self.A, self.B, self.SFA, self.SFB = [], [], [], []
        self.SFA_t, self.SFB_t, self.C = [], [], []
        for g in groups:
            self.A.append(_dev(g.A, self.device))
            self.B.append(_dev(g.B, self.device))
            self.SFA.append(_dev(g.SFA, self.device))
            self.SFB.append(_dev(g.SFB, self.device))
            self.SFA_t.append(torch.zeros(max(ops.sf_tiled_bytes(g.M, g.K), 16), dtype=torch.uint8,
                                          device=self.device))
            self.SFB_t.append(torch.zeros(max(ops.sf_tiled_bytes(g.N, g.K), 16), dtype=torch.uint8,
                                          device=self.device))
            self.C.append(torch.empty((g.M, g.N), dtype=torch.float16, device=self.device))
        self.relayout_items = []
        for i, (M, N, K) in enumerate(self.shapes):
            if M > 0:   # an empty group is skipped by the GEMM as well
                self.relayout_items.append((self.SFA[i], self.SFA_t[i], M, K))
                self.relayout_items.append((self.SFB[i], self.SFB_t[i], N, K))
        self.relayout_descs = ops.make_relayout_descs(self.relayout_items)
        self.descs = ops.make_group_descs(
            (self.A[i], self.B[i], self.SFA_t[i], self.SFB_t[i], self.C[i], M, N, K)
            for i, (M, N, K) in enumerate(self.shapes))

    def relayout(self, stream=None) -> None:
        ops.sf_relayout_group(None, stream=stream, descs=self.relayout_descs)

    def gemm(self, stream=None) -> None:
        ops.group_gemm(None, stream=stream, descs=self.descs)

    def step(self, stream=None) -> None:
        self.relayout(stream)
        self.gemm(stream)

    def outputs_fp16_bits(self):
        return [c.view(torch.int16).cpu().numpy().view(np.uint16) for c in self.C]

    @property
    def resident_bytes(self) -> int:
        ts = self.A + self.B + self.SFA + self.SFB + self.SFA_t + self.SFB_t + self.C
        return sum(t.numel() * t.element_size() for t in ts)
