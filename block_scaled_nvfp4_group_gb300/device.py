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
    SFA and SFB, then the grouped GEMM (nvfp4_relayout_and_gemm).  ``gemm()`` runs the GEMM alone on
    the tiled scales already produced."""

    def __init__(self, groups, device="cuda"):
        self.device = torch.device(device)
        self.shapes = [(g.M, g.N, g.K) for g in groups]
        self.A, self.B, self.SFA, self.SFB = [], [], [], []
        self.SFA_t, self.SFB_t, self.C = [], [], []
        # every input in one device buffer and every output in another (views
        # at 256-byte offsets), so a batch moves host <-> device in one copy
        # each way
        in_sizes = []
        for g in groups:
            in_sizes += [g.A.size, g.B.size, g.SFA.size, g.SFB.size]
        offs, total = [], 0
        for n in in_sizes:
            offs.append(total)
            total += (n + 255) // 256 * 256
        self.inputs = torch.zeros(max(total, 256), dtype=torch.uint8, device=self.device)
        host = np.zeros(max(total, 256), dtype=np.uint8)
        out_offs, out_total = [], 0
        for (M, N, K) in self.shapes:
            out_offs.append(out_total)
            out_total += (M * N * 2 + 255) // 256 * 256
        self.outputs = torch.empty(max(out_total, 256), dtype=torch.uint8, device=self.device)
        for i, g in enumerate(groups):
            views = []
            for j, arr in enumerate((g.A, g.B, g.SFA, g.SFB)):
                o = offs[4 * i + j]
                host[o:o + arr.size] = np.ascontiguousarray(arr).reshape(-1)
                views.append(self.inputs[o:o + arr.size])
            self.A.append(views[0])
            self.B.append(views[1])
            self.SFA.append(views[2])
            self.SFB.append(views[3])
            self.SFA_t.append(torch.zeros(max(ops.sf_tiled_bytes(g.M, g.K), 16), dtype=torch.uint8,
                                          device=self.device))
            self.SFB_t.append(torch.zeros(max(ops.sf_tiled_bytes(g.N, g.K), 16), dtype=torch.uint8,
                                          device=self.device))
            o = out_offs[i]
            self.C.append(self.outputs[o:o + g.M * g.N * 2].view(torch.float16).view(g.M, g.N))
        self.inputs.copy_(torch.from_numpy(host))
        self.relayout_items = []
        for i, (M, N, K) in enumerate(self.shapes):
            if M > 0:   # an empty group is skipped by the GEMM as well
                self.relayout_items.append((self.SFA[i], self.SFA_t[i], M, K))
                self.relayout_items.append((self.SFB[i], self.SFB_t[i], N, K))
        self.relayout_descs = ops.make_relayout_descs(self.relayout_items)
        self.descs = ops.make_group_descs(
            (self.A[i], self.B[i], self.SFA_t[i], self.SFB_t[i], self.C[i], M, N, K)
            for i, (M, N, K) in enumerate(self.shapes))
        self.step_descs = ops.make_step_descs(
            (self.A[i], self.B[i], self.SFA[i], self.SFB[i], self.SFA_t[i], self.SFB_t[i], self.C[i],
             M, N, K)
            for i, (M, N, K) in enumerate(self.shapes))

    def relayout(self, stream=None) -> None:
        ops.sf_relayout_group(None, stream=stream, descs=self.relayout_descs)

    def gemm(self, stream=None) -> None:
        ops.group_gemm(None, stream=stream, descs=self.descs)

    def step(self, stream=None) -> None:
        """The whole path in one library call (relayout, then the GEMM, whose
        A and B loads need not wait for the relayout to finish)."""
        ops.relayout_and_gemm(stream=stream, descs=self.step_descs)

    def outputs_fp16_bits(self):
        return [c.view(torch.int16).cpu().numpy().view(np.uint16) for c in self.C]

    @property
    def resident_bytes(self) -> int:
        ts = self.A + self.B + self.SFA + self.SFB + self.SFA_t + self.SFB_t + self.C
        return sum(t.numel() * t.element_size() for t in ts)
