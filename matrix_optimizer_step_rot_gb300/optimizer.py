"""PyTorch-side plumbing around the C ABI: device buffers for the state and
workspace blobs, stream handles, and exports.  No optimizer arithmetic here."""

from __future__ import annotations

from typing import Sequence, Tuple

import torch

from . import binding as B


class RotatedAdam:
    """Rotated-Adam step over a fixed list of float32 matrices.

    shapes: (m, n) per matrix; c_max: micro-group byte cap; state_format:
    ROT_STATE_FULL or ROT_STATE_COMPACT (bf16 moments, fp16 bases).  The state blob
    (M, v, U, V per matrix) and the workspace blob are torch uint8 tensors on
    `device`; the library writes them through raw pointers.
    """

    def __init__(self, shapes: Sequence[Tuple[int, int]], c_max: int, device="cuda",
                 beta1=0.9, beta2=0.999, eps=1e-8, lr=1e-3, rank_rtol=1e-3,
                 precision=B.ROT_PREC_3XTF32, state_format=B.ROT_STATE_FULL):
        self.plan = B.Plan(shapes, c_max, state_format=state_format)
        self.device = torch.device(device)
        sb, wb = self.plan.state_bytes()
        self.state = torch.empty(sb, dtype=torch.uint8, device=self.device)
        self.work = torch.empty(wb, dtype=torch.uint8, device=self.device)
        self.hyper = (float(beta1), float(beta2), float(eps), float(lr))
        self.rank_rtol = float(rank_rtol)
        self.precision = int(precision)
        B.rot_state_init(self.plan, self.state.data_ptr(), self._stream())

    def _stream(self, stream=None) -> int:
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        return int(s.cuda_stream)

    def step(self, W: Sequence[torch.Tensor], G: Sequence[torch.Tensor], refresh: bool,
             stream=None, precision=None) -> None:
        for w, g, (m, n) in zip(W, G, self.plan.shapes):
            assert w.dtype == torch.float32 and g.dtype == torch.float32
            assert w.is_contiguous() and g.is_contiguous() and tuple(w.shape) == (m, n)
        b1, b2, eps, lr = self.hyper
        B.rot_step(self.plan, [w.data_ptr() for w in W], [g.data_ptr() for g in G],
                   self.state.data_ptr(), self.work.data_ptr(), b1, b2, eps, lr, refresh,
                   self.precision if precision is None else int(precision), self.rank_rtol,
                   self._stream(stream))

    def export(self, item: int, which: int) -> torch.Tensor:
        m, n = self.plan.shapes[item]
        shape = {B.ROT_WHICH_M: (m, n), B.ROT_WHICH_V2: (m, n), B.ROT_WHICH_U: (m, m),
                 B.ROT_WHICH_V: (n, n)}[which]
        out = torch.empty(shape, dtype=torch.float32, device=self.device)
        B.rot_state_export(self.plan, self.state.data_ptr(), item, which, out.data_ptr(),
                           self._stream())
        return out

    def ranks(self, item: int) -> Tuple[int, int]:
        return B.rot_state_ranks(self.plan, self.state.data_ptr(), item, self._stream())

    def status(self) -> int:
        return B.rot_status(self.plan, self.state.data_ptr(), self._stream())
