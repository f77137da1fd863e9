"""Host-side spike protocol around the optimizer step.

"OPEN-1B: A Fully Auditable Training Run", §3.4.2: training clipped at a global norm of 1.0
and skipped five optimizer steps whenever the pre-clip gradient norm exceeded 5.  The pages
do not say whether the spiking step is one of the five or whether a spike inside the window
extends it.  Reading taken here: a step whose pre-clip norm exceeds the threshold (or is not
finite) skips its own update and the next span - 1, and every such step restarts the window.

A skipped step changes nothing in (w, m, v); it still produces a state hash, with the
training step in the image header.  AdamW's bias corrections count applied updates only.
The decision needs the norm on the host, so a step under this protocol synchronises once,
after the clip kernel.
"""
from __future__ import annotations

import math

from . import repstep as rs


class SpikeSkip:
    """Decides, from each step's pre-clip norm, whether to apply the update."""

    def __init__(self, threshold: float = 5.0, span: int = 5):
        if span < 1:
            raise ValueError("span must be >= 1")
        self.threshold = float(threshold)
        self.span = int(span)
        self.remaining = 0

    def apply(self, norm: float) -> bool:
        """True if this step's update is applied."""
        if not math.isfinite(norm) or norm > self.threshold:
            self.remaining = self.span - 1
            return False
        if self.remaining > 0:
            self.remaining -= 1
            return False
        return True

    def state(self) -> dict:
        return {"threshold": self.threshold, "span": self.span, "remaining": self.remaining}


class Stepper:
    """Training-loop driver: one call per training step, with the spike protocol.

    train_step numbers the steps (the image header's step); adam_step counts the updates
    actually applied (AdamW's t)."""

    def __init__(self, ctx: rs.Repstep, hparams: dict, policy: SpikeSkip | None = None,
                 adam_step: int = 0):
        self.ctx = ctx
        self.hp = dict(hparams)
        self.policy = policy or SpikeSkip()
        self.adam_step = adam_step
        import torch
        self._norm = torch.empty(1, dtype=torch.float32, device=ctx.device)

    def step(self, grads, w, m, v, train_step: int, root_out=None) -> dict:
        ctx = self.ctx
        ctx.reduce(grads)
        ctx.clip(self.hp["clip"], norm_out=self._norm)
        norm = float(self._norm.item())
        applied = self.policy.apply(norm)
        if applied:
            self.adam_step += 1
            hp = rs.hparams(lr=self.hp["lr"], beta1=self.hp["beta1"], beta2=self.hp["beta2"],
                            eps=self.hp["eps"], weight_decay=self.hp["wd"], clip=self.hp["clip"],
                            t=self.adam_step)
            ctx.adamw(w, m, v, hp)
            ctx.root(train_step, root_out=root_out)
        else:
            ctx.hash(train_step, w, m, v, root_out=root_out)
        return {"norm": norm, "applied": applied, "adam_step": self.adam_step}
