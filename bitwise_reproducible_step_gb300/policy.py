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

import json
import math
import os
import struct
import time

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


class StepLog:
    """Append-only JSON-lines record of a run, one line per training step.

    ("grow_a_language_model_checkpoints", "Cumulative training record": a sidecar file keeps
    one entry per step for the whole run and is never reset.)  Each line is written and
    flushed whole, so a crash leaves at most a missing last line, never a torn one in the
    middle; reopening the same path appends.  The norm is recorded with its fp32 bits and
    the state root in hex, so two runs can be compared bit for bit from their logs."""

    def __init__(self, path: str):
        self.path = str(path)

    def write(self, record: dict) -> None:
        line = json.dumps(record, sort_keys=True, allow_nan=True)
        if "\n" in line:
            raise ValueError("a record must serialise to one line")
        with open(self.path, "a", encoding="utf-8") as f:
            f.write(line + "\n")
            f.flush()
            os.fsync(f.fileno())

    def records(self) -> list[dict]:
        if not os.path.exists(self.path):
            return []
        with open(self.path, encoding="utf-8") as f:
            return [json.loads(ln) for ln in f if ln.strip()]


def f32_bits(x: float) -> str:
    """The fp32 bit pattern of x, as 8 hex digits."""
    return struct.pack("<f", x)[::-1].hex()


def root_hex(root: int) -> str:
    """A state root (the int64 bits of a u64) as 16 hex digits."""
    return f"{int(root) & (2**64 - 1):016x}"


class Stepper:
    """Training-loop driver: one call per training step, with the spike protocol.

    train_step numbers the steps (the image header's step); adam_step counts the updates
    actually applied (AdamW's t)."""

    def __init__(self, ctx: rs.Repstep, hparams: dict, policy: SpikeSkip | None = None,
                 adam_step: int = 0, log: StepLog | None = None):
        self.ctx = ctx
        self.hp = dict(hparams)
        self.policy = policy or SpikeSkip()
        self.adam_step = adam_step
        self.log = log
        import torch
        self._norm = torch.empty(1, dtype=torch.float32, device=ctx.device)
        self._root = torch.empty(1, dtype=torch.int64, device=ctx.device)

    def step(self, grads, w, m, v, train_step: int, root_out=None) -> dict:
        """One training step.  With a log, the step also waits for its root and appends
        {train_step, adam_step, applied, norm, norm_bits, root, ms, policy} to it."""
        ctx = self.ctx
        t0 = time.perf_counter()
        if self.log is not None and root_out is None:
            root_out = self._root
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
        out = {"norm": norm, "applied": applied, "adam_step": self.adam_step}
        if self.log is not None:
            ctx.sync()
            out["root"] = root_hex(int(root_out.reshape(-1)[0].item()))
            self.log.write({"train_step": int(train_step), "adam_step": self.adam_step,
                            "applied": applied, "norm": norm, "norm_bits": f32_bits(norm),
                            "root": out["root"], "ms": (time.perf_counter() - t0) * 1e3,
                            "policy": self.policy.state()})
        return out
