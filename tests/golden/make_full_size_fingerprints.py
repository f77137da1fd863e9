"""Write full_size_fingerprints.txt: the oracle's pre-clip norm bits and Merkle root of every
full-size step the GPU tests compare (tests/test_gpu_big.py), from the oracle alone.

The inputs are the seeded ones of bitwise_reproducible_step_gb300/inputs.py, generated with
torch's Philox generator on a CUDA device (so this script needs one); every number written
comes from the oracle's functions, run chunk-parallel on the host by tests/oracle_full.py.
Nothing of the CUDA step path is called.

    python tests/golden/make_full_size_fingerprints.py OUT.txt
"""
import os
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from bitwise_reproducible_step_gb300 import inputs as I  # noqa: E402
from tests import oracle_full as OF  # noqa: E402

HP = I.default_hparams()


def host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bench_segments(n):
    segs, e = [(0, False)], n // 20 | 1
    while e < n:
        segs.append((e, True))
        e += 16_777_216 + 3
        if e < n:
            segs.append((e, False))
            e += 4096
    return segs


def trajectory(wl, steps, variant, out, *, hash_mode=0, topologies=None):
    dev = torch.device("cuda", 0)
    w, m, v = I.gen_state(wl, device=dev)
    fo = OF.FullOracle(wl.n, wl.R, host(w), host(m), host(v), grad_dtype=wl.grad_dtype,
                       hash_mode=hash_mode)
    del w, m, v
    gdt = torch.bfloat16 if wl.grad_dtype == "bf16" else torch.float32
    grads = [torch.empty(wl.n, dtype=gdt, device=dev) for _ in range(wl.R)]
    for t in range(1, steps + 1):
        for r in range(wl.R):
            I.gen_grad(wl, t, r, device=dev, out=grads[r])
        kw = {}
        if topologies:
            nodes, gpn = topologies[t - 1]
            kw = dict(reducer="topology", nodes=nodes, gpus_per_node=gpn)
        rep = fo.step(grads, t, HP, None, **kw)
        out.append((wl.name, variant, t, rep["norm"]["oracle"], rep["root"]["oracle"]))
        print(out[-1], flush=True)
    fo.close()


def mid_run(wl, t, variant, out, *, reducer="tree", dp_shard=1, bf16w_ftz_segments=False):
    dev = torch.device("cuda", 0)
    n, R = wl.n, wl.R
    w, m, v = I.gen_state(wl, device=dev)
    kw = {}
    if variant == "mid_run_sweep_reference" or bf16w_ftz_segments:
        m.copy_(I.gen_grad(wl, 9, 0, device=dev))
        v.copy_(I.gen_grad(wl, 9, 1, device=dev).square())
    if bf16w_ftz_segments:
        w = w.to(torch.bfloat16)
        kw = dict(param_dtype="bf16", ftz=True, segments=bench_segments(n))
    fo = OF.FullOracle(n, R, host(w), host(m), host(v), **kw)
    del w, m, v
    grads = [I.gen_grad(wl, 1 if variant != "bf16w_decay_ftz_mid_run" else 3, r, device=dev)
             for r in range(R)]
    rep = fo.step(grads, t, HP, None, reducer=reducer, dp_shard=dp_shard)
    out.append((wl.name, variant, t, rep["norm"]["oracle"], rep["root"]["oracle"]))
    print(out[-1], flush=True)
    fo.close()


def main(path):
    t0 = time.time()
    W = I.WORKLOADS
    out = []
    c3, c4, c5 = W["flat1200m_r8_segscale"], W["flat268m_r32_topologies"], \
        W["flat3000m_r8_bf16_spiked_shards"]
    trajectory(c3, c3.steps, "default", out)
    trajectory(c3, 2, "audit", out, hash_mode=1)
    trajectory(c5, c5.steps, "default", out)
    trajectory(c4, c4.steps, "topologies", out, topologies=c4.topologies)
    mid_run(c4, 3, "mid_run_sweep_reference", out)
    mid_run(c4, 1, "paper_exact_4x8", out, reducer="alg1", dp_shard=8)
    mid_run(c3, 3, "bf16w_decay_ftz_mid_run", out, bf16w_ftz_segments=True)
    with open(path, "w") as f:
        f.write("# Pre-clip norm (fp32 bits) and Merkle root of each full-size step that\n"
                "# tests/test_gpu_big.py compares, from the oracle alone: written by\n"
                "# tests/golden/make_full_size_fingerprints.py (the oracle's functions run\n"
                "# chunk-parallel by tests/oracle_full.py) on the seeded inputs of\n"
                "# bitwise_reproducible_step_gb300/inputs.py, drawn with torch's Philox\n"
                f"# generator on a CUDA device (torch {torch.__version__}).\n"
                "# workload | variant | step | norm bits | root\n")
        for row in out:
            f.write(" | ".join(str(x) for x in row) + "\n")
    print(f"wrote {len(out)} fingerprints in {time.time() - t0:.0f} s")


if __name__ == "__main__":
    main(sys.argv[1])
