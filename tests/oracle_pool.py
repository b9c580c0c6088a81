"""The fp64 oracle fanned out over the host cores, for parity tests over whole batches.

The batch drivers of the oracle (verify_stochastic, verify_greedy, nkl_rows) run on
interleaved shares of the sequences in one process per core. Workers are started with
`spawn` (the calling process already holds a CUDA context, and a process forked from it
can hang), and read the logits from .npy files in a temporary directory (in /dev/shm
where it exists) through read-only memory maps, so every worker sees exactly the bytes
the GPU was given and nothing large crosses a pipe. Results come back as the drivers'
per-sequence dicts, merged into one.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import shutil
import sys
import tempfile

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(task):
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from oracle import oracle as O
    kind, files, small, kwargs, seqs = task
    arrays = {k: np.load(f, mmap_mode="r") for k, f in files.items()}
    a = {**arrays, **small}
    if kind == "stochastic":
        return O.verify_stochastic(a["target"], a["draft"], a["tokens"], a["cu_draft"], kwargs.pop("T"),
                                   a["u_accept"], a["u_sample"], kwargs.pop("dtype"), seqs=seqs, **kwargs)
    if kind == "greedy":
        return O.verify_greedy(a["target"], a["tokens"], a["cu_draft"], kwargs.pop("dtype"), seqs=seqs, **kwargs)
    if kind == "nkl":
        return O.nkl_rows(a["target"], a["draft"], a["cu_draft"], kwargs.pop("T"), kwargs.pop("dtype"), seqs=seqs,
                          **kwargs)
    raise ValueError(kind)


def oracle_batch(kind: str, w, seqs=None, nproc: int | None = None, **kwargs) -> dict:
    """The oracle's `kind` driver ("stochastic", "greedy" or "nkl") over sequences `seqs`
    (default: all) of workload w, on nproc processes (default: every host core).
    kwargs go to the driver (T defaults to w.T)."""
    seqs = list(range(w.B)) if seqs is None else list(seqs)
    if not seqs:
        return {}
    nproc = max(1, min(nproc or os.cpu_count() or 1, len(seqs)))
    kwargs = dict(kwargs)
    kwargs.setdefault("dtype", w.dtype)
    if kind != "greedy":
        kwargs.setdefault("T", w.T)
    base = "/dev/shm" if os.path.isdir("/dev/shm") and os.access("/dev/shm", os.W_OK) else None
    tmp = tempfile.mkdtemp(prefix="oracle_pool_", dir=base)
    try:
        files = {}
        for name in ("target", "draft"):
            f = os.path.join(tmp, name + ".npy")
            np.save(f, getattr(w, name))
            files[name] = f
        small = {"tokens": w.tokens, "cu_draft": w.cu_draft, "u_accept": w.u_accept, "u_sample": w.u_sample}
        shares = [seqs[r::nproc] for r in range(nproc)]
        tasks = [(kind, files, small, dict(kwargs), s) for s in shares if s]
        ctx = mp.get_context("spawn")
        with ctx.Pool(len(tasks)) as pool:
            parts = pool.map(_worker, tasks)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    out = {}
    for p in parts:
        out.update(p)
    return out
