"""Stored row statistics of the fp64 oracle for the full-size parity checks, and the script
that writes them.

At S >= 128K the expensive half of a backward check is the forward statistics of every query
row that sees the checked keys: LSE_i and D_i = <dO_i, O_i> need the row's whole score row and
O_i. They depend only on the seeded inputs, so this script computes them once with
oracle.attn_row_stats_ref (nothing else does arithmetic here) and stores them next to a
SHA-256 fingerprint of the exact input bytes they were computed from. The GPU tests check the
fingerprint, compare the CUDA path's LSE with the stored values on every covered row, and run
the cheap half (oracle.attn_group_from_stats_ref: dK, dV from the statistics) themselves.

The inputs of these workloads are drawn on the GPU (workloads.make_inputs), so the script runs
where a GPU is present:
    python -m tests.golden.attn_stats [workload ...]
It writes tests/golden/attn_stats_<workload>.npz.

What each file covers (batch 0, one kv-head and its q-heads):
  llama8b_s128k       kv-head 0, every row: the whole slice's dK/dV is checked.
  llama8b_s1m_hostkv  kv-head 7, rows from S - T - 128: the 256-key window straddling the
                      last trunk boundary, [S - T - 128, S - T + 128).
  gqa32b_s256k_peaky  kv-head 0, rows from j0: the 256-key window [j0, j0 + 256) around the
                      last trunk boundary n*T (j0 = n*T - 128) whose window holds one of the
                      x8 key rows.
"""
from __future__ import annotations

import hashlib
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))


def path(name: str) -> str:
    return os.path.join(HERE, f"attn_stats_{name}.npz")


def spec(name: str, peaky=None):
    """(kv-head, first row, key window) of the check for a workload. peaky: the scaled key
    positions (workloads.peaky_rows) for the peaky workload."""
    from workloads import WORKLOADS
    w = WORKLOADS[name]
    if name == "llama8b_s128k":
        return 0, 0, (0, w.S)
    if name == "llama8b_s1m_hostkv":
        j0 = w.S - w.seq_trunk - 128
        return 7, j0, (j0, j0 + 256)
    if name == "gqa32b_s256k_peaky":
        T = w.seq_trunk
        marks = set(int(p) for p in peaky)
        for n in range((w.S - 1) // T, 0, -1):
            if any(p in marks for p in range(n * T - 128, n * T + 128)):
                return 0, n * T - 128, (n * T - 128, n * T + 128)
        raise ValueError("no trunk boundary window holds a scaled key row")
    raise KeyError(name)


def fingerprint(q, k, v, do, kvh, row_lo) -> str:
    """SHA-256 over the bytes of the input slices the statistics depend on: q and dO rows
    [row_lo, S) of the kv-head's q-heads, all of k and v of the kv-head (batch 0)."""
    import torch
    Hq, Hkv = q.shape[2], k.shape[2]
    G = Hq // Hkv
    h = hashlib.sha256()
    for t, lo, hs in ((q, row_lo, slice(kvh * G, (kvh + 1) * G)), (k, 0, slice(kvh, kvh + 1)),
                      (v, 0, slice(kvh, kvh + 1)), (do, row_lo, slice(kvh * G, (kvh + 1) * G))):
        x = t[0, lo:, hs, :].contiguous().view(torch.int16).cpu().numpy()
        h.update(x.tobytes())
    return h.hexdigest()


def load(name: str):
    """The stored statistics: dict with lse, dvec [G, S - row_lo], row_lo, kvh, fingerprint."""
    with np.load(path(name)) as z:
        return {"lse": z["lse"], "dvec": z["dvec"], "row_lo": int(z["row_lo"]),
                "kvh": int(z["kvh"]), "fingerprint": str(z["fingerprint"])}


def write(name: str) -> str:
    import torch

    import oracle
    from workloads import WORKLOADS, make_inputs, peaky_rows
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    kvh, row_lo, _ = spec(name, peaky_rows(w) if w.peaky_frac > 0 else None)
    G = w.Hq // w.Hkv
    lse = np.empty((G, w.S - row_lo))
    dvec = np.empty((G, w.S - row_lo))
    for g in range(G):
        lse[g], dvec[g] = oracle.attn_row_stats_ref(q, k, v, do, 0, kvh * G + g, row_lo, w.S,
                                                    causal=w.causal, row_block=256)
    fp = fingerprint(q, k, v, do, kvh, row_lo)
    np.savez_compressed(path(name), lse=lse, dvec=dvec, row_lo=row_lo, kvh=kvh, fingerprint=fp)
    del q, k, v, do
    torch.cuda.empty_cache()
    return path(name)


if __name__ == "__main__":
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    names = sys.argv[1:] or ["llama8b_s128k", "llama8b_s1m_hostkv", "gqa32b_s256k_peaky"]
    for n in names:
        print(write(n), flush=True)
