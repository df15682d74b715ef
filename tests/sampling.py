"""Seeded query-row samples for full-size parity checks, and a process pool
that evaluates the fp64 oracle on them (test infrastructure only).

Row sample (per query head, 512 rows): a fixed set of boundary rows -- the
first rows, both sides of the local window w0 and of the pretrained window
w_pretrained, G-aligned rows around w_pretrained and L/2, the last rows --
then uniform draws without replacement up to 512, from
numpy.random.default_rng(1000 * workload_index + head).
"""

from __future__ import annotations

import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np


def boundary_rows(L: int, w0: int, wp: int, G: int) -> list[int]:
    cand = [0, 1, 2, w0 - 1, w0, w0 + 1, w0 + 2, wp - 1, wp, wp + 1, L // 2, L - 2, L - 1]
    for centre in (wp, L // 2):
        base = (centre // G) * G
        cand += [base - 1, base, base + 1, base + G - 1, base + G]
    return sorted({r for r in cand if 0 <= r < L})


def sample_rows(L: int, w0: int, wp: int, G: int, n: int, seed: int) -> np.ndarray:
    fixed = boundary_rows(L, w0, wp, G)
    if n >= L:
        return np.arange(L, dtype=np.int64)
    rng = np.random.default_rng(seed)
    rest = np.setdiff1d(np.arange(L, dtype=np.int64), np.asarray(fixed, dtype=np.int64))
    extra = rng.choice(rest, size=max(0, n - len(fixed)), replace=False)
    return np.sort(np.concatenate([np.asarray(fixed, dtype=np.int64), extra]))[:n]


def _worker(args):
    os.environ.setdefault("OMP_NUM_THREADS", "1")
    import oracle
    q, k, v, w0, wp, theta, rows, rounded = args
    return oracle.bifocal_prefill(q, k, v, w0, wp, theta, round_rotated_qk=rounded, rows=rows)


def oracle_prefill_rows(q, k, v, w0, wp, theta, rows, rounded, workers=None):
    """Oracle output on sampled rows, one process per KV head.

    q [1, L, Hq, d], k/v [1, L, Hkv, d] as float32 numpy arrays; rows [Hq, n].
    Returns (o [1, n, Hq, d], lse [1, Hq, n])."""
    _, L, Hq, d = q.shape
    Hkv = k.shape[2]
    grp = Hq // Hkv
    jobs = []
    for hk in range(Hkv):
        hs = slice(hk * grp, (hk + 1) * grp)
        jobs.append((q[:, :, hs], k[:, :, hk:hk + 1], v[:, :, hk:hk + 1], w0, wp, theta,
                     rows[hs], rounded))
    workers = workers or min(Hkv, os.cpu_count() or 1)
    ctx = mp.get_context("spawn")
    with cf.ProcessPoolExecutor(max_workers=workers, mp_context=ctx) as ex:
        res = list(ex.map(_worker, jobs))
    n = rows.shape[1]
    o = np.zeros((1, n, Hq, d))
    lse = np.zeros((1, Hq, n))
    for hk, (oh, lh) in enumerate(res):
        o[:, :, hk * grp:(hk + 1) * grp] = oh
        lse[:, hk * grp:(hk + 1) * grp] = lh
    return o, lse
