"""Full-size parity checks in row chunks (test infrastructure).

Every batch row of a chain workload is generated from its own seed
(``workloads.make_chain``), so a worker process can regenerate any chunk of
rows, run the float64 oracle on it and compare the library's outputs for
those rows, without the whole float64 workload (11.5 GB for C2's 4096
rounds) ever sitting in one process.

The pool uses the ``spawn`` start method: its workers never inherit a CUDA
context, and they touch only the CPU (the oracle and the input generator).
"""

from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np

from speculative_decoding_verification_48_gb300 import workloads as W


def _init_worker():
    # one thread per worker: the pool itself spreads the work over the cores
    import torch
    torch.set_num_threads(1)


def spawn_pool(workers: int | None = None):
    n = workers or max(1, min(12, (os.cpu_count() or 2) - 1))
    return mp.get_context("spawn").Pool(n, initializer=_init_worker)


def chunks(B: int, size: int):
    return [(r0, min(size, B - r0)) for r0 in range(0, B, size)]


def _gen(task):
    spec, r0, n = task
    return W.make_chain(**{**spec, "B": n, "row0": r0})


def generate(pool, spec: dict, size: int) -> W.ChainCase:
    """The whole workload of ``spec``, generated chunk by chunk in the pool."""
    parts = pool.map(_gen, [(spec, r0, n) for r0, n in chunks(spec["B"], size)])
    return W.concat_chain(parts, spec["name"])


def _compare(task):
    import oracle
    from oracle.compare import compare_chain
    spec, r0, n, outs, prob_tol = task
    case = W.make_chain(**{**spec, "B": n, "row0": r0})
    args = case.numpy64()
    ref = oracle.verify_chain(*args)
    toks, nacc, diag, st = outs
    cmp = compare_chain(args, ref, toks, nacc, st, diag, prob_tol=prob_tol)

    def shift(items):  # row indices of this chunk -> rows of the whole workload
        return [(x[0] + r0,) + tuple(x[1:]) for x in items]

    return dict(exact=cmp["exact"], boundary=shift(cmp["boundary"]),
                failures=shift(cmp["failures"]), diag_max_err=cmp["diag_max_err"],
                num_accepted=ref["num_accepted"], greedy=ref["greedy"], status=ref["status"])


def compare(pool, spec: dict, outputs, size: int, prob_tol: float) -> dict:
    """Compare library outputs (numpy tokens, num_accepted, diag, status for
    every row of ``spec``) with the oracle, chunk by chunk in the pool."""
    toks, nacc, diag, st = outputs
    tasks = [(spec, r0, n, (toks[r0:r0 + n], nacc[r0:r0 + n],
                            None if diag is None else diag[r0:r0 + n], st[r0:r0 + n]), prob_tol)
             for r0, n in chunks(spec["B"], size)]
    res = pool.map(_compare, tasks)
    return dict(rows=spec["B"], exact=sum(r["exact"] for r in res),
                boundary=[b for r in res for b in r["boundary"]],
                failures=[f for r in res for f in r["failures"]],
                diag_max_err=max(r["diag_max_err"] for r in res),
                num_accepted=np.concatenate([r["num_accepted"] for r in res]),
                greedy=np.concatenate([r["greedy"] for r in res]),
                status=np.concatenate([r["status"] for r in res]))
