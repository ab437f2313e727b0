"""Write margin_redraws.json: which rows of x are redrawn, and how often.

A row t of x is kept only if the oracle's fp64 top-k margin of its router
logits (k-th largest minus (k+1)-th largest) is at least 1e-3; otherwise it is
redrawn from the generator stream with the next attempt number.  The table
holds {layer name: {token: attempts}} for every layer shape in synth.CONFIGS.
Only the oracle and the generator are called here.

    python tests/golden/make_margin_redraws.py
"""
import json
import os
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

MARGIN = 1e-3


def margins(cfg, x, rw, rb, rows):
    chunks = np.array_split(rows, max(1, min(len(rows), 4 * (os.cpu_count() or 1))))
    chunks = [c for c in chunks if len(c)]

    def work(c):
        return oracle.router(np.ascontiguousarray(x[c]), rw, rb, cfg.top_k)["margin"]

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        parts = list(ex.map(work, chunks))
    return np.concatenate(parts)


def redraws(cfg):
    rw, rb = synth.router(cfg)
    attempts = np.zeros(cfg.T, np.uint32)
    x = synth.x_rows(cfg, attempts)
    rows = np.arange(cfg.T)
    while len(rows):
        m = margins(cfg, x, rw, rb, rows)
        bad = rows[m < MARGIN]
        attempts[bad] += 1
        if len(bad):
            x[bad] = synth.x_rows(cfg, attempts, rows=bad)
        rows = bad
    return {str(int(t)): int(attempts[t]) for t in np.nonzero(attempts)[0]}


def main():
    table = {}
    for cfg in synth.CONFIGS:
        table[cfg.name] = redraws(cfg)
        print(cfg.name, "redrawn rows:", len(table[cfg.name]), "of", cfg.T, flush=True)
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "margin_redraws.json"), "w") as f:
        json.dump(table, f, indent=0, sort_keys=True)


if __name__ == "__main__":
    main()
