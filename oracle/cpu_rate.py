"""Throughput of the oracle on one host core: one process of the bench's
all-cores CPU baseline.

TEST INFRASTRUCTURE, like the rest of oracle/: only the tests and the
bench's CPU-baseline leg run it; nothing on the GPU path imports it.  It
imports numpy and the oracle only, so a process starts in well under a
second.

    python -m oracle.cpu_rate BITS.npy W.npy T0 N START_AT BUDGET_S CHUNK

BITS.npy holds the workload's sources as bf16 bit patterns ([S, T, d],
uint16; widened exactly to fp64 here), W.npy the pseudo-query ([d], fp32).
The process takes tokens [T0, T0 + N), waits until the wall-clock time
START_AT (seconds since the epoch), runs `depth_attention` over CHUNK-token
pieces of them, wrapping around, for BUDGET_S seconds, and prints one JSON
line {"tokens": ..., "start": ..., "end": ...} (wall-clock times).
"""
from __future__ import annotations

import json
import sys
import time

import numpy as np

from .attnres_oracle import depth_attention


def run(bits_path: str, w_path: str, t0: int, n: int, start_at: float, budget_s: float, chunk: int) -> dict:
    bits = np.load(bits_path, mmap_mode="r")
    sl = np.ascontiguousarray(bits[:, t0:t0 + n])
    h = (sl.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    w = np.load(w_path).astype(np.float64)
    n = h.shape[1]
    delay = start_at - time.time()
    if delay > 0:
        time.sleep(delay)
    tokens, start = 0, 0
    t_start = time.time()
    c0 = time.perf_counter()
    while True:
        depth_attention(h[:, start:start + chunk], w)
        tokens += min(chunk, n - start)
        start = (start + chunk) % n
        if time.perf_counter() - c0 >= budget_s:
            break
    return {"tokens": tokens, "start": t_start, "end": t_start + (time.perf_counter() - c0)}


def main(argv: list[str]) -> int:
    if len(argv) != 7:
        print(__doc__, file=sys.stderr)
        return 2
    bits_path, w_path = argv[0], argv[1]
    t0, n = int(argv[2]), int(argv[3])
    start_at, budget_s, chunk = float(argv[4]), float(argv[5]), int(argv[6])
    print(json.dumps(run(bits_path, w_path, t0, n, start_at, budget_s, chunk)))
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))
