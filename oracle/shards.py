"""Run oracle calls over contiguous shards of their inputs in host threads.

TEST INFRASTRUCTURE ONLY, like the rest of this package: the test suite and the
CPU-baseline leg of ``bench.py`` use it to run the unchanged oracle functions on all
host cores.

Every 128-value INT8 block and every 32-value MX group is computed from its own values
alone ("feat(pcie_dma): add block-INT8 wire modes for AG, ring, and A2A", Summary;
"feat(pcie_dma): add INT8 and MXFP8 wire modes", Summary), and a row of the workloads
here is a whole number of blocks. So running an oracle function on each shard of rows
and placing the shards' results side by side gives exactly the bytes of one call on the
whole input. This module holds no arithmetic of the codec: it only cuts row ranges and
runs calls. ctypes releases the GIL around each C call, so the threads run in parallel.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # not Linux
        return max(1, os.cpu_count() or 1)


def row_ranges(rows: int, parts: int):
    """Split [0, rows) into at most `parts` contiguous, non-empty ranges of nearly equal
    size, in order."""
    parts = max(1, min(parts, rows))
    base, extra = divmod(rows, parts)
    out, lo = [], 0
    for p in range(parts):
        hi = lo + base + (1 if p < extra else 0)
        out.append((lo, hi))
        lo = hi
    return out if rows > 0 else []


def run_indexed(work, parts: int, threads: int = 0):
    """Call work(p) for p = 0 .. parts-1 on `threads` host threads (0: one per part).
    Returns the results in order; the first exception raised by any call is raised here."""
    threads = min(parts, threads or parts)
    if threads <= 1:
        return [work(p) for p in range(parts)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = [ex.submit(work, p) for p in range(parts)]
        return [f.result() for f in futs]


def run(work, rows: int, threads: int, parts: int = 0):
    """Call work(lo, hi) for every range of row_ranges(rows, parts or threads) on
    `threads` host threads (more parts than threads bounds each call's memory).
    Returns the results in range order."""
    ranges = row_ranges(rows, parts or threads)
    return run_indexed(lambda p: work(*ranges[p]), len(ranges), threads)
