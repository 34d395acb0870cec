"""Host logic on CPU: the key runs of a streaming call (``plan_key_runs``,
used by the host planner and by the graph-mode kernels) against the key
rows implied by the oracle's ring model -- the sink rows when used, ring
chunks max(0, c - W) .. c (.. c - 1 with the current chunk passed in) at
physical slot ``oracle.ring.slot_of(chunk, R)``, and the current chunk's own
tensor -- for every window the ring can hold.  Each visible row is covered
exactly once, adjacent runs are merged, and the tile numbering is the running
sum of whole 128-key tiles per run.  The harness is host code built with
nvcc; no GPU is touched."""

import os
import shutil
import subprocess
import tempfile
from collections import Counter

import pytest

from oracle.ring import slot_of

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def plans():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "plan")
        subprocess.run([nvcc, "-std=c++17", "-O1", "-o", exe, os.path.join(HERE, "host", "plan_key_runs_main.cu")],
                       check=True, capture_output=True)
        out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return [list(map(int, ln.split())) for ln in out.splitlines()]


def test_plans_cover_the_window_once(plans):
    assert len(plans) > 1000
    for p in plans:
        c, W, R, Lc, has_sink, use_sink, kcur, nseg, total = p[:9]
        segs = [tuple(p[9 + 4 * i: 13 + 4 * i]) for i in range(nseg)]
        assert 1 <= nseg <= 4 or (nseg == 0 and not use_sink and not kcur)
        expect = Counter()
        if use_sink:
            expect.update((0, r) for r in range(Lc))
        for x in range(max(0, c - W), c - kcur + 1):
            base = (has_sink + slot_of(x, R)) * Lc
            expect.update((0, r) for r in range(base, base + Lc))
        if kcur:
            expect.update((1, r) for r in range(Lc))
        got = Counter()
        for src, row0, nrows, _ in segs:
            got.update((src, r) for r in range(row0, row0 + nrows))
        assert got == expect, (p[:9], segs)
        # runs of the ring are merged when physically adjacent
        for a, b in zip(segs, segs[1:]):
            assert not (a[0] == b[0] == 0 and a[1] + a[2] == b[1]), (p[:9], segs)
        # tile numbering: running sum of whole tiles per run
        t = 0
        for src, row0, nrows, tile0 in segs:
            assert tile0 == t, (p[:9], segs)
            t += (nrows + 127) // 128
        assert total == t
