"""The seeded generators (synth/) give the same graph for any number of host
threads (counter-based draws, stable sorts), so a workload is identical on the
8-core container and the 16-core GPU host."""
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SNIPPET = """
import sys, numpy as np
sys.path.insert(0, {root!r})
import synth
r, c = synth.rmat(14, 0.57, 0.19, 0.19, 120000, 9)
w_r, w_c = synth.weblike(1 << 14, seed=4)
synth.permute_bfs(1 << 14, r, c, 9)
np.savez({out!r}, r=r, c=c, wr=w_r, wc=w_c)
"""


def _run(threads, out):
    env = dict(os.environ, K2T_SYNTH_THREADS=str(threads))
    subprocess.check_call([sys.executable, "-c", _SNIPPET.format(root=ROOT, out=out)], env=env)
    return np.load(out)


def test_generators_independent_of_thread_count(tmp_path):
    a = _run(1, str(tmp_path / "one.npz"))
    b = _run(7, str(tmp_path / "seven.npz"))
    for k in ("r", "c", "wr", "wc"):
        assert a[k].size > 0 and np.array_equal(a[k], b[k]), k
