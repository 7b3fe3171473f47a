"""Host logic of bench.py that needs no GPU: the build-traffic model behind
`roofline.traffic` reproduces the per-launch DRAM reads captured on the mid
workload (512^2 scan, 64^2 detector; ssb_gather, chunks 4 to 7 of a build:
100.77, 100.93, 100.89 and 67.15 MB, i.e. 3, 3, 3 and 2 lines of 128 bytes
per frame)."""
import importlib.util
import os

import numpy as np

from synth import configs as C

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _bf(name):
    import electron_microscopy_gb300 as ssb
    w = C.WORKLOADS[name]
    g, ab = C.geometry(w), C.aberrations(w)
    return g, np.asarray(ssb.bf_indices(g, ab), dtype=np.int64)


def test_gather_line_model_matches_mid_capture():
    b = _bench()
    g, bf = _bf("mid")
    lines = [len(np.unique((bf[c:c + b.BUILD_CHUNK_BF] * 2) // 128))
             for c in range(0, len(bf), b.BUILD_CHUNK_BF)]
    assert lines[4:8] == [3, 3, 3, 2]
    frames = g.n * g.n
    for nl, mb in zip(lines[4:8], (100.77, 100.93, 100.89, 67.15)):
        assert abs(nl * 128 * frames / 1e6 - mb) < 0.5


def test_build_traffic_full_workload():
    b = _bench()
    g, bf = _bf("full")
    t = b.build_traffic(g, bf, g.n)
    if t is None:  # the build kernels changed since the capture: no figure claimed
        return
    # gather reads 14.33 GB (the earlier full-size capture: 14.35 GB) + 1.250 MB per pixel written
    assert abs(t - (14.328e9 + len(bf) * 1.250e6)) < 0.01e9
    assert b.build_traffic(C.geometry(C.WORKLOADS["large"]), bf, 1024) is None
