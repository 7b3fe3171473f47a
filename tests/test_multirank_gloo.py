"""Sharded execution of the path across ranks, on CPU ranks over gloo.

The planes G(., k) are independent per bright-field pixel, and O(q), N(q)
and mean_k G(0,k) are sums over k.  So the build shards over k with no
exchange, and the reduction shards over k with one all-reduce (sum) of O, N
and the G(0,k) sum, after which any rank forms the image ("Tilt-corrected
SSB on CUDA", Where the time went: the reduction is a sum over BF pixels per
frequency; "Historical WebGPU G(q,k) memory experiment", Implementation: G is
built per BF pixel).  The per-BF phase moments shard the same way: each rank sums the angles of its
own BF pixels' images and their squares, and one all-reduce of those two
images gives the mean and variance over all pixels ("Historical WebGPU G(q,k)
memory experiment", Object-redraw fast path: the exact path is a mean over BF
pixels).  These tests run that plan on two gloo ranks with the oracle as the
per-rank compute and compare it with the single-process oracle.
"""
import os
import socket
import tempfile

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir, name):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import ssb_oracle as O
        from synth import configs as C
        from synth import forward as F
        d = F.make_numpy_dataset(name)
        g, ab = d["geom"], d["ab"]
        bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
        mine = np.array_split(bf, world)[rank]          # contiguous k shard
        G = O.build_G(d["frames"], mine)                  # no exchange
        Oq, Nq = O.reduce(G, g, ab, mine)
        band = O.band_indices(g, *C.BAND_INVA)
        sets = C.perturbed_sets(ab, 2, seed=4)
        Ob = [O.reduce(G, g, s, mine, entries=band) for s in sets]
        # one all-reduce of the partial sums
        parts = [torch.from_numpy(np.ascontiguousarray(Oq).view(np.float64).copy()),
                 torch.from_numpy(Nq.astype(np.int64)),
                 torch.tensor([float(np.sum(G[:, 0, 0].real)), float(len(mine))], dtype=torch.float64)]
        for o, nn in Ob:
            parts.append(torch.from_numpy(np.ascontiguousarray(o).view(np.float64).copy()))
            parts.append(torch.from_numpy(nn.astype(np.int64)))
        n = g.n
        s1, s2 = np.zeros((n, n)), np.zeros((n, n))
        for a, b in O.per_bf_images(G, g, ab, mine):    # this rank's BF pixels only
            t = np.arctan2(b, a)
            s1 += t
            s2 += t * t
        parts += [torch.from_numpy(s1), torch.from_numpy(s2)]
        for t in parts:
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
        if rank == 0:
            np.savez(os.path.join(out_dir, "reduced.npz"), *[t.numpy() for t in parts])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["tiny"])
def test_k_sharded_reduction_matches_single_process(name):
    from oracle import ssb_oracle as O
    from synth import configs as C
    from synth import forward as F

    with tempfile.TemporaryDirectory() as td:
        mp.start_processes(_rank_main, args=(2, _free_port(), td, name), nprocs=2, join=True,
                           start_method="spawn")
        z = np.load(os.path.join(td, "reduced.npz"))
        parts = [z[f"arr_{i}"] for i in range(len(z.files))]

    d = F.make_numpy_dataset(name)
    g, ab = d["geom"], d["ab"]
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    ref = O.reconstruct(d["frames"], g, ab, bf)
    n = g.n

    O_sh = parts[0].view(np.complex128)
    N_sh = parts[1]
    g0_sum, cnt = parts[2]
    assert int(cnt) == len(bf)
    np.testing.assert_array_equal(N_sh, ref["N"])
    assert np.linalg.norm(O_sh - ref["O"]) <= 1e-12 * np.linalg.norm(ref["O"])
    g0 = g0_sum / cnt
    assert abs(g0 - O.g0_mean(ref["G"]).real) <= 1e-12 * abs(g0)
    ph = O.phase_image(O_sh, N_sh, g0, n)
    np.testing.assert_allclose(ph, ref["phase"], rtol=0, atol=1e-12)

    band = O.band_indices(g, *C.BAND_INVA)
    sets = C.perturbed_sets(ab, 2, seed=4)
    for i, s in enumerate(sets):
        o_ref, n_ref = O.reduce(ref["G"], g, s, bf, entries=band)
        o_sh = parts[3 + 2 * i].view(np.complex128)
        n_sh = parts[4 + 2 * i]
        np.testing.assert_array_equal(n_sh, n_ref)
        assert np.linalg.norm(o_sh - o_ref) <= 1e-12 * max(np.linalg.norm(o_ref), 1e-300)
        assert abs(O.score(o_sh, n_sh) - O.score(o_ref, n_ref)) <= 1e-12 * max(O.score(o_ref, n_ref), 1e-300)

    # per-BF moments from the all-reduced angle sums
    mean_ref, var_ref = O.phase_moments(ref["G"], g, ab, bf)
    mean_sh = parts[7] / len(bf)
    var_sh = np.maximum(parts[8] / len(bf) - mean_sh * mean_sh, 0.0)
    np.testing.assert_allclose(mean_sh, mean_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(var_sh, var_ref, rtol=0, atol=1e-12)
