"""Benchmark: SSB G build + reconstruction + batched scoring on one GB300.

One step = one pass of the whole hot path over the full-size synthetic scan
(512^2 scan, 192^2 uint16 detector, ~9.35k bright-field pixels):
  ssb_build_G      frames -> G(q,k) half plane             (the build)
  ssb_reconstruct  one aberration set -> O, N, phase image (the recon)
  ssb_score_batch  8 aberration sets over the 0.2-0.9 1/A band -> scores

Prints one JSON line.  `value` is ms per step (device time, inputs resident
in HBM, max over ranks); `e2e` is the same step through the public API with
host buffers: the frames stay in pinned host memory and ssb_build_G_host
copies the bright-field box of every frame each step; the phase
image and the scores are copied out every step.  `--impl reference` times the CPU float64 oracle on a bounded sample of
the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "ms per SSB recon + G-build HBM GB/s (512^2 scan, 192^2 det, ~9.3k BF px)"

L2_BYTES = 129 * 1024 * 1024


def gpu_numa_node(index):
    """NUMA node of GPU `index` (sysfs of its PCI function), or None."""
    try:
        out = subprocess.run(["nvidia-smi", f"--id={index}", "--query-gpu=pci.bus_id", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=30).stdout.strip()
        bus = out.split()[0].lower()
        dom, rest = bus.split(":", 1)
        path = f"/sys/bus/pci/devices/{dom[-4:]}:{rest}/numa_node"
        node = int(open(path).read().strip())
        return node if node >= 0 else None
    except (OSError, ValueError, IndexError, subprocess.SubprocessError):
        return None


def bind_to_node(node):
    """Restrict this process to the CPUs of NUMA node `node` (so that pinned
    host buffers allocated afterwards are first touched there).  Returns the
    CPU list used, or None."""
    try:
        text = open(f"/sys/devices/system/node/node{node}/cpulist").read().strip()
    except OSError:
        return None
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    cpus &= os.sched_getaffinity(0)
    if not cpus:
        return None
    os.sched_setaffinity(0, cpus)
    return sorted(cpus)


# DRAM traffic of one n = 512 build (ssb_gather + ssb_plane512 on uint16
# frames), from per-kernel ncu captures on the mid workload (512^2 scan, 64^2
# detector; one kernel name and four launches per capture, dram__bytes_read
# and dram__bytes_write with --cache-control none) scaled to this workload:
#  * the gather reads, for every frame, each 128-byte line that its chunk of
#    60 bright-field pixels falls in; this count reproduced the captured reads
#    chunk by chunk (2 to 4 lines per frame), so it is evaluated here on the
#    actual BF list;
#  * the two kernels together write 1.250 MB per BF pixel (the 1.053 MB of
#    G's half plane plus cluster exchange slots evicted from L2), and the
#    plane kernel's reads of its chunk buffer hit L2.
# The figure belongs to the build kernels' source: if it has changed since the
# capture, no traffic is claimed.
BUILD_SOURCES_SHA = "38e4d35b23e3cbdc"
BUILD_WRITE_BYTES_PER_BF = 1.250e6
BUILD_CHUNK_BF = 60


def build_traffic(geom, bf, n):
    h = hashlib.sha256()
    for f in ("build.cu", "plane.cu"):
        with open(os.path.join(ROOT, "electron_microscopy_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    if n != 512 or h.hexdigest()[:16] != BUILD_SOURCES_SHA:
        return None
    bf = np.asarray(bf, dtype=np.int64)
    lines = sum(len(np.unique((bf[c:c + BUILD_CHUNK_BF] * 2) // 128)) for c in range(0, len(bf), BUILD_CHUNK_BF))
    return float(lines * 128 * n * n + len(bf) * BUILD_WRITE_BYTES_PER_BF)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="full", choices=["full", "large", "mid", "middet", "midlarge", "small", "tiny"])
    p.add_argument("--sets", type=int, default=8)
    p.add_argument("--e2e-steps", type=int, default=8)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-sweep", action="store_true", help="skip the B = 1, 2, 4, 8 scoring sweep")
    p.add_argument("--no-compact", action="store_true",
                   help="skip the compact-storage measurements (band copy, herm16)")
    p.add_argument("--cpu-sample-bf", type=int, default=0, help="BF pixels in the oracle sample (0: auto)")
    return p.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs its own full problem)
# ----------------------------------------------------------------------------

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1 and args.impl == "ours":
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(backend="nccl")
        pg = dist
    return ws, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def allmax(pg, x, device=None):
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------
# oracle (CPU float64) timing on a bounded sample
# ----------------------------------------------------------------------------

def oracle_sample(d, bf_all, band, sets, n_sample, cols_host):
    """Time the CPU oracle on `n_sample` BF pixels of the workload: G build,
    one reconstruction's reduction over the whole half plane and the 8-set band
    reduction, then scale to all BF pixels (every stage is linear in N_bf; the
    O(n^2 log n) image step is added once)."""
    from oracle import ssb_oracle as O
    g, ab = d["geom"], d["ab"]
    n = g.n
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(len(bf_all), size=n_sample, replace=False))
    bf = bf_all[pick]
    frames_sub = cols_host[:, pick].reshape(n, n, 1, n_sample)  # fake (n, n, 1, s) layout
    idx = np.arange(n_sample, dtype=np.int32)
    t0 = time.perf_counter()
    G = O.build_G(frames_sub, idx)
    t1 = time.perf_counter()
    Oq, Nq = O.reduce(G, g, ab, bf)
    t2 = time.perf_counter()
    O.phase_image(Oq, Nq, O.g0_mean(G), n)
    t3 = time.perf_counter()
    for s in sets:
        O.reduce(G, g, s, bf, entries=band)
    t4 = time.perf_counter()
    scale = len(bf_all) / n_sample
    per_step = (t1 - t0) * scale + (t2 - t1) * scale + (t3 - t2) + (t4 - t3) * scale
    return {"ms_per_step": per_step * 1e3, "sample_seconds": t4 - t0,
            "build_ms": (t1 - t0) * scale * 1e3, "recon_ms": ((t2 - t1) * scale + (t3 - t2)) * 1e3,
            "score_ms": (t4 - t3) * scale * 1e3, "n_sample": n_sample}


def _oracle_chunk(job):
    """One worker's share of the pooled oracle sample: G build, the
    reconstruction's reduction and the band reductions of every set for a
    subset of the sampled BF pixels (each is a sum over BF pixels)."""
    from oracle import ssb_oracle as O
    g, ab, bf, cols, band, sets = job
    n, s = g.n, len(bf)
    G = O.build_G(cols.reshape(n, n, 1, s), np.arange(s, dtype=np.int32))
    O.reduce(G, g, ab, bf)
    for st in sets:
        O.reduce(G, g, st, bf, entries=band)
    return s


def oracle_pool_sample(d, bf_all, band, sets, n_sample, cols_host, procs):
    """The same sample as oracle_sample, split over `procs` spawned worker
    processes (the oracle itself unchanged); wall time scaled to all BF
    pixels.  Returns ms per step."""
    import multiprocessing as mp
    g, ab = d["geom"], d["ab"]
    rng = np.random.default_rng(0)
    pick = np.sort(rng.choice(len(bf_all), size=n_sample, replace=False))
    parts = [p for p in np.array_split(pick, procs) if len(p)]
    jobs = [(g, ab, bf_all[p], np.ascontiguousarray(cols_host[:, p]), band, sets) for p in parts]
    ctx = mp.get_context("spawn")
    with ctx.Pool(len(jobs)) as pool:
        # workers started and importing before the clock; bounded waits so a
        # pool that cannot start reports instead of hanging the benchmark
        pool.map_async(int, range(len(jobs))).get(timeout=300)
        t0 = time.perf_counter()
        pool.map_async(_oracle_chunk, jobs).get(timeout=1800)
        t = time.perf_counter() - t0
    return t * (len(bf_all) / n_sample) * 1e3


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ----------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ----------------------------------------------------------------------------

def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    from synth import configs as C
    from synth import forward as F
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    d = F.make_torch_dataset(args.workload, device=dev) if args.workload in ("full", "large", "mid", "middet", "midlarge") \
        else F.make_numpy_dataset(args.workload)
    g, ab = d["geom"], d["ab"]
    from oracle import ssb_oracle as O
    bf = O.bf_indices(g, ab.tilt_x_rad, ab.tilt_y_rad)
    band = O.band_indices(g, *C.BAND_INVA)
    sets = C.perturbed_sets(ab, args.sets, seed=4)
    n = g.n
    if torch.is_tensor(d["frames"]):
        cols = d["frames"].view(n * n, -1).index_select(1, torch.from_numpy(bf).to(d["frames"].device).long())
        cols = cols.cpu().numpy().view(np.uint16)
    else:
        cols = d["frames"].reshape(n * n, -1)[:, bf]
    n_sample = args.cpu_sample_bf or max(1, min(len(bf), 16 if n >= 512 else 64))
    times = []
    info = None
    for i in range(args.warmup + args.steps):
        info = oracle_sample(d, bf, band, sets, n_sample, cols)
        if i >= args.warmup:
            times.append(info["ms_per_step"])
    v = statistics.mean(times)
    line = {"metric": METRIC, "value": v, "unit": "ms", "impl": "reference", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {n}^2 scan, {g.det_y}^2 uint16 detector, "
                                   f"{len(bf)} BF px; step = G build + 1 reconstruction + "
                                   f"{args.sets}-set band scoring",
                       "sample": f"{n_sample} of {len(bf)} BF pixels per step, scaled by N_bf"},
            "cpu_baseline": {"value": v, "unit": "ms", "cores": 1, "kind": "oracle",
                             "sample": f"{n_sample} BF pixels per step (all q), linear scaling to {len(bf)}"},
            "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def run_ours(args, ws, rank, local, pg):
    import torch
    import electron_microscopy_gb300 as ssb
    from synth import configs as C
    from synth import forward as F

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssb.load()

    d = F.make_torch_dataset(args.workload, device=dev) if args.workload in ("full", "large", "mid", "middet", "midlarge") \
        else None
    if d is None:
        dn = F.make_numpy_dataset(args.workload)
        fr = dn["frames"]
        fr_t = torch.from_numpy(fr.view(np.int16) if fr.dtype == np.uint16 else fr).to(dev)
        d = {**dn, "frames": fr_t, "max_count": int(fr.max())}
    frames = d["frames"]
    geom, ab = d["geom"], d["ab"]
    n, h = geom.n, geom.n // 2 + 1
    bf = ssb.bf_indices(geom, ab)
    n_bf = len(bf)
    bfd = torch.from_numpy(bf).to(dev)
    band = ssb.band_indices(geom, *C.BAND_INVA)
    band_d = torch.from_numpy(band).to(dev)
    nq = len(band)
    sets = C.perturbed_sets(ab, args.sets, seed=4)
    B = len(sets)

    G = torch.empty((n_bf, n, h), dtype=torch.complex64, device=dev)
    Od = torch.empty((n, h), dtype=torch.complex64, device=dev)
    Nd = torch.empty((n, h), dtype=torch.int32, device=dev)
    ph = torch.empty((n, n), dtype=torch.float32, device=dev)
    Ob = torch.empty((B, nq), dtype=torch.complex64, device=dev)
    Nb = torch.empty((B, nq), dtype=torch.int32, device=dev)
    sc = torch.empty((B,), dtype=torch.float64, device=dev)
    ws_b = ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_BUILD), dev)
    ws_r = ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_RECON), dev)
    ws_s = ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_SCORE, B, nq), dev)
    stream = torch.cuda.Stream(device=dev)

    def step(fr=None):
        ssb.build_G(frames if fr is None else fr, geom, bfd, G=G, ws=ws_b, stream=stream)
        ssb.reconstruct(G, geom, bfd, ab, O=Od, N=Nd, phase=ph, ws=ws_r, stream=stream)
        ssb.score_batch(G, geom, bfd, sets, band_d, O=Ob, N=Nb, score=sc, ws=ws_s, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()

    # timed region (device time on the launching stream)
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    clocks = ClockSampler(vis.split(",")[local] if vis else str(local))
    clocks.start()
    time.sleep(0.3)
    barrier(pg)
    torch.cuda.synchronize()
    l0 = ssb.launch_count()
    t_wall0 = time.perf_counter()
    for i in range(K):
        e0, e1, e2, e3 = ev[i]
        e0.record(stream)
        ssb.build_G(frames, geom, bfd, G=G, ws=ws_b, stream=stream)
        e1.record(stream)
        ssb.reconstruct(G, geom, bfd, ab, O=Od, N=Nd, phase=ph, ws=ws_r, stream=stream)
        e2.record(stream)
        ssb.score_batch(G, geom, bfd, sets, band_d, O=Ob, N=Nb, score=sc, ws=ws_s, stream=stream)
        e3.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    launches = ssb.launch_count() - l0
    barrier(pg)
    clk = clocks.stop()
    b_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(K)]
    r_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(K)]
    s_ms = [ev[i][2].elapsed_time(ev[i][3]) for i in range(K)]
    tot = ev[0][0].elapsed_time(ev[K - 1][3])
    ms_step = allmax(pg, tot / K, dev)

    # algorithmic work
    bytes_build = n_bf * n * n * (2 if frames.element_size() == 2 else 4) + n_bf * n * h * 8
    bytes_recon = n_bf * n * h * 8
    bytes_score = n_bf * nq * 8
    terms = int(Nb.sum().item())
    build_ms = statistics.mean(b_ms)
    recon_ms = statistics.mean(r_ms)
    score_ms = statistics.mean(s_ms)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peaks = json.load(open(peaks_path))
        hbm = float(peaks["hbm_gbs"])
        peak_src = "measured"
    else:
        hbm = 6800.0
        peak_src = "fallback"
    achieved = bytes_build / (build_ms * 1e-3) / 1e9
    traffic = build_traffic(geom, bf, n) if frames.element_size() == 2 else None

    # end to end through the public API with host buffers: the frames stay in
    # pinned host memory and ssb_build_G_host copies the bright-field box of
    # every frame each step; phase image and scores come back each step.  Two
    # lanes (stream, G, workspaces, outputs) alternate, so the copy of step
    # i + 1 runs while step i computes, as a pipeline over a series of scans
    # would run.
    e2e = None
    if not args.no_e2e:
        vis_e = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        numa = gpu_numa_node(vis_e.split(",")[local] if vis_e else local)
        cpus_before = os.sched_getaffinity(0)
        bound = bind_to_node(numa) if numa is not None else None
        host = torch.empty(frames.shape, dtype=frames.dtype, pin_memory=True)
        host.copy_(frames)  # first touch on the GPU's node
        os.sched_setaffinity(0, cpus_before)
        code = ssb.SSB_U16 if frames.element_size() == 2 else ssb.SSB_F32
        r_bf, c_bf = bf // geom.det_x, bf % geom.det_x
        box = (int(r_bf.min()), int(r_bf.max()), int(c_bf.min()), int(c_bf.max()))
        h2d = n * n * (box[1] - box[0] + 1) * (box[3] - box[2] + 1) * frames.element_size()
        E = max(2, args.e2e_steps)
        lanes = []
        for li in range(2):
            L = {"stream": stream if li == 0 else torch.cuda.Stream(device=dev),
                 "G": G if li == 0 else torch.empty_like(G),
                 "ws_h": ssb.Workspace(ssb.build_G_host_bytes(geom, bf, code), dev),
                 "ws_r": ws_r if li == 0 else ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_RECON), dev),
                 "ws_s": ws_s if li == 0 else ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_SCORE, B, nq),
                                                            dev),
                 "O": torch.empty_like(Od), "N": torch.empty_like(Nd), "ph": torch.empty_like(ph),
                 "Ob": torch.empty_like(Ob), "Nb": torch.empty_like(Nb), "sc": torch.empty_like(sc),
                 "ph_h": torch.empty(ph.shape, dtype=ph.dtype, pin_memory=True),
                 "sc_h": torch.empty(sc.shape, dtype=sc.dtype, pin_memory=True)}
            lanes.append(L)

        def e2e_step(L):
            st = L["stream"]
            ssb.build_G_host(host, geom, bf, bfd, G=L["G"], ws=L["ws_h"], stream=st)
            ssb.reconstruct(L["G"], geom, bfd, ab, O=L["O"], N=L["N"], phase=L["ph"], ws=L["ws_r"], stream=st)
            ssb.score_batch(L["G"], geom, bfd, sets, band_d, O=L["Ob"], N=L["Nb"], score=L["sc"], ws=L["ws_s"],
                            stream=st)
            with torch.cuda.stream(st):
                L["ph_h"].copy_(L["ph"], non_blocking=True)
                L["sc_h"].copy_(L["sc"], non_blocking=True)

        for L in lanes:  # warm-up (first use of each lane's workspaces)
            e2e_step(L)
        torch.cuda.synchronize()
        barrier(pg)
        t_stream = torch.cuda.Stream(device=dev)
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(t_stream)
        for L in lanes:
            L["stream"].wait_event(ea)
        for i in range(E):
            e2e_step(lanes[i % 2])
        for L in lanes:
            done = torch.cuda.Event()
            done.record(L["stream"])
            t_stream.wait_event(done)
        eb.record(t_stream)
        torch.cuda.synchronize()
        e2e_ms = allmax(pg, ea.elapsed_time(eb) / E, dev)
        # one call on its own (no pipelining): copy in, compute, results out
        L0 = lanes[0]
        ec, ed = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        lat = []
        for _ in range(2):
            torch.cuda.synchronize()
            ec.record(L0["stream"])
            e2e_step(L0)
            ed.record(L0["stream"])
            torch.cuda.synchronize()
            lat.append(ec.elapsed_time(ed))
        # the host link's ceiling in this run: one contiguous pinned copy of
        # the same number of bytes
        nel = h2d // frames.element_size()
        src_h = host.view(-1)[:nel]
        dst_d = torch.empty(nel, dtype=frames.dtype, device=dev)
        for _ in range(2):
            dst_d.copy_(src_h, non_blocking=True)
        ef, eg = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ef.record()
        dst_d.copy_(src_h, non_blocking=True)
        eg.record()
        torch.cuda.synchronize()
        link_GBs = h2d / (ef.elapsed_time(eg) * 1e-3) / 1e9
        del dst_d
        e2e = {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": ph.numel() * 4 + sc.numel() * 8, "steps": E,
               "latency_ms": min(lat), "link_GBs": link_GBs,
               "link_frac": h2d / (e2e_ms * 1e-3) / 1e9 / link_GBs,
               "link": "one contiguous pinned host-to-device copy of the step's bytes, timed in this run",
               "host_numa_node": numa, "host_cpus_bound": len(bound) if bound else None,
               "call": f"ssb_build_G_host (detector box rows {box[0]}..{box[1]}, columns {box[2]}..{box[3]} of "
                       f"{geom.det_y}x{geom.det_x}) + ssb_reconstruct + ssb_score_batch, phase and scores to host",
               "pipelining": "two streams alternate steps: the host-to-device copy of step i+1 overlaps step i"}
        del host, lanes

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cols = frames.view(n * n, -1).index_select(1, bfd.long()).cpu().numpy().view(np.uint16) \
            if frames.element_size() == 2 else frames.view(n * n, -1).index_select(1, bfd.long()).cpu().numpy()
        ns = min(n_bf, args.cpu_sample_bf or (96 if n >= 512 else 64))
        info = oracle_sample({"geom": geom, "ab": ab}, bf, band, sets, ns, cols)
        cpu = {"value": info["ms_per_step"], "unit": "ms", "cores": 1, "kind": "oracle",
               "sample": f"{ns} of {n_bf} BF pixels (all q, 1 recon + {B}-set band), scaled linearly by N_bf; "
                         f"{info['sample_seconds']:.1f} s of CPU work",
               "build_ms": info["build_ms"], "recon_ms": info["recon_ms"], "score_ms": info["score_ms"]}
        procs = cpu_threads()
        if procs > 1:
            try:
                v = oracle_pool_sample({"geom": geom, "ab": ab}, bf, band, sets, ns, cols, procs)
                cpu["pool"] = {"value": v, "unit": "ms", "cores": procs,
                               "sample": f"the same {ns} BF pixels split over {procs} spawned processes, wall "
                                         f"time scaled linearly by N_bf"}
            except Exception as exc:  # report, do not fail the benchmark
                cpu["pool"] = {"unavailable": f"{type(exc).__name__}: {exc}"}

    # the other stages against their binding units: the reconstruction streams
    # all of G (HBM); the 8-set scoring pass does one sincos (2 transcendental
    # results) per active term, against the sin/cos rate measured here by the
    # library's probe kernel (also the float32 FMA rate, context for the FFT)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    clk_mhz = (clk or {}).get("sm_mhz") or 2070.0
    with torch.cuda.stream(stream):
        rates = ssb.peak_rates(dev, stream=stream)
    xu_peak = rates["sincos_per_s"]
    fp32_peak = rates["fma_flops_per_s"]
    xu_ach = 2.0 * terms / (score_ms * 1e-3)
    def timed(run, reps=10, warm=3):
        """mean ms of `run` over `reps` calls, CUDA events on the launching stream"""
        for _ in range(warm):
            run()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def sweep(store, band_bytes):
        """B = 1, 2, 4, 8 sets per scoring pass over the band (10 passes each);
        store None: the complex64 half plane through ssb_score_batch"""
        out = {}
        for Bs in (1, 2, 4, 8):
            sub = sets[:Bs]
            Ob_s = torch.empty((Bs, nq), dtype=torch.complex64, device=dev)
            Nb_s = torch.empty((Bs, nq), dtype=torch.int32, device=dev)
            sc_s = torch.empty((Bs,), dtype=torch.float64, device=dev)
            ws_b2 = ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_SCORE, Bs, nq), dev)
            if store is None:
                run = lambda: ssb.score_batch(G, geom, bfd, sub, band_d, O=Ob_s, N=Nb_s, score=sc_s,  # noqa: E731
                                              ws=ws_b2, stream=stream)
            else:
                run = lambda: ssb.score_batch_g(store, geom, bfd, sub, band_d, O=Ob_s, N=Nb_s,  # noqa: E731
                                                score=sc_s, ws=ws_b2, stream=stream)
            t_ms = timed(run)
            terms_b = int(Nb_s.sum().item())
            out[str(Bs)] = {"ms": t_ms, "terms": terms_b, "terms_per_s": terms_b / (t_ms * 1e-3),
                            "xu_frac": 2.0 * terms_b / (t_ms * 1e-3) / xu_peak,
                            "hbm_frac": band_bytes / (t_ms * 1e-3) / 1e9 / hbm}
            del ws_b2
        return out

    # the batched-scoring configuration: B = 1, 2, 4, 8 sets per pass (after
    # the timed region)
    score_sweep = {} if args.no_sweep else sweep(None, bytes_score)

    # the depth-spread fit: the same 8 sets, each with a 136 A defocus spread
    # (the fit kernel's depth on the pages), one pass over the band
    score_depth = None
    if not args.no_sweep:
        depths = [136.0] * B
        t_dep = timed(lambda: ssb.score_batch_depth(G, geom, bfd, sets, depths, band_d, O=Ob, N=Nb, score=sc,
                                                    ws=ws_s, stream=stream))
        score_depth = {"ms": t_dep, "depth_A": 136.0, "sets": B, "terms": terms,
                       "terms_per_s": terms / (t_dep * 1e-3),
                       "xu_frac": 2.0 * terms / (t_dep * 1e-3) / xu_peak,
                       "note": "all sets at one spread with one tilt: the spread factor (a sine and a reciprocal) "
                               "once per active (q, k) pair, one sincos per active term; xu_frac counts the sincos "
                               "only",
                       "depth0_ms": score_ms}

    # compact G storage (measured after the timed region, not part of the
    # step): the band-compacted complex64 copy, and herm16 with one scale per
    # q row or per BF pixel -- the packing pass, the reconstruction from it and
    # the scoring sweep over its band copy.  Algorithmic bytes: what each pass
    # must read and write once.
    compact = None
    if not args.no_compact:
        compact = {}
        entries = n_bf * n * h
        Gb = torch.empty((n_bf, nq), dtype=torch.complex64, device=dev)
        src = ssb.GStore(G)
        t_band = timed(lambda: ssb.compact_band(src, geom, band_d, dst=Gb, stream=stream), reps=5)
        bb = n_bf * nq * 8
        compact["band_c64"] = {
            "copy_ms": t_band, "copy_GBs": 2 * bb / (t_band * 1e-3) / 1e9,
            "copy_hbm_frac": 2 * bb / (t_band * 1e-3) / 1e9 / hbm, "copy_algorithmic_bytes": 2 * bb,
            "score_sweep": sweep(ssb.GStore(Gb, band_compact=True), bb)}
        del Gb
        Oc, Nc, phc = torch.empty_like(Od), torch.empty_like(Nd), torch.empty_like(ph)
        for rows, name in ((1, "herm16_q_row"), (n, "herm16_bf")):
            W = torch.empty((n_bf, n, h), dtype=torch.int32, device=dev)
            S = torch.empty((n // rows, n_bf), dtype=torch.float32, device=dev)
            t_pack = timed(lambda: ssb.compact_G16(G, geom, rows, G16=W, scale=S, stream=stream), reps=5)
            st = ssb.GStore(W, ssb.G_SN16, S, rows)
            pack_bytes = entries * 8 + entries * 4 + S.numel() * 4
            t_rec = timed(lambda: ssb.reconstruct_g(st, geom, bfd, ab, O=Oc, N=Nc, phase=phc, ws=ws_r,
                                                    stream=stream))
            rec_bytes = entries * 4 + S.numel() * 4
            Wb = torch.empty((n_bf, nq), dtype=torch.int32, device=dev)
            ssb.compact_band(st, geom, band_d, dst=Wb, stream=stream)
            bb16 = n_bf * nq * 4
            compact[name] = {
                "rows_per_scale": rows,
                "pack_ms": t_pack, "pack_GBs": pack_bytes / (t_pack * 1e-3) / 1e9,
                "pack_hbm_frac": pack_bytes / (t_pack * 1e-3) / 1e9 / hbm, "pack_algorithmic_bytes": pack_bytes,
                "recon_ms": t_rec, "recon_GBs": rec_bytes / (t_rec * 1e-3) / 1e9,
                "recon_hbm_frac": rec_bytes / (t_rec * 1e-3) / 1e9 / hbm, "recon_algorithmic_bytes": rec_bytes,
                "band_score_sweep": sweep(ssb.GStore(Wb, ssb.G_SN16, S, rows, band_compact=True), bb16)}
            del W, S, Wb, st
        # per-BF phase moments (the exact mean(angle) path) from the complex64
        # half plane: G read once, every corrected plane through L2
        mom_mean = torch.empty((n, n), dtype=torch.float32, device=dev)
        mom_var = torch.empty((n, n), dtype=torch.float32, device=dev)
        ws_m = ssb.Workspace(ssb.workspace_bytes(geom, n_bf, ssb.OP_MOMENTS), dev)
        t_mom = timed(lambda: ssb.phase_moments(G, geom, bfd, ab, mean=mom_mean, var=mom_var, ws=ws_m,
                                                stream=stream), reps=5)
        gb = entries * 8
        compact["phase_moments"] = {"ms": t_mom, "G_GBs": gb / (t_mom * 1e-3) / 1e9,
                                    "G_hbm_frac": gb / (t_mom * 1e-3) / 1e9 / hbm,
                                    "atan2_per_s": n_bf * n * n / (t_mom * 1e-3),
                                    "planes_per_s": n_bf / (t_mom * 1e-3)}
        del ws_m
        torch.cuda.synchronize()

    stage_rooflines = {
        "reconstruct": {"bound": "hbm", "achieved": bytes_recon / (recon_ms * 1e-3) / 1e9, "peak": hbm,
                        "unit": "GB/s", "frac": bytes_recon / (recon_ms * 1e-3) / 1e9 / hbm,
                        "algorithmic_bytes": bytes_recon},
        "score": {"bound": "xu", "achieved": xu_ach / 1e9, "peak": xu_peak / 1e9, "unit": "Gop/s",
                  "frac": xu_ach / xu_peak, "ops": 2 * terms,
                  "peak_source": "measured in this run: ssb_peak_sincos (8 independent __sincosf chains per "
                                 f"thread, {rates['blocks']} CTAs x 256 threads)",
                  "derived_peak": 16.0 * sms * clk_mhz * 1e6 / 1e9,
                  "derived_source": f"16 sin/cos per clock per SM x {sms} SMs x {clk_mhz:.0f} MHz",
                  "hbm_frac": bytes_score / (score_ms * 1e-3) / 1e9 / hbm},
        "build_fp32": {"bound": "fp32 (context)", "peak": fp32_peak / 1e12, "unit": "TFLOP/s",
                       "peak_source": "measured in this run: ssb_peak_fma (8 independent FMA chains per thread)"},
    }

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": ms_step, "unit": "ms", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {n}^2 scan, {geom.det_y}^2 uint16 detector, {n_bf} BF px, "
                               f"band {nq} q, {B} sets",
                   "step": "ssb_build_G + ssb_reconstruct + ssb_score_batch(B=8)",
                   "l2": "inputs larger than L2 (frames %.1f GB, G %.2f GB); no flush" % (
                       frames.numel() * frames.element_size() / 1e9, n_bf * n * h * 8 / 1e9),
                   "parallelism": f"replicas x{ws}"},
        "stages": {"build_ms": build_ms, "build_GBs": achieved, "recon_ms": recon_ms,
                   "recon_GBs": bytes_recon / (recon_ms * 1e-3) / 1e9,
                   "score_ms": score_ms, "score_GBs": bytes_score / (score_ms * 1e-3) / 1e9,
                   "score_terms": terms, "score_terms_per_s": terms / (score_ms * 1e-3),
                   "max_count": d.get("max_count")},
        "stage_rooflines": stage_rooflines,
        "score_sweep": score_sweep,
        "score_depth": score_depth,
        "compact": compact,
        "roofline": {"bound": "hbm", "kernel": "ssb_build_G = ssb_gather + ssb_plane512<8> on two internal streams (one C-ABI call, timed on the caller's stream)", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                     "peak_source": peak_src, "algorithmic_bytes": bytes_build},
        "clocks": clk, "gpu_launches": launches, "wall_s_timed": t_wall,
        "e2e": e2e, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    ws, rank, local, pg = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, ws, rank)
        return run_ours(args, ws, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
