"""Benchmark of the sparse-KV reuse decode step on GB300.

One step = match + reservation + miss gather + attention for every unit of a
workload, through the C interface.  The headline workload is the largest one
that fits one GPU: 16-token head-wise pages, 32 requests x 8 kv-heads, GQA 4,
L = 131072 tokens (8192 pages), k = 128 pages, B = 512 page slots (~17 GB of
pinned host KV).  The other workloads (tiny, batch, multi-token prediction,
the million-token latent cache at four buffer sizes) are measured in the same
run and reported as sub-objects of the same JSON line.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload pages|batch|tiny|mtp|latent] [--slots B] [--no-others]

Units (request, kv-head) are independent, so N GPUs run N ranks, each with its
own contiguous range of requests (weak scaling: rank r holds requests
[r*R, (r+1)*R) of an N*R-request job, its host KV in the memory of its GPU's
NUMA node); there is no collective on the data path.  value = selected
entries of all ranks / the slowest rank's time.  `python bench.py --gpus N`
starts the N ranks itself; under torchrun it is one rank.

The timed pass runs the steps as they are served (captured step graphs, the
kernels of a step overlapping on three streams).  A second pass over the same
steps, with the library's events between kernels, enqueues each step on one
stream and gives every kernel's own time, for the per-kernel roofline figures.
"""
from __future__ import annotations

import argparse
import json
import os
import socket
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode steps/s & selected-KV entries/s per GB300; miss-gather GB/s vs pinned H2D"
FLUSH_BYTES = 256 << 20  # > 129 MB L2: written between timed steps
HEADLINE = "pages"
# the other workloads, in the same run: (name, slots override)
OTHERS = [("tiny", 0), ("batch", 0), ("mtp", 0), ("latent", 2048), ("latent", 4096),
          ("latent", 8192), ("latent", 16384)]


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--slots", type=int, default=0, help="override B (latent sweep)")
    ap.add_argument("--no-others", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ceilings", action="store_true")
    ap.add_argument("--skip-no-reuse", action="store_true",
                    help="skip the no-reuse and request-assignment passes (profiling runs)")
    ap.add_argument("--_dry", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def workload_for(name, slots=0):
    import workload as W
    w = W.get_workload(name)
    if slots:
        w = w.replace(slots=slots)
    return w


def describe(w) -> dict:
    return {"workload": f"{w.name}: {w.requests}x{w.kv_heads} units, GQA {w.q_per_kv}, "
                        f"L={w.context}, D={w.head_dim}, entry={w.entry_tokens} tok, "
                        f"k={w.k}, B={w.slots}, tokens/step={w.tokens_per_step}",
            "units": w.units, "k": w.k, "slots": w.slots, "context": w.context,
            "head_dim": w.head_dim, "q_per_kv": w.q_per_kv, "entry_tokens": w.entry_tokens,
            "tokens_per_step": w.tokens_per_step, "kv_shared": w.kv_shared,
            "l2": "flushed between timed steps (256 MiB write)",
            "timing": "CUDA events around each step on the launch stream, summed"}


# --------------------------------------------------------------- ranks
def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(args, argv) -> int:
    """Starts args.gpus copies of this script as ranks 0..N-1 (one per GPU,
    rendezvous on 127.0.0.1) and returns the largest exit code."""
    port = free_port()
    procs = []
    for r in range(args.gpus):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(args.gpus),
                   LOCAL_WORLD_SIZE=str(args.gpus), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + argv, env=env))
    return max(p.wait() for p in procs)


def rank_units(w, rank: int) -> int:
    """First unit of a rank's contiguous request range (weak scaling)."""
    return rank * w.units


def gpu_pci_id(torch, index: int):
    """PCI address of a CUDA device (domain:bus:device.function, as nvidia-smi
    prints it), or None."""
    p = torch.cuda.get_device_properties(index)
    dom, bus, dev = (getattr(p, a, None) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id"))
    if bus is None or dev is None:
        return None
    return f"{dom or 0:08x}:{bus:02x}:{dev:02x}.0"


def numa_node_of_gpu(pci):
    """NUMA node the GPU's PCI device reports (sysfs), or None."""
    if not pci:
        return None
    try:
        node = int(open(f"/sys/bus/pci/devices/{pci[4:]}/numa_node").read().strip())
    except (OSError, ValueError):
        return None
    return node if node >= 0 else None


def bind_to_numa(pci) -> dict:
    """Moves this process onto the CPUs of its GPU's NUMA node, so the pinned
    host KV it allocates (first touch) lands in that node's memory."""
    node = numa_node_of_gpu(pci)
    if node is None:
        return {"node": None, "cpus": None}
    try:
        text = open(f"/sys/devices/system/node/node{node}/cpulist").read().strip()
    except OSError:
        return {"node": node, "cpus": None}
    cpus = set()
    for part in text.split(","):
        if "-" in part:
            a, b = part.split("-")
            cpus.update(range(int(a), int(b) + 1))
        elif part:
            cpus.add(int(part))
    if not cpus:  # a memory-only node
        return {"node": node, "cpus": None}
    os.sched_setaffinity(0, cpus)
    return {"node": node, "cpus": len(cpus)}


# --------------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index  # nvidia-smi -i: a PCI address (or an index)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- our arm
def pinned_h2d_peak_gbs(torch) -> float:
    """Best of 5 cudaMemcpyAsync of 256 MiB from pinned host memory."""
    n = 256 << 20
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = max(best, n / (a.elapsed_time(b) * 1e-3) / 1e9)
    return best


def read_ceilings(torch, row_sizes_hbm, row_sizes_host) -> dict:
    """Read rate (GB/s) of rows at uniformly random positions, the step's row
    reads with nothing else in the way (avsg_read_rows): device rows over a
    4 GiB region, host rows over a 2 GiB mapped pinned region; best of two
    grid sizes and three runs each, the L2 flushed before each run."""
    from decode_serving_gb300 import avsg
    dev = torch.device("cuda")
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(4, dtype=torch.int32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    st = torch.cuda.current_stream()
    gen = torch.Generator(device=dev)
    gen.manual_seed(0x5EED)

    def rate(src, nrows, rb, nbytes):
        n = max(1, nbytes // rb)
        idx = torch.randint(0, nrows, (n,), dtype=torch.int32, device=dev, generator=gen)
        best = float("inf")
        for per_sm in (4, 8):
            for r in range(3):
                flush.fill_(r)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(st)
                avsg.avsg_read_rows(src, nrows, rb, idx.data_ptr(), n, sink.data_ptr(),
                                    per_sm * sms, st.cuda_stream)
                b.record(st)
                torch.cuda.synchronize()
                best = min(best, a.elapsed_time(b))
        return n * rb / (best * 1e-3) / 1e9

    out = {"hbm_gbs": {}, "host_gbs": {}}
    region = torch.empty(4 << 30, dtype=torch.uint8, device=dev)
    for rb in row_sizes_hbm:
        out["hbm_gbs"][str(rb)] = rate(region.data_ptr(), region.numel() // rb, rb, 256 << 20)
    del region
    torch.cuda.empty_cache()
    hb = 2 << 30
    ptr = avsg.avsg_host_alloc(hb)
    try:
        import ctypes
        ctypes.memset(ptr, 0x3C, hb)
        # one address for host and device: a mapped allocation under unified addressing
        for rb in row_sizes_host:
            out["host_gbs"][str(rb)] = rate(ptr, hb // rb, rb, 64 << 20)
    finally:
        avsg.avsg_host_free(ptr)
    out["how"] = ("avsg_read_rows over uniformly random row indices; device rows from a 4 GiB "
                  "region (256 MiB read), host rows from 2 GiB of mapped pinned memory (64 MiB read)")
    return out


def algorithmic_bytes(w, hits, misses, steps, num_sms=152) -> dict:
    """Bytes each kernel must move per launch (averaged over the timed steps).

    attention: slot id + K row + V row per selected entry, plus q and out
           (both passes together);
    match: id (4) + one 32-byte probe window (two 16-byte hash cells) +
           slot map (4) + hit-slot list (4) + hit flag (1) per selected id,
           + 8 per distinct miss (miss-set cell) + the hit bitmaps (1 bit per
           slot) + q read and copied;
    victims: tag and last_step (8 bytes) per slot + the hit bitmaps, + 40 per
           miss (miss-set cell, descriptor, last_step, cell -> slot, marker);
    commit: the slot map read (4 per selected id), + 112 per miss
           (descriptor, evicted and new tag, cell -> slot, slot map write,
           evicted-id and new-id probe windows);
    gather: one entry (K + V) per miss, read over the host link and written
           to HBM (host-link bytes are the read half);
    finish: the partials it merges (about 2 * SMs / pairs hit-pass partials
           and one miss-pass partial per pair) and the output;
    place: one entry per miss read from the staging area and written to its
           slot."""
    U, n_tok, k = w.units, w.tokens_per_step, w.k
    sel = U * n_tok * k
    miss_ps = misses / steps
    row_b = w.entry_k_bytes + w.entry_v_bytes
    attn = sel * 4 + sel * row_b + U * n_tok * w.q_per_kv * (w.head_dim + w.v_dim) * 4
    q_bytes = U * n_tok * w.q_per_kv * w.head_dim * 4
    match = sel * (4 + 32 + 4 + 4 + 1) + miss_ps * 8 + U * n_tok * w.slots / 8 + 2 * q_bytes
    victims = U * w.slots * 8 + U * n_tok * w.slots / 8 + miss_ps * 40
    gather_host = miss_ps * w.entry_bytes
    commit = sel * 4 + miss_ps * 112
    return {"attention": attn, "match": match, "victims": victims, "gather": 2 * gather_host,
            "gather_host_link": gather_host, "commit": commit,
            "finish": U * n_tok * (max(1, 2 * num_sms // (U * n_tok)) + 1) * w.q_per_kv
            * (w.v_dim + 2) * 4 + U * n_tok * w.q_per_kv * w.v_dim * 4,
            "place": 2 * gather_host}


def measure(args, w, rank, world, torch, steps, warmup, full):
    """Runs one workload on this rank's units: the timed pass (served as in
    use), the per-kernel pass, the no-reuse pass, and, when `full`, the e2e
    pass through the host-buffer entry point and the request-level gather."""
    import workload as W
    from decode_serving_gb300.session import PinnedArray, Session, make_config

    dev = torch.device("cuda", torch.cuda.current_device())
    total = warmup + steps
    ub = rank_units(w, rank)
    t0 = time.time()
    sel = W.selections(w, total, unit_base=ub)
    q = W.queries(w, total, unit_base=ub, units_total=world * w.units)
    hk = PinnedArray(W.host_kv_shape(w), np.uint16)
    hv = None if w.kv_shared else PinnedArray((w.units, w.num_entries, w.entry_tokens * w.v_dim),
                                              np.uint16)
    W.fill_host_kv(w, hk.array, hv.array if hv is not None else None, unit_base=ub)
    gen_s = time.time() - t0
    sel_d = torch.from_numpy(sel).to(dev)
    q_d = torch.from_numpy(q).to(dev)
    out = torch.empty((w.units, w.tokens_per_step, w.q_per_kv, w.v_dim), dtype=torch.float32,
                      device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def make(no_reuse=False, request_gather=False):
        cfg = make_config(w.requests, w.kv_heads, w.q_per_kv, w.num_entries, w.head_dim, w.v_dim,
                          w.slots, w.k, entry_tokens=w.entry_tokens, kv_shared=w.kv_shared,
                          max_tokens_per_step=w.tokens_per_step, no_reuse=no_reuse,
                          request_gather=request_gather)
        return Session(cfg, hk.ptr, hv.ptr if hv is not None else None)

    def timed_pass(sess, n_steps, profile, sample_clocks=True):
        for t in range(warmup):
            sess.step(t, sel_d[t], q_d[t], out, stream=sptr)
            flush.fill_(t & 0xFF)
        torch.cuda.synchronize()
        st0 = sess.stats()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clocks = ClockSampler(gpu_pci_id(torch, torch.cuda.current_device())
                              or torch.cuda.current_device())
        if sample_clocks:
            clocks.start()
        if profile:
            sess.profile(True)
        wall0 = time.perf_counter()
        for i in range(n_steps):
            t = warmup + i
            flush.fill_(t & 0xFF)
            evs[i][0].record(stream)
            sess.step(t, sel_d[t], q_d[t], out, stream=sptr)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        if world > 1:
            torch.distributed.barrier()
        ck = clocks.stop() if sample_clocks else None
        per = np.array([a.elapsed_time(b) for a, b in evs])
        prof = sess.profile_read() if profile else None
        if profile:
            sess.profile(False)
        st1 = sess.stats()
        return per, wall, prof, ck, st0, st1

    sess = make()
    info = sess.info()
    # the per-kernel pass first: the served pass then runs on a host store the
    # device has already read from (the first steps after a store is created
    # pay for first accesses to it)
    per_prof, _, prof, _, _, _ = timed_pass(sess, steps, True, sample_clocks=False)
    sess.reset()
    per, wall, _, clocks, st0, st1 = timed_pass(sess, steps, False, sample_clocks=full)
    assert st1.device_error == 0, st1.device_error
    hits, misses = st1.hits - st0.hits, st1.misses - st0.misses
    res = {"w": w, "steps": steps, "warmup": warmup, "gen_s": gen_s,
           "launches_per_step": sum(n for _, n in prof.values()) / max(1, steps),
           "host_us_per_step": 1e6 * wall / steps,
           "per_step_ms": per, "ms_per_step": float(per.sum() / steps), "wall_s": wall,
           "prof": prof, "ms_per_step_profiled": float(per_prof.sum() / steps),
           "clocks": clocks, "hits": hits, "misses": misses, "unique": hits + misses,
           "hit_rate_all": st1.hits / max(1, st1.unique_selected), "info": info}

    if full and not args.no_e2e:  # end to end through the host-buffer entry point
        sess.reset()
        sel_h = PinnedArray(sel.shape[1:], np.int32)
        q_h = PinnedArray(q.shape[1:], np.float32)
        out_h = PinnedArray(tuple(out.shape), np.float32)
        for t in range(warmup):
            sess.step(t, sel_d[t], q_d[t], out, stream=sptr)
        torch.cuda.synchronize()
        e2e_ms = 0.0
        for i in range(steps):
            t = warmup + i
            sel_h.array[...] = sel[t]
            q_h.array[...] = q[t]
            flush.fill_(t & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sess.step_host(t, sel_h.array, q_h.array, out_h.array, stream=sptr)
            b.record(stream)
            b.synchronize()
            e2e_ms += a.elapsed_time(b)
        res["e2e_ms"] = e2e_ms / steps
        res["e2e_h2d"] = sel[0].nbytes + q[0].nbytes
        res["e2e_d2h"] = out_h.array.nbytes
        for p in (sel_h, q_h, out_h):
            p.free()
    sess.close()

    # transfer assignment (AVSG page: even split of the miss transfers across
    # cores against request-level assignment): the same steps with one gather
    # CTA per request, the gather timed by the library's events as above
    res["assign"] = None
    if full and not args.skip_no_reuse:
        try:
            sess = make(request_gather=True)
        except Exception as exc:  # a shape without the staged gather
            res["assign"] = {"unavailable": str(exc)}
        else:
            a_steps = min(steps, 300)
            info_r = sess.info()
            _, _, prof_r, _, s0, s1 = timed_pass(sess, a_steps, True, sample_clocks=False)
            sess.close()
            res["assign"] = {"request": prof_r.get("gather"), "request_ctas": info_r.gather_ctas,
                             "request_misses": s1.misses - s0.misses, "steps": a_steps,
                             "even_ctas": info.gather_ctas}

    # no-reuse comparison: every selected row crosses the host link each step
    res["no_reuse_ms_per_step"] = None
    if not args.skip_no_reuse:
        nr_steps = min(steps, 200)
        sess = make(no_reuse=True)
        per_nr, _, _, _, _, _ = timed_pass(sess, nr_steps, False, sample_clocks=False)
        sess.close()
        res["no_reuse_ms_per_step"] = float(per_nr.sum() / nr_steps)
    hk.free()
    if hv is not None:
        hv.free()
    del sel_d, q_d, flush
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------- CPU oracle (baseline arm)
def _oracle_worker(name, slots, u0, u1, warmup, steps, budget_s):
    """One pool worker: the oracle (match, reservation, row copies, fp64
    attention) over units [u0, u1) of the workload, warmup untimed steps then
    up to `steps` timed steps or `budget_s` seconds."""
    import oracle
    import workload as W
    w = workload_for(name, slots)
    part = w.replace(requests=1, kv_heads=u1 - u0)  # the worker's units, drawn as [u0, u1)
    total = warmup + steps
    sel = W.selections(part, total, unit_base=u0)
    q = W.queries(part, total, unit_base=u0, units_total=w.units)
    hk = np.empty(W.host_kv_shape(part), np.uint16)
    hv = None if w.kv_shared else np.empty((part.units, w.num_entries, w.entry_tokens * w.v_dim),
                                           np.uint16)
    W.fill_host_kv(part, hk, hv, unit_base=u0)
    run = oracle.OracleRun(w.slots, hk, hv, w.head_dim, w.v_dim, w.softmax_scale)
    for t in range(warmup):
        run.step(t, sel[t], q[t])
    t0 = time.perf_counter()
    done = 0
    for t in range(warmup, total):
        run.step(t, sel[t], q[t])
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return {"seconds": el, "steps": done, "units": u1 - u0,
            "entries": done * (u1 - u0) * w.tokens_per_step * w.k}


def oracle_pool(name, slots, warmup, steps, budget_s) -> dict:
    """The oracle over every unit of a workload, units split into contiguous
    ranges over a process pool with one single-threaded worker per host core.
    Workers run side by side; the rate is the sum of their rates."""
    import multiprocessing as mp
    w = workload_for(name, slots)
    cores = os.cpu_count() or 1
    n = max(1, min(cores, w.units))
    bounds = [(i * w.units // n, (i + 1) * w.units // n) for i in range(n)]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                            "MKL_NUM_THREADS", "WORKLOAD_THREADS")}
    os.environ.update(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
                      WORKLOAD_THREADS="1")
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            parts = pool.starmap(_oracle_worker, [(name, slots, a, b, warmup, steps, budget_s)
                                                  for a, b in bounds])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    rate = sum(p["entries"] / p["seconds"] for p in parts if p["seconds"] > 0)
    step_s = max(p["seconds"] / max(1, p["steps"]) for p in parts)
    return {"entries_per_s": rate, "workers": n, "cores": cores, "ms_per_step": 1e3 * step_s,
            "steps": min(p["steps"] for p in parts), "seconds": max(p["seconds"] for p in parts),
            "units": w.units}


def cpu_baseline(args) -> dict:
    w = workload_for(args.workload, args.slots)
    r = oracle_pool(args.workload, args.slots, 0, w.steps, 15.0)
    return {"value": r["entries_per_s"], "unit": "selected entries/s", "cores": r["workers"],
            "kind": "oracle",
            "sample": f"all {w.units} units, steps 0..{r['steps'] - 1} or more from a cold buffer "
                      f"(15 s per worker), {r['workers']} single-threaded worker processes on "
                      f"{r['cores']} host cores, units split into contiguous ranges",
            "steps_per_s_full_batch": r["entries_per_s"] / (w.units * w.tokens_per_step * w.k)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = workload_for(args.workload, args.slots)
    r = oracle_pool(args.workload, args.slots, args.warmup, args.steps, 120.0)
    v = r["entries_per_s"]
    sample = (f"every unit of the workload ({w.units}), the whole hot path per unit (match, "
              f"reservation, row copies, fp64 attention), {r['steps']}+ timed steps after "
              f"{args.warmup} warm-up steps, {r['workers']} single-threaded worker processes "
              f"on {r['cores']} host cores")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "selected entries/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": r["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": describe(w),
            "cpu_baseline": {"value": v, "unit": "selected entries/s", "cores": r["workers"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "selected entries/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# --------------------------------------------------------------------- report
def measured_peaks() -> tuple:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "of measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "of fallback"


def ncu_traffic() -> dict:
    """DRAM bytes per launch from the committed ncu summary, keyed by
    (workload, kernel); an entry is used only while its kernel source is
    unchanged."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return out
    for ln in lines:
        f = ln.split()
        if len(f) != 5 or f[0].startswith("#"):
            continue
        wl, name, src, digest, nbytes = f
        try:
            h = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
        except OSError:
            continue
        if h == digest:
            out[(wl, name)] = float(nbytes)
    return out


def transfer_assignment(res, w, kernels):
    """Effective host-link bandwidth of the miss gather (miss bytes / gather
    time) with the even split over CTAs and with one CTA per request."""
    a = res.get("assign")
    if not a or "unavailable" in a or not a.get("request") or not a["request"][1]:
        return a
    even = kernels.get("gather")
    ms_total, n = a["request"]
    req_us = ms_total / n * 1e3
    req_bytes = a["request_misses"] / a["steps"] * w.entry_bytes
    req_gbs = req_bytes / (req_us * 1e-6) / 1e9
    out = {"request": {"ctas": a["request_ctas"], "gather_us": req_us, "gbs": req_gbs},
           "even": None, "even_over_request": None}
    if even:
        out["even"] = {"ctas": a["even_ctas"], "gather_us": even["avg_us"], "gbs": even["achieved"]}
        out["even_over_request"] = even["achieved"] / req_gbs if req_gbs else None
    return out


def kernel_table(res, h2d_peak, ceilings):
    """Per-kernel average time, algorithmic GB/s and roofline fractions."""
    w = res["w"]
    hbm_peak, peak_kind = measured_peaks()
    ab = algorithmic_bytes(w, res["hits"], res["misses"], res["steps"], res["info"].num_sms)
    traffic = ncu_traffic()
    kernels = {}
    prof = dict(res["prof"])
    passes = {}
    if prof.get("attention_miss", (0, 0))[1]:
        # two attention passes (hit rows beside the gather, then miss rows):
        # the attention roofline takes both launches of a step together
        (ha, hn), (ma, mn) = prof["attention"], prof.pop("attention_miss")
        prof["attention"] = (ha + ma, hn)
        passes = {"hit_pass_us": 1e3 * ha / hn, "miss_pass_us": 1e3 * ma / mn}
    row_ceiling = None
    if ceilings:
        row_ceiling = ceilings["hbm_gbs"].get(str(w.entry_k_bytes))
    for name, (ms_total, n) in prof.items():
        if not n or name not in ab:
            continue
        avg = ms_total / n
        if name == "gather":
            ach = ab["gather_host_link"] / (avg * 1e-3) / 1e9
            kernels[name] = {"bound": "host_link", "avg_us": avg * 1e3, "achieved": ach,
                             "peak": h2d_peak, "unit": "GB/s", "frac": ach / h2d_peak,
                             "peak_kind": "pinned cudaMemcpy H2D measured in this run",
                             "algorithmic_bytes": ab["gather_host_link"]}
            if ceilings and str(w.entry_k_bytes) in ceilings["host_gbs"]:
                c = ceilings["host_gbs"][str(w.entry_k_bytes)]
                kernels[name]["random_row_ceiling_gbs"] = c
                kernels[name]["frac_of_random_row_ceiling"] = ach / c
        else:
            ach = ab[name] / (avg * 1e-3) / 1e9
            kernels[name] = {"bound": "hbm", "avg_us": avg * 1e3, "achieved": ach, "peak": hbm_peak,
                             "unit": "GB/s", "frac": ach / hbm_peak, "peak_kind": peak_kind,
                             "algorithmic_bytes": ab[name],
                             "traffic": traffic.get((w.name, name))}
            if name == "attention" and row_ceiling:
                kernels[name]["random_row_ceiling_gbs"] = row_ceiling
                kernels[name]["frac_of_random_row_ceiling"] = ach / row_ceiling
            if name == "attention":
                kernels[name].update(passes)
    total_k = sum(v["avg_us"] for v in kernels.values())
    for v in kernels.values():
        v["share"] = v["avg_us"] / total_k if total_k else None
    return kernels, ab


def summarize(res, world, max_ms, h2d_peak, ceilings) -> dict:
    """The figures of one workload: latency, rates, hit rate, gather and
    attention rooflines, the host-link floor and the no-reuse comparison."""
    w = res["w"]
    kernels, ab = kernel_table(res, h2d_peak, ceilings)
    per = res["per_step_ms"]
    sel_step = w.units * w.tokens_per_step * w.k
    hbm_kernels = [n for n in ("match", "victims", "attention") if n in kernels]
    hbm_bytes = sum(ab[n] for n in hbm_kernels)
    hbm_us = sum(kernels[n]["avg_us"] for n in hbm_kernels)
    hbm_peak, peak_kind = measured_peaks()
    floor_us = ab["gather_host_link"] / (h2d_peak * 1e3) if h2d_peak else None
    att = kernels.get("attention", {})
    out = {
        "config": describe(w),
        "us_per_step": 1e3 * max_ms,
        "step_latency_us": {"median": 1e3 * float(np.median(per)),
                            "p99": 1e3 * float(np.percentile(per, 99)),
                            "max": 1e3 * float(per.max()),
                            "steps_over_1.5x_median": int((per > 1.5 * np.median(per)).sum())},
        "steps_per_s": 1e3 / max_ms,
        "selected_entries_per_s": world * sel_step * 1e3 / max_ms,
        "hit_rate": {"timed_steps": res["hits"] / max(1, res["unique"]),
                     "all_steps": res["hit_rate_all"]},
        "miss_gather": {"bytes_per_step": ab["gather_host_link"],
                        "gbs": kernels.get("gather", {}).get("achieved"),
                        "pinned_h2d_peak_gbs": h2d_peak,
                        "frac": kernels.get("gather", {}).get("frac"),
                        "frac_of_random_row_ceiling":
                            kernels.get("gather", {}).get("frac_of_random_row_ceiling")},
        "attention_hbm": {"gbs": att.get("achieved"), "frac": att.get("frac"),
                          "peak_kind": peak_kind,
                          "frac_of_random_row_ceiling": att.get("frac_of_random_row_ceiling")},
        "match_victims_attention_hbm": {
            "gbs": hbm_bytes / (hbm_us * 1e-6) / 1e9 if hbm_us else None,
            "frac": (hbm_bytes / (hbm_us * 1e-6) / 1e9) / hbm_peak if hbm_us else None},
        "link_floor": {"us": floor_us,
                       "step_over_floor": (1e3 * max_ms / floor_us) if floor_us else None,
                       "how": "miss bytes per step / pinned cudaMemcpy H2D peak"},
        "no_reuse": None if res["no_reuse_ms_per_step"] is None else {
            "us_per_step": 1e3 * res["no_reuse_ms_per_step"],
            "steps_per_s": 1e3 / res["no_reuse_ms_per_step"],
            "reuse_speedup": res["no_reuse_ms_per_step"] / max_ms},
        "kernels": kernels,
        "gpu_launches_per_step": res["launches_per_step"],
    }
    return out


def report_headline(args, res, world, max_ms, max_e2e_ms, h2d_peak, ceilings) -> dict:
    w = res["w"]
    K = args.steps
    summary = summarize(res, world, max_ms, h2d_peak, ceilings)
    kernels = summary["kernels"]
    att = kernels.get("attention")
    roof = None
    if att:
        roof = {"kernel": "attention", "bound": "hbm", "achieved": att["achieved"],
                "peak": att["peak"], "unit": "GB/s", "frac": att["frac"],
                "traffic": att.get("traffic"), "peak_kind": att["peak_kind"],
                "random_row_ceiling_gbs": att.get("random_row_ceiling_gbs"),
                "frac_of_random_row_ceiling": att.get("frac_of_random_row_ceiling")}
    g = kernels.get("gather")
    sel_step = w.units * w.tokens_per_step * w.k
    line = {
        "metric": METRIC, "value": summary["selected_entries_per_s"], "unit": "selected entries/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": max_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 K/V, fp32 accumulate", "data": "synthetic (seeded generator)",
        "config": summary["config"],
        "steps_per_s": summary["steps_per_s"],
        "step_latency_ms": {k: v / 1e3 for k, v in summary["step_latency_us"].items()},
        "host_wall_us_per_step": res["host_us_per_step"],
        "hit_rate": summary["hit_rate"], "miss_gather": summary["miss_gather"],
        "attention_hbm": summary["attention_hbm"],
        "match_victims_attention_hbm": summary["match_victims_attention_hbm"],
        "link_floor": summary["link_floor"],
        "transfer_assignment": transfer_assignment(res, w, kernels),
        "no_reuse": summary["no_reuse"],
        "roofline": roof,
        "host_link_roofline": None if not g else {
            "kernel": "gather", "bound": "host_link", "achieved": g["achieved"],
            "peak": g["peak"], "unit": "GB/s", "frac": g["frac"], "peak_kind": g["peak_kind"],
            "random_row_ceiling_gbs": g.get("random_row_ceiling_gbs"),
            "frac_of_random_row_ceiling": g.get("frac_of_random_row_ceiling")},
        "kernels": kernels,
        "kernel_timing": ("second pass over the same steps with library CUDA events between "
                          "kernels, each step on one stream (every kernel timed alone); that "
                          f"pass's ms_per_step: {res['ms_per_step_profiled']:.4f}"),
        "gpu_launches": int(round(res["launches_per_step"] * K)),
        "clocks": res["clocks"],
    }
    if max_e2e_ms is not None:
        line["e2e"] = {"value": world * sel_step * 1e3 / max_e2e_ms, "unit": "selected entries/s",
                       "h2d_bytes_per_step": res["e2e_h2d"], "d2h_bytes_per_step": res["e2e_d2h"],
                       "ms_per_step": max_e2e_ms, "entry_point": "avsg_step_host"}
    return line


def slowest_rank(torch, ms_per_step, e2e_ms, world, device):
    """Step time of the slowest rank (max over ranks); e2e likewise (None stays None)."""
    t = torch.tensor([ms_per_step, e2e_ms if e2e_ms is not None else 0.0], dtype=torch.float64,
                     device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t[0]), (float(t[1]) if e2e_ms is not None else None)


def whole_job_value(w, world, max_ms) -> float:
    """Selected entries of all ranks per second: every rank runs its own
    range of requests (units shard across GPUs with no exchange), so a step
    of the job is `world` ranges in the slowest rank's step time."""
    return world * w.units * w.tokens_per_step * w.k * 1e3 / max_ms


def dry_rank(args, rank, world):
    """The multi-rank path without a GPU (gloo): each rank takes its own
    request range, runs the oracle's state machine over it for the given
    steps, and the slowest rank's time makes the whole-job value."""
    import torch
    import oracle
    import workload as W
    if world > 1:
        torch.distributed.init_process_group("gloo")
    w = workload_for(args.workload, args.slots)
    ub = rank_units(w, rank)
    sel = W.selections(w, args.warmup + args.steps, unit_base=ub)
    hk = np.empty(W.host_kv_shape(w), np.uint16)
    hv = None if w.kv_shared else np.empty((w.units, w.num_entries, w.entry_tokens * w.v_dim),
                                           np.uint16)
    W.fill_host_kv(w, hk, hv, unit_base=ub)
    run = oracle.OracleRun(w.slots, hk, hv, w.head_dim, w.v_dim, w.softmax_scale)
    for t in range(args.warmup):
        run.step(t, sel[t], None, attention=False)
    t0 = time.perf_counter()
    for t in range(args.warmup, args.warmup + args.steps):
        run.step(t, sel[t], None, attention=False)
    ms = 1e3 * (time.perf_counter() - t0) / max(1, args.steps)
    t = torch.tensor([ms], dtype=torch.float64)
    units = torch.tensor([ub, ub + w.units], dtype=torch.int64)
    gathered = [torch.zeros(2, dtype=torch.int64) for _ in range(world)]
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_gather(gathered, units)
    else:
        gathered = [units]
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": world, "ms_per_step": float(t[0]),
                          "value": whole_job_value(w, world, float(t[0])),
                          "unit": "selected entries/s (oracle state machine, CPU)",
                          "rank_units": [g.tolist() for g in gathered]}), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse(argv)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        sys.exit(launch_ranks(args, argv))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args._dry:
        dry_rank(args, rank, world)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    numa = bind_to_numa(gpu_pci_id(torch, local))
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    __graft_entry__.build()
    h2d_peak = pinned_h2d_peak_gbs(torch)
    w = workload_for(args.workload, args.slots)
    ceilings = None
    if not args.no_ceilings and world == 1:
        ceilings = read_ceilings(torch, sorted({256, 512, 1152, 4096, 8192, w.entry_k_bytes}),
                                 sorted({512, 1152, 4096, 8192, w.entry_k_bytes}))
    res = measure(args, w, rank, world, torch, args.steps, args.warmup, full=True)
    h2d_after = pinned_h2d_peak_gbs(torch)  # a lower figure than before: the link was shared
    max_ms, max_e2e = slowest_rank(torch, res["ms_per_step"], res.get("e2e_ms"), world, "cuda")
    line = None
    if rank == 0:
        line = report_headline(args, res, world, max_ms, max_e2e, h2d_peak, ceilings)
        line["numa"] = numa
        line["pinned_h2d_gbs"] = {"before": h2d_peak, "after_headline": h2d_after,
                                  "how": "best of 5 cudaMemcpyAsync of 256 MiB from pinned memory"}
        if ceilings:
            line["read_ceilings"] = ceilings
    if world == 1 and not args.no_others:
        others = {}
        for name, slots in OTHERS:
            if name == w.name and (slots or w.slots) == w.slots:
                continue
            wo = workload_for(name, slots)
            key = f"{name}_B{wo.slots}" if name == "latent" else name
            r = measure(args, wo, rank, world, torch, min(args.steps, wo.steps) if name != "tiny"
                        else wo.steps, args.warmup, full=False)
            others[key] = summarize(r, world, r["ms_per_step"], h2d_peak, ceilings)
        line["other_workloads"] = others
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
