#!/usr/bin/env python
"""Throughput benchmark of the verify / overlap / E2E-TV hot path.

One *step* is one pass of the whole hot path over one batch of the
entropy-mix workload (B=32 rows, K=4 drafted positions, V=151936, bf16
logits, per-row sigma in {1, 2, 4}, draft = target + N(0, 0.7^2)):

  verify at T=1.0, verify at T=0.7 (both with per-position overlap),
  greedy verify at T=0, and the E2E-TV loss + draft-logit gradient at T=1.0.

Metric: verified draft positions ("rows") per second, B*K per verify call,
three verify calls per step; the E2E-TV call adds time but no rows.  Inputs
are resident in HBM and rotated over 8 copies of the batch (700 MB, above
the 129 MB L2), so every call reads its logits from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Prints ONE JSON line (rank 0).  Under torchrun each rank runs its own batch
(batch rows are independent: weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

B, K, V = 32, 4, 151936
SEED = 1235
TEMPS = (1.0, 0.7, 0.0)
N_ROT = 8
METRIC = "verify rows/s (B*K*V logits) and achieved HBM GB/s vs 8 TB/s roofline"
WORKLOAD = "entropy-mix verify step: B=32, K=4, V=151936 bf16, T in {1.0, 0.7, 0 greedy} + E2E-TV fwd+bwd at T=1"
L2_NOTE = "inputs rotated over 8 resident copies of the batch (700 MB > 129 MB L2)"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--single", choices=["verify", "greedy", "overlap", "e2e", "diag", "truncate", "ragged",
                                         "schedule", "relaxed", "tree"], default=None,
                    help="run only `--calls` calls of one entry point (an L2 flush before each): the "
                         "profiling target, prints no JSON")
    ap.add_argument("--shape", default="32,4,151936", help="B,K,V of --single")
    ap.add_argument("--temperature", type=float, default=1.0, help="T of --single verify")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--sweep", action="store_true",
                    help="time verify at B in {1,8,32,64,128,256} x K in {1,2,4,7,16}, V=151936 (one line per point)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def job_rate(ms_total_max, steps, ws, rows_per_step):
    """Whole-job rows/s: every rank verifies rows_per_step rows per step, and
    the job takes the slowest rank's time (weak scaling)."""
    return ws * rows_per_step / (ms_total_max / steps * 1e-3)


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if ident:
            cmd[1:1] = ["-i", ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        win = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not win and self.samples:  # a short timed region: take the closest samples
            win = [min(self.samples, key=lambda s: abs(s[0] - (t0 + t1) / 2))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[0]) for p in win if num(p[0]) is not None]
        mx = [num(p[1]) for p in win if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in win for i in range(4) if p[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


# ---------------------------------------------------------------------------
# ncu-measured traffic (null once the kernel sources changed)
# ---------------------------------------------------------------------------

def kernel_source_hash():
    """Hash of the sweep kernel's device code (the kernel the ncu traffic
    record describes); other kernels' sources do not change it."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "sampling_spec_verify_gb300", "csrc")
    for name in ("ptx.cuh", "sweep.cuh"):
        h.update(open(os.path.join(d, name), "rb").read())
    return h.hexdigest()[:16]


def measured_traffic(kernel_key):
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        db = json.load(open(path))
    except Exception:
        return None
    ent = db.get(kernel_key)
    if not ent or ent.get("src_hash") != kernel_source_hash():
        return None
    return ent.get("bytes_per_launch")


def hbm_peak():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def make_batches(seed):
    from sampling_spec_verify_gb300 import synth
    # same logits for every temperature; tokens drafted from q at that T
    return {T: synth.entropy_mix(seed=seed, temperature=T) for T in TEMPS}


def algorithmic_bytes():
    s = 2
    return {
        "verify": B * (K + 1) * V * s + B * K * V * s,
        "greedy": B * (K + 1) * V * s,
        "e2e": B * K * V * (s + s + 4),
    }


# ---------------------------------------------------------------------------
# CPU baseline: the fp64 oracle as it stands, on host cores
# ---------------------------------------------------------------------------

def oracle_step(batches, rows):
    import oracle
    from sampling_spec_verify_gb300 import synth
    w = batches[1.0]
    zt, zd = synth.f64(w.target[rows]), synth.f64(w.draft[rows])
    for T in TEMPS:
        x = batches[T]
        oracle.verify(zt, zd if T > 0 else None, x.draft_tokens[rows].numpy(), x.u_accept[rows].numpy(),
                      x.u_final[rows].numpy(), T)
    oracle.e2e_tv_loss(zt[:, :K], zd, 1.0)
    oracle.e2e_tv_grad(zt[:, :K], zd, 1.0)


_POOL_BATCHES = None


def _pool_init(seed):
    global _POOL_BATCHES
    torch.set_num_threads(1)
    _POOL_BATCHES = make_batches(seed)


def _pool_rows(rows):
    oracle_step(_POOL_BATCHES, rows)
    return len(rows)


def _single_threaded_children():
    # pool workers inherit the environment: one BLAS / OpenMP thread each
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"


def oracle_pool_rate(budget_s=12.0):
    """The oracle as it stands, one batch row per task, over a process pool
    of one worker per host core (spawned, so it is safe after CUDA starts).
    Returns (rows of the step per second, workers, rows done, seconds)."""
    import multiprocessing as mp
    n = os.cpu_count() or 1
    _single_threaded_children()
    ctx = mp.get_context("spawn")
    with ctx.Pool(n, initializer=_pool_init, initargs=(SEED,)) as pool:
        pool.map(_pool_rows, [[i % B] for i in range(n)], chunksize=1)  # every worker ready
        done, b = 0, 0
        t0 = time.time()
        while time.time() - t0 < budget_s:
            done += sum(pool.map(_pool_rows, [[(b + i) % B] for i in range(n)], chunksize=1))
            b += n
        dt = time.time() - t0
    return len(TEMPS) * K * done / dt, n, done, dt


def cpu_baseline(batches, budget_s=12.0):
    done_rows = 0
    t0 = time.time()
    b = 0
    while True:
        oracle_step(batches, [b % B])
        done_rows += 1
        b += 1
        if time.time() - t0 > budget_s:
            break
    dt = time.time() - t0
    one = len(TEMPS) * K * done_rows / dt
    rate, n, done, dtp = oracle_pool_rate(budget_s)
    return {"value": rate, "unit": "rows/s", "cores": n, "kind": "oracle",
            "sample": f"{done} batch rows of the step (3 verify calls + E2E-TV) in {dtp:.1f} s over a pool of "
                      f"{n} single-threaded numpy float64 workers, one row per task",
            "single_core": {"value": one, "cores": 1,
                            "sample": f"{done_rows} batch rows in {dt:.1f} s, one process"}}


def run_reference(args, ws, rank):
    """The oracle, timed as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    import multiprocessing as mp
    n = os.cpu_count() or 1
    _single_threaded_children()
    ctx = mp.get_context("spawn")
    budget_s = 120.0  # the timed steps stop here even if fewer than --steps ran
    with ctx.Pool(n, initializer=_pool_init, initargs=(SEED,)) as pool:
        # a step: one batch row per host core, the rows of the step's calls
        for i in range(max(1, min(args.warmup, 3))):
            pool.map(_pool_rows, [[(i * n + j) % B] for j in range(n)], chunksize=1)
        t0 = time.time()
        done = 0
        while done < max(1, args.steps) and (done == 0 or time.time() - t0 < budget_s):
            pool.map(_pool_rows, [[(done * n + j) % B] for j in range(n)], chunksize=1)
            done += 1
        dt = time.time() - t0
    value = len(TEMPS) * K * done * n / max(dt, 1e-9)
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": args.gpus, "steps": done,
            "steps_requested": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / done,
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD + f" ({n} batch rows per step, one per host core)", "B": B, "K": K,
                       "V": V},
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": n, "kind": "oracle",
                             "sample": f"{n} batch rows per step over a pool of {n} single-threaded numpy "
                                       f"float64 workers"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------

def run_native(args, ws, rank, local):
    import sampling_spec_verify_gb300 as ssv
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L = ssv.lib()
    batches = make_batches(SEED + rank)
    base = batches[1.0]
    stream = torch.cuda.current_stream(dev)
    sh = ctypes.c_void_p(stream.cuda_stream)

    # resident inputs: N_ROT copies of the batch's logits
    tgt = [base.target.to(dev) for _ in range(N_ROT)]
    drf = [base.draft.to(dev) for _ in range(N_ROT)]
    per_t = {T: (batches[T].draft_tokens.to(dev), batches[T].u_accept.to(dev), batches[T].u_final.to(dev))
             for T in TEMPS}
    outs = {T: (torch.empty((B, K + 1), dtype=torch.int32, device=dev), torch.empty((B,), dtype=torch.int32, device=dev),
                torch.empty((B, K), dtype=torch.float32, device=dev)) for T in TEMPS}
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    loss = torch.empty((1,), dtype=torch.float32, device=dev)
    alpha_e = torch.empty((B, K), dtype=torch.float32, device=dev)
    grad = torch.empty((B, K, V), dtype=torch.float32, device=dev)
    wsz_v = L.spec_verify_workspace_bytes(B, K, V)
    wsz_e = L.spec_e2e_tv_workspace_bytes(B, K, V)
    ws_v = torch.zeros(wsz_v, dtype=torch.uint8, device=dev)
    ws_e = torch.zeros(wsz_e, dtype=torch.uint8, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731

    # prebuilt C-ABI argument lists: call c of the rotation reads copy c % N_ROT
    calls = []  # (kind, args)
    for c in range(N_ROT):
        T = TEMPS[c % 4] if c % 4 < 3 else None
        t, d = tgt[c], drf[c]
        if T is None:
            calls.append(("e2e", (P(t), P(d), 1, B, K, K + 1, V, 1.0, 1.0, P(loss), P(alpha_e), P(grad), P(status),
                                  P(ws_e), wsz_e, sh)))
        else:
            y, ua, uf = per_t[T]
            o = outs[T]
            greedy = T == 0.0
            calls.append(("greedy" if greedy else "verify",
                          (P(t), None if greedy else P(d), 1, B, K, V, T, P(y), P(ua), P(uf), P(o[0]), P(o[1]),
                           None if greedy else P(o[2]), P(status), P(ws_v), wsz_v, sh)))
    fn = {"verify": L.spec_verify, "greedy": L.spec_verify, "e2e": L.spec_e2e_tv_fwd_bwd}
    kinds_per_step = ["verify", "verify", "greedy", "e2e"]
    launches_per_step = 5  # 3 verify kernels + E2E-TV sweep + E2E-TV gradient

    def step(i, ev=None):
        for j in range(4):
            kind, a = calls[(4 * i + j) % N_ROT]
            if ev is not None:
                ev[j][0].record(stream)
            rc = fn[kind](*a)
            if ev is not None:
                ev[j][1].record(stream)
            if rc != 0:
                raise RuntimeError(f"{kind} returned status {rc}")

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    # ---- timed region: K steps, events around every call ----
    n_ev = args.steps
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
           for _ in range(n_ev)]
    clocks = ClockSampler(dev.index) if rank == 0 else None
    time.sleep(0.5 if clocks else 0)
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i, evs[i])
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(ws)
    ms_total = e0.elapsed_time(e1)
    ms_total = max_over_ranks(ms_total, ws, dev)
    if clocks:
        time.sleep(0.3)
        clocks.stop()
    per_kind = {k: [] for k in ("verify", "greedy", "e2e")}
    for i in range(n_ev):
        for j in range(4):
            per_kind[kinds_per_step[j]].append(evs[i][j][0].elapsed_time(evs[i][j][1]))
    ms_step = ms_total / args.steps
    rows_per_step = len(TEMPS) * B * K
    value = job_rate(ms_total, args.steps, ws, rows_per_step)

    # ---- end to end through the public API, host buffers ----
    e2e = run_e2e(args, ssv, batches, dev, stream)

    if rank != 0:
        return
    abytes = algorithmic_bytes()
    peak, peak_kind = hbm_peak()
    avg = {k: statistics.mean(v) for k, v in per_kind.items()}
    share = {k: (sum(per_kind[k]) / max(sum(sum(v) for v in per_kind.values()), 1e-9)) for k in per_kind}
    # dominant single kernel by time: verify (two calls per step) vs the E2E pair
    dom = max(("verify", "greedy"), key=lambda k: sum(per_kind[k]))
    achieved = abytes[dom] / (avg[dom] * 1e-3) / 1e9
    key = {"verify": "sweep_kernel<Bf16,kVerify>@entropy B32K4V151936",
           "greedy": "sweep_kernel<Bf16,kVerifyGreedy>@entropy B32K4V151936"}[dom]
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": measured_traffic(key), "kernel": key, "peak_kind": peak_kind,
            "algorithmic_bytes_per_launch": abytes[dom], "avg_launch_us": 1e3 * avg[dom]}
    per_call = {k: {"avg_us": 1e3 * avg[k], "GB_s": abytes[k] / (avg[k] * 1e-3) / 1e9,
                    "frac_of_measured_hbm": abytes[k] / (avg[k] * 1e-3) / 1e9 / peak, "time_share": share[k]}
                for k in per_kind}
    line = {
        "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "K": K, "V": V, "l2": L2_NOTE, "rows_per_step": rows_per_step,
                   "parallelism": f"dp{ws} (independent batch rows per GPU)"},
        "roofline": roof, "per_call": per_call,
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
        "clocks": clocks.summary(t_wall0, t_wall1) if clocks else None,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(batches)
    print(json.dumps(line), flush=True)


def run_e2e(args, ssv, batches, dev, stream):
    """Whole steps from pinned host memory through the public API: H2D copy of
    the batch, the four calls, D2H of tokens / counts / overlaps / loss.  The
    copy of step i+1's inputs runs on a copy stream into the other of two
    device input sets while step i's kernels run: every step still copies
    its own inputs and reads back its own results."""
    base = batches[1.0]
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    th, dh = pin(base.target), pin(base.draft)
    hin = {T: (pin(batches[T].draft_tokens), pin(batches[T].u_accept), pin(batches[T].u_final)) for T in TEMPS}
    sets = []
    for _ in range(2):
        sets.append({"t": torch.empty_like(th, device=dev), "d": torch.empty_like(dh, device=dev),
                     "in": {T: tuple(torch.empty_like(x, device=dev) for x in hin[T]) for T in TEMPS}})
    outs = {T: ssv.VerifyOutput(torch.empty((B, K + 1), dtype=torch.int32, device=dev),
                                torch.empty((B,), dtype=torch.int32, device=dev),
                                torch.empty((B, K), dtype=torch.float32, device=dev) if T > 0 else None,
                                torch.zeros((1,), dtype=torch.int32, device=dev)) for T in TEMPS}
    eo = ssv.E2EOutput(torch.empty((1,), dtype=torch.float32, device=dev),
                       torch.empty((B, K), dtype=torch.float32, device=dev),
                       torch.empty((B, K, V), dtype=torch.float32, device=dev),
                       torch.zeros((1,), dtype=torch.int32, device=dev))
    hout = {T: (torch.empty((B, K + 1), dtype=torch.int32).pin_memory(),
                torch.empty((B,), dtype=torch.int32).pin_memory(),
                torch.empty((B, K), dtype=torch.float32).pin_memory()) for T in TEMPS}
    hloss = torch.empty((1,), dtype=torch.float32).pin_memory()
    h2d = th.numel() * 2 + dh.numel() * 2 + sum(x.numel() * x.element_size() for T in TEMPS for x in hin[T])
    d2h = 4 + sum(x.numel() * x.element_size() for T in TEMPS for x in (hout[T][:2] if T == 0 else hout[T]))
    copy_s = torch.cuda.Stream(dev)
    free = [torch.cuda.Event(), torch.cuda.Event()]  # the kernels are done with input set j
    for ev in free:
        ev.record(stream)

    def one(i):
        st = sets[i & 1]
        copy_s.wait_event(free[i & 1])
        with torch.cuda.stream(copy_s):
            st["t"].copy_(th, non_blocking=True)
            st["d"].copy_(dh, non_blocking=True)
            for T in TEMPS:
                for a, b_ in zip(st["in"][T], hin[T]):
                    a.copy_(b_, non_blocking=True)
        landed = torch.cuda.Event()
        landed.record(copy_s)
        stream.wait_event(landed)
        t, d = st["t"], st["d"]
        for T in TEMPS:
            y, ua, uf = st["in"][T]
            ssv.verify(t, d if T > 0 else None, y, ua, uf, T, out=outs[T], stream=stream)
        ssv.e2e_tv_fwd_bwd(t, d, 1.0, 1.0, K=K, out=eo, stream=stream)
        free[i & 1].record(stream)
        for T in TEMPS:
            hout[T][0].copy_(outs[T].tokens, non_blocking=True)
            hout[T][1].copy_(outs[T].n_accepted, non_blocking=True)
            if T > 0:
                hout[T][2].copy_(outs[T].alpha, non_blocking=True)
        hloss.copy_(eo.loss, non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    n = max(1, min(args.e2e_steps, args.steps))
    t0 = time.perf_counter()
    for i in range(n):
        one(i)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    # the last step's results, read on the host, check the pipeline
    ref_tok = outs[1.0].tokens.cpu()
    assert torch.equal(hout[1.0][0], ref_tok)
    return {"value": len(TEMPS) * B * K * n / dt, "unit": "rows/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "steps": n, "ms_per_step": 1e3 * dt / n,
            "overlap": "step i+1's H2D copy runs on a second stream during step i's kernels (two input sets)"}


def run_single(args):
    """A few calls of one entry point on the entropy-mix workload at --shape,
    each after a 512 MB L2 flush, for ncu captures of one launch."""
    import sampling_spec_verify_gb300 as ssv
    from sampling_spec_verify_gb300 import synth
    Bs, Ks, Vs = (int(v) for v in args.shape.split(","))
    dev = torch.device("cuda")
    T = 0.0 if args.single == "greedy" else (
        1.0 if args.single in ("overlap", "e2e", "diag", "truncate", "ragged", "schedule", "relaxed")
        else args.temperature)
    w = synth.entropy_mix(seed=SEED, temperature=T, B=Bs, K=Ks, V=Vs)
    t, d = w.target.to(dev), w.draft.to(dev)
    y, ua, uf = w.draft_tokens.to(dev), w.u_accept.to(dev), w.u_final.to(dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(args.calls):
        flush.zero_()
        if args.single in ("verify", "greedy"):
            ssv.verify(t, d if T > 0 else None, y, ua, uf, T)
        elif args.single == "overlap":
            ssv.overlap(t, d, 1.0, K=Ks)
        elif args.single == "diag":
            ssv.diagnostics(t, d, 1.0, K=Ks)
        elif args.single == "truncate":  # top-k 50, top-p 0.9 on the target tensor
            ssv.truncate_logits(t, 1.0, 50, 0.9)
        elif args.single == "ragged":  # every row verifies all of its positions, flattened
            offs = torch.arange(0, (Bs + 1) * (Ks + 1), Ks + 1, dtype=torch.int32, device=dev)
            ssv.verify_ragged(t.reshape(-1, Vs), d.reshape(-1, Vs), offs, y.reshape(-1), ua.reshape(-1), uf, 1.0)
        elif args.single == "relaxed":  # top-k 8, log-probability gap 3
            ssv.verify_relaxed(t, d, y, uf, 1.0, 8, 3.0)
        elif args.single == "tree":  # every row's K drafts as a chain-shaped tree over its K+1 slots
            par = torch.arange(-1, Ks - 1, dtype=torch.int32, device=dev).repeat(Bs, 1)
            ssv.tree_verify_greedy(t, par, y)
        elif args.single == "schedule":  # 1024 requests x 16 positions of prefix survivals
            g = torch.Generator(device=dev).manual_seed(SEED)
            a = torch.cumprod(torch.rand((1024, 16), generator=g, device=dev) * 0.7 + 0.3, dim=1)
            sps = 2000.0 / (1.0 + torch.arange(1024 * 17 + 1, device=dev, dtype=torch.float32) / 256.0)
            ssv.schedule_lengths(a, sps)
        else:
            ssv.e2e_tv_fwd_bwd(t, d, 1.0, 1.0, K=Ks)
    torch.cuda.synchronize()
    print("ok", args.single, Bs, Ks, Vs, T)


def run_sweep():
    """Verify at every point of the shape grid: N(0, 2^2) target logits,
    draft = target + N(0, 0.5^2), bf16, T = 1, drafted tokens from the
    draft; CUDA events around one call after a 512 MB L2 flush, median of 11."""
    import sampling_spec_verify_gb300 as ssv
    dev = torch.device("cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    peak, _ = hbm_peak()
    for Bs in (1, 8, 32, 64, 128, 256):
        for Ks in (1, 2, 4, 7, 16):
            g = torch.Generator(device=dev).manual_seed(Bs * 100 + Ks)
            t = (torch.randn((Bs, Ks + 1, V), device=dev, generator=g) * 2).to(torch.bfloat16)
            d = (t[:, :Ks].float() + 0.5 * torch.randn((Bs, Ks, V), device=dev, generator=g)).to(torch.bfloat16)
            gum = -torch.log(-torch.log(torch.rand((Bs, Ks, V), device=dev, generator=g).clamp_min(1e-20)))
            y = torch.argmax(d.float() + gum, dim=2).to(torch.int32)
            del gum
            ua = torch.rand((Bs, Ks), device=dev, generator=g)
            uf = torch.rand((Bs,), device=dev, generator=g)
            o = ssv.verify(t, d, y, ua, uf, 1.0)
            ts = []
            for i in range(13):
                flush.zero_()
                a, b = torch.cuda.Event(True), torch.cuda.Event(True)
                a.record()
                ssv.verify(t, d, y, ua, uf, 1.0, out=o)
                b.record()
                torch.cuda.synchronize()
                if i >= 2:
                    ts.append(a.elapsed_time(b) * 1e3)
            us = statistics.median(ts)
            by = Bs * (2 * Ks + 1) * V * 2
            print(json.dumps({"B": Bs, "K": Ks, "V": V, "us": round(us, 1), "rows_per_s": round(Bs * Ks / us * 1e6),
                              "GB_s": round(by / us / 1e3), "frac_of_measured_hbm": round(by / us / 1e3 / peak, 3)}),
                  flush=True)
            del t, d, y, o
            torch.cuda.empty_cache()


def main():
    args = parse()
    if args.sweep:
        run_sweep()
        return
    if args.single:
        run_single(args)
        return
    ws, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, ws, rank)
    else:
        run_native(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
