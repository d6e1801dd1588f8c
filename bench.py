"""Benchmark of the reproducible-operator hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. order-fixed FP32 GEMM, M = N = K = 8192, A, B ~ N(0, 1)        (headline)
  2. fixed-order mean of 16 contributor gradients of 2^28 fp32 + SGD in place
  3. SHA-256 Merkle commitment of a 2^30-element fp32 tensor (4 GiB), and of
     the GEMM output C (256 MiB), 4096-byte leaves
Every input is larger than the 129 MB L2, so no flush is needed between steps.

`value` is the GEMM's TFLOP/s (2*M*N*K per launch / its device time, CUDA
events on the launching stream); `parts` gives each stage's own throughput.
`e2e` is the same step from host memory through the library's host-buffer
calls (buffers from its huge-page host allocator), the copies inside the
timed region; its `value` is the GEMM's TFLOP/s measured that way, and
`whole_step` the whole step's time, with the host link's rate beside them.
`--impl reference` times the CPU oracle instead (on a bounded sample of the
same workload), printing the same JSON line with "impl": "reference".

Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(replicas, weak scaling); ranks share only a barrier and a max-reduction of
the elapsed time -- the path has no exchange step.

Other modes: `--sweep [part]` times every workload of a part (one JSON line
each); `--config N` runs one of the five workload configurations with the
Merkle roots of its results; `--tile c` / `--seed s` run the step with the
GEMM on tile configuration c (the roots do not change) or with shifted input
seeds; `--gemm-once` / `--attention-once` launch one GEMM or one sequence's
attention kernels a few times, for a profiler.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import verifiable_repops_gemm_gb300 as rp  # noqa: E402
from verifiable_repops_gemm_gb300 import inputs  # noqa: E402

METRIC = "Bit-exact fixed-order FP32 GEMM TFLOP/s vs FP32 peak; mean/commit HBM GB/s"
GEMM_N = 8192
SM_MAX_MHZ_NOMINAL = 2070.0          # GB300 maximum SM clock
FP32_LANES_PER_SM = 128              # FP32 CUDA cores per SM
# SHA-256 is bound by the integer ALU pipe (16 lanes per SM sub-partition, 64
# per SM).  Rotates (funnel shifts) and 3-input logic run only there; the adds
# and the schedule's two plain shifts can run on the integer multiply-add pipe
# instead (the kernel puts them there).  ALU-only operations of one compression:
# 64 rounds x (6 rotates + Sigma0/Sigma1 XOR3 + Ch + Maj) + 48 schedule words x
# (4 rotates + 2 XOR3) + 16 byte permutes of the message block.
ALU_LANES_PER_SM = 64
SHA_ALU_OPS_PER_COMPRESSION = 64 * 10 + 48 * 6 + 16
# every integer operation of a compression, were both pipes able to share them
# all (64 ALU + 64 multiply-add lanes): a looser figure, reported beside it
SHA_OPS_PER_COMPRESSION = 64 * 14 + 48 * 10 + 24
L2_BYTES = 129 * 10 ** 6
# GB300 HBM3e bandwidth as specified (nominal, not measured)
HBM_SPEC_GBS = 7900.0

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one GEMM
# launch at 8192^3 from one ncu capture of the tiled kernel, valid only for
# the kernel source it was taken on (sha256 of gemm_kernels.cuh).
# Integer-ALU instructions per SHA-256 compression as executed, from one ncu
# capture of repops_sha256_rate_probe (sm__inst_executed_pipe_alu.sum x 32 /
# compressions), valid only for the merkle.cu source it was taken on: the
# measured instruction bound of the commitment (the ALU pipe issuing these
# and nothing else).
SHA_ALU_INSTR = {"src_sha256": "af05b29961a133e97eea5debe9cd92cf231e9b3bcf1a6d137024bca3cf942c07",
                 "per_compression": 1023.23}
GEMM_TRAFFIC = {"src_sha256": "a18f733c4b730ab375a6ca15bf294ac6f4821df7e42a730824418dbbe26ae9fe",
                "bytes_per_launch": 3748467200 + 265021184}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "sm_max_mhz": SM_MAX_MHZ_NOMINAL}, "fallback"


def gemm_kernel_label():
    cfg = rp.gemm_auto_config(GEMM_N, GEMM_N, GEMM_N)
    ci = rp.gemm_config_info(cfg)
    return ("gemm_tma_ws_kernel config %d: %dx%d CTA tile, %d consumer threads + 1 producer warp, "
            "%dx%d per thread; A M-inner (row-major A transposed into scratch first, inside the timed "
            "call), B N-inner" % (cfg, ci["bm"], ci["bn"], ci["threads"], ci["tm"], ci["tn"]))


def kernel_source_sha(name="gemm_kernels.cuh"):
    p = os.path.join(ROOT, "verifiable_repops_gemm_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def sha_instruction_bound(comp_rate, sms, peaks):
    """The commitment against the ALU pipe issuing the ALU instructions a
    compression executes (ncu on the rate probe), while merkle.cu is the
    source they were counted on; else None."""
    if SHA_ALU_INSTR["src_sha256"] != kernel_source_sha("merkle.cu"):
        return None
    clk = peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL) * 1e6
    bound = sms * ALU_LANES_PER_SM * clk / SHA_ALU_INSTR["per_compression"] / 1e9
    return {"peak": bound, "unit": "Gcompressions/s", "frac": comp_rate / bound,
            "alu_instructions_per_compression": SHA_ALU_INSTR["per_compression"],
            "basis": "64 ALU lanes x %d SMs x %.0f MHz / the ALU instructions one compression executes "
                     "(ncu sm__inst_executed_pipe_alu on repops_sha256_rate_probe)"
                     % (sms, clk / 1e6)}


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during timing."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            props = torch.cuda.get_device_properties(self.dev)
            sel = "GPU-%s" % props.uuid if getattr(props, "uuid", None) else str(self.dev)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", sel, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- workload ----

def merkle_launches(nbytes, leaf=4096):
    """Kernel launches of one Merkle commitment (leaf kernel + reduce passes)."""
    leaves = -(-nbytes // leaf)
    n = -(-leaves // 128)
    launches = 1
    while n > 1:
        n = -(-n // 512)
        launches += 1
    return launches


def sha_compressions(nbytes, leaf=4096):
    """SHA-256 compressions of one commitment: 1 + leaf/64 per full leaf (the
    0x00 prefix and padding add one block), 2 per interior node."""
    leaves = -(-nbytes // leaf)
    assert nbytes % leaf == 0
    return leaves * (leaf // 64 + 1) + 2 * (leaves - 1)


class Workload:
    def __init__(self, dev, tile=-1, seed=0):
        # tile: the GEMM's tile configuration (-1: the automatic choice); seed:
        # added to every input seed (0: the seeds the roots below are quoted for)
        n = GEMM_N
        idx = inputs.SQUARE_SWEEP.index(n)
        self.tile = tile
        self.A = inputs.normal((n, n), 1.0, 10 + idx + seed, dev)
        self.B = inputs.normal((n, n), 1.0, 20 + idx + seed, dev)
        self.C = torch.empty((n, n), dtype=torch.float32, device=dev)
        nC, ln = inputs.MEAN_CONTRIBUTORS, inputs.MEAN_LEN
        self.grads = [inputs.normal((ln,), 1e-2, 200 + r + seed, dev) for r in range(nC)]
        self.theta = inputs.normal((ln,), 0.02, 199 + seed, dev)
        self.order = rp.sort_ids(inputs.contributor_ids(nC, 200 + seed))
        self.eta = 1e-3
        self.T = inputs.normal((inputs.MERKLE_ELEMS,), 0.02, 300 + seed, dev)
        self.tbytes = self.T.numel() * 4
        self.cbytes = self.C.numel() * 4
        ws = max(rp.merkle_workspace_bytes(self.tbytes), rp.merkle_workspace_bytes(self.cbytes), 16)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.root_T = torch.empty(32, dtype=torch.uint8, device=dev)
        self.root_C = torch.empty(32, dtype=torch.uint8, device=dev)
        self.gemm_flops = 2.0 * n * n * n
        self.mean_bytes = float((nC + 2) * ln * 4)
        # the GEMM call copies the row-major A into its M-inner scratch layout
        # (one transpose launch) and runs one GEMM kernel
        self.launches = 2 + 1 + merkle_launches(self.tbytes) + merkle_launches(self.cbytes)

    def step(self, s, ev=None):
        if ev: ev[0].record(s)
        rp.gemm(self.A, self.B, out=self.C, config=self.tile, stream=s)
        if ev: ev[1].record(s)
        rp.fixed_order_mean_sgd(self.grads, self.order, self.eta, self.theta, stream=s)
        if ev: ev[2].record(s)
        rp.merkle_sha256(self.T, 4096, out=self.root_T, workspace=self.ws, stream=s)
        rp.merkle_sha256(self.C, 4096, out=self.root_C, workspace=self.ws, stream=s)
        if ev: ev[3].record(s)


def dist_setup(backend=None, timeout_s=None):
    """Rank layout from the torchrun environment; joins the process group
    (NCCL on GPUs unless `backend` says otherwise) when there is more than one
    rank.  The group carries only a barrier and a max-reduction of times.  A
    rank that never reaches a collective makes the others' next collective
    fail after `timeout_s` (REPOPS_PG_TIMEOUT_S, default 600 s) instead of
    waiting forever."""
    import datetime
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        t = float(timeout_s if timeout_s is not None else os.environ.get("REPOPS_PG_TIMEOUT_S", "600"))
        torch.distributed.init_process_group(
            backend or ("nccl" if torch.cuda.is_available() else "gloo"), timeout=datetime.timedelta(seconds=t))
    return world, rank, local


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world, dev):
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle ----

def sha256_probe_rate(dev, sms, iters=500):
    """Compressions per second of the library's SHA-256 compression with its
    message in registers (repops_sha256_rate_probe: no loads, no tree), 8 CTAs
    of 128 threads per SM, iters + 1 compressions a thread, median of 5
    launches: the ceiling the Merkle kernels are measured against."""
    threads = sms * 8 * 128
    out = torch.empty((threads, 8), dtype=torch.int32, device=dev)
    rp.sha256_rate_probe(threads, iters, out=out)
    ts = []
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        rp.sha256_rate_probe(threads, iters, out=out)
        e1.record()
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    return threads * (iters + 1) / (statistics.median(ts) / 1e3) / 1e9


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def host_cores():
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def oracle_parallel(ex, cores, oracle, A, B, row0, grads, order, th, T):
    """One pass of the oracle, as it stands, over disjoint parts of a sample on
    `cores` threads (ctypes releases the GIL while the C oracle runs): one
    GEMM row each (rows row0 ..), a slice of the mean+SGD elements each, and a
    leaf-aligned slice of the Merkle bytes each (its subtree root).  Returns
    the three wall times."""
    n = A.shape[0]
    t0 = time.perf_counter()
    list(ex.map(lambda r: oracle.gemm(A[(row0 + r) % n:(row0 + r) % n + 1], B), range(cores)))
    t1 = time.perf_counter()
    m = th.size
    cuts = [m * c // cores for c in range(cores + 1)]
    list(ex.map(lambda c: oracle.mean_sgd([g[cuts[c]:cuts[c + 1]] for g in grads], order, 1e-3,
                                          th[cuts[c]:cuts[c + 1]]), range(cores)))
    t2 = time.perf_counter()
    leaves = T.size // 1024
    lc = [leaves * c // cores * 1024 for c in range(cores + 1)]
    list(ex.map(lambda c: oracle.merkle_root(T[lc[c]:lc[c + 1]], 4096), range(cores)))
    t3 = time.perf_counter()
    return t1 - t0, t2 - t1, t3 - t2


def cpu_oracle_sample(budget_s=12.0):
    """The oracle (as it stands) on a bounded sample of the step, on one thread
    and on every host core (the same calls over disjoint parts).

    GEMM: whole rows of the 8192^3 product (k-chains of length 8192), rows
    added until about half the budget is used on one thread, a quarter on all
    cores.  Mean+SGD: 2^22 elements of the 16-contributor update.  Merkle:
    256 MiB of the committed tensor."""
    import concurrent.futures as cf
    import oracle
    oracle.lib()
    n = GEMM_N
    idx = inputs.SQUARE_SWEEP.index(n)
    A = inputs.normal((n, n), 1.0, 10 + idx, "cpu").numpy()
    B = inputs.normal((n, n), 1.0, 20 + idx, "cpu").numpy()
    rows, t_gemm = 0, 0.0
    while t_gemm < budget_s * 0.5 and rows < n:
        t0 = time.perf_counter()
        oracle.gemm(A[rows:rows + 1], B)
        t_gemm += time.perf_counter() - t0
        rows += 1
    gemm_tflops = 2.0 * rows * n * n / t_gemm / 1e12
    m = 1 << 22
    grads = [inputs.normal((m,), 1e-2, 200 + r, "cpu").numpy() for r in range(16)]
    th = inputs.normal((m,), 0.02, 199, "cpu").numpy()
    order = oracle.sort_ids(inputs.contributor_ids(16, 200))
    t0 = time.perf_counter()
    oracle.mean_sgd(grads, order, 1e-3, th)
    t_mean = time.perf_counter() - t0
    mb = 256 << 20
    T = inputs.normal((mb // 4,), 0.02, 300, "cpu").numpy()
    t0 = time.perf_counter()
    oracle.merkle_root(T, 4096)
    t_merk = time.perf_counter() - t0
    cores = host_cores()
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        tg = tm = tk = 0.0
        passes = 0
        while tg < budget_s * 0.25 and passes * cores < n:
            g_, m_, k_ = oracle_parallel(ex, cores, oracle, A, B, passes * cores, grads, order, th, T)
            tg += g_; tm += m_; tk += k_
            passes += 1
    return {
        "gemm_tflops": gemm_tflops, "gemm_rows": rows, "gemm_s": t_gemm,
        "mean_gbs": 18 * m * 4 / t_mean / 1e9, "merkle_gbs": mb / t_merk / 1e9,
        "cores": cores,
        "all_cores": {"gemm_tflops": 2.0 * passes * cores * n * n / tg / 1e12,
                      "mean_gbs": 18 * m * 4 * passes / tm / 1e9, "merkle_gbs": mb * passes / tk / 1e9},
        "sample": ("GEMM: %d row(s) of the 8192^3 product on one thread (%.1f s), %d on %d threads "
                   "(%.1f s); mean+SGD: 2^22 elements x 16 contributors; Merkle: 256 MiB (on %d "
                   "threads: leaf-aligned slices, one subtree root each)"
                   % (rows, t_gemm, passes * cores, cores, tg, cores)),
    }


def run_reference(args):
    world, rank, _ = dist_setup("gloo")   # the oracle runs on host cores only
    if rank != 0:
        return
    import oracle
    oracle.lib()
    n = GEMM_N
    idx = inputs.SQUARE_SWEEP.index(n)
    A = inputs.normal((n, n), 1.0, 10 + idx, "cpu").numpy()
    B = inputs.normal((n, n), 1.0, 20 + idx, "cpu").numpy()
    m = 1 << 20
    grads = [inputs.normal((m,), 1e-2, 200 + r, "cpu").numpy() for r in range(16)]
    th = inputs.normal((m,), 0.02, 199, "cpu").numpy()
    order = oracle.sort_ids(inputs.contributor_ids(16, 200))
    T = inputs.normal(((32 << 20) // 4,), 0.02, 300, "cpu").numpy()

    import concurrent.futures as cf
    cores = host_cores()
    ex = cf.ThreadPoolExecutor(max_workers=cores)

    def step(i):
        # one GEMM row per core (8192 k-chains of 8192 each), the mean+SGD
        # elements and the Merkle bytes split across the cores
        return oracle_parallel(ex, cores, oracle, A, B, i * cores, grads, order, th, T)

    for i in range(args.warmup):
        step(i)
    tg = tm = tk = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        a, b, c = step(args.warmup + i)
        tg += a; tm += b; tk += c
    total = time.perf_counter() - t0
    ex.shutdown()
    val = 2.0 * n * n * cores * args.steps / tg / 1e12
    sample = ("per step: %d rows of the 8192^3 GEMM, mean+SGD over 2^20 elements x 16 "
              "contributors, Merkle of 32 MiB (leaf-aligned slices, one subtree root each); "
              "%d threads, one part each" % (cores, cores))
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "order-fixed fp32 GEMM 8192^3 + mean/SGD 16x2^28 + Merkle 4 GiB "
                               "(bounded CPU sample)", "parallelism": "replicas",
                   "l2": "inputs larger than L2"},
        "parts": {"mean_sgd": {"value": 18 * m * 4 * args.steps / tm / 1e9, "unit": "GB/s"},
                  "merkle": {"value": (32 << 20) * args.steps / tk / 1e9, "unit": "GB/s"}},
        "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "cpu_model": cpu_model(),
                         "sample": sample},
        "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------- ours ----

KEEP_SCRATCH_E2E = 2 << 30   # freed scratch the pool may keep mapped during the end-to-end steps


def run_e2e(w, dev, steps):
    """Same metric through the library's host-buffer entry points, all three
    parts from page-locked host memory: repops_gemm_f32_host (A and B in, C back,
    the copies overlapping the GEMM's row blocks), then
    repops_fixed_order_mean_sgd_host (16 gradients and theta in, theta back,
    chunk by chunk), then repops_merkle_sha256_host of T and of C (chunks in,
    roots back).  Every byte moves over the host link inside the timed
    region.  The host buffers come from the library's host allocator
    (rp.host_empty: page-locked, in transparent huge pages), which keeps the
    copies at the host link's rate where memory pinned in 64 KB pages lost up
    to two thirds of it at this step's 22 GB."""
    s = torch.cuda.Stream(device=dev)
    def pinned_copy(t):
        h = rp.host_empty(t.shape, t.dtype)
        h.copy_(t)
        return h
    # A, B and C (256 MiB each, below a 512 MB huge page) share one block, so
    # that they sit in huge pages without rounding each of them up to one
    hABC = rp.host_empty((3,) + tuple(w.A.shape), torch.float32)
    assert tuple(w.A.shape) == tuple(w.B.shape) == tuple(w.C.shape)
    hA, hB, hC = hABC[0], hABC[1], hABC[2]
    hA.copy_(w.A)
    hB.copy_(w.B)
    hg = [pinned_copy(g) for g in w.grads]
    hth = pinned_copy(w.theta)
    hT = pinned_copy(w.T)
    hroot = rp.host_empty((2, 32), torch.uint8)
    # the link probes copy from and to the step's own buffers (the output C is
    # written over by the first step): another GiB of host memory here cost
    # the step's first buffers their huge pages on a host with ~22 GiB of
    # huge-page blocks free
    link = host_link_rate(dev, s, src=hg[0], dst=hC)
    link["h2d_gradients_16gib"] = working_set_rate(dev, s, hg)
    huge = anon_huge_page_bytes()
    want_root_C = bytes(w.root_C.cpu().numpy())
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps + 1)]
    # a caller that runs step after step lets the scratch pool keep its memory
    # mapped across the per-step synchronisation (the default hands it back)
    rp.scratch_set_keep_bytes(KEEP_SCRATCH_E2E)
    try:
        torch.cuda.synchronize(dev)
        for i in range(steps + 1):          # the first pass is an untimed warm-up
            e = ev[i]
            e[0].record(s)
            rp.gemm_host(hA, hB, out=hC, stream=s)
            e[1].record(s)
            rp.fixed_order_mean_sgd_host(hg, w.order, w.eta, hth, stream=s)
            e[2].record(s)
            rp.merkle_sha256_host(hT, 4096, out=hroot[0], stream=s)
            rp.merkle_sha256_host(hC, 4096, out=hroot[1], stream=s)
            e[3].record(s)
            # the step's result read on the host: the roots
            e[3].synchronize()
            if bytes(hroot[1].numpy()) != want_root_C:
                raise RuntimeError("the host-buffer step's root of C differs from the device step's")
    finally:
        torch.cuda.synchronize(dev)
        rp.scratch_set_keep_bytes(0)
        rp.scratch_release()
    ev = ev[1:]
    tg = sum(e[0].elapsed_time(e[1]) for e in ev) / 1e3
    tm = sum(e[1].elapsed_time(e[2]) for e in ev) / 1e3
    tk = sum(e[2].elapsed_time(e[3]) for e in ev) / 1e3
    step_s = [e[0].elapsed_time(e[3]) / 1e3 for e in ev]
    h2d = 2 * w.A.numel() * 4 + (len(w.grads) + 1) * w.theta.numel() * 4 + w.tbytes + w.cbytes
    d2h = w.C.numel() * 4 + w.theta.numel() * 4 + 64
    return {"value": w.gemm_flops * steps / tg / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "parts": {"mean_sgd_gbs": w.mean_bytes * steps / tm / 1e9,
                      "merkle_gbs": (w.tbytes + w.cbytes) * steps / tk / 1e9},
            "whole_step": {"ms": 1e3 * statistics.mean(step_s), "ms_min": 1e3 * min(step_s),
                           "ms_max": 1e3 * max(step_s),
                           "steps_ms": [round(1e3 * x, 1) for x in step_s],
                           "parts_ms": [[round(e[0].elapsed_time(e[1]), 1), round(e[1].elapsed_time(e[2]), 1),
                                         round(e[2].elapsed_time(e[3]), 1)] for e in ev],
                           "host_bytes_moved_gbs": (h2d + d2h) * steps / sum(step_s) / 1e9,
                           "basis": "every part through a host-buffer C-ABI call (repops_gemm_f32_host, "
                                    "repops_fixed_order_mean_sgd_host, repops_merkle_sha256_host x 2) from "
                                    "page-locked huge-page host memory (repops_host_alloc); a synchronisation "
                                    "and a host read of the roots after every step; the scratch pool keeps "
                                    "%d GiB across steps (repops_scratch_set_keep_bytes); mean of the steps"
                                    % (KEEP_SCRATCH_E2E >> 30)},
            "host_link_gbs": link,
            "host_huge_page_bytes": huge,
            "steps": steps}


def working_set_rate(dev, s, bufs):
    """Host -> device rate over a whole set of host buffers, copied back to back
    into one device buffer (CUDA events, best of 2): the host link at the
    working set a step touches, which on a virtual machine can be far below
    the 1 GiB figure (address translation of the guest's memory)."""
    d = torch.empty(max(b.numel() * b.element_size() for b in bufs), dtype=torch.uint8, device=dev)
    total = sum(b.numel() * b.element_size() for b in bufs)
    best = None
    for _ in range(2):
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            for b in bufs:
                n = b.numel() * b.element_size()
                d[:n].copy_(b.view(-1).view(torch.uint8), non_blocking=True)
            e.record(s)
        e.synchronize()
        t = a.elapsed_time(e) / 1e3
        best = t if best is None else min(best, t)
    del d
    return total / best / 1e9


def anon_huge_page_bytes():
    """Bytes of this process's anonymous memory held in transparent huge pages
    (/proc/self/smaps_rollup), or None where the kernel does not say."""
    try:
        with open("/proc/self/smaps_rollup") as f:
            for line in f:
                if line.startswith("AnonHugePages:"):
                    return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def host_link_rate(dev, s, src, dst):
    """Host <-> device copy rate over one host buffer each way (src read,
    dst written: host memory of the end-to-end steps' kind, rp.host_empty),
    each direction timed alone (CUDA events, best of 3), sampled right before
    those steps: the end-to-end figures are bound by it."""
    hs, hd = src.view(-1).view(torch.uint8), dst.view(-1).view(torch.uint8)
    d = torch.empty(max(hs.numel(), hd.numel()), dtype=torch.uint8, device=dev)
    sizes = {"h2d": hs.numel(), "d2h": hd.numel()}
    out = {}
    for name, fn in (("h2d", lambda: d[:hs.numel()].copy_(hs, non_blocking=True)),
                     ("d2h", lambda: hd.copy_(d[:hd.numel()], non_blocking=True))):
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(s):
                a.record(s)
                fn()
                b.record(s)
            b.synchronize()
            t = a.elapsed_time(b) / 1e3
            best = t if best is None else min(best, t)
        out[name] = sizes[name] / best / 1e9
    del d
    return out


def run_ours(args):
    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    rp.load()
    peaks, peaks_kind = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    w = Workload(dev, args.tile, args.seed)
    s = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            w.step(s)
    torch.cuda.synchronize(dev)
    if rp.device_status(s) != 0:
        raise RuntimeError("a kernel reported a timed-out wait during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(s):
            start.record(s)
            for i in range(args.steps):
                w.step(s, evs[i])
            stop.record(s)
        torch.cuda.synchronize(dev)
        barrier(world)
    clocks = clk.summary()
    if rp.device_status(s) != 0:
        raise RuntimeError("a kernel reported a timed-out wait in the timed region")
    total_ms = start.elapsed_time(stop)
    gemm_ms = [e[0].elapsed_time(e[1]) for e in evs]
    mean_ms = [e[1].elapsed_time(e[2]) for e in evs]
    merk_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_max = max_over_ranks(total_ms, world, dev)
    gemm_max = max_over_ranks(sum(gemm_ms), world, dev)
    mean_max = max_over_ranks(sum(mean_ms), world, dev)
    merk_max = max_over_ranks(sum(merk_ms), world, dev)

    # the step's commitments right after the timed region: the roots of T and
    # of the GEMM output C (the same bits on every run of these seeds) and of
    # theta after warmup + steps updates
    theta_root = rp.merkle_sha256(w.theta)
    commitments = {"T_root": bytes(w.root_T.cpu().numpy()).hex(),
                   "C_root": bytes(w.root_C.cpu().numpy()).hex(),
                   "theta_root": bytes(theta_root.cpu().numpy()).hex(),
                   "theta_updates": args.warmup + args.steps}
    e2e = run_e2e(w, dev, args.e2e_steps) if args.e2e_steps > 0 else None
    probe_rate = sha256_probe_rate(dev, sms)   # outside the timed region
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_sample()

    if rank != 0:
        return
    gemm_avg_s = statistics.mean(gemm_ms) / 1e3
    achieved = w.gemm_flops / gemm_avg_s / 1e12
    peak = sms * FP32_LANES_PER_SM * peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL) * 1e6 / 1e12
    traffic = None
    if GEMM_TRAFFIC["src_sha256"] and GEMM_TRAFFIC["src_sha256"] == kernel_source_sha():
        traffic = GEMM_TRAFFIC["bytes_per_launch"]
    hbm = peaks.get("hbm_gbs", 6800.0)
    mean_gbs = w.mean_bytes * args.steps * world / (mean_max / 1e3) / 1e9
    merk_gbs = (w.tbytes + w.cbytes) * args.steps * world / (merk_max / 1e3) / 1e9
    value = w.gemm_flops * args.steps * world / (gemm_max / 1e3) / 1e12
    ncomp = sha_compressions(w.tbytes) + sha_compressions(w.cbytes)
    comp_rate = ncomp * args.steps / (merk_max / 1e3) / 1e9
    clk = peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL) * 1e6
    comp_peak = sms * ALU_LANES_PER_SM * clk / SHA_ALU_OPS_PER_COMPRESSION / 1e9
    comp_peak_shared = sms * 2 * ALU_LANES_PER_SM * clk / SHA_OPS_PER_COMPRESSION / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded torch generators)",
        "config": {"workload": "order-fixed fp32 GEMM 8192^3 (A,B ~ N(0,1)) + fixed-order mean/SGD "
                               "16 x 2^28 + SHA-256 Merkle of 4 GiB and of C, 4096-B leaves",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (129 MB); no flush",
                   "gemm_tile": "automatic" if args.tile < 0 else args.tile, "seed_offset": args.seed},
        "parts": {
            "gemm": {"value": value, "unit": "TFLOP/s", "ms": statistics.mean(gemm_ms)},
            "mean_sgd": {"value": mean_gbs, "unit": "GB/s", "ms": statistics.mean(mean_ms),
                         "roofline": {"bound": "hbm", "achieved": mean_gbs / world, "peak": hbm,
                                      "unit": "GB/s", "frac": mean_gbs / world / hbm,
                                      "peak_is": "the %s copy bandwidth (hbm_gbs: a STREAM-style copy), "
                                                 "which a read-mostly stream can slightly exceed" % peaks_kind,
                                      "spec_hbm_gbs": HBM_SPEC_GBS,
                                      "frac_of_spec_hbm": mean_gbs / world / HBM_SPEC_GBS,
                                      "basis": "(16 + 2) x 2^28 x 4 B per step"}},
            "merkle": {"value": merk_gbs, "unit": "GB/s", "ms": statistics.mean(merk_ms),
                       "sha256_compressions_per_step": ncomp,
                       "roofline": {"bound": "alu", "achieved": comp_rate, "peak": comp_peak,
                                    "unit": "Gcompressions/s", "frac": comp_rate / comp_peak,
                                    "basis": "64 ALU lanes x %d SMs x %.0f MHz / %d ALU-only operations per "
                                             "SHA-256 compression (rotates, 3-input logic, byte permutes; the "
                                             "adds run on the multiply-add pipe)"
                                             % (sms, peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL),
                                                SHA_ALU_OPS_PER_COMPRESSION),
                                    "frac_if_both_pipes_shared_all_ops": comp_rate / comp_peak_shared,
                                    "measured_ceiling": {
                                        "value": probe_rate, "unit": "Gcompressions/s",
                                        "basis": "repops_sha256_rate_probe: the same compression, message in "
                                                 "registers, no loads or tree, 8 x 128 threads per SM"},
                                    "frac_of_measured_ceiling": comp_rate / probe_rate,
                                    "measured_instruction_bound": sha_instruction_bound(comp_rate, sms, peaks)}},
        },
        "roofline": {"kernel": gemm_kernel_label(), "bound": "alu",
                     "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_basis": "%d SMs x 128 FP32 lanes x %.0f MHz (%s sm_max_mhz); one FP32 "
                                   "op per lane per clock: products and sums issue separately"
                                   % (sms, peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL), peaks_kind)},
        "clocks": clocks,
        "gpu_launches": w.launches * args.steps,
    }
    line["commitments"] = commitments
    if clocks.get("sm_mhz"):
        line["roofline"]["frac_at_sampled_clock"] = achieved / (
            sms * FP32_LANES_PER_SM * clocks["sm_mhz"] * 1e6 / 1e12)
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        allc = cpu["all_cores"]
        line["cpu_baseline"] = {"value": allc["gemm_tflops"], "unit": "TFLOP/s", "cores": cpu["cores"],
                                "kind": "oracle", "sample": cpu["sample"], "cpu_model": cpu_model(),
                                "parts": {"mean_sgd_gbs": allc["mean_gbs"],
                                          "merkle_gbs": allc["merkle_gbs"]},
                                "single_thread": {"value": cpu["gemm_tflops"], "cores": 1,
                                                  "parts": {"mean_sgd_gbs": cpu["mean_gbs"],
                                                            "merkle_gbs": cpu["merkle_gbs"]}}}
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """One JSON line per workload.  GEMM: the 256^3 case, the square sweep with
    B row- and column-major, the ragged 4097x1023x3001 case, and the 15 GEMMs
    of the decoder-layer set; then the row operators and the commitments.
    Each timed launch is bracketed by its own CUDA events and preceded by an L2
    flush (a 256 MiB write).  `args.sweep` picks one part or all of them."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rp.load()
    peaks, _ = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = sms * FP32_LANES_PER_SM * peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL) * 1e6 / 1e12
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    if args.sweep in ("all", "gemm"):
        run_sweep_gemm(dev, s, flush, peak)
    if args.sweep in ("all", "rowops"):
        run_sweep_rowops(dev, s, flush, peaks.get("hbm_gbs", 6800.0))
    if args.sweep in ("all", "commitments"):
        run_sweep_commitments(dev, s, flush)
    if args.sweep in ("all", "decoder"):
        run_sweep_decoder(dev, s, flush, peak)
    if args.sweep in ("all", "halfstore"):
        run_sweep_halfstore(dev, s, flush, peak, peaks.get("hbm_gbs", 6800.0))
    if args.sweep in ("all", "halfstore", "rolling"):
        run_sweep_rolling(dev, s, flush, peaks.get("hbm_gbs", 6800.0))
    if args.sweep in ("all", "train"):
        run_sweep_train(dev, s, flush, peak)
    if args.sweep == "decoder_step":
        run_decoder_step(dev, s, peak)


def run_config(c):
    """One workload configuration: one JSON line per workload, with the Merkle
    roots of the GEMM outputs (configurations 0 and 1) and of theta after the
    update (3); 4 times the 4 GiB commitment and prints the roots of the
    square-sweep outputs (the same for both B layouts)."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rp.load()
    peaks, _ = measured_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak = sms * FP32_LANES_PER_SM * peaks.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL) * 1e6 / 1e12
    hbm = peaks.get("hbm_gbs", 6800.0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream(device=dev)
    if c in (0, 1, 2):
        run_sweep_gemm(dev, s, flush, peak, parts=(c,), roots=c in (0, 1))
        return
    w = Workload(dev)

    def timed(fn, reps=10):
        with torch.cuda.stream(s):
            fn()
            evs = []
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    if c == 3:
        reps = 10
        ms = timed(lambda: rp.fixed_order_mean_sgd(w.grads, w.order, w.eta, w.theta, stream=s), reps)
        gbs = w.mean_bytes / ms / 1e6
        print(json.dumps({"config": 3, "workload": "fixed-order mean + SGD, 16 contributors x 2^28 (inputs above "
                          "L2)", "ms": ms, "gbs": gbs, "frac_of_measured_hbm": gbs / hbm,
                          "theta_updates": reps + 1, "theta_root": bytes(rp.merkle_sha256(w.theta).cpu().numpy()).hex()}),
              flush=True)
        return
    ms = timed(lambda: rp.merkle_sha256(w.T, 4096, out=w.root_T, workspace=w.ws, stream=s))
    print(json.dumps({"config": 4, "workload": "SHA-256 Merkle root of 2^30 fp32 (4 GiB), 4096-byte leaves",
                      "ms": ms, "gbs": w.tbytes / ms / 1e6,
                      "root": bytes(w.root_T.cpu().numpy()).hex()}), flush=True)
    del w
    for i, n in enumerate(inputs.SQUARE_SWEEP):
        A = inputs.normal((n, n), 1.0, 10 + i, dev)
        B = inputs.normal((n, n), 1.0, 20 + i, dev)
        r1 = bytes(rp.merkle_sha256(rp.gemm(A, B)).cpu().numpy()).hex()
        r2 = bytes(rp.merkle_sha256(rp.gemm(A, B.t().contiguous().t())).cpu().numpy()).hex()
        print(json.dumps({"config": 4, "workload": "Merkle root of the %d^3 GEMM output" % n, "root": r1,
                          "same_for_column_major_B": r1 == r2}), flush=True)
        del A, B


def run_sweep_gemm(dev, s, flush, peak, parts=(0, 1, 2), roots=False):
    """Every GEMM workload, L2 flushed before each timed launch, the median of
    at least 10 launches.  Beside each,
    the library's FP32 GEMM (torch.mm on cuBLAS, TF32 off: fused multiply-adds,
    no fixed order) on the same operands, timed the same way: the pages state
    their cost as the overhead of the order-fixed GEMM over that one."""

    def timed(fn, flops):
        reps = max(10, min(50, int(2e11 / max(flops, 1.0))))
        with torch.cuda.stream(s):
            for _ in range(3):
                fn()
            evs = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    def emit(name, A, B, extra=None):
        M, K = A.shape
        N = B.shape[1]
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
        flops = 2.0 * M * N * K
        ms = timed(lambda: rp.gemm(A, B, out=C, stream=s), flops)
        tf32 = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        try:
            lib_ms = timed(lambda: torch.mm(A, B, out=C), flops)
        finally:
            torch.backends.cuda.matmul.allow_tf32 = tf32
        cfg = rp.gemm_auto_config(M, N, K)
        chained = rp.gemm_auto_chained(M, N, K)
        kernel = ("small-output" if rp.gemm_small_output(M, N, K) else
                  "tiled config %d%s" % (cfg, ", chained k-split" if chained else ""))
        tf = flops / ms / 1e9
        rec = {"sweep": name, "M": M, "N": N, "K": K, "ms": ms,
               "tflops": tf, "frac_of_fp32_peak": tf / peak, "kernel": kernel,
               "library_fp32_gemm_ms": lib_ms, "overhead_vs_library": ms / lib_ms - 1.0}
        if chained:
            # the same configuration with one CTA per tile (no split)
            one_ms = timed(lambda: rp.gemm(A, B, out=C, config=cfg, stream=s), flops)
            rec["one_cta_per_tile_ms"] = one_ms
            rec["one_cta_per_tile_tflops"] = flops / one_ms / 1e9
        rec.update(extra or {})
        print(json.dumps(rec), flush=True)
        return flops, ms

    def root(A, B):
        # the Merkle root of the output (the same bits for every layout)
        return {"C_root": bytes(rp.merkle_sha256(rp.gemm(A, B)).cpu().numpy()).hex()} if roots else None

    if 0 in parts:
        A = inputs.uniform_pm1((256, 256), 0, dev)
        B = inputs.uniform_pm1((256, 256), 1, dev)
        emit("gemm 256^3 U[-1,1)", A, B, root(A, B))
    if 1 in parts:
        for i, n in enumerate(inputs.SQUARE_SWEEP):
            A = inputs.normal((n, n), 1.0, 10 + i, dev)
            B = inputs.normal((n, n), 1.0, 20 + i, dev)
            emit("gemm %d^3 B row-major" % n, A, B, root(A, B))
            Bc = B.t().contiguous().t()
            emit("gemm %d^3 B column-major" % n, A, Bc, root(A, Bc))
            del A, B, Bc
        M, N, K = inputs.RAGGED
        A = inputs.normal((M, K), 1.0, 30, dev)
        B = inputs.normal((K, N), 1.0, 31, dev)
        emit("gemm ragged 4097x1023x3001 (lda = 3001: operands repacked to a 16-byte pitch)", A, B, root(A, B))
    if 2 not in parts:
        return
    T, D = inputs.DECODER_TOKENS, inputs.DECODER_DIM
    X = inputs.normal((T, D), 1.0, 100, dev)
    tot_f = tot_ms = 0.0
    for li, (name, kin, nout) in enumerate(inputs.DECODER_LAYERS):
        Xin = X if kin == D else inputs.normal((T, kin), 1.0, 150 + li, dev)
        W = inputs.normal((kin, nout), 0.02, 110 + li, dev)
        dY = inputs.normal((T, nout), 1e-3, 120 + li, dev)
        for kind, a, b in (("forward Y=XW", Xin, W), ("dX=dY W^T", dY, W.t()), ("dW=X^T dY", Xin.t(), dY)):
            f, ms = emit("decoder %s %s" % (name, kind), a, b)
            tot_f += f
            tot_ms += ms
    print(json.dumps({"sweep": "decoder layer set, 15 GEMMs", "ms": tot_ms, "tflops": tot_f / tot_ms / 1e9,
                      "frac_of_fp32_peak": tot_f / tot_ms / 1e9 / peak}), flush=True)
    del X, Xin, W, dY


def run_sweep_rowops(dev, s, flush, hbm):
    """The order-fixed row operators on decoder-sized tensors: LayerNorm and
    RMSNorm over 16 x 4096 tokens x 2048, GeLU over 4096 x 8192 activations,
    softmax (plain, causal, causal backward) over 8 heads of 4096 x 4096
    scores, SwiGLU and its backward over 4096 x 8192, the rotary embedding of
    a 4096-token qkv matrix.  Bytes = the algorithmic reads and writes (HBM
    roofline); the L2 is flushed before each launch."""
    def ev_time(fn, reps=5):
        with torch.cuda.stream(s):
            fn()
            evs = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in evs) / reps

    def emit(name, nbytes, ms):
        gbs = nbytes / ms / 1e6
        print(json.dumps({"sweep": name, "ms": ms, "gbs": gbs, "frac_of_hbm": gbs / hbm}), flush=True)

    T, D = inputs.DECODER_TOKENS, inputs.DECODER_DIM
    X = inputs.normal((16 * T, D), 1.0, 100, dev)
    Y = torch.empty_like(X)
    g = inputs.normal((D,), 1.0, 101, dev)
    b = inputs.normal((D,), 0.1, 102, dev)
    emit("layernorm rows 65536 x 2048", 2 * X.numel() * 4,
         ev_time(lambda: rp.layernorm_rows(X, g, b, 1e-5, out=Y, stream=s)))
    emit("rmsnorm rows 65536 x 2048", 2 * X.numel() * 4,
         ev_time(lambda: rp.rmsnorm_rows(X, g, 1e-6, out=Y, stream=s)))
    del X, Y
    H = inputs.normal((T, 4 * D), 1.0, 103, dev)
    G = torch.empty_like(H)
    emit("gelu 4096 x 8192", 2 * H.numel() * 4, ev_time(lambda: rp.gelu(H, out=G, stream=s)))
    del H, G
    S = inputs.normal((8 * T, T), 3.0, 104, dev)
    P = torch.empty_like(S)
    emit("softmax rows 8 x 4096 x 4096", 2 * S.numel() * 4, ev_time(lambda: rp.softmax_rows(S, out=P, stream=s)))
    # the causal forms read and write each row's prefix only (the rest of the
    # output is written as +0): bytes = 2 x 4 x the prefix elements + 4 x the rest
    n, rows = T, 8 * T
    pre = rows // n * (n * (n + 1) // 2)
    causal_bytes = 8 * pre + 4 * (S.numel() - pre)
    emit("causal softmax rows 8 x 4096 x 4096", causal_bytes,
         ev_time(lambda: rp.softmax_rows(S, out=P, causal_first=0, causal_period=T, stream=s)))
    dP = inputs.normal((8 * T, T), 1.0, 105, dev)
    emit("causal softmax backward 8 x 4096 x 4096", 12 * pre + 4 * (S.numel() - pre),
         ev_time(lambda: rp.softmax_backward(P, dP, out=S, causal_first=0, causal_period=T, stream=s)))
    del S, P, dP
    # the Llama layer's element-wise operators at decoder sizes: SwiGLU over
    # [g | u] of 4096 x 2 x 8192, its backward, the rotary embedding of the 40
    # query and key heads of a 4096 x 3072 qkv matrix
    GU = inputs.normal((T, 8 * D), 2.0, 106, dev)
    A = torch.empty(T, 4 * D, device=dev)
    emit("swiglu 4096 x 8192 (reads g, u; writes h)", 3 * A.numel() * 4,
         ev_time(lambda: rp.swiglu(GU[:, :4 * D], GU[:, 4 * D:], out=A, stream=s)))
    DG, DU = torch.empty_like(A), torch.empty_like(A)
    emit("swiglu backward 4096 x 8192 (reads g, u, dh; writes dg, du)", 5 * A.numel() * 4,
         ev_time(lambda: rp.swiglu_backward(GU[:, :4 * D], GU[:, 4 * D:], A, dg=DG, du=DU, stream=s)))
    del GU, A, DG, DU
    Q = inputs.normal((T, 3 * D // 2), 1.0, 107, dev)
    cos, sin = rp.rope_table(T, rp.rope_frequencies(32, math.log(500000.0), dev))
    emit("rotary 4096 x 40 heads of 64 (in place)", 2 * T * 40 * 64 * 4,
         ev_time(lambda: rp.rope(Q, 40, cos, sin, stream=s)))
    del Q


def run_sweep_decoder(dev, s, flush, peak):
    """One decoder layer (Llama-3.2-1B sizes: d 2048, 32 query and 8 key/value
    heads of 64, MLP 8192) over two causal sequences of 2048 tokens, every
    step a library call.  The Llama layer (rotary embedding, SwiGLU MLP) and
    the GeLU layer (no rotary): the fused forward, the forward with its
    epilogues as separate steps, the training step (forward keeping the
    activations, then the backward pass); and the attention alone.  FLOPs
    count the causal band of the attention products.  Synthetic N(0, 0.02)
    weights; L2 flushed before each timed layer."""
    from verifiable_repops_gemm_gb300 import decoder
    llama = decoder.DecoderConfig()
    layers = (("llama layer (rotary, SwiGLU)", llama, ((True, False), (False, False))),
              ("GeLU layer", decoder.DecoderConfig(mlp="gelu", rope_base=0.0),
               ((True, False), (True, True), (False, False))))
    T = 2 * llama.seq_len
    x0 = inputs.normal((T, llama.d), 1.0, 301, dev)
    x = torch.empty_like(x0)
    dy0 = inputs.normal((T, llama.d), 1e-2, 302, dev)
    dy = torch.empty_like(dy0)

    def timed(fn, reps=5):
        with torch.cuda.stream(s):
            for _ in range(2):
                x.copy_(x0)
                fn()
            evs = []
            for _ in range(reps):
                x.copy_(x0)
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in evs) / reps

    for label, cfg, variants in layers:
        w = decoder.init_weights(cfg, 300, dev)
        ws = decoder.workspace(cfg, T, dev)
        flops = cfg.flops(T)
        for fused, ge in variants:
            what = ("fused residual/bias epilogues" if fused else "epilogues as separate steps") + \
                   (", GeLU in the GEMM epilogue" if ge else "")
            ms = timed(lambda: decoder.forward(x, w, cfg, fused=fused, gelu_epilogue=ge, work=ws))
            print(json.dumps({"sweep": "%s forward, %s" % (label, what), "tokens": T, "ms": ms,
                              "tokens_per_s": T / ms * 1e3, "tflops": flops / ms / 1e9,
                              "frac_of_fp32_peak": flops / ms / 1e9 / peak}), flush=True)
        if cfg is llama:
            S = cfg.seq_len
            attn_flops = 2 * 2.0 * (T // S) * cfg.heads * (S * (S + 1) / 2) * cfg.d_head
            ms = timed(lambda: decoder.attention(ws["qkv"], cfg, ws["attn"], ws["scores"], streams=ws["streams"],
                                                 fused=False))
            print(json.dumps({"sweep": "causal grouped-query attention, unfused (batched QK^T, softmax, banded PV)",
                              "tokens": T, "ms": ms, "tflops": attn_flops / ms / 1e9,
                              "frac_of_fp32_peak": attn_flops / ms / 1e9 / peak}), flush=True)
            ms = timed(lambda: decoder.attention(ws["qkv"], cfg, ws["attn"], ws["scores"], fused=True))
            print(json.dumps({"sweep": "causal grouped-query attention, fused kernel (one launch)",
                              "tokens": T, "ms": ms, "tflops": attn_flops / ms / 1e9,
                              "frac_of_fp32_peak": attn_flops / ms / 1e9 / peak}), flush=True)
            probs = torch.empty((T // S) * cfg.heads * S * S, device=dev)
            ms = timed(lambda: decoder.attention(ws["qkv"], cfg, ws["attn"], ws["scores"], probs=probs,
                                                 fused=True))
            print(json.dumps({"sweep": "causal grouped-query attention, fused kernel writing every probability",
                              "tokens": T, "ms": ms, "tflops": attn_flops / ms / 1e9,
                              "frac_of_fp32_peak": attn_flops / ms / 1e9 / peak}), flush=True)
            del probs
            ms = timed(lambda: decoder.forward(x, w, cfg, work=ws, fused_attention=True))
            print(json.dumps({"sweep": "%s forward, fused epilogues, fused attention kernel" % label, "tokens": T,
                              "ms": ms, "tokens_per_s": T / ms * 1e3, "tflops": flops / ms / 1e9,
                              "frac_of_fp32_peak": flops / ms / 1e9 / peak}), flush=True)
        # the training step: forward keeping its activations, then the backward
        # pass (every weight's gradient and dx): 3x the forward FLOPs
        saved = decoder.activations(cfg, T, dev)
        bws = decoder.backward_workspace(cfg, T, dev)
        ms_f = timed(lambda: decoder.forward(x, w, cfg, work=ws, save=saved))

        def step():
            decoder.forward(x, w, cfg, work=ws, save=saved)
            dy.copy_(dy0)
            decoder.backward(dy, w, cfg, saved, work=bws)
        ms = timed(step)
        print(json.dumps({"sweep": "%s training step (forward keeping activations + backward)" % label,
                          "tokens": T, "ms": ms, "forward_ms": ms_f, "tokens_per_s": T / ms * 1e3,
                          "tflops": 3 * flops / ms / 1e9, "frac_of_fp32_peak": 3 * flops / ms / 1e9 / peak}),
              flush=True)
        del saved, bws, ws, w


def run_decoder_step(dev, s, peak):
    """Exactly two training steps of the Llama layer (forward keeping the
    activations, then the backward pass), 2 x 2048 tokens: a short program whose
    every kernel launch a profiler can list (the first step warms up, the
    second is the one to read).  Not part of "all"."""
    from verifiable_repops_gemm_gb300 import decoder
    cfg = decoder.DecoderConfig()
    T = 2 * cfg.seq_len
    w = decoder.init_weights(cfg, 300, dev)
    ws = decoder.workspace(cfg, T, dev)
    saved = decoder.activations(cfg, T, dev)
    bws = decoder.backward_workspace(cfg, T, dev)
    x0 = inputs.normal((T, cfg.d), 1.0, 301, dev)
    dy0 = inputs.normal((T, cfg.d), 1e-2, 302, dev)
    x, dy = torch.empty_like(x0), torch.empty_like(dy0)
    ms = []
    with torch.cuda.stream(s):
        for _ in range(2):
            x.copy_(x0)
            dy.copy_(dy0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            decoder.forward(x, w, cfg, work=ws, save=saved)
            decoder.backward(dy, w, cfg, saved, work=bws)
            e1.record(s)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
    flops = 3 * cfg.flops(T)
    print(json.dumps({"sweep": "llama layer training step, 2 steps", "tokens": T, "ms": ms,
                      "tflops": flops / ms[-1] / 1e9, "frac_of_fp32_peak": flops / ms[-1] / 1e9 / peak}),
          flush=True)


def run_sweep_train(dev, s, flush, peak):
    """The verifiable training step end to end: 4 contributors (DIDs), each
    with 2 x 2048 tokens through 2 Llama-3.2-1B-sized decoder layers (rotary,
    SwiGLU), forward and backward; their gradients folded in DID order into
    the mean, SGD on the flat theta (122 M parameters) and the Merkle root of
    theta.  Synthetic inputs and upstream gradients; the step is timed as a
    whole and by part."""
    from verifiable_repops_gemm_gb300 import decoder, train
    cfg = decoder.DecoderConfig()
    T, layers, C = 2 * cfg.seq_len, 2, 4
    model = train.Model(cfg, layers, dev, seed=700)
    ws = train.Workspace(model, T, dev)
    grads = [model.gradient_buffer() for _ in range(C)]
    contribs = [(b"did:zoo:contributor-%02d" % c, inputs.normal((T, cfg.d), 1.0, 710 + c, dev),
                 inputs.normal((T, cfg.d), 1e-2, 720 + c, dev)) for c in range(C)]
    theta0 = model.theta.clone()

    def step():
        model.theta.copy_(theta0)
        return train.train_step(model, contribs, 1e-3, ws, grads)

    with torch.cuda.stream(s):
        step()
        torch.cuda.synchronize(dev)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        flush.zero_()
        model.theta.copy_(theta0)
        ev[0].record(s)
        for (did, x, dy), g in zip(contribs, grads):
            train.contributor_gradient(model, x, dy, g, ws)
        ev[1].record(s)
        order = rp.sort_ids([did for did, _, _ in contribs])
        rp.fixed_order_mean_sgd(grads, order, 1e-3, model.theta, stream=s)
        ev[2].record(s)
        root = rp.merkle_sha256(model.theta, stream=s)
        ev[3].record(s)
    torch.cuda.synchronize(dev)
    total = ev[0].elapsed_time(ev[3])
    flops = 3 * layers * C * cfg.flops(T)
    n = model.theta.numel()
    print(json.dumps({"sweep": "verifiable training step: 4 contributors x 2 decoder layers x 4096 tokens, "
                               "fixed-order mean + SGD over %d parameters, Merkle root of theta" % n,
                      "ms": total, "tokens_per_s": C * T / total * 1e3, "tflops": flops / total / 1e9,
                      "frac_of_fp32_peak": flops / total / 1e9 / peak,
                      "gradients_ms": ev[0].elapsed_time(ev[1]), "mean_sgd_ms": ev[1].elapsed_time(ev[2]),
                      "commit_ms": ev[2].elapsed_time(ev[3]), "root": bytes(root.cpu().numpy()).hex()[:16]}),
          flush=True)


def run_sweep_halfstore(dev, s, flush, peak, hbm):
    """Half-precision storage around the binary32 path: the mean + SGD step of
    the hot path (16 contributors x 2^28) with bfloat16 gradients next to
    float32 ones, a float32 -> bfloat16 conversion, the 8192^3 GEMM on
    bfloat16 operands.  L2 flushed before each timed launch."""
    def ev_time(fn, reps=5):
        with torch.cuda.stream(s):
            fn()
            evs = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in evs) / reps

    nC, n = inputs.MEAN_CONTRIBUTORS, inputs.MEAN_LEN
    theta = inputs.normal((n,), 0.02, 500, dev)
    order = list(range(nC))
    for name, dt, size in (("float32", torch.float32, 4), ("bfloat16", torch.bfloat16, 2)):
        grads = [inputs.normal((n,), 1e-2, 510 + r, dev).to(dt) for r in range(nC)]
        ms = ev_time(lambda: rp.fixed_order_mean_sgd(grads, order, 1e-3, theta, stream=s))
        nb = n * (nC * size + 8)
        print(json.dumps({"sweep": "mean + SGD 16 x 2^28, %s gradients" % name, "ms": ms, "gbs": nb / ms / 1e6,
                          "frac_of_hbm": nb / ms / 1e6 / hbm}), flush=True)
        del grads
    x = inputs.normal((n,), 1.0, 520, dev)
    y = torch.empty(n, dtype=torch.bfloat16, device=dev)
    ms = ev_time(lambda: rp.convert(x, torch.bfloat16, out=y, stream=s))
    print(json.dumps({"sweep": "convert 2^28 float32 -> bfloat16", "ms": ms, "gbs": n * 6 / ms / 1e6,
                      "frac_of_hbm": n * 6 / ms / 1e6 / hbm}), flush=True)
    del x, y, theta
    N = GEMM_N
    A = inputs.normal((N, N), 1.0, 530, dev).to(torch.bfloat16)
    B = inputs.normal((N, N), 1.0, 531, dev).to(torch.bfloat16)
    C = torch.empty(N, N, device=dev)
    ms = ev_time(lambda: rp.gemm_typed(A, B, out=C, stream=s), reps=3)
    tf = 2.0 * N ** 3 / ms / 1e9
    print(json.dumps({"sweep": "gemm 8192^3 on bfloat16 operands (widened, binary32 k-chain)", "ms": ms,
                      "tflops": tf, "frac_of_fp32_peak": tf / peak}), flush=True)
    del A, B, C


def run_sweep_rolling(dev, s, flush, hbm):
    """The rolling hash of a 8192 x 4096-word uint32 batch, window 32 (128 MiB
    read, 256 MiB of hashes written).  L2 flushed before each timed launch;
    the mean of 10 launches."""
    rows, width, win = 8192, 4096, 32
    g = torch.Generator(device=dev)
    g.manual_seed(540)
    words = torch.randint(-(1 << 31), 1 << 31, (rows, width), generator=g, dtype=torch.int64,
                          device=dev).to(torch.int32)
    out = torch.empty(rows, width - win + 1, dtype=torch.int64, device=dev)
    with torch.cuda.stream(s):
        rp.rolling_hash(words, win, out=out, stream=s)
        evs = []
        for _ in range(10):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s)
            rp.rolling_hash(words, win, out=out, stream=s)
            e1.record(s)
            evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    ms = sum(a.elapsed_time(b) for a, b in evs) / len(evs)
    nb = words.numel() * 4 + out.numel() * 8
    print(json.dumps({"sweep": "rolling hash 8192 x 4096 uint32 words, window 32", "ms": ms,
                      "hashes_per_s": out.numel() / ms * 1e3, "gbs": nb / ms / 1e6,
                      "frac_of_hbm": nb / ms / 1e6 / hbm}), flush=True)


def run_sweep_commitments(dev, s, flush):
    """Merkle root versus whole stored tree of the 4 GiB tensor, one inclusion
    proof and one membership check, and replayed blocks of the 16 x 2^28
    workload (mean + SGD, then the root of theta)."""
    def ev_time(fn, reps):
        with torch.cuda.stream(s):
            fn()
            evs = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(s)
                fn()
                e1.record(s)
                evs.append((e0, e1))
        torch.cuda.synchronize(dev)
        return sum(a.elapsed_time(b) for a, b in evs) / reps

    T = inputs.normal((inputs.MERKLE_ELEMS,), 0.02, 300, dev)
    nb = T.numel() * 4
    ws = torch.empty(rp.merkle_workspace_bytes(nb), dtype=torch.uint8, device=dev)
    root = torch.empty(32, dtype=torch.uint8, device=dev)
    tree = torch.empty((rp.load().repops_merkle_tree_bytes(nb, 4096) // 32, 32), dtype=torch.uint8, device=dev)
    ms = ev_time(lambda: rp.merkle_sha256(T, 4096, out=root, workspace=ws, stream=s), 5)
    print(json.dumps({"sweep": "merkle root 4 GiB", "ms": ms, "gbs": nb / ms / 1e6}), flush=True)
    ms = ev_time(lambda: rp.merkle_tree(T, 4096, tree=tree, root=root, stream=s), 5)
    print(json.dumps({"sweep": "merkle whole tree 4 GiB (2^21 - 1 nodes stored)", "ms": ms,
                      "gbs": nb / ms / 1e6}), flush=True)
    nleaves = nb // 4096
    idx = nleaves - 12345
    with torch.cuda.stream(s):
        proof = rp.merkle_proof(tree, nleaves, idx, stream=s)
    ms = ev_time(lambda: rp.merkle_proof(tree, nleaves, idx, stream=s), 20)
    leaf = T.view(torch.uint8)[idx * 4096:(idx + 1) * 4096]
    ms_v = ev_time(lambda: rp.merkle_verify(leaf, nleaves, idx, proof, root, stream=s), 20)
    with torch.cuda.stream(s):
        okt = rp.merkle_verify(leaf, nleaves, idx, proof, root, stream=s)
    torch.cuda.synchronize(dev)
    ok = int(okt.item())
    print(json.dumps({"sweep": "inclusion proof (20 siblings) and membership check", "proof_us": ms * 1e3,
                      "verify_us": ms_v * 1e3, "verified": ok}), flush=True)
    del T, tree, ws
    nC, ln = inputs.MEAN_CONTRIBUTORS, inputs.MEAN_LEN
    grads = [inputs.normal((ln,), 1e-2, 200 + r, dev) for r in range(nC)]
    theta = inputs.normal((ln,), 0.02, 199, dev)
    order = rp.sort_ids(inputs.contributor_ids(nC, 200))
    blocks = 3
    roots = torch.empty((blocks, 32), dtype=torch.uint8, device=dev)
    ms = ev_time(lambda: rp.replay([grads] * blocks, [order] * blocks, [1e-3] * blocks, theta, 4096,
                                   roots=roots, stream=s), 3) / blocks
    per_block = (nC + 2) * ln * 4 + ln * 4
    print(json.dumps({"sweep": "replay, per block: mean+SGD of 16 x 2^28 then root of theta (1 GiB)",
                      "ms_per_block": ms, "gbs": per_block / ms / 1e6}), flush=True)


def run_gemm_once(spec):
    """A few launches of one automatic-choice GEMM (M,N,K with N(0,1)
    operands, A row-major): for profiling one kernel in isolation.  Prints the
    kernel the automatic choice runs and the event time of the last launch."""
    M, N, K = (int(x) for x in spec.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rp.load()
    A = inputs.normal((M, K), 1.0, 1, dev)
    B = inputs.normal((K, N), 1.0, 2, dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    s = torch.cuda.Stream(device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        for i in range(3):
            if i == 2:
                e0.record(s)
            rp.gemm(A, B, out=C, stream=s)
        e1.record(s)
    torch.cuda.synchronize(dev)
    if rp.device_status(s) != 0:
        raise RuntimeError("a kernel reported a timed-out wait")
    print(json.dumps({"gemm": [M, N, K], "config": rp.gemm_auto_config(M, N, K),
                      "chained": rp.gemm_auto_chained(M, N, K), "ms": e0.elapsed_time(e1)}), flush=True)


def run_attention_once():
    """The unfused attention of one 2048-token sequence of the decoder layer
    (32 query / 8 key-value heads of 64): the scores QK^T with alpha 1/8 and
    the causal tile skip, the causal softmax, and P V over the band k <= i,
    three times: for profiling those kernels in isolation."""
    from verifiable_repops_gemm_gb300 import decoder
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rp.load()
    cfg = decoder.DecoderConfig()
    S, dh, kv, H = cfg.seq_len, cfg.d_head, cfg.kv_heads, cfg.heads
    qkv = inputs.normal((S, cfg.qkv_width), 1.0, 1, dev)
    k0, v0 = cfg.d, cfg.d + kv * dh
    sc = torch.empty((H, S, S), device=dev)
    out = torch.empty((S, cfg.d), device=dev)
    rows = slice(0, S)
    Q, K = decoder._heads(qkv, rows, 0, H, dh), decoder._kv(qkv, rows, k0, kv, dh)
    V, O = decoder._kv(qkv, rows, v0, kv, dh), decoder._heads(out, rows, 0, H, dh)
    for _ in range(3):
        rp.gemm_batched(Q, K.transpose(1, 2), out=sc, alpha=1.0 / 8.0, causal_first=0)
        rp.softmax_rows(sc.view(H * S, S), out=sc.view(H * S, S), causal_first=0, causal_period=S)
        rp.gemm_batched(sc, V, out=O, k_hi=0)
    torch.cuda.synchronize(dev)
    if rp.device_status() != 0:
        raise RuntimeError("a kernel reported a timed-out wait")
    print(json.dumps({"attention_once": "ok"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", nargs="?", const="all", default=None,
                    choices=("all", "gemm", "rowops", "commitments", "decoder", "halfstore", "rolling",
                             "train", "decoder_step"),
                    help="time every workload of a part (one JSON line each) instead of the step")
    ap.add_argument("--gemm-once", metavar="M,N,K", default=None,
                    help="three launches of one automatic-choice GEMM (for a profiler)")
    ap.add_argument("--attention-once", action="store_true",
                    help="three passes of one sequence's unfused attention kernels (for a profiler)")
    ap.add_argument("--config", type=int, choices=range(5), default=None,
                    help="one JSON line per workload of one of the five workload configurations: 0 the "
                         "256^3 GEMM, 1 the square sweep and the ragged GEMM, 2 the decoder GEMM set, 3 the "
                         "mean + SGD, 4 the Merkle commitments")
    ap.add_argument("--tile", type=int, default=-1,
                    help="the step's GEMM tile configuration (default -1: the automatic choice); the "
                         "commitments are the same for every one")
    ap.add_argument("--seed", type=int, default=0, help="added to every input seed of the step")
    args = ap.parse_args()
    if args.config is not None:
        run_config(args.config)
    elif args.attention_once:
        run_attention_once()
    elif args.gemm_once:
        run_gemm_once(args.gemm_once)
    elif args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
