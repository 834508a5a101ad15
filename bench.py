"""Benchmark of the batched speculative-decoding verify step on GB300.

One step = one verify call (one batch) of a named workload; the default is
B=64, k=5, V=128256 (Llama-3 vocabulary), bf16 target logits, T=1.  Every
call streams its inputs from HBM: large workloads cycle through enough
copies of their inputs to exceed twice the L2 (replayed from a CUDA graph);
workloads too small for that have the L2 flushed (a 2x-L2 read) before
every call, each call timed by its own pair of CUDA events.  Prints one JSON
line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload toy|zipf|benchmark|mixed|split_v]

--impl reference times the float64 CPU oracle on this host's cores on a
bounded sample of the same workload (the reference arm of this build: the
pages ship no GPU implementation); its steps cycle through all the
workload's rows.  Under torchrun with N > 1 every rank runs an independent
replica on its own GPU (rows are independent; no collective on the data
path) and the slowest rank's time counts.
"""
import argparse
import hashlib
import re
import glob
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "verify B=64 k=5 V=128256 bf16 T=1 (Llama-3 vocabulary, +8 spike, q=softmax(L+N(0,1)))"
WORKLOAD_NAME = "benchmark"
# what each named workload is (tests/ and the oracle use the same generators)
WORKLOADS_DESC = {
    "toy": "verify B=1 k=4 V=1000 fp32 T=1 (toy: L ~ N(0,2^2) iid, q = softmax(L + N(0,1)), fresh seeded inputs)",
    "zipf": "verify B=8 k=4 V=32000 bf16 T=0.8 (L ~ N(0,3^2) + 6 at one Zipf(1.1)-ranked token per row, "
            "q = softmax(L + N(0,1.5^2)))",
    "benchmark": WORKLOAD,
    "mixed": "verify B=256 k=8 V=128256 bf16 (rows 0..127 greedy T=0, rows 128..255 T=0.7; +8 spike; draft noise "
             "sigma ~ U(0.5,3) per row)",
    "split_v": "verify B=16 k=16 V=151936 fp32 T=1 (L ~ N(0,4^2), q = softmax(L + N(0,2^2)); split-vocabulary clusters)",
}
N_SETS = 4
MAX_SETS = 256  # more input copies than this: flush the L2 between calls instead
NOMINAL_HBM_GBS = 8000.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--graph-calls", type=int, default=100)
    p.add_argument("--variant", choices=["sample", "onehot", "tree", "filtered", "rollback"], default="sample",
                   help="onehot: the same workload verified as one-hot drafts (q = None); tree: greedy "
                        "verification of 16-node draft trees over the same vocabulary")
    p.add_argument("--top-k", type=int, default=None,
                   help="filtered variant: top_k of every row (default 40; above 64 the radix-select kernel)")
    p.add_argument("--top-p", type=float, default=None, help="filtered variant: top_p of every row (default 0.95)")
    p.add_argument("--workload", choices=list(WORKLOADS_DESC), default=WORKLOAD_NAME,
                   help="the named synthetic workload of the sample / onehot variants (and of the reference arm)")
    return p.parse_args(argv)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(value, world_size, device=None):
    """Max of a float over the ranks of the default process group."""
    if world_size <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def algorithmic_bytes(w, num_accepted, row_status, onehot=False):
    """Bytes the verify step must move for one call: every logit once, the
    draft-probability row at each rejected sampled position, the gathered
    q(x), x and accept uniforms, the draw uniform and temperature, and the
    outputs (num_accepted, out_tokens, row_status).  One-hot drafts read no
    q at all."""
    import numpy as np

    B, k, V = w.B, w.k, w.V
    esz = 2 if w.dtype == "bf16" else 4
    ok = (row_status & 0x2F) == 0
    rejected = ok & (w.T != 0) & (num_accepted < k)
    qrow = 0 if onehot else int(rejected.sum()) * V * 4
    return (B * (k + 1) * V * esz + qrow + B * k * (8 if onehot else 12) + B * 12 + B * (k + 2) * 4)


def rule_bytes(w, num_accepted, row_status, onehot=False):
    """Bytes the rule itself needs for one call: of each row's logits only
    positions 0..j (j = num_accepted: no test after the first rejection
    looks further), plus what algorithmic_bytes counts besides the logits.
    Rows that end in an error count every position."""
    import numpy as np

    B, k, V = w.B, w.k, w.V
    esz = 2 if w.dtype == "bf16" else 4
    ok = (row_status & 0x2F) == 0
    pos = np.where(ok, np.minimum(num_accepted, k) + 1, k + 1)
    return (algorithmic_bytes(w, num_accepted, row_status, onehot) - B * (k + 1) * V * esz
            + int(pos.sum()) * V * esz)


TREE_M = 16


def make_tree_workload(seed, B=64, M=TREE_M, V=128256):
    """Greedy draft trees over the benchmark vocabulary: logits as in the
    benchmark workload (N(0, 3^2) + an +8 spike per row, bf16), each node's
    parent uniform among the prefix and the earlier nodes, and its token the
    argmax of its parent's row with probability 0.8 (else uniform)."""
    import numpy as np

    from speculative_decoding_verification_57_gb300 import workloads as W

    rng = np.random.default_rng(seed)
    L = rng.normal(scale=3.0, size=(B, M + 1, V))
    L[np.arange(B)[:, None], np.arange(M + 1)[None, :], rng.integers(0, V, size=(B, M + 1))] += 8.0
    Lb = W.f32_to_bf16_bits(L.astype(np.float32))
    A = np.argmax(W.bf16_bits_to_f32(Lb), axis=-1)
    par = np.array([[int(rng.integers(-1, i)) for i in range(M)] for _ in range(B)], np.int32)
    tok = rng.integers(0, V, size=(B, M)).astype(np.int32)
    keep = rng.random((B, M)) < 0.8
    for b in range(B):
        for i in range(M):
            if keep[b, i]:
                tok[b, i] = A[b, par[b, i] + 1]
    return Lb, tok, par


# The sources each profiled kernel is built from: a committed ncu summary
# counts only while these are unchanged.
_CLUSTER_SOURCES = ["verify_cluster.cuh", "ptx.cuh", "exp2dd.cuh", "specv.cu"]
_WARP_SOURCES = ["verify_warp.cuh", "verify_cluster.cuh", "ptx.cuh", "exp2dd.cuh", "specv.cu"]
KERNEL_SOURCES = {
    "verify_cluster_kernel_B64_k5_V128256_bf16": _CLUSTER_SOURCES,
    "verify_row_kernel_toy_B1_k4_V1000_f32": _WARP_SOURCES,
    "verify_cluster_kernel_zipf_B8_k4_V32000_bf16": _CLUSTER_SOURCES,
    "verify_cluster_kernel_mixed_B256_k8_V128256_bf16": _CLUSTER_SOURCES,
    "verify_cluster_kernel_split_v_B16_k16_V151936_f32": _CLUSTER_SOURCES,
    "verify_cluster_kernel_onehot_B64_k5_V128256_bf16": _CLUSTER_SOURCES,
    "verify_cluster_kernel_tree_B64_M16_V128256_bf16": _CLUSTER_SOURCES,
    "verify_topk_kernel_B64_k5_V128256_bf16": ["verify_topk.cuh"] + _CLUSTER_SOURCES,
    "verify_topk_wide_kernel_B64_k5_V128256_bf16_K4096": ["verify_topk_wide.cuh", "verify_topk.cuh"] + _CLUSTER_SOURCES,
    "rollback_kernel_B4096_k8": ["rollback.cuh", "specv.cu"],
}


def _code_only(text):
    """A source file without its comments and blank lines: edits to comments
    leave a kernel, and so its profile, unchanged."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash(files):
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "speculative_decoding_verification_57_gb300", "csrc", name)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(name="verify_cluster_kernel_B64_k5_V128256_bf16"):
    """DRAM traffic per launch of a kernel from its committed ncu summary,
    if it was taken on the kernel's current sources."""
    if name not in KERNEL_SOURCES:
        return None
    path = os.path.join(ROOT, "profiles", name + ".json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_hash") != kernel_source_hash(KERNEL_SOURCES[name]):
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons over a window."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return None
        inside = [r for r in rows if self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        used = inside or rows
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in used:
            for name, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": sorted(reasons), "samples": len(used), "in_window": bool(inside)}


def small_v_kernel(B, sms):
    """The kernel the library runs for a vocabulary of at most 2048: one CTA
    of eight warps per row while the batch is at most twice the SM count,
    else one warp per row; SPECV_SMALLV=row|warp forces either."""
    env = os.environ.get("SPECV_SMALLV")
    if env in ("row", "warp"):
        return f"verify_{env}_kernel"
    return "verify_row_kernel" if B <= 2 * sms else "verify_warp_kernel"


def profile_name(workload, w, onehot=False, sms=152):
    """The committed ncu summary of a workload's verify kernel."""
    if workload == WORKLOAD_NAME:
        return "verify_cluster_kernel_onehot_B64_k5_V128256_bf16" if onehot else "verify_cluster_kernel_B64_k5_V128256_bf16"
    kern = small_v_kernel(w.B, sms) if w.V <= 2048 else "verify_cluster_kernel"
    return f"{kern}_{workload}_B{w.B}_k{w.k}_V{w.V}_{'bf16' if w.dtype == 'bf16' else 'f32'}"


def logits_tensor(w):
    """The workload's logits as a CPU tensor of their own type (bf16 or fp32)."""
    import numpy as np
    import torch

    if w.dtype == "bf16":
        return torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(w.logits)


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's name as /proc/cpuinfo gives it (x86: model name; Arm:
    implementer / part codes)."""
    import platform

    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model"):
        for line in info:
            if line.startswith(key):
                return line.split(":", 1)[1].strip()
    impl = next((l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")), "?")
    part = next((l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")), "?")
    return f"{platform.machine()} implementer {impl} part {part}"


def time_oracle(w, budget_s, max_rows=None, nthreads=None):
    """Rows/s of the float64 oracle over (a bounded sample of) workload w
    on nthreads host threads (default: all cores); also the oracle's
    outputs on that sample, for the comparison with the GPU's."""
    import oracle

    rows = w.B if max_rows is None else min(w.B, max_rows)
    sl = slice(0, rows)
    args = (w.logits[sl], None if w.q is None else w.q[sl], w.x[sl], w.u[sl], w.T[sl])
    cores = host_cores() if nthreads is None else nthreads
    ref = oracle.verify(*args, nthreads=cores)  # warm (page in)
    n, t0 = 0, time.perf_counter()
    while True:
        ref = oracle.verify(*args, nthreads=cores)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s and n >= 2:
            break
    return (rows * n / el, cores, f"{n} oracle calls x {rows} rows of the {w.name} workload, {el:.2f} s wall",
            ref)


def compare_rows(ref, got, keys=("num_accepted", "out_tokens", "row_status")):
    """Rows where the GPU's outputs differ from the oracle's (ref, computed
    in the CPU-baseline leg on the first len(ref) rows); with the oracle's
    boundary flags (a uniform within 1e-6 of a decision edge) when it has
    them."""
    import numpy as np

    rows = len(ref[keys[0]])
    same = np.ones(rows, bool)
    for kk in keys:
        a, r = np.asarray(got[kk])[:rows], np.asarray(ref[kk])
        same &= (a == r).reshape(rows, -1).all(1)
    out = {"rows": rows, "differ": int((~same).sum())}
    if "boundary" in ref:
        flagged = np.asarray(ref["boundary"]) != 0
        out["differ_unflagged"] = int((~same & ~flagged).sum())
        out["flagged"] = int(flagged.sum())
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from speculative_decoding_verification_57_gb300 import workloads as W

    import oracle

    name = args.workload
    w = W.make_workload(name)
    B = w.B
    cores = host_cores()

    def rows(a, b):
        q = None if w.q is None else w.q[a:b]
        return (w.logits[a:b], q, w.x[a:b], w.u[a:b], w.T[a:b])

    # the time of one row, from a warm call over the whole batch
    oracle.verify(*rows(0, B), nthreads=cores)
    t0 = time.perf_counter()
    oracle.verify(*rows(0, B), nthreads=cores)
    per_row = (time.perf_counter() - t0) / B
    # rows per step: the whole batch when all steps fit about two minutes,
    # else a window that moves on by its own length each step, so that
    # consecutive steps cover every row of the batch
    n = max(1, min(B, int(120.0 / (max(1, args.steps + args.warmup) * per_row))))

    def step(s):
        a = (s * n) % B
        if a + n <= B:
            oracle.verify(*rows(a, a + n), nthreads=cores)
        else:
            oracle.verify(*rows(a, B), nthreads=cores)
            oracle.verify(*rows(0, a + n - B), nthreads=cores)

    for s_ in range(max(0, args.warmup)):
        step(s_)
    t0 = time.perf_counter()
    for s_ in range(args.steps):
        step(s_)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = (f"each step: the oracle over {n} of the {B} rows of the {name} workload"
              + ("" if n == B else f" (a window moving {n} rows a step: the steps cover every row)"))
    line = {
        "impl": "reference", "metric": "verify rows/s", "value": value, "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOADS_DESC[name], "B": B, "k": w.k, "V": w.V,
                   "logits": "bf16" if w.dtype == "bf16" else "fp32", "rows_per_step": n},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import numpy as np
    import torch

    import speculative_decoding_verification_57_gb300 as sv
    from speculative_decoding_verification_57_gb300 import workloads as W

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    if args.variant == "tree":
        return run_tree(args, sv, dev, rank, ws, local, hbm_peak, peak_src)
    if args.variant == "filtered":
        return run_filtered(args, sv, dev, rank, ws, local, hbm_peak, peak_src)
    if args.variant == "rollback":
        return run_rollback(args, sv, dev, rank, ws, local, hbm_peak, peak_src)
    name = args.workload
    w = W.make_workload(name, seed=W.WORKLOADS[name][1] + 1000 * rank)
    onehot = args.variant == "onehot"
    if onehot:
        w = W.Workload(w.name, w.dtype, w.logits, None, w.x, w.u, w.T)
    B, k, V = w.B, w.k, w.V
    h = sv.specv_create(local, max_batch=B, max_k=k, vocab=V)
    L0 = logits_tensor(w)
    # enough copies of the inputs that a call never finds its own in the L2;
    # where that takes too many, the L2 is flushed before every call instead
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2 ** 20)
    set_bytes = w.logits.nbytes + (0 if onehot else w.q.nbytes)
    n_need = -(-int(2.05 * l2) // set_bytes)
    flushed = n_need > MAX_SETS
    n_sets = 1 if flushed else max(N_SETS, n_need)
    sets = []
    for _ in range(n_sets):
        sets.append(dict(L=L0.to(dev), q=None if onehot else torch.from_numpy(w.q).to(dev),
                         x=torch.from_numpy(w.x).to(dev), u=torch.from_numpy(w.u).to(dev),
                         T=torch.from_numpy(w.T).to(dev)))
    outs = [dict(num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                 out_tokens=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
                 row_status=torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(n_sets)]
    stream = torch.cuda.Stream(device=dev)

    def call(i):
        s_ = sets[i % n_sets]
        sv.specv_verify_sample(h, s_["L"], s_["q"], s_["x"], s_["u"], s_["T"], out=outs[i % n_sets], stream=stream)

    # outcome of the timed inputs (for the byte count), outside the timed region
    with torch.cuda.stream(stream):
        call(0)
    stream.synchronize()
    got = {kk: v.cpu().numpy() for kk, v in outs[0].items()}
    if np.any(got["row_status"] & sv.ST_ERROR_MASK):
        raise RuntimeError(f"verify reported data errors on the {name} inputs")
    alg = algorithmic_bytes(w, got["num_accepted"], got["row_status"], onehot)
    needed = rule_bytes(w, got["num_accepted"], got["row_status"], onehot)

    launches_before = sv.specv_launch_count(h)
    sampler = ClockSampler(local)
    if flushed:
        # each call alone: a 2x-L2 read (the L2 then holds clean lines of
        # another buffer, nothing to write back), then the call between its
        # own events
        flush = torch.ones(2 * l2 // 4, dtype=torch.int32, device=dev)
        flush_out = torch.empty((), dtype=torch.int64, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup)):
                torch.sum(flush, dim=0, out=flush_out)
                torch.cuda._sleep(200_000)
                call(i)
        stream.synchronize()
        launch_mode = f"direct launches, L2 flushed ({2 * l2 / 1e6:.0f} MB read) before each call"
        l2_desc = (f"L2 flushed before every call ({2 * l2 / 1e6:.0f} MB read, outside the call's event pair); "
                   "the sum of the per-call event times is the timed total")
        if rank == 0:
            sampler.start()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        sampler.mark("t0")
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                torch.sum(flush, dim=0, out=flush_out)
                # a ~100 us device-side pause after the flush: the host has
                # queued the call before the GPU reaches its first event
                torch.cuda._sleep(200_000)
                evs[i][0].record(stream)
                call(i)
                evs[i][1].record(stream)
        stream.synchronize()
        sampler.mark("t1")
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs)
    else:
        # capture G calls (cycling through the sets) into a CUDA graph
        G = max(1, min(max(args.graph_calls, n_sets), args.steps))

        def capture(ncalls):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.stream(stream):
                call(0)  # keep the capture stream warm
                stream.synchronize()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(ncalls):
                        call(i)
            return g

        rem = args.steps % G
        reps = args.steps // G
        try:
            g_main = capture(G)
            g_rem = capture(rem) if rem else None
            launch_mode = f"CUDA graph of {G} calls"
        except RuntimeError:
            # capture refused: time direct launches instead
            stream.synchronize()
            g_main = g_rem = None
            launch_mode = "direct launches"

        class Direct:
            def __init__(self, n):
                self.n = n

            def replay(self):
                for i in range(self.n):
                    call(i)

        if g_main is None:
            g_main = Direct(G)
            g_rem = Direct(rem) if rem else None
        with torch.cuda.stream(stream):
            for _ in range(max(1, (max(3, args.warmup) + G - 1) // G)):
                g_main.replay()
        stream.synchronize()
        l2_desc = f"rotating {n_sets} input sets ({n_sets * set_bytes / 1e9:.2f} GB) > 2x L2"
        if rank == 0:
            sampler.start()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        sampler.mark("t0")
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                g_main.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(stream)
        ev1.synchronize()
        sampler.mark("t1")
        torch.cuda.synchronize()
        ms = ev0.elapsed_time(ev1)
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    ms_max = reduce_max(ms, ws, dev)
    per_call_s = ms / 1e3 / args.steps
    value = B * args.steps * ws / (ms_max / 1e3)
    launches_timed = sv.specv_launch_count(h) - launches_before

    # end to end through the host-buffer entry point (pinned memory in/out)
    pin = dict(L=L0.pin_memory(), q=None if onehot else torch.from_numpy(w.q).pin_memory(), x=torch.from_numpy(w.x).pin_memory(),
               u=torch.from_numpy(w.u).pin_memory(), T=torch.from_numpy(w.T).pin_memory())
    host_out = dict(num_accepted=torch.empty(B, dtype=torch.int32).pin_memory(),
                    out_tokens=torch.empty((B, k + 1), dtype=torch.int32).pin_memory(),
                    row_status=torch.empty(B, dtype=torch.int32).pin_memory())
    for _ in range(3):
        sv.specv_verify_sample_host(h, pin["L"], pin["q"], pin["x"], pin["u"], pin["T"], out=host_out, stream=stream)
    if ws > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        sv.specv_verify_sample_host(h, pin["L"], pin["q"], pin["x"], pin["u"], pin["T"], out=host_out, stream=stream)
    e2e_s = reduce_max(time.perf_counter() - t0, ws, dev)
    # q is page-locked, so the kernel reads in place only the entries it needs: q at
    # the draft tokens and the rejecting rows' stop rows; the other inputs are copied
    q_in_place = 0 if onehot else (int(((got["num_accepted"] < k) & (w.T > 0)).sum()) * V * 4 + B * k * 4)
    h2d = sum(t.numel() * t.element_size() for kk, t in pin.items() if t is not None and kk != "q") + q_in_place
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    assert np.array_equal(host_out["num_accepted"].numpy(), got["num_accepted"])

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return 0

    cpu_value, cores, sample, ref = time_oracle(w, budget_s=1.5)
    cpu_one, _, _, _ = time_oracle(w, budget_s=1.0, max_rows=8, nthreads=1)
    parity = compare_rows(ref, got)
    achieved = alg / per_call_s / 1e9
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    traffic = measured_traffic(profile_name(name, w, onehot, sms))
    temps = sorted(set(float(t) for t in w.T))
    if V > 2048:
        launch_desc = specv_cluster_desc(sv, h, B, k, V)
    elif small_v_kernel(B, sms) == "verify_row_kernel":
        launch_desc = f"one CTA of 8 warps per row, {B} CTA{'' if B == 1 else 's'} (verify_row_kernel)"
    else:
        launch_desc = f"one warp per row, {(B + 1) // 2} CTAs of 2 warps (verify_warp_kernel)"
    line = {
        "metric": "verify rows/s",
        "value": value,
        "unit": "rows/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_max / args.steps,
        "us_per_call": 1e3 * ms_max / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": WORKLOADS_DESC[name] + (", one-hot drafts (q = None)" if onehot else ""), "name": name,
            "B": B, "k": k, "V": V, "logits": "bf16" if w.dtype == "bf16" else "fp32",
            "T": temps[0] if len(temps) == 1 else temps,
            "global_batch": B * ws, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
            "l2": l2_desc,
            "launch": f"{launch_mode}, {launch_desc}",
        },
        "logits_per_s": B * (k + 1) * V * args.steps * ws / (ms_max / 1e3),
        "roofline": {
            "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s", "frac": achieved / hbm_peak,
            "traffic": traffic, "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
            "algorithmic_bytes_per_launch": alg, "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
            # every logit counts once above; the rule reads no position after a
            # row's first rejection, and the kernel does not either
            "rule_bytes_per_launch": needed, "achieved_rule": needed / per_call_s / 1e9,
            "frac_rule": needed / per_call_s / 1e9 / hbm_peak,
        },
        "cpu_baseline": {"value": cpu_value, "unit": "rows/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "single_thread_value": cpu_one, "cpu_model": cpu_model(),
                         "gpu_outputs_vs_oracle": parity},
        "e2e": {"value": B * args.e2e_steps * ws / e2e_s, "unit": "rows/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                "q_bytes_read_in_place": q_in_place,
                "path": "specv_verify_sample_host (pinned host buffers: logits, x, u, T copied, q read in place "
                        "by the kernel; kernel + outputs copied back + sync per step)"},
        "gpu_launches": args.steps,
        "host_launch_calls": launches_timed,
        "mean_num_accepted": float(np.mean(got["num_accepted"])),
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_tree(args, sv, dev, rank, ws, local, hbm_peak, peak_src):
    """Greedy tree verification: rows/s over 16-node trees, V = 128256 bf16."""
    import numpy as np
    import torch


    Lb, tok, par = make_tree_workload(57100 + 1000 * rank)
    B, M1, V = Lb.shape
    M = M1 - 1
    h = sv.specv_create(local, max_batch=B, max_k=M, vocab=V)
    L0 = torch.from_numpy(Lb.view(np.int16)).view(torch.bfloat16)
    sets = [dict(L=L0.to(dev), t=torch.from_numpy(tok).to(dev), p=torch.from_numpy(par).to(dev))
            for _ in range(N_SETS)]
    outs = [dict(num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                 out_tokens=torch.empty((B, M + 1), dtype=torch.int32, device=dev),
                 path=torch.empty((B, M), dtype=torch.int32, device=dev),
                 row_status=torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(N_SETS)]
    stream = torch.cuda.Stream(device=dev)

    def call(i):
        s = sets[i % N_SETS]
        sv.specv_verify_tree_greedy(h, s["L"], s["t"], s["p"], out=outs[i % N_SETS], stream=stream)

    with torch.cuda.stream(stream):
        call(0)
    stream.synchronize()
    got = {kk: v.cpu().numpy() for kk, v in outs[0].items()}
    alg = B * M1 * V * 2 + B * M * 8 + B * 4 + B * M1 * 4 + B * M * 4 + B * 4
    G = max(1, min(args.graph_calls, args.steps))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        call(0)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                call(i)
    reps = max(1, args.steps // G)
    steps = reps * G
    with torch.cuda.stream(stream):
        for _ in range(max(1, (args.warmup + G - 1) // G)):
            g.replay()
    stream.synchronize()
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("t0")
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    sampler.mark("t1")
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    ms_max = reduce_max(ev0.elapsed_time(ev1), ws, dev)
    per_call_s = ms_max / 1e3 / steps
    # end to end: pinned host inputs copied in, outputs read back, every step
    pin = dict(L=L0.pin_memory(), t=torch.from_numpy(tok).pin_memory(), p=torch.from_numpy(par).pin_memory())
    host_out = {kk: torch.empty_like(v, device="cpu").pin_memory() for kk, v in outs[0].items()}
    e2e_steps = max(1, args.e2e_steps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            s = sets[0]
            s["L"].copy_(pin["L"], non_blocking=True)
            s["t"].copy_(pin["t"], non_blocking=True)
            s["p"].copy_(pin["p"], non_blocking=True)
            call(0)
            for kk in host_out:
                host_out[kk].copy_(outs[0][kk], non_blocking=True)
        stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, ws, dev)
    if rank != 0:
        return 0
    import oracle  # the CPU-baseline leg

    ref = oracle.tree_greedy(Lb[:8], tok[:8], par[:8])
    n, t1 = 0, time.perf_counter()
    while time.perf_counter() - t1 < 1.5 or n < 2:
        ref = oracle.tree_greedy(Lb[:8], tok[:8], par[:8])
        n += 1
    cpu_value = 8 * n / (time.perf_counter() - t1)
    parity = compare_rows(ref, got, keys=("num_accepted", "out_tokens", "path", "row_status"))
    achieved = alg / per_call_s / 1e9
    line = {
        "metric": "tree-verify rows/s", "value": B * steps * ws / (ms_max / 1e3), "unit": "rows/s", "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms_max / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"greedy tree verify B={B} M={M} nodes V={V} bf16 (random trees, 0.8 of tokens "
                               "the parent's argmax)", "B": B, "M": M, "V": V, "global_batch": B * ws,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": f"rotating {N_SETS} input sets ({N_SETS * Lb.nbytes / 1e9:.2f} GB) > 2x L2",
                   "launch": f"CUDA graph of {G} calls, {specv_cluster_desc(sv, h, B, M, V)}"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": measured_traffic("verify_cluster_kernel_tree_B64_M16_V128256_bf16"),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
                     "algorithmic_bytes_per_launch": alg},
        "cpu_baseline": {"value": cpu_value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} oracle calls x 8 rows, one thread", "gpu_outputs_vs_oracle": parity},
        "e2e": {"value": B * e2e_steps * ws / e2e_s, "unit": "rows/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out.values()),
                "steps": e2e_steps, "path": "pinned copies + specv_verify_tree_greedy + copies back, per step"},
        "gpu_launches": steps, "mean_num_accepted": float(np.mean(got["num_accepted"])), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


FILTER_TOP_K, FILTER_TOP_P = 40, 0.95


def run_filtered(args, sv, dev, rank, ws, local, hbm_peak, peak_src):
    """Sampled verification with top-k / top-p (default 40 / 0.95) on the
    target rows, on the benchmark workload (B=64, k=5, V=128256 bf16)."""
    import numpy as np
    import torch

    from speculative_decoding_verification_57_gb300 import workloads as W

    top_k = FILTER_TOP_K if args.top_k is None else args.top_k
    top_p = FILTER_TOP_P if args.top_p is None else args.top_p
    wide = top_k > 64
    w = W.make_workload(WORKLOAD_NAME, seed=W.WORKLOADS[WORKLOAD_NAME][1] + 1000 * rank)
    B, k, V = w.B, w.k, w.V
    tk = np.full(B, top_k, np.int32)
    tp = np.full(B, top_p, np.float32)
    h = sv.specv_create(local, max_batch=B, max_k=k, vocab=V)
    L0 = torch.from_numpy(w.logits.view(np.int16)).view(torch.bfloat16)
    host = dict(L=L0, q=torch.from_numpy(w.q), x=torch.from_numpy(w.x), u=torch.from_numpy(w.u),
                T=torch.from_numpy(w.T), tk=torch.from_numpy(tk), tp=torch.from_numpy(tp))
    sets = [{kk: v.to(dev) for kk, v in host.items()} for _ in range(N_SETS)]
    outs = [dict(num_accepted=torch.empty(B, dtype=torch.int32, device=dev),
                 out_tokens=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
                 row_status=torch.empty(B, dtype=torch.int32, device=dev)) for _ in range(N_SETS)]
    stream = torch.cuda.Stream(device=dev)

    def call(i, s=None, o=None):
        s = s or sets[i % N_SETS]
        sv.specv_verify_sample_filtered(h, s["L"], s["q"], s["x"], s["u"], s["T"], s["tk"], s["tp"],
                                        out=o or outs[i % N_SETS], stream=stream)

    with torch.cuda.stream(stream):
        call(0)
    stream.synchronize()
    got = {kk: v.cpu().numpy() for kk, v in outs[0].items()}
    if np.any(got["row_status"] & sv.ST_ERROR_MASK):
        raise RuntimeError("filtered verify reported data errors on the benchmark inputs")
    # every logit once; q read at the kept entries of the stop row (at most top_k per row); the
    # per-position q(x), x, u and T; top_k, top_p; outputs
    rejected = got["num_accepted"] < k
    alg = (B * (k + 1) * V * 2 + int(rejected.sum()) * min(top_k, V) * 4 + B * k * 12 + B * 12 + B * 8
           + B * (k + 2) * 4)
    G = max(1, min(args.graph_calls, args.steps))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        call(0)
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                call(i)
    reps = max(1, args.steps // G)
    steps = reps * G
    with torch.cuda.stream(stream):
        for _ in range(max(1, (args.warmup + G - 1) // G)):
            g.replay()
    stream.synchronize()
    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark("t0")
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    sampler.mark("t1")
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    ms_max = reduce_max(ev0.elapsed_time(ev1), ws, dev)
    per_call_s = ms_max / 1e3 / steps
    # end to end: pinned host inputs copied in, outputs read back, every step
    pin = {kk: v.pin_memory() for kk, v in host.items()}
    host_out = {kk: torch.empty_like(v, device="cpu").pin_memory() for kk, v in outs[0].items()}
    e2e_steps = max(1, args.e2e_steps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    # q stays in page-locked host memory: the kernel reads q at the draft tokens and at the
    # stop row's kept entries in place; the other inputs are copied
    e2e_set = dict(sets[0], q=pin["q"])
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            for kk in pin:
                if kk != "q":
                    sets[0][kk].copy_(pin[kk], non_blocking=True)
            call(0, s=e2e_set)
            for kk in host_out:
                host_out[kk].copy_(outs[0][kk], non_blocking=True)
        stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, ws, dev)
    assert np.array_equal(host_out["num_accepted"].numpy(), got["num_accepted"])
    q_in_place = B * k * 4 + int(rejected.sum()) * min(top_k, V) * 4
    if rank != 0:
        return 0
    import oracle  # the CPU-baseline leg

    cores = 1
    sl = slice(0, 8)
    oargs = (w.logits[sl], w.q[sl], w.x[sl], w.u[sl], w.T[sl], tk[sl], tp[sl])
    ref = oracle.verify_warped(*oargs)
    n, t1 = 0, time.perf_counter()
    while time.perf_counter() - t1 < 1.5 or n < 2:
        ref = oracle.verify_warped(*oargs)
        n += 1
    cpu_value = 8 * n / (time.perf_counter() - t1)
    parity = compare_rows(ref, got)
    achieved = alg / per_call_s / 1e9
    line = {
        "metric": "filtered-verify rows/s", "value": B * steps * ws / (ms_max / 1e3), "unit": "rows/s",
        "n_gpus": ws, "steps": steps, "warmup": args.warmup, "ms_per_step": ms_max / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD + f", top_k {top_k}, top_p {top_p}", "B": B, "k": k, "V": V,
                   "global_batch": B * ws, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": f"rotating {N_SETS} input sets ({N_SETS * (w.logits.nbytes + w.q.nbytes) / 1e9:.2f} GB) "
                         "> 2x L2",
                   "launch": f"CUDA graph of {G} calls, two launches a call: the top-64 kernel "
                             f"({B * min(k + 1, 8)} CTAs in clusters of {min(k + 1, 8)}) and the radix-select "
                             f"kernel ({B * min(k + 1, 16)} CTAs of 256 threads in clusters of {min(k + 1, 16)}); "
                             f"the rows are the {'second' if wide else 'first'}'s, the other's CTAs exit at once"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak,
                     "traffic": measured_traffic(f"verify_topk_wide_kernel_B64_k5_V128256_bf16_K{top_k}" if wide
                                                 else "verify_topk_kernel_B64_k5_V128256_bf16"),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
                     "algorithmic_bytes_per_launch": alg},
        "cpu_baseline": {"value": cpu_value, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} oracle calls x 8 rows, one thread", "gpu_outputs_vs_oracle": parity},
        "e2e": {"value": B * e2e_steps * ws / e2e_s, "unit": "rows/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for kk, t in pin.items() if kk != "q")
                + q_in_place, "q_bytes_read_in_place": q_in_place,
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out.values()),
                "steps": e2e_steps,
                "path": "pinned copies (logits, x, u, T, top_k, top_p) + specv_verify_sample_filtered with q read "
                        "in place from page-locked host memory + copies back, per step"},
        "gpu_launches": 2 * steps, "mean_num_accepted": float(np.mean(got["num_accepted"])), "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


RB_B, RB_K, RB_BS, RB_MB = 4096, 8, 16, 64


def run_rollback(args, sv, dev, rank, ws, local, hbm_peak, peak_src):
    """Paged-KV rollback after a verify step: B=4096 rows, k=8 drafts,
    16-position blocks, up to 64 blocks a row."""
    import numpy as np
    import torch

    from speculative_decoding_verification_57_gb300 import workloads as W

    B, k, bs, mb = RB_B, RB_K, RB_BS, RB_MB
    na, lens, tables, nb = W.make_rollback_batch(57200 + 1000 * rank, B, k, bs, mb)
    cap = B * mb
    h = sv.specv_create(local, max_batch=B, max_k=k, vocab=1024)
    base = {kk: torch.from_numpy(v).to(dev) for kk, v in dict(na=na, lens=lens, tables=tables, nb=nb).items()}
    work = {kk: v.clone() for kk, v in base.items()}
    free = torch.full((cap,), -1, dtype=torch.int32, device=dev)
    fc = torch.zeros(1, dtype=torch.int32, device=dev)
    st = torch.empty(B, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def reset():
        for kk in work:
            work[kk].copy_(base[kk], non_blocking=True)
        fc.zero_()

    def call():
        sv.specv_rollback(h, work["na"], k, work["lens"], work["tables"], work["nb"], bs, free, fc, row_status=st,
                          stream=stream)

    with torch.cuda.stream(stream):
        reset()
        call()
    stream.synchronize()
    got = dict(seq_lens=work["lens"].cpu().numpy(), block_tables=work["tables"].cpu().numpy(),
               num_blocks=work["nb"].cpu().numpy(), row_status=st.cpu().numpy(), free_list=free.cpu().numpy(),
               free_count=np.array([int(fc.item())]))
    popped = int(got["free_count"][0])
    # per row: read num_accepted, seq_len, num_blocks; write seq_len, num_blocks, status;
    # per popped block: read its table entry, write -1 there and the block into the free list
    alg = B * 24 + popped * 12 + 8
    # the call changes its inputs: every replay restores them first; the restore alone is
    # timed too and subtracted
    G = max(1, min(args.graph_calls, 50))

    def graph(with_call):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            reset()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(G):
                    reset()
                    if with_call:
                        call()
        return g

    g_both, g_reset = graph(True), graph(False)
    reps = max(1, args.steps // G)
    steps = reps * G

    def timed(g):
        with torch.cuda.stream(stream):
            for _ in range(max(3, args.warmup // G)):
                g.replay()
        stream.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(reps):
                g.replay()
            ev1.record(stream)
        ev1.synchronize()
        return ev0.elapsed_time(ev1)

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark("t0")
    ms_both = timed(g_both)
    sampler.mark("t1")
    ms_reset = timed(g_reset)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if rank == 0 else None
    ms = reduce_max(max(ms_both - ms_reset, 1e-6), ws, dev)
    per_call_s = ms / 1e3 / steps
    # end to end: pinned host state in, rollback, the changed state and the free list back
    pin = {kk: torch.from_numpy(v).pin_memory() for kk, v in dict(na=na, lens=lens, tables=tables, nb=nb).items()}
    host_out = {kk: torch.empty_like(work[kk], device="cpu").pin_memory() for kk in ("lens", "tables", "nb")}
    host_free = torch.empty_like(free, device="cpu").pin_memory()
    host_fc = torch.empty(1, dtype=torch.int32).pin_memory()
    e2e_steps = max(1, args.e2e_steps)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            for kk in pin:
                work[kk].copy_(pin[kk], non_blocking=True)
            fc.zero_()
            call()
            for kk in host_out:
                host_out[kk].copy_(work[kk], non_blocking=True)
            host_fc.copy_(fc, non_blocking=True)
            host_free[:popped].copy_(free[:popped], non_blocking=True)
        stream.synchronize()
    e2e_s = reduce_max(time.perf_counter() - t0, ws, dev)
    if rank != 0:
        return 0
    import oracle  # the CPU-baseline leg

    ref = oracle.rollback(na, k, lens, tables, nb, bs, np.full(cap, -1, np.int32), 0)
    n, t1 = 0, time.perf_counter()
    while time.perf_counter() - t1 < 1.5 or n < 2:
        ref = oracle.rollback(na, k, lens, tables, nb, bs, np.full(cap, -1, np.int32), 0)
        n += 1
    cpu_value = B * n / (time.perf_counter() - t1)
    same = all(np.array_equal(got[kk], ref[kk]) for kk in ("seq_lens", "block_tables", "num_blocks", "row_status",
                                                            "free_list")) and popped == ref["free_count"]
    parity = {"rows": B, "identical": bool(same)}
    achieved = alg / per_call_s / 1e9
    line = {
        "metric": "rollback rows/s", "value": B * steps * ws / (ms / 1e3), "unit": "rows/s", "n_gpus": ws,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"paged-KV rollback B={B} k={k} block_size={bs} max_blocks={mb} (lengths uniform "
                               "in [k, 1024], num_accepted uniform in 0..k)", "B": B, "k": k,
                   "global_batch": B * ws, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "inputs (1.1 MB) stay in L2; every call first restores them from a device copy, "
                         "that restore timed alone and subtracted",
                   "launch": f"CUDA graph of {G} calls, one CTA of 1024 threads"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": achieved / hbm_peak, "traffic": measured_traffic("rollback_kernel_B4096_k8"),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst)",
                     "algorithmic_bytes_per_launch": alg,
                     "note": "latency-bound: one CTA, one block-wide scan over the batch"},
        "cpu_baseline": {"value": cpu_value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} oracle calls x {B} rows, one thread", "gpu_outputs_vs_oracle": parity},
        "e2e": {"value": B * e2e_steps * ws / e2e_s, "unit": "rows/s",
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in pin.values()),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in host_out.values()) + 4 + popped * 4,
                "steps": e2e_steps, "path": "pinned copies + specv_rollback + copies back, per step"},
        "gpu_launches": steps, "blocks_freed_per_call": popped, "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    return 0


def specv_cluster_desc(sv, h, B, k, V):
    c = sv.specv_plan_cluster(h, 1, B, k, V)
    return f"{B * c} CTAs in clusters of {c}"


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
