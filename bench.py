"""Benchmark of the compressed-KV sparse-attention decode step on GB300.

One step = one ds4x_csa_decode_step call: CSA indexer score + exact top-512
over all N compressed rows of one layer, then sparse attention of the
64-head decode query over the 512 selected packed KV rows (batch 1).  Default workload: the long decode layer,
N = 1,048,576 rows (68-byte MXFP4 indexer rows, 583-byte KV rows, 64 indexer
heads x 128, 64 attention heads x 512), synthetic N(0,1) data packed by the
library's own cache writer.

Timing: W untimed warm-up steps, then exactly K steps replayed from CUDA
graphs, bracketed by a barrier and a device synchronise, timed with CUDA
events on the launching stream.  The steps rotate over L layer caches, and
the L layer steps of a token are one CUDA graph (K mod L steps are replayed
from one-step graphs); the time with one graph per step is reported beside
it.  Inputs larger than L2: L x 71.3 MB of indexer rows > 4 x the 129 MB
L2, so every step streams its rows from HBM.

Printed: one JSON line (rank 0).  `value` is compressed rows scored per second
over the whole job; `roofline` is the dominant kernel (the scorer entry
point) timed on its own over K graph replays; `e2e` times the same step
through the public API from pinned host buffers (append of the new row,
score, attention, result copied back); `cpu_baseline` is the float64 oracle
on the host cores (all cores over the whole workload; one core on a
262,144-row sample).  `--impl reference` times the oracle alone over the
whole workload on all host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn step latency (µs/layer) & compressed rows/s vs N; achieved HBM GB/s"
WORKLOADS = {"tiny": 4096, "mid": 131072, "long": 1048576}
EXTRA_WORKLOADS = ("sessions", "prefill", "hca", "window")  # parity configurations, measured on request
K_TOP = 512
HEADS = 64
FALLBACK_HBM_GBS = 6800.0


def step_bytes(n):
    """Algorithmic HBM bytes of one decode step (what the method must move)."""
    return scorer_bytes(n) + attn_bytes()


def scorer_bytes(n):
    # indexer rows + bf16 query + f32 weights + top-k indices and scores written
    return 68 * n + HEADS * 128 * 2 + HEADS * 4 + K_TOP * (4 + 4)


def attn_bytes():
    # gathered KV rows + index list + bf16 query + bf16 output + lse
    return K_TOP * 583 + K_TOP * 4 + HEADS * 512 * 2 + HEADS * 512 * 2 + HEADS * 4


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# Source files each timed kernel is built from: an ncu traffic figure is
# reported only while these are unchanged since the capture.
KERNEL_SOURCES = {
    "ds4x_index_score_topk": ("score_fused.cu", "select512.cuh", "tc_ptx.cuh", "ds4x_internal.cuh"),
    "ds4x_sparse_attn_decode": ("attn_decode.cu", "ds4x_internal.cuh"),
}


def kernel_sources_hash(kernel_name):
    csrc = os.path.join(ROOT, "compressed_kv_sparse_csa_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel_name]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    with open(os.path.join(ROOT, "include", "ds4x.h"), "rb") as fh:  # its constants, not its prose
        h.update(b"".join(ln for ln in fh.read().splitlines(True) if ln.startswith(b"#define")))
    return h.hexdigest()[:16]


def recorded_traffic(kernel_name):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
    except Exception:
        return None, None
    ent = rec.get(kernel_name)
    if not ent or ent.get("sources_hash") != kernel_sources_hash(kernel_name):
        return None, None
    return ent.get("dram_bytes_per_launch_full_size"), ent.get("note")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"ds4x_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            self.proc.wait(timeout=5)
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = sorted(float(r[1]) for r in rows if r[1].replace(".", "").isdigit())
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# CPU baseline / reference arm: the float64 oracle as it stands
# ---------------------------------------------------------------------------

def oracle_step_sample(n_rows, seed=1002):
    """Time one oracle decode step (score + top-512 + attention) over the
    first n_rows of the long-decode workload's distribution.  Returns seconds."""
    import numpy as np

    from oracle import codecs as C
    from oracle import indexer as I
    from oracle.attention import sparse_attn_decode
    from synth import decode_case

    case = decode_case(n_rows, seed)
    idx_rows = C.pack_idx_rows(case["idx_in"])
    t0 = time.perf_counter()
    idx, _, _ = I.score_topk(idx_rows, case["q_idx"], case["w"], K_TOP)
    t1 = time.perf_counter()
    # packing is not part of the step: pack just the selected KV rows, untimed
    kv_sel = C.pack_kv_rows(case["kv_in"][idx])
    t2 = time.perf_counter()
    sparse_attn_decode(kv_sel, np.arange(idx.shape[0]), case["q_attn"], 1.0 / math.sqrt(512.0))
    return (t1 - t0) + (time.perf_counter() - t2)


def run_oracle_subprocess(n_rows, reps):
    """Run the oracle in a single-threaded child process; returns list of seconds."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; import json; "
            f"print(json.dumps([bench.oracle_step_sample({n_rows}, seed=1002 + i) for i in range({reps})]))")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=1800)
    if out.returncode != 0:
        raise RuntimeError(out.stderr[-2000:])
    return json.loads(out.stdout.strip().splitlines()[-1])


def cpu_model():
    """The host CPU's model name (lscpu), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform

    return platform.machine()


def _oracle_score_chunk(task):
    """Pool worker: the oracle's scores of rows [a, b) of the shared packed rows."""
    from multiprocessing import shared_memory

    import numpy as np

    from oracle import indexer as I

    name, n, a, b, q_bits, w = task
    shm = shared_memory.SharedMemory(name=name)
    try:
        rows = np.ndarray((n, 68), dtype=np.uint8, buffer=shm.buf)
        return a, I.score_rows(rows[a:b], q_bits, w)
    finally:
        shm.close()


def oracle_step_all_cores(n_rows=1048576, reps=3, seed=1002, all_steps=False):
    """The oracle's decode step over every row of the long-decode workload on
    all host cores: the unchanged oracle scorer on one chunk of rows per
    process (one BLAS thread each, a spawn pool started before the timing),
    then the oracle's top-512 and attention in this process.  Returns
    (seconds per step, processes)."""
    import multiprocessing as mp
    from multiprocessing import shared_memory

    import numpy as np

    from oracle import codecs as C
    from oracle import indexer as I
    from oracle.attention import sparse_attn_decode
    from synth import decode_case

    procs = os.cpu_count() or 1
    case = decode_case(n_rows, seed)
    rows = C.pack_idx_rows(case["idx_in"])  # the cache contents (not timed)
    shm = shared_memory.SharedMemory(create=True, size=rows.nbytes)
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
    try:
        np.ndarray(rows.shape, dtype=np.uint8, buffer=shm.buf)[:] = rows
        for k in saved:
            os.environ[k] = "1"  # inherited by the spawned workers
        bounds = np.linspace(0, n_rows, 4 * procs + 1).astype(np.int64)
        tasks = [(shm.name, n_rows, int(a), int(b), case["q_idx"], case["w"]) for a, b in zip(bounds[:-1], bounds[1:])]
        secs = []
        with mp.get_context("spawn").Pool(procs) as pool:
            pool.map(_oracle_score_chunk, tasks[:procs])  # start-up and imports, not timed
            for _ in range(reps):
                t0 = time.perf_counter()
                parts = pool.map(_oracle_score_chunk, tasks)
                s = np.concatenate([p for _, p in sorted(parts, key=lambda x: x[0])])
                idx, _ = I.topk(s, K_TOP)
                t1 = time.perf_counter()
                kv_sel = C.pack_kv_rows(case["kv_in"][idx])  # packing is not part of the step
                t2 = time.perf_counter()
                sparse_attn_decode(kv_sel, np.arange(idx.shape[0]), case["q_attn"], 1.0 / math.sqrt(512.0))
                secs.append((t1 - t0) + (time.perf_counter() - t2))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        shm.close()
        shm.unlink()
    if all_steps:
        return secs, procs
    return sorted(secs)[len(secs) // 2], procs


def cpu_baseline(n_rows=262144, reps=5):
    secs = run_oracle_subprocess(n_rows, reps)
    t1 = sorted(secs)[len(secs) // 2]
    n_all = WORKLOADS["long"]
    t_all, procs = oracle_step_all_cores(n_all)
    return {"value": n_all / t_all, "unit": "rows/s", "cores": procs, "kind": "oracle",
            "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "sample": f"median of 3 oracle steps (score + top-512 + attention) over all {n_all} rows of the "
                      f"long-decode workload, numpy float64, the unchanged oracle scorer on {procs} processes "
                      f"(one per core, one BLAS thread each), top-512 and attention in one; {t_all:.2f} s each",
            "single_thread": {"value": n_rows / t1, "unit": "rows/s", "cores": 1,
                              "sample": f"median of {reps} oracle steps over {n_rows} rows of the same "
                                        f"distribution, 1 thread; {t1:.2f} s each"}}


def replay_plan(k, group):
    """Graph replays that run exactly k steps when a group graph runs `group`
    steps: (group replays, one-step replays), k // group and k % group."""
    return k // group, k % group


def max_over_ranks(values, dist, device):
    """Each timed quantity's maximum over the ranks (the job is as slow as
    its slowest replica); unchanged on one process."""
    if dist is None:
        return list(values)
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_value(world, n_rows, ms_per_step):
    """Whole-job throughput: every replica scores n_rows per step."""
    return world * n_rows / (ms_per_step * 1e-3)


def reference_arm(args, workload, n):
    """The oracle (the only other implementation of the path) on the host's
    cores: every step is the oracle's score + top-512 + attention over all n
    rows of the workload, the scorer on one process per core."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    secs, procs = oracle_step_all_cores(n, reps=args.warmup + args.steps, seed=1000 + list(WORKLOADS).index(workload),
                                        all_steps=True)
    timed = secs[args.warmup:]
    t = sum(timed)
    value = n * len(timed) / t
    sample = (f"all {n} rows of the {workload} decode workload per step, numpy float64 oracle, the scorer "
              f"on {procs} processes (one per core), top-512 and attention in one; host CPU {cpu_model()}")
    line = {"metric": METRIC, "value": value, "unit": "compressed rows/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload, "n_rows": n, "top_k": K_TOP},
            "cpu_baseline": {"value": value, "unit": "compressed rows/s", "cores": procs, "kind": "oracle",
                             "nproc": os.cpu_count(), "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": "compressed rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long", choices=sorted(WORKLOADS) + list(EXTRA_WORKLOADS))
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload in EXTRA_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the decode workloads only"}))
            return
        {"sessions": run_sessions, "prefill": run_prefill, "hca": run_hca, "window": run_window}[args.workload](args)
        return
    n = WORKLOADS[args.workload]
    if args.impl == "reference":
        reference_arm(args, args.workload, n)
        return

    import torch

    from compressed_kv_sparse_csa_gb300 import binding as B

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    L = args.layers
    scale = 1.0 / math.sqrt(512.0)

    # ---- resident inputs: L layer caches packed by the library's cache writer
    gen = torch.Generator(device=dev)
    layers = []
    with torch.cuda.stream(stream):
        for l in range(L):
            gen.manual_seed(1002 * 1000 + 97 * rank + l)
            idx_rows = torch.empty(n * 68, dtype=torch.uint8, device=dev)
            kv_rows = torch.empty(n * 583, dtype=torch.uint8, device=dev)
            chunk = 1 << 18
            for a in range(0, n, chunk):
                b = min(n, a + chunk)
                idx_in = torch.randn((b - a, 128), generator=gen, device=dev)
                kv_in = torch.randn((b - a, 512), generator=gen, device=dev)
                B.ds4x_cache_append(kv_rows, idx_rows, a, kv_in, idx_in, stream=stream)
            q_idx = torch.randn((HEADS, 128), generator=gen, device=dev).to(torch.bfloat16)
            w = torch.rand(HEADS, generator=gen, device=dev) / 8
            q_attn = torch.randn((HEADS, 512), generator=gen, device=dev).to(torch.bfloat16)
            layers.append({"idx_rows": idx_rows, "kv_rows": kv_rows, "q_idx": q_idx, "w": w, "q_attn": q_attn,
                           "out_idx": torch.empty(K_TOP, dtype=torch.int32, device=dev),
                           "out_score": torch.empty(K_TOP, dtype=torch.float32, device=dev),
                           "out": torch.empty((HEADS, 512), dtype=torch.bfloat16, device=dev)})
        ws_s = torch.empty(B.ds4x_index_score_topk_workspace(n, K_TOP), dtype=torch.uint8, device=dev)
        ws_d = torch.empty(B.ds4x_csa_decode_step_workspace(n, K_TOP), dtype=torch.uint8, device=dev)
        B.ds4x_workspace_init(ws_s, stream=stream)
        B.ds4x_workspace_init(ws_d, stream=stream)
    stream.synchronize()

    def step(l, score_only=False):
        c = layers[l]
        if score_only:
            B.ds4x_index_score_topk(c["idx_rows"], n, c["q_idx"], c["w"], K_TOP, c["out_idx"], c["out_score"], ws_s,
                                    stream=stream)
        else:  # the decode step: score + top-512, then attention over the selected rows
            B.ds4x_csa_decode_step(c["idx_rows"], c["kv_rows"], n, c["q_idx"], c["w"], K_TOP, c["q_attn"], scale,
                                   c["out_idx"], c["out_score"], c["out"], None, ws_d, stream=stream)

    # kernels each entry point launches: the fused scorer is one kernel, the
    # two-stage scorer two; attention is one cluster kernel
    two_stage = os.environ.get("DS4X_SCORER") == "two_stage"
    launches_per_step = {"score": 2 if two_stage else 1, "attn": 1}

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i % L)
    stream.synchronize()

    # The L layer steps of a decode token run back to back, as one CUDA graph
    # (a server captures a token's layers together); one graph per layer step
    # is kept for the remainder of K / L and for the per-step-graph figure.
    def capture(score_only):
        singles = []
        for l in range(L):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(l, score_only)
            singles.append(g)
        whole = torch.cuda.CUDAGraph()
        with torch.cuda.graph(whole, stream=stream):
            for l in range(L):
                step(l, score_only)
        return singles, whole

    step_graphs = capture(False)
    score_graphs = capture(True)

    def barrier():
        if dist is not None:
            dist.barrier()

    def timed(graphs, k, per_step_graphs=False):
        """Exactly k steps: k // L replays of the L-step graph and the first
        k % L single-step graphs (or k single-step graphs)."""
        singles, whole = graphs
        with torch.cuda.stream(stream):
            for g in singles:  # untimed replay of each graph once
                g.replay()
            whole.replay()
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            e0.record(stream)
            if per_step_graphs:
                for i in range(k):
                    singles[i % L].replay()
            else:
                n_whole, n_single = replay_plan(k, L)
                for _ in range(n_whole):
                    whole.replay()
                for i in range(n_single):
                    singles[i].replay()
            e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return e0.elapsed_time(e1)  # ms

    with ClockSampler(local) as clk:
        ms_total = timed(step_graphs, args.steps)
    clocks = clk.summary()
    ms_score = timed(score_graphs, args.steps)
    ms_total_1 = timed(step_graphs, args.steps, per_step_graphs=True)  # for comparison only

    # ---- end to end through the public API, host buffers, copies inside.
    # A step's inputs (the new row's 512 + 128 values, both queries, the head
    # weights) sit in one pinned block and cross in one copy; the attention
    # output and the indices come back in one copy (both ds4x_copy_async: a
    # kernel reading / writing the pinned host block).  The public calls of a
    # step (copy in, append, score + attend, copy out) are captured once per
    # layer as a CUDA graph, as a decode server would run them.
    e2e_steps = min(args.steps, 500)
    seg = [("kv", 512 * 4), ("idx", 128 * 4), ("q", HEADS * 128 * 2), ("w", HEADS * 4), ("qa", HEADS * 512 * 2)]
    offs, o = {}, 0
    for name, nb in seg:
        offs[name] = (o, nb)
        o += nb
    h_in = torch.empty(o, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(o, dtype=torch.uint8, device=dev)

    def part(buf, name, dtype, shape):
        a0, nb = offs[name]
        return buf[a0:a0 + nb].view(dtype).view(*shape)

    part(h_in, "kv", torch.float32, (1, 512)).copy_(torch.randn((1, 512)))
    part(h_in, "idx", torch.float32, (1, 128)).copy_(torch.randn((1, 128)))
    part(h_in, "q", torch.bfloat16, (HEADS, 128)).copy_(layers[0]["q_idx"].cpu())
    part(h_in, "w", torch.float32, (HEADS,)).copy_(layers[0]["w"].cpu())
    part(h_in, "qa", torch.bfloat16, (HEADS, 512)).copy_(layers[0]["q_attn"].cpu())
    d_kv, d_idx = part(d_in, "kv", torch.float32, (1, 512)), part(d_in, "idx", torch.float32, (1, 128))
    d_q, d_w = part(d_in, "q", torch.bfloat16, (HEADS, 128)), part(d_in, "w", torch.float32, (HEADS,))
    d_qa = part(d_in, "qa", torch.bfloat16, (HEADS, 512))
    out_bytes = HEADS * 512 * 2 + K_TOP * 4
    d_res = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    h_res = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    d_out = d_res[:HEADS * 512 * 2].view(torch.bfloat16).view(HEADS, 512)
    d_oidx = d_res[HEADS * 512 * 2:].view(torch.int32)
    h2d = o
    d2h = out_bytes

    def e2e_calls(l):
        c = layers[l]
        B.ds4x_copy_async(d_in, h_in, stream=stream)  # pinned host -> device, a kernel (no copy-engine hand-over)
        B.ds4x_cache_append(c["kv_rows"], c["idx_rows"], n - 1, d_kv, d_idx, stream=stream)
        B.ds4x_csa_decode_step(c["idx_rows"], c["kv_rows"], n, d_q, d_w, K_TOP, d_qa, scale, d_oidx, c["out_score"],
                               d_out, None, ws_d, stream=stream)
        B.ds4x_copy_async(h_res, d_res, stream=stream)  # device -> pinned host

    with torch.cuda.stream(stream):
        for l in range(L):
            e2e_calls(l)
    stream.synchronize()
    e2e_graphs = []
    for l in range(L):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e2e_calls(l)
        e2e_graphs.append(g)
    e2e_whole = torch.cuda.CUDAGraph()  # a token's L layer steps, each with its copies
    with torch.cuda.graph(e2e_whole, stream=stream):
        for l in range(L):
            e2e_calls(l)

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_graphs[i % L].replay()
        e2e_whole.replay()
        stream.synchronize()
        barrier()
        t0 = time.perf_counter()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        n_whole, n_single = replay_plan(e2e_steps, L)
        for _ in range(n_whole):
            e2e_whole.replay()
        for i in range(n_single):
            e2e_graphs[i].replay()
        e1.record(stream)
        stream.synchronize()
        barrier()
        ms_e2e = max(e0.elapsed_time(e1), 1e3 * (time.perf_counter() - t0))

    ms_step = ms_total / args.steps
    ms_sc = ms_score / args.steps
    ms_e2e_step = ms_e2e / e2e_steps
    ms_step_1 = ms_total_1 / args.steps
    ms_step, ms_sc, ms_e2e_step, ms_step_1 = max_over_ranks([ms_step, ms_sc, ms_e2e_step, ms_step_1], dist, dev)
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    sb = scorer_bytes(n)
    achieved = sb / (ms_sc * 1e-3) / 1e9
    traffic, tnote = recorded_traffic("ds4x_index_score_topk")
    line = {
        "metric": METRIC,
        "value": job_value(world, n, ms_step),
        "unit": "compressed rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16-in/fp32-acc (MXFP4 + E4M3/FP16 packed rows)",
        "data": "synthetic",
        "config": {"workload": f"{args.workload} decode, batch 1, one layer",
                   "n_rows": n, "top_k": K_TOP, "indexer_heads": HEADS, "attn_heads": HEADS,
                   "layer_caches_rotated": L,
                   "l2": f"inputs larger than L2: {L} layer caches x {68 * n / 1e6:.1f} MB indexer rows rotated",
                   "us_per_layer": ms_step * 1e3,
                   "graphs": f"the {L} layer steps of a token as one CUDA graph (K mod {L} steps as one-step graphs)",
                   "us_per_layer_one_graph_per_step": ms_step_1 * 1e3,
                   "achieved_step_gbs": step_bytes(n) / (ms_step * 1e-3) / 1e9,
                   "step_bytes": step_bytes(n),
                   "step_roofline_frac": (step_bytes(n) / (ms_step * 1e-3) / 1e9) / peak,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "scorer_path": "two_stage" if two_stage else "fused_tcgen05",
        "roofline": {"kernel": "ds4x_index_score_topk", "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                     "unit": "GB/s", "frac": achieved / peak, "traffic": traffic,
                     "traffic_note": tnote, "algorithmic_bytes_per_launch": sb, "us_per_launch": ms_sc * 1e3},
        "e2e": {"value": job_value(world, n, ms_e2e_step), "unit": "compressed rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "ms_per_step": ms_e2e_step,
                "path": f"the public calls of {L} layer steps as one CUDA graph, each step: ds4x_copy_async of "
                        "its packed inputs from pinned host memory (a kernel), ds4x_cache_append, "
                        "ds4x_csa_decode_step (score + top-512, attention), ds4x_copy_async of its output and "
                        "indices to pinned host memory"},
        "gpu_launches": args.steps * (launches_per_step["score"] + launches_per_step["attn"]),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_baseline()
        except Exception as e:  # report, never fake
            line["cpu_baseline"] = {"value": None, "error": str(e)[-300:]}
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()



# ---------------------------------------------------------------------------
# Extra workloads: micro-batched decode and chunked prefill
# ---------------------------------------------------------------------------

def _gpu_setup():
    import torch

    from compressed_kv_sparse_csa_gb300 import binding as B

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    return torch, B, dev, torch.cuda.Stream(device=dev)


def _timed_graph(torch, stream, graphs, steps, warmup=3):
    with torch.cuda.stream(stream):  # untimed warm-up replays
        for i in range(max(warmup, len(graphs))):
            graphs[i % len(graphs)].replay()
    stream.synchronize()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            graphs[i % len(graphs)].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps  # ms per step


GROUP = 8  # decode steps per CUDA graph (a token's layers back to back)


def _step_graphs(torch, stream, calls):
    """One-step graphs of each call (a closure launching one step) and graphs
    of GROUP consecutive steps (calls taken cyclically)."""
    singles = []
    for f in calls:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            f()
        singles.append(g)
    groups = []
    for j0 in range(0, len(calls), GROUP):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(j0, j0 + GROUP):
                calls[j % len(calls)]()
        groups.append(g)
    return singles, groups


def _timed_steps(torch, stream, graphs, steps, warmup=3, per_step_graphs=False):
    """ms per step over exactly `steps` steps: steps // GROUP group replays
    and steps % GROUP one-step replays (or one-step graphs throughout)."""
    singles, groups = graphs
    with torch.cuda.stream(stream):  # untimed warm-up replays
        for i in range(max(warmup, len(singles))):
            singles[i % len(singles)].replay()
        for g in groups:
            g.replay()
    stream.synchronize()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        if per_step_graphs:
            for i in range(steps):
                singles[i % len(singles)].replay()
        else:
            n_group, n_single = replay_plan(steps, GROUP)
            for i in range(n_group):
                groups[i % len(groups)].replay()
            for i in range(n_single):
                singles[i % len(singles)].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_sessions(args):
    """16 independent decode sessions (lengths uniform on [8192, 65536],
    seeded), one batched scorer launch and one batched attention launch per
    step; L layer copies rotated so the indexer rows exceed L2."""
    import numpy as np

    torch, B, dev, stream = _gpu_setup()
    rng = np.random.default_rng(1003)
    n_sess = 16
    lens = rng.integers(8192, 65536 + 1, size=n_sess)
    L = max(2, min(args.layers, 6))
    gen = torch.Generator(device=dev)
    layers = []
    with torch.cuda.stream(stream):
        for l in range(L):
            gen.manual_seed(3000 + l)
            idx_t, kv_t = [], []
            for nr in lens:
                nr = int(nr)
                it = torch.empty(nr * 68, dtype=torch.uint8, device=dev)
                kt = torch.empty(nr * 583, dtype=torch.uint8, device=dev)
                B.ds4x_cache_append(kt, it, 0, torch.randn((nr, 512), generator=gen, device=dev),
                                    torch.randn((nr, 128), generator=gen, device=dev), stream=stream)
                idx_t.append(it)
                kv_t.append(kt)
            layers.append({
                "idx": idx_t, "kv": kv_t,
                "idx_p": torch.tensor([t.data_ptr() for t in idx_t], dtype=torch.int64, device=dev),
                "kv_p": torch.tensor([t.data_ptr() for t in kv_t], dtype=torch.int64, device=dev),
                "n": torch.tensor([int(x) for x in lens], dtype=torch.int64, device=dev),
                "q": torch.randn((n_sess, 64, 128), generator=gen, device=dev).to(torch.bfloat16),
                "w": torch.rand((n_sess, 64), generator=gen, device=dev) / 8,
                "qa": torch.randn((n_sess, 64, 512), generator=gen, device=dev).to(torch.bfloat16),
                "oi": torch.empty((n_sess, K_TOP), dtype=torch.int32, device=dev),
                "out": torch.empty((n_sess, 64, 512), dtype=torch.bfloat16, device=dev)})
        ws_s = torch.empty(B.ds4x_index_score_topk_batched_workspace(n_sess, K_TOP), dtype=torch.uint8, device=dev)
        ws_a = torch.empty(B.ds4x_sparse_attn_decode_workspace(K_TOP), dtype=torch.uint8, device=dev)
        B.ds4x_workspace_init(ws_s, stream=stream)
        B.ds4x_workspace_init(ws_a, stream=stream)
    stream.synchronize()
    scale = 1.0 / math.sqrt(512.0)

    def step(c, score_only=False):
        B.ds4x_index_score_topk_batched(c["idx_p"], c["n"], c["q"], c["w"], K_TOP, c["oi"], None, ws_s, stream=stream)
        if not score_only:
            B.ds4x_sparse_attn_decode_batched(c["kv_p"], c["n"], c["oi"], K_TOP, c["qa"], scale, c["out"], None, ws_a,
                                              stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(layers[i % L])
    stream.synchronize()
    graphs = _step_graphs(torch, stream, [lambda c=c: step(c) for c in layers])
    sgraphs = _step_graphs(torch, stream, [lambda c=c: step(c, True) for c in layers])
    steps = min(args.steps, 1000)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ms = _timed_steps(torch, stream, graphs, steps, args.warmup)
    ms_sc = _timed_steps(torch, stream, sgraphs, steps, args.warmup)
    ms_1 = _timed_steps(torch, stream, graphs, steps, args.warmup, per_step_graphs=True)
    total = int(lens.sum())
    step_b = sum(step_bytes(int(x)) for x in lens)
    peak, kind = measured_peak()
    sb = sum(scorer_bytes(int(x)) for x in lens)
    print(json.dumps({
        "metric": "micro-batched decode step latency (us) & compressed rows/s",
        "value": total / (ms * 1e-3), "unit": "compressed rows/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-in/fp32-acc (MXFP4 + E4M3/FP16 packed rows)", "data": "synthetic",
        "config": {"workload": "16 decode sessions, lengths uniform on [8192, 65536] (seed 1003), batch 1 each",
                   "rows_total": total, "lengths": [int(x) for x in lens], "top_k": K_TOP, "layer_copies": L,
                   "us_per_step": ms * 1e3, "step_bytes": step_b,
                   "graphs": f"{GROUP} steps per CUDA graph (K mod {GROUP} as one-step graphs)", "us_per_step_one_graph_per_step": ms_1 * 1e3,
                   "step_roofline_frac": step_b / (ms * 1e-3) / 1e9 / peak},
        "roofline": {"kernel": "ds4x_index_score_topk_batched", "bound": "hbm",
                     "achieved": sb / (ms_sc * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": sb / (ms_sc * 1e-3) / 1e9 / peak, "traffic": None, "us_per_launch": ms_sc * 1e3,
                     "peak_kind": kind},
        "gpu_launches": steps * 2, "clocks": clk.summary()}), flush=True)


def run_hca(args):
    """Dense decode attention over every compressed row of a ratio-128 (HCA)
    layer at a 1M-token context: 8192 rows of 583 B, 64 heads; 40 layer
    copies (191 MB, above the 129 MB L2) rotated, one CUDA graph per layer
    (the tensor-core attention over 64 items of 128 rows, then the combine)."""
    torch, B, dev, stream = _gpu_setup()
    n, L = 8192, 40
    gen = torch.Generator(device=dev)
    gen.manual_seed(6006)
    layers = []
    with torch.cuda.stream(stream):
        for _ in range(L):
            kv = torch.empty(n * 583, dtype=torch.uint8, device=dev)
            B.ds4x_cache_append(kv, None, 0, torch.randn((n, 512), generator=gen, device=dev), None, stream=stream)
            layers.append({"kv": kv, "q": torch.randn((64, 512), generator=gen, device=dev).to(torch.bfloat16),
                           "out": torch.empty((64, 512), dtype=torch.bfloat16, device=dev)})
        ws = torch.empty(B.ds4x_dense_attn_decode_workspace(n), dtype=torch.uint8, device=dev)
        B.ds4x_workspace_init(ws, stream=stream)
    stream.synchronize()
    scale = 1.0 / math.sqrt(512.0)

    def step(c):
        B.ds4x_dense_attn_decode(c["kv"], n, c["q"], scale, c["out"], None, ws, stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(layers[i % L])
    stream.synchronize()
    graphs = _step_graphs(torch, stream, [lambda c=c: step(c) for c in layers])
    steps = min(args.steps, 2000)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ms = _timed_steps(torch, stream, graphs, steps, args.warmup)
    ms_1 = _timed_steps(torch, stream, graphs, steps, args.warmup, per_step_graphs=True)
    peak, kind = measured_peak()
    algo = n * 583 + 2 * 64 * 512 * 2  # the rows, the query, the output
    print(json.dumps({
        "metric": "HCA dense decode attention latency (us) & compressed rows/s",
        "value": n / (ms * 1e-3), "unit": "compressed rows/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-in/fp32-acc (E4M3/FP16 packed rows)", "data": "synthetic",
        "config": {"workload": "dense attention over 8192 ratio-128 rows (1M-token context), 64 heads",
                   "n_rows": n, "layer_copies": L, "l2": "inputs larger than L2: 40 x 4.8 MB rotated",
                   "us_per_step": ms * 1e3,
                   "graphs": f"{GROUP} steps per CUDA graph (K mod {GROUP} as one-step graphs)", "us_per_step_one_graph_per_step": ms_1 * 1e3},
        "roofline": {"kernel": "ds4x_dense_attn_decode", "bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": algo / (ms * 1e-3) / 1e9 / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": algo, "peak_kind": kind},
        "gpu_launches": steps * 2, "clocks": clk.summary()}), flush=True)


def run_window(args):
    """Decode attention over the 512 selected rows of a 1,048,576-row cache and
    all 256 live rows of the layer's raw sliding window, one softmax over
    both: 8 index lists and 8 rings rotated (the selected rows are random
    rows of the 611 MB cache, so they come from HBM), one CUDA graph each."""
    torch, B, dev, stream = _gpu_setup()
    n, L, w = 1048576, 8, 256
    gen = torch.Generator(device=dev)
    gen.manual_seed(7007)
    with torch.cuda.stream(stream):
        kv = torch.empty(n * 583, dtype=torch.uint8, device=dev)
        chunk = 1 << 18
        for a in range(0, n, chunk):
            B.ds4x_cache_append(kv, None, a, torch.randn((chunk, 512), generator=gen, device=dev), None, stream=stream)
        items = []
        for _ in range(L):
            ring = torch.empty(256 * 583, dtype=torch.uint8, device=dev)
            B.ds4x_cache_append(ring, None, 0, torch.randn((256, 512), generator=gen, device=dev), None, stream=stream)
            idx = torch.randperm(n, generator=gen, device=dev)[:K_TOP].to(torch.int32)
            items.append({"ring": ring, "idx": idx, "q": torch.randn((64, 512), generator=gen, device=dev).to(torch.bfloat16),
                          "out": torch.empty((64, 512), dtype=torch.bfloat16, device=dev)})
        ws = torch.empty(B.ds4x_window_sparse_attn_decode_workspace(), dtype=torch.uint8, device=dev)
        B.ds4x_workspace_init(ws, stream=stream)
    stream.synchronize()
    scale = 1.0 / math.sqrt(512.0)

    def step(c):
        B.ds4x_window_sparse_attn_decode(kv, n, c["idx"], K_TOP, c["ring"], 200, w, c["q"], scale, c["out"], None, ws,
                                         stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(items[i % L])
    stream.synchronize()
    graphs = _step_graphs(torch, stream, [lambda c=c: step(c) for c in items])
    steps = min(args.steps, 2000)
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        ms = _timed_steps(torch, stream, graphs, steps, args.warmup)
    ms_1 = _timed_steps(torch, stream, graphs, steps, args.warmup, per_step_graphs=True)
    peak, kind = measured_peak()
    # the selected and the window rows, the index list, the query, the output
    algo = (K_TOP + w) * 583 + K_TOP * 4 + 2 * 64 * 512 * 2
    print(json.dumps({
        "metric": "sparse + sliding-window decode attention latency (us)",
        "value": ms * 1e3, "unit": "us/call", "n_gpus": 1, "steps": steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16-in/fp32-acc (E4M3/FP16 packed rows)", "data": "synthetic",
        "config": {"workload": "512 selected rows of a 1,048,576-row cache + 256 live raw-window rows, 64 heads",
                   "n_rows": n, "window": w, "rotated": L,
                   "l2": "selected rows random over a 611 MB cache (above L2); 8 rings and index lists rotated",
                   "graphs": f"{GROUP} steps per CUDA graph (K mod {GROUP} as one-step graphs)", "us_per_step_one_graph_per_step": ms_1 * 1e3},
        "roofline": {"kernel": "ds4x_window_sparse_attn_decode", "bound": "hbm", "achieved": algo / (ms * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": algo / (ms * 1e-3) / 1e9 / peak, "traffic": None,
                     "algorithmic_bytes_per_launch": algo, "peak_kind": kind},
        # per call: the index-list set-up kernel, the attention over the two items, the finalize
        "gpu_launches": steps * 3, "clocks": clk.summary()}), flush=True)


def run_prefill(args):
    """One chunk of 2048 prefill query tokens over 65,536 history rows (query
    i sees rows t < 63,488 + i): query quantiser + per-query causal top-512 +
    per-query sparse attention."""
    torch, B, dev, stream = _gpu_setup()
    T, n, base = 2048, 65536, 63488
    per_launch = min(2 * torch.cuda.get_device_properties(dev).multi_processor_count, 512)  # query tokens per launch
    gen = torch.Generator(device=dev)
    gen.manual_seed(4004)
    with torch.cuda.stream(stream):
        idx_rows = torch.empty(n * 68, dtype=torch.uint8, device=dev)
        kv_rows = torch.empty(n * 583, dtype=torch.uint8, device=dev)
        B.ds4x_cache_append(kv_rows, idx_rows, 0, torch.randn((n, 512), generator=gen, device=dev),
                            torch.randn((n, 128), generator=gen, device=dev), stream=stream)
        q = torch.randn((T, 64, 128), generator=gen, device=dev)
        w = torch.rand((T, 64), generator=gen, device=dev) / 8
        qa = torch.randn((T, 64, 512), generator=gen, device=dev).to(torch.bfloat16)
        codes = torch.empty((T, 64, 128), dtype=torch.uint8, device=dev)
        scales = torch.empty((T, 64, 4), dtype=torch.uint8, device=dev)
        oi = torch.empty((T, K_TOP), dtype=torch.int32, device=dev)
        out = torch.empty((T, 64, 512), dtype=torch.bfloat16, device=dev)
        ws_s = torch.empty(B.ds4x_index_score_topk_prefill_workspace(n, T, K_TOP), dtype=torch.uint8, device=dev)
        ws_a = torch.empty(B.ds4x_sparse_attn_decode_workspace(K_TOP), dtype=torch.uint8, device=dev)
        B.ds4x_workspace_init(ws_s, stream=stream)
        B.ds4x_workspace_init(ws_a, stream=stream)
    stream.synchronize()
    scale = 1.0 / math.sqrt(512.0)

    def quant():
        B.ds4x_quantize_query_e4m3(q, codes, scales, stream=stream)

    def score():
        B.ds4x_index_score_topk_prefill(idx_rows, n, codes, scales, w, T, base, K_TOP, oi, None, ws_s, stream=stream)

    def attend():
        B.ds4x_sparse_attn_prefill(kv_rows, n, oi, T, K_TOP, qa, scale, out, None, ws_a, stream=stream)

    parts = {}
    with torch.cuda.stream(stream):
        for f in (quant, score, attend):
            f()
    stream.synchronize()
    steps = max(1, min(args.steps, 5))
    for name, fns in (("step", (quant, score, attend)), ("quant", (quant,)), ("score", (score,)),
                      ("attend", (attend,))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for f in fns:
                f()
        if name == "step":
            with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
                parts[name] = _timed_graph(torch, stream, [g], steps, args.warmup)
        else:
            parts[name] = _timed_graph(torch, stream, [g], steps, args.warmup)
    pairs = sum(min(n, base + i) for i in range(T))
    flop_score = pairs * 64 * 128 * 2.0          # q^ . k for every visible (query, row, head)
    flop_attn = T * 64 * K_TOP * 512 * 2.0 * 2   # logits and weighted sum
    peak_bf16 = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak_bf16 = float(json.load(f)["bf16_tflops"])
    except Exception:
        peak_bf16 = 1900.0
    peak_fp8 = 2.0 * peak_bf16  # FP8 dense nominal rate is twice bf16's
    print(json.dumps({
        "metric": "prefill chunk latency (ms) & query tokens/s",
        "value": T / (parts["step"] * 1e-3), "unit": "query tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": args.warmup, "ms_per_step": parts["step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "E4M3 x E2M1 block-scaled (scorer), bf16-in/fp32-acc (attention)", "data": "synthetic",
        "config": {"workload": "2048 prefill tokens x 64 heads over 65536 rows, causal base 63488",
                   "ms_quantize": parts["quant"], "ms_score_topk": parts["score"], "ms_attention": parts["attend"],
                   "visible_pairs": pairs},
        "roofline": {"kernel": "ds4x_index_score_topk_prefill", "bound": "tensor",
                     "achieved": flop_score / (parts["score"] * 1e-3) / 1e12,
                     "peak": peak_fp8, "unit": "TFLOP/s", "frac": flop_score / (parts["score"] * 1e-3) / 1e12 / peak_fp8,
                     "peak_kind": "measured bf16 burst x 2 (FP8 nominal ratio)", "traffic": None,
                     "attention_tflops": flop_attn / (parts["attend"] * 1e-3) / 1e12},
        # per step: the quantiser, a score and a top-k kernel per launch of up to
        # 2 x SMs query tokens (a pair per CTA), and one attention launch
        "gpu_launches": steps * (2 + 2 * ((T + per_launch - 1) // per_launch)), "clocks": clk.summary()}), flush=True)

if __name__ == "__main__":
    main()
