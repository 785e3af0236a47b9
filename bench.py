"""Benchmark of the paged-KV decode step on GB300.

One step = one pass of the whole hot path over one batch: the slot-mapped
append of each sequence's newest token fused into the decode
(``pkv_append_decode``; ``--separate`` runs ``pkv_append`` then
``pkv_decode_splitk``), with the split count from the heuristic.

The headline (no flags) is the largest configuration, the long-context
split-K decode: B=4, H=32, Hkv=8, D=128, bs=16, contexts of 32K/64K/96K/128K
tokens, 1.34 GB of K/V per call (phase 1 over 10 splits, then the combine).
Its JSON line carries ``sub_records`` for the other configurations, each
timed the same way in the same run: the Llama-3-8B-shaped step (B=32,
L~U[512,2048]), the large ragged batch (B=256, lognormal lengths), the
128-step append+decode loop and the tiny case.  ``--workload`` makes another
shape the headline (``--no-sub`` skips the records), ``--layout vllm`` uses
the vLLM cache layout.

The metric is KV bytes read per second (each token's K and V once, f16),
with decode tokens/s and microseconds per call alongside.  Workloads near
L2's size (the Llama-3-8B step reads 174 MB against a 129 MB L2) rotate four
independent pool sets between steps; the others read far more than L2 holds
per call.

``--impl reference`` times the CPU oracle on the host cores (each step one
whole decode call of the same workload, its sequences spread over one worker
process per sequence, at most one per core) and prints the same JSON line
with ``"impl": "reference"``.

Under ``torchrun`` (N>1) every rank runs its own replica on its own GPU (the
path has no exchange step); time is the max over ranks and ``value`` counts
the bytes all ranks processed.
"""

from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attn: KV HBM GB/s (% of ~8 TB/s), decode tokens/s, \u00b5s/call"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
WORKLOAD_DESC = {
    "llama8b": ("Llama-3-8B-shaped decode step: B=32, H=32, Hkv=8, D=128, bs=16, "
                "context_lens~U[512,2048], block tables drawn without replacement from a "
                "16384-block pool, f16 q/k/v ~N(0,1)"),
    "long": ("long-context split-K decode: B=4, H=32, Hkv=8, D=128, bs=16, context_lens "
             "{32768,65536,98304,131072}, one key per sequence x8, 24576-block pool"),
    "ragged": ("large ragged batch: B=256, H=28, Hkv=4, D=128, bs=32, lognormal context_lens "
               "(median 1024, sigma 1, clipped to [1,16384], 8 of length 1), 200000-block pool, "
               "f16 q/k/v ~N(0,0.5)"),
    "tiny": ("tiny paged decode: B=2, H=4, Hkv=2, D=64, bs=16, context_lens {17,40}, "
             "8-block pool"),
    "spec": ("speculative-decode verification: B=32, H=32, Hkv=8, D=128, bs=16, 4 draft tokens "
             "per sequence over a prefix ~U[508,2044] (pkv_varlen_attention_splitk, causal)"),
    "prefill": ("chunked prefill: B=4, H=32, Hkv=8, D=128, bs=16, 512 new tokens per sequence "
                "after a 2048-token prefix, causal (pkv_varlen_attention_splitk; tensor-bound)"),
    "prefill_one": ("chunked prefill of one sequence: B=1, H=32, Hkv=8, D=128, bs=16, 512 new "
                    "tokens after a 2048-token prefix, causal (pkv_varlen_attention_splitk; "
                    "tensor-bound)"),
    "spec_long": ("speculative-decode verification over long contexts: B=4, H=32, Hkv=8, D=128, "
                  "bs=16, 4 draft tokens per sequence after prefixes {32768,65536,98304,131072}-4, "
                  "24576-block pool (pkv_varlen_attention_splitk, causal)"),
    "qkv_prefill": ("fused QKV split + per-head RMS norm + rotary + paged append on the "
                    "Llama-3-8B attention shape: 4 sequences x 2048 new tokens (H=32, Hkv=8, "
                    "D=128, bs=16), f16 rows ~N(0,1) (pkv_qkv_norm_rope_append)"),
    "step_qkv": ("a whole attention step on the Llama-3-8B decode workload: the 32 new "
                 "tokens' fused QKV rows (RMS-normed q/k heads, rotary at position L-1, "
                 "keys/values appended) and the decode over the grown contexts, in one call "
                 "(pkv_qkv_norm_rope_append_decode); the two-launch form "
                 "(pkv_qkv_norm_rope_append then pkv_decode_splitk) timed beside it"),
    "loop": ("append+decode loop: MHA H=Hkv=16, D=64, bs=16, B=128, start context U[64,4096], "
             "128 steps of pkv_append (142 rows, 14 padding slots = -1, new blocks from a "
             "shuffled free list of 40000) then pkv_decode_splitk on one stream"),
}
N_SETS = 4  # default number of rotating pool sets (--sets)
BASE_QKV_SEED = 20261210

# DRAM bytes (read + write) of one decode launch on this workload, from a
# DRAM-only ncu pass over the workload's kernels (the hash of the kernel's sources at
# capture time: BASE_SOURCES, TC_SOURCES for "sources": "tc", PREFILL_SOURCES
# for "sources": "prefill").  Reported as null when those sources have
# changed since.
NCU_TRAFFIC = {
    # the long-context decode call, split-K phase 1
    # (10 splits, dram read 1,342,345,728 B + write 3,075,584 B) + the combine
    # (read 449,280 B)
    "long": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 1345870592, "num_splits": 10,
             "fused": False, "layout": "blocked",
             "kernel": "paged_decode_kernel<128,16,6,2,split> + splitk_combine_kernel<128>"},
    # the ragged decode call, phase 1 (8 splits, read
    # 810,166,016 B + write 6,290,176 B) + the combine (read 3,282,944 B)
    "ragged": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 819739136, "num_splits": 8,
               "fused": False, "layout": "blocked",
               "kernel": "paged_decode_kernel<128,32,6,2,split> + splitk_combine_kernel<128>"},
    # the fused append + single-pass decode launch,
    # dram read 175,223,808 B + write 3,140,608 B
    "llama8b": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 178364416, "num_splits": 1,
                "fused": True, "layout": "blocked",
                "kernel": "paged_decode_kernel<128,16,6,2,single,fused>"},
    # one paged_varlen_kernel launch (mma.sync),
    # read 174,704,640 B + write 3,002,112 B
    "spec": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 177706752, "num_splits": 1,
             "kernel": "paged_varlen_kernel<128,16,6,2,NT=2,blocked,single>"},
    # one paged_varlen_tc_kernel launch (tcgen05),
    # read 174,740,992 B + write 2,960,640 B
    "spec_tc": {"kernel_hash": "8a6b497ef88a907b", "sources": "tc", "bytes_per_launch": 177701632,
                "num_splits": 1, "kernel": "paged_varlen_tc_kernel<128,16,single>"},
    # the varlen split-K phase 1 (10 splits,
    # read 1,342,488,576 B + write 3,243,008 B) + the combine (read 2,674,176 B)
    "spec_long": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 1348405760,
                  "num_splits": 10,
                  "kernel": "paged_varlen_kernel<128,16,6,2,NT=2,blocked,split> + "
                            "varlen_combine_kernel<128>"},
    # tcgen05 phase 1 (read 1,342,530,816 B +
    # write 3,159,040 B) + the combine (read 2,674,688 B)
    "spec_long_tc": {"kernel_hash": "8a6b497ef88a907b", "sources": "tc",
                     "bytes_per_launch": 1348364544, "num_splits": 10,
                     "kernel": "paged_varlen_tc_kernel<128,16,split> + varlen_combine_kernel<128>"},
    # one paged_prefill_tc_kernel launch, dram read
    # 61,618,944 B + write 2,190,336 B
    "prefill": {"kernel_hash": "ca23019c848f6234", "sources": "prefill", "bytes_per_launch": 63809280,
                "num_splits": 1, "kernel": "paged_prefill_tc_kernel<16>"},
    # one qkv_norm_rope_kernel launch, dram read
    # 102,025,216 B + write 52,952,064 B (the rest of the writes stay in L2)
    "qkv_prefill": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 154977280,
                    "kernel": "qkv_norm_rope_kernel<128,16,3>"},
    # one-launch QKV step: the decode kernel with
    # the QKV norm + rotary + append folded in, dram read 175,252,736 B +
    # write 3,195,392 B
    "step_qkv": {"kernel_hash": "4141458843a655c8", "bytes_per_launch": 178448128,
                 "num_splits": 1, "kernel": "paged_decode_kernel<128,16,6,2,single,qkv>"},
}


def traffic_current(tr):
    """Whether a traffic entry's kernel sources still hash as captured."""
    files = {"tc": TC_SOURCES, "prefill": PREFILL_SOURCES}.get(tr.get("sources"), BASE_SOURCES)
    return tr.get("kernel_hash") == kernel_source_hash(files)


def ncu_traffic(workload, num_splits=None):
    """DRAM bytes per launch of the workload's dominant kernel from the
    committed ncu capture, or None once the kernels have changed since (or
    the split count differs from the captured one)."""
    tr = NCU_TRAFFIC.get(workload)
    if not tr or not traffic_current(tr):
        return None
    if "num_splits" in tr and num_splits != tr["num_splits"]:
        return None
    return tr["bytes_per_launch"]


# The CUDA sources a kernel is built from: every kernel but the tcgen05 ones
# (the varlen kernel adds varlen_tc.cuh, the prefill kernel prefill_tc.cuh as
# well) comes from these three.
BASE_SOURCES = ("kernels.cuh", "ptx.cuh", "pagedkv.cu")
TC_SOURCES = BASE_SOURCES + ("varlen_tc.cuh",)
PREFILL_SOURCES = BASE_SOURCES + ("varlen_tc.cuh", "prefill_tc.cuh")


def kernel_source_hash(files=BASE_SOURCES):
    """Hash of the given CUDA sources with comments and blank lines left out
    (a comment edit does not change a kernel; any code edit does)."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_decode_08_gb300", "csrc", f)) as fh:
            for line in fh:
                code = line.split("//", 1)[0].strip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor TFLOP/s measured on this machine (a burst of cuBLAS
    GEMMs); f16 runs at the same dense rate on these tensor cores."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"]), "measured (bf16 burst; f16 dense rate is the same)"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples (every `interval_ms`) while the timed region runs.
    begin() / end() mark the timed window inside a longer sampled stretch
    (a soak of untimed replays before it), so that the record holds both the
    samples under steady load and those that fell inside the window."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index, interval_ms=200):
        self.gpu_index = gpu_index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.window = None
        self.soak_steps = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def begin(self):
        self.window = [datetime.datetime.now(), None]

    def end(self):
        if self.window:
            self.window[1] = datetime.datetime.now()

    def soak(self, fn, seconds):
        """Run fn() (untimed work) for about `seconds`, to have the GPU at
        steady load when the timed window begins."""
        import torch

        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            for _ in range(8):
                fn()
                self.soak_steps += 1
            torch.cuda.synchronize()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(max(0.05, 1.25 * self.interval_ms / 1e3))
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons, in_window = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                mhz, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            sm.append(mhz)
            smax.append(mx)
            for name, val in zip(names, parts[6:10]):
                if val.lower() == "active":
                    reasons.add(name)
            if self.window and self.window[1]:
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                except ValueError:
                    continue
                if self.window[0] <= ts <= self.window[1]:
                    in_window += 1
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
               "reasons": sorted(reasons), "samples": len(sm),
               "interval_ms": self.interval_ms}
        if self.window:
            out["samples_in_timed_window"] = in_window
            out["soak_steps_before_window"] = self.soak_steps
        return out


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, dist=None, device="cpu"):
    """The largest `value` over all ranks (the job's time is its slowest
    rank's); returns `value` itself without a process group."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank, world, ms_per_step_max):
    """Whole-job GB/s: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_rank / (ms_per_step_max * 1e-3) / 1e9


def cpu_oracle_sample(w, seqs, kc, vc):
    import oracle

    t0 = time.perf_counter()
    oracle.decode_fast(w.q, kc, vc, w.block_tables, w.context_lens, w.scale, seqs=seqs)
    dt = time.perf_counter() - t0
    per_tok = 2 * w.num_kv_heads * w.head_dim * 2
    nbytes = sum(int(w.context_lens[s]) for s in seqs) * per_tok
    return nbytes, dt


# The oracle timed on the host: a fresh interpreter that never touches CUDA
# builds the workload once, then forks one worker per host core (forking is
# safe there: no GPU context exists in that process), at most one per
# sequence; each step is one whole decode call of the workload, its
# sequences spread over the workers.
_ORACLE_STATE = {}


def _oracle_one_seq(s):
    w, kc, vc = _ORACLE_STATE["w"], _ORACLE_STATE["kc"], _ORACLE_STATE["vc"]
    return cpu_oracle_sample(w, [s], kc, vc)[0]


def oracle_child_main(mode, name, steps, warmup, budget_s):
    import multiprocessing as mp

    from paged_kv_decode_08_gb300 import workloads as W

    w = W.make(name)
    kc, vc = W.host_pool(w)
    _ORACLE_STATE.update(w=w, kc=kc, vc=vc)
    # longest sequences first, so the pool's last tasks are the short ones
    seqs = sorted(range(w.num_seqs), key=lambda s: -int(w.context_lens[s]))
    procs = max(1, min(os.cpu_count() or 1, w.num_seqs))
    res = {"procs": procs, "num_seqs": w.num_seqs, "kv_mb": w.kv_bytes / 1e6}
    if mode == "baseline":  # one core: whole decode calls in this process
        tot_b, tot_t, calls = 0, 0.0, 0
        while tot_t < budget_s / 2:
            b, t = cpu_oracle_sample(w, seqs, kc, vc)
            tot_b, tot_t, calls = tot_b + b, tot_t + t, calls + 1
        res["one_core"] = {"bytes": tot_b, "seconds": tot_t, "calls": calls}
    with mp.get_context("fork").Pool(procs) as pool:
        def step():
            t0 = time.perf_counter()
            nb = sum(pool.map(_oracle_one_seq, seqs, chunksize=1))
            return nb, time.perf_counter() - t0

        for _ in range(warmup):
            step()
        tot_b, tot_t, calls = 0, 0.0, 0
        while (calls < steps) if mode == "reference" else (tot_t < budget_s / 2):
            b, t = step()
            tot_b, tot_t, calls = tot_b + b, tot_t + t, calls + 1
        res["all_cores"] = {"bytes": tot_b, "seconds": tot_t, "calls": calls}
    print(json.dumps(res), flush=True)


def run_oracle_child(mode, name, steps=0, warmup=1, budget_s=12.0):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = "1"
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-child", mode,
                          "--workload", name, "--steps", str(steps),
                          "--warmup", str(max(warmup, 3)), "--oracle-budget", str(budget_s)],
                         capture_output=True, text=True, env=env, timeout=1200)
    if res.returncode != 0:
        return None
    return json.loads(res.stdout.strip().splitlines()[-1])


def cpu_baseline_subprocess(name, budget_s=12.0):
    """The oracle on the host cores (one worker per sequence, at most one per
    core) and on one core, about budget_s of CPU time."""
    d = run_oracle_child("baseline", name, budget_s=budget_s)
    if d is None:
        return None
    a, o = d["all_cores"], d["one_core"]
    return {"value": a["bytes"] / a["seconds"] / 1e9, "unit": UNIT, "cores": d["procs"],
            "kind": "oracle",
            "sample": f"{a['calls']} full decode call(s) of the workload ({d['num_seqs']} "
                      f"sequences, {d['kv_mb']:.0f} MB of K/V each) in float64, sequences "
                      f"spread over {d['procs']} worker processes, {a['seconds']:.1f} s",
            "one_core": {"value": o["bytes"] / o["seconds"] / 1e9, "unit": UNIT, "cores": 1,
                         "sample": f"{o['calls']} full decode call(s) on one host thread, "
                                   f"{o['seconds']:.1f} s"}}


def run_reference(args):
    """The oracle on the host cores: each step one whole decode call of the
    workload, its sequences spread over one worker process per sequence (at
    most one per core)."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    name = args.workload
    d = run_oracle_child("reference", name, steps=args.steps, warmup=args.warmup)
    if d is None:
        print(json.dumps({"impl": "reference", "unavailable": "the oracle child process failed"}),
              flush=True)
        return
    a = d["all_cores"]
    value = a["bytes"] / a["seconds"] / 1e9
    sample = (f"whole decode calls ({d['num_seqs']} sequences, {d['kv_mb']:.0f} MB of K/V) per "
              f"step, float64 numpy oracle, sequences spread over {d['procs']} worker processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": a["calls"], "warmup": args.warmup, "ms_per_step": a["seconds"] / a["calls"] * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[name],
                   "sample_per_step": f"all {d['num_seqs']} sequences"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": d["procs"], "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_qkv(args):
    """The fused QKV split + norm + rotary + append step on a prefill-sized
    call.  Bytes per call: the rows read (q, k, v heads), the cos/sin rows read
    and the queries, keys and values written; rotating input sets keep the
    reads out of L2."""
    import numpy as np
    import torch

    from paged_kv_decode_08_gb300 import pagedkv as pk
    from paged_kv_decode_08_gb300 import workloads as W

    world, rank, local = dist_setup()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    H, Hkv, D, bs = 32, 8, 128, 16
    c = W.qkv_case(BASE_QKV_SEED, H, Hkv, D, bs, [2048] * 4, [0] * 4)
    n_sets = args.sets or N_SETS
    g = torch.Generator(device=dev)
    sets = []
    for r in range(n_sets):
        g.manual_seed(2000 + r)
        qkv = (torch.from_numpy(c.qkv).to(dev) if r == 0 else
               torch.randn(c.qkv.shape, generator=g, device=dev).to(torch.float16))
        shape = (c.num_blocks, Hkv, bs, D)
        sets.append({"qkv": qkv, "kc": torch.empty(shape, dtype=torch.float16, device=dev),
                     "vc": torch.empty(shape, dtype=torch.float16, device=dev),
                     "q_out": torch.empty((c.qkv.shape[0], H, D), dtype=torch.float16,
                                          device=dev)})
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qw, kw, cos, sin = t(c.q_norm_w), t(c.k_norm_w), t(c.cos), t(c.sin)
    cu, pos, bt = t(c.cu_seqlens_q), t(c.pos_offsets), t(c.block_tables)

    def call(i):
        st = sets[i % n_sets]
        pk.pkv_qkv_norm_rope_append(st["qkv"], qw, kw, cos, sin, st["kc"], st["vc"], cu, pos, bt,
                                    H, eps=c.eps, q_out=st["q_out"])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(n_sets):
            call(i)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(n_sets):
            call(i)
    rounds = max(1, args.steps // n_sets)
    for _ in range(max(1, args.warmup // n_sets)):
        graph.replay()
    torch.cuda.synchronize()
    flags = pk.pkv_read_device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after warm-up")
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        a.record()
        for _ in range(rounds):
            graph.replay()
        b.record()
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (rounds * n_sets)
    if rank != 0:
        return
    T = c.qkv.shape[0]
    nbytes = (T * (H + 2 * Hkv) * D * 2          # rows read
              + T * D * 4                          # cos and sin rows read (f32, D/2 each)
              + T * (H + 2 * Hkv) * D * 2)         # queries, keys and values written
    peak, peak_kind = measured_peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": job_throughput(nbytes, world, ms), "unit": UNIT,
        "n_gpus": world, "steps": rounds * n_sets, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC["qkv_prefill"], "launch": "CUDA graph, replayed",
                   "l2": f"{n_sets} rotating input sets; {nbytes / 1e6:.0f} MB moved per call"},
        "bytes_per_step": nbytes, "us_per_step": ms * 1e3,
        "tokens_per_s": world * T / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": "qkv_norm_rope_kernel (bytes read + written)",
                     "traffic": ncu_traffic("qkv_prefill")},
        "clocks": clocks.summary(), "gpu_launches": rounds * n_sets,
        "device_status_flags": pk.pkv_read_device_status(), "e2e": None, "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def run_step_qkv(args):
    """A whole attention step: the fused QKV split + norm + rotary + append of
    each sequence's new token, then the decode (two launches), timed as a
    graph of steps over rotating pool sets; the decode alone is timed beside
    it."""
    import numpy as np
    import torch

    from paged_kv_decode_08_gb300 import pagedkv as pk
    from paged_kv_decode_08_gb300 import workloads as W

    world, rank, local = dist_setup()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = W.make("llama8b")
    n_sets = args.sets or N_SETS
    sets = build_sets(w, dev, n_sets)
    lens = w.context_lens.astype(np.int64)
    c = W.qkv_case(BASE_QKV_SEED + 1, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size,
                   [1] * w.num_seqs, (lens - 1).tolist())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    qkv, qw, kw, cos, sin = t(c.qkv), t(c.q_norm_w), t(c.k_norm_w), t(c.cos), t(c.sin)
    cu, pos = t(c.cu_seqlens_q), t(c.pos_offsets)
    bt, cl = sets[0]["block_tables"], sets[0]["context_lens"]
    q = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float16, device=dev)
    out = torch.empty_like(q)
    S = pk.splits_for(q, sets[0]["k_cache"], bt, args.splits)
    scratch = pk.alloc_scratch(q, sets[0]["k_cache"], bt, args.splits)

    def step(i):
        st = sets[i % n_sets]
        pk.pkv_qkv_norm_rope_append(qkv, qw, kw, cos, sin, st["k_cache"], st["v_cache"], cu, pos,
                                    bt, w.num_heads, eps=c.eps, q_out=q)
        pk.pkv_decode_splitk(q, st["k_cache"], st["v_cache"], bt, cl, w.scale,
                             num_splits=args.splits, scratch=scratch, out=out)

    def fused(i):
        st = sets[i % n_sets]
        pk.pkv_qkv_norm_rope_append_decode(qkv, qw, kw, cos, sin, st["k_cache"], st["v_cache"],
                                           bt, cl, w.num_heads, w.scale, eps=c.eps,
                                           num_splits=args.splits, scratch=scratch, out=out)

    def decode_only(i):
        st = sets[i % n_sets]
        pk.pkv_decode_splitk(q, st["k_cache"], st["v_cache"], bt, cl, w.scale,
                             num_splits=args.splits, scratch=scratch, out=out)

    def capture(fn):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(n_sets):
                fn(i)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_sets):
                fn(i)
        return g

    g_step, g_fused, g_dec = capture(step), capture(fused), capture(decode_only)
    rounds = max(1, args.steps // n_sets)
    for _ in range(max(1, args.warmup // n_sets)):
        g_step.replay()
        g_fused.replay()
        g_dec.replay()
    torch.cuda.synchronize()
    flags = pk.pkv_read_device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after warm-up")

    def timed(g):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(rounds):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (rounds * n_sets)

    with ClockSampler(local) as clocks:
        two_ms = timed(g_step)
        ms = timed(g_fused)
        dec_ms = timed(g_dec)
    if rank != 0:
        return
    kv_bytes = w.kv_bytes
    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": job_throughput(kv_bytes, world, ms), "unit": UNIT,
        "n_gpus": world, "steps": rounds * n_sets, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC["step_qkv"], "num_splits": S,
                   "launch": f"CUDA graph of {n_sets} steps, replayed",
                   "l2": f"{n_sets} rotating pool sets"},
        "kv_bytes_per_step": kv_bytes, "us_per_step": ms * 1e3,
        "two_launch_us_per_step": two_ms * 1e3, "decode_us_per_call": dec_ms * 1e3,
        "decode_tokens_per_s": world * w.num_seqs / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": ("the step's single launch (QKV norm + rotary + append fused "
                                "into the decode)" if S <= 1 else
                                "the step (fused decode phase 1 + combine)"),
                     "traffic": ncu_traffic("step_qkv", S)},
        "clocks": clocks.summary(), "gpu_launches": rounds * n_sets * (1 + (S > 1)),
        "device_status_flags": pk.pkv_read_device_status(), "e2e": None, "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def build_sets(w, dev, n_sets, layout="blocked"):
    """Device pools for the workload: set 0 holds the generator's values, the
    others the same tables with fresh N(0,1) pools (distinct HBM bytes)."""
    import torch

    from paged_kv_decode_08_gb300 import workloads as W

    sets = []
    base = (W.to_device_vllm if layout == "vllm" else W.to_device)(w, dev, upto_last=True)
    sets.append(base)
    g = torch.Generator(device=dev)
    for r in range(1, n_sets):
        g.manual_seed(1000 + r)
        kc = torch.randn(base["k_cache"].shape, generator=g, device=dev).to(torch.float16)
        vc = torch.randn(base["v_cache"].shape, generator=g, device=dev).to(torch.float16)
        sets.append({**base, "k_cache": kc, "v_cache": vc})
    return sets


def run_loop(args):
    world, rank, local = dist_setup()
    line = measure_loop(args, local, world, rank)
    if line is not None:
        print(json.dumps(line), flush=True)


def measure_loop(args, local, world, rank):
    """The append+decode loop: every step appends one token per sequence
    (plus padding rows) and decodes over the grown contexts.  All 128 steps'
    inputs are uploaded first; the whole loop is one CUDA graph, replayed
    (re-appending the same rows to the same slots, so every replay does the
    same work).  Returns the JSON line (rank 0) or None."""
    import torch

    from paged_kv_decode_08_gb300 import pagedkv as pk
    from paged_kv_decode_08_gb300 import workloads as W

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    loop = W.AppendDecodeLoop()
    d0 = W.to_device(loop.initial_workload(), dev)
    kc, vc = d0["k_cache"], d0["v_cache"]
    steps = []
    for t in range(loop.steps):
        st = loop.step(t)
        steps.append({k: torch.from_numpy(getattr(st, k)).to(dev) for k in
                      ("k_new", "v_new", "slot_mapping", "q", "block_tables", "context_lens")})
    q0, bt0 = steps[0]["q"], steps[0]["block_tables"]
    S = pk.splits_for(q0, kc, bt0, args.splits)
    scratch = pk.alloc_scratch(q0, kc, bt0, args.splits)
    out = torch.empty_like(q0)

    def append(t):
        x = steps[t]
        pk.pkv_append(x["k_new"], x["v_new"], x["slot_mapping"], kc, vc)

    def decode(t):
        x = steps[t]
        pk.pkv_decode_splitk(x["q"], kc, vc, x["block_tables"], x["context_lens"], loop.scale,
                             num_splits=args.splits, scratch=scratch, out=out)

    def capture(fns):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for t in range(loop.steps):
                for f in fns:
                    f(t)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for t in range(loop.steps):
                for f in fns:
                    f(t)
        return g

    g_loop = capture([append, decode])
    g_append = capture([append])
    g_decode = capture([decode])
    reps = max(1, args.steps // loop.steps)
    for g in (g_loop, g_append, g_decode):
        g.replay()
    torch.cuda.synchronize()
    flags = pk.pkv_read_device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after warm-up")

    def timed(g):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / (reps * loop.steps)

    with ClockSampler(local) as clocks:
        step_ms = timed(g_loop)
        append_ms = timed(g_append)
        decode_ms = timed(g_decode)
    flags = pk.pkv_read_device_status()
    if rank != 0:
        return None
    kv_bytes = sum(loop.kv_bytes_per_step) / loop.steps
    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (decode_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": job_throughput(kv_bytes, world, step_ms), "unit": UNIT,
        "n_gpus": world, "steps": reps * loop.steps, "warmup": loop.steps,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC["loop"], "num_splits": S,
                   "launch": "CUDA graph of the 128-step loop, replayed",
                   "l2": f"{kv_bytes / 1e6:.0f} MB of K/V read per decode vs 129 MB L2"},
        "kv_bytes_per_step": kv_bytes,
        "decode_tokens_per_s": world * loop.num_seqs / (step_ms * 1e-3),
        "us_per_step": step_ms * 1e3, "append_us_per_step": append_ms * 1e3,
        "decode_us_per_call": decode_ms * 1e3, "pct_of_8TBs": 100.0 * achieved / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": "decode call", "traffic": None},
        "clocks": clocks.summary(), "gpu_launches": reps * loop.steps * (1 + (2 if S > 1 else 1)),
        "device_status_flags": flags, "e2e": None, "cpu_baseline": None,
    }
    return line


def run_varlen(args):
    line = measure_varlen(args, args.workload, args.varlen_tc)
    if line is not None:
        print(json.dumps(line), flush=True)


def measure_varlen(args, workload, tensor_path):
    """Speculative verification: 4 query tokens per sequence, causal, over
    the paged context (pkv_varlen_attention_splitk; the split count is the
    library's heuristic unless --splits forces one), on the mma.sync kernel
    or (tensor_path) the tcgen05 one.  Algorithmic bytes count each
    sequence's context once; a CTA covers max(1, 8 NT / G) queries (NT = 2
    n-tiles once a sequence has more than 8 query-head pairs), so the kernel
    reads a context ceil(q_len / that) times: once for 4 queries at G = 4.
    Returns rank 0's line (None on the other ranks)."""
    import torch

    from paged_kv_decode_08_gb300 import pagedkv as pk
    from paged_kv_decode_08_gb300 import workloads as W

    world, rank, local = dist_setup()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    prev_path = pk.pkv_set_varlen_tensor_path(1 if tensor_path else 0)
    try:
        return _measure_varlen(args, workload, tensor_path, pk, W, world, rank, local, dev)
    finally:
        pk.pkv_set_varlen_tensor_path(prev_path)


def _measure_varlen(args, workload, tensor_path, pk, W, world, rank, local, dev):
    import numpy as np
    import torch

    v = {"spec_long": W.spec_verify_long, "prefill": W.prefill_chunk,
         "prefill_one": W.prefill_one}.get(workload, W.spec_verify)()
    w = v.base
    n_sets = args.sets or N_SETS
    sets = build_sets(w, dev, n_sets)
    q = torch.from_numpy(v.q).to(dev)
    cu = torch.from_numpy(v.cu_seqlens_q).to(dev)
    pos = torch.from_numpy(v.pos_offsets).to(dev)
    out = torch.empty_like(q)
    S, n = pk._varlen_plan(q, sets[0]["k_cache"], sets[0]["block_tables"], v.max_q_len,
                           args.splits)
    scratch = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)

    def call(i):
        st = sets[i % n_sets]
        pk.pkv_varlen_attention_splitk(q, st["k_cache"], st["v_cache"], cu, pos,
                                       st["block_tables"], w.scale, max_q_len=v.max_q_len,
                                       num_splits=args.splits, scratch=scratch, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(n_sets):
            call(i)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n_sets):
            call(i)
    rounds = max(1, args.steps // n_sets)
    for _ in range(max(1, args.warmup // n_sets)):
        g.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        a.record()
        for _ in range(rounds):
            g.replay()
        b.record()
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (rounds * n_sets)
    if rank != 0:
        return None
    kv_bytes = w.kv_bytes
    G = w.group
    prefill = v.max_q_len * G >= 128 and w.head_dim == 128  # the prefill kernel, any S
    nt = 2 if v.max_q_len * G > 8 else 1
    per_cta = 2 * (128 // G) if prefill else max(1, 8 * nt // G)  # prefill: two 128-row tiles
    reads = -(-int(v.max_q_len) // per_cta)
    peak, peak_kind = measured_peaks()
    achieved = kv_bytes / (ms * 1e-3) / 1e9
    tc = prefill or (tensor_path and v.max_q_len * G > 8 and w.head_dim == 128)
    tr = NCU_TRAFFIC.get(workload + ("_tc" if tc and not prefill else ""))
    traffic = (tr["bytes_per_launch"] if tr and traffic_current(tr)
               and S == tr.get("num_splits") else None)
    line = {
        "metric": METRIC, "value": job_throughput(kv_bytes, world, ms), "unit": UNIT,
        "n_gpus": world, "steps": rounds * n_sets, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[workload], "launch": "CUDA graph, replayed",
                   "num_splits": S, "context_reads_per_call": reads,
                   "kernel_path": ("tcgen05 prefill" if prefill else
                                   "tcgen05" if tc else "mma.sync"),
                   "l2": f"{n_sets} rotating pool sets; {reads * kv_bytes / 1e6:.0f} MB read per call"},
        "kv_bytes_per_step": kv_bytes, "us_per_step": ms * 1e3,
        "query_tokens_per_s": world * v.total_q / (ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": (("paged_varlen_tc_kernel" if tc else "paged_varlen_kernel")
                                + (" split-K phase 1 + varlen_combine_kernel" if S > 1 else "")
                                + " (algorithmic bytes: each context once)"),
                     "bytes_read_frac": reads * achieved / peak, "traffic": traffic,
                     "traffic_kernel": tr["kernel"] if traffic is not None else None},
        "clocks": clocks.summary(), "gpu_launches": rounds * n_sets * (2 if S > 1 else 1),
        "device_status_flags": pk.pkv_read_device_status(), "e2e": None, "cpu_baseline": None,
    }
    if prefill:
        # tensor-bound: causal attention flops (4 D per query, head and
        # position it sees) over the measured dense f16/bf16 peak
        lens = v.pos_offsets.astype(np.int64)
        qls = np.diff(v.cu_seqlens_q).astype(np.int64)
        pairs = int(sum(ql * (p0 + 1) + ql * (ql - 1) // 2 for p0, ql in zip(lens, qls)))
        flops = 4.0 * w.head_dim * w.num_heads * pairs
        tpeak, tkind = measured_tensor_peak()
        tflops = flops / (ms * 1e-3) / 1e12
        line["flops_per_step"] = flops
        line["roofline"] = {
            "bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
            "frac": tflops / tpeak, "peak_source": tkind,
            "kernel": ("paged_prefill_tc_kernel" + (" split-K phase 1 + varlen_combine_kernel"
                                                     if S > 1 else "")
                       + " (algorithmic flops: the causal triangle, 4 * head_dim per "
                         "(query, head, position))"),
            "kv_gbs_contexts_once": achieved, "traffic": traffic}
    return line


def measure_step(args, name, dev, dist, world, rank, n_sets, want_e2e, want_cpu):
    """One decode step of workload `name` (the fused append + decode, or with
    --separate / --layout vllm the append then the decode), timed as CUDA
    graph replays over `n_sets` rotating pool sets, plus the decode call
    alone; with `want_e2e` also end to end from host buffers.  Returns the
    JSON line (rank 0) or None."""
    import torch

    from paged_kv_decode_08_gb300 import pagedkv as pk
    from paged_kv_decode_08_gb300 import workloads as W

    w = W.make(name)
    vllm = args.layout == "vllm"
    separate = args.separate or vllm  # no fused append on the vLLM layout
    sets = build_sets(w, dev, n_sets, args.layout)
    append_call = pk.pkv_append_vllm_layout if vllm else pk.pkv_append
    decode_call = pk.pkv_decode_vllm_layout if vllm else pk.pkv_decode_splitk
    k_new, v_new, slots = w.last_token_append()
    k_new_d = torch.from_numpy(k_new).to(dev)
    v_new_d = torch.from_numpy(v_new).to(dev)
    slots_d = torch.from_numpy(slots).to(dev)
    q, bt, cl = sets[0]["q"], sets[0]["block_tables"], sets[0]["context_lens"]
    S = pk.splits_for(q, sets[0]["k_cache"], bt, args.splits)
    scratch = pk.alloc_scratch(q, sets[0]["k_cache"], bt, args.splits)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()
    kv_bytes = w.kv_bytes
    launches_per_step = (1 if separate else 0) + (2 if S > 1 else 1)

    def step(i):
        st = sets[i % n_sets]
        if separate:
            append_call(k_new_d, v_new_d, slots_d, st["k_cache"], st["v_cache"])
            decode_call(q, st["k_cache"], st["v_cache"], bt, cl, w.scale,
                        num_splits=args.splits, scratch=scratch, out=out)
        else:
            pk.pkv_append_decode(k_new_d, v_new_d, slots_d, st["k_cache"], st["v_cache"], q, bt,
                                 cl, w.scale, num_splits=args.splits, scratch=scratch, out=out)

    def decode_only(i):
        st = sets[i % n_sets]
        decode_call(q, st["k_cache"], st["v_cache"], bt, cl, w.scale,
                    num_splits=args.splits, scratch=scratch, out=out)

    def capture(fn):
        """A CUDA graph of one round: fn(i) for every pool set in turn."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for i in range(n_sets):
                fn(i)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n_sets):
                fn(i)
        return g

    g_step = capture(step)
    g_decode = capture(decode_only)
    rounds = max(1, args.steps // n_sets)
    steps = rounds * n_sets
    for _ in range(max(1, args.warmup // n_sets)):
        g_step.replay()
        g_decode.replay()
    torch.cuda.synchronize()
    flags = pk.pkv_read_device_status()
    if flags:
        raise RuntimeError(f"device status flags {flags:#x} after warm-up")

    def timed(g):
        """Total ms over `rounds` back-to-back replays, and the ms of each
        replay (events between replays; the total spans first to last)."""
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(rounds + 1)]
        ev[0].record(stream)
        for r in range(rounds):
            g.replay()
            ev[r + 1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[-1]), [ev[r].elapsed_time(ev[r + 1]) for r in range(rounds)]

    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # clocks: sampled every 20 ms through an untimed soak of the same graph
    # (about 0.3 s, so the samples show the clocks under steady load) and the
    # timed window right after it
    with ClockSampler(dev.index, interval_ms=20) as clocks:
        clocks.soak(g_step.replay, 0.3)
        clocks.begin()
        total_ms, step_rounds = timed(g_step)
        decode_total_ms, decode_rounds = timed(g_decode)
        clocks.end()
    if dist is not None:
        dist.barrier()
    total_ms = max_over_ranks(total_ms, dist, dev)
    decode_total_ms = max_over_ranks(decode_total_ms, dist, dev)
    decode_ms = decode_total_ms / steps

    # end to end through the public API: each step copies its host inputs
    # (q, the new K/V rows, slots, block tables, lengths), packed in one
    # pinned buffer, to the device in one copy, runs the step on views of
    # that device buffer, and copies the output back to pinned memory.
    e2e = None
    if want_e2e:
        import numpy as np

        parts = [("q", np.ascontiguousarray(w.q)), ("k", np.ascontiguousarray(k_new)),
                 ("v", np.ascontiguousarray(v_new)), ("slots", np.ascontiguousarray(slots)),
                 ("bt", np.ascontiguousarray(w.block_tables)),
                 ("cl", np.ascontiguousarray(w.context_lens))]
        offs, cur = {}, 0
        for pname, a in parts:
            offs[pname] = cur
            cur += (a.nbytes + 255) // 256 * 256
        h_buf = torch.empty(cur, dtype=torch.uint8).pin_memory()
        for pname, a in parts:
            h_buf[offs[pname]:offs[pname] + a.nbytes] = torch.from_numpy(
                a.view(np.uint8).reshape(-1))
        d_buf = torch.empty(cur, dtype=torch.uint8, device=dev)

        def view(pname, a, dtype):
            return d_buf[offs[pname]:offs[pname] + a.nbytes].view(dtype).view(a.shape)

        d_q = view("q", w.q, torch.float16)
        d_k = view("k", k_new, torch.float16)
        d_v = view("v", v_new, torch.float16)
        d_s = view("slots", slots, torch.int32)
        d_bt = view("bt", w.block_tables, torch.int32)
        d_cl = view("cl", w.context_lens, torch.int32)
        h_out = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()
        h2d = sum(a.nbytes for _, a in parts)
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step(i):
            st = sets[i % n_sets]
            d_buf.copy_(h_buf, non_blocking=True)
            if separate:
                append_call(d_k, d_v, d_s, st["k_cache"], st["v_cache"], stream=stream)
                decode_call(d_q, st["k_cache"], st["v_cache"], d_bt, d_cl, w.scale,
                            num_splits=args.splits, scratch=scratch, out=out, stream=stream)
            else:
                pk.pkv_append_decode(d_k, d_v, d_s, st["k_cache"], st["v_cache"], d_q, d_bt,
                                     d_cl, w.scale, num_splits=args.splits, scratch=scratch,
                                     out=out, stream=stream)
            h_out.copy_(out, non_blocking=True)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(args.steps):
            e2e_step(i)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b), dist, dev)
        e2e = {"value": job_throughput(kv_bytes, world, e2e_ms / args.steps), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms / args.steps,
               "how": "direct Python calls each step: one pinned H2D copy of the packed step "
                      "inputs, the step, one D2H copy of the output"}
        if not separate:
            # the same steps with the kernels reading the pinned inputs and
            # writing the pinned output in place (no copies; pools on the GPU)
            h_view = {pname: h_buf[offs[pname]:offs[pname] + a.nbytes] for pname, a in parts}
            h_out2 = torch.empty(tuple(q.shape), dtype=torch.float16).pin_memory()

            def zc_step(i):
                st = sets[i % n_sets]
                rc = pk.lib.pkv_append_decode(
                    h_view["k"].data_ptr(), h_view["v"].data_ptr(), h_view["slots"].data_ptr(),
                    st["k_cache"].data_ptr(), st["v_cache"].data_ptr(), h_view["q"].data_ptr(),
                    h_view["bt"].data_ptr(), h_view["cl"].data_ptr(), w.num_seqs,
                    w.max_blocks_per_seq, w.num_blocks, float(w.scale), w.num_heads,
                    w.num_kv_heads, w.head_dim, w.block_size, h_out2.data_ptr(),
                    int(args.splits), scratch.data_ptr(), scratch.numel(), stream.cuda_stream)
                if rc != pk.PKV_OK:
                    raise RuntimeError(pk.last_error())

            for i in range(args.warmup):
                zc_step(i)
            torch.cuda.synchronize()
            a.record(stream)
            for i in range(args.steps):
                zc_step(i)
            b.record(stream)
            torch.cuda.synchronize()
            zc_ms = max_over_ranks(a.elapsed_time(b), dist, dev)
            e2e["zero_copy"] = {
                "value": job_throughput(kv_bytes, world, zc_ms / args.steps), "unit": UNIT,
                "ms_per_step": zc_ms / args.steps, "host_bytes_read_per_step": h2d,
                "host_bytes_written_per_step": d2h,
                "how": "the same steps through the C ABI with the packed inputs and the output "
                       "in page-locked host memory, read and written by the kernels in place "
                       "(no copies)"}

    flags = pk.pkv_read_device_status()
    if rank != 0:
        return None
    ms_per_step = total_ms / steps
    value = job_throughput(kv_bytes, world, ms_per_step)
    # The dominant kernel: the step's single fused launch when it is one
    # (pkv_append_decode, single pass), else the decode call (phase 1 +
    # combine when split) timed on its own.
    one_launch = not separate and S == 1
    kernel_ms = ms_per_step if one_launch else decode_ms
    achieved = kv_bytes / (kernel_ms * 1e-3) / 1e9
    peak, peak_kind = measured_peaks()
    traffic = None
    tr = NCU_TRAFFIC.get(name)
    if (tr and traffic_current(tr) and S == tr.get("num_splits")
            and one_launch == tr.get("fused", False) and tr.get("layout", "blocked") == args.layout):
        traffic = tr["bytes_per_launch"]
    cpu = cpu_baseline_subprocess(name) if want_cpu else None
    l2_bytes = n_sets * 2 * sets[0]["k_cache"].numel() * 2
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[name],
                   "step": (f"pkv_append_vllm_layout ({w.num_seqs} tokens) + "
                            "pkv_decode_vllm_layout (vLLM cache layout)" if vllm else
                            f"pkv_append ({w.num_seqs} tokens) + pkv_decode_splitk"
                            if separate else
                            f"pkv_append_decode (slot-mapped append of the {w.num_seqs} "
                            "newest tokens fused with the decode)")
                           + f", split count {'heuristic' if args.splits == 0 else 'forced'}",
                   "num_splits": S,
                   "launch": f"CUDA graph of {n_sets} step(s) (one per pool set), replayed",
                   "l2": (f"{n_sets} rotating pool set(s) ({l2_bytes / 1e9:.1f} GB; "
                          f"{kv_bytes / 1e6:.0f} MB of K/V read per step) vs 129 MB L2"
                          + ("" if n_sets > 1 else ": inputs larger than L2")),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "kv_bytes_per_step": kv_bytes,
        "decode_tokens_per_s": world * w.num_seqs / (ms_per_step * 1e-3),
        "us_per_step": ms_per_step * 1e3,
        "decode_us_per_call": decode_ms * 1e3,
        # per replay of the graph (n_sets steps), divided by n_sets
        "us_per_step_median": 1e3 * statistics.median(step_rounds) / n_sets,
        "us_per_step_min": 1e3 * min(step_rounds) / n_sets,
        "decode_us_median": 1e3 * statistics.median(decode_rounds) / n_sets,
        "decode_us_min": 1e3 * min(decode_rounds) / n_sets,
        "pct_of_8TBs": 100.0 * achieved / NOMINAL_HBM_GBS,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_kind,
                     "kernel": ("the step's single launch (fused append + single-pass decode), "
                                "timed as a graph of back-to-back steps" if one_launch else
                                "decode call (single-pass kernel, or split-K phase 1 + combine "
                                "when split), timed as a graph of back-to-back decode calls"),
                     "traffic": traffic,
                     "traffic_kernel": tr["kernel"] if traffic is not None else None},
        "clocks": clocks.summary(),
        "gpu_launches": launches_per_step * steps,
        "device_status_flags": flags,
        "e2e": e2e,
        "cpu_baseline": cpu,
    }
    return line


def sub_record(line, name):
    """The per-config summary kept beside the headline: time per call and
    step, bytes, roofline fraction and the clock record of that run."""
    peak, _ = measured_peaks()
    dec_us = line.get("decode_us_per_call", line["us_per_step"])
    kv = line["kv_bytes_per_step"]
    return {"workload": line["config"]["workload"], "name": name,
            "num_splits": line["config"].get("num_splits"),
            "us_per_call": dec_us, "us_per_step": line["us_per_step"], "kv_bytes": kv,
            "append_us_per_step": line.get("append_us_per_step"),
            "kv_gbs": kv / (dec_us * 1e-6) / 1e9,
            "frac": line["roofline"]["frac"], "frac_kernel": line["roofline"]["kernel"],
            "bound": line["roofline"]["bound"], "achieved": line["roofline"]["achieved"],
            "achieved_unit": line["roofline"]["unit"],
            "frac_of_decode_call": (kv / (dec_us * 1e-6) / 1e9 / peak
                                    if line["roofline"]["bound"] == "hbm" else None),
            "decode_tokens_per_s": line.get("decode_tokens_per_s"),
            "query_tokens_per_s": line.get("query_tokens_per_s"),
            "kernel_path": line["config"].get("kernel_path"),
            "traffic": line["roofline"].get("traffic"),
            "gpu_launches": line["gpu_launches"], "steps": line["steps"],
            "e2e": line.get("e2e"),
            "clocks": line["clocks"], "device_status_flags": line["device_status_flags"]}


def c_driver_record(steps=200, warmup=20):
    """The plain-C end-to-end driver (tests/c_abi/e2e_step.c) on the
    Llama-3-8B-shaped step: host buffers, one packed copy in, the step, the
    output copied back; reports the library's host time per call apart from
    Python.  None when it cannot be built or run."""
    from paged_kv_decode_08_gb300 import build

    try:
        exe = build.build_c_e2e()
        r = subprocess.run([exe, str(steps), str(warmup)], capture_output=True, text=True,
                           timeout=600)
    except (RuntimeError, OSError, subprocess.TimeoutExpired) as e:
        return {"unavailable": str(e).splitlines()[0][:200]}
    if r.returncode != 0:
        return {"unavailable": (r.stderr or r.stdout).strip()[:200]}
    return json.loads(r.stdout.strip().splitlines()[-1])


# Configurations timed beside the headline (name, rotating pool sets): the
# Llama-3-8B step reads 174 MB, near L2's 129 MB, so its pools rotate; the
# others read 0.8-1.3 GB per call, far above L2.
SUB_CONFIGS = [("llama8b", N_SETS, True), ("ragged", 1, False), ("loop", None, False),
               ("tiny", N_SETS, False), ("spec", N_SETS, False), ("spec_tc", N_SETS, False),
               ("prefill", N_SETS, False)]


def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)

    name = args.workload
    n_sets = args.sets if args.sets else (1 if name in ("long", "ragged") else N_SETS)
    line = measure_step(args, name, dev, dist, world, rank, n_sets, want_e2e=not args.no_e2e,
                        want_cpu=not args.no_cpu_baseline)
    torch.cuda.empty_cache()
    subs = []
    if not args.no_sub and world == 1 and name == "long":
        for sub, sets, e2e in SUB_CONFIGS:
            if sub == "loop":
                r = measure_loop(args, local, world, rank)
            elif sub in ("spec", "spec_tc"):
                r = measure_varlen(args, "spec", sub == "spec_tc")
            elif sub == "prefill":
                r = measure_varlen(args, "prefill", False)
            else:
                r = measure_step(args, sub, dev, None, world, rank, sets,
                                 want_e2e=e2e and not args.no_e2e, want_cpu=False)
            torch.cuda.empty_cache()
            if r is not None:
                subs.append(sub_record(r, sub))
    if rank == 0:
        line["sub_records"] = subs
        if not args.no_sub and world == 1 and name == "long":
            line["c_e2e_llama8b"] = c_driver_record()
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_profile(args):
    """A few plain calls of the step (no graph, no timing) for profiler
    captures: the workload over a compact pool (the blocks it reads,
    re-permuted; see workloads.compact_pool) so that a capture saves and
    restores little device memory.  `loop` runs its first steps (append of
    142 rows, then the decode)."""
    import torch

    from paged_kv_decode_08_gb300 import pagedkv as pk
    from paged_kv_decode_08_gb300 import workloads as W

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    n = args.ncu_calls
    pk.pkv_set_varlen_tensor_path(1 if args.varlen_tc else 0)
    if args.workload in ("spec", "spec_long", "prefill", "prefill_one"):
        import dataclasses

        v = {"spec_long": W.spec_verify_long, "prefill": W.prefill_chunk,
             "prefill_one": W.prefill_one}.get(args.workload, W.spec_verify)()
        v = dataclasses.replace(v, base=W.compact_pool(v.base))
        d = W.to_device(v.base, dev)
        q = torch.from_numpy(v.q).to(dev)
        cu = torch.from_numpy(v.cu_seqlens_q).to(dev)
        pos = torch.from_numpy(v.pos_offsets).to(dev)
        for _ in range(n):
            pk.pkv_varlen_attention_splitk(q, d["k_cache"], d["v_cache"], cu, pos,
                                           d["block_tables"], v.base.scale,
                                           max_q_len=v.max_q_len, num_splits=args.splits)
    elif args.workload == "loop":
        loop = W.AppendDecodeLoop()
        d0 = W.to_device(loop.initial_workload(), dev)
        kc, vc = d0["k_cache"], d0["v_cache"]
        for t in range(n):
            st = loop.step(t)
            x = {k: torch.from_numpy(getattr(st, k)).to(dev) for k in
                 ("k_new", "v_new", "slot_mapping", "q", "block_tables", "context_lens")}
            pk.pkv_append(x["k_new"], x["v_new"], x["slot_mapping"], kc, vc)
            pk.pkv_decode_splitk(x["q"], kc, vc, x["block_tables"], x["context_lens"], loop.scale,
                                 num_splits=args.splits)
    else:
        w = W.compact_pool(W.make(args.workload))
        d = W.to_device(w, dev, upto_last=True)
        k_new, v_new, slots = (torch.from_numpy(a).to(dev) for a in w.last_token_append())
        scratch = pk.alloc_scratch(d["q"], d["k_cache"], d["block_tables"], args.splits)
        out = torch.empty_like(d["q"])
        for _ in range(n):
            if args.separate:
                pk.pkv_append(k_new, v_new, slots, d["k_cache"], d["v_cache"])
                pk.pkv_decode_splitk(d["q"], d["k_cache"], d["v_cache"], d["block_tables"],
                                     d["context_lens"], w.scale, num_splits=args.splits,
                                     scratch=scratch, out=out)
            else:
                pk.pkv_append_decode(k_new, v_new, slots, d["k_cache"], d["v_cache"], d["q"],
                                     d["block_tables"], d["context_lens"], w.scale,
                                     num_splits=args.splits, scratch=scratch, out=out)
    torch.cuda.synchronize()
    flags = pk.pkv_read_device_status()
    print(json.dumps({"profile_calls": n, "workload": args.workload, "status_flags": flags}))
    if flags:
        raise SystemExit(f"device status flags {flags:#x}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--splits", type=int, default=0, help="0 = heuristic")
    ap.add_argument("--sets", type=int, default=0,
                    help="rotating pool sets (0 = 4 for workloads near L2's size, 1 for those "
                         "far above it)")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_DESC), default="long",
                    help="the headline workload (default: the long-context split-K decode, "
                         "the largest configuration)")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the per-configuration records timed beside the headline")
    ap.add_argument("--separate", action="store_true",
                    help="step = pkv_append then pkv_decode_splitk (two calls) instead of "
                         "the fused pkv_append_decode")
    ap.add_argument("--layout", choices=["blocked", "vllm"], default="blocked",
                    help="cache layout: [NB][Hkv][bs][D], or vLLM's K [NB][Hkv][D/8][bs][8] "
                         "with V [NB][Hkv][D][bs] (append and decode as two calls)")
    ap.add_argument("--varlen-tc", action="store_true",
                    help="spec / spec_long: run the tcgen05 varlen kernel "
                         "(pkv_set_varlen_tensor_path(1)) instead of the mma.sync one")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ncu-calls", type=int, default=0,
                    help="profiling mode: run this many plain calls of the step on a compact "
                         "pool, untimed, and exit")
    ap.add_argument("--oracle-child", choices=["baseline", "reference"], default=None,
                    help=argparse.SUPPRESS)
    ap.add_argument("--oracle-budget", type=float, default=12.0, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_child:
        oracle_child_main(args.oracle_child, args.workload, args.steps, args.warmup,
                          args.oracle_budget)
        return
    if args.ncu_calls:
        run_profile(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "ours" and args.workload == "loop":
        run_loop(args)
        return
    if args.impl == "ours" and args.workload == "step_qkv":
        run_step_qkv(args)
        return
    if args.impl == "ours" and args.workload == "qkv_prefill":
        run_qkv(args)
        return
    if args.impl == "ours" and args.workload in ("spec", "spec_long", "prefill", "prefill_one"):
        run_varlen(args)
        return
    if args.impl == "reference":
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[k] = "1"  # before numpy is first imported
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
