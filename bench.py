"""Benchmark of the MoE decode layer on one GB300 (replicas on N GPUs).

One step = one decode-layer call of the DeepSeek-V3-shaped layer (H=7168, 256
routed experts, top-8, I = I_s = 2048, FP8 E4M3 weights with fp32 128x128
block scales) at each of M = 1, 8 and 32 tokens, on distinct seeded inputs.
The weights (11.3 GB) are random-init and resident in HBM; L2 is flushed
before every layer call, outside the timed events: a 512 MB buffer is written
and then read back, so that the write-back of the flush's own dirty lines is
not charged to the layer.

Prints one JSON line: tokens/s over all layer calls (device time, CUDA
events), the per-M microseconds per layer and HBM GB/s, the roofline of the
expert kernel (algorithmic bytes / its measured duration vs the measured HBM
copy bandwidth), the end-to-end figure through the public API with host
buffers, the CPU oracle as a reported baseline (one core, and replicas on all
cores), clocks sampled during the timed region, and launch counts.  `extra`
times the other workloads the same way: the same layer at verify batch sizes
(M = 64, 128, 256), the layer with skewed routing and e8m0 scales (M = 1, 16,
128), the split-K eh_proj and the router GEMV alone at M = 1, 2, 4, 8, 16,
the MTP front, the LM head, the dense layer and a CUDA-graph decode chain,
with the oracle's time on one token of each workload beside them.

--impl reference times the CPU oracle alone, on the same workload (a bounded
sample per step), and prints the same kind of line with "impl": "reference".
"""

from __future__ import annotations

import os

# the oracle baseline is single-threaded: pin BLAS before numpy loads
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import ctypes
import hashlib
import json
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_decode_layer_bf16_gb300 import synth  # noqa: E402
from moe_decode_layer_bf16_gb300.dims import DSV3  # noqa: E402

MS = (1, 8, 32)
METRIC = "MoE decode layer tokens/s (DeepSeek-V3-shaped layer, M=1,8,32)"
UNIT = "tokens/s"
WORKLOAD = "deepseek-v3-shaped MoE decode layer, H=7168 E=256 k=8 I=Is=2048, M in {1,8,32}"
# bytes of one expert: fp8 w13 [2I,H] + w2 [H,I] + fp32 128x128 scales
EXPERT_BYTES = 2 * DSV3.inter * DSV3.hidden + DSV3.hidden * DSV3.inter + 4 * (
    (2 * DSV3.inter // 128) * (DSV3.hidden // 128) + (DSV3.hidden // 128) * (DSV3.inter // 128))
ROUTER_BYTES = DSV3.num_experts * DSV3.hidden * 2
# DRAM bytes (read + write) per activated expert of one launch of each expert
# kernel, from the ncu capture of profiles/experts_kernels_dsv3_e32_traffic.txt
# (the 32-expert profiling layer: experts_kernel at 1 and 8 tokens, 9 and 29
# experts active, the mean of the two per-expert figures; experts_tc_kernel at
# 32 tokens, 33 experts active), valid for the source whose
# code (comments and white space removed) has the SHA-256 given; the bench
# reports no traffic once a kernel's code differs from the captured one.
TRAFFIC_CAPTURE = {
    "experts.cu": {"code_sha256": "17d19129ee3d3d1e85b402138301d65921218ba69a2e5ad5d5b5c311cb89abff",
                   "bytes_per_expert": 44_148_562},
    "experts_tc.cu": {"code_sha256": "0513010fb4821d17177604fa276254241b5d02755c2e3798dc9f5a0fecd111fa",
                      "bytes_per_expert": 44_370_148},
}


def code_sha256(path):
    """SHA-256 of a CUDA source with its comments and white space removed."""
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return hashlib.sha256(re.sub(r"\s+", "", src).encode()).hexdigest()


def layer_bytes(M: int, unique: int) -> int:
    """Algorithmic HBM bytes of one layer call: the activated experts' and the
    shared expert's weights, the router weight, x/residual in, out/residual_out
    out (bf16), and the norm gain."""
    return (unique + 1) * EXPERT_BYTES + ROUTER_BYTES + 4 * M * DSV3.hidden * 2 + DSV3.hidden * 2


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """The SM clock and the clock-event (throttle) reasons of the GPU, sampled
    every 2 ms from a thread while the timed region runs (NVML through ctypes:
    a timed region of a few tens of milliseconds still gets tens of samples),
    or every 200 ms by nvidia-smi where NVML cannot be loaded.  Reads only."""

    PERIOD_S = 0.002
    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, local: int):
        self.samples, self.max_mhz, self.proc, self.thread = [], None, None, None
        self.stop_evt = threading.Event()
        try:
            self._start_nvml(local)
        except Exception:
            self.thread = None
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self._nvml_index(local)), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "200"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception:
                self.proc = None

    @staticmethod
    def _nvml_index(local: int) -> int:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
        if local < len(vis) and vis[local].strip().isdigit():
            return int(vis[local])
        return local

    def _start_nvml(self, local: int):
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit")
        h = ctypes.c_void_p()
        ok = False
        try:
            u = str(torch.cuda.get_device_properties(local).uuid)
            u = u if u.startswith("GPU-") else "GPU-" + u
            ok = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(self._nvml_index(local), ctypes.byref(h)) != 0:
            raise OSError("nvml handle")
        reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)

        def run():
            clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while not self.stop_evt.is_set():
                if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                        reasons_fn(h, ctypes.byref(rs)) == 0:
                    self.samples.append((float(clk.value), int(rs.value)))
                time.sleep(self.PERIOD_S)

        self.thread = threading.Thread(target=run, daemon=True)
        self.thread.start()

    def stop(self):
        if self.thread is not None:
            self.stop_evt.set()
            self.thread.join(timeout=5)
            if not self.samples:
                return None
            reasons = sorted({n for _, r in self.samples for b, n in self.REASONS.items() if r & b})
            return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                    "reasons": reasons, "samples": len(self.samples),
                    "source": f"nvml, {self.PERIOD_S * 1e3:g} ms"}
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [v.strip() for v in line.split(",")]
            if len(f) < 7:
                continue
            try:
                util = float(f[6])
                if util > 0:
                    sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[2:6]):
                if v.lower() == "active":
                    reasons.add(n)
        if not mx:
            return None
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(mx), "source": "nvidia-smi, 200 ms"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle

def _np(t):
    if t is None:
        return None
    t = t.detach().cpu()
    return t.float().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.numpy()


def oracle_layer_sample(seed: int = 0, skewed: bool = False):
    """The oracle's inputs for one token of the DeepSeek-V3-shaped layer: the
    token, the router (and, skewed, the selection bias and Zipf popularity
    with e8m0 scales), the shared expert, the gain and only the routed experts
    the token is routed to (drawn seeded per expert; on the GPU when there is
    one, which only draws random numbers).  Returns (dims, arrays dict)."""
    from oracle import moe_oracle as orc

    dims = DSV3.with_(e8m0=skewed)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    kw = dict(bias_std=0.5, zipf_s=1.1) if skewed else {}
    x, res = synth.make_tokens(1, dims.hidden, seed=seed, device=gen_dev, zipf=skewed)
    lw = synth.make_layer(dims, seed=seed, experts=[], device=gen_dev, **kw)
    a = {n: _np(lw[n]) for n in ("router_w", "sel_bias", "sw13", "sw13_s", "sw2", "sw2_s", "gain")}
    a["x"], a["res"] = _np(x), _np(res)
    _, _, _, ids, _ = orc.route(a["x"], a["router_w"], a["sel_bias"], dims.top_k, dims.routed_scaling)
    a["experts"] = np.asarray(sorted(set(ids.reshape(-1).tolist())), np.int64)
    for e in a["experts"]:
        for n, t in zip(("w13", "w13_s", "w2", "w2_s"), synth.make_expert(dims, int(e), seed=seed, device=gen_dev)):
            a[f"{n}_{e}"] = _np(t)
    return dims, a


def oracle_run(dims, a):
    """The oracle's M = 1 layer call on the arrays of oracle_layer_sample:
    seconds of the call alone."""
    from oracle import moe_oracle as orc

    ex = [int(e) for e in a["experts"]]
    L = orc.Layer(router_w=a["router_w"], sel_bias=a.get("sel_bias"),
                  w13={e: a[f"w13_{e}"] for e in ex}, w13_s={e: a[f"w13_s_{e}"] for e in ex},
                  w2={e: a[f"w2_{e}"] for e in ex}, w2_s={e: a[f"w2_s_{e}"] for e in ex},
                  sw13=a["sw13"], sw13_s=a["sw13_s"], sw2=a["sw2"], sw2_s=a["sw2_s"], gain=a["gain"],
                  top_k=dims.top_k, routed_scaling=dims.routed_scaling, swiglu_limit=dims.swiglu_limit,
                  rms_eps=dims.rms_eps, e8m0=dims.e8m0)
    t0 = time.perf_counter()
    orc.moe_decode_layer(L, a["x"], a["res"])
    return time.perf_counter() - t0


SAMPLE_DESC = "one M=1 layer call (router, 8 routed + shared expert dequantised and applied, boundary)"


def oracle_sample(seed: int = 0, skewed: bool = False):
    """One M=1 layer of the same shape on the CPU oracle.  Returns (seconds,
    description)."""
    dims, a = oracle_layer_sample(seed, skewed)
    return oracle_run(dims, a), SAMPLE_DESC


def _oracle_replica(path, barrier, out):
    # one process of the all-cores baseline: load the sample, wait for the
    # others, time the oracle call
    with np.load(path, allow_pickle=False) as z:
        a = {k: z[k] for k in z.files}
    barrier.wait()
    dt = oracle_run(DSV3, a)
    out.put(dt)


def oracle_all_cores(seed: int = 0):
    """The oracle as it stands, one replica per host core (spawned processes,
    each single-threaded), all on the same M = 1 sample, started together:
    tokens/s = replicas / the slowest replica's time."""
    import multiprocessing as mp

    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    dims, a = oracle_layer_sample(seed)
    with tempfile.TemporaryDirectory(dir="/dev/shm" if os.path.isdir("/dev/shm") else None) as d:
        path = os.path.join(d, "sample.npz")
        np.savez(path, **{k: v for k, v in a.items() if v is not None})
        ctx = mp.get_context("spawn")
        bar, q = ctx.Barrier(cores), ctx.Queue()
        procs = [ctx.Process(target=_oracle_replica, args=(path, bar, q)) for _ in range(cores)]
        for p in procs:
            p.start()
        dts = [q.get(timeout=600) for _ in range(cores)]
        for p in procs:
            p.join(timeout=60)
    return {"value": cores / max(dts), "unit": UNIT, "cores": cores, "kind": "oracle replicas",
            "sample": f"{cores} concurrent single-threaded replicas of the oracle, each on {SAMPLE_DESC}; "
                      f"slowest {max(dts):.2f} s, fastest {min(dts):.2f} s"}


def oracle_per_config(seed: int = 0):
    """The oracle on one token of each workload the bench times (one core)."""
    from oracle import moe_oracle as orc

    res = {}
    for name, skewed in (("deepseek_v3_uniform", False), ("deepseek_v3_skewed_e8m0", True)):
        dt, _ = oracle_sample(seed, skewed)
        res[name] = {"seconds": round(dt, 3), "tokens_per_s": round(1.0 / dt, 4), "sample": SAMPLE_DESC}
    for name, (N, K) in (("splitk_eh_proj", (7168, 14336)), ("router_gemv_fp32", (256, 7168))):
        a, w = synth.make_projection(1, N, K, seed=1,
                                     device="cuda" if torch.cuda.is_available() else "cpu")
        a, w = _np(a), _np(w)
        t0 = time.perf_counter()
        orc.projection(a, w, out_fp32=name.startswith("router"))
        dt = time.perf_counter() - t0
        res[name] = {"seconds": round(dt, 4), "tokens_per_s": round(1.0 / dt, 2),
                     "sample": f"M=1 projection [1,{K}] x [{N},{K}]^T"}
    return res


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        oracle_sample(seed=0)
    times = []
    for s in range(args.steps):
        dt, desc = oracle_sample(seed=s)
        times.append(dt)
    total = sum(times)
    value = args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "sample": "M=1 per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def timed(fn, flush_l2, reps, warm=1):
    """Device milliseconds of fn() per call (CUDA events on the current stream,
    L2 flushed before each call; the first `warm` calls untimed)."""
    times = []
    for i in range(warm + reps):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        if i >= warm:
            times.append(e0.elapsed_time(e1))
    return times


def splitk_proj(m, flush_l2, dev, N, K, Ms=(1, 2, 4, 8, 16), reps=20, fp32=False, peak=None):
    """The split-K BF16 projection Y[M, N] = A[M, K] W[N, K]^T, L2 flushed
    before every call: us and GB/s (weights + activations in + out)."""
    res = {}
    w = None
    for M in Ms:
        a, w_m = synth.make_projection(M, N, K, seed=M, device=dev)
        w = w_m if w is None else w
        c = torch.empty((M, N), dtype=torch.float32 if fp32 else torch.bfloat16, device=dev)
        ws = torch.zeros(m.splitk_gemm_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
        us = 1e3 * statistics.fmean(timed(lambda: m.splitk_gemm_bf16(a, w, c, ws), flush_l2, reps))
        nbytes = 2 * N * K + 2 * M * K + c.element_size() * M * N
        res[str(M)] = {"us": round(us, 2), "gbps": round(nbytes / us / 1e3, 1)}
        if peak:
            res[str(M)]["frac_of_measured"] = round(nbytes / us / 1e3 / peak, 3)
    del w
    torch.cuda.empty_cache()
    return res


def layer_block(m, dims, lw, Ms, flush_l2, dev, peak, reps=20, zipf=False, seed=500):
    """One layer's calls at each M (L2 flushed before every call): the plain
    call's us, tokens/s and GB/s of the layer's algorithmic bytes, and the
    expert kernel's us from a traced call (events between the kernels)."""
    lay = m.MoeDecodeLayer(dims, lw, max_tokens=max(Ms), device=dev)
    res = {}
    for M in Ms:
        x, r = synth.make_tokens(M, dims.hidden, seed=seed + M, device=dev, zipf=zipf)
        o, ro = torch.empty_like(x), torch.empty_like(r)
        ids = torch.empty((M, dims.top_k), dtype=torch.int32, device=dev)
        plain = timed(lambda: lay(x, r, o, ro, topk_ids=ids), flush_l2, reps)
        exp_ms = []
        for _ in range(reps):
            flush_l2()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            m.moe_decode_layer_traced(dims, lw, x, r, o, ro, lay.workspace, ev, topk_ids=ids)
            torch.cuda.synchronize()
            exp_ms.append(ev[1].elapsed_time(ev[2]))
        if lay.status() != m.MOE_OK:
            raise RuntimeError("layer status")
        unique = int(torch.unique(ids).numel())
        us, ue = 1e3 * statistics.fmean(plain), 1e3 * statistics.fmean(exp_ms)
        lb = layer_bytes(M, unique)
        res[str(M)] = {"us_per_layer": round(us, 2), "tokens_per_s": round(M * 1e6 / us, 1),
                       "unique_experts": unique, "layer_gbps": round(lb / us / 1e3, 1),
                       "frac_of_8TBs": round(lb / us / 1e3 / 8000.0, 3),
                       "frac_of_measured": round(lb / us / 1e3 / peak, 3),
                       "us_experts": round(ue, 2),
                       "experts_frac_of_measured": round((unique + 1) * EXPERT_BYTES / ue / 1e3 / peak, 3)}
    del lay
    torch.cuda.empty_cache()
    return res


def mtp_front(m, flush_l2, dev, Ms=(1, 4, 16), reps=20):
    """mtp_eh_front at DeepSeek-V3 sizes (H = 7168, vocabulary 129280,
    eh_proj [7168, 14336]), L2 flushed before every call."""
    H, V = 7168, 129280
    gen = torch.Generator(device=dev).manual_seed(1)
    embed = torch.randn(V, H, generator=gen, device=dev).to(torch.bfloat16)
    gains = (1 + 0.1 * torch.randn(2, H, generator=gen, device=dev)).to(torch.bfloat16)
    _, w = synth.make_projection(1, H, 2 * H, seed=3, device=dev)
    res = {}
    for M in Ms:
        ids = torch.randint(0, V, (M,), generator=gen, device=dev, dtype=torch.int32)
        hidden = torch.randn(M, H, generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty((M, H), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(m.mtp_eh_front_workspace_size(M, H), dtype=torch.uint8, device=dev)
        m.moe_workspace_init(ws)
        times = []
        for r in range(reps + 1):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            m.mtp_eh_front(ids, embed, hidden, gains[0], gains[1], 1e-6, w, out, ws)
            e1.record()
            torch.cuda.synchronize()
            if r:
                times.append(e0.elapsed_time(e1))
        if m.moe_device_status(ws) != m.MOE_OK:
            raise RuntimeError("mtp_eh_front status")
        us = 1e3 * statistics.fmean(times)
        nbytes = 2 * H * 2 * H + M * (2 * H * 3 + 2 * H * 2 * 2 + 4)  # weights; e, h in, A out + in, out
        res[str(M)] = {"us": round(us, 2), "gbps": round(nbytes / us / 1e3, 1)}
    del embed, w
    torch.cuda.empty_cache()
    return res


def dense_layer(m, flush_l2, dev, MS, reps=20):
    """A DeepSeek-V3 dense layer (num_experts = 0: the 18432-wide FP8 MLP in the
    shared-expert slot, no router) with its boundary, L2 flushed before every call."""
    from moe_decode_layer_bf16_gb300.dims import DSV3_DENSE as D
    lw = synth.make_layer(D, seed=21, device=dev)
    wbytes = sum(lw[n].numel() * lw[n].element_size() for n in ("sw13", "sw13_s", "sw2", "sw2_s"))
    res = {}
    for M in MS:
        lay = m.MoeDecodeLayer(D, lw, max_tokens=M, device=dev)
        x, r = synth.make_tokens(M, D.hidden, seed=400 + M, device=dev)
        o, ro = torch.empty_like(x), torch.empty_like(r)
        times = []
        for i in range(reps + 1):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            lay(x, r, o, ro)
            e1.record()
            torch.cuda.synchronize()
            if i:
                times.append(e0.elapsed_time(e1))
        if lay.status() != m.MOE_OK:
            raise RuntimeError("dense layer status")
        us = 1e3 * statistics.fmean(times)
        nbytes = wbytes + 4 * M * D.hidden * 2 + D.hidden * 2
        res[str(M)] = {"us_per_layer": round(us, 2), "tokens_per_s": round(M * 1e6 / us, 1),
                       "gbps": round(nbytes / us / 1e3, 1)}
    del lw
    torch.cuda.empty_cache()
    return res


def tp_rank_partial(m, dims, lw, Ms, flush_l2, dev, peak, Gs=(2, 4, 8), reps=20):
    """One rank's share of the layer under G-way tensor parallelism over each
    expert's intermediate dimension (rank 0's shard through
    moe_decode_layer_partial), and the boundary over G shares.  The all-reduce
    between GPUs is not part of it (one GPU)."""
    from moe_decode_layer_bf16_gb300 import tp
    res = {}
    for G in Gs:
        sd = tp.shard_dims(dims, G)
        shard = tp.shard_weights(dims, lw, 0, G)
        ws = torch.empty(m.moe_decode_workspace_size(sd, max(Ms)), dtype=torch.uint8, device=dev)
        m.moe_workspace_init(ws)
        per = {}
        for M in Ms:
            x, r = synth.make_tokens(M, dims.hidden, seed=700 + M, device=dev)
            mo = torch.empty((M, dims.hidden), dtype=torch.float32, device=dev)
            ids = torch.empty((M, dims.top_k), dtype=torch.int32, device=dev)
            us = 1e3 * statistics.fmean(
                timed(lambda: m.moe_decode_layer_partial(sd, shard, x, mo, ws, topk_ids=ids), flush_l2, reps))
            if m.moe_device_status(ws) != m.MOE_OK:
                raise RuntimeError("tp partial status")
            unique = int(torch.unique(ids).numel())
            nbytes = (unique + 1) * EXPERT_BYTES / G + ROUTER_BYTES + M * dims.hidden * (2 + 4)
            parts = torch.zeros((G, M, dims.hidden), dtype=torch.float32, device=dev)
            o, ro = torch.empty_like(x), torch.empty_like(r)
            ub = 1e3 * statistics.fmean(
                timed(lambda: m.moe_tp_boundary(parts, r, lw["gain"], o, ro, dims.rms_eps), flush_l2, reps))
            per[str(M)] = {"us_rank": round(us, 2), "rank_gbps": round(nbytes / us / 1e3, 1),
                           "rank_frac_of_measured": round(nbytes / us / 1e3 / peak, 3),
                           "us_boundary_over_G_shares": round(ub, 2)}
        res[f"G={G}"] = per
        del shard, ws
        torch.cuda.empty_cache()
    return res


def graph_chain(m, dims, lw0, MS, n_layers, reps, dev):
    """A decode chain captured as one CUDA graph: n_layers layers with distinct
    weights, each layer's out / residual_out feeding the next layer's x /
    residual, replayed back to back with no L2 flush (each layer's 11 GB of
    weights evicts the others').  Returns per M: us per layer, tokens/s, GB/s."""
    layers = [lw0] + [synth.make_layer(dims, seed=10 + i, device=dev) for i in range(n_layers - 1)]
    res = {}
    for M in MS:
        lay = m.MoeDecodeLayer(dims, lw0, max_tokens=M, device=dev)
        x0, r0 = synth.make_tokens(M, dims.hidden, seed=300 + M, device=dev)
        bufs = [(torch.empty_like(x0), torch.empty_like(r0)) for _ in range(n_layers)]
        ids = [torch.empty((M, dims.top_k), dtype=torch.int32, device=dev) for _ in range(n_layers)]

        def run():
            x, r = x0, r0
            for i, lw in enumerate(layers):
                o, ro = bufs[i]
                m.moe_decode_layer(dims, lw, x, r, o, ro, lay.workspace, topk_ids=ids[i])
                x, r = o, ro

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            run()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        if lay.status() != m.MOE_OK:
            raise RuntimeError("device status after graph replay")
        us = 1e3 * e0.elapsed_time(e1) / (reps * n_layers)
        nbytes = sum(layer_bytes(M, int(torch.unique(t).numel())) for t in ids) / n_layers
        res[str(M)] = {"us_per_layer": round(us, 2), "tokens_per_s": round(M * 1e6 / us, 1),
                       "layer_gbps": round(nbytes / us / 1e3, 1)}
        del g
    del layers[1:]
    torch.cuda.empty_cache()
    return res


def run_ours(args, world, rank, local):
    import moe_decode_layer_bf16_gb300 as m

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dims = DSV3.with_(num_experts=args.num_experts)
    MS = tuple(args.ms)
    if args.dense:
        # profiling aid: the dense layer alone (as in the `extra` measurement)
        fl = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

        def flush_dense():
            fl.zero_()
            fl.view(torch.int64).max()

        res = dense_layer(m, flush_dense, dev, MS, reps=max(1, args.steps))
        if rank == 0:
            print(json.dumps({"metric": "dense FP8 MLP layer (DeepSeek-V3 7168 x 18432) with its boundary, us",
                              "unit": "us", "steps": max(1, args.steps), "per_m": res}), flush=True)
        return 0
    lw = synth.make_layer(dims, seed=0, device=dev)
    layer = m.MoeDecodeLayer(dims, lw, max_tokens=max(MS), device=dev)
    inputs = {M: synth.make_tokens(M, dims.hidden, seed=100 + M, device=dev) for M in MS}
    outs = {M: (torch.empty_like(inputs[M][0]), torch.empty_like(inputs[M][1])) for M in MS}
    ids = {M: torch.empty((M, dims.top_k), dtype=torch.int32, device=dev) for M in MS}
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def flush_l2():
        # evict L2 (129 MB) by writing a 512 MB buffer, then read the buffer back
        # so that the flush's own dirty lines reach HBM before the timed region
        # rather than being written back while the layer streams its weights
        flush.zero_()
        flush.view(torch.int64).max()

    def call(M, events=None):
        x, res = inputs[M]
        out, ro = outs[M]
        if events is None:
            m.moe_decode_layer(dims, lw, x, res, out, ro, layer.workspace, topk_ids=ids[M])
        else:
            m.moe_decode_layer_traced(dims, lw, x, res, out, ro, layer.workspace, events, topk_ids=ids[M])

    # warm-up
    for _ in range(args.warmup):
        for M in MS:
            flush_l2()
            call(M)
    torch.cuda.synchronize()
    st = layer.status()
    if st != m.MOE_OK:
        raise RuntimeError(f"device status {st}")
    unique = {M: int(torch.unique(ids[M]).numel()) for M in MS}

    # timed region: each layer call bracketed by CUDA events (plain calls, so the
    # three kernels overlap their launches as in production)
    ev = {(s, M): [torch.cuda.Event(enable_timing=True) for _ in range(2)] for s in range(args.steps) for M in MS}
    clocks = Clocks(local)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        for M in MS:
            flush_l2()
            ev[(s, M)][0].record()
            call(M)
            ev[(s, M)][1].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    clk = clocks.stop()

    # per-kernel durations (router, experts, boundary) from traced calls: the
    # library records events between its three kernels on the launch stream
    tev = {(s, M): [torch.cuda.Event(enable_timing=True) for _ in range(4)] for s in range(args.steps) for M in MS}
    for s in range(args.steps):
        for M in MS:
            flush_l2()
            call(M, tev[(s, M)])
    torch.cuda.synchronize()

    per_m = {}
    total_ms = 0.0
    exp_ms_all, exp_bytes_all = 0.0, 0
    for M in MS:
        layer_ms = [ev[(s, M)][0].elapsed_time(ev[(s, M)][1]) for s in range(args.steps)]
        exp_ms = [tev[(s, M)][1].elapsed_time(tev[(s, M)][2]) for s in range(args.steps)]
        rt_ms = [tev[(s, M)][0].elapsed_time(tev[(s, M)][1]) for s in range(args.steps)]
        nm_ms = [tev[(s, M)][2].elapsed_time(tev[(s, M)][3]) for s in range(args.steps)]
        total_ms += sum(layer_ms)
        exp_ms_all += sum(exp_ms)
        eb = (unique[M] + 1) * EXPERT_BYTES
        exp_bytes_all += eb * args.steps
        lb = layer_bytes(M, unique[M])
        # (CUDA event stamps here tick in steps of about 2 us: a median is a
        # multiple of that, the mean resolves finer differences)
        us = 1e3 * statistics.fmean(layer_ms)
        per_m[str(M)] = {"us_per_layer": round(us, 2), "us_median": round(1e3 * statistics.median(layer_ms), 2),
                         "tokens_per_s": round(M * 1e6 / us, 1),
                         "unique_experts": unique[M], "layer_bytes": lb,
                         "layer_gbps": round(lb / us / 1e3, 1),
                         "us_router": round(1e3 * statistics.fmean(rt_ms), 2),
                         "us_experts": round(1e3 * statistics.fmean(exp_ms), 2),
                         "us_boundary": round(1e3 * statistics.fmean(nm_ms), 2)}
    # replicas: every rank runs the same steps; the job's time is the slowest rank's
    total_ms = max_over_ranks(total_ms, world)
    value = sum(MS) * args.steps * world / (total_ms / 1e3)

    peak, peak_kind = load_peaks()
    achieved = exp_bytes_all / (exp_ms_all / 1e3) / 1e9
    # which expert kernel each M runs (the library's choice)
    kern = {M: "experts_tc.cu" if m.moe_decode_layer_plan(dims, M)[0] == m.MOE_PATH_TCGEN05 else "experts.cu"
            for M in MS}
    traffic = None
    csrc = os.path.join(ROOT, "moe_decode_layer_bf16_gb300", "csrc")
    if all(code_sha256(os.path.join(csrc, f)) == c["code_sha256"] for f, c in TRAFFIC_CAPTURE.items()):
        # per launch, averaged over the launches like `achieved`
        traffic = round(sum(TRAFFIC_CAPTURE[kern[M]]["bytes_per_expert"] * (unique[M] + 1) for M in MS) / len(MS))
    for M in MS:
        per_m[str(M)]["frac_of_8TBs"] = round(per_m[str(M)]["layer_gbps"] / 8000.0, 3)
        per_m[str(M)]["frac_of_measured"] = round(per_m[str(M)]["layer_gbps"] / peak, 3)

    # end to end through the public API with host buffers
    h_in = {M: [t.cpu().pin_memory() for t in inputs[M]] for M in MS}
    h_out = {M: [torch.empty_like(t, device="cpu").pin_memory() for t in inputs[M]] for M in MS}
    d_in = {M: [torch.empty_like(t) for t in inputs[M]] for M in MS}
    e2e_ms = 0.0
    for rep in range(-1, args.steps):
        for M in MS:
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for d, h in zip(d_in[M], h_in[M]):
                d.copy_(h, non_blocking=True)
            out, ro = layer(d_in[M][0], d_in[M][1], out=outs[M][0], residual_out=outs[M][1])
            h_out[M][0].copy_(out, non_blocking=True)
            h_out[M][1].copy_(ro, non_blocking=True)
            e1.record()
            e1.synchronize()
            if rep >= 0:
                e2e_ms += e0.elapsed_time(e1)
    e2e_value = sum(MS) * args.steps / (e2e_ms / 1e3)
    io_bytes = sum(2 * M * dims.hidden * 2 for M in MS)

    extra = {}
    if not args.no_extras:
        def attempt(key, what, fn):
            # reported, not fatal: the headline does not depend on the extras
            if args.extras and key not in args.extras:
                return
            try:
                extra[key] = {"what": what, "per_m": fn()}
            except Exception as exc:
                extra[key] = {"what": what, "error": f"{type(exc).__name__}: {exc}"}

        attempt("verify_batches", "the same layer at verify / grouped batch sizes M = 64, 128, 256 (i.i.d. router "
                "logits: nearly every expert active), L2 flushed, mean of 20 (event stamps tick in about 2 us steps); us_experts from a traced call",
                lambda: layer_block(m, dims, lw, (64, 128, 256), flush_l2, dev, peak))
        if dims.num_experts == DSV3.num_experts:
            def skewed():
                d4 = DSV3.with_(e8m0=True)
                lw4 = synth.make_layer(d4, seed=4, device=dev, bias_std=0.5, zipf_s=1.1)
                try:
                    return layer_block(m, d4, lw4, (1, 16, 128), flush_l2, dev, peak, zipf=True, seed=600)
                finally:
                    del lw4
                    torch.cuda.empty_cache()

            attempt("skewed_e8m0", "the DeepSeek-V3-shaped layer with power-of-two (e8m0) scales, a selection bias "
                    "~N(0,0.5) and Zipf(1.1) expert popularity, M = 1, 16, 128, L2 flushed, mean of 20 (event stamps tick in about 2 us steps)",
                    skewed)
        attempt("splitk_eh_proj", "splitk_gemm_bf16 (split_k = 0: stream-K), MTP eh_proj N=7168 K=14336 "
                "(205.5 MB), L2 flushed, mean of 20 (event stamps tick in about 2 us steps)",
                lambda: splitk_proj(m, flush_l2, dev, 7168, 14336, peak=peak))
        attempt("router_gemv", "the router GEMV alone as the split-K projection's fp32 form, "
                "[M,7168] x [256,7168]^T -> fp32 logits (3.67 MB: launch-bound, its fraction of the HBM "
                "roofline is not meaningful), L2 flushed, mean of 20 (event stamps tick in about 2 us steps)",
                lambda: splitk_proj(m, flush_l2, dev, 256, 7168, fp32=True))
        if dims.num_experts == DSV3.num_experts:
            attempt("tp_rank_partial", "G-way tensor parallelism over each expert's intermediate dimension: one "
                    "rank's share of the layer (moe_decode_layer_partial on rank 0's shard, 1/G of every expert's "
                    "bytes) and the boundary over G shares (moe_tp_boundary); the all-reduce between GPUs is not "
                    "measured (one GPU), L2 flushed, mean of 20 (event stamps tick in about 2 us steps)",
                    lambda: tp_rank_partial(m, dims, lw, MS, flush_l2, dev, peak))
        attempt("graph_chain", "3 layers with distinct weights captured as one CUDA graph, each layer's outputs "
                "feeding the next, replayed back to back without L2 flushes",
                lambda: graph_chain(m, dims, lw, MS, 3, 10, dev))
        attempt("dense_layer", "DeepSeek-V3 dense layer (FP8 MLP 7168 x 18432, 396 MB) with its boundary, "
                "L2 flushed, mean of 20 (event stamps tick in about 2 us steps)", lambda: dense_layer(m, flush_l2, dev, MS))
        attempt("mtp_eh_front", "mtp_eh_front, H=7168, vocab 129280, eh_proj [7168, 14336] (205.5 MB), "
                "L2 flushed, mean of 20 (event stamps tick in about 2 us steps)", lambda: mtp_front(m, flush_l2, dev))
        attempt("splitk_lm_head", "splitk_gemm_bf16, LM head N=129280 K=7168 (1.85 GB), L2 flushed, mean of 20 (event stamps tick in about 2 us steps)",
                lambda: splitk_proj(m, flush_l2, dev, 129280, 7168, Ms=(1, 8), peak=peak))

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, desc = oracle_sample(seed=0)
        cpu = {"value": 1.0 / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc}
        try:
            cpu["all_cores"] = oracle_all_cores(seed=0)
        except Exception as exc:
            cpu["all_cores"] = {"error": f"{type(exc).__name__}: {exc}"}
        if not args.no_extras and (not args.extras or "oracle_per_config" in args.extras):
            try:
                extra["oracle_per_config"] = {"what": "the oracle (one core) on one token of each workload",
                                              "per_config": oracle_per_config(seed=0)}
            except Exception as exc:
                extra["oracle_per_config"] = {"error": f"{type(exc).__name__}: {exc}"}

    workload = WORKLOAD if (dims.num_experts == DSV3.num_experts and MS == (1, 8, 32)) else (
        f"profiling case: H=7168 E={dims.num_experts} k=8 I=Is=2048, M in {set(MS)}")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8",
        "data": "synthetic (seeded random-init weights and tokens)",
        "config": {"workload": workload, "tokens_per_step": sum(MS), "l2": "flushed before every layer call: 512 MB written, then read back (no dirty flush lines left)",
                   "weights": "fp8-e4m3 with fp32 128x128 block scales; router bf16; activations bf16 in/out",
                   "parallelism": "replicas" if world > 1 else "single GPU", "per_m": per_m,
                   "wall_s_timed": round(wall, 4)},
        "roofline": {"bound": "hbm",
                     "kernel": "expert kernels: " + ", ".join(
                         f"{'experts_tc_kernel' if kern[M] == 'experts_tc.cu' else 'experts_kernel'} at M={M}"
                         for M in MS),
                     "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": f"{peak_kind} HBM copy bandwidth", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": round(exp_bytes_all / (len(MS) * args.steps))},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": io_bytes, "d2h_bytes_per_step": io_bytes},
        "gpu_launches": sum(m.moe_decode_layer_plan(dims, M)[1] for M in MS) * args.steps,
        "timing": "value: events around each plain layer call; per-kernel us and roofline: a second, traced pass",
        "clocks": clk,
        "cpu_baseline": cpu,
        "extra": extra,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads (verify batches, skewed routing, split-K, router, graph chain, "
                         "dense layer, MTP front, LM head)")
    ap.add_argument("--extras", nargs="+", default=None,
                    help="run only these of the other workloads (by their keys in the JSON line's extra)")
    # profiling aids (smaller resident layer for multi-pass ncu captures)
    ap.add_argument("--num-experts", type=int, default=DSV3.num_experts)
    ap.add_argument("--ms", type=int, nargs="+", default=list(MS))
    ap.add_argument("--dense", action="store_true", help="time only the dense layer at --ms (one untimed call first)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
