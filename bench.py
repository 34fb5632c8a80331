#!/usr/bin/env python3
"""Benchmark of the BitNet b1.58 BitLinear forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama70b|...] [--impl ours|reference]

One step is one pass of the per-token hot path over every layer of the
workload: per-token int8 activation quantisation, then the ternary x int8
product with the fused gamma/s rescale, through the C ABI of libbitlinear.so.
Weights are packed once beforehand (the pages' "inference-ready pack"); the
packing kernels are timed in the same run and reported under "pack".

The default workload is the 70B-class layer pair at M = 1, 16 and 176 tokens
(the largest configuration that fits one GPU), so one line covers both halves
of the metric: the few-token layers are rated in GB/s against HBM, the
176-token layers in TOPS against the tensor pipe ("roofline.per_layer").

Timing: W warm-up steps, then the K steps, captured as one CUDA graph of the
public C-ABI calls, are replayed R times; each replay is bracketed by a
barrier and cuda.synchronize() on both sides and timed with CUDA events on the
launching stream, and ms_per_step is the median replay time / K (max over
ranks).  L2 (126 MB) is defeated by rotating every layer over copies of its
packed weights and activations whose total is more than twice L2.  After the
timed region the last step is re-run eagerly and its outputs must match bit
for bit ("verified").  The same K steps launched one call at a time (no
graph) give the "per_launch" figure.  Rank 0 prints one JSON line.

Under torchrun (N > 1) every rank runs its own replica of the workload (weak
scaling; the path has no data-path exchange) and value is the sum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
DEFAULT_WORKLOAD = "llama70b"
DEFAULT_STEPS = {"decode": 2000, "tiny": 2000, "skinny": 500, "prefill": 100, "llama70b": 50}
GRAPH_CHUNK = 500  # steps per captured graph
MIN_TIMED_S = 1.0  # replays of the K-step graph are repeated until about this long
MAX_REPLAYS = 200


# ---------------------------------------------------------------- helpers

# Rates of the legacy warp-level MMA on this GPU, measured with a register-only
# mma.sync loop over all SMs (m16n8k32 s8, m16n8k16 f16 with fp32 accumulate):
# the recompiled-kernel baseline a tcgen05 kernel is meant to beat.
LEGACY_MMA_SYNC = {"s8_tops": 139.5, "f16_tflops": 446.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_digest(files):
    h = hashlib.sha256()
    for rel in files:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, shape: str):
    """DRAM bytes per launch from the committed ncu summary, or None if absent
    or if the kernel's source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    for e in table.get("entries", []):
        if e.get("kernel") == kernel and e.get("shape") == shape:
            if e.get("source_digest") != kernel_source_digest(e.get("source_files", [])):
                return None
            return e.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                        rows.append(parts)
        except OSError:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        mx = [float(r[2]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if torch.cuda.is_available():
        torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend="nccl" if torch.cuda.is_available() else "gloo")
        return dist, rank, world, local
    return None, rank, world, local


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, value: float) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- accounting

def x_bytes(L) -> int:
    return 2 if L.x_dtype == "bf16" else 4


def tq5_row_bytes(K: int) -> int:
    """Bytes per row of the base-3 weight format (the library's rule, restated
    for the byte accounting): ceil(K/5) rounded up to 16."""
    return ((K + 4) // 5 + 15) // 16 * 16


def weight_bytes(L, fmt: str = "2bit") -> int:
    return L.N * tq5_row_bytes(L.K) if fmt == "tq5" else L.N * L.K // 4


def layer_bytes(L, fmt: str = "2bit") -> int:
    """Algorithmic HBM bytes of one layer step: read X, read the packed
    weights, write y (the per-token scales and gamma are counted too)."""
    return L.M * L.K * x_bytes(L) + weight_bytes(L, fmt) + 4 * L.M * L.N + 4 * L.M + 4


def forward_kernel_bytes(L, fused: bool, fmt: str = "2bit") -> int:
    """Algorithmic bytes of the timed forward kernel: packed W and y, plus
    x_q and s read (two-call path) or X read and x_q, s written (fused)."""
    act = L.M * L.K * (x_bytes(L) + 1) if fused else L.M * L.K
    return weight_bytes(L, fmt) + act + 4 * L.M + 4 * L.M * L.N + 4


def layer_ops(L) -> int:
    return 2 * L.M * L.N * L.K


def metric_for(wl) -> tuple[str, str]:
    if max(L.M for L in wl.layers) <= 4:
        return "BitLinear GEMV GB/s (HBM roofline)", "GB/s"
    if min(L.M for L in wl.layers) <= 4:
        return ("BitLinear GEMV GB/s & GEMM int8 TOPS: step TOPS (2MNK over all layers); per-layer GB/s or TOPS "
                "against the roofline each layer's intensity implies"), "TOPS"
    return "BitLinear GEMM int8 TOPS (tensor roofline)", "TOPS"


def layer_bound(ops: float, nbytes: float, peaks) -> str:
    """'hbm' where the layer's intensity (ops per algorithmic byte) lies below
    the ridge of the measured peaks, else 'tensor'."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return "hbm" if ops / nbytes < ridge else "tensor"


def layer_roofline(L, us: float, fused: bool, fmt: str, peaks, peak_src: str) -> dict:
    """One layer's forward kernel against the bound its intensity implies."""
    nbytes = forward_kernel_bytes(L, fused and gemv_fused_layer(L), fmt)
    ops = layer_ops(L)
    bound = layer_bound(ops, nbytes, peaks)
    if bound == "hbm":
        achieved, peak, unit = nbytes / (us * 1e-6) / 1e9, peaks["hbm_gbs"], "GB/s"
        src = f"{peak_src} hbm_gbs (copy)"
    else:
        achieved, peak, unit = ops / (us * 1e-6) / 1e12, peaks["bf16_tflops"], "TFLOP/s"
        src = f"{peak_src} bf16_tflops burst (kind::f16 runs at the bf16 rate)"
    return {"layer": f"M={L.M} K={L.K} N={L.N}", "bound": bound, "achieved": round(achieved, 1),
            "peak": peak, "unit": unit, "frac": round(achieved / peak, 4), "us": round(us, 3),
            "algorithmic_bytes": nbytes, "algorithmic_ops": ops, "intensity_op_per_byte": round(ops / nbytes, 2),
            "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1), "TOPS": round(ops / (us * 1e-6) / 1e12, 2),
            "peak_source": src}


def common_config(args, wl) -> dict:
    """The workload description shared by both arms' JSON lines."""
    return {"workload": args.workload,
            "layers": [f"M={L.M} K={L.K} N={L.N} X={L.x_dtype}" for L in wl.layers],
            "weights": ("base-3, five per byte (1.6 bits per weight)" if args.format == "tq5"
                        else "2-bit, four per byte"),
            "path": ("bitlinear_quant_act + bitlinear_forward_tq5" if args.format == "tq5" else
                     ("bitlinear_quant_forward_ws (one fused quantise+GEMV kernel for M <= 4; quantisation "
                      "writing the fp16 operand, then the tcgen05 GEMM otherwise)") if args.path == "fused"
                     else "bitlinear_quant_act + bitlinear_forward_lut (table-lookup GEMV)" if args.path == "lut"
                     else "bitlinear_quant_act + bitlinear_forward_ws"),
            "l2": "every layer rotates over copies of its packed weights and activations totalling more than "
                  "2x L2 (126 MiB); no L2 flush",
            "launch": "K steps captured as one CUDA graph of the C-ABI calls, replayed R times (median)",
            "parallelism": f"replicas x{args.gpus}"}


# ---------------------------------------------------------------- CPU oracle (baseline and reference arm)

_ORACLE_PACKED: dict = {}  # oracle-packed weights by (workload, weight seed, format)


def run_oracle(wl, budget_s: float, steps: int | None = None, warmup: int = 0, fmt: str = "2bit",
               omp: bool = False):
    """Time the oracle on a bounded sample of the per-token step: a fraction f
    of each layer's output rows (all tokens).  Returns (value, f, s/step,
    steps, threads)."""
    import oracle

    layers = []
    for i, L in enumerate(wl.layers):
        key = (wl.name, workloads.weight_seed(wl, i), fmt)
        if key not in _ORACLE_PACKED:
            W = workloads.layer_weights(wl, i).numpy()
            _ORACLE_PACKED[key] = oracle.pack_weights_tq5(W) if fmt == "tq5" else oracle.pack_weights(W)
        p, g = _ORACLE_PACKED[key]
        layers.append((L, p, g, workloads.x_as_f32_numpy(workloads.layer_activations(wl, i))))
    _, unit = metric_for(wl)

    def one(frac):
        work = 0.0
        for (L, p, g, X) in layers:
            rows = max(1, int(round(L.N * frac)))
            xq, s = oracle.quant_act(X, omp=omp)
            if fmt == "tq5":
                oracle.forward_tq5(p[:rows], g, xq, s, L.K)
            else:
                oracle.forward(p[:rows], g, xq, s, L.K, omp=omp)
            wrow = tq5_row_bytes(L.K) if fmt == "tq5" else L.K / 4
            work += (L.M * L.K * x_bytes(L) + rows * wrow + 4 * L.M * rows) if unit == "GB/s" \
                else 2.0 * L.M * rows * L.K
        return work

    t0 = time.perf_counter()
    one(0.02)
    t_small = time.perf_counter() - t0
    frac = 0.02
    if steps:
        n_total = steps
        frac = max(1.0 / max(L.N for L in wl.layers), min(1.0, budget_s / (steps * t_small / 0.02)))
    else:
        frac = min(1.0, max(0.02, 0.02 * budget_s / (20 * max(t_small, 1e-4))))
        t0 = time.perf_counter()
        one(frac)
        t_one = time.perf_counter() - t0
        n_total = max(1, int(budget_s / max(t_one, 1e-4)))
    for _ in range(warmup):
        one(frac)
    t0 = time.perf_counter()
    work = 0.0
    for _ in range(n_total):
        work += one(frac)
    dt = time.perf_counter() - t0
    return (work / dt / (1e9 if unit == "GB/s" else 1e12), frac, dt / n_total, n_total,
            oracle.num_threads(omp) if omp else 1)


def cpu_baseline(wl, fmt: str, budget_s: float) -> dict:
    """The oracle on the host: single-threaded, and its OpenMP build on every
    host thread (the same code; identical results)."""
    _, unit = metric_for(wl)
    v1, f1, s1, n1, _ = run_oracle(wl, budget_s=budget_s / 2, fmt=fmt)
    out = {"unit": unit, "kind": "oracle", "nproc": os.cpu_count()}
    single = {"value": round(v1, 4), "cores": 1,
              "sample": f"{n1} oracle steps on {f1:.2%} of each layer's output rows (all tokens), {n1 * s1:.1f} s"}
    if fmt == "tq5":  # the base-3 decode has no threaded loops
        out.update(single)
        return out
    vN, fN, sN, nN, thr = run_oracle(wl, budget_s=budget_s / 2, fmt=fmt, omp=True)
    out.update({"value": round(vN, 4), "cores": thr,
                "sample": f"{nN} oracle steps on {fN:.2%} of each layer's output rows (all tokens), "
                          f"OpenMP build on {thr} threads, {nN * sN:.1f} s",
                "single_thread": single})
    return out


# ---------------------------------------------------------------- GPU arm

def gemm_variant(L, num_sms: int) -> str:
    """Which forward kernel the library picks for a layer (the library's own
    rule, restated here only to label the bench line)."""
    if L.M <= 4 and L.K <= 32768:
        return "gemv_kernel"
    if L.M <= 64:
        return "gemm_f8_kernel"
    ntiles_m = -(-L.M // 256)
    bn = -(-(-(-L.M // ntiles_m)) // 16) * 16
    tiles = -(-L.N // 128) * ntiles_m
    if tiles >= 2 * num_sms and bn >= 128:
        return "gemm_tc_x16_persistent_kernel"
    return "gemm_f16_sk_kernel"


def gemv_fused_layer(L) -> bool:
    """True where bitlinear_quant_forward runs the layer as ONE kernel (the
    fused quantise + GEMV: at most 4 tokens and K <= 32768)."""
    return L.M <= 4 and L.K <= 32768


def graph_kernel_nodes(g) -> int | None:
    """Kernel nodes of a captured CUDA graph (the launches one replay makes),
    or None where the graph cannot be inspected."""
    try:
        import cuda.bindings.runtime as rt

        graph = rt.cudaGraph_t(init_value=g.raw_cuda_graph())
        err, _, n = rt.cudaGraphGetNodes(graph, numNodes=0)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        err, nodes, n = rt.cudaGraphGetNodes(graph, numNodes=n)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        count = 0
        for node in nodes[:n]:
            err, typ = rt.cudaGraphNodeGetType(node)
            if err != rt.cudaError_t.cudaSuccess:
                return None
            count += int(typ == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel)
        return count
    except Exception:  # noqa: BLE001 -- an inspection aid only
        return None


def timed_replays(graphs, K, stream, dist, sampler=None):
    """Replays the K-step graph(s) R times, each replay bracketed by a barrier
    and synchronize; returns (median ms per step over ranks, R, per-replay ms)."""
    def once():
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        a.record(stream)
        for g in graphs:
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        return a.elapsed_time(b)

    first = once()
    R = int(min(MAX_REPLAYS, max(5, math.ceil(MIN_TIMED_S * 1e3 / max(first, 1e-3)))))
    R = int(max_over_ranks(dist, R))  # every rank replays the same number of times
    times = [once() for _ in range(R)]
    med = statistics.median(times)
    return max_over_ranks(dist, med) / K, R, times


def run_gpu(args, dist, rank, world, local):
    import ternary_weight_06_b300 as bl

    wl = workloads.WORKLOADS[args.workload]
    metric, unit = metric_for(wl)
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    stream = torch.cuda.Stream(device=dev)  # graphs cannot be captured on the legacy default stream
    torch.cuda.set_stream(stream)
    tq5 = args.format == "tq5"
    fused = args.path == "fused" and not tq5  # the base-3 forward takes quantised activations
    nlayers = len(wl.layers)
    peaks, peak_src = load_peaks()

    # ---- resident inputs: pack each distinct weight matrix once (timed as the "pack" figure)
    packed, gammas, Xs, Xs_host, ys, xqs, ss = [], [], [], [], [], [], []
    pack_ms, pack_bytes = 0.0, 0
    by_seed = {}
    for i, L in enumerate(wl.layers):
        seed = workloads.weight_seed(wl, i)
        if seed not in by_seed:
            W = workloads.layer_weights(wl, i).to(dev)
            pack_fn = bl.bitlinear_pack_weights_tq5 if tq5 else bl.bitlinear_pack_weights
            pack_fn(W)  # warm
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            Wp, g = pack_fn(W)
            e1.record(stream)
            torch.cuda.synchronize()
            pack_ms += e0.elapsed_time(e1)
            pack_bytes += 2 * 4 * L.N * L.K + weight_bytes(L, args.format)
            del W
            by_seed[seed] = (Wp, g)
        Wp, g = by_seed[seed]
        packed.append(Wp)
        gammas.append(g)
        X = workloads.layer_activations(wl, i)
        Xs_host.append(X.pin_memory())
        Xs.append(X.to(dev))
        ys.append(None)  # views into one output buffer, below
        xqs.append(torch.empty((L.M, L.K), dtype=torch.int8, device=dev))
        ss.append(torch.empty((L.M,), dtype=torch.float32, device=dev))
    # every layer's y is a 256-byte aligned slice of one device buffer, so the
    # end-to-end run reads all outputs back with one copy
    y_offs, y_total = [], 0
    for L in wl.layers:
        y_offs.append(y_total)
        y_total += (4 * L.M * L.N + 255) // 256 * 256
    y_all = torch.empty((y_total,), dtype=torch.uint8, device=dev)
    for l, L in enumerate(wl.layers):
        ys[l] = y_all[y_offs[l]:y_offs[l] + 4 * L.M * L.N].view(torch.float32).view(L.M, L.N)
    # every layer rotates over enough copies of its packed weights and
    # activations that one pass over them is more than twice L2; layers that
    # share a weight matrix share its copies
    Rs, Wrot, rot_by_seed = [], [], {}
    for i, (p, x) in enumerate(zip(packed, Xs)):
        nbytes = p.numel() + x.numel() * x.element_size()
        R = min(512, max(2, math.ceil(2 * l2 / nbytes) + 1))
        Rs.append(R)
        seed = workloads.weight_seed(wl, i)
        have = rot_by_seed.setdefault(seed, [p])
        while len(have) < R:
            have.append(p.clone())
        Wrot.append(have)
    Xrot = [[x] + [x.clone() for _ in range(R - 1)] for x, R in zip(Xs, Rs)]
    # quantised activations of every copy, made on first use, for timing the
    # forward kernel alone on layers whose step runs quantise + forward
    XQrot = [None] * nlayers
    torch.cuda.synchronize()

    # one workspace serves every layer's call (the calls run in stream order)
    ws_bytes = max(bl.bitlinear_forward_workspace_bytes(L.M, L.N, L.K) for L in wl.layers)
    workspace = torch.empty((max(ws_bytes, 16),), dtype=torch.uint8, device=dev)

    def layer_call(l, r, X=None):
        if tq5:
            bl.bitlinear_quant_act(Xrot[l][r] if X is None else X, x_q=xqs[l], s=ss[l], stream=stream)
            bl.bitlinear_forward_tq5(Wrot[l][r], gammas[l], xqs[l], ss[l], y=ys[l], stream=stream)
        elif fused:
            bl.bitlinear_quant_forward_ws(Wrot[l][r], gammas[l], Xrot[l][r] if X is None else X, y=ys[l],
                                          x_q=xqs[l], s=ss[l], workspace=workspace, stream=stream)
        elif args.path == "lut":
            bl.bitlinear_quant_act(Xrot[l][r] if X is None else X, x_q=xqs[l], s=ss[l], stream=stream)
            bl.bitlinear_forward_lut(Wrot[l][r], gammas[l], xqs[l], ss[l], y=ys[l], stream=stream)
        else:
            bl.bitlinear_quant_act(Xrot[l][r] if X is None else X, x_q=xqs[l], s=ss[l], stream=stream)
            bl.bitlinear_forward_ws(Wrot[l][r], gammas[l], xqs[l], ss[l], y=ys[l], workspace=workspace, stream=stream)

    def step(i, X_override=None):
        for l in range(nlayers):
            layer_call(l, i % Rs[l], None if X_override is None else X_override[l])

    def kernel_call(l, r):
        """The layer's forward alone: the fused quantise+GEMV where the layer
        runs as one kernel, else the forward product (GEMV or GEMM) on
        activations quantised beforehand."""
        L = wl.layers[l]
        if fused and gemv_fused_layer(L):
            layer_call(l, r)
        elif tq5:
            xq, s = XQrot[l][r]
            bl.bitlinear_forward_tq5(Wrot[l][r], gammas[l], xq, s, y=ys[l], stream=stream)
        elif args.path == "lut":
            xq, s = XQrot[l][r]
            bl.bitlinear_forward_lut(Wrot[l][r], gammas[l], xq, s, y=ys[l], stream=stream)
        else:
            xq, s = XQrot[l][r]
            bl.bitlinear_forward_ws(Wrot[l][r], gammas[l], xq, s, y=ys[l], workspace=workspace, stream=stream)

    def prepare_kernel_inputs(l):
        L = wl.layers[l]
        if not (fused and gemv_fused_layer(L)) and XQrot[l] is None:
            XQrot[l] = [bl.bitlinear_quant_act(x, stream=stream) for x in Xrot[l]]
            torch.cuda.synchronize()

    K, Wm = args.steps, args.warmup
    for i in range(Wm):
        step(i)
    torch.cuda.synchronize()
    bl.bitlinear_check_device_error(stream)

    if args.eager:
        return run_gpu_eager(args, wl, step, K, stream, dist, world, unit, metric)

    # ---- capture: the K steps as graphs of at most GRAPH_CHUNK steps
    def capture(fn, n, keep=False):
        g = torch.cuda.CUDAGraph(keep_graph=keep)
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                fn(j)
        return g

    chunk = min(GRAPH_CHUNK, K)
    nfull, rem = divmod(K, chunk)
    g_full = capture(step, chunk, keep=True)
    g_rem = capture(step, rem) if rem else None
    g_full.replay()
    torch.cuda.synchronize()
    nodes = graph_kernel_nodes(g_full)
    if tq5:  # quantise + base-3 forward, one pass per 4 tokens
        rule = sum(1 + -(-L.M // 4) for L in wl.layers)
    elif args.path == "lut":  # quantise + table-lookup GEMV
        rule = 2 * len(wl.layers)
    else:  # fused GEMV 1; quantise + GEMV 2; quantise (writing the fp16 operand) + GEMM 2
        rule = sum((1 if fused else 2) if gemv_fused_layer(L) else (2 if fused else 3) for L in wl.layers)
    launches_per_step = nodes / chunk if nodes is not None else rule
    graphs = [g_full] * nfull + ([g_rem] if g_rem is not None else [])

    # ---- timed region
    sampler = ClockSampler(local)
    with sampler:
        ms_per_step, R, rep_ms = timed_replays(graphs, K, stream, dist)
    clocks = sampler.summary()
    bl.bitlinear_check_device_error(stream)

    # ---- the graph-replayed outputs must equal an eager re-run of the last step
    last = [y.clone() for y in ys]
    step(rem - 1 if rem else chunk - 1)  # graphs were captured with chunk-local step indices
    torch.cuda.synchronize()
    verified = all(torch.equal(a, b) for a, b in zip(last, ys))

    step_bytes = sum(layer_bytes(L, args.format) for L in wl.layers)
    step_ops = sum(layer_ops(L) for L in wl.layers)

    def rate(ms):
        return world * (step_bytes / (ms * 1e-3) / 1e9 if unit == "GB/s" else step_ops / (ms * 1e-3) / 1e12)

    value = rate(ms_per_step)

    # ---- the same K steps launched call by call (no graph)
    per_launch_ms = []
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(dist)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(K):
            step(i)
        b.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
        per_launch_ms.append(a.elapsed_time(b) / K)
    pl_ms = max_over_ranks(dist, statistics.median(per_launch_ms))

    # ---- each layer's forward alone, back to back from a CUDA graph on the
    # launching stream (CUDA events around the replays)
    kchunk = 200

    def graph_us(fn):
        g = capture(fn, kchunk)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(3):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) * 1e3 / (3 * kchunk)

    kern_us = []
    for l in range(nlayers):
        prepare_kernel_inputs(l)
        kern_us.append(graph_us(lambda j, l=l: kernel_call(l, j % Rs[l])))
    per_layer = []
    for l, L in enumerate(wl.layers):
        e = layer_roofline(L, kern_us[l], fused, args.format, peaks, peak_src)
        e["kernel"] = ("gemv_tq5_kernel" if tq5 else "gemv_lut_kernel" if args.path == "lut"
                       else gemm_variant(L, props.multi_processor_count))
        if args.path == "lut":
            e["note"] = "bitlinear_forward_lut on quantised activations"
        elif fused and gemv_fused_layer(L) and not tq5:
            e["note"] = "the timed kernel also quantises the activations (fused)"
        elif not gemv_fused_layer(L) and not tq5:
            e["note"] = "bitlinear_forward_ws on quantised activations: the fp16 expansion of x_q plus the GEMM"
        per_layer.append(e)
    dom = max(range(nlayers), key=lambda l: kern_us[l])
    roof = {k: per_layer[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac")}
    roof["traffic"] = (ncu_traffic(per_layer[dom]["kernel"].split(" ")[0], per_layer[dom]["layer"])
                       if not args.layers else None)
    roof["layer"] = per_layer[dom]["layer"]
    roof["kernel"] = per_layer[dom]["kernel"]
    roof["peak_source"] = per_layer[dom]["peak_source"]
    roof["dominant"] = "the layer with the largest forward time in the step"
    roof["per_layer"] = per_layer
    roof["how"] = (f"each layer's forward replayed {3 * kchunk} times back to back from a CUDA graph over its "
                   "rotating buffers; CUDA events on the launching stream; bound from the layer's intensity "
                   "(2MNK per algorithmic byte) against the ridge of the measured peaks")
    if roof["bound"] == "tensor":
        roof["vs_legacy_mma_sync"] = {"s8": round(roof["achieved"] / LEGACY_MMA_SYNC["s8_tops"], 2),
                                      "f16": round(roof["achieved"] / LEGACY_MMA_SYNC["f16_tflops"], 2),
                                      "rates": LEGACY_MMA_SYNC}

    # the per-token quantisation (a3) alone, per layer: X read, x_q and s written
    quant = []
    for l, L in enumerate(wl.layers):
        us = graph_us(lambda j, l=l: bl.bitlinear_quant_act(Xrot[l][j % Rs[l]], x_q=xqs[l], s=ss[l], stream=stream))
        nbytes = L.M * L.K * (Xs[l].element_size() + 1) + 4 * L.M
        quant.append({"us": round(us, 3), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                      "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4), "algorithmic_bytes": nbytes})
    bl.bitlinear_check_device_error(stream)

    # ---- the FFN pieces around each layer, timed the same way (outside the step):
    # the sub-layer RMS norm then the quantisation of the layer's X, and the
    # fused forward with and without the squared-ReLU epilogue
    ffn = {"rmsnorm_quant": [], "forward_us": [], "forward_relu2_us": [], "norm_forward_one_call_us": [],
           "norm_forward_two_calls_us": [], "forward_requant_us": [], "forward_then_quant_us": []}
    for l, L in enumerate(wl.layers):
        gain = torch.rand((L.K,), generator=torch.Generator().manual_seed(l), dtype=torch.float32).add_(0.5).to(dev)
        us = graph_us(lambda j, l=l, gain=gain: bl.bitlinear_rmsnorm_quant_act(
            Xrot[l][j % Rs[l]], gain=gain, x_q=xqs[l], s=ss[l], stream=stream))
        nbytes = L.M * L.K * (Xs[l].element_size() + 1) + 4 * L.M + 4 * L.K
        ffn["rmsnorm_quant"].append({"us": round(us, 3), "GB/s": round(nbytes / (us * 1e-6) / 1e9, 1),
                                     "frac": round(nbytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                                     "algorithmic_bytes": nbytes})
        for key, fl in (("forward_us", 0), ("forward_relu2_us", bl.BITLINEAR_RELU2)):
            if tq5:
                prepare_kernel_inputs(l)
                ffn[key].append(round(graph_us(lambda j, l=l, fl=fl: bl.bitlinear_forward_tq5(
                    Wrot[l][j % Rs[l]], gammas[l], XQrot[l][j % Rs[l]][0], XQrot[l][j % Rs[l]][1], y=ys[l],
                    flags=fl, stream=stream)), 3))
            else:
                ffn[key].append(round(graph_us(lambda j, l=l, fl=fl: bl.bitlinear_quant_forward_ws(
                    Wrot[l][j % Rs[l]], gammas[l], Xrot[l][j % Rs[l]], y=ys[l], x_q=xqs[l], s=ss[l],
                    workspace=workspace, flags=fl, stream=stream)), 3))
        if not tq5:
            # the FFN's second BitLinear: RMS norm + quantisation + forward in one call
            # (the normalising kernel writes the GEMM's operand) against the two calls
            def two_calls(j, l=l, gain=gain):
                bl.bitlinear_rmsnorm_quant_act(Xrot[l][j % Rs[l]], gain=gain, x_q=xqs[l], s=ss[l], stream=stream)
                bl.bitlinear_forward_ws(Wrot[l][j % Rs[l]], gammas[l], xqs[l], ss[l], y=ys[l], workspace=workspace,
                                        stream=stream)
            ffn["norm_forward_one_call_us"].append(round(graph_us(
                lambda j, l=l, gain=gain: bl.bitlinear_rmsnorm_quant_forward_ws(
                    Wrot[l][j % Rs[l]], gammas[l], Xrot[l][j % Rs[l]], gain=gain, y=ys[l], x_q=xqs[l], s=ss[l],
                    workspace=workspace, stream=stream)), 3))
            ffn["norm_forward_two_calls_us"].append(round(graph_us(two_calls), 3))
            # the FFN's first BitLinear with its squared-ReLU output quantised for the
            # next layer in the same call, against the two calls
            yq = torch.empty((L.M, L.N), dtype=torch.int8, device=dev)
            sy = torch.empty((L.M,), dtype=torch.float32, device=dev)

            def then_quant(j, l=l, yq=yq, sy=sy):
                bl.bitlinear_quant_forward_ws(Wrot[l][j % Rs[l]], gammas[l], Xrot[l][j % Rs[l]], y=ys[l], x_q=xqs[l],
                                              s=ss[l], workspace=workspace, flags=bl.BITLINEAR_RELU2, stream=stream)
                bl.bitlinear_quant_act(ys[l], x_q=yq, s=sy, stream=stream)
            ffn["forward_requant_us"].append(round(graph_us(
                lambda j, l=l, yq=yq, sy=sy: bl.bitlinear_quant_forward_requant_ws(
                    Wrot[l][j % Rs[l]], gammas[l], Xrot[l][j % Rs[l]], y=ys[l], x_q=xqs[l], s=ss[l], y_q=yq, s_y=sy,
                    workspace=workspace, flags=bl.BITLINEAR_RELU2, stream=stream)), 3))
            ffn["forward_then_quant_us"].append(round(graph_us(then_quant), 3))
            del yq, sy
    bl.bitlinear_check_device_error(stream)
    ffn["note"] = ("rmsnorm_quant: bitlinear_rmsnorm_quant_act on each layer's X with a per-channel gain, bytes = "
                   "X read + x_q write + s + gain, frac of the measured copy bandwidth; forward(_relu2)_us: "
                   + ("bitlinear_forward_tq5 (quantised activations)" if tq5 else "bitlinear_quant_forward_ws")
                   + " without and with BITLINEAR_RELU2; norm_forward_one_call_us: bitlinear_rmsnorm_quant_forward_ws "
                   "(the normalising kernel writes the GEMM operand) against norm_forward_two_calls_us: "
                   "bitlinear_rmsnorm_quant_act then bitlinear_forward_ws; forward_requant_us: "
                   "bitlinear_quant_forward_requant_ws with BITLINEAR_RELU2 (y also quantised to int8 in the same "
                   "call, read back from L2) against forward_then_quant_us: bitlinear_quant_forward_ws with "
                   "BITLINEAR_RELU2 then bitlinear_quant_act on y")

    # ---- the lookup-table GEMV beside the conditional-add GEMV, on the layers of
    # at most 4 tokens (both on quantised activations, graph-replayed)
    lut = []
    for l, L in enumerate(wl.layers):
        if tq5 or L.M > 4:
            continue
        if XQrot[l] is None:
            XQrot[l] = [bl.bitlinear_quant_act(x, stream=stream) for x in Xrot[l]]
            torch.cuda.synchronize()
        us_lut = graph_us(lambda j, l=l: bl.bitlinear_forward_lut(Wrot[l][j % Rs[l]], gammas[l], XQrot[l][j % Rs[l]][0],
                                                                  XQrot[l][j % Rs[l]][1], y=ys[l], stream=stream))
        us_add = graph_us(lambda j, l=l: bl.bitlinear_forward(Wrot[l][j % Rs[l]], gammas[l], XQrot[l][j % Rs[l]][0],
                                                              XQrot[l][j % Rs[l]][1], y=ys[l], stream=stream))
        nbytes = forward_kernel_bytes(L, False)
        lut.append({"layer": f"M={L.M} K={L.K} N={L.N}", "lut_us": round(us_lut, 3), "dp4a_us": round(us_add, 3),
                    "lut_GB/s": round(nbytes / (us_lut * 1e-6) / 1e9, 1),
                    "lut_frac": round(nbytes / (us_lut * 1e-6) / 1e9 / peaks["hbm_gbs"], 4),
                    "dp4a_GB/s": round(nbytes / (us_add * 1e-6) / 1e9, 1)})
    bl.bitlinear_check_device_error(stream)

    # ---- live re-ternarisation: every distinct latent matrix re-packed in place
    # (gamma + ternarise + pack), as a training step would after each update;
    # one graph of all the packs, replayed, median per step
    repack = None
    if not tq5 and args.repack:
        latents, outs = [], []
        for i, L in enumerate(wl.layers):
            seed = workloads.weight_seed(wl, i)
            if seed in [s_ for s_, _ in latents]:
                continue
            latents.append((seed, workloads.layer_weights(wl, i).to(dev)))
            outs.append((torch.empty((L.N, L.K // 4), dtype=torch.uint8, device=dev),
                         torch.empty((1,), dtype=torch.float32, device=dev),
                         torch.empty((bl.bitlinear_pack_workspace_bytes(L.N, L.K),), dtype=torch.uint8, device=dev)))

        def repack_all(_j):
            for (_, Wl), (Wp_, g_, ws_) in zip(latents, outs):
                bl.bitlinear_pack_weights(Wl, W_packed=Wp_, gamma=g_, workspace=ws_, stream=stream)

        repack_all(0)
        torch.cuda.synchronize()
        gr = capture(repack_all, 1)
        times = []
        for _ in range(7):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            gr.replay()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        rp_ms = statistics.median(times)
        rp_bytes = sum(2 * 4 * Wl.numel() + Wl.numel() // 4 for _, Wl in latents)
        repack = {"ms_per_step": round(rp_ms, 4), "GB/s": round(rp_bytes / (rp_ms * 1e-3) / 1e9, 1),
                  "frac": round(rp_bytes / (rp_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4), "matrices": len(latents),
                  "algorithmic_bytes": rp_bytes,
                  "how": "bitlinear_pack_weights of every distinct latent matrix (read twice, packed bytes "
                         "written), one CUDA graph replayed 7 times, median; frac of the measured copy bandwidth"}
        del latents, outs, gr
        torch.cuda.empty_cache()

    e2e = run_e2e(bl, wl, step, Xs_host, y_all, K, Wm, stream, dist, world, unit, step_bytes, step_ops)

    config = common_config(args, wl)
    return {
        "metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": config,
        "timing": {"replays": R, "graph_steps": K, "replay_ms": [round(t, 4) for t in rep_ms],
                   "rotation": {"copies_per_layer": Rs,
                                "MiB_per_layer": [round(R * (p.numel() + x.numel() * x.element_size()) / 2**20)
                                                  for R, p, x in zip(Rs, packed, Xs)],
                                "l2_MiB": round(l2 / 2**20)},
                   "kernel_sum_us": round(sum(kern_us), 3),
                   "how": "median over R replays of the K-step graph, each bracketed by barrier + synchronize"},
        "per_launch": {"value": round(rate(pl_ms), 2), "unit": unit, "ms_per_step": round(pl_ms, 6),
                       "how": "the K steps launched call by call without a graph, median of 3 runs"},
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * K)),
        "gpu_launches_how": ("kernel nodes counted in the captured step graph" if nodes is not None
                             else "counted by the library's routing rule"),
        "verified": verified,
        "clocks": clocks,
        "quant": {"per_layer": quant,
                  "note": "bitlinear_quant_act alone per layer, graph-replayed over the rotating X copies; bytes = "
                          "X read + x_q written + s, frac of the measured copy bandwidth"},
        "ffn": ffn,
        "repack": repack,
        "lut": {"per_layer": lut, "how": "bitlinear_forward_lut (table lookup) and bitlinear_forward (conditional-add "
                                         "GEMV) on quantised activations, graph-replayed; bytes = packed W + x_q + y"},
        "pack": {"ms": round(pack_ms, 4), "GB/s": round(pack_bytes / (pack_ms * 1e-3) / 1e9, 1),
                 "matrices": len(by_seed),
                 "note": "gamma + ternarise + pack of every distinct weight matrix (one call each), outside the step"},
    }


def run_gpu_eager(args, wl, step, K, stream, dist, world, unit, metric):
    """Timed region with eager launches only (for profilers; includes launch gaps)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(K):
        step(i)
    b.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(dist, a.elapsed_time(b)) / K
    step_bytes = sum(layer_bytes(L, args.format) for L in wl.layers)
    step_ops = sum(layer_ops(L) for L in wl.layers)
    value = world * (step_bytes / (ms * 1e-3) / 1e9 if unit == "GB/s" else step_ops / (ms * 1e-3) / 1e12)
    cfg = common_config(args, wl)
    cfg["launch"] = "eager (profiling mode)"
    return {"metric": metric, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "int8", "data": "synthetic", "config": cfg}


def run_e2e(bl, wl, step, Xs_host, y_all, K, Wm, stream, dist, world, unit, step_bytes, step_ops):
    """The same step through the public API with host buffers: each step copies
    every layer's X from one pinned host buffer to the device (one copy), runs
    the layer calls, and copies every y back into one pinned host buffer (one
    copy); replayed from CUDA graphs like the device-side number."""
    dev = y_all.device
    in_bytes = [x.numel() * x.element_size() for x in Xs_host]
    out_bytes = [4 * L.M * L.N for L in wl.layers]

    # 256-byte aligned slices of one staging buffer per direction
    def offsets(sizes):
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += (n + 255) // 256 * 256
        return offs, o
    in_off, in_total = offsets(in_bytes)
    h_in = torch.empty((in_total,), dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty((in_total,), dtype=torch.uint8, device=dev)
    h_out = torch.empty(y_all.shape, dtype=torch.uint8, pin_memory=True)
    for x, o, n in zip(Xs_host, in_off, in_bytes):
        h_in[o:o + n].copy_(x.reshape(-1).view(torch.uint8))
    Xd = [d_in[o:o + n].view(x.dtype).view(x.shape) for x, o, n in zip(Xs_host, in_off, in_bytes)]
    h2d = sum(in_bytes)
    d2h = sum(out_bytes)

    def e2e_step(i):
        d_in.copy_(h_in, non_blocking=True)
        step(i, X_override=Xd)
        h_out.copy_(y_all, non_blocking=True)

    for i in range(Wm):
        e2e_step(i)
    torch.cuda.synchronize()
    chunk = min(GRAPH_CHUNK, K)
    nfull, rem = divmod(K, chunk)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(n):
                e2e_step(j)
        return g

    g1 = capture(chunk)
    g2 = capture(rem) if rem else None
    g1.replay()
    torch.cuda.synchronize()
    ms, R, _ = timed_replays([g1] * nfull + ([g2] if g2 is not None else []), K, stream, dist)
    val = world * (step_bytes / (ms * 1e-3) / 1e9 if unit == "GB/s" else step_ops / (ms * 1e-3) / 1e12)
    return {"value": round(val, 2), "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms, 6), "replays": R,
            "how": "CUDA graphs of one pinned H2D copy of every layer's X + C-ABI calls + one D2H copy of every y; "
                   "median over R replays"}


# ---------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default="fused", choices=["fused", "separate", "lut"],
                    help="fused: bitlinear_quant_forward; separate: bitlinear_quant_act + bitlinear_forward; "
                         "lut: bitlinear_quant_act + bitlinear_forward_lut")
    ap.add_argument("--format", default="2bit", choices=["2bit", "tq5"],
                    help="weight format: 2-bit (four per byte) or base-3 (five per byte, the forward on x_q)")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step eagerly instead of from CUDA graphs (for profilers)")
    ap.add_argument("--layers", default="", help="comma-separated layer indices of the workload (default: all)")
    ap.add_argument("--cpu-seconds", type=float, default=20.0, help="budget of the oracle CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-repack", dest="repack", action="store_false",
                    help="skip the timing of the per-step re-ternarisation of the latent weights")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps is None:
        args.steps = DEFAULT_STEPS[args.workload]
    if args.layers:
        wl0 = workloads.WORKLOADS[args.workload]
        idx = [int(v) for v in args.layers.split(",")]
        if any(i < 0 or i >= len(wl0.layers) for i in idx):
            ap.error(f"--layers indexes 0..{len(wl0.layers) - 1}")
        workloads.WORKLOADS[args.workload] = workloads.select_layers(wl0, idx)

    dist, rank, world, local = dist_setup()
    wl = workloads.WORKLOADS[args.workload]
    metric, unit = metric_for(wl)

    if args.impl == "reference":
        # the reference arm is the CPU oracle (OpenMP build) on the host cores; rank 0 only
        if rank == 0:
            value, frac, sec_step, n, thr = run_oracle(wl, budget_s=120.0, steps=args.steps, warmup=args.warmup,
                                                       fmt=args.format, omp=args.format != "tq5")
            line = {"impl": "reference", "metric": metric, "value": round(value, 4), "unit": unit,
                    "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": round(sec_step * 1e3, 4), "higher_is_better": True, "scaling": "weak",
                    "vs_baseline": None, "dtype": "int8 x ternary -> int64 sums (fp32 rescale)",
                    "data": "synthetic", "config": common_config(args, wl),
                    "cpu_baseline": {"value": round(value, 4), "unit": unit, "cores": thr, "kind": "oracle",
                                     "nproc": os.cpu_count(),
                                     "sample": f"{frac:.4%} of each layer's output rows, all tokens, per step; "
                                               f"{'OpenMP build, ' if thr > 1 else ''}{thr} host threads"},
                    "e2e": {"value": round(value, 4), "unit": unit, "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the BitLinear kernels have no CPU path)")
    line = run_gpu(args, dist, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.eager:
        line["cpu_baseline"] = cpu_baseline(wl, args.format, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
