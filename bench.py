"""Benchmark of the MoE verification pass on GB300.

Workload: the DeepSeek-V3-shaped FP8-E4M3 layer (d 7168, 256 routed experts
top-8 with sigmoid gating, 1 shared expert, intermediate 2048, 128x128 fp32
block scales), n = 8 draft-tree tokens (BFS tree, 4 children under the root,
2 below; child = 0.6 parent + 0.8 eps).  Synthetic, seeded weights and
hidden states; weights resident in HBM.

One step = one verification pass through the C ABI (moe_verify_pass): router
scores, top-k and union plan in one launch, then the deduplicating expert FFN
(gate/up, down) and the combine, recorded once into a CUDA graph and
replayed.  `value` = union-expert bytes per pass (routed union + shared
expert, weights and scales) / device time per pass.  The expert bytes of one
pass (1.76 GB at U = 39) exceed the 129 MB L2, so passes run back to back
with no flush.

Also printed: the expert kernels' roofline against the measured HBM copy
bandwidth, the end-to-end number (hidden states copied from pinned host
memory, outputs copied back, every step), the oracle on the host cores, and
a dedup-vs-per-slot sweep over n = 1..64 with its crossover.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from moe_expert_ffn_gemv_gb300 import synth  # noqa: E402

CFG = synth.DSV3
N_TOKENS = 8
METRIC = "µs per MoE verify pass and union-byte HBM GB/s (% of GB300 peak) vs n tokens"
WORKLOAD = "deepseek-v3-shaped fp8-e4m3 moe layer, n=8 draft-tree tokens (rho=0.6), dedup verify pass"
NOMINAL_HBM_GBS = (7900.0, 8000.0)  # GB300 HBM3e nominal: 7.9 TB/s, "~8 TB/s"
FALLBACK_HBM_GBS = 6800.0
# E4M3: route + top-k + plan (fused, + the fp16 rows of h), gate/up, fp16 rows of a, down, combine
KERNELS_PER_PASS = 5
KERNELS_PER_DEDUP_CALL = 5  # E4M3: fp16 rows of h, gate/up, fp16 rows of a, down, combine


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-sweep", action="store_true", help="skip the n = 1..64 engine sweep")
    p.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    p.add_argument("--sweep-max", type=int, default=64)
    p.add_argument("--sweep-min", type=int, default=1)
    p.add_argument("--sweep-config", default=None, choices=sorted(synth.CONFIGS),
                   help="run only the dedup-vs-per-slot sweep on this layer shape")
    p.add_argument("--fit-config", default=None, choices=sorted(synth.CONFIGS),
                   help="fit the bandwidth cost model on this layer shape and test it")
    p.add_argument("--windows", type=int, default=4, help="routing windows to fit (and to test)")
    p.add_argument("--budget-config", default=None, choices=sorted(synth.CONFIGS),
                   help="expert-budget sweep (MoE-Spec) on this layer shape, then exit")
    p.add_argument("--budget-n", default="8,16,32,64", help="pass sizes of the budget sweep")
    p.add_argument("--select-config", default=None, choices=sorted(synth.CONFIGS),
                   help="EVICT / EcoSpec selection on 64-node trees of this layer, then exit")
    p.add_argument("--select-trees", type=int, default=64, help="trees in the selection batch")
    p.add_argument("--stack-config", default=None, choices=sorted(synth.CONFIGS),
                   help="multi-layer pass and best draft length on this layer shape, then exit")
    p.add_argument("--layers", type=int, default=8, help="MoE layers of the stack")
    p.add_argument("--max-drafts", type=int, default=15, help="largest K (n = K + 1 tokens)")
    p.add_argument("--t-draft", type=float, default=0.0,
                   help="draft cost of one position in µs (added as K * t_draft)")
    p.add_argument("--rho", type=float, default=None, help="chain/tree correlation for the sweep")
    p.add_argument("--sigma", type=float, default=None, help="tree noise for the sweep")
    p.add_argument("--experts", type=int, default=None,
                   help="routed experts of the layer (default: the shape's own); fewer make a "
                        "small profiling case")
    return p.parse_args()


# ------------------------------------------------------------- environment

def dist_setup(args=None):
    """One process per GPU (replicas only): NCCL when there is a GPU, gloo
    when there is none (the CPU tests of the replica path)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: float, ms_per_step: float, ws: int) -> float:
    """The whole job's throughput: every rank moves bytes_per_rank_step per
    step, and a step takes ms_per_step (the slowest rank's time)."""
    return ws * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def clocks_rejected(clocks) -> bool:
    """A timed region is rejected when its clock samples show a hardware or
    thermal slowdown, or a median SM clock below 85% of the maximum with no
    reason reported (power capping alone is kept)."""
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    reasons = set(clocks.get("reasons") or [])
    if reasons & bad:
        return True
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.85 * mx and not (reasons - {"unsampled"}))


def traffic_from_profile():
    """DRAM bytes per dedup call from the committed ncu summary, if it was
    taken on the current sources of the kernels that call runs (else None)."""
    path = os.path.join(ROOT, "profiles", "dedup_dsv3_fp8_n8.md")
    try:
        with open(path) as f:
            for line in f:
                if line.startswith("traffic_json:"):
                    j = json.loads(line.split(":", 1)[1])
                    if j.get("dedup_kernels_code_sha256") == code_hash(DEDUP_KERNEL_SOURCES):
                        return j.get("dram_bytes_per_dedup_call")
    except Exception:
        pass
    return None


# The sources of the kernels a moe_verify_dedup call runs (and the layout
# they read): what a recorded DRAM-traffic figure for that call depends on.
DEDUP_KERNEL_SOURCES = ("act_scale.cu", "act_scale.cuh", "combine.cu", "expert_tc.cu", "kernels.h",
                        "moe_common.cuh", "pack.cu")


def csrc_hash(names=None) -> str:
    """Hash of the kernel sources (all of csrc/, or the named files)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "moe_expert_ffn_gemv_gb300", "csrc")
    for name in sorted(names or os.listdir(d)):
        with open(os.path.join(d, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def strip_comments(src: str) -> str:
    """C/C++/CUDA source without its comments, each run of whitespace made
    one space: what the compiler sees, give or take the preprocessor.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def code_hash(names) -> str:
    """Hash of the named kernel sources with their comments left out, so
    that a recorded measurement stays tied to the code, not to its prose."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "moe_expert_ffn_gemv_gb300", "csrc")
    for name in sorted(names):
        with open(os.path.join(d, name), encoding="utf-8") as f:
            h.update(name.encode())
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


# -------------------------------------------------------------- workloads

def make_workload(device="cuda"):
    layer = synth.make_layer(CFG, seed=1, device=device)
    if layer.cfg.n_experts != CFG.n_experts:
        raise AssertionError("layer config mismatch")
    h = synth.make_hidden(CFG, 64, seed=3, device=device)   # the first n nodes of a 64-node tree
    return layer, h


def bench_config(U, union_bytes, ws):
    """The workload's config, the same on both arms."""
    return {"workload": WORKLOAD, "n_tokens": N_TOKENS, "d": CFG.d, "experts": CFG.n_experts,
            "top_k": CFG.top_k, "shared": CFG.n_shared, "inter": CFG.inter,
            "U": U, "union_bytes_per_pass": union_bytes,
            "l2": "inputs larger than L2 (union bytes per pass >> 129 MB), no flush",
            "parallelism": f"replicas x{ws}"}


def expert_bytes(mv, desc):
    wb, sb = mv.moe_expert_bytes(desc)
    return wb + sb


# ------------------------------------------------------------------- ours

def run_ours(args):
    ws, rank = dist_setup(args)
    from moe_expert_ffn_gemv_gb300 import binding as mv
    n = N_TOKENS
    layer, h_all = make_workload()
    h = h_all[:n].contiguous()
    vl = mv.VerifyLayer(layer, 64)
    eb = expert_bytes(mv, vl.desc)
    stream = torch.cuda.current_stream()

    for _ in range(max(args.warmup, 3)):
        vl.verify_pass(h, n)
    assert vl.last_error() == 0
    union_bytes = int(vl.plan.union_bytes[0])
    U = int(vl.plan.n_uniq[0])

    # the pass as one CUDA graph (route + plan, then the expert call); the
    # expert call alone as a second graph, for the roofline of its kernels
    g_pass = vl.capture_pass(h, n)
    g_route, g_exp = vl.capture(h, n)
    for _ in range(3):
        g_pass.replay()
        g_exp.replay()
    torch.cuda.synchronize()
    assert vl.last_error() == 0

    # timed region: K passes back to back, then K expert calls back to back,
    # each bracketed by events on the launching stream
    def timed_region():
        barrier(ws)
        torch.cuda.synchronize()
        with ClockSampler(torch.cuda.current_device()) as clk:
            t_start = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            t_start.record(stream)
            for i in range(args.steps):
                g_pass.replay()
            t_end.record(stream)
            d_start = torch.cuda.Event(enable_timing=True)
            d_end = torch.cuda.Event(enable_timing=True)
            d_start.record(stream)
            for i in range(args.steps):
                g_exp.replay()
            d_end.record(stream)
            torch.cuda.synchronize()
        barrier(ws)
        return t_start.elapsed_time(t_end), d_start.elapsed_time(d_end), clk.summary()

    pass_ms, dedup_ms, clocks = timed_region()
    # a region that saw a hardware or thermal slowdown, or SM clocks well below
    # their maximum with no reason given (a clock lock), is measured once more;
    # every rank takes the same decision
    if max_over_ranks(1.0 if clocks_rejected(clocks) else 0.0, ws) > 0:
        pass_ms, dedup_ms, clocks = timed_region()
        clocks["remeasured"] = True
    total_ms = max_over_ranks(pass_ms, ws)
    assert vl.last_error() == 0
    ms_per_step = total_ms / args.steps
    value = whole_job_gbs(union_bytes, ms_per_step, ws)

    # the spread of single passes: the same graph replayed K more times, each
    # replay between its own pair of events (outside the timed region above)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        g_pass.replay()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_pass = sorted(1e3 * evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))
    q = lambda f: per_pass[min(len(per_pass) - 1, int(f * (len(per_pass) - 1) + 0.5))]
    replays = {"median_us": round(statistics.median(per_pass), 2),
               "iqr_us": [round(q(0.25), 2), round(q(0.75), 2)], "replays": args.steps}

    # algorithmic bytes of one moe_verify_dedup call: union expert bytes + the
    # hidden states (bf16, read once), their fp16 rows (written and read
    # once), the intermediate a (bf16, written and read once per slot), the
    # per-slot fp32 outputs (written, read), y (bf16) and the gate weights
    slots = n * (CFG.top_k + CFG.n_shared)
    act_bytes = (n * CFG.d * 2 + 2 * n * CFG.d * 2 + 2 * slots * CFG.inter * 2
                 + 2 * slots * CFG.d * 4 + n * CFG.d * 2 + n * CFG.top_k * 4)
    alg_bytes = union_bytes + act_bytes
    dedup_avg = dedup_ms / args.steps
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / (dedup_avg * 1e-3) / 1e9

    # end to end through the public API, every step: pinned host h -> device,
    # the pass, y -> pinned host.  Steps are independent passes, so one
    # step's copies overlap another step's pass: two (h, y) buffer pairs with
    # a captured pass each, one stream per copy direction (so that the next
    # input need not queue behind the read-back of a pass still running), and
    # events that order each buffer's copy in, pass and read-back.
    h_host = h.cpu().pin_memory()
    y_host = [torch.empty(n, CFG.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    hb = [h.clone() for _ in range(2)]
    yb = [torch.empty(n, CFG.d, dtype=vl.y.dtype, device="cuda") for _ in range(2)]
    gx = [vl.capture_pass(hb[x], n, y=yb[x]) for x in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined(steps):
        ev_c, ev_y = [None, None], [None, None]
        for i in range(steps):
            x = i % 2
            with torch.cuda.stream(h2d):
                if ev_c[x] is not None:
                    h2d.wait_event(ev_c[x])       # the pass that read hb[x] is done
                hb[x].copy_(h_host, non_blocking=True)
                eh = torch.cuda.Event()
                eh.record(h2d)
            stream.wait_event(eh)
            if ev_y[x] is not None:
                stream.wait_event(ev_y[x])        # yb[x] has been read back
            gx[x].replay()
            ec = torch.cuda.Event()
            ec.record(stream)
            ev_c[x] = ec
            with torch.cuda.stream(d2h):
                d2h.wait_event(ec)
                y_host[x].copy_(yb[x], non_blocking=True)
                ey = torch.cuda.Event()
                ey.record(d2h)
                ev_y[x] = ey

    pipelined(4)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    e0.record(h2d)
    pipelined(args.steps)
    e1.record(d2h)
    torch.cuda.synchronize()
    assert vl.last_error() == 0
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws) / args.steps
    e2e_value = whole_job_gbs(union_bytes, e2e_ms, ws)

    cpu = None
    oracle_ns = []
    if not args.no_cpu and rank == 0 and ws == 1:
        cpu = cpu_baseline(layer, h, union_bytes)
        oracle_ns = [1, N_TOKENS, args.sweep_max]

    sweep = None
    if not args.no_sweep and rank == 0:
        sweep = engine_sweep(mv, layer, h_all, args.sweep_max, eb, oracle_ns=oracle_ns)

    if rank == 0:
        out = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": "GB/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3 weights x fp16 activations, fp32 accumulate",
            "data": "synthetic (seeded N(0,0.02^2) weights quantised per 128x128 block; tree hidden states)",
            "config": bench_config(U, union_bytes, ws),
            "us_per_pass": round(1e3 * ms_per_step, 2),
            "us_per_pass_single_replays": replays,
            "us_dedup_call": round(1e3 * dedup_avg, 2),
            "pct_of_nominal_whole_pass": {f"{g:.0f}_gbs": round(100 * value / ws / g, 1)
                                          for g in NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "peak_kind": peak_kind, "kernel": "moe_verify_dedup (gate/up + down + combine)",
                         "traffic": traffic_from_profile(),
                         "algorithmic_bytes_per_launch": alg_bytes},
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": n * CFG.d * 2, "d2h_bytes_per_step": n * CFG.d * 2,
                    "us_per_pass": round(1e3 * e2e_ms, 2),
                    "copies": "every step copies its h in and its y out (pinned host); "
                              "one step's copies overlap another step's pass "
                              "(two buffer pairs, a stream per copy direction)"},
            "gpu_launches": (KERNELS_PER_PASS + KERNELS_PER_DEDUP_CALL) * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "sweep": sweep,
        }
        print(json.dumps(out))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def flush_l2(buf_a, buf_b):
    buf_a.fill_(1)            # write more than L2 ...
    buf_b.sum()               # ... then read more than L2, so no dirty lines remain


def engine_sweep(mv, layer, h_all, n_max, eb, reps=5, n_min=1, cfg=None, oracle_ns=()):
    """µs per pass of each engine's expert call (after routing and planning,
    which are shared) for n = n_min..n_max, L2 flushed before each timed call;
    u_bar, r and the crossover as "Expert Bytes, Kernel Bandwidth and the Best
    Draft Length" defines them (moe_expert_ffn_gemv_gb300/crossover.py).
    For each n in oracle_ns, the oracle's time for the same pass on the host
    cores beside it (oracle_pass_times)."""
    from moe_expert_ffn_gemv_gb300 import crossover as X
    cfg = cfg or CFG
    vl = mv.VerifyLayer(layer, 64)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    a = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    b = torch.ones_like(a)
    stream = torch.cuda.current_stream()
    raw = []
    for n in range(n_min, n_max + 1):
        h = h_all[:n].contiguous()
        vl.route_plan(h, n)
        vl.dedup(h, n)
        vl.perslot(h, n)
        torch.cuda.synchronize()
        U = int(vl.plan.n_uniq[0])
        t = {}
        for eng in ("dedup", "perslot"):
            ts = []
            for _ in range(reps):
                flush_l2(a, b)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                (vl.dedup if eng == "dedup" else vl.perslot)(h, n)
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e-3)
            t[eng] = statistics.median(ts)
        assert vl.last_error() == 0
        raw.append(dict(n=n, U=U, t_dedup=t["dedup"], t_slot=t["perslot"]))
    an = X.analyse(raw, cfg.top_k, eb, cfg.n_shared)
    # consecutive-token reuse of the window: token n's experts already chosen
    # by the tokens before it (the routing of a token does not depend on the
    # pass size, so one routing of the largest pass gives every n)
    vl.route_plan(h_all[:n_max].contiguous(), n_max)
    torch.cuda.synchronize()
    reuse = [None] + X.consecutive_reuse(vl.ids_view(n_max).cpu().tolist())
    rows = [[a_["n"], a_["U"], round(1e6 * a_["t_dedup"], 1), round(1e6 * a_["t_slot"], 1),
             round(a_["u_bar"], 3), round(a_["r"], 3), round(a_["beta_dedup"] / 1e9, 1),
             round(a_["beta_slot"] / 1e9, 1),
             None if reuse[a_["n"] - 1] is None else round(reuse[a_["n"] - 1], 3),
             round(X.uniform_reuse(a_["n"], cfg.top_k, cfg.n_experts), 3)] for a_ in an]
    cols = ["n", "U", "us_dedup", "us_perslot", "u_bar", "r", "gbs_dedup_union",
            "gbs_perslot_requested", "reuse_rho", "reuse_rho_uniform"]
    extra = {}
    ns = sorted({m for m in oracle_ns if n_min <= m <= n_max})
    if ns:
        ot = oracle_pass_times(cfg, layer, h_all, ns)
        cols += ["oracle_ms_all_cores", "oracle_ms_1_thread"]
        for row in rows:
            o = ot["per_n"].get(row[0])
            row += [None, None] if o is None else [o["ms_all_cores"], o["ms_1_thread"]]
        extra["oracle_host"] = ot["host"]
    return {"columns": cols,
            "rows": rows,
            **extra,
            "crossover_n": X.crossover([a_["n"] for a_ in an], [a_["t_dedup"] for a_ in an],
                                       [a_["t_slot"] for a_ in an]),
            "criterion_agrees": all(a_["criterion_dedup_faster"] == a_["measured_dedup_faster"]
                                    for a_ in an),
            "l2": "flushed (2x L2 written then 2x L2 read) before each timed call"}


def run_fit(args):
    """--fit-config NAME: fit each engine's effective bandwidth per n on
    --windows routing windows, predict time and saving on as many held-out
    windows, and check the saving bound and the faster-kernel criterion."""
    from moe_expert_ffn_gemv_gb300 import binding as mv
    from moe_expert_ffn_gemv_gb300 import crossover as X
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS[args.fit_config]
    layer = synth.make_layer(cfg, seed=1, device="cuda")
    eb = sum(mv.moe_expert_bytes(mv.make_desc(cfg, 64)))
    vl = mv.VerifyLayer(layer, 64)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    fa = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    fb = torch.ones_like(fa)
    stream = torch.cuda.current_stream()

    def timed(fn, reps=3):
        ts = []
        for _ in range(reps):
            flush_l2(fa, fb)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    fit_w, test_w = [], []
    for w in range(2 * args.windows):
        h_all = synth.make_hidden(cfg, 64, seed=1000 + w, device="cuda", rho=args.rho,
                                  sigma=args.sigma)
        for n in range(1, args.sweep_max + 1):
            h = h_all[:n].contiguous()
            vl.route_plan(h, n)
            vl.dedup(h, n)
            vl.perslot(h, n)
            torch.cuda.synchronize()
            U = int(vl.plan.n_uniq[0])
            row = dict(n=n, U=U, t_dedup=timed(lambda: vl.dedup(h, n)),
                       t_slot=timed(lambda: vl.perslot(h, n)))
            (fit_w if w < args.windows else test_w).append(row)
    assert vl.last_error() == 0
    k, sh = cfg.top_k, cfg.n_shared
    model = X.fit_bandwidths(fit_w, k, eb, sh)
    # the per-slot engine's re-read cost against a unique read (eq. (4)
    # reading), over every window's per-slot times
    rr = X.fit_reread_cost(fit_w + test_w, k, sh)
    reread = {"c_u_us": round(1e6 * rr["c_u"], 3), "c_re_us": round(1e6 * rr["c_re"], 3),
              "c_re_over_c_u": round(rr["ratio"], 3), "t0_us": round(1e6 * rr["t0"], 2),
              "rms_us": round(1e6 * rr["rms"], 2), "points": rr["points"],
              "unique_read_gbs": round(eb / rr["c_u"] / 1e9, 1)}
    ev = X.evaluate(model, test_w, k, eb, sh)
    ns = sorted(model)
    med = lambda xs: statistics.median(xs) if xs else float("nan")
    s_meas = {n: med([e["saving"] for e in ev if e["n"] == n]) for n in ns}
    s_pred = {n: med([e["saving_hat"] for e in ev if e["n"] == n]) for n in ns}
    cross_meas = next((n for n in ns if s_meas[n] > 0), None)
    cross_pred = next((n for n in ns if s_pred[n] > 0), None)
    # (19): where the criterion is certain for the fit's eps, it must pick the faster kernel
    certain = agree = 0
    for e, w in zip(ev, test_w):
        m = model[w["n"]]
        ub = X.u_bar(w["U"], w["n"], k, sh)
        r_hat = m["beta_dedup"] / m["beta_slot"]
        if X.faster_kernel_is_certain(r_hat, ub, m["eps"]):
            certain += 1
            agree += (ub < r_hat) == (w["t_dedup"] < w["t_slot"])
    print(json.dumps({
        "fit_config": cfg.name, "windows_fit": args.windows, "windows_test": args.windows,
        "n_max": args.sweep_max,
        "model": {str(n): {"gbs_slot": round(model[n]["beta_slot"] / 1e9, 1),
                           "gbs_dedup": round(model[n]["beta_dedup"] / 1e9, 1),
                           "eps": round(model[n]["eps"], 4)} for n in ns},
        "saving_us": {str(n): [round(1e6 * s_meas[n], 2), round(1e6 * s_pred[n], 2)] for n in ns},
        "max_saving_error_us": round(1e6 * max(abs(e["saving"] - e["saving_hat"]) for e in ev), 2),
        "inside_bound_18": f"{sum(e['inside'] for e in ev)} of {len(ev)}",
        "sign_of_saving_predicted": f"{sum(e['sign_ok'] for e in ev)} of {len(ev)}",
        "criterion_19_certain_and_right": f"{agree} of {certain}",
        "crossover_measured": cross_meas, "crossover_predicted": cross_pred,
        "reread_cost": reread}))


def run_sweep_only(args):
    """--sweep-config NAME: the engine sweep alone on another layer shape."""
    from moe_expert_ffn_gemv_gb300 import binding as mv
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS[args.sweep_config]
    if args.experts:
        from dataclasses import replace
        cfg = replace(cfg, n_experts=args.experts, name=f"{cfg.name} ({args.experts} routed experts)")
    layer = synth.make_layer(cfg, seed=1, device="cuda")
    h_all = synth.make_hidden(cfg, 64, seed=3, device="cuda", rho=args.rho, sigma=args.sigma)
    eb = sum(mv.moe_expert_bytes(mv.make_desc(cfg, 64)))
    sw = engine_sweep(mv, layer, h_all, args.sweep_max, eb, n_min=args.sweep_min, cfg=cfg,
                      oracle_ns=[] if args.no_cpu else [1, 8, args.sweep_max])
    print(json.dumps({"sweep_config": cfg.name, "rho": args.rho if args.rho is not None else cfg.rho,
                      "sigma": args.sigma if args.sigma is not None else cfg.sigma,
                      "hidden": cfg.hidden, **sw}))


def run_budget(args):
    """--budget-config NAME: the verification-time expert budget (MoE-Spec)
    for n in --budget-n and B from the full union U down to a quarter of it
    and k: µs of the fused route + budgeted plan (against the plain one), µs
    and GB/s of the deduplicating expert call on the kept union bytes, and
    how far the output moves from the unbudgeted output (the cap is lossy):
    relative L2 distance and the largest element-relative deviation."""
    from moe_expert_ffn_gemv_gb300 import binding as mv
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS[args.budget_config]
    layer = synth.make_layer(cfg, seed=1, device="cuda")
    h_all = synth.make_hidden(cfg, 64, seed=3, device="cuda", rho=args.rho, sigma=args.sigma)
    eb = sum(mv.moe_expert_bytes(mv.make_desc(cfg, 64)))
    vl = mv.VerifyLayer(layer, 64)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    fa = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    fb = torch.ones_like(fa)
    stream = torch.cuda.current_stream()

    def timed(fn, reps=5):
        ts = []
        for _ in range(reps):
            flush_l2(fa, fb)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    rows = []
    for n in [int(x) for x in args.budget_n.split(",")]:
        h = h_all[:n].contiguous()
        vl.route_plan(h, n)
        y_full = vl.dedup(h, n).float().clone()
        U = int(vl.plan.n_uniq[0])
        t_plan_plain = timed(lambda: vl.route_plan(h, n))
        t_full = timed(lambda: vl.dedup(h, n))
        budgets = sorted({U, (3 * U) // 4, U // 2, U // 4, cfg.top_k}, reverse=True)
        for B in budgets:
            vl.route_plan(h, n, budget=B)
            y = vl.dedup(h, n, kept=True).float().clone()
            Uk = int(vl.plan.n_uniq[0])
            assert int(vl.routed_u[0]) == U and Uk == min(B, U)
            t_plan = timed(lambda: vl.route_plan(h, n, budget=B))
            t = timed(lambda: vl.dedup(h, n, kept=True))
            kept_bytes = (Uk + cfg.n_shared) * eb
            rms = float(y_full.pow(2).mean().sqrt())
            dev = (y - y_full).abs() / torch.clamp(y_full.abs(), min=rms)
            rows.append([n, U, B, round(1e6 * t_plan_plain, 1), round(1e6 * t_plan, 1),
                         round(1e6 * t_full, 1), round(1e6 * t, 1),
                         round(kept_bytes / t / 1e9, 1),
                         round(1 - kept_bytes / ((U + cfg.n_shared) * eb), 3),
                         float(f"{float((y - y_full).norm() / y_full.norm()):.4g}"),
                         float(f"{float(dev.max()):.4g}")])
    assert vl.last_error() == 0
    print(json.dumps({
        "budget_config": cfg.name, "rho": args.rho if args.rho is not None else cfg.rho,
        "sigma": args.sigma if args.sigma is not None else cfg.sigma, "hidden": cfg.hidden,
        "columns": ["n", "U", "B", "us_route_plan", "us_route_plan_budgeted", "us_dedup_full",
                    "us_dedup_budgeted", "gbs_kept_union", "union_bytes_saved",
                    "rel_l2_dev_from_full", "max_rel_dev_from_full"],
        "rows": rows,
        "l2": "flushed (2x L2 written then 2x L2 read) before each timed call; median of 5"}))


def draft_tree_batch(T, K, seed):
    """T draft trees of K nodes (the BFS tree shape of the hidden-state
    recipe) with draft probabilities: each parent's children share one
    Dirichlet(0.5) draw over (children + the rest of the vocabulary)."""
    import numpy as np
    par = np.array(synth.tree_parents(K), dtype=np.int32)
    rng = np.random.default_rng(seed)
    q = np.ones((T, K), dtype=np.float32)
    kids = {}
    for v in range(1, K):
        kids.setdefault(int(par[v]), []).append(v)
    for t in range(T):
        for p_, ch in kids.items():
            d = rng.dirichlet(np.full(len(ch) + 1, 0.5))
            q[t, ch] = np.sort(d[:-1])[::-1]  # the draft ranks its children by probability
    return np.broadcast_to(par, (T, K)).copy(), q


def run_select(args):
    """--select-config NAME: pre-verification selection on a batch of
    --select-trees draft trees of 64 nodes.

    - EVICT (utility-guided prefix): C(k) is this library's measured layer
      pass (route + plan + dedup) at n = k. It reports k* over the trees and
      the kernel's µs for the batch (20 calls in one CUDA graph).
    - EcoSpec (cost-aware selection), at gamma = 4, 8, 16, with the layer's
      own routing as the predicted sets (a perfect predictor). It reports the
      kernel's µs, the mean union of the selected nodes against the
      confidence-ranked top-gamma, and the measured verify pass of both node
      sets (L2 flushed, median of 3)."""
    import numpy as np
    from moe_expert_ffn_gemv_gb300 import binding as mv
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS[args.select_config]
    layer = synth.make_layer(cfg, seed=1, device="cuda")
    K, T = 64, args.select_trees
    par, q = draft_tree_batch(T, K, seed=11)
    vl = mv.VerifyLayer(layer, K)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    fa = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    fb = torch.ones_like(fa)
    stream = torch.cuda.current_stream()

    def timed(fn, reps=3, flush=True):
        ts = []
        for _ in range(reps):
            if flush:
                flush_l2(fa, fb)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    def verify_pass(h):
        n = h.shape[0]
        vl.route_plan(h, n)
        vl.dedup(h, n)

    hs = [synth.make_hidden(cfg, K, seed=100 + t, device="cuda") for t in range(T)]
    ids = []
    for h in hs:
        vl.route(h, K)
        ids.append(vl.ids_view(K).clone())
    ids = torch.stack(ids)                               # [T][K][k]
    # EVICT: C(k) from the measured pass on tree 0's first k nodes
    cost = np.array([timed(lambda: verify_pass(hs[0][:k].contiguous())) * 1e6
                     for k in range(1, K + 1)], dtype=np.float32)
    par_d = torch.from_numpy(par).cuda()
    q_d = torch.from_numpy(q).cuda()
    cost_d = torch.from_numpy(cost).cuda()

    def graph_us(call, reps=20):
        """µs per call: `reps` calls on preallocated buffers captured in one
        CUDA graph, so that host latency stays out of the device time."""
        call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                call()
        g.replay()
        torch.cuda.synchronize()
        return 1e6 * timed(g.replay, reps=5, flush=False) / reps

    ev_out = [torch.empty(T, K, dtype=torch.int32, device="cuda"),
              torch.empty(T, K, dtype=torch.float64, device="cuda"),
              torch.empty(T, K, dtype=torch.float64, device="cuda"),
              torch.empty(T, dtype=torch.int32, device="cuda")]
    out = {}
    t_ev = graph_us(lambda: mv.moe_evict_select(par_d, q_d, T, K, cost_d, *ev_out))
    k_star = mv.evict_select(par_d, q_d, cost_d)[0].cpu().numpy()
    out["evict"] = {"kernel_us_batch": round(t_ev, 2),
                    "k_star": {"min": int(k_star.min()), "median": float(np.median(k_star)),
                               "max": int(k_star.max())},
                    "cost_us_at_k": {str(k): round(float(cost[k - 1]), 1)
                                     for k in (1, 2, 4, 8, 16, 32, 64)}}
    order = mv.evict_select(par_d, q_d, cost_d)[1].cpu().numpy()
    pred = ids[:, :, None, :].contiguous()
    eco = []
    n_meas = min(T, 16)
    for gamma in (4, 8, 16):
        eco_out = [torch.empty(T, gamma, dtype=torch.int32, device="cuda"),
                   torch.empty(T, 1, (cfg.n_experts + 31) // 32, dtype=torch.int32, device="cuda"),
                   torch.empty(T, dtype=torch.int32, device="cuda")]
        t_k = graph_us(lambda: mv.moe_ecospec_select(par_d, q_d, pred, T, K, 1, cfg.n_experts,
                                                     cfg.top_k, gamma, 1e-6, None, *eco_out))
        sel, _, usz = mv.ecospec_select(par_d, q_d, pred, cfg.n_experts, gamma, 1e-6)
        sel = sel.cpu().numpy()
        ids_np = ids.cpu().numpy()
        u_eco = [len(set(ids_np[t][sel[t]].ravel().tolist())) for t in range(T)]
        u_conf = [len(set(ids_np[t][order[t, :gamma]].ravel().tolist())) for t in range(T)]
        assert u_eco == usz.cpu().tolist()
        t_eco = [timed(lambda: verify_pass(hs[t][torch.from_numpy(sel[t]).long().cuda()]
                                           .contiguous())) for t in range(n_meas)]
        t_conf = [timed(lambda: verify_pass(hs[t][torch.from_numpy(order[t, :gamma].copy())
                                                  .long().cuda()].contiguous()))
                  for t in range(n_meas)]
        eco.append({"gamma": gamma, "kernel_us_batch": round(t_k, 2),
                    "U_ecospec_mean": round(float(np.mean(u_eco)), 2),
                    "U_confidence_mean": round(float(np.mean(u_conf)), 2),
                    "us_verify_ecospec": round(1e6 * float(np.mean(t_eco)), 1),
                    "us_verify_confidence": round(1e6 * float(np.mean(t_conf)), 1),
                    "trees_timed": n_meas})
    out["ecospec"] = eco
    assert vl.last_error() == 0
    print(json.dumps({"select_config": cfg.name, "trees": T, "nodes": K,
                      "hidden": cfg.hidden, **out}))


def run_stack(args):
    """--stack-config NAME --layers L: the verify pass of L MoE layers (one
    CUDA graph per pass size) for K = 0..--max-drafts drafts (n = K + 1
    tokens of a chain or tree, the layer's recipe), over --windows hidden-
    state windows.  Reports per K the median stack time T_T(K) and the
    layer-averaged union U_bar ("The Limits of Speculation", eq. (5)); the
    cost model T_T = beta0(m) + alpha(m) U_bar per m (its eq. (4), no
    context term) and pooled over m (eq. (3)); and, with the step time
    V(K) = T_T(K) + K * --t-draft, the best draft length k*(a) under
    geometric acceptance, its staircase, a0 and the speedup
    ("Speculative Decoding for MoE Models: Expert Bytes, ...").  The
    calibrated step time (the pooled fit at each K's mean U_bar) gives
    k_hat*(a); its relative error delta feeds bound (20)."""
    import numpy as np
    from moe_expert_ffn_gemv_gb300 import binding as mv
    from moe_expert_ffn_gemv_gb300 import draft_length as D
    torch.cuda.set_device(0)
    cfg = synth.CONFIGS[args.stack_config]
    L, Kmax, W = args.layers, args.max_drafts, args.windows
    n_max = Kmax + 1
    st = mv.VerifyStack.synthetic(cfg, L, n_max, seed=1)
    hs = torch.empty(L, n_max, cfg.d, dtype=synth.torch_dtype(cfg.act), device="cuda")
    windows = [torch.stack([synth.make_hidden(cfg, n_max, seed=5000 + 100 * w + l, device="cuda",
                                              rho=args.rho, sigma=args.sigma)
                            for l in range(L)]) for w in range(W)]
    stream = torch.cuda.current_stream()
    rounds = []
    for K in range(Kmax + 1):
        n = K + 1
        hs.copy_(windows[0])
        g = st.capture(hs, n)
        for w in range(W):
            hs.copy_(windows[w])
            g.replay()  # warm
            ts = []
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1) * 1e3)
            rounds.append({"K": K, "m": n, "w": w, "t": statistics.median(ts),
                           "u_bar": D.layer_mean_union(st.unions())})
        del g
    assert st.last_error() == 0
    t_med = [statistics.median(r["t"] for r in rounds if r["K"] == K) for K in range(Kmax + 1)]
    u_mean = [statistics.mean(r["u_bar"] for r in rounds if r["K"] == K) for K in range(Kmax + 1)]
    per_m = D.fit_cost_model(rounds)
    pooled = D.fit_cost_model([dict(r, m=0) for r in rounds])[0]
    V = D.step_time(t_med, args.t_draft)
    V_hat = D.step_time([pooled["beta0"] + pooled["alpha"] * u for u in u_mean], args.t_draft)
    delta = max(abs(vh / v - 1) for vh, v in zip(V_hat, V))
    grid = [i / 100 for i in range(0, 100)]
    agree = sum(D.best_draft_length(a, V_hat) == D.best_draft_length(a, V) for a in grid)
    inside = sum(D.throughput(a, V, D.best_draft_length(a, V_hat))
                 >= D.bound_best_length(delta) * D.throughput(a, V, D.best_draft_length(a, V))
                 for a in grid)
    at = {}
    for a in (0.5, 0.6, 0.7, 0.8, 0.9):
        k = D.best_draft_length(a, V)
        at[str(a)] = {"k_star": k, "speedup": round(D.speedup(a, V, k), 3),
                      "moesd_speedup": round(D.moesd_speedup(D.expected_tokens(a, k), k,
                                                             args.t_draft, t_med), 3)}
    print(json.dumps({
        "stack_config": cfg.name, "layers": L, "windows": W, "t_draft_us": args.t_draft,
        "hidden": cfg.hidden, "rho": args.rho if args.rho is not None else cfg.rho,
        "sigma": args.sigma if args.sigma is not None else cfg.sigma,
        "per_K": [{"K": K, "us_stack": round(t_med[K], 1), "u_bar": round(u_mean[K], 2),
                   "us_per_layer": round(t_med[K] / L, 1)} for K in range(Kmax + 1)],
        "cost_model_per_m": {str(m): {"alpha_us": round(f["alpha"], 3),
                                      "beta0_us": round(f["beta0"], 1),
                                      "r2": None if f["r2"] != f["r2"] else round(f["r2"], 3)}
                             for m, f in per_m.items()},
        "cost_model_pooled": {"alpha_us": round(pooled["alpha"], 3),
                              "beta0_us": round(pooled["beta0"], 1),
                              "r2": round(pooled["r2"], 4)},
        "a0": round(D.a0(V), 4),
        "staircase": [[round(a_, 4), k] for a_, k in D.staircase(V)],
        "best_at": at,
        "calibrated": {"delta": round(delta, 4),
                       "k_star_agrees": f"{agree} of {len(grid)} acceptance values",
                       "inside_bound_20": f"{inside} of {len(grid)}"},
        "timing": "graph replay of the whole stack, median of 3 after one warm replay; the "
                  "stack's expert bytes exceed L2"}))


# ------------------------------------------------------------- cpu / oracle

def host_info():
    """The host's CPU model and core count (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"host_cores": os.cpu_count() or 1, "cpu_model": model or "unknown",
            "machine": os.uname().machine}


def oracle_inputs(layer, h, cfg=None):
    import numpy as np
    import oracle
    cfg = cfg or CFG
    cpu = layer.to("cpu")

    def nb(t):
        if t is None:
            return None
        t = t.contiguous()
        return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()
    ot = {synth.F32: oracle.F32, synth.BF16: oracle.BF16, synth.E4M3: oracle.E4M3}
    og = {synth.GATE_SOFTMAX: oracle.GATE_SOFTMAX,
          synth.GATE_SOFTMAX_RENORM: oracle.GATE_SOFTMAX_RENORM,
          synth.GATE_SIGMOID_RENORM: oracle.GATE_SIGMOID_RENORM}
    L = oracle.Layer(cfg.d, cfg.n_experts, cfg.top_k, cfg.inter, ot[cfg.act], ot[cfg.wtype],
                     og[cfg.gate], nb(cpu.wg), nb(cpu.w13), nb(cpu.w2), nb(cpu.s13),
                     nb(cpu.s2), nb(cpu.sh_w13), nb(cpu.sh_w2), nb(cpu.sh_s13), nb(cpu.sh_s2))
    return oracle, L, nb(h.cpu())


def oracle_pass_times(cfg, layer, h_all, ns, reps=1):
    """The oracle, as it stands, on the same seeded inputs: for each n, one
    whole n-token pass with its tokens split over all host cores (the oracle
    runs one token per thread, so it uses min(cores, n) threads), and the
    single-thread time of a pass, taken as n x one token's single-thread time
    (every token does the same work: all N router scores and k (+ shared)
    SwiGLU experts)."""
    oracle, L, hb = oracle_inputs(layer, h_all[:max(ns)].contiguous(), cfg)
    cores = os.cpu_count() or 1
    t1 = []
    for _ in range(3):
        t0 = time.perf_counter()
        oracle.verify(L, hb, tokens=[0], threads=1)
        t1.append(time.perf_counter() - t0)
    tok = statistics.median(t1)
    per_n = {}
    for n in ns:
        ts = []
        for _ in range(reps):
            t0 = time.perf_counter()
            oracle.verify(L, hb, tokens=list(range(n)), threads=cores)
            ts.append(time.perf_counter() - t0)
        per_n[n] = {"ms_all_cores": round(1e3 * statistics.median(ts), 1),
                    "threads": min(cores, n), "ms_1_thread": round(1e3 * n * tok, 1)}
    return {"per_n": per_n,
            "host": {**host_info(), "ms_1_thread_per_token": round(1e3 * tok, 1),
                     "method": "all cores: the pass itself, tokens split over threads; "
                               "1 thread: n x one token (median of 3)"}}


def cpu_baseline(layer, h, union_bytes, reps=3):
    """The oracle, as it stands, on the host cores: the whole n-token pass
    with its tokens split over threads (min(cores, n) threads), and the
    single-thread time of the same pass (n x one token's time)."""
    oracle, L, hb = oracle_inputs(layer, h)
    cores = os.cpu_count() or 1
    threads = min(cores, N_TOKENS)
    ts = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.verify(L, hb, threads=cores)
        ts.append(time.perf_counter() - t0)
    t = statistics.median(ts)
    t1 = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.verify(L, hb, tokens=[0], threads=1)
        t1.append(time.perf_counter() - t0)
    t_one = N_TOKENS * statistics.median(t1)
    host = host_info()
    return {"value": round(union_bytes / t / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle", **host,
            "sample": f"the whole {N_TOKENS}-token pass (fp64 per-token loop, one token per "
                      f"thread: {threads} threads on {host['host_cores']} cores), median of "
                      f"{reps}: {t:.2f} s per pass",
            "single_thread": {"value": round(union_bytes / t_one / 1e9, 4), "unit": "GB/s",
                              "s_per_pass": round(t_one, 2),
                              "sample": f"one token on one thread, median of {reps}, x "
                                        f"{N_TOKENS} tokens (each token does the same work)"}}


# ---------------------------------------------------------------- reference

def run_reference(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    device = "cuda" if torch.cuda.is_available() else "cpu"
    layer, h_all = make_workload(device)
    h = h_all[:N_TOKENS].contiguous()
    oracle, L, hb = oracle_inputs(layer, h)
    cores = os.cpu_count() or 1
    # union bytes of the pass, from the oracle's own routing
    hv = h.double().cpu().numpy()
    U = len({int(e) for t in range(N_TOKENS)
             for e in oracle.topk(oracle.router_scores(L, hv[t]), CFG.top_k)})
    wb, sb = oracle.expert_bytes(CFG.d, CFG.inter, oracle.E4M3)
    union_bytes = (U + CFG.n_shared) * (wb + sb)
    for _ in range(min(args.warmup, 1)):
        oracle.verify(L, hb, tokens=[0], threads=1)
    ts = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.verify(L, hb, threads=cores)
        ts.append(time.perf_counter() - t0)
    t = sum(ts) / len(ts)
    value = union_bytes / t / 1e9
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(1e3 * t, 1), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeds as ours)",
           "config": bench_config(U, union_bytes, ws),
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": min(cores, N_TOKENS),
                            "kind": "oracle", **host_info(),
                            "sample": f"the whole {N_TOKENS}-token pass per step, one token per "
                                      f"thread ({min(cores, N_TOKENS)} threads)"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def main():
    global CFG, WORKLOAD
    args = parse()
    if args.experts:
        from dataclasses import replace
        CFG = replace(CFG, n_experts=args.experts)
        WORKLOAD += f" ({args.experts} routed experts: profiling case)"
    if args.fit_config:
        run_fit(args)
    elif args.budget_config:
        run_budget(args)
    elif args.select_config:
        run_select(args)
    elif args.stack_config:
        run_stack(args)
    elif args.sweep_config:
        run_sweep_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
