"""Layer fwd+bwd throughput of the dropless MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixtral]
                    [--impl ours|reference] [--no-cpu-baseline]
    python bench.py --dispatch-ablation

One step = route + dispatch index + forward + backward of one layer over one
batch of synthetic, seeded inputs (all through the C ABI). Prints one JSON line
on rank 0. With N > 1 (torchrun), every rank runs an independent replica on its
own GPU (the layer has no exchange step), so scaling is weak.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from token_dispatch_grouped_gb300 import inputs as I  # noqa: E402

METRIC = "MoE layer fwd+bwd tokens/s and % of BF16 tensor peak on 1 GB300; peak act bytes"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")

# Algorithmic FLOPs per step of each kernel family, in units of TK*d*h
# (SwiGLU expert GEMMs: 18 TK d h in total; SonicMoE 3.4.5 counts (6 + 12) d n
# per token-expert). Non-gated experts have no W3: 12 TK d h in total.
GEMM_FLOP_UNITS = {"g1_up_swiglu": 4, "g2_down": 2, "g3_dh": 2, "g4_dw2": 2, "g5_dw13": 4,
                   "g6_dx": 4}
GEMM_FLOP_UNITS_NON_GATED = {"g1_up_act": 2, "g2_down": 2, "g3_dh_act": 2, "g4_dw2": 2,
                             "g5_dw13": 2, "g6_dx": 2}


def gemm_flop_units(s) -> dict:
    return GEMM_FLOP_UNITS if s.gated else GEMM_FLOP_UNITS_NON_GATED


def flops_per_step(s, rows=None) -> float:
    """Algorithmic FLOPs of one step; rows = routed rows (T*K for top-K routing)."""
    rows = s.T * s.K if rows is None else rows
    return sum(gemm_flop_units(s).values()) * rows * s.d * s.h + 6.0 * s.T * s.d * s.E


def memory_kernel_bytes(s) -> dict:
    """Algorithmic bytes per step of the memory-bound kernels: each operand read
    once and each result written once (the per-kernel byte table of the design
    notes). Kernel names are the launch names; D1-D3 count together."""
    T, d, E, K = s.T, s.d, s.E, s.K
    TK = T * K
    return {
        # the tensor-core router's split of W_g into bf16 parts counts with it
        "router": (("router", "router_wsplit"), T * d * 2 + E * d * 4 + TK * 8 + T * E * 4),
        "dispatch": (("dispatch_single", "dispatch_hist", "dispatch_scan", "dispatch_scatter"),
                     2 * TK * 4 + 2 * TK * 4 + (E + 1) * 4),
        "combine": (("combine",), TK * d * 2 + TK * 8 + T * d * 2),
        "dx_combine": (("dx_combine",), TK * d * 2 + TK * 8 + T * d * 2),
        # router weight gradient: x read once, dz and the row lists, dW_g written
        "router_dwg": (("router_dwg", "router_dwg_zero", "router_dwg_scatter", "router_dwg_mma",
                        "router_dwg_reduce"), T * d * 2 + TK * 12 + E * d * 4),
    }


def routing_stats(counts) -> dict:
    """Per-expert row counts of a routing: their spread, the empty experts, and the
    256-row M tiles that a CTA-pair GEMM over these rows runs against the tiles the
    same rows would fill if packed (the partial-tile cost of the row-tiled GEMMs).
    mma_rows_issued counts the rows the row-tiled GEMMs multiply in CTA-pair mode:
    whole 256-row tiles, a last partial tile above 128 rows as 256, and one of
    1..128 rows as a 128-row single-CTA tile; mma_rows_pairs_only is the same with
    every partial tile at 256 rows."""
    c = counts.to(torch.int64)
    rows = int(c.sum())
    rem = c % 256
    issued = (c // 256) * 256 + torch.where(rem > 128, 256, torch.where(rem > 0, 128, 0))
    return {"min_rows": int(c.min()), "max_rows": int(c.max()),
            "empty_experts": int((c == 0).sum()),
            "cv": float(c.float().std() / c.float().mean()),
            "m_tiles_256": int(((c + 255) // 256).sum()),
            "m_tiles_256_packed": (rows + 255) // 256,
            "routed_rows": rows,
            "mma_rows_issued": int(issued.sum()),
            "mma_rows_pairs_only": int(((c + 255) // 256 * 256).sum())}


PEAK_RULE = ("the burst bf16 peak applies when the timed region is shorter than 1 s or its "
             "median SM clock is within 3% of the maximum; otherwise the sustained peak")


def choose_bf16_peak(peaks: dict, timed_ms: float, clk: dict) -> tuple[float, str]:
    """The measured bf16 peak that a timed region is compared against: the burst
    figure for a short region or one that ran at full clock, the sustained
    figure (a seconds-long loop under the power cap) otherwise."""
    sm, smax = clk.get("sm_mhz"), clk.get("sm_max_mhz")
    at_max = sm is not None and smax is not None and sm >= 0.97 * smax
    if timed_ms < 1000.0 or at_max:
        return peaks["bf16"], "burst"
    return peaks["bf16_sus"], "sustained"


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return dict(hbm=p.get("hbm_gbs"), bf16=p.get("bf16_tflops"),
                    bf16_sus=p.get("bf16_tflops_sustained"), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------ distributed
def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world <= 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons; start() before the
    warm-up, mark() around the timed region, stop() keeps the samples taken
    inside the marked window (at least the one nearest to it)."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.win = [None, None]
        self.t_start = time.time()
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(dev_index), f"--query-gpu=timestamp,{self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def mark(self, i: int):
        self.win[i] = time.time()

    def stop(self) -> dict:
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.p.terminate()
        self.p.wait(timeout=10)
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        import datetime
        samples = []
        for r in rows:
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(r[1]), float(r[2]), [v.strip().lower() for v in r[4:8]]))
            except (ValueError, IndexError):
                continue
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        a, b = self.win
        inside = [x for x in samples if a is not None and a <= x[0] <= b]
        if not inside:  # window shorter than the sampling period: nearest sample
            mid = 0.5 * (a + b) if a is not None else samples[-1][0]
            inside = [min(samples, key=lambda x: abs(x[0] - mid))]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for x in inside for n, v in zip(names, x[3]) if v == "active"})
        return {"sm_mhz": statistics.median(x[1] for x in inside),
                "sm_max_mhz": max(x[2] for x in inside), "reasons": reasons,
                "samples": len(inside)}


# ------------------------------------------------------------------ oracle (CPU baseline)
def cpu_oracle_sample(s, inp, tokens: int) -> tuple[float, int]:
    """Times the CPU oracle (as it stands) on the first `tokens` tokens of the
    workload: route, dispatch, forward and backward. Returns (seconds, tokens)."""
    from oracle import moe_oracle as O
    sl = slice(0, tokens)
    t0 = time.perf_counter()
    O.layer_step(inp["x"][sl], inp["Wg"], inp["W1"], inp["W3"], inp["W2"], inp["dO"][sl], s.K,
                 inp.get("bias"), s.expert)
    return time.perf_counter() - t0, tokens


def cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def run_reference(args, s, name):
    """The oracle as the reference arm: each step is a bounded sample."""
    rank, world, _ = dist_setup(args.gpus)
    if rank != 0:
        return
    inp = I.make_layer_inputs(s, seed=0, with_bias=(name == "skew"))
    tok = args.ref_tokens
    for _ in range(args.warmup):
        cpu_oracle_sample(s, inp, tok)
    secs = 0.0
    for _ in range(args.steps):
        dt, _ = cpu_oracle_sample(s, inp, tok)
        secs += dt
    v = tok * args.steps / secs
    line = dict(metric=METRIC, value=v, unit="tokens/s", n_gpus=args.gpus, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * secs / args.steps, higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic", impl="reference",
                config=workload_config(s, name),
                cpu_baseline=dict(value=v, unit="tokens/s", cores=cores(), kind="oracle",
                                  sample=f"first {tok} tokens of the workload per step"),
                e2e=dict(value=v, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


def workload_config(s, name):
    return {"workload": f"{name}: T={s.T} d={s.d} E={s.E} K={s.K} h={s.h} expert={s.expert}",
            "T": s.T, "d": s.d, "E": s.E, "K": s.K, "h": s.h, "expert": s.expert,
            "global_batch_tokens": s.T,
            "l2": "working set > L2 (expert weights alone exceed 129 MB and are streamed every step)"}


# ------------------------------------------------------------------ dispatch ablation
def sort_dispatch(ids: torch.Tensor, E: int):
    """Sort-based dispatch index on the GPU with library kernels (torch's stable
    radix sort, a binary search for the offsets, a scatter for the inverse):
    the baseline the atomic-free build is compared with. Same outputs:
    expert_token_indices, expert_token_offsets, token_index_map (int32)."""
    T, K = ids.shape
    flat = ids.reshape(-1)
    keys, perm = torch.sort(flat, stable=True)
    eti = torch.div(perm, K, rounding_mode="floor").to(torch.int32)
    bounds = torch.arange(E + 1, device=ids.device, dtype=keys.dtype)
    offsets = torch.searchsorted(keys, bounds).to(torch.int32)
    tim = torch.empty_like(flat)
    tim[perm] = torch.arange(flat.numel(), device=ids.device, dtype=torch.int32)
    return eti, offsets, tim


def _graph_us(fn, reps: int) -> tuple[float, float]:
    """(CUDA-graph replay, eager) microseconds per call of fn, back to back."""
    st = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(reps):
        fn()
    b.record(st)
    torch.cuda.synchronize()
    eager = a.elapsed_time(b) * 1e3 / reps
    side = torch.cuda.Stream()
    side.wait_stream(st)
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    st.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a.record(st)
    g.replay()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / reps, eager


def run_dispatch_ablation(args):
    """The atomic-free dispatch build (D1-D3, one C-ABI call) against the
    sort-based baseline across token counts, expert counts, K and skew. One
    JSON line per case; both outputs are checked equal first."""
    from token_dispatch_grouped_gb300 import binding as B
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    peaks = load_peaks()
    for T in (4096, 32768, 262144):
        for E, K in ((8, 2), (64, 6), (128, 8)):
            for skew in (0.0, 1.2):
                ids = I.random_ids_gumbel(T, E, K, seed=T + E, skew=skew).to(dev)
                s = B.shape(T, 128, E, K, 128)
                ws = torch.empty(max(B.moe_workspace_size(s, B.MOE_WS_DISPATCH), 256),
                                 dtype=torch.uint8, device=dev)
                TK = T * K
                eti = torch.empty(TK, dtype=torch.int32, device=dev)
                off = torch.empty(E + 1, dtype=torch.int32, device=dev)
                tim = torch.empty(TK, dtype=torch.int32, device=dev)

                def ours():
                    B.moe_build_dispatch(s, ids, eti, off, tim, ws)

                def base():
                    return sort_dispatch(ids, E)

                ours()
                ref = base()
                torch.cuda.synchronize()
                same = (torch.equal(eti, ref[0]) and torch.equal(off, ref[1])
                        and torch.equal(tim, ref[2]))
                if B.moe_get_error() != B.MOE_OK or not same:
                    raise SystemExit(f"dispatch ablation: outputs differ at T={T} E={E} K={K}")
                g_ours, e_ours = _graph_us(ours, 20)
                g_sort, e_sort = _graph_us(base, 20)
                nbytes = 2 * TK * 4 + 2 * TK * 4 + (E + 1) * 4  # ids read twice, two maps written
                line = {"ablation": "dispatch_index", "T": T, "E": E, "K": K, "skew": skew,
                        "ours_us": g_ours, "sort_us": g_sort, "speedup": g_sort / g_ours,
                        "ours_eager_us": e_ours, "sort_eager_us": e_sort,
                        "ours_hbm_frac": nbytes / (g_ours * 1e-6) / 1e9 / peaks["hbm"],
                        "timing": "CUDA graph of 20 back-to-back calls; eager alongside",
                        "outputs_equal": True}
                print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="mixtral", choices=sorted(I.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-tokens", type=int, default=0, help="oracle sample size (0 = auto)")
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--combine", default="chunked", choices=["chunked", "slotwise"],
                    help="forward combine: chunked expert-output passes (moe_forward) or "
                         "fused into the down projection slot by slot (moe_forward_slotwise)")
    ap.add_argument("--routing", default="tc", choices=["tc", "tr"],
                    help="tc: top-K token choice; tr: token rounding of it (NR-f, --m-tile) "
                         "and the layer on the rounded rows")
    ap.add_argument("--m-tile", type=int, default=128)
    ap.add_argument("--dispatch-ablation", action="store_true",
                    help="time the dispatch build against a sort-based baseline and exit")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.dispatch_ablation:
        run_dispatch_ablation(args)
        return
    name = args.workload
    s = I.WORKLOADS[name]
    if args.impl == "reference":
        run_reference(args, s, name)
        return

    from token_dispatch_grouped_gb300 import binding as B
    from token_dispatch_grouped_gb300.layer import MoELayer, Routing

    rank, world, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = load_peaks()

    inp = I.make_layer_inputs(s, seed=0, with_bias=(name == "skew"))
    dv = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    L = MoELayer(s.T, s.d, s.E, s.K, s.h, device=dev, expert=s.expert)
    TK = s.T * s.K
    # Preallocated outputs (gradients are written, not accumulated).
    logits = torch.empty(s.T, s.E, dtype=torch.float32, device=dev)
    r = Routing(logits, torch.empty(s.T, s.K, dtype=torch.int32, device=dev),
                torch.empty(s.T, s.K, dtype=torch.float32, device=dev))
    from token_dispatch_grouped_gb300.layer import Dispatch
    dp = Dispatch(torch.empty(TK, dtype=torch.int32, device=dev),
                  torch.empty(s.E + 1, dtype=torch.int32, device=dev),
                  torch.empty(TK, dtype=torch.int32, device=dev))
    y = torch.empty(s.T, s.d, dtype=torch.bfloat16, device=dev)
    H = torch.empty(TK, L.hs, dtype=torch.bfloat16, device=dev)
    grads = L.alloc_grads()
    bias = dv["bias"]
    st = torch.cuda.current_stream(dev)

    fwd = B.moe_forward_slotwise if args.combine == "slotwise" else B.moe_forward

    def step(x, dy, y=y, dx=grads["dx"]):
        B.moe_route(L.s, x, dv["Wg"], bias, r.logits, r.ids, r.w, L.ws)
        B.moe_build_dispatch(L.s, r.ids, dp.eti, dp.offsets, dp.tim, L.ws)
        fwd(L.s, x, dv["W1"], dv["W3"], dv["W2"], r.ids, r.w, dp.eti, dp.offsets, dp.tim, y, H,
            L.ws)
        B.moe_backward(L.s, dy, x, dv["Wg"], dv["W1"], dv["W3"], dv["W2"], r.ids, r.w, dp.eti,
                       dp.offsets, dp.tim, H, dx, grads["dWg"], grads["dW1"],
                       grads["dW3"], grads["dW2"], grads["dS"], L.ws)

    rows_of_step = None
    if args.routing == "tr":
        # Token rounding of the top-K routing, then the layer on the rounded rows.
        from token_dispatch_grouped_gb300.layer import RowRouting
        m = args.m_tile
        cap = B.moe_rows_capacity(L.s, m)
        i32 = dict(dtype=torch.int32, device=dev)
        rr = RowRouting(cap, torch.empty(cap, **i32), torch.empty(s.E + 1, **i32),
                        torch.empty(cap, dtype=torch.float32, device=dev),
                        torch.empty(s.T + 1, **i32), torch.empty(cap, **i32),
                        torch.empty(cap, **i32))
        tr_ws = torch.empty(max(B.moe_token_rounding_workspace_size(L.s, m), 256),
                            dtype=torch.uint8, device=dev)
        rows_ws = torch.empty(max(B.moe_workspace_size_rows(L.s, cap, B.MOE_WS_FORWARD),
                                  B.moe_workspace_size_rows(L.s, cap, B.MOE_WS_BACKWARD)),
                              dtype=torch.uint8, device=dev)
        H = torch.empty(cap, L.hs, dtype=torch.bfloat16, device=dev)
        dS_row = torch.empty(cap, dtype=torch.float32, device=dev)

        def step(x, dy, y=y, dx=grads["dx"]):  # noqa: F811
            B.moe_route(L.s, x, dv["Wg"], bias, r.logits, r.ids, r.w, L.ws)
            B.moe_build_dispatch(L.s, r.ids, dp.eti, dp.offsets, dp.tim, L.ws)
            B.moe_token_rounding(L.s, m, r.logits, r.ids, dp.eti, dp.offsets, rr.eti, rr.offsets,
                                 rr.w_row, rr.tok_off, rr.tok_exp, rr.tok_rows, tr_ws)
            B.moe_forward_rows(L.s, cap, x, dv["W1"], dv["W3"], dv["W2"], rr.eti, rr.offsets,
                               rr.w_row, rr.tok_off, rr.tok_exp, rr.tok_rows, y, H, rows_ws)
            B.moe_backward_rows(L.s, cap, dy, x, dv["Wg"], dv["W1"], dv["W3"], dv["W2"], rr.eti,
                                rr.offsets, rr.w_row, rr.tok_off, rr.tok_exp, rr.tok_rows, H,
                                dx, grads["dWg"], grads["dW1"], grads["dW3"],
                                grads["dW2"], dS_row, rows_ws)

    # ---- memory: activation bytes of one fwd+bwd beyond inputs/weights/grads/outputs
    torch.cuda.synchronize(dev)
    base_alloc = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    step(dv["x"], dv["dO"])
    L.check_error()
    torch.cuda.synchronize(dev)
    routed_bytes = s.T * s.K * s.d * 2
    ws_f = B.moe_workspace_size(L.s, B.MOE_WS_FORWARD_SLOTWISE if args.combine == "slotwise"
                                else B.MOE_WS_FORWARD)
    ws_b = B.moe_workspace_size(L.s, B.MOE_WS_BACKWARD)
    saved = H.numel() * 2 + 3 * TK * 4 + (s.E + 1) * 4 + 2 * TK * 4
    memory = {"routed_buffer_bytes_not_allocated": routed_bytes,
              "saved_for_backward_bytes": saved,
              "saved_over_routed": saved / routed_bytes,
              "workspace_fwd_bytes": ws_f, "workspace_bwd_bytes": ws_b,
              "peak_activation_bytes": saved + max(ws_f, ws_b),
              "peak_activation_bytes_kind": "computed from the layout: saved tensors plus the "
                                            "larger workspace (all buffers are preallocated)",
              "peak_activation_over_routed": (saved + max(ws_f, ws_b)) / routed_bytes,
              # the down-projection chunk buffer (plus the segment table): the
              # forward workspace beyond the [rows, h] SwiGLU output
              "fwd_workspace_beyond_swiglu_output_bytes": ws_f - TK * s.h * 2,
              "allocator_peak_delta_bytes": torch.cuda.max_memory_allocated(dev) - base_alloc}

    # ---- device-resident timing
    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        step(dv["x"], dv["dO"])
    torch.cuda.synchronize(dev)
    L.check_error()
    launches0 = B.moe_launch_count()
    barrier(world)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    clocks.mark(0)
    e0.record(st)
    for _ in range(args.steps):
        step(dv["x"], dv["dO"])
    e1.record(st)
    torch.cuda.synchronize(dev)
    clocks.mark(1)
    barrier(world)
    ms = e0.elapsed_time(e1)
    launches = B.moe_launch_count() - launches0
    clk = clocks.stop()
    L.check_error()
    # Per-kernel breakdown in a separate pass of the same steps: two CUDA events
    # around every launch (recorded on its stream), so the timed pass above
    # carries no per-launch instrumentation.
    B.moe_timing_enable(True)
    for _ in range(args.steps):
        step(dv["x"], dv["dO"])
    torch.cuda.synchronize(dev)
    per_kernel = B.moe_timing_collect()
    B.moe_timing_enable(False)
    L.check_error()
    ms = max_over_ranks(ms, world)
    ms_step = ms / args.steps
    bf16_peak, peak_kind = choose_bf16_peak(peaks, ms, clk)
    value = world * s.T * args.steps / (ms / 1e3)
    if args.routing == "tr":
        rows_of_step = int(rr.offsets[-1].item())
    tflops = flops_per_step(s, rows_of_step) / (ms_step / 1e3) / 1e12

    # ---- roofline of the dominant kernel (event-timed over the timed region)
    top = max(per_kernel.items(), key=lambda kv: kv[1][1])
    kname, (klaunches, kms) = top
    roof = None
    units = gemm_flop_units(s)
    if kname in units:
        per_launch_flop = (units[kname] * (rows_of_step or TK) * s.d * s.h * args.steps
                           / klaunches)
        achieved = per_launch_flop / (kms / klaunches / 1e3) / 1e12
        peak = bf16_peak
        traffic = None
        traffic_note = "no capture of the current GEMM sources"
        if os.path.exists(PROFILE_TRAFFIC):
            with open(PROFILE_TRAFFIC) as f:
                tr = json.load(f)
            ent = tr.get(f"{kname}@{name}")
            if ent and ent.get("source_hash") == source_hash():
                traffic = ent["dram_bytes_per_launch"]
                traffic_note = ent.get("note", "profiles/traffic.json")
        roof = {"kernel": kname, "bound": "tensor", "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "frac_burst": achieved / peaks["bf16"],
                "frac_sustained": achieved / peaks["bf16_sus"],
                "peak_source": f"{peaks['src']} bf16 {peak_kind}", "peak_rule": PEAK_RULE,
                "traffic_source": traffic_note}
    kernels = {k: {"launches": n, "ms_per_step": t / args.steps} for k, (n, t) in per_kernel.items()}
    # HBM-bound kernels: algorithmic bytes / event-timed duration vs the measured copy peak
    memory_bound = {}
    for mk, (names, nbytes) in memory_kernel_bytes(s).items():
        ms_k = sum(per_kernel[n][1] for n in names if n in per_kernel) / args.steps
        if ms_k > 0:
            gbs = nbytes / (ms_k / 1e3) / 1e9
            memory_bound[mk] = {"bytes_per_step": nbytes, "ms_per_step": ms_k,
                                "achieved_gbs": gbs, "frac_of_hbm": gbs / peaks["hbm"],
                                "launches_per_step": sum(per_kernel[n][0] for n in names
                                                         if n in per_kernel) / args.steps}

    # ---- end to end: host buffers in, results out, through the same C ABI calls.
    # Every step copies its inputs from pinned host memory and its results back;
    # the copies run on two copy streams with double-buffered device inputs and
    # outputs, so step i+1's upload and step i's download overlap step i's (and
    # i+1's) compute, as an input pipeline would. The region is timed from an
    # event before the first upload to one after the last download.
    xh = inp["x"].pin_memory()
    dyh = inp["dO"].pin_memory()
    yh = [torch.empty(s.T, s.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dxh = [torch.empty(s.T, s.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(dv["x"]) for _ in range(2)]
    dyd = [torch.empty_like(dv["dO"]) for _ in range(2)]
    yd = [y, torch.empty_like(y)]
    dxd = [grads["dx"], torch.empty_like(grads["dx"])]
    up = torch.cuda.Stream(dev)
    down = torch.cuda.Stream(dev)

    def ev():
        return torch.cuda.Event()

    def e2e_run(n):
        in_ready = [None, None]
        in_free = [None, None]   # the step that read buffer b finished
        out_ready = [None, None]
        out_free = [None, None]  # the download of buffer b finished

        def upload(i):
            b = i % 2
            with torch.cuda.stream(up):
                if in_free[b] is not None:
                    up.wait_event(in_free[b])
                xd[b].copy_(xh, non_blocking=True)
                dyd[b].copy_(dyh, non_blocking=True)
                in_ready[b] = ev()
                in_ready[b].record(up)

        upload(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                upload(i + 1)
            st.wait_event(in_ready[b])
            if out_free[b] is not None:
                st.wait_event(out_free[b])
            step(xd[b], dyd[b], yd[b], dxd[b])
            in_free[b] = ev()
            in_free[b].record(st)
            out_ready[b] = in_free[b]
            with torch.cuda.stream(down):
                down.wait_event(out_ready[b])
                yh[i % 2].copy_(yd[b], non_blocking=True)
                dxh[i % 2].copy_(dxd[b], non_blocking=True)
                out_free[b] = ev()
                out_free[b].record(down)
        for e in out_free:
            if e is not None:
                st.wait_event(e)

    e2e_run(args.warmup)
    torch.cuda.synchronize(dev)
    barrier(world)
    up.wait_stream(st)
    down.wait_stream(st)
    e0.record(st)
    up.wait_event(e0)
    e2e_run(args.steps)
    e1.record(st)
    torch.cuda.synchronize(dev)
    barrier(world)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1), world)
    # The last step's downloaded results are the device results.
    last = (args.steps - 1) % 2
    if not (torch.equal(yh[last], yd[last].cpu()) and torch.equal(dxh[last], dxd[last].cpu())):
        raise RuntimeError("end-to-end results differ from the device buffers")
    e2e = {"value": world * s.T * args.steps / (ms_e2e / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": xh.numel() * 2 + dyh.numel() * 2,
           "d2h_bytes_per_step": yh[0].numel() * 2 + dxh[0].numel() * 2,
           "copies": "two copy streams, double-buffered inputs and outputs"}
    L.check_error()

    # ---- routing statistics
    routing = routing_stats((dp.offsets[1:] - dp.offsets[:-1]).cpu())

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok = args.cpu_tokens or max(8, min(s.T, 256 if s.d * s.h < 2 ** 26 else 64))
        dt, n = cpu_oracle_sample(s, inp, tok)
        cpu_base = {"value": n / dt, "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                    "sample": f"first {n} tokens of the {name} workload, one fwd+bwd, "
                              f"{dt:.1f} s (numpy float64, BLAS threads = all host cores)"}

    if rank == 0:
        line = dict(metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
                    warmup=args.warmup, ms_per_step=ms_step, higher_is_better=True,
                    scaling="weak", vs_baseline=None, dtype="bf16", data="synthetic",
                    config=dict(workload_config(s, name), combine=args.combine,
                                routing=args.routing,
                                **({"m_tile": args.m_tile, "rows": rows_of_step}
                                   if args.routing == "tr" else {})),
                    tflops=tflops,
                    frac_of_bf16_peak=tflops / bf16_peak,
                    frac_of_bf16_burst=tflops / peaks["bf16"],
                    frac_of_bf16_sustained=tflops / peaks["bf16_sus"],
                    peak_note=(f"{peaks['src']} bf16 {peak_kind} {bf16_peak} TFLOP/s "
                               f"(burst {peaks['bf16']}, sustained {peaks['bf16_sus']}); "
                               + PEAK_RULE),
                    memory=memory, roofline=roof, kernels=kernels, memory_bound=memory_bound,
                    hbm_peak_gbs=peaks["hbm"], routing=routing,
                    cpu_baseline=cpu_base, e2e=e2e, gpu_launches=launches, clocks=clk)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def source_hash() -> str:
    """Hash of the sources that define the GEMM kernels and their launches (the
    kernels whose DRAM traffic profiles/traffic.json records)."""
    import hashlib
    h = hashlib.sha1()
    for f in ("api.cu", "common.cuh", "gemm.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "token_dispatch_grouped_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


if __name__ == "__main__":
    main()
