"""Benchmark: verified tree tokens/s of the target-verify round on GB300.

One step = one full verify round (tv_build_ancestor_mask, tv_branch_compress, tv_tree_verify_attn,
tv_accept_walk, tv_refresh_commit) over one batch of synthetic requests.  Default workload: the
serving batch -- 64 requests with ragged prefixes U{1024..8192}, C4 + C128 + 128-token window,
64 query heads sharing one KV head, head dim 512, bf16, top-2 draft trees pruned to D = 8.

value  = whole-job verified tree tokens per second (sum over ranks of B * D per step / max time).
e2e    = the same metric through the C ABI: every step uploads its inputs from pinned host memory
         (on a copy stream, one step ahead) and reads its acceptance results back to the host.
roofline, hbm = the attention kernel's algorithmic flops / bytes per launch over its CUDA-event
         duration, against the measured peaks.
cpu_baseline = the fp64 CPU oracle on a bounded sample of the same workload (rank 0, N = 1).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
       [--workload serving|small|long|tiny] [--no-cpu-baseline]
Multi-GPU: launched by torchrun, one rank per GPU; each rank verifies its own batch (requests are
independent: replicas with no data-path collective, weak scaling).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


# the headline metric (both arms report it; its value is the verified tree tokens per second)
METRIC = "verified tree tokens/s and achieved HBM GB/s (% of peak), D=8 bs=64, 1 GB300"

WORKLOAD_DESC = {
    "serving": "serving batch: B=64, L~U{1024..8192}, D=8 (top-2 tree, 4 steps), H=64x1, d=512, "
               "C4+C128+W128, bf16",
    "small": "small: B=4, L=4096, D=6 (top-2, depth 3), H=64x1, d=512, C4+C128+W128, bf16",
    "long": "long context: B=8, L~U{65536..131072}, C128 + top-2048 C4 (device indexer in the "
            "round), W128, D=8, H=64x1, "
            "d=512, bf16",
    "tiny": "tiny fp32: B=1, L=256, C4 only, remainder tail, D=5, H=8x1, d=64",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOAD_DESC), default="serving")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--attn-kernel", choices=["auto", "simt", "tcgen05"], default="auto")
    ap.add_argument("--batch", type=int, default=None,
                    help="requests per GPU (default: the workload's own batch)")
    ap.add_argument("--sets", type=int, default=3,
                    help="rotating state copies (3 keeps every step's inputs out of L2)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the five calls directly instead of replaying a captured round")
    ap.add_argument("--sweep", action="store_true",
                    help="the budget sweep instead of the bench line: D x batch x {chain, tree} x "
                         "child-match probability at prefix 4096, one JSON line per cell")
    ap.add_argument("--copy-streams", type=int, default=1,
                    help="copy streams for the end-to-end uploads")
    ap.add_argument("--page-tokens", type=int, default=0,
                    help="keep the persistent cache in page pools of this many tokens per page "
                         "(a multiple of 512; pages scattered over the pool); 0 = contiguous")
    ap.add_argument("--draft", action="store_true",
                    help="draft-side tree attention instead of the bench line: per draft step of "
                         "a width-2 beam tree (B=64, serving cache geometry), one JSON line")
    ap.add_argument("--cpu-baseline-only", action="store_true",
                    help="print the oracle's CPU figure for the workload and exit (no GPU)")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle work in the CPU figure")
    ap.add_argument("--stage-chain", type=int, choices=[0, 1], default=0,
                    help="1: the branch call stages the cached chain's raw rows and C4 entries "
                         "and the refresh skips them")
    ap.add_argument("--cells", type=str, default=None,
                    help="with --sweep: comma-separated cell indices (default: all 64)")
    return ap.parse_args()


def make_workload(name, rank, batch=None):
    from tree_speculative_verify_gb300 import workloads
    seed = rank
    if name == "serving":
        return workloads.serving(seed=seed, B=batch or 64)
    if name == "small":
        return workloads.small(seed=seed)
    if name == "long":
        return workloads.long_context(seed=seed)
    return workloads.tiny(seed=seed)


# ---- accounting (host-side, from the workload's integers) -------------------------------------

def visible_counts(wl):
    """Per request and node: how many entries the node attends to, and the tail entries and
    scratch rows the round reads.  Pure bookkeeping for the roofline numerators."""
    out = []
    for b in range(wl.B):
        L = int(wl.L[b])
        par = [int(x) for x in wl.parents[b]]
        depth = [0] * wl.D
        for v in range(1, wl.D):
            depth[v] = depth[par[v]] + 1
        n4 = (wl.n_sel if wl.n_sel else L // 4) if 4 in wl.ms else 0
        n128 = L // 128 if 128 in wl.ms else 0
        closes = {m: [(L + depth[v] + 1) % m == 0 for v in range(wl.D)] for m in wl.ms}
        n_scr = sum(sum(c) for c in closes.values())
        m_min = 4 if 4 in wl.ms else 128
        per_node = []
        for v in range(wl.D):
            p = L + depth[v]
            lo = max(0, p - wl.W) if wl.tail_mode == "window" else m_min * (p // m_min)
            anc = []
            u = v
            while True:
                anc.append(u)
                if u == 0:
                    break
                u = par[u]
            n_tree = sum(1 for u in anc if L + depth[u] >= lo)
            n_scr_v = sum(1 for m in wl.ms for u in anc if u != v and closes[m][u])
            per_node.append(n4 + n128 + max(0, L - lo) + n_tree + n_scr_v)
        tail = min(L, wl.W) if wl.tail_mode == "window" else L - m_min * (L // m_min)
        out.append(dict(shared=n4 + n128, tail=tail, tree=wl.D, scr=n_scr, per_node=per_node))
    return out


def attention_accounting(wl):
    es = 2 if wl.dtype == "bf16" else 4
    counts = visible_counts(wl)
    kv_bytes = sum((c["shared"] + c["tail"] + c["tree"] + c["scr"]) * 2 * wl.d * es for c in counts)
    qo_bytes = 2 * wl.B * wl.D * wl.H * wl.d * es
    flops = sum(4 * wl.d * wl.H * n for c in counts for n in c["per_node"])
    return kv_bytes, qo_bytes, flops


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=p["hbm_gbs"], tc=p["bf16_tflops"], tc_sus=p["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sus=1700.0, source="fallback")


ATTN_SOURCES = {
    "tcgen05": ["tv_attn_tc.cu", "tv_attn_tc.cuh", "tv_sm100.cuh", "tv_attn_common.cuh",
                "tv_common.cuh"],
    "simt": ["tv_attn_simt.cu", "tv_attn_common.cuh", "tv_common.cuh"],
}


def sources_digest(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "tree_speculative_verify_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(key):
    """DRAM bytes per launch from a committed ncu summary under profiles/ (a line
    ``bench-record: {json}``), valid only while the kernel's sources are the ones it measured."""
    import glob
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                if not line.startswith("bench-record: "):
                    continue
                rec = json.loads(line[len("bench-record: "):])
                if rec.get("key") != key:
                    continue
                try:
                    if sources_digest(rec["sources"]) != rec["sources_sha256_16"]:
                        return None
                except OSError:
                    return None
                return rec
    return None


# ---- clocks -----------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- distributed ------------------------------------------------------------------------------

def dist_setup(n_gpus, backend="nccl"):
    """Rank / world from the torchrun environment; one process group per job (NCCL on GPUs; gloo
    serves the CPU tests of the multi-rank path)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}: launch N>1 with torchrun")
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, B, D, ms):
    """Whole-job verified tree tokens/s: every rank verifies B requests of D nodes per step; the
    job's step time is the slowest rank's."""
    return world * B * D / (ms * 1e-3)


# ---- the CPU oracle (baseline / reference arm) ------------------------------------------------

def oracle_setup(wl, requests):
    """Oracle-made compressed prefix of the sampled requests (state preparation, not timed)."""
    import oracle
    comp = {}
    for m in wl.ms:
        cap = wl.cap4 if m == 4 else wl.cap128
        CK = np.zeros((wl.B, cap, wl.d), dtype=np.float32)
        CV = np.zeros((wl.B, cap, wl.d), dtype=np.float32)
        for b in requests:
            L = int(wl.L[b])
            ck, cv = oracle.compress_prefix(wl.rawK[b, :L].float().numpy(),
                                            wl.rawV[b, :L].float().numpy(), L, m,
                                            wl.g[m].float().numpy(), wl.dtype)
            CK[b, :L // m], CV[b, :L // m] = ck, cv
        comp[m] = (CK, CV)
    return comp


class _Rows:
    def __init__(self, t):
        self.t = t

    def __getitem__(self, b):
        return self.t[b].float().numpy()


def oracle_round(wl, comp, requests):
    import oracle
    cfg = oracle.VerifyConfig(H=wl.H, d=wl.d, ms=wl.ms, W=wl.W, tail_mode=wl.tail_mode,
                              store=wl.dtype)
    g = {m: wl.g[m].float().numpy() for m in wl.ms}
    return oracle.verify_round(cfg, wl.parents, wl.L, _Rows(wl.Q), comp, wl.sel, _Rows(wl.rawK),
                               _Rows(wl.rawV), _Rows(wl.treeK), _Rows(wl.treeV), g, wl.draft,
                               wl.target, requests=requests)


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except ImportError:
        pass
    return os.cpu_count()


def cpu_model():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def cpu_baseline_single_thread(args, budget_s=8.0):
    """The same oracle sample with every BLAS / OpenMP pool limited to one thread (a child process,
    since the limits must be set before numpy loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only", "--workload",
           args.workload, "--cpu-budget", str(budget_s)]
    if args.batch:
        cmd += ["--batch", str(args.batch)]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=600)
        return json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None


def cpu_baseline(wl, budget_s=20.0):
    """Time the oracle's verify round on requests 0, 1, ... until ~budget_s of CPU work."""
    order = list(range(wl.B))
    comp = oracle_setup(wl, order)
    done, t_total = [], 0.0
    for b in order:
        t0 = time.perf_counter()
        oracle_round(wl, comp, [b])
        t_total += time.perf_counter() - t0
        done.append(b)
        if t_total >= budget_s:
            break
    value = len(done) * wl.D / t_total
    return {"value": value, "unit": "verified tree tokens/s", "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"fp64 numpy oracle, one verify round of {len(done)} of the {wl.B} requests "
                      f"(same workload, same seed), {t_total:.1f} s"}


def run_reference(args, world, rank):
    from tree_speculative_verify_gb300 import workloads  # noqa: F401  (inputs only)
    if rank != 0:
        return
    wl = make_workload(args.workload, 0)
    per_step = max(1, min(wl.B, 4))
    reqs = [list(range(i * per_step % wl.B, i * per_step % wl.B + per_step)) for i in range(
        args.warmup + args.steps)]
    reqs = [[b % wl.B for b in r] for r in reqs]
    comp = oracle_setup(wl, sorted({b for r in reqs for b in r}))
    for i in range(args.warmup):
        oracle_round(wl, comp, reqs[i])
    t0 = time.perf_counter()
    tokens = 0
    for i in range(args.steps):
        r = reqs[args.warmup + i]
        oracle_round(wl, comp, r)
        tokens += len(r) * wl.D
    dt = time.perf_counter() - t0
    value = tokens / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "verified tree tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "B_per_gpu": wl.B, "D": wl.D,
                   "H": wl.H, "d": wl.d, "sample_per_step": f"{per_step} of the {wl.B} requests"},
        "cpu_baseline": {"value": value, "unit": "verified tree tokens/s", "cores": cpu_threads(),
                         "kind": "oracle",
                         "sample": f"{per_step} requests of the workload per step"},
        "e2e": {"value": value, "unit": "verified tree tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---- our arm ------------------------------------------------------------------------------------

def run_ours(args, world, rank, local):
    from tree_speculative_verify_gb300 import _lib, build as tvbuild, engine
    tvbuild.build()
    kernel = {"auto": _lib.TV_ATTN_AUTO, "simt": _lib.TV_ATTN_SIMT,
              "tcgen05": _lib.TV_ATTN_TCGEN05}[args.attn_kernel]
    wl = make_workload(args.workload, rank, args.batch)
    n_sets = max(1, args.sets)
    shape = engine.shape_for(wl, kernel, stage_chain=args.stage_chain)
    stream = torch.cuda.current_stream()
    sets = []
    for i in range(n_sets):
        if args.page_tokens:
            # every copy gets the same (seeded) page table, so the first copy's shape -- which
            # holds the address of its table -- serves all of them
            shape_i, st = engine.alloc_paged(wl, args.page_tokens, kernel, seed=0)
            shape_i.stage_chain = args.stage_chain
            if i == 0:
                shape = shape_i
        else:
            st = engine.alloc_state(wl)
        rb = engine.alloc_round(wl, shape)
        engine.prefill(shape, st, rb, stream)
        sets.append((st, rb, st.L.clone()))
    torch.cuda.synchronize()
    for _, rb, _ in sets:
        if int(rb.status.item()) != 0:
            raise SystemExit(f"prefill failed: status {int(rb.status.item())}")
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]

    select = shape.n_sel > 0   # the sparse path picks its C4 entries on the device each round

    def step(i, timed=None):
        st, rb, L0 = sets[i % n_sets]
        st.L.copy_(L0, non_blocking=True)
        if select:
            engine.indexer(shape, st, rb, stream)
        engine.plan(shape, st, rb, stream)
        engine.branch_compress(shape, st, rb, stream)
        if timed is not None:
            timed[0].record(stream)
        engine.attention(shape, st, rb, None, stream)
        if timed is not None:
            timed[1].record(stream)
        engine.accept(shape, st, rb, stream)
        engine.refresh(shape, st, rb, stream)

    # the round as a CUDA graph per state copy (the L reset is captured with it); attention time
    # comes from a separate eager pass with events around the attention launch
    graphs = None
    if not args.no_graph:
        graphs = []
        for st, rb, L0 in sets:
            graphs.append(engine.RoundGraph(
                shape, st, rb, prologue=lambda st=st, L0=L0: st.L.copy_(L0, non_blocking=True),
                select=select))
    for i in range(args.warmup):
        if graphs:
            graphs[i % n_sets].replay()
        else:
            step(i)
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        if graphs:
            graphs[(args.warmup + k) % n_sets].replay()
        else:
            step(args.warmup + k, ev[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    # clocks under load: the same rounds replayed back to back for ~1.5 s while the sampler runs
    # (the timed steps alone last a few ms, too short for a 100 ms sampler)
    t_load = time.perf_counter()
    k = 0
    while time.perf_counter() - t_load < 1.5:
        for _ in range(50):
            if graphs:
                graphs[k % n_sets].replay()
            else:
                step(k)
            k += 1
        torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    if clk is not None:
        clk["under_load"] = f"{k} rounds replayed back to back over {time.perf_counter() - t_load:.1f} s"
    for st_, rb_, l0_ in sets:   # the replays committed rounds: back to the set's state
        st_.L.copy_(l0_)
    torch.cuda.synchronize()
    barrier(world)
    if graphs:
        for k in range(args.steps):
            step(args.warmup + k, ev[k])
        torch.cuda.synchronize()
    ms = t_start.elapsed_time(t_end) / args.steps
    ms = max_over_ranks(ms, world)
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    for _, rb, _ in sets:
        if int(rb.status.item()) != 0:
            raise SystemExit(f"device status {int(rb.status.item())} after the timed steps")

    # end to end through the C ABI: every step copies its inputs (queries, tree K/V, tree, tokens)
    # from pinned host memory and reads its result -- the acceptance outputs the host scheduler
    # continues from (accept length, path, bonus token, committed positions) -- back to the host.
    # The attention output O stays on the device, where the next layer consumes it.  Copies run on
    # their own stream, one step ahead, so step k+1's upload overlaps step k's round.
    def in_tensors(r_):
        return [r_.Q, r_.treeK, r_.treeV, r_.parents, r_.draft, r_.target] + (
            [r_.q_idx] if select else [])

    def out_tensors(r_):
        return [r_.accept_len, r_.path, r_.bonus, r_.committed]

    host_in = [t.cpu().pin_memory() for t in in_tensors(sets[0][1])]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in out_tensors(sets[0][1])]
                for _ in range(n_sets)]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    # uploads split over several copy streams (large inputs in slices along the batch), so that
    # more than one copy engine moves the step's inputs
    n_cs = max(1, args.copy_streams)
    copy_streams = [torch.cuda.Stream() for _ in range(n_cs)]
    freed = [torch.cuda.Event() for _ in range(n_sets)]     # the set's last round has finished
    landed = [[torch.cuda.Event() for _ in range(n_cs)] for _ in range(n_sets)]

    def e2e_upload(i):
        s_, r_, _ = sets[i % n_sets]
        pieces = []
        for dst, src in zip(in_tensors(r_), host_in):
            if dst.numel() * dst.element_size() >= (4 << 20) and dst.shape[0] >= n_cs:
                step_ = -(-dst.shape[0] // n_cs)
                pieces += [(dst[k:k + step_], src[k:k + step_]) for k in range(0, dst.shape[0], step_)]
            else:
                pieces.append((dst, src))
        for c, cs in enumerate(copy_streams):
            with torch.cuda.stream(cs):
                cs.wait_event(freed[i % n_sets])
                for dst, src in pieces[c::n_cs]:
                    dst.copy_(src, non_blocking=True)
                landed[i % n_sets][c].record(cs)

    def e2e_round(i):
        s_, r_, l_ = sets[i % n_sets]
        for ev_ in landed[i % n_sets]:
            stream.wait_event(ev_)
        if graphs:
            graphs[i % n_sets].replay()   # the captured round (its prologue resets L)
        else:
            s_.L.copy_(l_, non_blocking=True)
            engine.verify_round(shape, s_, r_, None, stream, select=select)
        for dst, src in zip(host_out[i % n_sets], out_tensors(r_)):
            dst.copy_(src, non_blocking=True)
        freed[i % n_sets].record(stream)

    def e2e_run(n, t0=None):
        if t0 is not None:
            for cs in copy_streams:
                cs.wait_event(t0)
        e2e_upload(0)
        for k in range(n):
            if k + 1 < n:
                e2e_upload(k + 1)
            e2e_round(k)

    for fe in freed:
        fe.record(stream)
    e2e_run(args.warmup)
    torch.cuda.synchronize()
    barrier(world)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps, e0)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    barrier(world)
    # the same end-to-end loop with the five C-ABI calls launched one by one every step (the host
    # side of every call -- validation, tensor-map encoding, launches -- inside the timed region)
    e2e_eager_ms = None
    if graphs:
        graphs_saved, graphs = graphs, None
        e2e_run(args.warmup)
        torch.cuda.synchronize()
        barrier(world)
        e2 = torch.cuda.Event(enable_timing=True)
        e3 = torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        e2e_run(args.steps, e2)
        e3.record(stream)
        torch.cuda.synchronize()
        e2e_eager_ms = max_over_ranks(e2.elapsed_time(e3) / args.steps, world)
        graphs = graphs_saved
        barrier(world)
    for k in range(min(args.steps, n_sets)):
        if int(host_out[k][0].min()) < 1:
            raise SystemExit("end-to-end step returned an accept length below 1")

    tokens_per_step = world * wl.B * wl.D
    value = job_throughput(world, wl.B, wl.D, ms)
    kv_bytes, qo_bytes, flops = attention_accounting(wl)
    pk = peaks()
    attn_s = attn_ms * 1e-3
    tc_name = "tcgen05" if _lib.tv_attn_kernel_for(shape) == _lib.TV_ATTN_TCGEN05 else "simt"
    traffic = traffic_record(f"attention_{tc_name}_{args.workload}")
    if traffic is not None:
        # captured on a smaller batch of the same workload; DRAM bytes scale with the KV read
        traffic = traffic["dram_bytes_per_launch"] * kv_bytes / traffic["algorithmic_bytes_per_launch"]
    tflops = flops / attn_s / 1e12
    gbs = kv_bytes / attn_s / 1e9
    line = {
        "metric": METRIC,
        "value": value, "unit": "verified tree tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": WORKLOAD_DESC[args.workload], "B_per_gpu": wl.B, "D": wl.D,
                   "H": wl.H, "d": wl.d, "attention_kernel": tc_name,
                   "l2": f"inputs larger than L2: {n_sets} rotating state copies, "
                         f"{kv_bytes / 1e6:.0f} MB KV per step each",
                   "parallelism": f"replicas x{world} (requests sharded, no collective)",
                   "cuda_graph": graphs is not None,
                   "refresh_skip": bool(args.stage_chain),
                   "kv_layout": (f"page pools, {args.page_tokens} tokens per page, pages scattered"
                                 if args.page_tokens else "contiguous per request")},
        "roofline": {"bound": "tensor", "achieved": tflops,
                     "peak": pk["tc"], "unit": "TFLOP/s", "frac": tflops / pk["tc"],
                     "traffic": traffic,
                     "kernel": f"tv_tree_verify_attn ({tc_name})",
                     "peak_source": f"{pk['source']} bf16 dense, burst (the kernel runs "
                                    "for ~0.2 ms per round)",
                     "algorithmic_flops_per_launch": flops},
        "hbm": {"achieved": gbs, "peak": pk["hbm"], "unit": "GB/s", "frac": gbs / pk["hbm"],
                "frac_of_8TBps": gbs / 8000.0, "algorithmic_bytes_per_launch": kv_bytes,
                "with_q_and_o_bytes": kv_bytes + qo_bytes,
                "note": "compressed KV + raw tail + tree + scratch rows, read once per request"},
        "attention_ms": attn_ms,
        "e2e": {"value": tokens_per_step / (e2e_ms * 1e-3), "unit": "verified tree tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "note": ("the captured round (engine.RoundGraph)" if graphs else
                         "the round launched call by call") + " through the C ABI; inputs "
                        f"uploaded from pinned host memory one step ahead on {n_cs} copy "
                        "stream(s); acceptance results read back each step"},
        "e2e_eager": None if e2e_eager_ms is None else {
            "value": tokens_per_step / (e2e_eager_ms * 1e-3), "unit": "verified tree tokens/s",
            "ms_per_step": e2e_eager_ms,
            "note": "the same end-to-end loop with the five C-ABI calls launched call by call "
                    "every step"},
        "gpu_launches": args.steps * launches_per_step(shape, tc_name),
        "clocks": clk,
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl)
        line["cpu_baseline"]["cpu_model"] = cpu_model()
        one = cpu_baseline_single_thread(args)
        if one is not None:
            line["cpu_baseline"]["single_thread"] = {"value": one["value"], "cores": 1,
                                                     "sample": one["sample"]}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_sweep(args):
    """Per cell: round time (CUDA graph replay, L2 flushed before each timed replay), attention
    time (eager launch between events), mean accepted length and committed tokens/s
    = sum of accepted lengths / round time."""
    from tree_speculative_verify_gb300 import _lib, build as tvbuild, engine, workloads
    tvbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")   # 256 MB > L2
    cells = workloads.sweep_cells()
    idx = range(len(cells)) if args.cells is None else [int(c) for c in args.cells.split(",")]
    rows = []
    for i in idx:
        c = cells[i]
        wl = workloads.sweep_cell(i, **c)
        shape = engine.shape_for(wl, stage_chain=args.stage_chain)
        st = engine.alloc_state(wl)
        rb = engine.alloc_round(wl, shape)
        engine.prefill(shape, st, rb, stream)
        L0 = st.L.clone()
        graph = engine.RoundGraph(shape, st, rb,
                                  prologue=lambda st=st, L0=L0: st.L.copy_(L0, non_blocking=True))
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        t_round, t_attn = [], []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            flush.fill_(2)
            st.L.copy_(L0)
            engine.plan(shape, st, rb, stream)
            engine.branch_compress(shape, st, rb, stream)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            engine.attention(shape, st, rb, None, stream)
            a1.record(stream)
            torch.cuda.synchronize()
            t_round.append(e0.elapsed_time(e1))
            t_attn.append(a0.elapsed_time(a1))
        if int(rb.status.item()) != 0:
            raise SystemExit(f"cell {i}: device status {int(rb.status.item())}")
        acc = rb.accept_len.cpu().numpy()
        ms = statistics.median(t_round)
        row = {"cell": i, "D": c["D"], "B": c["B"], "tree": c["kind"], "p": c["p"],
               "round_ms": ms, "attention_ms": statistics.median(t_attn),
               "mean_accept_len": float(acc.mean()), "refresh_skip": bool(args.stage_chain),
               "committed_tokens_per_s": float(acc.sum()) / (ms * 1e-3),
               "verified_tree_tokens_per_s": job_throughput(1, wl.B, wl.D, ms),
               "attention_kernel": "tcgen05" if _lib.tv_attn_kernel_for(shape) ==
               _lib.TV_ATTN_TCGEN05 else "simt"}
        rows.append(row)
        print(json.dumps(row), flush=True)
        del graph, st, rb
        torch.cuda.empty_cache()
    best = max(rows, key=lambda r: r["committed_tokens_per_s"])
    print(json.dumps({"sweep": "budget", "cells": len(rows), "steps": args.steps,
                      "warmup": args.warmup, "best_committed_tokens_per_s": best}), flush=True)


def run_draft(args):
    """Draft decode at draft-side shapes: for draft steps s = 1..3 the tree built so far
    (D_s = 1 + 2s nodes) goes through plan, scratch pad and attention; L2 flushed before each
    timed iteration; CUDA events around the three calls."""
    from tree_speculative_verify_gb300 import _lib, build as tvbuild, engine, workloads
    tvbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    base = workloads.draft_beam(B=args.batch or 64, steps=3)
    for s in range(1, 4):
        wl = workloads.draft_level(base, s)
        shape = engine.shape_for(wl)
        st = engine.alloc_state(wl)
        rb = engine.alloc_round(wl, shape)
        engine.prefill(shape, st, rb, stream)
        for _ in range(args.warmup):
            engine.draft_decode(shape, st, rb, None, stream)
        ts = []
        for _ in range(args.steps):
            flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            engine.draft_decode(shape, st, rb, None, stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        if int(rb.status.item()) != 0:
            raise SystemExit(f"draft step {s}: device status {int(rb.status.item())}")
        ms = statistics.median(ts)
        print(json.dumps({"draft_step": s, "B": wl.B, "D": wl.D, "ms": ms,
                          "draft_tree_tokens_per_s": wl.B * wl.D / (ms * 1e-3),
                          "attention_kernel": "tcgen05" if _lib.tv_attn_kernel_for(shape) ==
                          _lib.TV_ATTN_TCGEN05 else "simt"}), flush=True)
        del st, rb
        torch.cuda.empty_cache()


def launches_per_step(shape, kernel):
    # plan, branch compress, accept, refresh + attention: SIMT (partials, merge; + the indexer's
    # score and select kernels on the sparse path) or tensor cores (selection gather when a C4
    # selection list is given, request ranking, pair kernel, merge when the KV is split)
    from tree_speculative_verify_gb300 import _lib
    if kernel == "simt":
        return 6 + (2 if shape.n_sel > 0 else 0)
    gather = shape.B * shape.n_sel * 512 * 2 * 2
    split = _lib.tv_workspace_size(shape) > ((shape.B * 4 + 255) // 256) * 256 + gather
    # the ranking kernel runs unless the attention ranks the requests itself (contiguous dense
    # path, B <= 2048); + the indexer's score and select kernels and the selection gather on the
    # sparse path, and the gather of the C128 entries and raw tails from page pools
    ranking = shape.n_sel > 0 or shape.page_tokens > 0 or shape.B > 2048
    return (4 + 1 + (1 if ranking else 0) + (1 if split else 0) + (3 if shape.n_sel > 0 else 0)
            + (1 if shape.page_tokens > 0 else 0))


def main():
    args = parse()
    if args.cpu_baseline_only:
        wl = make_workload(args.workload, 0, args.batch)
        print(json.dumps(cpu_baseline(wl, args.cpu_budget)), flush=True)
        return
    if args.impl == "reference":
        world = int(os.environ.get("WORLD_SIZE", "1"))
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.draft:
        run_draft(args)
        return
    world, rank, local = dist_setup(args.gpus)
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
