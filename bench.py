"""Benchmark of the block-sparse top-k selection hot path on GB300.

One step = one pass of the whole hot path over one batch: the fused decode
selector (causal page count from seq_lens, top-k with forced init/local
blocks under IEEE totalOrder, token-major [T, H, K] ids) with the page-16
sparse block-table epilogue, in one kernel (``--path fused``, default), or
the same work as three launches (``--path unfused``: page counts, selector,
table builder).

Workload (default): long-context decode scaled so that its inputs exceed L2:
131072 requests x decode query length 1, 2 index heads, 1024-tile capacity,
topk 16, bf16 N(0,1) scores with one planted +8.0 block per row, seq_len
uniform in [16384, 131072] (128..1024 causal blocks), 1 init + 2 local
blocks, -inf beyond the causal bound, block table [131072, 1024].

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "selected rows/sec and achieved HBM GB/s (% of GB300 peak) for top-k select"
UNIT = "rows/s"
L2_BYTES = 129 * 1024 * 1024


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--path", choices=["fused", "unfused"], default="fused")
    p.add_argument("--requests", type=int, default=131072)
    p.add_argument("--topk", type=int, default=16)
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--e2e-chunks", type=int, default=8)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-configs", action="store_true")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the topk-64, index-score and attention measurements")
    p.add_argument("--extras-only", choices=["index_score", "attention", "prefill_heavy"],
                   default=None,
                   help="time only this call and print its record (for profiling)")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    return p.parse_args()


# --------------------------------------------------------------------------- dist

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- workload

def build_workload(args, device, rank):
    import synth
    import block_sparse_attention_topk_gb300 as bsa
    w = synth.long_decode(seed=1003 + 7919 * rank, device=device, B=args.requests, H=2,
                          M=1024, K=args.topk, dtype=torch.bfloat16)
    nvp = bsa.bsa_num_valid_pages_decode(w.seq_lens, w.dql)
    synth.fill_tail(w.scores, nvp, float("-inf"))
    synth.plant(w.scores, nvp, w.plant_u, w.plant_value)
    table = synth.random_block_table(w.B, w.M, seed=2003 + rank, device=device)
    torch.cuda.synchronize()
    return w, nvp, table


def algorithmic_bytes(w, nvp_host: np.ndarray, path: str) -> dict:
    """Algorithmic bytes, i.e. the bytes the method must move: the non-forced part of each row's causal prefix, the page-count or
    seq_len read, the id write, and for the table the block-table gathers and
    the table + ctx writes.  Rows whose causal prefix fits in topk read no
    scores."""
    K, H, I, L = w.K, w.H, w.num_init, w.num_local
    S = 2 if w.dtype == torch.bfloat16 else 4
    v = np.minimum(nvp_host.astype(np.int64), w.M)
    forced = np.minimum(v, I + L)
    nonforced = v - forced
    read = np.where(v > K, nonforced, 0) * S                    # per token, per head
    n = np.minimum(v, K)
    score_bytes = int(read.sum()) * H
    idx_bytes = w.T * H * K * 4
    meta_bytes = w.T * 4                                        # seq_len / page count
    gather_bytes = int(n.sum()) * H * 4
    table_bytes = w.T * H * (K * 8 * 4 + 4)
    select = score_bytes + idx_bytes + meta_bytes
    fused = select + gather_bytes + table_bytes
    return {"score_read": score_bytes, "select": select, "fused": fused,
            "table_builder": idx_bytes + meta_bytes + gather_bytes + table_bytes,
            "per_row_select": select / (w.T * H), "per_row_fused": fused / (w.T * H)}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


KERNEL_OF_PATH = {0: "select_kernel", 1: "select_kernel", 2: "group_select_kernel",
                  3: "pair_select_kernel", 4: "octet_select_kernel"}


def dominant_kernel(path_id: int, fused: bool) -> str:
    """Name of the selector kernel the launch policy picked."""
    name = KERNEL_OF_PATH[path_id]
    return name + " (fused sparse-table epilogue)" if fused else name


def select_source_sha() -> str:
    """First 16 hex digits of the sha256 of the selector's CUDA source."""
    import hashlib
    src = os.path.join(ROOT, "block_sparse_attention_topk_gb300", "csrc", "bsa_select.cu")
    return hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]


def read_traffic(path_name: str, kernel: str = "pair_select_kernel", topk: int = 16,
                 requests: int = 131072, traffic_file: str | None = None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on this kernel, topk and request count and still describes the current
    kernel source."""
    f = traffic_file or os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(f) as fh:
            d = json.load(fh)
        ent = d.get(path_name)
        if not ent:
            return None
        if (not ent.get("kernel", "").startswith(kernel + "<") or ent.get("topk") != topk
                or ent.get("requests") != requests):
            return None
        if ent.get("source_sha") != select_source_sha():
            return None
        return ent
    except (OSError, ValueError):
        return None


# --------------------------------------------------------------------------- ours

def run_ours(args):
    import block_sparse_attention_topk_gb300 as bsa
    world, rank, local = dist_setup(args)
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    bsa.lib()
    w, nvp, table = build_workload(args, device, rank)
    nvp_host = nvp.cpu().numpy()
    rows = w.T * w.H
    byt = algorithmic_bytes(w, nvp_host, args.path)
    K, I, L = w.K, w.num_init, w.num_local
    stream = torch.cuda.current_stream(device)

    out_idx = torch.empty((w.T, w.H, K), dtype=torch.int32, device=device)
    sparse_bt = torch.empty((w.T, w.H, K * 8), dtype=torch.int32, device=device)
    sparse_ctx = torch.empty((w.T, w.H), dtype=torch.int32, device=device)
    nvp_buf = torch.empty(w.T, dtype=torch.int32, device=device)

    def step(dominant_events=None):
        if args.path == "fused":
            if dominant_events:
                dominant_events[0].record(stream)
            bsa.bsa_topk_select_sparse_table(w.scores, w.seq_lens, w.dql, K, I, L, table,
                                             out_idx=out_idx, sparse_bt=sparse_bt,
                                             sparse_ctx=sparse_ctx)
            if dominant_events:
                dominant_events[1].record(stream)
            return 1
        bsa.bsa_num_valid_pages_decode(w.seq_lens, w.dql, out=nvp_buf)
        if dominant_events:
            dominant_events[0].record(stream)
        bsa.bsa_topk_select(w.scores, nvp_buf, K, I, L, out_idx=out_idx)
        if dominant_events:
            dominant_events[1].record(stream)
        bsa.bsa_build_sparse_block_table(out_idx, table, w.seq_lens, w.dql, sparse_bt=sparse_bt,
                                         sparse_ctx=sparse_ctx)
        return 3

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(device.index)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launches = 0
    t0.record(stream)
    for i in range(args.steps):
        launches += step(ev[i])
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(total_ms, world)
    ms_per_step = total_ms / args.steps
    rows_all = sum_over_ranks(float(rows), world)
    value = rows_all / (ms_per_step / 1e3)
    kern_avg_ms = statistics.mean(kern_ms)
    peak, peak_src = read_peaks()
    dom_bytes = byt["fused"] if args.path == "fused" else byt["select"]
    achieved = dom_bytes / (kern_avg_ms / 1e3) / 1e9
    pol = bsa.bsa_select_policy(rows, w.M, K, bsa.BSA_DTYPE_BF16,
                                torch.cuda.get_device_properties(device).multi_processor_count)
    kernel = KERNEL_OF_PATH[pol["path"]]
    traffic = read_traffic(args.path, kernel, K, w.B)

    # ---- the same workload at topk 64 (the long-context config's other topk) ----
    extra_topk = None
    if not args.no_extra and w.K != 64:
        extra_topk = topk_step(w, table, nvp_host, 64, device, stream, args)
    # ---- and in a buffer of the 8192-tile capture-time capacity ----
    extra_cap = None
    if not args.no_extra and world == 1:
        extra_cap = capacity_step(w, table, nvp_host, device, stream, args)

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, table, device, stream, rows, expect=(out_idx, sparse_ctx))
        e2e["value"] = sum_over_ranks(e2e["value"], world) if world > 1 else e2e["value"]

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 scores, planted block per row)",
        "config": {
            "workload": f"long_decode_scaled: {w.B} requests x dql 1, H={w.H}, max_k_tiles={w.M}, "
                        f"topk={K}, init={I}, local={L}, seq_len U[16384,131072]",
            "global_batch_rows": int(rows_all), "seq_len": "16384-131072 tokens",
            "path": args.path, "parallelism": f"weak x{world} (independent row shards)",
            "l2": "inputs larger than L2: "
                  f"{byt['score_read'] / 1e6:.0f} MB of scores read per step (L2 129 MB)"},
        "hbm_gbs_achieved": achieved,
        "hbm_frac_of_peak": achieved / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": peak_src,
                     "kernel": dominant_kernel(pol["path"], args.path == "fused"),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                     "traffic_note": None if traffic is None else traffic.get("note")},
        "kernel_ms": kern_avg_ms,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
    }
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        result["cpu_baseline"] = cpu_baseline(w, table, args.cpu_seconds)
    if extra_topk is not None:
        result["topk64_fused"] = extra_topk
    if extra_cap is not None:
        result["capacity8192_fused"] = extra_cap
    if rank == 0 and not args.no_extra and world == 1:
        result["index_score_select"] = index_score_step(device, args)
        result["sparse_decode_attention"] = attention_step(device, args)
    if rank == 0 and not args.no_configs and world == 1:
        result["per_config_latency_us"] = config_latencies(device)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def timed_launches(fn, stream, steps, warmup):
    """Mean CUDA-event duration (ms) of fn() on `stream`, after warm-up; the
    inputs exceed L2, so consecutive launches do not reuse cached data."""
    for _ in range(max(3, warmup)):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for a, b in ev:
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def topk_step(w, table, nvp_host, K, device, stream, args):
    """The fused step of the same long-context workload at another topk
    (same scores, lengths and block table)."""
    import block_sparse_attention_topk_gb300 as bsa
    from types import SimpleNamespace
    out_idx = torch.empty((w.T, w.H, K), dtype=torch.int32, device=device)
    sparse_bt = torch.empty((w.T, w.H, K * 8), dtype=torch.int32, device=device)
    sparse_ctx = torch.empty((w.T, w.H), dtype=torch.int32, device=device)

    def fn():
        bsa.bsa_topk_select_sparse_table(w.scores, w.seq_lens, w.dql, K, w.num_init, w.num_local,
                                         table, out_idx=out_idx, sparse_bt=sparse_bt,
                                         sparse_ctx=sparse_ctx)

    ms = timed_launches(fn, stream, max(10, args.steps // 2), args.warmup)
    wk = SimpleNamespace(K=K, H=w.H, num_init=w.num_init, num_local=w.num_local, dtype=w.dtype,
                         M=w.M, T=w.T)
    byt = algorithmic_bytes(wk, nvp_host, "fused")["fused"]
    peak, src = read_peaks()
    pol = bsa.bsa_select_policy(w.T * w.H, w.M, K, bsa.BSA_DTYPE_BF16,
                                torch.cuda.get_device_properties(device).multi_processor_count)
    achieved = byt / (ms / 1e3) / 1e9
    traffic = read_traffic(f"fused_topk{K}", KERNEL_OF_PATH[pol["path"]], K, w.B)
    return {"kernel": dominant_kernel(pol["path"], True), "topk": K, "kernel_ms": ms,
            "rows_per_s": w.T * w.H / (ms / 1e3), "algorithmic_bytes_per_launch": byt,
            "achieved_gbs": achieved, "peak_gbs": peak, "frac": achieved / peak,
            "peak_source": src,
            "traffic": None if traffic is None else traffic["dram_bytes_per_launch"]}


def capacity_step(w, table, nvp_host, device, stream, args, M=8192):
    """The same fused step with the scores held in a buffer of the 8192-tile
    capture-time capacity (rows 16 KB apart, at most 1024 valid tiles each):
    the policy's pair / octet path takes every row and its list of rows over
    2 KB stays empty.  The call's time covers the list counter's memset and
    both launches; the algorithmic bytes are those of the 1024-tile step."""
    from types import SimpleNamespace
    big = torch.full((w.T, w.H, M), float("-inf"), dtype=w.dtype, device=device)
    big[:, :, :w.M].copy_(w.scores)
    wk = SimpleNamespace(scores=big, seq_lens=w.seq_lens, dql=w.dql, num_init=w.num_init,
                         num_local=w.num_local, T=w.T, H=w.H, M=M, B=w.B, dtype=w.dtype)
    rec = topk_step(wk, table, nvp_host, w.K, device, stream, args)
    rec["workload"] = (f"{w.B} requests x dql 1, H={w.H}, max_k_tiles={M}, topk={w.K}, "
                       "seq_len U[16384,131072] (the headline rows in the capture-time capacity)")
    del big, wk
    torch.cuda.empty_cache()
    return rec


def index_score_bytes(seq, dql, H, D, M, K, valid_blocks):
    """Bytes the fused index score + select must move: the queries, the
    block-table entries and pooled keys of every causal block (once per
    request), the scores it writes for the causal blocks of each row, the
    sequence lengths and the ids.  The selection re-reads the scores it has
    just written from L2, which a separate score kernel would read from HBM."""
    T = seq.shape[0] * dql
    v_req = np.minimum(-(-np.maximum(seq.astype(np.int64), 0) // 128), M)
    rows_v = []
    for lq in range(dql):
        ln = np.maximum(seq.astype(np.int64) - dql + lq + 1, 0)
        rows_v.append(np.minimum(-(-ln // 128), M))
    score_entries = int(sum(x.sum() for x in rows_v)) * H
    return (T * H * D * 2 + int(v_req.sum()) * 4 + int(valid_blocks) * D * 2 +
            score_entries * 4 + seq.shape[0] * 4 + T * H * K * 4)


def index_score_step(device, args):
    """The fused index score + select on a long-context decode batch: 8192
    requests x query length 1, 2 index heads, index dim 128, 1024-tile
    capacity, seq_len U[16384, 131072], paged keys (a distinct physical block
    per causal block), topk 16."""
    import block_sparse_attention_topk_gb300 as bsa
    import synth
    B, dql, H, D, M, K = 8192, 1, 2, 128, 1024, 16
    g = synth.generator(4242, device)
    seq = torch.randint(16384, 131073, (B,), generator=g, device=device).to(torch.int32)
    nb = B * M
    table = synth.paged_block_table(B, M, nb, seed=4243, device=device)
    q, k = synth.index_inputs(4244, B * dql, H, D, nb, device=device)
    scores = torch.full((B * dql, H, M), float("-inf"), dtype=torch.float32, device=device)
    out_idx = torch.empty((B * dql, H, K), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)

    def fn():
        bsa.bsa_index_score_topk_select(q, k, table, seq, dql, K, 1, 2, M=M, scores=scores,
                                        out_idx=out_idx)

    ms = timed_launches(fn, stream, 10, args.warmup)
    seq_h = seq.cpu().numpy()
    valid = int(np.minimum(-(-seq_h.astype(np.int64) // 128), M).sum())
    byt = index_score_bytes(seq_h, dql, H, D, M, K, valid)
    peak, src = read_peaks()
    achieved = byt / (ms / 1e3) / 1e9
    return {"kernel": "index_score_select_kernel", "workload":
            f"{B} requests x dql {dql}, H={H}, D={D}, max_k_tiles={M}, topk={K}, "
            "seq_len U[16384,131072], paged bf16 keys",
            "kernel_ms": ms, "rows_per_s": B * dql * H / (ms / 1e3),
            "algorithmic_bytes_per_launch": byt, "achieved_gbs": achieved, "peak_gbs": peak,
            "frac": achieved / peak, "peak_source": src}


def attention_bytes(ctx, H, G, D, K):
    """Bytes the sparse decode attention must move: each row's key and value
    rows for its ctx tokens, its table entries, ctx, queries and output."""
    rows = ctx.size
    return (int(ctx.sum()) * D * 2 * 2 + rows * (K * 8 * 4 + 4) + rows * G * D * (2 + 4))


def attention_step(device, args):
    """Sparse decode attention over the tables of the fused-table workload
    shape: 128 requests x query length 4, 1 index head, topk 16, seq_len
    U[1, 65536] with ~5% padded, 4 query heads of dim 64 per KV head, a
    page-16 bf16 KV cache of 524288 pages (1 GB each for keys and values; the
    rows read about 260 MB of it per launch, more than L2 holds)."""
    import block_sparse_attention_topk_gb300 as bsa
    import synth
    B, dql, H, G, D, M, K = 128, 4, 1, 4, 64, 512, 16
    w = synth.fused_table(seed=1005, device=device, B=B, dql=dql, H=H, M=M, K=K)
    nvp = bsa.bsa_num_valid_pages_decode(w.seq_lens, dql)
    synth.fill_tail(w.scores, nvp, float("-inf"))
    _, bt, ctx = bsa.bsa_topk_select_sparse_table(w.scores, w.seq_lens, dql, K, 1, 1,
                                                  w.block_table, want_idx=False)
    num_pages = B * M * 8
    q = synth.normal_scores((B * dql, H, G, D), torch.bfloat16, seed=31, device=device)
    kc = synth.normal_scores((num_pages, 16, H, D), torch.bfloat16, seed=32, device=device)
    vc = synth.normal_scores((num_pages, 16, H, D), torch.bfloat16, seed=33, device=device)
    out = torch.empty((B * dql, H, G, D), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def fn():
        bsa.bsa_sparse_decode_attention(q, kc, vc, bt, ctx, out=out)

    ms = timed_launches(fn, stream, 10, args.warmup)
    byt = attention_bytes(ctx.cpu().numpy(), H, G, D, K)
    peak, src = read_peaks()
    achieved = byt / (ms / 1e3) / 1e9
    return {"kernel": "sparse_decode_attention_kernel", "workload":
            f"{B} requests x dql {dql}, H={H}, G={G}, D={D}, topk={K}, seq_len U[1,65536], "
            "tables from the fused select",
            "kernel_ms": ms, "rows_per_s": B * dql * H / (ms / 1e3),
            "algorithmic_bytes_per_launch": byt, "achieved_gbs": achieved, "peak_gbs": peak,
            "frac": achieved / peak, "peak_source": src}


def run_e2e(args, w, table, device, stream, rows, expect=None):
    """Host buffers in, host buffers out, through the same C-ABI call: the
    timed region holds the H2D copies of scores, seq_lens and block table,
    the fused call, and the D2H copies of ids, table and ctx.  The step is
    pipelined over request chunks on three streams (upload, compute,
    download), so a chunk's outputs come back while later inputs still go
    up; one step finishes before the next begins."""
    import block_sparse_attention_topk_gb300 as bsa
    K, I, L = w.K, w.num_init, w.num_local
    h_scores = w.scores.cpu().pin_memory()
    h_seq = w.seq_lens.cpu().pin_memory()
    h_table = table.cpu().pin_memory()
    h_idx = torch.empty((w.T, w.H, K), dtype=torch.int32).pin_memory()
    h_bt = torch.empty((w.T, w.H, K * 8), dtype=torch.int32).pin_memory()
    h_ctx = torch.empty((w.T, w.H), dtype=torch.int32).pin_memory()
    d_scores = torch.empty_like(w.scores)
    d_seq = torch.empty_like(w.seq_lens)
    d_table = torch.empty_like(table)
    d_idx = torch.empty((w.T, w.H, K), dtype=torch.int32, device=device)
    d_bt = torch.empty((w.T, w.H, K * 8), dtype=torch.int32, device=device)
    d_ctx = torch.empty((w.T, w.H), dtype=torch.int32, device=device)
    C = max(1, min(args.e2e_chunks, w.B))
    bounds = [(w.B * c // C, w.B * (c + 1) // C) for c in range(C)]
    up, comp, down = (torch.cuda.Stream(device) for _ in range(3))

    def one():
        start = torch.cuda.Event()
        start.record(stream)
        for st in (up, comp, down):
            st.wait_event(start)
        for r0, r1 in bounds:
            t0, t1 = r0 * w.dql, r1 * w.dql
            with torch.cuda.stream(up):
                d_scores[t0:t1].copy_(h_scores[t0:t1], non_blocking=True)
                d_seq[r0:r1].copy_(h_seq[r0:r1], non_blocking=True)
                d_table[r0:r1].copy_(h_table[r0:r1], non_blocking=True)
                e_up = torch.cuda.Event()
                e_up.record(up)
            comp.wait_event(e_up)
            with torch.cuda.stream(comp):
                bsa.bsa_topk_select_sparse_table(d_scores[t0:t1], d_seq[r0:r1], w.dql, K, I, L,
                                                 d_table[r0:r1], out_idx=d_idx[t0:t1],
                                                 sparse_bt=d_bt[t0:t1], sparse_ctx=d_ctx[t0:t1])
                e_c = torch.cuda.Event()
                e_c.record(comp)
            down.wait_event(e_c)
            with torch.cuda.stream(down):
                h_idx[t0:t1].copy_(d_idx[t0:t1], non_blocking=True)
                h_bt[t0:t1].copy_(d_bt[t0:t1], non_blocking=True)
                h_ctx[t0:t1].copy_(d_ctx[t0:t1], non_blocking=True)
        e_d = torch.cuda.Event()
        e_d.record(down)
        stream.wait_event(e_d)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.e2e_steps):
        one()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.e2e_steps
    if expect is not None:
        # the pipelined step returns what the device-resident step computed
        if not (torch.equal(h_idx, expect[0].cpu()) and torch.equal(h_ctx, expect[1].cpu())):
            raise RuntimeError("end-to-end outputs differ from the device-resident run")
    h2d = h_scores.numel() * h_scores.element_size() + h_seq.numel() * 4 + h_table.numel() * 4
    d2h = (h_idx.numel() + h_bt.numel() + h_ctx.numel()) * 4
    # the host link by itself: one plain pinned copy each way of the step's
    # largest input and output
    link = {}
    for name, src, dst in (("h2d", h_scores, d_scores), ("d2h", d_bt, h_bt)):
        for _ in range(2):
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        nbytes = src.numel() * src.element_size()
        link[name] = 3 * nbytes / (a.elapsed_time(b) / 1e3) / 1e9
    return {"value": rows / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "copy_gbs_in_step": (h2d + d2h) / (ms / 1e3) / 1e9,
            "link_gbs_alone": {"h2d": link["h2d"], "d2h": link["d2h"]},
            "steps": args.e2e_steps, "chunks": C, "kernel_launches_per_step": C}


def config_latencies(device, only=None):
    """Latency of one fused/select call on each workload as given (or on the
    one named `only`): the call is captured in a CUDA graph and each replay
    is timed with events (inputs resident in HBM; L2 flushed before each
    replay by writing 256 MB)."""
    import synth
    import block_sparse_attention_topk_gb300 as bsa
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.int32, device=device)
    out = {}
    cases = {
        "tiny_decode": synth.tiny_decode(device=device),
        "short_decode": synth.short_decode(device=device),
        "long_decode_k16": synth.long_decode(device=device, K=16),
        "long_decode_k64": synth.long_decode(device=device, K=64),
        "mixed_prefill_decode": synth.mixed_prefill_decode(device=device),
        "fused_table": synth.fused_table(device=device),
        # full capacity (1M-token contexts, 4096..8192 blocks): the split path
        "capacity_8192_split": synth.long_decode(device=device, B=64, H=2, M=8192, K=16,
                                                 min_len=524288, max_len=1048576),
        # prefill-heavy unified batch at the 8192-tile capacity: 32 decode rows
        # and two 8192-token prefill chunks (one at the end of a 1M context)
        "prefill_heavy_8192": synth.mixed_prefill_decode(
            device=device, H=4, M=8192, K=16, dtype=torch.bfloat16,
            prefill_prefix=(0, 8192 * 128 - 8192), decode_max_prefix=8192 * 128 - 1),
    }
    if only is not None:
        cases = {only: cases[only]}
    for name, w in cases.items():
        if w.seq_lens is not None:
            nvp = bsa.bsa_num_valid_pages_decode(w.seq_lens, w.dql)
        else:
            nvp = bsa.bsa_num_valid_pages_varlen(w.cu_seqlens_q, w.prefix_lens, w.T)
        synth.fill_tail(w.scores, nvp, float("-inf"))
        if w.plant_u is not None:
            synth.plant(w.scores, nvp, w.plant_u, w.plant_value)
        if name == "fused_table":
            def call():
                bsa.bsa_topk_select_sparse_table(w.scores, w.seq_lens, w.dql, w.K, w.num_init,
                                                 w.num_local, w.block_table)
        else:
            def call():
                bsa.bsa_topk_select(w.scores, nvp, w.K, w.num_init, w.num_local)
        for _ in range(5):
            call()
        torch.cuda.synchronize()
        # capture once, replay: the timed span holds the kernel(s) only
        graph = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream(device)
        with torch.cuda.stream(st):
            with torch.cuda.graph(graph, stream=st):
                call()
        torch.cuda.synchronize()
        times = []
        for _ in range(30):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            graph.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
        out[name] = {"median_us": statistics.median(times), "rows": w.T * w.H,
                     "call": "fused select+table" if name == "fused_table" else "select"}
    return out


# --------------------------------------------------------------------------- CPU

def cpu_baseline(w, table, seconds):
    """The oracle as it stands (single-threaded C), timed on the host on a
    bounded sample of the same workload's rows."""
    import oracle
    oracle.build()
    K, I, L = w.K, w.num_init, w.num_local
    chunk = 512
    done = 0
    t_spent = 0.0
    while t_spent < seconds and done < w.T:
        hi = min(w.T, done + chunk)
        sc = w.scores[done:hi].cpu()
        seq = w.seq_lens[done:hi].cpu().numpy()
        bt = table[done:hi].cpu().numpy()
        t0 = time.perf_counter()
        oracle.topk_select_sparse_table(sc, seq, w.dql, K, I, L, bt)
        t_spent += time.perf_counter() - t0
        done = hi
    rows = done * w.H
    return {"value": rows / t_spent, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"first {done} of {w.T} token rows ({rows} rows) of the same workload, "
                      f"fused select + table, {t_spent:.1f} s of single-thread CPU",
            "host_cores_available": os.cpu_count()}


def run_reference(args):
    """The reference arm: the CPU oracle timed on bounded samples of the same
    workload (the pages ship no runnable implementation)."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    import oracle
    import synth
    oracle.build()
    dev = "cpu"
    B = min(args.requests, 2048)
    w = synth.long_decode(seed=1003, device=dev, B=B, H=2, M=1024, K=args.topk)
    nvp = oracle.num_valid_pages_decode(w.seq_lens.numpy(), w.dql)
    synth.fill_tail(w.scores, torch.from_numpy(nvp), float("-inf"))
    synth.plant(w.scores, torch.from_numpy(nvp), w.plant_u, w.plant_value)
    table = synth.random_block_table(B, w.M, seed=2003)
    rows_per_step = 256
    times = []
    seq = w.seq_lens.numpy()
    tb = table.numpy()
    for i in range(args.warmup + args.steps):
        lo = (i * rows_per_step) % B
        hi = min(B, lo + rows_per_step)
        t0 = time.perf_counter()
        oracle.topk_select_sparse_table(w.scores[lo:hi], seq[lo:hi], 1, w.K, w.num_init,
                                        w.num_local, tb[lo:hi])
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = rows_per_step * w.H / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": {
                "workload": "long_decode_scaled (sampled): dql 1, H=2, max_k_tiles=1024, "
                            f"topk={w.K}, init=1, local=2, seq_len U[16384,131072]",
                "path": "fused select + table"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{rows_per_step} token rows x H=2 per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_extras_only(args):
    import block_sparse_attention_topk_gb300 as bsa
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    bsa.lib()
    if args.extras_only == "prefill_heavy":
        res = config_latencies(device, only="prefill_heavy_8192")["prefill_heavy_8192"]
    else:
        fn = index_score_step if args.extras_only == "index_score" else attention_step
        res = fn(device, args)
    print(json.dumps({args.extras_only: res}), flush=True)


if __name__ == "__main__":
    a = parse()
    if a.impl == "reference":
        run_reference(a)
    elif a.extras_only:
        run_extras_only(a)
    else:
        run_ours(a)
