"""Benchmark: decode-attention KV tokens/s and achieved HBM GB/s on one GB300.

Default workload: the hybrid 6-layer decode step (batch 256, 32 query heads,
lognormal lengths with median 4096 clipped to [256, 32768], layers 0-4 local
with window 1024, layer 5 global, buffer map {0,0,1,1,2,3}, page size 16).
One step = cai_kv_append of the current token into each of the 4 buffers,
then cai_mqa_decode for each of the 6 layers (split-KV decode + LSE combine).
Inputs are resident in HBM when the timed region starts; the KV read per step
(~0.77 GB) is larger than L2, and the KV loads carry an L2 evict-first hint.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl cai|reference] [--config 1..5]

Under torchrun (N > 1) every rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
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
import threading
import time
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention KV tokens/s and achieved HBM GB/s (% of peak) per GB300"
UNIT = "KV tokens/s"
BYTES_PER_TOKEN = 2 * 128 + 8  # int8 K + int8 V + two fp32 scales


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cai", choices=["cai", "reference"])
    ap.add_argument("--config", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--sigma", type=float, default=1.0)
    ap.add_argument("--num-splits", type=int, default=0)
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (testing only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--mixed", action="store_true",
                    help="continuous batching: 128 decode steps + 8 prefill chunks of 256 tokens in one launch")
    ap.add_argument("--dialogues", action="store_true",
                    help="cross-turn host KV cache on a synthetic multi-turn trace (hit rate, restore GB/s, TTFT)")
    ap.add_argument("--per-layer", action="store_true",
                    help="one decode launch per layer instead of all the step's layers in one launch")
    ap.add_argument("--local-ring", action="store_true",
                    help="keep each sequence of a local-only KV buffer in a ring of pages (window recycling)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--no-parity", action="store_true", help="skip the oracle check of the timed outputs")
    ap.add_argument("--no-extra", action="store_true",
                    help="default run only: skip the long-context (5) and append-prefill (4) sub-records")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ncu", action="store_true",
                    help="open the CUDA profiler window around the timed steps only (for ncu --profile-from-start off)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- work accounting

def layer_work(w, layer):
    """Attended tokens, pages and algorithmic HBM bytes of one decode launch."""
    W = w.layer_windows[layer]
    P = w.page_size
    L = np.asarray(w.ctx_len, dtype=np.int64)
    lo = np.maximum(0, L - W) if W > 0 else np.zeros_like(L)
    tokens = L - lo
    pages = np.where(tokens > 0, (L - 1) // P - lo // P + 1, 0)
    q_out = w.batch * w.num_q_heads * 128 * (2 + 4) + w.batch * 4
    bytes_ = int(tokens.sum()) * BYTES_PER_TOKEN + int(pages.sum()) * 4 + q_out
    return int(tokens.sum()), int(pages.sum()), bytes_


def append_bytes(w):
    # fp32 K and V rows read + int8 codes and scales written, per buffer
    return w.num_buffers * w.batch * w.n_new * (2 * 128 * 4 + BYTES_PER_TOKEN + 4)


def step_work(w):
    toks, byts = 0, 0
    for layer in range(len(w.layer_windows)):
        t, _, b = layer_work(w, layer)
        toks += t
        byts += b
    return toks, byts


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []          # (wall time, csv line)
        self.t_start = None
        self.t_end = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # sampling must be running before the timed region opens
            deadline = time.time() + 5.0
            while not self.lines and time.time() < deadline and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def start(self):
        self.t_start = time.time()

    def stop(self):
        self.t_end = time.time()
        if self.proc is not None:  # one more sample period so the last stretch is covered
            time.sleep(0.06)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        """Median SM clock and the throttle reasons seen during the timed region [start, stop]
        (the nearest earlier sample when the region is shorter than one sample period)."""
        lines = self.lines
        if self.t_start is not None and self.t_end is not None:
            inside = [x for x in lines if self.t_start <= x[0] <= self.t_end + 0.06]
            before = [x for x in lines if x[0] < self.t_start]
            lines = inside if inside else before[-1:]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def smi_index(device: int) -> int:
    """nvidia-smi index of a CUDA device, honouring CUDA_VISIBLE_DEVICES when it lists numbers."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p.strip() for p in vis.split(",") if p.strip()]
    if device < len(parts) and parts[device].isdigit():
        return int(parts[device])
    return device


# ----------------------------------------------------------------------------- peaks and profiles

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic(workload_tag: str):
    """DRAM bytes (read + write) of one step's decode launches from the committed ncu summary, if it
    matches the current kernel source and this workload; the same unit as roofline.achieved."""
    path = os.path.join(ROOT, "profiles", "decode_dram_traffic.txt")
    src = os.path.join(ROOT, "int8_mqa_decode_gb300", "csrc", "decode.cu")
    if not os.path.exists(path):
        return None
    info = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            info[k.strip()] = v.strip()
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if info.get("decode_cu_sha256") != sha or info.get("workload") != workload_tag:
        return None
    try:
        return float(info["dram_bytes_per_step"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- CPU oracle leg

L2_BYTES = 129 * 1024 * 1024  # GB300 L2
PARITY_ATOL = 2e-3  # max abs error of attention outputs against the float64 oracle


def sample_seqs(ctx_len, n_spaced):
    """Shortest, longest and about n_spaced more sequences evenly spaced by length."""
    order = np.argsort(ctx_len, kind="stable")
    picks = [int(order[0]), int(order[-1])] + [int(i) for i in order[1:-1:max(1, len(order) // n_spaced)]]
    return list(dict.fromkeys(picks))


class CpuOracle:
    """The oracle (as it stands) on host cores over a bounded sample of the workload's sequences."""

    def __init__(self, w, n_spaced: int = 14):
        import oracle
        import synth

        self.w = w
        self.picks = sample_seqs(w.ctx_len, n_spaced)
        # Inputs (codes, scales, queries) prepared untimed, like resident device inputs.
        self.items = []
        for b in self.picks:
            L = int(w.ctx_len[b])
            kv = {buf: oracle.seq_kv(w.seed, buf, b, L) for buf in range(w.num_buffers)}
            for layer in range(len(w.layer_windows)):
                qb = synth.q_rows(w.seed, synth.stream_q(layer), b, w.num_q_heads)
                W = w.layer_windows[layer]
                tokens = min(L, W) if W > 0 else L
                self.items.append((qb, kv[w.layer_to_buffer[layer]], L, W, tokens, b, layer))
        self.cores = os.cpu_count() or 1

    def parity(self, outs):
        """Max abs error of the GPU outputs (numpy [layer][B][Hq][128]) against the oracle on the
        sampled sequences, all layers."""
        import oracle
        from concurrent.futures import ThreadPoolExecutor

        w = self.w

        def one(item):
            qb, (kc, ks, vc, vs), L, W, _, b, layer = item
            ref, _ = oracle.decode_seq(qb, kc, ks, vc, vs, L, W, w.softmax_scale)
            return float(np.abs(outs[layer][b] - ref).max())

        with ThreadPoolExecutor(self.cores) as ex:
            worst = max(ex.map(one, self.items))
        ok = bool(worst <= PARITY_ATOL)
        return {"max_abs_err": worst, "n_seqs": len(self.picks), "layers": len(w.layer_windows),
                "atol": PARITY_ATOL, "ok": ok,
                "what": "outputs of the last timed step against the float64 oracle on the shortest, the longest and "
                        "evenly spaced sequences"}

    def run(self, seconds: float):
        import oracle
        from concurrent.futures import ThreadPoolExecutor

        w = self.w

        def one(item):
            qb, (kc, ks, vc, vs), L, W = item[:4]
            oracle.decode_seq(qb, kc, ks, vc, vs, L, W, w.softmax_scale)

        done_tokens, t0 = 0, time.perf_counter()
        with ThreadPoolExecutor(self.cores) as ex:
            while True:
                list(ex.map(one, self.items))
                done_tokens += sum(p[4] for p in self.items)
                if time.perf_counter() - t0 >= seconds:
                    break
        dt = time.perf_counter() - t0
        return {"value": done_tokens / dt, "unit": UNIT, "cores": self.cores, "kind": "oracle",
                "sample": f"{len(self.picks)} sequences (shortest, longest and evenly spaced by length) x "
                          f"{len(w.layer_windows)} layers of the same workload, repeated for {dt:.1f} s; float64 C "
                          f"oracle, {self.cores} threads over (sequence, layer)"}


# ----------------------------------------------------------------------------- GPU arm: append-prefill

def prefill_flops(w):
    """4*d FLOPs per (query row, attended key) pair: QK^T and PV, causal within the chunk."""
    prefix = np.asarray(w.ctx_len, dtype=np.int64) - w.n_new
    pairs = 0
    for p0 in prefix:
        for i in range(w.n_new):
            hi = int(p0) + i + 1
            lo = max(0, hi - w.layer_windows[0]) if w.layer_windows[0] > 0 else 0
            pairs += hi - lo
    return 4 * 128 * w.num_q_heads * pairs, pairs


def prefill_parity(w, out, seqs=None, tokens=(0, 1, 127, 128, 129, 254, 255)):
    """Max abs error of prefill outputs (numpy [B][n_new][Hq][128]) against the oracle on sampled
    sequences and new tokens (the first and last tokens of the chunk and those at the tile edges)."""
    import oracle
    import synth

    seqs = sample_seqs(w.ctx_len, 2) if seqs is None else seqs
    tokens = [t for t in tokens if t < w.n_new]
    worst = 0.0
    for b in seqs:
        L = int(w.ctx_len[b])
        kc, ks, vc, vs = oracle.seq_kv(w.seed, 0, b, L)
        qb = synth.q_rows(w.seed, synth.STREAM_Q_PREFILL, b, w.n_new * w.num_q_heads).reshape(w.n_new, w.num_q_heads, 128)
        ref, _ = oracle.prefill_seq(qb, kc, ks, vc, vs, L - w.n_new, w.layer_windows[0], w.softmax_scale, tokens)
        worst = max(worst, float(np.abs(out[b][tokens] - ref).max()))
    return {"max_abs_err": worst, "n_seqs": len(seqs), "tokens_per_seq": len(tokens), "atol": PARITY_ATOL,
            "ok": bool(worst <= PARITY_ATOL),
            "what": "outputs of the last timed call against the float64 oracle on sampled sequences and tokens"}


def prefill_launches(w):
    """Launches of one append + prefill step: the append, the dequant pass, the attention, and
    the merge of the last wave's key pieces when the q-tile pairs leave a partial wave."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    pairs = w.batch * -(-w.n_new * w.num_q_heads // 256)
    grid = min(pairs, sms)
    rem = pairs % grid
    return 3 + (1 if rem and grid // rem >= 2 else 0)


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["bf16_tflops_sustained"]), float(d["bf16_tflops"]), "measured"
    return 1700.0, 1900.0, "fallback"


def run_prefill(args, rank, world):
    import torch
    import harness
    import int8_mqa_decode_gb300 as cai
    import synth

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    import __graft_entry__
    __graft_entry__.build()
    seed = 1004 + 100 * rank
    w = synth.workload(4, seed=seed, batch=args.batch)
    cache = harness.PagedCache(w)
    cache.fill()
    q = cache.prefill_q()
    out = torch.empty(w.batch, w.n_new, w.num_q_heads, 128, device="cuda")
    ws = cache.prefill_workspace()
    kvs = [cache.step_kv(0)]
    prefix = (cache.ctx_len - w.n_new).to(torch.int32)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]

    def step(rec=None):
        k, v, start = kvs[0]
        cai.cai_kv_append(cache.pools[0], k, v, cache.table, start)
        if rec is not None:
            rec[0].record(stream)
        cai.cai_mqa_prefill_chunk(cache.pools[0], q, cache.table, prefix, 0, w.softmax_scale, ws, out)
        if rec is not None:
            rec[1].record(stream)

    # The step's KV pages (and the copy the dequant pass writes) fit in L2: L2 is flushed
    # between timed steps by a write of twice its size, outside each step's event pair.
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    with ClockSampler(smi_index(torch.cuda.current_device())) as clocks:
        torch.cuda.synchronize()
        if args.ncu:
            torch.cuda.profiler.start()
        clocks.start()
        # Pass 1, the step (append + prefill call), one event pair per step; pass 2, the same
        # steps with an event pair around the prefill call, for the kernels' duration.
        for s in range(args.steps):
            flush_buf.fill_(s & 255)
            step_ev[s][0].record(stream)
            step()
            step_ev[s][1].record(stream)
        torch.cuda.synchronize()
        if args.ncu:
            torch.cuda.profiler.stop()
        for s in range(args.steps):
            flush_buf.fill_(s & 255)
            step(ev[s])
        torch.cuda.synchronize()
        clocks.stop()
    ms = allreduce_max(sum(a.elapsed_time(b) for a, b in step_ev), world)
    kernel_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    parity = prefill_parity(w, out.cpu().numpy()) if rank == 0 and not args.no_parity else None
    flops, pairs = prefill_flops(w)
    sustained, burst, kind = bf16_peak()
    achieved = flops / (kernel_ms * 1e-3) / 1e12
    return {
        "metric": "append-prefill attention TFLOP/s (KV-query pairs / s)", "value": world * flops * args.steps / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 KV, bf16/fp16 MMA / fp32 accumulate", "data": "synthetic",
        "config": {"workload": w.name, "global_batch": w.batch * world, "kv_query_pairs_per_head": pairs,
                   "flops_per_step": flops, "parallelism": f"replicas x{world}",
                   "l2": "L2 flushed between timed steps (a write of twice its size, outside each step's event pair)"},
        "gpu_launches": prefill_launches(w) * args.steps,
        # The launches are timed alone (a sub-millisecond burst), so the burst peak is the
        # denominator; the sustained figure is kept for reference.
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s",
                     "frac": achieved / burst, "traffic": None, "peak_kind": kind + " bf16 burst",
                     "peak_sustained": sustained,
                     "kernel": "cai_mqa_prefill_chunk (dequant pass + tcgen05 attention)"},
        "clocks": clocks.summary(),
        "parity": parity,
    }


# ----------------------------------------------------------------------------- GPU arm: mixed batch

def run_mixed(args, rank, world):
    """Continuous batching: one varlen launch over 128 one-token decode steps (contexts
    U[1024, 8192]) and 8 prefill chunks of 256 tokens on 4096-token prefixes, against the
    same work as a decode launch plus a prefill launch."""
    import torch
    import harness
    import int8_mqa_decode_gb300 as cai
    import synth
    import synth.gpu as sgpu

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    import __graft_entry__
    __graft_entry__.build()
    seed = 1006 + 100 * rank
    n_dec, n_pf, chunk, Hq, P = 128, 8, 256, 32, 16
    dec_len = synth.uniform_int(seed, 3, n_dec, 1024, 8192)
    prefix = np.concatenate([dec_len - 1, np.full(n_pf, 4096)]).astype(np.int64)
    n_new = np.concatenate([np.ones(n_dec), np.full(n_pf, chunk)]).astype(np.int64)
    L = prefix + n_new
    B = n_dec + n_pf
    w = synth.Workload("mixed", B, Hq, P, L, [0], [0], n_new=1, seed=seed)
    cache = harness.PagedCache(w)
    cache.fill(upto=L)
    off = np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32)
    total = int(off[-1])
    q = torch.empty(total, Hq, 128, dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        qb = torch.empty(1, int(n_new[b]) * Hq, 128, dtype=torch.bfloat16, device="cuda")
        sgpu.q_rows(qb, seed, synth.STREAM_Q_PREFILL, b)
        q[off[b]:off[b + 1]] = qb.view(int(n_new[b]), Hq, 128)
    out = torch.empty(total, Hq, 128, device="cuda")
    off_d = torch.from_numpy(off).cuda()
    prefix_d = torch.from_numpy(prefix.astype(np.int32)).cuda()
    ws = cache.prefill_workspace()
    # the same work split: decode launch over the one-token sequences, prefill launch over the chunks
    q_dec = q[:n_dec]
    out_dec = torch.empty(n_dec, Hq, 128, device="cuda")
    ctx_dec = torch.from_numpy(L[:n_dec].astype(np.int32)).cuda()
    table_dec, table_pf = cache.table[:n_dec].contiguous(), cache.table[n_dec:].contiguous()
    ws_dec = torch.zeros(cai.cai_mqa_decode_workspace_size(n_dec, Hq, cache.max_pages_per_seq, P, 0, 0),
                         dtype=torch.uint8, device="cuda")
    q_pf = q[n_dec:].view(n_pf, chunk, Hq, 128)
    out_pf = torch.empty(n_pf, chunk, Hq, 128, device="cuda")
    prefix_pf = prefix_d[n_dec:].contiguous()
    ws_pf = torch.empty(cai.cai_mqa_prefill_workspace_size(n_pf, cache.max_pages_per_seq, P), dtype=torch.uint8,
                        device="cuda")

    def one_launch():
        cai.cai_mqa_prefill_varlen(cache.pools[0], q, off_d, chunk, cache.table, prefix_d, 0, w.softmax_scale, ws, out)

    def two_launches():
        cai.cai_mqa_decode(cache.pools, [0], 0, q_dec, table_dec, ctx_dec, 0, w.softmax_scale, 0, ws_dec, out_dec)
        cai.cai_mqa_prefill_chunk(cache.pools[0], q_pf, table_pf, prefix_pf, 0, w.softmax_scale, ws_pf, out_pf)

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(smi_index(torch.cuda.current_device())) as clocks:
            torch.cuda.synchronize()
            clocks.start()
            if args.ncu:
                torch.cuda.profiler.start()
            t0.record()
            for _ in range(args.steps):
                fn()
            t1.record()
            torch.cuda.synchronize()
            if args.ncu:
                torch.cuda.profiler.stop()
            clocks.stop()
        return allreduce_max(t0.elapsed_time(t1), world) / args.steps, clocks.summary()

    ms_one, clocks = timed(one_launch)
    ms_two, _ = timed(two_launches)
    torch.cuda.synchronize()
    diff = float((out[:n_dec] - out_dec).abs().max())
    pairs = float(np.sum(n_new * prefix + n_new * (n_new + 1) / 2)) * Hq  # (query row, attended key) pairs
    return {
        "metric": "continuous-batching step: new tokens/s (128 decode steps + 8 prefill chunks, one cai_mqa_prefill_varlen call)",
        "value": world * total / (ms_one * 1e-3), "unit": "new tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_one, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8 KV, bf16 QK / fp16 PV, fp32 accumulate", "data": "synthetic",
        "config": {"workload": f"mixed: {n_dec} decode (L~U[1024,8192]) + {n_pf} chunks of {chunk} on 4096, Hq={Hq}, "
                               f"P={P}", "new_tokens": total, "kv_query_pairs": pairs},
        "one_call": "cai_mqa_prefill_varlen: the chunks through the prefill kernel, then the one-token rows through "
                    "the decode kernel, which starts on the SMs that the prefill's last wave leaves",
        "two_launch_ms_per_step": ms_two, "decode_rows_max_abs_diff_vs_decode_path": diff,
        "tflops": 4 * 128 * pairs / (ms_one * 1e-3) / 1e12, "gpu_launches": 2 * args.steps, "clocks": clocks,
    }


# ----------------------------------------------------------------------------- GPU arm: cross-turn cache

def run_dialogues(args, rank, world):
    """Cross-turn KV cache on a synthetic multi-turn trace: D dialogues, T turns, U new tokens per
    turn.  Turn t brings (t+1)*U tokens; with the host cache the previous turns' whole pages are
    restored from host memory and only the rest is appended and prefilled, without it the whole
    dialogue is appended and prefilled.  Reports the hit rate (restored / prompt tokens), the restore
    rate and the time to first token per turn both ways (restore + append + prefill of the batch)."""
    import torch
    import harness
    import int8_mqa_decode_gb300 as cai
    import synth
    import synth.gpu as sgpu

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    import __graft_entry__
    __graft_entry__.build()
    D, T, U, Hq, P = 16, 4, 512, 32, 16
    seed = 1008 + 100 * rank
    max_len = T * U
    w = synth.Workload("dialogues", D, Hq, P, np.full(D, max_len), [0], [0], seed=seed)
    dev = harness.PagedCache(w)
    ids = [np.arange(d * 1000003, d * 1000003 + max_len, dtype=np.int32) for d in range(D)]
    host = cai.cai_host_cache_create(P, 1, D * max_len // P + 64)
    stream = torch.cuda.current_stream()
    ws = dev.prefill_workspace()
    scale = w.softmax_scale

    def kv_for(p0, n):
        k = torch.empty(D, n, 128, dtype=torch.float32, device="cuda")
        v = torch.empty_like(k)
        start = torch.full((D,), p0, dtype=torch.int32, device="cuda")
        sgpu.normal_rows(k, seed, synth.stream_k(0), 0, pos=start)
        sgpu.normal_rows(v, seed, synth.stream_v(0), 0, pos=start)
        return k, v, start

    def q_for(n):
        q = torch.empty(D, n * Hq, 128, dtype=torch.bfloat16, device="cuda")
        sgpu.q_rows(q, seed, synth.STREAM_Q_PREFILL, 0)
        return q.view(D, n, Hq, 128)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    # One untimed append + prefill first, so the first timed call pays no first-launch setup.
    k, v, start = kv_for(0, U)
    q = q_for(U)
    out = torch.empty(D, U, Hq, 128, device="cuda")
    cai.cai_kv_append(dev.pools[0], k, v, dev.table, start)
    cai.cai_mqa_prefill_chunk(dev.pools[0], q, dev.table, torch.zeros(D, dtype=torch.int32, device="cuda"), 0, scale,
                              ws, out)
    torch.cuda.synchronize()
    del k, v, q, out
    turns = []
    restored_tokens = prompt_tokens = restored_bytes = 0
    restore_ms_total = 0.0
    try:
        for t in range(T):
            L = (t + 1) * U
            # --- without the cache: the whole dialogue
            k, v, start = kv_for(0, L)
            q = q_for(L)
            out = torch.empty(D, L, Hq, 128, device="cuda")
            prefix = torch.zeros(D, dtype=torch.int32, device="cuda")
            torch.cuda.synchronize()
            a, b = ev(), ev()
            a.record(stream)
            cai.cai_kv_append(dev.pools[0], k, v, dev.table, start)
            cai.cai_mqa_prefill_chunk(dev.pools[0], q, dev.table, prefix, 0, scale, ws, out)
            b.record(stream)
            torch.cuda.synchronize()
            no_cache_ms = a.elapsed_time(b)
            del k, v, q, out
            # --- with the cache: restore the longest cached prefix, then append and prefill the rest
            n = [cai.cai_host_cache_match(host, ids[d][:L]) for d in range(D)]
            n0 = min(n)
            k, v, start = kv_for(n0, L - n0)
            q = q_for(L - n0)
            out = torch.empty(D, L - n0, Hq, 128, device="cuda")
            prefix = torch.full((D,), n0, dtype=torch.int32, device="cuda")
            torch.cuda.synchronize()
            a, r, b = ev(), ev(), ev()
            a.record(stream)
            if n0 > 0:  # the whole batch's cached prefixes in one call
                cai.cai_host_cache_restore_batch(host, ids, [n0] * D, dev.pools, [dev.table_np[d] for d in range(D)],
                                                 stream=stream)
            r.record(stream)
            cai.cai_kv_append(dev.pools[0], k, v, dev.table, start)
            cai.cai_mqa_prefill_chunk(dev.pools[0], q, dev.table, prefix, 0, scale, ws, out)
            b.record(stream)
            torch.cuda.synchronize()
            cache_ms = a.elapsed_time(b)
            rest_ms = a.elapsed_time(r)
            restored_tokens += D * n0
            prompt_tokens += D * L
            rb = D * (n0 // P) * cai.cai_page_bytes(P)
            restored_bytes += rb
            restore_ms_total += rest_ms
            # the turn's pages go back to the host cache (after the first token, not timed)
            for d in range(D):
                cai.cai_host_cache_store(host, ids[d][:L], dev.pools, dev.table_np[d], stream=stream)
            turns.append({"turn": t, "prompt_tokens": L, "restored_tokens": n0, "ttft_ms_cache": cache_ms,
                          "ttft_ms_no_cache": no_cache_ms, "restore_ms": rest_ms,
                          "restore_gbs": (rb / (rest_ms * 1e-3) / 1e9) if n0 else None})
            del k, v, q, out
        stats = cai.cai_host_cache_stats(host)
    finally:
        cai.cai_host_cache_destroy(host)
    cached = [x["ttft_ms_cache"] for x in turns[1:]]
    plain = [x["ttft_ms_no_cache"] for x in turns[1:]]
    return {
        "metric": "cross-turn KV cache: time to first token per turn (batch of dialogues), with / without the host cache",
        "value": statistics.mean(plain) / statistics.mean(cached), "unit": "x speed-up (turns 2..T)",
        "n_gpus": world, "steps": T, "warmup": 0, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 KV, bf16/fp16 MMA / fp32 accumulate", "data": "synthetic multi-turn trace",
        "config": {"workload": f"{D} dialogues x {T} turns x {U} new tokens, Hq={Hq}, P={P}, one KV buffer",
                   "parallelism": f"replicas x{world}"},
        "hit_rate_tokens": restored_tokens / prompt_tokens,
        "restore_gbs": restored_bytes / (restore_ms_total * 1e-3) / 1e9 if restore_ms_total else None,
        "turns": turns, "host_cache_stats": stats, "gpu_launches": None,
    }


# ----------------------------------------------------------------------------- GPU arm: decode

def run_gpu(args, rank, world):
    import torch
    import harness
    import int8_mqa_decode_gb300 as cai
    import synth

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    import __graft_entry__
    __graft_entry__.build()
    seed = (1000 + args.config) + 100 * rank
    w = synth.workload(args.config, seed=seed, sigma=args.sigma, batch=args.batch)
    cache = harness.PagedCache(w, local_ring=args.local_ring)
    cache.fill()
    nl = len(w.layer_windows)
    qs = [cache.decode_q(layer) for layer in range(nl)]
    outs = [torch.empty(w.batch, w.num_q_heads, 128, device="cuda") for _ in range(nl)]
    layered = nl > 1 and not args.per_layer
    wss = [cache.workspace(layer, args.num_splits) for layer in range(nl)]
    ws_layers = cache.layers_workspace(args.num_splits) if layered else None
    step_kv = [cache.step_kv(buf) for buf in range(w.num_buffers)]
    stream = torch.cuda.current_stream()
    n_events = 1 if layered else nl
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * n_events)] for _ in range(args.steps)]

    def step(record=None):
        cai.cai_kv_append_pools(cache.pools, [k for k, _, _ in step_kv], [v for _, v, _ in step_kv], cache.tables,
                                [s for _, _, s in step_kv])
        if layered:
            if record is not None:
                record[0].record(stream)
            cache.decode_layers(qs, outs, num_splits=args.num_splits, workspace=ws_layers)
            if record is not None:
                record[1].record(stream)
            return
        for layer in range(nl):
            if record is not None:
                record[2 * layer].record(stream)
            cai.cai_mqa_decode(cache.pools, w.layer_to_buffer, layer, qs[layer], cache.tables[w.layer_to_buffer[layer]],
                               cache.ctx_len, w.layer_windows[layer], w.softmax_scale, args.num_splits, wss[layer],
                               outs[layer])
            if record is not None:
                record[2 * layer + 1].record(stream)

    # Launches per step: the appends, the decode launch(es) and one combine per split layer.
    splits_layers = sum(
        1 for layer in range(nl)
        if cai.cai_mqa_decode_workspace_size(w.batch, w.num_q_heads, cache.max_pages_per_seq, w.page_size,
                                             w.layer_windows[layer], args.num_splits) > 256)
    launches_per_step = 1 + (1 if layered else nl) + splits_layers

    # A step whose KV fits in L2 twice over would read it back from L2 in the next step:
    # such workloads (the tiny and the local-layer ones) flush L2 between timed steps by
    # writing a buffer of twice its size, outside each step's own event pair.
    _, kv_bytes_step = step_work(w)
    flush_buf = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda")
                 if kv_bytes_step < 2 * L2_BYTES else None)
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)] if flush_buf is not None else None

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    barrier(world)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(smi_index(torch.cuda.current_device())) as clocks:
        torch.cuda.synchronize()
        if args.ncu:
            torch.cuda.profiler.start()
        clocks.start()
        # Pass 1, the step throughput: no events between the launches (an event between two
        # launches chained by programmatic dependent launch holds the second one back); with
        # an L2 flush between steps, one event pair per step and the flush outside it.
        t_start.record(stream)
        for s in range(args.steps):
            if flush_buf is not None:
                flush_buf.fill_(s & 255)
                step_ev[s][0].record(stream)
            step()
            if flush_buf is not None:
                step_ev[s][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        if args.ncu:
            torch.cuda.profiler.stop()
        # Pass 2, the same steps with an event pair around every decode launch: the kernel's
        # average launch duration for the roofline.
        for s in range(args.steps):
            if flush_buf is not None:
                flush_buf.fill_(s & 255)
            step(ev[s])
        torch.cuda.synchronize()
        clocks.stop()
    ms_total = (t_start.elapsed_time(t_end) if flush_buf is None
                else sum(a.elapsed_time(b) for a, b in step_ev))
    decode_ms = sum(ev[s][2 * l].elapsed_time(ev[s][2 * l + 1]) for s in range(args.steps) for l in range(n_events))
    ms_max = allreduce_max(ms_total, world)

    toks_step, bytes_step = step_work(w)
    value = world * toks_step * args.steps / (ms_max * 1e-3)
    peak, peak_kind = measured_peaks()
    achieved = bytes_step * args.steps / (decode_ms * 1e-3) / 1e9
    tag = f"config{args.config}-B{w.batch}-seed{seed}"
    traffic = profiled_traffic(tag)

    # Parity of the benchmarked step: the outputs of its last timed pass against the oracle.
    cpu = None
    parity = None
    if rank == 0 and not args.no_parity:
        cpu = CpuOracle(w, n_spaced=14 if args.config != 5 else 2)
        parity = cpu.parity([o.cpu().numpy() for o in outs])

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, w, cache, qs, outs, wss, step_kv, toks_step, world, layered)

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8 KV, fp16 MMA / fp32 accumulate",
        "data": "synthetic (seeded Irwin-Hall normals, lengths and permuted block tables)",
        "config": {"workload": w.name, "global_batch": w.batch * world, "seq_len": "lognormal" if args.config == 3
                   else "uniform", "kv_tokens_per_step": toks_step, "num_splits": args.num_splits or "auto",
                   "l2": ("KV read per step larger than L2 (129 MB); KV loads are L2 evict-first"
                          if flush_buf is None else
                          "L2 flushed between timed steps (a write of twice its size, outside each step's event pair)"),
                   "parallelism": f"replicas x{world} (independent sequences per GPU)",
                   "kv_pool_bytes": cache.pool_bytes(),
                   **({"local_ring_pages": [r for r in cache.ring if r]} if args.local_ring else {})},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": ("cai_mqa_decode_layers (all layers of the step in one launch, "
                                f"LSE combine of {splits_layers} split layer(s))" if layered else
                                f"cai_mqa_decode (split-KV decode + LSE combine), {nl} launch(es) per step"),
                     "timed_launches": (["decode_kernel"] if layered else ["decode_kernel"] * nl) +
                                       ["combine_kernel"] * splits_layers,
                     "algorithmic_bytes_per_step": bytes_step,
                     "bytes_note": "KV pages read once per attended layer (264 B per token, 4 B per page id), q and "
                                   "out; the append launch is outside the event pair and outside these bytes"},
        "step_algorithmic_bytes": bytes_step + append_bytes(w),
        "hbm_gbs_step": (bytes_step + append_bytes(w)) * args.steps / (ms_max * 1e-3) / 1e9,
        "queries_per_s": world * w.batch * args.steps / (ms_max * 1e-3),
        "clocks": clocks.summary(),
        "e2e": e2e,
        "parity": parity,
    }
    if rank == 0 and world == 1 and not args.no_cpu:
        result["cpu_baseline"] = (cpu or CpuOracle(w)).run(args.cpu_seconds)
    return result


def run_e2e(args, w, cache, qs, outs, wss, step_kv, toks_step, world, layered=False):
    """Same step through the public API with inputs in pinned host memory: every step copies its
    inputs host -> device and its outputs device -> host inside the timed region.  As a serving loop
    would, the step's inputs sit packed in one pinned buffer and go over in one copy, on their own
    stream, into one of two device buffers while the previous step computes; the outputs sit packed
    in one device buffer and come back in one copy on a third stream while the next step computes."""
    import torch
    import int8_mqa_decode_gb300 as cai

    nl = len(w.layer_windows)
    # Packed input layout: per layer q, then per buffer k, v, start; every piece 256-byte aligned.
    pieces = [q for q in qs] + [t for kv in step_kv for t in kv]
    offs, total = [], 0
    for t in pieces:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    for t, o in zip(pieces, offs):
        n = t.numel() * t.element_size()
        h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(2)]

    def views(buf):
        out = []
        for t, o in zip(pieces, offs):
            n = t.numel() * t.element_size()
            out.append(buf[o:o + n].view(t.dtype).view(t.shape))
        return out[:nl], [tuple(out[nl + 3 * i: nl + 3 * i + 3]) for i in range(len(step_kv))]

    d_views = [views(d_in[b]) for b in range(2)]
    o_numel = outs[0].numel()
    d_out = [torch.empty(nl * o_numel, dtype=outs[0].dtype, device="cuda") for _ in range(2)]
    d_out_views = [[d_out[b][l * o_numel:(l + 1) * o_numel].view(outs[0].shape) for l in range(nl)] for b in range(2)]
    h_out = torch.empty(nl * o_numel, dtype=outs[0].dtype).pin_memory()
    ws_layers = [cache.layers_workspace(args.num_splits) for _ in range(2)] if layered else None
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of slot b copied
    ev_used = [torch.cuda.Event() for _ in range(2)]  # kernels done with the inputs of slot b
    ev_done = [torch.cuda.Event() for _ in range(2)]  # outputs of slot b written
    ev_read = [torch.cuda.Event() for _ in range(2)]  # outputs of slot b copied out
    h2d = sum(t.numel() * t.element_size() for t in pieces)
    d2h = h_out.numel() * h_out.element_size()
    first_use = [True, True]

    def step(i):
        b = i & 1
        d_q, d_kv = d_views[b]
        with torch.cuda.stream(s_in):
            if not first_use[b]:
                s_in.wait_event(ev_used[b])
            d_in[b].copy_(h_in, non_blocking=True)
            ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        cai.cai_kv_append_pools(cache.pools, [dk for dk, _, _ in d_kv], [dv for _, dv, _ in d_kv], cache.tables,
                                [ds for _, _, ds in d_kv])
        if not first_use[b]:
            comp.wait_event(ev_read[b])
        if layered:
            cache.decode_layers(d_q, d_out_views[b], num_splits=args.num_splits, workspace=ws_layers[b])
        else:
            for layer in range(nl):
                cai.cai_mqa_decode(cache.pools, w.layer_to_buffer, layer, d_q[layer],
                                   cache.tables[w.layer_to_buffer[layer]], cache.ctx_len, w.layer_windows[layer],
                                   w.softmax_scale, args.num_splits, wss[layer], d_out_views[b][layer])
        ev_done[b].record(comp)
        ev_used[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            h_out.copy_(d_out[b], non_blocking=True)
            ev_read[b].record(s_out)
        first_use[b] = False

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.steps):
        step(i)
    comp.wait_stream(s_out)
    comp.wait_stream(s_in)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = allreduce_max(e0.elapsed_time(e1), world)
    return {"value": world * toks_step * args.steps / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms / args.steps,
            "copies": "pinned host buffers; the step's inputs packed into one buffer and copied in one transfer on "
                      "their own stream into one of two device buffers while the previous step computes; the "
                      "outputs packed in one device buffer and copied back in one transfer on a third stream"}


# ----------------------------------------------------------------------------- reference arm (the oracle)

def run_reference(args):
    import synth

    w = synth.workload(args.config, sigma=args.sigma, batch=args.batch)
    cpu = CpuOracle(w)
    per_step = max(1.0, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu.run(per_step / 2)
    vals, t0 = [], time.perf_counter()
    last = None
    for _ in range(args.steps):
        last = cpu.run(per_step)
        vals.append(last["value"])
    dt = time.perf_counter() - t0
    value = statistics.mean(vals)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "global_batch": w.batch, "sample": last["sample"]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                             "sample": last["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------------------------- distributed plumbing

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse()
    rank, world = dist_init()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if args.mixed:
        res = run_mixed(args, rank, world)
    elif args.dialogues:
        res = run_dialogues(args, rank, world)
    else:
        res = run_prefill(args, rank, world) if args.config == 4 else run_gpu(args, rank, world)
        if args.config == 3 and not args.no_extra and not args.per_layer and not args.local_ring and args.batch is None:
            res["extra"] = run_extra(args, rank, world)
    bad = [k for k, r in [("main", res), *((res.get("extra") or {}).items())]
           if isinstance(r, dict) and isinstance(r.get("parity"), dict) and not r["parity"]["ok"]]
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if bad:
        print(f"parity failed: {bad}", file=sys.stderr, flush=True)
        sys.exit(3)


def run_extra(args, rank, world):
    """The long-context global decode (workload 5, batch 1024) and the append-prefill chunk (workload 4,
    batch 16), each timed for a few steps after the headline step, with its roofline and an oracle check."""
    import copy
    import gc
    import torch

    extra = {}
    for cfg in (5, 4):
        gc.collect()
        torch.cuda.empty_cache()
        a = copy.copy(args)
        a.config, a.steps, a.warmup, a.no_e2e, a.no_cpu, a.num_splits = cfg, min(args.steps, 30), 3, True, True, 0
        r = run_prefill(a, rank, world) if cfg == 4 else run_gpu(a, rank, world)
        keep = ("value", "unit", "ms_per_step", "roofline", "parity", "clocks", "gpu_launches", "queries_per_s")
        extra[f"config{cfg}"] = {"workload": r["config"]["workload"], "steps": a.steps,
                                 **{k: r[k] for k in keep if k in r}}
    gc.collect()
    torch.cuda.empty_cache()
    return extra


if __name__ == "__main__":
    main()
