#!/usr/bin/env python3
"""Throughput of the GPT-2 pre-norm forward on GB300 through the C ABI.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--seed S]

A step is one pass of the whole forward path of the workload over one batch of
synthetic, seeded input already resident in device memory: the block
(LN1, c_attn, causal attention, c_proj + residual, LN2, c_fc + GELU, mlp
c_proj + residual), the full model (embedding, L blocks, ln_f, tied head) or
one cached decode step.  The default workload is the GPT-2-small block
(d=768, 12 heads, B=8, T=1024, bf16 storage, fp32 accumulate).

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events
on the launching stream; a barrier and a device synchronize bracket the K
steps; the per-step time is the maximum over ranks.  No step finds its inputs
in L2: the inputs of every workload are larger than L2.  The block workloads
rotate over R copies of their parameters and input (R x (weights + x) >= 2 x
L2, every copy read once per R steps); the full forward reads 250 MB of
weights and decode 3.3 GB of cached keys and values per step.  Under torchrun each rank runs an independent
replica of the workload (the forward has no cross-sequence exchange), so the
whole-job value is the sum of the ranks' tokens over the slowest rank's time.

One JSON line is printed by rank 0.  Beside the device-timed value it carries:
  e2e         the same metric through the C ABI with pinned host buffers: every
              step copies its input from pinned host memory and its result
              back; steps are pipelined over the device input/result slots
              (copies on their own streams overlap the neighbouring steps'
              compute), every copy inside the timed region; with it, the
              host link as this run's copies see it (GB/s each way and the
              copy time of one step) and the host's time to enqueue a step;
  workloads   the other configurations timed in the same run (the full
              GPT-2-small forward, the GPT-2-XL-shaped block, cached decode
              of the GPT-2-medium shape), each with its step time, tokens/s,
              end-to-end roofline fraction, top kernel and clock sample;
  roofline    the dominant kernel's achieved rate (its algorithmic flops or
              bytes per launch over its CUDA-event duration, measured in a
              second, profiled pass of K steps) against the measured peak;
  cpu_baseline  the fp64 oracle timed on the host cores on a bounded sample;
  clocks      SM clocks and throttle reasons sampled during the timed steps;
  ms_per_step_median  the median of the K step times (ms_per_step is their
              mean);
  eager_ms_per_step  for the graph-replayed decode step, the same step with
              its kernels launched one by one;
  graph_ms_per_step  for the other steps, launched one by one for the
              headline, the same steps replayed from CUDA graphs (one per
              input slot);
  cached_weights  for the block workloads, the same step with the fp16
              working copies of the weights made by an earlier call (what the
              per-call conversion from bf16 costs).
--impl reference times the oracle itself as the reference arm.
"""
from __future__ import annotations

import os

# The oracle's matrix products use numpy's BLAS: give it every host core
# (set before numpy is first imported).
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(os.cpu_count() or 1))

import argparse  # noqa: E402
import gc  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402
from concurrent.futures import ThreadPoolExecutor  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gpt_pre_norm_gb300 import synthetic as S  # noqa: E402

METRIC = "GPT-2 block/full-forward tokens/s at 1 GB300; achieved TFLOP/s vs bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}
TENSOR_KINDS = {"gemm_c_attn", "gemm_c_proj", "gemm_c_fc", "gemm_mlp_c_proj", "gemm_lm_head",
                "gemm_other", "attention_prefill"}
L2_BYTES_FALLBACK = 126 << 20  # GB300
TOPK = 8  # candidates per position of the top-k workload
# Configurations timed beside the default one (the GPT-2-small block).
EXTRA_WORKLOADS = ("forward_bf16_gpt2_small", "block_bf16_d1600", "decode_bf16_gpt2_medium")
# What the bf16 path computes in.
DTYPE_DETAIL = ("bf16 storage (weights, block input/output, KV cache); fp16 operands in the "
                "Linear products (activations written as fp16, weights converted from bf16); "
                "bf16 Q/K/V and probabilities in attention; fp32 accumulation and fp32 "
                "residual stream")


# ------------------------------------------------------------------ helpers --
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0, source="fallback")


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:12]


KERNEL_SOURCES = {
    "gemm": ["gpt_pre_norm_gb300/csrc/gemm_tc.cu", "gpt_pre_norm_gb300/csrc/gemm_smallm.cu",
             "gpt_pre_norm_gb300/csrc/device.cuh"],
    "attention_prefill": ["gpt_pre_norm_gb300/csrc/attn_tc.cu",
                          "gpt_pre_norm_gb300/csrc/device.cuh"],
    "attention_decode": ["gpt_pre_norm_gb300/csrc/attention.cu",
                         "gpt_pre_norm_gb300/csrc/device.cuh"],
    "row": ["gpt_pre_norm_gb300/csrc/rowwise.cu", "gpt_pre_norm_gb300/csrc/device.cuh"],
}


def kernel_family(kind: str) -> str:
    if kind.startswith("gemm"):
        return "gemm"
    if kind.startswith("attention_decode"):
        return "attention_decode"
    if kind.startswith("attention"):
        return "attention_prefill"
    return "row"


def ncu_traffic(kind: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = source_digest(KERNEL_SOURCES[kernel_family(kind)])
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kind \
                    and parts[1] == workload and parts[3] == digest:
                return float(parts[2])
    return None


def e2e_roofline(prof, peaks, steps, ms_step):
    """Sum over the step's kernels of each one's roofline time, max(algorithmic
    flops / tensor peak, algorithmic bytes / HBM peak), against the measured
    step time: the end-to-end fraction of the rooflines."""
    t_roof = 0.0
    for rec in prof.values():
        t_roof += max(rec["flops"] / (peaks["bf16_tflops"] * 1e12),
                      rec["bytes"] / (peaks["hbm_gbs"] * 1e9))
    t_roof = t_roof / steps * 1e3  # ms per step
    return {"sum_t_roof_ms": t_roof, "measured_ms": ms_step, "frac": t_roof / ms_step}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, v in enumerate(flags)
                          if v.lower() == "active"})
        mx = max(r[1] for r in rows)
        loaded = [r[0] for r in rows if r[0] > 0.5 * mx] or [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------- workloads --
def workload_flops(w: S.Workload) -> float:
    """Algorithmic flops of one step (dense products; causal attention pairs)."""
    d, B, T = w.d, w.B, w.T
    tp = w.t_past
    gemm = 2.0 * B * T * (3 * d * d + d * d + 4 * d * d + 4 * d * d)
    pairs = T * tp + 0.5 * T * (T + 1)
    attn = 4.0 * B * w.n_head * pairs * w.d_h
    per_layer = gemm + attn
    if w.kind == "block":
        return per_layer
    return w.n_layer * per_layer + 2.0 * B * T * d * w.n_vocab


def l2_bytes(torch, device) -> int:
    props = torch.cuda.get_device_properties(device)
    return int(getattr(props, "L2_cache_size", 0) or L2_BYTES_FALLBACK)


def nbytes(tensors) -> int:
    return sum(t.numel() * t.element_size() for t in tensors)


def to_dev_bf16(a: np.ndarray, torch, device):
    bits = S.bf16_bits(a).view(np.int16)
    return torch.from_numpy(bits).to(device).view(torch.bfloat16)


class Runner:
    """Builds one workload's device state and exposes step functions.

    Host-side generation of the synthetic weights (and of the decode
    workload's 1.6e9-value KV cache) runs on a thread pool: each tensor has
    its own random stream, so the values do not depend on the pool.

    Step i uses input/result slot i % slots.  A block workload's inputs (its
    weights and x) are smaller than L2, so it keeps `slots` copies of both,
    enough that all copies together are at least twice the L2 size: a copy
    is read again only after the others have been, and is gone from L2."""

    def __init__(self, w: S.Workload, seed: int, device, pool: ThreadPoolExecutor, l2: int):
        import torch
        from gpt_pre_norm_gb300 import binding as G
        self.G, self.torch, self.w, self.device = G, torch, w, device
        mode = G.GPT2_BF16 if w.dtype == "bf16" else G.GPT2_FP32
        dt = torch.bfloat16 if mode == G.GPT2_BF16 else torch.float32

        def todev(a):
            return to_dev_bf16(a, torch, device) if mode == G.GPT2_BF16 else \
                torch.from_numpy(a).to(device)

        self.ctx = G.Context(w.n_vocab, w.n_ctx, w.d, w.n_head, w.n_layer, mode, w.B, w.T)
        self.tokens = w.B * w.T
        self.cache = None
        self.graph = None
        # At least two device buffers for each step input and result, so that
        # the end-to-end steps can overlap copies with the neighbouring steps'
        # compute; a step replayed from a CUDA graph has fixed buffers (one slot).
        self.slots = 2
        if w.kind == "block":
            p = {k: todev(v) for k, v in S.block_params(w, seed).items()}
            x = todev(S.block_input(w, seed))
            per_copy = nbytes(p.values()) + nbytes([x])
            self.slots = max(2, -(-2 * l2 // per_copy))
            self.params = [p] + [{k: v.clone() for k, v in p.items()}
                                 for _ in range(self.slots - 1)]
            self.inp = [{"x": x}] + [{"x": x.clone()} for _ in range(self.slots - 1)]
            self.res = [torch.empty_like(x) for _ in range(self.slots)]
            self.inp_host = {"x": x.cpu().pin_memory()}
            self.res_host = [torch.empty(x.shape, dtype=dt).pin_memory()
                             for _ in range(self.slots)]
            self.l2_note = (f"inputs larger than L2, no flush: {self.slots} copies of the "
                            f"weights and x ({per_copy / 1e6:.1f} MB each) rotated, "
                            f"{self.slots * per_copy / 1e6:.0f} MB >= 2 x L2")
            return
        blocks = list(pool.map(lambda layer: S.block_params(w, seed, layer), range(w.n_layer)))
        p = S.embeddings(w, seed)
        tp = {k: todev(p[k]) for k in ("wte", "wpe", "lnf_g", "lnf_b")}
        tp["blocks"] = [{k: todev(v) for k, v in b.items()} for b in blocks]
        self.mp = G.ModelParams(tp)
        weights = nbytes([tp[k] for k in ("wte", "wpe", "lnf_g", "lnf_b")]) + \
            sum(nbytes(b.values()) for b in tp["blocks"])
        self.l2_note = (f"inputs larger than L2, no flush: {weights / 1e6:.0f} MB of weights "
                        "read every step")
        ids = S.token_ids(w, seed)
        ids_dev = torch.from_numpy(ids).to(device)
        self.inp = [{"ids": ids_dev}, {"ids": torch.empty_like(ids_dev)}]
        self.inp_host = {"ids": ids_dev.cpu().pin_memory()}
        if w.kind == "forward_loss":
            # targets: the next token of each sequence, none (-1) at the last position
            tg = np.concatenate([ids[:, 1:], np.full((w.B, 1), -1, ids.dtype)], axis=1)
            tg_dev = torch.from_numpy(np.ascontiguousarray(tg)).to(device)
            self.inp[0]["targets"] = tg_dev
            self.inp[1]["targets"] = torch.empty_like(tg_dev)
            self.inp_host["targets"] = tg_dev.cpu().pin_memory()
            self.res = [torch.empty((w.B, w.T), dtype=torch.float32, device=device)
                        for _ in range(2)]
        elif w.kind == "forward_topk":
            # [0]: the k largest logits, [1]: their ids (int32 bits)
            self.res = [torch.empty((2, w.B, w.T, TOPK), dtype=torch.float32, device=device)
                        for _ in range(2)]
        else:
            n_res = 1 if w.kind == "decode" else 2
            self.res = [torch.empty((w.B, w.T, w.n_vocab), dtype=torch.float32, device=device)
                        for _ in range(n_res)]
        self.res_host = [torch.empty(r.shape, dtype=r.dtype).pin_memory() for r in self.res]
        if w.kind == "decode":
            self.slots = 1
            # A generation loop reuses its weights every step: their fp16
            # working copies are made once (on the first step, before timing).
            G.gpt2_ctx_cache_weights(self.ctx, True)
            shape = (w.B, w.n_layer, 2, w.n_head, w.n_ctx, w.d_h)
            host = torch.empty(shape, dtype=torch.int16).pin_memory()
            hv = host.numpy()

            def fill(bl):
                b, layer = bl
                pk = S.past_kv(w, seed, b, layer)
                hv[b, layer, :, :, :w.t_past] = S.bf16_bits(pk).view(np.int16)

            list(pool.map(fill, [(b, layer) for b in range(w.B) for layer in range(w.n_layer)]))
            self.cache = G.KV(host.to(device).view(torch.bfloat16), w.t_past)
            kv_read = 2 * w.B * w.n_layer * 2 * w.n_head * w.t_past * w.d_h
            self.l2_note = (f"inputs larger than L2, no flush: {kv_read / 1e9:.1f} GB of cached "
                            f"keys and values and {weights / 1e6:.0f} MB of weights read "
                            "every step")

    # One step on input/result slot `s`, inputs resident on the device.
    def step(self, s: int = 0):
        G, w = self.G, self.w
        s %= self.slots
        inp, res = self.inp[s], self.res[s]
        if w.kind == "block":
            G.gpt2_block_forward(self.ctx, inp["x"], self.params[s], w.B, w.T, w.d, w.n_head,
                                 out=res)
        elif w.kind == "forward":
            G.gpt2_forward(self.ctx, inp["ids"], self.mp, w.B, w.T, logits=res)
        elif w.kind == "forward_topk":
            G.gpt2_forward_topk(self.ctx, inp["ids"], self.mp, w.B, w.T, TOPK, want_lse=False,
                                top_logits=res[0], top_ids=res[1].view(self.torch.int32))
        elif w.kind == "forward_loss":
            G.gpt2_forward_loss(self.ctx, inp["ids"], self.mp, w.B, w.T, targets=inp["targets"],
                                want_next=False, loss=res)
        else:
            self.cache.T_len = w.t_past
            G.gpt2_forward(self.ctx, inp["ids"], self.mp, w.B, w.T, past=self.cache,
                           present=self.cache, logits=res)

    # The block step on one weight set whose fp16 working copies an earlier call
    # made (the context's weight cache on): what the per-call conversion costs.
    def step_cached(self, s: int = 0):
        G, w = self.G, self.w
        s %= self.slots
        G.gpt2_block_forward(self.ctx, self.inp[s]["x"], self.params[0], w.B, w.T, w.d, w.n_head,
                             out=self.res[s])

    def capture_graph(self):
        torch = self.torch
        self.step()  # first call outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        self.graph = g

    def capture_slot_graphs(self):
        """One CUDA graph of the step per input/result slot (the same launches
        as step(s), replayed without host work)."""
        torch = self.torch
        graphs = []
        for s in range(self.slots):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self.step(s)
            graphs.append(g)
        torch.cuda.synchronize()
        return graphs

    def run(self, s: int = 0):
        if self.graph is not None:
            self.graph.replay()
        else:
            self.step(s)

    # The end-to-end step's copies: the step's inputs from pinned host memory
    # into slot s, and slot s's result back to pinned host memory.
    def stage_input(self, s: int):
        for k, t in self.inp[s].items():
            t.copy_(self.inp_host[k], non_blocking=True)

    def fetch_result(self, s: int):
        self.res_host[s].copy_(self.res[s], non_blocking=True)

    def e2e_bytes(self):
        h2d = sum(t.numel() * t.element_size() for t in self.inp[0].values())
        d2h = self.res[0].numel() * self.res[0].element_size()
        return h2d, d2h

    def close(self):
        self.torch.cuda.synchronize()
        self.graph = None
        self.ctx.close()


def reduce_over_ranks(times_ms, device):
    """Maximum of each per-step time over all ranks (the slowest rank sets the
    whole job's step time); a no-op without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(t) for t in times_ms]
    t = torch.tensor(times_ms, device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(tokens_per_rank, world_size, ms_per_step):
    """Whole-job tokens/s: every rank processes its own replica's tokens."""
    return tokens_per_rank * world_size / (ms_per_step / 1e3)


def timed_steps(fn, K, barrier, torch):
    """Per-step times (ms) of K steps fn(0) .. fn(K - 1), back to back."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier()
    torch.cuda.synchronize()
    for i in range(K):
        starts[i].record()
        fn(i)
        ends[i].record()
    torch.cuda.synchronize()
    barrier()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def timed_e2e(r, K, barrier, torch):
    """Mean time of K end-to-end steps: step i copies its input from pinned
    host memory into device slot i % slots (own stream), runs after that copy
    (compute stream), and copies its result back to pinned host memory (own
    stream); with two or more slots the copies of one step overlap the compute
    of its neighbours.  One event pair brackets all K steps, the last result
    copy included, so every copy is inside the timed region."""
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    n = r.slots
    ev_in = [torch.cuda.Event() for _ in range(K)]
    ev_done = [torch.cuda.Event() for _ in range(K)]
    ev_out = [torch.cuda.Event() for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(comp)
    h2d.wait_stream(comp)
    d2h.wait_stream(comp)
    t_host = time.perf_counter()
    for i in range(K):
        s = i % n
        with torch.cuda.stream(h2d):
            if i >= n:
                h2d.wait_event(ev_done[i - n])  # step i - n no longer reads slot s
            r.stage_input(s)
            ev_in[i].record(h2d)
        if i >= n:
            comp.wait_event(ev_out[i - n])      # slot s's last result copied out
        comp.wait_event(ev_in[i])
        r.run(s)
        ev_done[i].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[i])
            r.fetch_result(s)
            ev_out[i].record(d2h)
    comp.wait_stream(h2d)
    comp.wait_stream(d2h)
    end.record(comp)
    t_host = time.perf_counter() - t_host
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end) / K, t_host * 1e3 / K


def link_probe(r, torch, reps=5):
    """The host link as this run's end-to-end copies see it: the step's input
    copy (pinned host -> slot 0) alone, its result copy (slot 0 -> pinned
    host) alone, and the two at once on separate streams, each repeated reps
    times and timed with events.  Returns GB/s per direction and the copy time
    of one step at the concurrent rate, to set beside the device step time."""
    h2d_b, d2h_b = r.e2e_bytes()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(use_in, use_out):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(s_in)
        s_out.wait_event(a)
        for _ in range(reps):
            if use_in:
                with torch.cuda.stream(s_in):
                    r.stage_input(0)
            if use_out:
                with torch.cuda.stream(s_out):
                    r.fetch_result(0)
        s_in.wait_stream(s_out)
        b.record(s_in)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / reps  # seconds per repetition

    timed(True, True)  # first touch of the buffers
    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    out = {"h2d_gbs": h2d_b / t_in / 1e9, "d2h_gbs": d2h_b / t_out / 1e9,
           "both_gbs_per_direction": max(h2d_b, d2h_b) / t_both / 1e9,
           "copy_ms_per_step": t_both * 1e3}
    return out


# -------------------------------------------------------------- CPU oracle --
def oracle_sample(w: S.Workload, seed: int, T_sample: int):
    """A bounded sample of the workload for the fp64 oracle: one sequence of
    T_sample new tokens (block / forward), or one sequence's decode step.
    Returns (callable, tokens)."""
    from oracle import gpt2_oracle as O
    if w.kind == "block":
        p = S.block_params(w, seed)
        x = S.block_input(w, seed)[:1, :T_sample]
        return (lambda: O.block_forward(x, p, w.n_head)), T_sample
    p = S.model_params(w, seed)
    ids = S.token_ids(w, seed)[:1]
    if w.kind in ("forward", "forward_loss", "forward_topk"):
        ids = ids[:, :T_sample]
        if w.kind == "forward":
            return (lambda: O.forward(ids, p, w.n_head)), T_sample
        if w.kind == "forward_topk":
            return (lambda: O.top_k(O.forward(ids, p, w.n_head)[0], TOPK)), T_sample
        tg = np.concatenate([ids[:, 1:], np.full((1, 1), -1, ids.dtype)], axis=1)
        return (lambda: O.next_token_loss(O.forward(ids, p, w.n_head)[0], tg)), T_sample
    past = np.stack([S.past_kv(w, seed, 0, layer) for layer in range(w.n_layer)])[None]
    return (lambda: O.forward(ids, p, w.n_head, past=past)), 1


def time_oracle(w, seed, budget_s=15.0):
    T_sample = w.T
    fn, tokens = oracle_sample(w, seed, T_sample)
    t0 = time.perf_counter()
    fn()
    one = time.perf_counter() - t0
    reps = max(1, min(20, int(budget_s / max(one, 1e-3))))
    if reps > 1:
        t0 = time.perf_counter()
        for _ in range(reps):
            fn()
        one = (time.perf_counter() - t0) / reps
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    sample = (f"1 sequence x {tokens} token(s) of {w.name}"
              + (f" with a {w.t_past}-position cache" if w.kind == "decode" else "")
              + f", {reps} repetition(s), fp64 numpy")
    return {"value": tokens / one, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample}


def reference_arm(args, w):
    """The oracle as the reference arm: K timed steps of a bounded sample."""
    T_s = w.T if w.kind != "decode" else 1
    fn, tokens = oracle_sample(w, args.seed, T_s)
    t0 = time.perf_counter()
    fn()
    one = time.perf_counter() - t0
    budget = 150.0 / max(1, args.steps + args.warmup)
    if w.kind != "decode" and one > budget:
        T_s = max(16, int(w.T * budget / one))
        fn, tokens = oracle_sample(w, args.seed, T_s)
    for _ in range(max(0, args.warmup - 1)):
        fn()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        fn()
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = tokens / (ms / 1e3)
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", os.cpu_count() or 1))
    sample = f"1 sequence x {tokens} token(s) of {w.name} per step, fp64 numpy"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, args, "not applicable: host cores"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def workload_config(w, args, l2_note):
    cfg = {"workload": w.name, "kind": w.kind, "d": w.d, "n_head": w.n_head, "B": w.B, "T": w.T,
           "seed": args.seed, "l2": l2_note,
           "parallelism": f"replicas x{args.gpus}"}
    if w.kind != "block":
        cfg.update(n_layer=w.n_layer, n_vocab=w.n_vocab)
    if w.kind == "decode":
        cfg.update(t_past=w.t_past, cuda_graph=True,
                   weights="fp16 working copies made once before the timed steps")
    else:
        cfg.update(weights="bf16 -> fp16 working copies made inside every step")
    return cfg


def kernel_table(prof, peaks, steps):
    """Per kernel kind: launches, time, share of the step, achieved rate and
    its roofline fraction, the roofline being max(algorithmic flops / tensor
    peak, algorithmic bytes / HBM peak) per launch."""
    total = sum(x["ms"] for x in prof.values())
    out = {}
    for kind, rec in prof.items():
        n = rec["launches"]
        avg_s = rec["ms"] / 1e3 / n
        t_flop = rec["flops"] / n / (peaks["bf16_tflops"] * 1e12)
        t_byte = rec["bytes"] / n / (peaks["hbm_gbs"] * 1e9)
        e = {"launches_per_step": n / steps, "ms_per_launch": rec["ms"] / n,
             "share": rec["ms"] / total}
        if rec["flops"] > 0:
            e["tflops"] = rec["flops"] / n / avg_s / 1e12
        if rec["bytes"] > 0:
            e["gbs"] = rec["bytes"] / n / avg_s / 1e9
        if t_flop > 0 or t_byte > 0:
            e["bound"] = "tensor" if (kind in TENSOR_KINDS and t_flop >= t_byte) else "hbm"
            e["frac"] = max(t_flop, t_byte) / avg_s
        out[kind] = e
    return out


def roofline_entry(prof, peaks, workload):
    """The dominant kernel (most time per step) against its roofline."""
    top = max(prof, key=lambda k: prof[k]["ms"])
    rec = prof[top]
    n = rec["launches"]
    avg_s = rec["ms"] / 1e3 / n
    t_flop = rec["flops"] / n / (peaks["bf16_tflops"] * 1e12)
    t_byte = rec["bytes"] / n / (peaks["hbm_gbs"] * 1e9)
    if top in TENSOR_KINDS and t_flop >= t_byte:
        roof = {"bound": "tensor", "achieved": rec["flops"] / n / avg_s / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
        alg = rec["flops"] / n
    else:
        roof = {"bound": "hbm", "achieved": rec["bytes"] / n / avg_s / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s"}
        alg = rec["bytes"] / n
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = top
    roof["peak_source"] = peaks["source"]
    roof["traffic"] = ncu_traffic(top, workload)
    roof["algorithmic_per_launch"] = alg
    return roof


def measure(r, args, barrier, torch, G, e2e: bool):
    """Warm-up, K device-resident steps under the clock sampler, (decode) the
    same steps without the graph, (e2e) the pipelined end-to-end steps, and a
    profiled pass of K steps with every kernel bracketed by events."""
    if r.w.kind == "decode":
        r.capture_graph()
    for i in range(max(args.warmup, r.slots)):
        r.run(i)
    torch.cuda.synchronize()
    st = G.gpt2_sync_status(r.ctx)
    if st != G.GPT2_OK:
        raise SystemExit(f"{r.w.name}: device error after warm-up: {G.status_string(st)}")
    out = {}
    # The end-to-end steps run before the clock sampler's nvidia-smi starts:
    # host-memory copies issued just after such a process exits were held up
    # for 1-30 ms (4 of 40 end-to-end runs that followed one, 1 of 80
    # otherwise), while kernels ran at their usual speed.
    out["ms_e2e"], out["host_ms_e2e"] = timed_e2e(r, args.steps, barrier, torch) if e2e \
        else (None, None)
    out["link"] = link_probe(r, torch) if e2e else None
    with ClockSampler(torch.cuda.current_device()) as clk:
        out["times"] = timed_steps(r.run, args.steps, barrier, torch)
    out["clocks"] = clk.summary()
    out["ms_eager"] = None
    out["ms_graph"] = None
    if r.graph is not None:
        t = timed_steps(r.step, args.steps, barrier, torch)
        out["ms_eager"] = sum(t) / len(t)
    else:
        # The same steps replayed from CUDA graphs, one per slot.
        graphs = r.capture_slot_graphs()
        t = timed_steps(lambda i: graphs[i % len(graphs)].replay(), args.steps, barrier, torch)
        out["ms_graph"] = sum(t) / len(t)
        del graphs
    out["ms_cached"] = None
    if r.w.kind == "block" and r.w.dtype == "bf16":
        G.gpt2_ctx_cache_weights(r.ctx, True)
        r.step_cached(0)  # makes the copies
        t = timed_steps(r.step_cached, args.steps, barrier, torch)
        out["ms_cached"] = sum(t) / len(t)
        G.gpt2_ctx_cache_weights(r.ctx, False)
    G.gpt2_profile_enable(r.ctx, True)
    G.gpt2_profile_reset(r.ctx)
    timed_steps(r.step, args.steps, barrier, torch)
    out["prof"] = G.gpt2_profile_read(r.ctx)
    G.gpt2_profile_enable(r.ctx, False)
    st = G.gpt2_sync_status(r.ctx)
    if st != G.GPT2_OK:
        raise SystemExit(f"{r.w.name}: device error in the timed region: {G.status_string(st)}")
    return out


def workload_entry(w, r, m, peaks, args, ws, device):
    """The summary of one extra configuration for the `workloads` key."""
    ms, ms_med = reduce_over_ranks([sum(m["times"]) / len(m["times"]),
                                    statistics.median(m["times"])], device)
    e = {"config": workload_config(w, args, r.l2_note), "ms_per_step": ms, "ms_per_step_median": ms_med,
         "value": job_throughput(r.tokens, ws, ms), "unit": "tokens/s",
         "tflops": workload_flops(w) * ws / (ms / 1e3) / 1e12,
         "e2e_roofline": e2e_roofline(m["prof"], peaks, args.steps, ms),
         "roofline": roofline_entry(m["prof"], peaks, w.name),
         "kernels": kernel_table(m["prof"], peaks, args.steps),
         "gpu_launches": int(round(sum(v["launches"] for v in m["prof"].values()))),
         "clocks": m["clocks"]}
    if m["ms_eager"] is not None:
        e["eager_ms_per_step"] = reduce_over_ranks([m["ms_eager"]], device)[0]
    if m["ms_graph"] is not None:
        e["graph_ms_per_step"] = reduce_over_ranks([m["ms_graph"]], device)[0]
    if m["ms_cached"] is not None:
        e["cached_weights"] = cached_entry(r, m, ws, device)
    return e


def cached_entry(r, m, ws, device):
    ms = reduce_over_ranks([m["ms_cached"]], device)[0]
    return {"ms_per_step": ms, "value": job_throughput(r.tokens, ws, ms), "unit": "tokens/s",
            "note": "the same step on one weight set whose fp16 working copies an earlier call "
                    "made (weight cache on; x still rotated): the difference from ms_per_step is "
                    "the per-call bf16 -> fp16 weight conversion"}


# --------------------------------------------------------------------- main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="block_bf16_d768", choices=sorted(S.WORKLOADS))
    ap.add_argument("--extra", default=",".join(EXTRA_WORKLOADS),
                    help="comma-separated configurations timed after the main one "
                         "(default: the full forward, the XL block and decode; '' for none)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    w = S.WORKLOADS[args.workload]
    extras = [S.WORKLOADS[n] for n in args.extra.split(",") if n and n != w.name]
    ws, rank, local = dist_env()

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(reference_arm(args, w)), flush=True)
        return 0

    import torch
    if args.warmup < 3:
        args.warmup = 3
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    barrier = lambda: None  # noqa: E731
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        barrier = lambda: dist.barrier()  # noqa: E731

    from gpt_pre_norm_gb300 import binding as G
    pool = ThreadPoolExecutor(max_workers=os.cpu_count() or 4)
    l2 = l2_bytes(torch, device)
    peaks = load_peaks()

    r = Runner(w, args.seed + rank, device, pool, l2)
    m = measure(r, args, barrier, torch, G, e2e=True)
    times, prof = m["times"], m["prof"]
    ms, ms_e2e, ms_med = reduce_over_ranks(
        [sum(times) / len(times), m["ms_e2e"], statistics.median(times)], device)
    ms_eager = reduce_over_ranks([m["ms_eager"]], device)[0] if m["ms_eager"] is not None else None
    ms_graph = reduce_over_ranks([m["ms_graph"]], device)[0] if m["ms_graph"] is not None else None
    tokens_rank = r.tokens
    h2d, d2h = r.e2e_bytes()
    cached = cached_entry(r, m, ws, device) if m["ms_cached"] is not None else None
    l2_note, slots = r.l2_note, r.slots
    r.close()
    del r
    gc.collect()
    torch.cuda.empty_cache()

    # The other configurations, one after the other (each rank a replica).
    extra_entries = {}
    for we in extras:
        re_ = Runner(we, args.seed + rank, device, pool, l2)
        me = measure(re_, args, barrier, torch, G, e2e=False)
        extra_entries[we.name] = workload_entry(we, re_, me, peaks, args, ws, device)
        re_.close()
        del re_
        gc.collect()
        torch.cuda.empty_cache()
    pool.shutdown()
    if rank != 0:
        return 0

    value = job_throughput(tokens_rank, ws, ms)
    flops = workload_flops(w)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "ms_per_step_median": ms_med,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16/fp16" if w.dtype == "bf16" else "f32",
        "dtype_detail": DTYPE_DETAIL if w.dtype == "bf16" else "fp32 storage and arithmetic",
        "data": "synthetic",
        "config": workload_config(w, args, l2_note),
        "tflops": flops * ws / (ms / 1e3) / 1e12,
        "tflops_frac_of_bf16_peak": flops * ws / (ms / 1e3) / 1e12 / peaks["bf16_tflops"],
        "roofline": roofline_entry(prof, peaks, w.name),
        "e2e_roofline": e2e_roofline(prof, peaks, args.steps, ms),
        "e2e": {"value": job_throughput(tokens_rank, ws, ms_e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": f"{slots} device input/result slots; copies on their own "
                             "streams",
                "link": m["link"],
                "host_enqueue_ms_per_step": m["host_ms_e2e"]},
        "gpu_launches": int(round(sum(v["launches"] for v in prof.values()))),
        "clocks": m["clocks"],
        "kernels": kernel_table(prof, peaks, args.steps),
        "workloads": extra_entries,
    }
    if ms_eager is not None:
        line["eager_ms_per_step"] = ms_eager  # the same step without the CUDA graph
    if ms_graph is not None:
        line["graph_ms_per_step"] = ms_graph  # the same steps replayed from CUDA graphs
    if cached is not None:
        line["cached_weights"] = cached
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = time_oracle(w, args.seed)
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
