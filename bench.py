#!/usr/bin/env python
"""Dual-flow decode benchmark on B300: tokens/s of the decode step and achieved HBM bandwidth.

Default workload (--workload dense): the 24-layer dense dual-flow model (d_model 2048, 16/4 heads
of 128, SwiGLU 8192, vocab 32000), batch 32, every sequence with 4096 cached positions, bf16
storage / fp32 accumulation, synthetic seeded inputs generated in place. One step = one decode
step of both flows for the whole batch (embeddings -> 24 x {QKV + query coupling + RoPE + KV
append, shared-KV attention, O projection, gate/up + SwiGLU + b coupling, down + c coupling, with
RMSNorm carried between them} -> LM head), replayed as one CUDA graph through dualflow_step.
Other workloads: moe (16 layers, 16 experts, top-2 / top-4, batch 64), attn (attention-only layer,
batch 8, 2048 positions), paged (attention-only layer, batch 64, ragged 1k-32k positions, paged).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Under torchrun every rank runs its own replica (independent sequences: no data-path collective);
value = total tokens of all ranks / max-over-ranks step time. --impl reference times the CPU
fp64 oracle on a bounded sample of the same workload and scales it to the same metric.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "dual-flow decode tokens/s at 1 B300; achieved HBM GB/s vs ~8 TB/s roofline"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6400.0


class Replicas:
    """Multi-GPU mode: one replica of the decode path per rank. Sequences are independent and each
    sequence's cache lives with it, so the batch shards across ranks with no exchange on the data
    path; the only collectives are the timing bookkeeping around it: a barrier on both sides of
    every timed region and the maximum of each measured time over the ranks."""

    def __init__(self, rank: int = 0, world: int = 1, device=None):
        self.rank, self.world, self.device = rank, world, device

    @staticmethod
    def from_env() -> tuple[int, int, int]:
        """(RANK, WORLD_SIZE, LOCAL_RANK) as torchrun sets them; a single process without it."""
        env = os.environ
        return int(env.get("RANK", "0")), int(env.get("WORLD_SIZE", "1")), int(env.get("LOCAL_RANK", "0"))

    def barrier(self) -> None:
        if self.world > 1:
            import torch.distributed as dist
            dist.barrier()

    def max(self, *vals: float) -> list[float]:
        """Each value's maximum over the ranks (every rank gets the result)."""
        if self.world == 1:
            return [float(v) for v in vals]
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=self.device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return [float(x) for x in t.tolist()]

    def rate(self, units_per_rank: float, seconds: float) -> float:
        """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
        return self.world * units_per_rank / seconds


def step_percentiles(times_ms) -> dict:
    """p10 / p50 / p90 (nearest rank) of per-step times."""
    t = sorted(float(x) for x in times_ms)
    n = len(t)
    pick = lambda q: t[min(n - 1, max(0, -(-q * n // 100) - 1))]  # noqa: E731  nearest-rank percentile
    return {"n": n, "p10_ms": pick(10), "p50_ms": pick(50), "p90_ms": pick(90)}


def load_peaks() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def workload(name: str = "dense"):
    from dfsynth import workloads as W
    return {"dense": W.DENSE_24L_B32_L4096, "moe": W.MOE_16L_B64, "attn": W.ATTN_B8_L2048,
            "paged": W.PAGED_RAGGED_B64, "prefill": W.DENSE_24L_B32_L4096, "dense_paged": W.DENSE_PAGED_RAGGED_B32,
            "prefill_moe": W.MOE_16L_B64}[name]


PREFILL_TOKENS = 512  # prompt tokens per sequence of the prefill workload (from an empty cache)


def prefill_flops(w, n_tok: int) -> float:
    """Algorithmic FLOPs of the primary-only prefill of n_tok tokens per sequence from position 0:
    2 per weight element per row for the projections of every layer (a MoE layer: the router and
    the topk_primary experts each row chose), and the causal attention (2 x 2 x D per head per
    (query, attended key) pair)."""
    qkv = (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim * w.d_model
    mlp = 3 * w.ffn_hidden * w.d_model
    if w.n_experts > 0:
        mlp = w.n_experts * w.d_model + w.topk_primary * mlp
    layer = qkv + w.d_model * w.n_q_heads * w.head_dim + mlp
    rows = w.batch * n_tok
    pairs = w.batch * n_tok * (n_tok + 1) / 2
    return w.n_layers * (2.0 * layer * rows + 4.0 * w.head_dim * w.n_q_heads * pairs)


def step_bytes(w, experts_touched=None) -> dict:
    """Algorithmic HBM bytes of one step: every weight once (for MoE, the router and the experts
    some row selected, counted per layer), every cached K1/V1 element once, the appended entries,
    the gathered embedding rows and the fp32 logits."""
    from dfsynth import workloads as W
    es = 2 if w.dtype == "bf16" else 4
    weights = sum(s.numel for s in W.global_specs(w) if s.name in ("W_lm", "g_final")) * es
    for l in range(w.n_layers):
        for spec in W.layer_specs(w, l):
            if spec.name.endswith((".K", ".V")):
                continue
            n = spec.numel
            if spec.name.endswith((".We_gu", ".We_d")) and experts_touched is not None:
                n = n // w.n_experts * int(experts_touched[l])
            weights += n * es
    lens = w.seq_lens()
    kv_per_pos = w.n_kv_heads * w.head_dim * es * 2  # K and V
    kv_read = int(lens.sum()) * kv_per_pos * w.n_layers
    kv_write = w.batch * kv_per_pos * w.n_layers
    emb = 2 * w.batch * w.d_model * es
    logits = 2 * w.batch * w.vocab * 4
    # one attention launch reads positions 0..L_b (the appended one included), q, and writes o
    qo = 2 * w.batch * w.n_q_heads * w.head_dim * es
    attn = int((lens + 1).sum()) * kv_per_pos + 2 * qo
    return dict(total=weights + kv_read + kv_write + emb + logits, weights=weights, kv_read=kv_read,
                kv_write=kv_write, attention_per_launch=attn)


def family_bytes(w, experts_touched=None) -> dict:
    """Algorithmic HBM bytes per step of each kernel family of the decode step (the unit a family's
    roofline is taken on): its weights once (for MoE, the router and every touched expert's
    weights), the activations it reads and writes once, and for attention every cached K1/V1 entry
    once. Sums to at least step_bytes()['total'] (the activations are counted here only)."""
    es = 2
    B, d, F, V = w.batch, w.d_model, w.ffn_hidden, w.vocab
    M = 2 * B
    qd, kvd = w.q_dim, w.kv_dim
    nL = w.n_layers
    sb = step_bytes(w, experts_touched)
    out = {
        "norm": M * d * es + M * d * 4 + M * d * es,  # embedding rows, residual, first norm operand
        "qkv": nL * ((qd + 2 * kvd) * d * es + M * d * es + M * qd * es + B * 2 * kvd * es),
        "attention": nL * sb["attention_per_launch"],
        "o_proj": nL * (d * qd * es + M * qd * es + 2 * M * d * 4 + M * d * es),
        "lm_head": V * d * es + M * d * es + M * V * 4,
    }
    if w.n_experts == 0:
        out["gate_up"] = nL * (2 * F * d * es + M * d * es + M * F * es)
        out["down"] = nL * (d * F * es + M * F * es + 2 * M * d * 4 + M * d * es)
    else:
        E = w.n_experts
        touched = list(experts_touched) if experts_touched is not None else [E] * nL
        kmax = max(w.topk_primary, w.topk_aux)
        out["gate_up"] = sum(E * d * es + M * E * 4 + t_ * 2 * F * d * es + M * d * es + M * kmax * F * es
                             for t_ in touched)
        out["down"] = sum(t_ * d * F * es + M * kmax * F * es + M * kmax * d * 4 + 2 * M * d * 4 + M * d * es
                          for t_ in touched)
    return out


FAMILY_LAUNCHES = {"norm": 1, "lm_head": 1}  # per step; the per-layer families launch once per layer


def call_bytes(w) -> dict:
    """Algorithmic HBM bytes of one attention-only call: Wq once, K1/V1 of the cached positions
    once, q1 and h2 read, both flows' outputs written."""
    es = 2
    lens = w.seq_lens()
    kv = int(lens.sum()) * w.n_kv_heads * w.head_dim * es * 2
    wq = w.q_dim * w.d_model * es
    act = (w.batch * w.q_dim + w.batch * w.d_model + w.q_dim) * es
    out = 2 * w.batch * w.q_dim * es
    return dict(total=kv + wq + act + out, kv_read=kv, weights=wq)


def attention_traffic() -> float | None:
    """DRAM bytes per attention launch from the committed ncu summary, if the kernel is unchanged."""
    prof = os.path.join(ROOT, "profiles", "attention_dense_24l_b32_l4096.md")
    src = os.path.join(ROOT, "dual_flow_decode_dualflow_b300", "csrc", "attn_bf16.cu")
    try:
        txt = open(prof).read()
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    rec = dict(line.split(":", 1) for line in txt.splitlines() if line.startswith(("source_sha256:", "traffic_bytes_per_launch:")))
    if rec.get("source_sha256", "").strip() != sha:
        return None
    try:
        return float(rec["traffic_bytes_per_launch"].strip())
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def mark(self, start: bool):
        if start:
            self.t_start = time.time()
        else:
            self.t_end = time.time()

    def __enter__(self):
        self.t_start = self.t_end = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200", "-i",
                 str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        import datetime
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                clk, mxv = float(f[2]), float(f[3])
            except ValueError:
                continue
            if self.t_start is not None and not (self.t_start - 0.05 <= ts <= (self.t_end or ts) + 0.05):
                continue
            sm.append(clk)
            mx = mxv
            for n, v in zip(names, f[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


class PrefillOracleSample:
    """The CPU oracle's prefill on a bounded sample: one sequence, the first layer, the first
    n_sample prompt tokens from an empty cache; scaled to the workload by sequences, tokens and
    layers (the oracle's prefill runs one decode step per position, logits included)."""

    def __init__(self, w, n_sample: int, n_tok: int):
        import oracle as O
        from tests import gpu_harness as H
        self.O, self.w, self.n_sample, self.n_tok = O, w, n_sample, n_tok
        ws = w.replace(n_layers=1, batch=1)
        self.layers = [H.LazyLayers(ws)[0]]
        self.glob = {"E1": H.LazyRows(ws, "E1"), "E2": H.LazyRows(ws, "E2"), "W_lm": H.host_f64(ws, "W_lm"),
                     "g_final": H.host_f64(ws, "g_final")}
        self.hp = H.hparams(ws)
        self.prompt = np.random.default_rng(51).integers(0, w.vocab, size=(1, n_sample))

    def time(self) -> float:
        caches = [self.O.DenseCache(K=np.zeros((1, self.w.n_kv_heads, self.n_sample, self.w.head_dim)),
                                    V=np.zeros((1, self.w.n_kv_heads, self.n_sample, self.w.head_dim)))]
        t0 = time.perf_counter()
        self.O.prefill(self.hp, self.glob, self.layers, caches, self.prompt, np.zeros(1, dtype=np.int64))
        return time.perf_counter() - t0

    def full(self, seconds: float) -> float:
        # per position: one layer + the LM head of the oracle's step; scale to all layers + head
        return seconds * self.w.batch * (self.n_tok / self.n_sample) * (self.w.n_layers + 1) / 2

    def describe(self) -> str:
        return (f"oracle (numpy fp64) prefill of {self.n_sample} prompt tokens of 1 of {self.w.batch} sequences x 1 of "
                f"{self.w.n_layers} layers (+ the LM head its per-position steps compute), scaled to {self.n_tok} "
                f"tokens x {self.w.batch} sequences x (layers + 1)")


class OracleSample:
    """The CPU oracle on a bounded sample of the workload: the first `n_layers` layers and the
    sequences in `rows`, inputs drawn and widened beforehand. time_step() times one oracle decode
    step on a subset of those rows; full_step() scales it to the whole workload's step."""

    def __init__(self, w, rows, n_layers):
        import oracle as O
        from tests import gpu_harness as H
        self.O, self.w, self.rows, self.n_layers = O, w, list(rows), n_layers
        ws = w.replace(n_layers=n_layers)
        self.layers = [H.LazyLayers(ws)[l] for l in range(n_layers)]
        self.caches = []
        for l in range(n_layers):
            if ws.paged:  # the pages of the sampled sequences, drawn on first use
                self.caches.append(H.oracle_cache(ws, l))
                continue
            kc, vc = H.LazySeqCache(ws, f"L{l}.K"), H.LazySeqCache(ws, f"L{l}.V")
            self.caches.append(O.DenseCache({b: kc[b] for b in self.rows}, {b: vc[b] for b in self.rows}))
        self.glob = {"E1": H.LazyRows(ws, "E1"), "E2": H.LazyRows(ws, "E2"), "W_lm": H.host_f64(ws, "W_lm"),
                     "g_final": H.host_f64(ws, "g_final")}
        self.tokens, self.lens, self.hp = ws.tokens(), ws.seq_lens(), H.hparams(ws)

    def time_step(self, rows) -> float:
        t0 = time.perf_counter()
        self.O.decode_step(self.hp, self.glob, self.layers, self.caches, self.tokens, self.lens, aux_on=True,
                           mirror=True, rows=rows)
        return time.perf_counter() - t0

    def full_step(self, seconds: float, n_rows: int) -> float:
        # the LM head costs about one layer: scale (sample layers + head) to (all layers + head)
        return seconds * (self.w.batch / n_rows) * (self.w.n_layers + 1) / (self.n_layers + 1)

    def describe(self, n_rows: int) -> str:
        return (f"oracle (numpy fp64) decode step of both flows on {n_rows} of {self.w.batch} sequences x "
                f"{self.n_layers} of {self.w.n_layers} layers + LM head (inputs drawn beforehand), scaled to the "
                f"full step by sequences and by (layers + 1)")


def host_cpu() -> dict:
    """The host's CPU model and the cores this process may run on."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        cores = len(os.sched_getaffinity(0))
    except AttributeError:
        cores = os.cpu_count() or 1
    return {"model": model, "cores": cores}


def _openblas_calls():
    """(set_num_threads, get_num_threads) of the OpenBLAS that numpy loaded, found through its
    exported C entry points (the symbol names carry a suffix in numpy's own build), or None."""
    import ctypes
    paths = set()
    try:
        with open("/proc/self/maps") as f:
            for line in f:
                if "openblas" in line.lower() and ".so" in line:
                    paths.add(line.split()[-1])
    except OSError:
        return None
    names = ("scipy_openblas_set_num_threads64_", "openblas_set_num_threads64_", "scipy_openblas_set_num_threads",
             "openblas_set_num_threads")
    for path in sorted(paths):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for n in names:
            if hasattr(lib, n):
                getter = getattr(lib, n.replace("set_num_threads", "get_num_threads"), None)
                setter = getattr(lib, n)
                setter.argtypes, setter.restype = [ctypes.c_int], None
                if getter is not None:
                    getter.argtypes, getter.restype = [], ctypes.c_int
                return setter, getter
    return None


class OracleThreads:
    """Runs the oracle with its BLAS library on every core this process may use (the oracle's
    matrix products are where its time goes); `threads` is the count in effect inside, read back
    from the library."""

    def __enter__(self):
        np.zeros(1) @ np.zeros(1)  # numpy's BLAS is loaded
        self.cores = host_cpu()["cores"]
        self._restore = None
        calls = _openblas_calls()
        if calls is not None:
            setter, getter = calls
            before = getter() if getter is not None else None
            setter(self.cores)
            self.threads = getter() if getter is not None else self.cores
            if before is not None:
                self._restore = lambda: setter(before)
        else:
            self.threads = 1
        return self

    def __exit__(self, *exc):
        if self._restore is not None:
            self._restore()
        return False


def cpu_baseline_entry(value: float, unit: str, threads: int, sample: str, sample_s: float) -> dict:
    cpu = host_cpu()
    return {"value": value, "unit": unit, "cores": threads, "kind": "oracle", "sample": sample,
            "sample_seconds": sample_s, "host_cpu": cpu["model"], "host_cores": cpu["cores"],
            "parallelism": f"the oracle's BLAS calls on {threads} threads (numpy fp64); its Python loops on one"}


class AttentionOracleSample:
    """The CPU oracle's attention-only call on a bounded sample of the sequences of the workload,
    inputs drawn and widened beforehand (only the oracle's arithmetic is timed)."""

    def __init__(self, w, rows):
        import oracle as O
        from tests import gpu_harness as H
        self.O, self.w, self.rows = O, w, list(rows)
        self.hp = H.hparams(w)
        self.q1, self.h2 = H.host_f64(w, "q1"), H.host_f64(w, "h2")
        self.Wq, self.a = H.host_f64(w, "Wq"), H.host_f64(w, "a")
        self.lens = w.seq_lens()
        if w.paged:
            table, _ = w.page_table()
            kp, vp = H.LazyPages(w, "K"), H.LazyPages(w, "V")
            pids = {int(table[b, j]) for b in self.rows for j in range(-(-int(self.lens[b]) // w.page_size))}
            self.cache = O.PagedCache({p: kp[p] for p in pids}, {p: vp[p] for p in pids}, table, w.page_size)
        else:
            kc, vc = H.LazySeqCache(w, "K"), H.LazySeqCache(w, "V")
            self.cache = O.DenseCache({b: kc[b] for b in self.rows}, {b: vc[b] for b in self.rows})

    def time_rows(self, rows) -> float:
        t0 = time.perf_counter()
        self.O.attention_only_step(self.hp, self.q1, self.h2, self.Wq, self.a, self.cache, self.lens, aux_on=True,
                                   mirror=True, rows=rows)
        return time.perf_counter() - t0

    def full_call(self, seconds: float, rows) -> float:
        # cost grows with the cached positions attended: scale by the workload's total over the sample's
        return seconds * float(self.lens.sum()) / float(sum(int(self.lens[b]) for b in rows))

    def describe(self, rows) -> str:
        return (f"oracle (numpy fp64) attention-only call of both flows on sequences {list(rows)} of {self.w.batch} "
                f"(inputs drawn beforehand), scaled to the full call by cached positions")


def run_reference(args, w) -> dict:
    """The reference arm: the CPU oracle, as it stands, on the host's cores (its BLAS calls on every
    usable core), one bounded sample per step -- one sequence, rotating through the batch, over the
    first layer and the LM head; for an attention-only workload one sequence's attention call; for
    prefill one sequence's first prompt tokens over one layer. Each sample's seconds are measured;
    the line's time per step is those seconds scaled to the whole workload (extrapolated, stated as
    such in the line)."""
    per, raw = [], []
    with OracleThreads() as th:
        if args.workload in ("prefill", "prefill_moe"):
            samp = PrefillOracleSample(w, 8, PREFILL_TOKENS)
            for i in range(args.warmup + args.steps):
                t = samp.time()
                if i >= args.warmup:
                    raw.append(t)
                    per.append(samp.full(t))
            desc = samp.describe()
        elif w.kind == "attention":
            lens = w.seq_lens()
            order = [int(b) for b in np.argsort(lens)[: max(1, min(8, w.batch))]]  # the shortest: bounded time
            samp = AttentionOracleSample(w, order)
            for i in range(args.warmup + args.steps):
                rows = [order[i % len(order)]]
                t = samp.time_rows(rows)
                if i >= args.warmup:
                    raw.append(t)
                    per.append(samp.full_call(t, rows))
            desc = samp.describe(order)
        else:
            rows = list(range(min(8, w.batch)))
            samp = OracleSample(w, rows, 1)
            for i in range(args.warmup + args.steps):
                t = samp.time_step([rows[i % len(rows)]])
                if i >= args.warmup:
                    raw.append(t)
                    per.append(samp.full_step(t, 1))
            desc = samp.describe(1)
    s = statistics.median(per)
    if args.workload in ("prefill", "prefill_moe"):
        metric, unit, value = "primary-only prefill tokens/s at 1 B300", "prefill tokens/s", w.batch * PREFILL_TOKENS / s
        config = {"workload": f"prefill_{w.name}", "batch": w.batch, "prompt_tokens": PREFILL_TOKENS, "layers": w.n_layers}
    else:
        metric, value = METRIC, w.batch / s
        unit = "tokens/s" if w.kind == "step" else "sequence-steps/s (one layer)"
        config = {"workload": w.name, "batch": w.batch, "ctx": w.ctx_len or f"{w.ctx_lo}-{w.ctx_hi}",
                  "layers": w.n_layers}
    return {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s * 1e3,
            "ms_per_step_kind": "extrapolated: the median timed sample scaled to the whole workload's step",
            "sample_ms": {"median": statistics.median(raw) * 1e3, "min": min(raw) * 1e3, "max": max(raw) * 1e3,
                          "n": len(raw)},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": cpu_baseline_entry(value, unit, th.threads, desc, statistics.median(raw)),
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ours_attention(args, w, rank: int, world: int, local_rank: int) -> dict | None:
    """Attention-only workloads: one step = one dualflow_decode_attention call for the batch (the
    auxiliary query projection with coupling and RoPE, then the shared-KV attention). Inputs are
    rotated over enough copies that the working set of a round exceeds L2 three times over; the
    round of calls is replayed as a CUDA graph."""
    import torch

    import dual_flow_decode_dualflow_b300 as dfl
    from tests import gpu_harness as H

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    reps = Replicas(rank, world, dev)
    nb = call_bytes(w)
    copies = max(1, min(16, -(-3 * 126 * 2 ** 20 // nb["total"])))
    runs = [H.DeviceRun(w, dev) for _ in range(copies)]
    for r in runs:  # back-to-back calls write only o: each may start while the previous finishes
        dfl.dualflow_set_call_chaining(r.ctx, 1)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(2):
            for r in runs:
                r.attention(aux_on=1, stream=stream)
    stream.synchronize()
    for r in runs:
        st = dfl.dualflow_sync_status(r.ctx)
        if st != 0:
            raise RuntimeError(f"device status: {dfl.dualflow_status_string(st)}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
        for r in runs:
            r.attention(aux_on=1, stream=stream)
    rounds = max(1, args.steps // copies)
    steps = rounds * copies

    def timed(sampler=None):
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup // copies)):
                graph.replay()
        stream.synchronize()
        reps.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with (sampler if sampler is not None else _Null()):
            if sampler is not None:
                sampler.mark(True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(rounds):
                    graph.replay()
                e1.record(stream)
            e1.synchronize()
            if sampler is not None:
                sampler.mark(False)
        torch.cuda.synchronize()
        reps.barrier()
        (ms,) = reps.max(e0.elapsed_time(e1) / steps)
        return ms

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    ms = timed(sampler)
    # end to end: q1 and h2 from pinned host memory, the call, o back to host, every step
    r0 = runs[0]
    q1_h = r0.t["q1"].cpu().pin_memory()
    h2_h = r0.t["h2"].cpu().pin_memory()
    o_h = torch.empty(r0.o.shape, dtype=r0.o.dtype).pin_memory()
    e2e_steps = max(min(args.steps, 200), 3)
    for i in range(3 + e2e_steps):
        if i == 3:
            torch.cuda.synchronize()
            t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            r0.t["q1"].copy_(q1_h, non_blocking=True)
            r0.t["h2"].copy_(h2_h, non_blocking=True)
            r0.attention(aux_on=1, stream=stream)
            o_h.copy_(r0.o, non_blocking=True)
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    graph.reset()
    for r in runs:
        r.close()
    if rank != 0:
        return None
    peak, peak_kind = load_peaks()
    gbs = nb["total"] / (ms * 1e-3) / 1e9
    lens = w.seq_lens()
    rows = [int(b) for b in np.argsort(lens)[:2]]
    samp = AttentionOracleSample(w, rows)
    with OracleThreads() as th:
        raw_s = statistics.median(samp.time_rows(rows) for _ in range(3))
    cpu_s = samp.full_call(raw_s, rows)
    unit = "sequence-steps/s (one layer)"
    return {
        "metric": METRIC, "value": reps.rate(w.batch, ms * 1e-3), "unit": unit, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "accumulate": "f32",
        "data": "synthetic: seeded counter-hash generator, random-init weights of the workload's shapes",
        "config": {"workload": w.name, "d_model": w.d_model, "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "batch_per_gpu": w.batch,
                   "ctx": w.ctx_len or f"uniform {w.ctx_lo}-{w.ctx_hi}", "paged": w.paged,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"{copies} rotated input copies, {copies * nb['total'] / 1e6:.0f} MB per round vs 126 MB L2",
                   "launch": "round of calls replayed as a CUDA graph, each call chained to the previous one "
                             "(dualflow_set_call_chaining)"},
        "hbm": {"call_bytes": nb["total"], "achieved_gbs": gbs, "frac_of_8000": gbs / NOMINAL_HBM_GBS,
                f"frac_of_{peak_kind}": gbs / peak},
        "roofline": {"kernel": "dualflow_decode_attention call (Q2 projection + shared-KV attention)",
                     "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "bytes_per_launch": nb["total"],
                     "avg_launch_ms": ms, "traffic": None},
        "cpu_baseline": cpu_baseline_entry(w.batch / cpu_s, unit, th.threads, samp.describe(rows), raw_s),
        "e2e": {"value": reps.rate(w.batch, e2e_s), "unit": unit,
                "h2d_bytes_per_step": int((q1_h.numel() + h2_h.numel()) * 2), "d2h_bytes_per_step": int(o_h.numel() * 2),
                "api": "dualflow_decode_attention with q1, h2 copied from pinned host memory and o copied back, "
                       "stream sync per step"},
        "gpu_launches": 2 * steps, "launches_per_step": 2,
        "clocks": sampler.summary(),
    }


def run_ours_prefill(args, w, rank: int, world: int, local_rank: int) -> dict | None:
    """Primary-only prefill of PREFILL_TOKENS tokens per sequence from an empty cache, on the dense
    or the MoE model (the positions are rewritten by every repetition)."""
    import torch

    import dual_flow_decode_dualflow_b300 as dfl
    from tests import gpu_harness as H

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    reps = Replicas(rank, world, dev)
    run = H.DeviceRun(w, dev)
    stream = torch.cuda.Stream(device=dev)
    n_tok = PREFILL_TOKENS
    prompt_np = np.random.default_rng(52).integers(0, w.vocab, size=(w.batch, n_tok)).astype(np.int32)
    prompt = torch.from_numpy(prompt_np).to(dev)
    dfl.dualflow_prefill_reserve(run.ctx, w.batch * n_tok)
    steps = max(min(args.steps, 10), 3)

    def once(tokens):
        with torch.cuda.stream(stream):
            run.seq_len.zero_()
            dfl.dualflow_prefill(run.ctx, run.weights, run.kv, tokens, w.batch, n_tok, stream)

    for _ in range(args.warmup):
        once(prompt)
    stream.synchronize()
    reps.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with sampler:
        sampler.mark(True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                once(prompt)
            e1.record(stream)
        e1.synchronize()
        sampler.mark(False)
    torch.cuda.synchronize()
    reps.barrier()
    ms = e0.elapsed_time(e1) / steps
    st = dfl.dualflow_sync_status(run.ctx)
    if st != 0:
        raise RuntimeError(f"device status after the prefill: {dfl.dualflow_status_string(st)}")
    # end to end: the prompt copied from pinned host memory, the prefill, a synchronisation
    prompt_h = torch.from_numpy(prompt_np).pin_memory()
    prompt_d = torch.empty_like(prompt)
    e2e = []
    for i in range(3 + steps):
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            prompt_d.copy_(prompt_h, non_blocking=True)
        once(prompt_d)
        stream.synchronize()
        if i >= 3:
            e2e.append(time.perf_counter() - t0)
    ms, e2e_s = reps.max(ms, statistics.median(e2e))
    run.close()
    if rank != 0:
        return None
    flops = prefill_flops(w, n_tok)
    launches = 1 + (10 if w.n_experts else 5) * w.n_layers + 1  # embedding + layers + length advance
    peak = None
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, kind = float(json.load(f)["bf16_tflops_sustained"]), "measured sustained bf16 (cuBLAS 8192^3 loop)"
    except (OSError, KeyError, ValueError):
        peak, kind = 1400.0, "fallback sustained bf16"
    tflops = flops / (ms * 1e-3) / 1e12
    samp = PrefillOracleSample(w, 8, n_tok)
    with OracleThreads() as th:
        raw_s = statistics.median(samp.time() for _ in range(3))
    cpu_s = samp.full(raw_s)
    return {
        "metric": "primary-only prefill tokens/s at 1 B300", "value": reps.rate(w.batch * n_tok, ms * 1e-3),
        "unit": "prefill tokens/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32",
        "data": "synthetic: seeded counter-hash generator, random-init weights of the workload's shapes",
        "config": {"workload": f"prefill_{w.name}", "layers": w.n_layers, "d_model": w.d_model,
                   "batch_per_gpu": w.batch, "prompt_tokens": n_tok, "rows": w.batch * n_tok,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "compute-bound; weights re-read per 256-row block, no flush"},
        "roofline": {"kernel": f"whole prefill pass ({w.n_layers} x {{QKV, causal attention, O, "
                               + ("router, routing, gather, expert gate/up, expert down, combine})" if w.n_experts
                                  else "gate/up, down})"),
                     "bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s", "frac": tflops / peak,
                     "peak_kind": kind, "flops_per_step": flops, "traffic": None},
        "cpu_baseline": cpu_baseline_entry(w.batch * n_tok / cpu_s, "prefill tokens/s", th.threads, samp.describe(),
                                           raw_s),
        "e2e": {"value": reps.rate(w.batch * n_tok, e2e_s), "unit": "prefill tokens/s", "h2d_bytes_per_step": int(prompt_np.nbytes),
                "d2h_bytes_per_step": 0,
                "api": "dualflow_prefill with the prompt copied from pinned host memory, stream sync per call"},
        "gpu_launches": steps * launches, "launches_per_step": launches,
        "clocks": sampler.summary(),
    }


def run_ours(args, w, rank: int, world: int, local_rank: int) -> dict | None:
    import torch

    import dual_flow_decode_dualflow_b300 as dfl
    from tests import gpu_harness as H

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    reps = Replicas(rank, world, dev)
    run = H.DeviceRun(w, dev)
    stream = torch.cuda.Stream(device=dev)

    def timed(aux_on: int, steps: int, warmup: int, sampler=None):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                run.step(aux_on=aux_on, stream=stream)
        stream.synchronize()
        reps.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ctx = sampler if sampler is not None else _Null()
        with ctx:
            if sampler is not None:
                sampler.mark(True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                for _ in range(steps):
                    run.step(aux_on=aux_on, stream=stream)
                e1.record(stream)
            e1.synchronize()
            if sampler is not None:
                sampler.mark(False)
        torch.cuda.synchronize()
        reps.barrier()
        (ms,) = reps.max(e0.elapsed_time(e1) / steps)
        return ms

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    ms = timed(1, args.steps, args.warmup, sampler)
    st = dfl.dualflow_sync_status(run.ctx)
    if st != 0:
        raise RuntimeError(f"device status after the timed steps: {dfl.dualflow_status_string(st)}")
    experts_touched = None
    if w.n_experts > 0:  # distinct experts each layer's rows selected (their weights are read)
        kmax = max(w.topk_primary, w.topk_aux)
        ids = torch.empty((w.n_layers, 2, w.batch, kmax), dtype=torch.int32, device=dev)
        dfl.dualflow_expert_ids(run.ctx, ids, w.batch, stream)
        stream.synchronize()
        experts_touched = [len(set(x for x in ids[l].flatten().tolist() if x >= 0)) for l in range(w.n_layers)]
    _, launches = dfl.dualflow_profile_read(run.ctx)
    if args.quick:
        run.close()
        if rank == 0:
            return {"metric": METRIC, "value": reps.rate(w.batch, ms * 1e-3), "unit": "tokens/s",
                    "ms_per_step": ms, "steps": args.steps, "warmup": args.warmup, "n_gpus": world,
                    "config": {"workload": w.name, "layers": w.n_layers}, "note": "quick run (no extras)"}
        return None
    ms_primary = timed(0, max(args.steps // 2, 3), 3)

    # the distribution of single steps (an event between consecutive steps; outside the timed region)
    dist_steps = None
    try:
        n_d = 50
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_d + 1)]
        with torch.cuda.stream(stream):
            evs[0].record(stream)
            for i in range(n_d):
                run.step(aux_on=1, stream=stream)
                evs[i + 1].record(stream)
        evs[-1].synchronize()
        dist_steps = step_percentiles([evs[i].elapsed_time(evs[i + 1]) for i in range(n_d)])
    except Exception as exc:  # the distribution is a report only: never lose the run over it
        dist_steps = {"error": str(exc)[:200]}

    # per-kernel times inside the step: mode 2 = each launch's share of the pipelined step (device
    # end stamps, nothing serialised); mode 1 = CUDA event pairs around every launch (serialising:
    # each kernel's stand-alone duration, start-up included)
    nprof = max(min(args.steps, 50), 3)

    def profile(mode):
        dfl.dualflow_set_profiling(run.ctx, mode)
        fm = [0.0] * dfl.DF_PROF_FAMILIES
        fn = [0] * dfl.DF_PROF_FAMILIES
        with torch.cuda.stream(stream):
            for i in range(3 + nprof):
                run.step(aux_on=1, stream=stream)
                tt, nn = dfl.dualflow_profile_read(run.ctx)
                if i >= 3:
                    fm = [a + b for a, b in zip(fm, tt)]
                    fn = [a + b for a, b in zip(fn, nn)]
        dfl.dualflow_set_profiling(run.ctx, 0)
        return fm, fn

    fam_ms_graph, _ = profile(2)
    fam_ms, fam_n = profile(1)

    # end to end through the host-buffer decode call a user makes: the step's input tokens copied in
    # from pinned host memory, one decode step (step, mixture head, token choice, length advance),
    # the chosen tokens copied back, stream synchronised, every step; the length is restored before
    # each call so the context stays the workload's
    tok = torch.from_numpy(run.tokens_np.copy()).pin_memory()
    tok_out = torch.empty((1, w.batch), dtype=torch.int32).pin_memory()
    seq_keep = run.seq_len.clone()
    out = torch.empty((2, w.batch, w.vocab), dtype=torch.float32).pin_memory()

    e2e_i = [0]

    def e2e_call():
        if w.paged:  # the workload's pages end at slot L_b: no room to advance, logits out instead
            dfl.dualflow_step_host(run.ctx, run.weights, run.kv, tok, w.batch, out, 1, stream)
            return
        # every call advances the lengths by one; they are put back every 16 calls (the workload's
        # lengths stay within L_b .. L_b + 15, as in the decode-loop measurement below)
        if e2e_i[0] % 16 == 0:
            with torch.cuda.stream(stream):
                run.seq_len.copy_(seq_keep)
        e2e_i[0] += 1
        dfl.dualflow_generate_host(run.ctx, run.weights, run.kv, tok, w.batch, 1, tok_out, stream=stream)

    for _ in range(3):
        e2e_call()
    reps.barrier()
    e2e_steps = max(args.steps // 2, 3)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_call()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    # the same with the full logits [2, B, V] copied back every step instead of the tokens
    for _ in range(3):
        dfl.dualflow_step_host(run.ctx, run.weights, run.kv, tok, w.batch, out, 1, stream)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        dfl.dualflow_step_host(run.ctx, run.weights, run.kv, tok, w.batch, out, 1, stream)
    e2e_logits_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s, e2e_logits_s = reps.max(e2e_s, e2e_logits_s)

    # the decode loop: dualflow_generate (step, mixture head, greedy choice, length advance) for
    # gen_n tokens; the lengths are restored before each repetition so the context stays the
    # workload's
    gen_n, gen_reps = 16, 3
    gen = None
    if not w.paged and w.max_ctx - 1 - int(run.seq_len_np.max()) >= gen_n:
        seq0 = run.seq_len.clone()
        tok_out = torch.empty((gen_n, w.batch), dtype=torch.int32, device=dev)
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for r in range(2 + gen_reps):
                if r == 2:
                    g0.record(stream)
                run.seq_len.copy_(seq0)
                dfl.dualflow_generate(run.ctx, run.weights, run.kv, run.tokens, w.batch, gen_n, tok_out, run.logits,
                                      stream=stream)
            g1.record(stream)
            run.seq_len.copy_(seq0)
        g1.synchronize()
        gen_ms = g0.elapsed_time(g1) / (gen_reps * gen_n)
        st = dfl.dualflow_sync_status(run.ctx)
        if st != 0:
            raise RuntimeError(f"device status after the decode loop: {dfl.dualflow_status_string(st)}")
        gen = {"api": "dualflow_generate (greedy choice from the mixture head, in-loop length advance)",
               "tokens_per_loop": gen_n, "ms_per_token_step": gen_ms,
               "tokens_per_s": reps.rate(w.batch, gen_ms * 1e-3)}
    run.close()
    if rank != 0:
        return None

    peak, peak_kind = load_peaks()
    nb = step_bytes(w, experts_touched)
    step_gbs = nb["total"] / (ms * 1e-3) / 1e9
    att_ms = fam_ms[dfl.PROF_NAMES.index("attention")] / max(fam_n[dfl.PROF_NAMES.index("attention")], 1)
    att_gbs = nb["attention_per_launch"] / (att_ms * 1e-3) / 1e9
    prof_total = sum(fam_ms) / nprof
    graph_total = sum(fam_ms_graph) / nprof
    fb = family_bytes(w, experts_touched)
    families = {}
    for i, name in enumerate(dfl.PROF_NAMES):
        if not fam_n[i] or name not in fb:
            continue
        per_step = fam_n[i] // nprof
        ms_g, ms_s = fam_ms_graph[i] / nprof, fam_ms[i] / nprof
        gbs_g, gbs_s = fb[name] / (ms_g * 1e-3) / 1e9, fb[name] / (ms_s * 1e-3) / 1e9
        families[name] = {"launches_per_step": per_step, "bytes_per_step": fb[name],
                          "bytes_per_launch": fb[name] / per_step,
                          "in_graph": {"ms_per_step": ms_g, "share": ms_g / graph_total, "achieved_gbs": gbs_g,
                                       "frac": gbs_g / peak},
                          "serialised": {"ms_per_step": ms_s, "achieved_gbs": gbs_s, "frac": gbs_s / peak}}
    cpu_rows = list(range(min(8, w.batch)))
    samp = OracleSample(w, cpu_rows, min(6, w.n_layers))
    with OracleThreads() as th:
        raw_s = statistics.median(samp.time_step(cpu_rows) for _ in range(3))
    cpu_s = samp.full_step(raw_s, len(cpu_rows))
    cpu_desc = samp.describe(len(cpu_rows)) + " (median of 3 timings)"
    launches_per_step = int(sum(launches))
    res = {
        "metric": METRIC, "value": reps.rate(w.batch, ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32",
        "data": "synthetic: seeded counter-hash generator, random-init weights of the workload's shapes",
        "config": {"workload": w.name, "layers": w.n_layers, "d_model": w.d_model, "q_heads": w.n_q_heads,
                   "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "ffn_hidden": w.ffn_hidden,
                   "vocab": w.vocab, "batch_per_gpu": w.batch, "ctx": w.ctx_len,
                   "experts": w.n_experts, "topk": [w.topk_primary, w.topk_aux],
                   "experts_touched_per_layer": experts_touched,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: {nb['total'] / 1e9:.2f} GB per step vs 126 MB L2, no flush"},
        "hbm": {"step_bytes": nb["total"], "achieved_gbs": step_gbs, "frac_of_8000": step_gbs / NOMINAL_HBM_GBS,
                f"frac_of_{peak_kind}": step_gbs / peak},
        "primary_only": {"ms_per_step": ms_primary, "dual_over_primary": ms / ms_primary},
        "step_distribution": dist_steps,
        "roofline": {"kernel": "attn_bf16_kernel (shared-KV decode attention)", "bound": "hbm",
                     "achieved": att_gbs, "peak": peak, "unit": "GB/s", "frac": att_gbs / peak,
                     "peak_kind": f"{peak_kind} copy bandwidth", "bytes_per_launch": nb["attention_per_launch"],
                     "avg_launch_ms": att_ms,
                     "timing": "CUDA event pair around every launch in the replayed graph (serialising)",
                     "in_graph_achieved": families["attention"]["in_graph"]["achieved_gbs"],
                     "in_graph_frac": families["attention"]["in_graph"]["frac"],
                     # the committed ncu capture is of the dense workload's attention launch
                     "traffic": attention_traffic() if w.name == workload("dense").name else None},
        "roofline_families": {
            "note": ("per kernel family, against the measured copy bandwidth: in_graph = the family's share of the "
                     "pipelined step (device end stamps, dualflow_set_profiling mode 2; shares add up to the step), "
                     "serialised = CUDA event pairs around every launch (mode 1; each launch's stand-alone time)"),
            "peak_gbs": peak, "families": families},
        "kernel_ms_per_step": {n: fam_ms_graph[i] / nprof for i, n in enumerate(dfl.PROF_NAMES) if fam_n[i]},
        "kernel_ms_per_step_serialised": {n: fam_ms[i] / nprof for i, n in enumerate(dfl.PROF_NAMES) if fam_n[i]},
        "kernel_share": {n: fam_ms_graph[i] / nprof / graph_total for i, n in enumerate(dfl.PROF_NAMES) if fam_n[i]},
        "cpu_baseline": cpu_baseline_entry(w.batch / cpu_s, "tokens/s", th.threads, cpu_desc, raw_s),
        "e2e": {"value": reps.rate(w.batch, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": int(tok.numel() * 4),
                "d2h_bytes_per_step": int((out if w.paged else tok_out).numel() * 4),
                "api": ("dualflow_step_host (pinned host tokens in, host logits out, sync per step)" if w.paged else
                        "dualflow_generate_host, one step per call (pinned host tokens in, the step's chosen "
                        "tokens out, stream sync per step; the lengths advance by one per call and are put back "
                        "every 16 calls)")},
        "e2e_logits": {"value": reps.rate(w.batch, e2e_logits_s), "unit": "tokens/s",
                       "h2d_bytes_per_step": int(tok.numel() * 4), "d2h_bytes_per_step": int(out.numel() * 4),
                       "api": "dualflow_step_host (pinned host tokens in, host logits [2, B, V] out, sync per step)"},
        "generate": gen,
        "gpu_launches": launches_per_step * args.steps,
        "launches_per_step": launches_per_step,
        "clocks": sampler.summary(),
    }
    return res


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def sweep_topk_aux(w, ks, local_rank: int, steps: int = 20) -> list:
    """Decode-budget sweep of the auxiliary flow's expert fan-out (cost side only): the MoE step
    with topk_aux = k, timed with both flows and primary-only, and the distinct experts the
    step's rows touched per layer (their weights are read once each)."""
    import torch

    import dual_flow_decode_dualflow_b300 as dfl
    from tests import gpu_harness as H

    dev = torch.device("cuda", local_rank)
    out = []
    for k in ks:
        wk = w.replace(topk_aux=k)
        run = H.DeviceRun(wk, dev)
        stream = torch.cuda.Stream(device=dev)

        def timed(aux_on):
            with torch.cuda.stream(stream):
                for _ in range(3):
                    run.step(aux_on=aux_on, stream=stream)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(steps):
                    run.step(aux_on=aux_on, stream=stream)
                e1.record(stream)
            e1.synchronize()
            return e0.elapsed_time(e1) / steps

        ms_prim = timed(0)
        ms_dual = timed(1)
        kmax = max(wk.topk_primary, k)
        ids = torch.empty((wk.n_layers, 2, wk.batch, kmax), dtype=torch.int32, device=dev)
        dfl.dualflow_expert_ids(run.ctx, ids, wk.batch, stream)
        stream.synchronize()
        st = dfl.dualflow_sync_status(run.ctx)
        if st != 0:
            raise RuntimeError(f"device status in the topk_aux sweep: {dfl.dualflow_status_string(st)}")
        touched = [len(set(x for x in ids[l].flatten().tolist() if x >= 0)) for l in range(wk.n_layers)]
        nb = step_bytes(wk, touched)
        out.append({"topk_aux": k, "ms_per_step": ms_dual, "primary_only_ms": ms_prim,
                    "dual_over_primary": ms_dual / ms_prim, "experts_touched_mean": sum(touched) / len(touched),
                    "step_bytes": nb["total"], "hbm_gbs": nb["total"] / (ms_dual * 1e-3) / 1e9})
        run.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 600; 36 000 calls for the 18 us attention-only workload, so that the "
                         "timed region spans the 200 ms clock samples)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--layers", type=int, default=0,
                    help="profiling captures only: run the workload with this many layers")
    ap.add_argument("--quick", action="store_true", help="profiling captures only: time the step, skip the rest")
    ap.add_argument("--workload", choices=["dense", "moe", "attn", "paged", "prefill", "prefill_moe", "dense_paged"],
                    default="dense")
    ap.add_argument("--sweep-topk-aux", default="",
                    help="MoE only: comma-separated auxiliary fan-outs to time as well (cost side of the decode budget)")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = 36000 if args.workload == "attn" and args.impl == "ours" else 600
    args.warmup = max(args.warmup, 3)
    w = workload(args.workload)
    if args.layers:
        w = w.replace(n_layers=args.layers)
    rank, world, local_rank = Replicas.from_env()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, w)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    if args.workload in ("prefill", "prefill_moe"):
        res = run_ours_prefill(args, w, rank, world, local_rank)
    elif w.kind == "attention":
        res = run_ours_attention(args, w, rank, world, local_rank)
    else:
        res = run_ours(args, w, rank, world, local_rank)
        if res is not None and args.sweep_topk_aux and w.n_experts > 0:
            res["topk_aux_sweep"] = sweep_topk_aux(w, [int(k) for k in args.sweep_topk_aux.split(",")], local_rank)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
