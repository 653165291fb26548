"""Blended-prefill benchmark: TTFT and context tokens/s of the blend at r = 15 % against a
full prefill of the same prompt, with the roofline fractions of its kernels and of the
whole prefill.

Headline workload: the Yi-34B-shaped decoder (60 layers, d 7168, 56/8 heads, FFN 20480,
rotary base 5e6, bf16, random-init weights N(0, 0.02)) on 16 cached chunks of 512 tokens
+ a 128-token query (8320 tokens, Zipf(1.1) ids), gradual filtering to 15 %: the largest
of the pages' RAG shapes quoted at r = 15 % that fits one GPU.  The ``configs`` key adds,
each measured the same way, the Mistral-7B shape (3200 tokens), the Llama-7B shape with
its chunk KV staged from pinned host memory per layer (4128 tokens: ratio sweep, per-layer
overlap of loading and recompute, quantised staging, loading controller) and the
Llama-70B shape (4 requests x 8256 tokens over a pool of 64 chunks, r = 10 % and 20 %).
Synthetic inputs stand in for the RAG datasets of the pages.

One JSON line on rank 0.  Multi-GPU (torchrun): requests are independent units; a batch
of several requests is partitioned over the ranks (each blends its own requests with the
chunk pool replicated), a single-request workload runs one request per rank; no
collective on the data path.  The barrier and max-over-ranks timing use
torch.distributed for scalars only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "blended-prefill TTFT ms & context tok/s at r=15% vs full prefill; % roofline"
HEADLINE = "yi34b"
# (workload, ratios) of the other configurations, reported under "configs"
SECONDARY = (("mistral7b", (0.15,)), ("llama7b", (0.15,)), ("llama70b", (0.10, 0.20)))


def _sources_sha(paths):
    h = hashlib.sha256()
    for src in paths:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def _gemm_traffic():
    """DRAM bytes over algorithmic bytes of the projection GEMM, from the committed
    single-kernel ncu captures, while the kernel's sources are unchanged (else None)."""
    p = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if not d.get("source_sha256") or not d.get("ratio"):
        return None
    return d["ratio"] if _sources_sha(d["sources"]) == d["source_sha256"] else None


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the oracle's baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
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
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- flop / byte accounting
def gemm_flops(cfg, rows_R, rows_S):
    """Algorithmic flops of the projection GEMMs per layer (2 per multiply-add)."""
    d, qw, kvw, f = cfg.d_model, cfg.q_width, cfg.kv_width, cfg.ffn_dim
    out = {"qkv": 0.0, "oproj": 0.0, "gateup": 0.0, "down": 0.0}
    for R, S in zip(rows_R, rows_S):
        out["qkv"] += 2.0 * R * d * (qw + 2 * kvw)
        out["oproj"] += 2.0 * S * qw * d
        out["gateup"] += 2.0 * S * d * 2 * f
        out["down"] += 2.0 * S * f * d
    return out


def gemm_layer_bytes(cfg, R, S):
    """Bytes the projection GEMMs of one layer must move: weights once, A read, C written
    (q|k|v in fp32 where the layer checks its set (R != S), else rotated q, k, v in the model
    dtype straight from the epilogue; residual read + written; bf16 SwiGLU output)."""
    d, qw, kvw, f = cfg.d_model, cfg.q_width, cfg.kv_width, cfg.ffn_dim
    es = 2 if cfg.dtype == "bf16" else 4
    qkv_es = es if R == S else 4
    return (es * ((qw + 2 * kvw) * d + qw * d + 2 * f * d + f * d)
            + R * d * es + R * (qw + 2 * kvw) * qkv_es
            + S * qw * es + 2 * S * d * 4
            + S * d * es + S * f * es
            + S * f * es + 2 * S * d * 4)


def plan_rows(cfg, n_tokens, n_cached, n_query, ratios):
    """|R_i| and |S_i| per layer for one request (host-known sizes)."""
    import rag_non_prefix_gb300 as cb

    R, C = n_tokens, n_cached
    rows_R, rows_S = [], []
    for r in ratios:
        rows_R.append(R)
        if r >= 0:
            k = min(cb.k_for_ratio(r, n_cached), C)
            S, C = k + n_query, k
        else:
            S = R
        rows_S.append(S)
        R = S
    return rows_R, rows_S


def step_terms(cfg, rows_R, rows_S, pairs, kv_rows, checks, rerot_rows, peaks, link_bytes=None, link_gbs=None):
    """Per-layer algorithmic work and the roofline time of one prefill step.

    rows_R / rows_S: |R_i| and |S_i| summed over the step's requests; pairs[i]: sum over
    the queries q of S_i of (p_q + 1) (keys each attends to); kv_rows: fused-cache rows of
    all requests; checks[i]: cached candidates whose deviation is measured at layer i;
    rerot_rows: cached rows re-rotated at the start of the step (resident chunks).
    T_roof = sum_i max(F_i / P, B_i / BW) (+ per layer the host-link time of staged KV)
    + re-rotation and LM-head bytes / BW, P = sustained bf16, BW = HBM copy bandwidth.
    """
    es = 2 if cfg.dtype == "bf16" else 4
    kvw, H, dh = cfg.kv_width, cfg.n_heads, cfg.head_dim
    P = peaks["bf16_tflops_sustained"] * 1e12
    BW = peaks["hbm_gbs"] * 1e9
    t_roof, F_tot, B_tot, F_attn = 0.0, 0.0, 0.0, 0.0
    for i, (R, S) in enumerate(zip(rows_R, rows_S)):
        fa = 4.0 * H * dh * pairs[i]
        F = sum(gemm_flops(cfg, [R], [S]).values()) + fa
        B = (gemm_layer_bytes(cfg, R, S) + 2 * kv_rows * kvw * es  # attention reads the fused K and V once
             + S * 2 * kvw * es + checks[i] * 2 * kvw * es * 2)     # scatter; deviation reads fresh + cached
        t = max(F / P, B / BW)
        if link_bytes is not None:
            t = max(t, link_bytes / (link_gbs * 1e9))
        t_roof += t
        F_tot += F
        B_tot += B
        F_attn += fa
    extra = (4 * rerot_rows * kvw * es * len(rows_R) + cfg.vocab * cfg.d_model * es) / BW
    return {"t_roof_ms": (t_roof + extra) * 1e3, "flops": F_tot, "bytes": B_tot, "attn_flops": F_attn}


# ----------------------------------------------------------------------------- ranks
def max_over_ranks(values, world: int, device=None):
    """Element-wise maximum of per-rank scalars over all ranks (the slowest rank's times):
    ranks share no data, only this reduction and the barriers around the timed region."""
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def sum_over_ranks(value: float, world: int, device=None) -> float:
    """Sum of a per-rank scalar over all ranks (e.g. the tokens every rank processed)."""
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def shard_requests(n_requests: int, world: int, rank: int):
    """The requests of a batch that one rank blends: round-robin when the batch has at least
    one request per rank (the batch is partitioned, no request runs twice), else every
    request on every rank (each rank serves its own copy of the workload).  Returns the
    indices and whether the batch was partitioned."""
    if world > 1 and n_requests >= world:
        return list(range(rank, n_requests, world)), True
    return list(range(n_requests)), False


def job_throughput(units_all_ranks: float, ms_max: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's time."""
    return units_all_ranks / (ms_max * 1e-3)


# ----------------------------------------------------------------------------- one workload on the GPU
class Workload:
    """A workload's model, engine, cached chunks and requests on this rank's GPU."""

    def __init__(self, name, dev, world=1, rank=0, staged=None, decode_room=0):
        import torch

        import harness as hz
        import harness.device as hd
        import rag_non_prefix_gb300 as cb

        self.torch, self.hd, self.cb = torch, hd, cb
        self.spec = spec = hz.workload(name)
        self.cfg = cfg = spec.cfg
        self.dev = dev
        self.world = world
        self.req_idx, self.partitioned = shard_requests(len(spec.requests), world, rank)
        self.W = hd.device_weights(cfg, spec.seed)
        self.n_tok = [spec.n_tokens(r) for r in self.req_idx]
        self.n_cached = [spec.n_cached(r) for r in self.req_idx]
        self.T = sum(self.n_tok)
        self.decode_room = decode_room
        self.eng = cb.Engine(cfg, self.W, max_tokens=max(self.T, max(len(c) for c in spec.chunks)),
                             max_requests=len(self.req_idx), max_positions=max(self.n_tok) + 1 + decode_room)
        self.used = sorted({s.chunk for r in self.req_idx for s in spec.requests[r] if s.chunk >= 0})
        self.staged = staged if staged is not None else name == "llama7b"
        self.chunk_store, self.host_store = {}, {}
        for c in self.used:
            ids = hd.ids_tensor(spec.chunks[c])
            k, v = self.eng.precompute_chunk(ids)
            self.chunk_store[c] = (ids, k, v)
            self.eng.register_chunk(c, ids, k, v)
        if self.staged:  # the cached KV lives in page-locked host memory and is staged layer by layer
            for c in self.used:
                ids, k, v = self.chunk_store[c]
                self.host_store[c] = (ids, k.cpu().pin_memory(), v.cpu().pin_memory())
            self.register(on_host=True)
        self.copy_stream = torch.cuda.Stream() if self.staged else None
        self.stream = torch.cuda.current_stream()
        self.reqs = self.make_requests(want_sel=False)
        self.full_ids = [hd.ids_tensor(np.concatenate([s.ids for s in spec.requests[r]])) for r in self.req_idx]
        self.flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 512 MiB > L2
        torch.cuda.synchronize()

    def register(self, on_host: bool):
        for c in self.used:
            ids, k, v = (self.host_store if on_host else self.chunk_store)[c]
            self.eng.register_chunk(c, ids, k, v, on_host=on_host)

    def make_requests(self, want_sel=False, decode_room=0):
        out = []
        for r in self.req_idx:
            req = self.spec.requests[r]
            q = [s for s in req if s.chunk < 0][0]
            out.append(self.eng.make_request([s.chunk for s in req if s.chunk >= 0], self.hd.ids_tensor(q.ids),
                                             want_hidden=False, want_sel=want_sel, decode_room=decode_room))
        return out

    def blend_step(self, ratios, reqs=None, copy_stream="default", **kw):
        cs = self.copy_stream if copy_stream == "default" else copy_stream
        self.eng.blend_prefill(self.reqs if reqs is None else reqs, ratios, stream=self.stream, copy_stream=cs, **kw)

    def full_step(self):
        for ids in self.full_ids:
            self.eng.full_prefill(ids, want_hidden=False, stream=self.stream)

    def timed(self, fn, n, tag):
        torch = self.torch
        ts = []
        for _ in range(n):
            self.flush.fill_(1.0)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            torch.cuda.nvtx.range_push(tag)
            a.record(self.stream)
            fn()
            b.record(self.stream)
            torch.cuda.nvtx.range_pop()
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return ts

    def barrier(self):
        if self.world > 1:
            self.torch.distributed.barrier()
        self.torch.cuda.synchronize()

    def profiled(self, fn, level=1):
        """Per-phase device ms (and per-layer ms at level 2) of one run of fn."""
        self.eng.get_profile()
        self.eng.set_profiling(level)
        self.flush.fill_(1.0)
        self.torch.cuda.synchronize()
        fn()
        self.torch.cuda.synchronize()
        phases = self.eng.get_profile()
        layers = self.eng.get_layer_profile() if level & 2 else None
        self.eng.set_profiling(0)
        return phases, layers

    def close(self):
        self.torch.cuda.synchronize()
        self.eng.close()
        for name in ("reqs", "chunk_store", "host_store", "W", "full_ids", "flush", "eng"):
            setattr(self, name, None)
        self.torch.cuda.empty_cache()


def _phase_ms(phases):
    return {k: round(v["ms"], 4) for k, v in phases.items() if v["calls"]}


GEMM_PHASES = ("qkv", "oproj", "gateup", "down")


def measure(wl, ratio, schedule, steps, warmup, peaks, sample_clocks=False, full_from=None):
    """Blend and full prefill of one workload at one ratio: timed steps (CUDA events on the
    launching stream, 512 MiB written between steps), one profiled run of each, and the
    roofline fractions: the projection GEMMs and the attention against the sustained bf16
    peak, and the whole prefill as T_roof / TTFT.  ``full_from``: an earlier measurement of
    the same workload whose full-prefill timing and profile are reused (the full prefill does
    not depend on the ratio)."""
    cb = wl.cb
    cfg = wl.cfg
    ratios = cb.ratio_schedule(cfg.n_layers, ratio, schedule)
    for _ in range(warmup):
        wl.blend_step(ratios)
        if full_from is None:
            wl.full_step()
    wl.eng.get_status()
    wl.eng.get_profile()  # reset the launch counters
    sampler = None
    if sample_clocks:
        sampler = ClockSampler(wl.dev.index)
        sampler.start()
    wl.barrier()
    blend_ms = wl.timed(lambda: wl.blend_step(ratios), steps, "blend_timed")
    wl.barrier()
    counts = wl.eng.get_profile()
    full_ms = wl.timed(wl.full_step, steps, "full_timed") if full_from is None else full_from["full_runs"]
    wl.barrier()
    clocks = sampler.stop() if sampler else None
    wl.eng.get_status()
    # one profiled blend that also returns its sets (for the attention's key counts) and one
    # profiled full prefill
    sel_reqs = wl.make_requests(want_sel=True)
    ph_b, _ = wl.profiled(lambda: wl.blend_step(ratios, reqs=sel_reqs))
    ph_f = wl.profiled(wl.full_step)[0] if full_from is None else full_from["ph_full_raw"]
    L = cfg.n_layers
    pairs_b = [0.0] * L
    for req in sel_reqs:
        sel, cnt = req["sel"].cpu().numpy(), req["sel_count"].cpu().numpy()
        for i in range(L):
            pairs_b[i] += float(np.sum(sel[i, : cnt[i]].astype(np.float64) + 1.0))
    rows = [plan_rows(cfg, n, c, n - c, ratios) for n, c in zip(wl.n_tok, wl.n_cached)]
    rows_R = [sum(x[0][i] for x in rows) for i in range(L)]
    rows_S = [sum(x[1][i] for x in rows) for i in range(L)]
    checks = [0] * L  # cached candidates whose deviation a check layer measures: R_i minus the query
    for (rR, _), n, c in zip(rows, wl.n_tok, wl.n_cached):
        for i in range(L):
            if ratios[i] >= 0:
                checks[i] += rR[i] - (n - c)
    kv_rows = wl.T
    nc = sum(wl.n_cached)
    rows_full = [wl.T] * L
    pairs_full = [float(sum(n * (n + 1) / 2 for n in wl.n_tok))] * L
    tb = step_terms(cfg, rows_R, rows_S, pairs_b, kv_rows, checks, 0 if wl.staged else nc, peaks)
    tf = step_terms(cfg, rows_full, rows_full, pairs_full, kv_rows, [0] * L, 0, peaks)
    P = peaks["bf16_tflops_sustained"]

    def frac(flops, ms):
        if not ms:
            return None
        a = flops / (ms * 1e-3) / 1e12
        return {"achieved_tflops": round(a, 1), "frac": round(a / P, 4), "ms": round(ms, 4)}

    gb = sum(gemm_flops(cfg, rows_R, rows_S).values())
    gf = sum(gemm_flops(cfg, rows_full, rows_full).values())
    blend_mean, full_mean = max_over_ranks([statistics.mean(blend_ms), statistics.mean(full_ms)], wl.world, wl.dev)
    tokens_all = sum_over_ranks(wl.T, wl.world, wl.dev)
    return {
        "ratio": ratio, "ratios": ratios, "tokens": wl.T, "tokens_all_ranks": tokens_all,
        "blend_ms": blend_mean, "full_ms": full_mean, "blend_runs": blend_ms, "full_runs": full_ms,
        "blend_tok_s": job_throughput(tokens_all, blend_mean), "full_tok_s": job_throughput(tokens_all, full_mean),
        "speedup": full_mean / blend_mean, "phases_blend": _phase_ms(ph_b), "phases_full": _phase_ms(ph_f),
        "gemm_blend": frac(gb, sum(ph_b[p]["ms"] for p in GEMM_PHASES)), "gemm_flops_blend": gb,
        "gemm_full": frac(gf, sum(ph_f[p]["ms"] for p in GEMM_PHASES)),
        "attn_blend": frac(tb["attn_flops"], ph_b["attention"]["ms"]),
        "attn_full": frac(tf["attn_flops"], ph_f["attention"]["ms"]),
        "t_roof_blend_ms": tb["t_roof_ms"], "t_roof_full_ms": tf["t_roof_ms"],
        "roof_frac_blend": tb["t_roof_ms"] / blend_mean, "roof_frac_full": tf["t_roof_ms"] / full_mean,
        "gemm_launches_blend": sum(ph_b[p]["calls"] for p in GEMM_PHASES),
        "gemm_bytes_blend": sum(gemm_layer_bytes(cfg, R, S) for R, S in zip(rows_R, rows_S)),
        "launches_per_step": sum(v["launches"] for v in counts.values()) / max(1, steps),
        "clocks": clocks, "rows_R": rows_R, "rows_S": rows_S, "pairs_blend": pairs_b, "checks": checks,
        "ph_full_raw": ph_f,
    }


def summary(m):
    """The per-configuration entry of the JSON line."""
    r4 = lambda x: None if x is None else round(x, 4)  # noqa: E731
    return {"ratio": m["ratio"], "tokens": m["tokens"],
            "ttft_ms": {"blend": r4(m["blend_ms"]), "full_prefill": r4(m["full_ms"]),
                        "blend_median": r4(statistics.median(m["blend_runs"])),
                        "full_median": r4(statistics.median(m["full_runs"]))},
            "runs_ms": {"blend": [round(x, 3) for x in m["blend_runs"]], "full_prefill": [round(x, 3) for x in m["full_runs"]]},
            "speedup_vs_full_prefill": round(m["speedup"], 3),
            # on the medians too: a staged configuration's runs can stall on the host's copies
            "speedup_vs_full_prefill_median": round(statistics.median(m["full_runs"]) / statistics.median(m["blend_runs"]), 3),
            "context_tok_s": {"blend": round(m["blend_tok_s"], 1), "full_prefill": round(m["full_tok_s"], 1)},
            "gemm_roofline": {"blend": m["gemm_blend"], "full_prefill": m["gemm_full"]},
            "attention_roofline": {"blend": m["attn_blend"], "full_prefill": m["attn_full"]},
            "whole_prefill_roofline": {"blend": {"t_roof_ms": r4(m["t_roof_blend_ms"]), "frac": r4(m["roof_frac_blend"])},
                                       "full_prefill": {"t_roof_ms": r4(m["t_roof_full_ms"]),
                                                        "frac": r4(m["roof_frac_full"])}},
            "phase_ms": {"blend": m["phases_blend"], "full_prefill": m["phases_full"]},
            "clocks": m["clocks"]}


# ----------------------------------------------------------------------------- extras on the headline
def measure_decode(wl, ratios, steps, peaks):
    """Greedy decode steps after a blend of the same prompt (one token per request per step),
    each timed with CUDA events; a step streams every weight once, so its bound is HBM."""
    torch, cfg = wl.torch, wl.cfg
    dreqs = wl.make_requests(decode_room=wl.decode_room)
    wl.blend_step(ratios, reqs=dreqs)
    wl.eng.get_status()
    tok = torch.cat([r["first_token"] for r in dreqs]).to(torch.int32)
    for _ in range(4):
        tok = wl.eng.decode_step(dreqs, tok)
    torch.cuda.synchronize()
    ts = []
    wl.eng.get_profile()
    for _ in range(steps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(wl.stream)
        tok = wl.eng.decode_step(dreqs, tok)
        b.record(wl.stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    dprof = wl.eng.get_profile()
    ph, _ = wl.profiled(lambda: wl.eng.decode_step(dreqs, tok))
    wl.eng.get_status()
    ms = statistics.mean(ts)
    n_seq = len(dreqs)
    es = 2 if cfg.dtype == "bf16" else 4
    ctx_len = statistics.mean(r["n_tokens"] + r["decoded"] for r in dreqs)  # mid-run context
    wbytes = (cfg.n_layers * cfg.params_per_layer() + cfg.vocab * cfg.d_model) * es
    kvbytes = n_seq * cfg.n_layers * ctx_len * 2 * cfg.kv_width * es
    gbs = (wbytes + kvbytes) / (ms * 1e-3) / 1e9
    return {"steps": steps, "sequences": n_seq, "ms_per_step": round(ms, 4), "tok_s": round(n_seq / (ms * 1e-3), 1),
            "context_tokens": round(ctx_len, 1),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "bytes_per_step": int(wbytes + kvbytes),
                         "weight_bytes": int(wbytes), "kv_bytes": int(kvbytes),
                         "peak_source": f"{peaks['source']} HBM copy"},
            "launches_per_step": sum(v["launches"] for v in dprof.values()) / steps, "phase_ms": _phase_ms(ph)}


def measure_variants(wl, ratios, full_ms, steps):
    """The same prompt with the cosine deviation and with spatial seam repair (the 16
    tokens before every chunk boundary, recomputed from layer 0 on)."""
    out = {}
    for tag, kw in (("cosine_deviation", {"dev_mode": 3}), ("seam_repair_r16", {"seam_tokens": 16})):
        for _ in range(2):
            wl.blend_step(ratios, **kw)
        ts = wl.timed(lambda: wl.blend_step(ratios, **kw), steps, tag)
        out[tag] = {"ttft_ms": round(statistics.mean(ts), 4),
                    "speedup_vs_full_prefill": round(full_ms / statistics.mean(ts), 3)}
    wl.eng.get_status()
    return out


def measure_e2e(wl, ratios, steps):
    """The blend through the public API with host buffers: the query ids copied in from
    pinned host memory and the first tokens copied out, host-timed per step."""
    torch = wl.torch
    pinned_q = [r["query_ids"].cpu().pin_memory() for r in wl.reqs]
    host_tok = torch.empty(len(wl.reqs), dtype=torch.int32).pin_memory()
    e2e = []
    for _ in range(steps):
        wl.flush.fill_(1.0)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for r, pq in zip(wl.reqs, pinned_q):
            r["query_ids"].copy_(pq, non_blocking=True)
        wl.blend_step(ratios)
        for i, r in enumerate(wl.reqs):
            host_tok[i:i + 1].copy_(r["first_token"], non_blocking=True)
        torch.cuda.synchronize()
        e2e.append((time.perf_counter() - t) * 1e3)
    return statistics.mean(e2e), int(sum(pq.numel() * 4 for pq in pinned_q)), 4 * len(wl.reqs)


def measure_staging(wl, ratios, schedule, blend_staged_ms, full_ms, steps, peaks, codec=True):
    """Host-staged workloads: link bandwidth, T_load, T_recompute (the same blend with the
    chunks resident), the per-layer overlap of loading and recompute ([P1] パイプライン化の設計:
    T_layer ~ max(T_load, T_recompute), summed over the layers) measured with per-layer
    events of both streams, int8 / int4 quantised staging, and the loading controller."""
    torch, cb, cfg = wl.torch, wl.cb, wl.cfg
    ids0, kh, vh = wl.host_store[wl.used[0]]
    dst = torch.empty_like(kh, device=wl.dev)
    torch.cuda.synchronize()
    # the link's bandwidth: the best of three bursts of three copies (the host link is shared
    # with the box's other work; one slow burst is not the link)
    best_ms = None
    for _ in range(3):
        a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(wl.copy_stream):
            a_ev.record(wl.copy_stream)
            for _ in range(3):
                dst.copy_(kh, non_blocking=True)
            b_ev.record(wl.copy_stream)
        b_ev.synchronize()
        ms = a_ev.elapsed_time(b_ev)
        best_ms = ms if best_ms is None else min(best_ms, ms)
    del dst
    h2d_gbs = 3 * kh.numel() * kh.element_size() / (best_ms * 1e-3) / 1e9
    total_bytes = sum(2 * wl.host_store[s.chunk][1].numel() * wl.host_store[s.chunk][1].element_size()
                      for r in wl.req_idx for s in wl.spec.requests[r] if s.chunk >= 0)
    t_load = total_bytes / (h2d_gbs * 1e9) * 1e3
    # per-layer events of one staged blend (no phase events in that run): staging copies
    # (copy stream), compute (after the wait for the staged KV); begin and finish, which are
    # outside the layers, from a run with phase events
    _, lay = wl.profiled(lambda: wl.blend_step(ratios), level=2)
    ph_s, _ = wl.profiled(lambda: wl.blend_step(ratios), level=1)
    load_l, comp_l = lay["load_ms"], lay["compute_ms"]
    edge = ph_s.get("begin", {"ms": 0.0})["ms"] + ph_s.get("finish", {"ms": 0.0})["ms"]
    sum_max = sum(max(a, b) for a, b in zip(load_l, comp_l)) + edge
    overlap = {"sum_load_ms": round(sum(load_l), 3), "sum_compute_ms": round(sum(comp_l), 3),
               "begin_finish_ms": round(edge, 3), "sum_max_ms": round(sum_max, 3),
               "ttft_staged_ms": round(blend_staged_ms, 3), "ttft_over_sum_max": round(blend_staged_ms / sum_max, 3),
               "per_layer_load_ms": [round(x, 4) for x in load_l], "per_layer_compute_ms": [round(x, 4) for x in comp_l]}
    # the same blend with the cached KV resident in HBM: T_recompute
    wl.register(on_host=False)
    for _ in range(2):
        wl.blend_step(ratios, copy_stream=None)
    res_ms = statistics.mean(wl.timed(lambda: wl.blend_step(ratios, copy_stream=None), steps, "resident"))
    r0 = cb.ratio_schedule(cfg.n_layers, 0.0, schedule)
    for _ in range(2):
        wl.blend_step(r0, copy_stream=None)
    fixed_ms = statistics.mean(wl.timed(lambda: wl.blend_step(r0, copy_stream=None), steps, "r0"))
    wl.register(on_host=True)
    out = {"h2d_gbs": round(h2d_gbs, 1), "staged_bytes": total_bytes, "t_load_ms": round(t_load, 3),
           "t_recompute_ms": round(res_ms, 3), "max_load_recompute_ms": round(max(t_load, res_ms), 3),
           "ttft_staged_ms": round(blend_staged_ms, 3), "per_layer_overlap": overlap}
    # loading controller: the plan and the ratio it picks from the measured costs (link
    # bandwidth, full-prefill time per token, the blend's fixed recompute time at r = 0),
    # then the staged blend timed at that ratio against the plan's prediction
    model = {"link_bytes_per_s": h2d_gbs * 1e9, "link_latency_s": 0.0,
             "prefill_s_per_token": full_ms * 1e-3 / wl.T, "recompute_fixed_s": fixed_ms * 1e-3,
             "r_min": 0.05, "r_max": 0.20}
    req0 = wl.spec.requests[wl.req_idx[0]]
    infos = [wl.eng.chunk_info(s.chunk) for s in req0 if s.chunk >= 0]
    acts, r_star, t_load_p, t_rec_p = cb.cb_plan_loading(model, infos, wl.n_tok[0] - wl.n_cached[0])
    rat_star = cb.ratio_schedule(cfg.n_layers, r_star, schedule)
    for _ in range(2):
        wl.blend_step(rat_star)
    ts = wl.timed(lambda: wl.blend_step(rat_star), steps, "controller")
    out["controller"] = {"model": {k: round(v, 9) for k, v in model.items()}, "actions": acts,
                         "ratio": round(r_star, 4), "t_load_pred_ms": round(t_load_p * 1e3, 3),
                         "t_recompute_pred_ms": round(t_rec_p * 1e3, 3),
                         "ttft_pred_ms": round(max(t_load_p, t_rec_p) * 1e3, 3),
                         "ttft_measured_ms": round(statistics.mean(ts), 3), "fixed_ms_at_r0": round(fixed_ms, 3)}
    # the same chunks quantised (KIVI-style int8 / int4) in pinned host memory, staged
    # through a two-slot ring and decoded + re-rotated per layer on the GPU
    if codec:
        for bits in (8, 4):
            slot = 0
            for c in wl.used:
                ids, k, v = wl.chunk_store[c]
                blob = cb.cb_kv_encode(k, v, bits)
                torch.cuda.synchronize()
                hb = blob.cpu().pin_memory()
                wl.host_store[("q", bits, c)] = hb
                wl.eng.register_chunk_codec(c, ids, hb, bits, on_host=True)
            for r in wl.req_idx:
                slot = max(slot, sum(cb.cb_codec_layer_bytes(len(s.ids), cfg.n_kv_heads, cfg.head_dim, bits)
                                     for s in wl.spec.requests[r] if s.chunk >= 0))
            wl.eng.set_staging(2 * slot)
            for _ in range(2):
                wl.blend_step(ratios)
            ts = wl.timed(lambda: wl.blend_step(ratios), steps, f"codec{bits}")
            qbytes = sum(wl.host_store[("q", bits, s.chunk)].numel()
                         for r in wl.req_idx for s in wl.spec.requests[r] if s.chunk >= 0)
            out[f"int{bits}"] = {"staged_bytes": qbytes, "t_load_ms": round(qbytes / (h2d_gbs * 1e9) * 1e3, 3),
                                 "ttft_staged_ms": round(statistics.mean(ts), 3), "staging_slots": 2}
        wl.eng.get_status()
        wl.register(on_host=True)
    return out


def staged_roofline(m, wl, h2d_gbs, peaks):
    """Whole-prefill roofline of the staged blend: per layer also the host-link time of the
    layer's cached KV (T_roof = sum_i max(F_i / P, B_i / BW, KV_i / link))."""
    cfg = wl.cfg
    es = 2 if cfg.dtype == "bf16" else 4
    layer_kv = sum(wl.n_cached) * 2 * cfg.kv_width * es
    t = step_terms(cfg, m["rows_R"], m["rows_S"], m["pairs_blend"], wl.T, m["checks"], 0, peaks,
                   link_bytes=layer_kv, link_gbs=h2d_gbs)
    return {"t_roof_ms": round(t["t_roof_ms"], 4), "frac": round(t["t_roof_ms"] / m["blend_ms"], 4),
            "link_gbs": round(h2d_gbs, 1), "layer_kv_bytes": layer_kv}


def measure_sweep(wl, schedule, steps):
    """Blended TTFT at r in {0, 5, 10, 15, 20, 50, 100} %, each timed like the headline."""
    out = []
    for r in (0.0, 0.05, 0.10, 0.15, 0.20, 0.50, 1.0):
        rat = wl.cb.ratio_schedule(wl.cfg.n_layers, r, schedule)
        for _ in range(2):
            wl.blend_step(rat)
        ts = wl.timed(lambda: wl.blend_step(rat), steps, "sweep")
        out.append({"ratio": r, "ttft_ms": round(statistics.mean(ts), 4)})
    return out


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, world):
    import torch

    import rag_non_prefix_gb300 as cb
    from rag_non_prefix_gb300 import build as cbbuild

    cbbuild.build()
    cb.cb_set_launch_overlap(args.launch_overlap)
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks = _peaks()
    schedule = args.schedule
    wl = Workload(args.workload, dev, world, rank, staged=args.staged,
                  decode_room=args.decode_steps + 8 if args.decode_steps else 0)
    spec, cfg = wl.spec, wl.cfg
    sched = schedule or spec.schedule
    ratio = spec.ratio if args.ratio is None else args.ratio
    m = measure(wl, ratio, sched, args.steps, args.warmup, peaks, sample_clocks=True)
    ratios = m["ratios"]
    full_mean = m["full_ms"]
    n_small = max(3, min(args.steps, 5))
    sweep = measure_sweep(wl, sched, n_small) if args.sweep else None
    decode = measure_decode(wl, ratios, args.decode_steps, peaks) if args.decode_steps else None
    variants = measure_variants(wl, ratios, full_mean, n_small) if args.variants else None
    staging = (measure_staging(wl, ratios, sched, m["blend_ms"], full_mean, n_small, peaks, codec=args.codec)
               if wl.staged else None)
    if staging:
        staging["whole_prefill_roofline"] = staged_roofline(m, wl, staging["h2d_gbs"], peaks)
    e2e_ms, h2d, d2h = measure_e2e(wl, ratios, args.steps)
    e2e_ms = max_over_ranks([e2e_ms], world, dev)[0]
    # roofline of the dominant kernel: the tcgen05 projection GEMM over all its launches in a blend
    g = m["gemm_blend"]
    launches = m["gemm_launches_blend"]
    alg_per_launch = m["gemm_bytes_blend"] / max(1, launches)
    ratio_traffic = _gemm_traffic()
    nc_total = sum(wl.n_cached)
    es = 2 if cfg.dtype == "bf16" else 4
    rerot_bytes = 2 * cfg.n_layers * nc_total * cfg.kv_width * es  # K read + written (algorithmic; V copy not counted)
    moved_bytes = 2 * rerot_bytes  # what the kernel moves: K and V, each read and written
    begin_ms = m["phases_blend"].get("begin")
    T_all = m["tokens_all_ranks"]
    out = {
        "metric": METRIC,
        "value": round(m["blend_tok_s"], 1),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(m["blend_ms"], 4),
        "higher_is_better": True,
        "scaling": "strong" if wl.partitioned else "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (harness: random-init N(0,0.02) weights, Zipf(1.1) token ids)",
        "config": {"workload": f"{spec.name}: {cfg.n_layers}L d{cfg.d_model} H{cfg.n_heads}/{cfg.n_kv_heads} "
                               f"ffn{cfg.ffn_dim} theta{cfg.rope_theta:g} {cfg.dtype}; {len(wl.req_idx)} request(s) "
                               f"x {wl.n_tok[0]} tokens ({wl.n_cached[0]} cached); r={ratio} {sched}",
                   "ratio_schedule": [round(x, 4) for x in ratios], "tokens_per_step": wl.T,
                   "l2": "512 MiB buffer written between timed steps; weights > L2",
                   "parallelism": (f"requests partitioned over {world} ranks" if wl.partitioned
                                   else f"one request set per rank x{world}"),
                   "launch_overlap": bool(args.launch_overlap)},
        "ttft_ms": summary(m)["ttft_ms"],
        "speedup_vs_full_prefill": round(m["speedup"], 3),
        "full_prefill_tok_s": round(m["full_tok_s"], 1),
        "phase_ms": m["phases_blend"],
        "roofline": {"kernel": "projection GEMM: gemm_pair_kernel (tcgen05 cta_group::2) / gemm_bf16_tc (qkv, o, gate/up, down)", "bound": "tensor",
                     "achieved": g["achieved_tflops"] if g else None, "peak": peaks["bf16_tflops_sustained"],
                     "unit": "TFLOP/s", "frac": g["frac"] if g else None,
                     "traffic": round(ratio_traffic * alg_per_launch) if ratio_traffic else None,
                     "traffic_source": ("DRAM/algorithmic ratio of single-kernel ncu captures at one kept layer's "
                                        "shapes, times this step's algorithmic bytes per launch") if ratio_traffic
                     else "no capture of the current kernel",
                     "algorithmic_bytes_per_launch": round(alg_per_launch),
                     "peak_source": f"{peaks['source']} bf16 sustained", "launches": launches,
                     "flops": m["gemm_flops_blend"]},
        "rooflines": {k: v for k, v in summary(m).items()
                      if k in ("gemm_roofline", "attention_roofline", "whole_prefill_roofline")},
        "rerotate": None if wl.staged else {
            "bytes": rerot_bytes, "bytes_note": "algorithmic: K read + written, every layer (the V copy is not counted)",
            "moved_bytes": moved_bytes, "ms": begin_ms,
            "gbs": round(rerot_bytes / (begin_ms * 1e-3) / 1e9, 1) if begin_ms else None,
            "frac": round(rerot_bytes / (begin_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4) if begin_ms else None,
            "moved_gbs": round(moved_bytes / (begin_ms * 1e-3) / 1e9, 1) if begin_ms else None},
        "e2e": {"value": round(job_throughput(T_all, e2e_ms), 1), "unit": "tok/s", "ms": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(m["launches_per_step"] * args.steps),
        "sweep": sweep,
        "decode": decode,
        "variants": variants,
        "staging": staging,
        "clocks": m["clocks"],
    }
    wl.close()
    del wl
    if args.configs and world == 1:
        out["configs"] = []
        for name, rs in SECONDARY:
            if name == args.workload:
                continue
            w2 = Workload(name, dev, world, rank)
            s2 = w2.spec.schedule if schedule is None else schedule
            first = None
            for r in rs:
                m2 = measure(w2, r, s2, args.config_steps, 3, peaks, sample_clocks=True, full_from=first)
                first = first or m2
                e = {"workload": f"{name}: {w2.cfg.n_layers}L d{w2.cfg.d_model} H{w2.cfg.n_heads}/{w2.cfg.n_kv_heads} "
                                 f"ffn{w2.cfg.ffn_dim}; {len(w2.req_idx)} request(s) x {w2.n_tok[0]} tokens"
                                 + ("; chunk KV staged from pinned host memory" if w2.staged else ""),
                     "steps": args.config_steps, **summary(m2)}
                if first is not m2:
                    e["full_prefill_note"] = "full prefill timed once per workload (at the first ratio)"
                if w2.staged:
                    e["staging"] = measure_staging(w2, m2["ratios"], s2, m2["blend_ms"], m2["full_ms"],
                                                   args.config_steps, peaks, codec=args.codec)
                    e["whole_prefill_roofline"]["blend_staged"] = staged_roofline(m2, w2, e["staging"]["h2d_gbs"],
                                                                                  peaks)
                    e["sweep"] = measure_sweep(w2, s2, 3)
                out["configs"].append(e)
            w2.close()
            del w2
    return out, spec, cfg, ratios


# ----------------------------------------------------------------------------- oracle (CPU) samples
def _oracle_threads() -> int:
    t = os.environ.get("OPENBLAS_NUM_THREADS") or os.environ.get("OMP_NUM_THREADS")
    return int(t) if t else (os.cpu_count() or 1)


def oracle_samples(spec, ratios, kept_fraction=1.0, full_tokens=1024, with_full=True):
    """Times the oracle, as it stands, on bounded samples of the same workload and scales
    each to the whole prefill by algorithmic flops.

    * blend: one layer that keeps the recomputed set, i.e. the per-layer work of the blend
      after its last check layer: ``fixed_set_prefill`` of the model's first layer with the
      set S = the query + k cached tokens (k of the final ratio; ``kept_fraction`` < 1
      takes that share of them), which re-rotates the layer's cached K, projects S, scatters
      its K/V, attends causally over the fused cache and runs the output projection and MLP
      for S;
    * full prefill: ``full_prefill`` of the prompt's first ``full_tokens`` tokens through the
      model's first layer (by causality the first rows of the prompt's own prefill).
    Weights come from the harness's host generator; cached chunk KV is harness random data
    of the right shape (its values do not change the oracle's work).
    """
    import dataclasses

    import harness as hz
    import oracle.cacheblend as orc

    cfg = spec.cfg
    one = dataclasses.replace(cfg, n_layers=1)
    W = hz.HostWeights(one, spec.seed)
    W.layer(0)
    W.lm_head()
    req = spec.requests[0]
    caches = {}
    for s in req:
        if s.chunk < 0:
            continue
        n = len(s.ids) * cfg.n_kv_heads * cfg.head_dim
        shape = (1, len(s.ids), cfg.n_kv_heads, cfg.head_dim)
        caches[s.chunk] = (hz.gen_weight_fp32(0x5EED0000 + s.chunk, 0, n).reshape(shape).astype(np.float64),
                           hz.gen_weight_fp32(0x5EED8000 + s.chunk, 0, n).reshape(shape).astype(np.float64))
    n_tok, n_c = spec.n_tokens(0), spec.n_cached(0)
    n_q = n_tok - n_c
    rR, rS = plan_rows(cfg, n_tok, n_c, n_q, ratios)
    k = int(round((rS[-1] - n_q) * kept_fraction))
    S = np.concatenate([np.linspace(0, n_c - 1, k).astype(np.int64) if k else np.zeros(0, np.int64),
                        np.arange(n_c, n_tok)])
    storage = "bf16" if cfg.dtype == "bf16" else "f32"
    t = time.perf_counter()
    orc.fixed_set_prefill(one, W, req, caches, S, storage)
    dt_b = time.perf_counter() - t
    pos = S.astype(np.float64)

    def layer_flops(R, S_n, pairs):
        return sum(gemm_flops(cfg, [R], [S_n]).values()) + 4.0 * cfg.n_heads * cfg.head_dim * pairs

    f_sample = layer_flops(len(S), len(S), float(np.sum(pos + 1)))
    # the whole blend: every layer's projections, and attention with the kept set's key counts
    pairs_kept = float(np.sum(pos + 1)) / max(1, len(S)) * rS[-1]
    f_blend = sum(layer_flops(R, Sn, n_tok * (n_tok + 1) / 2 if i == 0 else pairs_kept * Sn / rS[-1])
                  for i, (R, Sn) in enumerate(zip(rR, rS)))
    est_b = dt_b * f_blend / f_sample
    out = {"value": round(n_tok / est_b, 3), "unit": "tok/s", "cores": _oracle_threads(), "kind": "oracle",
           "cpu_model": cpu_model(),
           "sample": (f"oracle blend: one kept layer of the workload (fixed_set_prefill of layer 0 with "
                      f"|S| = {len(S)} rows: the query + {k} cached tokens) in {dt_b:.2f} s, scaled by algorithmic "
                      f"flops to all {cfg.n_layers} layers of the blend: est. TTFT {est_b:.1f} s"),
           "sample_s": round(dt_b, 3), "est_ttft_s": round(est_b, 2), "estimate": True}
    if with_full:
        ids = np.concatenate([s.ids for s in req])[:full_tokens]
        t = time.perf_counter()
        orc.full_prefill(one, W, ids, storage)
        dt_f = time.perf_counter() - t
        nf = len(ids)
        f_smp = layer_flops(nf, nf, nf * (nf + 1) / 2)
        f_full = cfg.n_layers * layer_flops(n_tok, n_tok, n_tok * (n_tok + 1) / 2)
        est_f = dt_f * f_full / f_smp
        out["full_prefill"] = {"value": round(n_tok / est_f, 3), "unit": "tok/s", "sample_s": round(dt_f, 3),
                               "est_ttft_s": round(est_f, 2),
                               "sample": (f"oracle full prefill of the prompt's first {nf} tokens through one layer "
                                          f"in {dt_f:.2f} s, scaled by algorithmic flops to {n_tok} tokens x "
                                          f"{cfg.n_layers} layers: est. TTFT {est_f:.1f} s")}
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm (CPU, rank 0 only): each step one bounded sample (a
    quarter of one kept layer's recomputed rows), the rate scaled to the whole blend."""
    import harness as hz
    import oracle.cacheblend as orc
    from rag_non_prefix_gb300 import build as cbbuild

    for lib, srcs in cbbuild.HOST_LIBS.items():  # the harness's host generator (gcc; no GPU code)
        cbbuild._build_host(lib, srcs)
    spec = hz.workload(args.workload)
    cfg = spec.cfg
    ratio = spec.ratio if args.ratio is None else args.ratio
    ratios = orc.ratio_schedule(cfg.n_layers, ratio, args.schedule or spec.schedule)
    vals = []
    for i in range(args.warmup + args.steps):
        r = oracle_samples(spec, ratios, kept_fraction=0.25, with_full=False)
        if i >= args.warmup:
            vals.append(r)
    v = statistics.mean(x["value"] for x in vals)
    step_ms = statistics.mean(x["sample_s"] for x in vals) * 1e3
    cpu = dict(vals[-1])
    cpu["value"] = round(v, 3)
    return {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "tok/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "ratio_schedule": [round(x, 4) for x in ratios]},
            "estimate": {"value_is": "context tok/s of the whole blend, extrapolated by algorithmic flops from the "
                                     "timed sample; ms_per_step is the sample's measured wall time",
                         "est_ttft_s": round(spec.n_tokens(0) / v, 2)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(v, 3), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--ratio", type=float, default=None)
    ap.add_argument("--schedule", default=None, choices=[None, "fixed", "gradual"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="also time r in {0, 5, 10, 15, 20, 50, 100} %%")
    ap.add_argument("--staged", default=None, action=argparse.BooleanOptionalAction,
                    help="cached KV in pinned host memory, staged per layer (default: on for llama7b)")
    ap.add_argument("--decode-steps", type=int, default=32, help="timed greedy decode steps after the blend (0: none)")
    ap.add_argument("--codec", default=True, action=argparse.BooleanOptionalAction,
                    help="with staged chunks: also time int8 / int4 quantised staging")
    ap.add_argument("--variants", default=True, action=argparse.BooleanOptionalAction,
                    help="also time the cosine-deviation and seam-repair selection variants")
    ap.add_argument("--configs", default=True, action=argparse.BooleanOptionalAction,
                    help="also measure the other configurations (N = 1 only) under the key 'configs'")
    ap.add_argument("--config-steps", type=int, default=5, help="timed steps of each other configuration")
    ap.add_argument("--launch-overlap", default=True, action=argparse.BooleanOptionalAction,
                    help="programmatic dependent launch of the layer kernels (default: on)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    out, spec, cfg, ratios = run_ours(args, rank, world)
    if rank == 0:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = oracle_samples(spec, ratios)
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
