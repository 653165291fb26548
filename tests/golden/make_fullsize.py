"""Writes the oracle's blended-prefill outputs for the full-size workloads, for the GPU
parity tests (``tests/golden/fullsize_<name>.npz``).

Only ``oracle/`` computes; ``harness/`` supplies the seeded inputs.  Nothing here runs the
CUDA library.  The workloads are the four GPU-sized configurations of the pages' RAG
shapes, each at full width, head count, FFN size, rotary base, token count and batch:

* mistral7b -- Mistral-7B shape, 64-token prefix + 6 x 512 chunks + 64-token query, all 32 layers;
* llama7b   -- Llama-7B shape (MHA), 8 x 512 chunks + 32-token query, all 32 layers;
* yi34b     -- Yi-34B shape (rotary base 5e6), 16 x 512 chunks + 128-token query, first 6 layers;
* llama70b  -- Llama-70B shape, 4 requests of 32 pooled 256-token chunks + 64-token query,
  first 6 layers, at r = 10 % and r = 20 %.

Six layers hold layer 0 (every token), the four check layers of gradual filtering (layers
1-4) and one layer that keeps the last checked set, so every kind of layer is covered; the
oracle takes ~10 minutes per layer-pass at these widths on a few CPU cores, which is why
the two largest shapes stop there.

Stored per ratio and request: the selected set of every check layer, the hidden rows of
the last 16 query tokens and of 16 recomputed cached tokens drawn with a fixed seed (8 + 8
for the four-request batch), the 16 largest LM-head logits at the last position with their
token ids (the first token is the first id), and the oracle's wall time.

    python tests/golden/make_fullsize.py mistral7b llama7b yi34b llama70b
    python tests/golden/make_fullsize.py --full-prefill mistral7b

The second form stores the oracle's plain full prefill of the Mistral-7B-shaped prompt
(same model, all 32 layers), against which the GPU's own full prefill and a plain-PyTorch
bf16 witness are compared to measure the rounding floor of bf16 operands at full depth.
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import harness as hz  # noqa: E402
import oracle.cacheblend as orc  # noqa: E402

CASES = {
    "mistral7b": {"depth": None, "ratios": [0.15], "rows": 16},
    "llama7b": {"depth": None, "ratios": [0.15], "rows": 16},
    "yi34b": {"depth": 6, "ratios": [0.15], "rows": 16},
    "llama70b": {"depth": 6, "ratios": [0.10, 0.20], "rows": 8},
}
TOP_LOGITS = 16


def spec_of(name: str):
    spec = hz.workload(name)
    depth = CASES[name]["depth"]
    return spec if depth is None else hz.with_depth(spec, depth)


def path_of(name: str) -> str:
    return os.path.join(HERE, f"fullsize_{name}.npz")


def ratio_tag(r: float) -> str:
    return f"r{int(round(r * 100)):03d}"


def make(name: str) -> str:
    spec = spec_of(name)
    cfg = spec.cfg
    storage = "bf16" if cfg.dtype == "bf16" else "f32"
    n_rows = CASES[name]["rows"]
    W = hz.HostWeights(cfg, spec.seed)
    out = {"n_layers": np.int32(cfg.n_layers), "seed": np.int32(spec.seed),
           "n_requests": np.int32(len(spec.requests)),
           "ratios": np.array(CASES[name]["ratios"], dtype=np.float64)}
    t = time.perf_counter()
    caches = orc.precompute_all(cfg, W, spec, storage)
    # bf16-rounded values are exact in float32: halve the host memory the caches hold
    caches = {c: (k.astype(np.float32), v.astype(np.float32)) for c, (k, v) in caches.items()}
    out["precompute_s"] = np.float64(time.perf_counter() - t)
    print(f"{name}: {len(caches)} chunks precomputed in {out['precompute_s']:.0f} s", flush=True)
    for r in CASES[name]["ratios"]:
        tag = ratio_tag(r)
        ratios = orc.ratio_schedule(cfg.n_layers, r, spec.schedule)
        out[f"{tag}_schedule"] = np.array(ratios, dtype=np.float64)
        for q, segs in enumerate(spec.requests):
            t = time.perf_counter()
            res = orc.blend_prefill(cfg, W, segs, caches, ratios, storage)
            out[f"{tag}_q{q}_blend_s"] = np.float64(time.perf_counter() - t)
            for i in range(cfg.n_layers):
                if ratios[i] >= 0:
                    out[f"{tag}_q{q}_set_l{i}"] = res["sets"][i].astype(np.int32)
            rows = res["rows"]
            n_tok = sum(len(s.ids) for s in segs)
            n_query = len(segs[-1].ids)
            query_rows = np.arange(n_tok - min(n_rows, n_query), n_tok)
            cached_rows = rows[rows < n_tok - n_query]
            pick = np.random.default_rng(1000 * spec.seed + 10 * q + int(r * 100)).choice(
                len(cached_rows), size=min(n_rows, len(cached_rows)), replace=False)
            sample = np.sort(np.concatenate([cached_rows[pick], query_rows])).astype(np.int64)
            loc = np.searchsorted(rows, sample)
            assert np.array_equal(rows[loc], sample)
            out[f"{tag}_q{q}_rows"] = sample.astype(np.int32)
            out[f"{tag}_q{q}_hidden"] = res["hidden"][loc].astype(np.float32)
            logits = orc.lm_logits(cfg, W, res["hidden"][-1])
            top = np.lexsort((np.arange(len(logits)), -logits))[:TOP_LOGITS]
            assert int(top[0]) == res["first_token"]
            out[f"{tag}_q{q}_top_ids"] = top.astype(np.int32)
            out[f"{tag}_q{q}_top_logits"] = logits[top]
            print(f"{name} {tag} request {q}: blend {out[f'{tag}_q{q}_blend_s']:.0f} s, "
                  f"first token {res['first_token']}", flush=True)
    np.savez_compressed(path_of(name), **out)
    return path_of(name)


def full_path_of(name: str) -> str:
    return os.path.join(HERE, f"fullsize_{name}_full_prefill.npz")


def make_full(name: str, n_rows: int = 32) -> str:
    """The oracle's plain full prefill of the workload's first prompt (the full-recompute
    baseline): hidden rows of the last ``n_rows`` // 2 tokens and of as many earlier tokens
    drawn with a fixed seed, the top logits at the last token, and the wall time."""
    spec = spec_of(name)
    cfg = spec.cfg
    storage = "bf16" if cfg.dtype == "bf16" else "f32"
    W = hz.HostWeights(cfg, spec.seed)
    ids = np.concatenate([s.ids for s in spec.requests[0]])
    n = len(ids)
    t = time.perf_counter()
    res = orc.full_prefill(cfg, W, ids, storage)
    secs = time.perf_counter() - t
    tail = np.arange(n - n_rows // 2, n)
    early = np.sort(np.random.default_rng(7 * spec.seed).choice(n - n_rows // 2, n_rows // 2, replace=False))
    rows = np.concatenate([early, tail]).astype(np.int64)
    logits = orc.lm_logits(cfg, W, res["hidden"][-1])
    top = np.lexsort((np.arange(len(logits)), -logits))[:TOP_LOGITS]
    np.savez_compressed(full_path_of(name), n_layers=np.int32(cfg.n_layers), rows=rows.astype(np.int32),
                        hidden=res["hidden"][rows].astype(np.float32), top_ids=top.astype(np.int32),
                        top_logits=logits[top], full_prefill_s=np.float64(secs))
    print(f"{name}: full prefill of {n} tokens in {secs:.0f} s, first token {res['first_token']}", flush=True)
    return full_path_of(name)


if __name__ == "__main__":
    args = sys.argv[1:] or list(CASES)
    if args[0] == "--full-prefill":
        for n in args[1:]:
            print("wrote", make_full(n), flush=True)
    else:
        for n in args:
            print("wrote", make(n), flush=True)
