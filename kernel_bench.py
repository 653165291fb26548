"""Per-kernel timing of the library's hot kernels through the C ABI (CUDA events).

    python kernel_bench.py gemm --M 535 --N 28672 --K 4096 --mode swiglu
    python kernel_bench.py attention --H 32 --Hkv 8 --N 3200 --m 535 [--tiles 1|2] [--causal]
    python kernel_bench.py rerotate --rows 100352 --hkv 8
    python kernel_bench.py select --n 3136 --k 471
    python kernel_bench.py deviation --n 3200 --kvw 1024
    python kernel_bench.py codec --n 3136 --hkv 8 --bits 8
    python kernel_bench.py decode --layers 32 --steps 2

(`decode` builds the Mistral-7B-shaped model with --layers layers, blends the configuration-2
prompt, decodes 4 warm-up steps, then --steps steps inside the NVTX range "decode_prof" that
profilers can filter on.)

Operands are random device tensors sized like one layer of the Mistral-7B-shaped
workload; weight operands exceed the 129 MB L2 where the shape allows, and a 512 MiB
buffer is written between timed launches.  Prints one JSON line with the average
launch time and the achieved rate (TFLOP/s or GB/s of algorithmic traffic).
"""
from __future__ import annotations

import argparse
import json

import torch

import rag_non_prefix_gb300 as cb
from rag_non_prefix_gb300 import build as cbbuild


def _time(fn, iters, warmup=3, flush=None, batch=1):
    """Average and best time of one launch; with batch > 1, `batch` launches run back to
    back between the events and the time is divided by `batch` (launch gaps included, host
    launch latency hidden behind the queue)."""
    for _ in range(warmup):
        fn()
    ts = []
    for _ in range(iters):
        if flush is not None:
            flush.fill_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s = torch.cuda.current_stream()
        if batch > 1:
            torch.cuda._sleep(2_000_000)  # keeps the GPU busy while the launches queue up
        a.record(s)
        for _ in range(batch):
            fn()
        b.record(s)
        b.synchronize()
        ts.append(a.elapsed_time(b) / batch)
    return sum(ts) / len(ts), min(ts)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=["gemm", "attention", "rerotate", "select", "deviation", "codec", "decode"])
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--M", type=int, default=535)
    ap.add_argument("--N", type=int, default=28672)
    ap.add_argument("--K", type=int, default=4096)
    ap.add_argument("--mode", default="swiglu", choices=["store", "add", "swiglu"])
    ap.add_argument("--H", type=int, default=32)
    ap.add_argument("--Hkv", type=int, default=8)
    ap.add_argument("--m", type=int, default=535)
    ap.add_argument("--rows", type=int, default=32 * 3136)
    ap.add_argument("--hkv", type=int, default=8)
    ap.add_argument("--n", type=int, default=3136)
    ap.add_argument("--k", type=int, default=471)
    ap.add_argument("--kvw", type=int, default=1024)
    ap.add_argument("--bits", type=int, default=8)
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--tiles", type=int, default=0, help="attention: query tiles per CTA (0 by size, 1, 2)")
    ap.add_argument("--causal", action="store_true", help="attention: every position a query (full prefill)")
    ap.add_argument("--no-flush", action="store_true")
    ap.add_argument("--batch", type=int, default=1, help="launches per timed region")
    ap.add_argument("--no-stream-k", action="store_true", help="GEMM without scratch: whole tiles per CTA")
    ap.add_argument("--orientation", type=int, default=0,
                    help="GEMM tiles: 0 by the time model, 1 token rows, 2 weight rows, 16..256 weight rows "
                         "with that many tokens per tile")
    ap.add_argument("--pairing", type=int, default=0,
                    help="GEMM CTA pairs: 0 by the time model, 1 never, 2 clusters of one pair, 4 of two")
    a = ap.parse_args()
    cbbuild.build()
    torch.manual_seed(0)
    dev = torch.device("cuda")
    flush = None if a.no_flush else torch.empty(128 * 1024 * 1024, dtype=torch.float32, device=dev)
    out = {"kernel": a.kernel}
    if a.kernel == "gemm":
        M, N, K = a.M, a.N, a.K
        scr = None if a.no_stream_k else cb.gemm_scratch(dev)
        cb.cb_gemm_set_orientation(a.orientation)
        cb.cb_gemm_set_pairing(a.pairing)
        A = (torch.randn(M, K, device=dev) * 0.5).to(torch.bfloat16)
        if a.mode == "swiglu":
            G = (torch.randn(N // 2, K, device=dev) * 0.02).to(torch.bfloat16)
            U = (torch.randn(N // 2, K, device=dev) * 0.02).to(torch.bfloat16)
            C = torch.empty(M, N // 2, dtype=torch.bfloat16, device=dev)
            fn = lambda: cb.cb_gemm(A, G, C, 2, B2=U, scratch=scr)  # noqa: E731
        else:
            B = (torch.randn(N, K, device=dev) * 0.02).to(torch.bfloat16)
            C = torch.zeros(M, N, dtype=torch.float32, device=dev)
            fn = lambda: cb.cb_gemm(A, B, C, 1 if a.mode == "add" else 0, scratch=scr)  # noqa: E731
        avg, best = _time(fn, a.iters, a.warmup, flush, a.batch)
        fl = 2.0 * M * N * K
        out.update(shape=[M, N, K], mode=a.mode, stream_k=scr is not None, orientation=a.orientation, pairing=a.pairing,
                   plan=cb.cb_gemm_describe(M, N, K, {"store": 0, "add": 1, "swiglu": 2}[a.mode], 0 if scr is None else scr.numel()), ms=avg, best_ms=best, tflops=fl / (avg * 1e-3) / 1e12,
                   weight_bytes=N * K * 2)
    elif a.kernel == "attention":
        H, Hkv, N, m = a.H, a.Hkv, a.N, a.m
        pos = torch.sort(torch.randperm(N, device=dev)[:m]).values.to(torch.int32)
        q = torch.randn(m, H, 128, device=dev).to(torch.bfloat16)
        k = torch.randn(N, Hkv, 128, device=dev).to(torch.bfloat16)
        v = torch.randn(N, Hkv, 128, device=dev).to(torch.bfloat16)
        o = torch.empty_like(q)
        if a.causal:  # every position a query: the attention of a full prefill
            pos = torch.arange(N, device=dev, dtype=torch.int32)
            q = torch.randn(N, H, 128, device=dev).to(torch.bfloat16)
            o = torch.empty_like(q)
        cb.cb_attention_set_tiles(a.tiles)
        fn = lambda: cb.cb_attention(q, pos, k, v, o)  # noqa: E731
        avg, best = _time(fn, a.iters, a.warmup, flush, a.batch)
        cb.cb_attention_set_tiles(0)
        fl = 4.0 * H * 128 * float((pos.to(torch.float64) + 1).sum())
        out.update(shape=[H, Hkv, N, int(pos.numel())], tiles=a.tiles, ms=avg, best_ms=best,
                   tflops=fl / (avg * 1e-3) / 1e12)
    elif a.kernel == "rerotate":
        k = torch.randn(a.rows, a.hkv, 128, device=dev).to(torch.bfloat16)
        v = torch.randn(a.rows, a.hkv, 128, device=dev).to(torch.bfloat16)
        kd, vd = torch.empty_like(k), torch.empty_like(v)
        fn = lambda: cb.cb_rope_rerotate(k, kd, v, vd, 1234, 1e4)  # noqa: E731
        avg, best = _time(fn, a.iters, a.warmup, flush, a.batch)
        by = 4 * k.numel() * 2  # K and V, read and written
        out.update(rows=a.rows, ms=avg, best_ms=best, gbs=by / (avg * 1e-3) / 1e9, bytes=by)
    elif a.kernel == "select":
        d = torch.rand(a.n, device=dev)
        cand = torch.arange(a.n, dtype=torch.int32, device=dev)
        o = torch.empty(a.k, dtype=torch.int32, device=dev)
        fn = lambda: cb.cb_select_hkvd(d, cand, a.k, o)  # noqa: E731
        avg, best = _time(fn, a.iters, a.warmup, None, a.batch)
        out.update(n=a.n, k=a.k, ms=avg, best_ms=best)
    elif a.kernel == "deviation":
        kn = torch.randn(a.n, a.kvw, device=dev)
        vn = torch.randn(a.n, a.kvw, device=dev)
        kf = torch.randn(a.n, a.kvw, device=dev).to(torch.bfloat16)
        vf = torch.randn(a.n, a.kvw, device=dev).to(torch.bfloat16)
        dv = torch.empty(a.n, device=dev)
        fn = lambda: cb.cb_kv_deviation(kn, vn, kf, vf, None, 0, dv)  # noqa: E731
        avg, best = _time(fn, a.iters, a.warmup, flush, a.batch)
        by = a.n * a.kvw * (4 + 2) * 2
        out.update(n=a.n, ms=avg, best_ms=best, gbs=by / (avg * 1e-3) / 1e9, bytes=by)
    elif a.kernel == "codec":
        # decode + re-rotation of a quantised chunk of n tokens, all layers in one launch
        shape = (a.layers, a.n, a.hkv, 128)
        k = torch.randn(shape, device=dev).to(torch.bfloat16)
        v = torch.randn(shape, device=dev).to(torch.bfloat16)
        blob = cb.cb_kv_encode(k, v, a.bits)
        kd, vd = torch.empty_like(k), torch.empty_like(v)
        lib = cb.load_library()
        fn = lambda: cb._check(lib.cb_kv_decode(cb._ptr(blob), *shape, a.bits, 1234, 1e4, cb.CB_BF16,  # noqa: E731
                                                cb._ptr(kd), cb._ptr(vd), cb._stream(None)))
        avg, best = _time(fn, a.iters, a.warmup, flush, a.batch)
        by = blob.numel() + 2 * k.numel() * 2  # blob read, K and V written
        enc = lambda: cb.cb_kv_encode(k, v, a.bits, blob)  # noqa: E731
        eavg, _ = _time(enc, max(3, a.iters // 4), 1, flush, 1)
        out.update(shape=list(shape), bits=a.bits, ms=avg, best_ms=best, gbs=by / (avg * 1e-3) / 1e9, bytes=by,
                   blob_bytes=blob.numel(), encode_ms=eavg)
    elif a.kernel == "decode":
        import harness as hz
        import harness.device as hd

        base = hz.MODELS["mistral7b"]
        cfg = hz.ModelConfig(f"mistral7b_{a.layers}l", a.layers, base.d_model, base.n_heads, base.n_kv_heads,
                             base.head_dim, base.ffn_dim, base.vocab, base.rope_theta, base.rms_eps, base.dtype)
        hz.MODELS[cfg.name] = cfg
        spec = hz.make_prompt(cfg.name, 2, [512] * 6, 64, 0.15, "gradual", "zipf", prefix_len=64)
        W = hd.device_weights(cfg, spec.seed)
        n = spec.n_tokens(0)
        eng = cb.Engine(cfg, W, max_tokens=n, max_requests=1, max_positions=n + a.steps + 16)
        for sg in spec.requests[0]:
            if sg.chunk >= 0:
                ids = hd.ids_tensor(sg.ids)
                k, v = eng.precompute_chunk(ids)
                eng.register_chunk(sg.chunk, ids, k, v)
        qseg = [sg for sg in spec.requests[0] if sg.chunk < 0][0]
        req = eng.make_request([sg.chunk for sg in spec.requests[0] if sg.chunk >= 0], hd.ids_tensor(qseg.ids),
                               want_hidden=False, want_sel=False, decode_room=a.steps + 8)
        eng.blend_prefill([req], cb.ratio_schedule(cfg.n_layers, 0.15, "gradual"))
        tok = req["first_token"].clone()
        for _ in range(4):
            tok = eng.decode_step([req], tok)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.nvtx.range_push("decode_prof")
        ev[0].record()
        for _ in range(a.steps):
            tok = eng.decode_step([req], tok)
        ev[1].record()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        eng.get_status()
        out.update(layers=a.layers, context=n, steps=a.steps, ms_per_step=ev[0].elapsed_time(ev[1]) / a.steps)
    torch.cuda.synchronize()
    print(json.dumps(out))


if __name__ == "__main__":
    main()
