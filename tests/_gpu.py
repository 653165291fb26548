"""Shared set-up of the GPU parity tests: the CUDA path (through the C ABI) and the
oracle, each fed from the harness with the same seeds."""
from __future__ import annotations

import functools

import numpy as np
import torch

import harness as hz
import harness.device as hd
import oracle.cacheblend as orc
import rag_non_prefix_gb300 as cb
from rag_non_prefix_gb300 import build as cbbuild


@functools.lru_cache(maxsize=None)
def built():
    cbbuild.build()
    cb.load_library()
    return True


def storage_of(cfg) -> str:
    return "bf16" if cfg.dtype == "bf16" else "f32"


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


class GpuWorkload:
    """A workload on the GPU: weights, an engine, every chunk precomputed and registered."""

    def __init__(self, spec: hz.PromptSpec, on_host: bool = False, max_tokens=None, extra_positions: int = 0):
        built()
        self.spec = spec
        self.cfg = spec.cfg
        self.W = hd.device_weights(self.cfg, spec.seed)
        total = sum(spec.n_tokens(r) for r in range(len(spec.requests)))
        longest = max(max((len(c) for c in spec.chunks), default=0),
                      max(spec.n_tokens(r) for r in range(len(spec.requests))))
        self.eng = cb.Engine(self.cfg, self.W, max_tokens=max_tokens or max(total, longest),
                             max_requests=len(spec.requests), max_positions=longest + 1 + extra_positions)
        self.chunk_kv = {}
        used = sorted({s.chunk for req in spec.requests for s in req if s.chunk >= 0})
        for c in used:
            ids = hd.ids_tensor(spec.chunks[c])
            k, v = self.eng.precompute_chunk(ids)
            if on_host:
                k, v = k.cpu().pin_memory(), v.cpu().pin_memory()
            self.chunk_kv[c] = (ids, k, v)
            self.eng.register_chunk(c, ids, k, v, on_host=on_host)
        torch.cuda.synchronize()

    def requests(self):
        out = []
        for req in self.spec.requests:
            chunks = [s.chunk for s in req if s.chunk >= 0]
            q = [s for s in req if s.chunk < 0][0]
            out.append(self.eng.make_request(chunks, hd.ids_tensor(q.ids)))
        return out

    def blend(self, ratios, forced=None, copy_stream=None, dev_mode=0, seam_tokens=None):
        reqs = self.requests()
        self.eng.blend_prefill(reqs, ratios, dev_mode=dev_mode, forced=forced,
                               copy_stream=copy_stream, seam_tokens=seam_tokens)
        self.eng.get_status()
        torch.cuda.synchronize()
        return reqs


class OracleWorkload:
    """The same workload in the oracle (fp64, KV stored in the model dtype)."""

    def __init__(self, spec: hz.PromptSpec):
        self.spec = spec
        self.cfg = spec.cfg
        self.W = hz.HostWeights(self.cfg, spec.seed)
        self.storage = storage_of(self.cfg)
        self.caches = orc.precompute_all(self.cfg, self.W, spec, self.storage)

    def blend(self, r: int, ratios, force_sel=None, dev_mode=0):
        return orc.blend_prefill(self.cfg, self.W, self.spec.requests[r], self.caches, ratios, self.storage,
                                 dev_mode=dev_mode, force_sel=force_sel)

    def seam(self, r: int, seam_tokens: int):
        return orc.seam_repair_prefill(self.cfg, self.W, self.spec.requests[r], self.caches, seam_tokens,
                                       self.storage)

    def full(self, r: int):
        ids = np.concatenate([s.ids for s in self.spec.requests[r]])
        return orc.full_prefill(self.cfg, self.W, ids, self.storage)


def max_rel_err(gpu_rows: np.ndarray, ref_rows: np.ndarray) -> float:
    """max over rows t of ||g_t - o_t||_inf / ||o_t||_inf."""
    num = np.max(np.abs(gpu_rows - ref_rows), axis=1)
    den = np.maximum(np.max(np.abs(ref_rows), axis=1), 1e-30)
    return float(np.max(num / den))


def forced_from_oracle(res, n_cached: int, n_layers: int, ratios):
    """{check layer: [cached part of the oracle's S_i]} for the GPU's forced-selection mode."""
    out = {}
    for i in range(n_layers):
        if ratios[i] >= 0:
            S = res["sets"][i]
            out[i] = [[int(x) for x in S if x < n_cached]]
    return out


def bf16_operand_full_prefill(cfg, W, ids: np.ndarray, rounding="all") -> torch.Tensor:
    """A plain-PyTorch full prefill on the GPU that rounds to bf16 exactly the operands a bf16
    tensor-core path must round, and computes everything else in fp32 (TF32 off): the
    normalised rows x entering each projection, q / k / v after RoPE (the cache's K and V),
    the softmax probabilities P entering P.V (the row sum taken before rounding), the
    attention output entering the output projection, and the SwiGLU output entering the down
    projection; the residual stream stays fp32.

    It shares no code with the library or the oracle (library routines: matmul, rms_norm,
    silu).  Its distance to the oracle's fp64 prefill is the rounding floor of bf16 operands
    for the model's depth, against which the library's own error is judged.  rounding="none"
    (or False) gives the same prefill with no operand rounded (fp32 throughout);
    rounding="kv" rounds only K and V, as a bf16 cache stores them (the oracle's model of the
    path).  Returns the hidden states [N, d] (fp32)."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        if rounding is True:
            rounding = "all"
        elif rounding is False:
            rounding = "none"
        rnd = lambda t: t.to(torch.bfloat16).to(torch.float32)  # noqa: E731
        keep = lambda t: t  # noqa: E731
        bf = rnd if rounding == "all" else keep
        bkv = rnd if rounding in ("all", "kv") else keep
        dev = W["embed"].device
        t_ids = torch.from_numpy(np.asarray(ids, dtype=np.int64)).to(dev)
        N, d, H, Hkv, dh = len(ids), cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
        G, half = H // Hkv, dh // 2
        h = W["embed"][t_ids].float()
        inv = torch.pow(torch.tensor(float(cfg.rope_theta), dtype=torch.float64),
                        -2.0 * torch.arange(half, dtype=torch.float64) / dh)
        ang = torch.arange(N, dtype=torch.float64)[:, None] * inv[None, :]
        cos, sin = ang.cos().float().to(dev)[:, None, :], ang.sin().float().to(dev)[:, None, :]

        def rope(x):
            a, b = x[..., :half], x[..., half:]
            return torch.cat([a * cos - b * sin, b * cos + a * sin], dim=-1)

        later = torch.ones(N, N, dtype=torch.bool, device=dev).triu(1)  # key after query
        scale = 1.0 / float(np.sqrt(dh))
        for lw in W["layers"][: cfg.n_layers]:
            x = bf(torch.nn.functional.rms_norm(h, (d,), eps=cfg.rms_eps))
            q = bf(rope((x @ lw["wq"].float().T).view(N, H, dh)))
            k = bkv(rope((x @ lw["wk"].float().T).view(N, Hkv, dh)))
            v = bkv((x @ lw["wv"].float().T).view(N, Hkv, dh))
            att = torch.empty(N, H, dh, device=dev)
            for g in range(Hkv):
                s = torch.einsum("ngd,md->gnm", q[:, g * G:(g + 1) * G, :], k[:, g, :]) * scale
                s = s.masked_fill(later, float("-inf"))
                p = torch.exp(s - s.amax(dim=-1, keepdim=True))
                o = (bf(p) @ v[:, g, :]) / p.sum(dim=-1, keepdim=True)
                att[:, g * G:(g + 1) * G, :] = o.transpose(0, 1)
            h = h + bf(att.reshape(N, H * dh)) @ lw["wo"].float().T
            x2 = bf(torch.nn.functional.rms_norm(h, (d,), eps=cfg.rms_eps))
            act = bf(torch.nn.functional.silu(x2 @ lw["wgate"].float().T) * (x2 @ lw["wup"].float().T))
            h = h + act @ lw["wdown"].float().T
        return h
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
