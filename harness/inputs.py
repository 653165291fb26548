"""Seeded synthetic inputs for the blended-prefill path (weights, token ids, prompts).

This module serves both sides of every parity check: the CPU oracle and the CUDA
library read the same bytes from here.  It holds none of the method's arithmetic
(no normalisation, no projection, no rotary embedding, no attention): only the
model shapes, a counter-based random generator and the prompt layouts.

Generator
---------
Every random value is a pure function of (key, counter), so any element of any
tensor can be produced on its own, in any order, on the host (numpy, here) or on
the GPU (``harness/gen_kernel.cu``, the same definition in CUDA).  Both produce
identical bits; a GPU test checks that.

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014): the n-th draw of a
  stream with seed ``key`` is ``mix64(key + (n + 1) * GAMMA)``.
* A weight element with flat index ``e`` takes draws ``2e`` and ``2e + 1`` and
  cuts four 22-bit integers ``k0..k3`` out of them.  Their centred sum
  ``z = k0 + k1 + k2 + k3 - (2**23 - 2)`` is an Irwin-Hall(4) variate with
  variance ``2**44 / 3``; ``w = fp32(z) * fp32(std * sqrt(3) / 2**22)`` then has
  mean 0 and standard deviation ``std`` (0.02).  ``z`` is exact in fp32 and the
  product is one correctly rounded fp32 multiply, so host and device agree
  bit for bit.  Weights of bf16 models are rounded to bf16 (round to nearest,
  ties to even) from that fp32 value.
* Token ids are uniform over the vocabulary or Zipf(1.1) (P(id = k - 1)
  proportional to k**-1.1), drawn by inverse CDF from 53-bit uniforms.

Model and prompt shapes follow the workloads of the CacheBlend pages: chunks of
128-512 tokens retrieved for a RAG prompt, a system prefix, a user query, and
decoders shaped like Mistral-7B, Llama-7B, Yi-34B and Llama-70B.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK22 = np.uint64((1 << 22) - 1)
WEIGHT_STD = 0.02

# tensor ids inside one layer (row-major [out_features, in_features] each)
MAT_Q, MAT_K, MAT_V, MAT_O, MAT_GATE, MAT_UP, MAT_DOWN = range(7)
LAYER_MATS = ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")
GLOBAL_EMBED_LAYER = 0xFFFF  # embedding table [vocab, d]
GLOBAL_LM_LAYER = 0xFFFE  # LM head [vocab, d]


# --------------------------------------------------------------------------- generator
def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on uint64 arrays (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def draw(key: int, n: np.ndarray) -> np.ndarray:
    """The n-th 64-bit draw of stream ``key`` (vectorised over ``n``)."""
    n = np.asarray(n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + (n + np.uint64(1)) * GAMMA)


def stream_key(seed: int, a: int, b: int = 0) -> int:
    """Key of the stream for (seed, a, b): two chained draws, so streams never overlap."""
    k1 = int(draw(seed & 0xFFFFFFFFFFFFFFFF, np.array([a], dtype=np.uint64))[0])
    return int(draw(k1, np.array([b], dtype=np.uint64))[0])


def weight_scale(std: float = WEIGHT_STD) -> np.float32:
    return np.float32(std * math.sqrt(3.0) / float(1 << 22))


def gen_weight_fp32_numpy(key: int, start: int, count: int, std: float = WEIGHT_STD) -> np.ndarray:
    """fp32 weights for flat indices [start, start + count) of the stream ``key`` (numpy)."""
    e = np.arange(start, start + count, dtype=np.uint64)
    w0 = draw(key, e * np.uint64(2))
    w1 = draw(key, e * np.uint64(2) + np.uint64(1))
    s = (w0 & _MASK22) + ((w0 >> np.uint64(22)) & _MASK22) + (w1 & _MASK22) + ((w1 >> np.uint64(22)) & _MASK22)
    z = s.astype(np.int64) - ((1 << 23) - 2)
    return z.astype(np.float32) * weight_scale(std)


_HOST_LIB_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "harness",
                              "libsynth_host.so")
_HOST_LIB = None


def host_generator():
    """The C twin of the generator (``harness/libsynth_host.so``), or None when it is not built."""
    global _HOST_LIB
    if _HOST_LIB is None:
        if not os.path.exists(_HOST_LIB_PATH):
            return None
        lib = ctypes.CDLL(_HOST_LIB_PATH)
        lib.synth_weights_host.restype = ctypes.c_int
        lib.synth_weights_host.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                           ctypes.c_int, ctypes.c_void_p]
        _HOST_LIB = lib
    return _HOST_LIB


def gen_weight_fp32_c(key: int, start: int, count: int, std: float = WEIGHT_STD, as_bf16: bool = False) -> np.ndarray:
    """The same elements from the C generator (threads over the range); ``as_bf16`` rounds
    each to bf16 (nearest, ties to even) and returns the fp32 value of the bf16."""
    lib = host_generator()
    if lib is None:
        raise RuntimeError(f"{_HOST_LIB_PATH} is missing: run `python -m rag_non_prefix_gb300.build`")
    out = np.empty(count, dtype=np.float32)
    lib.synth_weights_host(key & 0xFFFFFFFFFFFFFFFF, start, count, float(weight_scale(std)), int(as_bf16),
                           out.ctypes.data)
    return out


def gen_weight_fp32(key: int, start: int, count: int, std: float = WEIGHT_STD) -> np.ndarray:
    """fp32 weights for flat indices [start, start + count) of the stream ``key``: the C
    generator for large ranges when it is built, numpy otherwise (identical bits)."""
    if count >= 1 << 16 and host_generator() is not None:
        return gen_weight_fp32_c(key, start, count, std)
    return gen_weight_fp32_numpy(key, start, count, std)


def fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_fp32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def uniform53(key: int, start: int, count: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits each."""
    d = draw(key, np.arange(start, start + count, dtype=np.uint64))
    return (d >> np.uint64(11)).astype(np.float64) * (1.0 / float(1 << 53))


# --------------------------------------------------------------------------- models
@dataclasses.dataclass(frozen=True)
class ModelConfig:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_theta: float = 10000.0
    rms_eps: float = 1e-5
    dtype: str = "bf16"  # "f32" or "bf16": weights, cached KV and GEMM inputs

    @property
    def q_width(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv_heads * self.head_dim

    def mat_shape(self, mat: int):
        d, qw, kw, f = self.d_model, self.q_width, self.kv_width, self.ffn_dim
        return [(qw, d), (kw, d), (kw, d), (d, qw), (f, d), (f, d), (d, f)][mat]

    def params_per_layer(self) -> int:
        return sum(int(np.prod(self.mat_shape(m))) for m in range(7))


MODELS: Dict[str, ModelConfig] = {
    # configuration 1: tiny CPU-checkable decoder, fp32
    "tiny": ModelConfig("tiny", 2, 256, 4, 4, 64, 1024, 1000, 1e4, 1e-5, "f32"),
    # configuration 2: Mistral-7B shape
    "mistral7b": ModelConfig("mistral7b", 32, 4096, 32, 8, 128, 14336, 32000, 1e4, 1e-5, "bf16"),
    # configuration 3: Llama-7B shape (MHA)
    "llama7b": ModelConfig("llama7b", 32, 4096, 32, 32, 128, 11008, 32000, 1e4, 1e-5, "bf16"),
    # configuration 4: Yi-34B shape
    "yi34b": ModelConfig("yi34b", 60, 7168, 56, 8, 128, 20480, 64000, 5e6, 1e-5, "bf16"),
    # configuration 5: Llama-70B shape
    "llama70b": ModelConfig("llama70b", 80, 8192, 64, 8, 128, 28672, 32000, 1e4, 1e-5, "bf16"),
    # reduced shapes for element-by-element parity (oracle finishes in seconds)
    "small_bf16": ModelConfig("small_bf16", 4, 512, 8, 2, 128, 1536, 2048, 1e4, 1e-5, "bf16"),
    "small_mha_bf16": ModelConfig("small_mha_bf16", 3, 512, 4, 4, 128, 1024, 1024, 1e4, 1e-5, "bf16"),
    "small_gqa_f32": ModelConfig("small_gqa_f32", 3, 256, 8, 2, 64, 768, 512, 1e4, 1e-5, "f32"),
}


def layer_weight_key(seed: int, layer: int, mat: int) -> int:
    return stream_key(seed, layer, mat)


def gen_matrix(cfg: ModelConfig, seed: int, layer: int, mat: int, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """One weight matrix (or a subset of its rows) as float32 values of the model dtype."""
    out_f, in_f = cfg.mat_shape(mat) if layer < GLOBAL_LM_LAYER else (cfg.vocab, cfg.d_model)
    key = layer_weight_key(seed, layer, mat)
    if rows is None and host_generator() is not None:
        return gen_weight_fp32_c(key, 0, out_f * in_f, as_bf16=cfg.dtype == "bf16").reshape(out_f, in_f)
    if rows is None:
        w = gen_weight_fp32(key, 0, out_f * in_f).reshape(out_f, in_f)
    else:
        rows = np.asarray(rows, dtype=np.int64)
        w = np.empty((len(rows), in_f), dtype=np.float32)
        for i, r in enumerate(rows):
            w[i] = gen_weight_fp32(key, int(r) * in_f, in_f)
    if cfg.dtype == "bf16":
        w = bf16_bits_to_fp32(fp32_to_bf16_bits(w))
    return w


def gen_embedding_rows(cfg: ModelConfig, seed: int, ids: np.ndarray) -> np.ndarray:
    """Rows ``ids`` of the embedding table [vocab, d] (only the rows that are needed)."""
    uniq, inv = np.unique(np.asarray(ids, dtype=np.int64), return_inverse=True)
    rows = gen_matrix(cfg, seed, GLOBAL_EMBED_LAYER, 0, rows=uniq)
    return rows[inv]


def gen_lm_head(cfg: ModelConfig, seed: int) -> np.ndarray:
    return gen_matrix(cfg, seed, GLOBAL_LM_LAYER, 0)


def gen_layer_weights(cfg: ModelConfig, seed: int, layer: int) -> Dict[str, np.ndarray]:
    return {name: gen_matrix(cfg, seed, layer, m) for m, name in enumerate(LAYER_MATS)}


class HostWeights:
    """Lazily generated host copy of a model's weights (float32 values, dtype-exact)."""

    def __init__(self, cfg: ModelConfig, seed: int, cache_layers: bool = True):
        self.cfg, self.seed, self.cache_layers = cfg, seed, cache_layers
        self._layers: Dict[int, Dict[str, np.ndarray]] = {}
        self._lm = None

    def layer(self, i: int) -> Dict[str, np.ndarray]:
        if i in self._layers:
            return self._layers[i]
        w = gen_layer_weights(self.cfg, self.seed, i)
        if self.cache_layers:
            self._layers[i] = w
        return w

    def embed(self, ids) -> np.ndarray:
        return gen_embedding_rows(self.cfg, self.seed, ids)

    def lm_head(self) -> np.ndarray:
        if self._lm is None:
            self._lm = gen_lm_head(self.cfg, self.seed)
        return self._lm


# --------------------------------------------------------------------------- token ids
_ZIPF_CDF: Dict[tuple, np.ndarray] = {}


def zipf_cdf(vocab: int, s: float = 1.1) -> np.ndarray:
    if (vocab, s) not in _ZIPF_CDF:
        p = np.arange(1, vocab + 1, dtype=np.float64) ** (-s)
        c = np.cumsum(p)
        _ZIPF_CDF[(vocab, s)] = c / c[-1]
    return _ZIPF_CDF[(vocab, s)]


def gen_token_ids(key: int, n: int, vocab: int, dist: str) -> np.ndarray:
    u = uniform53(key, 0, n)
    if dist == "uniform":
        ids = np.floor(u * vocab).astype(np.int64)
    elif dist == "zipf":
        ids = np.searchsorted(zipf_cdf(vocab), u, side="right").astype(np.int64)
    else:
        raise ValueError(dist)
    return np.minimum(ids, vocab - 1).astype(np.int32)


# --------------------------------------------------------------------------- prompts
@dataclasses.dataclass
class Segment:
    """One piece of a prompt: a cached chunk (``chunk`` = its pool index) or the query (chunk = -1)."""
    ids: np.ndarray
    chunk: int


@dataclasses.dataclass
class PromptSpec:
    """A workload: the model, a chunk pool and one or more requests built from it."""
    name: str
    model: str
    seed: int
    ratio: float
    schedule: str  # "fixed" or "gradual"
    chunks: List[np.ndarray]  # the pool of independently cached chunks (token ids)
    requests: List[List[Segment]]  # per request: [prefix chunk?][chunks...][query]
    id_dist: str
    depth: Optional[int] = None  # when set: only the model's first ``depth`` layers (same weights)

    @property
    def cfg(self) -> ModelConfig:
        c = MODELS[self.model]
        if self.depth is None:
            return c
        return dataclasses.replace(c, n_layers=self.depth, name=f"{c.name}@{self.depth}")

    def n_tokens(self, r: int = 0) -> int:
        return sum(len(s.ids) for s in self.requests[r])

    def n_cached(self, r: int = 0) -> int:
        return sum(len(s.ids) for s in self.requests[r] if s.chunk >= 0)


def _chunk_ids(seed: int, index: int, n: int, vocab: int, dist: str) -> np.ndarray:
    return gen_token_ids(stream_key(seed, 0x10000 + index, 1), n, vocab, dist)


def _query_ids(seed: int, request: int, n: int, vocab: int, dist: str) -> np.ndarray:
    return gen_token_ids(stream_key(seed, 0x20000 + request, 2), n, vocab, dist)


def make_prompt(model: str, seed: int, chunk_lens: Sequence[int], query_len: int, ratio: float,
                schedule: str = "gradual", id_dist: str = "zipf", prefix_len: int = 0,
                name: str = "custom") -> PromptSpec:
    """One request: [system prefix (a cached chunk at offset 0)] + chunks + query."""
    cfg = MODELS[model]
    lens = ([prefix_len] if prefix_len else []) + list(chunk_lens)
    chunks = [_chunk_ids(seed, i, n, cfg.vocab, id_dist) for i, n in enumerate(lens)]
    req = [Segment(c, i) for i, c in enumerate(chunks)]
    req.append(Segment(_query_ids(seed, 0, query_len, cfg.vocab, id_dist), -1))
    return PromptSpec(name, model, seed, ratio, schedule, chunks, [req], id_dist)


def make_pooled_batch(model: str, seed: int, pool: int, chunk_len: int, per_request: int,
                      n_requests: int, query_len: int, ratio: float, schedule: str = "gradual",
                      id_dist: str = "zipf", name: str = "pooled") -> PromptSpec:
    """Requests that each draw ``per_request`` distinct chunks from a shared pool (chunks recur)."""
    cfg = MODELS[model]
    chunks = [_chunk_ids(seed, i, chunk_len, cfg.vocab, id_dist) for i in range(pool)]
    reqs = []
    for r in range(n_requests):
        u = uniform53(stream_key(seed, 0x30000 + r, 3), 0, pool)
        order = np.argsort(u, kind="stable")[:per_request]
        segs = [Segment(chunks[int(c)], int(c)) for c in order]
        segs.append(Segment(_query_ids(seed, r, query_len, cfg.vocab, id_dist), -1))
        reqs.append(segs)
    return PromptSpec(name, model, seed, ratio, schedule, chunks, reqs, id_dist)


def workload(name: str) -> PromptSpec:
    """The five named workloads (shapes of the pages' RAG prompts) and reduced parity cases."""
    if name == "tiny":  # 2 x 128 cached + 32 query, uniform ids, r = 15 %, fixed schedule
        return make_prompt("tiny", 1, [128, 128], 32, 0.15, "fixed", "uniform", name=name)
    if name == "mistral7b":  # 64 prefix + 6 x 512 + 64 query, Zipf(1.1), r = 15 %
        return make_prompt("mistral7b", 2, [512] * 6, 64, 0.15, "gradual", "zipf", prefix_len=64, name=name)
    if name == "llama7b":  # 8 x 512 + 32 query (host-staged KV), Zipf(1.1), r = 15 % (swept)
        return make_prompt("llama7b", 3, [512] * 8, 32, 0.15, "gradual", "zipf", name=name)
    if name == "yi34b":  # 16 x 512 + 128 query
        return make_prompt("yi34b", 4, [512] * 16, 128, 0.15, "gradual", "zipf", name=name)
    if name == "llama70b":  # 4 requests x (32 of a pool of 64 chunks of 256) + 64 query
        return make_pooled_batch("llama70b", 5, 64, 256, 32, 4, 64, 0.10, name=name)
    if name == "small_bf16":  # several tiles and a ragged tail
        return make_prompt("small_bf16", 11, [160, 144, 176], 40, 0.15, "gradual", "zipf", prefix_len=32, name=name)
    if name == "small_mha_bf16":
        return make_prompt("small_mha_bf16", 12, [96, 128], 24, 0.2, "gradual", "zipf", name=name)
    if name == "small_gqa_f32":
        return make_prompt("small_gqa_f32", 13, [64, 80, 72], 20, 0.2, "gradual", "uniform", prefix_len=16, name=name)
    raise KeyError(name)


def with_depth(spec: PromptSpec, depth: int) -> PromptSpec:
    """The same prompts on the first ``depth`` layers of the model: every width, head count,
    FFN size, rotary base, token count and batch unchanged; layer i keeps its weights (they
    are keyed by (seed, layer, matrix)), as do the embedding and the LM head."""
    if not 1 <= depth <= MODELS[spec.model].n_layers:
        raise ValueError(depth)
    return dataclasses.replace(spec, depth=depth, name=f"{spec.name}@{depth}")


def ratio_for_k(k: int, n_cached: int) -> float:
    return k / n_cached
