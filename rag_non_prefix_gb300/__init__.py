"""Python binding of the GB300 blended-prefill library (include/cacheblend.h).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libcacheblend.so``.  PyTorch provides device memory and streams.  Importing this
package does not need a GPU; calling into the library does, and fails loudly when the
shared library has not been built (``python -m rag_non_prefix_gb300.build``).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcacheblend.so")

CB_F32, CB_BF16 = 0, 1
STATUS = {0: "CB_OK", 1: "CB_ERR_INVALID_ARG", 2: "CB_ERR_SHAPE", 3: "CB_ERR_DTYPE", 4: "CB_ERR_NOT_FOUND",
          5: "CB_ERR_WORKSPACE", 6: "CB_ERR_CUDA", 7: "CB_ERR_TIMEOUT", 8: "CB_ERR_NAN", 9: "CB_ERR_DEVICE",
          10: "CB_ERR_STATE"}
EXPORTED = ("cb_create", "cb_destroy", "cb_status_string", "cb_last_error", "cb_workspace_size", "cb_set_workspace",
            "cb_precompute_chunk", "cb_register_chunk", "cb_unregister_chunk", "cb_registered_chunks",
            "cb_rope_rerotate", "cb_kv_deviation", "cb_select_hkvd", "cb_gemm", "cb_gemm_scratch_size", "cb_attention",
            "cb_blend_prefill",
            "cb_full_prefill", "cb_blend_begin", "cb_fetch_kv", "cb_synchronize", "cb_prefill_layer",
            "cb_blend_layer", "cb_blend_finish", "cb_get_status", "cb_plan_counts", "cb_set_profiling",
            "cb_get_profile", "cb_get_layer_profile", "cb_gemm_noalloc", "cb_gemm_noalloc_error", "cb_gemm_noalloc_scratch_used", "cb_gemm_get_status", "cb_gemm_set_orientation", "cb_gemm_set_pairing", "cb_gemm_describe", "cb_attention_set_tiles", "cb_set_qkv_fusion",
            "cb_set_launch_overlap", "cb_codec_layer_bytes", "cb_kv_encode", "cb_kv_decode", "cb_register_chunk_codec",
            "cb_set_staging", "cb_chunk_hash", "cb_chunk_info_of", "cb_plan_loading", "cb_decode_step",
            "cb_ratio_schedule", "cb_k_for_ratio")
PHASES = ("begin", "staged_rot", "norm", "qkv", "rope", "deviation", "select", "scatter", "attention", "oproj",
          "gateup", "down", "finish")


class CacheBlendError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status
        self.name = STATUS.get(status, str(status))


class ModelCfg(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("d_model", C.c_int), ("n_heads", C.c_int), ("n_kv_heads", C.c_int),
                ("head_dim", C.c_int), ("ffn_dim", C.c_int), ("vocab", C.c_int), ("rope_theta", C.c_double),
                ("rms_eps", C.c_float), ("dtype", C.c_int), ("max_positions", C.c_int)]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p)] + [
        (n, C.POINTER(C.c_void_p)) for n in ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")]


CB_SELECT_HKVD, CB_SELECT_SEAM = 0, 1


class BlendParams(C.Structure):
    _fields_ = [("n_layers", C.c_int), ("layer_ratio_host", C.POINTER(C.c_double)), ("dev_mode", C.c_int),
                ("forced_sel_host", C.POINTER(C.POINTER(C.c_int32))), ("select_mode", C.c_int),
                ("seam_tokens", C.c_int)]


class Request(C.Structure):
    _fields_ = [("n_chunks", C.c_int), ("chunk_ids_host", C.POINTER(C.c_uint64)), ("query_ids", C.c_void_p),
                ("n_query", C.c_int), ("fused_k", C.c_void_p), ("fused_v", C.c_void_p), ("out_hidden", C.c_void_p),
                ("out_sel", C.c_void_p), ("out_sel_count", C.c_void_p), ("out_first_token", C.c_void_p),
                ("kv_capacity", C.c_int)]


class DecodeSeq(C.Structure):
    _fields_ = [("fused_k", C.c_void_p), ("fused_v", C.c_void_p), ("kv_capacity", C.c_int), ("n_past", C.c_int),
                ("out_hidden", C.c_void_p)]


class ChunkInfo(C.Structure):
    _fields_ = [("n_tokens", C.c_int), ("tier", C.c_int), ("bytes", C.c_double)]


class CostModel(C.Structure):
    _fields_ = [("link_bytes_per_s", C.c_double), ("link_latency_s", C.c_double),
                ("prefill_s_per_token", C.c_double), ("recompute_fixed_s", C.c_double),
                ("r_min", C.c_double), ("r_max", C.c_double)]


TIER_MISSING, TIER_DEVICE, TIER_HOST = -1, 0, 1
ACT_USE, ACT_LOAD, ACT_RECOMPUTE = 0, 1, 2


class Profile(C.Structure):
    _fields_ = [("ms", C.c_float * len(PHASES)), ("launches", C.c_int * len(PHASES)), ("calls", C.c_int * len(PHASES))]


_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libcacheblend.so (once) and declares the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m rag_non_prefix_gb300.build` "
                           "(there is no fallback implementation)")
    lib = C.CDLL(path)
    vp, i32p, st = C.c_void_p, C.c_void_p, C.c_int
    sig = {
        "cb_create": (st, [C.POINTER(ModelCfg), C.POINTER(Weights), C.POINTER(C.c_void_p)]),
        "cb_destroy": (st, [vp]),
        "cb_status_string": (C.c_char_p, [st]),
        "cb_last_error": (C.c_char_p, [vp]),
        "cb_workspace_size": (C.c_size_t, [vp, C.c_int, C.c_int]),
        "cb_set_workspace": (st, [vp, vp, C.c_size_t, C.c_int, C.c_int]),
        "cb_precompute_chunk": (st, [vp, i32p, C.c_int, vp, vp, vp]),
        "cb_register_chunk": (st, [vp, C.c_uint64, i32p, vp, vp, C.c_int, C.c_int]),
        "cb_unregister_chunk": (st, [vp, C.c_uint64]),
        "cb_registered_chunks": (C.c_int, [vp]),
        "cb_rope_rerotate": (st, [vp, vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, C.c_double, C.c_int, vp]),
        "cb_kv_deviation": (st, [vp, vp, vp, vp, i32p, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp]),
        "cb_select_hkvd": (st, [vp, i32p, C.c_int, C.c_int, i32p, i32p, vp]),
        "cb_gemm": (st, [vp, vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, vp, C.c_size_t, vp]),
        "cb_gemm_scratch_size": (C.c_size_t, []),
        "cb_gemm_set_orientation": (st, [C.c_int]),
        "cb_gemm_set_pairing": (st, [C.c_int]),
        "cb_gemm_describe": (st, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_size_t, C.c_char_p, C.c_size_t]),
        "cb_attention_set_tiles": (st, [C.c_int]),
        "cb_set_qkv_fusion": (st, [C.c_int]),
        "cb_set_launch_overlap": (st, [C.c_int]),
        "cb_gemm_noalloc": (st, [vp, vp, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, vp]),
        "cb_gemm_noalloc_error": (C.c_char_p, []),
        "cb_gemm_get_status": (st, [vp, C.c_int]),
        "cb_gemm_noalloc_scratch_used": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int]),
        "cb_attention": (st, [vp, i32p, C.c_int, vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp, C.c_int, vp]),
        "cb_codec_layer_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
        "cb_kv_encode": (st, [vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, vp, vp]),
        "cb_kv_decode": (st, [vp, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_int, C.c_double, C.c_int, vp, vp,
                              vp]),
        "cb_register_chunk_codec": (st, [vp, C.c_uint64, i32p, vp, C.c_int, C.c_int, C.c_int]),
        "cb_set_staging": (st, [vp, vp, C.c_size_t]),
        "cb_chunk_hash": (C.c_uint64, [C.POINTER(C.c_int32), C.c_int]),
        "cb_ratio_schedule": (st, [C.c_int, C.c_double, C.c_int, C.c_double, C.c_int, C.POINTER(C.c_double)]),
        "cb_k_for_ratio": (C.c_int, [C.c_double, C.c_int]),
        "cb_decode_step": (st, [vp, C.POINTER(DecodeSeq), C.c_int, vp, vp, vp]),
        "cb_chunk_info_of": (st, [vp, C.c_uint64, C.POINTER(ChunkInfo)]),
        "cb_plan_loading": (st, [C.POINTER(CostModel), C.POINTER(ChunkInfo), C.c_int, C.c_int, C.POINTER(C.c_int32),
                                 C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(C.c_double)]),
        "cb_blend_prefill": (st, [vp, C.POINTER(Request), C.c_int, C.POINTER(BlendParams), vp, vp]),
        "cb_full_prefill": (st, [vp, i32p, C.c_int, vp, vp, vp, i32p, vp]),
        "cb_blend_begin": (st, [vp, C.POINTER(Request), C.c_int, C.POINTER(BlendParams), vp]),
        "cb_fetch_kv": (st, [vp, C.c_int, vp]),
        "cb_synchronize": (st, [vp, C.c_int, C.c_int]),
        "cb_prefill_layer": (st, [vp, C.c_int, vp]),
        "cb_blend_layer": (st, [vp, C.c_int, vp]),
        "cb_blend_finish": (st, [vp, vp]),
        "cb_get_status": (st, [vp, vp, C.c_int]),
        "cb_plan_counts": (st, [vp, C.c_int, C.POINTER(C.c_int32)]),
        "cb_set_profiling": (st, [vp, C.c_int]),
        "cb_get_profile": (st, [vp, C.POINTER(Profile)]),
        "cb_get_layer_profile": (st, [vp, C.c_int, C.POINTER(C.c_float), C.POINTER(C.c_float)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(s) -> C.c_void_p:
    if s is None:
        s = torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream if hasattr(s, "cuda_stream") else int(s))


def _check(st: int, ctx=None):
    if st != 0:
        lib = load_library()
        msg = lib.cb_last_error(ctx).decode() if lib else ""
        raise CacheBlendError(st, msg)


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.bfloat16:
        return CB_BF16
    if t == torch.float32:
        return CB_F32
    raise CacheBlendError(3, f"unsupported dtype {t}")


# ----------------------------------------------------------------------------- host logic
def k_for_ratio(r: float, n_cached: int) -> int:
    """Cached tokens kept at a check layer (cb_k_for_ratio)."""
    return int(load_library().cb_k_for_ratio(float(r), int(n_cached)))


def ratio_schedule(n_layers: int, r: float, schedule: str = "gradual", r1: Optional[float] = None,
                   n_narrow: int = 3) -> List[float]:
    """Per-layer ratios of gradual filtering (cb_ratio_schedule)."""
    sched = {"fixed": 0, "gradual": 1}.get(schedule)
    if sched is None:
        raise ValueError(schedule)
    out = (C.c_double * max(1, n_layers))()
    _check(load_library().cb_ratio_schedule(int(n_layers), float(r), sched, -1.0 if r1 is None else float(r1),
                                            int(n_narrow), out))
    return [float(out[i]) for i in range(n_layers)]


# ----------------------------------------------------------------------------- standalone kernels
def cb_rope_rerotate(k_src: torch.Tensor, k_dst: torch.Tensor, v_src: Optional[torch.Tensor],
                     v_dst: Optional[torch.Tensor], delta_pos: int, theta: float, stream=None) -> None:
    lib = load_library()
    n, hkv, dh = k_src.shape
    _check(lib.cb_rope_rerotate(_ptr(k_src), _ptr(k_dst), _ptr(v_src), _ptr(v_dst), n, hkv, dh, int(delta_pos),
                                float(theta), _dtype_code(k_src.dtype), _stream(stream)))


def cb_kv_deviation(k_new: torch.Tensor, v_new: torch.Tensor, k_fus: torch.Tensor, v_fus: torch.Tensor,
                    idx: Optional[torch.Tensor], mode: int = 0, out: Optional[torch.Tensor] = None,
                    stream=None) -> torch.Tensor:
    lib = load_library()
    n = k_new.shape[0]
    width = k_new[0].numel() if n else k_fus[0].numel()
    out = torch.empty(n, dtype=torch.float32, device=k_new.device) if out is None else out
    _check(lib.cb_kv_deviation(_ptr(k_new), _ptr(v_new), _ptr(k_fus), _ptr(v_fus), _ptr(idx), n, width, mode,
                               _dtype_code(k_fus.dtype), _ptr(out), _stream(stream)))
    return out


def cb_select_hkvd(dev: torch.Tensor, cand: Optional[torch.Tensor], k: int, out: Optional[torch.Tensor] = None,
                   status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    lib = load_library()
    out = torch.empty(k, dtype=torch.int32, device=dev.device) if out is None else out
    _check(lib.cb_select_hkvd(_ptr(dev), _ptr(cand), dev.numel(), int(k), _ptr(out), _ptr(status), _stream(stream)))
    return out


_GEMM_SCRATCH = {}


def gemm_scratch(device=None) -> torch.Tensor:
    """A zero-filled scratch buffer for cb_gemm on ``device`` (one per device, reused)."""
    device = torch.device("cuda") if device is None else torch.device(device)
    key = device.index if device.index is not None else torch.cuda.current_device()
    if key not in _GEMM_SCRATCH:
        n = load_library().cb_gemm_scratch_size()
        _GEMM_SCRATCH[key] = torch.zeros(n, dtype=torch.uint8, device=torch.device("cuda", key))
    return _GEMM_SCRATCH[key]


def cb_gemm(A: torch.Tensor, B: torch.Tensor, C_out: torch.Tensor, epilogue: int = 0,
            B2: Optional[torch.Tensor] = None, scratch: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """C = A . B^T (epilogue 0), C += A . B^T (1), C = SiLU(A B^T) * (A B2^T) (2).
    ``scratch`` (see gemm_scratch) enables the stream-K schedule; None = whole tiles only."""
    lib = load_library()
    M, K = A.shape
    N = B.shape[0] * (2 if epilogue == 2 else 1)
    _check(lib.cb_gemm(_ptr(A), _ptr(B), _ptr(B2), _ptr(C_out), M, N, K, C_out.shape[1], epilogue,
                       _dtype_code(A.dtype), _ptr(scratch), 0 if scratch is None else scratch.numel(),
                       _stream(stream)))
    return C_out


def cb_gemm_set_orientation(orientation: int) -> None:
    """Process-wide tile orientation of the bf16 GEMMs: 0 by the library's time model,
    1 tokens as tile rows, 2 output features as tile rows (tuning and tests)."""
    _check(load_library().cb_gemm_set_orientation(int(orientation)))


def cb_gemm_set_pairing(pairing: int) -> None:
    """Process-wide CTA pairs for the bf16 GEMMs: 0 by the library's time model, 1 never,
    2 clusters of one pair, 4 clusters of two pairs (tuning and tests)."""
    _check(load_library().cb_gemm_set_pairing(int(pairing)))


def cb_gemm_describe(M: int, N: int, K: int, epilogue: int, scratch_bytes: int = 0) -> str:
    """The schedule a bf16 cb_gemm of this shape would run under the current hooks."""
    buf = C.create_string_buffer(256)
    _check(load_library().cb_gemm_describe(int(M), int(N), int(K), int(epilogue), int(scratch_bytes), buf, 256))
    return buf.value.decode()


def cb_set_qkv_fusion(enabled: bool) -> None:
    """Process-wide: Q/K/V projection with RoPE and the K/V scatter in one launch in the
    layers without a check (default), or the projection and the post-QKV kernel (tests)."""
    _check(load_library().cb_set_qkv_fusion(1 if enabled else 0))


def cb_attention_set_tiles(tiles: int) -> None:
    """Process-wide query tiles per CTA of the bf16 attention: 0 by the launch's size,
    1 or 2 forced (tuning and tests)."""
    _check(load_library().cb_attention_set_tiles(int(tiles)))


def cb_set_launch_overlap(enabled: bool) -> None:
    """Programmatic dependent launch of the blended-prefill kernels (process-wide, default on)."""
    _check(load_library().cb_set_launch_overlap(1 if enabled else 0))


def cb_gemm_noalloc(A: torch.Tensor, B: torch.Tensor, C_out: torch.Tensor, epilogue: int = 0,
                    B2: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """cb_gemm without scratch arguments: for callers that cannot allocate device memory
    (the library's built-in device array serves as stream-K scratch)."""
    lib = load_library()
    M, K = A.shape
    N = B.shape[0] * (2 if epilogue == 2 else 1)
    st = lib.cb_gemm_noalloc(_ptr(A), _ptr(B), _ptr(B2), _ptr(C_out), M, N, K, C_out.shape[1], epilogue,
                             _dtype_code(A.dtype), _stream(stream))
    if st != 0:
        raise CacheBlendError(st, lib.cb_gemm_noalloc_error().decode())
    return C_out


def cb_gemm_get_status(stream=None, timeout_ms: int = 10000) -> None:
    """Waits for ``stream`` and reads (and clears) the status word of the standalone GEMM
    calls on the current device; raises when a device-side wait gave up."""
    lib = load_library()
    st = lib.cb_gemm_get_status(_stream(stream), int(timeout_ms))
    if st != 0:
        raise CacheBlendError(st, lib.cb_gemm_noalloc_error().decode())


def cb_attention(q: torch.Tensor, q_pos: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                 out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    lib = load_library()
    m, H, dh = q.shape
    n_kv, hkv, _ = k.shape
    out = torch.empty_like(q) if out is None else out
    _check(lib.cb_attention(_ptr(q), _ptr(q_pos), m, _ptr(k), _ptr(v), n_kv, H, hkv, dh, _ptr(out),
                            _dtype_code(q.dtype), _stream(stream)))
    return out


def cb_chunk_hash(ids) -> int:
    """Content key of a chunk: FNV-1a 64 of its token ids (host sequence or tensor)."""
    if isinstance(ids, torch.Tensor):
        ids = ids.detach().to("cpu", torch.int32).tolist()
    arr = (C.c_int32 * max(1, len(ids)))(*[int(x) for x in ids])
    return int(load_library().cb_chunk_hash(arr, len(ids)))


def cb_plan_loading(model: Dict[str, float], chunks: Sequence[Dict[str, float]], n_query: int):
    """(actions, ratio, T_load, T_recompute) of one prompt; see cb_plan_loading in the header."""
    lib = load_library()
    m = CostModel(model["link_bytes_per_s"], model["link_latency_s"], model["prefill_s_per_token"],
                  model["recompute_fixed_s"], model["r_min"], model["r_max"])
    n = len(chunks)
    arr = (ChunkInfo * max(1, n))(*[ChunkInfo(int(c["n_tokens"]), int(c["tier"]), float(c["bytes"])) for c in chunks])
    acts = (C.c_int32 * max(1, n))()
    r, tl, tr = C.c_double(), C.c_double(), C.c_double()
    _check(lib.cb_plan_loading(C.byref(m), arr, n, int(n_query), acts, C.byref(r), C.byref(tl), C.byref(tr)))
    return [int(acts[i]) for i in range(n)], r.value, tl.value, tr.value


def cb_codec_layer_bytes(n_tok: int, n_kv_heads: int, head_dim: int, bits: int) -> int:
    return int(load_library().cb_codec_layer_bytes(n_tok, n_kv_heads, head_dim, bits))


def cb_kv_encode(k: torch.Tensor, v: torch.Tensor, bits: int, blob: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """Quantised chunk (uint8 blob) of k, v [L, n, Hkv, dh]: keys per channel, values per token."""
    lib = load_library()
    L, n, hkv, dh = k.shape
    nbytes = L * cb_codec_layer_bytes(n, hkv, dh, bits)
    blob = torch.empty(nbytes, dtype=torch.uint8, device=k.device) if blob is None else blob
    _check(lib.cb_kv_encode(_ptr(k), _ptr(v), L, n, hkv, dh, _dtype_code(k.dtype), int(bits), _ptr(blob),
                            _stream(stream)))
    return blob


def cb_kv_decode(blob: torch.Tensor, shape, bits: int, delta_pos: int, theta: float, dtype: torch.dtype,
                 stream=None):
    """Dequantised k, v [L, n, Hkv, dh] of a blob, keys re-rotated by ``delta_pos`` positions."""
    lib = load_library()
    L, n, hkv, dh = shape
    k = torch.empty(shape, dtype=dtype, device=blob.device)
    v = torch.empty_like(k)
    _check(lib.cb_kv_decode(_ptr(blob), L, n, hkv, dh, int(bits), int(delta_pos), float(theta), _dtype_code(dtype),
                            _ptr(k), _ptr(v), _stream(stream)))
    return k, v


# ----------------------------------------------------------------------------- model / engine
class Engine:
    """A cb_ctx bound to one model's device weights and a workspace.

    ``weights``: {"embed": [V, d], "lm_head": [V, d], "layers": [ {"wq", "wk", "wv", "wo",
    "wgate", "wup", "wdown"} ... ]} of device tensors in the model dtype (row-major
    [out, in]).  The engine keeps references so the tensors outlive the context.
    """

    def __init__(self, cfg, weights: Dict, max_tokens: int, max_requests: int = 1, max_positions: Optional[int] = None,
                 device="cuda"):
        self.lib = load_library()
        self.cfg = cfg
        self.dtype = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
        self.device = torch.device(device)
        self.weights = weights
        L = cfg.n_layers
        mc = ModelCfg(L, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn_dim, cfg.vocab,
                      float(cfg.rope_theta), float(cfg.rms_eps), CB_BF16 if cfg.dtype == "bf16" else CB_F32,
                      int(max_positions or max_tokens + 1))
        arrs = {}
        for name in ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown"):
            a = (C.c_void_p * L)(*[weights["layers"][i][name].data_ptr() for i in range(L)])
            arrs[name] = a
        self._arrs = arrs
        w = Weights(weights["embed"].data_ptr(), weights["lm_head"].data_ptr(),
                    *[C.cast(arrs[n], C.POINTER(C.c_void_p)) for n in ("wq", "wk", "wv", "wo", "wgate", "wup", "wdown")])
        ctx = C.c_void_p()
        _check(self.lib.cb_create(C.byref(mc), C.byref(w), C.byref(ctx)))
        self.ctx = ctx
        self.max_tokens, self.max_requests = max_tokens, max_requests
        nbytes = self.lib.cb_workspace_size(ctx, max_tokens, max_requests)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        _check(self.lib.cb_set_workspace(ctx, _ptr(self.workspace), nbytes, max_tokens, max_requests), ctx)
        self._chunks = {}
        self._keep = []

    def close(self):
        if getattr(self, "ctx", None):
            self.lib.cb_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- chunk cache
    def kv_shape(self, n: int):
        return (self.cfg.n_layers, n, self.cfg.n_kv_heads, self.cfg.head_dim)

    def precompute_chunk(self, ids: torch.Tensor, stream=None):
        n = ids.numel()
        k = torch.empty(self.kv_shape(n), dtype=self.dtype, device=self.device)
        v = torch.empty_like(k)
        _check(self.lib.cb_precompute_chunk(self.ctx, _ptr(ids), n, _ptr(k), _ptr(v), _stream(stream)), self.ctx)
        return k, v

    def register_chunk(self, chunk_id: int, ids: torch.Tensor, k: torch.Tensor, v: torch.Tensor, on_host: bool = False):
        _check(self.lib.cb_register_chunk(self.ctx, C.c_uint64(chunk_id), _ptr(ids), _ptr(k), _ptr(v), ids.numel(),
                                          int(on_host)), self.ctx)
        self._chunks[chunk_id] = (ids, k, v)

    def register_chunk_codec(self, chunk_id: int, ids: torch.Tensor, blob: torch.Tensor, bits: int,
                             on_host: bool = False):
        """Registers a quantised chunk (a blob from cb_kv_encode; pinned host memory if on_host)."""
        _check(self.lib.cb_register_chunk_codec(self.ctx, C.c_uint64(chunk_id), _ptr(ids), _ptr(blob), ids.numel(),
                                                int(bits), int(on_host)), self.ctx)
        self._chunks[chunk_id] = (ids, blob, None)

    def set_staging(self, nbytes: int):
        """Allocates (caller side) and binds the staging ring for host-resident quantised chunks."""
        self.staging = torch.empty(max(1, nbytes), dtype=torch.uint8, device=self.device) if nbytes else None
        _check(self.lib.cb_set_staging(self.ctx, _ptr(self.staging), nbytes if nbytes else 0), self.ctx)

    def chunk_info(self, chunk_id: int) -> Dict[str, float]:
        """Tier, tokens and load bytes of a registered chunk (tier -1 when missing)."""
        info = ChunkInfo()
        _check(self.lib.cb_chunk_info_of(self.ctx, C.c_uint64(chunk_id), C.byref(info)), self.ctx)
        return {"n_tokens": info.n_tokens, "tier": info.tier, "bytes": info.bytes}

    def unregister_chunk(self, chunk_id: int):
        _check(self.lib.cb_unregister_chunk(self.ctx, C.c_uint64(chunk_id)), self.ctx)
        self._chunks.pop(chunk_id, None)

    # -- requests
    def make_request(self, chunk_ids: Sequence[int], query_ids: torch.Tensor, want_hidden=True, want_sel=True,
                     decode_room: int = 0):
        """Buffers of one blend request; ``decode_room`` extra cache rows per layer leave room to
        decode that many tokens after the blend (cb_decode_step)."""
        n = sum(self._chunks[c][0].numel() for c in chunk_ids) + query_ids.numel()
        L, d = self.cfg.n_layers, self.cfg.d_model
        r = {
            "chunk_ids": list(chunk_ids), "query_ids": query_ids, "n_tokens": n, "kv_capacity": n + int(decode_room),
            "fused_k": torch.empty(self.kv_shape(n + int(decode_room)), dtype=self.dtype, device=self.device),
            "first_token": torch.full((1,), -1, dtype=torch.int32, device=self.device),
        }
        r["fused_v"] = torch.empty_like(r["fused_k"])
        r["hidden"] = torch.zeros((n, d), dtype=torch.float32, device=self.device) if want_hidden else None
        r["sel"] = torch.full((L, n), -1, dtype=torch.int32, device=self.device) if want_sel else None
        r["sel_count"] = torch.zeros(L, dtype=torch.int32, device=self.device) if want_sel else None
        return r

    def _c_requests(self, reqs):
        arr = (Request * len(reqs))()
        keep = []
        for i, r in enumerate(reqs):
            ids = (C.c_uint64 * max(1, len(r["chunk_ids"])))(*r["chunk_ids"])
            keep.append(ids)
            arr[i] = Request(len(r["chunk_ids"]), C.cast(ids, C.POINTER(C.c_uint64)), r["query_ids"].data_ptr(),
                             r["query_ids"].numel(), r["fused_k"].data_ptr(), r["fused_v"].data_ptr(),
                             None if r["hidden"] is None else r["hidden"].data_ptr(),
                             None if r["sel"] is None else r["sel"].data_ptr(),
                             None if r["sel_count"] is None else r["sel_count"].data_ptr(),
                             r["first_token"].data_ptr(), int(r.get("kv_capacity", 0)))
        return arr, keep

    def _c_params(self, ratios, dev_mode=0, forced=None, seam_tokens=None):
        """``seam_tokens`` (an int) selects spatial seam repair instead of the ratio schedule."""
        L = self.cfg.n_layers
        rat = (C.c_double * L)(*[float(x) for x in (ratios if ratios is not None else [-1.0] * L)])
        keep = [rat]
        fptr = None
        if forced is not None:
            # forced: {layer: [list per request of sorted cached token indices]}
            tbl = (C.POINTER(C.c_int32) * L)()
            for layer, per_req in forced.items():
                flat = []
                for lst in per_req:
                    flat.append(len(lst))
                    flat.extend(int(x) for x in lst)
                a = (C.c_int32 * len(flat))(*flat)
                keep.append(a)
                tbl[layer] = C.cast(a, C.POINTER(C.c_int32))
            keep.append(tbl)
            fptr = C.cast(tbl, C.POINTER(C.POINTER(C.c_int32)))
        seam = seam_tokens is not None
        return BlendParams(L, C.cast(rat, C.POINTER(C.c_double)), dev_mode, fptr,
                           CB_SELECT_SEAM if seam else CB_SELECT_HKVD, int(seam_tokens) if seam else 0), keep

    def blend_prefill(self, reqs, ratios, dev_mode=0, forced=None, stream=None, copy_stream=None, seam_tokens=None):
        arr, k1 = self._c_requests(reqs)
        params, k2 = self._c_params(ratios, dev_mode, forced, seam_tokens)
        _check(self.lib.cb_blend_prefill(self.ctx, arr, len(reqs), C.byref(params), _stream(stream),
                                         None if copy_stream is None else _stream(copy_stream)), self.ctx)
        return reqs

    def blend_begin(self, reqs, ratios, dev_mode=0, forced=None, stream=None, seam_tokens=None):
        arr, k1 = self._c_requests(reqs)
        params, k2 = self._c_params(ratios, dev_mode, forced, seam_tokens)
        _check(self.lib.cb_blend_begin(self.ctx, arr, len(reqs), C.byref(params), _stream(stream)), self.ctx)

    def fetch_kv(self, layer: int, copy_stream=None):
        _check(self.lib.cb_fetch_kv(self.ctx, layer, _stream(copy_stream)), self.ctx)

    def synchronize(self, layer: int, timeout_ms: int = 10000):
        _check(self.lib.cb_synchronize(self.ctx, layer, timeout_ms), self.ctx)

    def prefill_layer(self, layer: int, stream=None):
        _check(self.lib.cb_prefill_layer(self.ctx, layer, _stream(stream)), self.ctx)

    def blend_layer(self, layer: int, stream=None):
        _check(self.lib.cb_blend_layer(self.ctx, layer, _stream(stream)), self.ctx)

    def blend_finish(self, stream=None):
        _check(self.lib.cb_blend_finish(self.ctx, _stream(stream)), self.ctx)

    def full_prefill(self, ids: torch.Tensor, want_kv=False, want_hidden=True, stream=None):
        n = ids.numel()
        out = {"first_token": torch.full((1,), -1, dtype=torch.int32, device=self.device)}
        out["hidden"] = torch.zeros((n, self.cfg.d_model), dtype=torch.float32, device=self.device) if want_hidden else None
        if want_kv:
            out["k"] = torch.empty(self.kv_shape(n), dtype=self.dtype, device=self.device)
            out["v"] = torch.empty_like(out["k"])
        _check(self.lib.cb_full_prefill(self.ctx, _ptr(ids), n, _ptr(out.get("k")), _ptr(out.get("v")),
                                        _ptr(out["hidden"]), _ptr(out["first_token"]), _stream(stream)), self.ctx)
        return out

    def decode_step(self, reqs, tokens: torch.Tensor, out_tokens: Optional[torch.Tensor] = None, n_past=None,
                    out_hidden=None, stream=None) -> torch.Tensor:
        """One greedy decode step of the blended requests ``reqs`` (made with decode_room):
        tokens [n] enter at positions n_past[i] (default: each request's prompt length plus the
        steps it already decoded); returns the next tokens [n]."""
        n = len(reqs)
        out_tokens = torch.empty(n, dtype=torch.int32, device=self.device) if out_tokens is None else out_tokens
        arr = (DecodeSeq * n)()
        for i, r in enumerate(reqs):
            past = r["n_tokens"] + r.setdefault("decoded", 0) if n_past is None else int(n_past[i])
            arr[i] = DecodeSeq(r["fused_k"].data_ptr(), r["fused_v"].data_ptr(), int(r["kv_capacity"]), past,
                               None if out_hidden is None else out_hidden[i].data_ptr())
        _check(self.lib.cb_decode_step(self.ctx, arr, n, _ptr(tokens), _ptr(out_tokens), _stream(stream)), self.ctx)
        if n_past is None:
            for r in reqs:
                r["decoded"] += 1
        return out_tokens

    def get_status(self, stream=None, timeout_ms: int = 60000):
        _check(self.lib.cb_get_status(self.ctx, _stream(stream), timeout_ms), self.ctx)

    def set_profiling(self, enable):
        """0 / False off, 1 / True per-phase events, 2 per-layer events, 3 both."""
        _check(self.lib.cb_set_profiling(self.ctx, int(enable)), self.ctx)

    def get_layer_profile(self) -> Dict[str, List[float]]:
        """Per-layer staging (copy stream) and compute (compute stream) ms since the last call."""
        L = self.cfg.n_layers
        load, comp = (C.c_float * L)(), (C.c_float * L)()
        _check(self.lib.cb_get_layer_profile(self.ctx, L, load, comp), self.ctx)
        return {"load_ms": list(load), "compute_ms": list(comp)}

    def get_profile(self) -> Dict[str, Dict[str, float]]:
        """Per-phase device ms, launches and timed calls since the last call (waits for the events)."""
        p = Profile()
        _check(self.lib.cb_get_profile(self.ctx, C.byref(p)), self.ctx)
        return {name: {"ms": p.ms[i], "launches": p.launches[i], "calls": p.calls[i]} for i, name in enumerate(PHASES)}

    def plan_counts(self, request: int = 0) -> List[int]:
        a = (C.c_int32 * self.cfg.n_layers)()
        _check(self.lib.cb_plan_counts(self.ctx, request, a), self.ctx)
        return list(a)
