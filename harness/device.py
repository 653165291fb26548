"""Device-side copies of the harness inputs (same bits as harness/inputs.py).

Weights are generated directly in GPU memory by ``harness/libsynth.so`` (the generator
of inputs.py written in CUDA), so a 7B-140B parameter model needs no host round trip.
Token ids are small and are generated on the host and copied.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np
import torch

from . import inputs as hz

_LIB = None
_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(_PATH):
            raise RuntimeError(f"{_PATH} is missing: run `python -m rag_non_prefix_gb300.build`")
        _LIB = C.CDLL(_PATH)
        _LIB.synth_weights.restype = C.c_int
        _LIB.synth_weights.argtypes = [C.c_uint64, C.c_uint64, C.c_uint64, C.c_float, C.c_int, C.c_void_p, C.c_void_p]
    return _LIB


def synth_into(out: torch.Tensor, key: int, start: int = 0, std: float = hz.WEIGHT_STD) -> torch.Tensor:
    """Fills a contiguous fp32 or bf16 device tensor with elements [start, start + numel) of stream ``key``."""
    assert out.is_cuda and out.is_contiguous()
    as_bf16 = out.dtype == torch.bfloat16
    assert as_bf16 or out.dtype == torch.float32
    st = _lib().synth_weights(C.c_uint64(key & 0xFFFFFFFFFFFFFFFF), start, out.numel(), float(hz.weight_scale(std)),
                              int(as_bf16), out.data_ptr(), C.c_void_p(torch.cuda.current_stream().cuda_stream))
    if st != 0:
        raise RuntimeError(f"synth_weights failed with CUDA error {st}")
    return out


def torch_dtype(cfg: hz.ModelConfig):
    return torch.bfloat16 if cfg.dtype == "bf16" else torch.float32


def device_weights(cfg: hz.ModelConfig, seed: int, device="cuda", layers=None):
    """All weights of a model, generated on the device, as the binding's weight dict."""
    dt = torch_dtype(cfg)
    L = cfg.n_layers if layers is None else layers

    def mat(layer, m, shape):
        t = torch.empty(shape, dtype=dt, device=device)
        return synth_into(t, hz.layer_weight_key(seed, layer, m))

    out = {
        "embed": mat(hz.GLOBAL_EMBED_LAYER, 0, (cfg.vocab, cfg.d_model)),
        "lm_head": mat(hz.GLOBAL_LM_LAYER, 0, (cfg.vocab, cfg.d_model)),
        "layers": [],
    }
    for i in range(L):
        out["layers"].append({name: mat(i, m, cfg.mat_shape(m)) for m, name in enumerate(hz.LAYER_MATS)})
    return out


def ids_tensor(ids: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(device)
