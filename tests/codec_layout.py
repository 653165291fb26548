"""Reader of the quantised-chunk byte layout that include/cacheblend.h documents (at
cb_codec_layer_bytes), written from that description for the tests: it lets them compare the
library's blobs with the oracle's codes without calling back into the library."""
from __future__ import annotations

import numpy as np


def _r16(x: int) -> int:
    return (x + 15) // 16 * 16


def layer_layout(n: int, hkv: int, dh: int, bits: int):
    """Byte offsets of the six regions of one layer block and the block size."""
    rows = n * hkv
    codes = _r16(rows * dh * bits // 8)
    chan = _r16(hkv * dh * 4)
    per_row = _r16(rows * 4)
    off = {"k_codes": 0, "v_codes": codes, "k_scale": 2 * codes}
    off["k_zero"] = off["k_scale"] + chan
    off["v_scale"] = off["k_zero"] + chan
    off["v_zero"] = off["v_scale"] + per_row
    size = (off["v_zero"] + per_row + 255) // 256 * 256
    return off, size


def _unpack(b: np.ndarray, count: int, bits: int) -> np.ndarray:
    if bits == 8:
        return b[:count].astype(np.int64)
    lo = (b & 15).astype(np.int64)
    hi = (b >> 4).astype(np.int64)
    return np.stack([lo, hi], axis=-1).reshape(-1)[:count]


def parse_blob(blob: np.ndarray, L: int, n: int, hkv: int, dh: int, bits: int):
    """Codes, scales and minima of a blob, shaped like oracle.kv_encode's output."""
    off, size = layer_layout(n, hkv, dh, bits)
    assert blob.size == L * size, (blob.size, L * size)
    out = {k: [] for k in ("k_codes", "v_codes", "k_scale", "k_zero", "v_scale", "v_zero")}
    nb = n * hkv * dh * bits // 8
    for layer in range(L):
        blk = blob[layer * size:(layer + 1) * size]
        for name in ("k_codes", "v_codes"):
            out[name].append(_unpack(blk[off[name]:off[name] + nb], n * hkv * dh, bits).reshape(n, hkv, dh))
        for name, cnt, shape in (("k_scale", hkv * dh, (hkv, dh)), ("k_zero", hkv * dh, (hkv, dh)),
                                 ("v_scale", n * hkv, (n, hkv)), ("v_zero", n * hkv, (n, hkv))):
            out[name].append(blk[off[name]:off[name] + 4 * cnt].view(np.float32).reshape(shape))
    return {k: np.stack(v) for k, v in out.items()}
