"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin catches each one.

A pin that still passes with a wrong sign, a dropped term or an off-by-one is no pin.
"""
import numpy as np
import pytest

import oracle.cacheblend as ocb
from tests import test_oracle_pins as pins


def _rope_wrong_sign(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    n, _, dh = x.shape
    half = dh // 2
    pos = np.broadcast_to(np.asarray(pos, dtype=np.float64), (n,))
    ang = pos[:, None] * ocb.rope_inv_freq(dh, theta)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


def _rope_adjacent_pairs(x, pos, theta):
    x = np.asarray(x, dtype=np.float64)
    n, _, dh = x.shape
    pos = np.broadcast_to(np.asarray(pos, dtype=np.float64), (n,))
    ang = pos[:, None] * ocb.rope_inv_freq(dh, theta)[None, :]
    c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


_orig_attention = ocb.causal_attention


def _attention_off_by_one(q, q_pos, k, v):
    # excludes the diagonal key except at position 0
    return _orig_attention(q, [max(0, int(p) - 1) for p in q_pos], k, v)


_orig_dev = ocb.kv_deviation


def _deviation_k_only(k_new, v_new, k_fused, v_fused, mode=0):
    return _orig_dev(k_new, v_new, k_fused, v_fused, 1)


def _select_ties_high_index(dev32, cand, k):
    dev32 = np.asarray(dev32, np.float32)
    cand = np.asarray(cand, np.int64)
    if k <= 0:
        return np.zeros(0, np.int64)
    order = np.lexsort((-cand, -dev32.astype(np.float64)))
    return np.sort(cand[order[:k]])


def _mlp_no_residual(cfg, W, h, attn):
    n = h.shape[0]
    h = h + attn.reshape(n, cfg.q_width) @ W["wo"].astype(np.float64).T
    x = ocb.rms_norm(h, cfg.rms_eps)
    return (ocb.silu(x @ W["wgate"].T) * (x @ W["wup"].T)) @ W["wdown"].T


def _cosine_k_only(k_new, v_new, k_fused, v_fused, mode=0):
    if mode != 3:
        return _orig_dev(k_new, v_new, k_fused, v_fused, mode)
    z = np.zeros_like(np.asarray(v_new, np.float64))
    return _orig_dev(k_new, z, k_fused, z, 3)


def _seam_after_boundary(segments, seam_tokens):
    # the first R tokens after each chunk start instead of the last R before its end
    out, off = [], 0
    for seg in segments:
        n = len(seg.ids)
        if seg.chunk >= 0:
            out.extend(range(off, off + min(int(seam_tokens), n)))
        off += n
    return np.array(sorted(out), dtype=np.int64)


_orig_minmax = ocb._minmax_codes


def _codec_keys_per_token(x32, axis, bits):
    # groups along the other axis: keys per token instead of per channel
    return _orig_minmax(x32, 3 if axis == 1 else axis, bits)


def _codec_round_down(x32, axis, bits):
    codes, scale, mn = _orig_minmax(x32, axis, bits)
    q = np.zeros_like(x32)
    d = x32 - mn
    np.divide(d, np.broadcast_to(scale, d.shape), out=q, where=np.broadcast_to(scale > 0, d.shape))
    return np.clip(np.floor(q), 0, 2 ** bits - 1).astype(np.int64), scale, mn


def _fnv1_order(data):
    # FNV-1 (multiply, then xor) instead of FNV-1a
    h = ocb.FNV64_OFFSET
    for b in data:
        h = (h * ocb.FNV64_PRIME) & 0xFFFFFFFFFFFFFFFF
        h ^= b
    return h


_orig_plan = ocb.plan_loading


def _ratio_inverted(model, chunks, n_query):
    acts, r, t_load, t_rec = _orig_plan(model, chunks, n_query)
    r2 = model["r_max"] + model["r_min"] - r  # lower r on slow storage
    return acts, r2, t_load, model["recompute_fixed_s"] + r2 * (t_rec - model["recompute_fixed_s"]) / max(r, 1e-30)


_orig_decode = ocb.decode_step


def _decode_position_off_by_one(cfg, weights, Kf, Vf, n_past, token, storage="f64"):
    # RoPE and the causal bound at n_past + 1 while the K/V row still goes to n_past
    h = weights.embed(np.asarray([token])).astype(np.float64)
    for i in range(cfg.n_layers):
        W = weights.layer(i)
        q, k, v = ocb.project_qkv(cfg, W, h, [n_past + 1])
        Kf[i][n_past] = ocb.round_storage(k[0], storage)
        Vf[i][n_past] = ocb.round_storage(v[0], storage)
        h = ocb.output_and_mlp(cfg, W, h, ocb.causal_attention(q, [n_past], Kf[i], Vf[i]))
    return {"hidden": h[0], "token": ocb.first_token(cfg, weights, h[0])}


def _rms_no_eps_mean(x, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


MUTATIONS = [
    ("rerotate_keys", lambda k, d, t: np.asarray(k, np.float64), [pins.test_layer0_fresh_kv_equals_rerotated_cache]),
    ("rope_rotate", _rope_wrong_sign, [pins.test_rope_matches_complex_exponential]),
    ("rope_rotate", _rope_adjacent_pairs, [pins.test_rope_matches_complex_exponential]),
    ("causal_attention", _attention_off_by_one, [pins.test_attention_matches_torch_sdpa_with_sparse_queries]),
    ("kv_deviation", _deviation_k_only, [pins.test_deviation_closed_forms]),
    ("select_hkvd", _select_ties_high_index, [pins.test_select_exhaustive_small_with_ties]),
    ("output_and_mlp", _mlp_no_residual, [lambda: pins.test_full_prefill_matches_torch_library_decoder(pins.TINY)]),
    ("rms_norm", _rms_no_eps_mean, [pins.test_rms_norm_properties]),
    ("kv_deviation", _cosine_k_only, [pins.test_cosine_deviation_closed_forms]),
    ("seam_positions", _seam_after_boundary, [pins.test_seam_positions_hand_examples]),
    ("_minmax_codes", _codec_keys_per_token, [pins.test_codec_hand_example_fixes_the_axes]),
    ("_minmax_codes", _codec_round_down, [lambda: pins.test_codec_error_bound_and_extremes(8)]),
    ("fnv1a64", _fnv1_order, [pins.test_fnv1a64_published_vectors_and_chunk_key]),
    ("plan_loading", _ratio_inverted, [pins.test_ratio_rule_hides_recompute_under_the_load]),
    ("decode_step", _decode_position_off_by_one, [pins.test_decode_after_prefill_equals_a_longer_prefill]),
]


@pytest.mark.parametrize("name,fn,tests", MUTATIONS, ids=[f"{m[0]}-{i}" for i, m in enumerate(MUTATIONS)])
def test_planted_mistake_is_caught(monkeypatch, name, fn, tests):
    monkeypatch.setattr(ocb, name, fn)
    failed = 0
    for t in tests:
        try:
            t()
        except (AssertionError, FloatingPointError, ValueError):
            failed += 1
    assert failed == len(tests), f"mutation of {name} was not caught"

