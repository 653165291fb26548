"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU).

Each test ties an oracle function to something other than itself: a closed form,
an invariant, a special case that reduces to a library routine (torch SDPA,
complex exponentials, torch's bfloat16 conversion), brute force on tiny inputs,
or a number printed on the pages (tests/golden/kv_bytes.json).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import harness as hz
import oracle.cacheblend as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

TINY = hz.ModelConfig("pin_tiny", 3, 64, 4, 2, 16, 128, 100, 1e4, 1e-5, "f32")
TINY_MHA = hz.ModelConfig("pin_mha", 2, 48, 3, 3, 16, 96, 80, 500.0, 1e-5, "f32")


def _rng(seed=0):
    return np.random.default_rng(seed)


def _prompt(cfg, seed, lens, qlen, prefix=0):
    """A small prompt built with the harness generators for a custom model."""
    segs, chunks = [], []
    allens = ([prefix] if prefix else []) + list(lens)
    for i, n in enumerate(allens):
        ids = hz.gen_token_ids(hz.stream_key(seed, 100 + i), n, cfg.vocab, "uniform")
        chunks.append(ids)
        segs.append(hz.Segment(ids, i))
    segs.append(hz.Segment(hz.gen_token_ids(hz.stream_key(seed, 999), qlen, cfg.vocab, "uniform"), -1))
    return segs, chunks


def _caches(cfg, W, chunks, storage):
    return {i: orc.precompute_chunk(cfg, W, c, storage) for i, c in enumerate(chunks)}


def _concat(segs):
    return np.concatenate([s.ids for s in segs])


# ----------------------------------------------------------------------------- RoPE
def test_inv_freq_closed_form():
    f = orc.rope_inv_freq(128, 1e4)
    assert f[0] == 1.0
    assert np.allclose(f[1:] / f[:-1], 1e4 ** (-2.0 / 128), rtol=1e-14)
    assert math.isclose(f[-1], 1e4 ** (-126.0 / 128), rel_tol=1e-14)


def test_rope_group_property_and_identity():
    """R(a) R(b) = R(a + b) and R(0) = I (baseline property c, fp64 within 1e-6)."""
    x = _rng(1).standard_normal((7, 3, 64))
    for a, b in [(3, 5), (511, 2048), (0, 8191), (4096, 4096)]:
        lhs = orc.rope_rotate(orc.rope_rotate(x, a, 1e4), b, 1e4)
        rhs = orc.rope_rotate(x, a + b, 1e4)
        assert np.max(np.abs(lhs - rhs)) < 1e-6
    assert np.array_equal(orc.rope_rotate(x, 0, 1e4), x)
    assert np.array_equal(orc.rerotate_keys(x, 0, 5e6), x)


def test_rerotation_equals_encoding_at_shifted_position():
    """Re-rotating a key cached at p by delta equals encoding it at p + delta (property c)."""
    k = _rng(2).standard_normal((50, 4, 128))
    p = np.arange(50) * 7
    for delta in [1, 64, 3136, 8191]:
        cached = orc.rope_rotate(k, p, 1e4)
        assert np.max(np.abs(orc.rerotate_keys(cached, delta, 1e4) - orc.rope_rotate(k, p + delta, 1e4))) < 1e-6


def test_rope_matches_complex_exponential():
    """Pairs (x_i, x_{i+dh/2}) as complex numbers multiplied by exp(i * p * theta^(-2i/dh))."""
    x = _rng(3).standard_normal((9, 2, 32))
    pos = np.array([0, 1, 2, 5, 17, 100, 1000, 4095, 9000])
    half = 16
    z = x[..., :half] + 1j * x[..., half:]
    freq = 1e4 ** (-np.arange(half) * 2.0 / 32)
    z = z * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    ref = np.concatenate([z.real, z.imag], axis=-1)
    assert np.max(np.abs(orc.rope_rotate(x, pos, 1e4) - ref)) < 1e-12


def test_rope_relative_position_and_norm():
    q = _rng(4).standard_normal((1, 1, 64))
    k = _rng(5).standard_normal((1, 1, 64))
    dots = [float(np.sum(orc.rope_rotate(q, p + 9, 1e4) * orc.rope_rotate(k, p, 1e4))) for p in (0, 13, 700)]
    assert np.allclose(dots, dots[0], rtol=1e-10)
    r = orc.rope_rotate(q, 123, 1e4)
    assert math.isclose(np.linalg.norm(r), np.linalg.norm(q), rel_tol=1e-13)


# ----------------------------------------------------------------------------- pieces
def test_round_bf16_matches_torch():
    x = (_rng(6).standard_normal(20000) * np.exp(_rng(7).uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(orc.round_bf16(x.astype(np.float64)), ref)
    # ties go to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert orc.round_bf16(np.array([1 + 2 ** -8]))[0] == 1.0
    assert orc.round_bf16(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6


def test_rms_norm_properties():
    x = _rng(8).standard_normal((5, 256)) * 3
    y = orc.rms_norm(x, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-13)
    assert np.allclose(orc.rms_norm(7.5 * x, 0.0), y, rtol=1e-13)
    ref = F.rms_norm(torch.from_numpy(x), (256,), eps=1e-5).numpy()
    assert np.allclose(orc.rms_norm(x, 1e-5), ref, rtol=1e-12, atol=1e-14)


def test_attention_matches_torch_sdpa_with_sparse_queries():
    rng = _rng(9)
    N, H, Hkv, dh = 40, 6, 2, 16
    k = rng.standard_normal((N, Hkv, dh))
    v = rng.standard_normal((N, Hkv, dh))
    qpos = np.array([0, 3, 4, 17, 25, 39])
    q = rng.standard_normal((len(qpos), H, dh))
    out = orc.causal_attention(q, qpos, k, v)
    G = H // Hkv
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)  # [H, N, dh]
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)
    qt = torch.from_numpy(q).permute(1, 0, 2)  # [H, m, dh]
    mask = torch.from_numpy(np.arange(N)[None, :] <= qpos[:, None])  # [m, N]
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).permute(1, 0, 2).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_attention_across_query_blocks_matches_torch_sdpa():
    """Unsorted query positions spread over several query blocks (block = 4) of the oracle."""
    rng = _rng(12)
    N, H, Hkv, dh = 50, 8, 2, 16
    k = rng.standard_normal((N, Hkv, dh))
    v = rng.standard_normal((N, Hkv, dh))
    qpos = rng.permutation(N)[:19]
    q = rng.standard_normal((len(qpos), H, dh))
    out = orc.causal_attention(q, qpos, k, v, block=4)
    G = H // Hkv
    kt = torch.from_numpy(k).repeat_interleave(G, dim=1).permute(1, 0, 2)
    vt = torch.from_numpy(v).repeat_interleave(G, dim=1).permute(1, 0, 2)
    qt = torch.from_numpy(q).permute(1, 0, 2)
    mask = torch.from_numpy(np.arange(N)[None, :] <= qpos[:, None])
    ref = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask).permute(1, 0, 2).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


def test_attention_textbook_loops_and_edge_cases():
    rng = _rng(10)
    N, H, dh = 6, 2, 4
    k = rng.standard_normal((N, 1, dh))
    v = rng.standard_normal((N, 1, dh))
    q = rng.standard_normal((N, H, dh))
    out = orc.causal_attention(q, np.arange(N), k, v)
    for t in range(N):
        for h in range(H):
            s = [sum(q[t, h, e] * k[j, 0, e] for e in range(dh)) / 2.0 for j in range(t + 1)]
            w = [math.exp(a - max(s)) for a in s]
            z = sum(w)
            ref = [sum(w[j] / z * v[j, 0, e] for j in range(t + 1)) for e in range(dh)]
            assert np.allclose(out[t, h], ref, atol=1e-13)
    # the first position attends to itself only
    assert np.allclose(out[0, 0], v[0, 0], atol=1e-15)
    # attention weights sum to one: constant V rows give that constant back
    vc = np.ones_like(v) * 3.25
    assert np.allclose(orc.causal_attention(q, np.arange(N), k, vc), 3.25, atol=1e-13)


def test_attention_gqa_reduces_to_mha():
    rng = _rng(11)
    N, Hkv, G, dh = 12, 2, 3, 8
    k = rng.standard_normal((N, Hkv, dh))
    v = rng.standard_normal((N, Hkv, dh))
    q = rng.standard_normal((N, Hkv * G, dh))
    gqa = orc.causal_attention(q, np.arange(N), k, v)
    mha = orc.causal_attention(q, np.arange(N), np.repeat(k, G, axis=1), np.repeat(v, G, axis=1))
    assert np.allclose(gqa, mha, atol=1e-14)


# ----------------------------------------------------------------------------- decoder
def _torch_decoder(cfg, W, ids):
    """The same decoder written with torch library routines (complex RoPE, SDPA)."""
    n = len(ids)
    h = torch.from_numpy(W.embed(ids).astype(np.float64))
    pos = torch.arange(n, dtype=torch.float64)
    half = cfg.head_dim // 2
    freq = cfg.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / cfg.head_dim)
    rot = torch.polar(torch.ones(n, half, dtype=torch.float64), pos[:, None] * freq[None, :])

    def rope(x):  # x [n, heads, dh]
        z = torch.complex(x[..., :half], x[..., half:]) * rot[:, None, :]
        return torch.cat([z.real, z.imag], dim=-1)

    G = cfg.n_heads // cfg.n_kv_heads
    for i in range(cfg.n_layers):
        L = {k_: torch.from_numpy(v_.astype(np.float64)) for k_, v_ in W.layer(i).items()}
        x = F.rms_norm(h, (cfg.d_model,), eps=cfg.rms_eps)
        q = rope(F.linear(x, L["wq"]).view(n, cfg.n_heads, cfg.head_dim))
        k = rope(F.linear(x, L["wk"]).view(n, cfg.n_kv_heads, cfg.head_dim))
        v = F.linear(x, L["wv"]).view(n, cfg.n_kv_heads, cfg.head_dim)
        a = F.scaled_dot_product_attention(q.transpose(0, 1), k.repeat_interleave(G, 1).transpose(0, 1),
                                           v.repeat_interleave(G, 1).transpose(0, 1), is_causal=True)
        h = h + F.linear(a.transpose(0, 1).reshape(n, -1), L["wo"])
        x = F.rms_norm(h, (cfg.d_model,), eps=cfg.rms_eps)
        h = h + F.linear(F.silu(F.linear(x, L["wgate"])) * F.linear(x, L["wup"]), L["wdown"])
    logits = F.linear(F.rms_norm(h[-1:], (cfg.d_model,), eps=cfg.rms_eps), torch.from_numpy(W.lm_head().astype(np.float64)))
    return h.numpy(), int(torch.argmax(logits[0]))


@pytest.mark.parametrize("cfg", [TINY, TINY_MHA])
def test_full_prefill_matches_torch_library_decoder(cfg):
    W = hz.HostWeights(cfg, 77)
    ids = hz.gen_token_ids(hz.stream_key(77, 5), 23, cfg.vocab, "uniform")
    r = orc.full_prefill(cfg, W, ids, "f64")
    ref_h, ref_tok = _torch_decoder(cfg, W, ids)
    assert np.max(np.abs(r["hidden"] - ref_h)) < 1e-10 * np.max(np.abs(ref_h))
    assert r["first_token"] == ref_tok


def test_full_prefill_is_causal():
    W = hz.HostWeights(TINY, 3)
    ids = hz.gen_token_ids(hz.stream_key(3, 1), 30, TINY.vocab, "uniform")
    a = orc.full_prefill(TINY, W, ids, "f64")
    b = orc.full_prefill(TINY, W, ids[:17], "f64")
    assert np.allclose(a["hidden"][:17], b["hidden"], rtol=0, atol=1e-12)
    assert np.allclose(a["k"][:, :17], b["k"], atol=1e-12)


# ----------------------------------------------------------------------------- blend
def test_blend_full_recompute_equals_full_prefill():
    """(a) r = 100 %: every cached token is recomputed, which is a plain full prefill."""
    W = hz.HostWeights(TINY, 21)
    segs, chunks = _prompt(TINY, 21, [12, 10], 5, prefix=8)
    caches = _caches(TINY, W, chunks, "f64")
    ratios = orc.ratio_schedule(TINY.n_layers, 1.0, "fixed")
    b = orc.blend_prefill(TINY, W, segs, caches, ratios, "f64")
    f = orc.full_prefill(TINY, W, _concat(segs), "f64")
    assert np.array_equal(b["rows"], np.arange(len(_concat(segs))))
    assert np.max(np.abs(b["hidden"] - f["hidden"])) < 1e-11
    assert b["first_token"] == f["first_token"]
    assert np.max(np.abs(b["k"] - f["k"])) < 1e-11


def test_blend_zero_ratio_equals_full_kv_reuse():
    """(b) r = 0 %: only the query is recomputed over re-rotated cached KV."""
    W = hz.HostWeights(TINY, 22)
    segs, chunks = _prompt(TINY, 22, [9, 14, 7], 6)
    caches = _caches(TINY, W, chunks, "f64")
    for sched in ("fixed", "gradual"):
        b = orc.blend_prefill(TINY, W, segs, caches, orc.ratio_schedule(TINY.n_layers, 0.0, sched), "f64")
        u = orc.full_reuse(TINY, W, segs, caches, "f64")
        assert np.array_equal(b["rows"], u["rows"])
        assert np.max(np.abs(b["hidden"] - u["hidden"])) < 1e-11
        assert b["first_token"] == u["first_token"]


def test_full_reuse_differs_from_full_prefill():
    """Cross-chunk attention is missing in full reuse (the problem the method solves)."""
    W = hz.HostWeights(TINY, 23)
    segs, chunks = _prompt(TINY, 23, [9, 14], 6)
    caches = _caches(TINY, W, chunks, "f64")
    u = orc.full_reuse(TINY, W, segs, caches, "f64")
    f = orc.full_prefill(TINY, W, _concat(segs), "f64")
    assert np.max(np.abs(u["hidden"] - f["hidden"][u["rows"]])) > 1e-3


@pytest.mark.parametrize("r", [0.0, 0.15, 0.5])
def test_single_chunk_blend_equals_full_prefill(r):
    """One cached chunk at offset 0 is an exact prefix cache: the blend is exact for any r."""
    W = hz.HostWeights(TINY, 24)
    segs, chunks = _prompt(TINY, 24, [20], 6)
    caches = _caches(TINY, W, chunks, "f64")
    b = orc.blend_prefill(TINY, W, segs, caches, orc.ratio_schedule(TINY.n_layers, r, "gradual"), "f64")
    f = orc.full_prefill(TINY, W, _concat(segs), "f64")
    assert np.max(np.abs(b["hidden"] - f["hidden"][b["rows"]])) < 1e-11
    assert b["first_token"] == f["first_token"]


def test_first_chunk_tokens_have_zero_deviation():
    """(d) Tokens of the chunk at offset 0 see the same context as when cached: deviation 0."""
    W = hz.HostWeights(TINY, 25)
    segs, chunks = _prompt(TINY, 25, [11, 13], 4, prefix=9)
    caches = _caches(TINY, W, chunks, "f64")
    b = orc.blend_prefill(TINY, W, segs, caches, orc.ratio_schedule(TINY.n_layers, 0.3, "gradual", r1=0.9), "f64")
    assert len(b["devs"]) >= 2
    for layer, (cand, dev) in b["devs"].items():
        first = cand < 9
        assert first.any() and (~first).any()
        assert np.max(dev[first]) <= 1e-20 * max(1.0, float(np.mean(dev[~first])))
        assert np.min(dev[~first]) > 0.0


def test_layer0_fresh_kv_equals_rerotated_cache():
    """Layer-0 K/V depend only on (token, position): after re-rotation their deviation is 0."""
    W = hz.HostWeights(TINY, 26)
    segs, chunks = _prompt(TINY, 26, [12, 15, 10], 3)
    caches = _caches(TINY, W, chunks, "f64")
    Kf, Vf = orc.init_fused_cache(TINY, segs, caches, "f64")
    ids = _concat(segs)
    nc = 37
    q, k, v = orc.project_qkv(TINY, W.layer(0), W.embed(ids).astype(np.float64), np.arange(len(ids)))
    dev = orc.kv_deviation(k[:nc], v[:nc], Kf[0][:nc], Vf[0][:nc])
    assert np.max(dev) < 1e-24
    # but not at layer 1 for tokens after the first chunk
    b = orc.blend_prefill(TINY, W, segs, caches, orc.ratio_schedule(TINY.n_layers, 0.5, "fixed"), "f64")
    cand, d1 = b["devs"][1]
    assert np.max(d1[cand >= 12]) > 1e-6


def test_gradual_sets_are_nested_and_sized():
    W = hz.HostWeights(TINY, 27)
    segs, chunks = _prompt(TINY, 27, [16, 16, 16], 5, prefix=4)
    caches = _caches(TINY, W, chunks, "f64")
    ratios = orc.ratio_schedule(TINY.n_layers, 0.2, "gradual")
    b = orc.blend_prefill(TINY, W, segs, caches, ratios, "f64")
    nc = b["n_cached"]
    prev = None
    for i in range(TINY.n_layers):
        S = b["sets"][i]
        assert np.all(np.diff(S) > 0)
        assert set(range(nc, nc + 5)) <= set(S.tolist())
        if ratios[i] >= 0:
            assert len(S) == 5 + min(orc.k_for_ratio(ratios[i], nc), int(np.sum(prev < nc)))
        if prev is not None:
            assert set(S.tolist()) <= set(prev.tolist())
        prev = S


def test_forced_selection_is_followed():
    W = hz.HostWeights(TINY, 28)
    segs, chunks = _prompt(TINY, 28, [10, 10], 3)
    caches = _caches(TINY, W, chunks, "f64")
    ratios = orc.ratio_schedule(TINY.n_layers, 0.3, "fixed")
    forced = {1: np.array([2, 11, 15, 20, 21, 22])}
    b = orc.blend_prefill(TINY, W, segs, caches, ratios, "f64", force_sel=forced)
    assert np.array_equal(b["sets"][1], forced[1])
    assert np.array_equal(b["rows"], forced[1])


# ----------------------------------------------------------------------------- selection
def _brute_topk(dev32, cand, k):
    """Among all k-subsets, the one whose members all outrank every non-member."""
    n = len(cand)
    better = lambda a, b: (dev32[a] > dev32[b]) or (dev32[a] == dev32[b] and cand[a] < cand[b])  # noqa: E731
    hits = []
    for sub in itertools.combinations(range(n), k):
        rest = [j for j in range(n) if j not in sub]
        if all(better(a, b) for a in sub for b in rest):
            hits.append(sorted(cand[list(sub)]))
    assert len(hits) == 1
    return np.array(hits[0], dtype=np.int64)


def test_select_exhaustive_small_with_ties():
    rng = _rng(12)
    for trial in range(300):
        n = int(rng.integers(1, 9))
        dev = rng.integers(0, 4, n).astype(np.float32) * np.float32(0.5)  # many ties
        cand = np.sort(rng.choice(100, n, replace=False))
        for k in range(0, n + 1):
            got = orc.select_hkvd(dev, cand, k)
            assert np.array_equal(got, _brute_topk(dev, cand, k) if k else np.zeros(0, np.int64))


def test_select_matches_full_sort():
    rng = _rng(13)
    dev = rng.standard_normal(5000).astype(np.float32) ** 2
    dev[::7] = dev[3]  # ties
    cand = np.arange(5000) * 2 + 1
    for k in (1, 471, 4999, 5000):
        pairs = sorted(zip((-dev.astype(np.float64)).tolist(), cand.tolist()))
        ref = np.sort(np.array([c for _, c in pairs[:k]]))
        assert np.array_equal(orc.select_hkvd(dev, cand, k), ref)
    with pytest.raises(FloatingPointError):
        orc.select_hkvd(np.array([1.0, np.nan], np.float32), np.array([0, 1]), 1)


def test_deviation_closed_forms():
    rng = _rng(14)
    kn, vn, kf, vf = (rng.standard_normal((9, 2, 8)) for _ in range(4))
    full = orc.kv_deviation(kn, vn, kf, vf, 0)
    ref = np.linalg.norm(np.concatenate([(kn - kf).reshape(9, -1), (vn - vf).reshape(9, -1)], 1), axis=1) ** 2
    assert np.allclose(full, ref, rtol=1e-13)
    assert np.allclose(orc.kv_deviation(kn, vn, kf, vf, 1) + orc.kv_deviation(kn, vn, kf, vf, 2), full, rtol=1e-13)
    assert np.all(orc.kv_deviation(kn, vn, kn, vn) == 0)


def test_cosine_deviation_closed_forms():
    """mode 3 = 1 - cos of the concatenated K and V rows: 0 for a positive multiple, 2 for
    the negated row, 1 for an orthogonal one, scale-free, and on unit rows half the
    squared L2 deviation of mode 0 (||a - b||^2 = 2 (1 - cos))."""
    rng = _rng(15)
    kn, vn, kf, vf = (rng.standard_normal((9, 2, 8)) for _ in range(4))
    assert np.max(np.abs(orc.kv_deviation(3.0 * kf, 3.0 * vf, kf, vf, 3))) < 1e-14
    assert np.allclose(orc.kv_deviation(-kf, -vf, kf, vf, 3), 2.0, rtol=0, atol=1e-14)
    ek = np.zeros((2, 1, 4))
    ev = np.zeros((2, 1, 4))
    ek[0, 0, 0] = 1.0  # row 0: a = e0 (K part), b = e1 (V part): orthogonal
    fk = np.zeros((2, 1, 4))
    fv = np.zeros((2, 1, 4))
    fv[0, 0, 1] = 2.0
    ek[1, 0, 2], fk[1, 0, 2], fv[1, 0, 3] = 1.0, 1.0, 1.0  # row 1: cos = 1/sqrt(2)
    assert np.allclose(orc.kv_deviation(ek, ev, fk, fv, 3), [1.0, 1.0 - 1.0 / math.sqrt(2.0)], rtol=0, atol=1e-15)
    assert np.allclose(orc.kv_deviation(5.0 * kn, 5.0 * vn, 0.25 * kf, 0.25 * vf, 3),
                       orc.kv_deviation(kn, vn, kf, vf, 3), rtol=1e-12)

    def unit(k, v):
        nrm = np.sqrt(np.sum(k.reshape(9, -1) ** 2, 1) + np.sum(v.reshape(9, -1) ** 2, 1))[:, None, None]
        return k / nrm, v / nrm

    ku, vu = unit(kn, vn)
    kfu, vfu = unit(kf, vf)
    assert np.allclose(orc.kv_deviation(ku, vu, kfu, vfu, 0), 2.0 * orc.kv_deviation(ku, vu, kfu, vfu, 3),
                       rtol=1e-12)
    z = np.zeros((2, 1, 4))
    assert list(orc.kv_deviation(z, z, z, z, 3)) == [0.0, 0.0]
    assert list(orc.kv_deviation(z, z, fk, fv, 3)) == [1.0, 1.0]


def _seam_layout(lens, qlen):
    segs = [hz.Segment(np.arange(n) % 7, i) for i, n in enumerate(lens)]
    segs.append(hz.Segment(np.arange(qlen) % 5, -1))
    return segs


def test_seam_positions_hand_examples():
    """[P2] SelectiveRecompute: the R tokens just before each chunk boundary; chunks of 5, 3
    and 7 tokens sit at 0-4, 5-7 and 8-14, the query at 15-18."""
    segs = _seam_layout([5, 3, 7], 4)
    assert list(orc.seam_positions(segs, 2)) == [3, 4, 6, 7, 13, 14]
    assert list(orc.seam_positions(segs, 4)) == [1, 2, 3, 4, 5, 6, 7, 11, 12, 13, 14]
    assert list(orc.seam_positions(segs, 0)) == []
    assert list(orc.seam_positions(segs, 99)) == list(range(15))
    assert list(orc.seam_positions(_seam_layout([6], 2), 1)) == [5]


def test_seam_repair_limits():
    """R = 0 is full KV reuse; R covering every chunk recomputes everything (a full prefill);
    a lone chunk at offset 0 is an exact prefix cache, so any R gives the full prefill."""
    W = hz.HostWeights(TINY, 28)
    segs, chunks = _prompt(TINY, 28, [9, 14, 7], 6)
    caches = _caches(TINY, W, chunks, "f64")
    s0 = orc.seam_repair_prefill(TINY, W, segs, caches, 0, "f64")
    u = orc.full_reuse(TINY, W, segs, caches, "f64")
    assert np.array_equal(s0["rows"], u["rows"])
    assert np.max(np.abs(s0["hidden"] - u["hidden"])) < 1e-11
    f = orc.full_prefill(TINY, W, _concat(segs), "f64")
    s_all = orc.seam_repair_prefill(TINY, W, segs, caches, 14, "f64")
    assert np.array_equal(s_all["rows"], np.arange(36))
    assert np.max(np.abs(s_all["hidden"] - f["hidden"])) < 1e-11
    assert np.max(np.abs(s_all["k"] - f["k"])) < 1e-11 and s_all["first_token"] == f["first_token"]
    s4 = orc.seam_repair_prefill(TINY, W, segs, caches, 4, "f64")
    assert len(s4["rows"]) == 12 + 6
    assert np.max(np.abs(s4["hidden"][-6:] - f["hidden"][-6:])) > 1e-6  # still an approximation
    segs1, chunks1 = _prompt(TINY, 29, [20], 6)
    caches1 = _caches(TINY, W, chunks1, "f64")
    f1 = orc.full_prefill(TINY, W, _concat(segs1), "f64")
    for R in (1, 5):
        s = orc.seam_repair_prefill(TINY, W, segs1, caches1, R, "f64")
        assert np.max(np.abs(s["hidden"] - f1["hidden"][s["rows"]])) < 1e-11


# ----------------------------------------------------------------------------- KV codec
def test_codec_hand_example_fixes_the_axes():
    """Keys are grouped per channel over the tokens, values per token over the channels:
    tokens x channels [[0, 10], [1, 20], [3, 40]] give key codes 0, 85, 255 down each channel
    (int8) and value codes 0, 255 along each token."""
    x = np.array([[0.0, 10.0], [1.0, 20.0], [3.0, 40.0]], dtype=np.float32)[None, :, None, :]  # [1, 3, 1, 2]
    e8 = orc.kv_encode(x, x, 8)
    assert e8["k_codes"][0, :, 0, :].tolist() == [[0, 0], [85, 85], [255, 255]]
    assert e8["v_codes"][0, :, 0, :].tolist() == [[0, 255], [0, 255], [0, 255]]
    assert e8["k_zero"][0, 0].tolist() == [0.0, 10.0] and e8["v_zero"][0, :, 0].tolist() == [0.0, 1.0, 3.0]
    assert e8["k_scale"][0, 0].tolist() == [np.float32(3.0) / np.float32(255.0), np.float32(30.0) / np.float32(255.0)]
    e4 = orc.kv_encode(x, x, 4)
    assert e4["k_codes"][0, :, 0, :].tolist() == [[0, 0], [5, 5], [15, 15]]
    assert e4["v_codes"][0, :, 0, :].tolist() == [[0, 15], [0, 15], [0, 15]]


@pytest.mark.parametrize("bits", [4, 8])
def test_codec_error_bound_and_extremes(bits):
    """Round trip within half a step of each group; every group's minimum maps to code 0
    and its maximum to 2^b - 1."""
    rng = _rng(31 + bits)
    K = (rng.standard_normal((2, 37, 3, 16)) * rng.uniform(0.1, 5.0, (1, 1, 3, 16))).astype(np.float32)
    V = (rng.standard_normal((2, 37, 3, 16)) * rng.uniform(0.1, 5.0, (1, 37, 1, 1))).astype(np.float32)
    e = orc.kv_encode(K, V, bits)
    Kh, Vh = orc.kv_decode(e)
    lv = 2 ** bits - 1
    assert e["k_scale"].shape == (2, 3, 16) and e["v_scale"].shape == (2, 37, 3)
    assert np.all(np.abs(K - Kh) <= e["k_scale"][:, None] * 0.5 * (1 + 1e-5))
    assert np.all(np.abs(V - Vh) <= e["v_scale"][..., None] * 0.5 * (1 + 1e-5))
    assert np.all(e["k_codes"].min(axis=1) == 0) and np.all(e["k_codes"].max(axis=1) == lv)
    assert np.all(e["v_codes"].min(axis=3) == 0) and np.all(e["v_codes"].max(axis=3) == lv)
    # the error really is of the order of a step (the bound is not vacuous)
    assert np.max(np.abs(K - Kh) / e["k_scale"][:, None]) > 0.4


def test_codec_exact_on_grid_and_constant_groups():
    """Values on a power-of-two grid spanning the levels come back exactly; a constant group
    has scale 0, codes 0 and decodes exactly."""
    rng = _rng(33)
    q = rng.integers(0, 256, (1, 40, 2, 8)).astype(np.float32)
    q[:, 0], q[:, 1] = 0.0, 255.0  # every channel spans the full range
    K = (q * np.float32(2.0 ** -4) - np.float32(3.0)).astype(np.float32)
    e = orc.kv_encode(K, K, 8)
    assert np.array_equal(orc.kv_decode(e)[0], K.astype(np.float64))
    C = np.full((1, 5, 2, 8), 1.25, dtype=np.float32)
    e = orc.kv_encode(C, C, 4)
    assert np.all(e["k_scale"] == 0) and np.all(e["k_codes"] == 0) and np.all(e["v_codes"] == 0)
    Kd, Vd = orc.kv_decode(e)
    assert np.all(Kd == 1.25) and np.all(Vd == 1.25)


def test_ratio_schedule_and_k():
    assert orc.ratio_schedule(2, 0.15, "fixed") == [-1.0, 0.15]
    g = orc.ratio_schedule(32, 0.15, "gradual")
    assert g[0] == -1 and g[1] == pytest.approx(0.30) and g[4] == pytest.approx(0.15)
    assert g[2] == pytest.approx(0.25) and g[3] == pytest.approx(0.20) and all(x == -1 for x in g[5:])
    checks = [x for x in g if x >= 0]
    assert all(a >= b for a, b in zip(checks, checks[1:]))
    # k = ceil(r * Nc) for the named workloads
    assert orc.k_for_ratio(0.15, 256) == 39
    assert orc.k_for_ratio(0.15, 3136) == 471
    assert [orc.k_for_ratio(r, 4096) for r in (0, .05, .10, .15, .20, .50, 1.0)] == [0, 205, 410, 615, 820, 2048, 4096]
    assert orc.k_for_ratio(0.15, 8192) == 1229
    assert orc.k_for_ratio(0.10, 8192) == 820 and orc.k_for_ratio(0.20, 8192) == 1639


# ----------------------------------------------------------------------------- bytes / cost model
def test_kv_bytes_and_cost_model_match_printed_numbers():
    with open(os.path.join(GOLDEN, "kv_bytes.json")) as f:
        g = json.load(f)
    for row in g["per_token_kv_bytes"]:
        assert orc.kv_bytes_per_token(row["n_layers"], row["n_kv_heads"], row["head_dim"], row["elem_bytes"]) == row["bytes"]
    lk = g["loaded_kv"]
    assert abs(lk["tokens"] * lk["bytes_per_token"] / 2 ** 30 - lk["gib"]) < lk["gib_tol"]
    be = g["break_even"]
    assert abs(orc.break_even_bandwidth(be["bytes_per_token"], be["prefill_ms_per_token"] * 1e-3) / 1e9 - be["gbs"]) < be["gbs_tol"]
    ll = g["layer_load_llama7b_4k"]
    per_tok = orc.kv_bytes_per_token(ll["n_layers"], ll["n_kv_heads"], ll["head_dim"], ll["elem_bytes"])
    t = orc.t_load(ll["n_tokens"], per_tok, 1, ll["n_layers"], ll["ssd_gbs"] * 1e9)
    assert abs(t * 1e3 - ll["printed_ms"]) / ll["printed_ms"] < ll["rel_tol"]
    assert orc.pipelined_latency([1, 5, 2], [3, 3, 3]) == 11
    assert orc.t_recompute(0.15, 100.0) == pytest.approx(15.0)


# ----------------------------------------------------------------------------- loading controller
def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_fnv1a64_published_vectors_and_chunk_key():
    g = _golden("loading_controller.json")["fnv1a64_vectors"]
    for text, hexval in g.items():
        if text.startswith("_"):
            continue
        assert orc.fnv1a64(text.encode()) == int(hexval, 16), text
    ids = [1, 258, -1, 70000]
    raw = b"".join(int(x).to_bytes(4, "little", signed=True) for x in ids)
    assert orc.chunk_hash(ids) == orc.fnv1a64(raw)
    assert orc.chunk_hash(np.array(ids, dtype=np.int64)) == orc.chunk_hash(ids)
    keys = {orc.chunk_hash(hz.gen_token_ids(hz.stream_key(7, i), 64, 32000, "zipf")) for i in range(200)}
    assert len(keys) == 200
    assert orc.chunk_hash([1, 2]) != orc.chunk_hash([2, 1])


def test_load_or_recompute_follows_the_printed_break_even():
    """[P4] §5: 6,414 tokens (0.12 ms each), 28,672 B per token: load over 13.4 GB/s, recompute
    over 104 MB/s (about 1.8 s of transfer against 0.77 s of prefill)."""
    g = _golden("loading_controller.json")["break_even_cases"]
    n, t_tok = g["n_tokens"], g["prefill_s"] / g["n_tokens"]
    nbytes = n * g["bytes_per_token"]
    act = {"load": orc.ACT_LOAD, "recompute": orc.ACT_RECOMPUTE}
    assert orc.chunk_action(orc.TIER_HOST, n, nbytes, g["fast_link_bytes_per_s"], 0.0, t_tok) == act[g["fast_action"]]
    assert orc.chunk_action(orc.TIER_HOST, n, nbytes, g["slow_link_bytes_per_s"], 0.0, t_tok) == act[g["slow_action"]]
    assert abs(nbytes / g["slow_link_bytes_per_s"] - g["slow_load_s"]) < g["slow_load_tol"]
    # the threshold is the break-even bandwidth of the same section
    bw = orc.break_even_bandwidth(g["bytes_per_token"], t_tok)
    assert orc.chunk_action(orc.TIER_HOST, n, nbytes, bw * 1.01, 0.0, t_tok) == orc.ACT_LOAD
    assert orc.chunk_action(orc.TIER_HOST, n, nbytes, bw * 0.99, 0.0, t_tok) == orc.ACT_RECOMPUTE
    assert orc.chunk_action(orc.TIER_DEVICE, n, nbytes, 1.0, 0.0, t_tok) == orc.ACT_USE
    assert orc.chunk_action(orc.TIER_MISSING, n, nbytes, 1e12, 0.0, t_tok) == orc.ACT_RECOMPUTE


def test_ratio_rule_hides_recompute_under_the_load():
    """[P1] 閾値チューニング: slower storage raises r (up to r_max), faster storage lowers it (down
    to r_min, also when nothing is loaded); between the bounds the chosen r makes T_recompute
    equal T_load exactly.  A link so slow that recomputing beats loading loads nothing."""
    g = _golden("loading_controller.json")["ratio_rule"]
    base = {"link_latency_s": 0.0, "prefill_s_per_token": 1e-5, "recompute_fixed_s": 0.0,
            "r_min": g["r_min"], "r_max": g["r_max"]}
    chunks = [{"tier": orc.TIER_HOST, "n_tokens": 512, "bytes": 512 * 131072.0} for _ in range(8)]
    n_q = 32
    t_prefill = (8 * 512 + n_q) * 1e-5
    rs = []
    inside = 0
    for bw in (2e10, 7e10, 1.31e11, 2e11, 1e12):  # per-token load 6.6 .. 0.13 us < 10 us of prefill
        acts, r, t_load, t_rec = orc.plan_loading(dict(base, link_bytes_per_s=bw), chunks, n_q)
        assert all(a == orc.ACT_LOAD for a in acts)
        rs.append(r)
        if g["r_min"] < r < g["r_max"]:
            inside += 1
            assert abs(t_rec - t_load) < 1e-12 and abs(t_rec - r * t_prefill) < 1e-12
    assert rs[0] == g["r_max"] and rs[-1] == g["r_min"] and inside == 3
    assert all(a > b for a, b in zip(rs, rs[1:]))
    acts, r, t_load, _ = orc.plan_loading(dict(base, link_bytes_per_s=1e9), chunks, n_q)  # 131 us per token
    assert all(a == orc.ACT_RECOMPUTE for a in acts) and t_load == 0 and r == g["r_min"]
    fixed = dict(base, link_bytes_per_s=1.31e11, recompute_fixed_s=0.001)
    _, r_f, t_load_f, t_rec_f = orc.plan_loading(fixed, chunks, n_q)
    assert abs(t_rec_f - t_load_f) < 1e-12 and r_f < rs[2]  # a fixed recompute cost leaves less room
    assert orc.plan_loading(dict(base, link_bytes_per_s=1e9), [{"tier": orc.TIER_DEVICE, "n_tokens": 9, "bytes": 1.0}],
                            3)[1] == g["r_min"]


# ----------------------------------------------------------------------------- decode
def test_decode_after_prefill_equals_a_longer_prefill():
    """A decode step on the KV of a full prefill of ids[:-1], fed ids[-1], is the last row of a
    full prefill of ids; two steps extend it by the greedy token."""
    W = hz.HostWeights(TINY, 51)
    ids = hz.gen_token_ids(hz.stream_key(51, 1), 23, TINY.vocab, "uniform")
    f_short = orc.full_prefill(TINY, W, ids[:-1], "f64")
    cap = 30
    K = np.zeros((TINY.n_layers, cap, TINY.n_kv_heads, TINY.head_dim))
    V = np.zeros_like(K)
    K[:, :22], V[:, :22] = f_short["k"], f_short["v"]
    st = orc.decode_step(TINY, W, K, V, 22, int(ids[-1]), "f64")
    f_full = orc.full_prefill(TINY, W, ids, "f64")
    assert np.max(np.abs(st["hidden"] - f_full["hidden"][-1])) < 1e-11
    assert st["token"] == f_full["first_token"]
    assert np.max(np.abs(K[:, :23] - f_full["k"])) < 1e-11
    st2 = orc.decode_step(TINY, W, K, V, 23, st["token"], "f64")
    f2 = orc.full_prefill(TINY, W, np.append(ids, st["token"]), "f64")
    assert np.max(np.abs(st2["hidden"] - f2["hidden"][-1])) < 1e-11
    K2 = np.zeros_like(K)
    V2 = np.zeros_like(V)
    K2[:, :22], V2[:, :22] = f_short["k"], f_short["v"]
    assert orc.greedy_decode(TINY, W, K2, V2, 22, int(ids[-1]), 2, "f64") == [st["token"], st2["token"]]
