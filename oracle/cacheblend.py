"""CPU oracle of CacheBlend's blended prefill ("cached knowledge fusion").

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module: only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
use it.  It shares no code with the CUDA library; both read their inputs from
``harness`` (seeded generators, no method arithmetic).

Everything is computed in float64 with plain numpy (matrix products are the
only library primitive used as a step).  The one place where lower precision
enters on purpose is the KV *storage* dtype: the cached chunk KV and the fused
cache are rounded to the storage type (``"f64"``, ``"f32"`` or ``"bf16"``) when
written, because that is what a cache holds.

Pages cited (titles as published; sections by heading):

* [P1] "論文解説: CacheBlend - RAG向けKVキャッシュ融合によるLLM推論高速化"
  (0h-n0.github.io), an explainer of arXiv 2405.16444.
* [P2] "KVキャッシュを再利用してLLM推論を4.49倍高速化——KVBoostが切り拓く自宅サーバーLLMの新境地".
* [P3] "논문: CacheBlend: Fast Large Language Model Serving for RAG with Cached
  Knowledge Fusion" (jaehun.me).
* [P4] "LMCache: KV キャシを GPU の外へ" (ttlab.hopto.org).

Readings where the pages are silent or garbled (each is restated where used):

R1  RoPE pairs element i with element i + dh/2 ("rotate half"), inverse
    frequency theta**(-2i/dh), angles evaluated in float64.
R2  "Layer 1" of gradual filtering is the second layer (0-indexed 1): layer-0
    K/V depend only on (token, position), so their deviation is zero.
R3  Gradual filtering is a per-layer array of ratios of *all cached tokens*,
    non-increasing; a negative entry means "no check: keep the previous set".
    Layer 0 runs on every token, which supplies layer-1 inputs for the check.
R4  The deviation of token j is the squared L2 norm of the difference of the
    concatenated K (after re-rotation) and V rows over all KV heads.
R5  k_i = ceil(r_i * Nc - 1e-9) over the Nc cached tokens of the request,
    clamped to the cached candidates available; query tokens are always kept.
R6  Top-k order: deviation descending, then token index ascending.  The
    selected indices are returned in ascending order.
R7  Fresh K/V of candidates that are not selected are discarded.
R9  RMSNorm weight 1, eps 1e-5; no biases; untied LM head; no BOS token.
R14 Selection runs on the fp32-rounded deviations, so the CUDA selection can be
    compared bit for bit on the same fp32 array.
R17 The cosine deviation is 1 - cos over the concatenated K and V rows; a zero row
    against a zero row deviates by 0, against a non-zero row by 1.
R18 Spatial seam repair recomputes the last R tokens of every cached chunk (each
    ends at a boundary) plus the query, at every layer from layer 0 on.
R19 A quantised key group is one channel of one KV head of one layer over all the
    chunk's tokens ("per channel").
R20 A quantised value group is one token's row of one KV head of one layer, head_dim
    channels ("per token").
R22 The "text hash" that keys the chunk store is FNV-1a 64 over the chunk's token ids
    (little-endian int32 bytes): content only, independent of the chunk's position.
R23 Per chunk: device-resident -> use; host-resident -> load when bytes / bandwidth +
    latency is below n x prefill time per token, else recompute; missing -> recompute.
R24 The ratio chosen is the largest whose recompute time (fixed + r x T_prefill) fits
    under T_load, clamped to [r_min, r_max]; r_min when nothing is loaded.
R21 Quantisation is asymmetric min/max (as KIVI): scale = (max - min) / (2^b - 1), the
    minimum kept as the zero point, codes rounded half to even and clamped; a group
    whose values are all equal gets scale 0 and codes 0.

Parity pins (tests/test_oracle_*.py) tie every function here to something other
than itself: closed forms, invariants, the pages' printed byte counts, library
routines (torch SDPA, complex exponentials) and brute force on tiny inputs.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

STORAGE_TYPES = ("f64", "f32", "bf16")


# --------------------------------------------------------------------------- rounding
def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (8 significant bits), ties to even."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0), e - 8)


def round_storage(x: np.ndarray, storage: str) -> np.ndarray:
    """Values as a KV cache of type ``storage`` holds them."""
    if storage == "f64":
        return np.asarray(x, dtype=np.float64)
    if storage == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    if storage == "bf16":
        return round_bf16(x)
    raise ValueError(storage)


# --------------------------------------------------------------------------- RoPE
def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """Inverse frequencies theta**(-2i/dh), i < dh/2 (reading R1)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_rotate(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotary position embedding of rows x[n, heads, dh] at positions pos[n] (or one scalar).

    [P1] 技術的詳細 / 位置エンコーディングの更新: keys carry a rotation R(p) that depends on
    their position.  Element i is paired with element i + dh/2 (reading R1):
    (a, b) -> (a cos t - b sin t, b cos t + a sin t) with t = pos * inv_freq_i.
    """
    x = np.asarray(x, dtype=np.float64)
    n, _, dh = x.shape
    half = dh // 2
    pos = np.broadcast_to(np.asarray(pos, dtype=np.float64), (n,))
    ang = pos[:, None] * rope_inv_freq(dh, theta)[None, :]  # [n, half]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def rerotate_keys(k_cached: np.ndarray, delta: int, theta: float) -> np.ndarray:
    """K_new = R(delta) . K_cached for every row of a chunk moved by ``delta`` positions.

    [P1] 技術的詳細 / 位置エンコーディングの更新, the re-rotation equation: a chunk cached at
    positions 0..n-1 and placed at offset ``delta`` needs the extra rotation R(delta).
    """
    return rope_rotate(k_cached, delta, theta)


# --------------------------------------------------------------------------- decoder pieces
def rms_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x**2) + eps) per row; weight 1 (reading R9)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def causal_attention(q: np.ndarray, q_pos: Sequence[int], k: np.ndarray, v: np.ndarray,
                     block: int = 256) -> np.ndarray:
    """Causal scaled-dot-product attention of sparse queries over a KV cache.

    q[m, H, dh] are queries at global positions q_pos[m]; k, v[N, Hkv, dh] hold the
    cache.  Query t attends to cache rows 0..q_pos[t] with scale 1/sqrt(dh); head h
    reads KV head floor(h * Hkv / H) (grouped-query attention).  [P3] "어떤 토큰을
    다시 계산하는가": selected queries attend, under the causal mask, to all available
    K/V -- cached rows included.

    Written as softmax(q K^T / sqrt(dh) + M) V with M[t, j] = -inf for keys j after
    q_pos[t] (0 otherwise).  Query rows are independent; taking them ``block`` at a time
    only bounds the memory of the score matrix.
    """
    m, H, dh = q.shape
    Hkv = k.shape[1]
    G = H // Hkv
    out = np.zeros((m, H, dh), dtype=np.float64)
    scale = 1.0 / math.sqrt(dh)
    q_pos = np.asarray(q_pos, dtype=np.int64).reshape(m)
    for t0 in range(0, m, block):
        t1 = min(m, t0 + block)
        b = t1 - t0
        n = int(q_pos[t0:t1].max()) + 1  # keys any query of the block may see
        after = np.arange(n)[None, :] > q_pos[t0:t1, None]  # [b, n]: the causal mask
        for g in range(Hkv):  # query heads g*G .. g*G + G - 1 read KV head g
            qg = q[t0:t1, g * G:(g + 1) * G, :].reshape(b * G, dh)
            s = (qg @ k[:n, g, :].T).reshape(b, G, n) * scale
            s = np.where(after[:, None, :], -np.inf, s)
            s = s - s.max(axis=-1, keepdims=True)
            w = np.exp(s)
            w = w / w.sum(axis=-1, keepdims=True)
            out[t0:t1, g * G:(g + 1) * G, :] = (w.reshape(b * G, n) @ v[:n, g, :]).reshape(b, G, dh)
    return out


def project_qkv(cfg, W: Dict[str, np.ndarray], h: np.ndarray, pos: Sequence[int]):
    """x = RMSNorm(h); q, k, v = x W_q^T, x W_k^T, x W_v^T; RoPE on q and k at ``pos``."""
    n = h.shape[0]
    x = rms_norm(h, cfg.rms_eps)
    q = (x @ W["wq"].astype(np.float64).T).reshape(n, cfg.n_heads, cfg.head_dim)
    k = (x @ W["wk"].astype(np.float64).T).reshape(n, cfg.n_kv_heads, cfg.head_dim)
    v = (x @ W["wv"].astype(np.float64).T).reshape(n, cfg.n_kv_heads, cfg.head_dim)
    pos = np.asarray(pos)
    return rope_rotate(q, pos, cfg.rope_theta), rope_rotate(k, pos, cfg.rope_theta), v


def output_and_mlp(cfg, W: Dict[str, np.ndarray], h: np.ndarray, attn: np.ndarray) -> np.ndarray:
    """h += attn W_o^T; h += (SiLU(x W_gate^T) * (x W_up^T)) W_down^T with x = RMSNorm(h)."""
    n = h.shape[0]
    h = h + attn.reshape(n, cfg.q_width) @ W["wo"].astype(np.float64).T
    x = rms_norm(h, cfg.rms_eps)
    g = x @ W["wgate"].astype(np.float64).T
    u = x @ W["wup"].astype(np.float64).T
    return h + (silu(g) * u) @ W["wdown"].astype(np.float64).T


def lm_logits(cfg, weights, h_last: np.ndarray) -> np.ndarray:
    """Logits of the untied LM head over RMSNorm(h) of one hidden row (reading R9)."""
    x = rms_norm(np.asarray(h_last, dtype=np.float64)[None, :], cfg.rms_eps)[0]
    return weights.lm_head().astype(np.float64) @ x


def first_token(cfg, weights, h_last: np.ndarray) -> int:
    """argmax of the LM head over RMSNorm(h) of the last prompt token; ties -> lowest id."""
    return int(np.argmax(lm_logits(cfg, weights, h_last)))


# --------------------------------------------------------------------------- full prefill
def full_prefill(cfg, weights, ids: Sequence[int], storage: str = "f64", want_logits_token: bool = True):
    """Plain causal prefill of ``ids`` at positions 0..n-1 (the full-recompute baseline).

    Returns the final hidden states [n, d], the per-layer K (with RoPE) and V as the
    cache holds them (rounded to ``storage``), and the first generated token.
    [P1] 実験結果 / TTFT: "Full Recompute" is the baseline CacheBlend is compared with.
    """
    ids = np.asarray(ids)
    n = len(ids)
    pos = np.arange(n)
    h = weights.embed(ids).astype(np.float64)
    K = np.zeros((cfg.n_layers, n, cfg.n_kv_heads, cfg.head_dim))
    V = np.zeros_like(K)
    for i in range(cfg.n_layers):
        W = weights.layer(i)
        q, k, v = project_qkv(cfg, W, h, pos)
        K[i] = round_storage(k, storage)
        V[i] = round_storage(v, storage)
        attn = causal_attention(q, pos, K[i], V[i])
        h = output_and_mlp(cfg, W, h, attn)
    tok = first_token(cfg, weights, h[-1]) if want_logits_token else None
    return {"hidden": h, "k": K, "v": V, "first_token": tok}


def precompute_chunk(cfg, weights, ids: Sequence[int], storage: str):
    """A chunk's KV cache: the chunk prefilled alone from position 0.

    [P3] "어떤 문제를 해결하는가": each retrieved chunk is processed independently and its
    KV stored; [P1] 背景と動機: each document can be precomputed on its own.
    """
    r = full_prefill(cfg, weights, ids, storage, want_logits_token=False)
    return r["k"], r["v"]


# --------------------------------------------------------------------------- HKVD
def kv_deviation(k_new, v_new, k_fused, v_fused, mode: int = 0) -> np.ndarray:
    """KV deviation per token (readings R4, R17).

    [P1] 技術的詳細 / HKVD トークン選定: Delta_KV^(i)[j] = || KV_cached^(i)[j] - KV_full^(i)[j] ||_2.
    The squared norm ranks tokens the same way.  mode 0: K and V together;
    mode 1: K only; mode 2: V only.

    mode 3 is the cosine form of [P2] シーム修復戦略 / CacheBlendRecompute (a per-token
    cosine-similarity deviation): 1 - cos(a, b) of the concatenated K and V rows a
    (fresh) and b (fused cache).  Reading R17: two zero rows deviate by 0, a zero row
    against a non-zero one by 1.
    """
    n = k_new.shape[0]
    width = int(np.prod(k_new.shape[1:]))
    if mode == 3:
        a = np.concatenate([np.asarray(k_new, np.float64).reshape(n, width),
                            np.asarray(v_new, np.float64).reshape(n, width)], axis=1)
        b = np.concatenate([np.asarray(k_fused, np.float64).reshape(n, width),
                            np.asarray(v_fused, np.float64).reshape(n, width)], axis=1)
        ab = np.sum(a * b, axis=1)
        aa = np.sum(a * a, axis=1)
        bb = np.sum(b * b, axis=1)
        out = np.where((aa == 0) & (bb == 0), 0.0, 1.0)
        both = (aa > 0) & (bb > 0)
        out[both] = 1.0 - ab[both] / np.sqrt(aa[both] * bb[both])
        return out
    dk = (np.asarray(k_new, np.float64) - np.asarray(k_fused, np.float64)).reshape(n, width)
    dv = (np.asarray(v_new, np.float64) - np.asarray(v_fused, np.float64)).reshape(n, width)
    sk = np.sum(dk * dk, axis=1)
    sv = np.sum(dv * dv, axis=1)
    if mode == 0:
        return sk + sv
    if mode == 1:
        return sk
    if mode == 2:
        return sv
    raise ValueError(mode)


def select_hkvd(dev32: np.ndarray, cand: Sequence[int], k: int) -> np.ndarray:
    """The k candidates of highest deviation, as ascending token indices (readings R6, R14).

    [P1] 段階的フィルタリングスキーム: the HKVD tokens are the top r% by deviation.
    Order: deviation descending, then token index ascending.
    """
    dev32 = np.asarray(dev32, dtype=np.float32)
    cand = np.asarray(cand, dtype=np.int64)
    if np.any(np.isnan(dev32)):
        raise FloatingPointError("NaN deviation")
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    order = np.lexsort((cand, -dev32.astype(np.float64)))  # primary: -dev, secondary: index
    return np.sort(cand[order[:k]])


def k_for_ratio(r: float, n_cached: int) -> int:
    """k = ceil(r * Nc - 1e-9) (reading R5)."""
    if r <= 0:
        return 0
    return int(math.ceil(r * n_cached - 1e-9))


def ratio_schedule(n_layers: int, r: float, schedule: str = "gradual", r1: Optional[float] = None,
                   n_narrow: int = 3) -> List[float]:
    """Per-layer recompute ratios of gradual filtering (reading R3).

    [P1] 段階的フィルタリングスキーム: layer 1 recomputes r1 % of all tokens and measures
    their deviation; each later layer keeps a narrower share of the previous one.
    Layer 0: no check (all tokens).  Layer 1: r1.  Layers 2..1+n_narrow: linear from
    r1 down to r.  Later layers: no check (the set of the last checked layer is kept).
    ``fixed`` is r1 = r with no narrowing; ``gradual`` defaults to r1 = min(1, 2r).
    """
    out = [-1.0] * n_layers
    if n_layers < 2:
        return out
    if schedule == "fixed":
        out[1] = r
        return out
    if schedule != "gradual":
        raise ValueError(schedule)
    if r1 is None:
        r1 = min(1.0, 2.0 * r)
    out[1] = r1
    for j in range(1, n_narrow + 1):
        if 1 + j < n_layers:
            out[1 + j] = r1 + (r - r1) * j / n_narrow
    return out


# --------------------------------------------------------------------------- blended prefill
def _layout(segments):
    """Offsets of each segment and the cached-token mask of the concatenated prompt."""
    offs, ids, cached = [], [], []
    off = 0
    for seg in segments:
        offs.append(off)
        ids.append(np.asarray(seg.ids))
        cached.append(np.full(len(seg.ids), seg.chunk >= 0))
        off += len(seg.ids)
    return offs, np.concatenate(ids), np.concatenate(cached)


def init_fused_cache(cfg, segments, chunk_caches, storage: str):
    """Fused cache before any recompute: re-rotated cached K, copied V, NaN on query rows."""
    offs, ids, cached = _layout(segments)
    N = len(ids)
    Kf = np.full((cfg.n_layers, N, cfg.n_kv_heads, cfg.head_dim), np.nan)
    Vf = np.full_like(Kf, np.nan)
    for seg, off in zip(segments, offs):
        if seg.chunk < 0:
            continue
        Kc, Vc = chunk_caches[seg.chunk]
        n = len(seg.ids)
        for i in range(cfg.n_layers):
            Kf[i, off:off + n] = round_storage(rerotate_keys(Kc[i], off, cfg.rope_theta), storage)
            Vf[i, off:off + n] = round_storage(Vc[i], storage)
    return Kf, Vf


def blend_prefill(cfg, weights, segments, chunk_caches, ratios: Sequence[float], storage: str = "f64",
                  dev_mode: int = 0, force_sel: Optional[Dict[int, np.ndarray]] = None):
    """CacheBlend's blended prefill over independently cached chunks.

    Steps, in the pages' order ([P3] "어떤 토큰을 다시 계산하는가", per-layer flow; [P1]
    選択的再計算アルゴリズム, HKVD, 段階的フィルタリング, 位置エンコーディングの更新):

    1. concatenate the segments; re-rotate each cached chunk's K by its offset;
    2. layer 0 runs on every token (reading R3);
    3. at each layer i the tokens R_i whose layer input exists (R_i = S_{i-1}) get
       fresh q, k, v; at a check layer (ratio >= 0) the cached ones are ranked by
       deviation against the fused cache and the top k_i kept: S_i = Q u top-k;
       otherwise S_i = R_i;
    4. fresh K/V of S_i overwrite the fused cache (the rest is discarded, R7);
    5. queries of S_i attend causally over the whole fused cache;
    6. output projection and MLP for S_i; their hidden states go to layer i+1.

    ``force_sel`` maps a check layer to the full set S_i to use instead of the top-k.
    Returns the final hidden rows (of the last S), the sets, the deviations of each
    check layer, the fused cache and the first token.
    """
    offs, ids, cached = _layout(segments)
    N = len(ids)
    n_cached = int(cached.sum())
    Kf, Vf = init_fused_cache(cfg, segments, chunk_caches, storage)
    h = np.zeros((N, cfg.d_model))
    h[:] = weights.embed(ids).astype(np.float64)
    R = np.arange(N)
    sets, devs = {}, {}
    for i in range(cfg.n_layers):
        W = weights.layer(i)
        q, k, v = project_qkv(cfg, W, h[R], R)
        r_i = ratios[i]
        if r_i >= 0:
            is_c = cached[R]
            cand = R[is_c]
            dev = kv_deviation(k[is_c], v[is_c], Kf[i][cand], Vf[i][cand], dev_mode)
            dev32 = dev.astype(np.float32)
            devs[i] = (cand.copy(), dev32)
            if force_sel is not None and i in force_sel:
                S = np.asarray(force_sel[i], dtype=np.int64)
            else:
                kk = min(k_for_ratio(r_i, n_cached), len(cand))
                top = select_hkvd(dev32, cand, kk)
                S = np.union1d(top, R[~is_c]).astype(np.int64)
        else:
            S = R
        loc = np.searchsorted(R, S)
        assert np.array_equal(R[loc], S), "selected tokens must have a layer input"
        Kf[i][S] = round_storage(k[loc], storage)
        Vf[i][S] = round_storage(v[loc], storage)
        attn = causal_attention(q[loc], S, Kf[i], Vf[i])
        h[S] = output_and_mlp(cfg, W, h[S], attn)
        sets[i] = S
        R = S
    tok = first_token(cfg, weights, h[N - 1])
    return {"hidden": h[R], "rows": R, "sets": sets, "devs": devs, "k": Kf, "v": Vf,
            "first_token": tok, "n_cached": n_cached}


def full_reuse(cfg, weights, segments, chunk_caches, storage: str = "f64"):
    """Full KV reuse: only the query is computed, over the re-rotated cached KV.

    [P1] 実験結果 / 生成品質の評価 ("Full KV Reuse", no recompute); [P3] comparison table.
    """
    offs, ids, cached = _layout(segments)
    N = len(ids)
    Kf, Vf = init_fused_cache(cfg, segments, chunk_caches, storage)
    Q = np.nonzero(~cached)[0]
    h = weights.embed(ids[Q]).astype(np.float64)
    for i in range(cfg.n_layers):
        W = weights.layer(i)
        q, k, v = project_qkv(cfg, W, h, Q)
        Kf[i][Q] = round_storage(k, storage)
        Vf[i][Q] = round_storage(v, storage)
        attn = causal_attention(q, Q, Kf[i], Vf[i])
        h = output_and_mlp(cfg, W, h, attn)
    return {"hidden": h, "rows": Q, "first_token": first_token(cfg, weights, h[-1])}


def seam_positions(segments, seam_tokens: int) -> np.ndarray:
    """Tokens that spatial seam repair recomputes (reading R18).

    [P2] シーム修復戦略 / SelectiveRecompute: the R tokens just before each chunk
    boundary are encoded again with the whole context.  Every cached segment ends at a
    boundary (with the next chunk, or with the query after the last one), so these are
    the last min(R, n_c) tokens of every cached chunk c, in prompt positions, ascending.
    """
    offs, _, _ = _layout(segments)
    out = []
    for seg, off in zip(segments, offs):
        if seg.chunk < 0:
            continue
        n = len(seg.ids)
        r = min(int(seam_tokens), n)
        out.extend(range(off + n - r, off + n))
    return np.array(sorted(out), dtype=np.int64)


def fixed_set_prefill(cfg, weights, segments, chunk_caches, S, storage: str = "f64"):
    """Prefill over re-rotated chunk caches that recomputes one fixed token set S at every
    layer, layer 0 included (no deviation is measured, so no layer needs other tokens).

    Per layer: q, k, v of S; fresh K/V of S overwrite the fused cache; S attends causally
    over the whole fused cache; output projection and MLP for S.
    """
    offs, ids, cached = _layout(segments)
    N = len(ids)
    Kf, Vf = init_fused_cache(cfg, segments, chunk_caches, storage)
    S = np.asarray(S, dtype=np.int64)
    h = weights.embed(ids[S]).astype(np.float64)
    for i in range(cfg.n_layers):
        W = weights.layer(i)
        q, k, v = project_qkv(cfg, W, h, S)
        Kf[i][S] = round_storage(k, storage)
        Vf[i][S] = round_storage(v, storage)
        attn = causal_attention(q, S, Kf[i], Vf[i])
        h = output_and_mlp(cfg, W, h, attn)
    return {"hidden": h, "rows": S, "k": Kf, "v": Vf, "first_token": first_token(cfg, weights, h[-1])}


def seam_repair_prefill(cfg, weights, segments, chunk_caches, seam_tokens: int, storage: str = "f64"):
    """Spatial seam repair ([P2] SelectiveRecompute): the query and the R tokens before every
    chunk boundary are recomputed at every layer; all other tokens keep their re-rotated
    cached K/V."""
    offs, ids, cached = _layout(segments)
    S = np.union1d(seam_positions(segments, seam_tokens), np.nonzero(~cached)[0]).astype(np.int64)
    return fixed_set_prefill(cfg, weights, segments, chunk_caches, S, storage)


def decode_step(cfg, weights, Kf: np.ndarray, Vf: np.ndarray, n_past: int, token: int, storage: str = "f64"):
    """One greedy decoding step on a fused KV cache ([P3] flow: the response is generated
    from the fused KV; [P1] 実験結果 / スループット: decoding follows the blended prefill).

    The token ``token`` enters at position ``n_past``: per layer its q, k, v are computed
    (RoPE at n_past), its K/V are written to row n_past of the cache (rounded to the storage
    type), its query attends to rows 0..n_past, then output projection and MLP.  Kf, Vf
    [L, capacity, Hkv, dh] are updated in place.  Returns the final hidden state and the
    argmax of the LM head (the next token).
    """
    h = weights.embed(np.asarray([token])).astype(np.float64)
    pos = [int(n_past)]
    for i in range(cfg.n_layers):
        W = weights.layer(i)
        q, k, v = project_qkv(cfg, W, h, pos)
        Kf[i][n_past] = round_storage(k[0], storage)
        Vf[i][n_past] = round_storage(v[0], storage)
        attn = causal_attention(q, pos, Kf[i], Vf[i])
        h = output_and_mlp(cfg, W, h, attn)
    return {"hidden": h[0], "token": first_token(cfg, weights, h[0])}


def greedy_decode(cfg, weights, Kf: np.ndarray, Vf: np.ndarray, n_past: int, token: int, steps: int,
                  storage: str = "f64"):
    """``steps`` decode steps, each feeding the previous step's argmax; returns the tokens."""
    out = []
    for t in range(steps):
        r = decode_step(cfg, weights, Kf, Vf, n_past + t, token, storage)
        token = r["token"]
        out.append(token)
    return out


def precompute_all(cfg, weights, spec, storage: str, chunk_indices=None):
    """Chunk caches for every chunk a workload's requests use."""
    used = sorted({s.chunk for req in spec.requests for s in req if s.chunk >= 0})
    if chunk_indices is not None:
        used = [c for c in used if c in chunk_indices]
    return {c: precompute_chunk(cfg, weights, spec.chunks[c], storage) for c in used}


# --------------------------------------------------------------------------- KV codec
def _minmax_codes(x32: np.ndarray, axis, bits: int):
    """Asymmetric min/max quantisation of float32 values along ``axis`` (reading R21).

    scale = (max - min) / (2**bits - 1), code = clamp(rint((x - min) / scale), 0, 2**bits - 1)
    (code 0 where scale is 0).  Every step is one float32 operation, so the integer codes
    are decided in the precision the kernel uses.
    """
    levels = np.float32(2 ** bits - 1)
    mn = np.min(x32, axis=axis, keepdims=True)
    mx = np.max(x32, axis=axis, keepdims=True)
    scale = (mx - mn) / levels
    diff = x32 - mn
    q = np.zeros_like(x32)
    np.divide(diff, np.broadcast_to(scale, diff.shape), out=q, where=np.broadcast_to(scale > 0, diff.shape))
    codes = np.clip(np.rint(q), 0, float(levels)).astype(np.int64)
    return codes, scale.astype(np.float32), mn.astype(np.float32)


def kv_encode(K: np.ndarray, V: np.ndarray, bits: int) -> Dict[str, np.ndarray]:
    """KIVI-style asymmetric quantisation of a chunk's KV cache ([P2] KV量子化とメモリ管理 /
    非対称量子化: keys per channel, values per token; int8 or int4).

    K, V: [L, n, Hkv, dh] as the cache stores them.  Readings R19, R20: a key channel
    (layer, head, channel) is one group over the chunk's n tokens; a value group is one
    (layer, token, head) row of dh channels.  Returns the integer codes and the float32
    scale and minimum ("zero") of each group.
    """
    if bits not in (4, 8):
        raise ValueError(bits)
    K32 = np.asarray(K, dtype=np.float32)
    V32 = np.asarray(V, dtype=np.float32)
    kc, ks, kz = _minmax_codes(K32, 1, bits)   # over tokens: [L, 1, Hkv, dh]
    vc, vs, vz = _minmax_codes(V32, 3, bits)   # over channels: [L, n, Hkv, 1]
    return {"bits": bits, "k_codes": kc, "k_scale": ks[:, 0], "k_zero": kz[:, 0],
            "v_codes": vc, "v_scale": vs[..., 0], "v_zero": vz[..., 0]}


def kv_decode(enc: Dict[str, np.ndarray]):
    """Dequantised K, V [L, n, Hkv, dh] in float64: zero + code * scale of each group."""
    K = enc["k_zero"][:, None].astype(np.float64) + enc["k_codes"] * enc["k_scale"][:, None].astype(np.float64)
    V = enc["v_zero"][..., None].astype(np.float64) + enc["v_codes"] * enc["v_scale"][..., None].astype(np.float64)
    return K, V


# --------------------------------------------------------------------------- cost model
def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """Per-token KV size 2 * L * Hkv * dh * bytes ([P4] §4, §9-1: Qwen2.5-1.5B 28,672 B)."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes


def t_recompute(ratio: float, t_prefill: float) -> float:
    """[P1] パイプライン化の設計: T_recompute = r% x T_prefill."""
    return ratio * t_prefill


def t_load(n_tokens: int, kv_bytes_token: float, n_layers_loaded: int, n_layers: int, bandwidth: float) -> float:
    """[P1] パイプライン化の設計, T_load = PerTokenKVSize x L / StorageThroughput (reading R8:
    the KV bytes of the request's cached tokens for the layers loaded, over the bandwidth)."""
    return n_tokens * kv_bytes_token * (n_layers_loaded / n_layers) / bandwidth


def pipelined_latency(t_load_layers: Sequence[float], t_rec_layers: Sequence[float]) -> float:
    """[P3] "로딩과 재계산의 시간을 겹친다": T_layer ~ max(T_load, T_recompute), summed over layers."""
    return float(sum(max(a, b) for a, b in zip(t_load_layers, t_rec_layers)))


def break_even_bandwidth(kv_bytes_token: float, prefill_s_per_token: float) -> float:
    """[P4] §5: loading beats recomputing above BW* = KV bytes per token / prefill time per token."""
    return kv_bytes_token / prefill_s_per_token


# --------------------------------------------------------------------------- loading controller
FNV64_OFFSET = 0xCBF29CE484222325
FNV64_PRIME = 0x100000001B3


def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64-bit (Fowler, Noll, Vo): h = offset basis; per byte h = (h xor byte) * prime mod 2^64."""
    h = FNV64_OFFSET
    for b in data:
        h ^= b
        h = (h * FNV64_PRIME) & 0xFFFFFFFFFFFFFFFF
    return h


def chunk_hash(ids: Sequence[int]) -> int:
    """Content key of a chunk (reading R22): FNV-1a 64 of its token ids as little-endian int32 bytes.

    [P3] loading controller: the cache manager finds a chunk's KV by a hash of its text; [P1]
    vLLMとの統合: the hash table lives in CPU memory.  Content only, so the key does not depend
    on where the chunk sits in a prompt.
    """
    return fnv1a64(np.asarray(ids, dtype="<i4").tobytes())


TIER_MISSING, TIER_DEVICE, TIER_HOST = -1, 0, 1
ACT_USE, ACT_LOAD, ACT_RECOMPUTE = 0, 1, 2


def chunk_action(tier: int, n_tokens: int, nbytes: float, link_bytes_per_s: float, link_latency_s: float,
                 prefill_s_per_token: float) -> int:
    """Use, load or recompute one chunk (reading R23).

    [P4] §5 損益分岐: loading n tokens costs n x (KV bytes per token) / bandwidth + a fixed
    latency, recomputing them costs n x (prefill time per token); load only when that is
    cheaper.  A chunk already in device memory is used as it is; a missing one is recomputed.
    """
    if tier == TIER_DEVICE:
        return ACT_USE
    if tier == TIER_MISSING:
        return ACT_RECOMPUTE
    t_load = nbytes / link_bytes_per_s + link_latency_s
    return ACT_LOAD if t_load < n_tokens * prefill_s_per_token else ACT_RECOMPUTE


def plan_loading(model: Dict[str, float], chunks: Sequence[Dict[str, float]], n_query: int):
    """Loading plan of one prompt and the recompute ratio that hides under the load (reading R24).

    [P1] パイプライン化の設計: T_recompute = r% x T_prefill and T_load = KV bytes / storage
    throughput overlap, so a layer costs max(T_load, T_recompute) ([P3] "로딩과 재계산의 시간을
    겹친다").  [P1] 閾値チューニング: raise r on slow storage (the extra recompute hides under the
    load), lower it on fast storage, within the quality bounds [r_min, r_max].  Here
    T_recompute(r) = fixed + r x T_prefill with T_prefill = N x prefill time per token; the
    chosen r is the largest whose recompute still fits under T_load:
    r = clamp((T_load - fixed) / T_prefill, r_min, r_max), r_min when nothing is loaded.
    Returns (actions, r, T_load, T_recompute(r)).
    """
    actions = [chunk_action(c["tier"], c["n_tokens"], c["bytes"], model["link_bytes_per_s"],
                            model["link_latency_s"], model["prefill_s_per_token"]) for c in chunks]
    t_load = sum(c["bytes"] / model["link_bytes_per_s"] + model["link_latency_s"]
                 for c, a in zip(chunks, actions) if a == ACT_LOAD)
    n_total = sum(c["n_tokens"] for c in chunks) + n_query
    t_prefill = n_total * model["prefill_s_per_token"]
    if t_load <= 0 or t_prefill <= 0:
        r = model["r_min"]
    else:
        r = min(model["r_max"], max(model["r_min"], (t_load - model["recompute_fixed_s"]) / t_prefill))
    return actions, r, t_load, model["recompute_fixed_s"] + r * t_prefill
