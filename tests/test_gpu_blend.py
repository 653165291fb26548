"""End-to-end parity of the blended prefill (CUDA path through the C ABI vs the oracle)."""
import numpy as np
import pytest
import torch

import harness as hz
import harness.device as hd
import oracle.cacheblend as orc
import rag_non_prefix_gb300 as cb
from tests._gpu import GpuWorkload, OracleWorkload, forced_from_oracle, max_rel_err, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


def tol(cfg):
    return TOL[cfg.dtype]


@pytest.fixture(scope="module")
def tiny():
    spec = hz.workload("tiny")
    return spec, GpuWorkload(spec), OracleWorkload(spec)


@pytest.fixture(scope="module")
def small_bf16():
    spec = hz.workload("small_bf16")
    return spec, GpuWorkload(spec), OracleWorkload(spec)


def _sets(req, cfg):
    sel, cnt = req["sel"].cpu().numpy(), req["sel_count"].cpu().numpy()
    return {i: sel[i, : cnt[i]] for i in range(cfg.n_layers)}


# ----------------------------------------------------------------------------- chunk precompute / full prefill
@pytest.mark.parametrize("name", ["tiny", "small_gqa_f32", "small_bf16", "small_mha_bf16"])
def test_precompute_and_full_prefill_match_oracle(name):
    spec = hz.workload(name)
    g = GpuWorkload(spec)
    o = OracleWorkload(spec)
    t = tol(spec.cfg)
    for c, (ids, k, v) in g.chunk_kv.items():
        ok, ov = o.caches[c]
        for got, ref in ((to_np(k), ok), (to_np(v), ov)):
            err = np.max(np.abs(got - ref), axis=(2, 3)).max() / np.max(np.abs(ref))
            assert err < t, (c, err)
    ids = np.concatenate([s.ids for s in spec.requests[0]])
    full = g.eng.full_prefill(hd.ids_tensor(ids))
    torch.cuda.synchronize()
    ref = o.full(0)
    assert max_rel_err(to_np(full["hidden"]), ref["hidden"]) < t
    if spec.cfg.dtype == "f32":
        assert int(full["first_token"].item()) == ref["first_token"]


# ----------------------------------------------------------------------------- blend, fp32 (configuration 1)
def test_tiny_blend_matches_oracle(tiny):
    spec, g, o = tiny
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    req = g.blend(ratios)[0]
    ref = o.blend(0, ratios)
    sets = _sets(req, cfg)
    for i in range(cfg.n_layers):
        assert np.array_equal(sets[i], ref["sets"][i]), i
    rows = ref["rows"]
    got = to_np(req["hidden"])[rows]
    assert max_rel_err(got, ref["hidden"]) < 1e-4
    assert int(req["first_token"].item()) == ref["first_token"]
    assert len(rows) == 32 + 39


@pytest.mark.parametrize("schedule,r", [("gradual", 0.2), ("fixed", 0.5)])
def test_gqa_f32_blend_matches_oracle(schedule, r):
    spec = hz.workload("small_gqa_f32")
    g, o = GpuWorkload(spec), OracleWorkload(spec)
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, r, schedule)
    req = g.blend(ratios)[0]
    ref = o.blend(0, ratios)
    sets = _sets(req, cfg)
    for i in range(cfg.n_layers):
        assert np.array_equal(sets[i], ref["sets"][i]), i
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < 1e-4


# ----------------------------------------------------------------------------- blend, bf16
@pytest.mark.parametrize("orientation", [0, 1, 2], ids=["model", "token-rows", "weight-rows"])
def test_bf16_blend_forced_selection_matches_oracle(small_bf16, orientation):
    """Numerics alone: the GPU follows the oracle's sets (under each GEMM tile orientation:
    the q|k|v weights split along the output features, SwiGLU, residual add)."""
    cb.cb_gemm_set_orientation(orientation)
    try:
        _forced_bf16(small_bf16)
    finally:
        cb.cb_gemm_set_orientation(0)


@pytest.mark.parametrize("pairing", [2, 4], ids=["pairs", "two-pairs"])
def test_bf16_blend_on_cta_pairs_matches_oracle(small_bf16, pairing):
    """Numerics with every projection on CTA pairs (q|k|v across three weight tensors,
    output projection and down projection with the residual add, SwiGLU)."""
    cb.cb_gemm_set_pairing(pairing)
    try:
        _forced_bf16(small_bf16)
    finally:
        cb.cb_gemm_set_pairing(0)


@pytest.mark.parametrize("tiles", [1, 2], ids=["one-tile", "two-tiles"])
def test_bf16_blend_attention_kernels_match_oracle(small_bf16, tiles):
    """Numerics with each attention kernel forced (one or two query tiles per CTA)."""
    cb.cb_attention_set_tiles(tiles)
    try:
        _forced_bf16(small_bf16)
    finally:
        cb.cb_attention_set_tiles(0)


def _forced_bf16(small_bf16):
    spec, g, o = small_bf16
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    ref = o.blend(0, ratios)
    forced = forced_from_oracle(ref, ref["n_cached"], cfg.n_layers, ratios)
    req = g.blend(ratios, forced=forced)[0]
    sets = _sets(req, cfg)
    for i in range(cfg.n_layers):
        assert np.array_equal(sets[i], ref["sets"][i])
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < 2e-2


@pytest.mark.parametrize("name,schedule,pairing,tile", [("small_bf16", "gradual", 2, 0), ("small_mha_bf16", "fixed", 2, 0),
                                                      ("small_bf16", "gradual", 4, 192)],
                         ids=["gqa-pairs", "mha-pairs-fixed", "gqa-two-pair-clusters-pad-tile"])
def test_bf16_blend_fused_qkv_matches_separate_kernels(name, schedule, pairing, tile):
    """The layers without a check run Q/K/V, RoPE and the K/V scatter in the paired GEMM's
    epilogue; with the paired GEMM forced in both runs, the blend's sets, hidden rows and first
    token are bit for bit those of the projection followed by the post-QKV kernel (the same
    sums, the same rotation arithmetic, the same roundings).  The fixed schedule checks only
    layer 1, so every other layer takes the fused path; clusters of two pairs with 192-token
    tiles give layer 0's 552 rows three token tiles, the second pair of the last cluster unit a
    tile past the rows (nothing stored)."""
    spec = hz.workload(name)
    if schedule != spec.schedule:
        spec = hz.make_prompt(name, 12, [96, 128], 24, spec.ratio, schedule, "zipf", name=name + "_fixed")
    g = GpuWorkload(spec)
    cfg = spec.cfg
    ratios = [float(x) for x in orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)]
    outs = []
    cb.cb_gemm_set_pairing(pairing)
    cb.cb_gemm_set_orientation(tile)
    try:
        for fused in (True, False):
            cb.cb_set_qkv_fusion(fused)
            req = g.blend(ratios)[0]
            torch.cuda.synchronize()
            outs.append((to_np(req["hidden"]).copy(), _sets(req, cfg), int(req["first_token"].item())))
    finally:
        cb.cb_set_qkv_fusion(True)
        cb.cb_gemm_set_pairing(0)
        cb.cb_gemm_set_orientation(0)
    (h1, s1, t1), (h2, s2, t2) = outs
    assert np.array_equal(h1, h2)
    assert t1 == t2
    for i in range(cfg.n_layers):
        assert np.array_equal(s1[i], s2[i])


def test_bf16_blend_long_context_matches_oracle_and_repeats():
    """A 2176-token prompt on the reduced bf16 model: tiles reach 17 key blocks, so the
    attention of every layer splits its long tiles into two key ranges merged on the device.
    The GPU follows the oracle's sets and agrees with its hidden rows, and two runs agree bit
    for bit (the merge adds the two ranges in a fixed order)."""
    spec = hz.make_prompt("small_bf16", 31, [512] * 4, 32, 0.15, "gradual", "zipf", prefix_len=64, name="long")
    g, o = GpuWorkload(spec), OracleWorkload(spec)
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    ref = o.blend(0, ratios)
    forced = forced_from_oracle(ref, ref["n_cached"], cfg.n_layers, ratios)
    outs = []
    for _ in range(2):
        req = g.blend(ratios, forced=forced)[0]
        torch.cuda.synchronize()
        sets = _sets(req, cfg)
        for i in range(cfg.n_layers):
            assert np.array_equal(sets[i], ref["sets"][i])
        outs.append(to_np(req["hidden"])[ref["rows"]].copy())
    assert max_rel_err(outs[0], ref["hidden"]) < 2e-2
    assert np.array_equal(outs[0], outs[1])


def test_bf16_blend_selection_overlap(small_bf16):
    """Free-running selection: >= 99 % overlap of every checked set with the oracle's."""
    spec, g, o = small_bf16
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    ref = o.blend(0, ratios)
    req = g.blend(ratios)[0]
    sets = _sets(req, cfg)
    for i in range(cfg.n_layers):
        inter = len(np.intersect1d(sets[i], ref["sets"][i]))
        assert len(sets[i]) == len(ref["sets"][i])
        assert inter / len(ref["sets"][i]) >= 0.99, (i, inter, len(ref["sets"][i]))
    common = np.intersect1d(sets[cfg.n_layers - 1], ref["rows"])
    got = to_np(req["hidden"])[common]
    refh = ref["hidden"][np.searchsorted(ref["rows"], common)]
    assert max_rel_err(got, refh) < 2e-2


def test_mha_bf16_blend_forced(tmp_path):
    spec = hz.workload("small_mha_bf16")
    g, o = GpuWorkload(spec), OracleWorkload(spec)
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    ref = o.blend(0, ratios)
    req = g.blend(ratios, forced=forced_from_oracle(ref, ref["n_cached"], cfg.n_layers, ratios))[0]
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < 2e-2


# ----------------------------------------------------------------------------- selection variants
def test_cosine_deviation_blend(tiny):
    """dev_mode 3 (cosine): the checked sets overlap the oracle's, and under the oracle's
    sets the hidden states agree to fp32 rounding."""
    spec, g, o = tiny
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    ref = o.blend(0, ratios, dev_mode=3)
    req = g.blend(ratios, dev_mode=3)[0]
    sets = _sets(req, cfg)
    for i in range(cfg.n_layers):
        assert len(sets[i]) == len(ref["sets"][i])
        assert len(np.intersect1d(sets[i], ref["sets"][i])) / len(ref["sets"][i]) >= 0.97, i
    l2 = o.blend(0, ratios, dev_mode=0)
    assert not np.array_equal(l2["sets"][1], ref["sets"][1])  # the mode changes the choice
    forced = forced_from_oracle(ref, ref["n_cached"], cfg.n_layers, ratios)
    req = g.blend(ratios, forced=forced, dev_mode=3)[0]
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < 1e-4


@pytest.mark.parametrize("name,R", [("tiny", 16), ("tiny", 0), ("small_bf16", 16), ("small_bf16", 200)])
def test_seam_repair_matches_oracle(name, R):
    """Spatial seam repair: the same fixed set at every layer (layer 0 included) as the
    oracle's, and hidden states within the dtype's tolerance; R = 0 is full KV reuse and
    an R above every chunk length recomputes everything."""
    spec = hz.workload(name)
    g, o = GpuWorkload(spec), OracleWorkload(spec)
    cfg = spec.cfg
    ref = o.seam(0, R)
    req = g.blend(None, seam_tokens=R)[0]
    sets = _sets(req, cfg)
    for i in range(cfg.n_layers):
        assert np.array_equal(sets[i], ref["rows"]), i
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < tol(cfg)
    if cfg.dtype == "f32":
        assert int(req["first_token"].item()) == ref["first_token"]
    N = spec.n_tokens(0)
    if R == 0:
        assert len(ref["rows"]) == N - spec.n_cached(0)
    if R >= max(len(c) for c in spec.chunks):
        assert len(ref["rows"]) == N


# ----------------------------------------------------------------------------- special cases
def test_full_recompute_equals_full_prefill_on_gpu(small_bf16):
    """r = 100 %: the blend recomputes everything, which is the GPU's own full prefill."""
    spec, g, o = small_bf16
    cfg = spec.cfg
    req = g.blend(orc.ratio_schedule(cfg.n_layers, 1.0, "fixed"))[0]
    ids = np.concatenate([s.ids for s in spec.requests[0]])
    full = g.eng.full_prefill(hd.ids_tensor(ids))
    torch.cuda.synchronize()
    a, b = to_np(req["hidden"]), to_np(full["hidden"])
    assert max_rel_err(a, b) < 1e-2
    assert int(req["first_token"].item()) == int(full["first_token"].item())


def test_zero_ratio_equals_full_reuse_oracle(tiny):
    spec, g, o = tiny
    cfg = spec.cfg
    req = g.blend(orc.ratio_schedule(cfg.n_layers, 0.0, "fixed"))[0]
    ref = orc.full_reuse(cfg, o.W, spec.requests[0], o.caches, "f32")
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < 1e-4


def test_host_staged_chunks_are_bit_identical(small_bf16):
    spec, g, o = small_bf16
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    resident = g.blend(ratios)[0]
    gh = GpuWorkload(spec, on_host=True)
    cs = torch.cuda.Stream()
    staged = gh.blend(ratios, copy_stream=cs)[0]
    assert torch.equal(resident["hidden"], staged["hidden"])
    assert torch.equal(resident["fused_k"], staged["fused_k"])
    assert torch.equal(resident["sel"], staged["sel"])


def test_layer_profile_of_a_staged_blend(small_bf16):
    """Per-layer events (profiling level 2): every layer of a host-staged blend has staging
    copies on the copy stream and compute on the compute stream; a resident blend stages
    nothing; phase events alone (level 1) record no layer; the profile drains on reading."""
    spec, g, o = small_bf16
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    gh = GpuWorkload(spec, on_host=True)
    cs = torch.cuda.Stream()
    for level, staged in ((2, True), (2, False), (1, True)):
        eng = gh if staged else g
        eng.eng.get_layer_profile()
        eng.eng.set_profiling(level)
        out = eng.blend(ratios, copy_stream=cs if staged else None)[0]
        lay = eng.eng.get_layer_profile()
        eng.eng.set_profiling(0)
        eng.eng.get_profile()
        if level == 1:
            assert max(lay["load_ms"]) == 0 and max(lay["compute_ms"]) == 0
            continue
        assert all(x > 0 for x in lay["compute_ms"]), lay
        if staged:
            assert all(x > 0 for x in lay["load_ms"]), lay
        else:
            assert max(lay["load_ms"]) == 0
        assert eng.eng.get_layer_profile()["compute_ms"] == [0.0] * cfg.n_layers
        assert out["sel_count"].cpu().tolist() == g.eng.plan_counts(0)


def test_per_layer_api_matches_whole_call(small_bf16):
    spec, g, o = small_bf16
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    whole = g.blend(ratios)[0]
    reqs = g.requests()
    g.eng.blend_begin(reqs, ratios)
    for i in range(cfg.n_layers):
        g.eng.blend_layer(i)
    g.eng.blend_finish()
    g.eng.get_status()
    torch.cuda.synchronize()
    assert torch.equal(whole["hidden"], reqs[0]["hidden"])
    assert g.eng.plan_counts(0) == whole["sel_count"].cpu().tolist()


def test_batched_requests_match_single():
    """Two requests sharing chunks (a pooled batch) give the same result as one at a time."""
    base = hz.make_pooled_batch("small_bf16", 21, 6, 96, 3, 2, 24, 0.2, name="pool")
    g = GpuWorkload(base)
    cfg = base.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, base.ratio, base.schedule)
    both = g.blend(ratios)
    for r in range(2):
        req = base.requests[r]
        one = g.eng.make_request([s.chunk for s in req if s.chunk >= 0], hd.ids_tensor(req[-1].ids))
        g.eng.blend_prefill([one], ratios)
        torch.cuda.synchronize()
        assert max_rel_err(to_np(one["hidden"])[to_np(one["sel"])[-1][: int(one["sel_count"][-1])].astype(int)],
                           to_np(both[r]["hidden"])[to_np(both[r]["sel"])[-1][: int(both[r]["sel_count"][-1])].astype(int)]) < 1e-2


# ----------------------------------------------------------------------------- errors and waits
def test_errors_are_reported_not_raised_on_device(tiny):
    spec, g, o = tiny
    cfg = spec.cfg
    eng = g.eng
    bad = eng.make_request([0, 1], hd.ids_tensor(spec.requests[0][-1].ids))
    bad["chunk_ids"] = [0, 12345]
    with pytest.raises(cb.CacheBlendError) as e:
        eng.blend_prefill([bad], orc.ratio_schedule(cfg.n_layers, 0.15, "fixed"))
    assert e.value.name == "CB_ERR_NOT_FOUND"
    # a NaN in a cached chunk reaches the deviation: the call reports CB_ERR_NAN, no trap
    ids, k, v = g.chunk_kv[1]
    k2 = k.clone()
    k2[1, 5] = float("nan")
    eng.register_chunk(99, ids, k2, v)
    req = eng.make_request([0, 99], hd.ids_tensor(spec.requests[0][-1].ids))
    eng.blend_prefill([req], orc.ratio_schedule(cfg.n_layers, 0.15, "fixed"))
    with pytest.raises(cb.CacheBlendError) as e:
        eng.get_status()
    assert e.value.name == "CB_ERR_NAN"
    eng.unregister_chunk(99)
    eng.get_status()  # cleared


def test_synchronize_deadline_on_a_stalled_copy_stream(small_bf16):
    spec, g, o = small_bf16
    gh = GpuWorkload(spec, on_host=True)
    cfg = spec.cfg
    cs = torch.cuda.Stream()
    reqs = gh.requests()
    gh.eng.blend_begin(reqs, orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule))
    with torch.cuda.stream(cs):
        torch.cuda._sleep(int(2e9))  # about a second of spinning on the copy stream (bounded)
    gh.eng.fetch_kv(0, cs)
    with pytest.raises(cb.CacheBlendError) as e:
        gh.eng.synchronize(0, timeout_ms=1)
    assert e.value.name == "CB_ERR_TIMEOUT"
    gh.eng.synchronize(0, timeout_ms=30000)
    for i in range(1, cfg.n_layers):
        gh.eng.fetch_kv(i, cs)
    for i in range(cfg.n_layers):
        gh.eng.prefill_layer(i)
    gh.eng.blend_finish()
    gh.eng.get_status()
    torch.cuda.synchronize()


# ----------------------------------------------------------------------------- degenerate prompts
def _custom(model, seed, lens, qlen, ratio=0.2, schedule="gradual"):
    return hz.make_prompt(model, seed, lens, qlen, ratio, schedule, "uniform", name=f"edge{seed}")


@pytest.mark.parametrize("model", ["tiny", "small_bf16"])
def test_prompt_without_chunks_is_a_full_prefill(model):
    """No cached chunk: every token is query, recomputed at every layer; the blend is the
    full prefill of the query (the oracle's blend with Nc = 0 is checked too)."""
    spec = _custom(model, 41, [], 37)
    g, o = GpuWorkload(spec), OracleWorkload(spec)
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, 0.2, "gradual")
    req = g.blend(ratios)[0]
    ref = o.blend(0, ratios)
    full = o.full(0)
    assert np.array_equal(ref["rows"], np.arange(37))
    assert np.max(np.abs(ref["hidden"] - full["hidden"])) < 1e-9 * max(1.0, np.max(np.abs(full["hidden"])))
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < tol(cfg)
    sel, cnt = req["sel"].cpu().numpy(), req["sel_count"].cpu().numpy()
    assert all(cnt[i] == 37 and np.array_equal(sel[i, :37], np.arange(37)) for i in range(cfg.n_layers))


@pytest.mark.parametrize("model", ["tiny", "small_bf16"])
def test_one_token_chunks_and_a_one_token_query(model):
    """Chunks of one token (re-rotation rows of one, deviation of single rows) and a query of
    one token: the sets and hidden states follow the oracle."""
    spec = _custom(model, 42, [1, 1, 5, 1, 130], 1, ratio=0.5)
    g, o = GpuWorkload(spec), OracleWorkload(spec)
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, 0.5, "gradual")
    ref = o.blend(0, ratios)
    forced = forced_from_oracle(ref, ref["n_cached"], cfg.n_layers, ratios)
    req = g.blend(ratios, forced=forced)[0]
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < tol(cfg)
    if cfg.dtype == "f32":
        free = g.blend(ratios)[0]
        sel, cnt = free["sel"].cpu().numpy(), free["sel_count"].cpu().numpy()
        for i in range(cfg.n_layers):
            assert np.array_equal(sel[i, : cnt[i]], ref["sets"][i]), i


def test_prompt_at_max_positions():
    """The longest prompt the rotary table allows (N = max_positions) blends; one more token is
    refused before anything runs."""
    import rag_non_prefix_gb300 as cb_

    spec = _custom("small_bf16", 43, [200, 111], 9)
    N = spec.n_tokens(0)
    g = GpuWorkload(spec, max_tokens=N)
    # GpuWorkload sizes max_positions to N + 1: an engine with max_positions = N exactly
    eng = cb_.Engine(spec.cfg, g.W, max_tokens=N, max_requests=1, max_positions=N)
    for c, (ids, k, v) in g.chunk_kv.items():
        eng.register_chunk(c, ids, k, v)
    q = hd.ids_tensor(spec.requests[0][-1].ids)
    r = eng.make_request([0, 1], q)
    eng.blend_prefill([r], orc.ratio_schedule(spec.cfg.n_layers, 0.2, "gradual"))
    eng.get_status()
    torch.cuda.synchronize()
    assert int(r["first_token"].item()) >= 0
    longer = eng.make_request([0, 1], hd.ids_tensor(np.concatenate([spec.requests[0][-1].ids, [3]])))
    with pytest.raises(cb_.CacheBlendError) as e:
        eng.blend_prefill([longer], orc.ratio_schedule(spec.cfg.n_layers, 0.2, "gradual"))
    assert e.value.name in ("CB_ERR_SHAPE", "CB_ERR_WORKSPACE")
