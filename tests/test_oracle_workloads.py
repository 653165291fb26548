"""The oracle on the named workloads that it finishes in seconds (no GPU)."""
import numpy as np

import harness as hz
import oracle.cacheblend as orc


def test_tiny_workload_blend_and_baselines():
    spec = hz.workload("tiny")
    cfg = spec.cfg
    W = hz.HostWeights(cfg, spec.seed)
    caches = orc.precompute_all(cfg, W, spec, "f32")
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    b = orc.blend_prefill(cfg, W, spec.requests[0], caches, ratios, "f32")
    assert b["n_cached"] == 256 and len(b["rows"]) == 39 + 32
    f = orc.full_prefill(cfg, W, np.concatenate([s.ids for s in spec.requests[0]]), "f32")
    u = orc.full_reuse(cfg, W, spec.requests[0], caches, "f32")
    # the blend sits between full reuse and full prefill on the query rows
    q = slice(len(b["rows"]) - 32, None)
    err_blend = np.abs(b["hidden"][q] - f["hidden"][256:]).max()
    err_reuse = np.abs(u["hidden"] - f["hidden"][256:]).max()
    assert err_blend < err_reuse


def test_harness_is_deterministic_and_shaped():
    a = hz.workload("mistral7b")
    b = hz.workload("mistral7b")
    assert a.n_tokens() == 3200 and a.n_cached() == 3136
    for sa, sb in zip(a.requests[0], b.requests[0]):
        assert np.array_equal(sa.ids, sb.ids)
    w1 = hz.gen_weight_fp32(hz.layer_weight_key(2, 3, 1), 1000, 5000)
    w2 = hz.gen_weight_fp32(hz.layer_weight_key(2, 3, 1), 0, 6000)[1000:]
    assert np.array_equal(w1, w2)
    assert abs(float(np.std(hz.gen_weight_fp32(7, 0, 200000))) - 0.02) < 2e-4
    p = hz.workload("llama70b")
    assert len(p.requests) == 4 and all(len({s.chunk for s in r if s.chunk >= 0}) == 32 for r in p.requests)
    assert all(hz.workload(n).n_tokens() for n in ("llama7b", "yi34b"))
