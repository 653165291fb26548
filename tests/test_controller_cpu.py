"""The loading controller's host code in the library against the oracle (no GPU needed):
content keys bit for bit, and per-chunk actions, ratio, T_load and T_recompute on random
prompts, including the degenerate ones (no chunk, nothing loaded, everything clamped)."""
import numpy as np
import pytest

import harness as hz
import oracle.cacheblend as orc
import rag_non_prefix_gb300 as cb


def test_chunk_hash_matches_oracle():
    for i, n in enumerate([0, 1, 2, 7, 128, 512, 4099]):
        ids = hz.gen_token_ids(hz.stream_key(41, i), n, 64000, "zipf")
        assert cb.cb_chunk_hash(ids) == orc.chunk_hash(ids), n
    extreme = [0, -1, 2 ** 31 - 1, -2 ** 31, 255, 256]
    assert cb.cb_chunk_hash(extreme) == orc.chunk_hash(extreme)


def _random_prompt(rng, n_chunks):
    tiers = rng.choice([orc.TIER_DEVICE, orc.TIER_HOST, orc.TIER_MISSING], n_chunks, p=[0.3, 0.6, 0.1])
    chunks = []
    for t in tiers:
        n = int(rng.integers(16, 1024))
        chunks.append({"tier": int(t), "n_tokens": n, "bytes": float(n * rng.choice([28672, 131072, 4096 * 2 * 2]))})
    return chunks


@pytest.mark.parametrize("seed", range(40))
def test_plan_loading_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    model = {"link_bytes_per_s": float(10 ** rng.uniform(8, 12)), "link_latency_s": float(rng.choice([0.0, 1e-4, 2e-3])),
             "prefill_s_per_token": float(10 ** rng.uniform(-6, -4)), "recompute_fixed_s": float(rng.uniform(0, 5e-3)),
             "r_min": 0.05, "r_max": float(rng.choice([0.2, 0.5, 1.0]))}
    chunks = _random_prompt(rng, int(rng.integers(0, 40)))
    n_q = int(rng.integers(0, 200))
    got = cb.cb_plan_loading(model, chunks, n_q)
    ref = orc.plan_loading(model, chunks, n_q)
    assert got[0] == ref[0]
    for a, b in zip(got[1:], ref[1:]):
        assert a == pytest.approx(b, rel=1e-12, abs=1e-15)


def test_plan_loading_rejects_bad_models():
    good = {"link_bytes_per_s": 1e10, "link_latency_s": 0.0, "prefill_s_per_token": 1e-5, "recompute_fixed_s": 0.0,
            "r_min": 0.05, "r_max": 0.2}
    for key, bad in (("link_bytes_per_s", 0.0), ("prefill_s_per_token", -1.0), ("r_max", 0.01), ("r_max", 1.5),
                     ("link_latency_s", -1.0)):
        with pytest.raises(cb.CacheBlendError) as e:
            cb.cb_plan_loading(dict(good, **{key: bad}), [], 1)
        assert e.value.name == "CB_ERR_INVALID_ARG"
    with pytest.raises(cb.CacheBlendError):
        cb.cb_plan_loading(good, [{"tier": 7, "n_tokens": 3, "bytes": 1.0}], 1)
