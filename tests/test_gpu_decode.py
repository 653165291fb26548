"""Decode on the fused cache (CUDA path through the C ABI) against the oracle's decode step.

The oracle decodes from the GPU's own cache (copied to the host) and is fed the GPU's tokens,
so each step's numerics are compared on identical inputs; the argmax is compared wherever the
oracle's top two logits are further apart than the dtype's error."""
import numpy as np
import pytest
import torch

import harness as hz
import harness.device as hd
import oracle.cacheblend as orc
from tests._gpu import GpuWorkload, OracleWorkload, built, max_rel_err, storage_of, to_np

pytestmark = pytest.mark.gpu

TOL = {"f32": 1e-4, "bf16": 2e-2}


@pytest.fixture(scope="module", autouse=True)
def _build():
    built()


def _margin(cfg, W, h):
    x = orc.rms_norm(np.asarray(h, np.float64)[None, :], cfg.rms_eps)[0]
    logits = np.sort(W.lm_head().astype(np.float64) @ x)
    return logits[-1] - logits[-2], float(np.max(np.abs(logits)))


def _oracle_cache(req, cfg):
    return to_np(req["fused_k"]).copy(), to_np(req["fused_v"]).copy()


def _check_steps(g, o, reqs, steps):
    """Greedy decode of ``steps`` tokens for every request on the GPU and, request by request,
    in the oracle from the GPU's post-blend cache with the GPU's tokens as inputs."""
    cfg = g.cfg
    n = len(reqs)
    caches = [_oracle_cache(r, cfg) for r in reqs]
    tok = torch.cat([r["first_token"] for r in reqs]).to(torch.int32)
    hid = torch.zeros((n, cfg.d_model), dtype=torch.float32, device="cuda")
    fed = [[int(x) for x in tok.cpu()]]
    got_h, got_t = [], []
    for _ in range(steps):
        tok = g.eng.decode_step(reqs, tok, out_hidden=hid)
        torch.cuda.synchronize()
        got_h.append(to_np(hid).copy())
        got_t.append([int(x) for x in tok.cpu()])
        fed.append(got_t[-1])
    g.eng.get_status()
    t = TOL[cfg.dtype]
    for i, r in enumerate(reqs):
        K, V = caches[i]
        for s in range(steps):
            st = orc.decode_step(cfg, o.W, K, V, r["n_tokens"] + s, fed[s][i], storage_of(cfg))
            err = max_rel_err(got_h[s][i][None, :], st["hidden"][None, :])
            assert err < t, (i, s, err)
            gap, scale = _margin(cfg, o.W, st["hidden"])
            if gap > 4 * t * scale:
                assert got_t[s][i] == st["token"], (i, s)
    return got_t


@pytest.mark.parametrize("name", ["tiny", "small_bf16", "small_gqa_f32"])
def test_decode_after_blend_matches_oracle(name):
    """Four greedy steps after a blend (split key ranges at these lengths)."""
    spec = hz.workload(name)
    g, o = GpuWorkload(spec, extra_positions=8), OracleWorkload(spec)
    cfg = spec.cfg
    req = spec.requests[0]
    r = g.eng.make_request([s.chunk for s in req if s.chunk >= 0], hd.ids_tensor(req[-1].ids), decode_room=4)
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    g.eng.blend_prefill([r], ratios)
    g.eng.get_status()
    torch.cuda.synchronize()
    _check_steps(g, o, [r], 4)


def test_decode_after_short_prefill_equals_longer_prefill():
    """One key range (a 20-token context): decoding ids[-1] after a full prefill of ids[:-1]
    gives the last hidden row of the GPU's full prefill of ids, to fp32 rounding."""
    spec = hz.workload("tiny")
    g = GpuWorkload(spec)
    cfg = spec.cfg
    ids = hz.gen_token_ids(hz.stream_key(77, 1), 21, cfg.vocab, "uniform")
    short = g.eng.full_prefill(hd.ids_tensor(ids[:-1]), want_kv=True)
    cap = 24
    K = torch.zeros((cfg.n_layers, cap, cfg.n_kv_heads, cfg.head_dim), dtype=short["k"].dtype, device="cuda")
    V = torch.zeros_like(K)
    K[:, :20], V[:, :20] = short["k"], short["v"]
    r = {"fused_k": K, "fused_v": V, "kv_capacity": cap, "n_tokens": 20}
    hid = torch.zeros((1, cfg.d_model), dtype=torch.float32, device="cuda")
    tok = g.eng.decode_step([r], hd.ids_tensor(ids[-1:]), out_hidden=hid)
    full = g.eng.full_prefill(hd.ids_tensor(ids), want_kv=True)
    torch.cuda.synchronize()
    assert max_rel_err(to_np(hid), to_np(full["hidden"])[-1:]) < 1e-4
    assert int(tok.item()) == int(full["first_token"].item())
    assert max_rel_err(to_np(K[:, 20]).reshape(cfg.n_layers, -1), to_np(full["k"][:, 20]).reshape(cfg.n_layers, -1)) < 1e-4


def test_batched_decode_matches_oracle_per_request():
    """Two requests of a pooled batch decode together (one GEMM per weight, one attention
    launch); each follows the oracle on its own cache."""
    base = hz.make_pooled_batch("small_bf16", 21, 6, 96, 3, 2, 24, 0.2, name="pool")
    g, o = GpuWorkload(base, extra_positions=8), OracleWorkload(base)
    cfg = base.cfg
    reqs = [g.eng.make_request([s.chunk for s in rq if s.chunk >= 0], hd.ids_tensor(rq[-1].ids), decode_room=3)
            for rq in base.requests]
    g.eng.blend_prefill(reqs, orc.ratio_schedule(cfg.n_layers, base.ratio, base.schedule))
    g.eng.get_status()
    torch.cuda.synchronize()
    _check_steps(g, o, reqs, 3)


def test_decode_rejects_a_full_cache():
    import rag_non_prefix_gb300 as cb

    spec = hz.workload("tiny")
    g = GpuWorkload(spec, extra_positions=8)
    req = spec.requests[0]
    r = g.eng.make_request([s.chunk for s in req if s.chunk >= 0], hd.ids_tensor(req[-1].ids), decode_room=1)
    g.eng.blend_prefill([r], orc.ratio_schedule(spec.cfg.n_layers, spec.ratio, spec.schedule))
    tok = g.eng.decode_step([r], r["first_token"])
    with pytest.raises(cb.CacheBlendError) as e:
        g.eng.decode_step([r], tok)
    assert e.value.name == "CB_ERR_SHAPE"
    g.eng.get_status()
