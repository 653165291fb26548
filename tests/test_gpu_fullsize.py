"""Parity at the full sizes the bench runs (Mistral-7B-shaped workload, bench launch
configuration): per-kernel checks on sampled outputs the oracle computes one by one, and
end-to-end properties that hold at any size."""
import numpy as np
import pytest
import torch

import harness as hz
import harness.device as hd
import oracle.cacheblend as orc
import rag_non_prefix_gb300 as cb
from tests._gpu import GpuWorkload, built, max_rel_err, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    built()


@pytest.mark.parametrize("M,N,K,mode", [
    (535, 6144, 4096, 0),   # q|k|v of a 15 % layer
    (3200, 6144, 4096, 0),  # layer 0 / check layer
    (535, 4096, 4096, 1),           # output projection + residual
    (535, 28672, 4096, 2),          # gate/up + SiLU-mul
    (535, 4096, 14336, 1),          # down projection + residual
    (884, 57344, 8192, 2),          # Llama-70B-shaped gate/up, 820 + 64 rows
])
def test_gemm_full_size_sampled_rows(M, N, K, mode):
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    rows = np.unique(np.concatenate([[0, 1, M - 1], np.random.default_rng(M).choice(M, 13)]))
    if mode == 2:
        G = (torch.randn(N // 2, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        U = (torch.randn(N // 2, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        C = torch.empty(M, N // 2, dtype=torch.bfloat16, device="cuda")
        cb.cb_gemm(A, G, C, 2, B2=U, scratch=cb.gemm_scratch())
        a = to_np(A[rows])
        ref = orc.silu(a @ to_np(G).T) * (a @ to_np(U).T)
        tol = 2 ** -7
    else:
        B = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        C0 = torch.randn(M, N, device="cuda", generator=g)
        C = C0.clone()
        cb.cb_gemm(A, B, C, mode, scratch=cb.gemm_scratch())
        ref = to_np(A[rows]) @ to_np(B).T + (to_np(C0[rows]) if mode == 1 else 0)
        tol = 1e-4
    torch.cuda.synchronize()
    got = to_np(C[rows])
    assert np.max(np.abs(got - ref)) <= tol * np.max(np.abs(ref)) + 1e-5


@pytest.fixture(scope="module")
def mistral():
    return GpuWorkload(hz.workload("mistral7b"))


def _sets(req, L):
    sel, cnt = req["sel"].cpu().numpy(), req["sel_count"].cpu().numpy()
    return [sel[i, : cnt[i]] for i in range(L)]


def test_mistral7b_blend_properties(mistral):
    spec, g = mistral.spec, mistral
    cfg = spec.cfg
    ratios = cb.ratio_schedule(cfg.n_layers, 0.15, "gradual")
    req = g.blend(ratios)[0]
    N, Nc, Q = spec.n_tokens(), spec.n_cached(), spec.n_tokens() - spec.n_cached()
    sets = _sets(req, cfg.n_layers)
    plan = g.eng.plan_counts(0)
    expect = [N] + [orc.k_for_ratio(r, Nc) + Q for r in ratios[1:5]] + [orc.k_for_ratio(0.15, Nc) + Q] * (cfg.n_layers - 5)
    assert plan == expect and [len(s) for s in sets] == expect
    prev = None
    for s in sets:
        assert np.all(np.diff(s) > 0) and set(range(Nc, N)) <= set(s.tolist())
        if prev is not None:
            assert set(s.tolist()) <= set(prev.tolist())
        prev = s
    h = to_np(req["hidden"])[sets[-1]]
    assert np.all(np.isfinite(h))
    assert 0 <= int(req["first_token"].item()) < cfg.vocab


def test_mistral7b_full_recompute_equals_full_prefill(mistral):
    spec, g = mistral.spec, mistral
    cfg = spec.cfg
    req = g.blend(cb.ratio_schedule(cfg.n_layers, 1.0, "fixed"))[0]
    ids = np.concatenate([s.ids for s in spec.requests[0]])
    full = g.eng.full_prefill(hd.ids_tensor(ids), want_kv=True)
    torch.cuda.synchronize()
    assert max_rel_err(to_np(req["hidden"]), to_np(full["hidden"])) < 1e-3
    assert int(req["first_token"].item()) == int(full["first_token"].item())
    assert torch.equal(req["fused_k"], full["k"]) or max_rel_err(
        to_np(req["fused_k"][-1].reshape(len(ids), -1)), to_np(full["k"][-1].reshape(len(ids), -1))) < 1e-2


def test_mistral7b_blend_is_closer_to_full_prefill_than_reuse(mistral):
    """The method's premise on this workload: recomputing the HKVD tokens moves the query's
    final hidden states toward the full prefill, relative to reusing every cached KV."""
    spec, g = mistral.spec, mistral
    cfg = spec.cfg
    Nc, N = spec.n_cached(), spec.n_tokens()
    blend = g.blend(cb.ratio_schedule(cfg.n_layers, 0.15, "gradual"))[0]
    reuse = g.blend(cb.ratio_schedule(cfg.n_layers, 0.0, "fixed"))[0]
    ids = np.concatenate([s.ids for s in spec.requests[0]])
    full = g.eng.full_prefill(hd.ids_tensor(ids))
    torch.cuda.synchronize()
    ref = to_np(full["hidden"])[Nc:N]
    e_blend = max_rel_err(to_np(blend["hidden"])[Nc:N], ref)
    e_reuse = max_rel_err(to_np(reuse["hidden"])[Nc:N], ref)
    assert e_blend < e_reuse, (e_blend, e_reuse)
