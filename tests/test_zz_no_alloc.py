"""cb_gemm_noalloc: the projection GEMM for callers that cannot allocate device memory.

Callers held to a fixed device budget after start-up, or running inside a framework
that owns every allocation, cannot hand the GEMM a scratch buffer.  This entry point
keeps its stream-K scratch in a built-in device array instead.  The tests call it
through the C ABI twice in a row (the array keeps the previous call's contents) and
compare with cb_gemm given its own caller-allocated scratch, at the GEMM tolerance of
the other GPU tests.  This file is collected last and builds what it needs itself, so
it passes alone in a fresh process and after every other test.
"""
import numpy as np
import pytest
import torch

import rag_non_prefix_gb300 as cb
from tests._gpu import built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    built()


# (M, N, K, epilogue): stream-K splits over 16 CTAs (4 output tiles), which fit the
# built-in array, and a data-parallel shape that needs no scratch at all
SHAPES = [(64, 512, 28672, 1), (48, 512, 14336, 0), (64, 512, 8192, 2), (1024, 4096, 4096, 1)]


@pytest.mark.parametrize("M,N,K,epi", SHAPES)
def test_noalloc_gemm_matches_cb_gemm_on_two_calls(M, N, K, epi):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N + K)
    A = (torch.randn(M, K, device="cuda", generator=g) * 0.5).to(torch.bfloat16)
    if epi == 2:
        B = (torch.randn(N // 2, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        B2 = (torch.randn(N // 2, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        make = lambda: torch.zeros(M, N // 2, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    else:
        B = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        B2 = None
        C0 = torch.randn(M, N, device="cuda", generator=g)
        make = lambda: C0.clone()  # noqa: E731
    ref = make()
    cb.cb_gemm(A, B, ref, epi, B2=B2, scratch=cb.gemm_scratch())
    outs = []
    for _ in range(2):  # the second call finds the first call's partial tiles in the array
        o = make()
        cb.cb_gemm_noalloc(A, B, o, epi, B2=B2)
        outs.append(o)
    torch.cuda.synchronize()
    r = to_np(ref)
    tol = (2 ** -7 if epi == 2 else 1e-4) * np.max(np.abs(r)) + 1e-6
    for o in outs:
        assert np.max(np.abs(to_np(o) - r)) <= tol


def test_noalloc_gemm_rejects_a_split_larger_than_its_array():
    # 16 output tiles would be split over 128 CTAs: 16 MiB of partial tiles
    A = torch.zeros(200, 14336, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(2048, 14336, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(200, 2048, dtype=torch.float32, device="cuda")
    need = cb.load_library().cb_gemm_scratch_size()
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_gemm_noalloc(A, B, C, 0)
    assert e.value.name == "CB_ERR_WORKSPACE" and "built-in array" in str(e.value)
    assert need > 0
