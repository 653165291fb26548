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

STATIC_BYTES = (4 << 20) + 1024  # CB_GEMM_STATIC_SCRATCH_BYTES


@pytest.fixture(scope="module", autouse=True)
def _build():
    built()


# (M, N, K, epilogue, uses the array): stream-K splits of 4 output tiles over 16 CTAs;
# a split that asks for more slots than the array holds with unlimited scratch (narrowed
# to the array's 32); a decode row (the GEMV, no scratch); a q|k|v projection of 480
# selected tokens of the Mistral-7B shape; whole output tiles (no scratch)
SHAPES = [(64, 512, 28672, 1, True), (48, 512, 14336, 0, True), (64, 512, 8192, 2, True),
          (200, 2048, 14336, 0, None), (1, 4096, 4096, 0, False), (480, 6144, 4096, 0, None),
          (1024, 4096, 4096, 1, False)]


@pytest.mark.parametrize("M,N,K,epi,uses", SHAPES)
def test_noalloc_gemm_matches_cb_gemm_on_two_calls(M, N, K, epi, uses):
    lib = cb.load_library()
    used = lib.cb_gemm_noalloc_scratch_used(M, N, K, epi, cb.CB_BF16)
    assert used <= STATIC_BYTES
    if uses is not None:
        assert (used > 0) == uses, used
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
    cb.cb_gemm_get_status()  # no device-side wait gave up
    assert lib.cb_gemm_noalloc_error() == b""
    r = to_np(ref)
    tol = (2 ** -7 if epi == 2 else 1e-4) * np.max(np.abs(r)) + 1e-6
    for o in outs:
        assert np.max(np.abs(to_np(o) - r)) <= tol


def test_noalloc_gemm_reports_bad_arguments_with_a_message():
    A = torch.zeros(8, 100, dtype=torch.bfloat16, device="cuda")  # K % 64 != 0
    B = torch.zeros(128, 100, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(8, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(cb.CacheBlendError) as e:
        cb.cb_gemm_noalloc(A, B, C, 0)
    assert e.value.name == "CB_ERR_SHAPE" and "K % 64" in str(e.value)
