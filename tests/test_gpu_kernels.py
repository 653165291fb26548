"""Per-kernel parity of the CUDA path (through the C ABI) against the oracle."""
import numpy as np
import pytest
import torch

import harness as hz
import harness.device as hd
import oracle.cacheblend as orc
import rag_non_prefix_gb300 as cb
from tests._gpu import built, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    built()


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).cuda()


def _f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


# ----------------------------------------------------------------------------- harness
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_device_generator_matches_host_bits(dtype):
    key = hz.layer_weight_key(5, 3, 2)
    t = torch.empty(300_001, dtype=dtype, device="cuda")
    hd.synth_into(t, key, start=12345)
    host = hz.gen_weight_fp32(key, 12345, 300_001)
    if dtype == torch.bfloat16:
        ref = hz.fp32_to_bf16_bits(host)
        got = t.view(torch.int16).cpu().numpy().view(np.uint16)
    else:
        ref = host.view(np.uint32)
        got = t.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, ref)


# ----------------------------------------------------------------------------- re-rotation
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,hkv,dh,delta,theta", [(1, 1, 64, 3, 1e4), (37, 4, 64, 128, 1e4), (512, 8, 128, 3136, 1e4),
                                                  (333, 2, 128, 8191, 1e4), (64, 8, 128, 0, 1e4),
                                                  # the Yi-34B shape's rotary base, chunks up to its last offset
                                                  (512, 8, 128, 7680, 5e6), (128, 8, 128, 8320, 5e6),
                                                  (512, 8, 128, 512, 5e6)])
def test_rerotate_matches_oracle(dtype, n, hkv, dh, delta, theta):
    rng = np.random.default_rng(n + delta)
    k = rng.standard_normal((n, hkv, dh)).astype(np.float32)
    v = rng.standard_normal((n, hkv, dh)).astype(np.float32)
    mk = _bf16 if dtype == "bf16" else _f32
    ks, vs = mk(k), mk(v)
    kd, vd = torch.empty_like(ks), torch.empty_like(vs)
    cb.cb_rope_rerotate(ks, kd, vs, vd, delta, theta)
    torch.cuda.synchronize()
    kin = to_np(ks)
    ref = orc.rerotate_keys(kin, delta, theta)
    got = to_np(kd)
    if dtype == "bf16":
        ref = orc.round_storage(ref, "bf16")
        # one bf16 ulp of the largest element bounds the difference of two roundings
        assert np.max(np.abs(got - ref)) <= 2 ** -7 * np.max(np.abs(ref))
        assert np.mean(got == ref) > 0.97
    else:
        assert np.max(np.abs(got - ref)) <= 2e-6 * max(1.0, np.max(np.abs(ref)))
    assert torch.equal(vd, vs)
    if delta == 0:
        assert torch.equal(kd, ks)


def test_rerotate_in_place_and_key_only():
    rng = np.random.default_rng(7)
    k = _bf16(rng.standard_normal((100, 8, 128)))
    ref = k.clone()
    out = torch.empty_like(k)
    cb.cb_rope_rerotate(ref, out, None, None, 777, 1e4)
    cb.cb_rope_rerotate(k, k, None, None, 777, 1e4)
    torch.cuda.synchronize()
    assert torch.equal(k, out)


# ----------------------------------------------------------------------------- deviation
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1, 2])
def test_deviation_matches_oracle(dtype, mode):
    rng = np.random.default_rng(11 + mode)
    n, N, kvw = 300, 520, 1024
    kn = rng.standard_normal((n, kvw)).astype(np.float32)
    vn = rng.standard_normal((n, kvw)).astype(np.float32)
    kf = rng.standard_normal((N, kvw)).astype(np.float32)
    vf = rng.standard_normal((N, kvw)).astype(np.float32)
    idx = np.sort(rng.choice(N, n, replace=False)).astype(np.int32)
    mk = _bf16 if dtype == "bf16" else _f32
    kft, vft = mk(kf), mk(vf)
    dev = cb.cb_kv_deviation(_f32(kn), _f32(vn), kft, vft, torch.from_numpy(idx).cuda(), mode)
    torch.cuda.synchronize()
    ref = orc.kv_deviation(kn.astype(np.float64), vn.astype(np.float64), to_np(kft)[idx], to_np(vft)[idx], mode)
    assert np.max(np.abs(dev.cpu().numpy() - ref) / ref) < 1e-5


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cosine_deviation_matches_oracle(dtype):
    """mode 3 (1 - cos of [k; v]) on rows far apart (dev ~ 1) and close together
    (dev ~ 1e-3, where fp32 sums lose the most relative accuracy), plus zero rows."""
    rng = np.random.default_rng(17)
    n, N, kvw = 300, 520, 1024
    kf = rng.standard_normal((N, kvw)).astype(np.float32)
    vf = rng.standard_normal((N, kvw)).astype(np.float32)
    idx = np.sort(rng.choice(N, n, replace=False)).astype(np.int32)
    near = np.arange(n) % 2 == 0
    kn = rng.standard_normal((n, kvw)).astype(np.float32)
    vn = rng.standard_normal((n, kvw)).astype(np.float32)
    kn[near] = kf[idx[near]] + 0.05 * kn[near]
    vn[near] = vf[idx[near]] + 0.05 * vn[near]
    kn[1], vn[1] = 0.0, 0.0  # a zero fresh row against a non-zero cached one: 1
    mk = _bf16 if dtype == "bf16" else _f32
    kft, vft = mk(kf), mk(vf)
    dev = cb.cb_kv_deviation(_f32(kn), _f32(vn), kft, vft, torch.from_numpy(idx).cuda(), 3)
    torch.cuda.synchronize()
    ref = orc.kv_deviation(kn.astype(np.float64), vn.astype(np.float64), to_np(kft)[idx], to_np(vft)[idx], 3)
    got = dev.cpu().numpy().astype(np.float64)
    assert got[1] == 1.0 and ref[1] == 1.0
    assert np.max(np.abs(got - ref)) < 4e-6, np.max(np.abs(got - ref))
    assert np.max(ref[near]) < 5e-3 and np.min(ref[~near]) > 0.5


# ----------------------------------------------------------------------------- selection (bit-exact)
def _select_case(dev32, cand, k):
    d = torch.from_numpy(dev32).cuda()
    c = None if cand is None else torch.from_numpy(cand.astype(np.int32)).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cb.cb_select_hkvd(d, c, k, status=st)
    torch.cuda.synchronize()
    ref = orc.select_hkvd(dev32, np.arange(len(dev32)) if cand is None else cand, k)
    return out.cpu().numpy(), ref, int(st.item())


@pytest.mark.parametrize("n,k", [(1, 1), (7, 3), (256, 39), (3136, 471), (3200, 941), (8192, 1229), (8192, 8192),
                                 (65536, 6554), (1000, 0), (4099, 4098)])
def test_select_is_bit_exact(n, k):
    rng = np.random.default_rng(n * 7 + k)
    dev = (rng.standard_normal(n) ** 2).astype(np.float32)
    cand = np.sort(rng.choice(4 * n + 10, n, replace=False))
    got, ref, st = _select_case(dev, cand, k)
    assert st == 0
    assert np.array_equal(got, ref)


def test_select_ties_and_zero_deviation():
    rng = np.random.default_rng(3)
    dev = rng.integers(0, 5, 4000).astype(np.float32)  # heavy ties
    dev[:500] = 0.0  # a first chunk: deviation 0
    for k in (1, 17, 500, 3500, 3999):
        got, ref, st = _select_case(dev, None, k)
        assert np.array_equal(got, ref)


def test_select_nan_sets_status_without_fault():
    dev = np.ones(100, dtype=np.float32)
    dev[17] = np.nan
    d = torch.from_numpy(dev).cuda()
    st_t = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cb.cb_select_hkvd(d, None, 10, status=st_t)
    torch.cuda.synchronize()
    assert int(st_t.item()) & 1
    assert 17 not in out.cpu().numpy().tolist()


# ----------------------------------------------------------------------------- GEMM
def _gemm_ref(a, b):
    return a.astype(np.float64) @ b.astype(np.float64).T


@pytest.fixture(params=[0, 1, 2], ids=["model", "token-rows", "weight-rows"])
def orientation(request):
    """Runs a GEMM test under each tile orientation (process-wide setting, reset after)."""
    cb.cb_gemm_set_orientation(request.param)
    yield request.param
    cb.cb_gemm_set_orientation(0)


@pytest.mark.parametrize("sk", [False, True], ids=["whole-tiles", "stream-k"])
@pytest.mark.parametrize("M,N,K", [(1, 128, 64), (2, 6144, 4096), (3, 6144, 4096), (8, 1024, 14336), (71, 256, 512), (128, 384, 256), (300, 768, 1024), (535, 1024, 4096),
                                   (1000, 512, 320), (535, 4096, 4096), (535, 4096, 14336), (3000, 6144, 512),
                                   (128, 4096, 14336), (256, 4096, 4096), (200, 2560, 8192), (64, 1024, 28672)])
def test_gemm_bf16_store_and_add(M, N, K, sk, orientation):
    scr = cb.gemm_scratch() if sk else None
    rng = np.random.default_rng(M + N + K)
    A = _bf16(rng.standard_normal((M, K)))
    B = _bf16(rng.standard_normal((N, K)) * 0.02)
    C0 = _f32(rng.standard_normal((M, N)))
    ref = _gemm_ref(to_np(A), to_np(B))
    out = torch.full((M, N), np.nan, dtype=torch.float32, device="cuda")
    cb.cb_gemm(A, B, out, epilogue=0, scratch=scr)
    acc = C0.clone()
    cb.cb_gemm(A, B, acc, epilogue=1, scratch=scr)
    torch.cuda.synchronize()
    if sk:  # the flags at the head of the scratch are left zeroed for the next call
        assert int(scr[:1024].view(torch.int32).abs().sum().item()) == 0
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(to_np(out) - ref)) < 1e-4 * scale
    assert np.max(np.abs(to_np(acc) - (ref + to_np(C0)))) < 1e-4 * max(scale, 1.0) + 1e-5


@pytest.mark.parametrize("sk", [False, True], ids=["whole-tiles", "stream-k"])
@pytest.mark.parametrize("M,F,K", [(1, 14336, 4096), (2, 2048, 1024), (5, 64, 128), (8, 2048, 1024), (130, 128, 256), (535, 384, 512), (535, 14336, 4096), (96, 2048, 4096),
                                   (3200, 1024, 256), (1005, 3584, 1024)])
def test_gemm_bf16_swiglu(M, F, K, sk, orientation):
    rng = np.random.default_rng(M + F)
    A = _bf16(rng.standard_normal((M, K)))
    G = _bf16(rng.standard_normal((F, K)) * 0.05)
    U = _bf16(rng.standard_normal((F, K)) * 0.05)
    out = torch.zeros((M, F), dtype=torch.bfloat16, device="cuda")
    cb.cb_gemm(A, G, out, epilogue=2, B2=U, scratch=cb.gemm_scratch() if sk else None)
    torch.cuda.synchronize()
    g = _gemm_ref(to_np(A), to_np(G))
    u = _gemm_ref(to_np(A), to_np(U))
    ref = orc.silu(g) * u
    assert np.max(np.abs(to_np(out) - ref)) <= 2 ** -7 * np.max(np.abs(ref)) + 1e-6


@pytest.mark.parametrize("ldc_extra", [0, 8, 136], ids=["dense", "pitch+8", "pitch+136"])
def test_gemm_bf16_strided_output(ldc_extra, orientation):
    """Output rows with a pitch larger than N (the tile stores go through a tensor map
    with that pitch): columns past N stay untouched."""
    M, N, K = 535, 1024, 512
    rng = np.random.default_rng(7)
    A = _bf16(rng.standard_normal((M, K)))
    B = _bf16(rng.standard_normal((N, K)) * 0.02)
    ref = _gemm_ref(to_np(A), to_np(B))
    big = torch.full((M, N + ldc_extra), 3.0, dtype=torch.float32, device="cuda")
    cb.cb_gemm(A, B, big, epilogue=1, scratch=cb.gemm_scratch())
    torch.cuda.synchronize()
    got = to_np(big)
    assert np.max(np.abs(got[:, :N] - (ref + 3.0))) < 1e-4 * np.max(np.abs(ref)) + 1e-5
    assert np.all(got[:, N:] == 3.0)


def test_gemm_stream_k_is_deterministic():
    rng = np.random.default_rng(99)
    A = _bf16(rng.standard_normal((200, 14336)))  # 32 tiles: the stream-K schedule
    B = _bf16(rng.standard_normal((4096, 14336)) * 0.02)
    outs = []
    for _ in range(3):
        o = torch.zeros((200, 4096), dtype=torch.float32, device="cuda")
        cb.cb_gemm(A, B, o, 1, scratch=cb.gemm_scratch())
        outs.append(o)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


@pytest.fixture(params=[(2, 0), (4, 0), (2, 16), (4, 16), (2, 240), (4, 240), (4, 256)],
                ids=["pair-model", "two-pairs-model", "pair-16", "two-pairs-16", "pair-240", "two-pairs-240",
                     "two-pairs-256"])
def pairing(request):
    """Runs a GEMM test on CTA pairs (clusters of one or two pairs), with the time model's
    token tile or a forced one (process-wide settings, reset after)."""
    cl, bt = request.param
    cb.cb_gemm_set_pairing(cl)
    cb.cb_gemm_set_orientation(bt)
    yield request.param
    cb.cb_gemm_set_pairing(0)
    cb.cb_gemm_set_orientation(0)


@pytest.mark.parametrize("M,N,K", [(1, 256, 64), (17, 256, 128), (71, 256, 512), (300, 768, 1024), (535, 1024, 4096),
                                   (1000, 512, 320), (535, 4096, 4096), (3000, 6144, 512), (256, 4096, 4096),
                                   (200, 2560, 8192), (64, 1024, 28672), (1357, 1024, 1024), (4400, 512, 256)])
def test_gemm_bf16_pairs_store_and_add(M, N, K, pairing):
    """CTA-pair tiles against fp64: every token tile (a ragged last one, a pad tile of the
    second pair when the token tiles are odd), both weight halves, K of one or many stages."""
    rng = np.random.default_rng(M + N + K + 1)
    A = _bf16(rng.standard_normal((M, K)))
    B = _bf16(rng.standard_normal((N, K)) * 0.02)
    C0 = _f32(rng.standard_normal((M, N)))
    ref = _gemm_ref(to_np(A), to_np(B))
    out = torch.full((M, N), np.nan, dtype=torch.float32, device="cuda")
    cb.cb_gemm(A, B, out, epilogue=0)
    acc = C0.clone()
    cb.cb_gemm(A, B, acc, epilogue=1)
    torch.cuda.synchronize()
    scale = np.max(np.abs(ref))
    assert np.max(np.abs(to_np(out) - ref)) < 1e-4 * scale
    assert np.max(np.abs(to_np(acc) - (ref + to_np(C0)))) < 1e-4 * max(scale, 1.0) + 1e-5


@pytest.mark.parametrize("M,F,K", [(2, 2048, 1024), (130, 128, 256), (535, 384, 512), (535, 14336, 4096),
                                   (96, 2048, 4096), (3200, 1024, 256), (1005, 3584, 1024), (1357, 640, 1024)])
def test_gemm_bf16_pairs_swiglu(M, F, K, pairing):
    rng = np.random.default_rng(M + F + 1)
    A = _bf16(rng.standard_normal((M, K)))
    G = _bf16(rng.standard_normal((F, K)) * 0.05)
    U = _bf16(rng.standard_normal((F, K)) * 0.05)
    out = torch.zeros((M, F), dtype=torch.bfloat16, device="cuda")
    cb.cb_gemm(A, G, out, epilogue=2, B2=U)
    torch.cuda.synchronize()
    g = _gemm_ref(to_np(A), to_np(G))
    u = _gemm_ref(to_np(A), to_np(U))
    ref = orc.silu(g) * u
    assert np.max(np.abs(to_np(out) - ref)) <= 2 ** -7 * np.max(np.abs(ref)) + 1e-6


def test_gemm_pairs_are_deterministic_and_match_single_ctas():
    """The paired kernel sums each output in the same k order on every run; against the
    single-CTA kernel it agrees to fp32 rounding of the same sums."""
    rng = np.random.default_rng(5)
    A = _bf16(rng.standard_normal((1357, 2048)))
    B = _bf16(rng.standard_normal((2048, 2048)) * 0.02)
    outs = {}
    try:
        for mode in (1, 2, 4):
            cb.cb_gemm_set_pairing(mode)
            runs = []
            for _ in range(2):
                o = torch.zeros((1357, 2048), dtype=torch.float32, device="cuda")
                cb.cb_gemm(A, B, o, 0)
                runs.append(o)
            torch.cuda.synchronize()
            assert torch.equal(runs[0], runs[1])
            outs[mode] = to_np(runs[0])
    finally:
        cb.cb_gemm_set_pairing(0)
    scale = np.max(np.abs(outs[1]))
    assert np.max(np.abs(outs[2] - outs[1])) < 1e-5 * scale
    assert np.max(np.abs(outs[4] - outs[1])) < 1e-5 * scale


@pytest.mark.parametrize("M,N,K", [(1, 64, 8), (2, 100, 36), (4, 100, 36), (8, 256, 1024), (77, 200, 96), (288, 1024, 256)])
def test_gemm_f32_all_epilogues(M, N, K):
    rng = np.random.default_rng(M * 3 + N)
    A = _f32(rng.standard_normal((M, K)))
    B = _f32(rng.standard_normal((N, K)) * 0.05)
    U = _f32(rng.standard_normal((N, K)) * 0.05)
    ref = _gemm_ref(to_np(A), to_np(B))
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    cb.cb_gemm(A, B, out, 0)
    sw = torch.empty((M, N), dtype=torch.float32, device="cuda")
    cb.cb_gemm(A, B, sw, 2, B2=U)
    torch.cuda.synchronize()
    assert np.max(np.abs(to_np(out) - ref)) < 1e-5 * np.max(np.abs(ref))
    swr = orc.silu(ref) * _gemm_ref(to_np(A), to_np(U))
    assert np.max(np.abs(to_np(sw) - swr)) < 1e-5 * np.max(np.abs(swr))


# ----------------------------------------------------------------------------- attention
@pytest.mark.parametrize("tiles", [1, 2], ids=["one-tile", "two-tiles"])
@pytest.mark.parametrize("H,Hkv,N,m", [(8, 2, 300, 70), (4, 4, 200, 130), (32, 8, 3200, 535), (56, 8, 700, 50),
                                       (64, 8, 260, 33), (8, 8, 64, 64), (56, 8, 8320, 1357), (32, 8, 1000, 96)])
def test_attention_bf16_matches_oracle(H, Hkv, N, m, tiles):
    """Both kernels: one query tile per CTA, and two tiles of one KV head per CTA (odd and
    even tile counts, tiles of different lengths, the Yi-34B shape at its kept-layer size)."""
    rng = np.random.default_rng(H * N + m)
    pos = np.sort(rng.choice(N, m, replace=False)).astype(np.int32)
    q = _bf16(rng.standard_normal((m, H, 128)))
    k = _bf16(rng.standard_normal((N, Hkv, 128)))
    v = _bf16(rng.standard_normal((N, Hkv, 128)))
    cb.cb_attention_set_tiles(tiles)
    try:
        out = cb.cb_attention(q, torch.from_numpy(pos).cuda(), k, v)
        torch.cuda.synchronize()
    finally:
        cb.cb_attention_set_tiles(0)
    sample = np.arange(m) if m <= 80 else np.unique(np.concatenate([np.arange(8), rng.choice(m, 40), [m - 1]]))
    ref = orc.causal_attention(to_np(q)[sample], pos[sample], to_np(k), to_np(v))
    got = to_np(out)[sample]
    # per query row and head: ||g - o||_inf / ||o||_inf (bf16 probabilities and output:
    # a few 2^-9 relative errors per element)
    err = np.max(np.abs(got - ref), axis=2) / np.maximum(np.max(np.abs(ref), axis=2), 1e-30)
    assert np.max(err) < 2e-2, float(np.max(err))


@pytest.mark.parametrize("H,Hkv,dh,N,m", [(4, 4, 64, 288, 71), (8, 2, 64, 252, 40), (2, 1, 128, 100, 100)])
def test_attention_f32_matches_oracle(H, Hkv, dh, N, m):
    rng = np.random.default_rng(H + dh + m)
    pos = np.sort(rng.choice(N, m, replace=False)).astype(np.int32)
    q = _f32(rng.standard_normal((m, H, dh)))
    k = _f32(rng.standard_normal((N, Hkv, dh)))
    v = _f32(rng.standard_normal((N, Hkv, dh)))
    out = cb.cb_attention(q, torch.from_numpy(pos).cuda(), k, v)
    torch.cuda.synchronize()
    ref = orc.causal_attention(to_np(q), pos, to_np(k), to_np(v))
    assert np.max(np.abs(to_np(out) - ref)) < 1e-5 * np.max(np.abs(ref))
