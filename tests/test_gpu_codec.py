"""KV codec on the GPU (through the C ABI) against the oracle: the encoder bit for bit, the
fused decode + re-rotation to the storage type's rounding, and blends over quantised chunks
(device-resident and staged from pinned host memory through the staging ring)."""
import numpy as np
import pytest
import torch

import harness as hz
import oracle.cacheblend as orc
import rag_non_prefix_gb300 as cb
from tests._gpu import GpuWorkload, OracleWorkload, built, forced_from_oracle, max_rel_err, to_np
from tests.codec_layout import parse_blob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _build():
    built()


def _dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def _kv(rng, shape, dtype):
    """Keys with per-channel spreads and values with per-token spreads (the shapes KIVI's axes
    are chosen for), stored in the model dtype."""
    L, n, hkv, dh = shape
    k = rng.standard_normal(shape) * rng.uniform(0.05, 3.0, (L, 1, hkv, dh)) + rng.uniform(-1, 1, (L, 1, hkv, dh))
    v = rng.standard_normal(shape) * rng.uniform(0.05, 3.0, (L, n, hkv, 1))
    return _dev(k, dtype), _dev(v, dtype)


CASES = [(1, 1, 1, 64), (2, 37, 2, 64), (2, 512, 8, 128), (3, 129, 4, 128)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("shape", CASES, ids=[f"L{c[0]}n{c[1]}h{c[2]}d{c[3]}" for c in CASES])
def test_encode_is_bit_exact(dtype, bits, shape):
    rng = np.random.default_rng(sum(shape) * 10 + bits + (dtype == "bf16"))
    k, v = _kv(rng, shape, dtype)
    blob = cb.cb_kv_encode(k, v, bits)
    torch.cuda.synchronize()
    got = parse_blob(blob.cpu().numpy(), *shape, bits)
    ref = orc.kv_encode(to_np(k).astype(np.float32), to_np(v).astype(np.float32), bits)
    for name in ("k_codes", "v_codes"):
        assert np.array_equal(got[name], ref[name]), name
    for name in ("k_scale", "k_zero", "v_scale", "v_zero"):
        assert np.array_equal(got[name].view(np.uint32), ref[name].astype(np.float32).view(np.uint32)), name


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bits", [8, 4])
@pytest.mark.parametrize("delta", [0, 777, 8191])
def test_decode_rerotate_matches_oracle(dtype, bits, delta):
    shape = (2, 300, 8, 128) if dtype == "bf16" else (2, 97, 4, 64)
    rng = np.random.default_rng(5 + bits + delta)
    k, v = _kv(rng, shape, dtype)
    blob = cb.cb_kv_encode(k, v, bits)
    kd, vd = cb.cb_kv_decode(blob, shape, bits, delta, 1e4, k.dtype)
    torch.cuda.synchronize()
    enc = orc.kv_encode(to_np(k).astype(np.float32), to_np(v).astype(np.float32), bits)
    K, V = orc.kv_decode(enc)
    storage = "bf16" if dtype == "bf16" else "f32"
    refk = orc.round_storage(np.stack([orc.rerotate_keys(K[i], delta, 1e4) for i in range(shape[0])]), storage)
    refv = orc.round_storage(V, storage)
    gk, gv = to_np(kd), to_np(vd)
    if dtype == "bf16":
        # two roundings of values that agree to fp32 differ by one bf16 ulp at most: of the
        # element for V, of the head row's largest element for the rotated K (a rotation may
        # cancel an element down to far below its inputs)
        assert np.all(np.abs(gv - refv) <= 2 ** -7 * np.abs(refv))
        assert np.all(np.abs(gk - refk) <= 2 ** -7 * np.max(np.abs(refk), axis=-1, keepdims=True))
        assert np.mean(gk == refk) > 0.97 and np.mean(gv == refv) > 0.97
    else:
        scale = max(1.0, float(np.max(np.abs(refk))))
        assert np.max(np.abs(gk - refk)) <= 4e-6 * scale
        assert np.max(np.abs(gv - refv)) <= 4e-6 * max(1.0, float(np.max(np.abs(refv))))
    # the quantisation error itself is what the codec promises: half a step per group
    kin = to_np(k)
    err = np.abs(K - kin) / np.maximum(enc["k_scale"][:, None], 1e-30)
    assert np.max(err) <= 0.5 + 1e-3


# ----------------------------------------------------------------------------- blends over quantised chunks
class CodecWorkload:
    """The GPU workload with every chunk re-registered as a quantised blob (device or pinned host)."""

    def __init__(self, spec, bits, on_host=False, slots=2):
        self.g = GpuWorkload(spec)
        self.bits = bits
        self.blobs = {}
        slot = 0
        for c, (ids, k, v) in self.g.chunk_kv.items():
            blob = cb.cb_kv_encode(k, v, bits)
            torch.cuda.synchronize()
            if on_host:
                blob = blob.cpu().pin_memory()
            self.blobs[c] = blob
            self.g.eng.register_chunk_codec(c, ids, blob, bits, on_host=on_host)
        if on_host:
            cfg = spec.cfg
            for req in spec.requests:
                per = sum(cb.cb_codec_layer_bytes(len(s.ids), cfg.n_kv_heads, cfg.head_dim, bits)
                          for s in req if s.chunk >= 0)
                slot = max(slot, per)
            self.g.eng.set_staging(slots * slot)
        self.slot_bytes = slot


class OracleCodec(OracleWorkload):
    """The oracle over its own chunk caches quantised and dequantised by its codec."""

    def __init__(self, spec, bits):
        super().__init__(spec)
        self.caches = {c: orc.kv_decode(orc.kv_encode(K.astype(np.float32), V.astype(np.float32), bits))
                       for c, (K, V) in self.caches.items()}


@pytest.fixture(scope="module")
def small_bf16_spec():
    return hz.workload("small_bf16")


@pytest.mark.parametrize("bits", [8, 4])
def test_codec_blend_matches_oracle(small_bf16_spec, bits):
    """Resident quantised chunks: under the oracle's sets the hidden states agree within the
    bf16 tolerance, the free-running sets overlap the oracle's, and the blend differs from the
    unquantised one (the codec really is in the path)."""
    spec = small_bf16_spec
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    w = CodecWorkload(spec, bits)
    o = OracleCodec(spec, bits)
    ref = o.blend(0, ratios)
    req = w.g.blend(ratios, forced=forced_from_oracle(ref, ref["n_cached"], cfg.n_layers, ratios))[0]
    assert max_rel_err(to_np(req["hidden"])[ref["rows"]], ref["hidden"]) < 2e-2
    free = w.g.blend(ratios)[0]
    sel, cnt = free["sel"].cpu().numpy(), free["sel_count"].cpu().numpy()
    for i in range(cfg.n_layers):
        s = sel[i, : cnt[i]]
        assert len(s) == len(ref["sets"][i])
        assert len(np.intersect1d(s, ref["sets"][i])) / len(ref["sets"][i]) >= 0.97, i
    plain = GpuWorkload(spec).blend(ratios)[0]
    assert not torch.equal(plain["fused_k"], free["fused_k"])


@pytest.mark.parametrize("bits,slots", [(8, 1), (8, 2), (4, 3)])
def test_staged_codec_chunks_are_bit_identical(small_bf16_spec, bits, slots):
    """Host-resident quantised chunks staged through a ring of 1, 2 or 3 slots give exactly the
    result of the same blobs resident in device memory."""
    spec = small_bf16_spec
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    res = CodecWorkload(spec, bits).g.blend(ratios)[0]
    host = CodecWorkload(spec, bits, on_host=True, slots=slots)
    cs = torch.cuda.Stream()
    staged = host.g.blend(ratios, copy_stream=cs)[0]
    assert torch.equal(res["fused_k"], staged["fused_k"])
    assert torch.equal(res["fused_v"], staged["fused_v"])
    assert torch.equal(res["hidden"], staged["hidden"])


def test_staging_ring_rules(small_bf16_spec):
    """A fetch that would overwrite a slot still in use is refused; a missing or too small
    staging buffer is refused at begin; the per-layer API in the right order works."""
    spec = small_bf16_spec
    cfg = spec.cfg
    ratios = orc.ratio_schedule(cfg.n_layers, spec.ratio, spec.schedule)
    host = CodecWorkload(spec, 8, on_host=True, slots=2)
    eng = host.g.eng
    cs = torch.cuda.Stream()
    reqs = host.g.requests()
    eng.blend_begin(reqs, ratios)
    eng.fetch_kv(0, cs)
    eng.fetch_kv(1, cs)
    with pytest.raises(cb.CacheBlendError) as e:
        eng.fetch_kv(2, cs)  # slot 0 is still waiting for layer 0's decode
    assert e.value.name == "CB_ERR_STATE"
    for i in range(cfg.n_layers):
        eng.prefill_layer(i)
        if i + 2 < cfg.n_layers:
            eng.fetch_kv(i + 2, cs)
    eng.blend_finish()
    eng.get_status()
    torch.cuda.synchronize()
    whole = host.g.blend(ratios, copy_stream=cs)[0]
    assert torch.equal(whole["hidden"], reqs[0]["hidden"])
    eng.set_staging(host.slot_bytes - 256)
    with pytest.raises(cb.CacheBlendError) as e:
        host.g.blend(ratios, copy_stream=cs)
    assert e.value.name == "CB_ERR_WORKSPACE"


# ----------------------------------------------------------------------------- loading controller
def test_chunk_info_and_plan_over_the_registry(small_bf16_spec):
    """cb_chunk_info_of reports each registered chunk's tier and load bytes (bf16 KV, or the
    quantised blob), missing ids as missing; keyed by cb_chunk_hash, the registry finds a
    chunk by its content, and the plan over those infos is the oracle's."""
    spec = small_bf16_spec
    cfg = spec.cfg
    g = GpuWorkload(spec)
    eng = g.eng
    ids0, k0, v0 = g.chunk_kv[0]
    key = cb.cb_chunk_hash(spec.chunks[0])
    assert key == orc.chunk_hash(spec.chunks[0])
    eng.register_chunk(key, ids0, k0.cpu().pin_memory(), v0.cpu().pin_memory(), on_host=True)
    info = eng.chunk_info(key)
    n0 = len(spec.chunks[0])
    assert info == {"n_tokens": n0, "tier": cb.TIER_HOST,
                    "bytes": float(2 * cfg.n_layers * n0 * cfg.n_kv_heads * cfg.head_dim * 2)}
    assert eng.chunk_info(1)["tier"] == cb.TIER_DEVICE
    assert eng.chunk_info(0xDEADBEEF) == {"n_tokens": 0, "tier": cb.TIER_MISSING, "bytes": 0.0}
    ids1, k1, v1 = g.chunk_kv[1]
    blob = cb.cb_kv_encode(k1, v1, 4)
    torch.cuda.synchronize()
    eng.register_chunk_codec(77, ids1, blob, 4)
    n1 = len(spec.chunks[1])
    assert eng.chunk_info(77)["bytes"] == cfg.n_layers * cb.cb_codec_layer_bytes(n1, cfg.n_kv_heads, cfg.head_dim, 4)
    infos = [eng.chunk_info(c) for c in (key, 1, 77, 0xDEADBEEF)]
    model = {"link_bytes_per_s": 2e11, "link_latency_s": 1e-5, "prefill_s_per_token": 2e-6,
             "recompute_fixed_s": 1e-4, "r_min": 0.05, "r_max": 0.2}
    got = cb.cb_plan_loading(model, infos, 40)
    ref = orc.plan_loading(model, infos, 40)
    assert got[0] == ref[0] and got[0][1:] == [cb.ACT_USE, cb.ACT_USE, cb.ACT_RECOMPUTE]
    assert got[1] == pytest.approx(ref[1], rel=1e-12)
