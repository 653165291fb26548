"""The C-ABI library loads and exports every symbol include/cacheblend.h declares; the
binding's struct layouts match the C compiler's; host-side planning agrees with the
oracle's reading of the pages (no GPU, no compute calls)."""
import ctypes as C
import os
import re
import subprocess

import pytest

import rag_non_prefix_gb300 as cb
from rag_non_prefix_gb300 import build as cbbuild
import oracle.cacheblend as orc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cacheblend.h")


@pytest.fixture(scope="module")
def lib():
    cbbuild.build()
    return cb.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cb_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 20
    out = subprocess.run(["nm", "-D", "--defined-only", cb.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (cb_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    assert sorted(cb.EXPORTED) == names
    for n in names:
        assert hasattr(lib, n)


def test_status_strings_without_gpu(lib):
    assert lib.cb_status_string(0) == b"ok"
    assert lib.cb_status_string(4) == b"chunk id not registered"
    assert lib.cb_registered_chunks(None) == 0


def test_struct_layout_matches_c_compiler(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "cacheblend.h"\n'
        "int main(void){\n"
        'printf("%zu %zu %zu %zu %zu\\n", sizeof(cb_model_cfg), offsetof(cb_model_cfg, rope_theta),'
        " offsetof(cb_model_cfg, rms_eps), offsetof(cb_model_cfg, dtype), offsetof(cb_model_cfg, max_positions));\n"
        'printf("%zu %zu %zu %zu\\n", sizeof(cb_request), offsetof(cb_request, n_query), offsetof(cb_request, out_first_token), offsetof(cb_request, kv_capacity));\n'
        'printf("%zu %zu %zu\\n", sizeof(cb_decode_seq), offsetof(cb_decode_seq, n_past), offsetof(cb_decode_seq, out_hidden));\n'
        'printf("%zu %zu %zu %zu %zu\\n", sizeof(cb_blend_params), offsetof(cb_blend_params, dev_mode),'
        " offsetof(cb_blend_params, forced_sel_host), offsetof(cb_blend_params, select_mode),"
        " offsetof(cb_blend_params, seam_tokens));\n"
        'printf("%zu\\n", sizeof(cb_weights));\nreturn 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    m = cb.ModelCfg
    assert lines[0].split() == [str(v) for v in (C.sizeof(m), m.rope_theta.offset, m.rms_eps.offset, m.dtype.offset,
                                                 m.max_positions.offset)]
    r = cb.Request
    assert lines[1].split() == [str(v) for v in (C.sizeof(r), r.n_query.offset, r.out_first_token.offset,
                                                 r.kv_capacity.offset)]
    ds = cb.DecodeSeq
    assert lines[2].split() == [str(v) for v in (C.sizeof(ds), ds.n_past.offset, ds.out_hidden.offset)]
    p = cb.BlendParams
    assert lines[3].split() == [str(v) for v in (C.sizeof(p), p.dev_mode.offset, p.forced_sel_host.offset,
                                                 p.select_mode.offset, p.seam_tokens.offset)]
    assert lines[4].strip() == str(C.sizeof(cb.Weights))


@pytest.mark.parametrize("L,r,sched", [(2, 0.15, "fixed"), (32, 0.15, "gradual"), (60, 0.15, "gradual"),
                                       (80, 0.1, "gradual"), (80, 0.2, "gradual"), (4, 0.5, "gradual"),
                                       (32, 0.0, "gradual"), (32, 1.0, "fixed")])
def test_host_schedule_matches_oracle(lib, L, r, sched):
    """cb_ratio_schedule / cb_k_for_ratio (C) against the oracle's reading R3 / R5, value for value."""
    assert cb.ratio_schedule(L, r, sched) == orc.ratio_schedule(L, r, sched)
    for nc in (1, 255, 256, 3136, 4096, 8192):
        for x in cb.ratio_schedule(L, r, sched):
            assert cb.k_for_ratio(x, nc) == orc.k_for_ratio(x, nc)


@pytest.mark.parametrize("L,r,r1,n", [(32, 0.15, 0.6, 5), (6, 0.1, 0.1, 3), (3, 0.2, None, 4), (60, 0.05, 1.0, 0)])
def test_host_schedule_options_match_oracle(lib, L, r, r1, n):
    assert cb.ratio_schedule(L, r, "gradual", r1=r1, n_narrow=n) == orc.ratio_schedule(L, r, "gradual", r1=r1,
                                                                                        n_narrow=n)


def test_host_schedule_rejects_bad_ratios(lib):
    for args in ((8, -0.1, "gradual"), (8, 1.5, "fixed")):
        with pytest.raises(cb.CacheBlendError):
            cb.ratio_schedule(*args)
    with pytest.raises(cb.CacheBlendError):  # r1 below r
        cb.ratio_schedule(8, 0.3, "gradual", r1=0.2)
    with pytest.raises(ValueError):
        cb.ratio_schedule(8, 0.3, "linear")


def test_tuning_hooks_reject_bad_values(lib):
    for bad in (-1, 3, 7):
        assert lib.cb_attention_set_tiles(bad) == 1  # CB_ERR_INVALID_ARG
    for ok in (0, 1, 2, 0):
        assert lib.cb_attention_set_tiles(ok) == 0
    for bad in (-1, 2):
        assert lib.cb_set_qkv_fusion(bad) == 1
    for ok in (0, 1):
        assert lib.cb_set_qkv_fusion(ok) == 0
    assert lib.cb_gemm_set_orientation(3) == 1 and lib.cb_gemm_set_orientation(0) == 0
    for bad in (-1, 3, 5, 8):
        assert lib.cb_gemm_set_pairing(bad) == 1
    for ok in (1, 2, 4, 0):
        assert lib.cb_gemm_set_pairing(ok) == 0
    assert lib.cb_k_for_ratio(0.0, 100) == 0 and lib.cb_k_for_ratio(0.15, 3136) == 471


def test_gemm_describe_reports_a_schedule_without_a_gpu():
    """The schedule query is host logic: on a machine without a GPU no CTA-pair cluster can be
    resident, so the single-CTA schedule is reported; its fields follow the header."""
    line = cb.cb_gemm_describe(1357, 7168, 7168, 1, 1 << 30)
    assert line.startswith(("single ", "pairs ")) and "model_us=" in line
    assert cb.cb_gemm_describe(0, 7168, 7168, 1) == "empty"
    with pytest.raises(cb.CacheBlendError):
        cb.cb_gemm_describe(4, 8, 8, 3)


def test_library_fails_loudly_when_missing(tmp_path):
    with pytest.raises(RuntimeError):
        cb._lib = None
        try:
            cb.load_library(str(tmp_path / "nope.so"))
        finally:
            cb._lib = None


def test_codec_layer_bytes_follow_the_documented_layout():
    """cb_codec_layer_bytes (a host-side size query) against the byte layout the header documents."""
    from tests.codec_layout import layer_layout

    lib = cb.load_library()
    for n, hkv, dh, bits in [(1, 1, 64, 8), (1, 1, 64, 4), (37, 2, 64, 4), (512, 8, 128, 8), (512, 32, 128, 4),
                             (129, 4, 128, 8), (3, 3, 64, 4)]:
        assert lib.cb_codec_layer_bytes(n, hkv, dh, bits) == layer_layout(n, hkv, dh, bits)[1]
    assert lib.cb_codec_layer_bytes(10, 2, 96, 8) == 0 and lib.cb_codec_layer_bytes(10, 2, 128, 2) == 0
