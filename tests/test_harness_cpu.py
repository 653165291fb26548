"""The harness's host generators agree bit for bit: the C twin (threads over the range)
against the numpy definition, in fp32 and bf16, at arbitrary starts and extreme keys."""
import numpy as np
import pytest

import harness as hz
from rag_non_prefix_gb300 import build as cbbuild


@pytest.fixture(scope="module", autouse=True)
def host_lib():
    for lib, srcs in cbbuild.HOST_LIBS.items():
        cbbuild._build_host(lib, srcs)
    assert hz.host_generator() is not None


@pytest.mark.parametrize("key,start,count", [
    (0, 0, 1),
    (123, 0, 100_003),
    (0xFFFFFFFFFFFFFFFF, 10**9, 70_001),
    (hz.layer_weight_key(4, 59, hz.MAT_DOWN), 20480 * 7168 - 5000, 5000),
    (hz.layer_weight_key(5, hz.GLOBAL_LM_LAYER, 0), 3 * 2**31 + 17, 1 << 17),
])
def test_c_generator_matches_numpy_bits(key, start, count):
    ref = hz.gen_weight_fp32_numpy(key, start, count)
    got = hz.gen_weight_fp32_c(key, start, count)
    assert np.array_equal(ref.view(np.uint32), got.view(np.uint32))
    ref16 = hz.bf16_bits_to_fp32(hz.fp32_to_bf16_bits(ref))
    got16 = hz.gen_weight_fp32_c(key, start, count, as_bf16=True)
    assert np.array_equal(ref16.view(np.uint32), got16.view(np.uint32))


def test_gen_matrix_rows_equal_whole_matrix():
    cfg = hz.MODELS["small_bf16"]
    whole = hz.gen_matrix(cfg, 11, 2, hz.MAT_UP)
    rows = np.array([0, 7, 1535])
    assert np.array_equal(hz.gen_matrix(cfg, 11, 2, hz.MAT_UP, rows=rows), whole[rows])
    # statistics of the definition: mean 0, standard deviation 0.02
    assert abs(float(whole.mean())) < 2e-4
    assert abs(float(whole.std()) - 0.02) < 2e-4
