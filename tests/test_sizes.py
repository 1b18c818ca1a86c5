"""Size arithmetic printed on the pages (CPU): bits per weight of MXFP4 and
NVFP4, and the Qwen3-8B NVFP4 checkpoint's code and scale bytes that the
36-layer weight-set workload reproduces."""
import numpy as np

import oracle as ora
from block_scaled_fp4_e2m1_gb300 import workloads
from golden_util import load


def test_bits_per_weight():
    s = load("sizes.txt")
    n = 16 * 32 * 10
    packed, scales, _ = ora.nvfp4_quantize(np.zeros(n, np.float32))
    assert (packed.nbytes + scales.nbytes) * 8 / n == float(s["nvfp4_bits_per_weight"][0])
    mp, ms = ora.mxfp4_quantize(np.zeros((1, n), np.float32))
    assert (mp.nbytes + ms.nbytes) * 8 / n == float(s["mxfp4_bits_per_weight"][0])


def test_qwen3_8b_weight_set_bytes():
    """hiren.me "Where the missing speed went": 6.95 billion FP4 weights =
    3.47 GB of codes + 0.43 GB of FP8 scales."""
    s = load("sizes.txt")
    shapes = workloads.qwen3_8b_weight_shapes()
    n = sum(r * c for r, c in shapes)
    assert n == 6_945_767_424
    assert round(n / 1e9, 2) == float(s["nvfp4_weights_billion"][0])
    assert round(n / 2 / 1e9, 2) == float(s["nvfp4_codes_gb"][0])
    assert round(n / 16 / 1e9, 2) == float(s["nvfp4_scales_gb"][0])
