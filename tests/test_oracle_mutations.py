"""Planted mistakes in the oracle must each fail a named pin (no GPU).

Each ORC_PLANT value compiles oracle.cpp with one plausible mistake (a wrong
shift order, a dropped term, a reciprocal scale, ties-to-even rounding, a
missing floor, a transposed output, a lost scale, int16 overflow, a wrong row
scale, a wrong epilogue order, a missing ReLU, a dropped input scale, a scale
product associated the other way). The test proves the pins are strong enough
to notice each one.
"""

import os
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle
from tests import pins

PLANTS = {
    1: ["pin_i2s_hand_decode"],            # unpacker shift order reversed
    2: ["pin_i2s_hand_pack"],              # packer shift order reversed
    3: ["pin_i2s_pow2_special_case"],      # row sum not subtracted
    4: ["pin_quant_golden"],               # reciprocal (127/amax) stored as scale
    5: ["pin_quant_golden"],               # ties to even
    6: ["pin_quant_golden"],               # no 1e-5 amax floor
    7: ["pin_i2s_pow2_special_case"],      # output written transposed
    8: ["pin_i8s_permute_cont"],           # permute/cont loses the scale
    9: ["pin_i2s_headroom"],               # accumulator narrowed to int16
    10: ["pin_i2s_pow2_special_case"],     # every row uses row 0's scale
    11: ["pin_i8s_mul_mat_add_special_case"],  # bias added before scaling
    12: ["pin_i8s_mul_mat_add_special_case"],  # ReLU dropped
    13: ["pin_i8s_mul_mat_add_special_case"],  # activation scale dropped
    14: ["pin_i8s_add_scaled_pow2"],       # second input read with the first's scale
    15: ["pin_i8s_rms_norm_closed_forms"],  # mean square without the scale
    16: ["pin_i8s_rms_norm_closed_forms"],  # mean over ne0 - 1
    17: ["pin_i8s_im2col_asym"],           # right pad used as the left pad
    18: ["pin_i8s_depthwise_pow2"],        # kernel taps reversed (convolution)
    19: ["pin_w8a8_mul_mat_pow2"],         # row scale dropped
    20: ["pin_w8a8_weight_quant"],         # weight ties rounded away from zero
    21: ["pin_i2s_epilogue_association"],  # (dot - row_sum) * w_scale * act_scale, left to right
    22: ["pin_i8s_epilogue_association"],  # acc * w_scale * x_scale, left to right
    23: ["pin_w8a8_epilogue_association"],  # aScale * (bScale * C)
}


@pytest.fixture(scope="module")
def planted():
    d = tempfile.mkdtemp(prefix="oracle_plants_")
    paths = {k: os.path.join(d, f"liboracle_plant{k}.so") for k in PLANTS}
    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        list(ex.map(lambda k: oracle.build(paths[k], plant=k), PLANTS))
    return {k: oracle.Oracle(p) for k, p in paths.items()}


@pytest.mark.parametrize("plant", sorted(PLANTS))
def test_plant_is_caught(planted, plant):
    o = planted[plant]
    for name in PLANTS[plant]:
        with pytest.raises(AssertionError):
            getattr(pins, name)(o)
