"""The algorithmic bytes behind every GB/s figure bench.py reports, checked
against a count of the tensors each call reads or writes once, built from the
shapes include/rq.h documents (element counts times element sizes), for the
workloads the bench times."""
import numpy as np

import bench


def _bytes(*tensors):
    """Sum of numel * itemsize over (shape, itemsize) pairs."""
    return sum(int(np.prod(shape)) * size for shape, size in tensors)


def test_fp8_call_bytes():
    r, h = 65536, 1024
    read = _bytes(((r, h), 2), ((r, h), 2), ((h,), 2), ((1,), 4))  # x, residual, weight, scale
    written = _bytes(((r, h), 2), ((r, h), 1))                       # residual', codes
    assert bench.alg_bytes_fp8(r, h) == read + written == 469_764_100


def test_nvfp4_call_bytes():
    r, h = 16384, 7168
    read = _bytes(((r, h), 2), ((r, h), 2), ((h,), 2), ((1,), 4))
    # residual', norm out, packed codes (two per byte), one E4M3 scale per 16
    written = _bytes(((r, h), 2), ((r, h), 2), ((r, h // 2), 1), ((r, h // 16), 1))
    assert bench.alg_bytes_nvfp4(r, h) == read + written == 1_005_598_724


def test_qk_call_bytes():
    t, hq, hk, d = 4096, 16, 8, 128
    # q, k heads; one fp32 cos/sin table row and one int32 position per token;
    # two weights and two scales; dense FP8 codes out
    read = _bytes(((t, hq, d), 2), ((t, hk, d), 2), ((t, d), 4), ((t,), 4), ((d,), 2), ((d,), 2),
                  ((1,), 4), ((1,), 4))
    written = _bytes(((t, hq, d), 1), ((t, hk, d), 1))
    assert bench.alg_bytes_qk(t, hq, hk, d) == read + written == 39_862_792


def test_step_rows_and_bytes():
    assert bench.ROWS_PER_STEP == 65536 + 4096 * 24 + 16384
    assert bench.STEP_BYTES == 469_764_100 + 39_862_792 + 1_005_598_724
