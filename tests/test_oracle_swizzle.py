"""CPU checks of the oracle's GEMM-facing block-scale layout.

The pages size the NVFP4 scale tensor for the GEMM that consumes it but do
not print its layout, so the layout is the consumer's: the 128 x 4-tile
order that a block-scaled NVFP4 GEMM (cuBLASLt, 16-element blocks, E4M3
scales) reads.  Its byte order is pinned on the GPU by feeding the oracle's
output to that GEMM (tests/test_gpu_swizzle.py).  Here, without a GPU:

- the byte of each scale agrees with offsets worked by hand from the
  documented 128 x 4 block layout (tests/golden/nvfp4_swizzle_offsets.txt);

- the padded size agrees with the shape rule torch applies before it calls
  that GEMM (its meta kernel, which runs on the CPU), and any other size is
  refused by it;
- the layout moves every scale to its own byte, exactly once, and every
  other byte is a zero.
"""
import numpy as np
import pytest
import torch

import oracle as O

SHAPES = [(1, 32), (127, 96), (128, 64), (129, 80), (130, 96), (300, 1056), (257, 7168)]


def _meta_gemm(m, n, k, sa_bytes, sb_bytes):
    fp4 = torch.float4_e2m1fn_x2
    a = torch.empty(m, k // 2, dtype=fp4, device="meta")
    b = torch.empty(n, k // 2, dtype=fp4, device="meta").t()
    sa = torch.empty(sa_bytes, dtype=torch.float8_e4m3fn, device="meta")
    sb = torch.empty(sb_bytes, dtype=torch.float8_e4m3fn, device="meta")
    return torch._scaled_mm(a, b, sa, sb, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("rows,hidden", [(r, h) for r, h in SHAPES if h % 32 == 0])
def test_padded_size_is_the_gemm_shape_rule(rows, hidden):
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.skip("this torch has no packed FP4 dtype")
    n = 144  # the other operand: a multiple of 16 rows, as the GEMM asks
    sa = O.nvfp4_swizzled_scale_bytes(rows, hidden)
    sb = O.nvfp4_swizzled_scale_bytes(n, hidden)
    out = _meta_gemm(rows, n, hidden, sa, sb)
    assert tuple(out.shape) == (rows, n)
    for wrong in (sa - 1, sa + 4, rows * (hidden // 16)):
        if wrong == sa:
            continue
        with pytest.raises(RuntimeError):
            _meta_gemm(rows, n, hidden, wrong, sb)


@pytest.mark.parametrize("rows,hidden", SHAPES[:6])
def test_each_scale_moves_to_one_byte_and_padding_is_zero(rows, hidden):
    nb = hidden // 16
    size = O.nvfp4_swizzled_scale_bytes(rows, hidden)
    assert size == -(-rows // 128) * 128 * (-(-nb // 4) * 4)
    # one scale at a time set to a nonzero byte: exactly one output byte
    # changes, and no two scales share a byte
    seen = set()
    zero = np.zeros((rows, nb), np.uint8)
    assert not O.nvfp4_swizzle_scales(zero, hidden).any()
    picks = [(r, c) for r in range(rows) for c in range(nb)]
    if len(picks) > 600:
        rng = np.random.default_rng(7)
        picks = [picks[i] for i in rng.choice(len(picks), 600, replace=False)]
    for r, c in picks:
        sf = zero.copy()
        sf[r, c] = 0x3C
        out = O.nvfp4_swizzle_scales(sf, hidden)
        where = np.flatnonzero(out)
        assert where.size == 1 and out[where[0]] == 0x3C
        assert where[0] not in seen
        seen.add(int(where[0]))


def test_values_survive_and_rows_of_tiles_are_contiguous():
    rows, hidden = 300, 1056
    nb = hidden // 16
    rng = np.random.default_rng(3)
    sf = rng.integers(1, 127, size=(rows, nb), dtype=np.uint8)
    out = O.nvfp4_swizzle_scales(sf, hidden)
    # the multiset of bytes is the scales plus zeros for the padding
    pad = out.size - sf.size
    assert np.array_equal(np.sort(out)[pad:], np.sort(sf.ravel()))
    assert np.count_nonzero(out == 0) == pad
    # the scales of rows 0..127 fill the first row of tiles and no byte of it
    # comes from a later row
    per_tile_row = 128 * (-(-nb // 4) * 4)
    first = O.nvfp4_swizzle_scales(np.where(np.arange(rows)[:, None] < 128, sf, 0), hidden)
    assert np.array_equal(first[:per_tile_row], out[:per_tile_row])
    assert not first[per_tile_row:].any()


def _golden_cases():
    """Cases of tests/golden/nvfp4_swizzle_offsets.txt: (rows, hidden, size,
    [(r, c, offset)], [padding offsets])."""
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "nvfp4_swizzle_offsets.txt")
    cases = []
    with open(path) as f:
        for line in f:
            w = line.split()
            if not w or w[0].startswith("#"):
                continue
            if w[0] == "case":
                cases.append((int(w[1]), int(w[2]), int(w[3]), [], []))
            elif w[0] == "at":
                cases[-1][3].append((int(w[1]), int(w[2]), int(w[3])))
            elif w[0] == "pad":
                cases[-1][4].append(int(w[1]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: "%dx%d" % (c[0], c[1]))
def test_byte_offsets_match_the_hand_worked_golden(case):
    """Where each scale lands, against offsets worked by hand from the
    documented 128 x 4 block layout (row of tiles outermost; inside a tile
    (r, c) at 16 * (r mod 32) + 4 * (r div 32) + c)."""
    rows, hidden, size, at, pad = case
    nb = hidden // 16
    assert O.nvfp4_swizzled_scale_bytes(rows, hidden) == size
    # every scale a distinct nonzero byte, so a byte identifies its (r, c)
    ids = (np.arange(rows * nb) % 251 + 1).astype(np.uint8).reshape(rows, nb)
    out = O.nvfp4_swizzle_scales(ids, hidden)
    assert out.size == size
    for r, c, off in at:
        assert out[off] == ids[r, c], "scale (%d, %d) is not at byte %d" % (r, c, off)
        # and nowhere else among the bytes holding its id within its own tile
        tile = off // 512
        same = np.flatnonzero(out[tile * 512:(tile + 1) * 512] == ids[r, c]) + tile * 512
        assert off in same
    for off in pad:
        assert out[off] == 0, "padding byte %d is not zero" % off
