"""Helpers of the GPU parity tests: device tensors from generator bits,
guarded output buffers, and the tolerance checks the fused path promises.

Tolerances (stated for the fused path): residual' bit-exact; norm output
within 1 ulp of the dtype; FP8 codes, NVFP4 block scales and E2M1 codes at
least 99.9 % identical and never more than one code step apart; NVFP4
dequantised values within one quantisation step of the block.  Only the fp32
order of the sum of squares may differ from the oracle, so wherever the
kernel's own norm output equals the oracle's, the quantised bytes must be
identical, and the kernel's codes must equal the oracle's quantiser applied
to the kernel's norm output.
"""
import numpy as np
import torch

from tests import pins

GUARD = 256
POISON = 0xA5


def dev16(a, dt):
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.bfloat16 if dt == "bf16" else torch.float16).cuda()


def host16(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def host8(t):
    return t.detach().cpu().numpy()


def f32dev(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


class Guarded:
    """An output tensor inside a buffer with poisoned guard bytes around it."""

    def __init__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((n + 2 * GUARD,), POISON, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + n].view(dtype).view(shape)
        self.n = n

    def guards_intact(self):
        b = self.buf.cpu().numpy()
        return bool(np.all(b[:GUARD] == POISON) and np.all(b[GUARD + self.n:] == POISON))


def assert_norm_within_ulp(y_gpu, y_ref, dt):
    a = pins.bits_to_f64(y_gpu, dt)
    b = pins.bits_to_f64(y_ref, dt)
    bad = ~(np.abs(a - b) <= pins.ulp(b, dt))
    assert not bad.any(), "norm output more than 1 ulp off at %d places" % int(bad.sum())


def assert_codes(c_gpu, c_ref, sign_bit, what, min_same=0.999):
    c_gpu = np.asarray(c_gpu)
    c_ref = np.asarray(c_ref)
    if c_ref.size == 0:
        return
    same = float(np.mean(c_gpu == c_ref))
    assert same >= min_same, "%s: only %.5f identical" % (what, same)
    steps = pins.code_steps(c_gpu, c_ref, sign_bit)
    assert steps.max() <= 1, "%s: %d codes more than one step apart" % (what, int((steps > 1).sum()))


def split_nibbles(packed):
    packed = np.asarray(packed, np.uint8)
    return np.stack([packed & 0xF, packed >> 4], axis=-1).reshape(packed.shape[0], -1)


def assert_nvfp4(p_gpu, sf_gpu, p_ref, sf_ref, y_ref, gs, dt):
    assert_codes(sf_gpu, sf_ref, 0x80, "block scales")
    assert_codes(split_nibbles(p_gpu), split_nibbles(p_ref), 0x8, "E2M1 codes")
    # dequantised error within one step (largest E2M1 gap, 2, times sf / gs)
    e2m1 = pins.e2m1_table()
    e4m3 = pins.e4m3_table()
    sfv = e4m3[np.asarray(sf_gpu)]
    deq = e2m1[split_nibbles(p_gpu)] * np.repeat(sfv, 16, axis=1) / gs
    yv = pins.bits_to_f64(y_ref, dt)
    step = np.repeat(2.0 * sfv / gs, 16, axis=1)
    # against y, the bound needs a normal, unsaturated block scale (an
    # oversized global scale saturates the E4M3 scale at 448 and then the
    # E2M1 codes at 6; a subnormal scale has too few bits to keep every
    # element within one step of y, on either side)
    normal = np.repeat((sfv >= 2.0 ** -6) & (sfv < 448.0), 16, axis=1)
    err = np.abs(deq - yv)
    assert np.all(err[normal] <= step[normal] * (1 + 1e-6)), "dequant error above one block step"
    # in those other blocks, against the oracle's own dequantised values:
    # equal wherever the scale byte and the code are the oracle's, and
    # otherwise within one step of the larger of the two block scales
    sfr = e4m3[np.asarray(sf_ref)]
    deq_ref = e2m1[split_nibbles(p_ref)] * np.repeat(sfr, 16, axis=1) / gs
    same = (np.repeat(np.asarray(sf_gpu) == np.asarray(sf_ref), 16, axis=1) &
            (split_nibbles(p_gpu) == split_nibbles(p_ref)))
    other = ~normal
    assert np.array_equal(deq[other & same], deq_ref[other & same]), \
        "dequantised value differs from the oracle's with the same codes"
    step2 = np.repeat(2.0 * np.maximum(sfv, sfr) / gs, 16, axis=1)
    diff = np.abs(deq - deq_ref)
    assert np.all(diff[other] <= step2[other] * (1 + 1e-6)), \
        "dequantised value more than one step from the oracle's in a subnormal or saturated block"
