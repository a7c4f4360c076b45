"""The contract's primitives on the GPU against the C emulator, over whole input ranges.

Each primitive is evaluated on the device for every fp32 bit pattern of a range
and folded into a position-weighted 64-bit sum (rlk_debug_primitive_hash); the
emulator forms the same sum.  Equal sums mean equal bits on every input of the
range (a single differing output changes the sum).  Ranges: exp on +0 and on
every negative fp32 down to -inf (the contract only forms arguments <= 0),
both as the scalar function and in the two-lane packed form the kernels use;
log on [1, 2^21] (every root sum of a tile tree); rsqrt on [2^-40, 2^40].
NaN inputs are outside the contract's domain and not compared.

A second opinion on accuracy: on a strided sample of each range, the contract's
values (the emulator's, which the device equals bit for bit) lie within 3 ulp of
CUDA's own expf / logf / rsqrtf as torch evaluates them on the device (each side
is within 2 ulp of the true value).
"""
import functools

import numpy as np
import pytest
import torch

from oracle import emulator as E

pytestmark = pytest.mark.gpu

RANGES = {
    "exp": [(0x00000000, 1), (0x80000000, 0xFF800000 - 0x80000000 + 1)],
    "exp_x2": [(0x00000000, 1), (0x80000000, 0xFF800000 - 0x80000000 + 1)],
    "log": [(0x3F800000, 0x4A000000 - 0x3F800000 + 1)],
    "rsqrt": [(0x2B800000, 0x53800000 - 0x2B800000 + 1)],
}


@functools.lru_cache(maxsize=None)
def emulator_hash(function, first, count):
    # the packed form must equal the scalar function, so both compare with it
    return E.primitive_hash(function, first, count)


@pytest.mark.slow
@pytest.mark.parametrize("which", sorted(RANGES))
def test_primitive_bits_equal_emulator_on_every_input(rlk, cuda_device, which):
    for first, count in RANGES[which]:
        gpu = rlk.primitive_hash(which, first, count, cuda_device)
        cpu = emulator_hash("exp" if which == "exp_x2" else which, first, count)
        assert gpu == cpu, (which, hex(first), count, hex(gpu), hex(cpu))


def test_hash_sees_a_shifted_range(rlk, cuda_device):
    """Over inputs whose outputs vary (exp on [-0.5, ...)), moving the range by one bit
    pattern changes the sum, and the emulator agrees with the device on both."""
    a = rlk.primitive_hash("exp", 0xBF000000, 1 << 20, cuda_device)
    b = rlk.primitive_hash("exp", 0xBF000001, 1 << 20, cuda_device)
    assert a != b
    assert a == E.primitive_hash("exp", 0xBF000000, 1 << 20)
    assert b == E.primitive_hash("exp", 0xBF000001, 1 << 20)


SAMPLES = {  # (first bit pattern, last, the emulator's scalar function, torch's)
    "exp": (0xC2AC0000, 0x80000001, E.exp, torch.exp),       # [-86, -2^-149]
    "log": (0x3F800000, 0x4A000000, E.log, torch.log),       # [1, 2^21]
    "rsqrt": (0x2B800000, 0x53800000, E.rsqrt, torch.rsqrt),  # [2^-40, 2^40]
}


@pytest.mark.parametrize("which", sorted(SAMPLES))
def test_primitives_within_3_ulp_of_cuda_math(cuda_device, which):
    lo, hi, contract, cuda_fn = SAMPLES[which]
    a, b = min(lo, hi), max(lo, hi)
    bits = np.unique(np.concatenate([np.linspace(a, b, 1 << 17).astype(np.uint32),
                                     np.array([a, b], dtype=np.uint32)]))
    x = bits.view(np.float32)
    ours = np.array([contract(float(v)) for v in x], dtype=np.float32)
    theirs = cuda_fn(torch.from_numpy(x.copy()).to(cuda_device)).cpu().numpy()
    # all values of one sign, so the ulp distance is the distance of the bit patterns
    assert np.all(np.isfinite(ours)) and np.all(ours >= 0) and np.all(theirs >= 0)
    ulps = np.abs(ours.view(np.int32).astype(np.int64) - theirs.view(np.int32).astype(np.int64))
    assert ulps.max() <= 3, (which, int(ulps.max()), float(x[ulps.argmax()]))
