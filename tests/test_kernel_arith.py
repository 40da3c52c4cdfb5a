"""Arithmetic shortcuts the CUDA kernels take, checked on the CPU against the
oracle over every input they can see (no GPU needed).

q8_0 key blocks ("PolyKV" section 2, the q8_0 key format): the encoder forms
the fp16 block scale as fp16(fl32(max|k|) * fl32(1/127)) instead of an IEEE
division.  Over all 32,640 finite bf16 maxima that must give the oracle's
scale, the fp16 nearest to the real max|k|/127, including the fp16 subnormal
range and the overflow to Inf (reported as a range error).
"""
import numpy as np

import oracle as O


def _kernel_block_scale(m_bits):
    m = (np.asarray(m_bits, dtype=np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore"):
        return (m * (np.float32(1.0) / np.float32(127.0))).astype(np.float16).view(np.uint16)


def test_q8_block_scale_product_matches_oracle_for_every_bf16_maximum():
    m_bits = np.arange(0, 0x7F80, dtype=np.uint32)
    got = _kernel_block_scale(m_bits)
    block = np.zeros(32, dtype=np.uint16)
    for i, b in enumerate(m_bits):
        block[5] = b
        block[17] = b | 0x8000  # a negative key of the same magnitude
        sb, bad, rng = O.k_block_scale(block)
        assert not bad
        assert int(got[i]) == sb, (hex(int(b)), hex(int(got[i])), hex(sb))
        assert rng == ((sb & 0x7C00) == 0x7C00)


def test_q8_block_scale_plain_division_would_differ_in_fp32():
    # The fp32 product and fp32 quotient differ for some maxima; only the
    # fp16 results agree, so the identity above is not a tautology.
    m = (np.arange(0x0080, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    q = m / np.float32(127.0)
    r = m * (np.float32(1.0) / np.float32(127.0))
    assert np.count_nonzero(q != r) > 0
