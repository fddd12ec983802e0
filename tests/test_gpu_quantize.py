"""quantize_q_fp8 on the GPU is bit-exact against the oracle quantizer over
every bf16 bit pattern (normals, subnormals, +-0, +-inf, NaNs) and descales
that exercise ties, saturation and underflow."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("descale", [1.0, 3.7 / 448, 2.0 ** -10, 1000.0, 0.0123456, 1.0 / 3.0,
                                     35.0 / 448, 5.0, 3.0 / 64, 0.75, 2.0 ** -64, 2.0 ** 64, 2.0 ** -65, 2.0 ** 65,
                                     1e-30, 3.1e18, (1 - 2.0 ** -24) * 4, (9 * 2 ** 20 - 3) * 2.0 ** -27,
                                     (13 * 2 ** 20 + 7) * 2.0 ** -23])
def test_quantize_all_bf16_patterns_bit_exact(descale):
    import fp8_paged_attention_gb300 as fp8pa
    bits = np.arange(65536, dtype=np.uint16)
    q = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    d = torch.tensor([descale], dtype=torch.float32, device="cuda")
    got = fp8pa.quantize_q_fp8(q, d).cpu().numpy()
    want = oracle.quantize_q(bits, float(np.float32(descale)))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(int(bits[i])), hex(int(got[i])), hex(int(want[i]))) for i in bad[:10]]


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 4097])
def test_quantize_ragged_lengths_and_unaligned(n):
    import fp8_paged_attention_gb300 as fp8pa
    rng = np.random.default_rng(n)
    x = torch.from_numpy(rng.standard_normal(n + 3).astype(np.float32)).to(torch.bfloat16).cuda()
    d = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    for off in (0, 1):  # offset 1 forces the unaligned scalar path
        src = x[off:off + n]
        out = torch.full((n + 1,), 0xAA, dtype=torch.uint8, device="cuda")
        fp8pa.quantize_q_fp8(src.contiguous() if off == 0 else src, d, out=out[off:off + n])
        want = oracle.quantize_q(src.cpu().view(torch.int16).numpy().view(np.uint16), 0.01)
        assert np.array_equal(out[off:off + n].cpu().numpy(), want)
        if off == 0:
            assert out[n].item() == 0xAA   # no write past the end


@pytest.mark.parametrize("descale", [3.7 / 448, 35.0 / 448])
def test_quantize_input_larger_than_one_grid_pass_bit_exact(descale):
    """An input larger than one pass of the quantizer's grid (4096 blocks x 256
    threads x 8 elements), which loads four vectors per thread before
    converting, with a partial last pass and a scalar tail (length not a
    multiple of 8): every element, of random bit patterns (NaNs and
    infinities included), against the oracle."""
    import fp8_paged_attention_gb300 as fp8pa
    n = 4096 * 256 * 8 * 2 + 8 * 12345 + 5
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 65536, size=n, dtype=np.uint16)
    q = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    d = torch.tensor([descale], dtype=torch.float32, device="cuda")
    got = fp8pa.quantize_q_fp8(q, d).cpu().numpy()
    want = oracle.quantize_q(bits, float(np.float32(descale)))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(int(i), hex(int(bits[i])), hex(int(got[i])), hex(int(want[i]))) for i in bad[:10]]
