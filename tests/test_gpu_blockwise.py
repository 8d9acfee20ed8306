"""The blockwise 8-bit codec on the GPU against the oracle, bit for bit (GPU)."""

import numpy as np
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from int8_mixed_precision_04_b300 import binding, build
    build.build()
    binding.load()


def _state(n, block, seed):
    """fp32 optimizer-state-like values: a different magnitude per block, an
    all-zero block, exact ties and exact quotients in another."""
    rng = np.random.default_rng(seed)
    nb = (n + block - 1) // block
    mag = 10.0 ** rng.uniform(-9, 3, size=nb)
    x = (rng.standard_normal(n) * np.repeat(mag, block)[:n]).astype(np.float32)
    if nb > 2:
        x[block:2 * block] = 0
    if nb > 3 and n >= 3 * block + 4:
        s = np.float32(2.0 ** -7)
        k = rng.integers(-126, 127, size=block - 1)
        seg = (k + 0.5 * rng.integers(0, 2, size=block - 1)) * s
        x[2 * block] = 127 * s
        x[2 * block + 1:3 * block] = seg[: min(block - 1, n - 2 * block - 1)]
    return x


@pytest.mark.parametrize("n", [1, 7, 8, 256 * 37 + 45, 2048 * 5 + 3, (1 << 22) + 5])
@pytest.mark.parametrize("block", [64, 256, 512, 2048])
def test_blockwise_parity(orc, n, block):
    import torch

    from int8_mixed_precision_04_b300 import binding
    x = _state(n, block, seed=n + block)
    xd = torch.from_numpy(x).cuda()
    q, a = binding.quantize_blockwise(xd, block)
    y = binding.dequantize_blockwise(q, a, block)
    q_o, a_o = orc.quantize_blockwise(x, block)
    y_o = orc.dequantize_blockwise(q_o, a_o, block)
    assert np.array_equal(a.cpu().numpy(), a_o)
    qg = q.cpu().numpy()
    bad = np.nonzero(qg != q_o)[0]
    assert bad.size == 0, f"codes differ at {bad[:8]} (of {bad.size})"
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_o.view(np.uint32))


def test_blockwise_decode_of_oracle_codes(orc):
    """The decoder on codes it did not produce (the oracle's)."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    x = _state(100003, 128, seed=5)
    q_o, a_o = orc.quantize_blockwise(x, 128)
    y = binding.dequantize_blockwise(torch.from_numpy(q_o).cuda(), torch.from_numpy(a_o).cuda(), 128)
    assert np.array_equal(y.cpu().numpy().view(np.uint32),
                          orc.dequantize_blockwise(q_o, a_o, 128).view(np.uint32))


@pytest.mark.parametrize("block", [64, 256, 2048])
def test_blockwise_huge_values(orc, block):
    """States near the top of fp32's range (|x| up to FLT_MAX), where 127 x
    and q a overflow fp32 unless the block is rescaled: codes, scales and
    decoded values equal the oracle's bit for bit, and the absmax codes to
    +-127."""
    import torch

    from int8_mixed_precision_04_b300 import binding
    rng = np.random.default_rng(block)
    nb = 40
    n = nb * block - 3
    fmax = float(np.finfo(np.float32).max)
    mag = np.concatenate([[fmax, 3e38, 2.0 ** 121, 2.0 ** 120, 1.3e36, 2.0 ** 119],
                          10.0 ** rng.uniform(30, 38.5, size=nb - 6)])
    mag = np.minimum(mag, fmax)
    x = (rng.uniform(-1, 1, size=n) * np.repeat(mag, block)[:n]).astype(np.float32)
    for b in range(nb):  # each block reaches its magnitude exactly, some negative
        i = b * block + int(rng.integers(0, min(block, n - b * block)))
        x[i] = np.float32(mag[b] if b % 3 else -mag[b])
    assert np.isfinite(x).all()
    xd = torch.from_numpy(x).cuda()
    q, a = binding.quantize_blockwise(xd, block)
    y = binding.dequantize_blockwise(q, a, block)
    q_o, a_o = orc.quantize_blockwise(x, block)
    y_o = orc.dequantize_blockwise(q_o, a_o, block)
    assert np.array_equal(a.cpu().numpy(), a_o)
    assert np.array_equal(q.cpu().numpy(), q_o)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y_o.view(np.uint32))
    assert np.isfinite(y_o).all()
    qo = q_o.astype(np.int64)
    for b in range(nb):
        seg = np.abs(x[b * block:(b + 1) * block])
        j = int(np.argmax(seg))
        assert abs(qo[b * block + j]) == 127
