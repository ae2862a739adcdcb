"""The synthetic weight quantizers (harness steps, not part of the drafter): the
FP4 buffer layout and round-trip error, decoded by the oracle."""
import numpy as np
import torch

from block_diffusion_drafter_fc_gb300 import synth as S
from oracle import dflash_oracle as O


def test_fp4_buffer_size_and_roundtrip_error():
    g = torch.Generator().manual_seed(0)
    w = torch.randn(37, 512, generator=g) * 0.02
    q, s = S.quantize_fp4_rows(w)
    assert q.dtype == torch.uint8 and q.numel() == S.fp4_nbytes(37, 512) == 37 * 256 + 48 * 32
    d = O.decode(q.numpy(), "fp4", s.numpy())
    wb = w.double().numpy().reshape(37, 32, 16)
    amax = np.abs(wb).max(axis=2)
    # E2M1 steps are at most 2 between 4 and 6 (half a step = 1/6 of the block
    # maximum) plus the E4M3 rounding of the block scale (2^-4 relative)
    err = np.abs(d.reshape(37, 32, 16) - wb).max(axis=2) / amax
    assert err.max() <= 1 / 6 * (1 + 2 ** -4) + 2 ** -4


def test_fp4_exact_grid_roundtrips():
    """Weights that are already E2M1 values times a power-of-two block scale (the
    block maximum 6 x scale) come back up to the f32 rounding of the row scale."""
    g = np.random.default_rng(1)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    n, k = 20, 256
    v = grid[g.integers(0, 8, size=(n, k))] * np.where(g.random((n, k)) < 0.5, -1, 1)
    v.reshape(n, k // 16, 16)[:, :, 0] = 6.0          # every block reaches 6
    bscale = 2.0 ** g.integers(-3, 3, size=(n, k // 16))
    w = v * np.repeat(bscale, 16, axis=1) * 2.0 ** -7
    q, s = S.quantize_fp4_rows(torch.from_numpy(w).float())
    d = O.decode(q.numpy(), "fp4", s.numpy())
    assert np.all(np.abs(d - w) <= 2.0 ** -22 * np.abs(w))
    assert np.array_equal(d == 0, w == 0)


def test_fp4_zero_rows():
    w = torch.zeros(3, 64)
    w[1, 5] = 0.25
    q, s = S.quantize_fp4_rows(w)
    d = O.decode(q.numpy(), "fp4", s.numpy())
    assert s[0] == 1.0 and s[2] == 1.0
    assert np.array_equal(d[[0, 2]], np.zeros((2, 64)))
    assert abs(d[1, 5] - 0.25) <= 2.0 ** -22 and np.count_nonzero(d[1]) == 1
