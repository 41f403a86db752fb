"""Fractal flatten / unflatten on the GPU through the C ABI vs the oracle.

A permutation of whole token rows: the result must be bit-exact."""
import numpy as np
import pytest
import torch

from oracle import nabla_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def nabla():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    from block_sparse_attention_nablat_gb300 import nabla as N

    try:
        N.load()
    except RuntimeError:
        __graft_entry__.build()
        N.load()
    return N


CASES = [
    # B, T, H, W, h, D, P, dtype
    (1, 2, 4, 4, 1, 8, 2, torch.float32),      # the golden fixture's shape, tiny rows
    (2, 3, 16, 24, 2, 64, 8, torch.bfloat16),  # ragged patch grid (2 x 3 patches)
    (1, 4, 8, 8, 4, 128, 8, torch.float32),
    (1, 1, 6, 10, 3, 32, 2, torch.bfloat16),   # rows of 192 bytes
    (1, 24, 64, 64, 24, 128, 8, torch.bfloat16),  # the 720p-like latent: 98,304 tokens
]


@pytest.mark.parametrize("B,T,H,W,h,D,P,dt", CASES)
def test_fractal_matches_oracle_and_round_trips(nabla, B, T, H, W, h, D, P, dt):
    g = torch.Generator().manual_seed(B * 1000 + T * 100 + H + W)
    x = torch.randn((B, T, H, W, h, D), generator=g).to(dt)
    xd = x.to(DEV)
    y = nabla.nabla_fractal_flatten(xd, P)
    back = nabla.nabla_fractal_unflatten(y, T, H, W, P)
    torch.cuda.synchronize()
    assert nabla.nabla_get_last_device_status() == 0
    # compare the raw bits (bf16 has no numpy dtype)
    bits = torch.int16 if dt == torch.bfloat16 else torch.int32
    ref = O.fractal_flatten(x.view(bits).numpy(), P)
    assert np.array_equal(y.cpu().view(bits).numpy(), ref)
    assert torch.equal(back.cpu().view(bits), x.view(bits))


def test_fractal_patch_size_one_is_a_plain_copy(nabla):
    x = torch.randn((1, 2, 3, 5, 2, 8), device=DEV)
    y = nabla.nabla_fractal_flatten(x, 1)
    assert torch.equal(y, x.reshape(1, 30, 2, 8))


@pytest.mark.parametrize("bad", ["ragged", "row_bytes", "overlap"])
def test_fractal_rejects_bad_arguments(nabla, bad):
    x = torch.zeros((1, 1, 8, 8, 2, 8), device=DEV)
    with pytest.raises(RuntimeError):
        if bad == "ragged":
            nabla.nabla_fractal_flatten(x, 3)  # 8 is not a multiple of 3
        elif bad == "row_bytes":
            nabla.nabla_fractal_flatten(torch.zeros((1, 1, 8, 8, 1, 3), device=DEV), 8)  # 12 B rows
        else:
            nabla.nabla_fractal_flatten(x, 8, out=x.view(1, 64, 2, 8))
