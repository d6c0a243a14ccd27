"""kda_linear (the in_proj / o_proj projections) against the projection
oracle: bf16 outputs within one bf16 step of the correctly rounded product,
plus the fp32 accumulation's share (2^-14 of sum |x_k w_k|); the in_proj and
o_proj shapes of the 12-head layer through the 16-row mma.sync tile (rows <=
16) and every tcgen05 tile shape (more rows), ragged column tails (odd N),
ragged K, K splits, a strided x."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import linear_attention_decode_03_gb300 as kda
from linear_attention_decode_03_gb300.inputs import to_bf16_bits
from oracle import linear as OL
from tests import gpu_harness as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.build()
    kda.load_library()


def _check(rows, K, N, seed, wscale=0.02, xcols=None):
    rng = np.random.default_rng(seed)
    x = to_bf16_bits(rng.normal(0.0, 1.0, size=(rows, xcols or K)).astype(np.float32))
    w = to_bf16_bits(rng.normal(0.0, wscale, size=(N, K)).astype(np.float32))
    xd = G.bf16_np_to_torch(x, "cuda")[:, :K]
    wd = G.bf16_np_to_torch(w, "cuda")
    y = G.torch_bf16_to_np(kda.linear(xd, wd))
    assert kda.kda_linear_check() == 0
    ref = OL.linear(np.ascontiguousarray(x[:, :K]), w)
    scale = OL.abs_products(np.ascontiguousarray(x[:, :K]), w)
    g, r = G.bf16_value(y), G.bf16_value(ref)
    ulp = np.maximum(np.abs(r), 1e-30) * 2.0 ** -7
    bound = ulp + 2.0 ** -14 * scale
    diff = np.abs(g - r)
    assert np.all(np.isfinite(g))
    assert np.all(diff <= bound), f"worst {diff.max()} (bound there {bound.flat[np.argmax(diff - bound)]})"
    return np.mean(y != ref)


@pytest.mark.parametrize("rows", [1, 8, 64])
def test_in_proj_shape(rows):
    # x [rows, 7168] . W_in [6284, 7168]^T -> the packed projection row (pitch 6284 at 12 heads)
    _check(rows, 7168, 6284, seed=rows)


@pytest.mark.parametrize("rows", [1, 64, 256])
def test_o_proj_shape(rows):
    # core_out [rows, 1536] . W_o [7168, 1536]^T; 256 rows: two tcgen05 row tiles
    _check(rows, 1536, 7168, seed=100 + rows, wscale=0.05)


def test_in_proj_tensor_core_tiles():
    # 160 rows: tcgen05 tiles, a full 128-row tile and a 32-row one (rows past 160 zero-filled)
    _check(160, 7168, 6284, seed=160)


def test_several_row_tiles_ragged_tail_and_strided_x():
    _check(130, 256, 99, seed=7, xcols=320)   # 2 row tiles (the second 2 rows), one 99-column tile


@pytest.mark.parametrize("rows,K,N", [(16, 512, 77), (17, 384, 77), (5, 200, 45), (20, 328, 70), (1, 8, 33),
                                     (3, 7168, 1154), (2, 128, 5000), (300, 256, 600), (257, 1536, 300)])
def test_row_tile_boundaries_ragged_k_and_k_splits(rows, K, N):
    # 16 rows: the mma.sync one-tile shape; 17: tcgen05 tiles; K = 200, 328, 8 end in a
    # partial k stage (zero-filled past K); 1154 columns (the 2-head in_proj)
    # split K eight ways; K = 128 is a single stage, so no split; 300 and 257 rows: three
    # tcgen05 row tiles, the last one mostly past the end
    _check(rows, K, N, seed=rows * 1000 + N, xcols=K + 8)


# Shapes that the launcher's time model sends (on 152 SMs) to each tcgen05 tile instance,
# unsplit and with a K split, every one with a ragged last column tile and (most) a ragged
# last k stage, so that every instance and both epilogues are compared with the oracle:
# rows x columns of the tile, K split
TILE_SHAPES = [
    (17, 328, 1000),      # 128 x 128, C = 6
    (17, 200, 19648),     # 128 x 192, C = 1
    (17, 1000, 6439),     # 128 x 192, C = 4
    (130, 200, 14986),    # 128 x 256, C = 1
    (17, 1000, 10324),    # 128 x 256, C = 3
    (130, 200, 19648),    # 256 x 192, C = 1
    (130, 8200, 4829),    # 256 x 192, C = 5
    (257, 200, 16540),    # 256 x 256, C = 1
    (130, 7176, 7160),    # 256 x 256, C = 5
]


@pytest.mark.parametrize("rows,K,N", TILE_SHAPES)
def test_each_tile_shape(rows, K, N):
    _check(rows, K, N, seed=rows + N, xcols=K + 8)


def test_rejects_bad_shapes():
    x = torch.zeros((4, 100), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((8, 100), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kda.KdaError):
        kda.linear(x, w)  # K = 100: weight rows of 200 bytes, not a multiple of 16


def test_host_memory_rejected():
    """kda_linear reads x and W through tensor maps and writes y with plain
    stores, on this GPU's own memory only: pinned or pageable host buffers,
    for any operand, are rejected with KDA_EINVAL before anything is enqueued."""
    rows, K, N = 4, 256, 64
    xd = torch.zeros((rows, K), dtype=torch.bfloat16, device="cuda")
    wd = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    yd = torch.zeros((rows, N), dtype=torch.bfloat16, device="cuda")
    for host in (torch.zeros((rows * N + N * K,), dtype=torch.bfloat16).pin_memory(),
                 torch.zeros((rows * N + N * K,), dtype=torch.bfloat16)):
        hp = host.data_ptr()
        for args in ((hp, wd.data_ptr(), yd.data_ptr()), (xd.data_ptr(), hp, yd.data_ptr()),
                     (xd.data_ptr(), wd.data_ptr(), hp)):
            x, w, y = args
            with pytest.raises(kda.KdaError) as ei:
                kda.kda_linear(x, rows, K, w, N, K, y, N)
            assert ei.value.code == -1
    kda.linear(xd, wd, yd)
    assert kda.kda_linear_check() == 0
