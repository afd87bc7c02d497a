"""GPU tests of wo_pack / wo_unpack: bit-exact round trips and the packed
layout itself, byte for byte, against a numpy construction written here from
the layout's definition (include/wo.h, csrc/wo_common.cuh)."""
import numpy as np
import pytest

import oracle
from helpers import to_device_u8

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def wo():
    import weight_only_quantized_fpa_gb300 as w
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w.load_library()
    return w


def expected_packed(codes: np.ndarray, bits: int) -> np.ndarray:
    """Packed bytes from integer codes [n, k], built from the layout's
    definition: 512-byte tiles of 16 channels x KT codes ordered
    [n/16][k/KT]; lane L = 4g + t holds 16 bytes."""
    n, k = codes.shape
    KT = 32 if bits == 8 else 64
    out = np.zeros((n // 16, k // KT, 32, 16), dtype=np.uint8)
    g = np.arange(32) // 4
    t = np.arange(32) % 4
    if bits == 8:
        for b in range(16):
            s, w, j = b >> 3, (b >> 2) & 1, b & 3
            row = g + 8 * (j >> 1)                 # [32]
            kk = 16 * s + 2 * t + 8 * w + (j & 1)  # [32]
            blk = codes.reshape(n // 16, 16, k // KT, KT)
            out[:, :, :, b] = blk[:, row, :, kk].transpose(1, 2, 0)
    else:
        words = np.zeros((n // 16, k // KT, 32, 4), dtype=np.uint32)
        blk = codes.reshape(n // 16, 16, k // KT, KT).astype(np.uint32)
        for s in range(4):
            for p in range(8):
                R, h = p & 3, p >> 2
                row = g + 8 * (R & 1)
                kk = 16 * s + 2 * t + 8 * (R >> 1) + h
                words[:, :, :, s] |= blk[:, row, :, kk].transpose(1, 2, 0) << np.uint32(4 * p)
        out = words.view(np.uint8).reshape(n // 16, k // KT, 32, 16)
    return out.reshape(-1)


def rowmajor_bytes(codes, bits):
    if bits == 8:
        return codes.astype(np.uint8)
    return oracle.pack_nibbles(codes)


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("n,k", [(64, 64), (256, 512), (192, 320)])
def test_pack_layout_matches_definition(wo, bits, n, k):
    rng = np.random.default_rng(n * 7 + k + bits)
    codes = rng.integers(0, 16 if bits == 4 else 256, size=(n, k))
    src = to_device_u8(rowmajor_bytes(codes, bits))
    packed = wo.pack(src, n, k, bits)
    torch.cuda.synchronize()
    assert np.array_equal(packed.cpu().numpy(), expected_packed(codes, bits))


@pytest.mark.parametrize("bits,n,k", [
    (4, 13312, 2048), (4, 2048, 6656), (4, 3072, 2048), (4, 131072, 2048),
    (8, 4608, 3584), (8, 3584, 18944), (8, 2816, 4096), (8, 4096, 1408), (4, 256, 512)])
def test_pack_round_trip_bit_exact(wo, bits, n, k):
    gen = torch.Generator(device="cuda").manual_seed(n + k + bits)
    shape = (n, k) if bits == 8 else (n, k // 2)
    src = torch.randint(0, 256, shape, dtype=torch.uint8, device="cuda", generator=gen)
    packed = wo.pack(src, n, k, bits)
    back = wo.unpack(packed, n, k, bits)
    torch.cuda.synchronize()
    assert torch.equal(back, src)
    assert packed.numel() == src.numel()


def test_pack_is_a_permutation_of_bytes_for_int8(wo):
    n, k = 128, 256
    src = torch.arange(n * k, device="cuda", dtype=torch.int64).remainder(251).to(torch.uint8)
    src = src.reshape(n, k)
    packed = wo.pack(src, n, k, 8)
    torch.cuda.synchronize()
    a = np.sort(packed.cpu().numpy())
    b = np.sort(src.cpu().numpy().reshape(-1))
    assert np.array_equal(a, b)


def test_pack_errors_do_not_launch(wo):
    src = torch.zeros((100, 512), dtype=torch.uint8, device="cuda")
    dst = torch.zeros(100 * 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(wo.WoError):
        wo.wo_pack(src, dst, 100, 512, 8)
