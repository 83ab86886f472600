"""GPU parity: the packer is byte-identical to the oracle's packer, the
device decode routine gives back the codes byte for byte, and the device-side
input generator equals the host one."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Mat, SEED, dev, qmv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,K,bits", [(1, 64, 2), (3, 128, 2), (33, 1024, 2), (257, 2048, 4),
                                      (5, 5376, 4), (7, 5376, 8), (64, 96, 8), (100, 14336, 2)])
def test_packer_bit_exact(N, K, bits):
    codes = synth.codes(SEED, f"pk{N}x{K}b{bits}", N, K, bits)
    scales = synth.scales(SEED, f"pk{N}x{K}b{bits}", N, K // 32)
    p = qmv().Pack(N, K, bits, 32).pack_weights(codes.to(dev()), scales.to(dev()))
    torch.cuda.synchronize()
    words = p.words.cpu().numpy().view(np.uint32).reshape(N, K * bits // 32)
    assert np.array_equal(words, oracle.pack(codes.numpy(), bits))
    assert np.array_equal(p.scales.cpu().numpy().view(np.uint16),
                          scales.numpy().view(np.uint16).ravel())
    back = qmv().qmv_unpack_codes(p)
    torch.cuda.synchronize()
    assert np.array_equal(back.cpu().numpy(), codes.numpy())


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_decode_every_word_pattern(bits):
    # every 16-bit half pattern in both halves of a word: 65536 words
    K = 32 // bits * 1024
    w = np.arange(65536, dtype=np.uint32)
    words = (w | (w[::-1] << 16)).reshape(64, -1)
    codes = oracle.unpack(words, K, bits)
    p = qmv().Pack(64, K, bits, 32).pack_weights(torch.from_numpy(codes).to(dev()),
                                                 torch.zeros(64, K // 32, dtype=torch.float16,
                                                             device=dev()))
    back = qmv().qmv_unpack_codes(p)
    torch.cuda.synchronize()
    assert np.array_equal(p.words.cpu().numpy().view(np.uint32).reshape(words.shape), words)
    assert np.array_equal(back.cpu().numpy(), codes)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_device_generator_matches_host(bits):
    N, K = 300, 2048
    rows = np.array([0, 5, 299])
    a = synth.codes(SEED, "gen", N, K, bits, device=dev()).cpu().numpy()
    b = synth.codes(SEED, "gen", N, K, bits).numpy()
    assert np.array_equal(a, b)
    assert np.array_equal(a[rows], synth.codes(SEED, "gen", N, K, bits, rows=rows).numpy())
    s1 = synth.scales(SEED, "gen", N, 64, device=dev()).cpu().numpy()
    s2 = synth.scales(SEED, "gen", N, 64).numpy()
    assert np.array_equal(s1.view(np.uint16), s2.view(np.uint16))
    assert s2.min() >= np.float16(0.005) and s2.max() <= np.float16(0.02)


@pytest.mark.parametrize("N,K,bits,group", [(300, 2048, 2, 32), (257, 5376, 4, 32), (65, 2048, 8, 2048)])
def test_saved_pack_reloads_bit_exact(tmp_path, N, K, bits, group):
    # save = header + the packed words and scales as the packer left them;
    # reload into fresh device buffers, bind without packing, and the matvec
    # is bit-identical to the original pack's (and to the oracle in exact mode)
    from gpu_util import acts, bits_equal, first_diff, to_dev
    q = qmv()
    m = Mat(f"save{N}x{K}b{bits}", N, K, bits, group)
    path = tmp_path / "w.qmvpack"
    with open(path, "wb") as f:
        f.write(m.pack.header())
        f.write(m.pack.words.cpu().numpy().tobytes())
        f.write(m.pack.scales.cpu().numpy().tobytes())
    blob = path.read_bytes()
    r = q.Pack.from_header(blob[:q.QMV_PACK_HEADER_BYTES])
    assert (r.N, r.K, r.bits, r.group) == (N, K, bits, group)
    assert len(blob) == q.QMV_PACK_HEADER_BYTES + r.codes_bytes + r.scales_bytes
    off = q.QMV_PACK_HEADER_BYTES
    words = torch.frombuffer(bytearray(blob[off:off + r.codes_bytes]), dtype=torch.int32).to(dev())
    scales = torch.frombuffer(bytearray(blob[off + r.codes_bytes:]), dtype=torch.float16).to(dev())
    r.bind_packed(words, scales)
    x, _, _ = acts(f"save{N}x{K}", 1, K)
    y0 = q.qmv_gemv(m.pack, to_dev(x), mode=q.QMV_EXACT)
    y1 = q.qmv_gemv(r, to_dev(x), mode=q.QMV_EXACT)
    torch.cuda.synchronize()
    assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
    codes, sc = m.host()
    ref = oracle.gemv(codes, sc, group, x)
    got = y1.cpu().numpy()
    assert bits_equal(got, ref), first_diff(got, ref)
    assert q.qmv_device_error(clear=True) == 0
