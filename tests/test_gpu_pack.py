"""Weight repack on the GPU: the packed layout decodes back to the oracle's fields."""
import numpy as np
import pytest
import torch

from oracle import q4k_blocks

pytestmark = pytest.mark.gpu


def _bf16(u):
    return (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("n,k,seed", [(256, 512, 0), (128, 256, 1), (384, 768, 2)])
def test_pack_layout_round_trip(n, k, seed):
    from quantized_prefill_gemm_gb300 import inputs, q4k

    from tests.gpu_common import to_dev

    blocks = inputs.q4k_blocks(n, k, seed)
    packed = q4k.q4k_pack_weights(to_dev(blocks), n, k)
    torch.cuda.synchronize()
    pk = packed.cpu().numpy()
    f = q4k_blocks.decode(blocks)
    kc, ksb, nt = k // 32, k // 256, n // 128
    align = lambda v: (v + 1023) // 1024 * 1024
    off_sc = align(n * k // 2)
    off_d = align(off_sc + n * kc)
    off_ndm = align(off_d + n * ksb * 4)
    # quants: [nt][kc][128][16 B]; word i = k-group i; nibble at bits 4j -> k 8i+2j, 16+4j -> 8i+2j+1
    nib = pk[: n * k // 2].reshape(nt, kc, 128, 4, 4).view(np.uint32)[..., 0]  # [nt][kc][128][4 words]
    q = np.zeros((nt, kc, 128, 32), np.uint8)
    for i in range(4):
        for j in range(4):
            q[..., 8 * i + 2 * j] = (nib[..., i] >> (4 * j)) & 15
            q[..., 8 * i + 2 * j + 1] = (nib[..., i] >> (16 + 4 * j)) & 15
    q = q.transpose(0, 2, 1, 3).reshape(n, k)
    assert np.array_equal(q, f["q"])
    sc = pk[off_sc: off_sc + n * kc].reshape(nt, kc, 128).transpose(0, 2, 1).reshape(n, kc)
    assert np.array_equal(sc, f["sc"])
    d = pk[off_d: off_d + n * ksb * 4].view(np.float32).reshape(nt, ksb, 128).transpose(0, 2, 1).reshape(n, ksb)
    assert np.array_equal(d.astype(np.float64), q4k_blocks.f16_bits_to_f64(f["d_bits"]))
    ndm = pk[off_ndm: off_ndm + 4 * n * kc].view(np.uint16).reshape(2, n, kc)
    want = -np.repeat(q4k_blocks.f16_bits_to_f64(f["dmin_bits"]), 8, axis=1) * f["m"].astype(np.float64)
    got = _bf16(ndm[0]) + _bf16(ndm[1])
    assert np.all(np.abs(got - want) <= 2.0 ** -16 * np.abs(want))
    # small-M sections: the 6-bit m per (row, chunk) and the fp32 dmin per (row, super-block)
    off_mq = align(off_ndm + 4 * n * kc)
    off_dmn = align(off_mq + n * kc)
    mq = pk[off_mq: off_mq + n * kc].reshape(nt, kc, 128).transpose(0, 2, 1).reshape(n, kc)
    assert np.array_equal(mq, f["m"])
    dmn = pk[off_dmn: off_dmn + n * ksb * 4].view(np.float32).reshape(nt, ksb, 128).transpose(0, 2, 1).reshape(n, ksb)
    assert np.array_equal(dmn.astype(np.float64), q4k_blocks.f16_bits_to_f64(f["dmin_bits"]))
    assert packed.numel() == align(off_dmn + n * ksb * 4)
