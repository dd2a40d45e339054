"""kv_append on the GPU: bit-exact against the oracle's byte copy.

The whole cache is compared, so slots the append must not touch are checked
to keep their sentinel contents.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import bf16_tensor_bits, cuda_or_skip, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,S,Hkv,D", [(1, 256, 1, 128), (64, 2048, 1, 256), (32, 64, 40, 128),
                                       (7, 33, 3, 64), (128, 16, 8, 128)])
def test_append_bit_exact(B, S, Hkv, D):
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    r = np.random.default_rng(B * 1000 + S)
    kc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    vc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    kn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    vn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    pos = r.integers(0, S, B).astype(np.int32)
    pos[0] = S - 1
    ek, ev, skipped = oracle.kv_append(kc, vc, kn, vn, pos)
    assert skipped == 0
    dk, dv = to_dev_bf16(kc, dev), to_dev_bf16(vc, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.kv_append(dk, dv, to_dev_bf16(kn, dev), to_dev_bf16(vn, dev),
                  torch.from_numpy(pos).to(dev), status=status)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_bits(dk), ek)
    assert np.array_equal(bf16_tensor_bits(dv), ev)
    assert status.item() == 0


def test_append_out_of_range_pos_is_skipped_and_flagged():
    import torch
    import kv_cache_decode_gb300 as kvd
    dev = cuda_or_skip()
    B, S, Hkv, D = 5, 8, 2, 64
    r = np.random.default_rng(9)
    kc = r.integers(0, 2**16, (B, S, Hkv, D), dtype=np.uint16)
    vc = kc[::-1].copy()
    kn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    vn = r.integers(0, 2**16, (B, Hkv, D), dtype=np.uint16)
    pos = np.array([0, -1, 8, 7, 100], np.int32)
    ek, ev, skipped = oracle.kv_append(kc, vc, kn, vn, pos)
    assert skipped == 3
    dk, dv = to_dev_bf16(kc, dev), to_dev_bf16(vc, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kvd.kv_append(dk, dv, to_dev_bf16(kn, dev), to_dev_bf16(vn, dev),
                  torch.from_numpy(pos).to(dev), status=status)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_tensor_bits(dk), ek)
    assert np.array_equal(bf16_tensor_bits(dv), ev)
    assert status.item() == kvd.STATUS_POS_OUT_OF_RANGE
