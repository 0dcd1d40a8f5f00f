"""Repack, unpack and dequantise on the GPU against the CPU oracle (byte/bit exact)."""
import numpy as np
import pytest

import oracle
from mixed_precision_w4a16_gb300 import synth
import w4a16_testlib as tl

pytestmark = pytest.mark.gpu

SHAPES = [(128, 128, 128), (256, 256, 128), (1024, 1024, 128), (512, 384, -1), (4096, 4096, 128),
          (11008, 256, 128), (1024, 640, 1024)]


@pytest.fixture(scope="module")
def w():
    return tl.lib()


@pytest.mark.parametrize("K,N,G", SHAPES)
def test_repack_matches_oracle_bytes(w, K, N, G):
    q, s = synth.make_weights(K, N, G, seed=K * 7 + N)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    ref_packed, ref_sp = oracle.repack(q, s, G)
    got = packed.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, ref_packed)
    assert np.array_equal(sp.cpu().numpy().view(np.uint16).ravel(), ref_sp.view(np.uint16))
    assert w.w4a16_get_status() == 0


@pytest.mark.parametrize("K,N,G", SHAPES)
def test_unpack_round_trip(w, K, N, G):
    q, s = synth.make_weights(K, N, G, seed=K + 3 * N)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    q2, s2 = w.unpack(packed, sp, K, N, G)
    assert np.array_equal(q2.cpu().numpy(), q)
    assert np.array_equal(s2.cpu().numpy().view(np.uint16), s.view(np.uint16))


@pytest.mark.parametrize("K,N,G", SHAPES)
def test_dequant_bit_exact(w, K, N, G):
    q, s = synth.make_weights(K, N, G, seed=K + N + 1)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    bhat = w.dequant(packed, sp, K, N, G)
    ref = oracle.dequant_fp16_bits(q, s, G)
    assert np.array_equal(bhat.cpu().numpy().view(np.uint16), ref)


def test_dequant_extreme_scales_bit_exact(w):
    # scales near the FP16 range ends: products overflow to inf or land in subnormals;
    # both sides round the same exact product once.
    K, N, G = 256, 256, 128
    q, _ = synth.make_weights(K, N, G, seed=99)
    rng = np.random.default_rng(5)
    pool = np.array([65504.0, 8192.0, 6e-8, 2.0 ** -24, 2.0 ** -14, 1.0 / 3, -0.5, 0.0, 1e-5], np.float16)
    s = rng.choice(pool, size=(K // G, N)).astype(np.float16)
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    bhat = w.dequant(packed, sp, K, N, G)
    assert np.array_equal(bhat.cpu().numpy().view(np.uint16), oracle.dequant_fp16_bits(q, s, G))


def test_code_range_is_flagged_not_trapped(w):
    K, N, G = 128, 128, 128
    q, s = synth.make_weights(K, N, G, seed=1)
    q[5, 7] = 16
    q[100, 127] = 255
    _, _, packed, sp = tl.device_layer(w, q, s, G)
    assert w.w4a16_get_status() == 4  # W4A16_ERR_CODE_RANGE
    assert w.w4a16_get_status() == 0  # read-and-clear
    # the other codes were packed normally (bad ones masked to 4 bits)
    q2, _ = w.unpack(packed, sp, K, N, G)
    expect = q & 15
    assert np.array_equal(q2.cpu().numpy(), expect)


def test_repack_rejects_bad_arguments(w):
    torch = tl.torch_mod()
    q = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.zeros((1, 128), dtype=torch.float16, device="cuda")
    packed = torch.empty(128 * 128 // 8, dtype=torch.int32, device="cuda")
    sp = torch.empty_like(s)
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_repack(q, s, 128, 128, 64, packed, sp)
    assert e.value.status == 3
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_repack(q.data_ptr() + 1, s, 128, 128, 128, packed, sp)
    assert e.value.status == 9
    with pytest.raises(w.W4A16Error) as e:
        w.w4a16_repack(q, s, 128, 64, 128, packed, sp)
    assert e.value.status == 2
