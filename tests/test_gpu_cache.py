"""GPU parity of kivi_append_flush: prefill, streaming and varlen appends give a
cache state bit-identical to the oracle's token-by-token append; capacity and
length errors leave the sequence unchanged and set the status word."""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
from gpu_util import assert_state_equal, configs, dev_tensor
from synth import to_dtype_bits

pytestmark = pytest.mark.gpu


def rand_kv(rng, H, n, D, dtype):
    K = rng.standard_normal((H, n, D))
    K[:, :, :4] *= 20
    V = rng.standard_normal((H, n, D))
    V[:, rng.random(n) < 0.02, :] *= 10
    return to_dtype_bits(K, dtype), to_dtype_bits(V, dtype)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("L", [1, 127, 128, 159, 160, 161, 192, 1000, 2048 + 17])
def test_prefill_bitexact(bits, dtype, L):
    H = 2
    kcfg, ocfg = configs(bits, dtype, 2 * H, H)
    rng = np.random.default_rng(L + 7 * bits)
    K, V = rand_kv(rng, H, L, 128, dtype)
    cap = 2048
    cache = kivi.KVCache(kcfg, 1, cap)
    cache.append(dev_tensor(K, dtype)[None], dev_tensor(V, dtype)[None])
    ref = oracle.SeqCache(ocfg, cap)
    assert ref.append(K, V) == oracle.OK
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    assert_state_equal(cache, 0, ref)


@pytest.mark.parametrize("bits", [2, 4])
def test_streaming_equals_oracle_every_step(bits):
    """Decode-style appends of one token (and random chunks) across several flushes."""
    H, dtype = 2, "f16"
    kcfg, ocfg = configs(bits, dtype, H, H)
    rng = np.random.default_rng(11 + bits)
    n = 420
    K, V = rand_kv(rng, H, n, 128, dtype)
    Kd, Vd = dev_tensor(K, dtype), dev_tensor(V, dtype)
    cache = kivi.KVCache(kcfg, 1, 512)
    ref = oracle.SeqCache(ocfg, 512)
    t = 0
    while t < n:
        m = 1 if t < 250 else int(rng.integers(1, 40))
        m = min(m, n - t)
        cache.append(Kd[:, t:t + m].contiguous()[None], Vd[:, t:t + m].contiguous()[None])
        assert ref.append(np.ascontiguousarray(K[:, t:t + m]), np.ascontiguousarray(V[:, t:t + m])) == oracle.OK
        t += m
        if t % 32 == 0 or t > 250:
            assert_state_equal(cache, 0, ref)
    assert_state_equal(cache, 0, ref)


def test_varlen_batch_with_zero_new_tokens():
    H, dtype = 2, "bf16"
    kcfg, ocfg = configs(2, dtype, 8, H)
    rng = np.random.default_rng(12)
    nseq, cap = 5, 1024
    cache = kivi.KVCache(kcfg, nseq, cap)
    refs = [oracle.SeqCache(ocfg, cap) for _ in range(nseq)]
    for rnd in range(4):
        ns = [int(x) for x in rng.integers(0, 300, nseq)]
        ns[rnd % nseq] = 0
        ks, vs = [], []
        for b in range(nseq):
            K, V = rand_kv(rng, H, ns[b], 128, dtype)
            ks.append(dev_tensor(K, dtype))
            vs.append(dev_tensor(V, dtype))
            assert refs[b].append(K, V) == oracle.OK
        cache.append(ks, vs)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    for b in range(nseq):
        assert_state_equal(cache, b, refs[b])


def test_capacity_overflow_sets_status_and_leaves_sequence_unchanged():
    H, dtype = 1, "f16"
    kcfg, ocfg = configs(2, dtype, 1, H)
    rng = np.random.default_rng(13)
    cache = kivi.KVCache(kcfg, 2, 64)
    refs = [oracle.SeqCache(ocfg, 64) for _ in range(2)]
    K, V = rand_kv(rng, H, 200, 128, dtype)
    cache.append([dev_tensor(K, dtype)] * 2, [dev_tensor(V, dtype)] * 2)
    for r in refs:
        assert r.append(K, V) == oracle.OK
    K2, V2 = rand_kv(rng, H, 30, 128, dtype)                 # sequence 0 would need 96 packed tokens
    K3, V3 = rand_kv(rng, H, 10, 128, dtype)                 # sequence 1 stays within capacity
    cache.append([dev_tensor(K2, dtype), dev_tensor(K3, dtype)], [dev_tensor(V2, dtype), dev_tensor(V3, dtype)])
    assert refs[0].append(K2, V2) == oracle.ERR_CAPACITY
    assert refs[1].append(K3, V3) == oracle.OK
    torch.cuda.synchronize()
    assert int(cache.status.item()) == kivi.ERR_CAPACITY
    assert_state_equal(cache, 0, refs[0])
    assert_state_equal(cache, 1, refs[1])


def test_count_above_max_new_is_a_length_error():
    kcfg, _ = configs(2, "f16", 1, 1)
    cache = kivi.KVCache(kcfg, 1, 64)
    k = torch.zeros((1, 40, 128), dtype=torch.float16, device="cuda")
    kp = torch.tensor([k.data_ptr()], dtype=torch.int64, device="cuda")
    nn = torch.tensor([40], dtype=torch.int32, device="cuda")
    cache.append_ptrs(kp, kp, nn, 16)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == kivi.ERR_LENGTH
    assert int(cache.kv_len.item()) == 0


def test_nothing_packed_beyond_n_packed():
    """The library packs a group exactly when the residual reaches R+G: after every
    append the packed buffers past n_packed(L) keep a sentinel."""
    H, dtype = 2, "f16"
    kcfg, ocfg = configs(2, dtype, 2, H)
    rng = np.random.default_rng(14)
    cache = kivi.KVCache(kcfg, 1, 256)
    for name in ("k_codes", "v_codes"):
        getattr(cache, name).fill_(0xAB)
    for name in ("k_scale", "k_zero", "v_scale", "v_zero"):
        getattr(cache, name).fill_(-21555)          # 0xABCD
    K, V = rand_kv(rng, H, 330, 128, dtype)
    Kd, Vd = dev_tensor(K, dtype), dev_tensor(V, dtype)
    L = 0
    for n in [100, 27, 1, 30, 2] + [1] * 120 + [50]:
        cache.append(Kd[:, L:L + n].contiguous()[None], Vd[:, L:L + n].contiguous()[None])
        L += n
        P = oracle.n_packed(ocfg, L)
        got = cache.seq_numpy(0)
        assert np.all(got["k_codes"][:, P:] == 0xAB) and np.all(got["v_codes"][:, P:] == 0xAB), L
        assert np.all(got["k_scale"][:, P // 32:] == 0xABCD) and np.all(got["v_zero"][:, P:] == 0xABCD), L
