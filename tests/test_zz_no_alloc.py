"""kivi_decode_attn_static: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: their device memory is
already reserved by another allocator (a serving framework's pool), or they run
on a latency-critical path that must not allocate or free (cudaFree synchronizes
the device), or they sit behind a plugin interface that passes only inputs and
outputs. kivi_decode_attn_static serves them with a fixed workspace inside the
library. This test calls it through the C ABI, twice in a row, and checks its
output against kivi_decode_attn with a caller workspace, within the attention
tolerance of the other tests. The file name makes pytest collect it last.
"""
import ctypes

import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import synth
from gpu_util import ATTN_TOL, configs, dev_tensor

pytestmark = pytest.mark.gpu


def _lib():
    L = kivi.lib()
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    L.kivi_decode_attn_static.argtypes = [ctypes.POINTER(kivi._Cfg), I32, P, P, P, P, ctypes.c_float, I32, P, P]
    L.kivi_decode_attn_static.restype = I32
    return L


def test_static_workspace_matches_caller_workspace():
    wl = synth.Workload("noalloc", 3, 16, 4, 128, (9000, 300, 20000), "f16", seed=77)
    kcfg, _ = configs(2, "f16", 16, 4)
    cache = kivi.KVCache(kcfg, 3, 20000)
    ks, vs = [], []
    for b in range(3):
        K, V = wl.kv_seq(b, 0, wl.lengths[b])
        ks.append(dev_tensor(K, "f16"))
        vs.append(dev_tensor(V, "f16"))
    cache.append(ks, vs)
    q = dev_tensor(wl.query(0), "f16")
    want = cache.decode(q, softmax_scale=wl.softmax_scale)         # caller-provided workspace
    L = _lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):                                              # two calls in a row share the array
        out = torch.full_like(want, float("nan"))
        rc = L.kivi_decode_attn_static(kcfg.c(), 3, cache.seqs.data_ptr(), cache.kv_len.data_ptr(), q.data_ptr(),
                                       out.data_ptr(), wl.softmax_scale, cache.max_len,
                                       cache.status.data_ptr(), stream)
        assert rc == kivi.OK, kivi.status_string(rc)
        torch.cuda.synchronize()
        assert int(cache.status.item()) == 0
        err = float((out - want).abs().max().item())
        assert err <= ATTN_TOL, err


def test_static_workspace_rejects_sizes_beyond_its_maximum():
    kcfg, _ = configs(2, "f16", 32, 8)
    L = _lib()
    nseq, max_len = 4096, 131072
    assert kcfg.decode_workspace_bytes(nseq, max_len) > (16 << 20)
    one = ctypes.c_void_p(16)
    rc = L.kivi_decode_attn_static(kcfg.c(), nseq, one, one, one, one, 0.1, max_len, one, None)
    assert rc == kivi.ERR_WORKSPACE


def test_static_workspace_query_group_8():
    """Query group 8 runs on the multi-query kernel; the fixed workspace serves it too."""
    wl = synth.Workload("noalloc8", 2, 16, 2, 128, (5000, 700), "bf16", seed=78)
    kcfg, _ = configs(2, "bf16", 16, 2)
    cache = kivi.KVCache(kcfg, 2, 5024)
    cache.append([dev_tensor(wl.kv_seq(b, 0, wl.lengths[b])[0], "bf16") for b in range(2)],
                 [dev_tensor(wl.kv_seq(b, 0, wl.lengths[b])[1], "bf16") for b in range(2)])
    q = dev_tensor(wl.query(0), "bf16")
    want = cache.decode(q, softmax_scale=wl.softmax_scale)
    out = torch.full_like(want, float("nan"))
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = _lib().kivi_decode_attn_static(kcfg.c(), 2, cache.seqs.data_ptr(), cache.kv_len.data_ptr(), q.data_ptr(),
                                        out.data_ptr(), wl.softmax_scale, cache.max_len, cache.status.data_ptr(),
                                        stream)
    assert rc == kivi.OK, kivi.status_string(rc)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    assert float((out - want).abs().max().item()) <= ATTN_TOL
