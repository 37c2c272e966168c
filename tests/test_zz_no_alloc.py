"""kivi_decode_attn_static: decode attention for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc: their device memory is
already reserved by another allocator (a serving framework's pool), or they run
on a latency-critical path that must not allocate or free (cudaFree synchronizes
the device), or they sit behind a plugin interface that passes only inputs and
outputs. kivi_decode_attn_static serves them with a fixed workspace inside the
library. These tests call it through the C ABI, twice in a row, and require its
output to equal kivi_decode_attn with a caller workspace bit for bit (both run the
same kernels on the same plan; a stale ticket or record left in the shared array
would show up as a difference) and to match the oracle within the attention
tolerance of the other tests. The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, configs, dev_tensor

pytestmark = pytest.mark.gpu


def _lib():
    L = kivi.lib()
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    L.kivi_decode_attn_static.argtypes = [ctypes.POINTER(kivi._Cfg), I32, P, P, P, P, ctypes.c_float, I32, P, P]
    L.kivi_decode_attn_static.restype = I32
    return L


def _run(wl, dtype, nseq_cap):
    kcfg, ocfg = configs(2, dtype, wl.num_q_heads, wl.num_kv_heads)
    cache = kivi.KVCache(kcfg, wl.batch, nseq_cap)
    ks, vs, refs = [], [], []
    for b in range(wl.batch):
        K, V = wl.kv_seq(b, 0, wl.lengths[b])
        ks.append(dev_tensor(K, dtype))
        vs.append(dev_tensor(V, dtype))
        ref = oracle.SeqCache(ocfg, nseq_cap)
        assert ref.append(K, V) == oracle.OK
        refs.append(ref)
    cache.append(ks, vs)
    q_np = wl.query(0)
    q = dev_tensor(q_np, dtype)
    want = cache.decode(q, softmax_scale=wl.softmax_scale)          # caller-provided workspace
    torch.cuda.synchronize()
    oerr = max(float(np.max(np.abs(want[b].cpu().numpy() - refs[b].decode(q_np[b], wl.softmax_scale))))
               for b in range(wl.batch))
    assert oerr <= ATTN_TOL, oerr
    L = _lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):                                              # two calls in a row share the array
        out = torch.full_like(want, float("nan"))
        rc = L.kivi_decode_attn_static(kcfg.c(), wl.batch, cache.seqs.data_ptr(), cache.kv_len.data_ptr(),
                                       q.data_ptr(), out.data_ptr(), wl.softmax_scale, cache.max_len,
                                       cache.status.data_ptr(), stream)
        assert rc == kivi.OK, kivi.status_string(rc)
        torch.cuda.synchronize()
        assert int(cache.status.item()) == 0
        assert torch.equal(out, want), float((out - want).abs().max().item())


def test_static_workspace_matches_caller_workspace():
    """Query group 4: the persistent decode kernel."""
    wl = synth.Workload("noalloc", 3, 16, 4, 128, (9000, 300, 20000), "f16", seed=77)
    _run(wl, "f16", 20000)


def test_static_workspace_query_group_8():
    """Query group 8, bf16 inputs."""
    wl = synth.Workload("noalloc8", 2, 16, 2, 128, (5000, 700), "bf16", seed=78)
    _run(wl, "bf16", 5024)


def test_static_workspace_query_group_6():
    """Query group 6: decode on the multi-query kernel, whose tickets the entry point also clears."""
    wl = synth.Workload("noalloc6", 3, 12, 2, 128, (4000, 33, 7000), "f16", seed=79)
    _run(wl, "f16", 7040)


def test_static_workspace_rejects_sizes_beyond_its_maximum():
    kcfg, _ = configs(2, "f16", 32, 8)
    L = _lib()
    nseq, max_len = 4096, 131072
    assert kcfg.decode_workspace_bytes(nseq, max_len) > (16 << 20)
    one = ctypes.c_void_p(16)
    rc = L.kivi_decode_attn_static(kcfg.c(), nseq, one, one, one, one, 0.1, max_len, one, None)
    assert rc == kivi.ERR_WORKSPACE
