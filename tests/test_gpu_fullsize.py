"""GPU parity at the full sizes of the large workloads, in the launch configuration
the benchmark uses (whole batch per call). Inputs are drawn on the GPU with the
generator's counters; the sampled sequences' inputs are copied to the host and given
to the oracle, which checks the packed cache bit-exact and the attention outputs of
every query head of those sequences within 2e-3.

  * Llama-3-8B GQA decode: 64 sequences x 32768 tokens, 32/8 heads, bf16, 2-bit
  * long varlen (Mistral-7B shape): 32 sequences, 1024..131072 tokens, fp16, 2-bit
  * streaming append: 16 sequences, 16384-token prefill then 512 decode steps of
    append + attention, 2-bit and 4-bit; the cache is checked bit-exact after every
    flush and attention every 16 steps.
  * the Llama-3-8B GQA batch with the other settings the benchmark takes: G = 64 with
    R = 64, and 4-bit keys with 2-bit values; and its verification step with four draft
    tokens (multi-query attention over the whole batch).
"""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, assert_state_equal, configs, dev_tensor, host_bits, record_error

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draw_seq(wl, b, t0, n):
    """K, V of sequence b, positions [t0, t0+n), all kv heads: [Hkv][n][D] on the GPU."""
    K = torch.stack([synth.torch_kv_head_major(wl, b, h, t0, n, "k", DEV) for h in range(wl.num_kv_heads)])
    V = torch.stack([synth.torch_kv_head_major(wl, b, h, t0, n, "v", DEV) for h in range(wl.num_kv_heads)])
    return K.contiguous(), V.contiguous()


def prefill(cache, wl, lengths, keep=()):
    """Prefill every sequence (eight at a time); returns host copies of the sequences in `keep`."""
    B = wl.batch
    kept = {}
    for b0 in range(0, B, 8):
        bs = list(range(b0, min(B, b0 + 8)))
        ks, vs = {}, {}
        for b in bs:
            ks[b], vs[b] = draw_seq(wl, b, 0, lengths[b])
            if b in keep:
                kept[b] = (host_bits(ks[b]), host_bits(vs[b]))
        empty = torch.empty((wl.num_kv_heads, 0, wl.head_dim), dtype=ks[bs[0]].dtype, device=DEV)
        cache.append([ks.get(b, empty) for b in range(B)], [vs.get(b, empty) for b in range(B)])
        torch.cuda.synchronize()
        del ks, vs
    assert int(cache.status.item()) == 0
    return kept


def oracle_seq(ocfg, cap, K, V):
    r = oracle.SeqCache(ocfg, cap)
    assert r.append(K, V) == oracle.OK
    return r


def check_heads(out_b, ref, q_b, scale):
    want = ref.decode(q_b, scale)
    err = float(np.max(np.abs(out_b - want)))
    record_error(err)
    assert err <= ATTN_TOL, err


def test_llama3_8b_gqa_full_size():
    wl = synth.workload(2)
    L = wl.lengths[0]
    kcfg, ocfg = configs(2, "bf16", 32, 8)
    cache = kivi.KVCache(kcfg, wl.batch, L)
    sample = (0, 37, 63)
    kept = prefill(cache, wl, wl.lengths, keep=sample)
    q = wl.query(0)
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV)
    out = cache.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0 and np.isfinite(out).all()
    for b in sample:
        ref = oracle_seq(ocfg, L, *kept[b])
        assert_state_equal(cache, b, ref)
        check_heads(out[b], ref, q[b], wl.softmax_scale)


def test_long_varlen_full_size():
    wl = synth.workload(4)
    lengths = wl.lengths
    cap = ((max(lengths) + 31) // 32) * 32
    kcfg, ocfg = configs(2, "f16", 32, 8)
    cache = kivi.KVCache(kcfg, wl.batch, cap)
    order = np.argsort(lengths)
    sample = (int(order[-1]), int(order[0]), int(order[len(order) // 2]))
    kept = prefill(cache, wl, lengths, keep=sample)
    q = wl.query(0)
    qd = torch.from_numpy(q.view(np.int16)).view(torch.float16).to(DEV)
    out = cache.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0 and np.isfinite(out).all()
    for b in sample:
        ref = oracle_seq(ocfg, cap, *kept[b])
        assert_state_equal(cache, b, ref)
        check_heads(out[b], ref, q[b], wl.softmax_scale)



@pytest.mark.parametrize("kb,vb,G,R", [(2, 2, 64, 64), (4, 2, 32, 128)])
def test_llama3_8b_gqa_full_size_variants(kb, vb, G, R):
    wl = synth.workload(2)
    L = wl.lengths[0]
    kcfg, ocfg = configs(2, "bf16", 32, 8, G=G, R=R, kb=kb, vb=vb)
    cache = kivi.KVCache(kcfg, wl.batch, L)
    sample = (0, 63)
    kept = prefill(cache, wl, wl.lengths, keep=sample)
    q = wl.query(0)
    qd = torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV)
    out = cache.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0 and np.isfinite(out).all()
    for b in sample:
        ref = oracle_seq(ocfg, L, *kept[b])
        assert_state_equal(cache, b, ref)
        check_heads(out[b], ref, q[b], wl.softmax_scale)


@pytest.mark.parametrize("nq", [2, 4])
def test_verification_step_full_size(nq):
    """Draft tokens (two or four: the decode kernel, one stream per query and kv head)
    appended to every sequence in one call, then their queries attend causally
    (kivi_decode_multi_attn over the whole batch)."""
    wl = synth.workload(2)
    L, B = wl.lengths[0], wl.batch
    cap = L + 32
    kcfg, ocfg = configs(2, "bf16", 32, 8)
    cache = kivi.KVCache(kcfg, B, cap)
    sample = (0, 41, 63)
    kept = prefill(cache, wl, wl.lengths, keep=sample)
    kn, vn = zip(*(draw_seq(wl, b, L, nq) for b in range(B)))
    cache.append(list(kn), list(vn))
    qb = np.stack([np.stack([wl.query(i, b) for i in range(nq)]) for b in range(B)])   # [B][nq][Hq][D]
    out = cache.decode_multi(dev_tensor(qb, "bf16"), softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0 and np.isfinite(out).all()
    for b in sample:
        K = np.concatenate([kept[b][0], host_bits(kn[b])], axis=1)
        V = np.concatenate([kept[b][1], host_bits(vn[b])], axis=1)
        ref = oracle_seq(ocfg, cap, K, V)
        assert_state_equal(cache, b, ref)
        err = float(np.max(np.abs(out[b] - ref.decode_multi(qb[b], wl.softmax_scale))))
        record_error(err)
        assert err <= ATTN_TOL, err

@pytest.mark.parametrize("bits", [2, 4])
def test_streaming_append_full_size(bits):
    wl = synth.workload(3).replace(bits=bits)
    L0, steps, B = wl.lengths[0], wl.steps, wl.batch
    cap = ((L0 + steps + 31) // 32) * 32
    kcfg, ocfg = configs(bits, "f16", 32, 8)
    cache = kivi.KVCache(kcfg, B, cap)
    sample = (0, 11)
    kept = prefill(cache, wl, wl.lengths, keep=sample)
    refs = {b: oracle_seq(ocfg, cap, *kept[b]) for b in sample}
    for b in sample:
        assert_state_equal(cache, b, refs[b])
    # the new tokens of every step, drawn up front: [steps][B][Hkv][1][D]
    H, D = wl.num_kv_heads, wl.head_dim
    kn = torch.empty((steps, B, H, 1, D), dtype=torch.float16, device=DEV)
    vn = torch.empty_like(kn)
    for b in range(B):
        K, V = draw_seq(wl, b, L0, steps)
        kn[:, b, :, 0] = K.transpose(0, 1)
        vn[:, b, :, 0] = V.transpose(0, 1)
    kn_h = {b: host_bits(kn[:, b]) for b in sample}
    vn_h = {b: host_bits(vn[:, b]) for b in sample}
    ones = torch.ones(B, dtype=torch.int32, device=DEV)
    for s in range(steps):
        kp = torch.tensor([kn[s, b].data_ptr() for b in range(B)], dtype=torch.int64, device=DEV)
        vp = torch.tensor([vn[s, b].data_ptr() for b in range(B)], dtype=torch.int64, device=DEV)
        cache.append_ptrs(kp, vp, ones, 1)
        q = wl.query(s)
        out = cache.decode(torch.from_numpy(q.view(np.int16)).view(torch.float16).to(DEV),
                           softmax_scale=wl.softmax_scale)
        for b in sample:
            assert refs[b].append(np.ascontiguousarray(kn_h[b][s]), np.ascontiguousarray(vn_h[b][s])) == oracle.OK
        flushed = (L0 + s + 1 - wl.residual) % wl.group == 0
        if flushed or s % 16 == 15 or s == steps - 1:
            torch.cuda.synchronize()
            assert int(cache.status.item()) == 0
            for b in sample:
                if flushed:
                    assert_state_equal(cache, b, refs[b])
                if s % 16 == 15 or s == steps - 1:
                    check_heads(out[b].cpu().numpy(), refs[b], q[b], wl.softmax_scale)
    for b in sample:
        assert refs[b].L == L0 + steps
        assert oracle.n_packed(ocfg, refs[b].L) == 16256 + 32 * (steps // 32)


def test_maximum_sequence_count():
    """The largest batch the ABI takes (65535 sequences): mostly residual-only sequences
    of 0..47 tokens and 1 % of 150..199 (a packed group or two), one kv head, query group
    4. Prefill, one decode step (append + flush + attention); a seeded sample of sequences
    is checked against the oracle, every output is finite."""
    n, H, g, D = 65535, 1, 4, 128
    rng = np.random.default_rng(2024)
    lengths = rng.integers(0, 48, size=n)
    long = rng.random(n) < 0.01
    lengths[long] = rng.integers(150, 200, size=int(long.sum()))
    lengths[:4] = (0, 1, 159, 160)
    lengths[-1] = 199
    kcfg, ocfg = configs(2, "f16", g * H, H)
    cache = kivi.KVCache(kcfg, n, 96)
    tot = int(lengths.sum())
    K = synth.to_dtype_bits(rng.standard_normal((H, tot, D)) * np.where(np.arange(D) < 3, 20.0, 1.0), "f16")
    V = synth.to_dtype_bits(rng.standard_normal((H, tot, D)), "f16")
    Kd, Vd = dev_tensor(K, "f16"), dev_tensor(V, "f16")
    offs = np.concatenate([[0], np.cumsum(lengths)])
    # one [H][L_b][D] view per sequence, contiguous because H == 1
    cache.append([Kd[:, offs[b]:offs[b + 1]] for b in range(n)], [Vd[:, offs[b]:offs[b + 1]] for b in range(n)])
    step_k = synth.to_dtype_bits(rng.standard_normal((H, 1, D)), "f16")
    step_v = synth.to_dtype_bits(rng.standard_normal((H, 1, D)), "f16")
    kn, vn = dev_tensor(step_k, "f16"), dev_tensor(step_v, "f16")
    cache.append([kn] * n, [vn] * n)
    q = synth.to_dtype_bits(rng.standard_normal((n, g * H, D)), "f16")
    scale = 1.0 / np.sqrt(D)
    out = cache.decode(dev_tensor(q, "f16"), softmax_scale=scale).cpu().numpy()
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    assert np.all(np.isfinite(out))
    sample = sorted(set([0, 1, 2, 3, n - 1] + [int(x) for x in rng.choice(n, 60, replace=False)] +
                        [int(x) for x in np.flatnonzero(long)[:10]]))
    worst = 0.0
    for b in sample:
        r = oracle.SeqCache(ocfg, 96)
        assert r.append(np.ascontiguousarray(K[:, offs[b]:offs[b + 1]]),
                        np.ascontiguousarray(V[:, offs[b]:offs[b + 1]])) == oracle.OK
        assert r.append(step_k, step_v) == oracle.OK
        assert_state_equal(cache, b, r)
        worst = max(worst, float(np.max(np.abs(out[b] - r.decode(q[b], scale)))))
    record_error(worst)
    assert worst <= ATTN_TOL, worst
