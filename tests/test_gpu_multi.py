"""GPU parity of kivi_decode_multi_attn (the n_query newest tokens of each sequence
attending causally to the packed cache) against the oracle's fp64 multi-query
attention: max |out - oracle| <= 2e-3 over every output element, for both code widths
and their mix, G = 32 and 64, query groups 1/2/4/8 and n_query from 1 to 32 / group,
at the edge lengths of the packed / residual split; the paged layout equal to the
contiguous one bit for bit; short sequences and bad lengths."""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, configs, dev_tensor, record_error

pytestmark = pytest.mark.gpu


def build(wl, kcfg, ocfg, cap, paged=False):
    cache = kivi.KVCache(kcfg, wl.batch, cap, paged=paged, page_seed=3, spare_pages=2)
    refs, ks, vs = [], [], []
    for b, L in enumerate(wl.lengths):
        K, V = wl.kv_seq(b, 0, L)
        ks.append(dev_tensor(K, wl.dtype))
        vs.append(dev_tensor(V, wl.dtype))
        r = oracle.SeqCache(ocfg, cap)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    cache.append(ks, vs)
    return cache, refs


def queries(wl, nq, step=0):
    """[nseq][nq][Hq][D] bit patterns: the queries of the nq newest tokens."""
    return np.stack([np.stack([wl.query(step + i, b) for i in range(nq)]) for b in range(wl.batch)])


def check(wl, cache, refs, nq, step=0):
    qb = queries(wl, nq, step)
    out = cache.decode_multi(dev_tensor(qb, wl.dtype), softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0
    worst = 0.0
    for b, r in enumerate(refs):
        want = r.decode_multi(qb[b], wl.softmax_scale)
        worst = max(worst, float(np.max(np.abs(out[b] - want))))
    record_error(worst)
    assert worst <= ATTN_TOL, worst
    return out


CASES = [  # (k_bits, v_bits, G, R, query group, n_query)
    (2, 2, 32, 128, 4, 1), (2, 2, 32, 128, 4, 2), (2, 2, 32, 128, 4, 4), (2, 2, 32, 128, 4, 8),
    (2, 2, 32, 128, 1, 3), (2, 2, 32, 128, 1, 16), (2, 2, 32, 128, 1, 32), (2, 2, 32, 128, 2, 5),
    (2, 2, 32, 128, 8, 1), (2, 2, 32, 128, 8, 4), (4, 4, 32, 128, 4, 4), (4, 4, 32, 128, 8, 2),
    (2, 2, 64, 64, 4, 4), (4, 2, 64, 64, 2, 7), (2, 4, 32, 64, 4, 8), (4, 2, 32, 128, 1, 12),
    (2, 4, 64, 128, 8, 3), (4, 4, 64, 64, 1, 1),
    # several queries at groups 4 and 8 run on the decode kernel: one stream per query and kv
    # head (the cases above at groups 1 and 2 with more than two queries run on the
    # multi-query kernel)
    (4, 2, 64, 64, 4, 2), (2, 4, 32, 64, 4, 2), (4, 4, 64, 128, 4, 2), (4, 2, 64, 128, 4, 8),
    (2, 2, 32, 128, 4, 3), (4, 4, 64, 64, 4, 5), (2, 2, 32, 128, 8, 3),
    # two queries at groups 1 and 2 also run on the decode kernel
    (2, 2, 32, 128, 1, 2), (4, 4, 64, 64, 2, 2), (2, 4, 32, 128, 2, 2),
]


@pytest.mark.parametrize("kb,vb,G,R,g,nq", CASES)
def test_multi_query_edge_lengths(kb, vb, G, R, g, nq):
    dtype = ("f16", "bf16")[(kb + vb + g + nq) % 2]
    H = 2
    base = {nq, nq + 1, 31, 32, 33, R - 1, R, R + 1, R + G - 1, R + G, R + G + 1, R + 2 * G + nq, 700, 1000 + G // 2}
    lengths = tuple(sorted(L for L in base if L >= nq))
    wl = synth.Workload("multi", len(lengths), g * H, H, 128, lengths, dtype, seed=300 + g + nq + G + kb)
    kcfg, ocfg = configs(2, dtype, g * H, H, G=G, R=R, kb=kb, vb=vb)
    cache, refs = build(wl, kcfg, ocfg, 1024)
    check(wl, cache, refs, nq)


@pytest.mark.parametrize("g,nq", [(4, 4), (8, 2), (1, 8)])
def test_multi_query_long_sequences_many_splits(g, nq):
    """Sequences long enough for several packed splits (1024..4096 tokens each), mixed
    lengths in one batch."""
    H = 2
    lengths = (9000, 4099, 12345, 300)
    wl = synth.Workload("multi-long", len(lengths), g * H, H, 128, lengths, "bf16", seed=400 + g)
    kcfg, ocfg = configs(2, "bf16", g * H, H)
    cache, refs = build(wl, kcfg, ocfg, 12352)
    check(wl, cache, refs, nq)


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16])
def test_multi_query_one_query_matches_decode(g):
    """n_query = 1 is decode attention: both entry points agree with the oracle and with
    each other, bit for bit for query groups 1, 2, 4 and 8 (which run the decode kernel)."""
    H = 2
    lengths = (1, 150, 1000, 5000)
    wl = synth.Workload("multi-one", len(lengths), g * H, H, 128, lengths, "f16", seed=410 + g)
    kcfg, ocfg = configs(2, "f16", g * H, H)
    cache, refs = build(wl, kcfg, ocfg, 5120)
    out = check(wl, cache, refs, 1)
    dec = cache.decode(dev_tensor(queries(wl, 1)[:, 0], "f16"), softmax_scale=wl.softmax_scale).cpu().numpy()
    if g <= 8:
        assert np.array_equal(out[:, 0], dec)
    else:
        assert np.max(np.abs(out[:, 0] - dec)) <= 1e-4


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_one_query_empty_sequence_is_a_length_error(g):
    """With n_query = 1 an empty sequence is a length error (NaN rows, KIVI_ERR_LENGTH),
    where decode gives zeros; the other sequences of the batch are unaffected."""
    H = 2
    lengths = (0, 7, 300)
    wl = synth.Workload("one-empty", len(lengths), g * H, H, 128, lengths, "bf16", seed=450 + g)
    kcfg, ocfg = configs(2, "bf16", g * H, H)
    cache, refs = build(wl, kcfg, ocfg, 320)
    qb = queries(wl, 1)
    out = cache.decode_multi(dev_tensor(qb, "bf16"), softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == kivi.ERR_LENGTH
    assert np.all(np.isnan(out[0]))
    for b in (1, 2):
        err = float(np.max(np.abs(out[b] - refs[b].decode_multi(qb[b], wl.softmax_scale))))
        record_error(err)
        assert err <= ATTN_TOL, err
    cache.status.zero_()
    dec = cache.decode(dev_tensor(qb[:, 0], "bf16"), softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0
    assert np.array_equal(dec[0], np.zeros_like(dec[0]))


@pytest.mark.parametrize("kb,vb,G,R,nq", [(2, 2, 32, 128, 4), (4, 2, 64, 64, 4), (2, 2, 32, 128, 2),
                                          (4, 2, 64, 64, 2)])
def test_multi_query_after_streaming_appends_and_paged_layout(kb, vb, G, R, nq):
    """Verification steps as a speculative decoder runs them: append n_query draft tokens,
    verify them, repeat (with flushes in between); the paged cache gives the same output
    bit for bit."""
    H, g = 2, 4
    lengths = (130, 300, 1000)
    wl = synth.Workload("multi-stream", len(lengths), g * H, H, 128, lengths, "bf16", seed=420 + G)
    kcfg, ocfg = configs(2, "bf16", g * H, H, G=G, R=R, kb=kb, vb=vb)
    cap = 1536
    cont, refs = build(wl, kcfg, ocfg, cap)
    paged, _ = build(wl, kcfg, ocfg, cap, paged=True)
    pos = list(lengths)
    for step in range(12):
        kn, vn = [], []
        for b in range(wl.batch):
            K, V = wl.kv_seq(b, pos[b], nq)
            kn.append(dev_tensor(K, "bf16"))
            vn.append(dev_tensor(V, "bf16"))
            assert refs[b].append(K, V) == oracle.OK
            pos[b] += nq
        cont.append(kn, vn)
        paged.append(kn, vn)
        oc = check(wl, cont, refs, nq, step=10 * step)
        qb = dev_tensor(queries(wl, nq, 10 * step), "bf16")
        op = paged.decode_multi(qb, softmax_scale=wl.softmax_scale).cpu().numpy()
        assert np.array_equal(oc, op), step


@pytest.mark.parametrize("g,nq", [(4, 6), (4, 2), (2, 6)])
def test_multi_query_bad_lengths(g, nq):
    """kv_len below n_query: NaN rows and KIVI_ERR_LENGTH for that sequence only (at query
    group 4 on the decode kernel, at group 2 on the multi-query kernel); n_query * group
    above 32 is refused before launch."""
    H = 1
    lengths = (nq - 1, 200)
    wl = synth.Workload("multi-bad", len(lengths), g * H, H, 128, lengths, "f16", seed=430)
    kcfg, ocfg = configs(2, "f16", g * H, H)
    cache, refs = build(wl, kcfg, ocfg, 256)
    qb = queries(wl, nq)
    out = cache.decode_multi(dev_tensor(qb, "f16"), softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == kivi.ERR_LENGTH
    assert np.all(np.isnan(out[0]))
    want = refs[1].decode_multi(qb[1], wl.softmax_scale)
    assert np.max(np.abs(out[1] - want)) <= ATTN_TOL
    with pytest.raises(kivi.KiviError):
        cache.decode_multi(dev_tensor(np.zeros((2, 32 // g + 1, g, 128), np.uint16), "f16"))


@pytest.mark.parametrize("g,nq", [(4, 2), (4, 3), (2, 3)])
def test_decode_and_multi_query_share_one_workspace(g, nq):
    """kivi_decode_attn and kivi_decode_multi_attn alternate on one cache and one workspace
    (the binding keeps one per cache). With 64 (sequence, kv head) streams the tickets fill
    the first 256 bytes exactly; at query group 4 the queries run the decode kernel over
    nq x 64 streams, at group 2 the multi-query kernel (next to the decode kernel's decode).
    Neither call may leave the other's counters or records disturbed, and decode repeats bit
    for bit."""
    H = 8
    lengths = (700, 1000, 150, 3000, 64, 2000, 999, 128)
    wl = synth.Workload("shared-ws", len(lengths), g * H, H, 128, lengths, "f16", seed=440)
    kcfg, ocfg = configs(2, "f16", g * H, H)
    cache, refs = build(wl, kcfg, ocfg, 3008)
    q1 = dev_tensor(wl.query(5), "f16")
    first = cache.decode(q1, softmax_scale=wl.softmax_scale).cpu().numpy()
    for step in range(3):
        check(wl, cache, refs, nq, step=step)
        again = cache.decode(q1, softmax_scale=wl.softmax_scale).cpu().numpy()
        assert int(cache.status.item()) == 0
        assert np.array_equal(first, again), step
    for b, r in enumerate(refs):
        err = float(np.max(np.abs(first[b] - r.decode(wl.query(5)[b], wl.softmax_scale))))
        record_error(err)
        assert err <= ATTN_TOL, err


@pytest.mark.parametrize("g,nq", [(4, 2), (8, 2), (2, 2), (2, 3)])
def test_plans_with_different_stream_counts_share_one_workspace(g, nq):
    """Calls whose plans count different streams alternate on one workspace: two queries
    run the decode kernel with two streams per kv head next to one-stream decode, and three
    queries at group 2 run the multi-query kernel next to the decode kernel. The
    sequences are long enough that the first CTA writes a partial record right after the
    tickets, so a record region overlapping another plan's tickets would corrupt the next
    call (8000 tokens: about 41 schedule units per CTA, past a stream's 32 units of setup,
    so the first CTA holds packed tiles of stream 0; the multi-query kernel splits each
    sequence nine ways). Every output stays within the bound, and decode repeats bit for
    bit."""
    H = 8
    lengths = (8000,) * 6 + (7000, 6500)
    wl = synth.Workload("plans-ws", len(lengths), g * H, H, 128, lengths, "f16", seed=460 + g)
    kcfg, ocfg = configs(2, "f16", g * H, H)
    cache, refs = build(wl, kcfg, ocfg, 8000)
    q1 = dev_tensor(wl.query(7), "f16")
    first = cache.decode(q1, softmax_scale=wl.softmax_scale).cpu().numpy()
    for step in range(3):
        check(wl, cache, refs, nq, step=step)
        again = cache.decode(q1, softmax_scale=wl.softmax_scale).cpu().numpy()
        assert int(cache.status.item()) == 0
        assert np.array_equal(first, again), step
    for b in (0, 7):
        err = float(np.max(np.abs(first[b] - refs[b].decode(wl.query(7)[b], wl.softmax_scale))))
        record_error(err)
        assert err <= ATTN_TOL, err
