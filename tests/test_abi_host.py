"""The C-ABI library on a host without a GPU: it loads, exports every symbol that
include/kivi.h declares, and its host-only logic (sizes, n_packed, argument
validation, status strings) behaves as documented. No compute call is made."""
import ctypes
import os
import re

import pytest

import bit_asymmetric_kv_kivi_gb300 as kivi
from bit_asymmetric_kv_kivi_gb300 import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "kivi.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kivi.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kivi_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "kivi_decode_attn" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert lib.kivi_abi_version() == 3


def test_status_strings(lib):
    for s in range(7):
        assert kivi.status_string(s) and kivi.status_string(s) != "unknown status"
    assert kivi.status_string(99) == "unknown status"


def test_seq_bytes_and_n_packed(lib):
    import oracle
    for kb, vb, G, R in ((2, 2, 32, 128), (4, 4, 32, 128), (2, 4, 64, 64), (4, 2, 64, 128), (2, 4, 32, 64)):
        for dt in (kivi.F16, kivi.BF16):
            cfg = kivi.Config(k_bits=kb, v_bits=vb, group=G, residual=R, num_q_heads=32, num_kv_heads=8, dtype=dt)
            ocfg = oracle.Cfg(k_bits=kb, v_bits=vb, group=G, residual=R, num_q_heads=32, num_kv_heads=8, dtype=dt)
            for cap in (0, 64, 4096, 32768):
                assert cfg.seq_bytes(cap) == oracle.seq_bytes(ocfg, cap)
                assert sum(cfg.seq_buffer_bytes(cap)) == cfg.seq_bytes(cap)
            kc, ks, kz, vc, vs, vz, kr, vr = cfg.seq_buffer_bytes(4096)
            assert kc == 8 * 4096 * 128 * kb // 8 and vc == 8 * 4096 * 128 * vb // 8
            assert ks == kz == 8 * (4096 // G) * 128 * 2 and vs == vz == 8 * 4096 * (128 // G) * 2
            assert kr == vr == 8 * (R + G) * 128 * 2
            for L in (0, 1, 63, 64, 127, 128, 159, 160, 161, 1024, 16384 + 511):
                assert cfg.n_packed(L) == oracle.n_packed(ocfg, L)
    assert kivi.Config(group=16).seq_bytes(64) == -1
    assert kivi.Config(group=64).seq_bytes(32) == -1          # capacity not a multiple of G
    assert kivi.Config().n_packed(-1) == -1


@pytest.mark.parametrize("bad", [dict(bits=3), dict(k_bits=8), dict(v_bits=1), dict(group=48), dict(group=128),
                                 dict(residual=100), dict(group=64, residual=96), dict(group=64, head_dim=96),
                                 dict(head_dim=96 + 1), dict(head_dim=512), dict(num_q_heads=6, num_kv_heads=4),
                                 dict(dtype=7), dict(residual=0), dict(num_kv_heads=0)])
def test_bad_config_rejected_before_launch(lib, bad):
    cfg = kivi.Config(**bad).c()
    P = ctypes.c_void_p
    one = P(16)
    assert lib.kivi_quant_keys(cfg, 1, 32, one, one, one, one, None) == kivi.ERR_ARG
    assert lib.kivi_quant_values(cfg, 1, 32, one, one, one, one, None) == kivi.ERR_ARG
    assert lib.kivi_append_flush(cfg, 1, one, one, one, one, one, 1, one, None) == kivi.ERR_ARG
    assert lib.kivi_decode_attn(cfg, 1, one, one, one, one, 0.1, 10, one, 1 << 20, one, None) == kivi.ERR_ARG
    assert lib.kivi_decode_workspace_bytes(cfg, 1, 100) == 0


def test_bad_arguments_rejected_before_launch(lib):
    cfg = kivi.Config(num_q_heads=4, num_kv_heads=1).c()
    P = ctypes.c_void_p
    one, null = P(16), None
    # NULL pointers, negative sizes, tokens not a multiple of G
    assert lib.kivi_quant_keys(cfg, 1, 32, null, one, one, one, None) == kivi.ERR_ARG
    assert lib.kivi_quant_keys(cfg, 1, 48, one, one, one, one, None) == kivi.ERR_ARG
    assert lib.kivi_quant_values(cfg, -1, 32, one, one, one, one, None) == kivi.ERR_ARG
    assert lib.kivi_append_flush(cfg, 2, null, one, one, one, one, 1, one, None) == kivi.ERR_ARG
    assert lib.kivi_append_flush(cfg, 2, one, one, one, one, one, -1, one, None) == kivi.ERR_ARG
    assert lib.kivi_append_flush(cfg, 2, one, one, one, one, one, 1, null, None) == kivi.ERR_ARG
    assert lib.kivi_decode_attn(cfg, 2, one, one, null, one, 0.1, 10, one, 1 << 20, one, None) == kivi.ERR_ARG
    assert lib.kivi_decode_attn(cfg, 2, one, one, one, one, float("nan"), 10, one, 1 << 20, one, None) == kivi.ERR_ARG
    # workspace too small
    need = lib.kivi_decode_workspace_bytes(cfg, 2, 5000)
    assert need > 0
    assert lib.kivi_decode_attn(cfg, 2, one, one, one, one, 0.1, 5000, one, need - 1, one, None) == kivi.ERR_WORKSPACE
    assert lib.kivi_decode_attn(cfg, 2, one, one, one, one, 0.1, 5000, null, need, one, None) == kivi.ERR_WORKSPACE
    # decode supports head_dim 128 and Hq/Hkv up to 32
    assert lib.kivi_decode_attn(kivi.Config(head_dim=64).c(), 1, one, one, one, one, 0.1, 10, one, 1 << 20,
                                one, None) == kivi.ERR_UNSUPPORTED
    assert lib.kivi_decode_attn(kivi.Config(num_q_heads=33).c(), 1, one, one, one, one, 0.1, 10, one, 1 << 20,
                                one, None) == kivi.ERR_UNSUPPORTED
    # zero-sized calls are no-ops that touch nothing
    assert lib.kivi_quant_keys(cfg, 0, 32, null, null, null, null, None) == kivi.OK
    assert lib.kivi_append_flush(cfg, 0, null, null, null, null, null, 0, null, None) == kivi.OK
    assert lib.kivi_decode_attn(cfg, 0, null, null, null, null, 0.1, 0, null, 0, null, None) == kivi.OK


def test_multi_query_arguments_rejected_before_launch(lib):
    cfg = kivi.Config(num_q_heads=8, num_kv_heads=2).c()
    P = ctypes.c_void_p
    one = P(16)
    need = lib.kivi_decode_multi_workspace_bytes(cfg, 2, 4, 5000)
    assert lib.kivi_decode_multi_workspace_bytes(cfg, 2, 8, 5000) > need >= lib.kivi_decode_multi_workspace_bytes(cfg, 2, 3, 5000) > 0
    # one query with a query group of 4 runs the decode kernel, with its workspace
    assert lib.kivi_decode_multi_workspace_bytes(cfg, 2, 1, 5000) == lib.kivi_decode_workspace_bytes(cfg, 2, 5000)
    assert lib.kivi_decode_multi_workspace_bytes(cfg, 2, 0, 5000) == 0
    call = lambda nq, ws=need: lib.kivi_decode_multi_attn(cfg, 2, one, one, nq, one, one, 0.1, 5000, one, ws, one, None)
    assert call(0) == kivi.ERR_ARG
    assert call(9) == kivi.ERR_UNSUPPORTED          # 9 queries x group 4 > 32 (query, head) pairs
    assert call(4, need - 1) == kivi.ERR_WORKSPACE
    assert lib.kivi_decode_multi_attn(kivi.Config(head_dim=64).c(), 1, one, one, 1, one, one, 0.1, 10, one, 1 << 20,
                                      one, None) == kivi.ERR_UNSUPPORTED
    assert lib.kivi_decode_multi_attn(cfg, 0, None, None, 4, None, None, 0.1, 0, None, 0, None, None) == kivi.OK



def test_decode_workspace_plans_by_query_group(lib):
    """The workspace each query group needs, from the documented plans: tickets for two
    streams per (sequence, kv head) in every plan, then fewer than 2 S + 1024 records of
    g (D + 4) floats, S the number of streams: one per kv head for decode at query groups
    1, 2, 4 and 8, one per query and kv head for multi-query calls at groups 4 and 8 and for
    two queries at groups 1 and 2. Other groups and other multi-query calls take the
    multi-query plan, whose size depends on max_kv_len."""
    nseq, H, D = 3, 8, 128
    tickets = ((2 * nseq * H * 4 + 255) // 256) * 256
    for g in (1, 2, 4, 8):
        cfg = kivi.Config(num_q_heads=g * H, num_kv_heads=H).c()
        want = tickets + (2 * nseq * H + 1024) * g * (D + 4) * 4
        assert lib.kivi_decode_workspace_bytes(cfg, nseq, 5000) == want, g
        assert lib.kivi_decode_multi_workspace_bytes(cfg, nseq, 1, 5000) == want, g
    for g, nqs in ((4, range(2, 9)), (8, range(2, 5))):
        cfg = kivi.Config(num_q_heads=g * H, num_kv_heads=H).c()
        for nq in nqs:
            S = nseq * H * nq
            want = tickets + (2 * S + 1024) * g * (D + 4) * 4
            assert lib.kivi_decode_multi_workspace_bytes(cfg, nseq, nq, 5000) == want, (g, nq)
    for g in (1, 2):   # two queries at groups 1 and 2: the decode kernel; more: the multi-query plan
        cfg = kivi.Config(num_q_heads=g * H, num_kv_heads=H).c()
        want = tickets + (2 * nseq * H * 2 + 1024) * g * (D + 4) * 4
        assert lib.kivi_decode_multi_workspace_bytes(cfg, nseq, 2, 5000) == want, g
        assert lib.kivi_decode_multi_workspace_bytes(cfg, nseq, 3, 5000) != lib.kivi_decode_multi_workspace_bytes(cfg, nseq, 3, 50000)
    cfg16 = kivi.Config(num_q_heads=16 * H, num_kv_heads=H).c()
    assert lib.kivi_decode_workspace_bytes(cfg16, nseq, 5000) == lib.kivi_decode_multi_workspace_bytes(cfg16, nseq, 1, 5000)

def test_cfg_struct_matches_header(tmp_path):
    """The binding's kivi_cfg fields: same size and offsets as the C struct."""
    import subprocess
    src = tmp_path / "cfg.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "kivi.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %zu\\n", sizeof(kivi_cfg), '
                   'offsetof(kivi_cfg, k_bits), offsetof(kivi_cfg, v_bits), offsetof(kivi_cfg, group), '
                   'offsetof(kivi_cfg, dtype)); return 0; }\n')
    exe = tmp_path / "cfg"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    size, kb, vb, grp, dt = map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                                     check=True).stdout.split())
    C = kivi._Cfg
    assert size == ctypes.sizeof(C)
    assert (kb, vb, grp, dt) == (C.k_bits.offset, C.v_bits.offset, C.group.offset, C.dtype.offset)
    c = kivi.Config(k_bits=4, v_bits=2, group=64, residual=64).c()
    assert (c.k_bits, c.v_bits, c.group, c.residual) == (4, 2, 64, 64)


def test_seq_record_layout_matches_header(tmp_path):
    """The binding writes kivi_seq records by hand; their size and field offsets must be
    those of the C struct (compiled here from include/kivi.h)."""
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "kivi.h"\n'
                   'int main(void) { printf("%zu %zu %zu %zu %d\\n", sizeof(kivi_seq), '
                   'offsetof(kivi_seq, cap_tokens), offsetof(kivi_seq, flags), '
                   'offsetof(kivi_seq, block_table), KIVI_SEQ_PAGED); return 0; }\n')
    exe = tmp_path / "layout"
    import subprocess
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    size, cap_off, flags_off, table_off, paged = map(int, subprocess.run([str(exe)], capture_output=True, text=True,
                                                                         check=True).stdout.split())
    assert size == kivi.SEQ_STRUCT_BYTES
    assert cap_off == 8 * len(kivi.SEQ_FIELDS) and flags_off == cap_off + 4 and table_off == cap_off + 8
    assert paged == kivi.SEQ_PAGED


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "llama3_8b_kv_bytes.txt")


def test_kv_bytes_plain_matches_the_pages_llama3_8b_table(lib):
    """kivi_kv_bytes_plain against the table printed under Figure 3 of "KV-Cache
    Quantization: I Ran the Experiments So You Don't Have To", "Component 1"
    (Llama-3-8B: 32 layers, 8 kv heads, head_dim 128; decimal GB, one request)."""
    rows = [[float(x) for x in line.split()] for line in open(GOLDEN)
            if line.strip() and not line.startswith("#")]
    assert len(rows) == 4
    for ctx, *gb in rows:
        for bits, want in zip((16, 8, 4, 2), gb):
            got = kivi.kv_bytes_plain(32, 8, 128, bits, int(ctx)) / 1e9
            assert round(got, 2) == want, (ctx, bits, got, want)


def test_kv_bytes_plain_prose_figures(lib):
    """The same section's prose: 128 KiB per token at fp16, about 275 GB for 64 requests at
    32K tokens and about 69 GB at 4-bit; "The memory math (verified)": 17.18 GB (fp16) and
    4.29 GB (4-bit) at 131072 tokens."""
    assert kivi.kv_bytes_plain(32, 8, 128, 16, 1) == 128 * 1024
    assert round(kivi.kv_bytes_plain(32, 8, 128, 16, 32768, 64) / 1e9) == 275
    assert round(kivi.kv_bytes_plain(32, 8, 128, 4, 32768, 64) / 1e9) == 69
    assert round(kivi.kv_bytes_plain(32, 8, 128, 16, 131072) / 1e9, 2) == 17.18
    assert round(kivi.kv_bytes_plain(32, 8, 128, 4, 131072) / 1e9, 2) == 4.29


def test_kv_bytes_plain_rejects_bad_input(lib):
    for bad in [(32, 8, 128, 3, 1, 1), (32, 8, 128, 32, 1, 1), (-1, 8, 128, 2, 1, 1), (32, 8, 128, 2, -5, 1),
                (32, 8, 128, 16, 1 << 40, 1 << 30)]:
        assert kivi.kv_bytes_plain(*bad) == -1, bad
    assert kivi.kv_bytes_plain(32, 8, 128, 2, 0, 7) == 0


def test_no_unsynchronised_static_state_in_the_library_sources():
    """The header says the only state kept between calls is per-device launch settings in
    atomic slots. Every function-scope or file-scope `static` variable in the CUDA sources
    must therefore be constant, atomic, or device memory (the fixed workspace of
    kivi_decode_attn_static, whose host-side address cache is guarded by a mutex)."""
    csrc = os.path.join(os.path.dirname(_build.__file__), "csrc")
    pat = re.compile(r"\bstatic\s+(?!constexpr\b|const\b|inline\b|__device__\b|__host__\b|__forceinline__\b)"
                     r"([A-Za-z_][\w:<>]*)\s+([A-Za-z_]\w*)\s*(\[|=|;)")
    bad = []
    for name in sorted(os.listdir(csrc)):
        text = re.sub(r"//[^\n]*", "", open(os.path.join(csrc, name)).read())
        for m in pat.finditer(text):
            if not m.group(1).startswith("std::atomic"):
                bad.append(f"{name}: {m.group(0)}")
    assert not bad, bad
