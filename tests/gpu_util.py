"""Helpers shared by the GPU parity tests: moving generator bit patterns to the
device, and comparing library caches with oracle caches."""
import numpy as np
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}
KIVI_DT = {"f16": kivi.F16, "bf16": kivi.BF16}
ORC_DT = {"f16": oracle.F16, "bf16": oracle.BF16}
ATTN_TOL = 2e-3   # max |out - oracle| over every output element (fp32 accumulation vs fp64)
ERRORS: dict = {}  # test id -> largest attention error seen (printed in the terminal summary)


def record_error(err: float) -> None:
    import os
    name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    ERRORS[name] = max(ERRORS.get(name, 0.0), float(err))


def dev_tensor(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """uint16 bit patterns -> torch tensor of `dtype` on `device` (same bits)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(TORCH_DT[dtype]).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def configs(bits, dtype, hq, h, D=128, R=128, G=32, kb=None, vb=None):
    """Library and oracle configs of one setting (kb / vb default to bits)."""
    kb = bits if kb is None else kb
    vb = bits if vb is None else vb
    return (kivi.Config(k_bits=kb, v_bits=vb, head_dim=D, num_q_heads=hq, num_kv_heads=h, dtype=KIVI_DT[dtype],
                        residual=R, group=G),
            oracle.Cfg(k_bits=kb, v_bits=vb, head_dim=D, num_q_heads=hq, num_kv_heads=h, dtype=ORC_DT[dtype],
                       residual=R, group=G))


def assert_state_equal(cache: "kivi.KVCache", b: int, ref: "oracle.SeqCache") -> None:
    """Packed history bit-exact for tokens below n_packed, live ring slots bit-exact, kv_len equal."""
    got = cache.seq_numpy(b)
    L = ref.L
    assert got["kv_len"] == L, (got["kv_len"], L)
    P = oracle.n_packed(ref.cfg, L)
    G = ref.cfg.group
    for name in ("k_codes", "v_codes", "v_scale", "v_zero"):
        np.testing.assert_array_equal(got[name][:, :P], getattr(ref, name)[:, :P], err_msg=name)
    for name in ("k_scale", "k_zero"):
        np.testing.assert_array_equal(got[name][:, :P // G], getattr(ref, name)[:, :P // G], err_msg=name)
    ring = ref.cfg.ring
    slots = [p % ring for p in range(P, L)]
    for name in ("k_res", "v_res"):
        np.testing.assert_array_equal(got[name][:, slots], getattr(ref, name)[:, slots], err_msg=name)
