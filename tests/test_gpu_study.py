"""The attention-error study run through the library's GPU codec equals the same study
through the oracle's quantizers (the codes are bit-exact, so the dequantized caches are
identical; only fp64 summation order differs)."""
import pytest

import study
from test_oracle_study import study as oracle_study

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("workload,group", [(1, 32), (2, 32), (2, 64)])
def test_gpu_study_equals_oracle_study(workload, group):
    res = study.run(workload=workload, seqs=1, tokens=512, group=group)
    ref = oracle_study(workload, seqs=1, T=512, group=group)
    assert res["tokens"] == 512
    for r in res["rows"]:
        want = ref[(r["scheme"], r["bits"])]
        got = (r["score_rel_l2"], r["prob_tv"], r["out_rel_l2"])
        for a, b in zip(got, want):
            assert abs(a - b) <= 1e-9 + 1e-6 * abs(b), (r, want)
