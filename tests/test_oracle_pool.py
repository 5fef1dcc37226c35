"""The multi-process oracle harness used by the full-size parity tests.

It must report, per head, exactly the error a direct oracle call gives, and
find a planted mistake on the head where it was planted. CPU only.
"""
import numpy as np
import torch

import oracle
import oracle_pool
import workloads as W


def test_pool_matches_direct_oracle_and_finds_planted_error(tmp_path):
    q, k, v, do = W.make_inputs(W.TINY, seed=11, B=2, H=2, Lq=40, Lk=33, d=64)
    scale = 0.125
    ro, rl = oracle.forward(q, k, v, scale)
    rdq, rdk, rdv = oracle.backward(q, k, v, do, scale)
    # "GPU outputs": the oracle's values rounded to bf16, one element of head
    # (1, 0) of dK off by 0.5.
    o, dq, dk, dv = (torch.tensor(x).to(torch.bfloat16) for x in (ro, rdq, rdk, rdv))
    dk[1, 0, 7, 3] += 0.5
    lse = torch.tensor(rl, dtype=torch.float32)
    heads = [(b, h) for b in range(2) for h in range(2)]
    errs = oracle_pool.head_errors(dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv),
                                   heads, scale, True, str(tmp_path), workers=2)
    assert set(errs) == set(heads)
    for (b, h), e in errs.items():
        sl = (slice(b, b + 1), slice(h, h + 1))
        direct = float(np.abs(dk[sl].double().numpy() - rdk[sl]).max())
        assert e["dk"] == direct
        assert e["o"] <= 2.0 ** -8 * np.abs(ro[sl]).max()
        assert e["lse"] <= 1e-6
    worst = oracle_pool.worst(errs)
    assert worst["dk"][1] == (1, 0) and 0.45 < worst["dk"][0] < 0.55
    assert max(e["dk"] for bh, e in errs.items() if bh != (1, 0)) < 0.02
    assert errs[(1, 0)]["dk_n_over_flat"] == 1 and worst["dk_n_over_flat"] == 1
    # the rounding-model option: the planted element exceeds its limit, the
    # bf16-rounded oracle values do not
    errs = oracle_pool.head_errors(dict(q=q, k=k, v=v, do=do, o=o, lse=lse, dq=dq, dk=dk, dv=dv),
                                   heads, scale, True, str(tmp_path), workers=2, model=True)
    assert errs[(1, 0)]["dk_n_over_model"] == 1
    assert all(e["dq_n_over_model"] == 0 and e["dv_n_over_model"] == 0 for e in errs.values())
    assert all(e["dk_n_over_model"] == 0 for bh, e in errs.items() if bh != (1, 0))
