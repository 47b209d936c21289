"""The process pool the full-size parity tests use (CPU only): its per-head
error sums equal a direct comparison, and a planted error in one element of
one head is found."""
import math

import numpy as np

import oracle
from sdpa_inputs import make_random
from tests.oracle_pool import backward_head, forward_head, make_pool


def test_pool_error_sums_equal_a_direct_comparison():
    B, H, N, d = 1, 3, 70, 16
    q, k, v, do = (make_random((B, H, N, d), 900 + i) for i in range(4))
    s = 1 / math.sqrt(d)
    O, lse = oracle.attention_forward(q, k, v, s, True)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, s, True)
    O = O.astype(np.float32)
    O[0, 2, 33, 5] += 0.25  # planted error: one element of one head
    tasks = [(q[0, h], k[0, h], v[0, h], do[0, h], O[0, h], lse[0, h], dq[0, h], dk[0, h], dv[0, h], s, True, h)
             for h in range(H)]
    pool, n = make_pool(1 << 20)
    assert n >= 1
    with pool:
        parts = pool.map(backward_head, tasks)
        fparts = pool.map(forward_head, [t[:3] + t[4:6] + (s, True, 0, d, t[-1]) for t in tasks])
    assert [p["o_max"] > 0.2 for p in parts] == [False, False, True]
    assert abs(max(p["o_max"] for p in parts) - 0.25) < 1e-6
    assert parts[2]["o_max_at"][:2] == (33, 5) and parts[2]["head"] == 2
    direct = np.abs(O.astype(np.float64) - oracle.attention_forward(q, k, v, s, True)[0])
    assert abs(sum(p["o_sum"] for p in parts) - direct.sum()) < 1e-9
    assert sum(p["o_n"] for p in parts) == direct.size
    for p, fp in zip(parts, fparts):
        assert p["o_max"] == fp["o_max"] and p["pad_zero"]
        for g in ("dq", "dk", "dv"):
            assert p[g + "_head"] < 1e-6  # float32 rounding of the oracle's own values
